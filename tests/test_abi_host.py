"""Host-side tests of the C ABI: no GPU needed, nothing is launched.

The library must load, export every function include/rkv.h declares, compute
the adaptive split on the host exactly as the oracle does, and reject bad
arguments before touching the device.
"""
import ctypes
import os
import re

import pytest

from oracle import rkv_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rkv():
    from two_stage_kv_snapkv_gb300 import build_lib
    build_lib.build()
    from two_stage_kv_snapkv_gb300 import rkv as mod
    return mod


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "rkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = _declared_functions()
    for n in ("rkv_split_ratio", "rkv_prefill_evict", "rkv_append_page_summary", "rkv_decode_hsa"):
        assert n in names


def test_library_exports_every_declared_symbol(rkv):
    lib = rkv.lib()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared_functions()) <= set(rkv.EXPORTED) | set(_declared_functions())


@pytest.mark.parametrize("L,budget,P,k1o", [
    (4096, 256, 16, 64), (32768, 512, 16, 0), (109000, 256, 16, 0), (65536, 4096, 16, 0),
    (8192, 2048, 32, 0), (32768, 2048, 32, 0), (20000, 2048, 32, 0), (300, 256, 16, 0), (200, 256, 16, 0),
    (1 << 20, 256, 64, 0), (1000, 1000, 16, 0), (999, 7, 16, 0), (5000, 100, 16, 128)])
def test_host_split_matches_oracle(rkv, L, budget, P, k1o):
    a = rkv.rkv_split_ratio(L, budget, 128, P, 32, k1o)
    b = O.split_ratio(L, budget, 128, P, 32, k1o)
    for key in ("keep1", "k1", "k2", "pool_kernel"):
        assert a[key] == b[key], key
    for key in ("c", "r", "c1", "c2"):
        assert a[key] == pytest.approx(b[key], rel=1e-12), key


def test_host_split_pool_kernel_matches_the_workloads(rkv):
    # the C ABI's default pooling kernel reproduces the sizes the benchmark workloads fix
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pool_kernel_workloads.json")))
    for c in g["cases"]:
        s = rkv.rkv_split_ratio(c["prompt_len"], c["budget"], 128, c["page_size"], 32, 0)
        assert s["pool_kernel"] == c["pool_kernel"], c["workload"]
        if "k1" in c:
            assert s["k1"] == c["k1"], c["workload"]


def test_split_rejects_bad_sizes(rkv):
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_split_ratio(0, 256)
    assert e.value.status == rkv.RKV_ERR_INVALID_ARG


def _fake_cache(rkv, **kw):
    base = dict(k_pages=0x10000, v_pages=0x20000, page_table=0x30000, seq_len=0x40000, kmax=0x50000,
                kmin=0x60000, error_word=0x70000, B=2, Hkv=2, head_dim=128, page_size=16, max_pages=64,
                num_phys_pages=128)
    base.update(kw)
    return rkv.RkvCacheStruct(**base)


def _decode_call(rkv, cache, Hq=8, k1=(64, 64), k2=(4, 4), ws_bytes=None, q=0x80000, out=0x90000, ws=0xA0000):
    lib = rkv.lib()
    if ws_bytes is None:
        ws_bytes = lib.rkv_decode_workspace_size(cache.B, Hq, cache.Hkv, cache.max_pages)
    i32 = ctypes.c_int32 * len(k1)
    return lib.rkv_decode_hsa(ctypes.byref(cache), ctypes.c_void_p(q), Hq, i32(*k1), i32(*k2), ctypes.c_float(0.088),
                              ctypes.c_void_p(out), None, None, 0, ctypes.c_void_p(ws), ws_bytes, None)


@pytest.mark.parametrize("kw,Hq,k1,k2,expect", [
    (dict(head_dim=64), 8, (64, 64), (4, 4), "UNSUPPORTED"),
    (dict(page_size=8), 8, (64, 64), (4, 4), "UNSUPPORTED"),
    (dict(max_pages=60), 8, (64, 64), (4, 4), "INVALID_ARG"),
    (dict(kmax=0x50004), 8, (64, 64), (4, 4), "INVALID_ARG"),
    (dict(error_word=0), 8, (64, 64), (4, 4), "INVALID_ARG"),
    (dict(), 6, (64, 64), (4, 4), "UNSUPPORTED"),       # group size 3
    (dict(), 7, (64, 64), (4, 4), "INVALID_ARG"),       # not a multiple of Hkv
    (dict(), 8, (0, 64), (4, 4), "INVALID_ARG"),
    (dict(), 8, (64, 129), (4, 4), "INVALID_ARG"),
    (dict(), 8, (64, 64), (4, 0), "INVALID_ARG"),
])
def test_decode_rejects_bad_arguments_without_launching(rkv, kw, Hq, k1, k2, expect):
    before = rkv.rkv_launch_count()
    st = _decode_call(rkv, _fake_cache(rkv, **kw), Hq=Hq, k1=k1, k2=k2)
    assert st == getattr(rkv, "RKV_ERR_" + expect), rkv.rkv_last_error()
    assert rkv.rkv_last_error()
    assert rkv.rkv_launch_count() == before


def test_decode_rejects_small_workspace(rkv):
    cache = _fake_cache(rkv)
    need = rkv.lib().rkv_decode_workspace_size(2, 8, 2, 64)
    assert _decode_call(rkv, cache, ws_bytes=need - 1) == rkv.RKV_ERR_WORKSPACE


def test_prefill_rejects_bad_arguments_without_launching(rkv):
    lib = rkv.lib()
    cache = _fake_cache(rkv)
    i32 = ctypes.c_int32 * 2
    ws_need = lib.rkv_prefill_workspace_size(2, 8, 2, 32, 1024)

    def call(L=(1024, 900), keep=(200, 200), kp=(7, 7), w=32, Hq=8, stride=256, ws=ws_need, pooled=None):
        return lib.rkv_prefill_evict(ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000), ctypes.c_void_p(0x300000),
                                     2, Hq, w, 1024, i32(*L), i32(*keep), i32(*kp), ctypes.c_float(0.088),
                                     ctypes.byref(cache), ctypes.c_void_p(0x400000), stride,
                                     pooled, ctypes.c_void_p(0x500000), ws, None)

    before = rkv.rkv_launch_count()
    assert call(L=(1025, 900)) == rkv.RKV_ERR_INVALID_ARG          # longer than max_prompt_len
    assert call(keep=(20, 200)) == rkv.RKV_ERR_INVALID_ARG         # keep1 < window
    assert call(keep=(200, 901)) == rkv.RKV_ERR_INVALID_ARG        # keep1 > prompt
    assert call(kp=(6, 7)) == rkv.RKV_ERR_INVALID_ARG              # even pooling kernel
    assert call(kp=(257, 7)) == rkv.RKV_ERR_INVALID_ARG
    assert call(w=33) == rkv.RKV_ERR_UNSUPPORTED                   # G*w > 128
    assert call(stride=100) == rkv.RKV_ERR_INVALID_ARG             # kept_stride < keep1
    assert call(ws=ws_need - 16) == rkv.RKV_ERR_WORKSPACE
    assert call(keep=(1025, 200), L=(1024, 900)) == rkv.RKV_ERR_INVALID_ARG
    assert call(pooled=ctypes.c_void_p(0x600004)) == rkv.RKV_ERR_INVALID_ARG   # misaligned
    # capacity: 64 pages x 16 tokens = 1024 >= keep1, so only the launch would be left
    assert rkv.rkv_launch_count() == before


def test_append_rejects_bad_arguments(rkv):
    lib = rkv.lib()
    cache = _fake_cache(rkv)
    assert lib.rkv_append_page_summary(ctypes.byref(cache), None, None, 0, None) == rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_append_page_summary(ctypes.byref(cache), ctypes.c_void_p(0x1000), None, 1, None) == \
        rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_append_page_summary(ctypes.byref(cache), None, None, 64 * 16 + 1, None) == rkv.RKV_ERR_INVALID_ARG


def test_recall_rejects_bad_arguments_without_launching(rkv):
    """The recall diagnostic validates on the host: nothing launches on a bad call."""
    import ctypes
    c = rkv.RkvCacheStruct()
    c.B, c.Hkv, c.head_dim, c.page_size, c.max_pages, c.num_phys_pages = 1, 1, 128, 16, 8, 8
    fake = ctypes.c_void_p(4096)
    for name in ("k_pages", "v_pages", "page_table", "seq_len", "kmax", "kmin", "error_word", "step_sync"):
        setattr(c, name, fake)
    n0 = rkv.rkv_launch_count()
    kt = (ctypes.c_int32 * 1)(16)
    # Hq not a multiple of Hkv... group of 3
    st = rkv.lib().rkv_exact_topk_recall(ctypes.byref(c), fake, 3, fake, 4, kt, 0.088, fake, fake, None)
    assert st == rkv.RKV_ERR_UNSUPPORTED
    # NULL recall output
    st = rkv.lib().rkv_exact_topk_recall(ctypes.byref(c), fake, 4, fake, 4, kt, 0.088, None, None, None)
    assert st == rkv.RKV_ERR_INVALID_ARG and "NULL" in rkv.rkv_last_error()
    # negative token budget
    kt[0] = -1
    st = rkv.lib().rkv_exact_topk_recall(ctypes.byref(c), fake, 4, fake, 4, kt, 0.088, fake, fake, None)
    assert st == rkv.RKV_ERR_INVALID_ARG
    assert rkv.rkv_launch_count() == n0


@pytest.mark.parametrize("L,budget,P", [(32768, 512, 16), (8192, 2048, 32), (100, 256, 16), (109000, 256, 16)])
def test_host_split_mt_matches_oracle(rkv, L, budget, P):
    from oracle import rkv_oracle as O
    got = rkv.rkv_split_ratio_mt(L, budget, 128, P)
    ref = O.split_ratio_mt(L, budget, 128, P)
    for key in ("keep1", "k1", "k2", "pool_kernel"):
        assert got[key] == ref[key], key
    for key in ("c", "r", "c1", "c2"):
        assert abs(got[key] - ref[key]) <= 1e-12 * max(1.0, abs(ref[key])), key


def test_prefill_chunk_rejects_bad_arguments_without_launching(rkv):
    lib = rkv.lib()
    cache = _fake_cache(rkv)
    i32 = ctypes.c_int32 * 2

    def call(m=(300, 100), held=(0, 0), keep=(200, 200), kp=(7, 7), w=32, Hq=8, stride=256, chunk_max=512,
             ws=None):
        if ws is None:
            total = max(h + c for h, c in zip(held, m))
            ws = lib.rkv_prefill_chunk_workspace_size(2, Hq, 2, w, total)
        return lib.rkv_prefill_chunk(ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000), ctypes.c_void_p(0x300000),
                                     2, Hq, w, chunk_max, i32(*m), i32(*held), i32(*keep), i32(*kp),
                                     ctypes.c_float(0.088), ctypes.byref(cache), ctypes.c_void_p(0x400000), stride,
                                     ctypes.c_void_p(0x500000), ws, None)

    before = rkv.rkv_launch_count()
    assert call(m=(20, 100)) == rkv.RKV_ERR_INVALID_ARG             # chunk shorter than the window
    assert call(m=(513, 100)) == rkv.RKV_ERR_INVALID_ARG            # longer than chunk_max
    assert call(held=(-1, 0)) == rkv.RKV_ERR_INVALID_ARG            # negative held length
    assert call(held=(1025, 0)) == rkv.RKV_ERR_INVALID_ARG          # more held than the pages hold
    assert call(keep=(20, 200)) == rkv.RKV_ERR_INVALID_ARG          # keep1 < window
    assert call(keep=(2000, 200), held=(1000, 0)) == rkv.RKV_ERR_INVALID_ARG   # survivors beyond capacity
    assert call(stride=150) == rkv.RKV_ERR_INVALID_ARG              # kept_stride < min(keep1, held + chunk)
    assert call(kp=(8, 7)) == rkv.RKV_ERR_INVALID_ARG               # even pooling kernel
    assert call(w=33) == rkv.RKV_ERR_UNSUPPORTED                    # G*w > 128
    need = lib.rkv_prefill_chunk_workspace_size(2, 8, 2, 32, 300)
    assert call(ws=need - 16) == rkv.RKV_ERR_WORKSPACE
    # the chunked workspace adds the gathered K and V to the single-shot one
    assert lib.rkv_prefill_chunk_workspace_size(2, 8, 2, 32, 300) > lib.rkv_prefill_workspace_size(2, 8, 2, 32, 300)
    assert rkv.rkv_launch_count() == before


def test_sparq_rejects_bad_arguments_without_launching(rkv):
    lib = rkv.lib()
    i32 = ctypes.c_int32 * 2

    def call(cache=None, k1=(32, 32), kt=(64, 64), stride=0, ws=None, sel=None, keys=None, keys_bytes=0):
        cache = cache or _fake_cache(rkv)
        if ws is None:
            ws = lib.rkv_sparq_workspace_size(2, 8, 2, cache.max_pages, cache.page_size)
        return lib.rkv_decode_sparq(ctypes.byref(cache), ctypes.c_void_p(0x80000), 8, i32(*k1), i32(*kt),
                                    ctypes.c_float(0.088), ctypes.c_void_p(0x90000), None, sel, stride,
                                    keys, keys_bytes, ctypes.c_void_p(0xA0000), ws, None)

    before = rkv.rkv_launch_count()
    assert call(k1=(0, 32)) == rkv.RKV_ERR_INVALID_ARG
    assert call(k1=(129, 32)) == rkv.RKV_ERR_INVALID_ARG
    assert call(kt=(0, 64)) == rkv.RKV_ERR_INVALID_ARG
    assert call(sel=ctypes.c_void_p(0xB0000), stride=63) == rkv.RKV_ERR_INVALID_ARG
    assert call(ws=16) == rkv.RKV_ERR_WORKSPACE
    assert call(cache=_fake_cache(rkv, max_pages=4096, num_phys_pages=8192)) == rkv.RKV_ERR_UNSUPPORTED  # 64K tokens
    assert call(cache=_fake_cache(rkv, page_size=8)) == rkv.RKV_ERR_UNSUPPORTED
    # the channel-major key copy: too small, or misaligned
    c = _fake_cache(rkv)
    need = lib.rkv_sparq_keys_size(2, 2, c.max_pages, c.page_size)
    assert call(keys=ctypes.c_void_p(0xC0000), keys_bytes=need - 1) == rkv.RKV_ERR_WORKSPACE
    assert call(keys=ctypes.c_void_p(0xC0008), keys_bytes=need) == rkv.RKV_ERR_INVALID_ARG
    assert rkv.rkv_launch_count() == before


def test_sparq_keys_size_is_the_record_and_a_block_per_unit(rkv):
    """[B*Hkv] int32 lengths padded to 256 bytes, then [B*Hkv][128][max_pages*P] bf16."""
    lib = rkv.lib()
    for B, Hkv, mp, P in ((1, 2, 8, 16), (16, 8, 304, 32), (64, 8, 16384, 64)):
        units = B * Hkv
        assert lib.rkv_sparq_keys_size(B, Hkv, mp, P) == (units * 4 + 255) // 256 * 256 + units * 128 * mp * P * 2
    assert lib.rkv_sparq_keys_size(0, 2, 8, 16) == 0


def test_decode_step_host_rejects_bad_arguments_without_launching(rkv):
    lib = rkv.lib()
    cache = _fake_cache(rkv, step_sync=0x78000)
    i32 = ctypes.c_int32 * 2
    need = lib.rkv_step_host_staging_size(2, 8, 2)
    ws = lib.rkv_decode_workspace_size(2, 8, 2, cache.max_pages)

    def call(staging=0xC0000, nbytes=need, host_in=0xD0000, k1=(32, 32)):
        return lib.rkv_decode_step_host(ctypes.byref(cache), ctypes.c_void_p(host_in), ctypes.c_void_p(0xE0000), 8,
                                        i32(*k1), i32(4, 4), ctypes.c_float(0.088), ctypes.c_void_p(staging), nbytes,
                                        ctypes.c_void_p(0xA0000), ws, None)

    before = rkv.rkv_launch_count()
    assert need == 2 * (8 + 4) * 128 * 2 + 2 * 8 * 128 * 4   # the packed inputs (256-aligned), then out
    assert call(nbytes=need - 1) == rkv.RKV_ERR_WORKSPACE
    assert call(staging=0xC0008) == rkv.RKV_ERR_INVALID_ARG
    assert call(host_in=0) == rkv.RKV_ERR_INVALID_ARG
    assert call(k1=(0, 32)) == rkv.RKV_ERR_INVALID_ARG
    assert rkv.rkv_launch_count() == before


def test_page_pools_too_large_for_32_bit_rows_are_rejected(rkv):
    cache = _fake_cache(rkv, num_phys_pages=1 << 22, Hkv=8, page_size=64)   # 2^31 rows
    assert _decode_call(rkv, cache) == rkv.RKV_ERR_UNSUPPORTED
