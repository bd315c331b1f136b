"""The allocation-free decode entry point (rkv_decode_hsa_noalloc).

It serves callers that cannot allocate device memory when they call, such as a
plug-in inside an engine that owns all device memory, or a latency-critical loop
that must never reach cudaMalloc.  It must give the same results as
rkv_decode_hsa with a caller workspace, call after call, while sharing one
built-in scratch array, and must refuse caches too large for that array.

This file is named to be collected last, so a run that stops at the first failure
has run every other test before it.
"""
import ctypes

import pytest
import torch

from two_stage_kv_snapkv_gb300 import workloads as W

from rkv_check import ATOL_OUT, DeviceRun

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from two_stage_kv_snapkv_gb300 import build_lib
    build_lib.build()
    from two_stage_kv_snapkv_gb300 import rkv as mod
    return mod


def _noalloc(rkv, cache, q, k1, k2, out, ch, pg):
    lib = rkv.lib()
    i32 = ctypes.c_int32 * len(k1)
    return lib.rkv_decode_hsa_noalloc(ctypes.byref(cache.struct), ctypes.c_void_p(q.data_ptr()), q.shape[1],
                                      i32(*k1), i32(*k2), ctypes.c_float(1.0 / 128 ** 0.5),
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ch.data_ptr()),
                                      ctypes.c_void_p(pg.data_ptr()), pg.shape[-1],
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_decode_two_calls(rkv):
    # the four-kernel path is the one that keeps its scratch in the workspace
    old = rkv.rkv_decode_path(1)
    try:
        _compare_two_calls(rkv)
    finally:
        rkv.rkv_decode_path(old)


def _compare_two_calls(rkv):
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.prefill()
    dev = run.dev
    for step in range(2):   # two calls in a row share the same scratch
        d = W.decode_tensors(wl, step, run.seed, 0, dev)
        rkv.rkv_append_page_summary(run.cache, d["k_new"].unsqueeze(2).contiguous(),
                                    d["v_new"].unsqueeze(2).contiguous(), 1)
        outs = []
        for use_noalloc in (False, True):
            out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device=dev)
            ch = torch.full((wl.B, wl.Hkv, 128), -9, dtype=torch.int32, device=dev)
            pg = torch.full((wl.B, wl.Hkv, max(run.k2) + 1), -9, dtype=torch.int32, device=dev)
            if use_noalloc:
                st = _noalloc(rkv, run.cache, d["q"], run.k1, run.k2, out, ch, pg)
                assert st == rkv.RKV_OK, rkv.rkv_last_error()
            else:
                rkv.rkv_decode_hsa(run.cache, d["q"], run.k1, run.k2, out, sel_channels=ch, sel_pages=pg,
                                   workspace=run.dws)
            outs.append((out, ch, pg))
        torch.cuda.synchronize()
        (o1, c1, p1), (o2, c2, p2) = outs
        assert torch.equal(c1, c2) and torch.equal(p1, p2)
        assert torch.isfinite(o2).all()
        assert float((o1 - o2).abs().max()) <= ATOL_OUT
    st, bits = run.status()
    assert st == rkv.RKV_OK, bits


def test_noalloc_rejects_caches_beyond_its_scratch(rkv):
    # 256 sequences x 8 query heads need 2048 x 64 split partials of 512 B: > 32 MiB.
    # The cache, query and output are real (small) device allocations, so even if the
    # size check ever let this call through, no kernel would touch unmapped memory.
    lib = rkv.lib()
    B, Hq, Hkv, max_pages = 256, 8, 1, 64
    need = lib.rkv_decode_workspace_size(B, Hq, Hkv, max_pages)
    if need <= 32 << 20:
        pytest.fail(f"this case no longer exceeds the 32 MiB scratch ({need} bytes); pick a larger one")
    dev = torch.device("cuda")
    cache = rkv.PagedCache(B, Hkv, 16, max_pages, dev, fill=0.0)
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device=dev)
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device=dev)
    k = (ctypes.c_int32 * B)(*([32] * B))
    torch.cuda.synchronize()
    before = rkv.rkv_launch_count()
    st = lib.rkv_decode_hsa_noalloc(ctypes.byref(cache.struct), ctypes.c_void_p(q.data_ptr()), Hq, k, k,
                                    ctypes.c_float(0.088), ctypes.c_void_p(out.data_ptr()), None, None, 0,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == rkv.RKV_ERR_WORKSPACE
    assert "32 MiB" in rkv.rkv_last_error()
    assert rkv.rkv_launch_count() == before
