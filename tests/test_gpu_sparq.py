"""GPU parity of the SparQ-only step (rkv_decode_sparq: HSA with one-token pages)
against the oracle's sparq_decode_unit, on caches built by the stage-1 prefill.

Channel and token sets are exact up to the fp32 tie band; the attention output is
compared with the oracle evaluated on the GPU's token set (max-abs 2e-3)."""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from two_stage_kv_snapkv_gb300 import workloads as W

from rkv_check import ATOL_OUT, DeviceRun, OracleUnit, check_topk, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from two_stage_kv_snapkv_gb300 import build_lib
    build_lib.build()
    from two_stage_kv_snapkv_gb300 import rkv as mod
    return mod


def _keys_block(rkv, run, keys_t, b, g):
    """[128][n] channel-major view of unit (b, g) in the key copy (float64 on the CPU)."""
    units = run.cache.B * run.cache.Hkv
    cap = run.cache.max_pages * run.cache.page_size
    off = (units * 4 + 255) // 256 * 256
    blk = keys_t[off:].view(torch.bfloat16).view(units, 128, cap)
    return f64(blk[b * run.cache.Hkv + g])


def _sparq_steps(rkv, wl, k_tokens, units=None, steps=None, seed=0x5EED, gen_device="cpu", tail="nan",
                 keys_t=False):
    run = DeviceRun(wl, rkv, seed=seed, gen_device=gen_device, tail=tail)
    run.prefill()
    if units is None:
        units = [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    checks = [OracleUnit(run, b, g) for b, g in units]
    for u in checks:
        u.check_prefill(run)
    G = wl.G
    ws = rkv.sparq_workspace(wl.B, wl.Hq, wl.Hkv, run.cache.max_pages, wl.page_size)
    stride = max(k_tokens) + 1
    kt = rkv.sparq_keys(run.cache, run.dev) if keys_t else None
    errs = []
    for step in range(wl.steps if steps is None else steps):
        d = W.decode_tensors(wl, step, seed, 0, run.dev)
        rkv.rkv_append_page_summary(run.cache, d["k_new"].unsqueeze(2).contiguous(),
                                    d["v_new"].unsqueeze(2).contiguous(), 1)
        out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device=run.dev)
        ch = torch.full((wl.B, wl.Hkv, 128), -9, dtype=torch.int32, device=run.dev)
        tk = torch.full((wl.B, wl.Hkv, stride), -9, dtype=torch.int32, device=run.dev)
        rkv.rkv_decode_sparq(run.cache, d["q"], run.k1, k_tokens, out, sel_channels=ch, sel_tokens=tk, workspace=ws,
                             keys_t=kt)
        for u in checks:
            b, g = u.b, u.g
            u.Kc = np.concatenate([u.Kc[: u.n], f64(d["k_new"][b, g])[None]])
            u.Vc = np.concatenate([u.Vc[: u.n], f64(d["v_new"][b, g])[None]])
            u.n += 1
            qg = f64(d["q"][b, g * G:(g + 1) * G])
            k1 = run.k1[b]
            gch = ch[b, g, :k1].cpu().numpy()
            check_topk(gch, O.channel_select(qg, k1)[1], k1, what="channel set")
            gch = np.sort(gch)
            # the token scores on the GPU's channel set, then the token set
            sig = O.page_scores(qg, *O.page_summaries(u.Kc, u.n, 1), gch)
            kk = min(k_tokens[b], u.n)
            got = tk[b, g, :kk].cpu().numpy().astype(np.int64)
            assert np.all(np.diff(got) > 0), "token list not ascending"
            if kk < stride:
                assert int(tk[b, g, kk].item()) == -1
            check_topk(got, sig, kk, what="token set")
            ref = O.sparq_decode_unit(qg, u.Kc, u.Vc, u.n, k1, k_tokens[b], tokens_override=got)["out"]
            err = float(np.abs(f64(out[b, g * G:(g + 1) * G]) - ref).max())
            errs.append(err)
            assert err <= ATOL_OUT, f"attention max-abs error {err}"
            if kt is not None:  # the copy holds every cached key, bit for bit
                np.testing.assert_array_equal(_keys_block(rkv, run, kt, b, g)[:, :u.n].T, u.Kc[:u.n])
    st, bits = run.status()
    assert st == rkv.RKV_OK, bits
    return max(errs)


SMALL = {
    "gqa4_ragged": (W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16,
                             steps=6, pool_kernel=5), [64, 100]),
    "gqa1_p32": (W.custom(B=1, Hq=2, Hkv=2, prompt_lens=[513], budget=48, window=16, page_size=32, steps=4,
                          pool_kernel=3), [37]),
    "gqa8_few_tokens": (W.custom(B=1, Hq=8, Hkv=1, prompt_lens=[900], budget=80, window=16, page_size=16, steps=3,
                                 pool_kernel=9), [5]),
    "needles": (W.custom(B=1, Hq=8, Hkv=2, prompt_lens=[3000], budget=128, window=32, page_size=16, steps=3,
                         pool_kernel=7, needles_per_head=2), [128]),
}


@pytest.mark.parametrize("keys_t", [False, True], ids=["rows", "keys_t"])
@pytest.mark.parametrize("name", list(SMALL))
def test_sparq_small(rkv, name, keys_t):
    wl, kt = SMALL[name]
    _sparq_steps(rkv, wl, kt, keys_t=keys_t)


def test_sparq_keys_copy_restarts_when_its_record_is_ahead(rkv):
    """A record above the cache's length (the cache was refilled shorter) makes the
    next call copy every position again; a zeroed copy is rebuilt the same way."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.prefill()
    kt = rkv.sparq_keys(run.cache, run.dev)
    units = wl.B * wl.Hkv
    cap = run.cache.max_pages * wl.page_size
    d = W.decode_tensors(wl, 0, run.seed, 0, run.dev)
    out = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device=run.dev)
    rkv.rkv_decode_sparq(run.cache, d["q"], run.k1, [64, 64], out, keys_t=kt)
    n = run.cache.seq_len.cpu().numpy()
    rec = kt[:units * 4].view(torch.int32)
    assert rec.cpu().tolist() == [int(n[u // wl.Hkv]) for u in range(units)]
    ref = kt.clone()
    # scramble the block and push every record past the end: the next call recopies all
    off = (units * 4 + 255) // 256 * 256
    kt[off:] = 0x55
    rec.fill_(cap)
    rkv.rkv_decode_sparq(run.cache, d["q"], run.k1, [64, 64], out, keys_t=kt)
    for b in range(wl.B):
        for g in range(wl.Hkv):
            nb = int(n[b])
            np.testing.assert_array_equal(_keys_block(rkv, run, kt, b, g)[:, :nb], _keys_block(rkv, run, ref, b, g)[:, :nb])
    assert rec.cpu().tolist() == [int(n[u // wl.Hkv]) for u in range(units)]
    assert run.status()[0] == rkv.RKV_OK


def test_sparq_every_token_is_dense_attention(rkv):
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[300, 420], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    assert _sparq_steps(rkv, wl, [5000, 5000]) <= ATOL_OUT


def test_sparq_ties_go_to_lower_tokens(rkv):
    """Every prompt key is the same vector, so all but the appended tokens tie."""
    wl = W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[800], budget=64, window=8, page_size=16, steps=2, pool_kernel=3)
    run = DeviceRun(wl, rkv)
    k = run.inputs["k"]
    k[0, :, :800] = k[0, :, :1].clone()
    run.gpu_in["k"] = k.to(run.dev)
    run.prefill()
    u = OracleUnit(run, 0, 0)
    u.check_prefill(run)
    d = W.decode_tensors(wl, 0, 0x5EED, 0, run.dev)
    rkv.rkv_append_page_summary(run.cache, d["k_new"].unsqueeze(2).contiguous(), d["v_new"].unsqueeze(2).contiguous(),
                                1)
    out = torch.empty((1, 4, 128), dtype=torch.float32, device=run.dev)
    tk = torch.full((1, 1, 41), -9, dtype=torch.int32, device=run.dev)
    rkv.rkv_decode_sparq(run.cache, d["q"], run.k1, [40], out, sel_tokens=tk)
    got = tk[0, 0, :40].cpu().numpy()
    Kc = np.concatenate([u.Kc, f64(d["k_new"][0, 0])[None]])
    qg = f64(d["q"][0])
    res = O.sparq_decode_unit(qg, Kc, Kc, u.n + 1, run.k1[0], 40)
    np.testing.assert_array_equal(got, res["pages"])
    assert run.status()[0] == rkv.RKV_OK


def test_sparq_workload2_sampled(rkv):
    """Workload 2 at full size: 32K prompt, the same token budget as HSA (k2 x P)."""
    wl = W.workload(2)
    wl.steps = 3
    _sparq_steps(rkv, wl, [512], units=[(0, 0), (0, 6)], gen_device="cuda", tail="zero")


def test_sparq_workload2_keys_t_sampled(rkv):
    wl = W.workload(2)
    wl.steps = 3
    _sparq_steps(rkv, wl, [512], units=[(0, 1), (0, 7)], gen_device="cuda", tail="zero", keys_t=True)


def test_sparq_workload4_sampled(rkv):
    wl = W.workload(4)
    wl.steps = 2
    longest = int(np.argmax(wl.prompt_lens))
    _sparq_steps(rkv, wl, [2048] * wl.B, units=[(longest, 3), (0, 0)], gen_device="cuda", tail="zero")


def test_sparq_workload4_keys_t_sampled(rkv):
    wl = W.workload(4)
    wl.steps = 2
    longest = int(np.argmax(wl.prompt_lens))
    _sparq_steps(rkv, wl, [2048] * wl.B, units=[(longest, 5), (3, 2)], gen_device="cuda", tail="zero", keys_t=True)
