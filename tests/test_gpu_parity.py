"""GPU parity: librkv against the CPU oracle on the same seeded inputs.

Small cases run the whole path (prefill, every decode step) unit by unit; the
full-size workloads run in the launch configuration the bench uses and are
checked on sampled (sequence, KV head) units.
"""

import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from two_stage_kv_snapkv_gb300 import workloads as W

from rkv_check import ATOL_OUT, DeviceRun, OracleUnit, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from two_stage_kv_snapkv_gb300 import build_lib
    build_lib.build()
    from two_stage_kv_snapkv_gb300 import rkv as mod
    return mod


SMALL = {
    # several tiles and a ragged tail, GQA 4, two sequences of different length
    "gqa4_ragged": W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16,
                            steps=20, pool_kernel=5),
    "gqa1": W.custom(B=1, Hq=2, Hkv=2, prompt_lens=[513], budget=48, window=16, page_size=16, steps=6,
                     pool_kernel=3),
    "gqa8_w16": W.custom(B=1, Hq=8, Hkv=1, prompt_lens=[900], budget=80, window=16, page_size=16, steps=5,
                         pool_kernel=9),
    "gqa2_p32": W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[1200, 333], budget=96, window=8, page_size=32, steps=40,
                         pool_kernel=7),
    "p64_outliers": W.custom(B=1, Hq=8, Hkv=2, prompt_lens=[2000], budget=128, window=32, page_size=64, steps=70,
                             pool_kernel=15, outlier_channels=4, sinks=4),
    "w1_kernel1": W.custom(B=1, Hq=1, Hkv=1, prompt_lens=[300], budget=40, window=1, page_size=16, steps=3,
                           pool_kernel=1),
    "no_eviction": W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[100], budget=256, window=8, page_size=16, steps=4,
                            pool_kernel=3),
    "prompt_equals_window": W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[16, 40], budget=8, window=16, page_size=16,
                                     steps=3, pool_kernel=3),
    "needles": W.custom(B=1, Hq=8, Hkv=2, prompt_lens=[3000], budget=128, window=32, page_size=16, steps=8,
                        pool_kernel=7, needles_per_head=2),
    "k1_small": W.custom(B=3, Hq=8, Hkv=2, prompt_lens=[640, 1500, 64], budget=64, window=8, page_size=16,
                         steps=10, pool_kernel=5, k1=16),
}


@pytest.fixture(params=["fused", "split"])
def path(rkv, request):
    """Run a test on each decode implementation (one fused launch / four kernels)."""
    old = rkv.rkv_decode_path(-1)
    rkv.rkv_decode_path(2 if request.param == "fused" else 1)
    yield request.param
    rkv.rkv_decode_path(old)


def _run_small(rkv, wl, check_every=1, api="step"):
    run = DeviceRun(wl, rkv, api=api)
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
        u.check_cache(run)
    errs = []
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            errs.append(u.step(run, d, out, ch, pg, check_cache=(step % check_every == 0))["err"])
    st, bits = run.status()
    assert st == rkv.RKV_OK, (st, bits)
    return max(errs) if errs else 0.0


@pytest.mark.parametrize("api", ["step", "separate"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_end_to_end(rkv, path, name, api):
    err = _run_small(rkv, SMALL[name], api=api)
    assert err <= ATOL_OUT


def test_tiny_workload_end_to_end(rkv, path):
    """Workload 1: 4K prompt, GQA 4, needles, 16 decode steps, every step checked."""
    wl = W.workload(1)
    run = DeviceRun(wl, rkv)
    run.prefill()
    units = [OracleUnit(run, 0, g) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
        u.check_cache(run)
    hits = 0
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            u.step(run, d, out, ch, pg, check_cache=True)
    st, _ = run.status()
    assert st == rkv.RKV_OK


def test_full_selection_is_dense_attention(rkv, path):
    """k1 = 128 and k2 >= pages: HSA is exact attention over every cached token."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[600, 450], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.k1 = [128, 128]
    run.k2 = [4096, 4096]
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(2) for g in range(2)]
    for u in units:
        u.check_prefill(run)
    d, out, ch, pg = run.decode_step(0)
    for u in units:
        u.step(run, d, out, ch, pg)
        G = wl.G
        qg = f64(d["q"][u.b, u.g * G:(u.g + 1) * G])
        dense = O.sparse_attention(qg, u.Kc, u.Vc, u.n, np.arange(-(-u.n // 16)), 16)
        np.testing.assert_allclose(f64(out[u.b, u.g * G:(u.g + 1) * G]), dense, atol=ATOL_OUT)


def test_append_equals_rebuild_on_gpu(rkv, path):
    """Incremental appends, then a from-scratch rebuild by the library: bit-identical summaries."""
    wl = W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[600, 600], budget=64, window=8, page_size=16, steps=37,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.prefill()
    for step in range(wl.steps):
        run.decode_step(step)
    c = run.cache
    n = int(c.seq_len[0].item())
    assert c.seq_len.tolist() == [n, n] and n % 16 != 0
    NP = -(-n // 16)
    inc_max, inc_min = c.kmax[..., :NP].clone(), c.kmin[..., :NP].clone()
    c.kmax.fill_(float("nan"))
    c.kmin.fill_(float("nan"))
    c.seq_len.zero_()
    for chunk in (17, 5, n - 22):          # uneven chunks; the tokens are already in their pages
        rkv.rkv_append_page_summary(c, None, None, chunk)
    assert c.seq_len.tolist() == [n, n]
    assert torch.equal(c.kmax[..., :NP], inc_max) and torch.equal(c.kmin[..., :NP], inc_min)
    st, _ = run.status()
    assert st == rkv.RKV_OK


@pytest.mark.parametrize("L", [3000, 700])
def test_prefill_select_with_large_tie_groups(rkv, L):
    """Prompt keys take only two values, so hundreds of scores tie exactly at the top-k
    boundary: the kept set must be exactly the oracle's (ties go to lower positions)."""
    wl = W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[L], budget=128, window=8, page_size=16, steps=1, pool_kernel=1)
    run = DeviceRun(wl, rkv)
    k = run.inputs["k"]
    a, bvec = k[0, 0, 0].clone(), k[0, 0, 1].clone()
    pattern = (torch.arange(L) % 3 == 0)
    k[0, 0, :L][pattern] = a
    k[0, 0, :L][~pattern] = bvec
    run.gpu_in["k"] = k.to(run.dev)
    run.prefill()
    u = OracleUnit(run, 0, 0)
    kept = run.kept[0, 0, : run.keep1[0]].cpu().numpy()
    np.testing.assert_array_equal(kept, u.res["kept"][0])
    assert run.status()[0] == rkv.RKV_OK


@pytest.mark.parametrize("L,budget", [(1500, 256), (3000, 2048), (6000, 4096), (12000, 8192), (20000, 16384)])
def test_decode_select_with_tied_page_scores(rkv, path, L, budget):
    """Every prompt key is the same vector, so every page of the compressed cache but the
    one taking the new tokens has the same Kmax/Kmin and the same bound.  The top-k2
    boundary then falls inside a group of equal scores (about 50, 170, 340, 690 or 1200
    pages: every kind of select the fused step has, from the counting ranks to the
    looping histogram select) and the tied pages must go to the lowest page indices, as
    in the oracle."""
    wl = W.custom(B=1, Hq=8, Hkv=2, prompt_lens=[L], budget=budget, window=16, page_size=16, steps=2,
                  pool_kernel=3)
    run = DeviceRun(wl, rkv)
    k = run.inputs["k"]
    k[0, :, :L] = k[0, :, :1].clone()
    run.gpu_in["k"] = k.to(run.dev)
    run.prefill()
    units = [OracleUnit(run, 0, g) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            r = u.step(run, d, out, ch, pg)
            sig, kk = r["sig"], len(r["pages"])
            desc = np.sort(sig)[::-1]
            assert kk < len(sig) and desc[kk - 1] == desc[kk], "no tie at the boundary"
            ref = np.sort(np.lexsort((np.arange(len(sig)), -sig))[:kk])
            np.testing.assert_array_equal(r["pages"], ref)
    assert run.status()[0] == rkv.RKV_OK


def test_channel_ties_go_to_lower_channels(rkv, path):
    """Every channel of the decode query has the same magnitude (signs vary), so all
    128 channel scores tie exactly: the channel set must be channels 0 .. k1-1."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 900], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)

    def flat_q(d):
        d["q"] = torch.where(d["q"] >= 0, 0.75, -0.75).to(d["q"].dtype)

    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step, edit=flat_q)
        for u in units:
            u.step(run, d, out, ch, pg)
            k1 = run.k1[u.b]
            np.testing.assert_array_equal(ch[u.b, u.g, :k1].cpu().numpy(), np.arange(k1))
    assert run.status()[0] == rkv.RKV_OK


def test_channel_scores_beyond_fp32_are_ranked_exactly(rkv, path):
    """In every channel one query head of a group holds 1.0 and the other 2^-30 (1 + c % 7):
    the fp32 sums all round to 1.0, so the channels are ranked on their exact (fp64)
    sums, as the oracle ranks them: the k1 chosen channels are those with the largest
    c % 7, ties to the lower channel."""
    wl = W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[700, 900], budget=64, window=8, page_size=16, steps=2,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
    tiny = torch.tensor([2.0 ** -30 * (1 + c % 7) for c in range(128)])

    def split_q(d):
        q = torch.empty_like(d["q"])
        q[:, 0::2] = 1.0
        q[:, 1::2] = tiny.to(q.dtype).to(q.device)
        d["q"] = q

    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step, edit=split_q)
        for u in units:
            u.step(run, d, out, ch, pg)
            k1 = run.k1[u.b]
            want = sorted(sorted(range(128), key=lambda c: (-(c % 7), c))[:k1])
            np.testing.assert_array_equal(ch[u.b, u.g, :k1].cpu().numpy(), np.array(want))
    assert run.status()[0] == rkv.RKV_OK


def test_deterministic(rkv, path):
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[900, 700], budget=64, window=8, page_size=16, steps=3,
                  pool_kernel=5)
    outs = []
    for _ in range(2):
        run = DeviceRun(wl, rkv)
        run.prefill()
        res = [run.kept.clone(), run.pooled.clone()]
        for s in range(wl.steps):
            d, out, ch, pg = run.decode_step(s)
            res += [out.clone(), pg.clone()]
        outs.append(res)
    for a, b in zip(*outs):
        assert torch.equal(a.nan_to_num(), b.nan_to_num())


def test_long_slices_with_few_pages(rkv, path):
    """A page capacity of 1024 makes every launch take the long-slice kernel (chosen
    channels staged after the select, the histogram top-k2) while the sequences hold
    40-70 pages: short slices and small page counts through that kernel, every unit
    checked against the oracle at every step."""
    wl = W.custom(B=4, Hq=8, Hkv=2, prompt_lens=[3000, 2200, 1500, 700], budget=256, window=8, page_size=16,
                  steps=4, pool_kernel=7)
    run = DeviceRun(wl, rkv, max_pages_req=1024)
    assert run.cache.max_pages >= 1024
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            assert u.step(run, d, out, ch, pg, check_cache=True)["err"] <= ATOL_OUT
    assert run.status()[0] == rkv.RKV_OK
    assert max(run.k2) < min((k + wl.steps) // wl.page_size for k in run.keep1)   # a real page selection


def test_decode_loop_graph_matches_eager(rkv, path):
    """Every decode step of two layers captured as one CUDA graph (as the bench replays
    the decode loop; the fused steps chained by programmatic launch, each step of a
    layer reading the cache the previous one appended to) gives the eager results bit
    for bit: outputs, selections and the cache with its summaries."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16, steps=12,
                  pool_kernel=5)

    def setup():
        runs = [DeviceRun(wl, rkv, layer=layer) for layer in range(2)]
        for r in runs:
            r.prefill()
        ins = [[W.decode_tensors(wl, t, r.seed, r.layer, r.dev) for t in range(wl.steps)] for r in runs]
        outs = [[(torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device=r.dev),
                  torch.full((wl.B, wl.Hkv, 128), -9, dtype=torch.int32, device=r.dev),
                  torch.full((wl.B, wl.Hkv, max(r.k2) + 1), -9, dtype=torch.int32, device=r.dev))
                 for _ in range(wl.steps)] for r in runs]
        torch.cuda.synchronize()
        return runs, ins, outs

    def loop(runs, ins, outs):
        for t in range(wl.steps):
            for r, i, o in zip(runs, ins, outs):
                d = i[t]
                rkv.rkv_decode_step(r.cache, d["q"], d["k_new"], d["v_new"], r.k1, r.k2, o[t][0],
                                    sel_channels=o[t][1], sel_pages=o[t][2], workspace=r.dws)

    eager = setup()
    loop(*eager)
    torch.cuda.synchronize()

    graph = setup()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        loop(*graph)
    g.replay()
    torch.cuda.synchronize()

    def bits(t):   # bitwise view: NaN fills compare equal to themselves
        return t.view({torch.bfloat16: torch.int16, torch.float32: torch.int32}.get(t.dtype, t.dtype))

    for re, rg in zip(eager[0], graph[0]):
        assert re.status()[0] == rkv.RKV_OK and rg.status()[0] == rkv.RKV_OK
        for name in ("k_pages", "v_pages", "kmax", "kmin", "seq_len"):
            assert torch.equal(bits(getattr(re.cache, name)), bits(getattr(rg.cache, name))), name
    for oe, og in zip(eager[2], graph[2]):
        for t, (te, tg) in enumerate(zip(oe, og)):
            for a, b in zip(te, tg):
                assert torch.equal(bits(a), bits(b)), t


def test_bad_page_id_is_flagged_not_faulted(rkv, path):
    wl = W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[400], budget=64, window=8, page_size=16, steps=1, pool_kernel=3)
    run = DeviceRun(wl, rkv)
    run.prefill()
    assert run.status()[0] == rkv.RKV_OK
    run.k2 = [1000]        # every page is attended, so the bad entry is used
    run.cache.page_table[0, 1] = run.cache.num_phys_pages + 7
    run.decode_step(0)
    st, bits = run.status()
    assert st == rkv.RKV_ERR_DEVICE_DATA and bits & rkv.DEVERR_PAGE_ID
    assert run.status() == (rkv.RKV_OK, 0)   # the word was cleared


def test_capacity_overflow_is_flagged(rkv, path):
    wl = W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[400], budget=64, window=8, page_size=16, steps=1, pool_kernel=3)
    run = DeviceRun(wl, rkv)
    run.prefill()
    cap = run.cache.max_pages * 16
    run.cache.seq_len.fill_(cap)
    d, out, ch, pg = run.decode_step(0)        # the append does not fit: flagged, length kept
    st, bits = run.status()
    assert st == rkv.RKV_ERR_DEVICE_DATA and bits & rkv.DEVERR_CAPACITY
    assert int(run.cache.seq_len[0].item()) == cap


def test_bounded_wait_runs_out_and_reports_timeout(rkv):
    """The failure path of every bounded device wait: a wait on an mbarrier that nothing
    arrives on runs out, sets the timeout bit, and the host reads RKV_ERR_TIMEOUT; the
    context stays usable and the next decode step is clean and correct."""
    wl = W.custom(B=1, Hq=4, Hkv=1, prompt_lens=[400], budget=64, window=8, page_size=16, steps=1, pool_kernel=3)
    run = DeviceRun(wl, rkv)
    run.prefill()
    unit = OracleUnit(run, 0, 0)
    unit.check_prefill(run)
    assert run.status() == (rkv.RKV_OK, 0)
    for limit_ns in (2_000, 200_000):
        rkv.rkv_selftest_bounded_wait(run.cache, limit_ns)
        st, bits = run.status()
        assert st == rkv.RKV_ERR_TIMEOUT and bits == rkv.DEVERR_TIMEOUT, (st, bits)
        assert run.status() == (rkv.RKV_OK, 0)   # the word was cleared
    with pytest.raises(rkv.RkvError):
        rkv.rkv_selftest_bounded_wait(run.cache, 0)
    d, out, ch, pg = run.decode_step(0)
    assert unit.step(run, d, out, ch, pg, check_cache=True)["err"] <= ATOL_OUT
    assert run.status() == (rkv.RKV_OK, 0)


@pytest.mark.parametrize("name", ["gqa4_ragged", "gqa2_p32", "p64_outliers"])
def test_quest_only_small(rkv, path, name):
    """Quest-only (the summary page's ablation of HSA's halves): every channel bounds
    the pages (k1 = 128) while only k2 < NP pages are attended.  Channel and page sets
    and the output against the oracle's HSA at k1 = d."""
    wl = SMALL[name]
    run = DeviceRun(wl, rkv)
    run.k1 = [128] * wl.B
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            res = u.step(run, d, out, ch, pg, check_cache=(step % 4 == 0))
            assert len(res["pages"]) < res["sig"].shape[0], "every page selected: not a Quest-only case"
            assert np.array_equal(np.sort(ch[u.b, u.g].cpu().numpy()), np.arange(128))
    assert run.status() == (rkv.RKV_OK, 0)


def test_quest_only_workload4_sampled(rkv, path):
    """Quest-only at full size: workload 4's batch with k1 = 128, sampled units."""
    wl = W.workload(4)
    longest = int(np.argmax(wl.prompt_lens))
    shortest = int(np.argmin(wl.prompt_lens))
    assert _sampled_full(rkv, 4, [(longest, 3), (shortest, 0)], {0, 255}, k1=128) <= ATOL_OUT


# ------------------------------------------------------------------ full-size workloads
def _sampled_full(rkv, n, units, steps_checked, gen_device="cuda", layer=0, k1=None):
    wl = W.workload(n)
    run = DeviceRun(wl, rkv, gen_device=gen_device, tail="zero", layer=layer)
    if k1 is not None:
        run.k1 = [k1] * wl.B
    run.prefill()
    checks = [OracleUnit(run, b, g) for b, g in units]
    for u in checks:
        u.check_prefill(run)
        u.check_cache(run)
    errs = []
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        if step in steps_checked:
            for u in checks:
                errs.append(u.step(run, d, out, ch, pg, check_cache=True)["err"])
        else:
            for u in checks:   # keep the oracle's cache in step without re-checking
                G = wl.G
                u.Kc = np.concatenate([u.Kc[: u.n], f64(d["k_new"][u.b, u.g])[None]])
                u.Vc = np.concatenate([u.Vc[: u.n], f64(d["v_new"][u.b, u.g])[None]])
                u.n += 1
    st, bits = run.status()
    assert st == rkv.RKV_OK, bits
    return max(errs)


def test_workload2_llama_layer_32k(rkv):
    assert _sampled_full(rkv, 2, [(0, 0), (0, 5)], {0, 63, 127}) <= ATOL_OUT


def test_workload3_extreme_ratio_109k(rkv):
    assert _sampled_full(rkv, 3, [(0, 3)], {0, 63}) <= ATOL_OUT


def test_workload4_batched_ragged(rkv, path):
    wl = W.workload(4)
    longest = int(np.argmax(wl.prompt_lens))
    shortest = int(np.argmin(wl.prompt_lens))
    assert _sampled_full(rkv, 4, [(longest, 1), (shortest, 6)], {0, 255}) <= ATOL_OUT


def test_flat_scoring_split_with_a_window_only_prompt(rkv):
    """128 units whose key tiles do not divide into the resident slots take the flat
    scoring split (equal shares of all units' tiles, runs crossing unit boundaries); one
    prompt is only its window, so it has no pass-2 tiles at all.  The units on both
    sides of it and that unit itself match the oracle (kept sets, pooled scores, cache,
    decode steps)."""
    lens = [8192] * 7 + [32] + [8192] * 8
    wl = W.custom(B=16, Hq=32, Hkv=8, prompt_lens=lens, budget=1024, window=32, page_size=16, steps=2,
                  pool_kernel=15)
    run = DeviceRun(wl, rkv, gen_device="cuda", tail="zero")
    run.prefill()
    checks = [OracleUnit(run, b, g) for b, g in [(6, 7), (7, 0), (7, 7), (8, 0), (15, 7)]]
    for u in checks:
        u.check_prefill(run)
        u.check_cache(run)
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in checks:
            assert u.step(run, d, out, ch, pg, check_cache=True)["err"] <= ATOL_OUT
    assert run.status()[0] == rkv.RKV_OK


def test_workload5_one_layer_sampled(rkv):
    assert _sampled_full(rkv, 5, [(0, 0), (7, 7)], {0, 63}) <= ATOL_OUT


def test_workload5_last_layer_sampled(rkv):
    """Layer 31 of the 32-layer workload: its own seeded keys, outlier channels and sinks."""
    assert _sampled_full(rkv, 5, [(3, 2)], {0, 63}, layer=31) <= ATOL_OUT


# ------------------------------------------------------------------ Exact-TopK recall diagnostic
@pytest.mark.parametrize("name", ["gqa4_ragged", "gqa8_w16", "gqa2_p32", "needles"])
def test_exact_topk_recall_matches_oracle(rkv, name):
    """Recall and mass of the GPU's page selection against the oracle's exact top-K,
    after every decode step.  The top-K may differ only by tokens whose exact score is
    within 1e-5 relative of the K-th score."""
    wl = SMALL[name]
    run = DeviceRun(wl, rkv)
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
    P = wl.page_size
    k_tokens = [k2 * P for k2 in run.k2]
    for step in range(min(wl.steps, 6)):
        d, out, ch, pg = run.decode_step(step)
        rec, mass = rkv.rkv_exact_topk_recall(run.cache, d["q"], pg, k_tokens)
        rec, mass = rec.cpu().numpy(), mass.cpu().numpy()
        for u in units:
            r = u.step(run, d, out, ch, pg)
            qg = f64(d["q"][u.b, u.g * wl.G:(u.g + 1) * wl.G])
            ref = O.exact_topk_recall(qg, u.Kc, u.n, r["pages"], P, k_tokens[u.b])
            e, K = ref["scores"], ref["K"]
            kth = np.sort(e)[::-1][K - 1] if K else 0.0
            band = int(np.sum(np.abs(e - kth) <= 1e-5 * abs(kth))) if K < u.n else 0
            got_hits = rec[u.b, u.g] * K
            assert abs(got_hits - ref["hits"]) <= band + 1e-3, (name, step, u.b, u.g, got_hits, ref["hits"], band)
            assert abs(mass[u.b, u.g] - ref["mass"]) <= 1e-4 + band / max(K, 1), (mass[u.b, u.g], ref["mass"])
    assert run.status()[0] == rkv.RKV_OK


def test_exact_topk_recall_full_selection_is_one(rkv):
    """Every page selected (k2 >= pages): recall and mass are exactly one."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[600, 450], budget=64, window=8, page_size=16, steps=1,
                  pool_kernel=5)
    run = DeviceRun(wl, rkv)
    run.k2 = [4096, 4096]
    run.prefill()
    d, out, ch, pg = run.decode_step(0)
    rec, mass = rkv.rkv_exact_topk_recall(run.cache, d["q"], pg, [64, 64])
    assert torch.all(rec == 1.0) and torch.allclose(mass, torch.ones_like(mass))


# ------------------------------------------------------------------ RocketKV-MT
def test_mt_small_end_to_end(rkv, path):
    """RocketKV-MT: nothing evicted, HSA over the whole prompt plus the new tokens."""
    wl = W.custom(B=2, Hq=8, Hkv=2, prompt_lens=[700, 1000], budget=64, window=8, page_size=16, steps=12,
                  pool_kernel=5, mt=True, name="mt_small")
    run = DeviceRun(wl, rkv)
    assert run.keep1 == [700, 1000]
    run.prefill()
    units = [OracleUnit(run, b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    for u in units:
        u.check_prefill(run)
        np.testing.assert_array_equal(u.kept, np.arange(u.L))
        u.check_cache(run)
    for step in range(wl.steps):
        d, out, ch, pg = run.decode_step(step)
        for u in units:
            u.step(run, d, out, ch, pg, check_cache=(step % 4 == 0))
    assert run.status()[0] == rkv.RKV_OK


def test_workload6_mt_batched_sampled(rkv):
    wl = W.workload(6)
    longest = int(np.argmax(wl.prompt_lens))
    assert _sampled_full(rkv, 6, [(longest, 2), (0, 5)], {0, 255}) <= ATOL_OUT


@pytest.mark.parametrize("name", ["gqa4_ragged", "no_eviction"])
def test_prefill_with_host_v_matches(rkv, name):
    """rkv_prefill_evict with V in pinned host memory (read through its device mapping)
    fills the cache exactly as with V on the device; a host K is refused."""
    wl = SMALL[name]
    runs = [DeviceRun(wl, rkv), DeviceRun(wl, rkv)]
    runs[0].prefill()
    g = runs[1].gpu_in
    v_host = runs[1].inputs["v"].contiguous().pin_memory()
    rkv.rkv_prefill_evict(g["q_win"], g["k"], v_host, g["prompt_len"], runs[1].keep1, runs[1].kp, runs[1].cache,
                          runs[1].kept, pooled_scores=runs[1].pooled)
    torch.cuda.synchronize()
    a, b = runs[0].cache, runs[1].cache
    assert torch.equal(runs[0].kept, runs[1].kept)
    assert torch.equal(a.seq_len, b.seq_len)
    for x, y in ((a.kmax, b.kmax), (a.kmin, b.kmin)):
        assert torch.equal(x.nan_to_num(), y.nan_to_num())
    # every page a sequence uses holds the same K and V rows
    for bb in range(wl.B):
        n = int(a.seq_len[bb])
        for pg in range((n + wl.page_size - 1) // wl.page_size):
            phys = int(a.page_table[bb, pg])
            cnt = min(wl.page_size, n - pg * wl.page_size)
            assert torch.equal(a.k_pages[phys, :, :cnt], b.k_pages[phys, :, :cnt])
            assert torch.equal(a.v_pages[phys, :, :cnt], b.v_pages[phys, :, :cnt])
    k_host = runs[1].inputs["k"].contiguous().pin_memory()
    with pytest.raises(rkv.RkvError):
        rkv.rkv_prefill_evict(g["q_win"], k_host, v_host, g["prompt_len"], runs[1].keep1, runs[1].kp,
                              runs[1].cache, runs[1].kept)
    for r in runs:
        assert r.status()[0] == rkv.RKV_OK


def test_decode_step_from_host_buffers_matches(rkv):
    """rkv_decode_step_host (host inputs and output) computes what rkv_decode_step does."""
    wl = SMALL["gqa4_ragged"]
    runs = [DeviceRun(wl, rkv), DeviceRun(wl, rkv)]
    for r in runs:
        r.prefill()
    staging = rkv.step_host_staging(wl.B, wl.Hq, wl.Hkv)
    for step in range(5):
        d = W.decode_tensors(wl, step, runs[0].seed, 0, runs[0].dev)   # the same draws as decode_step's
        host_in = torch.cat([d[k].contiguous().view(-1) for k in ("q", "k_new", "v_new")]).cpu().view(torch.uint8)
        host_in = host_in.pin_memory()
        host_out = torch.full((wl.B, wl.Hq, 128), float("nan")).pin_memory()
        rkv.rkv_decode_step_host(runs[1].cache, host_in, host_out, wl.Hq, runs[1].k1, runs[1].k2, staging,
                                 runs[1].dws)
        _, out, _, _ = runs[0].decode_step(step)
        torch.cuda.synchronize()
        assert torch.equal(host_out, out.cpu())
    assert torch.equal(runs[0].cache.seq_len, runs[1].cache.seq_len)
    for r in runs:
        assert r.status()[0] == rkv.RKV_OK
