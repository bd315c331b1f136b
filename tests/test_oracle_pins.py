"""Pins for the CPU oracle: each check ties it to something other than itself.

The checks come from what the RocketKV pages fix (the worked split example,
the page-bound invariant, append == rebuild), from closed forms and invariants,
from special cases that reduce to a library routine (scipy max filter, torch
SDPA, a plain argsort of raw logits), and from pure-Python brute force on tiny
inputs.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.ndimage
import torch

from oracle import rkv_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    """Round an fp64 array to bf16 values (kept as fp64), like the real inputs."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _rand(shape, seed, scale=1.0):
    return _bf16(np.random.default_rng(seed).standard_normal(shape) * scale)


# ---------------------------------------------------------------- a1: split
def test_split_worked_example():
    g = json.load(open(os.path.join(GOLD, "split_worked_example.json")))
    budget = 512
    s = O.split_ratio(g["c"] * budget, budget, 128, 16, 32)
    assert s["c"] == pytest.approx(64.0, abs=1e-12)
    assert round(s["c1"], 1) == g["stage1_ratio_1dp"]
    assert round(s["c2"], 1) == g["stage2_ratio_1dp"]


@pytest.mark.parametrize("c", [1 / 8, 0.5, 1.0, 2.0, 16.0, 64.0, 1000.0, 1024.0, 4096.0, 2.0 ** 20])
def test_split_clip_ends_and_product(c):
    g = json.load(open(os.path.join(GOLD, "split_worked_example.json")))
    budget = 256
    s = O.split_ratio(int(round(c * budget)), budget, 128, 16, 32)
    if c <= 1.0:
        assert s["r"] == g["r_floor"]
    elif c >= 1024.0:
        assert s["r"] == g["r_ceiling"]
    else:
        assert s["r"] == pytest.approx(0.2 + 0.06 * math.log2(c), abs=1e-12)
    # the two stage ratios multiply back to the overall ratio (c^r * c^(1-r) = c)
    assert s["c1"] * s["c2"] == pytest.approx(s["c"], rel=1e-12)


def test_split_share_grows_with_ratio():
    # small c leaves stage 1 near the 0.2 floor; large c moves it toward 0.8
    rs = [O.split_ratio(int(c * 256), 256, 128, 16, 32)["r"] for c in (2, 4, 64, 400)]
    assert all(a < b for a, b in zip(rs, rs[1:]))
    assert rs[0] < 0.3 and rs[-1] > 0.7


def test_split_niah_ratio():
    g = json.load(open(os.path.join(GOLD, "niah_ratio.json")))
    s = O.split_ratio(g["prompt_len"], g["budget"], 128, 16, 32)
    assert s["c"] > g["ratio_above"]
    assert 0.72 < s["r"] < 0.8           # not clipped: log2(425.8) < 10


def test_default_pool_kernel_matches_the_workloads():
    # the only sizes anything fixes: the three benchmark workloads that state a pooling
    # kernel (4K -> 7, 32K -> 31, 109K -> 63); the rule must reproduce each of them, and
    # the tiny workload's k1 = 64 must come out of the derived split without an override
    g = json.load(open(os.path.join(GOLD, "pool_kernel_workloads.json")))
    for c in g["cases"]:
        assert O.default_pool_kernel(c["prompt_len"]) == c["pool_kernel"], c["workload"]
        s = O.split_ratio(c["prompt_len"], c["budget"], 128, c["page_size"], 32)
        assert s["pool_kernel"] == c["pool_kernel"], c["workload"]
        if "k1" in c:
            assert s["k1"] == c["k1"], c["workload"]
    # the kernel is keyed by prompt length, not by the ratio: the same prompt at another
    # budget pools alike, and the 4K and 109K prompts at equal c differ
    assert O.split_ratio(32768, 2048, 128, 32, 32)["pool_kernel"] == 31
    assert O.split_ratio(4096, 16, 128, 16, 32)["pool_kernel"] == 7
    assert O.split_ratio(109000, 6812, 128, 16, 32)["pool_kernel"] == 63


def test_split_derived_sizes():
    # readings (keep1 = round(L/c1), k2 = budget/P, k1 from sqrt(c2)) on the workloads
    cases = [  # L, budget, P, k1_override -> keep1, k1, k2
        (4096, 256, 16, 64, 1209, 64, 16),
        (32768, 512, 16, 0, 3191, 48, 32),
        (109000, 256, 16, 0, 1361, 48, 16),
        (65536, 4096, 16, 0, 19349, 64, 256),
    ]
    for L, budget, P, k1o, keep1, k1, k2 in cases:
        s = O.split_ratio(L, budget, 128, P, 32, k1o)
        assert (s["keep1"], s["k1"], s["k2"]) == (keep1, k1, k2)
    # derived k1 reproduces the tiny workload's given k1 = 64 without the override
    assert O.split_ratio(4096, 256, 128, 16, 32)["k1"] == 64
    # keep1 never exceeds the prompt nor drops below the budget
    assert O.split_ratio(200, 256, 128, 16, 32)["keep1"] == 200
    assert O.split_ratio(300, 256, 128, 16, 32)["keep1"] == 290     # c=1.17, c1=1.034
    # L / c1 = budget * c / c^r = budget * c2: the survivors are the budget times stage 2's ratio
    for L in (5000, 32768, 1 << 20):
        s = O.split_ratio(L, 256, 128, 16, 32)
        assert abs(s["keep1"] - 256 * s["c2"]) <= 0.5 + 1e-9


# ---------------------------------------------------------------- a2: window scores
def _window_case(seed, Hq=4, Hkv=2, w=5, L=40, d=16):
    q = _rand((Hq, w, d), seed)
    k = _rand((Hkv, L, d), seed + 1)
    return q, k


def test_window_row_sums_invariant():
    q, k = _window_case(1)
    Hq, w, _ = q.shape
    Hkv = k.shape[0]
    A = O.window_column_scores(q, k)
    np.testing.assert_allclose(A.sum(axis=1), np.full(Hkv, w * (Hq // Hkv)), rtol=1e-13)


def test_window_zero_query_closed_form_and_gqa_mapping():
    # heads 0,1 (group 0) get zero queries -> uniform weights over visible keys;
    # heads 2,3 (group 1) are random.  An interleaved head->group mapping fails this.
    q, k = _window_case(2, Hq=4, Hkv=2, w=5, L=40)
    q[0:2] = 0.0
    A = O.window_column_scores(q, k)
    L, w, G = 40, 5, 2
    expect = np.empty(L)
    for t in range(L):
        expect[t] = G * sum(1.0 / (L - w + j + 1) for j in range(w) if t <= L - w + j)
    np.testing.assert_allclose(A[0], expect, rtol=1e-13)
    assert not np.allclose(A[1], expect)


def test_window_causal_decomposition():
    # w window rows == w single-row scorings, row j on the keys it may see (t <= L-w+j)
    q, k = _window_case(3)
    Hq, w, _ = q.shape
    Hkv, L, _ = k.shape
    A = O.window_column_scores(q, k)
    acc = np.zeros_like(A)
    for j in range(w):
        n_vis = L - w + j + 1
        Aj = O.window_column_scores(q[:, j:j + 1, :], k[:, :n_vis, :])
        acc[:, :n_vis] += Aj
    np.testing.assert_allclose(A, acc, rtol=1e-12, atol=1e-15)


def test_window_scores_bruteforce():
    Hq, Hkv, w, L, d = 2, 1, 2, 6, 3
    q, k = _window_case(4, Hq=Hq, Hkv=Hkv, w=w, L=L, d=d)
    S = O.window_scores(q, k)
    ref = [0.0] * (L - w)
    for h in range(Hq):
        for j in range(w):
            pos = L - w + j
            logits = []
            for t in range(pos + 1):
                dot = 0.0
                for c in range(d):
                    dot += q[h, j, c] * k[0, t, c]
                logits.append(dot / math.sqrt(d))
            m = max(logits)
            den = sum(math.exp(z - m) for z in logits)
            for t in range(L - w):
                ref[t] += math.exp(logits[t] - m) / den
    np.testing.assert_allclose(S[0], ref, rtol=1e-12)


# ---------------------------------------------------------------- a3: pooling
@pytest.mark.parametrize("kernel", [1, 3, 7, 31, 63])
@pytest.mark.parametrize("n", [1, 5, 40, 100])
def test_max_pool_matches_scipy(kernel, n):
    S = np.random.default_rng(kernel * 1000 + n).random((2, n))
    # 'nearest' edge replication only repeats in-range values, so for a max it is
    # the same as ignoring out-of-range positions
    ref = scipy.ndimage.maximum_filter1d(S, size=kernel, axis=-1, mode="nearest")
    np.testing.assert_array_equal(O.max_pool(S, kernel), ref)


# ---------------------------------------------------------------- a4: selection
def test_select_single_query_is_topk_of_raw_logits():
    # w=1, G=1, kernel 1: softmax is monotone, so stage 1 keeps the top logits
    L, d, keep1 = 64, 16, 10
    q = _rand((1, 1, d), 5)
    k = _rand((1, L, d), 6)
    res = O.prefill_evict_unit(q, k, keep1, 1)
    logits = k[0, : L - 1] @ q[0, 0]
    top = np.sort(np.argsort(-logits, kind="stable")[: keep1 - 1])
    np.testing.assert_array_equal(res["kept"][0], np.concatenate([top, [L - 1]]))


def test_select_invariants_with_planted_ties():
    L, w, keep1 = 50, 4, 12
    S = np.round(np.random.default_rng(7).random(L - w) * 5) / 5   # many exact ties
    kept = O.select_kept(S, keep1, L, w)
    assert len(kept) == keep1 and np.all(np.diff(kept) > 0)
    assert set(range(L - w, L)) <= set(kept.tolist())
    pre = kept[kept < L - w]
    rest = np.setdiff1d(np.arange(L - w), pre)
    assert S[pre].min() >= S[rest].max()
    kth = S[pre].min()
    # among tokens tied at the boundary score the lower positions were kept
    tied_kept = pre[S[pre] == kth]
    tied_out = rest[S[rest] == kth]
    if len(tied_out):
        assert tied_kept.max() < tied_out.min()


# ---------------------------------------------------------------- a6: summaries
def test_summaries_append_equals_rebuild():
    P, d = 16, 8
    Kc = _rand((70, d), 8)
    kmax, kmin = O.page_summaries(Kc, 33, P)
    n = 33
    for step in [1, 1, 1, 5, 14, 1, 14]:
        kmax, kmin = O.append_summaries(kmax, kmin, Kc, n, step, P)
        n += step
        rmax, rmin = O.page_summaries(Kc, n, P)
        np.testing.assert_array_equal(kmax, rmax)
        np.testing.assert_array_equal(kmin, rmin)
    assert n == 70


def test_summaries_membership_and_bounds():
    P, d, n = 8, 6, 29
    Kc = _rand((32, d), 9)
    Kc[n:] = np.nan                           # unfilled tail must not be read
    kmax, kmin = O.page_summaries(Kc, n, P)
    assert kmax.shape == (d, 4) and np.all(np.isfinite(kmax))
    for p in range(4):
        tok = Kc[p * P: min(n, (p + 1) * P)]
        for c in range(d):
            col = tok[:, c].tolist()
            assert kmax[c, p] in col and kmin[c, p] in col
            assert all(kmin[c, p] <= x <= kmax[c, p] for x in col)


# ---------------------------------------------------------------- a7: channels
def test_channel_select_topk_with_ties():
    d, G, k1 = 16, 2, 5
    q = np.zeros((G, d))
    a_target = np.array([3, 1, 4, 1, 5, 9, 2, 6, 5, 3, 5, 8, 9, 7, 9, 3], dtype=float)
    q[0] = a_target * np.where(np.arange(d) % 2, 1, -1)   # |q| carries the score
    chans, a = O.channel_select(q, k1)
    np.testing.assert_array_equal(a, a_target)
    # by (score desc, channel asc): 9@5, 9@12, 9@14, 8@11, 7@13
    np.testing.assert_array_equal(chans, [5, 11, 12, 13, 14])
    chans2, _ = O.channel_select(q, 8)     # then 6@7, 5@4, 5@8 (5@10 loses the tie)
    np.testing.assert_array_equal(chans2, [4, 5, 7, 8, 11, 12, 13, 14])


# ---------------------------------------------------------------- a8: page bound
def test_page_bound_is_upper_bound_bruteforce():
    G, d, n, P, k1 = 3, 16, 45, 8, 5
    q = _rand((G, d), 10, scale=2.0)
    Kc = _rand((n, d), 11)
    kmax, kmin = O.page_summaries(Kc, n, P)
    chans, _ = O.channel_select(q, k1)
    per = O.page_scores(q, kmax, kmin, chans, per_head=True)
    tot = O.page_scores(q, kmax, kmin, chans)
    np.testing.assert_allclose(per.sum(axis=0), tot, rtol=1e-14)
    for p in range(per.shape[1]):
        for t in range(p * P, min(n, (p + 1) * P)):
            partial = [sum(q[h, i] * Kc[t, i] for i in chans) for h in range(G)]
            for h in range(G):
                assert per[h, p] >= partial[h] - 1e-12
            assert tot[p] >= sum(partial) - 1e-12


def test_page_score_single_token_pages_closed_form():
    # with one token per page Kmax = Kmin = k, so the bound is the exact partial dot
    G, d, n, k1 = 2, 16, 9, 6
    q = _rand((G, d), 12)
    Kc = _rand((n, d), 13)
    kmax, kmin = O.page_summaries(Kc, n, 1)
    chans, _ = O.channel_select(q, k1)
    tot = O.page_scores(q, kmax, kmin, chans)
    exact = np.array([sum(q[h, i] * Kc[t, i] for h in range(G) for i in chans) for t in range(n)])
    np.testing.assert_allclose(tot, exact, rtol=1e-13, atol=1e-13)


def test_page_score_sign_picks_max_or_min():
    d, k1 = 8, 8
    Kc = _rand((4, d), 14)
    kmax, kmin = O.page_summaries(Kc, 4, 4)
    qp = np.abs(_rand((1, d), 15)) + 0.5
    chans, _ = O.channel_select(qp, k1)
    assert O.page_scores(qp, kmax, kmin, chans)[0] == pytest.approx(float(qp[0] @ kmax[:, 0]))
    assert O.page_scores(-qp, kmax, kmin, chans)[0] == pytest.approx(float(-qp[0] @ kmin[:, 0]))


# ---------------------------------------------------------------- a9: top-k2
def test_topk_pages_ties_and_all():
    s = np.array([1.0, 3.0, 2.0, 3.0, 0.5, 3.0])
    np.testing.assert_array_equal(O.topk_pages(s, 2), [1, 3])
    np.testing.assert_array_equal(O.topk_pages(s, 4), [1, 2, 3, 5])
    np.testing.assert_array_equal(O.topk_pages(s, 10), np.arange(6))


# ---------------------------------------------------------------- a10: attention
def _sdpa(q, K, V, scale):
    qt = torch.from_numpy(q)[None, :, None, :]                 # [1, G, 1, d]
    Kt = torch.from_numpy(K)[None, None].expand(1, q.shape[0], -1, -1)
    Vt = torch.from_numpy(V)[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return o[0, :, 0, :].numpy()


def test_hsa_full_selection_equals_sdpa():
    # k1 = d and k2 = every page: HSA is full attention over the survivors
    G, d, n, P = 4, 32, 50, 16
    q = _rand((G, d), 16, scale=1.5)
    Kc = _rand((64, d), 17)
    Vc = _rand((64, d), 18)
    Kc[n:] = np.nan
    Vc[n:] = np.nan
    kmax, kmin = O.page_summaries(Kc, n, P)
    res = O.hsa_decode_unit(q, Kc, Vc, n, kmax, kmin, P, k1=d, k2=100)
    np.testing.assert_array_equal(res["pages"], np.arange(4))
    ref = _sdpa(q, Kc[:n], Vc[:n], 1.0 / math.sqrt(d))
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-13)


def test_sparse_attention_on_selected_pages_equals_sdpa():
    G, d, n, P = 2, 16, 40, 8
    q = _rand((G, d), 19)
    Kc = _rand((n, d), 20)
    Vc = _rand((n, d), 21)
    pages = np.array([1, 3, 4])
    out = O.sparse_attention(q, Kc, Vc, n, pages, P, scale=0.3)
    tok = np.concatenate([np.arange(p * P, (p + 1) * P) for p in pages])
    np.testing.assert_allclose(out, _sdpa(q, Kc[tok], Vc[tok], 0.3), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- SparQ-only (one-token pages)
def test_sparq_scores_are_partial_dot_products():
    """The token score is the group's partial dot product over the chosen channels,
    computed here token by token in pure Python."""
    G, d, n = 3, 16, 23
    q = _rand((G, d), 30, scale=1.3)
    Kc = _rand((n, d), 31)
    Vc = _rand((n, d), 32)
    k1 = 5
    res = O.sparq_decode_unit(q, Kc, Vc, n, k1, k_tokens=7)
    chans = res["channels"]
    assert len(chans) == k1
    for t in range(n):
        s = 0.0
        for h in range(G):
            for i in chans:
                s += float(q[h, i]) * float(Kc[t, i])
        assert abs(res["page_score"][t] - s) <= 1e-12 * (1 + abs(s))
    order = sorted(range(n), key=lambda t: (-res["page_score"][t], t))[:7]
    np.testing.assert_array_equal(res["pages"], sorted(order))


def test_sparq_all_tokens_equals_sdpa():
    G, d, n = 4, 32, 37
    q = _rand((G, d), 33)
    Kc = _rand((n, d), 34)
    Vc = _rand((n, d), 35)
    res = O.sparq_decode_unit(q, Kc, Vc, n, k1=8, k_tokens=n + 5)
    np.testing.assert_array_equal(res["pages"], np.arange(n))
    np.testing.assert_allclose(res["out"], _sdpa(q, Kc, Vc, 1.0 / math.sqrt(d)), rtol=1e-12, atol=1e-13)


def test_sparq_with_every_channel_ranks_by_the_full_dot_product():
    G, d, n = 2, 16, 30
    q = _rand((G, d), 36)
    Kc = _rand((n, d), 37)
    res = O.sparq_decode_unit(q, Kc, Kc, n, k1=d, k_tokens=6)
    full = (q.sum(axis=0) @ Kc.T)
    np.testing.assert_allclose(res["page_score"], full, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(res["pages"], np.sort(np.argsort(-full, kind="stable")[:6]))


# ---------------------------------------------------------------- end to end (qualitative)
def test_planted_needle_survives_and_is_selected():
    Hq, Hkv, w, L, d, P = 4, 1, 8, 512, 64, 16
    rng = np.random.default_rng(22)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    k = _bf16(rng.standard_normal((Hkv, L, d)))
    v = _bf16(rng.standard_normal((Hkv, L, d)))
    needle = 300
    k[0, needle] = _bf16(2 * math.sqrt(d) * u)
    q = _bf16(rng.standard_normal((Hq, w, d)) + math.sqrt(d) * u)
    res = O.prefill_evict_unit(q, k, keep1=64, pool_kernel=7)
    kept = res["kept"][0]
    assert needle in kept
    Kc, Vc = k[0, kept], v[0, kept]
    kmax, kmin = O.page_summaries(Kc, 64, P)
    qd = _bf16(rng.standard_normal((Hq, d)) + math.sqrt(d) * u)
    dec = O.hsa_decode_unit(qd, Kc, Vc, 64, kmax, kmin, P, k1=16, k2=1)
    assert int(np.where(kept == needle)[0][0]) // P in dec["pages"].tolist()


# ------------------------------------------------------------------ exact top-K recall diagnostic
def _rand_unit(rng, G=4, n=70, d=128):
    q = rng.standard_normal((G, d))
    K = rng.standard_normal((n, d))
    return q, K


def test_exact_scores_sum_to_group_size():
    """Each head's attention over the cached tokens sums to one: the group sum is G."""
    rng = np.random.default_rng(11)
    for G in (1, 2, 4, 8):
        q, K = _rand_unit(rng, G=G, n=53)
        e = O.exact_token_scores(q, K, 53)
        assert e.shape == (53,) and np.all(e >= 0)
        assert abs(e.sum() - G) < 1e-12


def test_exact_scores_one_head_is_softmax():
    """With one head the score is the softmax of the scaled logits (scipy's softmax)."""
    import scipy.special
    rng = np.random.default_rng(12)
    q, K = _rand_unit(rng, G=1, n=40)
    e = O.exact_token_scores(q, K, 40)
    ref = scipy.special.softmax(K @ q[0] / math.sqrt(128))
    np.testing.assert_allclose(e, ref, rtol=1e-12, atol=1e-15)


def test_recall_all_pages_and_own_pages_is_one():
    rng = np.random.default_rng(13)
    q, K = _rand_unit(rng, n=70)
    P, Kt = 16, 24
    r = O.exact_topk_recall(q, K, 70, np.arange(5), P, Kt)
    assert r["recall"] == 1.0 and abs(r["mass"] - 1.0) < 1e-15 and r["K"] == Kt
    own = np.unique(r["top"] // P)
    r2 = O.exact_topk_recall(q, K, 70, own, P, Kt)
    assert r2["recall"] == 1.0
    missing = np.setdiff1d(np.arange(5), own)
    if missing.size:   # pages holding none of the top-K add nothing
        r3 = O.exact_topk_recall(q, K, 70, missing, P, Kt)
        assert r3["recall"] == 0.0 and r3["mass"] == 0.0


def test_recall_whole_cache_budget_closed_form():
    """K >= n: every token is in the top-K, so recall is the covered share of the
    tokens and the mass is the covered share of the group's total mass G."""
    rng = np.random.default_rng(14)
    G, n, P = 4, 61, 16
    q, K = _rand_unit(rng, G=G, n=n)
    pages = np.array([0, 2, 3])
    r = O.exact_topk_recall(q, K, n, pages, P, 10_000)
    covered = [t for t in range(n) if t // P in set(pages.tolist())]
    assert r["K"] == n and r["recall"] == len(covered) / n
    e = O.exact_token_scores(q, K, n)
    assert abs(r["mass"] - e[covered].sum() / G) < 1e-12


def test_recall_brute_force_tiny():
    """Pure-Python ranking of the scores on tiny inputs, with planted ties."""
    rng = np.random.default_rng(15)
    for trial in range(20):
        n, P, Kt = int(rng.integers(5, 30)), 4, int(rng.integers(1, 12))
        q, K = _rand_unit(rng, G=2, n=n, d=128)
        if trial % 4 == 0:
            K[1] = K[3]            # equal keys: equal scores, the lower index ranks first
        pages = rng.choice(-(-n // P), size=max(1, -(-n // P) // 2), replace=False)
        r = O.exact_topk_recall(q, K, n, pages, P, Kt)
        e = r["scores"]
        ranked = sorted(range(n), key=lambda t: (-float(e[t]), t))
        top = ranked[:min(Kt, n)]
        hits = [t for t in top if t // P in set(int(x) for x in pages)]
        assert r["top"].tolist() == sorted(top)
        assert r["hits"] == len(hits) and r["recall"] == len(hits) / len(top)


# ------------------------------------------------------------------ RocketKV-MT split
def test_split_mt_keeps_the_prompt_and_gives_stage2_the_ratio():
    for L, budget, P in [(32768, 512, 16), (8192, 2048, 32), (100, 256, 16)]:
        s = O.split_ratio_mt(L, budget, 128, P)
        assert s["keep1"] == L and s["c1"] == 1.0 and s["r"] == 0.0
        assert abs(s["c1"] * s["c2"] - L / budget) < 1e-12
        assert s["k2"] == max(1, budget // P)
        # k1 takes the same rule as the two-stage split would at c2 = c
        k1 = 16 * round(128 / (16 * math.sqrt(L / budget)))
        assert s["k1"] == min(max(k1, 16), 128)
    assert O.split_ratio_mt(32768, 512, 128, 16, k1_override=40)["k1"] == 40


# ------------------------------------------------------------------ chunked prefill
def _chunks(rng, Hq=4, Hkv=2, w=8, lens=(100, 60, 90), d=128):
    q = [rng.standard_normal((Hq, w, d)) for _ in lens]
    k = [rng.standard_normal((Hkv, m, d)) for m in lens]
    v = [rng.standard_normal((Hkv, m, d)) for m in lens]
    return q, k, v


def test_chunked_single_chunk_is_prefill_evict():
    rng = np.random.default_rng(21)
    q, k, v = _chunks(rng, lens=(150,))
    r = O.prefill_chunked_unit(q, k, v, keep1=64, pool_kernel=5)
    ref = O.prefill_evict_unit(q[0], k[0], 64, 5)["kept"]
    np.testing.assert_array_equal(r["history"][0]["kept"], ref)
    for g in range(2):
        np.testing.assert_array_equal(r["K"][g], k[0][g, ref[g]])
        np.testing.assert_array_equal(r["V"][g], v[0][g, ref[g]])


def test_chunked_under_budget_keeps_everything():
    rng = np.random.default_rng(22)
    q, k, v = _chunks(rng, lens=(20, 30, 10))
    r = O.prefill_chunked_unit(q, k, v, keep1=64, pool_kernel=5)
    assert all(h["kept"] is None for h in r["history"]) and [h["held"] for h in r["history"]] == [20, 50, 60]
    np.testing.assert_array_equal(r["K"], np.concatenate(k, axis=1))


def test_chunked_invariants():
    """The held length never exceeds keep1 after an eviction, the chunk's window is
    always kept, and the kept indices are ascending."""
    rng = np.random.default_rng(23)
    w, keep1 = 8, 64
    q, k, v = _chunks(rng, w=w, lens=(100, 60, 90, 9))
    r = O.prefill_chunked_unit(q, k, v, keep1=keep1, pool_kernel=5)
    held = 0
    for c, h in enumerate(r["history"]):
        before = held + k[c].shape[1]
        if h["kept"] is not None:
            assert h["held"] == keep1
            for g in range(2):
                kept = h["kept"][g]
                assert np.all(np.diff(kept) > 0)
                np.testing.assert_array_equal(kept[-w:], np.arange(before - w, before))
        else:
            assert h["held"] == before <= keep1
        held = h["held"]


def test_chunked_with_no_early_eviction_is_single_shot():
    """When no chunk but the last one overflows keep1, chunking changes nothing: the
    result equals one stage-1 eviction over the whole prompt with the last chunk's
    window."""
    rng = np.random.default_rng(24)
    q, k, v = _chunks(rng, lens=(30, 25, 90))
    r = O.prefill_chunked_unit(q, k, v, keep1=64, pool_kernel=5)
    assert [h["kept"] is None for h in r["history"]] == [True, True, False]
    K, V = np.concatenate(k, axis=1), np.concatenate(v, axis=1)
    ref = O.prefill_evict_unit(q[-1], K, 64, 5)["kept"]
    for g in range(2):
        np.testing.assert_array_equal(r["K"][g], K[g, ref[g]])
        np.testing.assert_array_equal(r["V"][g], V[g, ref[g]])


def test_chunked_survivors_keep_prompt_order():
    """Every held row is a row of the prompt, each at most once, in prompt order; an
    evicted token never returns."""
    rng = np.random.default_rng(25)
    q, k, v = _chunks(rng, lens=(120, 70, 45, 80))
    r = O.prefill_chunked_unit(q, k, v, keep1=64, pool_kernel=3)
    K = np.concatenate(k, axis=1)
    for g in range(2):
        pos = [int(np.flatnonzero((K[g] == row).all(axis=1))[0]) for row in r["K"][g]]
        assert np.all(np.diff(pos) > 0)
        # positions evicted by the first chunk's eviction are gone for good
        first = set(O.prefill_evict_unit(q[0], k[0], 64, 3)["kept"][g].tolist())
        assert all(p >= 120 or p in first for p in pos)
