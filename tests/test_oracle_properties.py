"""Randomised properties of the CPU oracle (hypothesis; CPU only).

Each property is a characterisation that does not restate the oracle's code: the
page bound against brute-force partial dot products, selections against the
order they must respect, summaries against their membership, the split against
its own identities.  They widen the fixed pins of test_oracle_pins.py to random
shapes, sizes, ties and page sizes.
"""
import math

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

from oracle import rkv_oracle as O  # noqa: E402

_SETTINGS = settings(max_examples=60, deadline=None)


def _keys(seed, shape, levels=None):
    """N(0,1) values, or small integers when `levels` is set (many exact ties)."""
    r = np.random.default_rng(seed)
    if levels:
        return r.integers(-levels, levels + 1, size=shape).astype(np.float64)
    return r.standard_normal(shape)


@_SETTINGS
@given(G=st.integers(1, 4), d=st.sampled_from([8, 16]), n=st.integers(1, 70),
       P=st.sampled_from([1, 2, 4, 8, 16, 32]), k1f=st.floats(0.05, 1.0), seed=st.integers(0, 2**31),
       ties=st.booleans())
def test_page_bound_dominates_every_token(G, d, n, P, k1f, seed, ties):
    """Each head's page bound is >= that head's partial dot product with every valid
    token of the page, over the chosen channels; the GQA bound is the sum."""
    k1 = max(1, int(round(k1f * d)))
    q = _keys(seed, (G, d), 3 if ties else None)
    Kc = _keys(seed + 1, (n, d), 2 if ties else None)
    kmax, kmin = O.page_summaries(Kc, n, P)
    chans, _ = O.channel_select(q, k1)
    per = O.page_scores(q, kmax, kmin, chans, per_head=True)
    tot = O.page_scores(q, kmax, kmin, chans)
    assert per.shape == (G, math.ceil(n / P))
    for t in range(n):
        p = t // P
        part = q[:, chans] @ Kc[t, chans]
        assert np.all(per[:, p] >= part - 1e-9)
        assert tot[p] >= part.sum() - 1e-9
    # a one-token page is bounded exactly
    if P == 1:
        np.testing.assert_allclose(tot, (q[:, chans] @ Kc[:n, chans].T).sum(axis=0), atol=1e-9)


@_SETTINGS
@given(NP=st.integers(1, 80), k2=st.integers(1, 90), seed=st.integers(0, 2**31), levels=st.sampled_from([0, 1, 3]))
def test_topk_pages_respects_score_then_index(NP, k2, seed, levels):
    """min(k2, NP) ascending pages; every taken page outscores every other, and among
    equal scores at the boundary the lower pages are the taken ones."""
    s = _keys(seed, (NP,), levels or None)
    sel = O.topk_pages(s, k2)
    assert len(sel) == min(k2, NP) and np.all(np.diff(sel) > 0)
    rest = np.setdiff1d(np.arange(NP), sel)
    if len(sel) and len(rest):
        assert s[sel].min() >= s[rest].max()
        boundary = s[sel].min()
        tied_in = sel[s[sel] == boundary]
        tied_out = rest[s[rest] == boundary]
        if len(tied_out):
            assert tied_in.max() < tied_out.min()


@_SETTINGS
@given(G=st.integers(1, 8), d=st.sampled_from([8, 16, 128]), k1f=st.floats(0.01, 1.0), seed=st.integers(0, 2**31),
       ties=st.booleans())
def test_channel_select_respects_magnitude_then_index(G, d, k1f, seed, ties):
    k1 = max(1, int(round(k1f * d)))
    q = _keys(seed, (G, d), 2 if ties else None)
    chans, a = O.channel_select(q, k1)
    np.testing.assert_allclose(a, [sum(abs(q[h, i]) for h in range(G)) for i in range(d)])
    assert len(chans) == k1 and np.all(np.diff(chans) > 0)
    rest = np.setdiff1d(np.arange(d), chans)
    if len(rest):
        assert a[chans].min() >= a[rest].max()
        b = a[chans].min()
        if np.any(a[rest] == b):
            assert chans[a[chans] == b].max() < rest[a[rest] == b].min()


@_SETTINGS
@given(n_old=st.integers(1, 60), n_new=st.integers(0, 40), P=st.sampled_from([1, 3, 8, 16]),
       seed=st.integers(0, 2**31))
def test_summaries_are_members_and_append_equals_rebuild(n_old, n_new, P, seed):
    d = 8
    Kc = _keys(seed, (n_old + n_new, d), 4)
    kmax, kmin = O.page_summaries(Kc, n_old, P)
    full = O.page_summaries(Kc, n_old + n_new, P)
    inc = O.append_summaries(kmax, kmin, Kc, n_old, n_new, P)
    np.testing.assert_array_equal(inc[0], full[0])
    np.testing.assert_array_equal(inc[1], full[1])
    for p in range(full[0].shape[1]):
        tok = Kc[p * P: min(n_old + n_new, (p + 1) * P)]
        for c in range(d):   # each summary value is one of the page's own values, and bounds them all
            assert full[0][c, p] in tok[:, c] and full[1][c, p] in tok[:, c]
            assert np.all(tok[:, c] <= full[0][c, p]) and np.all(tok[:, c] >= full[1][c, p])


@_SETTINGS
@given(L=st.integers(64, 200000), frac=st.floats(0.001, 1.0), P=st.sampled_from([16, 32, 64]))
def test_split_identities(L, frac, P):
    """c1 c2 = c, r inside its clip range and equal to the formula there, and the sizes
    stay inside their ranges."""
    w = 32
    budget = max(w + 1, int(L * frac))
    budget -= budget % P
    if budget <= w or budget > L:
        return
    s = O.split_ratio(L, budget, 128, P, w)
    c = L / budget
    assert s["c1"] * s["c2"] == pytest.approx(c, rel=1e-12)
    assert 0.2 <= s["r"] <= 0.8
    if 1.0 < c < 2 ** 10:
        assert s["r"] == pytest.approx(0.2 + 0.06 * math.log2(c)) or s["r"] in (0.2, 0.8)
    assert max(budget, w) <= s["keep1"] <= L
    assert s["k2"] == budget // P
    assert 16 <= s["k1"] <= 128 and s["k1"] % 16 == 0
