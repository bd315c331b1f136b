"""GPU parity of chunked prefill (rkv_prefill_chunk) against the oracle.

Each chunk joins the survivors held so far and SnapKV++ re-enforces keep1 over the
held sequence (RocketKV, [adapted] summary, "Evidence": the stage-1 budget holds
across chunked-prefill calls).  The oracle follows the GPU's validated kept set from
chunk to chunk, as the single-shot tests do, so a boundary swap inside the fp32 tie
band cannot make the later chunks diverge; the cache (pages, summaries, seq_len) is
compared bit for bit after every chunk.
"""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from two_stage_kv_snapkv_gb300 import workloads as W

from rkv_check import ATOL_OUT, check_topk, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from two_stage_kv_snapkv_gb300 import build_lib
    build_lib.build()
    from two_stage_kv_snapkv_gb300 import rkv as mod
    return mod


CASES = {
    # sequence 0 evicts from the first chunk on, sequence 1 only from the second;
    # chunk lengths are ragged (not multiples of the 128-key tile or the page)
    "gqa4_two_seqs": dict(B=2, Hq=8, Hkv=2, window=8, page_size=16, keep1=[200, 300], pool_kernel=[5, 7],
                          chunks=[[300, 100], [150, 250], [77, 501]]),
    # GQA 1, window 16, pages of 32, a chunk exactly the window long
    "gqa1_w16": dict(B=1, Hq=2, Hkv=2, window=16, page_size=32, keep1=[96], pool_kernel=[3],
                     chunks=[[64], [129], [16], [700]]),
    # keep1 larger than everything held until the last chunk
    "late_eviction": dict(B=1, Hq=4, Hkv=1, window=8, page_size=16, keep1=[600], pool_kernel=[9],
                          chunks=[[200], [200], [150], [400]]),
}


def _chunk_inputs(case: dict, c: int, seed: int) -> dict:
    lens = case["chunks"][c]
    wl = W.custom(B=case["B"], Hq=case["Hq"], Hkv=case["Hkv"], prompt_lens=lens, budget=64,
                  window=case["window"], page_size=case["page_size"], steps=1)
    return W.prefill_tensors(wl, seed, layer=c, device="cpu", tail="nan")


def _run_chunks(rkv, case: dict, seed: int = 0x5EED, held_len_offset: int = 0):
    dev = torch.device("cuda")
    B, Hq, Hkv, w, P = case["B"], case["Hq"], case["Hkv"], case["window"], case["page_size"]
    G = Hq // Hkv
    keep1, kp = case["keep1"], case["pool_kernel"]
    max_pages = (max(keep1) + 2 + P - 1) // P
    max_pages = (max_pages + 7) // 8 * 8
    pt = W.page_table(B, max_pages, seed, dev, spare=3)
    cache = rkv.PagedCache(B, Hkv, P, max_pages, dev, page_table=pt, num_phys_pages=B * max_pages + 3,
                           fill=float("nan"))
    kept = torch.full((B, Hkv, max(keep1)), -7, dtype=torch.int32, device=dev)
    held = [np.zeros((Hkv, 0, 128)) for _ in range(B)]      # the oracle's held keys per sequence
    held_v = [np.zeros((Hkv, 0, 128)) for _ in range(B)]
    chunks_k, chunks_v, qs = [[] for _ in range(B)], [[] for _ in range(B)], [[] for _ in range(B)]
    swaps = 0
    for c in range(len(case["chunks"])):
        inp = _chunk_inputs(case, c, seed)
        lens = case["chunks"][c]
        held_len = [h.shape[1] + held_len_offset for h in held]
        kept.fill_(-7)
        rkv.rkv_prefill_chunk(inp["q_win"].to(dev), inp["k"].to(dev), inp["v"].to(dev), lens, held_len, keep1, kp,
                              cache, kept)
        if held_len_offset:
            return cache
        for b in range(B):
            m = lens[b]
            kc, vc = f64(inp["k"][b, :, :m]), f64(inp["v"][b, :, :m])
            chunks_k[b].append(kc)
            chunks_v[b].append(vc)
            qs[b].append(f64(inp["q_win"][b]))
            K = np.concatenate([held[b], kc], axis=1)
            V = np.concatenate([held_v[b], vc], axis=1)
            n = K.shape[1]
            keep = min(keep1[b], n)
            newK, newV = [], []
            for g in range(Hkv):
                got = kept[b, g, :keep].cpu().numpy().astype(np.int64)
                if keep < kept.shape[-1]:
                    assert np.all(kept[b, g, keep:].cpu().numpy() == -7), "kept_idx written past keep1"
                assert np.all(np.diff(got) > 0), "kept positions not ascending"
                if n <= keep1[b]:
                    np.testing.assert_array_equal(got, np.arange(n))
                else:
                    ref = O.prefill_evict_unit(qs[b][-1][g * G:(g + 1) * G], K[g:g + 1], keep1[b], kp[b])
                    np.testing.assert_array_equal(got[keep - w:], np.arange(n - w, n))
                    swaps += check_topk(got[: keep - w], ref["pooled"][0], keep - w,
                                        what=f"chunk {c} seq {b} head {g} kept set")
                newK.append(K[g, got])
                newV.append(V[g, got])
            held[b], held_v[b] = np.stack(newK), np.stack(newV)
            # the cache equals the held tokens and their summaries, bit for bit
            Kg, Vg = cache.token_kv(b, keep)
            np.testing.assert_array_equal(f64(Kg), held[b])
            np.testing.assert_array_equal(f64(Vg), held_v[b])
            NP = -(-keep // P)
            for g in range(Hkv):
                kmax, kmin = O.page_summaries(held[b][g], keep, P)
                np.testing.assert_array_equal(f64(cache.kmax[b, g, :, :NP]), kmax)
                np.testing.assert_array_equal(f64(cache.kmin[b, g, :, :NP]), kmin)
            assert int(cache.seq_len[b].item()) == keep
        st, bits = rkv.rkv_get_device_status(cache)
        assert st == rkv.RKV_OK and bits == 0
    if swaps == 0:
        # with no boundary swap the whole chain is the oracle's own chunked prefill
        for b in range(B):
            ref = O.prefill_chunked_unit(qs[b], chunks_k[b], chunks_v[b], keep1[b], kp[b])
            np.testing.assert_array_equal(ref["K"], held[b])
            np.testing.assert_array_equal(ref["V"], held_v[b])
    return cache, held, held_v


@pytest.mark.parametrize("name", list(CASES))
def test_chunked_prefill_matches_oracle(rkv, name):
    _run_chunks(rkv, CASES[name])


def test_chunked_prefill_then_decode(rkv):
    """Decode over a cache built by chunks: HSA output within tolerance of the oracle."""
    case = CASES["gqa4_two_seqs"]
    cache, held, held_v = _run_chunks(rkv, case)
    B, Hq, Hkv, P = case["B"], case["Hq"], case["Hkv"], case["page_size"]
    G = Hq // Hkv
    wl = W.custom(B=B, Hq=Hq, Hkv=Hkv, prompt_lens=[sum(ch[b] for ch in case["chunks"]) for b in range(B)],
                  budget=64, window=case["window"], page_size=P, steps=3)
    k1, k2 = [32] * B, [4] * B
    dws = rkv.decode_workspace(B, Hq, Hkv, cache.max_pages)
    for step in range(wl.steps):
        d = W.decode_tensors(wl, step, 0x5EED, 0, "cuda")
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        pg = torch.full((B, Hkv, 5), -9, dtype=torch.int32, device="cuda")
        ch = torch.full((B, Hkv, 128), -9, dtype=torch.int32, device="cuda")
        rkv.rkv_decode_step(cache, d["q"], d["k_new"], d["v_new"], k1, k2, out, sel_channels=ch, sel_pages=pg,
                            workspace=dws)
        for b in range(B):
            held[b] = np.concatenate([held[b], f64(d["k_new"][b])[:, None]], axis=1)
            held_v[b] = np.concatenate([held_v[b], f64(d["v_new"][b])[:, None]], axis=1)
            n = held[b].shape[1]
            for g in range(Hkv):
                qg = f64(d["q"][b, g * G:(g + 1) * G])
                kmax, kmin = O.page_summaries(held[b][g], n, P)
                gch = ch[b, g, :k1[b]].cpu().numpy()
                check_topk(gch, O.channel_select(qg, k1[b])[1], k1[b], what="channel set")
                gch = np.sort(gch)
                sig = O.page_scores(qg, kmax, kmin, gch)
                kk = min(k2[b], kmax.shape[1])
                pages = pg[b, g, :kk].cpu().numpy().astype(np.int64)
                check_topk(pages, sig, kk, what="page set")
                ref = O.sparse_attention(qg, held[b][g], held_v[b][g], n, pages, P)
                err = float(np.abs(f64(out[b, g * G:(g + 1) * G]) - ref).max())
                assert err <= ATOL_OUT, f"attention max-abs error {err}"
    st, _ = rkv.rkv_get_device_status(cache)
    assert st == rkv.RKV_OK


def test_chunked_prefill_flags_a_stale_held_len(rkv):
    """held_len that disagrees with the cache's seq_len is reported, not acted on silently."""
    case = dict(CASES["gqa1_w16"], chunks=[[64]])
    cache = _run_chunks(rkv, case, held_len_offset=16)
    st, bits = rkv.rkv_get_device_status(cache)
    assert st == rkv.RKV_ERR_DEVICE_DATA and bits & rkv.DEVERR_SEQ_LEN


def _chunked_full(rkv, n: int, units, chunk_tokens: int = 8192, seed: int = 0x5EED):
    """A bench workload prefilled in chunks as the bench times it (the same plan, the
    same launches), with sampled (sequence, KV head) units checked after every chunk."""
    from rkv_check import splits_for
    dev = torch.device("cuda")
    wl = W.workload(n)
    s = splits_for(wl, rkv)
    keep1, kp = [x["keep1"] for x in s], [x["pool_kernel"] for x in s]
    P, G, w = wl.page_size, wl.G, wl.window
    prompt = W.prefill_tensors(wl, seed, 0, dev, tail="zero")
    plan = W.chunk_plan(wl, chunk_tokens)
    max_pages = (max(keep1) + P - 1) // P + 8
    cache = rkv.PagedCache(wl.B, wl.Hkv, P, max_pages, dev, page_table=W.page_table(wl.B, (max_pages + 7) // 8 * 8,
                                                                                       seed, dev))
    kept = torch.full((wl.B, wl.Hkv, max(keep1)), -7, dtype=torch.int32, device=dev)
    held_len = [0] * wl.B
    held = {u: (np.zeros((0, 128)), np.zeros((0, 128))) for u in units}
    for c in range(len(plan)):
        ch = W.chunk_tensors(wl, prompt, plan, c, seed, 0, dev)
        rkv.rkv_prefill_chunk(ch["q_win"], ch["k"], ch["v"], ch["chunk_len"], held_len, keep1, kp, cache, kept)
        for (b, g) in units:
            m = plan[c][b]
            K = np.concatenate([held[(b, g)][0], f64(ch["k"][b, g, :m])])
            V = np.concatenate([held[(b, g)][1], f64(ch["v"][b, g, :m])])
            nn = K.shape[0]
            keep = min(keep1[b], nn)
            got = kept[b, g, :keep].cpu().numpy().astype(np.int64)
            assert np.all(np.diff(got) > 0)
            if nn > keep1[b]:
                ref = O.prefill_evict_unit(f64(ch["q_win"][b, g * G:(g + 1) * G]), K[None], keep1[b], kp[b])
                np.testing.assert_array_equal(got[keep - w:], np.arange(nn - w, nn))
                check_topk(got[: keep - w], ref["pooled"][0], keep - w, what=f"chunk {c} unit {(b, g)}")
            else:
                np.testing.assert_array_equal(got, np.arange(nn))
            held[(b, g)] = (K[got], V[got])
            Kg, Vg = cache.token_kv(b, keep)
            np.testing.assert_array_equal(f64(Kg[g]), K[got])
            np.testing.assert_array_equal(f64(Vg[g]), V[got])
            kmax, kmin = O.page_summaries(K[got], keep, P)
            NP = kmax.shape[1]
            np.testing.assert_array_equal(f64(cache.kmax[b, g, :, :NP]), kmax)
            np.testing.assert_array_equal(f64(cache.kmin[b, g, :, :NP]), kmin)
        held_len = [min(k, h + m) for k, h, m in zip(keep1, held_len, plan[c])]
        assert cache.seq_len.tolist() == held_len
    st, bits = rkv.rkv_get_device_status(cache)
    assert st == rkv.RKV_OK, bits


def test_chunked_workload2_llama_layer_32k(rkv):
    _chunked_full(rkv, 2, [(0, 0), (0, 5)])


def test_chunked_workload4_batched_ragged(rkv):
    wl = W.workload(4)
    _chunked_full(rkv, 4, [(int(np.argmax(wl.prompt_lens)), 2), (int(np.argmin(wl.prompt_lens)), 7)])
