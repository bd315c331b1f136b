"""Host-side checks of the seeded input generators and the bench's request plans (CPU)."""
import torch

from two_stage_kv_snapkv_gb300 import workloads as W


def test_chunk_plan_partitions_every_prompt():
    """Chunked prefill plans: the same number of chunks for every sequence, each at
    least the window long, summing to the prompt length."""
    for n in (1, 2, 3, 4, 5, 6):
        wl = W.workload(n)
        plan = W.chunk_plan(wl, 8192)
        assert len(plan) >= 1
        for b, L in enumerate(wl.prompt_lens):
            lens = [c[b] for c in plan]
            assert sum(lens) == L
            assert min(lens) >= wl.window
            assert max(lens) - min(lens) <= 1          # near-equal cuts
    # a prompt too short for the requested chunk count falls back to fewer chunks
    wl = W.custom(B=1, prompt_lens=[50], window=16)
    assert W.chunk_plan(wl, 8) == [[16], [17], [17]]   # 7 chunks of ~8 would be shorter than w


def test_chunk_tensors_cut_the_prompt():
    wl = W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[300, 170], window=8)
    prompt = W.prefill_tensors(wl, 7, 0, "cpu")
    plan = W.chunk_plan(wl, 128)
    got_k = [[], []]
    for c in range(len(plan)):
        ch = W.chunk_tensors(wl, prompt, plan, c, 7, 0, "cpu")
        assert ch["chunk_len"] == plan[c]
        assert ch["k"].shape == (2, 2, max(plan[c]), 128)
        for b in range(2):
            got_k[b].append(ch["k"][b, :, :plan[c][b]])
            assert torch.count_nonzero(ch["k"][b, :, plan[c][b]:]) == 0   # padding rows are zero
        if c == len(plan) - 1:
            assert torch.equal(ch["q_win"], prompt["q_win"])               # the prompt's own window
        else:
            assert not torch.equal(ch["q_win"], prompt["q_win"])
    for b, L in enumerate(wl.prompt_lens):
        assert torch.equal(torch.cat(got_k[b], dim=1), prompt["k"][b, :, :L])


def test_generators_are_seeded_and_layer_specific():
    wl = W.workload(1)
    a = W.prefill_tensors(wl, 11, 0, "cpu")
    b = W.prefill_tensors(wl, 11, 0, "cpu")
    c = W.prefill_tensors(wl, 11, 1, "cpu")
    assert torch.equal(a["k"], b["k"]) and torch.equal(a["q_win"], b["q_win"])
    assert not torch.equal(a["k"], c["k"])
    d0 = W.decode_tensors(wl, 0, 11, 0, "cpu")
    d1 = W.decode_tensors(wl, 1, 11, 0, "cpu")
    assert not torch.equal(d0["q"], d1["q"])


def test_page_table_is_a_permutation():
    pt = W.page_table(4, 24, seed=3, spare=5)
    ids = pt.flatten().tolist()
    assert len(set(ids)) == len(ids) == 96
    assert min(ids) >= 0 and max(ids) < 4 * 24 + 5


def test_benchmark_workload_shapes():
    """The six workloads have the shapes of the configurations they stand in for."""
    w = [W.workload(n) for n in range(1, 7)]
    assert (w[0].B, w[0].Hq, w[0].Hkv, w[0].prompt_lens, w[0].budget, w[0].window, w[0].page_size,
            w[0].steps, w[0].pool_kernel, w[0].k1, w[0].needles_per_head) == (1, 8, 2, [4096], 256, 32, 16, 16, 7, 64, 4)
    assert (w[1].B, w[1].Hq, w[1].Hkv, w[1].prompt_lens, w[1].budget, w[1].page_size, w[1].steps, w[1].pool_kernel,
            w[1].outlier_channels, w[1].sinks) == (1, 32, 8, [32768], 512, 16, 128, 31, 4, 4)
    assert (w[2].prompt_lens, w[2].budget, w[2].steps, w[2].pool_kernel, w[2].needles_per_head) == \
        ([109000], 256, 64, 63, 1)
    assert (w[3].B, w[3].budget, w[3].page_size, w[3].steps) == (16, 2048, 32, 256)
    assert all(8192 <= L <= 32768 for L in w[3].prompt_lens) and len(set(w[3].prompt_lens)) > 8
    assert (w[4].B, w[4].prompt_lens, w[4].budget, w[4].layers, w[4].steps) == (8, [65536] * 8, 4096, 32, 64)
    assert w[5].mt and w[5].prompt_lens == w[3].prompt_lens and not w[3].mt
    for x in w:
        assert x.d == 128 and x.Hq % x.Hkv == 0


def test_outlier_channels_and_sinks_scale_the_plain_draw():
    """Outlier channels (per KV head) and the first tokens' keys are the plain N(0,1)
    draw times 8, rounded to bf16; everything else is the plain draw."""
    plain = W.custom(B=1, Hq=4, Hkv=2, prompt_lens=[256], window=8)
    wl = W.custom(B=1, Hq=4, Hkv=2, prompt_lens=[256], window=8, outlier_channels=4, sinks=4)
    a = W.prefill_tensors(plain, 5, 0, "cpu")["k"].float()
    b = W.prefill_tensors(wl, 5, 0, "cpu")["k"].float()
    big = (b != a)
    for h in range(2):
        # the scaled channels of head h: 4 of them, over every token past the sinks
        chans = big[0, h, 4:].any(dim=0).nonzero().flatten().tolist()
        assert len(chans) == 4
        sel = b[0, h, 4:, chans]
        assert torch.equal(sel, (a[0, h, 4:, chans] * 8).to(torch.bfloat16).float())
        assert 6.0 < float(sel.std()) < 10.0 and float(b[0, h, 4:, [c for c in range(128) if c not in chans]].std()) < 1.3
        # sink rows: every channel x8 (outlier channels x64)
        x = a[0, h, :4].clone()
        x[:, chans] = (x[:, chans] * 8).to(torch.bfloat16).float()
        assert torch.equal(b[0, h, :4], (x * 8).to(torch.bfloat16).float())
    d0, d1 = W.decode_tensors(plain, 3, 5, 0, "cpu"), W.decode_tensors(wl, 3, 5, 0, "cpu")
    diff = (d0["k_new"] != d1["k_new"])[0]
    assert int(diff.sum()) <= 8 and torch.equal(d0["q"], d1["q"]) and torch.equal(d0["v_new"], d1["v_new"])


def test_needles_are_planted_and_the_queries_lean_towards_them():
    """Needle keys are 2 sqrt(d) u_h at seeded prefix positions; the window and decode
    queries of the heads in group h carry sqrt(d) u_h on top of N(0,1)."""
    wl = W.custom(B=2, Hq=4, Hkv=2, prompt_lens=[300, 200], window=8, needles_per_head=3)
    p = W.prefill_tensors(wl, 9, 0, "cpu")
    k = p["k"].float()
    for b, L in enumerate(wl.prompt_lens):
        for h in range(2):
            norms = k[b, h, :L].norm(dim=1)
            hits = (norms > 20.0).nonzero().flatten().tolist()   # 2 sqrt(128) = 22.6
            assert 1 <= len(hits) <= 3 and max(hits) < L - wl.window
            u = k[b, h, hits[0]] / k[b, h, hits[0]].norm()
            for t in hits:
                assert torch.allclose(k[b, h, t], k[b, h, hits[0]])
            for qh in (2 * h, 2 * h + 1):
                cos = (p["q_win"][b, qh].float() @ u) / p["q_win"][b, qh].float().norm(dim=1)
                assert float(cos.mean()) > 0.6
            dq = W.decode_tensors(wl, 0, 9, 0, "cpu")["q"][b, 2 * h].float()
            assert float(dq @ u / dq.norm()) > 0.5
        assert torch.count_nonzero(k[b, :, L:]) == 0   # rows past the prompt
