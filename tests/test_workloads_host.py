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
