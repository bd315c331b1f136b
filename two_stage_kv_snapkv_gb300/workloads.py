"""Seeded synthetic inputs for the RocketKV hot path.

This module only draws input tensors; it holds none of the method's arithmetic,
so both the CUDA path and the CPU oracle can be fed from it.  It depends on
torch only (no CUDA library), and draws on whatever device it is given: the
caller copies the same bytes to the other side.

The workloads stand in for the long-context benchmarks the RocketKV pages
evaluate on (Needle-in-a-Haystack, LongBench, RULER, SCBench with
Llama3.1-8B-Instruct): Llama3.1-8B-shaped attention layers (32 query / 8 KV
heads, head_dim 128, bf16), random keys/values with planted structure
(needle keys aligned to the queries, outlier channels, attention sinks).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def seed_for(*parts) -> int:
    """Mix integers / strings into one 63-bit torch seed (deterministic)."""
    h = 0x5EED
    for p in parts:
        if isinstance(p, str):
            for ch in p.encode():
                h = _splitmix64(h ^ ch)
        else:
            h = _splitmix64(h ^ (int(p) & _MASK64))
    return h & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, seed: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """N(0,1) samples drawn in fp32 and rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x.to(dtype)


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    prompt_lens: list            # per sequence
    budget: int
    window: int
    page_size: int
    steps: int
    pool_kernel: Optional[int] = None    # None: the library's default rule
    k1: Optional[int] = None             # None: derived from the split
    needles_per_head: int = 0
    outlier_channels: int = 0            # per KV head, keys scaled x8
    sinks: int = 0                       # first tokens, keys scaled x8
    layers: int = 1
    mt: bool = False                     # RocketKV-MT: no stage-1 eviction

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def Lmax(self) -> int:
        return max(self.prompt_lens)


def _uniform_lengths(B, lo, hi, seed):
    g = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def workload(n: int, seed: int = 0x5EED) -> Workload:
    """The benchmark workloads of this project, by number 1..6 (6: workload 4's batch
    under RocketKV-MT, HSA over the whole un-evicted prompts)."""
    if n == 1:   # tiny single layer, GQA 4, 4 needles per KV head
        return Workload("tiny_4k_gqa4", 1, 8, 2, 128, [4096], 256, 32, 16, 16,
                        pool_kernel=7, k1=64, needles_per_head=4)
    if n == 2:   # Llama3.1-8B-shaped layer, 32K prompt
        return Workload("llama8b_layer_32k", 1, 32, 8, 128, [32768], 512, 32, 16, 128,
                        pool_kernel=31, outlier_channels=4, sinks=4)
    if n == 3:   # extreme ratio, 109K prompt, 1 needle per KV head
        return Workload("llama8b_layer_109k", 1, 32, 8, 128, [109000], 256, 32, 16, 64,
                        pool_kernel=63, outlier_channels=4, sinks=4, needles_per_head=1)
    if n == 4:   # batched serving, 16 ragged sequences 8K..32K
        lens = _uniform_lengths(16, 8192, 32768, seed_for(seed, 4, "lengths"))
        return Workload("llama8b_batch16_8k_32k", 16, 32, 8, 128, lens, 2048, 32, 32, 256,
                        outlier_channels=4, sinks=4)
    if n == 5:   # 32-layer decode, batch 8, 64K prompts
        return Workload("llama8b_32layer_b8_64k", 8, 32, 8, 128, [65536] * 8, 4096, 32, 16, 64,
                        outlier_channels=4, sinks=4, layers=32)
    if n == 6:   # workload 4's batch with nothing evicted (RocketKV-MT)
        lens = _uniform_lengths(16, 8192, 32768, seed_for(seed, 4, "lengths"))
        return Workload("llama8b_batch16_8k_32k_mt", 16, 32, 8, 128, lens, 2048, 32, 32, 256,
                        outlier_channels=4, sinks=4, mt=True)
    raise ValueError(f"no workload {n}")


def custom(B=1, Hq=4, Hkv=2, d=128, prompt_lens=(512,), budget=64, window=8, page_size=16,
           steps=4, pool_kernel=5, k1=None, needles_per_head=0, outlier_channels=0, sinks=0,
           name="custom", mt=False) -> Workload:
    """A small workload for parity tests (sizes the oracle finishes in seconds)."""
    pl = list(prompt_lens)
    if len(pl) == 1 and B > 1:
        pl = pl * B
    return Workload(name, B, Hq, Hkv, d, pl, budget, window, page_size, steps,
                    pool_kernel=pool_kernel, k1=k1, needles_per_head=needles_per_head,
                    outlier_channels=outlier_channels, sinks=sinks, mt=mt)


# ---------------------------------------------------------------- structure
def _needle_dirs(wl: Workload, seed: int, layer: int) -> torch.Tensor:
    """One seeded unit direction per KV head, [Hkv, d] fp32 (CPU)."""
    u = torch.randn(wl.Hkv, wl.d, generator=_gen(seed_for(seed, layer, "needle_dir"), "cpu"))
    return u / u.norm(dim=1, keepdim=True)


def _needle_positions(wl: Workload, seed: int, layer: int) -> list:
    """Per (b, KV head): needle positions in the prefix [0, L_b - w)."""
    out = []
    for b in range(wl.B):
        g = _gen(seed_for(seed, layer, "needle_pos", b), "cpu")
        L = wl.prompt_lens[b]
        n_prefix = L - wl.window
        per = []
        for _h in range(wl.Hkv):
            per.append([int(x) for x in torch.randint(0, n_prefix, (wl.needles_per_head,), generator=g)])
        out.append(per)
    return out


def _outlier_channels(wl: Workload, seed: int, layer: int) -> torch.Tensor:
    """[Hkv, outlier_channels] channel ids (CPU, int64)."""
    g = _gen(seed_for(seed, layer, "outliers"), "cpu")
    return torch.stack([torch.randperm(wl.d, generator=g)[: wl.outlier_channels] for _ in range(wl.Hkv)])


def _scale_outliers(k: torch.Tensor, chans: torch.Tensor):
    """k: [..., Hkv, T, d] in place: x8 on each head's outlier channels."""
    for h in range(chans.shape[0]):
        for c in chans[h].tolist():
            k[..., h, :, c] *= 8


def prefill_tensors(wl: Workload, seed: int = 0x5EED, layer: int = 0, device="cpu",
                    tail: str = "zero") -> dict:
    """Prompt tensors: q_win [B,Hq,w,d], k/v [B,Hkv,Lmax,d] (bf16), prompt_len list.

    Rows at or beyond a sequence's prompt length are filled with ``tail``
    ("zero" or "nan"); the library must never use them.
    """
    B, Hq, Hkv, d, w, Lmax = wl.B, wl.Hq, wl.Hkv, wl.d, wl.window, wl.Lmax
    q_win = normal((B, Hq, w, d), seed_for(seed, layer, "q_win"), device)
    k = normal((B, Hkv, Lmax, d), seed_for(seed, layer, "k"), device)
    v = normal((B, Hkv, Lmax, d), seed_for(seed, layer, "v"), device)
    if wl.outlier_channels:
        chans = _outlier_channels(wl, seed, layer)
        kf = k.float()
        _scale_outliers(kf, chans)
        k = kf.to(torch.bfloat16)
    if wl.sinks:
        k[:, :, : wl.sinks, :] = (k[:, :, : wl.sinks, :].float() * 8).to(torch.bfloat16)
    if wl.needles_per_head:
        u = _needle_dirs(wl, seed, layer).to(device)
        pos = _needle_positions(wl, seed, layer)
        for b in range(B):
            for h in range(Hkv):
                for t in pos[b][h]:
                    k[b, h, t, :] = (2.0 * math.sqrt(d) * u[h]).to(torch.bfloat16)
        # window queries of every head in group h lean towards the needle direction
        qf = q_win.float()
        for h in range(Hq):
            qf[:, h] += math.sqrt(d) * u[h // wl.G]
        q_win = qf.to(torch.bfloat16)
    for b in range(B):
        L = wl.prompt_lens[b]
        if L < Lmax:
            fill = float("nan") if tail == "nan" else 0.0
            k[b, :, L:, :] = fill
            v[b, :, L:, :] = fill
    return dict(q_win=q_win.contiguous(), k=k.contiguous(), v=v.contiguous(),
                prompt_len=list(wl.prompt_lens))


def chunk_plan(wl: Workload, chunk_tokens: int) -> list:
    """Chunk lengths for a chunked prefill of the workload's prompts: [chunk][b].

    Every prompt is cut into the same number of near-equal chunks, ceil(Lmax /
    chunk_tokens) of them, fewer where a chunk would be shorter than the window.
    """
    nc = max(1, -(-wl.Lmax // chunk_tokens))
    while nc > 1 and min(wl.prompt_lens) // nc < wl.window:
        nc -= 1
    bounds = [[(L * i) // nc for i in range(nc + 1)] for L in wl.prompt_lens]
    return [[bb[c + 1] - bb[c] for bb in bounds] for c in range(nc)]


def chunk_tensors(wl: Workload, prompt: dict, plan: list, c: int, seed: int = 0x5EED, layer: int = 0,
                  device="cpu") -> dict:
    """Chunk c of a chunked prefill: its keys and values cut from the prompt's
    ([B,Hkv,max chunk,d], zero-padded), and its observation window -- the prompt's
    own for the last chunk, fresh seeded queries for the others."""
    B, Hkv, d = wl.B, wl.Hkv, wl.d
    cmax = max(plan[c])
    k = torch.zeros((B, Hkv, cmax, d), dtype=torch.bfloat16, device=device)
    v = torch.zeros_like(k)
    for b in range(B):
        s = sum(plan[i][b] for i in range(c))
        m = plan[c][b]
        k[b, :, :m] = prompt["k"][b, :, s:s + m]
        v[b, :, :m] = prompt["v"][b, :, s:s + m]
    if c == len(plan) - 1:
        q = prompt["q_win"]
    else:
        q = normal((B, wl.Hq, wl.window, d), seed_for(seed, layer, "q_win_chunk", c), device)
    return dict(q_win=q, k=k, v=v, chunk_len=list(plan[c]))


def decode_tensors(wl: Workload, step: int, seed: int = 0x5EED, layer: int = 0, device="cpu") -> dict:
    """One decode step's inputs: q [B,Hq,d], k_new / v_new [B,Hkv,d] (bf16)."""
    B, Hq, Hkv, d = wl.B, wl.Hq, wl.Hkv, wl.d
    q = normal((B, Hq, d), seed_for(seed, layer, "dec_q", step), device)
    kn = normal((B, Hkv, d), seed_for(seed, layer, "dec_k", step), device)
    vn = normal((B, Hkv, d), seed_for(seed, layer, "dec_v", step), device)
    if wl.outlier_channels:
        chans = _outlier_channels(wl, seed, layer)
        kf = kn.float().unsqueeze(2)
        _scale_outliers(kf, chans)
        kn = kf.squeeze(2).to(torch.bfloat16)
    if wl.needles_per_head:
        u = _needle_dirs(wl, seed, layer).to(device)
        qf = q.float()
        for h in range(Hq):
            qf[:, h] += math.sqrt(d) * u[h // wl.G]
        q = qf.to(torch.bfloat16)
    return dict(q=q.contiguous(), k_new=kn.contiguous(), v_new=vn.contiguous())


def page_table(B: int, max_pages: int, seed: int = 0x5EED, device="cpu", spare: int = 0) -> torch.Tensor:
    """[B, max_pages] int32 physical page ids: a seeded shuffle of B*max_pages+spare ids.

    The shuffle makes every page gather truly indirect.
    """
    n_phys = B * max_pages + spare
    perm = torch.randperm(n_phys, generator=_gen(seed_for(seed, "pages"), "cpu"))[: B * max_pages]
    return perm.view(B, max_pages).to(torch.int32).to(device)
