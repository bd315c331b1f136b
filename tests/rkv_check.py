"""Shared helpers of the GPU parity tests: run the library on seeded inputs and
compare with the CPU oracle.

Comparison rules (the tolerances the hot path is held to):
  * page summaries and cache contents: bit-exact;
  * kept-token / channel / page sets: exact, except elements whose oracle score lies
    within 1e-5 relative of the oracle's k-th score (near ties, where fp32 on the
    GPU and fp64 in the oracle may order differently);
  * attention outputs: max-abs 2e-3 against the oracle evaluated on the GPU's
    page set (bf16 inputs, fp32 accumulation).
"""
from __future__ import annotations


import numpy as np
import torch

from oracle import rkv_oracle as O
from two_stage_kv_snapkv_gb300 import workloads as W

REL_TIE = 1e-5
ATOL_OUT = 2e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def check_topk(gpu_idx, scores: np.ndarray, k: int, rel: float = REL_TIE, what: str = "") -> int:
    """Assert a GPU top-k set is a valid top-k of the oracle scores; return #tie swaps."""
    gpu_idx = np.asarray(gpu_idx).astype(np.int64)
    assert len(gpu_idx) == k, f"{what}: {len(gpu_idx)} selected, expected {k}"
    assert len(set(gpu_idx.tolist())) == k, f"{what}: duplicate selections"
    if k == 0:
        return 0
    assert gpu_idx.min() >= 0 and gpu_idx.max() < len(scores), f"{what}: index out of range"
    order = np.lexsort((np.arange(len(scores)), -scores))
    ref = set(order[:k].tolist())
    kth = scores[order[k - 1]]
    diff = set(gpu_idx.tolist()) ^ ref
    band = rel * abs(kth)
    bad = [i for i in diff if abs(scores[i] - kth) > band]
    assert not bad, f"{what}: {len(bad)} selections outside the tie band, kth={kth!r}: " + \
        str([(i, scores[i], i in ref) for i in sorted(bad)[:6]])
    return len(diff)


def splits_for(wl: W.Workload, rkv) -> list:
    out = []
    for L in wl.prompt_lens:
        if wl.mt:
            s = rkv.rkv_split_ratio_mt(L, wl.budget, wl.d, wl.page_size, wl.k1 or 0)
        else:
            s = rkv.rkv_split_ratio(L, wl.budget, wl.d, wl.page_size, wl.window, wl.k1 or 0)
        if wl.pool_kernel:
            s["pool_kernel"] = wl.pool_kernel
        out.append(s)
    return out


class DeviceRun:
    """One layer of a workload on the GPU: inputs, cache, prefill, decode steps."""

    def __init__(self, wl: W.Workload, rkv, seed: int = 0x5EED, layer: int = 0, gen_device="cpu",
                 tail="nan", fill=float("nan"), api: str = "step", max_pages_req: int = 0):
        self.wl, self.rkv, self.seed, self.layer = wl, rkv, seed, layer
        self.api = api   # "step": rkv_decode_step; "separate": rkv_append_page_summary + rkv_decode_hsa
        self.dev = torch.device("cuda")
        self.inputs = W.prefill_tensors(wl, seed, layer, gen_device, tail=tail)
        self.gpu_in = {k: (v.to(self.dev) if torch.is_tensor(v) else v) for k, v in self.inputs.items()}
        self.splits = splits_for(wl, rkv)
        self.keep1 = [s["keep1"] for s in self.splits]
        self.k1 = [s["k1"] for s in self.splits]
        self.k2 = [s["k2"] for s in self.splits]
        self.kp = [s["pool_kernel"] for s in self.splits]
        P = wl.page_size
        max_pages = (max(self.keep1) + wl.steps + P - 1) // P
        max_pages = (max_pages + 7) // 8 * 8
        if max_pages_req:   # a larger page capacity than the request needs
            max_pages = max(max_pages, (max_pages_req + 7) // 8 * 8)
        spare = 5
        pt = W.page_table(wl.B, max_pages, seed, self.dev, spare=spare)
        self.cache = rkv.PagedCache(wl.B, wl.Hkv, P, max_pages, self.dev, page_table=pt,
                                    num_phys_pages=wl.B * max_pages + spare, fill=fill)
        self.kept = torch.full((wl.B, wl.Hkv, max(self.keep1)), -7, dtype=torch.int32, device=self.dev)
        self.pooled = torch.full((wl.B, wl.Hkv, wl.Lmax), float("nan"), dtype=torch.float32, device=self.dev)
        self.dws = rkv.decode_workspace(wl.B, wl.Hq, wl.Hkv, self.cache.max_pages, self.dev)

    def prefill(self):
        g = self.gpu_in
        self.rkv.rkv_prefill_evict(g["q_win"], g["k"], g["v"], g["prompt_len"], self.keep1, self.kp, self.cache,
                                   self.kept, pooled_scores=self.pooled)

    def decode_step(self, step: int, edit=None):
        """One decode step; `edit(d)` may change the step's tensors before the call."""
        wl = self.wl
        d = W.decode_tensors(wl, step, self.seed, self.layer, self.dev)
        if edit is not None:
            edit(d)
        out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device=self.dev)
        ch = torch.full((wl.B, wl.Hkv, 128), -9, dtype=torch.int32, device=self.dev)
        pg = torch.full((wl.B, wl.Hkv, max(self.k2) + 1), -9, dtype=torch.int32, device=self.dev)
        if self.api == "step":
            self.rkv.rkv_decode_step(self.cache, d["q"], d["k_new"], d["v_new"], self.k1, self.k2, out,
                                     sel_channels=ch, sel_pages=pg, workspace=self.dws)
        else:
            self.rkv.rkv_append_page_summary(self.cache, d["k_new"].unsqueeze(2).contiguous(),
                                             d["v_new"].unsqueeze(2).contiguous(), 1)
            self.rkv.rkv_decode_hsa(self.cache, d["q"], self.k1, self.k2, out, sel_channels=ch, sel_pages=pg,
                                    workspace=self.dws)
        return d, out, ch, pg

    def status(self):
        return self.rkv.rkv_get_device_status(self.cache)


class OracleUnit:
    """The oracle's view of one (sequence, KV head): stage 1 on the prompt, then the
    compressed cache built from the GPU's (validated) kept set and grown per step."""

    def __init__(self, run: DeviceRun, b: int, g: int):
        wl = run.wl
        self.b, self.g, self.wl = b, g, wl
        G = wl.G
        L = wl.prompt_lens[b]
        self.L = L
        q = f64(run.inputs["q_win"][b, g * G:(g + 1) * G])
        k = f64(run.inputs["k"][b, g:g + 1, :L])
        self.v_all = f64(run.inputs["v"][b, g, :L])
        self.k_all = k[0]
        self.res = O.prefill_evict_unit(q, k, run.keep1[b], run.kp[b])
        self.keep1 = run.keep1[b]

    def check_prefill(self, run: DeviceRun) -> int:
        wl, b, g = self.wl, self.b, self.g
        Lp = self.L - wl.window
        gp = run.pooled[b, g, :Lp].double().cpu().numpy()
        ref = self.res["pooled"][0]
        evicts = any(k < L for k, L in zip(run.keep1, wl.prompt_lens))
        if Lp > 0 and evicts:   # when no sequence evicts, the scoring (and S') is skipped
            scale = max(float(ref.max()), 1e-30)
            err = np.abs(gp - ref)
            assert np.all(err <= 1e-4 * np.abs(ref) + 1e-6 * scale), \
                f"pooled scores differ: max rel {float((err / (np.abs(ref) + 1e-30)).max())}"
        kept = run.kept[b, g, :self.keep1].cpu().numpy().astype(np.int64)
        assert np.all(np.diff(kept) > 0), "kept positions not ascending"
        np.testing.assert_array_equal(kept[self.keep1 - wl.window:], np.arange(Lp, self.L))
        swaps = check_topk(kept[: self.keep1 - wl.window], ref, self.keep1 - wl.window, what="stage-1 kept set")
        self.kept = kept
        self.Kc = self.k_all[kept].copy()
        self.Vc = self.v_all[kept].copy()
        self.n = self.keep1
        return swaps

    def check_cache(self, run: DeviceRun):
        """Cache pages and summaries equal the oracle's, bit for bit."""
        b, g, P = self.b, self.g, self.wl.page_size
        K, V = run.cache.token_kv(b, self.n)
        np.testing.assert_array_equal(f64(K[g]), self.Kc[: self.n])
        np.testing.assert_array_equal(f64(V[g]), self.Vc[: self.n])
        kmax, kmin = O.page_summaries(self.Kc, self.n, P)
        NP = kmax.shape[1]
        np.testing.assert_array_equal(f64(run.cache.kmax[b, g, :, :NP]), kmax)
        np.testing.assert_array_equal(f64(run.cache.kmin[b, g, :, :NP]), kmin)
        assert int(run.cache.seq_len[b].item()) == self.n

    def step(self, run: DeviceRun, d: dict, out, ch, pg, check_cache=False) -> dict:
        wl, b, g, P = self.wl, self.b, self.g, self.wl.page_size
        G = wl.G
        self.Kc = np.concatenate([self.Kc[: self.n], f64(d["k_new"][b, g])[None]])
        self.Vc = np.concatenate([self.Vc[: self.n], f64(d["v_new"][b, g])[None]])
        self.n += 1
        if check_cache:
            self.check_cache(run)
        qg = f64(d["q"][b, g * G:(g + 1) * G])
        kmax, kmin = O.page_summaries(self.Kc, self.n, P)
        k1, k2 = run.k1[b], run.k2[b]
        chans, a = O.channel_select(qg, k1)
        gch = ch[b, g, :k1].cpu().numpy()
        check_topk(gch, a, k1, what="channel set")
        assert np.all(ch[b, g, k1:].cpu().numpy() == -1)
        gch = np.sort(gch)
        sig = O.page_scores(qg, kmax, kmin, gch)
        NP = kmax.shape[1]
        kk = min(k2, NP)
        gpages = pg[b, g, :kk].cpu().numpy().astype(np.int64)
        assert np.all(np.diff(gpages) > 0), "page set not ascending"
        if pg.shape[-1] > kk:
            assert int(pg[b, g, kk].item()) == -1
        swaps = check_topk(gpages, sig, kk, what="page set")
        ref = O.sparse_attention(qg, self.Kc, self.Vc, self.n, gpages, P)
        got = f64(out[b, g * G:(g + 1) * G])
        err = float(np.abs(got - ref).max())
        assert err <= ATOL_OUT, f"attention max-abs error {err}"
        return dict(err=err, swaps=swaps, sig=sig, pages=gpages)
