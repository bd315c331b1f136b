#!/usr/bin/env python
"""Benchmark of the RocketKV decode-time hot path on one GB300 (or N, one per rank).

One bench step is one pass of the whole hot path over one request of the
workload: the adaptive split, stage-1 SnapKV++ eviction of the prompt
(rkv_prefill_evict, which also builds the page summaries), then every decode step
(rkv_decode_step: append the new token + the HSA step, one launch).  Inputs are seeded,
synthetic and resident in HBM before timing.  L2 is flushed (a 256 MB write)
before the prefill, and before every decode step whose compulsory bytes fit in L2,
outside the timed intervals.  Steps that read more than L2 holds (the batch-16
workloads) and the multi-layer workload, whose layers stream far more than L2
between two steps of a layer, run back to back: their inputs are larger than L2.

The metric is decode steps per second per layer over the whole job, prefill time
included: decode_steps * K / sum(pass time).  Each pass's prefill runs as a CUDA
graph; its decode steps run as one graph (the decode loop) where they run back to
back, else one graph a step with the L2 flush between them.  CUDA events on the
launching stream time each graph.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2]
    python bench.py --impl reference     # the CPU oracle, timed on this host
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from two_stage_kv_snapkv_gb300 import workloads as W  # noqa: E402

METRIC = "HSA decode steps/s per layer & achieved HBM GB/s vs GB300 peak; prefill evict ms"
UNIT = "decode steps/s per layer"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5,
                    help="1..6 (5, the default: 32 Llama3.1-8B-shaped layers, batch 8, 64K prompts; 2: one layer, 32K "
                         "prompt; 4: batch 16, 8K-32K prompts; 6: workload 4's batch under RocketKV-MT)")
    ap.add_argument("--seed", type=int, default=0x5EED)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-decode-steps", type=int, default=0, help="decode steps per oracle sample (0: all)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="repeat the oracle sample until this much CPU time")
    ap.add_argument("--flush-steps", choices=["auto", "always"], default="auto",
                    help="flush L2 before every decode step of a one-layer workload: always, or (auto) only when a "
                         "step's compulsory bytes fit in L2")
    ap.add_argument("--flush", choices=["write", "clean"], default="write",
                    help="L2 flush before timed intervals: write a 256 MB buffer (default), or write it and then read "
                         "another 256 MB buffer so no dirty line is left for the timed kernel to write back (clean)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batch-16 (workload 4) decode measurement added to the default workload's line")
    ap.add_argument("--prefill-chunk", type=int, default=8192,
                    help="also time a chunked prefill of the same prompts with chunks of about this many tokens "
                         "(0: skip)")
    ap.add_argument("--one-layer", action="store_true", help="run only layer 0 of a multi-layer workload")
    ap.add_argument("--mode", choices=["hsa", "quest", "sparq"], default="hsa",
                    help="decode selection: HSA (default), Quest-only (every channel), SparQ-only (one-token pages)")
    ap.add_argument("--ncu-every-kernel", action="store_true",
                    help="one eager launch of every library kernel, no warm-up (for an ncu launch list)")
    ap.add_argument("--ncu", action="store_true", help="one plain pass, no graphs (for an ncu launch list)")
    ap.add_argument("--decode-path", choices=["auto", "split", "fused"], default="auto",
                    help="decode implementation: one fused launch per step (auto/fused) or four kernels")
    return ap.parse_args()


# --------------------------------------------------------------------------- peaks / clocks
def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(hbm_gbs=6800.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.skip = 0
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        # start timing only once the sampler is writing (nvidia-smi takes a moment to
        # start), so that a short timed region still gets its samples; at most 3 s
        t0 = time.time()
        while self.proc is not None and self.proc.poll() is None and time.time() - t0 < 3.0:
            if os.path.getsize(self.tmp.name) > 0:
                break
            time.sleep(0.01)
        with open(self.tmp.name) as f:   # samples taken before the timed region
            self.skip = sum(1 for line in f if line.endswith("\n"))
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if len(rows) > self.skip:   # keep only the samples taken during the timed region
            rows = rows[self.skip:]
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit()) if rows else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=smax, reasons=reasons,
                    samples=len(rows))


# --------------------------------------------------------------------------- workload setup
class Setup:
    """Everything one rank needs for K passes of one workload (layer 0)."""

    def __init__(self, wl: W.Workload, rkv, seed: int, dev, layer: int = 0, share: "Setup | None" = None,
                 mode: str = "hsa"):
        self.wl, self.rkv, self.dev, self.seed, self.layer, self.mode = wl, rkv, dev, seed, layer, mode
        self.inp = W.prefill_tensors(wl, seed, layer, dev, tail="zero")
        self.dec = [W.decode_tensors(wl, t, seed, layer, dev) for t in range(wl.steps)]
        for d in self.dec:
            d["k_new"] = d["k_new"].unsqueeze(2).contiguous()
            d["v_new"] = d["v_new"].unsqueeze(2).contiguous()
        self.splits = []
        for L in wl.prompt_lens:
            if wl.mt:
                s = rkv.rkv_split_ratio_mt(L, wl.budget, wl.d, wl.page_size, wl.k1 or 0)
            else:
                s = rkv.rkv_split_ratio(L, wl.budget, wl.d, wl.page_size, wl.window, wl.k1 or 0)
            if wl.pool_kernel:
                s["pool_kernel"] = wl.pool_kernel
            self.splits.append(s)
        self.keep1 = [s["keep1"] for s in self.splits]
        # Quest-only: HSA with every channel; SparQ-only: one-token pages, the same token budget
        self.k1 = [s["k1"] if mode != "quest" else wl.d for s in self.splits]
        self.k2 = [s["k2"] for s in self.splits]
        self.k_tokens = [k * wl.page_size for k in self.k2]
        self.kp = [s["pool_kernel"] for s in self.splits]
        P = wl.page_size
        max_pages = (max(self.keep1) + wl.steps + P - 1) // P
        max_pages = (max_pages + 7) // 8 * 8
        pt = W.page_table(wl.B, max_pages, seed, dev)
        self.cache = rkv.PagedCache(wl.B, wl.Hkv, P, max_pages, dev, page_table=pt)
        self.kept = torch.empty((wl.B, wl.Hkv, max(self.keep1)), dtype=torch.int32, device=dev)
        # layers run one after another on one stream, so they can share the scratch
        self.pws = share.pws if share else rkv.prefill_workspace(wl.B, wl.Hq, wl.Hkv, wl.window, wl.Lmax, dev)
        self.dws = share.dws if share else rkv.decode_workspace(wl.B, wl.Hq, wl.Hkv, self.cache.max_pages, dev)
        self.sws = self.skt = None
        if mode == "sparq":
            self.sws = share.sws if share else rkv.sparq_workspace(wl.B, wl.Hq, wl.Hkv, self.cache.max_pages, P, dev)
            # the channel-major key copy SparQ scores from (per layer: it holds the keys)
            self.skt = rkv.sparq_keys(self.cache, dev)
        self.out = torch.empty((wl.steps, wl.B, wl.Hq, 128), dtype=torch.float32, device=dev)
        self.flush_buf = share.flush_buf if share else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        # read after the write, so the flush leaves L2 holding clean lines of this buffer
        # instead of 129 MB of dirty ones that the timed kernel would have to write back
        self.flush_read = share.flush_read if share else torch.ones(256 << 20, dtype=torch.uint8, device=dev)
        self.flush_mode = share.flush_mode if share else "write"

    # one call each, on the current stream
    def prefill(self):
        i = self.inp
        self.rkv.rkv_prefill_evict(i["q_win"], i["k"], i["v"], i["prompt_len"], self.keep1, self.kp, self.cache,
                                   self.kept, workspace=self.pws)
        if self.skt is not None:   # the cache was rewritten: the key copy starts empty
            self.skt[:self.wl.B * self.wl.Hkv * 4].zero_()

    def decode(self, t: int):
        d = self.dec[t]
        self.step(d["q"], d["k_new"], d["v_new"], self.out[t])

    def step(self, q, k_new, v_new, out):
        """One decode step of this mode: append the token, then select and attend."""
        if self.mode == "sparq":
            self.rkv.rkv_append_page_summary(self.cache, k_new, v_new, 1)
            self.rkv.rkv_decode_sparq(self.cache, q, self.k1, self.k_tokens, out, workspace=self.sws,
                                      keys_t=self.skt)
        else:
            self.rkv.rkv_decode_step(self.cache, q, k_new, v_new, self.k1, self.k2, out, workspace=self.dws)

    def flush(self):
        """Evict L2 before a timed interval: write a 256 MB buffer (twice L2); in the
        "clean" mode, then read another 256 MB buffer so the write's dirty lines are
        written back here rather than inside the timed kernel."""
        self.flush_buf.zero_()
        if self.flush_mode == "clean":
            self.flush_read.view(torch.int64).max()

    # ------------------------------------------------------------ byte accounting
    def decode_bytes(self, t: int) -> dict:
        """Compulsory HBM bytes of decode step t, by kernel (the method must move these)."""
        wl = self.wl
        P = wl.page_size
        summ = kv = sync = 0
        for b in range(wl.B):
            n = self.keep1[b] + t + 1
            NP = -(-n // P)
            if self.mode == "sparq":
                # the chosen channels of every key from the channel-major copy, the chosen
                # tokens' K and V rows; the copy takes the step's new key (at the first
                # step every key: its build), read as a row and written along the channels
                summ += wl.Hkv * n * self.k1[b] * 2
                kv += wl.Hkv * min(self.k_tokens[b], n) * 128 * 2 * 2
                sync += wl.Hkv * (n if t == 0 else 1) * 128 * 2 * 2
            else:
                summ += wl.Hkv * 2 * self.k1[b] * NP * 2
                kv += wl.Hkv * min(self.k2[b], NP) * P * 128 * 2 * 2
        q = wl.B * wl.Hq * 128 * 2
        out = wl.B * wl.Hq * 128 * 4
        append = wl.B * wl.Hkv * (128 * 2 * 2 * 2 + 128 * 2 * 2 * 2)   # new k,v read+write, summaries
        total = summ + kv + q + out + append
        total += sync
        return dict(hsa_score=summ + q, hsa_attend=kv + q + out, append_small=append, hsa_step=total,
                    sparq_score=summ + q, sparq_attend=kv + q + out, sparq_keys_sync=sync, step_total=total)

    def prefill_bytes(self) -> dict:
        """Stage-1 bytes per layer: `compulsory` reads the prompt's keys once and reads
        and writes the survivors' K and V (what the method must move); `moved` is what
        the two scoring passes (row statistics, then column sums) actually stream, the
        keys twice."""
        wl = self.wl
        # stage-1 scoring reads K once per pass; without eviction (RocketKV-MT) it is skipped
        kbytes = 0 if wl.mt else sum(wl.Hkv * L * 128 * 2 for L in wl.prompt_lens)
        surv = sum(wl.Hkv * k * 128 * 2 * 2 * 2 for k in self.keep1)   # K+V read and written
        return dict(snap_stats=kbytes, snap_colsum=kbytes, snap_compact=surv, compulsory=kbytes + surv,
                    moved=2 * kbytes + surv)


def selection_recall(setup: Setup) -> dict:
    """Exact-TopK recall of HSA's page choice on this workload (outside any timed region):
    one eager pass, the library's recall diagnostic after the first and the last decode
    step, over every (sequence, KV head)."""
    rkv, wl = setup.rkv, setup.wl
    stride = max(setup.k2) + 1
    pg = torch.empty((wl.B, wl.Hkv, stride), dtype=torch.int32, device=setup.dev)
    k_tokens = [k * wl.page_size for k in setup.k2]
    setup.prefill()
    rec, mass = [], []
    for t in range(wl.steps):
        d = setup.dec[t]
        rkv.rkv_decode_step(setup.cache, d["q"], d["k_new"], d["v_new"], setup.k1, setup.k2, setup.out[t],
                            sel_pages=pg, workspace=setup.dws)
        if t in (0, wl.steps - 1):
            r, m = rkv.rkv_exact_topk_recall(setup.cache, d["q"], pg, k_tokens)
            rec.append(r.flatten())
            mass.append(m.flatten())
    r, m = torch.cat(rec).double(), torch.cat(mass).double()
    return dict(token_recall_mean=round(float(r.mean()), 4), token_recall_min=round(float(r.min()), 4),
                mass_recall_mean=round(float(m.mean()), 4), mass_recall_min=round(float(m.min()), 4),
                k_tokens=self_or_range(k_tokens), steps=[0, wl.steps - 1],
                what="share of the exact top-k_tokens tokens (attention summed over the GQA group) and of their "
                     "attention mass inside the pages HSA selected")


def chunked_prefill(setup: Setup, stream, chunk_tokens: int, reps: int) -> dict:
    """The same prompts prefilled in chunks (rkv_prefill_chunk per chunk, the stage-1
    budget re-enforced at every chunk), outside the main timed region: one CUDA graph
    per request, L2 flushed before each replay, 3 untimed replays first."""
    rkv, wl = setup.rkv, setup.wl
    plan = W.chunk_plan(wl, chunk_tokens)
    chunks = [W.chunk_tensors(wl, setup.inp, plan, c, setup.seed, 0, setup.dev) for c in range(len(plan))]
    cache = rkv.PagedCache(wl.B, wl.Hkv, wl.page_size, setup.cache.max_pages, setup.dev,
                           page_table=setup.cache.page_table)
    kept = torch.empty_like(setup.kept)
    held = [[0] * wl.B]
    for c in range(len(plan)):
        held.append([min(k, h + m) for k, h, m in zip(setup.keep1, held[c], plan[c])])
    total = max(h + m for c in range(len(plan)) for h, m in zip(held[c], plan[c]))
    ws = rkv.prefill_chunk_workspace(wl.B, wl.Hq, wl.Hkv, wl.window, total, setup.dev)

    def run():
        cache.seq_len.zero_()
        for c, ch in enumerate(chunks):
            rkv.rkv_prefill_chunk(ch["q_win"], ch["k"], ch["v"], ch["chunk_len"], held[c], setup.keep1, setup.kp,
                                  cache, kept, workspace=ws)

    run()
    torch.cuda.synchronize()
    st, bits = rkv.rkv_get_device_status(cache, stream)
    if st != rkv.RKV_OK or cache.seq_len.tolist() != held[-1]:
        raise RuntimeError(f"chunked prefill: device status {st} bits {bits}")
    n0 = rkv.rkv_launch_count()
    g = capture(run, stream)
    launches = rkv.rkv_launch_count() - n0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for i in range(reps + 3):
        setup.flush()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        stream.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    return dict(chunk_tokens=chunk_tokens, chunks=len(plan), chunk_len=self_or_range([m for p in plan for m in p]),
                ms=round(statistics.mean(times), 4), launches=launches, replays=reps,
                what="whole request: every chunk gathered with the survivors, scored, re-evicted to keep1 and "
                     "written back to the pages")


def ncu_every_kernel(setup: Setup) -> None:
    """One launch of every kernel of the library on this workload, eagerly and with no
    warm-up, for an ncu launch list with DRAM counters (`--ncu-every-kernel`): stage 1,
    the fused and the four-kernel decode steps, a multi-token append, the recall
    diagnostic, the SparQ-only step and two chunks of a chunked prefill."""
    rkv, wl = setup.rkv, setup.wl
    setup.prefill()                       # the six stage-1 kernels
    rkv.rkv_decode_path(2)
    setup.decode(0)                       # the fused step
    rkv.rkv_decode_path(1)
    setup.decode(1)                       # append_small + the four-kernel decode
    n_new = 2 * wl.page_size
    kn = W.normal((wl.B, wl.Hkv, n_new, wl.d), W.seed_for(setup.seed, "ncu_append"), setup.dev)
    rkv.rkv_append_page_summary(setup.cache, kn, kn, n_new)   # append_pages + append_advance
    stride = max(setup.k2) + 1
    pg = torch.empty((wl.B, wl.Hkv, stride), dtype=torch.int32, device=setup.dev)
    d = setup.dec[2]
    rkv.rkv_decode_hsa(setup.cache, d["q"], setup.k1, setup.k2, setup.out[2], sel_pages=pg, workspace=setup.dws)
    rkv.rkv_exact_topk_recall(setup.cache, d["q"], pg, [k * wl.page_size for k in setup.k2])
    if setup.cache.max_pages * wl.page_size <= 32768:   # the token path's limit
        rkv.rkv_decode_sparq(setup.cache, d["q"], setup.k1, [k * wl.page_size for k in setup.k2], setup.out[2])
        # with the channel-major key copy: sparq_keys_sync + the copy's scoring
        rkv.rkv_decode_sparq(setup.cache, d["q"], setup.k1, [k * wl.page_size for k in setup.k2], setup.out[2],
                             keys_t=rkv.sparq_keys(setup.cache, setup.dev))
    rkv.rkv_decode_path(0)
    plan = W.chunk_plan(wl, 8192)
    cache = rkv.PagedCache(wl.B, wl.Hkv, wl.page_size, setup.cache.max_pages, setup.dev,
                           page_table=setup.cache.page_table)
    held = [0] * wl.B
    for c in range(min(2, len(plan))):    # chunk_gather + the stage-1 kernels
        ch = W.chunk_tensors(wl, setup.inp, plan, c, setup.seed, 0, setup.dev)
        rkv.rkv_prefill_chunk(ch["q_win"], ch["k"], ch["v"], ch["chunk_len"], held, setup.keep1, setup.kp, cache,
                              setup.kept)
        held = [min(k, h + m) for k, h, m in zip(setup.keep1, held, plan[c])]
    torch.cuda.synchronize()
    for cch in (setup.cache, cache):
        st, bits = rkv.rkv_get_device_status(cch)
        if st != rkv.RKV_OK:
            raise RuntimeError(f"device status {st} bits {bits}")


def capture(fn, stream) -> torch.cuda.CUDAGraph:
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


# --------------------------------------------------------------------------- CPU oracle timing
def sample_units(wl: W.Workload, max_units: int = 4) -> list:
    """The (sequence, KV head) units an oracle sample runs: every unit of a small
    workload, else `max_units` of them spread over the batch and the heads."""
    units = [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    if len(units) <= 8:
        return units
    step = len(units) / max_units
    return [units[int(i * step + step / 2) % len(units)] for i in range(max_units)]


def oracle_sample(setup, decode_steps: int, units=None) -> dict:
    """Time the oracle on this host over `units` ((b, g) pairs of layer 0; default all):
    each unit's stage-1 prefill (with its summary build), then `decode_steps` decode
    steps of those units (append + HSA).  Returns the measured seconds and the
    per-unit times, and the whole layer's decode steps/s extrapolated from them:
    steps / (units of the layer x (prefill + steps x decode step)), every unit of a
    layer being the same work."""
    import numpy as np

    from oracle import rkv_oracle as O

    wl = setup.wl
    units = list(units) if units is not None else [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    G = wl.G
    f = lambda t: t.detach().cpu().double().numpy()  # noqa: E731
    # the sampled units' inputs, widened before timing
    ins = []
    for b, g in units:
        L = wl.prompt_lens[b]
        ins.append((b, g, f(setup.inp["q_win"][b, g * G:(g + 1) * G]), f(setup.inp["k"][b, g:g + 1, :L]),
                    f(setup.inp["v"][b, g, :L])))
    steps_in = []
    for t in range(decode_steps):
        d = setup.dec[t]
        steps_in.append((f(d["q"]), f(d["k_new"][:, :, 0]), f(d["v_new"][:, :, 0])))
    t0 = time.perf_counter()
    state = []
    for b, g, q_win, k, v in ins:
        res = O.prefill_evict_unit(q_win, k, setup.keep1[b], setup.kp[b])
        kept = res["kept"][0]
        Kc, Vc = k[0, kept], v[kept]
        state.append([b, g, Kc, Vc, O.page_summaries(Kc, len(kept), wl.page_size)])
    t_prefill = time.perf_counter() - t0
    t1 = time.perf_counter()
    for q, kn, vn in steps_in:
        for u in state:
            b, g, Kc, Vc, (kmax, kmin) = u
            n_old = len(Kc)
            Kc = np.concatenate([Kc, kn[b, g][None]])
            Vc = np.concatenate([Vc, vn[b, g][None]])
            kmax, kmin = O.append_summaries(kmax, kmin, Kc, n_old, 1, wl.page_size)
            if setup.mode == "sparq":
                O.sparq_decode_unit(q[b, g * G:(g + 1) * G], Kc, Vc, n_old + 1, setup.k1[b], setup.k_tokens[b])
            else:
                O.hsa_decode_unit(q[b, g * G:(g + 1) * G], Kc, Vc, n_old + 1, kmax, kmin, wl.page_size,
                                  setup.k1[b], setup.k2[b])
            u[2], u[3], u[4] = Kc, Vc, (kmax, kmin)
    t_dec = time.perf_counter() - t1
    nu = len(units)
    pre_u = t_prefill / nu
    dec_u = t_dec / (nu * max(1, decode_steps))
    layer_s = wl.B * wl.Hkv * (pre_u + wl.steps * dec_u)
    return dict(value=wl.steps / layer_s, seconds=t_prefill + t_dec, units=nu, decode_steps=decode_steps,
                prefill_s_per_unit=pre_u, decode_s_per_unit_step=dec_u)


def oracle_sample_text(wl: W.Workload, o: dict, reps: int, seconds: float) -> str:
    return (f"{reps} x (oracle prefill + {o['decode_steps']} of {wl.steps} decode steps of {o['units']} of the "
            f"{wl.B * wl.Hkv} (sequence, KV head) units of layer 0), {seconds:.1f} s measured in total; value "
            f"extrapolated to the whole layer as steps / ({wl.B * wl.Hkv} units x (prefill + {wl.steps} x decode "
            f"step) per unit), every unit and every layer being the same work")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- main arms
def run_ours(args, rank: int, world: int, dev, workload: int = 0, extras: bool = True) -> dict:
    """The bench line of one workload (args.workload unless `workload` is given).
    With extras off only the timed passes and the per-kernel figures are taken (no
    recall diagnostic, chunked prefill, end-to-end run or CPU oracle)."""
    from two_stage_kv_snapkv_gb300 import rkv

    wl = W.workload(workload or args.workload, args.seed)
    rkv.rkv_decode_path({"auto": 0, "split": 1, "fused": 2}[args.decode_path])
    seed = rank_seed(args.seed, rank)
    nl = 1 if args.one_layer else wl.layers
    setup = Setup(wl, rkv, seed, dev, mode=args.mode)
    setup.flush_mode = args.flush
    # a multi-layer workload keeps every layer resident: stage 1 for all of them, then
    # each decode step runs HSA for every layer in turn, as a model's decode step does
    layers = [setup] + [Setup(wl, rkv, seed, dev, layer=l, share=setup, mode=args.mode) for l in range(1, nl)]
    multi = nl > 1
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)

    if args.ncu_every_kernel:
        ncu_every_kernel(setup)
        return {}

    def prefill_all():
        for s in layers:
            s.prefill()

    def decode_all(t: int):
        for s in layers:
            s.decode(t)

    # eager warm-up (sets kernel attributes, checks the path runs)
    prefill_all()
    for t in range(wl.steps):
        decode_all(t)
    torch.cuda.synchronize()
    for s in layers:
        st, bits = rkv.rkv_get_device_status(s.cache, stream)
        if st != rkv.RKV_OK:
            raise RuntimeError(f"layer {s.layer}: device status {st} bits {bits}")

    if args.ncu:
        setup.prefill()
        for t in range(wl.steps):
            setup.decode(t)
        torch.cuda.synchronize()
        return {}

    # graphs: one for the prefill (every layer), one per decode step (every layer)
    n0 = rkv.rkv_launch_count()
    g_pre = capture(prefill_all, stream)
    n1 = rkv.rkv_launch_count()
    g_dec = [capture(lambda t=t: decode_all(t), stream) for t in range(wl.steps)]
    launches_per_pass = rkv.rkv_launch_count() - n0
    launches_per_step = (rkv.rkv_launch_count() - n1) / wl.steps
    # instrumented copies: library events around every kernel launch
    rkv.profile_enable(True)
    gi_pre = capture(prefill_all, stream)
    gi_dec = [capture(lambda t=t: decode_all(t), stream) for t in range(wl.steps)]
    rkv.profile_enable(False)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * (wl.steps + 1))]

    # Between decode steps L2 is flushed unless a step's compulsory bytes exceed L2 (the
    # timing rule's other option: inputs larger than L2), or the layers evict it: several
    # layers stream far more than L2 between two steps of a layer.  A flush before every
    # step also leaves L2 full of the flush's dirty lines, which the step then writes back.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    step_mb = statistics.mean(setup.decode_bytes(t)["step_total"] for t in range(wl.steps)) / 1e6
    flush_steps = not multi and (args.flush_steps == "always" or step_mb * 1e6 <= l2_bytes)

    # Steps that run back to back also run as one graph, the decode loop: every step of
    # every layer, each launch chained to the one before by programmatic launch, as a
    # serving engine replays its decode graphs.  One graph a step instead adds a graph
    # launch (a few us) to every step of a single-layer workload.
    g_loop = None if flush_steps else capture(lambda: [decode_all(t) for t in range(wl.steps)], stream)

    def one_pass(pre, dec, flush_each=flush_steps, loop=None):
        setup.flush()
        ev[0].record(stream)
        pre.replay()
        ev[1].record(stream)
        if loop is not None:
            ev[2].record(stream)
            loop.replay()
            ev[3].record(stream)
            stream.synchronize()
            per = ev[2].elapsed_time(ev[3]) / wl.steps
            return ev[0].elapsed_time(ev[1]), [per] * wl.steps
        for t in range(wl.steps):
            if flush_each:   # one layer whose steps fit in L2: every step starts cold
                setup.flush()
            ev[2 + 2 * t].record(stream)
            dec[t].replay()
            ev[3 + 2 * t].record(stream)
        stream.synchronize()
        pre_ms = ev[0].elapsed_time(ev[1])
        dec_ms = [ev[2 + 2 * t].elapsed_time(ev[3 + 2 * t]) for t in range(wl.steps)]
        return pre_ms, dec_ms

    for _ in range(args.warmup):
        one_pass(g_pre, g_dec, loop=g_loop)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    pre_all, dec_all = [], []
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for _ in range(args.steps):
            p, d = one_pass(g_pre, g_dec, loop=g_loop)
            pre_all.append(p)
            dec_all.append(d)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary()
    pass_ms = [p + sum(d) for p, d in zip(pre_all, dec_all)]
    total_ms, value = whole_job_value(sum(pass_ms), wl.steps * nl, args.steps, world, dev)

    # per-kernel durations from the instrumented graphs (same work, same flushes)
    rkv.profile_reset()
    for _ in range(args.steps):
        one_pass(gi_pre, gi_dec)
        rkv.profile_accumulate()
    prof = {k: v for k, v in rkv.profile_read().items() if v[0] > 0}
    rkv.profile_release()

    peaks = measured_peaks()
    step_bytes = [setup.decode_bytes(t) for t in range(wl.steps)]
    pb = setup.prefill_bytes()

    def algo_bytes(kind):
        if kind in ("hsa_score", "hsa_attend", "append_small", "hsa_step", "sparq_score", "sparq_attend",
                    "sparq_keys_sync"):
            return statistics.mean(sb[kind] for sb in step_bytes)
        if kind in pb:
            return pb[kind]
        return None

    kernels = {}
    for k, (n, ms) in prof.items():
        avg_ms = ms / n
        ab = algo_bytes(k)
        kernels[k] = dict(launches=n, avg_us=round(avg_ms * 1e3, 3), share=round(ms / sum(v[1] for v in prof.values()), 4),
                          algo_bytes=ab, achieved_gbs=(round(ab / (avg_ms * 1e-3) / 1e9, 1) if ab else None))
    dec_mean_ms = statistics.mean(x for d in dec_all for x in d) / nl   # one layer's decode step
    if g_loop is not None and launches_per_step == nl and "hsa_step" in kernels:
        # the decode loop holds only hsa_step launches, back to back: its event time
        # divided by the launches is the kernel's own average duration, which the event
        # nodes of the instrumented copy (one per launch) would serialise and inflate
        hk = kernels["hsa_step"]
        hk["avg_us_instrumented"] = hk["avg_us"]
        hk["avg_us"] = round(dec_mean_ms * 1e3, 3)
        hk["achieved_gbs"] = round(hk["algo_bytes"] / (dec_mean_ms * 1e-3) / 1e9, 1)
        hk["duration_from"] = "uninstrumented decode loop graph: event time / hsa_step launches"
    dominant = max(kernels, key=lambda k: kernels[k]["avg_us"] * kernels[k]["launches"])
    dk = kernels[dominant]
    traffic = recorded_traffic(str(wl.name), dominant)
    roofline = dict(bound="hbm", kernel=dominant, achieved=dk["achieved_gbs"], peak=peaks["hbm_gbs"],
                    unit="GB/s", frac=(round(dk["achieved_gbs"] / peaks["hbm_gbs"], 4) if dk["achieved_gbs"] else None),
                    traffic=traffic, peak_source=peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"
                    if peaks["source"] == "measured" else "fallback 6.8 TB/s")

    step_total = statistics.mean(sb["step_total"] for sb in step_bytes)
    pre_layer_ms = statistics.mean(pre_all) / nl
    res = dict(
        metric=METRIC, value=round(value, 2), unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=round(statistics.mean(pass_ms), 4), higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16", data="synthetic (seeded normal bf16 with the workload's shapes, outlier channels, sinks and needles)",
        config=workload_config(wl, setup.keep1, setup.k1, setup.k2, setup.kp, args.decode_path, world, nl,
                               args.mode, args.flush, None if flush_steps else (step_mb, l2_bytes / 1e6)),
        prefill_evict_ms=round(pre_layer_ms, 4),
        decode_us_per_step=round(dec_mean_ms * 1e3, 3),
        decode_achieved_gbs=round(step_total / (dec_mean_ms * 1e-3) / 1e9, 1),
        decode_compulsory_mb_per_step=round(step_total / 1e6, 3),
        prefill_achieved_gbs=round(pb["compulsory"] / (pre_layer_ms * 1e-3) / 1e9, 1),
        prefill_compulsory_mb=round(pb["compulsory"] / 1e6, 2),
        prefill_traffic_ratio=round(pb["moved"] / pb["compulsory"], 3),
        roofline=roofline, kernels=kernels, gpu_launches=int(launches_per_pass * args.steps),
        clocks=dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"], reasons=clocks["reasons"],
                    samples=clocks["samples"]),
    )
    if g_loop is not None:
        # the same steps as one graph each (a graph launch before every step), and for a
        # single layer with L2 flushed before every step too, for comparison
        dec_g = []
        for _ in range(args.steps):
            dec_g += one_pass(g_pre, g_dec, flush_each=False)[1]
        res["decode_us_per_step_graph_per_step"] = round(statistics.mean(dec_g) * 1e3 / nl, 3)
    if not multi and not flush_steps:
        dec_fl = []
        for _ in range(args.steps):
            dec_fl += one_pass(g_pre, g_dec, flush_each=True)[1]
        res["decode_us_per_step_l2_flushed"] = round(statistics.mean(dec_fl) * 1e3, 3)
    if multi:
        res["prefill_all_layers_ms"] = round(statistics.mean(pre_all), 4)
        res["decode_all_layers_us_per_step"] = round(dec_mean_ms * nl * 1e3, 3)
        res["memory_gb"] = dict(prompt_kv=round(nl * 2 * wl.Hkv * sum(wl.prompt_lens) * 256 / 1e9, 2),
                                cache_pages=round(sum(s.cache.nbytes() for s in layers) / 1e9, 2))
    if not extras:
        return res
    res["selection"] = selection_recall(setup) if args.mode != "sparq" else dict(
        skipped="the recall diagnostic takes a page selection; SparQ-only selects tokens")
    if args.prefill_chunk > 0:
        res["chunked_prefill"] = chunked_prefill(setup, stream, args.prefill_chunk, max(args.steps, 3))
    if rank == 0 and not args.no_e2e:
        res["e2e"] = run_e2e(setup, args, stream, rkv)
        if multi:
            res["e2e"]["layers"] = 1   # layer 0 alone, through the host buffers
    if rank == 0 and not args.no_cpu_baseline:
        steps = args.cpu_decode_steps or wl.steps
        units = sample_units(wl)
        vals, secs, reps = [], 0.0, 0
        while secs < args.cpu_seconds and reps < 100:
            o = oracle_sample(setup, steps, units)
            vals.append(o["value"])
            secs += o["seconds"]
            reps += 1
            if secs + o["seconds"] > 3 * args.cpu_seconds:
                break
        res["cpu_baseline"] = dict(value=round(statistics.mean(vals), 3), unit=UNIT, cores=host_cores(),
                                   kind="oracle", sample=oracle_sample_text(wl, o, reps, secs))
    return res


def workload_config(wl: W.Workload, keep1, k1, k2, kp, decode_path: str, world: int, layers: int = 1,
                    mode: str = "hsa", flush: str = "write", step_over_l2=None) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    how = ("256 MB write, then a 256 MB read of another buffer, so no dirty line is left for the timed work "
           "to write back" if flush == "clean" else "256 MB write")
    if layers > 1:
        step = (f"one request over {layers} layers: split + prefill evict of every layer + every decode step "
                f"(append + HSA for each layer in turn); value counts layer-steps")
        l2 = (f"flushed ({how}) before the prefill; not between decode steps: each step streams "
              f"{layers} layers' caches, far more than L2, so every layer starts cold; flush not timed")
    elif step_over_l2:
        step = "one request: split + prefill evict + every decode step (append + HSA)"
        l2 = (f"flushed ({how}) before the prefill; not between decode steps: a step's compulsory bytes "
              f"({step_over_l2[0]:.1f} MB) exceed L2 ({step_over_l2[1]:.1f} MB), so its inputs are larger than "
              f"L2; flush not timed (decode_us_per_step_l2_flushed: the same steps with a flush before each)")
    else:
        step = "one request: split + prefill evict + every decode step (append + HSA)"
        l2 = f"flushed ({how}) before the prefill and before every decode step; flush not timed"
    return dict(workload=wl.name, B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, head_dim=wl.d, prompt_len=wl.prompt_lens[0]
                if wl.B == 1 else f"{min(wl.prompt_lens)}..{max(wl.prompt_lens)}", budget=wl.budget,
                window=wl.window, page_size=wl.page_size, decode_steps=wl.steps, layers=layers,
                keep1=self_or_range(keep1), k1=self_or_range(k1), k2=self_or_range(k2),
                pool_kernel=self_or_range(kp), split="RocketKV-MT (nothing evicted)" if wl.mt else "two-stage",
                step=step, l2=l2, timing=("CUDA graphs: the prefill, then the decode loop (every step of every layer, "
                                          "launches chained by programmatic launch); CUDA events on the launching "
                                          "stream around each" if step_over_l2 or layers > 1 else
                                          "CUDA graphs: the prefill, then one per decode step (L2 flushed between "
                                          "them); CUDA events on the launching stream around each"),
                decode_path=decode_path, parallelism=f"replica x{world}" if world > 1 else "single GPU",
                mode={"hsa": "HSA", "quest": "Quest-only (HSA, k1 = every channel)",
                      "sparq": "SparQ-only (one-token pages, k2 x P tokens)"}[mode])


def whole_job_value(total_ms: float, decode_steps: int, passes: int, world: int, device) -> tuple:
    """Max timed total over the ranks, and the whole-job decode steps/s it gives.

    Every rank runs its own independent request (weak scaling, no data exchange), so
    the job processed world * decode_steps * passes decode steps in the slowest rank's
    time.  Returns (max total ms, decode steps per second)."""
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    total = float(t.item())
    return total, world * decode_steps * passes / (total / 1e3)


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own request: the shards are independent sequences."""
    return seed + rank


def self_or_range(xs):
    return xs[0] if len(set(xs)) == 1 else f"{min(xs)}..{max(xs)}"


# the headers every kernel source includes: part of each kernel's code
KERNEL_HEADERS = ("two_stage_kv_snapkv_gb300/csrc/rkv_device.cuh", "two_stage_kv_snapkv_gb300/csrc/rkv_internal.h",
                  "include/rkv.h")


def _source_sha(rel: str) -> str:
    """sha256 (first 16 hex digits) of a kernel source file followed by KERNEL_HEADERS;
    a kernel's recorded DRAM counters stay valid while this is unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in (rel, *KERNEL_HEADERS) if rel else ():
        path = os.path.join(ROOT, f)
        if not os.path.exists(path):
            return ""
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16] if rel else ""


def recorded_traffic(workload: str, kernel: str, path: str = "") -> int | None:
    """DRAM bytes per launch of `kernel` at `workload` from the committed ncu record
    (profiles/traffic.json), or None when there is no entry or the kernel's sources
    have changed since it was captured."""
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        ent = json.load(f).get(workload, {}).get(kernel)
    if not ent or ent.get("source_sha") != _source_sha(ent.get("source_file", "")):
        return None
    return ent["bytes_per_launch"]


def run_e2e(setup: Setup, args, stream, rkv) -> dict:
    """The same request through the public API from pinned host buffers, inside the timed
    region: the prompt copied in, then every step's inputs taken from and its output
    returned to host memory."""
    wl = setup.wl
    host = {k: setup.inp[k].cpu().pin_memory() for k in ("q_win", "k", "v")}
    # a step's three inputs packed into one pinned buffer (q | k_new | v_new), so each
    # step takes one host-to-device copy; the device side views the same packing
    names = ("q", "k_new", "v_new")
    sizes = [setup.dec[0][k].numel() * 2 for k in names]
    offs = [0, sizes[0], sizes[0] + sizes[1]]
    hdec = []
    for d in setup.dec:
        buf = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
        for k, o, n in zip(names, offs, sizes):
            buf[o:o + n].copy_(d[k].cpu().contiguous().view(-1).view(torch.uint8))
        hdec.append(buf)
    ddev = torch.empty(sum(sizes), dtype=torch.uint8, device=setup.dev)
    dd = {k: ddev[o:o + n].view(torch.bfloat16).view(setup.dec[0][k].shape) for k, o, n in zip(names, offs, sizes)}
    hout = torch.empty((wl.steps, wl.B, wl.Hq, 128), dtype=torch.float32).pin_memory()
    # q_win and K are copied to the device (the scoring reads K twice, by the tensor
    # engine); V stays in pinned host memory: stage 1 reads only the kept rows of V,
    # once, through the buffer's device mapping
    dq = {k: torch.empty_like(setup.inp[k]) for k in ("q_win", "k")}
    v_kept = sum(wl.Hkv * k1 * 128 * 2 for k1 in setup.keep1)
    h2d = sum(host[k].numel() * host[k].element_size() for k in dq) + v_kept + wl.steps * sum(sizes)
    d2h = hout.numel() * 4
    host_step = setup.mode != "sparq"
    staging = rkv.step_host_staging(wl.B, wl.Hq, wl.Hkv, setup.dev)

    def one():
        for k in dq:
            dq[k].copy_(host[k], non_blocking=True)
        rkv.rkv_prefill_evict(dq["q_win"], dq["k"], host["v"], wl.prompt_lens, setup.keep1, setup.kp, setup.cache,
                              setup.kept, workspace=setup.pws)
        for t in range(wl.steps):
            if host_step:   # one call: the fused step on the host buffers
                rkv.rkv_decode_step_host(setup.cache, hdec[t], hout[t], wl.Hq, setup.k1, setup.k2, staging,
                                         setup.dws)
            else:
                ddev.copy_(hdec[t], non_blocking=True)
                setup.step(dd["q"], dd["k_new"], dd["v_new"], setup.out[t])
                hout[t].copy_(setup.out[t], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(args.steps):
        setup.flush()
        e0.record(stream)
        one()
        e1.record(stream)
        stream.synchronize()
        times.append(e0.elapsed_time(e1))
    return dict(value=round(wl.steps * len(times) / (sum(times) / 1e3), 2), unit=UNIT, h2d_bytes_per_step=int(h2d),
                d2h_bytes_per_step=int(d2h), ms_per_request=round(statistics.mean(times), 4),
                step=(f"one bench step is one request: the prompt's window queries and keys copied in, the prefill "
                      f"(which reads the kept rows of V from pinned host memory), then {wl.steps} decode steps, each "
                      "taking its inputs from and returning its output to host memory; the byte counts are per "
                      "request"),
                h2d_prompt_bytes=int(h2d - wl.steps * sum(sizes)), h2d_bytes_per_decode_step=int(sum(sizes)),
                d2h_bytes_per_decode_step=int(d2h // wl.steps),
                path=("python binding -> C ABI rkv_decode_step_host, eager, pinned host buffers (per call the "
                      "fused step reads the packed inputs and writes the output through the buffers' device "
                      "mapping; copy in, step, copy out where they are not mapped)") if host_step else
                     "python binding -> C ABI, eager launches, pinned host buffers (one input copy per step)")


def run_reference(args, rank: int, world: int) -> dict:
    """The CPU oracle as the reference arm: each step is a bounded sample of the request."""
    if rank != 0:
        return {}
    wl = W.workload(args.workload, args.seed)

    class _Split:
        pass

    from oracle import rkv_oracle as O

    setup = _Split()
    setup.wl = wl
    setup.inp = W.prefill_tensors(wl, args.seed, 0, "cpu", tail="zero")
    setup.dec = []
    for t in range(wl.steps):
        d = W.decode_tensors(wl, t, args.seed, 0, "cpu")
        d["k_new"] = d["k_new"].unsqueeze(2)
        d["v_new"] = d["v_new"].unsqueeze(2)
        setup.dec.append(d)
    if wl.mt:
        sp = [O.split_ratio_mt(L, wl.budget, wl.d, wl.page_size, wl.k1 or 0) for L in wl.prompt_lens]
    else:
        sp = [O.split_ratio(L, wl.budget, wl.d, wl.page_size, wl.window, wl.k1 or 0) for L in wl.prompt_lens]
    setup.keep1 = [s["keep1"] for s in sp]
    setup.mode = args.mode
    setup.k1 = [s["k1"] if args.mode != "quest" else wl.d for s in sp]
    setup.k2 = [s["k2"] for s in sp]
    setup.k_tokens = [k * wl.page_size for k in setup.k2]
    setup.kp = [wl.pool_kernel or s["pool_kernel"] for s in sp]
    units = sample_units(wl)
    # one bench step = one bounded sample: the sampled units' prefill and every decode step
    for _ in range(args.warmup):
        oracle_sample(setup, 1, units[:1])
    vals, secs = [], []
    for _ in range(args.steps):
        o = oracle_sample(setup, wl.steps, units)
        vals.append(o["value"])
        secs.append(o["seconds"])
    value = statistics.mean(vals)
    return dict(impl="reference", metric=METRIC, value=round(value, 3), unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(1e3 * statistics.mean(secs), 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic (seeded)",
                config=workload_config(wl, setup.keep1, setup.k1, setup.k2, setup.kp, args.decode_path, world,
                                       wl.layers, args.mode, args.flush),
                step=("one bounded sample of the request (ms_per_step is its measured wall time; value is the "
                      "whole layer's rate extrapolated from it, see cpu_baseline.sample)"),
                cpu_baseline=dict(value=round(value, 3), unit=UNIT, cores=host_cores(), kind="oracle",
                                  sample=oracle_sample_text(wl, o, args.steps, sum(secs))),
                e2e=dict(value=round(value, 3), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    res = run_ours(args, rank, world, dev)
    if res and args.workload == 5 and not args.no_extra and not args.one_layer and args.mode == "hsa":
        # the batch-16 serving workload (8K-32K prompts), measured in the same run: its
        # decode step, and the fused step's roofline there
        torch.cuda.empty_cache()
        w4 = run_ours(args, rank, world, dev, workload=4, extras=False)
        if w4:
            res["workload4"] = dict(workload=w4["config"]["workload"], value=w4["value"], unit=UNIT,
                                    ms_per_step=w4["ms_per_step"], decode_us_per_step=w4["decode_us_per_step"],
                                    prefill_evict_ms=w4["prefill_evict_ms"],
                                    decode_achieved_gbs=w4["decode_achieved_gbs"], roofline=w4["roofline"],
                                    l2=w4["config"]["l2"],
                                    decode_us_per_step_l2_flushed=w4.get("decode_us_per_step_l2_flushed"),
                                    clocks=w4["clocks"], gpu_launches=w4["gpu_launches"])
    if rank == 0 and res:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
