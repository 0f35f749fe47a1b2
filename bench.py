#!/usr/bin/env python
"""Benchmark of the top-k block-sparse GQA attention hot path on one B300.

Default workload (decode GQA): batch 8, Hq 32, Hkv 8, d 128, context 32768,
KV block 64 (512 blocks), top-k 32 + sink + local, bf16, 1% needle blocks.
One step = the whole decode hot path over one batch: append the new token's
K/V and refresh its block sketch (a1), score every block and select the top-k
(a2 + a3), sparse split-KV attention over the selected blocks (a4).

Prints ONE JSON line.  `value` = bytes the step must move (selected K/V blocks
+ sketch scan + append) / device time per step, with inputs resident in HBM;
8 input sets (distinct K/V caches) are rotated so that no step finds its
blocks in L2.  `e2e` = the same bytes / wall time per step through the C-ABI
decode-step call with pinned host q/k_new/v_new/out, copies included.

The same line carries a `prefill` list with the two prefill workloads, each
timed as whole steps on the full workload: sketch-selected prefill (batch 2,
Hq 32, Hkv 8, context 131072: sketch build + tile scoring/top-k + tcgen05
sparse prefill) and oracle-mass prefill (batch 1, Hq 16, Hkv 2, context 32768:
tcgen05 mass + top-k + sparse prefill), with tensor-core rooflines.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload c2|c3] [--prefill-steps P] [--prefill-only]
                    [--prefill-B B --prefill-L L]   (smaller prefill case for profiling)
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
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- workloads

def workload(name):
    import synth
    return synth.WORKLOADS[name]


def decode_bytes(wl, cnt_np, L):
    """Algorithmic bytes of one decode step (selected K/V + sketch scan + append)."""
    es = wl.esize
    kv = 0
    for c in cnt_np.reshape(-1):
        kv += int(c) * wl.Bk * wl.d * es * 2
    groups = wl.B * wl.Hkv
    sketch = groups * wl.nb * wl.d * 4
    touched_rows = (L - 1) % wl.Bk + 1
    append = groups * (wl.T * wl.d * es * 2 + touched_rows * wl.d * es + wl.d * 4)
    return kv, sketch, append


def _sub_workload(wl, x, ngroups):
    """The first `ngroups` (batch, kv-head) groups of the workload, as a smaller workload."""
    if ngroups <= wl.Hkv:
        sub = wl.replace(B=1, Hkv=ngroups, Hq=ngroups * wl.G)
        return sub, x.q[:1, :, : ngroups * wl.G], x.k[:1, :ngroups], x.v[:1, :ngroups]
    nbatch = ngroups // wl.Hkv
    return wl.replace(B=nbatch), x.q[:nbatch], x.k[:nbatch], x.v[:nbatch]


def oracle_decode_sample(wl, x, ngroups):
    """One CPU-oracle decode step (sketch -> score -> select -> attend) on the first
    `ngroups` groups.  Returns (seconds, algorithmic bytes)."""
    import numpy as np

    import oracle
    sub, q, k, v = _sub_workload(wl, x, ngroups)
    t0 = time.perf_counter()
    idx, cnt, _, _ = oracle.decode_select(q, k, sub)
    rows = np.array([(b, t, h) for b in range(sub.B) for t in range(sub.T) for h in range(sub.Hq)])
    oracle.attend(q, k, v, sub.Hkv, sub.L, sub.L - sub.T, sub.Bk, sub.scale, rows, idx, cnt)
    dt = time.perf_counter() - t0
    kv, sk, ap = decode_bytes(sub, cnt, sub.L)
    return dt, kv + sk + ap


def _sample_sizes(wl):
    sizes = [1]
    while sizes[-1] < wl.Hkv:
        sizes.append(min(wl.Hkv, sizes[-1] * 2))
    b = 2
    while b <= wl.B:
        sizes.append(b * wl.Hkv)
        b *= 2
    if sizes[-1] != wl.B * wl.Hkv:
        sizes.append(wl.B * wl.Hkv)
    return sizes


def cpu_oracle_decode(wl, x, budget_s):
    """Time the CPU oracle on a bounded sample (the first groups of the batch) for about budget_s
    seconds.  Returns (GB/s, cores, sample text)."""
    import oracle
    ng = 1
    dt, _ = oracle_decode_sample(wl, x, ng)
    for cand in _sample_sizes(wl)[1:]:
        if dt * cand / ng > budget_s / 3:
            break
        ng = cand
        dt, _ = oracle_decode_sample(wl, x, ng)
    reps = max(1, int(budget_s // max(dt, 1e-3)))
    total_t, total_b = 0.0, 0
    for _ in range(reps):
        t, b = oracle_decode_sample(wl, x, ng)
        total_t += t
        total_b += b
    sample = "%d of %d groups, full context %d, %d rep(s)" % (ng, wl.B * wl.Hkv, wl.L, reps)
    return total_b / total_t / 1e9, oracle.threads(), sample


# ------------------------------------------------------------------ our arm

def max_over_ranks(t_ms, device, world):
    """The job's time is the slowest rank's (replicas run independent batches; no data-path
    collective, only this reduction of the timing)."""
    if world <= 1:
        return float(t_ms)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(t_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_value(step_bytes_per_rank, world, ms_per_step):
    """GB/s over all ranks: every rank moves step_bytes_per_rank per step (weak scaling)."""
    return step_bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


def bench_decode(args, wl, rank, world, steps=None, rotate=None, cpu_seconds=None):
    """One decode workload as whole steps (append + select + decode), CUDA graphs over `rotate`
    resident input sets; per-kernel times, the decode kernel's roofline, the end-to-end leg through
    the C ABI with pinned host buffers, and (rank 0) the CPU oracle on a bounded sample."""
    import numpy as np
    import torch

    import synth
    import top_block_sparse_pooled_b300 as sa

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    x = synth.make_inputs(wl.replace(seed=wl.seed + 100 * rank))
    R = rotate or args.rotate
    steps = steps or args.steps
    cpu_seconds = args.cpu_seconds if cpu_seconds is None else cpu_seconds
    bf = wl.dtype == "bf16"

    def up(a):
        import numpy as np
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        return t.to(dev)

    q0, k0, v0 = up(x.q), up(x.k), up(x.v)
    pos = wl.L - wl.T
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, 0, False, wl.k)
    dtype_code = sa.SA_BF16 if bf else sa.SA_F32
    ws_bytes = sa.sa_decode_step_workspace_bytes(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, dtype_code, kmax)
    sets = []
    for r in range(R):
        kc, vc = k0.clone(), v0.clone()
        sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device=dev)
        sa.sa_build_sketch(kc, wl.L, wl.Bk, sk)
        sets.append(dict(
            q=q0.clone(), kc=kc, vc=vc, sk=sk,
            k_new=k0[:, :, pos:].permute(0, 2, 1, 3).contiguous(),
            v_new=v0[:, :, pos:].permute(0, 2, 1, 3).contiguous(),
            idx=torch.empty((wl.B, wl.Hkv, 1, kmax), dtype=torch.int32, device=dev),
            cnt=torch.empty((wl.B, wl.Hkv, 1), dtype=torch.int32, device=dev),
            out=torch.empty_like(q0),
            ws=torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)))
    del k0, v0

    def step(s):
        sa.sa_decode_step(s["q"], s["k_new"], s["v_new"], s["kc"], s["vc"], s["sk"], wl.L, wl.Bk, wl.k, wl.scale,
                          s["idx"], s["cnt"], s["out"], s["ws"])

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(sets[i % R])
    torch.cuda.synchronize()
    if sa.sa_device_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    cnt_np = sets[0]["cnt"].cpu().numpy()
    kv_b, sk_b, ap_b = decode_bytes(wl, cnt_np, wl.L)
    step_bytes = kv_b + sk_b + ap_b

    def capture(fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f in fns:
                f()
        return g

    def graph_us(g, calls, reps):
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda._sleep(20_000_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (calls * reps)

    # the step as CUDA graphs of GS consecutive steps cycling through the R input sets (at least
    # 32 steps per graph, so that the boundaries between replays, where one step cannot start
    # early behind the previous one, are rare)
    GS = R * max(1, 32 // R)
    g_full = capture([lambda s=s: step(s) for s in sets * (GS // R)])
    K = steps
    rem = K % GS
    g_rem = capture([lambda i=i: step(sets[i % R]) for i in range(rem)]) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // GS)):
            g_full.replay()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(20_000_000)  # keep the device busy while the host queues the replays
        ev0.record(stream)
        for _ in range(K // GS):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), dev, world)
    ms_per_step = t_ms / K
    value = whole_job_value(step_bytes, world, ms_per_step)

    # ---- per-kernel times, each from a CUDA graph of 4*R back-to-back calls
    def dec(s):
        sa.sa_decode(s["q"], s["kc"], s["vc"], s["idx"], s["cnt"], wl.L, wl.Bk, wl.scale, s["out"], s["ws"])

    def sel(s):
        sa.sa_select_topk(sa.SA_SELECT_SKETCH, s["q"], s["sk"], None, wl.Hkv, wl.L, wl.L, wl.Bk, 0, False, wl.k, 0,
                          1, wl.scale, s["idx"], s["cnt"])

    def app(s):
        sa.sa_append_kv(s["k_new"], s["v_new"], s["kc"], s["vc"], pos, wl.Bk, s["sk"])

    def seld(s):  # top-delta selection (threshold from the sink and local blocks), same budget as a cap
        sa.sa_select_topdelta(s["q"], s["sk"], None, wl.Hkv, wl.L, wl.L, wl.Bk, 0.3, wl.k, wl.scale, s["idx"],
                              s["cnt"])

    def fused(s):  # selection and attention in one launch (the step's kernel for these shapes)
        sa.sa_select_decode(s["q"], s["sk"], s["kc"], s["vc"], wl.L, wl.Bk, wl.k, wl.scale, s["idx"], s["cnt"],
                            s["out"])

    fused_ok = bf and wl.G * wl.T <= 16 and wl.Bk == 64
    # the step's append runs inside the same launch when the new rows lie in the local block
    fused_append = fused_ok and (wl.L - wl.T) // wl.Bk == (wl.L - 1) // wl.Bk
    reps = max(10, min(500, K // (4 * R)))
    kern_us = {}
    legs = [("append", app), ("select", sel), ("decode", dec)]
    if fused_ok:
        legs.append(("select_decode", fused))
    legs.append(("select_topdelta", seld))
    for name, fn in legs:
        g = capture([lambda s=s, fn=fn: fn(s) for s in sets * 4])
        kern_us[name] = round(graph_us(g, 4 * R, reps), 3)
    torch.cuda.synchronize()
    topdelta_blocks = float(sets[-1]["cnt"].float().mean().item())  # blocks kept per group at delta 0.3
    with torch.cuda.stream(stream):
        for s_ in sets:  # back to the top-k selection for the end-to-end leg below
            sel(s_)
    torch.cuda.synchronize()
    dec_ms = kern_us["decode"] * 1e-3
    dec_gbs = kv_b / (dec_ms * 1e-3) / 1e9
    # the step's dominant kernel: the fused selection + attention (sketch scan + selected K/V), or,
    # for shapes without it, the attention kernel
    if fused_append:  # the step is one launch: its time is the step time of the timed region
        top_ms, top_bytes = ms_per_step, step_bytes
        top_name = ("sa_decode_step (seldec_kernel: cache append, sketch scoring, top-k and sparse attention in "
                    "one launch)")
    elif fused_ok:
        top_ms, top_bytes = kern_us["select_decode"] * 1e-3, kv_b + sk_b
        top_name = "sa_select_decode (seldec_kernel: sketch scoring, top-k and sparse attention in one launch)"
    else:
        top_ms, top_bytes = dec_ms, kv_b
        top_name = "sa_decode (decode_split_kernel + decode_combine_kernel)"
    top_gbs = top_bytes / (top_ms * 1e-3) / 1e9

    # ---- end to end through the C ABI with pinned host buffers
    hq = sets[0]["q"].cpu().pin_memory()
    hkn = sets[0]["k_new"].cpu().pin_memory()
    hvn = sets[0]["v_new"].cpu().pin_memory()
    hout = torch.empty(hq.shape, dtype=hq.dtype).pin_memory()
    ne = min(K, 2000)
    with torch.cuda.stream(stream):
        # one prepared call per rotated input set (the binding marshals the arguments once)
        steps = [sa.DecodeStep(hq, hkn, hvn, s["kc"], s["vc"], s["sk"], wl.L, wl.Bk, wl.k, wl.scale, s["idx"],
                               s["cnt"], hout, s["ws"], host_io=True, stream=stream) for s in sets]
        for i in range(2 * R + 5):  # every set seen twice: its step graph is captured before timing
            steps[i % R]()
        stream.synchronize()
        t0 = time.perf_counter()
        for i in range(ne):
            steps[i % R]()
            stream.synchronize()  # the next token needs this one's output
        t_e2e = (time.perf_counter() - t0) / ne
    es = wl.esize
    h2d = hq.numel() * es + hkn.numel() * es * 2
    d2h = hout.numel() * es

    res = {
        "metric": "sparse-attn decode KV GB/s (% HBM peak)",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic: seeded N(0,1) q/k/v, %d needle blocks per group (keys + %g * q_hat)" % (wl.needles,
                                                                                                    wl.alpha),
        "config": {
            "workload": "%s decode: B=%d T=%d Hq=%d Hkv=%d d=%d L=%d block=%d top-k=%d + sink + local" % (
                wl.name, wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, wl.L, wl.Bk, wl.k),
            "step": ("append+sketch refresh, score+top-k select and sparse decode in one launch" if fused_append else
                     "append+sketch refresh, then score+top-k select and sparse decode in one launch" if fused_ok else
                     "append+sketch refresh, score+top-k select, split-KV sparse decode") + (
                " (CUDA graphs of %d steps over %d input sets)" % (GS, R)),
            "bytes_per_step": {"selected_kv": kv_b, "sketch_scan": sk_b, "append": ap_b},
            "l2": "%d resident input sets rotated (%.1f GB of K/V); no step reuses L2 from the previous" % (
                R, R * x.k.nbytes * 2 / 1e9),
        },
        "pct_hbm_peak": round(100 * value / peaks["hbm_gbs"], 2),
        "roofline": {
            "kernel": top_name,
            "bound": "hbm",
            "achieved": round(top_gbs, 2),
            "peak": peaks["hbm_gbs"],
            "peak_source": peak_src,
            "unit": "GB/s",
            "frac": round(top_gbs / peaks["hbm_gbs"], 4),
            "traffic": None,
            "avg_launch_us": round(top_ms * 1e3, 3),
            "algorithmic_bytes_per_launch": top_bytes,
        },
        "decode_roofline": {
            "kernel": "sa_decode alone (selected K/V given): " + (
                "seldec_kernel, one cluster per group" if fused_ok and 2 * wl.B * wl.Hkv <= 148 else
                "decode_mma_kernel" if fused_ok else "decode_split_kernel + decode_combine_kernel"),
            "bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peaks["hbm_gbs"], "peak_source": peak_src,
            "unit": "GB/s", "frac": round(dec_gbs / peaks["hbm_gbs"], 4), "avg_launch_us": round(dec_ms * 1e3, 3),
            "algorithmic_bytes_per_launch": kv_b,
        },
        "e2e": {"value": round(step_bytes / t_e2e / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(t_e2e * 1e3, 4)},
        "kernels_us": kern_us,
        "topdelta": {"delta": 0.3, "cap": wl.k, "mean_blocks_kept_per_group": round(topdelta_blocks, 2),
                     "select_us": kern_us["select_topdelta"]},
        "gpu_launches": K * (1 if fused_append else 2 if fused_ok else 4),
        "clocks": clocks,
    }
    if rank == 0 and args.cpu_baseline and cpu_seconds > 0:
        gbs, cores, sample = cpu_oracle_decode(wl, x, cpu_seconds)
        res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": sample}
        if wl.name == "c1":  # the small parity config also on one core
            import oracle
            oracle.set_threads(1)
            try:
                gbs1, cores1, sample1 = cpu_oracle_decode(wl, x, min(cpu_seconds, 5.0))
            finally:
                oracle.set_threads(cores)
            res["cpu_baseline_1core"] = {"value": round(gbs1, 4), "unit": "GB/s", "cores": cores1, "kind": "oracle",
                                         "sample": sample1}
    if bf and wl.G * wl.T <= 16:
        res["roofline"]["traffic"] = _stored_traffic("decode_%s_traffic.txt" % wl.name, DECODE_SOURCES)
    return res


def _leg_summary(r):
    """A secondary decode workload's result, without the keys that only the headline line carries."""
    keep = ("value", "unit", "ms_per_step", "steps", "dtype", "config", "pct_hbm_peak", "roofline", "decode_roofline",
            "e2e", "kernels_us", "gpu_launches", "clocks", "cpu_baseline", "cpu_baseline_1core")
    out = {k: r[k] for k in keep if k in r}
    out["metric"] = r["metric"]
    return out


def _events_ms(fn, reps, stream):
    """Median over reps of the CUDA-event time of fn() on `stream` (one launch sequence each).  A
    sleep kernel queued first keeps the device busy while the host enqueues fn(), so the events
    time the device work, not the host's launch overhead."""
    import torch
    ts = []
    with torch.cuda.stream(stream):
        fn()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
    ts.sort()
    return ts[len(ts) // 2]


def cpu_oracle_prefill(wl, x, budget_s, executed_flop):
    """The CPU oracle's prefill step on a seeded sample of (group, tile) units, extrapolated to the
    whole workload: each part of the step is scaled by the share of its work the sample holds
    (sketch-mode scores by causal blocks x rows, dense mass by causal pairs, sparse attention by
    selected tiles; the fp64 sketch of the keys is timed in full).  Returns the executed sparse-
    attention TFLOP of the full GPU step divided by the extrapolated CPU step time."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(4242)
    groups = wl.B * wl.Hkv
    all_c = np.array([oracle.causal_blocks(i, wl.Qt, wl.Bk, wl.L) for i in range(wl.nq)], dtype=np.float64)
    budget_i = np.array([oracle.prefill_budget(i, wl.k, wl.frac_num, wl.frac_den, wl.Qt, wl.Bk, wl.L)
                         for i in range(wl.nq)], dtype=np.float64)
    sel_i = np.minimum(all_c, budget_i + 2)  # selected blocks per tile (forced included)
    t_sketch = 0.0
    sketch = None
    if wl.mode != "mass":
        t0 = time.perf_counter()
        sketch = oracle.block_means(x.k, wl.L, wl.Bk)
        t_sketch = time.perf_counter() - t0
    n = 4
    t_score = t_sel = t_att = 0.0
    while True:
        units = [(int(rng.integers(groups)), int(rng.integers(wl.nq))) for _ in range(n)]
        t0 = time.perf_counter()
        if wl.mode == "mass":
            sc = oracle.mass(x.q, x.k, wl.Hkv, wl.L, 0, wl.Qt, wl.Bk, wl.scale, units)
        else:
            sc = oracle.prefill_scores(x.q, sketch, wl.Hkv, wl.Qt, wl.Bk, wl.scale, units)
        t1 = time.perf_counter()
        idx, cnt, _, _ = oracle.prefill_select(x.q, x.k, wl, units, scores=sc)
        t2 = time.perf_counter()
        rows = np.array([(g // wl.Hkv, t, (g % wl.Hkv) * wl.G + h) for g, i in units
                         for t in range(i * wl.Qt, min((i + 1) * wl.Qt, wl.L)) for h in range(wl.G)], dtype=np.int64)
        full_idx = -np.ones((groups * wl.nq, idx.shape[1]), dtype=np.int32)  # the sampled units' selections
        full_cnt = np.zeros((groups * wl.nq,), dtype=np.int32)
        for u, (g, i) in enumerate(units):
            full_idx[g * wl.nq + i] = idx[u]
            full_cnt[g * wl.nq + i] = cnt[u]
        oracle.attend(x.q, x.k, x.v, wl.Hkv, wl.L, 0, wl.Bk, wl.scale, rows, full_idx, full_cnt, nsel=wl.nq,
                      rows_per_sel=wl.Qt)
        t3 = time.perf_counter()
        t_score, t_sel, t_att = t1 - t0, t2 - t1, t3 - t2
        if t3 - t0 > budget_s / 4 or n >= 4096:
            break
        n *= 2
    ii = np.array([i for _, i in units])
    share_c = all_c[ii].sum() / (groups * all_c.sum())          # causal blocks (scores, mass)
    share_s = sel_i[ii].sum() / (groups * sel_i.sum())          # selected tiles (attention)
    step_s = t_sketch + (t_score + t_sel) / share_c + t_att / share_s
    sample = "%d random (group, tile) units of %d; %s; scaled to the whole step by causal blocks and " \
             "selected tiles (extrapolated)" % (len(units), groups * wl.nq,
                                                "dense fp64 mass" if wl.mode == "mass" else
                                                "fp64 sketch of all keys timed in full")
    return {"value": round(executed_flop / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
            "kind": "oracle", "sample": sample, "extrapolated": True, "step_s": round(step_s, 3)}


def bench_prefill(wl, steps, peaks, peak_src, cpu_seconds=0.0, full_size=True):
    """One prefill step = (sketch build + sketch select | oracle mass + mass select) + sparse prefill,
    on the full workload.  Returns a dict with per-kernel times and tensor-core rooflines (stored DRAM
    traffic per launch only at the full, unmodified workload)."""
    import numpy as np
    import torch

    import synth
    import top_block_sparse_pooled_b300 as sa

    dev = torch.device("cuda", torch.cuda.current_device())
    x = synth.make_inputs(wl)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = up(x.q), up(x.k), up(x.v)
    kmax = sa.sa_select_kmax(wl.L, wl.Bk, wl.Qt, True, wl.k, wl.frac_num, wl.frac_den)
    idx = torch.empty((wl.B, wl.Hkv, wl.nq, kmax), dtype=torch.int32, device=dev)
    cnt = torch.empty((wl.B, wl.Hkv, wl.nq), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.Stream(device=dev)
    if wl.mode == "mass":
        mass = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device=dev)

        def score():
            sa.sa_oracle_mass(q, k, wl.Qt, wl.Bk, wl.scale, mass, None)

        def select():
            sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                              wl.frac_num, wl.frac_den, wl.scale, idx, cnt, d=wl.d, dtype=sa.SA_BF16, B=wl.B,
                              Tq=wl.L, Hq=wl.Hq)
    else:
        sk = torch.empty((wl.B, wl.Hkv, wl.nb, wl.d), dtype=torch.float32, device=dev)
        tile_scores = torch.empty((wl.B, wl.Hkv, wl.nq, wl.nb), dtype=torch.float32, device=dev)

        def score():
            sa.sa_build_sketch(k, wl.L, wl.Bk, sk)

        def select():
            sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, tile_scores, wl.Hkv, wl.L, wl.L, wl.Bk, wl.Qt, True, wl.k,
                              wl.frac_num, wl.frac_den, wl.scale, idx, cnt)

    def attend():
        sa.sa_prefill(q, k, v, idx, cnt, wl.Qt, wl.Bk, wl.scale, out)

    def step():
        score()
        select()
        attend()

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    if sa.sa_device_status() != 0:
        raise RuntimeError("device status word set during prefill warm-up")
    t_step = _events_ms(lambda: [step() for _ in range(steps)], 1, stream) / steps
    reps = max(3, steps)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    t_score = _events_ms(score, reps, stream)
    score_clocks = sampler.stop()
    t_select = _events_ms(select, reps, stream)
    sampler.start()
    t_attend = _events_ms(attend, reps, stream)
    attend_clocks = sampler.stop()
    pairs = int(cnt.sum().item())  # (group, tile, block) triples executed
    tile_flops = 4 * wl.d * wl.Qt * wl.Bk  # QK^T + PV of one 128 x 128 tile, one head
    executed = pairs * wl.G * tile_flops
    causal_tiles = wl.B * wl.Hkv * sum(min(i + 1, wl.nb) for i in range(wl.nq))
    dense = causal_tiles * wl.G * tile_flops
    achieved = executed / (t_attend * 1e-3) / 1e12
    res = {
        "workload": "%s %s prefill: B=%d Hq=%d Hkv=%d d=%d L=%d qtile=%d block=%d, %s top-%d%%+sink+diagonal" % (
            wl.name, wl.mode, wl.B, wl.Hq, wl.Hkv, wl.d, wl.L, wl.Qt, wl.Bk,
            "oracle-mass" if wl.mode == "mass" else "mean-key sketch", round(100 * wl.frac_num / wl.frac_den)),
        "ms_per_step": round(t_step, 4),
        "steps": steps,
        "kernels_ms": {"score": round(t_score, 4), "select": round(t_select, 4), "prefill": round(t_attend, 4)},
        "selected_tiles": pairs,
        "causal_tiles": causal_tiles,
        "executed_tflop": round(executed / 1e12, 4),
        "dense_causal_tflop": round(dense / 1e12, 3),
        "tflops_executed": round(achieved, 2),
        "tflops_dense_equivalent": round(dense / (t_attend * 1e-3) / 1e12, 1),
        "roofline": {"kernel": "sa_prefill (prefill_kernel, tcgen05)", "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "peak_source": peak_src + " bf16 burst", "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": _stored_traffic("prefill_%s_traffic.txt" % wl.name, PREFILL_SOURCES)
                     if full_size else None,
                     "avg_launch_ms": round(t_attend, 4), "algorithmic_flop_per_launch": executed,
                     "clocks": attend_clocks},
        "l2": "inputs %.2f GB resident, larger than L2" % ((q.numel() + k.numel() + v.numel()) * 2 / 1e9),
    }
    if wl.mode == "mass":
        mass_flops = 2 * 2 * wl.d * wl.Qt * wl.Bk * wl.G * causal_tiles
        res["mass_roofline"] = {"kernel": "sa_oracle_mass (mass_kernel, tcgen05)", "bound": "tensor",
                                "achieved": round(mass_flops / (t_score * 1e-3) / 1e12, 2),
                                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": round(mass_flops / (t_score * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                                "traffic": _stored_traffic("mass_%s_traffic.txt" % wl.name, MASS_SOURCES)
                                if full_size else None,
                                "algorithmic_flop_per_launch": mass_flops, "clocks": score_clocks}
    del q, k, v, out
    torch.cuda.empty_cache()
    if cpu_seconds > 0:
        res["cpu_baseline"] = cpu_oracle_prefill(wl, x, cpu_seconds, executed)
    del x
    return res


def bench_length_sweep(lengths, k_ref, L_ref, exponent, reps=20):
    """Decode (B=1, T=4, Hq=32, Hkv=8, d=128, block 64) across context lengths with the
    length-aware budget k(L) = ceil(k_ref * (L / L_ref)^exponent).  Each rep: L2 flushed
    (256 MB write, untimed), then sketch select + sparse decode timed with CUDA events."""
    import numpy as np
    import torch

    import synth
    import top_block_sparse_pooled_b300 as sa
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rows = []
    for L in lengths:
        k = sa.sa_budget_sublinear(L, 64, k_ref, L_ref, exponent)
        nb = (L + 63) // 64
        wl = synth.WORKLOADS["c3"].replace(L=L, k=k, needles=max(1, round(0.005 * nb)))
        x = synth.make_inputs(wl)

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        q, kc, vc = up(x.q), up(x.k), up(x.v)
        del x
        sk = torch.empty((1, wl.Hkv, nb, wl.d), dtype=torch.float32, device=dev)
        sa.sa_build_sketch(kc, L, 64, sk)
        kmax = sa.sa_select_kmax(L, 64, 0, False, k)
        idx = torch.empty((1, wl.Hkv, 1, kmax), dtype=torch.int32, device=dev)
        cnt = torch.empty((1, wl.Hkv, 1), dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = torch.zeros(sa.sa_decode_workspace_bytes(1, wl.T, wl.Hq, wl.Hkv, wl.d, kmax), dtype=torch.uint8,
                         device=dev)
        ts = []
        for r in range(reps + 3):
            flush.fill_(r & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            sa.sa_select_topk(sa.SA_SELECT_SKETCH, q, sk, None, wl.Hkv, L, L, 64, 0, False, k, 0, 1, wl.scale, idx,
                              cnt)
            sa.sa_decode(q, kc, vc, idx, cnt, L, 64, wl.scale, out, ws)
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        kv = int(cnt.sum().item()) * 64 * wl.d * 2 * 2
        sketch_bytes = wl.Hkv * nb * wl.d * 4
        us = float(np.median(ts))
        rows.append({"L": L, "k": k, "blocks_per_group": int(cnt[0, 0, 0].item()),
                     "kept_fraction": round(int(cnt[0, 0, 0].item()) / nb, 4), "select_plus_decode_us": round(us, 2),
                     "bytes": kv + sketch_bytes, "GB_s": round((kv + sketch_bytes) / us / 1e3, 1)})
        del q, kc, vc, sk, out, ws
        torch.cuda.empty_cache()
    if sa.sa_device_status() != 0:
        raise RuntimeError("device status word set during the length sweep")
    return {"sweep": "length-aware budget", "budget": "k(L) = ceil(%d * (L / %d)^%g)" % (k_ref, L_ref, exponent),
            "workload": "decode B=1 T=4 Hq=32 Hkv=8 d=128 block 64, bf16, 0.5% needle blocks", "rows": rows}


def bench_tokens(reps, peaks, peak_src):
    """Head-collapsed token-level decode ("How Much Dense Attention is Necessary?" Sec. 2.1-2.2) on one
    256K-token sequence (B=1, T=4, Hq=32, Hkv=8, d=128): dense token mass averaged over all heads and
    queries, top-2048 tokens (+ sink and newest), attention over them shared by every kv head.  Each
    rep flushes L2 (256 MB write, untimed) and times each call with CUDA events."""
    import numpy as np
    import torch

    import synth
    import top_block_sparse_pooled_b300 as sa
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = synth.WORKLOADS["c3"].replace(k=2048)
    x = synth.make_inputs(wl)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q, kc, vc = up(x.q), up(x.k), up(x.v)
    del x
    B, T, Hq, Hkv, d, L = wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, wl.L
    R = (Hq // Hkv) * T
    tws = torch.empty(sa.sa_token_mass_workspace_bytes(B, T, Hq, Hkv, L), dtype=torch.uint8, device=dev)
    mass = torch.empty((B, L), dtype=torch.float32, device=dev)
    kmax = sa.sa_select_kmax(L, 1, 0, False, wl.k)
    idx = torch.empty((B, 1, 1, kmax), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, 1, 1), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    dws = torch.zeros(sa.sa_decode_workspace_bytes(B, T, Hq, Hkv, d, kmax), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    calls = {
        "token_mass": lambda: sa.sa_token_mass_decode(q, kc, L, wl.scale, mass, tws),
        "token_select": lambda: sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass.reshape(B, 1, 1, L), 1, L, L, 1,
                                                  0, False, wl.k, 0, 1, 1.0, idx, cnt, d=d, dtype=sa.SA_F32, B=B,
                                                  Tq=1, Hq=1),
        "decode_tokens": lambda: sa.sa_decode_tokens(q, kc, vc, idx.reshape(B, kmax), cnt.reshape(B), L, wl.scale,
                                                     out, dws),
    }
    ts = {name: [] for name in calls}
    for r in range(reps + 2):
        for name, fn in calls.items():
            flush.fill_(r & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                ts[name].append(e0.elapsed_time(e1) * 1e3)
    if sa.sa_device_status() != 0:
        raise RuntimeError("device status word set during the token-level leg")
    us = {name: round(float(np.median(v)), 2) for name, v in ts.items()}
    mass_bytes = B * Hkv * L * d * 2 + 2 * B * Hkv * R * L * 4 + B * L * 4
    sel = int(cnt.sum().item())
    dec_bytes = sel * Hkv * d * 2 * 2
    ach = mass_bytes / (us["token_mass"] * 1e-6) / 1e9
    return {
        "workload": "token-level head-collapsed decode: B=%d T=%d Hq=%d Hkv=%d d=%d L=%d, top-%d tokens + sink + "
                    "newest, shared by the kv heads (bf16)" % (B, T, Hq, Hkv, d, L, wl.k),
        "kernels_us": us,
        "step_us": round(sum(us.values()), 2),
        "token_mass_roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                                "peak_source": peak_src, "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                                "bytes": mass_bytes,
                                "bytes_note": "K read once + base-2 logits written and read back + mass written"},
        "decode_tokens": {"tokens_per_row": sel // B, "bytes": dec_bytes,
                          "GB_s": round(dec_bytes / (us["decode_tokens"] * 1e-6) / 1e9, 1)},
        "l2": "flushed before every timed call (256 MB write, untimed)",
    }


def bench_prefill_tokens(reps, peaks, peak_src):
    """Per-query (b_sel = 1) head-collapsed prefill ("How Much Dense Attention is Necessary?" Sec. 2.1):
    per-query token mass averaged over the heads, per-query top-256 tokens (+ token 0 and the query's
    own), causal attention over each query's tokens; B=1, L=4096, Hq=32, Hkv=8, d=128.  L2 flushed
    before every timed call (256 MB write, untimed)."""
    import numpy as np
    import torch

    import synth
    import top_block_sparse_pooled_b300 as sa
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = synth.WORKLOADS["c5"].replace(B=1, L=4096, k=256, needles=4)
    x = synth.make_inputs(wl)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q, kc, vc = up(x.q), up(x.k), up(x.v)
    del x
    B, Hq, Hkv, d, L = wl.B, wl.Hq, wl.Hkv, wl.d, wl.L
    mws = torch.empty(sa.sa_token_mass_prefill_workspace_bytes(B, L, Hq, Hkv), dtype=torch.uint8, device=dev)
    mass = torch.empty((B, L, L), dtype=torch.float32, device=dev)
    kmax = sa.sa_select_kmax(L, 1, 1, True, wl.k)
    idx = torch.empty((B, 1, L, kmax), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, 1, L), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    pws = torch.zeros(sa.sa_prefill_tokens_workspace_bytes(B, L, Hq, Hkv, d, kmax), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    calls = {
        "token_mass_prefill": lambda: sa.sa_token_mass_prefill(q, kc, wl.scale, mass, mws),
        "token_select": lambda: sa.sa_select_topk(sa.SA_SELECT_MASS, None, None, mass.reshape(B, 1, L, L), 1, L, L,
                                                  1, 1, True, wl.k, 0, 1, 1.0, idx, cnt, d=d, dtype=sa.SA_F32, B=B,
                                                  Tq=L, Hq=1),
        "prefill_tokens": lambda: sa.sa_prefill_tokens(q, kc, vc, idx.reshape(B, L, kmax), cnt.reshape(B, L),
                                                       wl.scale, out, pws),
    }
    ts = {name: [] for name in calls}
    for r in range(reps + 2):
        for name, fn in calls.items():
            flush.fill_(r & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                ts[name].append(e0.elapsed_time(e1) * 1e3)
    if sa.sa_device_status() != 0:
        raise RuntimeError("device status word set during the per-query prefill leg")
    us = {name: round(float(np.median(v)), 2) for name, v in ts.items()}
    # causal logits written and read back (L(L+1)/2 per head), the mass written, K read
    mass_bytes = 2 * B * Hq * (L * (L + 1) // 2) * 4 + B * L * L * 4 + B * Hkv * L * d * 2
    ach = mass_bytes / (us["token_mass_prefill"] * 1e-6) / 1e9
    sel = int(cnt.sum().item())
    # the tensor-core path attends each 128-query tile over the 128-key blocks that hold any of its
    # queries' tokens (each query over its own tokens only): its executed tiles, from the lists
    ih, ch = idx.reshape(B, L, kmax).cpu().numpy(), cnt.reshape(B, L).cpu().numpy()
    tiles = 0
    for b in range(B):
        for i0 in range(0, L, 128):
            blocks = set()
            for t in range(i0, min(i0 + 128, L)):
                row = ih[b, t, :ch[b, t]]
                blocks.update((row[(row >= 0) & (row <= t)] // 128).tolist())
            tiles += len(blocks)
    executed = tiles * Hq * 4 * d * 128 * 128  # QK^T + PV per (tile, block, head)
    return {
        "workload": "per-query (b_sel = 1) head-collapsed prefill: B=%d L=%d Hq=%d Hkv=%d d=%d, top-%d tokens per "
                    "query + token 0 + the query's own (bf16)" % (B, L, Hq, Hkv, d, wl.k),
        "kernels_us": us,
        "step_us": round(sum(us.values()), 2),
        "token_mass_roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                                "peak_source": peak_src, "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                                "bytes": mass_bytes,
                                "bytes_note": "causal base-2 logits written and read back, mass written, K read"},
        "prefill_tokens": {"kernel": "prefill_kernel<true> (tcgen05): 128-query tiles over the 128-key blocks "
                                     "holding their queries' tokens, per-query token masks",
                           "tokens_selected": sel, "executed_tiles": tiles, "executed_tflop": round(executed / 1e12, 4),
                           "tflops_executed": round(executed / (us["prefill_tokens"] * 1e-6) / 1e12, 1),
                           "frac_of_bf16_peak": round(executed / (us["prefill_tokens"] * 1e-6) / 1e12
                                                      / peaks["bf16_tflops"], 4)},
        "l2": "flushed before every timed call (256 MB write, untimed)",
    }


# Sources of each measured kernel: a stored DRAM-traffic figure is reported only while their hash
# still matches the one recorded beside it (null once the kernel has changed).
DECODE_SOURCES = ("k_seldec.cu", "k_select.cu", "k_decode_mma.cu", "sa_ptx.cuh")
PREFILL_SOURCES = ("k_prefill.cu", "sa_tc.cuh", "sa_f32x2.cuh", "sa_ptx.cuh")
MASS_SOURCES = ("k_mass.cu", "sa_tc.cuh", "sa_f32x2.cuh", "sa_ptx.cuh")


def _kernel_hash(sources=DECODE_SOURCES):
    """Hash of a kernel's sources (stored DRAM traffic is used while it matches)."""
    import hashlib
    h = hashlib.sha256()
    for fn in sources:
        with open(os.path.join(ROOT, "top_block_sparse_pooled_b300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _stored_traffic(name, sources):
    """DRAM bytes per launch from profiles/<name> (an ncu capture summary), or None when the file is
    missing or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    t = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            key, val = line.split(":", 1)
            t[key.strip()] = val.strip()
    if t.get("kernel_source_hash") != _kernel_hash(sources):
        return None
    try:
        return int(t["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def bench_reference(args, wl, rank, world):
    """The CPU oracle as it stands, on the same workload; each step is the oracle's decode
    step on a bounded sample (a prefix of the batch) so that K steps take a few minutes."""
    import oracle
    import synth
    if rank != 0:
        return None
    x = synth.make_inputs(wl)
    budget = max(0.002, 150.0 / max(1, args.steps + args.warmup))
    ng = 1
    dt, _ = oracle_decode_sample(wl, x, ng)
    for cand in _sample_sizes(wl)[1:]:
        if dt * cand / ng > budget:
            break
        ng = cand
        dt, _ = oracle_decode_sample(wl, x, ng)
    for _ in range(max(0, args.warmup - 1)):
        oracle_decode_sample(wl, x, ng)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        t, b = oracle_decode_sample(wl, x, ng)
        tot_t += t
        tot_b += b
    value = tot_b / tot_t / 1e9
    sample = "%d of %d groups per step, full context %d" % (ng, wl.B * wl.Hkv, wl.L)
    return {
        "impl": "reference",
        "metric": "sparse-attn decode KV GB/s (% HBM peak)",
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same generator and seed as the CUDA arm)",
        "config": {"workload": "%s decode: B=%d T=%d Hq=%d Hkv=%d d=%d L=%d block=%d top-k=%d + sink + local" % (
            wl.name, wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, wl.L, wl.Bk, wl.k)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=["c1", "c2", "c3"])
    ap.add_argument("--rotate", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-decode-legs", dest="decode_legs", action="store_false",
                    help="skip the c3 / c1 decode legs after the headline workload")
    ap.add_argument("--prefill-steps", type=int, default=5,
                    help="steps of each prefill leg (c5 sketch-selected, c4 oracle-mass); 0 skips them")
    ap.add_argument("--prefill-only", action="store_true", help="run only the prefill legs (profiling)")
    ap.add_argument("--prefill-workload", default="both", choices=["both", "c4", "c5"],
                    help="with --prefill-only: which prefill leg to run (profiling one workload)")
    ap.add_argument("--sweep-length", action="store_true",
                    help="decode across context lengths with the length-aware budget (separate report)")
    ap.add_argument("--prefill-B", type=int, default=0, help="override the prefill legs' batch (profiling)")
    ap.add_argument("--prefill-L", type=int, default=0, help="override the prefill legs' context (profiling)")
    ap.add_argument("--tokens-reps", type=int, default=5,
                    help="timed reps of the token-level decode leg (0 skips it)")
    ap.add_argument("--tokens-only", action="store_true", help="run only the token-level decode leg")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    wl = workload(args.workload)
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    if args.impl == "reference":
        res = bench_reference(args, wl, rank, world)
    else:
        def pf_wl(name):
            w = workload(name)
            if args.prefill_B:
                w = w.replace(B=args.prefill_B)
            if args.prefill_L:
                w = w.replace(L=args.prefill_L)
            return w

        if args.sweep_length:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            res = bench_length_sweep([16384, 32768, 65536, 131072, 262144], 80, 262144, 0.5)
        elif args.tokens_only:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            peaks, src = load_peaks()
            res = {"tokens": bench_tokens(max(1, args.tokens_reps), peaks, src),
                   "prefill_tokens": bench_prefill_tokens(max(1, args.tokens_reps), peaks, src)}
        elif args.prefill_only:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            peaks, src = load_peaks()
            names = ("c5", "c4") if args.prefill_workload == "both" else (args.prefill_workload,)
            res = {"prefill": [bench_prefill(pf_wl(n), max(1, args.prefill_steps), peaks, src,
                                             full_size=not (args.prefill_B or args.prefill_L)) for n in names]}
        else:
            res = bench_decode(args, wl, rank, world)
            if args.decode_legs and res is not None:
                # the other decode workloads, same step definition: c3 (256K context, 4 query tokens)
                # and c1 (fp32, 4K context; 128 rotated sets so that no step finds its blocks in L2)
                res["decode_legs"] = []
                for name, rot in (("c3", 8), ("c1", 128)):
                    if name == wl.name:
                        continue
                    leg = bench_decode(args, workload(name), rank, world, steps=min(args.steps, 4000), rotate=rot,
                                       cpu_seconds=min(args.cpu_seconds, 8.0))
                    res["decode_legs"].append(_leg_summary(leg))
            if args.prefill_steps > 0 and res is not None:
                peaks, src = load_peaks()
                cs = min(args.cpu_seconds, 10.0) if (args.cpu_baseline and rank == 0) else 0.0
                res["prefill"] = [bench_prefill(pf_wl(n), args.prefill_steps, peaks, src, cs,
                                                 full_size=not (args.prefill_B or args.prefill_L))
                                   for n in ("c5", "c4")]
                res["gpu_launches"] += 4 * args.prefill_steps * 2
            if args.tokens_reps > 0 and res is not None:
                peaks, src = load_peaks()
                res["tokens"] = bench_tokens(args.tokens_reps, peaks, src)
                res["prefill_tokens"] = bench_prefill_tokens(args.tokens_reps, peaks, src)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
