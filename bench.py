#!/usr/bin/env python
"""Benchmark: useful (unmasked) attention TFLOP/s of one forward + backward step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input: the planner and
forward kernel (out, lse), then the backward planner, preprocess, backward kernel and dq
conversion (dq, dk, dv).  Useful FLOPs per step = (4 + 10) * d * Hq * V, V = visible
(query, key) pairs under union semantics (forward: two GEMMs, backward: five, 2 flops per
multiply-add); masked work inside partial tiles is not counted.

Default workload: 65536 packed tokens, Hq 16 / Hkv 4, d 128, one CAUSAL slice over all
tokens plus two FULL slices over a 4096-token prefix (bf16 N(0,1), seed 3).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--impl reference times the float64 CPU oracle (a deliberately slow baseline) on a bounded
sample of the same workload.  With N > 1 (torchrun), every rank runs an independent replica
of the workload on its own GPU: the attention has no cross-GPU exchange.
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "unmasked attention TFLOP/s fwd/bwd on 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def headline_peak(peaks: dict, clocks: dict):
    """(peak TFLOP/s, name) for the headline fractions: the burst cuBLAS bf16 figure unless the
    median SM clock of the timed region was nearer the clock the sustained figure was measured
    at (its median under load) than the maximum, then the sustained figure; without that
    record, the burst figure unless the clock was below 97 % of the maximum.  No clock record:
    the sustained figure."""
    peak_burst = float(peaks.get("bf16_tflops", 1900.0))
    peak_sust = float(peaks.get("bf16_tflops_sustained", peak_burst))
    sust_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    at_max = False
    if clocks.get("sm_mhz") is not None and clocks.get("sm_max_mhz"):
        thr = 0.5 * (float(sust_mhz) + clocks["sm_max_mhz"]) if sust_mhz else 0.97 * clocks["sm_max_mhz"]
        at_max = clocks["sm_mhz"] >= thr
    return (peak_burst, "bf16_tflops (burst)") if at_max else (peak_sust, "bf16_tflops_sustained")


def visible_pairs(w: W.Workload) -> int:
    """Exact visible-pair count from the slice list (per-row interval union, host-side)."""
    # Rows are processed in blocks; each row's visible set is the union of one interval per
    # slice that covers it.  Pure counting, no attention arithmetic.
    total = w.total
    qr = np.asarray(w.q_ranges, dtype=np.int64).reshape(-1, 2)
    kr = np.asarray(w.k_ranges, dtype=np.int64).reshape(-1, 2)
    ty = np.asarray(w.types, dtype=np.int64)
    keep = (qr[:, 0] < qr[:, 1]) & (kr[:, 0] < kr[:, 1])
    qr, kr, ty = qr[keep], kr[keep], ty[keep]
    n = 0
    for r0 in range(0, total, 8192):
        rows = np.arange(r0, min(total, r0 + 8192))[:, None]
        sel = (qr[:, 0] < rows[-1, 0] + 1) & (qr[:, 1] > r0)
        if not sel.any():
            continue
        qs, qe, ks, ke, t = qr[sel, 0], qr[sel, 1], kr[sel, 0], kr[sel, 1], ty[sel]
        inside = (rows >= qs) & (rows < qe)
        hi = np.where(t == 1, np.minimum(ke, rows + ke - qe + 1), ke)
        lo = np.broadcast_to(ks, hi.shape)
        hi = np.where(inside, np.maximum(hi, lo), lo)
        order = np.argsort(np.where(hi > lo, lo, 1 << 60), axis=1, kind="stable")
        lo_s = np.take_along_axis(lo, order, 1)
        hi_s = np.take_along_axis(hi, order, 1)
        cur = np.full(rows.shape[0], -1, dtype=np.int64)
        for c in range(lo_s.shape[1]):
            a, b = lo_s[:, c], hi_s[:, c]
            valid = b > a
            st = np.maximum(a, cur)
            n += int(np.where(valid, np.maximum(0, b - st), 0).sum())
            cur = np.where(valid, np.maximum(cur, b), cur)
    return n


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.gpu, self.path, self.proc = gpu_index, path, None

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                s = float(parts[1].split()[0]); mx = float(parts[2].split()[0])
            except ValueError:
                continue
            smax = mx
            sm.append(s)
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"]}
        loaded = [x for x in sm if x >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def smi_index(cuda_index: int) -> int:
    """nvidia-smi index of a CUDA device (honours CUDA_VISIBLE_DEVICES when it lists indices)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if cuda_index < len(ids) and ids[cuda_index].isdigit():
        return int(ids[cuda_index])
    return cuda_index


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host float over ranks (host-side timing reduction, not a data-path collective)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_inputs(w: W.Workload):
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    qr, kr, ty = W.ranges_tensors(w.padded())
    return q, k, v, do, qr, kr, ty


def run_ours(args, w: W.Workload, rank: int, world: int, local: int):
    import flexible_mask_attention_range_gb300 as ffa
    from flexible_mask_attention_range_gb300 import build as ffa_build
    ffa_build.ensure_built()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    V = visible_pairs(w)
    fl_fwd = 4.0 * w.d * w.hq * V
    fl_bwd = 10.0 * w.d * w.hq * V
    q_h, k_h, v_h, do_h, qr_h, kr_h, ty_h = make_inputs(w)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    qr, kr, ty = (t.to(dev) for t in (qr_h, kr_h, ty_h))
    out = torch.empty_like(q)
    lse = torch.empty(w.hq, w.total, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    R = qr.shape[0]
    wsf = torch.empty(ffa.ffa_fwd_workspace_size(w.total, w.total, w.hq, w.hkv, w.d, R), dtype=torch.uint8,
                      device=dev)
    wsb = torch.empty(ffa.ffa_bwd_workspace_size(w.total, w.total, w.hq, w.hkv, w.d, R), dtype=torch.uint8,
                      device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = w.softmax_scale

    def step():
        ffa.ffa_fwd(q, k, v, qr, kr, ty, scale, w.softcap, out=out, lse=lse, workspace=wsf, status=status)
        ffa.ffa_bwd(q, k, v, out, lse, do, qr, kr, ty, scale, w.softcap, dq=dq, dk=dk, dv=dv, workspace=wsb,
                    status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    # ---- device-timed region: K steps, events around every main kernel launch
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    # torch creates events lazily: record each once so the handle exists; the library then
    # re-records it around its kernel launch on the same stream
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock_dir = os.environ.get("FFA_BENCH_CLOCKS_DIR", tempfile.gettempdir())
    clock_path = os.path.join(clock_dir, f"bench_clocks_rank{rank}.csv")
    os.makedirs(os.path.dirname(clock_path), exist_ok=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(smi_index(dev.index), clock_path) as clk:
        time.sleep(0.3)
        t0.record()
        for i in range(K):
            ffa.ffa_set_kernel_events(*ev[i])
            step()
        t1.record()
        ffa.ffa_set_kernel_events()
        torch.cuda.synchronize()
        time.sleep(0.2)
    barrier(world)
    ms_total = t0.elapsed_time(t1)
    ms_step = max_over_ranks(ms_total / K, world)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    clocks = clk.summary()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    value = world * (fl_fwd + fl_bwd) / (ms_step * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers (pinned), copies timed.
    # Every step uploads its inputs (q, k, v, dO, ranges) from pinned host memory and
    # downloads its results (out, lse, dq, dk, dv); uploads run on one copy stream, downloads
    # on another, and compute on the current stream, with two device buffer sets so step
    # i+1's upload and step i-1's download overlap step i's kernels.
    q_p, k_p, v_p, do_p = (t.pin_memory() for t in (q_h, k_h, v_h, do_h))
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (out, lse, dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in (q_p, k_p, v_p, do_p, qr_h, kr_h, ty_h))
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    E = max(3, K)  # pipeline fill (first upload) and drain (last download) amortised over K steps
    sets = []
    for _ in range(2):
        ins = [torch.empty_like(t) for t in (q, k, v, do, qr, kr, ty)]
        outs = [torch.empty_like(t) for t in (out, lse, dq, dk, dv)]
        sets.append((ins, outs))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)

    def e2e_run(n):
        done = [None, None]     # compute finished with set b (inputs and outputs)
        drained = [None, None]  # download of set b finished
        last = None
        for i in range(n):
            b = i % 2
            ins, outs = sets[b]
            with torch.cuda.stream(up):
                if done[b] is not None:
                    up.wait_event(done[b])
                for dst, src in zip(ins, (q_p, k_p, v_p, do_p, qr_h, kr_h, ty_h)):
                    dst.copy_(src, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            main.wait_stream(up)
            if drained[b] is not None:
                main.wait_event(drained[b])
            qi, ki, vi, doi, qri, kri, tyi = ins
            oo, ll, dqo, dko, dvo = outs
            ffa.ffa_fwd(qi, ki, vi, qri, kri, tyi, scale, w.softcap, out=oo, lse=ll, workspace=wsf, status=status)
            ffa.ffa_bwd(qi, ki, vi, oo, ll, doi, qri, kri, tyi, scale, w.softcap, dq=dqo, dk=dko, dv=dvo,
                        workspace=wsb, status=status)
            done[b] = torch.cuda.Event()
            done[b].record(main)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                for dst, src in zip(host_out, outs):
                    dst.copy_(src, non_blocking=True)
                drained[b] = torch.cuda.Event()
                drained[b].record(down)
                last = drained[b]
        main.wait_event(last)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    up.wait_stream(main)
    down.wait_stream(main)
    e0.record(main)
    up.wait_event(e0)
    down.wait_event(e0)
    e2e_run(E)
    e1.record(main)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, world)
    e2e_value = world * (fl_fwd + fl_bwd) / (e2e_ms * 1e-3) / 1e12

    bwd_tf = fl_bwd / (bwd_ms * 1e-3) / 1e12
    fwd_tf = fl_fwd / (fwd_ms * 1e-3) / 1e12
    peak_burst = float(peaks.get("bf16_tflops", 1900.0))
    peak_sust = float(peaks.get("bf16_tflops_sustained", peak_burst))
    peak_t, peak_kind = headline_peak(peaks, clocks)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "total_seqlen": w.total, "num_heads_q": w.hq, "num_heads_kv": w.hkv,
                   "head_dim": w.d, "slices": len(w.types), "softcap": w.softcap, "visible_pairs": V,
                   "pass": "fwd+bwd", "l2": "inputs larger than L2 (q alone is "
                   f"{w.total * w.hq * w.d * 2 / 2**20:.0f} MiB)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2),
        "fwd_kernel_ms": round(fwd_ms, 4), "bwd_kernel_ms": round(bwd_ms, 4),
        "frac_of_peak": {"fwd": round(fwd_tf / peak_t, 4), "bwd": round(bwd_tf / peak_t, 4),
                         "step": round(value / world / peak_t, 4), "peak": f"{peak_kind} of {peak_src}",
                         "fwd_of_burst": round(fwd_tf / peak_burst, 4), "bwd_of_burst": round(bwd_tf / peak_burst, 4),
                         "fwd_of_sustained": round(fwd_tf / peak_sust, 4),
                         "bwd_of_sustained": round(bwd_tf / peak_sust, 4)},
        "roofline": {"kernel": "ffa_bwd_kernel", "bound": "tensor", "achieved": round(bwd_tf, 2),
                     "peak": peak_t, "unit": "TFLOP/s", "frac": round(bwd_tf / peak_t, 4),
                     "traffic": kernel_traffic(w.name, "ffa_bwd_kernel"),
                     "peak_source": f"{peak_kind} of {peak_src} (median SM clock {clocks.get('sm_mhz')} MHz)"},
        "roofline_fwd": {"kernel": "ffa_fwd_kernel", "bound": "tensor", "achieved": round(fwd_tf, 2),
                         "peak": peak_t, "unit": "TFLOP/s", "frac": round(fwd_tf / peak_t, 4),
                         "traffic": kernel_traffic(w.name, "ffa_fwd_kernel")},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "copies": "pinned, own streams, overlapped with compute"},
        "gpu_launches": K * GPU_LAUNCHES_PER_STEP,
        "clocks": clocks,
    }
    return result, (q_h, k_h, v_h, do_h)


# planner (slices, rows, order) + forward; planner (slices, cols, order) + pre + backward + convert
GPU_LAUNCHES_PER_STEP = 4 + 6


def algorithmic_bytes(w: W.Workload):
    """Bytes a pass must move at least: forward reads Q, K, V and writes O (bf16) and LSE
    (f32); backward reads Q, K, V, O, dO, LSE and D and writes dQ, dK, dV."""
    qb = w.total * w.hq * w.d * 2
    kb = w.total * w.hkv * w.d * 2
    row = w.total * w.hq * 4
    fwd = qb + 2 * kb + qb + row
    bwd = 3 * qb + 2 * kb + 2 * row + qb + 2 * kb
    return fwd, bwd


def time_calls(w: W.Workload, calls: int, phase: str):
    """`calls` forward and/or backward calls of one workload, each timed with CUDA events
    (whole call and main kernel), L2 flushed before each; a fixed launch sequence for
    profilers (ncu -s / -c count the main-kernel launches of these calls)."""
    import flexible_mask_attention_range_gb300 as ffa
    from flexible_mask_attention_range_gb300 import build as ffa_build
    ffa_build.ensure_built()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q_h, k_h, v_h, do_h, qr_h, kr_h, ty_h = make_inputs(w)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    qr, kr, ty = (t.to(dev) for t in (qr_h, kr_h, ty_h))
    out = torch.empty_like(q)
    lse = torch.empty(w.hq, w.total, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    do_fwd = phase in ("fwd", "both") or not w.backward
    do_bwd = phase in ("bwd", "both") and w.backward
    t = {"fwd": [], "bwd": []}
    if not do_fwd:  # the backward needs out and lse
        ffa.ffa_fwd(q, k, v, qr, kr, ty, w.softmax_scale, w.softcap, out=out, lse=lse, status=st)
    for _ in range(calls):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        if do_fwd:
            flush.zero_()
            ev[0].record()
            ffa.ffa_fwd(q, k, v, qr, kr, ty, w.softmax_scale, w.softcap, out=out, lse=lse, status=st)
            ev[1].record()
        if do_bwd:
            flush.zero_()
            ev[2].record()
            ffa.ffa_bwd(q, k, v, out, lse, do, qr, kr, ty, w.softmax_scale, w.softcap, dq=dq, dk=dk, dv=dv,
                        status=st)
            ev[3].record()
        torch.cuda.synchronize()
        if do_fwd:
            t["fwd"].append(ev[0].elapsed_time(ev[1]))
        if do_bwd:
            t["bwd"].append(ev[2].elapsed_time(ev[3]))
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    return {"workload": w.name, "calls": calls,
            **{f"{ph}_ms_median": round(statistics.median(x), 4) for ph, x in t.items() if x}}


def time_decode(ffa, dw, dev, flush, iters: int, warm: int):
    """Whole ffa_fwd_decode calls on a decoding batch (packing, slices, attention, merge,
    unpacking), L2 flushed before each; milliseconds of the timed calls."""
    q_h, k_h, v_h = dw.draw()
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    qr, kr, ty = (torch.tensor(x, dtype=torch.int32, device=dev) for x in dw.slices())
    out = torch.empty_like(q)
    lse = torch.empty(dw.hq, dw.total_q, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None
    t = []
    for i in range(warm + iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        e0.record()
        out, lse = ffa.ffa_fwd_decode(q, k, v, qr, kr, ty, max_seqlen_q=dw.q_len, out=out, lse=lse, workspace=ws,
                                      status=st)
        e1.record()
        torch.cuda.synchronize()
        if i >= warm:
            t.append(e0.elapsed_time(e1))
    if int(st.item()) != 0:
        raise RuntimeError(f"{dw.name}: device status {int(st.item())}")
    return t


def per_config(ffa, dev, peaks, iters: int = 10, warm: int = 3):
    """Every workload of the project timed alone on this GPU: the whole forward call (planner,
    kernel, merge) and backward call (planner, preprocess, kernel, dq conversion) with CUDA
    events on the launching stream, L2 flushed (a 256 MiB write) before every timed call;
    medians of `iters` calls after `warm` untimed ones.  The main kernels alone are timed with
    the library's event hook in the same calls."""
    peak_b = float(peaks.get("bf16_tflops", 1900.0))
    peak_s = float(peaks.get("bf16_tflops_sustained", peak_b))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {}
    for name in W.ORDER:
        w = W.get(name)
        V = visible_pairs(w)
        q_h, k_h, v_h, do_h, qr_h, kr_h, ty_h = make_inputs(w)
        q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
        qr, kr, ty = (t.to(dev) for t in (qr_h, kr_h, ty_h))
        out = torch.empty_like(q)
        lse = torch.empty(w.hq, w.total, dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        R = qr.shape[0]
        wsf = torch.empty(ffa.ffa_fwd_workspace_size(w.total, w.total, w.hq, w.hkv, w.d, R), dtype=torch.uint8,
                          device=dev)
        wsb = torch.empty(ffa.ffa_bwd_workspace_size(w.total, w.total, w.hq, w.hkv, w.d, R), dtype=torch.uint8,
                          device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        t = {"fwd": [], "bwd": [], "fwd_kernel": [], "bwd_kernel": []}
        for i in range(warm + iters):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
            for e in ev:
                e.record()
            flush.zero_()
            ffa.ffa_set_kernel_events(ev[2], ev[3], None, None)
            ev[0].record()
            ffa.ffa_fwd(q, k, v, qr, kr, ty, w.softmax_scale, w.softcap, out=out, lse=lse, workspace=wsf, status=st)
            ev[1].record()
            if w.backward:
                flush.zero_()
                ffa.ffa_set_kernel_events(None, None, ev[6], ev[7])
                ev[4].record()
                ffa.ffa_bwd(q, k, v, out, lse, do, qr, kr, ty, w.softmax_scale, w.softcap, dq=dq, dk=dk, dv=dv,
                            workspace=wsb, status=st)
                ev[5].record()
            ffa.ffa_set_kernel_events()
            torch.cuda.synchronize()
            if i >= warm:
                t["fwd"].append(ev[0].elapsed_time(ev[1]))
                t["fwd_kernel"].append(ev[2].elapsed_time(ev[3]))
                if w.backward:
                    t["bwd"].append(ev[4].elapsed_time(ev[5]))
                    t["bwd_kernel"].append(ev[6].elapsed_time(ev[7]))
        if int(st.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(st.item())}")
        fb, bb = algorithmic_bytes(w)
        e = {"visible_pairs": V, "tokens": w.total, "heads": f"{w.hq}/{w.hkv}", "d": w.d, "softcap": w.softcap,
             "slices": len(w.types)}
        for ph, flop, byt in (("fwd", 4.0 * w.d * w.hq * V, fb), ("bwd", 10.0 * w.d * w.hq * V, bb)):
            if not t[ph]:
                continue
            ms = statistics.median(t[ph])
            kms = statistics.median(t[ph + "_kernel"])
            tf = flop / (ms * 1e-3) / 1e12
            ktf = flop / (kms * 1e-3) / 1e12
            e[ph] = {"ms": round(ms, 4), "us": round(ms * 1e3, 1), "tflops": round(tf, 2),
                     "frac_burst": round(tf / peak_b, 4), "frac_sustained": round(tf / peak_s, 4),
                     "hbm_gbs": round(byt / (ms * 1e-3) / 1e9, 1), "algorithmic_bytes": byt,
                     "kernel_ms": round(kms, 4), "kernel_tflops": round(ktf, 2),
                     "kernel_frac_burst": round(ktf / peak_b, 4)}
        res[name] = e
        del q, k, v, do, out, lse, dq, dk, dv, wsf, wsb
        torch.cuda.empty_cache()
    for name, dw in W.DECODE.items():
        ms = statistics.median(time_decode(ffa, dw, dev, flush, iters, warm))
        kv_bytes = 2 * dw.total_k * dw.hkv * dw.d * 2
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        res[name] = {"sequences": dw.n_seq, "new_tokens": dw.q_len, "keys_per_sequence": dw.kv_len,
                     "heads": f"{dw.hq}/{dw.hkv}", "d": dw.d, "ms": round(ms, 4), "us": round(ms * 1e3, 1),
                     "kv_bytes": kv_bytes, "hbm_gbs": round(gbs, 1),
                     "frac_hbm": round(gbs / float(peaks.get("hbm_gbs", 6800.0)), 4)}
        torch.cuda.empty_cache()
    res["_timing"] = (f"median of {iters} calls after {warm} warm-up calls; L2 flushed (256 MiB write) before "
                      "every timed call; 'ms' = whole call (planner included), 'kernel_ms' = main kernel alone; "
                      f"peaks: burst {peak_b}, sustained {peak_s} TFLOP/s")
    return res


# DRAM bytes per launch of the main kernels (dram__bytes_read.sum + dram__bytes_write.sum from
# one ncu capture of this benchmark's full-size workload; the capture command is in
# profiles/).  Each entry carries the hash of the kernel's sources at capture time: once a
# source changes the figure no longer describes the kernel, and `traffic` is reported null.
TRAFFIC = {
    # (workload, kernel): (bytes per launch, source hash at capture)
    ("long_causal_64k_prefix", "ffa_fwd_kernel"): (1856736000 + 238412032, "388d8b2834b203d0"),
    ("long_causal_64k_prefix", "ffa_bwd_kernel"): (23225705728 + 11979547904, "743ef98528ce98e7"),
    ("sliding_32k_softcap", "ffa_fwd_kernel"): (541080320 + 240462336, "388d8b2834b203d0"),
    ("sliding_32k_softcap", "ffa_bwd_kernel"): (2695739392 + 1358949376, "743ef98528ce98e7"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources that define a main kernel (its .cu plus the shared headers)."""
    import hashlib
    csrc = os.path.join(ROOT, "flexible_mask_attention_range_gb300", "csrc")
    unit = {"ffa_fwd_kernel": "ffa_fwd.cu", "ffa_bwd_kernel": "ffa_bwd.cu"}[kernel]
    h = hashlib.sha256()
    for f in (unit, "ffa_ptx.cuh", "ffa_internal.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_traffic(workload: str, kernel: str):
    e = TRAFFIC.get((workload, kernel))
    if e is None or e[1] != kernel_source_hash(kernel):
        return None
    return e[0]


def oracle_sample(w: W.Workload, inputs, rows: np.ndarray):
    """Time the float64 oracle on a bounded sample: forward + dq for the given rows."""
    import oracle as O
    q, k, v, do = inputs
    t0 = time.perf_counter()
    O.forward(q, k, v, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale, softcap=w.softcap,
              rows=rows)
    O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale, softcap=w.softcap,
               rows=rows)
    dt = time.perf_counter() - t0
    # useful flops of the sample: forward 4 d Hq per visible pair, dq-only backward 6 d Hq
    qr = np.asarray(w.q_ranges, dtype=np.int64).reshape(-1, 2)
    kr = np.asarray(w.k_ranges, dtype=np.int64).reshape(-1, 2)
    ty = np.asarray(w.types)
    pairs = 0
    for i in rows:
        ivs = []
        for (qs, qe), (ks, ke), t in zip(qr, kr, ty):
            if qs <= i < qe and ks < ke:
                hi = min(ke, i + ke - qe + 1) if t == 1 else ke
                if hi > ks:
                    ivs.append((ks, hi))
        ivs.sort()
        cur = -1
        for a, b in ivs:
            a = max(a, cur)
            if b > a:
                pairs += b - a
            cur = max(cur, b)
    flops = (4.0 + 6.0) * w.d * w.hq * pairs
    return dt, flops


# about 15 s of float64 oracle work on the 64K workload on the GPU host (about 0.04 s per row)
CPU_BASELINE_ROWS = 384


def cpu_threads() -> int:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def sample_rows(w: W.Workload, n: int, seed: int):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(w.total, size=n, replace=False))


def oracle_report(names, single_thread_names):
    """The float64 oracle timed on this host's cores for each workload: the whole forward (and
    backward where the workload has one) for the small ones, a seeded sample of 128 query rows
    (forward + dq over each row's full key set) for the large ones, with the time of the full
    pass extrapolated by useful flops.  Workloads in `single_thread_names` are timed again in a
    child process restricted to one BLAS thread."""
    import oracle as O
    res = {"host_cores": os.cpu_count(), "blas_threads": cpu_threads()}
    for name in names:
        w = W.get(name)
        V = visible_pairs(w)
        q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
        full = (4.0 + (10.0 if w.backward else 0.0)) * w.d * w.hq * V
        if w.total <= 16384:
            t0 = time.perf_counter()
            O.forward(q, k, v, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale, softcap=w.softcap)
            tf = time.perf_counter() - t0
            tb = 0.0
            if w.backward:
                t0 = time.perf_counter()
                O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale,
                           softcap=w.softcap)
                tb = time.perf_counter() - t0
            res[name] = {"kind": "full pass", "fwd_s": round(tf, 3), "bwd_s": round(tb, 3) if w.backward else None,
                         "tflops": full / (tf + tb) / 1e12}
        else:
            rows = sample_rows(w, 128, 7)
            dt, fl = oracle_sample(w, (q, k, v, do), rows)
            res[name] = {"kind": "128 sampled rows, forward + dq", "sample_s": round(dt, 3), "tflops": fl / dt / 1e12,
                         "extrapolated_full_fwd_bwd_s": round(dt * full / fl, 1)}
    if single_thread_names:
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-report", "--oracle-configs",
                            ",".join(single_thread_names), "--oracle-single", ""], env=env, capture_output=True,
                           text=True, check=True)
        res["single_thread"] = json.loads(r.stdout.strip().splitlines()[-1])
    return res


def run_reference(args, w: W.Workload):
    inputs = make_inputs(w)[:4]
    rows_per_step = 24
    for i in range(args.warmup):
        oracle_sample(w, inputs, sample_rows(w, rows_per_step, 1000 + i))
    times, flops = [], []
    for i in range(args.steps):
        dt, fl = oracle_sample(w, inputs, sample_rows(w, rows_per_step, i))
        times.append(dt)
        flops.append(fl)
    value = sum(flops) / sum(times) / 1e12
    cores = cpu_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "total_seqlen": w.total, "num_heads_q": w.hq, "num_heads_kv": w.hkv,
                   "head_dim": w.d, "pass": "fwd+bwd(dq) on sampled rows"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step (forward + dq over each "
                                   "row's full key set, all heads), float64 numpy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_causal_64k_prefix", choices=sorted(W.ALL) + sorted(W.DECODE))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload table")
    ap.add_argument("--oracle-report", action="store_true",
                    help="time the float64 oracle on the host cores for every workload and exit")
    ap.add_argument("--calls", type=int, default=0,
                    help="time N forward (and backward) calls of --workload alone and exit (profiling aid)")
    ap.add_argument("--phase", choices=["fwd", "bwd", "both"], default="both")
    ap.add_argument("--oracle-configs", default=",".join(W.ORDER))
    ap.add_argument("--oracle-single", default="tiny_256,page1_2048_gqa,docs_16k",
                    help="workloads also timed on one BLAS thread (empty: none)")
    args = ap.parse_args()
    if args.oracle_report:
        names = [x for x in args.oracle_configs.split(",") if x]
        single = [x for x in args.oracle_single.split(",") if x]
        print(json.dumps(oracle_report(names, single)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.calls > 0 and args.workload in W.DECODE:
        import flexible_mask_attention_range_gb300 as ffa
        dev = torch.device("cuda", 0)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        t = time_decode(ffa, W.DECODE[args.workload], dev, flush, args.calls, 0)
        print(json.dumps({"workload": args.workload, "calls": args.calls, "ms_median": statistics.median(t)}))
        return
    w = W.get(args.workload)
    if args.calls > 0:
        print(json.dumps(time_calls(w, args.calls, args.phase)), flush=True)
        return
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    result, inputs = run_ours(args, w, rank, world, local)
    if world == 1 and not args.no_per_config:
        import flexible_mask_attention_range_gb300 as ffa
        result["per_config"] = per_config(ffa, torch.device("cuda", 0), load_peaks()[0])
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            n_rows = CPU_BASELINE_ROWS
            rows = sample_rows(w, n_rows, 77)
            dt, fl = oracle_sample(w, inputs, rows)
            result["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": UNIT, "cores": cpu_threads(),
                                      "kind": "oracle", "seconds": round(dt, 2),
                                      "sample": f"{n_rows} random query rows (forward + dq over each row's "
                                                "full key set, all heads), float64 numpy"}
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
