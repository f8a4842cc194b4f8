#!/usr/bin/env python3
"""Benchmark of the TND attention score-gradient on B300.

One step = one tnd_attn_grad call (prepass, main gradient kernel, dSink
reduction when a sink is present) over one batch of the synthetic workload,
inputs already resident in HBM.  Metric: mask-adjusted attention-grad TFLOP/s,
FLOP = sum over sequences and query heads of 10 * D * (kept (q, kv) pairs)
(five GEMMs of 2*D FLOP per kept pair: S, dP, dV, dK, dQ; dropout does not
reduce the count), and its fraction of the measured dense BF16 peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 the script runs under torchrun: every rank processes its own copy
of the workload (independent replicas, no collective on the data path), the
timed region is bracketed by barriers and rank 0 reports the maximum over
ranks.  --impl reference times the fp64 CPU oracle on the host cores on a
bounded sample of the same workload (the reference arm of this project).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention-grad TFLOP/s (mask-adjusted) & % of B300 dense BF16 tensor peak"
DEFAULT_WORKLOAD = "causal_varlen_bf16"
FLUSH_BYTES = 256 << 20
# one oracle sample (forward + gradient in fp64 on the host cores): about
# ORACLE_TARGET_S of work, never more than ORACLE_MAX_S; the same sample for
# the cpu_baseline leg and every step of the reference arm
ORACLE_TARGET_S = 3.0
ORACLE_MAX_S = 8.0
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def max_over_ranks(x: float, dist, dev) -> float:
    """The largest of every rank's x: the time of the slowest replica (x
    itself with one process)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flop_per_replica: float, ms: float) -> float:
    """Whole-job throughput: every replica's FLOP over the slowest replica's time."""
    return world * flop_per_replica / (ms * 1e-3) / 1e12


def kept_pairs(wl) -> int:
    """Kept (q-row, kv-row) pairs summed over sequences and query heads,
    counted row by row from the sparseMode definitions."""
    total = 0
    for sq, skv in zip(wl.seqlens_q, wl.seqlens_kv):
        i = np.arange(sq, dtype=np.int64)
        lo = np.zeros(sq, dtype=np.int64)
        hi = np.full(sq, skv - 1, dtype=np.int64)
        if wl.sparse_mode == 2:
            hi = np.minimum(hi, i)
        elif wl.sparse_mode == 3:
            hi = np.minimum(hi, i + skv - sq)
        elif wl.sparse_mode == 4:
            lo = np.maximum(lo, i - wl.pre_tokens)
            hi = np.minimum(hi, i + wl.next_tokens)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total * wl.nq


def grad_flop(wl) -> float:
    return 10.0 * wl.d * kept_pairs(wl)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of `kernel` on
    `workload`, if it was taken on the current kernel source (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    rec = {}
    for line in text.splitlines():
        if line.startswith("- ") and ": " in line:
            k, v = line[2:].split(": ", 1)
            rec[k.strip()] = v.strip()
    src = os.path.join(ROOT, "attention_backward_tnd_b300", "csrc", rec.get("source", ""))
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if sha != rec.get("source_sha256_16") or rec.get("workload") is None:
        return None
    try:
        return {"bytes_per_launch": float(rec["dram_bytes_per_launch"]), "workload": rec["workload"]}
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every millisecond by
    an NVML thread; summary() keeps the samples taken inside the marked timed
    region (None when NVML is unavailable)."""

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []          # (host time, sm MHz, max MHz, reason bits)
        self.t0 = self.t1 = None
        self._stop = False
        self._thread = None
        self._handle = None

    def _open(self):
        """NVML through the driver's own library (ctypes), present wherever the driver is."""
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        props = torch.cuda.get_device_properties(self.dev)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(0), ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML device handle")
        self._nv, self._handle = nv, h
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reason_fn = fn if fn is not None else nv.nvmlDeviceGetCurrentClocksThrottleReasons

    def _sample(self):
        import ctypes
        sm, mx, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        nv, h = self._nv, self._handle
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) != 0:      # NVML_CLOCK_SM = 1
            return None
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        self._reason_fn(h, ctypes.byref(rs))
        return float(sm.value), float(mx.value), int(rs.value)

    def _run(self):
        while not self._stop:
            x = self._sample()
            if x is not None:
                self.samples.append((time.perf_counter(),) + x)
            time.sleep(0.001)

    def __enter__(self):
        import threading
        try:
            self._open()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        except Exception:
            self._thread = None
        return self

    def mark(self, start: bool):
        if start:
            self.t0 = time.perf_counter()
        else:
            self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return None
        inside = [x for x in self.samples if self.t0 is not None and self.t1 is not None and self.t0 <= x[0] <= self.t1]
        rows = inside or self.samples[-3:]
        bits = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
                "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
        reasons = sorted({name for _, _, _, r in rows for name, b in bits.items() if r & b})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows), "in_timed_region": bool(inside), "source": "nvml"}


def workload_config(wl, l2_note=True):
    cfg = {"workload": wl.name, "dtype": wl.dtype, "B": wl.batch, "T": wl.tq, "Nq": wl.nq, "Nkv": wl.nkv,
           "D": wl.d, "sparse_mode": wl.sparse_mode, "pre_tokens": wl.pre_tokens, "next_tokens": wl.next_tokens,
           "keep_prob": wl.keep_prob, "sink": wl.has_sink, "seed": wl.seed,
           "seqlens": wl.seqlens_q if wl.batch <= 16 else f"{wl.batch} sequences",
           "kept_pairs": kept_pairs(wl)}
    if l2_note:
        cfg["l2"] = "flushed between timed steps (256 MiB write, outside the per-step events)"
    return cfg


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl, inp, target_s: float, max_s: float):
    """Times the fp64 oracle (forward + gradient) on whole sequences taken in
    order until about target_s of work; returns (TFLOP/s, seconds, sample text,
    threads used)."""
    import oracle
    oracle.build()
    chosen, est = [], 0.0
    rate = 1.0e9 * max(1, os.cpu_count() or 1)       # rough fp64 flop/s for sizing only
    for b in range(wl.batch):
        sub = workloads.custom(wl.name, wl.dtype, [wl.seqlens_q[b]], [wl.seqlens_kv[b]], wl.nq, wl.nkv, wl.d,
                               scale=wl.scale, keep_prob=wl.keep_prob, pre_tokens=wl.pre_tokens,
                               next_tokens=wl.next_tokens, sparse_mode=wl.sparse_mode, has_sink=wl.has_sink)
        cost = kept_pairs(sub) * wl.d * 14.0 / rate
        if chosen and est + cost > target_s:
            break
        chosen.append(b)
        est += cost
        if est >= target_s:
            break
    heads = wl.nq
    # shrink to fewer kv groups if even one sequence is far too large
    while est > max_s and heads > wl.nq // wl.nkv:
        heads //= 2
        est /= 2
    hs = (0, max(heads - heads % (wl.nq // wl.nkv), wl.nq // wl.nkv))
    b0 = chosen[0]
    row_lo = None
    if est > max_s:  # keep a suffix of query rows (exact for dQ of those rows)
        keep_frac = max_s / est
        row_lo = [int(wl.seqlens_q[b] * (1 - keep_frac)) if b in chosen else wl.seqlens_q[b] for b in range(wl.batch)]
    p = oracle.problem_from_workload(wl, drop_mask=inp.mask, sink=inp.sink, heads=hs, row_lo=(
        row_lo if row_lo is not None else [0 if b in chosen else wl.seqlens_q[b] for b in range(wl.batch)]))
    t0 = time.perf_counter()
    oracle.fwd_grad(p, inp.q64, inp.k64, inp.v64, inp.dy64)
    dt = time.perf_counter() - t0
    # mask-adjusted pairs actually covered by the sample
    pairs = 0
    for b in chosen:
        sq, skv = wl.seqlens_q[b], wl.seqlens_kv[b]
        sub = workloads.custom(wl.name, wl.dtype, [sq], [skv], 1, 1, wl.d, keep_prob=wl.keep_prob,
                               pre_tokens=wl.pre_tokens, next_tokens=wl.next_tokens, sparse_mode=wl.sparse_mode)
        rows = kept_rows(sub)
        lo = 0 if row_lo is None else row_lo[b]
        pairs += int(rows[lo:].sum()) * (hs[1] - hs[0])
    units = len(chosen) * max(1, (hs[1] - hs[0]) // (wl.nq // wl.nkv))
    threads = min(os.cpu_count() or 1, units)
    text = (f"sequences {chosen} (lengths {[wl.seqlens_q[b] for b in chosen]}), query heads [{hs[0]}, {hs[1]})"
            + ("" if row_lo is None else ", query-row suffix") + f": {pairs} kept pairs, forward + gradient in fp64")
    return 10.0 * wl.d * pairs / dt / 1e12, dt, text, threads


def kept_rows(wl):
    sq, skv = wl.seqlens_q[0], wl.seqlens_kv[0]
    i = np.arange(sq, dtype=np.int64)
    lo = np.zeros(sq, dtype=np.int64)
    hi = np.full(sq, skv - 1, dtype=np.int64)
    if wl.sparse_mode == 2:
        hi = np.minimum(hi, i)
    elif wl.sparse_mode == 3:
        hi = np.minimum(hi, i + skv - sq)
    elif wl.sparse_mode == 4:
        lo = np.maximum(lo, i - wl.pre_tokens)
        hi = np.minimum(hi, i + wl.next_tokens)
    return np.maximum(hi - lo + 1, 0)


def run_reference(args, wl, rank):
    if rank != 0:
        return
    inp = workloads.make_inputs(wl)
    for _ in range(args.warmup):
        oracle_sample(wl, inp, target_s=ORACLE_TARGET_S, max_s=ORACLE_MAX_S)
    vals, secs, text, threads = [], [], "", 1
    for _ in range(args.steps):
        v, dt, text, threads = oracle_sample(wl, inp, target_s=ORACLE_TARGET_S, max_s=ORACLE_MAX_S)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, l2_note=False),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "threads_used": threads,
                             "kind": "oracle", "sample": text},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the library on the GPU
# ---------------------------------------------------------------------------

def run_ours(args, wl, rank, world, local_rank):
    import torch
    import attention_backward_tnd_b300 as tnd
    from attention_backward_tnd_b300 import build as tbuild

    tbuild.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    inp = workloads.make_inputs(wl, with_fp64=(rank == 0 and world == 1))
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[wl.dtype]

    def to_dev(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    q, k, v, dy = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.dy))
    sink = None if inp.sink is None else torch.from_numpy(inp.sink).to(dev)
    mask = None if inp.mask is None else torch.from_numpy(inp.mask).to(dev)
    cu_q, cu_kv = wl.cu_q, wl.cu_kv
    out, smax, ssum = tnd.fwd(q, k, v, cu_q, cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens,
                              wl.sparse_mode, mask, sink)
    nbytes = tnd.grad_workspace_bytes(q, k, cu_q, cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens,
                                      wl.sparse_mode, mask is not None, sink is not None)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
            torch.empty(wl.nq, dtype=torch.float32, device=dev) if sink is not None else None)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        tnd.grad(q, k, v, dy, out, smax, ssum, cu_q, cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens,
                 wl.next_tokens, wl.sparse_mode, mask, sink, workspace=ws, outputs=outs)

    # the timed steps run without the library's per-kernel events (they would
    # sit between its kernels on the stream); a second, profiled pass below
    # gives the per-kernel device times
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 0) == tnd.TND_OK
    assert tnd.tnd_attn_set_option(tnd.TND_OPT_GRAD_PATH, 1 if args.grad_path == "cuda_core" else 0) == tnd.TND_OK
    for _ in range(max(args.warmup, 0)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    st = tnd.device_status(ws)
    if st != tnd.TND_OK:
        raise SystemExit(f"device status after warm-up: {tnd.tnd_status_string(st)}")
    tnd.tnd_attn_profile_read(reset=True)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        time.sleep(0.05)
        wall0 = time.perf_counter()
        clk.mark(True)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize()
        clk.mark(False)
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    st = tnd.device_status(ws)
    if st != tnd.TND_OK:
        raise SystemExit(f"device status after timed steps: {tnd.tnd_status_string(st)}")
    # per-kernel device times: the same steps again with the library's events
    tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 1)
    tnd.tnd_attn_profile_read(reset=True)
    prof_steps = max(1, min(args.steps, 50))
    for i in range(prof_steps):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    prof = tnd.tnd_attn_profile_read(reset=True)
    tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 0)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step = max_over_ranks(float(statistics.median(step_ms)), dist, dev)
    flop = grad_flop(wl)
    value = job_tflops(world, flop, ms_per_step)
    # the library's kernels in the timed region: per-step launches of the profiled pass x steps
    launches = int(round(sum(n for _, n in prof.values()) / prof_steps)) * args.steps
    kernels = {name: {"ms_per_launch": ms / n, "launches": n} for name, (ms, n) in prof.items() if n}
    main = max(kernels, key=lambda kname: kernels[kname]["ms_per_launch"] * kernels[kname]["launches"])
    main_ms = kernels[main]["ms_per_launch"]
    peaks, peak_src = load_peaks()
    achieved = flop / (main_ms * 1e-3) / 1e12
    if main.startswith("grad_tc"):
        bound, peak, peak_kind = "tensor", float(peaks["bf16_tflops"]), f"bf16 dense, burst ({peak_src})"
    else:
        # CUDA-core path: FP32 FMA issue bound, 128 FP32 lanes per SM x 2 FLOP
        # per FMA x SM count x maximum SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = float(peaks.get("sm_max_mhz", 2032.0))
        bound, peak = "alu", sms * 128 * 2 * mhz * 1e6 / 1e12
        peak_kind = f"fp32 FMA, {sms} SMs x 128 lanes x 2 x {mhz:.0f} MHz (derived)"
    traffic = traffic_record(main, wl.name)

    # the forward (not part of the metric): device time per call, same inputs
    tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 1)
    tnd.tnd_attn_profile_read(reset=True)
    fwd_outs = (torch.empty_like(out), torch.empty_like(smax), torch.empty_like(ssum))
    for _ in range(max(3, min(args.steps, 20))):
        flush.fill_(3)
        tnd.fwd(q, k, v, cu_q, cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens, wl.next_tokens, wl.sparse_mode, mask,
                sink)
    torch.cuda.synchronize()
    fprof = {n: (ms, c) for n, (ms, c) in tnd.tnd_attn_profile_read(reset=True).items() if c and n.startswith("fwd")}
    del fwd_outs
    fwd_name = max(fprof, key=lambda n: fprof[n][1]) if fprof else None
    forward = None
    if fwd_name:
        fms = fprof[fwd_name][0] / fprof[fwd_name][1]
        forward = {"kernel": fwd_name, "ms_per_call": fms,
                   "tflops": 4.0 * wl.d * kept_pairs(wl) / (fms * 1e-3) / 1e12,
                   "flop": "4 * D per kept pair (S = Q K^T and O = P V)"}

    # the same steps with deterministic computing off (dQ contributions added
    # in arrival order): reported beside the default, deterministic figures
    arrival = None
    if main.startswith("grad_tc"):
        assert tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 0) == tnd.TND_OK
        try:
            for _ in range(max(args.warmup, 0)):
                flush.fill_(1)
                step()
            a_ms = []
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                starts[i].record()
                step()
                ends[i].record()
            torch.cuda.synchronize()
            a_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
            tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 1)
            tnd.tnd_attn_profile_read(reset=True)
            for i in range(prof_steps):
                flush.fill_(i & 0xFF)
                step()
            torch.cuda.synchronize()
            aprof = tnd.tnd_attn_profile_read(reset=True)
        finally:
            tnd.tnd_attn_set_option(tnd.TND_OPT_PROFILE, 0)
            tnd.tnd_attn_set_option(tnd.TND_OPT_DETERMINISTIC, 1)
        st = tnd.device_status(ws)
        if st != tnd.TND_OK:
            raise SystemExit(f"device status after arrival-order steps: {tnd.tnd_status_string(st)}")
        a_step = float(statistics.median(a_ms))
        a_main = aprof[main][0] / aprof[main][1]
        arrival = {"ms_per_step": a_step, "value": flop / (a_step * 1e-3) / 1e12, "main_ms": a_main,
                   "main_frac": flop / (a_main * 1e-3) / 1e12 / peak,
                   "note": "deterministic computing off: each (q block, head)'s dQ contributions are added in "
                           "arrival order (not bitwise repeatable); value and roofline above are the default, "
                           "deterministic order"}

    # end to end: pinned host inputs -> device, gradient, device -> pinned host outputs
    host_in = [t.cpu().pin_memory() for t in (q, k, v, dy, out, smax, ssum)]
    dev_in = [q, k, v, dy, out, smax, ssum]
    if sink is not None:
        host_in.append(sink.cpu().pin_memory())
        dev_in.append(sink)
    if mask is not None:
        host_in.append(mask.cpu().pin_memory())
        dev_in.append(mask)
    host_out = [t.cpu().pin_memory() for t in outs if t is not None]
    dev_out = [t for t in outs if t is not None]
    h2d = int(sum(t.numel() * t.element_size() for t in host_in))
    d2h = int(sum(t.numel() * t.element_size() for t in host_out))
    e2e_steps = max(4, min(args.steps, 12))
    # two device buffer sets, pipelined over three streams: step i's inputs go
    # up while step i-1 computes and step i-2's results come down (the copy
    # engines run both directions at once); every step still copies all its
    # inputs in and all its results out
    n_in = 7
    dev_sets = [(dev_in, dev_out), ([torch.empty_like(d) for d in dev_in], [torch.empty_like(d) for d in dev_out])]
    host_out_sets = [host_out, [torch.empty_like(h).pin_memory() for h in host_out]]
    comp = torch.cuda.current_stream()
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step_on(ins, outs_):
        q_, k_, v_, dy_, o_, m_, l_ = ins[:n_in]
        extra = ins[n_in:]
        sink_ = extra[0] if sink is not None else None
        mask_ = extra[-1] if mask is not None else None
        tnd.grad(q_, k_, v_, dy_, o_, m_, l_, cu_q, cu_kv, wl.scale, wl.keep_prob, wl.pre_tokens,
                 wl.next_tokens, wl.sparse_mode, mask_, sink_, workspace=ws,
                 outputs=tuple(outs_) + ((None,) if sink is None else ()))

    def e2e_run(n, start):
        for s_ in (s_up, s_down):
            s_.wait_event(start)
        for i in range(n):
            b_ = i % 2
            ins, outs_ = dev_sets[b_]
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(ev_comp[b_])          # step i-2 has read this input set
                for hsrc, d in zip(host_in, ins):
                    d.copy_(hsrc, non_blocking=True)
                ev_in[b_].record(s_up)
            comp.wait_event(ev_in[b_])
            if i >= 2:
                comp.wait_event(ev_out[b_])               # step i-2's results have been read out
            step_on(ins, outs_)
            ev_comp[b_].record(comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_comp[b_])
                for d, hdst in zip(outs_, host_out_sets[b_]):
                    hdst.copy_(d, non_blocking=True)
                ev_out[b_].record(s_down)
        for b_ in range(min(n, 2)):
            comp.wait_event(ev_out[b_])

    warm = torch.cuda.Event()
    warm.record(comp)
    e2e_run(2, warm)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    e2e_run(e2e_steps, e0)
    e1.record(comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    e2e_value = job_tflops(world, flop, e2e_ms)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded N(0,1) inputs; forward O/max/sum "
            "from this library's forward)",
            "config": dict(workload_config(wl), grad_path=args.grad_path,
                           parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
            "pct_of_bf16_peak": 100.0 * (value / world) / float(peaks["bf16_tflops"]), "peak_source": peak_src,
            "roofline": {"bound": bound, "kernel": main, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": None if traffic is None else traffic["bytes_per_launch"],
                         "peak_kind": peak_kind},
            "kernels": kernels,
            "kernels_note": f"device time per launch from a separate pass of {prof_steps} steps with per-kernel "
                            "events (the timed steps run without them)",
            "forward": forward,
            "arrival_order": arrival,
            "gpu_launches": launches,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "steps": e2e_steps,
                    "schedule": "pinned host buffers; each step's inputs copied in, its dq/dk/dv(/dsink) copied "
                                "out; two device buffer sets, uploads / gradient / downloads on three streams "
                                "so that consecutive steps overlap"},
            "clocks": clk.summary(),
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            v_cpu, dt, text, threads = oracle_sample(wl, inp, target_s=ORACLE_TARGET_S, max_s=ORACLE_MAX_S)
            line["cpu_baseline"] = {"value": v_cpu, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                    "threads_used": threads, "kind": "oracle", "sample": text, "seconds": dt}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.WORKLOAD_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--grad-path", default="auto", choices=["auto", "cuda_core"],
                    help="auto: tensor-core kernel where it applies; cuda_core: the CUDA-core kernels")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workloads.workload(args.workload)
    if args.impl == "reference":
        run_reference(args, wl, rank)
    else:
        run_ours(args, wl, rank, world, local_rank)


if __name__ == "__main__":
    main()
