"""Benchmark of exact tiled attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole path over one batch of the workload: for every
causal setting the workload runs, fa_fwd then the three fa_bwd stages
(preprocess, main, finalize), all through the C ABI of libfa.so.  Inputs are
resident in device memory; L2 is flushed (a 256 MiB write) between steps,
outside the timed events.  The timed step is one CUDA graph holding those
launches (captured once, replayed every step; the causal settings, which share
only the inputs, are two concurrent branches of it), bracketed by CUDA events
on the launching stream; a separate pass launches the kernels one by one and brackets
every forward and every backward main kernel (the dominant kernel) with
events, which gives the breakdown and the roofline figure.  FLOPs follow the usual
convention: forward 4 B H N^2 d, backward 2.5 x forward, halved for causal,
scaled by the kept-tile fraction for a block mask.

`e2e` is the same metric measured end to end: per step the inputs are copied
from pinned host memory, the path runs, and every output is copied back to
pinned host memory, all inside the timed region (copies overlap neighbouring
steps' kernels on their own streams).

`cpu_baseline` times the fp64 CPU oracle on the host cores on a bounded sample
of the same workload (a subset of heads), scaled to the same unit.

With --impl reference the oracle itself is the timed arm (each step one bounded
sample of the workload on the host cores).

Multi-GPU (torchrun, one process per GPU): every rank runs its own copy of the
workload (independent batches: weak scaling, no collective on the data path);
the reported time is the max over ranks (max_over_ranks) and the value counts
every rank's work (job_value), for the device-timed and the end-to-end numbers.

With --fp8 a step is the FP8 forward with incoherent processing instead: one
fa_fp8_quantize of Q, K, V (randomised Hadamard rotation, power-of-two block
scales, e4m3 codes) and one fa_fwd_fp8 per causal setting; the FLOPs are the
forward's, the roofline kernel is fwd_fp8_kernel against the FP8 tensor peak
(the measured bf16 peak times the nominal FP8/BF16 ratio 4.5/2.25 = 2), and the
CPU baseline and the reference arm run the oracle's FP8 forward.

Options beyond the contract's: --fp8, --fwd-splits S (key-range slices of the forward;
0 lets the library choose), --no-graph (time separately launched kernels),
--dropout P (dropout of the attention weights, off in the workloads; the FLOP
count is unchanged), --no-cpu-baseline, --e2e-steps K.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attention fwd/bwd TFLOP/s at N=2k–23.4k, d=64/128; "
          "% of GB300 BF16 tensor peak")
DEFAULT_WORKLOAD = "bf16_b4h12_n2048"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-graph", action="store_true",
                    help="time separately launched kernels instead of one CUDA graph per step")
    ap.add_argument("--fwd-splits", type=int, default=0,
                    help="key-range slices of the forward (0: the library's choice for this GPU)")
    ap.add_argument("--fp8", action="store_true",
                    help="measure the FP8 forward with incoherent processing (rotation + block "
                         "quantisation + forward) instead of the 16-bit forward + backward")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout probability of the attention weights (0: none, the workloads' "
                         "own setting); the FLOP count is unchanged")
    return ap.parse_args()


def kept_fraction(mask, causal: bool) -> float:
    """Visited (query, key) pairs relative to N^2 under the FLOP convention."""
    if mask is None:
        return 0.5 if causal else 1.0
    import numpy as np
    m = np.asarray(mask, dtype=bool)
    if causal:
        m = np.tril(m)
    return float(m.mean())


def workload_flops(w, mask) -> dict:
    dense = 4.0 * w.B * w.H * w.N * w.N * w.d
    out = {}
    for c in w.causal:
        f = dense * kept_fraction(mask, c)
        out[c] = {"fwd": f, "bwd": 2.5 * f}
    return out


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms in the background."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu):
        self.gpu = gpu
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [s for (t, s) in self.samples if self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not inside:
            inside = [s for (_, s) in self.samples]
        sm, mx, power, reasons = [], [], [], set()
        for s in inside:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def oracle_sample(w, inp, heads: int, dropout: float = 0.0):
    """fp64 oracle forward + backward on the first `heads` heads; returns (flops, s, threads)."""
    import oracle
    B, H = w.B, w.H
    sel = [(b, h) for b in range(B) for h in range(H)][:heads]
    x = {n: inp[n].double().numpy() for n in ("q", "k", "v", "do")}
    flops = workload_flops(w, inp["mask"])
    total = 0.0
    t = time.perf_counter()
    for (b, h) in sel:
        sl = lambda n: x[n][b:b + 1, h:h + 1]
        mh = oracle.head_mask(inp["mask"], b, h, w.N, w.mask_block)
        for c in w.causal:
            oracle.attention_fwd(sl("q"), sl("k"), sl("v"), w.scale, causal=c, mask=mh,
                                 mask_block=w.mask_block, dropout_p=dropout, seed=1)
            oracle.attention_bwd(sl("q"), sl("k"), sl("v"), sl("do"), w.scale, causal=c, mask=mh,
                                 mask_block=w.mask_block, dropout_p=dropout, seed=1)
            total += (flops[c]["fwd"] + flops[c]["bwd"]) / (B * H)
    return total, time.perf_counter() - t, oracle.num_threads()


def heads_for_seconds(w, target_s: float) -> int:
    """Heads that keep the oracle near target_s (it runs at roughly 1 GFLOP/s per core
    on this convention's FLOPs)."""
    cores = os.cpu_count() or 8
    f = workload_flops(w, None)
    per_head = sum(v["fwd"] + v["bwd"] for v in f.values()) / (w.B * w.H)
    n = int(target_s * cores * 1.0e9 / max(per_head, 1.0))
    return max(1, min(n, w.B * w.H))


def config_of(w, fwd_splits=None, dropout=0.0):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
            "causal": list(w.causal), "block_mask_p": w.mask_p, "fwd_splits": fwd_splits,
            "dropout_p": dropout,
            "passes": "fwd+bwd per causal setting",
            "l2": "flushed between steps (256 MiB write outside the timed events)"}


def run_reference(args, w, rank):
    import synth
    if rank != 0:
        return
    inp = synth.workload_inputs(w)
    # the whole reference run stays within a few minutes whatever K is
    heads = heads_for_seconds(w, min(1.5, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, inp, max(1, heads // 4), args.dropout)
    tot_f, tot_s, cores = 0.0, 0.0, 1
    for _ in range(args.steps):
        f, s, cores = oracle_sample(w, inp, heads, args.dropout)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e12
    sample = (f"fp64 oracle, forward + backward of {heads} of {w.B * w.H} heads per step "
              f"({w.name}, causal settings {list(w.causal)})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, dropout=args.dropout),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


KERNEL_SOURCES = {"bwd_main": ("bwd_tc.cu", "ptx.cuh", "internal.h"),
                  "fwd_fp8": ("fwd_fp8.cu", "fp8.h", "ptx.cuh", "internal.h")}


def kernel_source_digest(kernel: str = "bwd_main") -> str:
    """Digest of the sources a kernel is built from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_io_aware_26_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) recorded in
    profiles/traffic.json for this workload and this exact kernel source; None otherwise."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[workload][kernel]
        if t.get("source_digest") != kernel_source_digest(kernel):
            return None
        return t["bytes_per_launch"]
    except Exception:
        return None


def fwd(fa, r, q, k, v, o, lse, stream):
    """The forward of one run: fa_fwd, or fa_fwd_split when the run uses slices."""
    if r["splits"] > 1:
        fa.fwd_split_raw(r["p"], q, k, v, o, lse, r["splits"], r["fws"], stream)
    else:
        fa.fwd_raw(r["p"], q, k, v, o, lse, stream)


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest x over all ranks of the process group (x itself with one rank): a
    multi-rank step takes as long as its slowest rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank (weak scaling, one
    replica of the workload per GPU) in at most `seconds` (the max over ranks)."""
    return units_per_rank * world / seconds


FP8_METRIC = ("attention FP8 forward TFLOP/s (rotation + block quantisation + forward), "
              "% of GB300 FP8 tensor peak")


def read_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def oracle_fp8_sample(w, inp, heads: int, signs):
    """The oracle's FP8 path (quantise + forward) on the first `heads` heads; returns
    (forward flops, seconds, threads)."""
    import oracle
    sel = [(b, h) for b in range(w.B) for h in range(w.H)][:heads]
    x = {n: inp[n].double().numpy() for n in ("q", "k", "v")}
    flops = workload_flops(w, inp["mask"])
    total = 0.0
    t = time.perf_counter()
    for (b, h) in sel:
        sl = lambda n: x[n][b:b + 1, h:h + 1]
        tq = oracle.fp8_quantize(sl("q"), sl("k"), sl("v"), signs)
        mh = oracle.head_mask(inp["mask"], b, h, w.N, w.mask_block)
        for c in w.causal:
            oracle.fp8_attention_fwd(tq, w.scale, causal=c, mask=mh, mask_block=w.mask_block)
            total += flops[c]["fwd"] / (w.B * w.H)
    return total, time.perf_counter() - t, oracle.num_threads()


def fp8_heads_for_seconds(w, target_s: float) -> int:
    cores = os.cpu_count() or 8
    per_head = sum(v["fwd"] for v in workload_flops(w, None).values()) / (w.B * w.H)
    return max(1, min(int(target_s * cores * 2.0e9 / max(per_head, 1.0)), w.B * w.H))


def fp8_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
            "causal": list(w.causal), "block_mask_p": w.mask_p,
            "passes": "fa_fp8_quantize once, then fa_fwd_fp8 per causal setting",
            "rotation": "randomised Sylvester-Hadamard, signs PCG64(1)",
            "quantisation": "e4m3, one power-of-two scale per 128-row block",
            "l2": "flushed between steps (256 MiB write outside the timed events)"}


def run_fp8(args, w, rank, world, local):
    """The --fp8 measurement (see the module docstring)."""
    import torch
    import synth
    signs_cpu = synth.rotation_signs(w.d, 1)
    inp = synth.make_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, qkv_scale=w.qkv_scale,
                            ar1_rho=w.ar1_rho, mask_p=w.mask_p, mask_block=w.mask_block,
                            backward=False)
    if args.impl == "reference":
        if rank != 0:
            return
        heads = max(1, fp8_heads_for_seconds(w, min(1.5, 120.0 / max(1, args.steps + args.warmup))))
        sg = signs_cpu.double().numpy()
        for _ in range(args.warmup):
            oracle_fp8_sample(w, inp, 1, sg)
        tot_f = tot_s = 0.0
        cores = 1
        for _ in range(args.steps):
            f, s_, cores = oracle_fp8_sample(w, inp, heads, sg)
            tot_f += f
            tot_s += s_
        value = tot_f / tot_s / 1e12
        print(json.dumps({
            "impl": "reference", "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": fp8_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"fp64 oracle FP8 quantise + forward of {heads} of "
                                       f"{w.B * w.H} heads per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    import exact_io_aware_26_gb300 as fa
    fa.load()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    signs = signs_cpu.to(dev)
    mask = None if inp["mask"] is None else torch.as_tensor(inp["mask"]).to(dev)
    flops = workload_flops(w, inp["mask"])
    step_flops = sum(f["fwd"] for f in flops.values())
    stream = torch.cuda.current_stream()
    t8 = fa.fp8_quantize(q, k, v, signs, stream)
    outs = {c: (torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev))
            for c in w.causal}

    def quant(s):
        fa.fp8_quantize(q, k, v, signs, s, out=t8)

    def fwd8(c, s):
        fa.attention_fwd_fp8_codes(t8, w.scale, causal=c, block_mask=mask, mask_block=w.mask_block,
                                   dtype=q.dtype, out=outs[c][0], lse=outs[c][1], stream=s)

    def step(s, evq=None, evf=None):
        if evq is not None:
            evq[0].record(s)
        quant(s)
        if evq is not None:
            evq[1].record(s)
        for i, c in enumerate(w.causal):
            if evf is not None:
                evf[i][0].record(s)
            fwd8(c, s)
            if evf is not None:
                evf[i][1].record(s)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    W = max(args.warmup, 3)
    for _ in range(W):
        step(stream)
    torch.cuda.synchronize()
    if fa.get_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")
    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)
    ev_step = [(E(), E()) for _ in range(K)]
    ev_q = [(E(), E()) for _ in range(K)]
    ev_f = [[(E(), E()) for _ in w.causal] for _ in range(K)]
    uuid = getattr(torch.cuda.get_device_properties(local), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(0)
    for i in range(K):  # per-kernel pass
        flush.zero_()
        step(stream, ev_q[i], ev_f[i])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    for i in range(K):  # timed pass: whole steps
        flush.zero_()
        ev_step[i][0].record(stream)
        step(stream)
        ev_step[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark(1)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    if fa.get_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after the timed region")
    total_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev_step) / 1000.0, dist, dev)
    q_s = sum(a.elapsed_time(b) for a, b in ev_q) / 1000.0
    f_s = sum(a.elapsed_time(b) for row in ev_f for a, b in row) / 1000.0
    value = job_value(step_flops * K, world, total_s) / 1e12
    bf16_peak, peak_src = read_peaks()
    peak = 2.0 * bf16_peak
    hbm, hbm_src = read_hbm_peak()
    fwd_tflops = step_flops * K / f_s / 1e12
    elems = w.B * w.H * w.N * w.d
    T = (w.N + 127) // 128
    quant_bytes = 3 * elems * 2 + 3 * elems * 1 + 3 * w.B * w.H * T * 4  # read 16-bit, write e4m3 + scales
    quant_gbs = quant_bytes * K / q_s / 1e9

    # end to end: pinned host Q, K, V in, O and LSE out, every step
    host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
    host_out = {c: (torch.empty(q.shape, dtype=q.dtype).pin_memory(),
                    torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()) for c in w.causal}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(o.numel() * o.element_size() + l.numel() * l.element_size()
              for o, l in host_out.values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(n):
        for _ in range(n):
            with torch.cuda.stream(s_in):
                for nm, t in (("q", q), ("k", k), ("v", v)):
                    t.copy_(host_in[nm], non_blocking=True)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)  # the previous step's outputs have been copied out
            step(stream)
            s_out.wait_stream(stream)
            s_in.wait_stream(stream)  # inputs are overwritten only after this step read them
            with torch.cuda.stream(s_out):
                for c in w.causal:
                    host_out[c][0].copy_(outs[c][0], non_blocking=True)
                    host_out[c][1].copy_(outs[c][1], non_blocking=True)

    e2e_steps(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_steps(args.e2e_steps)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e = {"value": job_value(step_flops * args.e2e_steps, world, e2e_s) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "timing": "host clock around all steps, synchronised on both sides",
           "overlap": "input copies on one stream, output copies on another"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        heads = fp8_heads_for_seconds(w, 15.0)
        f, s_, cores = oracle_fp8_sample(w, inp, heads, signs_cpu.double().numpy())
        cpu = {"value": f / s_ / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"fp64 oracle FP8 quantise + forward of {heads} of {w.B * w.H} heads, "
                         f"{s_:.1f} s"}
    if rank == 0:
        launches = K * len(w.causal)
        print(json.dumps({
            "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": 1000.0 * total_s / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3",
            "dtype_detail": f"e4m3 operands, fp32 accumulation; {w.dtype} in and out",
            "data": "synthetic", "config": fp8_config(w),
            "breakdown": {"fwd_fp8_tflops": fwd_tflops, "fwd_fp8_frac_of_fp8_peak": fwd_tflops / peak,
                          "step_frac_of_fp8_peak": value / world / peak,
                          "quantize_us": 1e6 * q_s / K, "quantize_gbs": quant_gbs,
                          "quantize_frac_of_hbm": quant_gbs / hbm,
                          "hbm_peak_gbs": hbm, "hbm_peak_source": hbm_src},
            "roofline": {"kernel": "fwd_fp8_kernel", "bound": "tensor", "achieved": fwd_tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": fwd_tflops / peak,
                         "peak_source": ("measured bf16 burst x 2 (nominal FP8/BF16 ratio), "
                                         "MEASURED_PEAKS.json" if peak_src == "measured"
                                         else "fallback bf16 burst x 2"),
                         "traffic": measured_traffic(w.name, "fwd_fp8"),
                         "algorithmic_flops_per_launch": step_flops * K / launches},
            "clocks": clk, "e2e": e2e,
            "gpu_launches": K * (1 + len(w.causal)),
            "cpu_baseline": cpu}), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(fa, inp, runs, flops, steps, dev, stream, dist=None, world=1):
    """Same metric with host buffers.  Every step copies its inputs from pinned host
    memory, runs the path, and copies every output back to pinned host memory.  The
    copies run on their own streams with double-buffered device tensors, so step i's
    input copy and step i-1's output copy overlap step i's kernels; as in the timed
    step, each causal setting runs on a stream of its own, and its outputs are copied
    back on a copy stream of its own as soon as its kernels are done."""
    import torch
    names_in = ("q", "k", "v", "do")
    names_out = ("o", "lse", "dq", "dk", "dv")
    host_in = {n: inp[n].pin_memory() for n in names_in}
    dev_in = [{n: torch.empty_like(inp[n], device=dev) for n in names_in} for _ in range(2)]
    dev_out = [[{n: torch.empty_like(r[n]) for n in names_out} for r in runs] for _ in range(2)]
    host_out = [{n: torch.empty(r[n].shape, dtype=r[n].dtype).pin_memory() for n in names_out}
                for r in runs]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for ho in host_out for t in ho.values())
    s_h2d = torch.cuda.Stream(dev)
    s_comp = [stream] + [torch.cuda.Stream(dev) for _ in runs[1:]]
    s_d2h = [torch.cuda.Stream(dev) for _ in runs]
    E = lambda: torch.cuda.Event(enable_timing=False)

    def run(n):
        ev_h2d = [E() for _ in range(n)]
        ev_comp = [[E() for _ in runs] for _ in range(n)]
        ev_d2h = [[E() for _ in runs] for _ in range(n)]
        for i in range(n):
            bsel = i % 2
            if i >= 2:
                for ev in ev_comp[i - 2]:
                    s_h2d.wait_event(ev)  # inputs of set bsel no longer read
            with torch.cuda.stream(s_h2d):
                for nm in names_in:
                    dev_in[bsel][nm].copy_(host_in[nm], non_blocking=True)
            ev_h2d[i].record(s_h2d)
            x = dev_in[bsel]
            for j, (r, o) in enumerate(zip(runs, dev_out[bsel])):
                cs = s_comp[j]
                cs.wait_event(ev_h2d[i])
                if i >= 2:
                    cs.wait_event(ev_d2h[i - 2][j])  # outputs of set bsel copied out
                fwd(fa, r, x["q"], x["k"], x["v"], o["o"], o["lse"], cs)
                fa.bwd_preprocess(r["p"], o["o"], x["do"], r["ws"], cs)
                fa.bwd_main(r["p"], x["q"], x["k"], x["v"], x["do"], o["lse"], o["dk"], o["dv"],
                            r["ws"], cs)
                fa.bwd_finalize(r["p"], o["dq"], o["dk"], o["dv"], r["ws"], cs)
                ev_comp[i][j].record(cs)
                s_d2h[j].wait_event(ev_comp[i][j])
                with torch.cuda.stream(s_d2h[j]):
                    for nm in names_out:
                        host_out[j][nm].copy_(o[nm], non_blocking=True)
                ev_d2h[i][j].record(s_d2h[j])

    run(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    run(steps)
    issued = time.perf_counter() - t0  # the host's time to enqueue the steps
    torch.cuda.synchronize()
    s = time.perf_counter() - t0
    if dist:
        dist.barrier()
    s = max_over_ranks(s, dist, dev)
    step_flops = sum(f["fwd"] + f["bwd"] for f in flops.values())
    return {"value": job_value(step_flops * steps, world, s) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "host clock around all steps, synchronised on both sides",
            "host_issue_ms_per_step": 1000.0 * issued / steps,
            "overlap": "copies on their own streams, double-buffered device tensors; one "
                       "compute and one copy-back stream per causal setting"}


def main():
    args = parse()
    import torch
    import synth

    w = synth.WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.fp8:
        run_fp8(args, w, rank, world, local)
        return
    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import exact_io_aware_26_gb300 as fa
    lib = fa.load()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    inp = synth.workload_inputs(w)
    dev = torch.device("cuda", local)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    mask = None if inp["mask"] is None else torch.as_tensor(inp["mask"]).to(dev)
    flops = workload_flops(w, inp["mask"])
    step_flops = sum(f["fwd"] + f["bwd"] for f in flops.values())

    runs = []
    for c in w.causal:
        p, keep = fa.make_params(q, w.scale, c, mask, w.mask_block, args.dropout, seed=1)
        ws = torch.empty(int(lib.fa_bwd_workspace_size(ctypes.byref(p))), dtype=torch.uint8,
                         device=dev)
        splits = args.fwd_splits if args.fwd_splits > 0 else fa.num_splits(p)
        fws = None
        if splits > 1:
            fws = torch.empty(fa.split_workspace_bytes(p, splits), dtype=torch.uint8, device=dev)
        runs.append(dict(causal=c, p=p, keep=keep, splits=splits, fws=fws, o=torch.empty_like(q),
                         lse=torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
                         dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q),
                         ws=ws))
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def run_one(i, r, s, ev_main=None, ev_fwd=None):
        if ev_fwd is not None:
            ev_fwd[i][0].record(s)
        fwd(fa, r, q, k, v, r["o"], r["lse"], s)
        if ev_fwd is not None:
            ev_fwd[i][1].record(s)
        fa.bwd_preprocess(r["p"], r["o"], do, r["ws"], s)
        if ev_main is not None:
            ev_main[i][0].record(s)
        fa.bwd_main(r["p"], q, k, v, do, r["lse"], r["dk"], r["dv"], r["ws"], s)
        if ev_main is not None:
            ev_main[i][1].record(s)
        fa.bwd_finalize(r["p"], r["dq"], r["dk"], r["dv"], r["ws"], s)

    def step(s, ev_main=None, ev_fwd=None):
        for i, r in enumerate(runs):
            run_one(i, r, s, ev_main, ev_fwd)

    def step_branches(s):
        # the causal settings are independent (same inputs, separate outputs and
        # workspaces): one branch each, forked from and joined to `s`
        if len(runs) == 1:
            run_one(0, runs[0], s)
            return
        fork = torch.cuda.Event()
        fork.record(s)
        side_streams = [torch.cuda.Stream(dev) for _ in runs[1:]]
        for b in side_streams:
            b.wait_event(fork)
        run_one(0, runs[0], s)
        for i, (r, b) in enumerate(zip(runs[1:], side_streams), start=1):
            run_one(i, r, b)
        for b in side_streams:
            join = torch.cuda.Event()
            join.record(b)
            s.wait_event(join)

    W = max(args.warmup, 3)
    for _ in range(W):
        step(stream)
    torch.cuda.synchronize()
    if fa.get_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")

    # The step as one CUDA graph (its kernels launched back to back, without
    # the host in between); the per-kernel breakdown comes from a pass of
    # separately launched, separately timed kernels.
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.graph(graph, stream=side):
                step_branches(torch.cuda.current_stream())
            stream.wait_stream(side)
            graph.replay()
            torch.cuda.synchronize()
            if fa.get_status() != fa.FA_OK:
                raise RuntimeError("device status not OK after the graph's first replay")
        except RuntimeError as e:
            print(f"# CUDA graph capture failed ({e}); timing launched steps", file=sys.stderr)
            graph = None

    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)
    ev_step = [(E(), E()) for _ in range(K)]
    ev_kstep = [(E(), E()) for _ in range(K)]
    ev_main = [[(E(), E()) for _ in runs] for _ in range(K)]
    ev_fwd = [[(E(), E()) for _ in runs] for _ in range(K)]
    uuid = getattr(torch.cuda.get_device_properties(local), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark(0)
    # per-kernel pass
    for i in range(K):
        flush.zero_()
        ev_kstep[i][0].record(stream)
        step(stream, ev_main[i], ev_fwd[i])
        ev_kstep[i][1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    # timed pass: the whole step
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev_step[i][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(stream)
        ev_step[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks.mark(1)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    status = fa.get_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status {status} after the timed region")

    total_s = sum(a.elapsed_time(b) for a, b in ev_step) / 1000.0
    launched_s = sum(a.elapsed_time(b) for a, b in ev_kstep) / 1000.0
    main_s = sum(a.elapsed_time(b) for row in ev_main for a, b in row) / 1000.0
    fwd_s = sum(a.elapsed_time(b) for row in ev_fwd for a, b in row) / 1000.0
    total_s = max_over_ranks(total_s, dist, dev)

    peak, peak_src = read_peaks()
    launches = K * len(runs)
    bwd_flops = sum(flops[r["causal"]]["bwd"] for r in runs) * K
    fwd_flops = sum(flops[r["causal"]]["fwd"] for r in runs) * K
    achieved = bwd_flops / main_s / 1e12
    fwd_tflops = fwd_flops / fwd_s / 1e12
    value = job_value(step_flops * K, world, total_s) / 1e12

    e2e = run_e2e(fa, inp, runs, flops, args.e2e_steps, dev, stream, dist, world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        heads = heads_for_seconds(w, 15.0)
        f, s, cores = oracle_sample(w, inp, heads, args.dropout)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"fp64 oracle forward + backward of {heads} of {w.B * w.H} heads "
                         f"(causal settings {list(w.causal)}), {s:.1f} s"}

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": 1000.0 * total_s / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": dict(config_of(w, [r["splits"] for r in runs], args.dropout),
                           launch=("one CUDA graph per step, the causal settings as concurrent "
                                   "branches" if len(runs) > 1 else "one CUDA graph per step")
                           if graph is not None else "kernels launched one by one"),
            "breakdown": {
                "fwd_tflops": fwd_tflops, "bwd_main_tflops": achieved,
                "fwd_frac_of_bf16_peak": fwd_tflops / peak,
                "bwd_main_frac_of_bf16_peak": achieved / peak,
                "step_frac_of_bf16_peak": value / world / peak,
                "wall_s_timed_region": wall,
                "ms_per_step_launched_one_by_one": 1000.0 * launched_s / K},
            "roofline": {"kernel": "bwd_tc_kernel (backward main)", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_source": ("measured bf16 burst, MEASURED_PEAKS.json"
                                         if peak_src == "measured" else "fallback bf16 burst"),
                         "traffic": measured_traffic(w.name, "bwd_main"),
                         "algorithmic_flops_per_launch": bwd_flops / launches},
            "clocks": clk, "e2e": e2e,
            "gpu_launches": K * sum(4 + (r["splits"] > 1) for r in runs),
            "cpu_baseline": cpu}), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
