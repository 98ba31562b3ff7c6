#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path (forward + backward) on GB300.

One step = fa_fwd + fa_bwd (preprocess, main, postprocess) over the causal
B=4, H=16, N=8192, d=128 bf16 workload (the configuration the throughput
target is quoted on), inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

FLOP convention: forward 4*B*H*N^2*d (halved when causal), backward 2.5x the
forward.  Multi-GPU: one process per GPU (torchrun), each runs an independent
replica of the workload (the method has no exchange step); value = all
replicas' FLOPs / the slowest rank's time.

The reference arm (--impl reference) is the fp64 CPU oracle on the host cores,
timed on a bounded sample (whole heads) of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
NOMINAL_PEAK_TFLOPS = 2250.0


def flops_fwd(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_hash(paths, root=None):
    """Hash of the kernel sources' code: comments and whitespace are dropped, so that an edit
    of comments alone keeps a DRAM-traffic record of the compiled kernel valid."""
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(root or ROOT, p), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "fwd": ["exact_attention_49_gb300/csrc/fa_fwd.cu", "exact_attention_49_gb300/csrc/sm103.cuh"],
    "bwd_main": ["exact_attention_49_gb300/csrc/fa_bwd.cu", "exact_attention_49_gb300/csrc/sm103.cuh"],
}


def dram_traffic(kernel, workload_name):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current source of that kernel and scaled to this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    if rec.get("full_workload") != workload_name:
        return None
    return rec.get("bytes_per_launch_full_workload")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_tflops(flop_per_replica_step: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every replica's work over the slowest rank's time."""
    return flop_per_replica_step * world * steps / (max_ms * 1e-3) / 1e12


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_oracle_sample(w, q, k, v, do, budget_s=12.0, max_heads=8):
    """Time the fp64 oracle (fwd + bwd) on whole heads of the workload, one K/V
    group at a time, until about budget_s seconds of CPU work; returns
    (TFLOP/s, seconds, heads, threads)."""
    from oracle import reference as ref
    grp = w.H // w.Hkv
    f_head = flops_fwd(1, 1, w.N, w.d, w.causal) * 3.5
    t0 = time.perf_counter()
    heads = 0
    g = 0
    while heads < max_heads:
        b, kv = divmod(g, w.Hkv)
        if b >= w.B:
            break
        hs = slice(kv * grp, (kv + 1) * grp)
        q64 = q[b:b + 1, hs].double().numpy()
        k64 = k[b:b + 1, kv:kv + 1].double().numpy()
        v64 = v[b:b + 1, kv:kv + 1].double().numpy()
        do64 = do[b:b + 1, hs].double().numpy()
        ref.attn_fwd(q64, k64, v64, w.causal, w.scale)
        ref.attn_bwd(q64, k64, v64, do64, w.causal, w.scale)
        heads += grp
        g += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return f_head * heads / dt / 1e12, dt, heads, ref.num_threads()


def run_reference(args, w):
    ws, rank, _ = dist_setup()
    if args.gpus != ws:
        raise SystemExit("bench.py --gpus %d but WORLD_SIZE=%d" % (args.gpus, ws))
    if rank != 0:
        return 0
    import torch
    from exact_attention_49_gb300.inputs import workload_inputs
    from oracle import reference as ref
    q, k, v, do = workload_inputs(w)
    grp = w.H // w.Hkv
    f_step = flops_fwd(1, grp, w.N, w.d, w.causal) * 3.5
    q64 = q[0:1, 0:grp].double().numpy()
    k64 = k[0:1, 0:1].double().numpy()
    v64 = v[0:1, 0:1].double().numpy()
    do64 = do[0:1, 0:grp].double().numpy()

    def step():
        ref.attn_fwd(q64, k64, v64, w.causal, w.scale)
        ref.attn_bwd(q64, k64, v64, do64, w.causal, w.scale)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    val = f_step * args.steps / dt / 1e12
    sample = ("one K/V group (%d query head%s) of the workload, forward + backward, per step"
              % (grp, "" if grp == 1 else "s"))
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": ref.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, fwd_only=False):
    return {"workload": w.name + (", forward only" if fwd_only else ", forward + backward"), "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N,
            "d": w.d, "causal": w.causal, "softmax_scale": "1/sqrt(d)", "seed": w.seed,
            "inputs": "Q,K,V,dO i.i.d. N(0,1) rounded to bf16",
            "l2": "inputs larger than L2: Q,K,V,dO together %d MiB, each of Q,K,V,O,dO,dQ,dK,dV %d MiB "
                  "(L2 is 129 MB)" % (4 * w.B * w.H * w.N * w.d * 2 >> 20, w.B * w.H * w.N * w.d * 2 >> 20),
            "parallelism": "replicas"}


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from exact_attention_49_gb300 import binding as fa
    from exact_attention_49_gb300.inputs import workload_inputs

    ws, rank, local = dist_setup()
    if args.gpus != ws:
        raise SystemExit("bench.py --gpus %d but WORLD_SIZE=%d: launch one process per GPU with "
                         "python -m torch.distributed.run --nproc-per-node %d bench.py --gpus %d"
                         % (args.gpus, ws, args.gpus, args.gpus))
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fa.lib()
    dev = torch.device("cuda", local)
    q_h, k_h, v_h, do_h = workload_inputs(w)
    B, H, Hkv, N, d, causal, scale = w.B, w.H, w.Hkv, w.N, w.d, int(w.causal), w.scale
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    det = int(args.deterministic)
    fwd_only = args.fwd_only or not w.backward
    if args.poly_exp is not None and fa.fa_set_option("poly_exp", args.poly_exp) != fa.FA_OK:
        raise SystemExit("bad --poly-exp %r" % args.poly_exp)
    if args.bwd_2cta is not None and fa.fa_set_option("bwd_2cta", args.bwd_2cta) != fa.FA_OK:
        raise SystemExit("bad --bwd-2cta %r" % args.bwd_2cta)
    if args.fwd_2cta is not None and fa.fa_set_option("fwd_2cta", args.fwd_2cta) != fa.FA_OK:
        raise SystemExit("bad --fwd-2cta %r" % args.fwd_2cta)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d, det)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def check(name, st):
        if st != fa.FA_OK:
            raise fa.FAError(name, st)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(e=None):
        if e is not None:
            e[0].record(stream)
        check("fa_fwd", fa.fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, stream))
        if e is not None:
            e[1].record(stream)
        if fwd_only:
            if e is not None:
                e[2].record(stream)
                e[3].record(stream)
            return
        check("fa_bwd_preprocess", fa.fa_bwd_preprocess(o, do, lse, B, H, Hkv, N, d, det, wsp, ws_bytes, stream))
        if e is not None:
            e[2].record(stream)
        check("fa_bwd_main", fa.fa_bwd_main(q, k, v, do, lse, dk, dv, B, H, Hkv, N, d, causal, scale, det, wsp,
                                            ws_bytes, stream))
        if e is not None:
            e[3].record(stream)
        check("fa_bwd_postprocess", fa.fa_bwd_postprocess(dq, B, H, Hkv, N, d, det, wsp, ws_bytes, stream))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise fa.FAError("device status after warm-up", st)

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(ev[i])
        stop.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
    clocks = clk.summary()
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise fa.FAError("device status after the timed steps", st)
    total_ms = start.elapsed_time(stop)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    main_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps
    total_ms = max_over_ranks(total_ms, dev)
    ms_step = total_ms / args.steps
    f_fwd = flops_fwd(B, H, N, d, w.causal)
    f_bwd = 0.0 if fwd_only else 2.5 * f_fwd
    value = throughput_tflops(f_fwd + f_bwd, ws, args.steps, total_ms)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region.
    # Every step copies its four inputs from pinned host memory and reads its five results back
    # into pinned host memory.  The copies run on their own streams, on two sets of device and
    # host buffers, so step i's host-to-device copies overlap step i-1's kernels and step i-1's
    # read-back overlaps step i's kernels (the usual copy/compute pipeline of a training or
    # serving loop); the timed region runs from before the first copy to the end of the last
    # read-back.
    ins = (q_h, k_h, v_h) if fwd_only else (q_h, k_h, v_h, do_h)
    h2d = sum(x.numel() * x.element_size() for x in ins)
    out_shapes = [(q_h.shape, q_h.dtype), ((B, H, N), torch.float32)]
    if not fwd_only:
        out_shapes += [(q_h.shape, q_h.dtype), (k_h.shape, k_h.dtype), (v_h.shape, v_h.dtype)]
    d2h = sum(math.prod(sh) * torch.empty((), dtype=dt).element_size() for sh, dt in out_shapes)
    e2e_steps = max(4, min(args.steps, 40))
    e2e_value = None
    if not args.no_e2e:
        h_in = [x.pin_memory() for x in ins]
        sets = []
        for _ in range(2):
            d_in = [torch.empty_like(x, device=dev) for x in ins]
            d_out = [torch.empty(sh, dtype=dt, device=dev) for sh, dt in out_shapes]
            h_out = [torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in out_shapes]
            sets.append((d_in, d_out, h_out))
        s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_compute(d_in, d_out):
            qq, kk, vv = d_in[:3]
            oo, ll = d_out[:2]
            check("fa_fwd", fa.fa_fwd(qq, kk, vv, oo, ll, B, H, Hkv, N, d, causal, scale, stream))
            if fwd_only:
                return
            dd = d_in[3]
            gq, gk, gv = d_out[2:]
            check("fa_bwd_preprocess", fa.fa_bwd_preprocess(oo, dd, ll, B, H, Hkv, N, d, det, wsp, ws_bytes, stream))
            check("fa_bwd_main", fa.fa_bwd_main(qq, kk, vv, dd, ll, gk, gv, B, H, Hkv, N, d, causal, scale, det, wsp,
                                                ws_bytes, stream))
            check("fa_bwd_postprocess", fa.fa_bwd_postprocess(gq, B, H, Hkv, N, d, det, wsp, ws_bytes, stream))

        def e2e_run(n):
            in_free = [None, None]   # compute of the step that last used the set's inputs is done
            out_free = [None, None]  # read-back of the step that last used the set's outputs is done
            begin = torch.cuda.Event()
            begin.record(stream)
            s_h2d.wait_event(begin)
            last = None
            for i in range(n):
                d_in, d_out, h_out = sets[i & 1]
                with torch.cuda.stream(s_h2d):
                    if in_free[i & 1] is not None:
                        s_h2d.wait_event(in_free[i & 1])
                    for dst, src in zip(d_in, h_in):
                        dst.copy_(src, non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(s_h2d)
                stream.wait_event(ready)
                if out_free[i & 1] is not None:
                    stream.wait_event(out_free[i & 1])
                e2e_compute(d_in, d_out)
                done = torch.cuda.Event()
                done.record(stream)
                in_free[i & 1] = done
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(done)
                    for dst, src in zip(h_out, d_out):
                        dst.copy_(src, non_blocking=True)
                    last = torch.cuda.Event()
                    last.record(s_d2h)
                out_free[i & 1] = last
            stream.wait_event(last)

        e2e_run(2)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        st = fa.fa_last_device_status(stream)
        if st != fa.FA_OK:
            raise fa.FAError("device status after the end-to-end steps", st)
        e2e_value = throughput_tflops(f_fwd + f_bwd, ws, e2e_steps, max_over_ranks(e0.elapsed_time(e1), dev))
        # the pipelined results are the step's results: the last read-back equals the device-resident run
        if not torch.equal(sets[(e2e_steps - 1) & 1][2][0], o.cpu()):
            raise SystemExit("end-to-end output differs from the device-resident step")

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = measured_peaks()
    timed_s = total_ms * 1e-3
    peak_key = "bf16_tflops_sustained" if timed_s > 1.0 else "bf16_tflops"
    peak = float(peaks[peak_key])
    dominant = "bwd_main" if (main_ms >= fwd_ms and not fwd_only) else "fwd"
    dom_ms = main_ms if dominant == "bwd_main" else fwd_ms
    dom_flops = f_bwd if dominant == "bwd_main" else f_fwd
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    pair = d == 128 and fa.fa_get_option("bwd_2cta") == 1
    bwd_kernel = ("bwd256_kernel" if d == 256 else "bwd_pair_kernel" if pair
                  else "bwd_main_kernel<%d, %d>" % (d, det))
    fwd_kernel = ("fwd_pair_kernel" if d == 128 and fa.fa_get_option("fwd_2cta") == 1
                  else "fwd_kernel<%d, 0>" % d)
    dom_kernel = {"fwd": fwd_kernel, "bwd_main": bwd_kernel}[dominant]
    roofline = {"bound": "tensor", "kernel": dom_kernel, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": dram_traffic(dominant, w.name) if d == 128 and not det and "pair" not in dom_kernel else None,
                "peak_source": "%s %s (%s)" % (peak_src, peak_key, "MEASURED_PEAKS.json" if peak_src == "measured"
                                               else "profiling recipe fallback")}

    # ---- CPU baseline: the oracle on this host's cores, bounded sample (skipped when the budget is 0)
    cpu = None
    if args.cpu_budget > 0:
        cpu_val, cpu_s, cpu_heads, cores = cpu_oracle_sample(w, q_h, k_h, v_h, do_h, budget_s=args.cpu_budget)
        cpu = {"value": cpu_val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "%d whole heads (forward + backward, fp64) of the workload, %.1f s" % (cpu_heads, cpu_s)}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w, fwd_only),
        "pct_of_peak": {"measured_bf16": value / ws / peak, "nominal_2250": value / ws / NOMINAL_PEAK_TFLOPS},
        "fwd": {"ms": fwd_ms, "tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
                "frac_of_nominal_2250": f_fwd / (fwd_ms * 1e-3) / 1e12 / NOMINAL_PEAK_TFLOPS},
        "bwd": None if fwd_only else {
            "ms": ms_step - fwd_ms, "tflops": f_bwd / ((ms_step - fwd_ms) * 1e-3) / 1e12, "main_ms": main_ms,
            "frac_of_nominal_2250": f_bwd / ((ms_step - fwd_ms) * 1e-3) / 1e12 / NOMINAL_PEAK_TFLOPS},
        "deterministic": bool(det),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": None if e2e_value is None else {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                                               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                                               "copies": "pinned host buffers, own streams, overlapped with the "
                                                         "neighbouring steps' kernels"},
        "gpu_launches": (1 if fwd_only else 4) * args.steps,
        "poly_exp": fa.fa_get_option("poly_exp"),
        "bwd_2cta": fa.fa_get_option("bwd_2cta"),
        "fwd_2cta": fa.fa_get_option("fwd_2cta"),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# Decoding workloads (split-KV forward, fa_fwd_splitkv): B, Hq, Hkv, Nq, Nk, d, causal.
DECODE = {
    "D1": ("D1 decode B8 Hq32 Hkv8 Nq1 Nk16384 d128 causal", 8, 32, 8, 1, 16384, 128),
    "D2": ("D2 decode B8 Hq32 Hkv8 Nq1 Nk65536 d128 causal", 8, 32, 8, 1, 65536, 128),
    "D3": ("D3 decode B32 Hq32 Hkv8 Nq1 Nk8192 d128 causal", 32, 32, 8, 1, 8192, 128),
    "D4": ("D4 decode B8 Hq32 Hkv8 Nq4 Nk16384 d128 causal", 8, 32, 8, 4, 16384, 128),
    "D5": ("D5 decode B8 Hq32 Hkv32 Nq1 Nk16384 d128 causal", 8, 32, 32, 1, 16384, 128),
}


def run_decode(args):
    """Time the split-KV forward on a decoding workload: HBM-bound (K and V are streamed once
    per K/V head), so the line reports the K/V bytes per second against the measured HBM
    copy bandwidth.  L2 is flushed (a 256 MiB write) before every timed step.  The step is
    replayed from a CUDA graph, as a decoding loop runs it; the direct call is timed too."""
    import torch
    from exact_attention_49_gb300 import binding as fa
    from exact_attention_49_gb300.inputs import make_inputs
    name, B, H, Hkv, Nq, Nk, d = DECODE[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q, k, v, _ = make_inputs(B, H, Hkv, Nq, d, seed=7, Nk=Nk)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, 0)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    scale = d ** -0.5

    def split():
        # (the current stream at call time: inside a graph capture that is the capture stream)
        st = fa.fa_fwd_splitkv(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, 1, scale, 0, ws, ws_bytes,
                               torch.cuda.current_stream().cuda_stream)
        if st != fa.FA_OK:
            raise fa.FAError("fa_fwd_splitkv", st)

    def onepass():
        st = fa.fa_fwd_qk(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, 1, scale, stream)
        if st != fa.FA_OK:
            raise fa.FAError("fa_fwd_qk", st)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        with ClockSampler(0) as clk:
            for _ in range(steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts), clk.summary()

    ms_direct, _ = timed(split, args.steps)
    # A decoding loop replays its step as a CUDA graph (the split-KV kernel and the merge, no
    # host launch latency between them); the line's value is that replay.
    for _ in range(args.warmup):
        split()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        split()
    ms, clocks = timed(graph.replay, args.steps)
    ms_one, _ = timed(onepass, max(3, args.steps // 3))
    st = fa.fa_last_device_status()
    if st != fa.FA_OK:
        raise fa.FAError("device status after the timed steps", st)
    kv_bytes = 2 * B * Hkv * Nk * d * 2
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    line = {
        "metric": "decode K/V bytes streamed per second (bf16, 1×GB300)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "Hq": H, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d, "causal": True,
                   "l2": "256 MiB written before every timed step", "splits": "library choice",
                   "kv_bytes_per_step": kv_bytes},
        "roofline": {"bound": "hbm", "kernel": "fwd_kernel (split-KV) + fwd_combine_kernel", "achieved": gbs,
                     "peak": peak, "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                     "peak_source": ("measured hbm_gbs (MEASURED_PEAKS.json)" if src == "measured"
                                     else "fallback 6.8 TB/s")},
        "one_pass_forward_ms": ms_one, "speedup_vs_one_pass": ms_one / ms,
        "launch": "CUDA graph replay of fa_fwd_splitkv", "direct_launch_ms": ms_direct,
        "direct_launch_gbs": kv_bytes / (ms_direct * 1e-3) / 1e9,
        "gpu_launches": 2 * args.steps if ws_bytes > 0 else args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fp8(args, w):
    """Time the FP8 forward (fa_fwd_fp8, d = 128) on a workload, with the quantisation
    (fa_fp8_quantize, incoherent processing on) timed separately.  Throughput is the forward FLOP
    count over the attention kernel's time, against the dense FP8 peak taken as twice the
    measured bf16 peak (the nominal fp8 / bf16 ratio)."""
    import torch
    from exact_attention_49_gb300 import binding as fa
    from exact_attention_49_gb300.inputs import workload_inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q, k, v, _ = (t.to(dev) for t in workload_inputs(w))
    B, H, Hkv, N, d = w.B, w.H, w.Hkv, w.N, w.d
    signs = torch.tensor([1.0 if (i * 2654435761) % 7 < 4 else -1.0 for i in range(d)], dtype=torch.float32,
                         device=dev)
    need = fa.fa_fp8_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def quant():
        st = fa.fa_fp8_quantize(q, k, v, signs, B, H, Hkv, N, d, ws, need, stream)
        if st != fa.FA_OK:
            raise fa.FAError("fa_fp8_quantize", st)

    def attn():
        st = fa.fa_fwd_fp8(ws, need, o, lse, B, H, Hkv, N, d, int(w.causal), w.scale, stream)
        if st != fa.FA_OK:
            raise fa.FAError("fa_fwd_fp8", st)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_q = timed(quant, max(3, args.steps // 4))
    with ClockSampler(0) as clk:
        ms = timed(attn, args.steps)
    clocks = clk.summary()
    st = fa.fa_last_device_status(stream)
    if st != fa.FA_OK:
        raise fa.FAError("device status", st)
    f = flops_fwd(B, H, N, d, w.causal)
    peaks, src = measured_peaks()
    peak = 2.0 * float(peaks["bf16_tflops"])
    tf = f / (ms * 1e-3) / 1e12
    line = {"metric": "FP8 attention forward TFLOP/s (e4m3, 1×GB300)", "value": tf, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": config_of(w, fwd_only=True), "quantize_ms": ms_q,
            "roofline": {"bound": "tensor", "kernel": "fwd_fp8_kernel", "achieved": tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": tf / peak, "traffic": None,
                         "peak_source": "2 x %s bf16_tflops (nominal fp8/bf16 ratio)" % src},
            "frac_of_nominal_4500": tf / 4500.0, "gpu_launches": args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 200 steps of the default workload keep the timed region near 0.7 s, long enough for the
    # clock sampler (every 20 ms) to see it under load
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="C3")
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling on a smaller case)")
    ap.add_argument("--seq", type=int, default=65536, help="N for the long-context workload C5")
    ap.add_argument("--head-dim", type=int, default=128, help="d for the long-context workload C5")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward alone")
    ap.add_argument("--poly-exp", type=int, default=None, help="exp2 split: columns of 32 on the FMA polynomial")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--bwd-2cta", type=int, default=None, choices=[0, 1],
                    help="backward main stage on CTA pairs (1) or one CTA per key tile (0); default: library's")
    ap.add_argument("--fp8", action="store_true", help="time the FP8 forward (d = 128) instead")
    ap.add_argument("--fwd-2cta", type=int, default=None, choices=[0, 1],
                    help="forward on CTA pairs with P in shared memory (1) or one CTA per block (0); default: library's")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in DECODE:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "decoding workloads are timed for the GPU path only"}))
            return 0
        return run_decode(args)
    from exact_attention_49_gb300.inputs import WORKLOADS, long_context
    w = long_context(args.seq, args.head_dim) if args.workload == "C5" else WORKLOADS[args.workload]
    if args.batch:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch, name=w.name.replace("B%d " % w.B, "B%d " % args.batch))
    if args.impl == "reference":
        return run_reference(args, w)
    if args.fp8:
        return run_fp8(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
