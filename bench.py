#!/usr/bin/env python
"""Benchmark of the leak-free causal MXFP8 attention forward hot path.

One step = the whole path on one batch of synthetic bf16 inputs already resident in HBM: the
one-launch MXFP8 quantisation of Q and K (rowwise) and V (columnwise + token-normalised), and the
attention forward (O bf16 + LSE).  Default workload: B=1, Hq=16, Hkv=4, S=32768, D=128,
BSHD (the S=32K forward the pages quote).  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torchrun as independent replicas (the forward has no exchange step).
`--impl reference` times the CPU oracle on a bounded sample of the same workload.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal MXFP8 attn fwd TFLOP/s and % of MXFP8 tensor peak at S=32K, 1×GB300"
# The pages' own-block forward at B=1, 16/4 heads, S=32K: 2.797 ms (B200, cuDNN + Triton, including
# quantisation and launch) -> 2*1*16*32768^2*128 / 2.797 ms.
PAGES_OWN_BLOCK_TFLOPS = 2.0 * 16 * 32768 ** 2 * 128 / 2.797e-3 / 1e12
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 vs 2.25 PFLOP/s)


def max_over_ranks(x, world, device):
    """The maximum of a per-rank float over all ranks (the slowest replica sets the job's time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, ms):
    """Throughput of the whole job: every rank's FLOPs over the (max-over-ranks) step time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="gqa_s32k_h16_kv4")
    ap.add_argument("--p-terms", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
# CPU oracle sample (the reference arm and the cpu_baseline leg)

def oracle_sample_step(w, q, k, v, hq, rows):
    """Oracle as it stands on a bounded sample: query head hq, the given query rows, quantising
    exactly the operands those rows read.  Returns algorithmic FLOPs of the sample."""
    import numpy as np
    from oracle import attention as A
    from oracle import mx
    from block_scaled_causal_gb300 import inputs as I

    g = w.Hq // w.Hkv
    hk = hq // g
    kmax = int(max(rows)) + 1
    kpad = ((kmax + 31) // 32) * 32
    f64 = lambda t: I.to_bshd(t, w.layout).float().numpy().astype(np.float64)
    qb = f64(q[:, :, hq:hq + 1])       # head axis is 2 in both layouts
    kb = f64(k[:, :, hk:hk + 1])
    vb = f64(v[:, :, hk:hk + 1])
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb[:, rows]))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb[:, :kmax]))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb[:, :kpad]))[:, :kmax]
    vt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb[:, :kmax]))
    qfull = np.zeros((w.B, kmax, 1, w.D))
    qfull[:, rows] = qh
    A.causal_attention(qfull, kh, vc, vt, w.scale, rows=rows, chunk=64)
    return float(sum(4.0 * w.D * (int(r) + 1) for r in rows)) * w.B


def sample_rows(S, n, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(S, size=n, replace=False))


def run_oracle_steps(w, q, k, v, steps, warmup, rows_per_step):
    flops = 0.0
    t_total = 0.0
    times = []
    for it in range(warmup + steps):
        rows = sample_rows(w.S, rows_per_step, it)
        hq = it % w.Hq
        t0 = time.perf_counter()
        f = oracle_sample_step(w, q, k, v, hq, rows)
        dt = time.perf_counter() - t0
        if it >= warmup:
            flops += f
            t_total += dt
            times.append(dt)
    return flops / t_total / 1e12, t_total, times


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


# ------------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(gpu_id)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def recorded_traffic():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu summary, valid only
    while the kernel source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_gqa_s32k_h16_kv4.md")
    src = os.path.join(ROOT, "block_scaled_causal_gb300", "csrc", "attn_fwd.cu")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"attn_fwd_cu_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m.group(1)) if cur == h.group(1) else None


def main():
    args = parse()
    import torch

    from block_scaled_causal_gb300 import inputs as I

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = I.WORKLOADS[args.workload]
    flops = w.flops

    if args.impl == "reference":
        if rank != 0:
            return
        q, k, v = I.make_qkv(w)
        value, t_total, times = run_oracle_steps(w, q, k, v, args.steps, args.warmup, rows_per_step=8)
        sample = ("per step: 8 query rows drawn uniformly from S=%d for one query head (cycling), with the "
                  "rowwise/columnwise/token-normalised quantisation of exactly the Q rows and K/V tokens "
                  "they read; FLOPs = 4*D*(i+1) per row" % w.S)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
                                                "D": w.D, "layout": "BSHD" if w.layout == 0 else "SBHD"},
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    from block_scaled_causal_gb300 import _binding as ops

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    q_cpu, k_cpu, v_cpu = I.make_qkv(w)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    B, S, Hq, Hkv, D = w.B, w.S, w.Hq, w.Hkv, w.D
    u8 = dict(dtype=torch.uint8, device=dev)
    qq = torch.empty(q.shape, **u8)
    qs = torch.empty((B, Hq, S, D // 32), **u8)
    kq = torch.empty(k.shape, **u8)
    ks = torch.empty((B, Hkv, S, D // 32), **u8)
    vt = torch.empty((B, Hkv, D, S), **u8)
    vsc = torch.empty((B, Hkv, S // 32, D), **u8)
    vtn = torch.empty(v.shape, **u8)
    vtn_sc = torch.empty((B, Hkv, S), **u8)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    o8 = torch.empty(q.shape, **u8)
    o8_sc = torch.empty((B, Hq, S, D // 32), **u8)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)   # 256 MB > L2
    stream = torch.cuda.current_stream(dev)

    def step(p_terms, ev_mid, out8=False):
        ops.mxfp8_quantize_qkv(q, k, v, w.layout, out=(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc), stream=stream)
        ev_mid.record(stream)
        if out8:   # MXFP8 O (E4M3 + one UE8M0 scale per 32 d) instead of BF16 O
            ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, w.layout, w.scale, p_terms=p_terms,
                                      lse=lse, stream=stream, o8_out=True, bf16_out=False, o8=o8, o_sc=o8_sc)
        else:
            ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, w.layout, w.scale, p_terms=p_terms,
                                      o=o, lse=lse, stream=stream)

    def timed(p_terms, steps, warmup, out8=False):
        for _ in range(warmup):
            step(p_terms, torch.cuda.Event(enable_timing=True), out8)
        evs = []
        for _ in range(steps):
            flush.zero_()                                   # L2 flushed between steps, outside the events
            e0 = torch.cuda.Event(enable_timing=True)
            ev_mid = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(p_terms, ev_mid, out8)
            e1.record(stream)
            evs.append((e0, ev_mid, e1))
        return evs

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    gpu_id = local
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    t_wall0 = time.perf_counter()
    evs = timed(args.p_terms, args.steps, args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(c) for a, _, c in evs]
    attn_ms = [b.elapsed_time(c) for _, b, c in evs]
    quant_ms = [a.elapsed_time(b) for a, b, _ in evs]
    ms_per_step = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    value = whole_job_tflops(flops, world, ms_per_step)
    attn_avg = sum(attn_ms) / len(attn_ms)

    # the same step with two E4M3 terms for P
    evs2 = timed(2, max(3, args.steps // 2), 2)
    torch.cuda.synchronize()
    ms2 = max_over_ranks(sum(a.elapsed_time(c) for a, _, c in evs2) / len(evs2), world, dev)
    attn2 = sum(b.elapsed_time(c) for _, b, c in evs2) / len(evs2)
    # backward on decoded operands (BF16 MMAs), inputs resident: the forward's O and LSE and a dO
    g_do = torch.Generator(device="cpu").manual_seed(3)
    d_o = torch.randn(q.shape, generator=g_do, dtype=torch.float32).to(torch.bfloat16).to(dev)
    dq_, dk_, dv_ = (torch.empty(t.shape, dtype=torch.bfloat16, device=dev) for t in (q, k, k))
    step(args.p_terms, torch.cuda.Event(enable_timing=True))     # O, LSE of these inputs
    for _ in range(2):
        ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, d_o, w.layout, w.scale, dq=dq_, dk=dk_, dv=dv_,
                          stream=stream)
    bwd_ms = []
    for _ in range(max(3, args.steps // 4)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, d_o, w.layout, w.scale, dq=dq_, dk=dk_, dv=dv_,
                          stream=stream)
        e1.record(stream)
        bwd_ms.append((e0, e1))
    torch.cuda.synchronize()
    bwd_avg = max_over_ranks(sum(a.elapsed_time(b) for a, b in bwd_ms) / len(bwd_ms), world, dev)
    # the same step writing MXFP8 O instead of BF16 O
    evs8 = timed(args.p_terms, max(3, args.steps // 2), 2, out8=True)
    torch.cuda.synchronize()
    ms8 = max_over_ranks(sum(a.elapsed_time(c) for a, _, c in evs8) / len(evs8), world, dev)
    attn8 = sum(b.elapsed_time(c) for _, b, c in evs8) / len(evs8)

    # end to end through the public call with host buffers (pinned), copies inside the timed region.
    # Pipelined: step i's host->device copy runs on one copy stream while step i-1 computes, and its
    # device->host copy on another while step i+1 computes (two device buffer sets).  The events span
    # the first timed copy to the last, fill and drain included.  The serial form (copy in, compute,
    # copy out, one stream) is reported beside it.
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.pin_memory() for t in (q_cpu, k_cpu, v_cpu))
        oh = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        lh = [torch.empty((B, Hq, S), dtype=torch.float32).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        d2h = oh[0].numel() * 2 + lh[0].numel() * 4
        dq_in = [(q, k, v), tuple(torch.empty_like(t) for t in (q, k, v))]
        dq_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
        s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        torch.cuda.synchronize()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def pipelined(n, ev_start=None, ev_end=None):
            for i in range(n):
                bi = i % 2
                with torch.cuda.stream(s_in):
                    if i == 0 and ev_start is not None:
                        ev_start.record(s_in)
                    if i >= 2:
                        s_in.wait_event(ev_comp[bi])          # step i-2 has read these inputs
                    for dst, src in zip(dq_in[bi], (qh, kh, vh)):
                        dst.copy_(src, non_blocking=True)
                    ev_in[bi].record(s_in)
                s_comp.wait_event(ev_in[bi])
                if i >= 2:
                    s_comp.wait_event(ev_out[bi])             # step i-2's outputs are on the host
                with torch.cuda.stream(s_comp):
                    ops.forward(*dq_in[bi], w.layout, w.scale, p_terms=args.p_terms, o=dq_out[bi][0],
                                lse=dq_out[bi][1], stream=s_comp)
                ev_comp[bi].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[bi])
                    oh[bi].copy_(dq_out[bi][0], non_blocking=True)
                    lh[bi].copy_(dq_out[bi][1], non_blocking=True)
                    ev_out[bi].record(s_out)
                    if i == n - 1 and ev_end is not None:
                        ev_end.record(s_out)

        pipelined(args.warmup)
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipelined(args.steps, t_start, t_end)
        torch.cuda.synchronize()
        e_pipe = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world, dev)
        # serial form
        e_ms = []
        for it in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            c = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            oo, ll = ops.forward(q, k, v, w.layout, w.scale, p_terms=args.p_terms, o=o, lse=lse, stream=stream)
            oh[0].copy_(oo, non_blocking=True)
            lh[0].copy_(ll, non_blocking=True)
            c.record(stream)
            if it >= args.warmup:
                e_ms.append((a, c))
        torch.cuda.synchronize()
        e_serial = max_over_ranks(sum(a.elapsed_time(c) for a, c in e_ms) / len(e_ms), world, dev)
        e2e = {"value": whole_job_tflops(flops, world, e_pipe), "unit": "TFLOP/s", "ms_per_step": e_pipe,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "form": "copies pipelined with compute over two streams (inputs larger than L2, rewritten by "
                       "each step's copy)",
               "serial": {"value": whole_job_tflops(flops, world, e_serial), "ms_per_step": e_serial}}

    if rank != 0:
        return
    bf16_peak, hbm_peak, peak_kind = measured_peaks()
    fp8_peak = bf16_peak * FP8_OVER_BF16
    achieved = flops / (attn_avg * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": recorded_traffic(),
                "kernel": "attn_fwd_kernel", "attn_ms": attn_avg,
                "peak_note": "%s bf16 burst %.1f TFLOP/s x nominal fp8/bf16 ratio 2" % (peak_kind, bf16_peak)}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        val, t_total, _ = run_oracle_steps(w, q_cpu, k_cpu, v_cpu, steps=6, warmup=0, rows_per_step=16)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": "6 x (16 query rows drawn uniformly from S=%d, one query head each, with the "
                         "quantisation of exactly the operands they read); %.1f s of CPU time; numpy fp64, "
                         "matmul on OpenBLAS threads" % (w.S, t_total)}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_OWN_BLOCK_TFLOPS, "dtype": "mxfp8_e4m3", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "S": S, "Hq": Hq, "Hkv": Hkv, "D": D,
                   "layout": "BSHD" if w.layout == 0 else "SBHD", "p_terms": args.p_terms,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MB write outside the per-step events)"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "quant_ms": sum(quant_ms) / len(quant_ms),
        "attn_ms": attn_avg,
        "p_terms2": {"ms_per_step": ms2, "attn_ms": attn2, "value": whole_job_tflops(flops, world, ms2)},
        "mxfp8_o": {"ms_per_step": ms8, "attn_ms": attn8, "value": whole_job_tflops(flops, world, ms8)},
        "bwd": {"bwd_ms": bwd_avg, "fwd_bwd_ms": ms_per_step + bwd_avg,
                "tflops": whole_job_tflops(2.5 * flops, world, bwd_avg),
                "note": "backward on decoded operands, BF16 MMAs; FLOPs = 2.5 x forward"},
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
