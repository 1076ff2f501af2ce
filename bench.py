#!/usr/bin/env python
"""Benchmark of exact attention (forward + backward) on GB300 through the C ABI.

One step = fa_fwd + fa_bwd over one batch of the workload (seeded bf16 N(0,1)
inputs already resident in HBM).  Prints ONE JSON line on rank 0:

  value        algorithmic TFLOP/s of the whole job (forward 4*d, backward 10*d
               per visible (query, key) pair and query head; causal halves it)
  e2e          the same metric through the C ABI with pinned HOST buffers: each
               step copies Q, K, V, dO in and O, LSE, dQ, dK, dV out (two device
               buffer sets; copies of neighbouring steps overlap the kernels)
  roofline     the dominant kernel (largest device time): algorithmic FLOPs (or
               bytes) per launch / its mean launch time, from a second timed
               region of K steps in which the library records CUDA events around
               each of its launches on the launching stream, against the measured
               bf16 tensor peak (or HBM copy rate): whichever of the two gives the
               kernel's algorithmic work the longer time is its bound
  cpu_baseline the fp64 oracle timed on the host cores on a bounded sample
  clocks       SM clocks and throttle reasons sampled during the timed region

--impl reference runs the fp64 CPU oracle as the reference arm instead.
Multi-GPU (torchrun): independent replicas, one per GPU ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from exact_io_aware_tcgen05_gb300.inputs import attention_inputs  # noqa: E402
from exact_io_aware_tcgen05_gb300.workloads import (BENCH_DEFAULT, INCOHERENT_SEED,  # noqa: E402
                                                    WORKLOADS, visible_pairs)

METRIC = "attention fwd/bwd TFLOP/s (bf16, causal-halved) and % of GB300 dense BF16 peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# Algorithmic FLOPs per visible pair and query head, split by kernel: the
# forward's two products; of the backward's five products (S recomputed, dP,
# dV, dK, dQ) the fused kernel performs all five; on the split path the dK/dV
# kernel performs four and the dQ kernel contributes dQ (its second S and dP
# are recomputation and not counted).
KERNEL_FLOPS_PER_PAIR_D = {"fa_fwd": 4, "fa_bwd_fused": 10, "fa_bwd_dkdv": 8, "fa_bwd_dq": 2}
# the products each kernel issues, per visible pair and unit of d (the dQ kernel rebuilds
# S and dP before dQ = dS K: 3 products; the others issue exactly what they are credited)
KERNEL_EXECUTED_FLOPS_PER_PAIR_D = {"fa_fwd": 4, "fa_bwd_fused": 10, "fa_bwd_dkdv": 8, "fa_bwd_dq": 6}
HBM_KERNELS = ("fa_bwd_preprocess", "fa_bwd_dq_convert")
KERNEL_SOURCES = {"fa_fwd": ("fa_fwd.cu",), "fa_bwd_fused": ("fa_bwd_fused.cu", "fa_bwd_common.cuh"),
                  "fa_bwd_dkdv": ("fa_bwd.cu", "fa_bwd_common.cuh"),
                  "fa_bwd_dq": ("fa_bwd.cu", "fa_bwd_common.cuh"),
                  "fa_bwd_preprocess": ("fa_bwd.cu", "fa_bwd_common.cuh"),
                  "fa_bwd_dq_convert": ("fa_bwd_fused.cu", "fa_bwd_common.cuh")}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-events", action="store_true",
                    help="skip the second timed region with per-kernel events (no roofline)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--bwd-path", choices=["auto", "split", "fused"], default="auto",
                    help="backward path (fa_bwd_set_path): auto, the library's default choice; "
                         "split (dK/dV and dQ kernels); fused (one kernel)")
    ap.add_argument("--fwd-heads", type=int, default=0,
                    help="query heads per forward CTA (fa_fwd_set_heads): 0, the library's "
                         "choice; else a divisor of the GQA group")
    ap.add_argument("--dq-heads", type=int, default=0,
                    help="query heads per dQ CTA of the split backward (fa_bwd_set_dq_heads): "
                         "0, the library's choice; else a divisor of the GQA group")
    return ap.parse_args()


def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over all ranks of the default process group (identity
    when there is none or it has one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput of `world` replicas, each doing flops_per_rank_step per step,
    when the slowest rank takes ms_per_step per step."""
    return world * flops_per_rank_step / (ms_per_step / 1e3) / 1e12


def binding_roof(tflop: float, nbytes: float, peak_tflops: float, peak_gbs: float) -> str:
    """The roof that binds a kernel: "tensor" if its algorithmic FLOPs need at least as
    long at the tensor peak as its algorithmic bytes need at the HBM rate, else "hbm"."""
    return "tensor" if tflop / peak_tflops >= nbytes / 1e9 / peak_gbs else "hbm"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# headers every kernel is compiled with: a change there also changes the kernel
SHARED_SOURCES = ("fa_ptx.cuh", "fa_seq.cuh", "fa_kernels.h")


def source_sha(kernel: str) -> str:
    """SHA-256 (first 16 hex digits) of the kernel's source file and the shared headers."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        with open(os.path.join(ROOT, "exact_io_aware_tcgen05_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(workload, {}).get(kernel)
    if not e or e.get("source_sha") != source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = tempfile.TemporaryFile(mode="w+")

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- oracle

def oracle_pass(w, q, k, v, do, L: int, n_kv: int) -> None:
    """One fp64 oracle pass (forward, and backward if the workload has one) over the first
    L tokens of one sequence for key/value heads 0..n_kv-1 and their query heads.
    q, do: [tokens, Hq', d]; k, v: [tokens, Hkv', d] float64 views of that sequence."""
    import oracle
    G = w.Hq // w.Hkv
    if w.p_drop > 0:
        # the dropout oracle (dense, numpy)
        from oracle import dropout as odrop
        from exact_io_aware_tcgen05_gb300.workloads import DROPOUT_OFFSET, DROPOUT_SEED
        kw = dict(causal=w.causal, window=w.window, scale=w.scale, p_drop=w.p_drop,
                  seed=DROPOUT_SEED, offset=DROPOUT_OFFSET)
        qq, kk, vv = q[None, :L, :G * n_kv], k[None, :L, :n_kv], v[None, :L, :n_kv]
        odrop.attention_fwd(qq, kk, vv, **kw)
        if w.backward:
            odrop.attention_bwd(qq, kk, vv, do[None, :L, :G * n_kv], **kw)
        return
    for g in range(n_kv):
        qg = q[:L, g * G:(g + 1) * G].transpose(1, 0, 2)
        oracle.fwd_group(qg, k[:L, g], v[:L, g], w.causal, w.window, w.scale)
        if w.backward:
            oracle.bwd_group(qg, k[:L, g], v[:L, g], do[:L, g * G:(g + 1) * G].transpose(1, 0, 2),
                             w.causal, w.window, w.scale)


def oracle_sample(w, x, target_s: float):
    """Time the fp64 oracle (forward, and backward if the workload has one) on a sample of
    sequence 0: a prefix of it for the query heads of key/value head 0, grown until the run
    takes about target_s seconds; once the prefix is the whole sequence, further key/value
    heads (with their query heads) join.  Returns (TFLOP/s, threads, description, seconds,
    prefix length, key/value heads)."""
    import oracle
    oracle.build()
    G = w.Hq // w.Hkv
    L_full = w.seq_lengths()[0]
    cu = w.cu_seqlens()
    q = oracle.sequence_views(x["q"], 0, cu, slice(0, w.Hq))
    k = oracle.sequence_views(x["k"], 0, cu, slice(0, w.Hkv))
    v = oracle.sequence_views(x["v"], 0, cu, slice(0, w.Hkv))
    do = oracle.sequence_views(x["dout"], 0, cu, slice(0, w.Hq)) if w.backward else None

    def run(L, n_kv):
        t0 = time.perf_counter()
        oracle_pass(w, q, k, v, do, L, n_kv)
        return time.perf_counter() - t0

    L, n_kv = min(256, L_full), 1
    t = run(L, n_kv)
    while L < L_full and t < target_s / 3:
        L_new = min(L_full, int(L * max(1.25, min(4.0, math.sqrt(target_s / max(t, 1e-3))))))
        L_new = max(L + 1, L_new)
        L, t = L_new, run(L_new, n_kv)
    if L == L_full and t < target_s / 2 and w.Hkv > 1:
        n_kv = min(w.Hkv, max(2, int(target_s / max(t, 1e-3))))
        t = run(L, n_kv)
    flops = (14 if w.backward else 4) * w.d * G * n_kv * visible_pairs(L, w.causal, w.window)
    desc = (f"sequence 0, first {L} of {L_full} tokens, query heads 0..{G * n_kv - 1} "
            f"(key/value heads 0..{n_kv - 1}), "
            f"{'forward + backward' if w.backward else 'forward'} in fp64"
            + (f", dropout {w.p_drop}" if w.p_drop > 0 else ""))
    return flops / t / 1e12, oracle.threads(), desc, t, L, n_kv


# ------------------------------------------------------------ reference arm

def run_reference(args, w):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    x = attention_inputs(w.q_shape, w.kv_shape, args.seed, with_dout=w.backward,
                         dtype="bf16" if w.dtype == "fp8" else w.dtype)
    total = args.steps + args.warmup
    per_step = min(10.0, max(0.3, 120.0 / max(total, 1)))   # whole run within a few minutes
    _, threads, desc, _, L, n_kv = oracle_sample(w, x, per_step)
    import oracle
    G = w.Hq // w.Hkv
    cu = w.cu_seqlens()
    q = oracle.sequence_views(x["q"], 0, cu, slice(0, G * n_kv))[:L]
    do = oracle.sequence_views(x["dout"], 0, cu, slice(0, G * n_kv))[:L] if w.backward else None
    k = oracle.sequence_views(x["k"], 0, cu, slice(0, n_kv))[:L]
    v = oracle.sequence_views(x["v"], 0, cu, slice(0, n_kv))[:L]
    times = []
    for i in range(total):
        t0 = time.perf_counter()
        oracle_pass(w, q, k, v, do, L, n_kv)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    flops = (14 if w.backward else 4) * w.d * G * n_kv * visible_pairs(L, w.causal, w.window)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "cpu run; no L2 involved"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def served_heads(w, fp8: bool, bwd: bool, fused: bool):
    """(forward, dQ) query heads per CTA of a run on this thread's settings; dQ is None
    without a split backward."""
    import exact_io_aware_tcgen05_gb300 as fa
    q = (w.B, w.Hq, w.Hkv, w.N, w.d, int(w.causal), w.window, w.total_tokens if w.packed else 0)
    one = fp8 or w.p_drop > 0
    fwd = 1 if one else fa.fa_fwd_heads(*q)
    dq = None if (not bwd or fused) else (1 if w.p_drop > 0 else fa.fa_bwd_dq_heads(*q))
    return fwd, dq


def workload_config(w, l2_note):
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
           "causal": w.causal, "window": w.window, "packed": w.packed,
           "total_tokens": w.total_tokens, "scale": "1/sqrt(d)",
           "inputs": (f"{w.dtype} iid N(0,1), seed 0" if w.dtype != "fp8" else
                      "bf16 iid N(0,1), seed 0, quantised to e4m3 before the timed region"
                      + (" (Q, K rotated first: incoherent processing)" if w.incoherent else "")),
           "l2": l2_note}
    if w.packed:
        cfg["lengths"] = list(w.lengths)
    if w.p_drop > 0:
        cfg["p_drop"] = w.p_drop
    return cfg


# ----------------------------------------------------------------- our arm

def run_ours(args, w):
    import torch
    rank, world, local_rank = dist_info()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from exact_io_aware_tcgen05_gb300 import build as libbuild
    libbuild.build()
    import exact_io_aware_tcgen05_gb300 as fa
    fa.load()

    bwd = w.backward          # forward-only workloads time fa_fwd alone
    fp8 = w.dtype == "fp8"
    x = attention_inputs(w.q_shape, w.kv_shape, args.seed, with_dout=bwd,
                         dtype="bf16" if fp8 else w.dtype)
    dtype_code = fa.FA_DTYPE_F16 if w.dtype == "f16" else fa.FA_DTYPE_BF16
    from exact_io_aware_tcgen05_gb300.workloads import DROPOUT_OFFSET, DROPOUT_SEED
    if w.p_drop > 0:
        def fwd_call(*a):
            fa.fa_fwd_dropout(dtype_code, w.p_drop, DROPOUT_SEED, DROPOUT_OFFSET, *a)

        def bwd_call(*a):
            fa.fa_bwd_dropout(dtype_code, w.p_drop, DROPOUT_SEED, DROPOUT_OFFSET, *a)
    else:
        def fwd_call(*a):
            fa.fa_fwd_typed(dtype_code, *a)

        def bwd_call(*a):
            fa.fa_bwd_typed(dtype_code, *a)

    def pinned(a):
        if a.dtype == np.float16:
            return torch.from_numpy(a).pin_memory()
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()

    h_in = {n: pinned(x[n]) for n in (("q", "k", "v", "dout") if bwd else ("q", "k", "v"))}
    d_in = {n: t.to(dev) for n, t in h_in.items()}
    cu = None if not w.packed else torch.from_numpy(w.cu_seqlens()).to(dev)
    T = w.total_tokens if w.packed else 0
    o = torch.empty_like(d_in["q"])
    lse = torch.empty(w.lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(d_in["q"]), torch.empty_like(d_in["k"]),
                  torch.empty_like(d_in["v"]))
    ws_size = {"auto": fa.fa_bwd_workspace_size, "split": fa.fa_bwd_workspace_size_min,
               "fused": fa.fa_bwd_workspace_size_fused}[args.bwd_path]
    ws_bytes = ws_size(w.B, w.Hq, w.Hkv, w.N, w.d, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fa.fa_bwd_set_path({"auto": fa.FA_BWD_AUTO, "split": fa.FA_BWD_SPLIT,
                        "fused": fa.FA_BWD_FUSED}[args.bwd_path])
    fa.fa_bwd_set_dq_heads(args.dq_heads)
    fa.fa_fwd_set_heads(args.fwd_heads)
    fused = bwd and fa.fa_bwd_path(w.B, w.Hq, w.Hkv, w.N, w.d, int(w.causal), w.window, T,
                                   ws_bytes) == fa.FA_BWD_FUSED
    bwd_kernels = 3
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    geo = (w.B, w.Hq, w.Hkv, w.N, w.d, int(w.causal), w.window, cu, T, w.scale)
    fwd_call_e2e = fwd_call
    if fp8:
        # The fp8 forward's inputs are its e4m3 operands: quantised once here, like the
        # bf16 inputs are made resident before the timed region.  The end-to-end steps
        # quantise their own bf16 inputs every step (two operand sets, one per buffer set).
        nb = fa.fa_fp8_scale_blocks(w.B, w.N, T, w.packed)
        vt_tokens = fa.fa_fp8_vt_tokens(w.B, w.N, T, w.packed)

        def fp8_buffers():
            return (torch.empty(w.q_shape, dtype=torch.uint8, device=dev),
                    torch.empty((w.Hq, nb), dtype=torch.float32, device=dev),
                    torch.empty(w.kv_shape, dtype=torch.uint8, device=dev),
                    torch.empty((w.Hkv, nb), dtype=torch.float32, device=dev),
                    torch.empty((w.Hkv, w.d, vt_tokens), dtype=torch.uint8, device=dev),
                    torch.empty((w.Hkv, w.B), dtype=torch.float32, device=dev))

        def quantise(q, k, v, ops, st):
            if w.incoherent:
                fa.fa_fp8_quantize_qk_incoherent(q, ops[0], ops[1], nb, w.B, w.Hq, w.N, w.d, cu, T,
                                                 INCOHERENT_SEED, st)
                fa.fa_fp8_quantize_qk_incoherent(k, ops[2], ops[3], nb, w.B, w.Hkv, w.N, w.d, cu,
                                                 T, INCOHERENT_SEED, st)
            else:
                fa.fa_fp8_quantize_qk(q, ops[0], ops[1], nb, w.B, w.Hq, w.N, w.d, cu, T, st)
                fa.fa_fp8_quantize_qk(k, ops[2], ops[3], nb, w.B, w.Hkv, w.N, w.d, cu, T, st)
            fa.fa_fp8_quantize_v(v, ops[4], ops[5], vt_tokens, w.B, w.Hkv, w.N, w.d, cu, T, st)

        fp8_ops = [fp8_buffers(), fp8_buffers()]
        quantise(d_in["q"], d_in["k"], d_in["v"], fp8_ops[0], s)
        e2e_set = {}

        def fwd_call(q, k, v, o_, lse_, *rest):
            fa.fa_fwd_fp8(*fp8_ops[0], nb, vt_tokens, o_, lse_, *rest)

        def fwd_call_e2e(q, k, v, o_, lse_, *rest):
            ops = fp8_ops[e2e_set.get(q.data_ptr(), 0)]
            quantise(q, k, v, ops, rest[-1])
            fa.fa_fwd_fp8(*ops, nb, vt_tokens, o_, lse_, *rest)

    def step(ev_f=None, ev_b=None):
        if ev_f is not None:
            fa.fa_set_launch_events(ev_f)
        fwd_call(d_in["q"], d_in["k"], d_in["v"], o, lse, *geo, s)
        if not bwd:
            return
        if ev_b is not None:
            fa.fa_set_launch_events(ev_b)
        bwd_call(d_in["q"], d_in["k"], d_in["v"], o, lse, d_in["dout"], dq, dk, dv, *geo, ws,
                 ws_bytes, s)

    in_bytes = sum(t.numel() * 2 for t in d_in.values()) + o.numel() * 2
    flush = in_bytes < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    l2_note = (f"L2 flushed between steps (write of {2 * L2_BYTES >> 20} MiB outside the step events)"
               if flush else f"inputs larger than L2 ({in_bytes >> 20} MiB per step); no flush")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    fa.fa_device_status(s)

    K = args.steps
    ev_f = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    ev_b = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)] if bwd else [None] * K
    for e in sum(ev_f, []) + (sum(ev_b, []) if bwd else []):
        e.record(stream)      # instantiate the CUDA events
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)] if flush else None
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()

    def timed_region(with_kernel_events):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            if flush:
                scratch.fill_(float(i))
                step_ev[i][0].record(stream)
            if with_kernel_events:
                step(ev_f[i], ev_b[i])
            else:
                step()
            if flush:
                step_ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        fa.fa_device_status(s)
        if flush:
            return sum(a.elapsed_time(b) for a, b in step_ev)
        return t_start.elapsed_time(t_end)

    # Region 1 (the reported value): K steps exactly as a user runs them.
    elapsed = timed_region(False)
    # Region 2 (per-kernel durations for the roofline): K more steps with the
    # library recording caller-owned CUDA events around each of its launches on
    # the launching stream.  On the split path, events between the backward's
    # launches keep its dQ kernel from overlapping the end of the dK/dV kernel, so
    # this region is not used for the step time.
    kern_ms = None
    if not args.no_kernel_events:
        timed_region(True)
        kern_ms = {"fa_fwd": [a.elapsed_time(b) for a, b in ev_f]}
        if bwd:
            kern_ms["fa_bwd_preprocess"] = [e[0].elapsed_time(e[1]) for e in ev_b]
            if fused:
                kern_ms["fa_bwd_fused"] = [e[1].elapsed_time(e[2]) for e in ev_b]
                kern_ms["fa_bwd_dq_convert"] = [e[2].elapsed_time(e[3]) for e in ev_b]
            else:
                kern_ms["fa_bwd_dkdv"] = [e[1].elapsed_time(e[2]) for e in ev_b]
                kern_ms["fa_bwd_dq"] = [e[2].elapsed_time(e[3]) for e in ev_b]
    clocks = sampler.stop()
    elapsed = max_over_ranks(elapsed, dev)
    ms_per_step = elapsed / K
    fwd_flops, bwd_flops = w.fwd_flops(), (w.bwd_flops() if bwd else 0)
    value = job_tflops(fwd_flops + bwd_flops, world, ms_per_step)

    # ---- end to end through the C ABI with host buffers
    # Each step copies its inputs in from pinned host memory and its results out.
    # Two sets of device buffers let step k+1's input copy and step k-1's output
    # copy overlap step k's kernels (three streams, ordered by events).
    E = max(1, args.e2e_steps)
    d_out0 = {"o": o, "lse": lse}
    if bwd:
        d_out0.update(dq=dq, dk=dk, dv=dv)
    h_out = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in d_out0.items()}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    d_ins = [d_in, {n: torch.empty_like(t) for n, t in d_in.items()}]
    if fp8:
        e2e_set.update({d_ins[0]["q"].data_ptr(): 0, d_ins[1]["q"].data_ptr(): 1})
    d_outs = [d_out0, {n: torch.empty_like(t) for n, t in d_out0.items()}]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}

    def e2e_step(k):
        b = k & 1
        di, do_ = d_ins[b], d_outs[b]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev["comp"][b])          # step k-2 done reading di
            for n in h_in:
                di[n].copy_(h_in[n], non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if k >= 2:
            stream.wait_event(ev["out"][b])             # step k-2's results copied out
        fwd_call_e2e(di["q"], di["k"], di["v"], do_["o"], do_["lse"], *geo, s)
        if bwd:
            bwd_call(di["q"], di["k"], di["v"], do_["o"], do_["lse"], di["dout"], do_["dq"],
                     do_["dk"], do_["dv"], *geo, ws, ws_bytes, s)
        ev["comp"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            for n in h_out:
                h_out[n].copy_(do_[n], non_blocking=True)
            ev["out"][b].record(s_out)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0.record(s_in)
    for k in range(E):
        e2e_step(k)
    s_out.wait_event(ev["comp"][(E - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    fa.fa_device_status(s)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, dev)
    e2e_value = job_tflops(fwd_flops + bwd_flops, world, e2e_ms)

    # ---- roofline of the dominant kernel
    peaks, peak_src = measured_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # e4m3 products: the measured bf16 figure times the nominal fp8 / bf16 ratio (4.5 / 2.25)
    peak_mult = 2.0 if fp8 else 1.0
    peak_tf *= peak_mult
    peak_gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kernels, roof, fwd_tf, bwd_tf = None, None, None, None
    if not args.no_kernel_events:
        pairs_heads = w.visible_pairs_per_head() * w.Hq
        kernels = {}
        for name, times in kern_ms.items():
            mean = sum(times) / len(times)
            entry = {"ms_mean": mean, "ms_median": statistics.median(times), "launches": len(times),
                     "share": None}
            if name in KERNEL_FLOPS_PER_PAIR_D:
                fl = KERNEL_FLOPS_PER_PAIR_D[name] * w.d * pairs_heads
                entry["algorithmic_tflop_per_launch"] = fl / 1e12
                entry["tflops"] = fl / (mean / 1e3) / 1e12
                ex = KERNEL_EXECUTED_FLOPS_PER_PAIR_D[name] * w.d * pairs_heads
                entry["executed_tflop_per_launch"] = ex / 1e12
                entry["executed_tflops"] = ex / (mean / 1e3) / 1e12
            by = w.kernel_io_bytes(name, fused)
            entry["algorithmic_bytes_per_launch"] = by
            entry["gbs"] = by / (mean / 1e3) / 1e9
            entry["bound"] = binding_roof(entry.get("algorithmic_tflop_per_launch", 0.0), by,
                                          peak_tf, peak_gbs)
            kernels[name] = entry
        tot = sum(k["ms_mean"] for k in kernels.values())
        for k in kernels.values():
            k["share"] = k["ms_mean"] / tot
        dom = max(kernels, key=lambda n: kernels[n]["ms_mean"])
        of = " of measured" if peak_src == "measured" else " of fallback"
        if kernels[dom]["bound"] == "tensor":
            roof = {"kernel": dom, "bound": "tensor", "achieved": kernels[dom]["tflops"], "peak": peak_tf,
                    "unit": "TFLOP/s", "frac": kernels[dom]["tflops"] / peak_tf,
                    "peak_source": f"{peak_src} bf16_tflops (burst)" + (" x 2 (nominal fp8 / bf16)" if fp8 else "") + of}
        else:
            roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak_gbs,
                    "unit": "GB/s", "frac": kernels[dom]["gbs"] / peak_gbs,
                    "peak_source": f"{peak_src} hbm_gbs (copy)" + of}
        roof["traffic"] = recorded_traffic(dom, w.name)
        fwd_tf = fwd_flops / (kernels["fa_fwd"]["ms_mean"] / 1e3) / 1e12
        bwd_tf = None
        if bwd:
            # the backward's kernels overlap: its time is the step minus the forward
            bwd_ms = ms_per_step - kernels["fa_fwd"]["ms_mean"]
            bwd_tf = bwd_flops / (bwd_ms / 1e3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, threads, desc, secs, _, _ = oracle_sample(w, x, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": secs}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else w.dtype,
            "data": "synthetic",
            "config": workload_config(w, l2_note),
            "pct_of_peak": value / world / peak_tf,
            "fwd_tflops": fwd_tf, "fwd_pct_of_peak": (fwd_tf / peak_tf) if fwd_tf else None,
            "bwd_tflops": bwd_tf, "bwd_pct_of_peak": (bwd_tf / peak_tf) if bwd_tf else None,
            "roofline": roof, "kernels": kernels, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E},
            "gpu_launches": world * K * (1 + (bwd_kernels if bwd else 0)), "clocks": clocks,
            "bwd_path": ("fused" if fused else "split") if bwd else None,
        }
        # query heads per CTA the kernels served: the library's choice, or the count the
        # options above forced (dropout and fp8 forwards serve one head per CTA)
        line["fwd_heads"], line["dq_heads"] = served_heads(w, fp8, bwd, fused)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
