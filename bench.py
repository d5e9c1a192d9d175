"""Benchmark of the tiled FlashAttention forward on GB300.

Workload (one "step" = one forward over one batch): dense causal attention,
B=2, H=16, Sq=Skv=2048, D=Dv=128, bf16 Q/K/V drawn N(0,1), scale 1/sqrt(128),
fp32 LSE output.  Metric: algorithmic TFLOP/s = 2 (D + Dv) x unmasked
(query, key) pairs / time, also reported as ms per call and as a fraction of
the measured dense bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With the default workload (c2) the line also carries a "workloads" entry for
the other workloads (c3 GQA causal ragged, c4 block-sparse, c5 top-k sparse
MLA), each timed the same way after the benchmark line's own timed region.

N > 1 runs one process per GPU (torchrun); every rank runs its own replica of
the workload (the forward shards over (b, h) with no exchange), so the
scaling is weak and the whole-job value is the sum over ranks.
The reference arm times the fp64 CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense BF16 tensor peak; ms/call"
L2_BYTES = 129 * 2 ** 20


KERNEL_SOURCES = {
    # device code of each kernel: the headers its translation unit pulls in
    "dense": ("fa_ptx.cuh", "fa_tiled.cuh"),
    "topk": ("fa_ptx.cuh", "fa_tiled.cuh", "fa_mla.cuh"),
}


def kernel_source_hash(kind: str = "dense") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_fa_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "sm_max_mhz": 2070.0}, "fallback"


def dram_traffic(workload: str):
    """ncu DRAM bytes per launch for the current kernel sources, else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload)
    kind = "topk" if workload == "c5" else "dense"
    if not e or e.get("kernel_source_hash") != kernel_source_hash(kind):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        load = [s for s in sm] or [None]
        return {"sm_mhz": statistics.median(load) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


WORKLOADS = {
    "c2": (2, "dense causal attention forward, B=2 H=16 Sq=Skv=2048 D=Dv=128, bf16 Q/K/V ~ N(0,1), "
              "scale 1/sqrt(128), fp32 LSE"),
    "c3": (3, "GQA causal ragged attention forward, B=4 Hq=32 Hkv=8 S=4096 D=Dv=128, "
              "seqlens [4096, 3001, 517, 14], bf16"),
    "c4": (4, "block-sparse attention forward, B=1 H=16 S=16384 D=Dv=128, fp16, per (head, query "
              "block) the diagonal + 15 random KV blocks of 128 (causal inside the diagonal block)"),
    "c5": (5, "top-k sparse MLA forward, T=4096 tokens, 128 query heads, one latent KV head, "
              "D=576 (512 latent + 64 rope), Dv=512, 2048 key slots per token, bf16"),
}


def max_over_ranks(dist, values, device):
    """Element-wise maximum of per-rank values over all ranks (the whole job
    is as slow as its slowest rank); values unchanged without a process group."""
    if dist is None:
        return [float(x) for x in values]
    import torch
    t = torch.tensor([float(x) for x in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Throughput of all ranks together: every rank runs one step's work in
    ms_per_step (replicas, weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def workload_problem(name="c2", mla_tokens=4096):
    from attention_forward_fa_gb300 import workloads as W
    if name == "c5" and mla_tokens != 4096:
        return W.sparse_mla(name=f"sparse_mla_T{mla_tokens}", T=mla_tokens, seed=1005)
    return W.config(WORKLOADS[name][0])


def workload_desc(p, name="c2"):
    from attention_forward_fa_gb300 import workloads as W
    mask = {W.MASK_NONE: "none", W.MASK_CAUSAL: "causal",
            W.MASK_CAUSAL_DIAG_BLOCK: "causal inside the diagonal block"}[p.mask]
    d = {"workload": WORKLOADS[name][1], "B": p.B, "Hq": p.Hq, "Hkv": p.Hkv, "Sq": p.Sq,
         "Skv": p.Skv, "D": p.D, "Dv": p.Dv, "mask": mask, "rescale_threshold": 0.0}
    if p.topk_idx is not None:
        d["topk"] = int(p.topk_idx.shape[-1])
        if p.Sq != 4096:
            d["workload"] = d["workload"].replace("T=4096", f"T={p.Sq}")
    return d


def oracle_rows(p, q, k, v, b, h, rows):
    """Time the fp64 oracle on `rows` of head (b, h); returns (algorithmic
    flops of those rows, seconds)."""
    from oracle import attention as A
    t0 = time.perf_counter()
    A.attention_fwd(q, k, v, p.scale, mask=p.mask, seqlens=p.seqlens, rows=rows,
                    heads=np.array([h]), batches=np.array([b]))
    el = time.perf_counter() - t0
    kv = p.Skv if p.seqlens is None else int(p.seqlens[b])
    keys = np.minimum(rows + 1, kv) if p.mask == 1 else np.full(rows.size, kv)
    return 2.0 * (p.D + p.Dv) * float(keys.sum()), el


def row_sample(p, n_rows, step_index):
    """n_rows rows spread evenly over [0, Sq) (so the causal work per row
    matches the whole workload), shifted per step; head and batch rotate."""
    stride = max(1, p.Sq // n_rows)
    off = step_index % stride
    rows = np.arange(off, p.Sq, stride)[:n_rows]
    bh = step_index % (p.B * p.Hq)
    return rows, bh // p.Hq, bh % p.Hq


def oracle_timed(p, seconds):
    """Oracle throughput on a bounded sample: consecutive row samples until
    `seconds` of CPU work have passed.  Returns (flops, seconds, rows)."""
    q, k, v = p.q(), p.k(), p.v()
    f_tot = t_tot = 0.0
    n = 0
    i = 0
    while t_tot < seconds:
        rows, b, h = row_sample(p, 256, i)
        f, t = oracle_rows(p, q, k, v, b, h, rows)
        f_tot += f
        t_tot += t
        n += rows.size
        i += 1
    return f_tot, t_tot, n


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    p = workload_problem()
    from attention_forward_fa_gb300 import workloads as W
    q, k, v = p.q(), p.k(), p.v()
    # size each step so that warm-up + K steps take about a minute
    rows0, b0, h0 = row_sample(p, 64, 0)
    _, t64 = oracle_rows(p, q, k, v, b0, h0, rows0)
    per_row = max(t64 / 64, 1e-6)
    budget = 60.0 / max(1, args.steps + args.warmup)
    n_rows = int(min(p.Sq, max(1, budget / per_row)))
    for i in range(args.warmup):
        rows, b, h = row_sample(p, n_rows, i)
        oracle_rows(p, q, k, v, b, h, rows)
    t_tot = f_tot = 0.0
    for i in range(args.steps):
        rows, b, h = row_sample(p, n_rows, args.warmup + i)
        f, t = oracle_rows(p, q, k, v, b, h, rows)
        f_tot += f
        t_tot += t
    value = f_tot / t_tot / 1e12
    sample = (f"each step = {n_rows} query rows (spread over the sequence) of one (b, h) head "
              f"of the workload, fp64 numpy oracle materialising S and P; the full workload is "
              f"{W.algorithmic_flops(p) / 1e9:.2f} GFLOP")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_desc(p),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class Prepared:
    """Device buffers of one workload: rotating input / output sets larger than
    L2 together, and the fa_fwd arguments."""

    def __init__(self, p, dev):
        import torch
        import attention_forward_fa_gb300 as fa
        self.p = p
        bf16 = p.dtype == "bf16"
        self.bf16 = bf16
        dt = torch.bfloat16 if bf16 else torch.float16
        self.dt = dt

        def up(bits):
            return torch.from_numpy(bits.view(np.int16).copy()).to(dev).view(dt)

        def up_i32(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        self.q0, self.k0 = up(p.q_bits), up(p.k_bits)
        self.v0 = None if p.v_from_k else up(p.v_bits)
        self.seqlens = up_i32(p.seqlens)
        self.blk = self.tk = None
        if p.kv_block_idx is not None:
            bi = up_i32(p.kv_block_idx)
            nb, hh, nqb, ms = bi.shape
            self.blk = (bi, ms, 128, hh * nqb * ms, nqb * ms if hh > 1 else 0)
        if p.topk_idx is not None:
            ti = up_i32(p.topk_idx)
            self.tk = (ti, ti.shape[-1], ti.shape[-2] * ti.shape[-1])
        # top-k with a bf16 key latent: the latent (V is part of it) is
        # converted to fp16 by a separate pass; a bf16 V of the other paths is
        # converted inside the attention kernel
        self.conv_pass = bf16 and p.v_from_k
        self.n_conv = self.k0.numel() if self.conv_pass else 0
        mode = p.mask | (fa.FA_V_FROM_K if p.v_from_k else 0)
        if not bf16:
            mode |= fa.FA_DTYPE_FP16
        elif self.conv_pass:
            mode |= fa.FA_V_FP16
        self.mode = mode
        self.threshold = 0.0   # rescale_threshold of every call (log2 units; 0 = exact max)
        o_bytes = 2 * p.B * p.Hq * p.Sq * p.Dv + 4 * p.B * p.Hq * p.Sq
        v_n = 0 if self.v0 is None else self.v0.numel()
        self.per_set = 2 * (self.q0.numel() + self.k0.numel() + v_n) + 2 * self.n_conv + o_bytes
        self.n_sets = max(2, int(np.ceil(2.5 * L2_BYTES / self.per_set)))
        self.sets = []
        for _ in range(self.n_sets):
            o = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=dt, device=dev)
            lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device=dev)
            q, k = self.q0.clone(), self.k0.clone()
            v = None if self.v0 is None else self.v0.clone()
            c16 = torch.empty(k.shape, dtype=torch.float16, device=dev) if self.conv_pass else None
            self.sets.append((q, k, v, c16, o, lse))

    def step(self, i, strm, ev=None):
        """One step = the whole hot path: one fa_fwd launch, plus for a bf16
        top-k latent the conversion pass before it (issued through the C ABI on
        its own so that the attention kernel can be timed alone)."""
        import attention_forward_fa_gb300 as fa
        p = self.p
        ssp = strm.cuda_stream
        q, k, v, c16, o, lse = self.sets[i % self.n_sets]
        if ev:
            ev[0].record(strm)
        if self.conv_pass:
            code = fa.fa_convert_v_fp16(k, c16, self.n_conv, ssp)
            if code != 0:
                raise RuntimeError(fa.fa_strerror(code))
        if ev:
            ev[1].record(strm)
        code = fa.fa_fwd(q, c16 if self.conv_pass else k, v, o, lse, p.B, p.Hq, p.Hkv, p.Sq,
                         p.Skv, p.D, p.Dv, p.scale, self.mode, self.seqlens, self.blk, self.tk,
                         self.threshold, ssp)
        if code != 0:
            raise RuntimeError(fa.fa_strerror(code))
        if ev:
            ev[2].record(strm)


def timed_steps(prep, steps, warmup, soak, dist, local, no_graph=False):
    """Warm-up, an untimed soak (clocks sampled under load from its start),
    then exactly `steps` steps between a barrier + synchronize on both sides.
    Returns (total ms, mean attention-kernel ms, mean conversion ms, clocks,
    graph used)."""
    import torch
    import attention_forward_fa_gb300 as fa
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        prep.step(i, stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else local)
    sampler.start()
    t_soak = time.perf_counter()
    i = 0
    while time.perf_counter() - t_soak < soak:
        for _ in range(20):
            prep.step(i, stream)
            i += 1
        torch.cuda.synchronize()
    # A step that is one launch (every workload but a bf16 top-k latent) runs
    # as a CUDA graph of the K launches, captured beforehand: the events around
    # the replay then time K launches of that one kernel, so its average launch
    # duration is the step time.  A two-launch step runs eagerly with events
    # around each launch.
    use_graph = not prep.conv_pass and not no_graph
    evs = None
    graph = None
    if use_graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            prep.step(0, cap)
            cap.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                for s_ in range(steps):
                    prep.step(s_, cap)
        torch.cuda.synchronize()
    else:
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    if use_graph:
        graph.replay()
    else:
        for s_ in range(steps):
            prep.step(s_, stream, evs[s_])
    t_all1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    status = fa.fa_check_status()
    if status != 0:
        raise RuntimeError("device status after timed region: " + fa.fa_strerror(status))
    total_ms = t_all0.elapsed_time(t_all1)
    if use_graph:
        kern_avg_ms = total_ms / steps
        conv_avg_ms = 0.0
    else:
        kern_ms = [e[1].elapsed_time(e[2]) for e in evs]
        conv_ms = [e[0].elapsed_time(e[1]) for e in evs]
        kern_avg_ms = sum(kern_ms) / len(kern_ms)
        conv_avg_ms = sum(conv_ms) / len(conv_ms)
    del graph
    return total_ms, kern_avg_ms, conv_avg_ms, clocks, use_graph


def kernel_name(p):
    bf16 = p.dtype == "bf16"
    if p.topk_idx is not None:
        return f"fa_mla_topk_kernel<{'bf16' if bf16 else 'fp16'}>"
    return (f"fa_fwd_tiled_kernel<{p.D},{'bf16' if bf16 else 'fp16'},{4 if p.D == 128 else 6}"
            f"{',convert-V' if bf16 else ''}>")


def time_workload(args, dev, dist, world, local, peak, name, p, threshold=0.0, traffic=True):
    """One workload entry: the path on problem `p` (workload `name`'s shape) at
    `threshold`, timed like the benchmark line with its own clock record: ms
    per call, algorithmic TFLOP/s, fraction of the peak, and the DRAM bytes
    per launch of the latest ncu capture of that kernel (null when its sources
    changed since, or when the capture is of another configuration)."""
    from attention_forward_fa_gb300 import workloads as W
    flops = W.algorithmic_flops(p)
    prep = Prepared(p, dev)
    prep.threshold = threshold
    total_ms, kern_ms, conv_ms, clocks, graph = timed_steps(
        prep, args.workload_steps, 5, args.workload_soak, dist, local)
    total_ms, kern_ms = max_over_ranks(dist, [total_ms, kern_ms], dev)
    ms = total_ms / args.workload_steps
    achieved = flops / (kern_ms * 1e-3) / 1e12
    cfg = workload_desc(p, name)
    cfg["rescale_threshold"] = threshold
    e = {"config": cfg, "algorithmic_gflop": flops / 1e9,
         "ms_per_call": ms, "tflops": whole_job_tflops(world, flops, ms),
         "kernel": kernel_name(p), "kernel_ms": kern_ms,
         "kernel_tflops": achieved, "frac": achieved / peak, "steps": args.workload_steps,
         "timing": "CUDA graph of the steps" if graph else "eager, events around each launch",
         "clocks": clocks, "traffic": dram_traffic(name) if traffic else None}
    if e["traffic"] is not None:
        e["dram_gbs"] = e["traffic"] / (kern_ms * 1e-3) / 1e9
    if prep.conv_pass:
        e["other_kernel"] = {"name": "fa_convert_v_kernel (bf16 -> fp16 copy of the key latent)",
                             "avg_ms": conv_ms}
    return e


def other_workloads(args, dev, dist, world, local, peak):
    """The same path on the other workloads (one fa_fwd call per step, threshold
    0, the given slot order); the top-k workload also at the lazy threshold and
    with every token's slot order reversed (the four runs the pages measure it
    in); and the benchmark's workload at the lazy threshold."""
    import dataclasses
    import numpy as np
    import torch
    out = {}
    for name in ("c3", "c4", "c5"):
        p = workload_problem(name)
        out[name] = time_workload(args, dev, dist, world, local, peak, name, p)
        torch.cuda.empty_cache()
        if name == "c5":
            # self key last, invalid slots first; the same valid pairs
            rev = dataclasses.replace(p, name=p.name + "_reversed",
                                      topk_idx=np.ascontiguousarray(p.topk_idx[:, :, ::-1]))
            for key, prob, thr in (("c5_threshold_8", p, 8.0), ("c5_reversed", rev, 0.0),
                                   ("c5_reversed_threshold_8", rev, 8.0)):
                e = time_workload(args, dev, dist, world, local, peak, name, prob, thr,
                                  traffic=False)
                e["config"]["slot_order"] = "reversed" if prob is rev else "given"
                out[key] = e
                torch.cuda.empty_cache()
            out["c5"]["config"]["slot_order"] = "given"
            # the exact running max's cost on the top-k workload
            out["c5_threshold_8"]["exact_max_cost"] = (out["c5"]["ms_per_call"] /
                                                       out["c5_threshold_8"]["ms_per_call"] - 1)
    # the benchmark's workload at the lazy threshold (8 log2 units) instead of
    # the exact running max: the cost of the exact max, which the pages put at
    # about 4 % of the forward on this GPU
    out["c2_threshold_8"] = time_workload(args, dev, dist, world, local, peak, "c2",
                                          workload_problem("c2"), 8.0, traffic=False)
    torch.cuda.empty_cache()
    return out


def backward_workload(args, dev, dist, world, local, peak, dtype="bf16"):
    """fa_bwd on the benchmark's workload (B2 H16 S2048 D128 causal, bf16, or
    the same draws rounded to fp16 with dtype="fp16"),
    after one fa_fwd_o_lo call that provides o, its residual and the LSE, with
    a seeded upstream gradient: K calls between a barrier + synchronize, CUDA
    events around them, clocks sampled from an untimed soak on.  Reported
    against the backward's algorithmic work, 2.5x the forward's (S, dP, dV,
    dQ, dK: 2 D + 4 Dv ... = 1280 flops per unmasked pair at D = Dv = 128)."""
    import numpy as np
    import torch
    import attention_forward_fa_gb300 as fa
    from attention_forward_fa_gb300 import workloads as W
    p = workload_problem("c2") if dtype == "bf16" else W.config(2, dtype=dtype)
    flops = 2.5 * W.algorithmic_flops(p)
    tdt = torch.bfloat16 if p.dtype == "bf16" else torch.float16
    to = lambda bits: torch.from_numpy(bits.view(np.int16).copy()).to(dev).view(tdt)  # noqa: E731
    q, k, v = to(p.q_bits), to(p.k_bits), to(p.v_bits)
    dout = to(W.upstream_grad((p.B, p.Hq, p.Sq, p.Dv), p.dtype, seed=2001))
    causal = p.mask == W.MASK_CAUSAL
    o, lse, o_lo = fa.flash_attention_forward(q, k, v, scale=p.scale, causal=causal, o_lo=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def call():
        fa.flash_attention_backward(q, k, v, o, lse, dout, o_lo=o_lo, scale=p.scale, causal=causal,
                                    dq=dq, dk=dk, dv=dv)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else local)
    sampler.start()
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < args.workload_soak:
        call()
        torch.cuda.synchronize()
    steps = max(3, min(args.workload_steps, 20))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    status = fa.fa_check_status()
    if status != 0:
        raise RuntimeError("device status after the backward: " + fa.fa_strerror(status))
    ms = max_over_ranks(dist, [e0.elapsed_time(e1) / steps], dev)[0]
    achieved = flops / (ms * 1e-3) / 1e12
    cfg = workload_desc(p, "c2")
    cfg["dtype"] = p.dtype
    if p.dtype != "bf16":
        cfg["workload"] = cfg["workload"].replace("bf16", p.dtype)
    cfg["pass"] = "backward: dQ, dK, dV from q, k, v, o + o_lo, LSE and a seeded N(0,1) upstream gradient"
    return {"config": cfg,
            "algorithmic_gflop": flops / 1e9, "ms_per_call": ms,
            "tflops": whole_job_tflops(world, flops, ms), "frac": achieved / peak, "steps": steps,
            "kernel": f"fa_bwd: d_row, then per batch of (KV head, group head) planes cuBLAS {p.dtype} "
                      f"tensor-core GEMMs (fp32 accumulation) for S, dP and, with P and dS as {p.dtype} "
                      "hi + lo pairs, dV, dQ, dK; this library's P, dS and conversion kernels",
            "timing": "eager, events around the K calls", "clocks": clocks}


def run_ours(args, world, rank, local):
    import torch
    import attention_forward_fa_gb300 as fa
    from attention_forward_fa_gb300 import build as fa_build
    from attention_forward_fa_gb300 import workloads as W

    if rank == 0 or world == 1:
        fa_build.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        if rank != 0:
            fa_build.build()  # no-op once rank 0 built it (mtime check)
        dist.barrier()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.backward:
        # the backward entry of the c2 line on its own (a short run to profile)
        peaks, _ = measured_peaks()
        args.workload_steps, args.workload_soak = args.steps, args.soak
        # fp16 tensor-core products run at the bf16 rate: the same peak
        e = backward_workload(args, dev, dist, world, local, float(peaks["bf16_tflops"]),
                              dtype="fp16" if args.fp16 else "bf16")
        if rank == 0:
            print(json.dumps({"metric": "attention bwd TFLOP/s on 1 GB300 (algorithmic) and % of dense "
                                        "BF16 tensor peak; ms/call",
                              "value": e["tflops"], "unit": "TFLOP/s", "n_gpus": world,
                              "steps": e["steps"], "warmup": 3, "ms_per_step": e["ms_per_call"],
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "fp16" if args.fp16 else "bf16", "data": "synthetic",
                              **{k: e[k] for k in e
                                                                      if k not in ("tflops", "steps")}}))
        if dist:
            dist.destroy_process_group()
        return 0
    p = workload_problem(args.workload, args.mla_tokens)
    flops = W.algorithmic_flops(p)
    prep = Prepared(p, dev)
    bf16, dt = prep.bf16, prep.dt
    q0, k0, v0 = prep.q0, prep.k0, prep.v0
    seqlens, blk, tk = prep.seqlens, prep.blk, prep.tk
    sets, n_sets, per_set, conv_pass = prep.sets, prep.n_sets, prep.per_set, prep.conv_pass

    total_ms, kern_avg_ms, conv_avg_ms, clocks, use_graph = timed_steps(
        prep, args.steps, args.warmup, args.soak, dist, local, args.no_graph)
    total_ms, kern_avg_ms = max_over_ranks(dist, [total_ms, kern_avg_ms], dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, flops, ms_per_step)
    stream = torch.cuda.current_stream()

    # end to end through the public entry point with host buffers
    pin = lambda x: x.cpu().pin_memory()  # noqa: E731
    hq, hk = pin(q0), pin(k0)
    hv = None if v0 is None else pin(v0)
    ho = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=dt).pin_memory()
    hl = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32).pin_memory()
    h2d = 2 * (hq.numel() + hk.numel() + (0 if hv is None else hv.numel()))
    d2h = ho.numel() * 2 + hl.numel() * 4
    e2e_mode = p.mask | (fa.FA_V_FROM_K if p.v_from_k else 0) | (0 if bf16 else fa.FA_DTYPE_FP16)

    # Two device input/output sets and three streams (copy in, compute, copy
    # out), so that the upload of step i+1 and the download of step i-1 overlap
    # the kernel of step i; every step still moves its own inputs in and its own
    # result out inside the timed region.
    e2e_sets = [sets[0], sets[1 % len(sets)]]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    s_cmp = stream

    def e2e_run(n):
        done_cmp = [None, None]
        done_out = [None, None]
        for i in range(n):
            dq, dk, dv, _, do, dl = e2e_sets[i & 1]
            with torch.cuda.stream(s_in):
                if done_cmp[i & 1] is not None:
                    s_in.wait_event(done_cmp[i & 1])      # the kernel of step i-2 read this set
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                if hv is not None:
                    dv.copy_(hv, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_cmp.wait_event(ev_in)
            if done_out[i & 1] is not None:
                s_cmp.wait_event(done_out[i & 1])          # step i-2's result was read out
            code = fa.fa_fwd(dq, dk, dv, do, dl, p.B, p.Hq, p.Hkv, p.Sq, p.Skv, p.D, p.Dv, p.scale,
                             e2e_mode, seqlens, blk, tk, 0.0, s_cmp.cuda_stream)
            if code != 0:
                raise RuntimeError(fa.fa_strerror(code))
            ev_c = torch.cuda.Event()
            ev_c.record(s_cmp)
            done_cmp[i & 1] = ev_c
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                ho.copy_(do, non_blocking=True)
                hl.copy_(dl, non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
            done_out[i & 1] = ev_o

    e2e_run(3)
    torch.cuda.synchronize()
    n_e2e = max(3, min(args.steps, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(n_e2e)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    e2e_ms = max_over_ranks(dist, [e2e_ms], dev)[0]
    e2e_value = whole_job_tflops(world, flops, e2e_ms)

    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    # the other workloads, timed after the benchmark line's own region (every
    # rank takes part: their barriers and max over ranks are the same)
    del prep, sets
    others = None
    if args.workload == "c2" and not args.no_workloads:
        others = other_workloads(args, dev, dist, world, local, peak)
        others["bwd_c2"] = backward_workload(args, dev, dist, world, local, peak)
        # the exact running max's cost: this line's time over the lazy threshold's, minus 1
        others["c2_threshold_8"]["exact_max_cost"] = ms_per_step / others["c2_threshold_8"]["ms_per_call"] - 1
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    achieved = flops / (kern_avg_ms * 1e-3) / 1e12
    cfg = workload_desc(p, args.workload)
    cfg.update({"timing": ("CUDA graph of the K steps (captured before the timed region), "
                           "events around its replay" if use_graph else
                           "eager launches, CUDA events around each launch"),
                "parallelism": f"replicas x{world} (no exchange)",
                "l2": f"{n_sets} rotating input/output sets of {per_set / 2**20:.0f} MiB "
                      f"(> 2 x 129 MiB L2), no flush",
                "algorithmic_gflop_per_step": flops / 1e9})
    kernel = kernel_name(p)
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_source": f"{peak_src} bf16_tflops (burst); the fp16 products run at the same "
                           f"nominal rate",
            "traffic": dram_traffic(args.workload), "kernel": kernel,
            "kernel_source_hash": kernel_source_hash("topk" if args.workload == "c5" else "dense"),
            "kernel_avg_ms": kern_avg_ms}
    if conv_pass:
        roof["other_kernel"] = {"name": "fa_convert_v_kernel (bf16 -> fp16 copy of the key latent)",
                                "avg_ms": conv_avg_ms}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if bf16 else "fp16", "data": "synthetic", "config": cfg,
            "pct_of_bf16_peak": 100.0 * achieved / peak, "roofline": roof,
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": (2 if conv_pass else 1) * args.steps}
    if others is not None:
        line["workloads"] = others
    if world == 1 and not args.no_cpu_baseline and args.workload == "c2":
        f, t, n = oracle_timed(p, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": f / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} query rows of the same workload (256-row samples spread over the "
                      f"sequence, rotating heads), fp64 numpy oracle materialising S and P, "
                      f"{t:.1f} s; algorithmic flops of those rows / time"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load before timing")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mla-tokens", type=int, default=4096,
                    help="tokens of the top-k workload (c5); smaller values for profiling captures")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps eagerly with events around each launch")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the entries of the other workloads (c3, c4, c5) in the c2 line")
    ap.add_argument("--workload-steps", type=int, default=100,
                    help="timed steps of each other workload")
    ap.add_argument("--workload-soak", type=float, default=1.0,
                    help="seconds of untimed load before each other workload's timing")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c2",
                    help="c2 (default) is the benchmark line; the others time the same path "
                         "on the other workloads")
    ap.add_argument("--backward", action="store_true",
                    help="time only the backward (fa_bwd) on the c2 workload, its own JSON line")
    ap.add_argument("--fp16", action="store_true",
                    help="with --backward: the same workload's draws rounded to fp16")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
