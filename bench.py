#!/usr/bin/env python
"""Benchmark of the W4A16 fused MoE forward (INT4 weights, group 32, bf16
activations) at the MoE dimensions of the pages' benchmark: E=384 experts,
hidden 7168, intermediate 2048, top-8.

One "step" = one fused forward (align, gather, gate/up GEMM, down GEMM,
finalize) over one batch of seeded synthetic tokens with all 384 experts'
packed weights resident in HBM. The headline line is the decode workload
(M = 1 token, uniform router logits); the M sweep of the pages' table
(1, 9, 32, 90, 256, 512, 1024 uniform and Zipf-skewed) is reported under
"sweep" with each batch's roofline fraction.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); the timed region is bracketed by barriers and
the slowest rank's time is reported. ``--impl reference`` times the CPU oracle
(float64 numpy) on the host cores instead.
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

from int4_weight_only_moe_gb300 import inputs  # noqa: E402

HEADLINE = "decode"
SWEEP = ["decode", "small9", "small32", "small90", "plateau256", "plateau512", "large_uniform",
         "large_zipf"]
METRIC = "MoE tokens/sec and µs/call vs M (1–1024); % HBM / tensor-pipe roofline"
L2_FLUSH_BYTES = 512 << 20
KERNELS = ["align", "gather", "gemm_gateup", "gemm_down", "finalize"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def expert_bytes(K, N, G=32):
    """Packed INT4 codes + bf16 scales of one expert: (gate/up, down)."""
    w1 = 2 * N * K // 2 + 2 * N * (K // G) * 2
    w2 = K * N // 2 + K * (N // G) * 2
    return w1, w2


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value: float, device) -> float:
    """Largest ``value`` over all ranks (the slowest replica sets the time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def file_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


GEMM_SOURCES = ("gemm.cu", "ptx.cuh", "layout.cuh", "kernels.cuh", "small_route.cuh", "stream_k.cuh")
GEMV_SOURCES = ("gemv.cu", "ptx.cuh", "layout.cuh", "kernels.cuh", "small_route.cuh", "stream_k.cuh")


def kernel_sources_hash(files=GEMM_SOURCES):
    """Hash of a kernel's sources (the kernel file and the headers it includes)."""
    csrc = os.path.join(ROOT, "int4_weight_only_moe_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        path = os.path.join(csrc, f)
        if os.path.exists(path):
            h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(record="gemm_gateup_decode_ncu.json", files=GEMM_SOURCES):
    """DRAM bytes per launch of the dominant kernel at the headline workload, from the
    committed ncu record under profiles/, valid only while the kernel's sources are
    unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sources_sha256_16") != kernel_sources_hash(files):
        return None
    v = rec.get("dram_bytes_per_launch_full_size")
    return float(v) if v is not None else None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- GPU arm


class GpuBench:
    def __init__(self, device, experts=None):
        import torch

        import int4_weight_only_moe_gb300 as pkg
        self.torch, self.pkg = torch, pkg
        wl = inputs.WORKLOADS[HEADLINE]
        self.E, self.K, self.N, self.topk = experts or wl.E, wl.K, wl.N, wl.topk
        self.device = device
        q1, s1, q2, s2 = inputs.all_expert_weights(self.E, self.K, self.N)
        self.moe = pkg.MoEW4A16(self.E, self.K, self.N, self.topk)
        d = [torch.from_numpy(a).to(device) for a in (q1, s1.view(np.int16), q2, s2.view(np.int16))]
        self.moe.pack(*d)
        torch.cuda.synchronize()
        del d, q1, s1, q2, s2
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.stream = torch.cuda.current_stream()

    def step_inputs(self, wl, n):
        """Per step: device hidden states and their routing by the library's router
        kernel (outside any timed region)."""
        torch = self.torch
        out = []
        for s in range(n):
            h, logits = inputs.workload_inputs(wl, step=s)
            d_logits = torch.from_numpy(logits).to(self.device)
            if wl.E != self.E:  # a resident expert set smaller than the workload's: route among them
                d_logits = d_logits[:, :self.E].contiguous()
            ids, w = self.moe.route(d_logits)
            out.append((torch.from_numpy(h.view(np.int16)).to(self.device), ids, w))
        return out

    def flush(self):
        self.flush_buf.zero_()

    def time_forward(self, wl, steps, warmup, profile=False, barrier=None, flush=True):
        """Per-step device time (ms) of the forward, L2 flushed before every step
        (unless ``flush`` is false: the hot-L2 number)."""
        torch, pkg = self.torch, self.pkg
        data = self.step_inputs(wl, steps + warmup)
        out = torch.empty((wl.M, self.K), dtype=torch.bfloat16, device=self.device)
        self.moe.ensure_workspace(wl.M)
        pkg.moe_w4a16_set_option(self.moe.handle, pkg.OPT_PROFILE, 1 if profile else 0)
        for i in range(warmup):
            self.moe.forward(*data[i], out=out)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        ktimes = []
        if barrier:
            barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            if flush:
                self.flush()
            ev[i][0].record()
            self.moe.forward(*data[warmup + i], out=out)
            ev[i][1].record()
            if profile:
                ktimes.append(pkg.moe_w4a16_kernel_times(self.moe.handle))
        torch.cuda.synchronize()
        if barrier:
            barrier()
        pkg.moe_w4a16_set_option(self.moe.handle, pkg.OPT_PROFILE, 0)
        status = self.moe.status()
        if status != 0:
            raise RuntimeError(f"device status word {status} after {wl.name}")
        ms = [a.elapsed_time(b) for a, b in ev]
        return ms, ktimes, data

    def time_graph(self, wl, steps, warmup):
        """Per-step device time (ms) of the forward captured once in a CUDA graph and
        replayed, L2 flushed before every replay; each step's inputs are copied into
        the graph's static buffers before the flush, outside the timed region."""
        torch = self.torch
        data = self.step_inputs(wl, steps + warmup)
        static = [t.clone() for t in data[0]]
        out = torch.empty((wl.M, self.K), dtype=torch.bfloat16, device=self.device)
        self.moe.ensure_workspace(wl.M)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                self.moe.forward(*static, out=out)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.moe.forward(*static, out=out)
        for i in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            for dst, src in zip(static, data[warmup + i]):
                dst.copy_(src)
            self.flush()
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        status = self.moe.status()
        if status != 0:
            raise RuntimeError(f"device status word {status} after graph replays of {wl.name}")
        del g
        return [a.elapsed_time(b) for a, b in ev]

    def time_e2e(self, wl, steps, warmup):
        """Same metric through the host-buffer C-ABI call (H2D + forward + D2H)."""
        torch = self.torch
        host = []
        for h, ids, w in self.step_inputs(wl, steps + warmup):
            host.append((h.cpu().pin_memory(), ids.cpu().pin_memory(), w.cpu().pin_memory()))
        out = torch.empty((wl.M, self.K), dtype=torch.int16).pin_memory()
        for i in range(warmup):
            self.moe.forward_host(*host[i], out)
        ms = []
        for i in range(steps):
            self.flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            self.moe.forward_host(*host[warmup + i], out)  # synchronises before returning
            ms.append((time.perf_counter() - t0) * 1e3)
        h2d = wl.M * self.K * 2 + 2 * wl.M * self.topk * 4
        d2h = wl.M * self.K * 2
        return ms, h2d, d2h


def roofline_entry(wl, us, active, hbm_gbs, tc_tflops):
    w1b, w2b = expert_bytes(wl.K, wl.N)
    t_hbm = active * (w1b + w2b) / (hbm_gbs * 1e9) * 1e6
    t_tc = 2.0 * wl.M * wl.topk * 3 * wl.N * wl.K / (tc_tflops * 1e12) * 1e6
    t_star = max(t_hbm, t_tc)
    t_hbm8 = active * (w1b + w2b) / 8e12 * 1e6  # the same roof at 8 TB/s
    return {"M": wl.M, "routing": wl.routing, "active_experts": int(active), "us_per_call": round(us, 2),
            "tok_per_s": round(wl.M / (us * 1e-6), 1), "us_per_token": round(us / wl.M, 3),
            "roofline_us": round(t_star, 2), "binding_roof": "hbm" if t_hbm >= t_tc else "tensor",
            "frac_of_roofline": round(t_star / us, 4),
            "frac_of_roofline_8000_gbs": round(max(t_hbm8, t_tc) / us, 4)}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
        __graft_entry__.build()
    hbm_gbs, tc_tflops, peak_src = peaks()
    # the oracle's worker pool starts before any GPU work (spawned processes)
    cpu_pool = OraclePool() if (not args.no_cpu_baseline and world == 1 and rank == 0) else None
    gb = GpuBench(device)
    wl = inputs.WORKLOADS[HEADLINE]
    barrier = dist.barrier if world > 1 else None

    with ClockSampler(local_rank) as clk:
        ms, _, data = gb.time_forward(wl, args.steps, args.warmup, barrier=barrier)
    total_ms = reduce_max(sum(ms), device)
    ms_step = total_ms / args.steps
    value = world * wl.M * args.steps / (total_ms * 1e-3)

    # kernel breakdown (events between kernels), roofline of the dominant kernel
    _, ktimes, _ = gb.time_forward(wl, args.steps, args.warmup, profile=True)
    kmean = [statistics.mean(k[i] for k in ktimes) for i in range(len(KERNELS))]
    ids_all = np.stack([d[1].cpu().numpy() for d in data[args.warmup:]])
    active = float(np.mean([len(np.unique(x)) for x in ids_all]))
    w1b, w2b = expert_bytes(wl.K, wl.N)
    # The dominant kernel: for M * topk <= 32 both GEMMs run as one launch (its
    # time falls between the events after the gather and after the down GEMM);
    # otherwise the gate/up GEMM. Algorithmic bytes: the routed experts' packed
    # weights and scales, the activation rows read, the intermediate written (and,
    # fused, read back) and the output accumulator.
    fused = False  # (the fused small-batch launch is off by default)
    gemv = wl.M * wl.topk <= 256  # (by default such a batch runs its products on the CUDA cores)
    if fused:
        dom_name = "gemm_fused (gate/up + down, one cooperative launch)"
        dom_bytes = (active * (w1b + w2b) + wl.M * wl.K * 2 + 2 * wl.M * wl.topk * wl.N * 2
                     + wl.M * wl.K * 4 + wl.M * wl.K * 2)
        dom_ms = kmean[2] + kmean[3]
    elif gemv:
        # the CUDA-core gate/up kernel: weights and scales, the activation step rows
        # (288 bytes per row and step: 128 16-bit values and 4 group headers) read,
        # h written twice (step rows for the down kernel, blocked fp16 for read-back)
        dom_name = "gemv_gateup (CUDA cores)"
        dom_bytes = (active * w1b + wl.M * wl.topk * (wl.K // 128) * 288
                     + wl.M * wl.topk * (wl.N * 2 + (wl.N // 128) * 288))
        dom_ms = kmean[2]
    else:
        dom_name = "gemm_gateup"
        dom_bytes = active * w1b + wl.M * wl.K * 2 + wl.M * wl.topk * wl.N * 2
        dom_ms = kmean[2]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    if gemv:
        traffic = recorded_traffic("gemv_gateup_decode_ncu.json", GEMV_SOURCES)
    else:
        traffic = recorded_traffic("gemm_fused_decode_ncu.json" if fused else "gemm_gateup_decode_ncu.json")

    # timing detail of the headline workload: spread, hot L2, graph-captured launches
    hot_ms, _, _ = gb.time_forward(wl, args.steps, args.warmup, flush=False)
    graph_ms = gb.time_graph(wl, args.steps, args.warmup)
    q = np.percentile(np.array(ms) * 1e3, [10, 50, 90])
    timing = {"eager_flushed_us": {"p10": round(q[0], 2), "p50": round(q[1], 2), "p90": round(q[2], 2)},
              "eager_hot_l2_us_p50": round(statistics.median(hot_ms) * 1e3, 2),
              "graph_flushed_us_p50": round(statistics.median(graph_ms) * 1e3, 2)}

    e2e_ms, h2d, d2h = gb.time_e2e(wl, max(3, args.steps), args.warmup)
    e2e_value = wl.M / (statistics.mean(e2e_ms) * 1e-3) * world

    sweep = {}
    if not args.no_sweep:
        for name in SWEEP:
            w = inputs.WORKLOADS[name]
            sms, _, sdata = gb.time_forward(w, args.sweep_steps, 3)
            act = float(np.mean([len(np.unique(d[1].cpu().numpy())) for d in sdata[3:]]))
            sweep[name] = roofline_entry(w, statistics.median(sms) * 1e3, act, hbm_gbs, tc_tflops)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32+f32" if wl.M * wl.topk <= 256 else "f16",
        "dtype_detail": "INT4 weights: at most 256 routed slots (decode) exact int32 dot products of the codes "
                        "with 16-bit block-fixed-point activations (CUDA cores, dp2a), one f32 rounding per "
                        "group of 32; larger batches f16 tensor-core operands, f32 accumulate; bf16 in/out",
        "data": "synthetic (seeded random INT4 weights for all 384 experts, N(0,1) bf16 hidden, "
                "uniform router logits -> top-8 renormalised by the library's router)",
        "config": headline_config(wl, world),
        # for M * topk <= 32 the library runs the routing and the gather as one
        # kernel: 4 launches per forward
        "gpu_launches": (len(KERNELS) - (1 if wl.M * wl.topk <= 32 else 0)) * args.steps,
        "kernel_ms": {k: round(v, 5) for k, v in zip(KERNELS, kmean)},
        "roofline": {"kernel": dom_name, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm_gbs, "unit": "GB/s", "frac": round(achieved / hbm_gbs, 4),
                     "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                     "frac_of_8000_gbs": round(achieved / 8000.0, 4),
                     "algorithmic_bytes_per_launch": int(dom_bytes),
                     "traffic": traffic},
        "whole_forward_roofline": roofline_entry(wl, ms_step * 1e3, active, hbm_gbs, tc_tflops),
        "timing": timing,
        "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(statistics.mean(e2e_ms), 4)},
        "clocks": clk.summary(),
        "sweep": sweep,
    }
    if cpu_pool is not None:
        line["cpu_baseline"] = cpu_baseline(cpu_pool, args.cpu_samples)
        cpu_pool.close()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# --------------------------------------------------------------------------- CPU oracle arm
#
# The oracle (float64 numpy) is timed expert by expert: a call's experts are
# independent, so a pool of worker processes (one BLAS thread each, "spawn" start
# method) runs them concurrently on the host cores. Each worker regenerates the
# seeded inputs and its expert's weights untimed and times only the oracle's
# arithmetic (dequantise, SwiGLU MLP, weighted sum) for the tokens routed to it.

_ROUTED = {}


def _routed(fields, step):
    key = (fields, step)
    if key not in _ROUTED:
        import oracle
        wl = inputs.Workload(*fields)
        hidden, logits = inputs.workload_inputs(wl, step=step)
        ids, w = oracle.route(logits, wl.topk)
        _ROUTED.clear()
        _ROUTED[key] = (hidden, ids, w.astype(np.float32))
    return _ROUTED[key]


def _oracle_expert_seconds(task):
    """Seconds of oracle arithmetic for expert ``e``'s share of one call."""
    import oracle
    fields, step, e = task
    wl = inputs.Workload(*fields)
    hidden, ids, w = _routed(fields, step)
    weights = inputs.expert_weights(int(e), wl.K, wl.N)
    masked = np.where(ids == e, ids, -1).astype(np.int32)
    toks = np.unique(np.nonzero(ids == e)[0])
    t0 = time.perf_counter()
    oracle.moe_forward(hidden, masked, w, None, None, None, None, tokens=toks,
                       expert_source=lambda _e: weights)
    return time.perf_counter() - t0


def _fields(wl):
    return (wl.name, wl.E, wl.K, wl.N, wl.topk, wl.M, wl.routing, wl.zipf_s)


class OraclePool:
    """Worker processes for the oracle, one BLAS thread each."""

    def __init__(self, procs=None):
        import multiprocessing as mp
        self.procs = procs or max(1, min(os.cpu_count() or 1, 16))
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        self.pool = mp.get_context("spawn").Pool(self.procs)

    def close(self):
        self.pool.close()
        self.pool.join()

    def call_seconds(self, wl, step, experts):
        """Per-expert seconds for ``experts`` of ``wl``'s call at ``step``."""
        return self.pool.map(_oracle_expert_seconds, [(_fields(wl), step, int(e)) for e in experts])


def oracle_call(pool, wl, step):
    """Wall seconds of one whole oracle call: its experts run concurrently, so the
    call takes as long as the busiest worker's share (experts dealt round-robin)."""
    import oracle
    _, logits = inputs.workload_inputs(wl, step=step)
    experts = np.unique(oracle.route(logits, wl.topk)[0])
    secs = pool.call_seconds(wl, step, experts)
    loads = [sum(secs[i::pool.procs]) for i in range(pool.procs)]
    return max(loads), len(experts)


def cpu_baseline_sweep(pool, max_experts=16):
    """Oracle throughput for every workload of the sweep on a bounded sample: up to
    ``max_experts`` of a call's routed experts are timed (one per worker); the call's
    time is their mean times its expert count, spread over the pool's workers."""
    import oracle
    out = {}
    for name in SWEEP:
        wl = inputs.WORKLOADS[name]
        _, logits = inputs.workload_inputs(wl)
        experts = np.unique(oracle.route(logits, wl.topk)[0])
        sample = experts[np.linspace(0, len(experts) - 1, min(max_experts, len(experts))).astype(int)]
        secs = pool.call_seconds(wl, 0, sample)
        per_expert = float(np.mean(secs))
        wall = per_expert * -(-len(experts) // pool.procs)
        out[name] = {"M": wl.M, "s_per_call": round(wall, 3), "tok_per_s": round(wl.M / wall, 4),
                     "cpu_s_per_expert": round(per_expert, 4), "active_experts": int(len(experts)),
                     "sampled_experts": int(len(sample))}
    return out


def cpu_baseline(pool, steps):
    """The headline (decode) oracle throughput plus the sweep, on ``pool.procs`` cores."""
    wl = inputs.WORKLOADS[HEADLINE]
    walls = [oracle_call(pool, wl, s)[0] for s in range(steps)]
    return {"value": round(wl.M * steps / sum(walls), 4), "unit": "tokens/s", "cores": pool.procs,
            "kind": "oracle",
            "sample": f"{steps} decode steps (M=1, 8 routed experts each) of the float64 numpy oracle, "
                      f"experts run concurrently on {pool.procs} worker processes with one BLAS "
                      "thread each; input and weight generation untimed. sweep: per workload, up to "
                      "16 routed experts timed and the call extrapolated to all its experts",
            "sweep": cpu_baseline_sweep(pool)}


def headline_config(wl, world):
    return {"workload": "decode: E=384 K=7168 N=2048 top-8 INT4 g32, M=1 token per step",
            "M": wl.M, "E": wl.E, "K": wl.K, "N": wl.N, "topk": wl.topk, "group_size": 32,
            "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB write)",
            "inputs_per_step": "distinct seeded hidden/routing each step",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    wl = inputs.WORKLOADS[HEADLINE]
    pool = OraclePool()
    try:
        for s in range(args.warmup):
            oracle_call(pool, wl, s)
        secs = [oracle_call(pool, wl, args.warmup + s)[0] for s in range(args.steps)]
    finally:
        pool.close()
    total = sum(secs)
    value = wl.M * args.steps / total
    cores = min(pool.procs, 8)  # a decode call has 8 experts: at most 8 workers are busy
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": headline_config(wl, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} decode steps of the float64 numpy oracle (route, "
                                   "dequantise the 8 routed experts, SwiGLU, weighted sum), experts "
                                   "concurrently on worker processes with one BLAS thread each"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A few forwards of one workload for profiler captures (ncu): no timing, no
    extras. ``--experts`` shrinks the resident expert set to keep captures small."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    gb = GpuBench(torch.device("cuda", 0), experts=args.experts)
    wl = inputs.WORKLOADS[args.workload]
    if args.experts:
        from dataclasses import replace
        wl = replace(wl, E=args.experts)
    data = gb.step_inputs(wl, args.warmup + args.steps)
    out = torch.empty((wl.M, gb.K), dtype=torch.bfloat16, device="cuda")
    gb.moe.ensure_workspace(wl.M)
    if args.tensor_cores:  # the tensor-core kernels for every batch size
        import int4_weight_only_moe_gb300 as pkg
        pkg.moe_w4a16_set_option(gb.moe.handle, pkg.OPT_GEMV_SMALL_BATCH, 0)
    for h, ids, w in data:
        gb.flush()
        gb.moe.forward(h, ids, w, out=out)
    torch.cuda.synchronize()
    assert gb.moe.status() == 0
    print(f"profile case {wl.name} E={wl.E} M={wl.M}: {len(data)} forwards", flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-samples", type=int, default=3)
    ap.add_argument("--profile-case", action="store_true",
                    help="only run --warmup + --steps forwards of --workload (for ncu)")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--experts", type=int, default=None,
                    help="resident experts in --profile-case (default: the workload's E)")
    ap.add_argument("--tensor-cores", action="store_true",
                    help="--profile-case: run the products on the tensor cores whatever the batch size")
    args = ap.parse_args(argv)
    if args.profile_case:
        return run_profile_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
