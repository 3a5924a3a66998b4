"""Benchmark of the DeepSeekMoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one moe_layer_forward over T tokens of the chosen workload (default: the 16B-like layer,
T = 16384, d = 2048, 2 shared + 64 routed experts of width 1408, top-6): router, permutation,
gather, gate/up and down expert GEMMs, combine and balance statistics. Inputs are seeded
synthetic tensors of the workload's shape, resident in HBM when the timed region starts. Each
step is timed on its own with CUDA events on the launching stream; L2 is flushed (a 512 MB
write) between steps, outside the timed events. Under torchrun every rank runs its own batch of
T tokens (independent replicas, weak scaling); the reported time is the maximum over ranks.

``--impl reference`` times the fp64 CPU oracle on bounded samples of the same workload instead.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s at 16B-like shape"
UNIT = "tokens/s"


def flops_per_token(sh) -> float:
    """Algorithmic FLOPs per token: router 2*d*N', and three GEMMs of 2*d*I per active expert."""
    return 6.0 * sh.d * sh.inter * (sh.n_shared + sh.top_k) + 2.0 * sh.d * sh.n_routed


def gate_up_flops(sh, T, with_shared=True) -> float:
    """FLOPs of the gate/up GEMM over the routed groups, plus the shared group's when
    with_shared."""
    shared = sh.n_shared if with_shared and not sh.drop_shared else 0
    return 4.0 * sh.d * sh.inter * T * (shared + sh.top_k)


def workload_config(sh, T, world, graph=False) -> dict:
    """The `config` object of a bench line; both arms describe the workload the same way."""
    return {"workload": sh.name, "T": T, "d": sh.d, "n_shared": sh.n_shared,
            "n_routed": sh.n_routed, "inter": sh.inter, "top_k": sh.top_k,
            "global_batch": T * world, "parallelism": f"replicas x{world}",
            "l2": "flushed between timed steps (512 MB write outside the events)",
            "launch": "CUDA graph replay of moe_layer_forward" if graph
                      else "direct moe_layer_forward calls",
            "inputs": "seeded Gaussian tensors of the workload's shape"}


def gate_up_bytes(sh, T, counts, with_shared=True) -> float:
    """Algorithmic DRAM bytes of one gate/up launch: the gate and up weights of every routed
    expert that received a token (and of the shared experts when with_shared), the A rows it
    reads (T K' routed rows and, with the shared experts, the T rows of u) and the activations
    it writes."""
    es = 4 if sh.dtype == "f32" else 2
    shared = sh.n_shared if with_shared and not sh.drop_shared else 0
    touched = int(sum(1 for c in counts if c > 0))
    weights = (shared + touched) * 2 * sh.inter * sh.d * es
    a_rows = T * sh.top_k + (T if shared else 0)
    act = (T * sh.top_k + T * shared) * sh.inter * es
    return float(weights + a_rows * sh.d * es + act)


def gate_up_traffic(workload: str, kernel: str = "gemm_gate_up"):
    """DRAM bytes (read + write) of one gate/up GEMM launch (`kernel`: gemm_gate_up over all
    groups, gemm_gate_up_routed over the routed groups only) from the committed ncu summary, or
    None when the workload was not captured."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic_full_size.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 5 and not line.startswith("#") and parts[0] == workload \
                    and parts[1] == kernel:
                return int(parts[2]) + int(parts[3])
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


def layer_roofline(sh, T, counts, hbm_gbs, bf16_tf) -> dict:
    """Roofline of one layer call: the slower of its algorithmic FLOPs at the bf16 peak and its
    algorithmic bytes at the HBM copy bandwidth. The bytes are the weights it must read (shared
    experts, centroids, and every routed expert that received a token), u in, h out, and the
    routing outputs (indices and gates)."""
    es = 4 if sh.dtype == "f32" else 2
    touched = int(sum(1 for c in counts if c > 0))
    shared = 0 if sh.drop_shared else sh.n_shared
    weights = (shared + touched) * 3 * sh.inter * sh.d * es + sh.n_routed * sh.d * es
    acts = 2 * T * sh.d * es + T * sh.top_k * 8
    flops = flops_per_token(sh) * T
    t_flop = flops / (bf16_tf * 1e12)
    t_bytes = (weights + acts) / (hbm_gbs * 1e9)
    return {"bound": "tensor" if t_flop >= t_bytes else "hbm",
            "roofline_ms": 1e3 * max(t_flop, t_bytes), "flops": flops,
            "bytes": float(weights + acts)}


def rank_token_seed(sh, rank: int) -> int:
    """Each rank draws its own token batch; the expert weights are the same on every rank."""
    return sh.seed + 7919 * rank


def max_over_ranks(values, world: int, device=None):
    """Element-wise maximum over the ranks of the default process group (identity for 1 rank)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ------------------------------------------------------------------------------ clocks ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="moe_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- reference ----

def oracle_sample_rate(sh, n_tokens: int, seed: int = 0):
    """Oracle tokens/s on n_tokens of the workload (each token routed on its own, all its
    experts applied, fp64). Returns (tokens/s, seconds, threads)."""
    import numpy as np

    import oracle
    oracle.build()
    cfg = oracle.OracleCfg.from_shape(sh, T=n_tokens)
    inputs = moe_inputs.make_inputs(sh, T=n_tokens, seed=sh.seed + 1000 + seed)
    t0 = time.perf_counter()
    oracle.forward_tokens(cfg, inputs, np.arange(n_tokens))
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt, oracle.threads()


def run_reference(args, sh, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    n_tok = max(1, int(args.ref_tokens))
    cfg = oracle.OracleCfg.from_shape(sh, T=n_tok)
    inputs = moe_inputs.make_inputs(sh, T=n_tok, seed=sh.seed + 1000)
    toks = np.arange(n_tok)
    for _ in range(args.warmup):
        oracle.forward_tokens(cfg, inputs, toks)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward_tokens(cfg, inputs, toks)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n_tok * args.steps / total
    sample = (f"{n_tok} tokens of the {sh.name} workload per step (per-token routing over "
              f"{sh.n_routed} experts + {sh.n_shared + sh.top_k} SwiGLU experts, fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(sh, sh.T, world, graph=False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------------------- ours ----

def run_ours(args, sh, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import fine_grained_moe_softmax_b300 as moe

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T = sh.T
    inputs = moe_inputs.make_inputs(sh, seed=rank_token_seed(sh, rank))
    cfg = moe.MoEConfig.from_shape(sh)
    layer = moe.MoELayer(cfg, inputs["centroids"], inputs["w_gate"], inputs["w_up"],
                         inputs["w_down"], inputs["bias"], device=dev)
    u_host = inputs["u"].pin_memory()
    u = u_host.to(dev)
    del inputs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        layer.forward(u)
    torch.cuda.synchronize(dev)
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {moe.moe_status_string(status)} after warm-up")
    graph, graph_kernels = (layer.capture(u) if args.graph else (None, 0))
    if graph is not None:
        for _ in range(max(args.warmup, 3)):
            graph.replay()
        torch.cuda.synchronize(dev)

    def step():
        if graph is not None:
            graph.replay()
        else:
            layer.forward(u)

    # ---- device-resident timing: every step timed on its own, L2 flushed in between ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if graph is None:
        moe.moe_profile_enable(True, args.steps)
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = moe.moe_launch_count()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    launches = moe.moe_launch_count() - launches0 + graph_kernels * args.steps
    if graph is not None:   # stage times come from a separate profiled pass of direct calls
        moe.moe_profile_enable(True, args.steps)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            layer.forward(u)
        torch.cuda.synchronize(dev)
    stage_ms, n_prof = moe.moe_profile_read()
    gu_launch_ms, _, n_split = moe.moe_profile_read_gate_up()
    moe.moe_profile_enable(False)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)

    # ---- end to end through host buffers. Every step copies its T tokens in from pinned host
    # memory, runs the layer call and copies h and the two losses out to pinned host memory. The
    # copies run on their own streams with double-buffered device buffers, so step i's input copy
    # and step i-1's output copy overlap the layer calls; the timed region spans the first input
    # copy to the last output copy. ----
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    u_devs = [torch.empty_like(u) for _ in range(2)]
    h_devs = [torch.empty(T, sh.d, dtype=u.dtype, device=dev) for _ in range(2)]
    loss_devs = [torch.empty(2, dtype=torch.float32, device=dev) for _ in range(2)]
    h_hosts = [torch.empty(T, sh.d, dtype=u.dtype).pin_memory() for _ in range(2)]
    loss_hosts = [torch.empty(2, dtype=torch.float32).pin_memory() for _ in range(2)]

    def e2e_run(n_steps):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        copied = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(h2d)
        for i in range(n_steps):
            b = i % 2
            if i >= 2:
                h2d.wait_event(done[b])        # step i-2 has finished reading u_devs[b]
            with torch.cuda.stream(h2d):
                u_devs[b].copy_(u_host, non_blocking=True)
                in_ready[b].record(h2d)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(copied[b])   # step i-2's outputs have left h_devs[b]
            layer.forward(u_devs[b], h=h_devs[b], stream=stream)
            loss_devs[b].copy_(layer.losses)
            done[b].record(stream)
            d2h.wait_event(done[b])
            with torch.cuda.stream(d2h):
                h_hosts[b].copy_(h_devs[b], non_blocking=True)
                loss_hosts[b].copy_(loss_devs[b], non_blocking=True)
                copied[b].record(d2h)
        t1.record(d2h)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    e2e_run(max(args.warmup, 3))
    barrier()
    e2e_ms = e2e_run(args.steps)
    barrier()
    clk = clocks.stop()
    status = layer.device_status()
    if status != 0:
        raise RuntimeError(f"device status {moe.moe_status_string(status)} after timing")

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world, dev)
    if rank != 0:
        return

    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = load_peaks()
    counts_host = layer.counts.cpu().tolist()
    tokens = T * world * args.steps
    value = tokens / (total_ms / 1e3)
    e2e_value = tokens / (e2e_ms / 1e3)
    roof = dominant_roofline(sh, T, counts_host, gu_launch_ms, n_prof, n_split)
    layer_tflops = flops_per_token(sh) * T / (total_ms / args.steps / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": sh.dtype, "data": "synthetic",
        "config": workload_config(sh, T, world, graph=graph is not None),
        "roofline": roof,
        "layer_roofline": {"achieved_tflops": layer_tflops, "frac_of_bf16_peak":
                           layer_tflops / bf16_tf, "flops_per_token": flops_per_token(sh)},
        "stage_ms_per_step": {k: v / max(n_prof, 1) for k, v in stage_ms.items()},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * sh.d * u.element_size(),
                "d2h_bytes_per_step": T * sh.d * u.element_size() + 8,
                "copies": "pinned host buffers; input and output copies on their own streams, "
                          "overlapping the neighbouring steps' layer calls"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    lr = layer_roofline(sh, T, counts_host, hbm_gbs, bf16_tf)
    line["layer_roofline"].update({"bound": lr["bound"], "roofline_ms": lr["roofline_ms"],
                                   "frac": lr["roofline_ms"] / (total_ms / args.steps)})
    if world == 1 and not args.no_per_config and args.tokens is None and not args.graph \
            and sh.name == "16b_bf16":
        del layer, graph, flush
        torch.cuda.empty_cache()
        pc_clocks = ClockSampler(local_rank)
        pc_clocks.start()
        time.sleep(0.3)
        runs = [measure_workload(name, g, args.per_config_steps, 3, dev) for name, g in PER_CONFIG]
        line["per_config"] = {"runs": runs, "clocks": pc_clocks.stop()}
    if world == 1 and not args.no_cpu_baseline:
        n = args.cpu_tokens
        rate, secs, threads = oracle_sample_rate(sh, n)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"{n} tokens of the {sh.name} workload, fp64 oracle, "
                                          f"{secs:.1f} s"}
    print(json.dumps(line), flush=True)


def dominant_roofline(sh, T, counts, gu_launch_ms, n_prof, n_split) -> dict:
    """`roofline` of the dominant launch, the gate/up GEMM over the routed groups (over every
    group when the shared group was not split off into a launch of its own), from its summed
    CUDA-event time over n_prof profiled calls. Bound: whichever of its FLOPs at the bf16 peak
    and its algorithmic bytes at the HBM copy bandwidth takes longer."""
    hbm_gbs, bf16_tf, _, peak_src = load_peaks()
    split = n_split > 0
    if n_split not in (0, n_prof):
        raise RuntimeError(f"{n_split} of {n_prof} profiled calls split the gate/up GEMM")
    kname = "gemm_gate_up_routed" if split else "gemm_gate_up"
    traffic = gate_up_traffic(sh.name, kname)
    gu_ms = gu_launch_ms / max(n_prof, 1)
    gu_flops = gate_up_flops(sh, T, with_shared=not split)
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12
    gu_bytes = gate_up_bytes(sh, T, counts, with_shared=not split)
    hbm_bound = gu_bytes / (hbm_gbs * 1e9) > gu_flops / (bf16_tf * 1e12)
    gu_gbs = gu_bytes / (gu_ms / 1e3) / 1e9
    kernel = "gemm_tc_kernel (gate/up + SwiGLU epilogue, " + \
        ("routed groups; the shared group runs in a launch of its own)" if split else "all groups)")
    if hbm_bound:
        roof = {"bound": "hbm", "kernel": kernel,
                "achieved": gu_gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gu_gbs / hbm_gbs,
                "traffic": traffic, "peak_source": f"{peak_src} HBM copy",
                "algorithmic_bytes": gu_bytes}
    else:
        roof = {"bound": "tensor", "kernel": kernel,
                "achieved": gu_tflops, "peak": bf16_tf, "unit": "TFLOP/s",
                "frac": gu_tflops / bf16_tf, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 burst"}
    roof["traffic_source"] = (
        "profiles/gemm_traffic_full_size.txt: dram__bytes_read.sum + dram__bytes_write.sum of "
        f"this launch ({kname}) from an earlier one-pass ncu capture at full size, not this run"
        if traffic is not None else "not captured for this workload")
    roof["launch_ms"] = gu_ms
    return roof


# Workloads timed beside the headline in the default run: (name, CUDA-graph replay).
PER_CONFIG = [("2b_bf16", False), ("145b_zipf_bf16", False), ("16b_decode_bf16", False),
              ("16b_decode_bf16", True), ("2b_half_activated_bf16", False),
              ("2b_gshard_top2_bf16", False)]


def measure_workload(name, graph, steps, warmup, dev) -> dict:
    """ms per layer call of one more workload on this GPU (L2 flushed between steps, CUDA events
    on the launching stream), its layer roofline fraction and its dominant launch's fraction."""
    import torch

    import fine_grained_moe_softmax_b300 as moe
    sh = moe_inputs.CONFIGS[name]
    T = sh.T
    inputs = moe_inputs.make_inputs(sh)
    layer = moe.MoELayer(moe.MoEConfig.from_shape(sh), inputs["centroids"], inputs["w_gate"],
                         inputs["w_up"], inputs["w_down"], inputs["bias"], device=dev)
    u = inputs["u"].to(dev)
    del inputs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        layer.forward(u)
    torch.cuda.synchronize(dev)
    if layer.device_status() != 0:
        raise RuntimeError(f"{name}: device status after warm-up")
    g = layer.capture(u)[0] if graph else None
    if g is not None:
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        if g is not None:
            g.replay()
        else:
            layer.forward(u)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    moe.moe_profile_enable(True, steps)
    for i in range(steps):
        flush.fill_(i & 0xFF)
        layer.forward(u)
    torch.cuda.synchronize(dev)
    stage_ms, n_prof = moe.moe_profile_read()
    gu_launch_ms, _, n_split = moe.moe_profile_read_gate_up()
    moe.moe_profile_enable(False)
    if layer.device_status() != 0:
        raise RuntimeError(f"{name}: device status after timing")
    counts = layer.counts.cpu().tolist()
    hbm_gbs, bf16_tf, _, _ = load_peaks()
    lr = layer_roofline(sh, T, counts, hbm_gbs, bf16_tf)
    out = {"workload": name, "T": T,
           "launch": "CUDA graph replay of moe_layer_forward" if graph
                     else "direct moe_layer_forward calls",
           "steps": steps, "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
           "layer_roofline": {"bound": lr["bound"], "roofline_ms": lr["roofline_ms"],
                              "frac": lr["roofline_ms"] / ms},
           "dominant_launch": dominant_roofline(sh, T, counts, gu_launch_ms, n_prof, n_split),
           "stage_ms_per_step (direct calls)": {k: v / max(n_prof, 1)
                                                for k, v in stage_ms.items()}}
    del layer, g, flush, u
    torch.cuda.empty_cache()
    return out


def backward_flops_per_token(sh) -> float:
    """GEMM FLOPs one moe_layer_backward call executes per token: the forward it recomputes
    (router 2 d N', gate/up 4 d I (Ks+K'), routed down 2 d I K') and the gradients (router 2 x
    2 d N', input gradients 6 d I (Ks+K'), weight gradients 6 d I (Ks+K'))."""
    A = sh.n_shared + sh.top_k
    return (2.0 * sh.d * sh.n_routed * 3 + 4.0 * sh.d * sh.inter * A + 2.0 * sh.d * sh.inter *
            sh.top_k + 12.0 * sh.d * sh.inter * A)


def run_backward(args, sh):
    """Times moe_layer_backward (gradients of sum dh.h + the balance losses), or with --train a
    training step: moe_layer_forward_train then moe_layer_backward_saved; one JSON line."""
    import torch

    import fine_grained_moe_softmax_b300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inputs = moe_inputs.make_inputs(sh)
    layer = moe.MoELayer(moe.MoEConfig.from_shape(sh), inputs["centroids"], inputs["w_gate"],
                         inputs["w_up"], inputs["w_down"], inputs["bias"], device=dev,
                         backward=True)
    u = inputs["u"].to(dev)
    g = torch.Generator().manual_seed(sh.seed + 5)
    dh = torch.randn(sh.T, sh.d, generator=g).to(torch.bfloat16).to(dev)
    del inputs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    train = bool(getattr(args, "train", False))

    def step():
        if train:
            layer.forward_train(u)
            layer.backward_saved(u, dh)
        else:
            layer.backward(u, dh)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    n0 = moe.moe_launch_count()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    launches = moe.moe_launch_count() - n0
    clk = clocks.stop()
    if moe.moe_device_status(layer.ws_bwd) != 0:
        raise RuntimeError("device status after the backward")
    total_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    _, bf16_tf, _, peak_src = load_peaks()
    # a training step executes the forward (router, gate/up, down of routed and shared rows) and
    # the gradients; the recomputing backward executes the same minus the shared down GEMM
    fpt = backward_flops_per_token(sh) + (2.0 * sh.d * sh.inter * sh.n_shared if train else 0.0)
    tflops = fpt * sh.T / (total_ms / args.steps / 1e3) / 1e12
    metric = ("MoE-layer training step tokens/s (forward keeping its state, then all gradients)"
              if train else
              "MoE-layer backward tokens/s (gradients of u, centroids, bias, all experts)")
    note = ("moe_layer_forward_train + moe_layer_backward_saved per step" if train else
            "one call recomputes the forward it needs")
    print(json.dumps({
        "metric": metric,
        "value": sh.T * args.steps / (total_ms / 1e3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "dtype": sh.dtype, "data": "synthetic",
        "config": {"workload": sh.name, "T": sh.T, "d": sh.d, "n_shared": sh.n_shared,
                   "n_routed": sh.n_routed, "inter": sh.inter, "top_k": sh.top_k,
                   "note": note},
        "executed_tflops": tflops, "frac_of_bf16_peak": tflops / bf16_tf,
        "peak_source": f"{peak_src} bf16 burst", "gpu_launches": launches, "clocks": clk}),
        flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="16b_bf16", choices=sorted(moe_inputs.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=4096)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--train", action="store_true",
                    help="time a training step: forward keeping its state, then the gradients")
    ap.add_argument("--backward", action="store_true",
                    help="time the layer backward instead of the forward (1 GPU)")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of the layer call instead of direct calls")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads timed beside the 16B-like headline")
    ap.add_argument("--per-config-steps", type=int, default=10)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (small profiling captures only; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    sh = moe_inputs.CONFIGS[args.config]
    if args.tokens is not None:
        sh = sh.with_(T=args.tokens, name=f"{sh.name}_T{args.tokens}")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    try:
        if args.backward or args.train:
            run_backward(args, sh)
        elif args.impl == "reference":
            run_reference(args, sh, rank, world)
        else:
            run_ours(args, sh, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
