#!/usr/bin/env python3
"""Benchmark of the routed MoE layer on GB300: MoE-layer tokens/s.

Default workload: one qwen3_moe-geometry MoE layer at decode, T = 1 token
(d_model 2048, d_ff 768, 128 experts, top-8, Q8_0 SwiGLU experts, fp32
activations).  One step = one full layer forward (router, top-k, bucketing,
gate/up, down + combine) through the C ABI, replayed from a CUDA graph.
Steps rotate over R independently seeded layers (each with its own x), so the
40 MB of expert weights a step touches are not L2-resident: the reuse
distance is R-1 layers x 40 MB, far above the 129 MB L2.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle
instead (the plain fp64 definition of the layer, on this host's cores).

Multi-GPU: the layer has no exchange step at this scale, so N GPUs run N
independent replicas (weak scaling); timing is barrier-bracketed and the
max over ranks is taken.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_mixture_experts_router_gb300 import binding, synth  # noqa: E402

def row_bytes(wl, K: int) -> int:
    """HBM bytes of one weight row of K values: per 32, 32 int8 (Q8_0) or 16
    bytes of nibbles (Q4_0), plus one fp16 scale."""
    return (K // 32) * (18 if wl.wfmt == "q4" else 34)


NEAR_TIE = 1e-5  # adjacent top-(k+1) logit gap (fp64) below which a token's selection is a near-tie


def near_tie_tokens(x: torch.Tensor, Wr: torch.Tensor, bias, k: int) -> int:
    """Tokens whose fp64 router logits have an adjacent gap < NEAR_TIE among
    their k+1 largest: the tokens whose selection fp32 rounding may decide."""
    lg = x.double().cpu().numpy() @ Wr.double().cpu().numpy().T
    if bias is not None:
        lg = lg + bias.double().cpu().numpy()[None, :]
    s = -np.sort(-lg, axis=1)[:, :k + 1]
    return int(((s[:, :-1] - s[:, 1:]) < NEAR_TIE).any(axis=1).sum()) if s.shape[1] > 1 else 0


def expert_bytes(wl) -> int:
    """HBM bytes of one expert's three quantised matrices (values + scales)."""
    return 2 * wl.d_ff * row_bytes(wl, wl.d_model) + wl.d_model * row_bytes(wl, wl.d_ff)


def wfmt_of(wl) -> int:
    return binding.MOE_WFMT_Q4_0 if wl.wfmt == "q4" else binding.MOE_WFMT_Q8_0


def fmt_name(wl) -> str:
    return "Q4_0" if wl.wfmt == "q4" else "Q8_0"


# ------------------------------------------------------------------ dist ----
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(steps: int, units_per_step: int, ws: int, max_ms: float) -> float:
    """Whole-job throughput: units every rank processed / the slowest rank's time."""
    return steps * units_per_step * ws / (max_ms / 1e3)


def max_over_ranks(v: float, ws: int, device) -> float:
    """Max of a host float over all ranks (timing only, not a data path)."""
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is under load."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [p for (t, p) in self.rows if t0 <= t <= t1] or [p for (_, p) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


def cpu_info():
    """(CPU model, logical cores).  x86 /proc/cpuinfo has "model name"; Arm
    (e.g. NVIDIA Grace) has only implementer / part codes there, so lscpu's
    "Model name" is tried first, then the Arm codes are named."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    impl = part = None
    try:
        for ln in open("/proc/cpuinfo"):
            key = ln.split(":", 1)[0].strip().lower()
            if model is None and key in ("model name", "cpu model"):
                model = ln.split(":", 1)[1].strip()
            elif key == "cpu implementer" and impl is None:
                impl = ln.split(":", 1)[1].strip()
            elif key == "cpu part" and part is None:
                part = ln.split(":", 1)[1].strip()
    except OSError:
        pass
    arm_parts = {("0x41", "0xd4f"): "Arm Neoverse V2 (NVIDIA Grace)", ("0x41", "0xd40"): "Arm Neoverse V1",
                 ("0x41", "0xd0c"): "Arm Neoverse N1"}
    if impl is not None and part is not None:
        named = arm_parts.get((impl.lower(), part.lower()), f"Arm CPU implementer {impl} part {part}")
        if model is None or model.lower() in ("-", "unknown"):
            model = named
        elif named not in model:
            model = f"{model} ({named})"
    return model or "unknown", os.cpu_count()


# ----------------------------------------------------------- CPU oracle ----
def oracle_tokens_per_s(wl, layer_host, x_all: np.ndarray, budget_s: float = 12.0, max_s: float = 30.0):
    """Time the fp64 oracle (as it stands) on batches of independent tokens of
    the workload until ~budget_s of CPU work; returns (tokens/s, tokens, threads)."""
    import oracle
    orc = oracle.get()
    threads = orc.num_threads()
    batch = max(1, threads) * min(max(1, wl.T), 4)
    done, t_used = 0, 0.0
    i = 0
    while t_used < budget_s:
        rows = np.arange(i, i + batch) % x_all.shape[0]
        xb = x_all[rows]
        t0 = time.perf_counter()
        orc.moe_layer(xb, layer_host["Wr"], layer_host["bias"], layer_host["gate"], layer_host["up"],
                      layer_host["down"], wl.d_model, wl.d_ff, wl.E, wl.k, residual=wl.residual,
                      fmt=wfmt_of(wl))
        t_used += time.perf_counter() - t0
        done += batch
        i += batch
        if t_used > max_s:
            break
    return done / t_used, done, threads, t_used


# ------------------------------------------------------------ reference ----
def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[args.workload or "decode_t1"]
    w = synth.make_layer(wl, 0, "cpu")
    host = {k: (None if v is None else v.numpy()) for k, v in w.items()}
    import oracle
    orc = oracle.get()
    threads = orc.num_threads()
    per_step = max(1, threads)           # independent decode tokens per step, one per core
    xs = synth.make_x(wl, "cpu", step=0, T=per_step * (args.steps + args.warmup)).double().numpy()

    def step(i):
        xb = xs[i * per_step:(i + 1) * per_step]
        orc.moe_layer(xb, host["Wr"], host["bias"], host["gate"], host["up"], host["down"], wl.d_model, wl.d_ff,
                      wl.E, wl.k, residual=wl.residual, fmt=wfmt_of(wl))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    tokens = args.steps * per_step
    value = tokens / dt
    model, ncpu = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, qwen3_moe geometry)",
        "config": workload_config(wl, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} steps x {per_step} independent T=1 tokens, layer 0, "
                                   f"{model}, {ncpu} host cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "MoE-layer tokens/s (decode T=1/64, prefill T=1024); HBM GB/s & TC % of peak"


def _cudart():
    """The CUDA runtime already loaded by torch (for graph introspection)."""
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def new_graph():
    try:
        return torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        return torch.cuda.CUDAGraph()


def graph_kernel_nodes(g):
    """Kernel nodes in a captured step graph (every kernel in it is one of ours), or None."""
    try:
        raw = ctypes.c_void_p(int(g.raw_cuda_graph()))
    except Exception:
        return None
    rt = _cudart()
    if rt is None:
        return None
    n = ctypes.c_size_t(0)
    if rt.cudaGraphGetNodes(raw, None, ctypes.byref(n)) != 0:
        return None
    nodes = (ctypes.c_void_p * n.value)()
    if rt.cudaGraphGetNodes(raw, nodes, ctypes.byref(n)) != 0:
        return None
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        if rt.cudaGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0:
            return None
        kernels += t.value == 0  # cudaGraphNodeTypeKernel
    return kernels



def workload_config(wl, args, rot=None):
    rot = args.rot if rot is None else rot
    mb = f" as {wl.T // wl.microbatch} microbatches of {wl.microbatch} tokens (one layer call each)" \
        if wl.microbatch else ""
    return {"workload": f"{wl.name}: one MoE layer, T={wl.T}{mb}, d_model={wl.d_model}, d_ff={wl.d_ff}, E={wl.E}, "
                        f"top-{wl.k}, {fmt_name(wl)} SwiGLU experts, {wl.act} expert inputs"
                        f"{', Zipf router bias' if wl.zipf else ''}",
            "tokens_per_step": wl.T, "layers_rotated": rot,
            "l2": f"inputs larger than L2: steps rotate over {rot} seeded layers "
                  f"({rot} x {wl.E} experts x {expert_bytes(wl)} B resident)",
            "parallelism": f"replicas x{args.gpus}",
            "graph": "the layer forward captured as a CUDA graph per step; the K steps timed as one graph launch "
                     f"per step and as one launch per {rot} rotating steps (K mod {rot} steps as single graphs), "
                     "the faster reported (timed_loop)"}


def expert_path_name(wl, tc_path: bool) -> str:
    if tc_path:
        return f"moe_expert_ffn_q8 (tcgen05 gate/up + down, {fmt_name(wl)} dequant fused, combine fused)"
    return f"moe_expert_ffn_q8 (gate/up + down, {fmt_name(wl)} fused, combine fused)"


def time_loops(stream, graphs, g_all, steps: int):
    """The K steps timed two ways on `stream`: one graph launch per step, and
    (when there is a rotation graph) one launch per rotation with the K mod R
    leftover steps as single graphs.  Returns {name: ms}."""
    R = len(graphs)
    loops = {}
    names = ["per_step_graphs"] + (["one_graph_per_rotation"] if g_all is not None and steps >= R else [])
    for name in names:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if name == "one_graph_per_rotation":
            for _ in range(steps // R):
                g_all.replay()
            for i in range(steps - (steps // R) * R):
                graphs[i].replay()
        else:
            for i in range(steps):
                graphs[i % R].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        loops[name] = e0.elapsed_time(e1)
    return loops


# ------------------------------------------------------------------ ours ----
def measure_layer(wl, args, ws, rank, dev, sampler, rot: int, steps: int, warmup: int, cpu_budget: float,
                  e2e_variants: bool = False):
    """One MoE layer per step (T tokens, or T / microbatch layer calls), the
    steps rotating over `rot` seeded layers.  Returns the bench record."""
    act = binding.MOE_ACT_BF16 if wl.act == "bf16" else binding.MOE_ACT_F32
    mb = wl.microbatch or wl.T
    tc_path = act == binding.MOE_ACT_BF16 and mb * wl.k >= 128
    R = rot
    layers, xs, outs, wss = [], [], [], []
    host0 = None
    near = 0
    for r in range(R):
        w = synth.make_layer(wl, r, dev)
        if r == 0 and rank == 0 and ws == 1 and cpu_budget > 0:
            host0 = {k: (None if v is None else v.cpu().numpy()) for k, v in w.items()}
        layers.append(binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"],
                                                w["Wr"], w["bias"], wfmt=wfmt_of(wl)))
        xs.append(synth.make_x(wl, dev, step=r))
        near += near_tie_tokens(xs[-1], w["Wr"], w["bias"], wl.k)
        del w
        outs.append(torch.empty(wl.T, wl.d_model, dtype=torch.float32, device=dev))
        wss.append(binding.workspace(mb, layers[-1], act, 0, dev))
    torch.cuda.synchronize()
    P = mb * wl.k
    nmb = wl.T // mb
    # split buffers for the per-kernel (expert FFN) timing pass, first microbatch
    idxs = [torch.empty(mb, wl.k, dtype=torch.int32, device=dev) for _ in range(R)]
    wtss = [torch.empty(mb, wl.k, dtype=torch.float32, device=dev) for _ in range(R)]
    offs = [torch.empty(wl.E + 1, dtype=torch.int32, device=dev) for _ in range(R)]
    pts = [torch.empty(P, dtype=torch.int32, device=dev) for _ in range(R)]
    pss = [torch.empty(P, dtype=torch.int32, device=dev) for _ in range(R)]
    poss = [torch.empty(P, dtype=torch.int32, device=dev) for _ in range(R)]
    outs2 = [torch.empty(mb, wl.d_model, dtype=torch.float32, device=dev) for _ in range(R)]

    stream = torch.cuda.Stream(device=dev)
    L = binding.load()
    st = lambda: torch.cuda.current_stream().cuda_stream  # noqa: E731

    def step_call(r, x=None):
        x = xs[r] if x is None else x
        for m in range(nmb):
            binding.layer_forward(x[m * mb:(m + 1) * mb], layers[r], act, 0, wl.residual,
                                  out=outs[r][m * mb:(m + 1) * mb], ws=wss[r])

    def rb_call(r):
        binding._check("moe_route", L.moe_route(binding._ptr(xs[r]), mb, layers[r].ref(), binding._ptr(idxs[r]),
                                                binding._ptr(wtss[r]), binding.ctypes.c_void_p(st())))
        binding._check("moe_bucket", L.moe_bucket(binding._ptr(idxs[r]), mb, wl.k, wl.E, binding._ptr(offs[r]),
                                                  binding._ptr(pts[r]), binding._ptr(pss[r]), binding._ptr(poss[r]),
                                                  None, binding.ctypes.c_void_p(st())))

    def ffn_call(r):
        binding.expert_ffn_q8(xs[r][:mb], layers[r], offs[r], pts[r], pss[r], wtss[r], act, True, wl.residual,
                              ws=wss[r], out=outs2[r])

    # eager warm-up (also sets kernel attributes outside capture), then capture
    with torch.cuda.stream(stream):
        for r in range(R):
            step_call(r)
            rb_call(r)
            ffn_call(r)
    torch.cuda.synchronize()
    g_step, g_rb, g_ffn = [], [], []
    for r in range(R):
        for lst, fn in ((g_step, step_call), (g_rb, rb_call), (g_ffn, ffn_call)):
            g = new_graph()
            with torch.cuda.graph(g, stream=stream):
                fn(r)
            lst.append(g)
    torch.cuda.synchronize()
    g_all = new_graph()
    with torch.cuda.graph(g_all, stream=stream):
        for r in range(R):
            step_call(r)
    torch.cuda.synchronize()

    per_step = [graph_kernel_nodes(g) for g in g_step]
    if all(v is not None for v in per_step):
        launches = int(sum(per_step[i % R] for i in range(steps)))
        launches_src = "kernel nodes of the captured step graphs"
    else:
        launches, launches_src = None, "graph introspection unavailable"

    # distinct experts per rotation slot and microbatch (for the algorithmic bytes)
    xbytes = wl.T * wl.d_model * 4
    n_active = [int((np.diff(offs[r].cpu().numpy()) > 0).sum()) for r in range(R)]
    ffn_bytes = [n * expert_bytes(wl) + 2 * mb * wl.d_model * 4 for n in n_active]  # weights + x in + out
    step_bytes = [nmb * (b + wl.E * wl.d_model * 4 + (wl.E * 4 if wl.zipf else 0)) for b in ffn_bytes]

    with torch.cuda.stream(stream):
        for i in range(warmup):
            g_step[i % R].replay()
        g_all.replay()  # the rotation graph's first launch (upload) stays out of the timed loop
        torch.cuda.synchronize()
        t_soak = time.time()
        i = 0
        while time.time() - t_soak < args.soak:
            for _ in range(20):
                g_step[i % R].replay()
                i += 1
            torch.cuda.synchronize()
        t_clk0 = time.time()
        barrier(ws)
        torch.cuda.synchronize()
        loops = time_loops(stream, g_step, g_all, steps)
        barrier(ws)
        t_clk1 = time.time()
    timing = min(loops, key=loops.get)
    ms_local = loops[timing]
    clocks = sampler.summary(t_clk0 - 0.5, t_clk1 + 0.05)
    ms = max_over_ranks(ms_local, ws, dev)
    value = job_rate(steps, wl.T, ws, ms)

    # One kernel node per step means the whole layer ran as the fused
    # single-launch decode kernel: that kernel is the roofline subject, timed
    # over the timed loop (each step: the kernel and the memset before it).
    fused_step = per_step[0] is not None and all(v == 1 for v in per_step) and nmb == 1

    # per-kernel pass: events around the expert FFN (gate/up + down) on the launch stream
    with torch.cuda.stream(stream):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            r = i % R
            evs[i][2].record(stream)
            g_rb[r].replay()
            evs[i][0].record(stream)
            g_ffn[r].replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    ffn_ms_mean = float(np.mean([a.elapsed_time(b) for a, b, _ in evs]))
    rb_ms = float(np.mean([c.elapsed_time(a) for a, _, c in evs]))
    ffn_alg = float(np.mean([ffn_bytes[i % R] for i in range(steps)]))
    peaks = load_peaks()
    achieved = ffn_alg / (ffn_ms_mean / 1e3) / 1e9
    flops = 2.0 * mb * wl.k * 3 * wl.d_model * wl.d_ff            # expert contractions per FFN call
    roofline = {"kernel": expert_path_name(wl, tc_path),
                "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": ffn_alg, "launch_ms": ffn_ms_mean,
                "launch_ms_note": f"CUDA events around the expert FFN call on its stream, mean of {steps}"
                                  + (f" (first microbatch of {mb} tokens)" if nmb > 1 else ""),
                "traffic": load_traffic(f"moe_expert_ffn_q8 {wl.name}")}
    if fused_step:
        fused_ms = ms_local / steps
        step_alg0 = float(np.mean([step_bytes[i % R] for i in range(steps)]))
        fa = step_alg0 / (fused_ms / 1e3) / 1e9
        kname = "decode_split_kernel"
        roofline = {"kernel": f"{kname} (whole layer: router, top-k, bucketing, {fmt_name(wl)} "
                              "gate/up + down, combine; one cooperative launch)",
                    "bound": "hbm", "achieved": fa, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": fa / peaks["hbm_gbs"], "peak_source": peaks["source"],
                    "algorithmic_bytes_per_launch": step_alg0, "launch_ms": fused_ms,
                    "launch_ms_note": "per step of the timed loop (CUDA events on the launch stream): the step "
                                      "graph's kernel node" + (" and the memset of its barrier words"
                                                               if kname == "decode_fused_kernel" else ""),
                    "traffic": load_traffic(f"{kname} {wl.name}"),
                    "expert_ffn_three_kernel_path": {"achieved": achieved, "frac": achieved / peaks["hbm_gbs"],
                                                     "launch_ms": ffn_ms_mean}}
    if tc_path:
        tf = flops / (ffn_ms_mean / 1e3) / 1e12
        roofline["tensor"] = {"achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                              "frac": tf / peaks["bf16_tflops"], "flops_per_launch": flops,
                              "note": "arithmetic intensity below the bf16 ridge: HBM binds"}
    step_alg = float(np.mean([step_bytes[i % R] for i in range(steps)]))
    layer_gbs = step_alg / (ms_local / steps / 1e3) / 1e9

    # end to end through the C ABI: every step copies x in from pinned host
    # memory on the layer's stream, runs the layer and copies out back, in
    # that order on one stream (the fixed protocol reported as e2e.value)
    xh = [x.cpu().pin_memory() for x in xs]
    oh = torch.empty(wl.T, wl.d_model, dtype=torch.float32).pin_memory()

    def e2e_serial() -> float:
        with torch.cuda.stream(stream):
            for i in range(min(warmup, 10)):
                xs[i % R].copy_(xh[i % R], non_blocking=True)
                g_step[i % R].replay()
                oh.copy_(outs[i % R], non_blocking=True)
            torch.cuda.synchronize()
            barrier(ws)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(steps):
                r = i % R
                xs[r].copy_(xh[r], non_blocking=True)
                g_step[r].replay()
                oh.copy_(outs[r], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            barrier(ws)
        return max_over_ranks(a.elapsed_time(b), ws, dev)

    tokens = steps * wl.T * ws
    e2e_ms = e2e_serial()
    e2e = {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": xbytes,
           "d2h_bytes_per_step": xbytes,
           "method": "fixed protocol: x copied in from pinned host memory (cudaMemcpyAsync on the layer's stream), "
                     "the layer's step graph, out copied back to pinned host memory; serial on one stream"}
    if e2e_variants:
        # context only: the layer reading x straight from the pinned host
        # buffer (GB300's host memory is coherent with the GPU over NVLink-C2C)
        g_host = []
        with torch.cuda.stream(stream):
            for r in range(R):
                step_call(r, xh[r])
            torch.cuda.synchronize()
            for r in range(R):
                g = new_graph()
                with torch.cuda.graph(g, stream=stream):
                    step_call(r, xh[r])
                g_host.append(g)
            torch.cuda.synchronize()
            for i in range(min(warmup, 10)):
                g_host[i % R].replay()
            torch.cuda.synchronize()
            barrier(ws)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(steps):
                g_host[i % R].replay()
                oh.copy_(outs[i % R], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            barrier(ws)
        hx_ms = max_over_ranks(a.elapsed_time(b), ws, dev)
        e2e["context_variants_tokens_per_s"] = {
            "layer reads x from the pinned host buffer, out copied back": tokens / (hx_ms / 1e3)}

    cpu_base = None
    if host0 is not None:
        xa = synth.make_x(wl, "cpu", step=1000, T=256).double().numpy()
        tps, done, threads, secs = oracle_tokens_per_s(wl, host0, xa, budget_s=cpu_budget, max_s=2.5 * cpu_budget)
        model, ncpu = cpu_info()
        cpu_base = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                    "sample": f"{done} independent tokens of layer 0 in {secs:.1f} s (batches of "
                              f"{threads * min(max(1, wl.T), 4)}), {model}, {ncpu} host cores"}

    del g_step, g_rb, g_ffn, g_all, layers, xs, outs, wss
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": steps,
        "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if tc_path else "f32",
        "data": f"synthetic (seeded, qwen3_moe geometry, random-init {fmt_name(wl)})",
        "config": workload_config(wl, args, R),
        "layer_hbm_gbs": layer_gbs,
        "timed_loops_ms": loops, "timed_loop": timing,
        "near_ties": {"tokens": near, "of": R * wl.T, "gap": NEAR_TIE,
                      "note": "tokens of the rotating inputs whose fp64 top-(k+1) logits have an adjacent gap "
                              "below the threshold; their selection may follow fp32 rounding"},
        "separate_path_ms": {"route_and_bucket": rb_ms, "expert_ffn": ffn_ms_mean},
        "roofline": roofline, "cpu_baseline": cpu_base, "e2e": e2e,
        "gpu_launches": launches, "gpu_launches_source": launches_src, "clocks": clocks,
    }


class StackWeights:
    """The 48 resident layers of the stack workloads (they share weights and
    routers: the same seeds), generated once."""

    def __init__(self, wl, dev, keep_host0: bool):
        self.layers, self.host0 = [], None
        for l in range(wl.layers):
            w = synth.make_layer(wl, l, dev)
            if l == 0 and keep_host0:
                self.host0 = {k: (None if v is None else v.cpu().numpy()) for k, v in w.items()}
            self.layers.append(binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"],
                                                         w["down"], w["Wr"], w["bias"], wfmt=wfmt_of(wl)))
            del w
        torch.cuda.synchronize()


def measure_stack(wl, args, ws, rank, dev, sampler, sw: StackWeights, steps: int, warmup: int, cpu_budget: float):
    """The 48-layer stack: every layer resident, one CUDA graph per step running
    x_{l+1} = x_l + MoE_l(x_l) through all layers (residual chaining through two
    ping-pong buffers).  tokens/s = T / t_stack."""
    act = binding.MOE_ACT_BF16 if wl.act == "bf16" else binding.MOE_ACT_F32
    tc_path = act == binding.MOE_ACT_BF16 and wl.T * wl.k >= 128
    L = wl.layers
    layers = sw.layers
    x0 = synth.make_x(wl, dev, step=0)
    bufs = [torch.empty_like(x0), torch.empty_like(x0)]
    wsb = binding.workspace(wl.T, layers[0], act, 0, dev)
    offs = [torch.empty(wl.E + 1, dtype=torch.int32, device=dev) for _ in range(L)]
    torch.cuda.synchronize()  # everything above was made on the default stream
    stream = torch.cuda.Stream(device=dev)

    def stack_call(record_offsets=False):
        bufs[0].copy_(x0)  # this step's input
        for l in range(L):
            binding.layer_forward(bufs[l % 2], layers[l], act, 0, True, out=bufs[(l + 1) % 2], ws=wsb,
                                  offsets_out=offs[l] if record_offsets else None)

    with torch.cuda.stream(stream):
        stack_call(record_offsets=True)
        stack_call()
    torch.cuda.synchronize()
    g = new_graph()
    with torch.cuda.graph(g, stream=stream):
        stack_call()
    torch.cuda.synchronize()
    n_active = [int((np.diff(o.cpu().numpy()) > 0).sum()) for o in offs]
    xbytes = wl.T * wl.d_model * 4
    step_bytes = sum(n * expert_bytes(wl) + 2 * xbytes + wl.E * wl.d_model * 4 for n in n_active)
    kn = graph_kernel_nodes(g)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        t_soak = time.time()
        while time.time() - t_soak < args.soak:
            g.replay()
            torch.cuda.synchronize()
        t_clk0 = time.time()
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        t_clk1 = time.time()
    ms_local = e0.elapsed_time(e1)
    clocks = sampler.summary(t_clk0 - 0.5, t_clk1 + 0.05)
    ms = max_over_ranks(ms_local, ws, dev)
    tokens = steps * wl.T * ws
    value = job_rate(steps, wl.T, ws, ms)

    # dominant kernel: the expert FFN of each layer, timed alone (routing first, outside the events)
    P = wl.T * wl.k
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev)
    wts = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
    pt = torch.empty(P, dtype=torch.int32, device=dev)
    ps = torch.empty(P, dtype=torch.int32, device=dev)
    po = torch.empty(P, dtype=torch.int32, device=dev)
    off = torch.empty(wl.E + 1, dtype=torch.int32, device=dev)
    out2 = torch.empty_like(x0)
    Lb = binding.load()
    st = lambda: torch.cuda.current_stream().cuda_stream  # noqa: E731
    ffn_ms, ffn_alg = [], []
    with torch.cuda.stream(stream):
        for rep in range(2):
            for l in range(L):
                binding._check("moe_route", Lb.moe_route(binding._ptr(x0), wl.T, layers[l].ref(), binding._ptr(idx),
                                                         binding._ptr(wts), binding.ctypes.c_void_p(st())))
                binding._check("moe_bucket", Lb.moe_bucket(binding._ptr(idx), wl.T, wl.k, wl.E, binding._ptr(off),
                                                           binding._ptr(pt), binding._ptr(ps), binding._ptr(po), None,
                                                           binding.ctypes.c_void_p(st())))
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                binding.expert_ffn_q8(x0, layers[l], off, pt, ps, wts, act, True, True, ws=wsb, out=out2)
                b.record(stream)
                torch.cuda.synchronize()
                if rep > 0:
                    ffn_ms.append(a.elapsed_time(b))
                    na = int((np.diff(off.cpu().numpy()) > 0).sum())
                    ffn_alg.append(na * expert_bytes(wl) + 2 * xbytes)
    peaks = load_peaks()
    ffn_ms_mean = float(np.mean(ffn_ms))
    alg = float(np.mean(ffn_alg))
    achieved = alg / (ffn_ms_mean / 1e3) / 1e9
    roofline = {"kernel": expert_path_name(wl, tc_path),
                "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": alg, "launch_ms": ffn_ms_mean, "traffic": None,
                "timed_over": f"{len(ffn_ms)} launches, every layer of the stack (CUDA events on the launch stream)"}
    if tc_path:
        flops = 2.0 * wl.T * wl.k * 3 * wl.d_model * wl.d_ff
        tf = flops / (ffn_ms_mean / 1e3) / 1e12
        roofline["tensor"] = {"achieved": tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                              "frac": tf / peaks["bf16_tflops_sustained"], "flops_per_launch": flops,
                              "peak_note": "sustained bf16 figure (kernel timed inside a long step)"}

    # end to end: pinned x in, the stack, the final hidden state out
    xh = x0.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            x0.copy_(xh, non_blocking=True)
            g.replay()
            oh.copy_(bufs[L % 2], non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    e2e_ms = max_over_ranks(a.elapsed_time(b), ws, dev)

    cpu_base = None
    if sw.host0 is not None and cpu_budget > 0:
        xa = synth.make_x(wl, "cpu", step=1000, T=256).double().numpy()
        tps, done, threads, secs = oracle_tokens_per_s(wl, sw.host0, xa, budget_s=cpu_budget,
                                                       max_s=2.5 * cpu_budget)
        model, ncpu = cpu_info()
        cpu_base = {"value": tps / L, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                    "sample": f"layer 0 of the stack timed on {done} independent tokens in {secs:.1f} s; "
                              f"stack rate = layer rate / {L} (extrapolated), {model}, {ncpu} host cores"}
    del g
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": steps,
        "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if tc_path else "f32",
        "data": f"synthetic (seeded, qwen3_moe geometry, random-init {fmt_name(wl)})",
        "config": {"workload": f"{wl.name}: {L}-layer MoE stack with residual, T={wl.T}, d_model={wl.d_model}, "
                               f"d_ff={wl.d_ff}, E={wl.E}, top-{wl.k}, Zipf router bias, "
                               f"{'bf16' if tc_path else 'f32'} expert inputs",
                   "tokens_per_step": wl.T, "layers": L,
                   "l2": f"inputs larger than L2: {L} resident layers x {wl.E} experts x {expert_bytes(wl)} B",
                   "parallelism": f"replicas x{ws}", "graph": f"one CUDA graph per step ({L} layers)"},
        "stack_hbm_gbs": step_bytes / (ms_local / steps / 1e3) / 1e9,
        "roofline": roofline, "cpu_baseline": cpu_base,
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": xbytes,
                "d2h_bytes_per_step": xbytes,
                "method": "fixed protocol: x copied in from pinned host memory, the stack's step graph, the final "
                          "hidden state copied back; serial on one stream"},
        "gpu_launches": None if kn is None else kn * steps,
        "gpu_launches_source": "kernel nodes of the captured step graph" if kn is not None
        else "graph introspection unavailable",
        "clocks": clocks,
    }


# The default run: the headline workload (decode T = 1), then every other
# workload of the metric as a sub-record of the same line.
SUITE_LAYERS = ["decode_t64_zipf", "prefill_t768", "prefill_t1024", "prefill_t2048_mb1024", "prefill_t2048"]
SUITE_STACKS = ["stack48_t1", "stack48_t64", "stack48_t1024"]
# the 4-bit expert format (Q4_0) at the same geometry, beside its Q8_0 rows
SUITE_Q4 = ["decode_t1_q4", "decode_t64_zipf_q4", "prefill_t1024_q4"]


def run_ours(args, ws, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    sampler = ClockSampler(local)
    sampler.start()
    t_start = time.time()
    try:
        name = args.workload or "decode_t1"
        wl = synth.WORKLOADS[name]
        keep_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
        if wl.layers > 1:
            sw = StackWeights(wl, dev, keep_cpu)
            line = measure_stack(wl, args, ws, rank, dev, sampler, sw, args.steps, args.warmup,
                                 args.cpu_budget if keep_cpu else 0.0)
            del sw
        else:
            line = measure_layer(wl, args, ws, rank, dev, sampler, args.rot, args.steps, args.warmup,
                                 args.cpu_budget if keep_cpu else 0.0, e2e_variants=True)
        if args.workload is None and not args.headline_only:
            subs = {}
            sub_cpu = args.sub_cpu_budget if keep_cpu else 0.0
            for n in SUITE_LAYERS + SUITE_Q4:
                torch.cuda.empty_cache()
                subs[n] = measure_layer(synth.WORKLOADS[n], args, ws, rank, dev, sampler, args.sub_rot,
                                        args.steps, args.warmup, sub_cpu)
            torch.cuda.empty_cache()
            sw = StackWeights(synth.WORKLOADS[SUITE_STACKS[0]], dev, keep_cpu)
            for n in SUITE_STACKS:
                subs[n] = measure_stack(synth.WORKLOADS[n], args, ws, rank, dev, sampler, sw,
                                        max(3, args.steps // 4), args.warmup, sub_cpu)
            del sw
            torch.cuda.empty_cache()
            line["workloads"] = subs
            line["workloads_note"] = ("every workload of the metric, and the Q4_0 expert format at three of "
                                      "them, measured in this run with the same K / W (the stacks with K/4 "
                                      f"steps); value and ms_per_step above are {name}'s")
        line["bench_wall_s"] = time.time() - t_start
    finally:
        sampler.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_arena(args, ws, rank, local):
    """The 48-layer stack served from an expert arena: every expert's blob in
    page-locked host memory, `slots` of them in HBM.  Each layer admits its
    routed experts (LRU) before its FFN and the GPU copies the misses in over
    NVLink-C2C; one CUDA graph per step; every step is a new token (its own x),
    so routing, and with it residency, moves.  tokens/s = 1 / t_stack."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.workload]
    S = args.slots or wl.arena_slots
    L = wl.layers
    act = binding.MOE_ACT_F32
    binding.load()
    t_setup = time.time()
    ar, routers, host0 = None, [], None
    for l in range(L):
        w = synth.make_layer(wl, l, dev)
        if l == 0 and rank == 0 and ws == 1 and not args.no_cpu_baseline:
            host0 = {k: (None if v is None else v.cpu().numpy()) for k, v in w.items()}
        lay = binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"], w["Wr"],
                                        w["bias"], wfmt=wfmt_of(wl))
        if ar is None:
            ar = binding.Arena(lay, L, S, dev)
        ar.pack_layer(l, lay)
        routers.append((w["Wr"], w["bias"]))
        torch.cuda.synchronize()
        del w, lay
    setup_s = time.time() - t_setup
    als = [ar.layer(wr, b) for wr, b in routers]
    NX = 4096
    X = synth.make_x(wl, dev, step=0, T=NX)              # one new token per step, cycling over 4096
    xin = torch.empty(1, wl.d_model, dtype=torch.float32, device=dev)
    bufs = [torch.empty_like(xin), torch.empty_like(xin)]
    wsb = binding.workspace(1, als[0], act, 0, dev)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)

    def stack_call():
        bufs[0].copy_(xin)
        for l in range(L):
            binding.layer_forward_arena(bufs[l % 2], als[l], ar, l, act, 0, True, out=bufs[(l + 1) % 2], ws=wsb)

    with torch.cuda.stream(stream):
        xin.copy_(X[0:1])
        stack_call()
    torch.cuda.synchronize()
    g = new_graph()
    with torch.cuda.graph(g, stream=stream):
        stack_call()
    torch.cuda.synchronize()
    kn = graph_kernel_nodes(g)
    step_i = [0]

    def step():
        xin.copy_(X[step_i[0] % NX:step_i[0] % NX + 1])
        step_i[0] += 1
        g.replay()

    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        t_soak = time.time()
        while time.time() - t_soak < args.soak:
            step()
            torch.cuda.synchronize()
        s0 = ar.stats()
        t_clk0 = time.time()
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        t_clk1 = time.time()
    ms_local = e0.elapsed_time(e1)
    sampler.stop()
    clocks = sampler.summary(t_clk0 - 0.5, t_clk1 + 0.05)
    s1 = ar.stats()
    ms = max_over_ranks(ms_local, ws, dev)
    value = job_rate(args.steps, 1, ws, ms)
    d_hit, d_miss = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
    d_bytes = s1["bytes_in"] - s0["bytes_in"]

    # the same graph with the token repeated: every admission hits (routing repeats)
    nrep = min(args.steps, 200)
    with torch.cuda.stream(stream):
        xin.copy_(X[0:1])
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        h0 = ar.stats()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(nrep):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
    hit_ms = a.elapsed_time(b) / nrep
    assert ar.stats()["misses"] == h0["misses"]

    # the miss path alone: empty arena, one layer's 8 routed experts all missing
    Lb = binding.load()
    off = torch.zeros(wl.E + 1, dtype=torch.int32, device=dev)
    smap = torch.empty(wl.E, dtype=torch.int32, device=dev)
    copy_ms, copy_bytes = [], []
    with torch.cuda.stream(stream):
        for rep in range(12):
            ar.reset()
            offs = np.zeros(wl.E + 1, dtype=np.int32)
            sel = np.random.default_rng(rep).choice(wl.E, wl.k, replace=False)
            cnt = np.zeros(wl.E, dtype=np.int32)
            cnt[sel] = 1
            offs[1:] = np.cumsum(cnt)
            off.copy_(torch.from_numpy(offs))
            torch.cuda.synchronize()
            m0 = ar.stats()["bytes_in"]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            binding._check("moe_arena_admit", Lb.moe_arena_admit(
                binding._ptr(ar.state), rep % L, binding._ptr(off), wl.k,
                binding.ctypes.c_void_p(ar.host_blobs.data_ptr()), als[rep % L].ref(), binding._ptr(smap), None,
                binding.ctypes.c_void_p(stream.cuda_stream)))
            b.record(stream)
            torch.cuda.synchronize()
            if rep >= 2:
                copy_ms.append(a.elapsed_time(b))
                copy_bytes.append(ar.stats()["bytes_in"] - m0)
    copy_ms_mean = float(np.mean(copy_ms))
    copy_gbs = float(np.mean(copy_bytes)) / (copy_ms_mean / 1e3) / 1e9
    # the host link measured the plain way: one copy-engine transfer of 1 GiB pinned -> device
    hsrc = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    ddst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        best = None
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ddst.copy_(hsrc, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            t = a.elapsed_time(b)
            best = t if best is None else min(best, t)
    h2d_gbs = (1 << 30) / (best / 1e3) / 1e9
    del hsrc, ddst
    ar.reset()

    cpu_base = None
    if host0 is not None:
        xa = synth.make_x(wl, "cpu", step=1000, T=256).double().numpy()
        tps, done, threads, secs = oracle_tokens_per_s(wl, host0, xa, budget_s=args.cpu_budget)
        model, ncpu = cpu_info()
        cpu_base = {"value": tps / L, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                    "sample": f"layer 0 of the stack timed on {done} independent tokens in {secs:.1f} s; "
                              f"stack rate = layer rate / {L} (extrapolated; the oracle has every expert in "
                              f"host memory, no arena), {model}, {ncpu} host cores"}
    if rank == 0:
        per_step_bytes = d_bytes / args.steps
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": f"synthetic (seeded, qwen3_moe geometry, random-init {fmt_name(wl)})",
            "config": {"workload": f"{wl.name}: {L}-layer MoE stack with residual, T=1 (a new token each step), "
                                   f"d_model={wl.d_model}, d_ff={wl.d_ff}, E={wl.E}, top-{wl.k}, Zipf router bias, "
                                   f"experts served from an arena of {S} HBM slots "
                                   f"({100.0 * S / (L * wl.E):.2f}% of {L * wl.E} experts resident)",
                       "tokens_per_step": 1, "layers": L, "slots": S,
                       "l2": f"inputs larger than L2: {L} x {wl.E} experts of {expert_bytes(wl)} B behind "
                             f"{S} slots ({S * expert_bytes(wl) / 1e9:.2f} GB)",
                       "parallelism": f"replicas x{ws}", "graph": f"one CUDA graph per step ({L} layers)"},
            "arena": {"hit_rate": d_hit / max(1, d_hit + d_miss), "hits_per_step": d_hit / args.steps,
                      "misses_per_step": d_miss / args.steps, "bytes_in_per_step": per_step_bytes,
                      "blob_bytes": ar.blob_bytes, "all_hit_ms_per_step": hit_ms,
                      "miss_cost_ms_per_step": ms / args.steps - hit_ms,
                      "host_blobs_gb": L * wl.E * ar.blob_bytes / 1e9, "setup_s": setup_s},
            "roofline": {"kernel": "arena_copy_kernel (missed blobs, page-locked host memory -> HBM slots, "
                                   "read by the GPU over NVLink-C2C; with the one-CTA admission before it)",
                         "bound": "host link", "achieved": copy_gbs, "peak": h2d_gbs, "unit": "GB/s",
                         "frac": copy_gbs / h2d_gbs,
                         "peak_source": "measured in this run: one 1 GiB cudaMemcpyAsync, page-locked host -> "
                                        "device (copy engines), best of 5",
                         "algorithmic_bytes_per_launch": float(np.mean(copy_bytes)), "launch_ms": copy_ms_mean,
                         "traffic": None,
                         "timed_over": f"{len(copy_ms)} admissions of {wl.k} missed experts into an empty arena"},
            "cpu_baseline": cpu_base,
            "gpu_launches": None if kn is None else kn * args.steps,
            "gpu_launches_source": "kernel nodes of the captured step graph" if kn is not None
            else "graph introspection unavailable",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_ab_reuse(args, ws, rank, local):
    """Paired A/B of the reuse-ordering traversal (MOE_FLAG_REUSE_ORDER) on a
    prefill workload, with the protocol of
    expxa.com/research/reuse-ordering-qualification ("Method and limits"):
    pairs alternate AB / BA, the paired ratio candidate / baseline per pair,
    the median paired change, and a 95% interval from 20,000 paired bootstrap
    resamples; adopted only if the median is at least 2% faster and the
    interval lies wholly below parity (the pages' predeclared bar)."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.workload or "prefill_t1024"]
    act = binding.MOE_ACT_BF16 if wl.act == "bf16" else binding.MOE_ACT_F32
    binding.load()
    R = args.rot
    layers, xs, outs, wss = [], [], [], []
    for r in range(R):
        w = synth.make_layer(wl, r, dev)
        layers.append(binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"],
                                                w["Wr"], w["bias"], wfmt=wfmt_of(wl)))
        del w
        xs.append(synth.make_x(wl, dev, step=r))
        outs.append(torch.empty(wl.T, wl.d_model, dtype=torch.float32, device=dev))
        wss.append(binding.workspace(wl.T, layers[-1], act, 0, dev))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    for name, flags in (("A", 0), ("B", binding.MOE_FLAG_REUSE_ORDER)):
        def call(flags=flags):
            for r in range(R):
                binding.layer_forward(xs[r], layers[r], act, flags, False, out=outs[r], ws=wss[r])
        with torch.cuda.stream(stream):
            call()
        torch.cuda.synchronize()
        g = new_graph()
        with torch.cuda.graph(g, stream=stream):
            call()
        graphs[name] = g
    torch.cuda.synchronize()
    reps = max(1, args.steps // (2 * args.pairs))

    def trial(name):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                graphs[name].replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * R)  # ms per layer call

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        trial("A")
        trial("B")
    t_clk0 = time.time()
    ta, tb = [], []
    for i in range(args.pairs):
        order = ("A", "B") if i % 2 == 0 else ("B", "A")
        res = {n: trial(n) for n in order}
        ta.append(res["A"])
        tb.append(res["B"])
    t_clk1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_clk0 - 0.5, t_clk1 + 0.05)
    ratio = np.array(tb) / np.array(ta)
    rng = np.random.default_rng(20000)
    boot = np.median(ratio[rng.integers(0, len(ratio), size=(20000, len(ratio)))], axis=1)
    lo, hi = np.percentile(boot, [2.5, 97.5])
    med = float(np.median(ratio))
    adopt = bool(med <= 0.98 and hi < 1.0)
    if rank == 0:
        mb = float(np.median(tb))
        line = {
            "metric": METRIC, "value": wl.T / (mb / 1e3), "unit": "tokens/s", "n_gpus": ws,
            "steps": 2 * args.pairs * reps * R, "warmup": args.warmup, "ms_per_step": mb,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if act == binding.MOE_ACT_BF16 else "f32",
            "data": f"synthetic (seeded, qwen3_moe geometry, random-init {fmt_name(wl)})",
            "config": workload_config(wl, args),
            "ab_reuse_order": {
                "baseline": "chunk-major units (default)", "candidate": "MOE_FLAG_REUSE_ORDER (bands of 4 row tiles)",
                "pairs": args.pairs, "order": "alternating AB / BA", "layer_calls_per_trial": reps * R,
                "baseline_ms_median": float(np.median(ta)), "candidate_ms_median": mb,
                "median_paired_change": med - 1.0, "ci95": [float(lo) - 1.0, float(hi) - 1.0],
                "bootstrap_resamples": 20000,
                "bar": "median paired change <= -2% and the 95% interval wholly below parity",
                "adopted": adopt},
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    return 0


def sources_sha1(paths) -> str:
    """sha1 over the concatenated bytes of the given repo files (in order)."""
    import hashlib
    h = hashlib.sha1()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()


def load_traffic(key: str):
    """DRAM bytes per launch from a committed ncu capture, or None when a
    source of the kernel changed since the counters were taken."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[key]
        if sources_sha1(rec["sources"]) != rec["sources_sha1"]:
            return None
    except (OSError, KeyError, ValueError):
        return None
    return float(rec["dram_bytes_per_launch"])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(synth.WORKLOADS),
                    help="one workload only (default: decode T=1 with every workload of the metric as sub-records)")
    ap.add_argument("--rot", type=int, default=16, help="seeded layers the steps rotate over")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--slots", type=int, default=0, help="arena slots (arena workloads; 0: the workload's)")
    ap.add_argument("--ab-reuse-order", action="store_true",
                    help="paired A/B of the reuse-ordering traversal instead of the throughput line")
    ap.add_argument("--pairs", type=int, default=16)
    ap.add_argument("--headline-only", action="store_true", help="only the headline workload (no sub-records)")
    ap.add_argument("--sub-rot", type=int, default=4, help="seeded layers the sub-record workloads rotate over")
    ap.add_argument("--sub-cpu-budget", type=float, default=4.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, ws, rank)
        if args.ab_reuse_order:
            return run_ab_reuse(args, ws, rank, local)
        if args.workload and synth.WORKLOADS[args.workload].arena_slots > 0:
            return run_arena(args, ws, rank, local)
        return run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
