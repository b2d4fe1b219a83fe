"""Benchmark of the fused MoE layer (forward + backward, BF16) on GB300.

One step = one forward and one backward of the whole layer (router top-k,
layout, gather, [a|b] GEMM + SwiGLU, down GEMM, combine; gather, u GEMM +
SwiGLU backward, dx GEMM, dx reduce, router gradient, dWd and dWg/dWu GEMMs)
over T=4096 tokens, hidden 7168, expert width 2048, 256 experts, top-8, with
Zipf(1.1) routing skew (synthetic seeded inputs; random weights).

Prints one JSON line.  Under torchrun every rank runs its own copy of the
workload (token-parallel replicas: no data-path collective); timing is the
maximum over ranks.  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
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

from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs  # noqa: E402

METRIC = "MoE layer tokens/s fwd+bwd (BF16, MXFP8) on 1 GB300; % of roofline"
SHAPE = dict(T=4096, d=7168, F=2048, E=256, k=8)
MX_SHAPE = dict(T=16384)   # the MXFP8 forward configuration: same layer, 16384 tokens
ALPHA = 1.1
SEED = 0
WORKLOAD = "moe_layer_fwd_bwd_bf16_T4096_d7168_F2048_E256_top8_zipf1.1"


# ----------------------------------------------------------------------------- distributed helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def launch_ranks(args, argv) -> int:
    """`--gpus N` (N > 1) outside a launcher: start N ranks on this node, one
    per GPU, with torch.distributed.run on 127.0.0.1 and the same arguments,
    and return its exit status.  Rank 0 prints the JSON line."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def bench_dry_run(args):
    """The rank plumbing alone, without a GPU (gloo): each rank times a short
    host wait of its own length, then barrier and max over ranks as in the
    timed runs; rank 0 prints the line.  Checks the launcher and the timing
    exchange on a machine without GPUs."""
    ws, rank, _ = dist_env()
    init_dist(ws, "gloo")
    barrier(ws)
    t0 = time.perf_counter()
    time.sleep(0.01 * (1 + rank))
    el = max_over_ranks((time.perf_counter() - t0) * 1e3, ws, torch.device("cpu"))
    barrier(ws)
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": ws, "max_rank_ms": round(el, 3),
                          "config": {"parallelism": f"replicas{ws}"}}), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    """Largest value of x over all ranks (host-side timing exchange only)."""
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- roofline bookkeeping
def algorithmic_bytes(shape, R: int, e_act: int):
    """Compulsory HBM bytes per launch of each kernel (bf16 = 2 B).

    Weight reads count only the ``e_act`` experts that received at least one
    routed row: an expert with no rows need not be read.  Weight-gradient
    writes count all E experts, since an idle expert's dW is still written
    (zeros).  Activation terms count R routed rows, padding excluded; a token
    row that is gathered k times is counted once where the gather is served
    by L2 (the ring megakernel reads X once per token from HBM)."""
    T, d, F, E = shape["T"], shape["d"], shape["F"], shape["E"]
    Wa = e_act * F * d * 2     # one weight tensor, active experts only
    Wall = E * F * d * 2       # one weight-gradient tensor, all experts
    return {
        # one-launch forward: also reads the logits and writes Y (routing and
        # combine run inside it)
        "fwd_megakernel": 3 * Wa + T * d * 2 + R * 2 * F * 2 + R * d * 2 + T * shape["E"] * 4 + T * d * 2,
        "gemm_up_swiglu": 2 * Wa + R * d * 2 + R * 3 * F * 2,
        "gemm_down": Wa + R * F * 2 + R * d * 2,
        "gemm_bwd_u_swiglu": Wa + R * d * 2 + R * 2 * F * 2 + R * 3 * F * 2,
        "gemm_bwd_dx": 2 * Wa + R * 2 * F * 2 + R * d * 2,
        "gemm_wgrad_down": Wall + R * d * 2 + R * F * 2,
        "gemm_wgrad_gate_up": 2 * Wall + R * 2 * F * 2 + R * d * 2,
    }


def layer_roofline(shape, peaks, e_act: int):
    """Roofline time of one fwd+bwd: max(FLOPs / bf16 peak, compulsory bytes / HBM peak).

    Compulsory bytes: the active experts' weights read in the forward and again
    in the backward, every expert's weight gradient written once, and the
    layer's own inputs and outputs."""
    T, d, F, E, k = (shape[n] for n in ("T", "d", "F", "E", "k"))
    R = T * k
    flops = 18.0 * R * d * F
    Wa = 3.0 * e_act * F * d * 2
    Wall = 3.0 * E * F * d * 2
    act = T * d * 2 * 4 + T * E * 4 * 2   # X, dY in; Y, dX out; logits in, dlogits out
    byts = 2 * Wa + Wall + act
    t_tc = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    return {"flops": flops, "bytes": byts, "t_ms": max(t_tc, t_hbm) * 1e3,
            "bound": "hbm" if t_hbm >= t_tc else "tensor"}


# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, mean
# over the launches) from one single-pass ncu launch-list capture of this
# bench's default workload.  The figures hold only for the GEMM sources they
# were taken on: their digest is kept beside them, and any change to those
# sources makes measured_traffic() report null until a new capture is taken.
NCU_TRAFFIC = {
    "workload": WORKLOAD,
    "csrc_sha256": "2b67d396b0083f3c8f356e821589e1ebb991c02e7b1f81df11974171b3cbe150",
    "bytes": {
        "gemm_up_swiglu": 11549616282,
        "gemm_down": 5641070285,
        "gemm_bwd_u_swiglu": 6876470170,
        "gemm_bwd_dx": 10699051725,
        "gemm_wgrad_down": 8508401101,
        "gemm_wgrad_gate_up": 16121594010,
    },
}


# The files that define the GEMM kernels the traffic figures belong to.
GEMM_SOURCES = ("gemm.cuh", "ptx.cuh", "gemm_fwd.cu", "gemm_bwd.cu")


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines (string literals kept):
    a comment cannot change a kernel, so it does not change the digest."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                       # string literal, escapes kept
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def csrc_digest() -> str:
    """sha256 over the code (comments stripped) of the GEMM kernels' sources."""
    import hashlib
    src = os.path.join(ROOT, "mixture_experts_layer_19_gb300", "csrc")
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        h.update(name.encode())
        with open(os.path.join(src, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    t = NCU_TRAFFIC
    if workload != t["workload"] or kernel not in t["bytes"] or csrc_digest() != t["csrc_sha256"]:
        return None
    return t["bytes"][kernel]


def active_experts(plan, saved, T):
    """Number of experts that received at least one routed row, read from the
    plan's own routing of the last forward."""
    counts = plan.routing(saved, T)["counts"]
    return int((counts > 0).sum().item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- CPU oracle timing
class _HostWeights:
    """Per-expert host copies (float32, exact widening of bf16) of device weights."""

    def __init__(self, W, experts):
        self.cache = {int(e): W[int(e)].float().cpu().numpy() for e in experts}

    def __getitem__(self, e):
        return self.cache[int(e)]


def oracle_sample(inp, tokens, k):
    """Prepare the oracle's inputs for a sub-batch of tokens (host copies)."""
    from oracle import moe_ref
    tokens = torch.as_tensor(np.asarray(tokens), device=inp.X.device)
    logits = inp.logits[tokens].double().cpu().numpy()
    idx, _ = moe_ref.route(logits, k)
    experts = sorted(set(idx.reshape(-1).tolist()) | {0})
    return {
        "X": inp.X[tokens].double().cpu().numpy(), "logits": logits,
        "dY": inp.dY[tokens].double().cpu().numpy(),
        "Wg": _HostWeights(inp.Wg, experts), "Wu": _HostWeights(inp.Wu, experts),
        "Wd": _HostWeights(inp.Wd, experts), "n": int(tokens.numel()), "experts": len(experts) - 1,
    }


def run_oracle(s, k):
    from oracle import moe_ref
    Y, ctx = moe_ref.forward(s["X"], s["logits"], s["Wg"], s["Wu"], s["Wd"], k)
    g = moe_ref.backward(s["dY"], s["X"], s["logits"], s["Wg"], s["Wu"], s["Wd"], ctx, sparse_dw=True)
    return Y, g


def cpu_cores():
    return len(os.sched_getaffinity(0))


def set_blas_threads(n):
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(n)
    except Exception:
        return None


# ----------------------------------------------------------------------------- main arms
def bench_gpu(args):
    from mixture_experts_layer_19_gb300 import moe
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    shape = dict(SHAPE)
    if args.experts:
        shape["E"] = args.experts   # smaller layer for profiler captures only
    if args.tokens:
        shape["T"] = args.tokens
    T, d, F, E, k = (shape[n] for n in ("T", "d", "F", "E", "k"))
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=SEED + rank, alpha=ALPHA, device=dev)
    flags = moe.MOE_DEBUG_TIMING
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, device=local, debug_flags=flags))
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    grads = {
        "dX": torch.empty((T, d), dtype=torch.bfloat16, device=dev),
        "dWg": torch.empty((E, F, d), dtype=torch.bfloat16, device=dev),
        "dWu": torch.empty((E, F, d), dtype=torch.bfloat16, device=dev),
        "dWd": torch.empty((E, d, F), dtype=torch.bfloat16, device=dev),
        "dg": torch.empty((T, k), dtype=torch.float32, device=dev),
        "dlogits": torch.empty((T, E), dtype=torch.float32, device=dev),
    }
    stream = torch.cuda.current_stream(dev)

    def step(X, logits, dY):
        plan.forward(X, logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        plan.backward(dY, X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

    for _ in range(args.warmup):
        step(inp.X, inp.logits, inp.dY)
    torch.cuda.synchronize(dev)
    if plan.device_status() != 0:
        raise RuntimeError("device status set during warm-up")
    plan.kernel_times()  # discard warm-up records
    e_act = active_experts(plan, saved, T)
    plan.kernel_times()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(inp.X, inp.logits, inp.dY)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    ktimes = plan.kernel_times()
    status = plan.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_per_step = elapsed_ms / args.steps
    value = ws * T * args.steps / (elapsed_ms / 1e3)

    # ---- roofline of the dominant kernel (largest share of device time)
    peaks = load_peaks()
    R = T * k
    ab = algorithmic_bytes(shape, R, e_act)
    gemm_names = [n for n in ktimes if n in ab]
    dom = max(gemm_names, key=lambda n: ktimes[n][0])
    dom_ms = ktimes[dom][0] / ktimes[dom][1]
    achieved = ab[dom] / (dom_ms / 1e3) / 1e9
    workload = WORKLOAD if not (args.experts or args.tokens) else f"profile_T{T}_E{E}"
    traffic = measured_traffic(dom, workload)
    roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "peak_source": peaks["source"] + " hbm_gbs (STREAM copy)",
            "algorithmic_bytes": ab[dom], "avg_launch_ms": round(dom_ms, 4)}
    per_kernel = {n: {"achieved_gbs": round(ab[n] / (ktimes[n][0] / ktimes[n][1] / 1e3) / 1e9, 1),
                      "frac": round(ab[n] / (ktimes[n][0] / ktimes[n][1] / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                      "algorithmic_bytes": ab[n], "traffic": measured_traffic(n, workload)}
                  for n in gemm_names}
    total_dev = sum(v[0] for v in ktimes.values())
    kernels = {n: {"ms_per_step": round(v[0] / args.steps, 4), "launches": v[1],
                   "share": round(v[0] / total_dev, 4)} for n, v in sorted(ktimes.items(), key=lambda x: -x[1][0])}
    launches = int(sum(v[1] for v in ktimes.values()))
    lr = layer_roofline(shape, peaks, e_act)

    # ---- end-to-end through the public API with host buffers
    e2e = None if args.no_e2e else bench_e2e(args, plan, inp, Y, saved, grads, stream, dev, ws)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "T": T, "d": d, "F": F, "E": E, "k": k, "zipf_alpha": ALPHA,
                   "seed": SEED, "tokens_per_gpu": T, "experts_active": e_act, "parallelism": f"replicas{ws}",
                   "launch": plan.info(),
                   "l2": "inputs larger than L2 (22.5 GB of expert weights streamed per pass, 129 MB L2)"},
        "roofline": roof,
        "kernel_rooflines": per_kernel,
        "layer_roofline": {"bound": lr["bound"], "t_ms": round(lr["t_ms"], 4),
                           "frac": round(lr["t_ms"] / ms_per_step, 4),
                           "note": "max(18*R*d*F / sustained bf16 peak, active experts' weights read twice "
                                   "+ all dW written + I/O / HBM peak)"},
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    ref = {"Y": Y.clone(), **{n: v.clone() for n, v in grads.items()}}
    out["graph_replay"] = bench_graph(args, inp, ref, dev, ws)
    del ref
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(inp, k, args.cpu_tokens)
    if not args.no_ring:
        out["ring_pipeline"] = bench_ring(args, plan, inp, Y, saved, grads, stream, dev, ws)
    out["router_gemm"] = bench_router(args, plan, inp, stream, dev, ws, peaks)
    if not args.no_ep:
        out["virtual_rank_ep"] = bench_ep(args, plan, inp, Y, saved, grads, stream, dev, ws)
    if not args.no_mx:
        del plan, inp, grads, saved, Y
        torch.cuda.empty_cache()
        out["mxfp8_forward"] = [bench_mx_forward(args, dev, ws, peaks, alpha) for alpha in (0.0, ALPHA)]
        # the largest configuration (T=32768, tensor-bound) is part of every run
        grid = [(Tm, a) for Tm in (2048, 8192, 32768) for a in (0.0, 1.1, 1.5)] if args.sweep else \
            ([(args.tokens, ALPHA)] if args.tokens else [(8192, ALPHA), (32768, ALPHA)])
        out["mxfp8_fwd_bwd"] = [bench_mx_fwd_bwd(args, dev, ws, peaks, Tm, a) for Tm, a in grid]
        big = [m for m in out["mxfp8_fwd_bwd"] if m["T"] == 32768 and m["zipf_alpha"] == ALPHA]
        if big:
            m = big[0]
            gg = m["grouped_gemms"]["all_six"]["frac"]
            lf = m["layer_roofline"]["frac"]
            out["largest_config_target"] = {
                "workload": m["workload"], "grouped_gemms_frac_of_fp8_peak": gg, "layer_frac_of_roofline": lf,
                "layer_bound": m["layer_roofline"]["bound"], "targets": {"grouped_gemms": 0.6, "layer": 0.5},
                "met": bool(gg >= 0.6 and lf >= 0.5),
                "note": "the six block-scaled expert GEMMs' padding-free FLOPs over their summed device time, "
                        "against 2 x the measured sustained bf16 peak"}
        if not args.tokens:
            out["mxfp8_minibatch_sweep"] = bench_minibatch_sweep(args, dev, ws)
    if not args.no_nv:
        from mixture_experts_layer_19_gb300 import moe
        if args.no_mx:
            del plan, inp, grads, saved, Y
            torch.cuda.empty_cache()
        out["nvfp4_forward"] = [bench_mx_forward(args, dev, ws, peaks, ALPHA, prec=moe.MOE_NVFP4)]
        out["nvfp4_fwd_bwd"] = [bench_mx_fwd_bwd(args, dev, ws, peaks, Tn, ALPHA, prec=moe.MOE_NVFP4)
                                for Tn in ((args.tokens,) if args.tokens else (4096, 8192))]
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def bench_ep(args, plan_one, inp, Y, saved, grads, stream, dev, ws, ranks=8):
    """The same fwd+bwd step as expert parallelism over `ranks` virtual ranks
    on the one GPU (pull dispatch / push combine and their reverses as
    flag-signalled cooperative launches); bitwise equal to the headline path."""
    from mixture_experts_layer_19_gb300 import moe
    c = plan_one.cfg
    plan = moe.Plan(moe.Config(T_max=c.T_max, d=c.d, F=c.F, E=c.E, k=c.k, device=dev.index, ep_ranks=ranks,
                               debug_flags=moe.MOE_DEBUG_TIMING))

    def step():
        plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    plan.kernel_times()
    steps = max(3, args.steps // 2)
    barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if plan.device_status() != 0:
        raise RuntimeError("device status set in the virtual-rank EP step")
    kt = plan.kernel_times()
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev) / steps
    res = {"ranks": ranks, "ms_per_step": round(ms, 4),
           "value": round(ws * inp.X.shape[0] / (ms / 1e3), 1), "unit": "tokens/s",
           "exchange_ms": {n: round(v[0] / steps, 4) for n, v in kt.items() if n.startswith("ep_")}}
    del plan
    return res


def bench_graph(args, inp, ref, dev, ws):
    """The same fwd+bwd step captured once as a CUDA graph and replayed (a plan
    without per-kernel timing events, so the graph holds only the layer's
    kernels); the replayed outputs must equal the eager step's bitwise."""
    from mixture_experts_layer_19_gb300 import moe
    T, d = inp.X.shape
    E, F = inp.Wg.shape[0], inp.Wg.shape[1]
    k = ref["dg"].shape[1]
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, device=dev.index or 0))
    saved = plan.new_saved(T)
    Y = torch.empty_like(ref["Y"])
    grads = {n: torch.empty_like(ref[n]) for n in ("dX", "dWg", "dWu", "dWd", "dg", "dlogits")}
    stream = torch.cuda.Stream(dev)

    def step():
        plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    if plan.device_status() != 0:
        raise RuntimeError("device status set during the graph replays")
    same = torch.equal(Y, ref["Y"]) and all(torch.equal(grads[n], ref[n]) for n in grads)
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    res = {"ms_per_step": round(elapsed_ms / args.steps, 4),
           "value": round(ws * T * args.steps / (elapsed_ms / 1e3), 1), "unit": "tokens/s",
           "bitwise_equal_to_eager": bool(same),
           "note": "one fwd+bwd step captured once as a CUDA graph (no per-kernel timing events) and replayed"}
    del graph, plan, saved, Y, grads
    torch.cuda.empty_cache()
    return res


def bench_router(args, plan, inp, stream, dev, ws, peaks):
    """Router GEMM in front of the layer (logits = X Wr^T) and its backward
    (dX += dlogits Wr, dWr = dlogits^T X) on the headline shape."""
    c = plan.cfg
    T = inp.X.shape[0]
    gen = torch.Generator(device=dev).manual_seed(SEED + 1)
    Wr = (torch.randn((c.E, c.d), generator=gen, device=dev) / math.sqrt(c.d)).to(torch.bfloat16)
    dlog = torch.randn((T, c.E), generator=gen, device=dev)
    dX = torch.zeros((T, c.d), dtype=torch.bfloat16, device=dev)
    dWr = torch.empty((c.E, c.d), dtype=torch.bfloat16, device=dev)
    logits = torch.empty((T, c.E), dtype=torch.float32, device=dev)
    steps = max(3, args.steps // 2)
    res = {}
    for name, fn in (("forward", lambda: plan.router_forward(inp.X, Wr, logits, stream=stream)),
                     ("backward", lambda: plan.router_backward(inp.X, Wr, dlog, dX, dWr, stream=stream))):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        barrier(ws)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev) / steps
        flops = (2 if name == "forward" else 4) * T * c.E * c.d
        res[name] = {"ms": round(ms, 4), "tflops": round(flops / (ms / 1e3) / 1e12, 1)}
    plan.kernel_times()
    if plan.device_status() != 0:
        raise RuntimeError("device status set in the router GEMM")
    res["shape"] = {"T": T, "E": c.E, "d": c.d}
    return res


def bench_ring(args, plan_sep, inp, Y, saved, grads, stream, dev, ws):
    """The bf16 schedules on the headline workload, forward alone and the
    whole fwd+bwd step: separate kernels (the default), the ring pipeline as
    one launch per direction (forward megakernel with routing and combine
    inside; backward megakernel with the dY gather, u and dx GEMMs, dX sums
    and router gradient inside; the weight gradients after it), and the ring
    forward between separate routing / combine launches.  All are bitwise
    identical to one another."""
    from mixture_experts_layer_19_gb300 import moe
    c = plan_sep.cfg
    res = {}
    schedules = (("separate", plan_sep), ("ring_one_launch", None), ("ring_multi_launch", None))
    flag_of = {"ring_one_launch": moe.MOE_DEBUG_RING_MEGAKERNEL,
               "ring_multi_launch": moe.MOE_DEBUG_RING_MEGAKERNEL | moe.MOE_DEBUG_MULTI_LAUNCH}
    steps = max(3, args.steps // 2)

    def timed(plan, fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        plan.kernel_times()
        barrier(ws)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if plan.device_status() != 0:
            raise RuntimeError("device status set in the ring measurement")
        kt = plan.kernel_times()
        return round(max_over_ranks(ev0.elapsed_time(ev1), ws, dev) / steps, 4), \
            {n: round(v[0] / steps, 4) for n, v in sorted(kt.items(), key=lambda x: -x[1][0])}

    for name, plan in schedules:
        own = plan is None
        if own:
            plan = moe.Plan(moe.Config(T_max=c.T_max, d=c.d, F=c.F, E=c.E, k=c.k, device=dev.index,
                                       debug_flags=flag_of[name] | moe.MOE_DEBUG_TIMING))

        def fwd():
            plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)

        def step():
            fwd()
            plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

        f_ms, f_k = timed(plan, fwd)
        s_ms, s_k = timed(plan, step)
        res[name] = {"fwd_ms": f_ms, "fwd_kernels": f_k, "fwd_bwd_ms": s_ms, "fwd_bwd_kernels": s_k}
        if own:
            del plan
    return res


def _block_format(prec):
    """(name, kernel-name tag, tensor-peak multiple of bf16, bytes per weight value incl. scales, dtype)."""
    from mixture_experts_layer_19_gb300 import moe
    if prec == moe.MOE_NVFP4:
        return ("nvfp4", "nv", 6.0, 0.5 + 1 / 16,
                "e2m1 + e4m3 scale per 16 + fp32 tensor scale (fp32 accumulate, bf16 out)")
    return "mxfp8", "mx", 2.0, 1 + 1 / 32, "e4m3+e8m0 (fp32 accumulate, bf16 out)"


def bench_mx_forward(args, dev, ws, peaks, alpha, prec=None):
    """Block-scaled forward of the layer at T=16384 (uniform or Zipf routing):
    quantising gather, block-scaled [a|b] GEMM + SwiGLU + h re-quantisation,
    block-scaled down GEMM, combine; MXFP8 (with the ring megakernel beside
    the default schedule) or NVFP4.  Weight quantisation (once per optimiser
    step) is timed on its own and is not part of the step."""
    from mixture_experts_layer_19_gb300 import moe
    prec = moe.MOE_MXFP8 if prec is None else prec
    fname, tag, mult, wbytes, dtype = _block_format(prec)
    # --tokens / --experts shrink the layer for profiler captures only
    T, d, F, k = args.tokens or MX_SHAPE["T"], SHAPE["d"], SHAPE["F"], SHAPE["k"]
    E = args.experts or SHAPE["E"]
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=SEED, alpha=alpha, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run(flags, steps):
        plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, device=dev.index,
                                   debug_flags=moe.MOE_DEBUG_TIMING | flags))
        # the first call also pays for loading the kernels; time the second
        plan.quantize_weights(inp.Wg, inp.Wu, inp.Wd, stream=stream)
        torch.cuda.synchronize(dev)
        plan.kernel_times()
        plan.quantize_weights(inp.Wg, inp.Wu, inp.Wd, stream=stream)
        wq = plan.kernel_times()
        saved = plan.new_saved(T)
        Y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup):
            plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        torch.cuda.synchronize(dev)
        plan.kernel_times()
        barrier(ws)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if plan.device_status() != 0:
            raise RuntimeError(f"device status set in the {fname} forward")
        el = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
        kt = plan.kernel_times()
        e_act = active_experts(plan, saved, T)
        del plan, saved, Y
        return el, kt, wq, e_act

    # default schedule (separate kernels); for MXFP8 the ring megakernel beside it
    el, kt, wq, e_act = run(0, args.steps)
    R = T * k
    tpeak = mult * peaks["bf16_tflops_sustained"]      # nominal fp8 (x2) / fp4 (x6) : bf16 dense ratio
    up_ms = kt[f"gemm_{tag}_up_swiglu"][0] / kt[f"gemm_{tag}_up_swiglu"][1]
    dn_ms = kt[f"gemm_{tag}_down"][0] / kt[f"gemm_{tag}_down"][1]
    up_tf = 4.0 * R * d * F / (up_ms / 1e3) / 1e12
    dn_tf = 2.0 * R * d * F / (dn_ms / 1e3) / 1e12
    ms = el / args.steps
    t_tc = 6.0 * R * d * F / (tpeak * 1e12) * 1e3
    t_hbm = (3.0 * e_act * F * d * wbytes + T * d * 2 * 2 + T * E * 4) / (peaks["hbm_gbs"] * 1e9) * 1e3
    res = {
        "workload": f"moe_layer_fwd_{fname}_T{T}_d{d}_F{F}_E{E}_top{k}_zipf{alpha:g}", "experts_active": e_act,
        "value": round(ws * T * args.steps / (el / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
        "dtype": dtype,
        "roofline": {"kernel": f"gemm_{tag}_up_swiglu", "bound": "tensor", "achieved": round(up_tf, 1),
                     "peak": round(tpeak, 1), "unit": "TFLOP/s", "frac": round(up_tf / tpeak, 4),
                     "traffic": None,
                     "peak_source": peaks["source"] + f" bf16_tflops_sustained x {mult:g} (nominal "
                                                      f"{'fp4' if tag == 'nv' else 'fp8'}:bf16 ratio)"},
        "down_gemm": {"achieved": round(dn_tf, 1), "unit": "TFLOP/s", "frac": round(dn_tf / tpeak, 4)},
        "layer_roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "t_ms": round(max(t_tc, t_hbm), 4),
                           "frac": round(max(t_tc, t_hbm) / ms, 4)},
        "kernels": {n: {"ms_per_step": round(v[0] / args.steps, 4), "launches": v[1]} for n, v in kt.items()},
        "weight_quant_ms": round(wq.get("quant_weights", (0.0, 0))[0], 3),
    }
    if prec == moe.MOE_MXFP8:
        el_ring, ktr, _, _ = run(moe.MOE_DEBUG_RING_MEGAKERNEL, max(3, args.steps // 2))
        mk_ms = ktr["fwd_megakernel_mx"][0] / ktr["fwd_megakernel_mx"][1]
        mk_tf = 6.0 * R * d * F / (mk_ms / 1e3) / 1e12
        res["ring_megakernel"] = {"ms_per_step": round(el_ring / max(3, args.steps // 2), 4),
                                  "megakernel_ms": round(mk_ms, 4), "achieved": round(mk_tf, 1), "unit": "TFLOP/s",
                                  "frac": round(mk_tf / tpeak, 4), "flops": "6*R*d*F per launch"}
    del inp
    torch.cuda.empty_cache()
    return res


def _alloc_grads(T, d, F, E, k, dev):
    return {
        "dX": torch.empty((T, d), dtype=torch.bfloat16, device=dev),
        "dWg": torch.empty((E, F, d), dtype=torch.bfloat16, device=dev),
        "dWu": torch.empty((E, F, d), dtype=torch.bfloat16, device=dev),
        "dWd": torch.empty((E, d, F), dtype=torch.bfloat16, device=dev),
        "dg": torch.empty((T, k), dtype=torch.float32, device=dev),
        "dlogits": torch.empty((T, E), dtype=torch.float32, device=dev),
    }


def bench_mx_fwd_bwd(args, dev, ws, peaks, T, alpha, prec=None):
    """Block-scaled (MXFP8 or NVFP4) forward + backward at T tokens: every
    expert GEMM block-scaled (forward, dgrad, and the weight gradients with
    their operands quantised along the tokens).  Layer roofline:
    max(18RdF / fp8 or fp4 peak, (quantised weights fwd + bwd orientation +
    bf16 dW) / HBM)."""
    from mixture_experts_layer_19_gb300 import moe
    prec = moe.MOE_MXFP8 if prec is None else prec
    fname, _, mult, wbytes, _ = _block_format(prec)
    d, F, k = SHAPE["d"], SHAPE["F"], SHAPE["k"]
    E = args.experts or SHAPE["E"]
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=SEED, alpha=alpha, device=dev)
    plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, device=dev.index,
                               debug_flags=moe.MOE_DEBUG_TIMING))
    stream = torch.cuda.current_stream(dev)
    plan.quantize_weights(inp.Wg, inp.Wu, inp.Wd, stream=stream)
    saved = plan.new_saved(T)
    Y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    grads = _alloc_grads(T, d, F, E, k, dev)

    def step():
        plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
        plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    plan.kernel_times()
    barrier(ws)
    steps = max(3, args.steps // 2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if plan.device_status() != 0:
        raise RuntimeError(f"device status set in the {fname} fwd+bwd")
    el = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    kt = plan.kernel_times()
    e_act = active_experts(plan, saved, T)
    R = T * k
    tpeak = mult * peaks["bf16_tflops_sustained"]
    t_tc = 18.0 * R * d * F / tpeak / 1e12 * 1e3
    # quantised weights of the active experts in both orientations, bf16 dW of every expert
    t_hbm = (2 * 3.0 * e_act * F * d * wbytes + 3.0 * E * F * d * 2) / (peaks["hbm_gbs"] * 1e9) * 1e3
    ms = el / steps
    # each expert GEMM against the dense tensor peak of its format (padding-free FLOPs)
    tag = "nv" if prec == moe.MOE_NVFP4 else "mx"
    gemm_flops = {"up_swiglu": 4, "down": 2, "bwd_u_swiglu": 2, "bwd_dx": 4, "wgrad_down": 2, "wgrad_gate_up": 4}
    gemms = {}
    for kind, mul in gemm_flops.items():
        name = f"gemm_{tag}_{kind}"
        if name in kt:
            g_ms = kt[name][0] / kt[name][1]
            tf = mul * R * d * F / (g_ms / 1e3) / 1e12
            gemms[name] = {"ms": round(g_ms, 4), "achieved": round(tf, 1), "unit": "TFLOP/s",
                           "frac": round(tf / tpeak, 4)}
    g_tot_ms = sum(v["ms"] for v in gemms.values())
    all_tf = 18.0 * R * d * F / (g_tot_ms / 1e3) / 1e12 if g_tot_ms else 0.0
    res = {"workload": f"moe_layer_fwd_bwd_{fname}_T{T}_zipf{alpha:g}", "T": T, "zipf_alpha": alpha,
           "experts_active": e_act,
           "value": round(ws * T * steps / (el / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "layer_roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "t_ms": round(max(t_tc, t_hbm), 4),
                              "frac": round(max(t_tc, t_hbm) / ms, 4)},
           "grouped_gemms": {"peak": round(tpeak, 1), "unit": "TFLOP/s",
                             "peak_source": peaks["source"] + f" bf16_tflops_sustained x {mult:g}",
                             "all_six": {"ms": round(g_tot_ms, 4), "achieved": round(all_tf, 1),
                                         "frac": round(all_tf / tpeak, 4)},
                             "per_kind": gemms},
           "kernels": {n: round(v[0] / steps, 4) for n, v in sorted(kt.items(), key=lambda x: -x[1][0])}}
    del plan, inp, saved, Y, grads
    torch.cuda.empty_cache()
    return res


def bench_minibatch_sweep(args, dev, ws, T=8192, alphas=(0.0, 1.1, 1.5), prec=None,
                          rows=(512, 1024, 2048, 0, 4096, 8192)):
    """Layer step time versus the ring pipeline's minibatch size (rows per
    ring slot fill; 0 = the two-wave floor), forward + backward, for each
    routing skew: the ring megakernel forward's time and the whole step's."""
    from mixture_experts_layer_19_gb300 import moe
    prec = moe.MOE_MXFP8 if prec is None else prec
    fname = {moe.MOE_BF16: "bf16", moe.MOE_MXFP8: "mxfp8", moe.MOE_NVFP4: "nvfp4"}[prec]
    d, F, E, k = SHAPE["d"], SHAPE["F"], SHAPE["E"], SHAPE["k"]
    stream = torch.cuda.current_stream(dev)
    steps = max(3, args.steps // 4)
    out = []
    for alpha in alphas:
        inp = make_inputs(LayerShape(T, d, F, E, k), seed=SEED, alpha=alpha, device=dev)
        grads = _alloc_grads(T, d, F, E, k, dev)
        for mb in rows:
            plan = moe.Plan(moe.Config(T_max=T, d=d, F=F, E=E, k=k, prec=prec, minibatch_rows=mb,
                                       device=dev.index,
                                       debug_flags=moe.MOE_DEBUG_RING_MEGAKERNEL | moe.MOE_DEBUG_TIMING))
            if prec != moe.MOE_BF16:
                plan.quantize_weights(inp.Wg, inp.Wu, inp.Wd, stream=stream)
            saved = plan.new_saved(T)
            Y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)

            def step():
                plan.forward(inp.X, inp.logits, inp.Wg, inp.Wu, inp.Wd, Y=Y, saved=saved, stream=stream)
                plan.backward(inp.dY, inp.X, inp.Wg, inp.Wu, inp.Wd, saved, out=grads, stream=stream)

            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize(dev)
            plan.kernel_times()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(steps):
                step()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            if plan.device_status() != 0:
                raise RuntimeError("device status set in the minibatch sweep")
            kt = plan.kernel_times()
            mk = [n for n in kt if n.startswith("fwd_megakernel")]
            info = plan.info()
            out.append({"zipf_alpha": alpha, "minibatch_rows": mb if mb else "two-wave floor",
                        "minibatch_tiles": info["minibatch_tiles"],
                        "step_ms": round(max_over_ranks(ev0.elapsed_time(ev1), ws, dev) / steps, 4),
                        "megakernel_ms": round(sum(kt[n][0] for n in mk) / steps, 4)})
            del plan, saved, Y
        del inp, grads
        torch.cuda.empty_cache()
    return {"workload": f"{fname} fwd+bwd with the ring megakernel forward, T={T}, d={d}, F={F}, E={E}, top{k}",
            "points": out}


def bench_e2e(args, plan, inp, Y, saved, grads, stream, dev, ws):
    """Same fwd+bwd through the public API with pinned HOST inputs and results:
    each step copies X, logits, dY host->device and Y, dX device->host.

    The copies run on a second stream against double-buffered device inputs
    and outputs, ordered by events: step i+1's inputs arrive while step i
    computes, and step i's results leave while step i+1 computes.  Every
    step's copies are inside the timed region (the region ends when the last
    result is on the host)."""
    hX = inp.X.cpu().pin_memory()
    hL = inp.logits.cpu().pin_memory()
    hdY = inp.dY.cpu().pin_memory()
    hY = torch.empty_like(hX).pin_memory()
    hdX = torch.empty_like(hX).pin_memory()
    copy = torch.cuda.Stream(dev)
    bufs = []
    for b in range(2):
        bufs.append({"X": torch.empty_like(inp.X), "L": torch.empty_like(inp.logits),
                     "dY": torch.empty_like(inp.dY), "Y": Y if b == 0 else torch.empty_like(Y),
                     "dX": grads["dX"] if b == 0 else torch.empty_like(grads["dX"]),
                     "in_ready": torch.cuda.Event(), "computed": torch.cuda.Event(), "drained": torch.cuda.Event()})
    for b in bufs:      # nothing is pending on either buffer yet
        b["computed"].record(stream)
        b["drained"].record(copy)
    out = dict(grads)

    def h2d(b):
        with torch.cuda.stream(copy):
            copy.wait_event(b["computed"])            # the previous step on b has read its inputs
            b["X"].copy_(hX, non_blocking=True)
            b["L"].copy_(hL, non_blocking=True)
            b["dY"].copy_(hdY, non_blocking=True)
            b["in_ready"].record(copy)

    def compute(b):
        stream.wait_event(b["in_ready"])
        stream.wait_event(b["drained"])               # the previous results in b reached the host
        out["dX"] = b["dX"]
        plan.forward(b["X"], b["L"], inp.Wg, inp.Wu, inp.Wd, Y=b["Y"], saved=saved, stream=stream)
        plan.backward(b["dY"], b["X"], inp.Wg, inp.Wu, inp.Wd, saved, out=out, stream=stream)
        b["computed"].record(stream)

    def d2h(b):
        with torch.cuda.stream(copy):
            copy.wait_event(b["computed"])
            hY.copy_(b["Y"], non_blocking=True)
            hdX.copy_(b["dX"], non_blocking=True)
            b["drained"].record(copy)

    def run(n):
        h2d(bufs[0])
        for i in range(n):
            cur, nxt = bufs[i % 2], bufs[(i + 1) % 2]
            compute(cur)
            if i + 1 < n:
                h2d(nxt)
            d2h(cur)

    run(max(1, args.warmup // 2))
    torch.cuda.synchronize(dev)
    plan.kernel_times()
    barrier(ws)
    t0 = time.perf_counter()
    run(args.steps)
    torch.cuda.synchronize(dev)
    barrier(ws)
    el = time.perf_counter() - t0
    plan.kernel_times()
    el = max_over_ranks(el, ws, dev)
    T = inp.X.shape[0]
    h2d_bytes = hX.numel() * 2 + hL.numel() * 4 + hdY.numel() * 2
    d2h_bytes = hY.numel() * 2 + hdX.numel() * 2
    return {"value": round(ws * T * args.steps / el, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d_bytes),
            "d2h_bytes_per_step": int(d2h_bytes),
            "copies": "on a second stream, double-buffered, overlapped with the neighbouring steps' compute"}


def cpu_baseline(inp, k, n_tokens):
    cores = cpu_cores()
    lim = set_blas_threads(cores)
    toks = np.arange(n_tokens)
    s = oracle_sample(inp, toks, k)
    t0 = time.perf_counter()
    run_oracle(s, k)
    el = time.perf_counter() - t0
    del lim
    return {"value": round(n_tokens / el, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of the first {n_tokens} tokens of the same workload as one batch "
                      f"({s['experts']} experts touched; {el:.1f} s)"}


def bench_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    shape = dict(SHAPE)
    T, d, F, E, k = (shape[n] for n in ("T", "d", "F", "E", "k"))
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp = make_inputs(LayerShape(T, d, F, E, k), seed=SEED, alpha=ALPHA, device=dev)
    cores = cpu_cores()
    set_blas_threads(cores)
    per = args.ref_tokens
    samples = [oracle_sample(inp, np.arange(i * per, (i + 1) * per) % T, k)
               for i in range(args.warmup + args.steps)]
    for s in samples[:args.warmup]:
        run_oracle(s, k)
    t0 = time.perf_counter()
    for s in samples[args.warmup:]:
        run_oracle(s, k)
    el = time.perf_counter() - t0
    value = per * args.steps / el
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T, "d": d, "F": F, "E": E, "k": k, "zipf_alpha": ALPHA,
                   "seed": SEED, "tokens_per_step": per},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 oracle fwd+bwd of {per} consecutive tokens of the workload"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=128, help="tokens in the timed CPU-oracle sample")
    ap.add_argument("--ref-tokens", type=int, default=1, help="tokens per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiler captures on a smaller layer)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiler captures on a smaller layer)")
    ap.add_argument("--no-mx", action="store_true", help="skip the MXFP8 measurements")
    ap.add_argument("--no-nv", action="store_true", help="skip the NVFP4 measurements")
    ap.add_argument("--no-ring", action="store_true", help="skip the ring-pipeline line (forward and fwd+bwd)")
    ap.add_argument("--no-ep", action="store_true", help="skip the virtual-rank expert-parallel line")
    ap.add_argument("--sweep", action="store_true",
                    help="MXFP8 fwd+bwd over T in {2048, 8192, 32768} x zipf {0, 1.1, 1.5} and a minibatch sweep")
    ap.add_argument("--dry-run", action="store_true",
                    help="start the ranks and exchange timings on the CPU (gloo) without any GPU work")
    argv = sys.argv[1:] if argv is None else list(argv)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args, argv))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws != args.gpus:
        ap.error(f"--gpus {args.gpus} but the launcher started {ws} ranks")
    if args.dry_run:
        bench_dry_run(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
