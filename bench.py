#!/usr/bin/env python
"""Benchmark of the routed SwiGLU expert layer: one step = schedule + forward + backward.

Default workload: the imbalance / granularity sweep at Zipf s = 1 in BF16 -- T=8192 tokens,
H=4096, I=1536, E=128 experts, top-8, expert loads skewed by Gumbel-top-k sampling on
-ln(e+1) logits -- with synthetic seeded inputs.  The same line carries two further objects timed
the same way: "mxfp8" (the same sweep in MXFP8) and "ep64_shard" (the per-GPU shard of an EP64
layer in MXFP8: 16,384 routed rows onto 4 experts, H=7168, I=2048, Zipf 1.2).  Prints ONE JSON line
(rank 0):
  value     tokens/s of the whole job (all ranks), inputs resident in HBM, CUDA events on the
            launching stream, max over ranks.  The step runs as in training: captured once as a
            CUDA graph (every launch through the C ABI) and replayed; "step" also reports the same
            K steps launched eagerly from the host (--no-graph times those instead);
  e2e       the same metric through the C ABI with host (pinned) inputs: H2D of x, ids, weights,
            dY and D2H of out, dX, d_topk_weights for every timed step, double-buffered over a
            copy stream so transfers overlap the neighbouring steps' compute (one graph per buffer
            set);
  roofline  the dominant kernel's algorithmic flops (or bytes) per launch over its average launch
            time, measured live with per-launch CUDA events (the library's trace hook), against
            the measured peak;
  cpu_baseline  the CPU oracle's layer loops built in fp32 at -O3 (OpenMP over all host cores),
            timed on a bounded token sample; the fp64 build stays the parity reference.
``--impl reference`` times the oracle alone (the reference arm; rank 0 only).

Multi-GPU (torchrun): every rank runs an independent data-parallel shard of the same shape (its
own tokens); the layer has no collective, so N ranks are N replicas (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s on 1×GB300 (BF16, MXFP8); % of tensor/HBM peak"
UNIT = "tokens/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="sweep_zipf1")
    p.add_argument("--extra", default="mxfp8=sweep_zipf1_mx,ep64_shard=mxfp8_ep64_shard",
                   help="further workloads timed into objects of the same line (key=workload,...; '' for none)")
    p.add_argument("--minibatch", type=int, default=512)
    p.add_argument("--macrobatch", type=int, default=2048)
    p.add_argument("--num-ctas", type=int, default=0, help="persistent GEMM grid (0: one CTA per SM)")
    p.add_argument("--static-tiles", action="store_true",
                   help="static round-robin GEMM tiles instead of cluster launch control")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU seconds of the oracle sample")
    return p.parse_args()


# ------------------------------------------------------------------------------------------------
# distributed plumbing
# ------------------------------------------------------------------------------------------------
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def aggregate_tokens_per_s(tokens_per_rank: int, ws: int, ms_max: float) -> float:
    """Whole-job throughput of the replicas: every rank processes its own shard of tokens_per_rank
    (weak scaling); the job takes as long as the slowest rank."""
    return tokens_per_rank * ws / (ms_max * 1e-3)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.marks = {}

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="mok_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            except ValueError:
                ts = 0.0
            try:
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        t0, t1 = self.marks.get("t0"), self.marks.get("t1")
        timed = [r for r in rows if t0 is not None and t0 - 0.05 <= r["ts"] <= t1 + 0.05]
        window = "timed region"
        if len(timed) < 3:  # short timed region: use every sample of the benchmark run
            timed, window = rows, "whole benchmark run (timed region shorter than the sampling period)"
        if not timed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in timed:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        loaded = [r["sm"] for r in timed if r["power"] > 200.0] or [r["sm"] for r in timed]
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": max(r["smax"] for r in timed),
                "reasons": sorted(reasons), "samples": len(timed), "window": window,
                "power_w_max": max(r["power"] for r in timed)}


# ------------------------------------------------------------------------------------------------
# algorithmic work per kernel (flops for tensor-core kernels, bytes for the HBM-bound ones)
# ------------------------------------------------------------------------------------------------
def kernel_work(w, e_active: int) -> dict:
    """Algorithmic (flops, HBM bytes, operand type) of one launch of each kernel.  Bytes count each
    tensor the kernel must read or write once: gathered rows R (not the padded rows), the weights of
    the experts that received rows, the fp32 weight gradients of every expert.  MXFP8 operands
    count 1 + 1/32 bytes per element (E4M3 code + its share of the E8M0 scale)."""
    R, H, I, T, K, E = w.R, w.H, w.I, w.T, w.K, w.E
    b16 = 2
    work = {
        # combine / dX reduce: routed rows read + weights/indices + token rows written
        "combine": (0, R * H * b16 + T * K * 8 + T * H * b16, None),
        "dx_reduce": (0, R * H * b16 + T * K * 4 + T * H * b16, None),
    }
    if w.precision == "mxfp8":
        mx = 1 + 1 / 32
        wts = e_active * H * I * mx  # one quantised weight matrix of the active experts
        work.update({
            # reads Xq, Wg, Wu; writes g, u (fp32), a (bf16) and its MX copy
            "gemm_fwd_gateup": (4 * R * H * I, R * H * mx + 2 * wts + R * 2 * I * 4 + R * I * (b16 + mx), "e4m3"),
            "gemm_fwd_down": (2 * R * H * I, R * I * mx + wts + R * H * b16, "e4m3"),
            # reads dYq, Wd^T, g, u (fp32), a_q; writes [dg | du] quantised along I and along the rows,
            # s*a quantised along the rows, dS partials
            "gemm_dgrad1": (2 * R * H * I, R * H * mx + wts + R * 2 * I * 4 + R * I * b16
                            + 2 * R * 2 * I * mx + R * I * mx + R * (I // 128) * 4, "e4m3"),
            "gemm_dgrad2": (4 * R * H * I, R * 2 * I * mx + 2 * wts + R * H * b16, "e4m3"),
            # block-scaled on the operands quantised along the routed rows; fp32 dW of every expert
            "gemm_wgrad_gu": (4 * R * H * I, R * 2 * I * mx + R * H * mx + 2 * E * I * H * 4, "e4m3"),
            "gemm_wgrad_d": (2 * R * H * I, R * H * mx + R * I * mx + E * H * I * 4, "e4m3"),
            # gather: unique token rows read once; routed rows written quantised along H and along the rows
            "gather_x": (0, T * H * b16 + 2 * R * H * mx, None),
            "gather_dy": (0, T * H * b16 + 2 * R * H * mx, None),
            # three weight-scale matrices re-tiled into atoms per launch (read + write)
            "mx_scale_atoms": (0, 2 * 3 * E * H * I / 32, None),
        })
    else:
        wts = e_active * H * I * b16
        work.update({
            "gemm_fwd_gateup": (4 * R * H * I, R * H * b16 + 2 * wts + R * 2 * I * b16 + R * I * b16, "bf16"),
            "gemm_fwd_down": (2 * R * H * I, R * I * b16 + wts + R * H * b16, "bf16"),
            "gemm_dgrad1": (2 * R * H * I, R * H * b16 + wts + R * 2 * I * b16 + R * I * b16 + R * 3 * I * b16,
                            "bf16"),
            "gemm_dgrad2": (4 * R * H * I, R * 2 * I * b16 + 2 * wts + R * H * b16, "bf16"),
            "gemm_wgrad_gu": (4 * R * H * I, R * 2 * I * b16 + R * H * b16 + 2 * E * I * H * 4, "bf16"),
            "gemm_wgrad_d": (2 * R * H * I, R * H * b16 + R * I * b16 + E * H * I * 4, "bf16"),
            "gather_x": (0, T * H * b16 + R * H * b16, None),
            "gather_dy": (0, T * H * b16 + R * H * b16, None),
        })
    return work


# dense tensor-core peak of an operand type relative to bf16 (nominal 4.5 vs 2.25 PFLOP/s for e4m3)
TENSOR_RATIO = {"bf16": 1.0, "e4m3": 2.0}


def roofline_of(flops, nbytes, ms, peaks, kind="bf16"):
    """The kernel's bound is the larger of its tensor time (at the measured bf16 peak times the
    nominal ratio of its operand type) and its HBM time at the measured copy bandwidth."""
    tpeak = peaks["bf16_tflops"] * TENSOR_RATIO[kind or "bf16"]
    t_tensor = flops / (tpeak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    sec = ms * 1e-3
    if t_tensor >= t_hbm:
        return dict(bound="tensor", achieved=flops / sec / 1e12, peak=tpeak, unit="TFLOP/s",
                    frac=t_tensor / sec, operands=kind)
    return dict(bound="hbm", achieved=nbytes / sec / 1e9, peak=peaks["hbm_gbs"], unit="GB/s", frac=t_hbm / sec)


def _code_only(text: str) -> bytes:
    """Source text without comments, trailing blanks and empty lines: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/|//[^\n]*", "", text, flags=re.S)
    return "\n".join(l.rstrip() for l in text.splitlines() if l.strip()).encode()


def src_hash() -> str:
    """Hash of the CUDA sources of the layer kernels and the ABI header (code only), keying the
    stored ncu counters (all of them belong to layer kernels; the router's file is left out)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_layer_build_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and f != "mok_router.cu":
            h.update(_code_only(open(os.path.join(csrc, f)).read()))
    h.update(_code_only(open(os.path.join(ROOT, "include", "mok.h")).read()))
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def traffic_for(kernel: str, workload: str):
    if not os.path.exists(PROFILE_TRAFFIC):
        return None, "no ncu capture committed"
    d = json.load(open(PROFILE_TRAFFIC))
    e = d.get(workload, {}).get(kernel)
    if not e:
        return None, "kernel not captured"
    if e.get("src_hash") != src_hash():
        return None, "kernel changed since the counters were taken"
    return e["dram_bytes_per_launch"], e.get("note", "")


# ------------------------------------------------------------------------------------------------
# CPU oracle timing
# ------------------------------------------------------------------------------------------------
def oracle_sample_args(d, tokens: int):
    from mixture_experts_layer_build_gb300 import inputs
    ids = d["topk_ids"][:tokens].numpy()
    s = d["topk_weights"][:tokens].numpy()
    x = inputs.bits(d["x"][:tokens])
    dY = inputs.bits(d["dY"][:tokens])
    return ids, s, x, dY


def time_oracle_step(d, wbits, tokens: int) -> float:
    """One oracle fwd + bwd of the first `tokens` tokens.  wbits = (Wg, Wu, Wd) bf16 bit patterns
    for the BF16 layer loops (their fp32 -O3 build), or a dict of pre-quantised copies for the
    MXFP8 oracle (fp64; it has no fp32 build)."""
    import oracle
    ids, s, x, dY = oracle_sample_args(d, tokens)
    t0 = time.perf_counter()
    if isinstance(wbits, dict):
        E, I = d["Wg"].shape[0], d["Wg"].shape[1]
        oracle.layer_mx(ids, s, x, dY, wbits, E, I)
    else:
        Wg, Wu, Wd = wbits
        oracle.step_f32(ids, s, x, Wg, Wu, Wd, dY)
    return time.perf_counter() - t0


def oracle_kind(wbits) -> str:
    return ("fp64 MXFP8 oracle (C loops, OpenMP)" if isinstance(wbits, dict)
            else "the oracle's layer loops in fp32, gcc -O3 -fopenmp")


def calibrate_oracle_tokens(d, wbits, target_s: float, T: int) -> tuple[int, float]:
    """Token count whose oracle fwd+bwd takes about target_s, from a linear fit through 8- and
    32-token runs (the oracle's fixed cost is the dense dW initialisation)."""
    a, b = min(8, T), min(32, T)
    ta = time_oracle_step(d, wbits, a)
    tb = time_oracle_step(d, wbits, b)
    slope = (tb - ta) / (b - a) if b > a else tb / max(b, 1)
    if slope <= 0:
        slope = tb / b
    fixed = max(ta - slope * a, 0.0)
    tokens = int(max(a, min(T, (target_s - fixed) / slope)))
    return tokens, tb


def cores_used():
    import oracle
    return oracle.num_threads()


# ------------------------------------------------------------------------------------------------
def reference_arm(args, rank, ws):
    """The oracle timed as it stands (fp64 C loops, all host cores), step = fwd + bwd of a bounded
    token sample of the workload."""
    if rank != 0:
        return
    from mixture_experts_layer_build_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    d = inputs.make(w, seed=0)
    wbits = (inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
    if w.precision == "mxfp8":
        import oracle
        wbits = oracle.mx_weights(*wbits)
    per_step_budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    tokens, _ = calibrate_oracle_tokens(d, wbits, per_step_budget, w.T)
    for _ in range(args.warmup):
        time_oracle_step(d, wbits, tokens)
    times = [time_oracle_step(d, wbits, tokens) for _ in range(args.steps)]
    t = float(np.mean(times))
    value = tokens / t
    cores = cores_used()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64" if isinstance(wbits, dict) else "f32",
        "data": "synthetic", "config": config_of(w, args, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"fwd+bwd of the first {tokens} of {w.T} tokens per step (all their routed "
                                   f"rows, full dW), {oracle_kind(wbits)}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


WORKLOAD_TITLES = {
    "tiny": "tiny layer",
    "bf16_e64": "near-uniform softmax routing",
    "dsv3_e256": "DeepSeek-V3-style layer, all 256 experts resident, per-expert router bias",
    "mxfp8_ep64_shard": "per-GPU shard of an EP64 layer (2048 tokens x top-8 onto 4 local experts, Zipf 1.2)",
    "sweep_zipf0": "imbalance / granularity sweep at Zipf s=0",
    "sweep_zipf1": "imbalance / granularity sweep at Zipf s=1",
    "sweep_zipf2": "imbalance / granularity sweep at Zipf s=2",
    "sweep_zipf0_mx": "imbalance / granularity sweep at Zipf s=0",
    "sweep_zipf1_mx": "imbalance / granularity sweep at Zipf s=1",
    "sweep_zipf2_mx": "imbalance / granularity sweep at Zipf s=2",
}


def config_of(w, args, n):
    wbytes = 3 * w.E * w.H * w.I * 2
    title = WORKLOAD_TITLES.get(w.name, w.name)
    return {"workload": f"{title}, {w.precision.upper()}: T={w.T} H={w.H} I={w.I} E={w.E} top-{w.K}, router "
                        f"{w.router}, seeded synthetic ({w.name})", "T": w.T, "H": w.H, "I": w.I, "E": w.E, "K": w.K,
            "global_batch": w.T * n, "minibatch_rows": args.minibatch, "macrobatch_rows": args.macrobatch,
            "parallelism": f"replicas x{n} (independent data-parallel shards; the layer has no collective)",
            "l2": f"inputs larger than L2: {wbytes / 1e6:.0f} MB of expert weights streamed every step, no flush"}


def fp32_alu_tflops(dev, peaks) -> float:
    """fp32 fused multiply-add peak of the CUDA cores: SMs x 128 fp32 lanes x 2 flops x the maximum
    SM clock (the device's SM count; the clock from the measured peaks, else 2070 MHz)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def capture_step(fn, stream):
    """One CUDA graph of the layer step fn (schedule, forward, backward: every launch through the C
    ABI).  The step allocates nothing and reads nothing back, so it captures as is; each replay
    rebuilds the schedule on the device from whatever the captured input buffers hold."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_router(args, mok, w, d, cfg, dev, stream, peaks) -> dict:
    """Router forward (logits, top-k) and backward (W transposed, g and dx, dW and d_bias) on the
    workload's own router draws, with the schedule built from the router's ids; CUDA events
    around K steps after W warm-ups, then the per-kernel event trace."""
    x = d["x"].to(dev)
    Wr = d["Wr"].to(dev)
    b = None if d["router_bias"] is None else d["router_bias"].to(dev)
    T, H, E, K = w.T, w.H, w.E, w.K
    shape = mok.make_shape(T, H, w.I, E, K)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    wts = torch.empty((T, K), dtype=torch.float32, device=dev)
    dtopk = torch.randn((T, K), generator=torch.Generator().manual_seed(5)).to(dev)
    dw = torch.empty((H, E), dtype=torch.float32, device=dev)
    db = torch.empty((E,), dtype=torch.float32, device=dev) if b is not None else None
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    rws = torch.empty(mok.mok_router_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    sws = mok.alloc_workspace(cfg, shape, device=dev)
    with torch.cuda.stream(stream):
        mok.mok_router_forward(shape, x, Wr, b, logits, ids, wts, stream)
        sched = mok.mok_build_schedule(cfg, shape, ids, wts, sws, stream)

    def fwd():
        mok.mok_router_forward(shape, x, Wr, b, logits, ids, wts, stream)

    def bwd():
        mok.mok_router_backward(sched, x, Wr, ids, wts, dtopk, dw, db, dx, False, rws, stream)

    res = {"note": "router step before the layer (logits x W_r + b, softmax top-k, renormalised weights; "
                   "backward to W_r, b and x); timed on its own, not part of the layer step"}
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fwd()
            bwd()
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    e[0].record(stream)
    for _ in range(args.steps):
        fwd()
    e[1].record(stream)
    for _ in range(args.steps):
        bwd()
    e[2].record(stream)
    torch.cuda.synchronize()
    res["fwd_ms"] = e[0].elapsed_time(e[1]) / args.steps
    res["bwd_ms"] = e[1].elapsed_time(e[2]) / args.steps
    res["ms_per_step"] = res["fwd_ms"] + res["bwd_ms"]
    tr = mok.Tracer(capacity=8 * args.steps + 16)
    with tr:
        for _ in range(args.steps):
            fwd()
            bwd()
    per = {}
    for name, t in tr.records():
        p = per.setdefault(name, [0.0, 0])
        p[0] += t
        p[1] += 1
    kern = {k: {"avg_ms": v[0] / v[1], "launches": v[1]} for k, v in per.items()}
    if "router_logits" in kern:  # fp32 fused multiply-adds on the CUDA cores: ALU-bound
        ms = kern["router_logits"]["avg_ms"]
        tf = 2.0 * T * H * E / (ms * 1e-3) / 1e12
        alu = fp32_alu_tflops(dev, peaks)
        kern["router_logits"].update({"tflops": tf, "bound": "alu", "peak_tflops": alu, "frac": tf / alu})
    hbm = peaks["hbm_gbs"]
    # unique bytes: W^T read once by dx (its K rows per token are L2 hits), x read once by dW
    byts = {"router_topk": T * E * 4 + T * K * 8, "router_transpose": 2 * H * E * 2,
            "router_dx": T * K * 12 + E * H * 2 + T * H * 2, "router_dw": T * K * 8 + T * H * 2 + H * E * 4}
    for k, nb in byts.items():
        if k in kern:
            g = nb / (kern[k]["avg_ms"] * 1e-3) / 1e9
            kern[k].update({"gbs": g, "bound": "hbm", "frac": g / hbm})
    res["kernels"] = kern
    return res


def time_schedule_in_graph(mok, layer, ids, s, stream, step_ms, n=20, reps=10) -> dict:
    """The schedule's cost as it runs inside the step's graph: one CUDA graph of n back-to-back
    mok_build_schedule calls on the step's routing (three dependent launches each), replayed reps
    times; per build, against the graph-replayed step (the pages' budget: under 3 %)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            layer.schedule(ids, s, stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (reps * n)
    return {"ms_per_build": ms, "share_of_step": ms / step_ms,
            "how": f"graph of {n} builds in a row, {reps} replays"}


def time_quantize(args, mok, Wg, Wu, Wd, stream, peaks) -> dict:
    """mok_mxfp8_quantize on the forward weight copies (Wg, Wu along H; Wd along I), the call a
    training loop makes after each optimiser step: CUDA events around K sets of the three calls
    after W warm-ups, outputs preallocated.  Each element moves 2 bytes in and 1 + 1/32 out."""
    mats = [Wg.reshape(-1, Wg.shape[-1]), Wu.reshape(-1, Wu.shape[-1]), Wd.reshape(-1, Wd.shape[-1])]
    outs = [(torch.empty(m.shape, dtype=torch.uint8, device=m.device),
             torch.empty((m.shape[0], m.shape[1] // 32), dtype=torch.uint8, device=m.device)) for m in mats]

    def one():
        for m, (q, sc) in zip(mats, outs):
            mok.mok_mxfp8_quantize(m, q, sc, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    n = sum(m.numel() for m in mats)
    nbytes = n * (2 + 1 + 1 / 32)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "mxfp8_quantize", "ms_per_set": ms, "elements": n, "bytes": nbytes, "gbs": gbs,
            "bound": "hbm", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
            "what": "the three forward weight copies (Wg, Wu along H; Wd along I), inputs larger than L2"}


def ours(args, rank, ws, local_rank, name, with_router=True):
    """Every measurement of one workload: the step from a CUDA graph and eagerly, the per-kernel
    event trace and roofline, the router step (workloads with a softmax router), and e2e through
    the C ABI with host buffers."""
    from mixture_experts_layer_build_gb300 import inputs, mok

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = inputs.WORKLOADS[name]
    d = inputs.make(w, seed=rank, weight_device=str(dev))
    x, ids, s, dY = (d[k].to(dev) for k in ("x", "topk_ids", "topk_weights", "dY"))
    Wg, Wu, Wd = d["Wg"], d["Wu"], d["Wd"]
    mxfp8 = w.precision == "mxfp8"
    cfg = mok.make_config(args.minibatch, max(args.macrobatch, args.minibatch), args.num_ctas,
                          precision=mok.MOK_MXFP8 if mxfp8 else mok.MOK_BF16,
                          flags=mok.MOK_FLAG_STATIC_TILES if args.static_tiles else 0)
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg, device=dev)
    if mxfp8:  # weights are pre-quantised once, outside the step (the caller's optimiser step)
        mx = mok.quantize_weights(Wg.to(dev), Wu.to(dev), Wd.to(dev))
        weights = mok.weights_struct(mx=mx)
    else:
        weights = mok.weights_struct(Wg, Wu, Wd)
    stream = torch.cuda.Stream(device=dev)

    def step(xx=x, ii=ids, ss=s, dd=dY):
        layer.schedule(ii, ss, stream)
        layer.forward(xx, weights, stream)
        layer.backward(dd, weights, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    # the step as it runs in training: one CUDA graph, replayed (eager launches if capture fails)
    graph, graph_error = None, None
    if not args.no_graph:
        try:
            graph = capture_step(step, stream)
            with torch.cuda.stream(stream):
                for _ in range(2):
                    graph.replay()
            torch.cuda.synchronize()
        except Exception as ex:  # reported in the JSON line; the eager step is timed instead
            graph, graph_error = None, f"{type(ex).__name__}: {str(ex)[:200]}"
    run = graph.replay if graph is not None else step
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                fn()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return max_over_ranks(a.elapsed_time(b) / args.steps, ws, dev)

    # ---- timed region: inputs resident in HBM, K replays of the step ----
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    ms_max = timed(run)
    clocks.mark("t1")
    status = mok.mok_read_device_status(layer.sched, stream)
    # the same K steps launched one kernel at a time from the host, for comparison
    eager_ms = timed(step) if graph is not None else ms_max
    step_mode = {"mode": "cuda_graph" if graph is not None else "eager",
                 "eager_ms_per_step": eager_ms, "eager_value": aggregate_tokens_per_s(w.T, ws, eager_ms)}
    if graph_error:
        step_mode["graph_error"] = graph_error
    if graph is not None:
        step_mode["schedule"] = time_schedule_in_graph(mok, layer, ids, s, stream, ms_max)

    # ---- per-kernel times: the same K steps with the library's event trace ----
    tr = mok.Tracer(capacity=20 * args.steps + 64)
    with tr:
        for _ in range(args.steps):
            step()
    recs = tr.records()
    launches_per_step = len(recs) / args.steps
    per = {}
    for kname, t in recs:
        p = per.setdefault(kname, [0.0, 0])
        p[0] += t
        p[1] += 1
    traced_total = sum(v[0] for v in per.values())
    kernels = {k: {"avg_ms": v[0] / v[1], "launches": v[1], "share": v[0] / traced_total} for k, v in per.items()}
    e_active = int(torch.unique(ids).numel())
    work = kernel_work(w, e_active)
    peaks, peak_src = load_peaks()
    for k, v in kernels.items():
        if k in work:
            fl, nb, kd = work[k]
            if fl:
                v["tflops"] = fl / (v["avg_ms"] * 1e-3) / 1e12
            v["gbs"] = nb / (v["avg_ms"] * 1e-3) / 1e9
            rf = roofline_of(fl, nb, v["avg_ms"], peaks, kd)
            v["bound"], v["frac"] = rf["bound"], rf["frac"]
    dom = max((k for k in kernels if k in work), key=lambda k: kernels[k]["avg_ms"] * kernels[k]["launches"])
    fl, nb, kd = work[dom]
    traffic, tnote = traffic_for(dom, name)
    roof = roofline_of(fl, nb, kernels[dom]["avg_ms"], peaks, kd)
    roof.update({"traffic": traffic, "kernel": dom,
                 "peak_source": (f"{peak_src} (burst bf16 GEMM / STREAM copy)" if peak_src == "measured"
                                 else "fallback") + (" x2 nominal e4m3/bf16" if kd == "e4m3" else ""),
                 "traffic_note": tnote, "algorithmic_flops_per_launch": fl, "algorithmic_bytes_per_launch": nb})

    # ---- the router step before the layer (timed on its own; not part of the layer step) ----
    router = time_router(args, mok, w, d, cfg, dev, stream, peaks) if with_router and "Wr" in d else None
    # ---- the weight quantiser (MXFP8; outside the layer step, like the router) ----
    quant = time_quantize(args, mok, Wg.to(dev), Wu.to(dev), Wd.to(dev), stream, peaks) if mxfp8 else None

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its own inputs host->device and its results device->host inside the timed
    # region.  Inputs and outputs are double-buffered, uploads on one copy stream and downloads on
    # another, so step i+1's uploads, step i-1's downloads and step i's compute all overlap (the
    # usual prefetching input pipeline; the two directions of the host link run concurrently).
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    host_in = [pin(d["x"]), pin(d["topk_ids"]), pin(d["topk_weights"]), pin(d["dY"])]
    host_out = [[torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((w.T, w.K), dtype=torch.float32).pin_memory()] for _ in range(2)]
    dev_in = [[torch.empty_like(t, device=dev) for t in (x, ids, s, dY)] for _ in range(2)]
    dev_out = [dict(out=torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev),
                    grads=mok.Grads.empty(w.T, w.H, w.I, w.E, w.K, device=dev)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    copy_stream = torch.cuda.Stream(device=dev)   # host -> device
    down_stream = torch.cuda.Stream(device=dev)   # device -> host
    ev_in = [torch.cuda.Event() for _ in range(2)]      # uploads of buffer b landed
    ev_done = [torch.cuda.Event() for _ in range(2)]    # compute on buffer b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]     # downloads of buffer b finished

    def upload(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(ev_done[b])  # buffer b's previous step has consumed its inputs
            for dst, src in zip(dev_in[b], host_in):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(copy_stream)

    def abi_step(b):  # the step on buffer set b, through the C ABI entry points
        def fn():
            xx, ii, ss, dd = dev_in[b]
            sch = mok.mok_build_schedule(layer.cfg, layer.shape, ii, ss, layer.ws, stream)
            mok.mok_forward(sch, xx, weights, dev_out[b]["out"], layer.ctx, stream)
            mok.mok_backward(sch, layer.ctx, dd, weights, dev_out[b]["grads"], stream)
        return fn

    # one CUDA graph per buffer set when the resident-input step ran from a graph
    steps_b = [capture_step(abi_step(b), stream).replay if graph is not None else abi_step(b) for b in range(2)]

    def compute(i):
        b = i % 2
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # buffer b's previous results have been downloaded
            steps_b[b]()
            ev_done[b].record(stream)

    def download(i):
        b = i % 2
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(ev_done[b])
            o, g = dev_out[b]["out"], dev_out[b]["grads"]
            for dst, src in zip(host_out[b], (o, g.dx, g.d_topk_weights)):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(down_stream)

    def e2e_run(n):
        # issue order keeps both streams busy: upload(i+1) before compute(i)'s results are fetched
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
            download(i)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(copy_stream)
    e2e_run(args.steps)
    down_stream.wait_stream(stream)
    down_stream.wait_stream(copy_stream)
    e1.record(down_stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    clk = clocks.stop()

    result = None
    if rank == 0:
        tokens_per_s = aggregate_tokens_per_s(w.T, ws, ms_max)
        result = {
            "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp8" if mxfp8 else "bf16",
            "data": "synthetic (seeded; random-init expert weights)",
            "config": config_of(w, args, ws),
            "tflops": w.flops() / (ms_max * 1e-3) / 1e12,
            "roofline": roof,
            "kernels": kernels,
            "e2e": {"value": w.T * ws / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "launches_per_step": launches_per_step,
            "clocks": clk,
            "device_status": status,
            "step": step_mode,
        }
        if router is not None:
            result["router"] = router
        if quant is not None:
            result["quantize"] = quant
    return result, d, w


def parse_extra(spec: str):
    out = []
    for item in (spec or "").split(","):
        item = item.strip()
        if item:
            key, _, wl = item.partition("=")
            out.append((key.strip(), wl.strip()))
    return out


# keys of a further workload's object (its full kernel table stays on the headline only)
EXTRA_KEYS = ("metric", "value", "unit", "ms_per_step", "dtype", "config", "tflops", "roofline", "e2e",
              "gpu_launches", "launches_per_step", "clocks", "device_status", "step", "quantize")


def main():
    args = parse()
    rank, ws, local_rank = dist_init()
    if args.impl == "reference":
        reference_arm(args, rank, ws)
        return
    res, d, w = ours(args, rank, ws, local_rank, args.workload)
    extras = {}
    for key, wl in parse_extra(args.extra):
        if wl == args.workload:
            continue
        r2, _, _ = ours(args, rank, ws, local_rank, wl, with_router=False)
        torch.cuda.empty_cache()
        if rank == 0:
            extras[key] = {k: r2[k] for k in EXTRA_KEYS if k in r2}
            extras[key]["kernels"] = {k: {kk: v[kk] for kk in ("avg_ms", "bound", "frac", "tflops", "gbs") if kk in v}
                                      for k, v in r2["kernels"].items()}
    if rank == 0:
        res.update(extras)
        if ws == 1 and not args.no_cpu_baseline:
            from mixture_experts_layer_build_gb300 import inputs
            wbits = (inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
            if w.precision == "mxfp8":
                import oracle
                wbits = oracle.mx_weights(*wbits)
            tokens, _ = calibrate_oracle_tokens(d, wbits, args.cpu_seconds, w.T)
            t = time_oracle_step(d, wbits, tokens)
            res["cpu_baseline"] = {"value": tokens / t, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                                   "sample": f"fwd+bwd of the first {tokens} of {w.T} tokens (all their routed rows, "
                                             f"full dW), {oracle_kind(wbits)}, {t:.1f} s"}
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
