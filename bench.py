"""Benchmark: layer-streamed training step (forward + backward, every weight
streamed from pinned host memory, every gradient streamed back) on the
LLaMA-3.1-8B-shaped decoder, one GPU per process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference] [--workload llama8b|...]

Prints one JSON line (rank 0). Multi-GPU runs are independent replicas (each
GPU trains its own batch through its own context; nothing is exchanged), so
`value` is the sum of tokens over all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (layers, hidden, heads, kv_heads, head_dim, ffn, vocab, theta, B, S, K, bf16 host params)
    "llama8b": (32, 4096, 32, 8, 128, 14336, 128256, 5e5, 2, 4096, 4, True),
    "llama8b_long": (32, 4096, 32, 8, 128, 14336, 128256, 5e5, 1, 16384, 8, True),
    "small": (8, 1024, 16, 16, 64, 2816, 32000, 1e4, 4, 2048, 4, False),
    "tiny": (2, 64, 4, 4, 16, 172, 256, 1e4, 2, 32, 1, False),
    # Qwen3-235B-style mixture-of-experts layers, the first 8 of 94 (host RAM bound)
    "qwen3_moe": (8, 4096, 64, 4, 128, 0, 151936, 1e6, 1, 4096, 2, True),
}
# Mixture-of-experts workloads: (experts, top-k, expert FFN width)
MOE = {"qwen3_moe": (128, 8, 1536)}
NORM_EPS = {"qwen3_moe": 1e-6}
METRIC = "train tokens/sec (fwd+bwd, weights streamed from host) at 8B shape; % roofline"
_T0 = time.time()


def log(msg: str) -> None:
    sys.stderr.write(f"[bench +{time.time() - _T0:7.1f}s] {msg}\n")
    sys.stderr.flush()


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
                    if v.lower() in ("active", "1", "0x1"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def model_flops(shape, B, S, moe=None):
    """Algorithmic work of one step, as counted for the roofline: per decoder
    layer 2*T*P_lin for each of forward, recompute, input-gradient and
    weight-gradient products, plus causal attention (forward, recompute and
    2.5x backward); head 4 GEMM-equivalents (two logit passes, dX, dW).
    With experts (moe = (E, k, Fe)) a token passes through the router and k
    experts: P_lin counts those, not all E (the streamed bytes do)."""
    L, h, nq, nkv, d, F, V = shape[:7]
    T = B * S
    P_lin = h * (nq * d) * 2 + 2 * h * (nkv * d) + 3 * h * F
    if moe:
        E, k, Fe = moe
        P_lin += E * h + k * 3 * Fe * h
    A = 2.0 * B * nq * d * S * (S + 1)
    layer = 2.0 * T * P_lin * 4 + A * (1 + 1 + 2.5)
    head = 4 * 2.0 * T * V * h
    return layer, head, P_lin


def layer_params(shape, moe=None):
    """Matrix parameters of one decoder layer as streamed (all experts)."""
    L, h, nq, nkv, d, F, V = shape[:7]
    p = h * (nq * d) * 2 + 2 * h * (nkv * d) + 3 * h * F
    if moe:
        E, k, Fe = moe
        p += E * h + E * 3 * Fe * h
    return p


def moe_gemm_algorithmic_bytes(shape, B, S, K, head_rows, moe, fuse_top=True):
    """gemm_algorithmic_bytes for mixture-of-experts layers: attention
    projections as in the dense layer; router; per expert its rows of the
    gate|up and down products (bf16 operands, fp32 routed outputs and weight
    gradients), every expert's weights read once per product kind. Launch
    count assumes every expert receives rows."""
    L, h, nq, nkv, d, F, V = shape[:7]
    E, k, Fe = moe
    T = B * S
    R = T * k
    qkv = (nq + 2 * nkv) * d
    fwd = ((T * h + qkv * h + T * qkv) * 2 + (T * nq * d + h * nq * d) * 2 + T * h * 8 +
           (T * h + E * h) * 2 + T * E * 4 +                       # router logits (fp32)
           (R * h + E * 2 * Fe * h + R * 2 * Fe + R * Fe) * 2 +      # gate|up, writes g|u and act
           (R * Fe + E * h * Fe) * 2 + R * h * 4)                   # down, fp32 routed outputs
    bwd = ((R * h + R * Fe) * 2 + E * h * Fe * 4 +                  # dWd
           (R * h + E * h * Fe) * 2 + 2 * R * 2 * Fe * 2 +          # d act -> (dg, du) in place
           (R * 2 * Fe + R * h) * 2 + E * 2 * Fe * h * 4 +          # dWgu
           (R * 2 * Fe + E * 2 * Fe * h) * 2 + R * h * 4 +          # d routed inputs
           (T * E + E * h) * 2 + T * h * 8 +                        # dm += dr Wr
           (T * E + T * h) * 2 + E * h * 4 +                        # dWr
           (T * h + T * nq * d) * 2 + h * nq * d * 4 +              # dWo
           (T * h + h * nq * d + T * nq * d) * 2 +                  # do
           (T * qkv + T * h) * 2 + qkv * h * 4 +                    # dWqkv
           (T * qkv + qkv * h) * 2 + T * h * 4)                     # dx
    slices = (V + head_rows - 1) // head_rows
    head = 0
    for i in range(slices):
        Rr = min(head_rows, V - i * head_rows)
        head += 2 * ((T * h + Rr * h) * 2 + T * Rr * 4)
        head += (T * Rr + Rr * h) * 2 + T * h * (4 if i == 0 else 8)
        head += (T * Rr + T * h) * 2 + Rr * h * 4
    top = L - K * ((L + K - 1) // K - 1)
    n_fwd = L + (L - top if fuse_top else L)
    return n_fwd * fwd + L * bwd + head, (3 + 2 * E) * n_fwd + (6 + 4 * E) * L + 4 * slices


def gemm_algorithmic_bytes(shape, B, S, K, head_rows, fuse_top=True):
    """Operand and result bytes of every GEMM launch of one step: each operand
    read once and each result written once (bf16 activations and weights,
    fp32 weight gradients and residual outputs; read-modify-write where the
    epilogue adds to or rewrites its output). Returns (bytes, launches)."""
    L, h, nq, nkv, d, F, V = shape[:7]
    T = B * S
    qkv = (nq + 2 * nkv) * d
    fwd = ((T * h + qkv * h + T * qkv) * 2 +                       # QKV (+RoPE), bf16 out
           (T * nq * d + h * nq * d) * 2 + T * h * 8 +              # O-proj, fp32 residual add
           (T * h + 2 * F * h + 2 * T * F + T * F) * 2 +           # gate-up, writes g|u and act
           (T * F + h * F) * 2 + T * h * 8)                        # down, fp32 residual add
    bwd = ((T * h + T * F) * 2 + h * F * 4 +                       # dWd
           (T * h + h * F) * 2 + 2 * T * 2 * F * 2 +               # d act -> (dg, du) in place over (g, u)
           (2 * T * F + T * h) * 2 + 2 * F * h * 4 +               # dWg|Wu
           (2 * T * F + 2 * F * h) * 2 + T * h * 4 +               # dm
           (T * h + T * nq * d) * 2 + h * nq * d * 4 +             # dWo
           (T * h + h * nq * d + T * nq * d) * 2 +                 # do
           (T * qkv + T * h) * 2 + qkv * h * 4 +                   # dWqkv
           (T * qkv + qkv * h) * 2 + T * h * 4)                    # dx
    slices = (V + head_rows - 1) // head_rows
    head = 0
    for i in range(slices):
        R = min(head_rows, V - i * head_rows)
        head += 2 * ((T * h + R * h) * 2 + T * R * 4)              # logits, pass 1 and pass 2
        head += (T * R + R * h) * 2 + T * h * (4 if i == 0 else 8)  # dX, accumulated over slices
        head += (T * R + T * h) * 2 + R * h * 4                     # dW of the slice
    top = L - K * ((L + K - 1) // K - 1)                            # layers of the top block
    n_fwd = L + (L - top if fuse_top else L)
    return n_fwd * fwd + L * bwd + head, 4 * n_fwd + 8 * L + 4 * slices


def max_over_ranks(values, dist, device):
    """Element-wise maximum over all ranks (the slowest replica sets the
    time); identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_throughput(world, tokens_per_step, steps, seconds):
    """Whole-job tokens/s: every replica processes its own batch each step."""
    return world * tokens_per_step * steps / seconds


def head_slice_rows(shape, esz, moe=None):
    """Rows of an LM-head vocab slice: the fewest equal slices (multiples of
    256 rows) whose bytes fit one packed decoder layer (as the library sizes
    them)."""
    L, h, nq, nkv, d, F, V = shape[:7]
    layer = (2 * h + layer_params(shape, moe)) * esz
    ns = max(1, (V * h * esz + layer - 1) // layer)
    while True:
        r = min(V, (((V + ns - 1) // ns) + 255) // 256 * 256)
        if r * h * esz <= layer or r <= 256:
            return r
        ns += 1


# DRAM bytes (read + written) of each GEMM launch of the 8B step, one launch
# of each shape captured cold-cache by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum) with `kbench gemm --shape <name>`; the summary,
# commands and algorithmic bytes are in
# profiles/gemm_dram_traffic_8b_step_shapes.md. Taken with the GEMM kernels
# as committed with that summary; when the GEMM kernels change, the figure
# must be captured again.
GEMM_TRAFFIC_8B = {
    "qkv_rope": 301616384, "o_proj": 508946432, "gate_up": 1629239552, "down": 1530027520, "dWd": 1100619520,
    "dact_swiglu": 1536381184, "dWgu": 3216824320, "dm": 3643644928, "dWo": 336235776, "do": 201520128,
    "dWqkv": 525138688, "dx": 559515136, "head_logits": 2931604992, "head_dX": 5587098624,
    "head_dW": 5480545024,
}
# Launches of each per step at the 8B configuration (32 layers, K=4, top
# block not recomputed; three vocab slices of the head).
GEMM_LAUNCHES_8B = {"qkv_rope": 60, "o_proj": 60, "gate_up": 60, "down": 60, "dWd": 32, "dact_swiglu": 32,
                    "dWgu": 32, "dm": 32, "dWo": 32, "do": 32, "dWqkv": 32, "dx": 32, "head_logits": 6,
                    "head_dX": 3, "head_dW": 3}


def gemm_traffic_per_launch_8b() -> float:
    """DRAM bytes per GEMM launch of one 8B step: the per-shape captures
    weighted by each shape's launches."""
    n = sum(GEMM_LAUNCHES_8B.values())
    return sum(GEMM_TRAFFIC_8B[k] * GEMM_LAUNCHES_8B[k] for k in GEMM_LAUNCHES_8B) / n


def numa_pages(addrs) -> dict:
    """Pages per NUMA node of the mappings that contain the given host
    addresses (from /proc/self/numa_maps; empty when unavailable)."""
    out = {}
    try:
        with open("/proc/self/numa_maps") as f:
            lines = f.read().splitlines()
    except OSError:
        return out
    starts = sorted((int(l.split()[0], 16), l) for l in lines)
    for name, a in addrs.items():
        best = None
        for st, l in starts:
            if st <= a:
                best = l
            else:
                break
        if best:
            out[name] = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in best.split()
                         if kv.startswith("N") and "=" in kv}
    return out


def host_link_probe(torch, nbytes=436 * 2**20):
    """Pinned H2D alone, D2H alone, and both at once (GB/s), from fresh
    torch pinned buffers. Each copy is timed with CUDA events on its own
    stream, so the concurrent run gives one figure per direction (best of
    five)."""
    host_a = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host_b = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def run(h2d, d2h, reps=5):
        best_h = best_d = 1e9
        for _ in range(reps):
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            if h2d:
                ev[0].record(s1)
                with torch.cuda.stream(s1):
                    dev_a.copy_(host_a, non_blocking=True)
                ev[1].record(s1)
            if d2h:
                ev[2].record(s2)
                with torch.cuda.stream(s2):
                    host_b.copy_(dev_b, non_blocking=True)
                ev[3].record(s2)
            torch.cuda.synchronize()
            if h2d:
                best_h = min(best_h, ev[0].elapsed_time(ev[1]) / 1e3)
            if d2h:
                best_d = min(best_d, ev[2].elapsed_time(ev[3]) / 1e3)
        return best_h, best_d

    t_h2d, _ = run(True, False)
    _, t_d2h = run(False, True)
    t_bh, t_bd = run(True, True)
    out = {"h2d_gbs": nbytes / t_h2d / 1e9, "d2h_gbs": nbytes / t_d2h / 1e9,
           "h2d_concurrent_gbs": nbytes / t_bh / 1e9, "d2h_concurrent_gbs": nbytes / t_bd / 1e9}
    del host_a, host_b, dev_a, dev_b
    return out


def replay_summary(r: dict) -> dict:
    """Totals and distribution of a copy-only replay of the weight stream."""
    g = np.asarray(r["copy_gbs"], dtype=np.float64)
    return {"copies": r["n_copies"], "gbs": r["bytes"] / max(r["ms"], 1e-9) / 1e6,
            "copy_gbs_min": float(g.min()) if g.size else None,
            "copy_gbs_p10": float(np.percentile(g, 10)) if g.size else None,
            "copy_gbs_p50": float(np.percentile(g, 50)) if g.size else None,
            "slow_copies_below_100gbs": int(np.sum(g < 100.0))}


def _oracle_timed_step(shape, n_layers, vocab, S, seed, moe=None, eps=1e-5):
    """Seconds of one single-threaded oracle step of a model with the given
    layer count and vocabulary (the workload's widths) at B=1, S."""
    import oracle
    import seedgen
    L, h, nq, nkv, d, F, V, theta = shape[:8]
    E, k, Fe = moe or (0, 0, 0)
    cfg = oracle.Config(n_layers, h, nq, nkv, d, F, vocab, theta, eps, E, k, Fe)
    packed = np.zeros(oracle.packed_bytes(cfg, True), np.uint8)
    offs = []
    for unit, t, name, shp, is_gain in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, True)
        offs.append((unit, t, off, int(np.prod(shp)), is_gain))
    seedgen.fill_packed_params(packed.ctypes.data, offs, True, seed)
    tok, lab = seedgen.tokens_and_labels(1, S, vocab, seed + 1)
    t0 = time.perf_counter()
    oracle.forward_backward(cfg, packed, tok, lab, bf16=True)
    return time.perf_counter() - t0


def _oracle_timed_attention(shape, S, seed):
    """Seconds of the oracle's causal attention forward + backward over all
    heads of one sequence of length S."""
    import oracle
    import seedgen
    L, h, nq, nkv, d = shape[:5]
    q, do = (seedgen.normal(S * nq * d, seed + i, 9, 1.0).reshape(1, S, nq, d) for i in (0, 1))
    k, v = (seedgen.normal(S * nkv * d, seed + i, 9, 1.0).reshape(1, S, nkv, d) for i in (2, 3))
    t0 = time.perf_counter()
    oracle.attention(q, k, v, do)
    return time.perf_counter() - t0


class CpuFit:
    """The single-threaded CPU oracle timed on pieces of one training step
    of the workload and extrapolated to the whole step (each piece one
    oracle call on one thread, run one after another):
      - one decoder layer of the workload's widths with a 256-entry
        vocabulary (head negligible) at B=1, S=S1 and S=S2: t = c0 + c1 S,
        c0 the work done once per call (the oracle transposes every weight
        matrix for its forward products), c1 the work per token (its loops
        stream every weight matrix once per token in each of the forward,
        input-gradient and weight-gradient products);
      - causal attention forward + backward over all heads of one sequence
        at S_attn: a S_attn^2, extrapolated quadratically in the sequence
        length (the S1/S2 layers hold a negligible attention part);
      - the LM head and loss: the same three loop nests over V*h weights
        instead of the layer's P_lin, so c0 and c1 scaled by V*h / P_lin
        (the softmax over the vocabulary adds O(V) per token, negligible).
    step(B, S) = L (c0 + c1 T + a S^2 B) + (V h / P_lin)(c0 + c1 T), T = B S."""

    def __init__(self, shape, moe=None, eps=1e-5, seed=5, S1=8, S2=40, S_attn=512):
        self.shape, self.moe, self.eps, self.seed = shape, moe, eps, seed
        self.S1, self.S2, self.S_attn = S1, S2, S_attn
        t1 = _oracle_timed_step(shape, 1, 256, S1, seed, moe, eps)
        t2 = _oracle_timed_step(shape, 1, 256, S2, seed, moe, eps)
        self.c1 = max(0.0, (t2 - t1) / (S2 - S1))
        self.c0 = max(0.0, t1 - self.c1 * S1)
        self.t_attn = _oracle_timed_attention(shape, S_attn, seed)
        self.a = self.t_attn / S_attn ** 2
        L, h, nq, nkv, d, F, V = shape[:7]
        self.head_ratio = V * h / layer_params(shape, moe)
        self.cpu_seconds = t1 + t2 + self.t_attn

    def step_seconds(self, B, S, scale=1.0):
        L = self.shape[0]
        T = B * S
        lin = self.c0 + self.c1 * T
        return scale * (L * (lin + self.a * S * S * B) + self.head_ratio * lin)

    def resample(self):
        """Re-time the cheapest piece (attention at S_attn); its ratio to
        the fitted value rescales the extrapolated step."""
        return _oracle_timed_attention(self.shape, self.S_attn, self.seed) / self.t_attn

    def describe(self, B, S):
        L = self.shape[0]
        return (f"single-threaded fp32 oracle timed on one layer of the workload's widths (256-entry vocabulary) at "
                f"B=1, S={self.S1} and S={self.S2} and on causal attention forward+backward over all heads at "
                f"S={self.S_attn}; extrapolated to {L} layers and the LM head at B={B}, S={S}: linear terms linearly "
                f"in tokens (the head as the layer's per-weight cost times V*h), attention quadratically in sequence "
                f"length (extrapolated; {self.cpu_seconds:.1f} s of CPU work; host has {os.cpu_count()} cores)")


def cpu_oracle_full_step(shape, B, S, seed=5, moe=None, eps=1e-5, bf16=False):
    """Time one whole step of the CPU oracle (single thread) at the workload's
    own size (only for workloads where that takes seconds, e.g. the tiny
    decoder). Returns (tokens/s, seconds)."""
    import oracle
    import seedgen
    L, h, nq, nkv, d, F, V, theta = shape[:8]
    E, k, Fe = moe or (0, 0, 0)
    cfg = oracle.Config(L, h, nq, nkv, d, F, V, theta, eps, E, k, Fe)
    packed = np.zeros(oracle.packed_bytes(cfg, bf16), np.uint8)
    offs = []
    for unit, t, name, shp, is_gain in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, bf16)
        offs.append((unit, t, off, int(np.prod(shp)), is_gain))
    seedgen.fill_packed_params(packed.ctypes.data, offs, bf16, seed)
    tok, lab = seedgen.tokens_and_labels(B, S, V, seed + 1)
    t0 = time.perf_counter()
    oracle.forward_backward(cfg, packed, tok, lab, bf16=bf16)
    t1 = time.perf_counter() - t0
    return B * S / t1, t1


FULL_STEP_BASELINE = {"tiny"}  # workloads whose CPU baseline is a whole oracle step


def run_reference(args, shape, B, S):
    """The reference arm: the CPU oracle as it stands, timed on this host.
    The whole-step workloads time one oracle step per step; the others fit
    the piecewise model once (CpuFit) and re-time its cheapest piece each
    step, rescaling the extrapolated step by it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    full = args.workload in FULL_STEP_BASELINE
    moe, eps = MOE.get(args.workload), NORM_EPS.get(args.workload, 1e-5)
    vals = []
    fit = None if full else CpuFit(shape, moe=moe, eps=eps)
    for i in range(args.warmup + args.steps):
        if full:
            v, t1 = cpu_oracle_full_step(shape, B, S, seed=100 + i, moe=moe, eps=eps,
                                         bf16=bool(WORKLOADS[args.workload][11]))
        else:
            v = B * S / fit.step_seconds(B, S, fit.resample())
        if i >= args.warmup:
            vals.append(v)
    value = float(np.median(vals))
    sample = (f"whole step of the {args.workload} workload at B={B}, S={S}, single-threaded fp32 oracle" if full else
              fit.describe(B, S) + "; each step re-times the attention piece and rescales by it")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "global_batch": B, "seq_len": S, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="llama8b", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fuse-top", action="store_true", help="recompute the top block too")
    ap.add_argument("--serial", action="store_true", help="ablation: serialise weight copies and compute")
    ap.add_argument("--no-page-touch", action="store_true",
                    help="ablation: no host page touches ahead of the weight copies (MT_PAGE_TOUCH=0)")
    ap.add_argument("--optimizer", nargs="?", const="sync", choices=["sync", "async"], default=None,
                    help="time train steps with the host AdamW: sync = mt_train_step (each unit updated as its "
                         "gradients land), async = mt_train_step_async (staleness 1); allocates three fp32 copies "
                         "of the model on the host, so use it with --layers at the 8B widths")
    ap.add_argument("--param-dtype", default=None, choices=["bf16", "fp8"],
                    help="host weight format of the bf16 workloads: bf16 (the default) or fp8 (E4M3 codes with one "
                         "scale per row, dequantised to bf16 on the device: half the streamed weight bytes)")
    ap.add_argument("--grad-dtype", default="fp32", choices=["fp32", "bf16"],
                    help="dtype of the streamed host gradients (bf16 halves the D2H bytes)")
    ap.add_argument("--layers", type=int, default=None, help="diagnostic override of the layer count")
    ap.add_argument("--seq", type=int, default=None, help="diagnostic override of the sequence length")
    ap.add_argument("--batch", type=int, default=None, help="diagnostic override of the batch")
    args = ap.parse_args()
    wl = list(WORKLOADS[args.workload])
    if args.layers:
        wl[0] = args.layers
    if args.seq:
        wl[9] = args.seq
    if args.batch:
        wl[8] = args.batch
    shape, (B, S, K, bf16) = tuple(wl[:8]), wl[8:]
    K = min(K, shape[0])
    fp8 = args.param_dtype == "fp8"
    if fp8 and not bf16:
        sys.exit("--param-dtype fp8 applies to the bf16 workloads")
    if args.impl == "reference":
        return run_reference(args, shape, B, S)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    os.environ.setdefault("MT_TRACE", "1")
    if args.no_fuse_top:
        os.environ["MT_FUSE_TOP_BLOCK"] = "0"
    if args.serial:
        os.environ["MT_SERIAL"] = "1"
    if args.no_page_touch:
        os.environ["MT_PAGE_TOUCH"] = "0"
    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    import layer_streamed_gb300 as mt
    import seedgen
    mt.build()
    L, h, nq, nkv, d, F, V, theta = shape
    moe = MOE.get(args.workload)
    E, k_top, Fe = moe or (0, 0, 0)
    eps = NORM_EPS.get(args.workload, 1e-5)
    grad_dtype = mt.MT_BF16 if args.grad_dtype == "bf16" else mt.MT_F32
    if args.optimizer and grad_dtype != mt.MT_F32:
        sys.exit("the host optimizer takes fp32 gradients")
    pdt = mt.MT_FP8 if fp8 else (mt.MT_BF16 if bf16 else mt.MT_F32)
    cfg = mt.make_cfg(L, h, nq, nkv, d, F, V, theta, eps, B, S, K, pdt, E, k_top, Fe, grad_dtype)
    budget = mt.mt_required_budget(cfg)
    log(f"workload {args.workload} L={L} B={B} S={S} K={K}: device arena {budget / 2**30:.2f} GiB")
    arena = torch.empty(budget, dtype=torch.uint8, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(3)]
    sess = mt.Session(mt.ModelShape(L, h, nq, nkv, d, F, V, theta, eps, E, k_top, Fe), B, S, K,
                      pdt, device_budget=budget, device_arena=arena.data_ptr(),
                      streams=[s.cuda_stream for s in streams], grad_dtype=grad_dtype)
    # Parameters: N(0, 0.02) matrices, unit RMSNorm gains, per-rank seed.
    offs = []
    fill_dt = mt.MT_BF16 if bf16 else mt.MT_F32  # FP8 params are quantised from seeded bf16 values
    for unit in range(L + 2):
        nt = 1 if unit == 0 else (9 if unit <= L else 2)
        for t in range(nt):
            off, nbytes = sess.offset(unit, t, fill_dt)
            is_gain = (unit >= 1 and unit <= L and t in (0, 5)) or (unit == L + 1 and t == 0)
            offs.append((unit, t, off, nbytes // (2 if bf16 else 4), is_gain))
    log(f"context created; pinned host params {sess.param_bytes / 2**30:.2f} GiB, grads {sess.grad_bytes / 2**30:.2f} GiB")
    t0 = time.perf_counter()
    if fp8:
        src = np.zeros(mt.mt_packed_bytes(cfg, mt.MT_BF16), np.uint8)
        seedgen.fill_packed_params(src.ctypes.data, offs, True, seed=21 + rank)
        mt.mt_quantize_params_fp8(cfg, src.ctypes.data, mt.MT_BF16, sess.params_ptr, 0)
        del src
    else:
        seedgen.fill_packed_params(sess.params_ptr, offs, bf16, seed=21 + rank)
    init_s = time.perf_counter() - t0
    tok, lab = seedgen.tokens_and_labels(B, S, V, seed=22 + rank)

    log(f"parameters filled in {init_s:.1f} s")
    if args.optimizer:
        master = np.zeros(sess.grad_bytes // 4, np.float32)
        for unit, t, off, n, is_gain in offs:
            o32, _ = sess.offset(unit, t, mt.MT_F32)
            src = np.frombuffer((ctypes.c_uint8 * (n * (2 if bf16 else 4))).from_address(sess.params_ptr + off),
                                np.uint16 if bf16 else np.float32)
            master[o32 // 4:o32 // 4 + n] = ((src.astype(np.uint32) << 16).view(np.float32) if bf16 else src)
        sess.bind_optimizer(mt.adamw_cfg(1e-4, 0.9, 0.95, 1e-8, 0.1), master)
        del master
        log(f"optimizer bound: {3 * sess.grad_bytes / 2**30:.1f} GiB of fp32 master and moments")
    step_fn = {None: sess.step, "sync": sess.train_step, "async": sess.train_step_async}[args.optimizer]
    placement = numa_pages({"params": sess.params_ptr, "grads": sess.grads_ptr})
    log(f"pinned pages per NUMA node: {placement}")
    link = host_link_probe(torch)
    log(f"host link {link}")
    # the same weight stream, copies only, from the bound parameter buffer:
    # with nothing else running, then with the host page touches of the step
    replay_before = replay_summary(sess.replay_weight_stream(K))
    log(f"weight-stream replay from the bound buffer: {replay_before}")
    replay_touch = replay_summary(sess.replay_weight_stream(K, mt.MT_REPLAY_TOUCH))
    log(f"weight-stream replay with page touches: {replay_touch}")
    for i in range(args.warmup):
        t1 = time.perf_counter()
        step_fn(tok, lab, K)
        log(f"warmup step {i}: {time.perf_counter() - t1:.3f} s")
    comp, d2h_stream = streams[0], streams[2]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    agg = {}
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    ev0.record(comp)
    losses = []
    copy_p = []   # per step: min, p10, p50 of the weight copies' GB/s
    host_ms = []  # per step: wall time of the call minus its device span (host preparation and finishing)
    for _ in range(args.steps):
        t_call = time.perf_counter()
        losses.append(step_fn(tok, lab, K))
        call_ms = (time.perf_counter() - t_call) * 1e3
        st = sess.stats()
        host_ms.append(call_ms - st["step_ms"])
        copy_p.append((st["h2d_copy_gbs_min"], st["h2d_copy_gbs_p10"], st["h2d_copy_gbs_p50"]))
        for k, v in st.items():
            if isinstance(v, list):
                agg[k] = [a + b for a, b in zip(agg.get(k, [0.0] * len(v)), v)]
            else:
                agg[k] = agg.get(k, 0) + v
    ev1.record(d2h_stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    log(f"timed {args.steps} steps in {wall:.3f} s")
    clk = clocks.stop()
    # Kernel durations for the roofline: one more step, outside the timed
    # region, with every GEMM/attention launch bracketed by CUDA events on the
    # compute stream (events around launches stall the copy pipeline, so the
    # timed steps run without them).
    replay_r = sess.replay_weight_stream(K)
    replay_after = replay_summary(replay_r)
    log(f"weight-stream replay after the timed steps: {replay_after}")
    sess.set_tracing(2, 1)
    sess.step(tok, lab, K)
    kst = sess.stats()
    sess.set_tracing(1, 16)
    log(f"instrumented step: {kst['n_gemm']} GEMM launches {kst['gemm_ms']:.1f} ms, "
        f"{kst['n_attn']} attention launches {kst['attn_ms']:.1f} ms")
    dev_ms = ev0.elapsed_time(ev1)
    dev_ms, wall = max_over_ranks([dev_ms, wall], dist, "cuda")
    if dist:
        if rank != 0:
            dist.destroy_process_group()
            sess.close()
            return
    T = B * S
    steps = args.steps
    value = replica_throughput(world, T, steps, dev_ms / 1e3)
    e2e = replica_throughput(world, T, steps, wall)
    peaks, peak_kind = read_peaks()
    gemm_tflops = kst["gemm_flop"] / (kst["gemm_ms"] / 1e3) / 1e12 if kst.get("gemm_ms") else None
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    layer_f, head_f, P_lin = model_flops(shape, B, S, moe)
    P_bytes = layer_params(shape, moe)  # streamed matrix parameters of a layer
    step_flop = L * layer_f + head_f
    # Roofline of the whole step: per unit, the slower of its work at the
    # tensor-core peak and its streamed bytes at the measured host link.
    h2d_bw = link["h2d_concurrent_gbs"] * 1e9
    d2h_bw = link["d2h_concurrent_gbs"] * 1e9
    per_step_h2d = agg["h2d_bytes"] / steps
    per_step_d2h = agg["d2h_bytes"] / steps
    layer_h2d = per_step_h2d * (L * P_bytes * 2) / max(1.0, (L * P_bytes * 2 + 2 * V * h * 2)) / L
    gsz = 2.0 if args.grad_dtype == "bf16" else 4.0  # bytes per streamed gradient element
    t_layer = max(layer_f / (peak_tf * 1e12), layer_h2d / h2d_bw, gsz * (P_bytes + 2 * h) / d2h_bw)
    t_head = max(head_f / (peak_tf * 1e12), (per_step_h2d - L * layer_h2d) / h2d_bw, (2.0 * V * h * gsz) / d2h_bw)
    t_roof = L * t_layer + t_head
    ms_per_step = dev_ms / steps
    rows = head_slice_rows(shape, 2 if bf16 else 4, moe)
    if moe:
        gemm_bytes, gemm_launches = moe_gemm_algorithmic_bytes(shape, B, S, K, rows, moe,
                                                               fuse_top=not args.no_fuse_top)
    else:
        gemm_bytes, gemm_launches = gemm_algorithmic_bytes(shape, B, S, K, rows, fuse_top=not args.no_fuse_top)
    traffic_known = (args.workload == "llama8b" and (L, B, S, K) == (32, 2, 4096, 4) and bf16
                     and not args.no_fuse_top and kst["n_gemm"] == sum(GEMM_LAUNCHES_8B.values()))
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "global_batch": B * world, "seq_len": S, "checkpoint_every": K,
                   "layers": L, "hidden": h, "heads": f"{nq}q/{nkv}kv x {d}", "ffn": F, "vocab": V,
                   "host_params": "fp8 (E4M3, row scales)" if fp8 else ("bf16" if bf16 else "fp32"),
                   "host_grads": args.grad_dtype,
                   "parallelism": f"replicas x{world}",
                   **({"experts": f"{E} x SwiGLU {Fe}, top-{k_top}, softmax router"} if moe else {}),
                   "l2": "inputs larger than L2 (every step streams all weights from host)",
                   "optimizer_step": f"host AdamW included ({args.optimizer})" if args.optimizer else "none (fwd+bwd)"},
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(per_step_h2d + 2 * T * 4),
                "d2h_bytes_per_step": int(per_step_d2h + 4)},
        "gpu_launches": int(agg["n_launches"]),
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": (gemm_tflops / peak_tf) if gemm_tflops else None,
                     "traffic": gemm_traffic_per_launch_8b() if traffic_known else None,
                     "traffic_unit": "bytes per launch (ncu, cold cache, per-shape captures weighted by the "
                                     "step's launches)",
                     "algorithmic_bytes_per_launch": gemm_bytes / max(1, gemm_launches),
                     "kernel": "gemm_pair_kernel / gemm_kernel (tcgen05; all GEMM launches of one step, "
                               "event-timed per launch)",
                     "launches": kst["n_gemm"], "avg_launch_ms": kst["gemm_ms"] / max(1, kst["n_gemm"]),
                     "peak_kind": f"{peak_kind} bf16_tflops_sustained"},
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "t_measured_ms": ms_per_step, "frac": t_roof * 1e3 / ms_per_step,
                          "model_tflops_per_s": step_flop / (ms_per_step / 1e3) / 1e12,
                          "h2d_hidden_frac": agg["h2d_hidden_frac"] / steps,
                          "d2h_hidden_frac": agg["d2h_hidden_frac"] / steps,
                          "attn_tflops": (kst["attn_flop"] / (kst["attn_ms"] / 1e3) / 1e12) if kst.get("attn_ms")
                          else None,
                          "gemm_ms_per_step": kst["gemm_ms"], "attn_ms_per_step": kst["attn_ms"],
                          "compute_busy_ms_per_step": agg["compute_busy_ms"] / steps,
                          "host_ms_per_step": float(np.median(host_ms)),
                          # effective rates of the step's own copies (bytes / summed copy time)
                          "h2d_copy_gbs": agg["h2d_bytes"] / max(1e-9, agg["h2d_ms"]) / 1e6,
                          "d2h_copy_gbs": agg["d2h_bytes"] / max(1e-9, agg["d2h_ms"]) / 1e6},
        # where the copy time goes: per phase of the step, the in-step copy
        # rates; per copy, their spread; and the same weight stream replayed
        # with nothing beside it, from the bound buffer, before the warm-up
        # and after the timed steps
        "link_diagnostics": {
            "in_step_gbs_by_phase": {
                ph: {"h2d": (agg["h2d_phase_bytes"][i] / agg["h2d_phase_ms"][i] / 1e6) if agg["h2d_phase_ms"][i] else None,
                     "d2h": (agg["d2h_phase_bytes"][i] / agg["d2h_phase_ms"][i] / 1e6) if agg["d2h_phase_ms"][i] else None}
                for i, ph in enumerate(("forward", "head", "recompute", "backward"))},
            "in_step_h2d_copy_gbs": {"min": float(np.min([c[0] for c in copy_p])),
                                     "p10_median_over_steps": float(np.median([c[1] for c in copy_p])),
                                     "p50_median_over_steps": float(np.median([c[2] for c in copy_p]))},
            "replay_bound_buffer_before": replay_before,
            "replay_bound_buffer_with_page_touch": replay_touch,
            "replay_bound_buffer_after": replay_after,
            "page_touch_threads": int(os.environ.get("MT_PAGE_TOUCH", "4")),
            "page_touch_ms_per_step": agg["page_touch_ms"] / steps,
            "probe_fresh_buffer": link,
            "host_numa_node_of_gpu": replay_r["host_numa_node"],
        },
        "optimizer": ({"kind": "host AdamW, " + ("per-unit as gradients land (mt_train_step)"
                                                  if args.optimizer == "sync" else
                                                  "staleness 1, units published as they land (mt_train_step_async)"),
                       "ms_per_step": agg["optimizer_ms"] / steps,
                       "exposed_ms_per_step": agg["optimizer_exposed_ms"] / steps,
                       "params_per_s": (sess.grad_bytes / 4) / (agg["optimizer_ms"] / steps / 1e3)
                       if agg.get("optimizer_ms") else None} if args.optimizer else None),
        "host_link": link,
        "host_numa_pages": placement,
        "clocks": clk,
        "loss": losses[-1],
        "init_s": init_s,
    }
    sess.close()  # frees the pinned model before the oracle sample
    del arena
    if not args.no_cpu_baseline and world == 1:
        log("timing the CPU oracle sample")
        if args.workload in FULL_STEP_BASELINE and not (args.layers or args.seq or args.batch):
            v, t1 = cpu_oracle_full_step(shape, B, S, moe=moe, eps=eps, bf16=bf16)
            sample = (f"whole step of the {args.workload} workload at B={B}, S={S} ({t1:.2f} s single-threaded "
                      f"fp32 oracle); host has {os.cpu_count()} cores")
        else:
            fit = CpuFit(shape, moe=moe, eps=eps)
            v = B * S / fit.step_seconds(B, S)
            sample = fit.describe(B, S)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
