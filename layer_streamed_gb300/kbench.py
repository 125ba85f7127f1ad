"""Kernel benchmark CLI: time one layer-template kernel at a given shape.

  python -m layer_streamed_gb300.kbench gemm --mode nt --M 8192 --N 28672 --K 4096 [--reps 20]
  python -m layer_streamed_gb300.kbench gemm --shape dm        (one of the 8B step's GEMM launches)
  python -m layer_streamed_gb300.kbench attn --B 2 --S 4096 --heads 32 --kv-heads 8 --head-dim 128 [--bwd]
  python -m layer_streamed_gb300.kbench norm --T 8192 --h 4096 [--bwd]
  python -m layer_streamed_gb300.kbench moe --T 4096 --h 4096 --experts 128 --top-k 8 --expert-ffn 1536

Inputs are random bf16 tensors on the current GPU (larger than L2 at the 8B
shapes); each launch is timed with CUDA events on the launching stream after
warm-up. Prints one JSON line with the per-launch time and TFLOP/s (GB/s
of algorithmic traffic for the norms). The qkv_rope shape goes through
mt_op_gemm_rope, which rebuilds the cos/sin table on every call (about
0.08 ms at S = 4096); the training step builds it once per sequence length,
so its QKV projection is the GEMM alone.
"""
from __future__ import annotations

import argparse
import json

import torch

import layer_streamed_gb300 as mt


def _time(fn, reps: int, warmup: int = 3) -> float:
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


# The GEMM launches of one decoder layer of the 8B step (T = 8192 tokens,
# hidden 4096, q|k|v 6144, FFN 14336) and of one LM-head vocab slice (42752
# rows): name -> (mode, M, N, K, output / fused epilogue), N counting the
# columns the launch writes (gate-up: g and u).
STEP_SHAPES_8B = {
    "qkv_rope": ("nt", 8192, 6144, 4096, "rope"),
    "o_proj": ("nt", 8192, 4096, 4096, "f32add"),
    "gate_up": ("nt", 8192, 28672, 4096, "gated"),
    "down": ("nt", 8192, 4096, 14336, "f32add"),
    "dWd": ("tn", 4096, 14336, 8192, "f32"),
    "dact_swiglu": ("nn", 8192, 14336, 4096, "swiglu_bwd"),
    "dWgu": ("tn", 28672, 4096, 8192, "f32"),
    "dm": ("nn", 8192, 4096, 28672, "f32"),
    "dWo": ("tn", 4096, 4096, 8192, "f32"),
    "do": ("nn", 8192, 4096, 4096, "bf16"),
    "dWqkv": ("tn", 6144, 4096, 8192, "f32"),
    "dx": ("nn", 8192, 4096, 6144, "f32"),
    "head_logits": ("nt", 8192, 42752, 4096, "f32"),
    "head_dX": ("nn", 8192, 4096, 42752, "f32add"),
    "head_dW": ("tn", 42752, 4096, 8192, "f32"),
}
# Launches of each in one step at the 8B configuration (32 layers, K = 4,
# top block not recomputed: 60 forward passes of a layer, 32 backward; three
# vocab slices, each with two logits passes, one dX and one dW product).
STEP_LAUNCHES_8B = {"qkv_rope": 60, "o_proj": 60, "gate_up": 60, "down": 60, "dWd": 32, "dact_swiglu": 32,
                    "dWgu": 32, "dm": 32, "dWo": 32, "do": 32, "dWqkv": 32, "dx": 32, "head_logits": 6,
                    "head_dX": 3, "head_dW": 3}


def bench_gemm(args) -> dict:
    if args.shape:
        args.mode, args.M, args.N, args.K, args.out = STEP_SHAPES_8B[args.shape]
    M, N, K = args.M, args.N, args.K
    mode = {"nt": mt.MT_GEMM_NT, "nn": mt.MT_GEMM_NN, "tn": mt.MT_GEMM_TN}[args.mode]
    a_shape = (M, K) if args.mode in ("nt", "nn") else (K, M)
    b_shape = (N, K) if args.mode == "nt" else (K, N)
    A = torch.randn(a_shape, device="cuda").to(torch.bfloat16)
    B = (torch.randn(b_shape, device="cuda") * 0.02).to(torch.bfloat16)
    out = args.out
    if out in ("bf16", "f32", "f32add"):
        epi = {"bf16": mt.MT_EPI_BF16, "f32": mt.MT_EPI_F32, "f32add": mt.MT_EPI_F32_ADD}[out]
        C = torch.empty((M, N), device="cuda", dtype=torch.bfloat16 if out == "bf16" else torch.float32)
        add = torch.randn((M, N), device="cuda") if out == "f32add" else None
        fn = lambda: mt.mt_op_gemm(mode, epi, A, B, C, add, M, N, K, a_shape[1], b_shape[1], N)
    elif out == "rope":  # q|k|v with RoPE on the first (n_q + n_kv) heads of 128 (S = 4096 per sequence)
        C = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        tab = torch.empty(4096 * 128, device="cuda")
        fn = lambda: mt.mt_op_gemm_rope(A, B, C, M, N, K, K, K, N, tab, 4096, 128, 5e5, N - 1024)
    elif out == "gated":  # g|u with act = silu(g) u: N = 2F
        F = N // 2
        GU = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        ACT = torch.empty((M, F), device="cuda", dtype=torch.bfloat16)
        fn = lambda: mt.mt_op_gemm_swiglu(A, B, GU, ACT, M, F, K, K, K, F)
    elif out == "swiglu_bwd":  # d(act) = dY Wd turned into (dg, du) over g|u in place: N = F
        GU = torch.randn((M, 2 * N), device="cuda").to(torch.bfloat16)
        fn = lambda: mt.mt_op_gemm_swiglu_bwd(A, B, GU, M, N, K, K, N, N)
    else:
        raise SystemExit(f"unknown output {out}")
    ms = _time(fn, args.reps)
    flop = 2.0 * M * N * K
    return {"kernel": "gemm", "shape": args.shape, "mode": args.mode, "M": M, "N": N, "K": K, "out": out, "ms": ms,
            "tflops": flop / ms / 1e9}


def bench_attn(args) -> dict:
    B, S, nq, nkv, d = args.B, args.S, args.heads, args.kv_heads, args.head_dim
    T, qd, kd = B * S, nq * d, nkv * d
    ld = qd + 2 * kd
    qkv = torch.randn((T, ld), device="cuda").to(torch.bfloat16)
    o = torch.empty((T, qd), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B * nq * S, device="cuda")
    fwd = lambda: mt.mt_op_attention_fwd(qkv, qkv[:, qd:], qkv[:, qd + kd:], o, lse, B, S, nq, nkv, d, ld, ld, qd)
    flop = 2.0 * B * nq * d * S * (S + 1)  # causal Q K^T and P V
    if not args.bwd:
        ms = _time(fwd, args.reps)
        return {"kernel": "attention_fwd", "B": B, "S": S, "heads": nq, "kv_heads": nkv, "head_dim": d, "ms": ms,
                "tflops": flop / ms / 1e9}
    fwd()
    do = torch.randn((T, qd), device="cuda").to(torch.bfloat16)
    dqkv = torch.empty_like(qkv)
    ws = torch.empty(mt.mt_op_attention_bwd_workspace(B, S, nq), device="cuda")
    bwd = lambda: mt.mt_op_attention_bwd(qkv, qkv[:, qd:], qkv[:, qd + kd:], o, do, lse, dqkv, dqkv[:, qd:],
                                         dqkv[:, qd + kd:], ws, B, S, nq, nkv, d, ld, ld, qd)
    ms = _time(bwd, args.reps)
    return {"kernel": "attention_bwd", "B": B, "S": S, "heads": nq, "kv_heads": nkv, "head_dim": d, "ms": ms,
            "tflops": 2.5 * flop / ms / 1e9}


def bench_norm(args) -> dict:
    T, h = args.T, args.h
    x = torch.randn((T, h), device="cuda")
    w = 1.0 + 0.1 * torch.randn(h, device="cuda")
    dy, res = torch.randn((T, h), device="cuda"), torch.randn((T, h), device="cuda")
    y = torch.empty((T, h), device="cuda", dtype=torch.bfloat16)
    rstd = torch.empty(T, device="cuda")
    mt.mt_op_rmsnorm_fwd(x, w, y, rstd, T, h, 1e-5)
    dx, dxb, dw = torch.empty_like(x), torch.empty((T, h), device="cuda", dtype=torch.bfloat16), torch.empty_like(w)
    ws = torch.empty(mt.mt_op_rmsnorm_bwd_workspace(T, h), device="cuda")
    if args.bwd:
        ms = _time(lambda: mt.mt_op_rmsnorm_bwd(x, w, rstd, dy, res, dx, dxb, dw, ws, T, h), args.reps)
        nbytes = T * h * (4 * 3 + 4 + 2)  # read x, dy, residual; write dx fp32 and bf16
    else:
        ms = _time(lambda: mt.mt_op_rmsnorm_fwd(x, w, y, rstd, T, h, 1e-5), args.reps)
        nbytes = T * h * (4 + 2)
    return {"kernel": "rmsnorm_bwd" if args.bwd else "rmsnorm_fwd", "T": T, "h": h, "ms": ms,
            "gbs": nbytes / ms / 1e6}


def bench_moe(args) -> dict:
    """Mixture-of-experts FFN forward (mt_op_moe_ffn_fwd): router, routing,
    grouped gate|up and down expert GEMMs, combine. TFLOP/s counts the
    routed rows' expert products and the router."""
    T, h, E, k, Fe = args.T, args.h, args.experts, args.top_k, args.expert_ffn
    m = torch.randn((T, h), device="cuda").to(torch.bfloat16)
    wr = (torch.randn((E, h), device="cuda") * 0.02).to(torch.bfloat16)
    wgu = (torch.randn((E, 2 * Fe, h), device="cuda") * 0.02).to(torch.bfloat16)
    wd = (torch.randn((E, h, Fe), device="cuda") * 0.02).to(torch.bfloat16)
    resid = torch.zeros((T, h), device="cuda")
    out = torch.empty((T, h), device="cuda")
    route = torch.empty((T, k), device="cuda", dtype=torch.int32)
    ws = torch.empty(mt.mt_op_moe_workspace(T, h, E, k, Fe), device="cuda", dtype=torch.uint8)
    ms = _time(lambda: mt.mt_op_moe_ffn_fwd(m, wr, wgu, wd, resid, out, route, ws, T, h, E, k, Fe), args.reps)
    flop = 2.0 * T * E * h + 2.0 * T * k * 3 * Fe * h
    return {"kernel": "moe_ffn_fwd", "T": T, "h": h, "experts": E, "top_k": k, "expert_ffn": Fe, "ms": ms,
            "tflops": flop / ms / 1e9}


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="op", required=True)
    g = sub.add_parser("gemm")
    g.add_argument("--mode", default="nt", choices=["nt", "nn", "tn"])
    g.add_argument("--M", type=int, default=8192)
    g.add_argument("--N", type=int, default=28672)
    g.add_argument("--K", type=int, default=4096)
    g.add_argument("--out", default="bf16", choices=["bf16", "f32", "f32add", "rope", "gated", "swiglu_bwd"])
    g.add_argument("--shape", default=None, choices=sorted(STEP_SHAPES_8B),
                   help="one of the 8B step's GEMM launches (sets mode, M, N, K and the epilogue)")
    g.add_argument("--reps", type=int, default=20)
    a = sub.add_parser("attn")
    a.add_argument("--B", type=int, default=2)
    a.add_argument("--S", type=int, default=4096)
    a.add_argument("--heads", type=int, default=32)
    a.add_argument("--kv-heads", type=int, default=8)
    a.add_argument("--head-dim", type=int, default=128)
    a.add_argument("--bwd", action="store_true")
    a.add_argument("--reps", type=int, default=20)
    n = sub.add_parser("norm")
    n.add_argument("--T", type=int, default=8192)
    n.add_argument("--h", type=int, default=4096)
    n.add_argument("--bwd", action="store_true")
    n.add_argument("--reps", type=int, default=20)
    e = sub.add_parser("moe")
    e.add_argument("--T", type=int, default=4096)
    e.add_argument("--h", type=int, default=4096)
    e.add_argument("--experts", type=int, default=128)
    e.add_argument("--top-k", type=int, default=8)
    e.add_argument("--expert-ffn", type=int, default=1536)
    e.add_argument("--reps", type=int, default=20)
    args = ap.parse_args()
    mt.build()
    res = {"gemm": bench_gemm, "attn": bench_attn, "norm": bench_norm, "moe": bench_moe}[args.op](args)
    res["device_error"] = mt.mt_op_device_error()
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
