"""The step's GEMM launches at the full 8B shape (8192 tokens, hidden 4096,
FFN 14336, 32 q / 8 kv heads x 128), in the launch configuration the step
uses (256-wide tiles on SM pairs), checked on sampled outputs that the oracle
computes one by one, element by element (tests/bounds.py: acc(K) for the fp32
sums, U16 per bf16 rounding):
  - the input gradient of the gate-up projection, NN with K = 28672;
  - the weight gradient of the gate-up projection, TN over the 8192 tokens;
  - the gate-up projection with SwiGLU in its epilogue;
  - the q|k|v projection with RoPE in its epilogue (B = 2, S = 4096);
  - the down-projection input gradient with the SwiGLU backward in its
    epilogue.
The operands are drawn on the device with torch's seeded generator (the same
values go to both sides) to keep the host work of a full-size test short.
"""
import numpy as np
import pytest

import oracle
from tests.bounds import U16, U32, acc, check, pair_sum, silu_parts
from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu

T, H, F, NQ, NKV, D = 8192, 4096, 14336, 32, 8, 128
N_SAMPLES = 2000


def _bf16(torch, shape, gen, std):
    return (torch.randn(shape, generator=gen, device="cuda") * std).to(torch.bfloat16)


def _host(t):
    return t.float().cpu().numpy()


def _samples(seed, M, N):
    rng = np.random.default_rng(seed)
    return rng.integers(0, M, N_SAMPLES), rng.integers(0, N, N_SAMPLES)


def test_nn_input_gradient_k28672():
    """dm = d(g|u) [8192, 28672] x Wgu [28672, 4096] (fp32 out)."""
    torch, mt = need_gpu()
    gen = torch.Generator(device="cuda").manual_seed(301)
    A = _bf16(torch, (T, 2 * F), gen, 0.05)
    B = _bf16(torch, (2 * F, H), gen, 0.02)
    C = torch.empty((T, H), device="cuda")
    mt.mt_op_gemm(mt.MT_GEMM_NN, mt.MT_EPI_F32, A, B, C, None, T, H, 2 * F, 2 * F, H, H)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    rows, cols = _samples(302, T, H)
    a, b = _host(A), _host(B)
    got = C.cpu().numpy()[rows, cols]
    ref = oracle.matmul_sampled("nn", a, b, rows, cols)
    check(got, ref, acc(2 * F) * oracle.matmul_sampled("nn", np.abs(a), np.abs(b), rows, cols), "dm")


def test_tn_weight_gradient_over_8192_tokens():
    """dWgu [28672, 4096] = d(g|u)^T [8192, 28672]^T x m [8192, 4096] (fp32)."""
    torch, mt = need_gpu()
    gen = torch.Generator(device="cuda").manual_seed(311)
    A = _bf16(torch, (T, 2 * F), gen, 0.05)
    B = _bf16(torch, (T, H), gen, 1.0)
    C = torch.empty((2 * F, H), device="cuda")
    mt.mt_op_gemm(mt.MT_GEMM_TN, mt.MT_EPI_F32, A, B, C, None, 2 * F, H, T, 2 * F, H, H)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    rows, cols = _samples(312, 2 * F, H)
    a, b = _host(A), _host(B)
    got = C.cpu().numpy()[rows, cols]
    ref = oracle.matmul_sampled("tn", a, b, rows, cols)
    check(got, ref, acc(T) * oracle.matmul_sampled("tn", np.abs(a), np.abs(b), rows, cols), "dWgu")


def test_gate_up_projection_with_swiglu_epilogue():
    """g|u = m [8192, 4096] [Wg; Wu]^T [28672, 4096], act = silu(g) u."""
    torch, mt = need_gpu()
    gen = torch.Generator(device="cuda").manual_seed(321)
    X = _bf16(torch, (T, H), gen, 1.0)
    W = _bf16(torch, (2 * F, H), gen, 0.02)
    GU = torch.empty((T, 2 * F), dtype=torch.bfloat16, device="cuda")
    ACT = torch.empty((T, F), dtype=torch.bfloat16, device="cuda")
    mt.mt_op_gemm_swiglu(X, W, GU, ACT, T, F, H, H, H, F)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    rows, cols = _samples(322, T, F)
    x, w = _host(X), _host(W)
    g = oracle.matmul_sampled("nt", x, w, rows, cols)
    u = oracle.matmul_sampled("nt", x, w, rows, cols + F)
    eg = acc(H) * oracle.matmul_sampled("nt", np.abs(x), np.abs(w), rows, cols)
    eu = acc(H) * oracle.matmul_sampled("nt", np.abs(x), np.abs(w), rows, cols + F)
    a_ref, _, _ = oracle.swiglu(g, u)
    gu = _host(GU)
    check(gu[rows, cols], g, U16 * np.abs(g) + (1 + U16) * eg, "g")
    check(gu[rows, cols + F], u, U16 * np.abs(u) + (1 + U16) * eu, "u")
    _, silu_g, dsilu_mag = silu_parts(g)
    e_act = dsilu_mag * np.abs(u) * eg + np.abs(silu_g) * eu
    check(_host(ACT)[rows, cols], a_ref, (U16 + 1e-5) * np.abs(a_ref) + (1 + U16) * e_act, "act")


def test_qkv_projection_with_rope_epilogue():
    """q|k|v = a [8192, 4096] Wqkv^T [6144, 4096] with RoPE (theta 5e5) on the
    40 q and k heads at position row % 4096; 48 whole sampled rows, rotated
    by the oracle at their positions."""
    torch, mt = need_gpu()
    B, S, theta = 2, 4096, 5e5
    N = (NQ + 2 * NKV) * D
    gen = torch.Generator(device="cuda").manual_seed(331)
    A = _bf16(torch, (T, H), gen, 1.0)
    W = _bf16(torch, (N, H), gen, 0.02)
    C = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    tab = torch.empty(S * D, device="cuda")
    mt.mt_op_gemm_rope(A, W, C, T, N, H, H, H, N, tab, S, D, theta, (NQ + NKV) * D)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    rng = np.random.default_rng(332)
    rows = np.sort(rng.choice(T, 48, replace=False))
    a, w = _host(A), _host(W)
    rr, cc = np.repeat(rows, N), np.tile(np.arange(N), rows.size)
    prod = oracle.matmul_sampled("nt", a, w, rr, cc).reshape(rows.size, NQ + 2 * NKV, D)
    err = (acc(H) * oracle.matmul_sampled("nt", np.abs(a), np.abs(w), rr, cc)).reshape(prod.shape)
    # rotate the sampled rows at their own positions: place them in a
    # [B, S, heads, D] array and let the oracle rotate it
    full = np.zeros((B, S, NQ + NKV, D), np.float32)
    full[rows // S, rows % S] = prod[:, :NQ + NKV]
    ref = prod.copy()
    ref[:, :NQ + NKV] = oracle.rope(full, theta)[rows // S, rows % S]
    bound = err.copy()
    bound[:, :NQ + NKV] = pair_sum(err[:, :NQ + NKV]) + 4 * U32 * pair_sum(np.abs(prod[:, :NQ + NKV]))
    got = _host(C)[rows].reshape(prod.shape)
    check(got, ref, U16 * np.abs(ref) + (1 + U16) * bound, "qkv+rope")


def test_down_input_gradient_with_swiglu_backward_epilogue():
    """dact = dh [8192, 4096] Wd [4096, 14336]; (g, u) overwritten in place by
    dg = dact u silu'(g), du = dact silu(g)."""
    torch, mt = need_gpu()
    gen = torch.Generator(device="cuda").manual_seed(341)
    dY = _bf16(torch, (T, H), gen, 0.05)
    Wd = _bf16(torch, (H, F), gen, 0.02)
    GU = _bf16(torch, (T, 2 * F), gen, 1.0)
    gu0 = _host(GU)
    mt.mt_op_gemm_swiglu_bwd(dY, Wd, GU, T, F, H, H, F, F)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    rows, cols = _samples(342, T, F)
    dy, wd = _host(dY), _host(Wd)
    dact = oracle.matmul_sampled("nn", dy, wd, rows, cols)
    e_da = acc(H) * oracle.matmul_sampled("nn", np.abs(dy), np.abs(wd), rows, cols)
    g, u = gu0[rows, cols], gu0[rows, cols + F]
    _, dg_ref, du_ref = oracle.swiglu(g, u, dact)
    _, silu_g, dsilu_mag = silu_parts(g)
    out = _host(GU)
    check(out[rows, cols], dg_ref,
          U16 * np.abs(dg_ref) + (1 + U16) * dsilu_mag * np.abs(u) * (e_da + 1e-5 * np.abs(dact)), "dg")
    check(out[rows, cols + F], du_ref,
          U16 * np.abs(du_ref) + (1 + U16) * np.abs(silu_g) * (e_da + 1e-5 * np.abs(dact)), "du")
