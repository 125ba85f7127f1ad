"""GPU parity of the layer-template kernels against the CPU oracle.

Inputs are seeded normals rounded to bf16, so both sides see exactly the same
operand values; the oracle accumulates in double. Every output is checked
element by element against a bound derived from the arithmetic
(tests/bounds.py: U16 = 2^-8 per bf16 rounding, acc(K) for an fp32 sum of K
products, magnitudes from the oracle run on absolute values), and as a whole
by relative L2 error: fp32 outputs <= 1e-4; one bf16 rounding (at most 2^-8
relative per element, RMS about 1.1e-3) <= 6e-3; outputs that pass through
another bf16 rounding (attention probabilities, SwiGLU) <= 1.5e-2.
"""
import math

import numpy as np
import pytest

import oracle
import seedgen
from tests.bounds import U16, U32, acc, attention_magnitudes, check, pair_sum, silu_parts
from tests.common import bf16_round, rel_l2
from tests.gpu_util import from_dev, need_gpu, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _normal(shape, seed, std=1.0):
    return seedgen.normal(int(np.prod(shape)), seed, 7, std).reshape(shape)


def ATT_O(o_ref, o_abs, S):
    """Attention output: the bf16 rounding of P (and the row sum formed from
    the unrounded P) move each term of sum_j P_ij v_j by at most 2 U16 of
    P_ij |v_j|, the fp32 sums add acc(S), and the result is rounded once."""
    return U16 * np.abs(o_ref) + (2 * U16 + acc(S)) * o_abs


def ATT_G(g_ref, g_abs):
    """Attention gradients: bf16 roundings of P, dS and the forward output
    (five U16 of the magnitude sums, see attention_magnitudes) and one
    rounding of the result."""
    return U16 * np.abs(g_ref) + 5 * U16 * g_abs


GEMM_SHAPES = [
    (128, 256, 64),     # one tile
    (64, 192, 64),      # smaller than a tile (the tiny decoder's QKV)
    (200, 300, 136),    # ragged M, N, K
    (1000, 520, 328),   # several tiles, ragged
    (2048, 4096, 200),  # enough tiles for the 256-wide variant, ragged K
]


@pytest.mark.parametrize("mode", ["nt", "nn", "tn"])
@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_modes_against_oracle(mode, shape):
    torch, mt = need_gpu()
    M, N, K = shape
    a_shape = (M, K) if mode in ("nt", "nn") else (K, M)
    b_shape = (N, K) if mode == "nt" else (K, N)
    # operands are stored with row strides padded to 8 elements (TMA needs
    # 16-byte strides); only the logical a_shape/b_shape part is used
    pad = lambda n: (n + 7) // 8 * 8
    A_st = np.zeros((a_shape[0], pad(a_shape[1])), np.float32)
    B_st = np.zeros((b_shape[0], pad(b_shape[1])), np.float32)
    A_st[:, :a_shape[1]] = _normal(a_shape, M + 1)
    B_st[:, :b_shape[1]] = _normal(b_shape, N + 2)
    A, a32 = to_dev_bf16(torch, A_st)
    B, b32 = to_dev_bf16(torch, B_st)
    a32, b32 = a32[:, :a_shape[1]], b32[:, :b_shape[1]]
    ref = oracle.matmul(mode, a32, b32)
    ab = oracle.matmul(mode, np.abs(a32), np.abs(b32))  # sum_k |a||b| per output
    e_acc = acc(K) * ab
    add = _normal((M, N), 5)
    mode_id = {"nt": mt.MT_GEMM_NT, "nn": mt.MT_GEMM_NN, "tn": mt.MT_GEMM_TN}[mode]
    lda, ldb = A_st.shape[1], B_st.shape[1]
    # fp32 out
    C = torch.full((M, N), float("nan"), device="cuda")
    mt.mt_op_gemm(mode_id, mt.MT_EPI_F32, A, B, C, None, M, N, K, lda, ldb, N)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    assert rel_l2(from_dev(C), ref) < 1e-4
    check(from_dev(C), ref, e_acc, "fp32")
    # fp32 out = addend + acc, in place
    C2 = to_dev_f32(torch, add)
    mt.mt_op_gemm(mode_id, mt.MT_EPI_F32_ADD, A, B, C2, C2, M, N, K, lda, ldb, N)
    assert rel_l2(from_dev(C2), ref + add) < 1e-4
    check(from_dev(C2), ref + add, e_acc + 2 * U32 * (np.abs(ref + add) + np.abs(add)), "fp32 + addend")
    # bf16 out
    Cb = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    mt.mt_op_gemm(mode_id, mt.MT_EPI_BF16, A, B, Cb, None, M, N, K, lda, ldb, N)
    assert rel_l2(from_dev(Cb), ref) < 6e-3
    check(from_dev(Cb), ref, U16 * np.abs(ref) + (1 + U16) * e_acc, "bf16")


def test_gemm_strided_operands_and_unaligned_output():
    """Row strides larger than the logical width, and an fp32 output whose row
    stride is not a multiple of 4 elements (element-wise store path)."""
    torch, mt = need_gpu()
    M, N, K = 130, 172, 96
    A_full, a32 = to_dev_bf16(torch, _normal((M, K + 32), 11))
    B_full, b32 = to_dev_bf16(torch, _normal((N, K + 8), 12))
    ref = oracle.matmul("nt", a32[:, :K], b32[:, :K])
    C = torch.zeros((M, N + 1), device="cuda")
    mt.mt_op_gemm(mt.MT_GEMM_NT, mt.MT_EPI_F32, A_full, B_full, C, None, M, N, K, K + 32, K + 8, N + 1)
    assert rel_l2(from_dev(C)[:, :N], ref) < 1e-4
    check(from_dev(C)[:, :N], ref, acc(K) * oracle.matmul("nt", np.abs(a32[:, :K]), np.abs(b32[:, :K])))
    assert np.all(from_dev(C)[:, N] == 0)


def test_gemm_rejects_misaligned_strides():
    torch, mt = need_gpu()
    A = torch.zeros((64, 70), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), device="cuda")
    with pytest.raises(mt.MtError):
        mt.mt_op_gemm(mt.MT_GEMM_NT, mt.MT_EPI_F32, A, A, C, None, 64, 64, 70, 70, 70, 64)


def test_gemm_sampled_at_full_8b_qkv_shape():
    """The 8B QKV projection (M=8192 tokens, N=6144, K=4096), checked on 2000
    sampled outputs computed one by one by the oracle."""
    torch, mt = need_gpu()
    M, N, K = 8192, 6144, 4096
    A, a32 = to_dev_bf16(torch, _normal((M, K), 3, 0.5))
    B, b32 = to_dev_bf16(torch, _normal((N, K), 4, 0.02))
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mt.mt_op_gemm(mt.MT_GEMM_NT, mt.MT_EPI_F32, A, B, C, None, M, N, K, K, K, N)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, M, 2000), rng.integers(0, N, 2000)
    ref = oracle.matmul_sampled("nt", a32, b32, rows, cols)
    ab = oracle.matmul_sampled("nt", np.abs(a32), np.abs(b32), rows, cols)
    got = from_dev(C)[rows, cols]
    check(got, ref, acc(K) * ab)


@pytest.mark.parametrize("T,h,with_res", [(77, 320, True), (45, 1800, False), (33, 4096, True), (9, 6000, True)])
def test_rmsnorm_forward_backward(T, h, with_res):
    """Widths that select each per-thread vector count of the backward
    kernel (h/4 up to 256, 512, 1024, 2048 float4), ragged row counts (odd
    rows in the last block), with and without the residual input."""
    torch, mt = need_gpu()
    eps = 1e-5
    x = _normal((T, h), 21)
    w = 1.0 + 0.1 * _normal((h,), 22)
    dy = _normal((T, h), 23)
    res = _normal((T, h), 24)
    X, W = to_dev_f32(torch, x), to_dev_f32(torch, w)
    Y = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    R = torch.empty(T, device="cuda")
    mt.mt_op_rmsnorm_fwd(X, W, Y, R, T, h, eps)
    y_ref, r_ref = oracle.rmsnorm_fwd(x, w, eps)
    assert rel_l2(from_dev(Y), y_ref) < 6e-3
    assert rel_l2(from_dev(R), r_ref) < 1e-5
    # rstd from an fp32 sum of h squares and a reciprocal square root (a few ulp)
    e_r = acc(h) + 4 * U32
    check(from_dev(R), r_ref, e_r * np.abs(r_ref), "rstd")
    check(from_dev(Y), y_ref, (U16 + (1 + U16) * (e_r + 4 * U32)) * np.abs(y_ref), "y")
    DX = torch.empty((T, h), device="cuda")
    DXb = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    DW = torch.empty(h, device="cuda")
    ws = torch.empty(mt.mt_op_rmsnorm_bwd_workspace(T, h), device="cuda")
    if not with_res:
        res = np.zeros_like(res)
    mt.mt_op_rmsnorm_bwd(X, W, R, to_dev_f32(torch, dy), to_dev_f32(torch, res) if with_res else None, DX, DXb, DW,
                         ws, T, h)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(x, w, dy, eps)
    assert rel_l2(from_dev(DX), dx_ref + res) < 1e-5
    assert rel_l2(from_dev(DXb), dx_ref + res) < 6e-3
    assert rel_l2(from_dev(DW), dw_ref) < 1e-5
    # dx = rstd w dy - x rstd^3 (1/h) sum_j w_j dy_j x_j (+ res): the terms'
    # magnitudes times the relative error of rstd (three powers of it), of the
    # row sum and of a few fp32 operations
    r64 = r_ref.astype(np.float64)[:, None]
    t1 = r64 * np.abs(w * dy)
    t2 = np.abs(x) * r64 ** 3 * np.mean(np.abs(w * dy * x), axis=1, keepdims=True)
    e_dx = (3 * e_r + acc(h) + 8 * U32) * (t1 + t2) + 2 * U32 * (np.abs(dx_ref + res) + np.abs(res))
    check(from_dev(DX), dx_ref + res, e_dx, "dx")
    check(from_dev(DXb), dx_ref + res, U16 * np.abs(dx_ref + res) + (1 + U16) * e_dx, "dx bf16")
    check(from_dev(DW), dw_ref, (e_r + acc(T) + 4 * U32) * np.sum(np.abs(dy * x) * r64, axis=0), "dw")


@pytest.mark.parametrize("d", [16, 64, 128])
def test_rope_forward_and_inverse(d):
    torch, mt = need_gpu()
    B, S, nq, nkv, theta = 2, 37, 4, 2, 5e5
    width = (nq + 2 * nkv) * d
    x = _normal((B * S, width), 31 + d)
    X, x32 = to_dev_bf16(torch, x)
    tab = torch.empty(S * d, device="cuda")
    mt.mt_op_rope(X, tab, B, S, width, 0, nq + nkv, d, theta, 1)
    got = from_dev(X).reshape(B, S, nq + 2 * nkv, d)
    xin = x32.reshape(B, S, nq + 2 * nkv, d)[:, :, :nq + nkv]
    ref = oracle.rope(xin, theta)
    assert rel_l2(got[:, :, :nq + nkv], ref) < 6e-3
    # one bf16 rounding of x cos - x' sin formed in fp32 from fp32 cos/sin
    check(got[:, :, :nq + nkv], ref, U16 * np.abs(ref) + 4 * U32 * pair_sum(np.abs(xin)), "rope")
    np.testing.assert_array_equal(got[:, :, nq + nkv:], x32.reshape(B, S, -1, d)[:, :, nq + nkv:])  # v untouched
    mt.mt_op_rope(X, tab, B, S, width, 0, nq + nkv, d, theta, -1)
    assert rel_l2(from_dev(X), x32) < 1e-2
    # forward then inverse: the forward's rounding error rotated back, plus
    # the second rounding
    back = from_dev(X).reshape(B, S, nq + 2 * nkv, d)[:, :, :nq + nkv]
    check(back, xin, U16 * np.abs(xin) + (2 * U16 + 8 * U32) * pair_sum(pair_sum(np.abs(xin))), "rope inverse")


@pytest.mark.parametrize("F,ld", [(172, 176), (256, 256)])
def test_swiglu_forward_backward(F, ld):
    torch, mt = need_gpu()
    T = 53
    g, u, da = _normal((T, F), 41), _normal((T, F), 42), _normal((T, F), 43)
    gu = np.zeros((T, 2 * ld), np.float32)
    gu[:, :F], gu[:, ld:ld + F] = g, u
    GU, gu32 = to_dev_bf16(torch, gu)
    DA = np.zeros((T, ld), np.float32)
    DA[:, :F] = da
    DAd, da32 = to_dev_bf16(torch, DA)
    ACT = torch.full((T, ld), 7.0, dtype=torch.bfloat16, device="cuda")
    mt.mt_op_swiglu_fwd(GU, ACT, T, F, ld)
    g32, u32 = gu32[:, :F], gu32[:, ld:ld + F]
    a_ref, dg_ref, du_ref = oracle.swiglu(g32, u32, da32[:, :F])
    act = from_dev(ACT)
    assert rel_l2(act[:, :F], a_ref) < 6e-3
    assert np.all(act[:, F:] == 0)
    # one bf16 rounding of fp32 products; the exponential is a few ulp; silu'
    # can cancel, so its bound uses the magnitude of its terms
    _, _, dsilu_mag = silu_parts(g32)
    check(act[:, :F], a_ref, (U16 + 1e-5) * np.abs(a_ref), "act")
    mt.mt_op_swiglu_bwd(GU, DAd, T, F, ld)
    out = from_dev(GU)
    assert rel_l2(out[:, :F], dg_ref) < 6e-3
    assert rel_l2(out[:, ld:ld + F], du_ref) < 6e-3
    check(out[:, :F], dg_ref, U16 * np.abs(dg_ref) + 1e-5 * np.abs(da32[:, :F] * u32) * dsilu_mag, "dg")
    check(out[:, ld:ld + F], du_ref, (U16 + 1e-5) * np.abs(du_ref), "du")


@pytest.mark.parametrize("d,S,nq,nkv", [(16, 32, 4, 4), (64, 200, 4, 2), (128, 130, 8, 2), (128, 1, 2, 1),
                                         (128, 300, 16, 1)])
def test_attention_forward_backward(d, S, nq, nkv):
    torch, mt = need_gpu()
    B = 2
    q, k, v, do = (_normal((B, S, n, d), 50 + i) for i, n in enumerate((nq, nkv, nkv, nq)))
    Q, q32 = to_dev_bf16(torch, q)
    Kd, k32 = to_dev_bf16(torch, k)
    Vd, v32 = to_dev_bf16(torch, v)
    DO, do32 = to_dev_bf16(torch, do)
    O = torch.empty((B, S, nq, d), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((B, nq, S), device="cuda")
    mt.mt_op_attention_fwd(Q, Kd, Vd, O, LSE, B, S, nq, nkv, d, nq * d, nkv * d, nq * d)
    o_ref, lse_ref, *_ = oracle.attention(q32, k32, v32)
    o_abs, dq_abs, dk_abs, dv_abs = attention_magnitudes(q32, k32, v32, do32)
    assert rel_l2(from_dev(O), o_ref) < 1.5e-2
    check(from_dev(O), o_ref, ATT_O(o_ref, o_abs, S), "o")
    check(from_dev(LSE), lse_ref, 1e-3, "lse")
    dQ = torch.empty_like(Q)
    dK = torch.empty_like(Kd)
    dV = torch.empty_like(Vd)
    ws = torch.empty(mt.mt_op_attention_bwd_workspace(B, S, nq), device="cuda")
    mt.mt_op_attention_bwd(Q, Kd, Vd, O, DO, LSE, dQ, dK, dV, ws, B, S, nq, nkv, d, nq * d, nkv * d, nq * d)
    _, _, dq_ref, dk_ref, dv_ref = oracle.attention(q32, k32, v32, do32)
    assert rel_l2(from_dev(dQ), dq_ref) < 2e-2
    assert rel_l2(from_dev(dK), dk_ref) < 2e-2
    assert rel_l2(from_dev(dV), dv_ref) < 2e-2
    check(from_dev(dQ), dq_ref, ATT_G(dq_ref, dq_abs), "dq")
    check(from_dev(dK), dk_ref, ATT_G(dk_ref, dk_abs), "dk")
    check(from_dev(dV), dv_ref, ATT_G(dv_ref, dv_abs), "dv")
    assert mt.mt_op_device_error() == 0


def test_attention_growing_scores_rescale_per_warp():
    """Rows whose scores keep growing along the keys (so the running maximum
    jumps in later tiles) interleaved with rows whose scores shrink, over
    several 128-key tiles: neighbouring rows of one warp need different
    online-softmax rescaling decisions."""
    torch, mt = need_gpu()
    B, S, nq, nkv, d = 1, 640, 2, 1, 128
    rng = np.random.default_rng(7)
    u = rng.normal(size=d)
    u /= np.linalg.norm(u)
    ramp = np.linspace(0.0, 1.0, S)[:, None]
    k = (ramp * 6.0 * u[None, :] + 0.3 * rng.normal(size=(S, d))).reshape(B, S, nkv, d)
    sign = np.where(np.arange(S) % 2 == 0, 1.0, -1.0)[:, None, None]
    q = (sign * 6.0 * u[None, None, :] + 0.3 * rng.normal(size=(S, nq, d))).reshape(B, S, nq, d)
    v = rng.normal(size=(B, S, nkv, d))
    Q, q32 = to_dev_bf16(torch, q)
    Kd, k32 = to_dev_bf16(torch, k)
    Vd, v32 = to_dev_bf16(torch, v)
    O = torch.empty((B, S, nq, d), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((B, nq, S), device="cuda")
    mt.mt_op_attention_fwd(Q, Kd, Vd, O, LSE, B, S, nq, nkv, d, nq * d, nkv * d, nq * d)
    o_ref, lse_ref, *_ = oracle.attention(q32, k32, v32)
    assert mt.mt_op_device_error() == 0
    assert rel_l2(from_dev(O), o_ref) < 1.5e-2
    o_abs = oracle.attention(q32, k32, np.abs(v32))[0]
    check(from_dev(O), o_ref, ATT_O(o_ref, o_abs, S), "o")
    check(from_dev(LSE), lse_ref, 2e-3 * np.max(np.abs(lse_ref)), "lse")


@pytest.mark.parametrize("d,nq,nkv", [(128, 4, 2), (64, 4, 4), (16, 4, 2)])
def test_qkv_gemm_with_fused_rope(d, nq, nkv):
    """q|k|v = a W^T with RoPE on the q and k heads in the epilogue, against
    the oracle's product followed by its rotation."""
    torch, mt = need_gpu()
    B, S, h, theta = 2, 150, 256, 5e5
    N = (nq + 2 * nkv) * d
    A, a32 = to_dev_bf16(torch, _normal((B * S, h), 91))
    W, w32 = to_dev_bf16(torch, _normal((N, h), 92, 0.05))
    C = torch.empty((B * S, N), dtype=torch.bfloat16, device="cuda")
    tab = torch.empty(S * d, device="cuda")
    mt.mt_op_gemm_rope(A, W, C, B * S, N, h, h, h, N, tab, S, d, theta, (nq + nkv) * d)
    ref = oracle.matmul("nt", a32, w32).reshape(B, S, nq + 2 * nkv, d)
    ref_rot = ref.copy()
    ref_rot[:, :, :nq + nkv] = oracle.rope(ref[:, :, :nq + nkv], theta)
    assert rel_l2(from_dev(C).reshape(B, S, -1, d), ref_rot) < 6e-3
    # the fp32 accumulator's error, rotated (pairs mixed) on the q and k
    # heads, then one bf16 rounding
    e = acc(h) * oracle.matmul("nt", np.abs(a32), np.abs(w32)).reshape(B, S, nq + 2 * nkv, d)
    e[:, :, :nq + nkv] = pair_sum(e[:, :, :nq + nkv]) + 4 * U32 * pair_sum(np.abs(ref[:, :, :nq + nkv]))
    check(from_dev(C).reshape(B, S, -1, d), ref_rot, U16 * np.abs(ref_rot) + (1 + U16) * e, "qkv+rope")


@pytest.mark.parametrize("d", [128, 64, 16])
def test_attention_backward_with_fused_inverse_rope(d):
    """dq, dk of the RoPE'd attention come out rotated back: compare with the
    oracle's attention backward followed by its inverse rotation."""
    torch, mt = need_gpu()
    B, S, nq, nkv, theta = 2, 150, 4, 2, 1e4
    q, k, v, do = (_normal((B, S, n, d), 95 + i) for i, n in enumerate((nq, nkv, nkv, nq)))
    Q, q32 = to_dev_bf16(torch, q)
    Kd, k32 = to_dev_bf16(torch, k)
    Vd, v32 = to_dev_bf16(torch, v)
    DO, do32 = to_dev_bf16(torch, do)
    O = torch.empty((B, S, nq, d), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((B, nq, S), device="cuda")
    mt.mt_op_attention_fwd(Q, Kd, Vd, O, LSE, B, S, nq, nkv, d, nq * d, nkv * d, nq * d)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Kd), torch.empty_like(Vd)
    ws = torch.empty(mt.mt_op_attention_bwd_workspace(B, S, nq), device="cuda")
    tab = torch.empty(S * d, device="cuda")
    mt.mt_op_attention_bwd_rope(Q, Kd, Vd, O, DO, LSE, dQ, dK, dV, ws, B, S, nq, nkv, d, nq * d, nkv * d, nq * d,
                                tab, theta)
    _, _, dq_ref, dk_ref, dv_ref = oracle.attention(q32, k32, v32, do32)
    _, dq_abs, dk_abs, dv_abs = attention_magnitudes(q32, k32, v32, do32)
    dq_rot, dk_rot = oracle.rope(dq_ref, theta, -1), oracle.rope(dk_ref, theta, -1)
    assert rel_l2(from_dev(dQ), dq_rot) < 2e-2
    assert rel_l2(from_dev(dK), dk_rot) < 2e-2
    assert rel_l2(from_dev(dV), dv_ref) < 2e-2
    check(from_dev(dQ), dq_rot, ATT_G(dq_rot, pair_sum(dq_abs)), "dq")
    check(from_dev(dK), dk_rot, ATT_G(dk_rot, pair_sum(dk_abs)), "dk")
    check(from_dev(dV), dv_ref, ATT_G(dv_ref, dv_abs), "dv")


def test_attention_full_8b_shape_sliced():
    """The step's attention launches at the 8B shape (B=2, S=4096, 32 query /
    8 KV heads x 128, theta 5e5): the forward, then the backward with the
    inverse rotation fused. Every (sequence, KV group) pair is an independent
    causal attention problem (4 query heads over one KV head), so two of them
    (the first and the last) are checked element by element against the
    oracle solving that problem whole; the other pairs' outputs are checked
    to be finite."""
    torch, mt = need_gpu()
    B, S, nq, nkv, d, theta = 2, 4096, 32, 8, 128, 5e5
    grp = nq // nkv
    q, k, v, do = (_normal((B, S, n, d), 130 + i) for i, n in enumerate((nq, nkv, nkv, nq)))
    Q, q32 = to_dev_bf16(torch, q)
    Kd, k32 = to_dev_bf16(torch, k)
    Vd, v32 = to_dev_bf16(torch, v)
    DO, do32 = to_dev_bf16(torch, do)
    O = torch.empty((B, S, nq, d), dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty((B, nq, S), device="cuda")
    mt.mt_op_attention_fwd(Q, Kd, Vd, O, LSE, B, S, nq, nkv, d, nq * d, nkv * d, nq * d)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Kd), torch.empty_like(Vd)
    ws = torch.empty(mt.mt_op_attention_bwd_workspace(B, S, nq), device="cuda")
    tab = torch.empty(S * d, device="cuda")
    mt.mt_op_attention_bwd_rope(Q, Kd, Vd, O, DO, LSE, dQ, dK, dV, ws, B, S, nq, nkv, d, nq * d, nkv * d, nq * d,
                                tab, theta)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    o, lse, dq, dk, dv = (from_dev(t) for t in (O, LSE, dQ, dK, dV))
    for b, g in ((0, 0), (B - 1, nkv - 1)):
        hs = slice(g * grp, (g + 1) * grp)
        qs, ks, vs, dos = q32[b:b + 1, :, hs], k32[b:b + 1, :, g:g + 1], v32[b:b + 1, :, g:g + 1], do32[b:b + 1, :, hs]
        o_ref, lse_ref, dq_ref, dk_ref, dv_ref = oracle.attention(qs, ks, vs, dos)
        o_abs, dq_abs, dk_abs, dv_abs = attention_magnitudes(qs, ks, vs, dos)
        dq_rot, dk_rot = oracle.rope(dq_ref, theta, -1), oracle.rope(dk_ref, theta, -1)
        assert rel_l2(o[b:b + 1, :, hs], o_ref) < 1.5e-2, (b, g)
        assert rel_l2(dq[b:b + 1, :, hs], dq_rot) < 2e-2, (b, g)
        assert rel_l2(dk[b:b + 1, :, g:g + 1], dk_rot) < 2e-2, (b, g)
        assert rel_l2(dv[b:b + 1, :, g:g + 1], dv_ref) < 2e-2, (b, g)
        check(o[b:b + 1, :, hs], o_ref, ATT_O(o_ref, o_abs, S), f"o {b},{g}")
        check(lse[b:b + 1, hs], lse_ref, 1e-3, f"lse {b},{g}")
        check(dq[b:b + 1, :, hs], dq_rot, ATT_G(dq_rot, pair_sum(dq_abs)), f"dq {b},{g}")
        check(dk[b:b + 1, :, g:g + 1], dk_rot, ATT_G(dk_rot, pair_sum(dk_abs)), f"dk {b},{g}")
        check(dv[b:b + 1, :, g:g + 1], dv_ref, ATT_G(dv_ref, dv_abs), f"dv {b},{g}")
    for t in (o, lse, dq, dk, dv):
        assert np.all(np.isfinite(t))


@pytest.mark.parametrize("M,F,K,u_off", [(300, 384, 256, 384), (130, 172, 64, 176), (2048, 1536, 512, 1536)])
def test_gated_gemm_fuses_swiglu(M, F, K, u_off):
    """g|u = x [Wg;Wu]^T with act = silu(g) u formed from the fp32 products."""
    torch, mt = need_gpu()
    X, x32 = to_dev_bf16(torch, _normal((M, K), 101))
    Wst = np.zeros((2 * u_off, K), np.float32)
    Wst[:F] = _normal((F, K), 102, 0.05)
    Wst[u_off:u_off + F] = _normal((F, K), 103, 0.05)
    W, w32 = to_dev_bf16(torch, Wst)
    GU = torch.zeros((M, 2 * u_off), dtype=torch.bfloat16, device="cuda")
    ACT = torch.zeros((M, u_off), dtype=torch.bfloat16, device="cuda")
    mt.mt_op_gemm_swiglu(X, W, GU, ACT, M, F, K, K, K, u_off)
    g = oracle.matmul("nt", x32, w32[:F])
    u = oracle.matmul("nt", x32, w32[u_off:u_off + F])
    a_ref, _, _ = oracle.swiglu(g, u)
    gu = from_dev(GU)
    assert rel_l2(gu[:, :F], g) < 6e-3
    assert rel_l2(gu[:, u_off:u_off + F], u) < 6e-3
    assert rel_l2(from_dev(ACT)[:, :F], a_ref) < 6e-3
    eg = acc(K) * oracle.matmul("nt", np.abs(x32), np.abs(w32[:F]))
    eu = acc(K) * oracle.matmul("nt", np.abs(x32), np.abs(w32[u_off:u_off + F]))
    check(gu[:, :F], g, U16 * np.abs(g) + (1 + U16) * eg, "g")
    check(gu[:, u_off:u_off + F], u, U16 * np.abs(u) + (1 + U16) * eu, "u")
    # act = silu(g) u from the fp32 accumulators: their errors carried
    # through silu' and silu, then one bf16 rounding
    _, silu_g, dsilu_mag = silu_parts(g)
    e_act = dsilu_mag * np.abs(u) * eg + np.abs(silu_g) * eu
    check(from_dev(ACT)[:, :F], a_ref, (U16 + 1e-5) * np.abs(a_ref) + (1 + U16) * e_act, "act")


@pytest.mark.parametrize("M,F,K,u_off", [(300, 384, 256, 384), (130, 172, 64, 176)])
def test_down_dgrad_fuses_swiglu_backward(M, F, K, u_off):
    """dact = dY Wd with (g, u) replaced in place by (dg, du) from fp32 dact."""
    torch, mt = need_gpu()
    dY, dy32 = to_dev_bf16(torch, _normal((M, K), 111))
    Wd_st = np.zeros((K, u_off), np.float32)
    Wd_st[:, :F] = _normal((K, F), 112, 0.05)
    Wd, wd32 = to_dev_bf16(torch, Wd_st)
    gu0 = np.zeros((M, 2 * u_off), np.float32)
    gu0[:, :F] = _normal((M, F), 113)
    gu0[:, u_off:u_off + F] = _normal((M, F), 114)
    GU, gu32 = to_dev_bf16(torch, gu0)
    mt.mt_op_gemm_swiglu_bwd(dY, Wd, GU, M, F, K, K, u_off, u_off)
    dact = oracle.matmul("nn", dy32, wd32[:, :F])
    g32, u32 = gu32[:, :F], gu32[:, u_off:u_off + F]
    _, dg_ref, du_ref = oracle.swiglu(g32, u32, dact)
    out = from_dev(GU)
    assert rel_l2(out[:, :F], dg_ref) < 6e-3
    assert rel_l2(out[:, u_off:u_off + F], du_ref) < 6e-3
    # d(act) from an fp32 accumulator, times u silu'(g) and silu(g), then one
    # bf16 rounding
    e_da = acc(K) * oracle.matmul("nn", np.abs(dy32), np.abs(wd32[:, :F]))
    _, silu_g, dsilu_mag = silu_parts(g32)
    check(out[:, :F], dg_ref,
          U16 * np.abs(dg_ref) + (1 + U16) * (dsilu_mag * np.abs(u32) * (e_da + 1e-5 * np.abs(dact))), "dg")
    check(out[:, u_off:u_off + F], du_ref,
          U16 * np.abs(du_ref) + (1 + U16) * np.abs(silu_g) * (e_da + 1e-5 * np.abs(dact)), "du")


@pytest.mark.parametrize("V", [1000, 1003])
def test_lmhead_cross_entropy(V):
    """Vocab a multiple of 4 (16-byte logit loads) and not (scalar tails)."""
    torch, mt = need_gpu()
    T, h = 96, 128
    X, x32 = to_dev_bf16(torch, _normal((T, h), 61))
    W, w32 = to_dev_bf16(torch, _normal((V, h), 62, 0.1))
    lab = np.random.default_rng(1).integers(0, V, T).astype(np.int32)
    LAB = torch.from_numpy(lab).cuda()
    dX = torch.empty((T, h), device="cuda")
    dW = torch.empty((V, h), device="cuda")
    loss = torch.zeros(1, device="cuda")
    ws = torch.empty(mt.mt_op_lmhead_ce_workspace(T, V, h), dtype=torch.uint8, device="cuda")
    mt.mt_op_lmhead_ce(X, W, LAB, 1.0 / T, dX, dW, loss, ws, T, V, h)
    z = oracle.matmul("nt", x32, w32)
    l_ref, dz = oracle.cross_entropy(z, lab)
    assert abs(float(loss.item()) - l_ref) < 1e-4 * abs(l_ref)
    dzb = bf16_round(dz)
    dx_ref, dw_ref = oracle.matmul("nn", dzb, w32), oracle.matmul("tn", dzb, x32)
    assert rel_l2(from_dev(dX), dx_ref) < 6e-3
    assert rel_l2(from_dev(dW), dw_ref) < 6e-3
    # the kernel rounds its own fp32 dlogits to bf16: each may land one bf16
    # step (2 U16) away from the rounded oracle value; then fp32 sums over the
    # vocab (dX) or the tokens (dW)
    dza = np.abs(dz)
    check(from_dev(dX), dx_ref, (2 * U16 + acc(V)) * oracle.matmul("nn", dza, np.abs(w32)), "dX")
    check(from_dev(dW), dw_ref, (2 * U16 + acc(T)) * oracle.matmul("tn", dza, np.abs(x32)), "dW")
