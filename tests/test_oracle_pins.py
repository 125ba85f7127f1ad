"""Pins of the CPU oracle against what the mathematics fixes (no GPU).

Each test checks the oracle against something other than itself: finite
differences, closed forms, invariants, special cases that reduce to a
textbook formula evaluated independently here, or brute force on tiny inputs.
Together they are chosen so that a plausible slip in the oracle (a dropped
residual, a wrong softmax scale, an off-by-one causal mask, interleaved
instead of half-split RoPE pairs, a wrong GQA mapping, swapped gate/up, a
missing RMSNorm epsilon, a wrong loss scale) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.common import TINY, TINY_GQA, make_params, make_tokens, params_f64, rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Layout
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [False, True])
def test_layout_alignment_order_and_no_overlap(bf16):
    cfg = TINY
    prev_end = 0
    prev_unit = -1
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, bf16)
        assert off % 256 == 0
        if unit != prev_unit:
            assert off % 4096 == 0, name
            prev_unit = unit
        assert off >= prev_end
        assert nb == int(np.prod(shape)) * (2 if bf16 else 4)
        prev_end = off + nb
    assert oracle.packed_bytes(cfg, bf16) >= prev_end
    assert oracle.packed_bytes(cfg, bf16) % 4096 == 0


# --------------------------------------------------------------------------
# Whole-model gradient by central finite differences (fp64)
# --------------------------------------------------------------------------
def _fd_check(cfg, seed_w, seed_t, n_per_tensor=5, eps=1e-4):
    B, S = 2, 32
    packed = make_params(cfg, seed_w)
    p64 = params_f64(cfg, packed)
    tok, lab = make_tokens(cfg, B, S, seed_t)
    loss, g = oracle.forward_backward_f64(cfg, p64, tok, lab)
    rng = np.random.default_rng(seed_w)
    worst = 0.0
    used = np.unique(tok)
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, False)
        base, n = off // 4, nb // 4
        if name == "embed":
            rows = rng.choice(used, n_per_tensor)
            idx = rows * cfg.hidden + rng.integers(0, cfg.hidden, n_per_tensor)
        else:
            idx = rng.integers(0, n, n_per_tensor)
        for i in idx:
            p = p64.copy()
            p[base + i] += eps
            lp, _ = oracle.forward_backward_f64(cfg, p, tok, lab)
            p[base + i] -= 2 * eps
            lm, _ = oracle.forward_backward_f64(cfg, p, tok, lab)
            fd = (lp - lm) / (2 * eps)
            an = g[base + i]
            err = abs(fd - an) / max(abs(fd), abs(an), 1e-6)
            worst = max(worst, err)
            assert err < 1e-5, (name, int(i), fd, an)
    return worst


def test_fd_tiny():
    _fd_check(TINY, 1, 2)


def test_fd_tiny_gqa():
    _fd_check(TINY_GQA, 3, 4)


def test_f32_matches_f64():
    cfg = TINY
    packed = make_params(cfg, 1)
    tok, lab = make_tokens(cfg, 2, 32, 2)
    l32, g32 = oracle.forward_backward(cfg, packed, tok, lab)
    l64, g64 = oracle.forward_backward_f64(cfg, params_f64(cfg, packed), tok, lab)
    assert abs(l32 - l64) / l64 < 1e-5
    assert rel_l2(g32, g64) < 1e-4


def test_bf16_host_params_widen_exactly():
    """bf16 host params give the same result as their exact fp32 widening."""
    cfg = TINY
    p16 = make_params(cfg, 5, bf16=True)
    p32 = np.zeros(oracle.packed_bytes(cfg, False), dtype=np.uint8)
    v16, v32 = oracle.unpack(cfg, p16, True), oracle.unpack(cfg, p32, False)
    for k in v16:
        v32[k][...] = (v16[k].astype(np.uint32) << 16).view(np.float32)
    tok, lab = make_tokens(cfg, 2, 32, 6)
    la, ga = oracle.forward_backward(cfg, p16, tok, lab, bf16=True)
    lb, gb = oracle.forward_backward(cfg, p32, tok, lab, bf16=False)
    assert la == lb
    assert np.array_equal(ga, gb)


# --------------------------------------------------------------------------
# Loss anchoring
# --------------------------------------------------------------------------
def test_zero_head_gives_ln_vocab():
    cfg = TINY
    g = _golden("closed_forms.json")
    packed = make_params(cfg, 7)
    oracle.unpack(cfg, packed)["w_out"][...] = 0.0
    tok, lab = make_tokens(cfg, 2, 32, 8)
    loss, grads = oracle.forward_backward(cfg, packed, tok, lab)
    assert abs(loss - g["ln_256"]["value"]) < 1e-3
    assert abs(math.log(cfg.vocab) - g["ln_256"]["value"]) < 1e-12
    # The CE gradient rows sum to zero over the vocabulary, so the columns of
    # dW_out sum to zero.
    dW = oracle.unpack(cfg, grads)["w_out"]
    assert np.abs(dW.sum(axis=0)).max() < 1e-6


def test_cross_entropy_hand_example():
    g = _golden("closed_forms.json")["ce_example"]
    z = np.array(g["logits"], dtype=np.float32)
    lab = np.array(g["labels"], dtype=np.int32)
    loss, dz = oracle.cross_entropy(z, lab, scale=1.0)
    assert abs(loss - g["loss_sum"]) < 1e-5
    np.testing.assert_allclose(dz, np.array(g["dz_sum"]), atol=1e-6)


def test_microbatch_gradients_sum_to_whole_batch():
    """Sum over microbatches with scale 1/T_total == whole batch (the RoundPipe
    user guide, 输入分割与 microbatch 执行: per-microbatch losses and gradients add up
    to those of the summed batch loss)."""
    cfg = TINY_GQA
    packed = make_params(cfg, 9)
    tok, lab = make_tokens(cfg, 4, 16, 10)
    T = tok.size
    lw, gw = oracle.forward_backward(cfg, packed, tok, lab, scale=1.0 / T)
    ls, gs = 0.0, np.zeros_like(gw)
    for i in range(4):
        l, gi = oracle.forward_backward(cfg, packed, tok[i:i + 1], lab[i:i + 1], scale=1.0 / T)
        ls += l
        gs += gi
    assert abs(ls - lw) < 1e-5
    assert rel_l2(gs, gw) < 1e-5


# --------------------------------------------------------------------------
# Closed forms and special cases of single operations
# --------------------------------------------------------------------------
def test_attention_single_position_returns_v():
    rng = np.random.default_rng(0)
    q = rng.normal(size=(3, 1, 4, 8)).astype(np.float32)
    k = rng.normal(size=(3, 1, 2, 8)).astype(np.float32)
    v = rng.normal(size=(3, 1, 2, 8)).astype(np.float32)
    o, lse, *_ = oracle.attention(q, k, v)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=1e-6)
    np.testing.assert_allclose(o[:, :, 1], v[:, :, 0], rtol=1e-6)  # heads 0,1 -> kv 0
    np.testing.assert_allclose(o[:, :, 2], v[:, :, 1], rtol=1e-6)  # heads 2,3 -> kv 1
    np.testing.assert_allclose(o[:, :, 3], v[:, :, 1], rtol=1e-6)


def test_attention_zero_query_is_causal_running_mean():
    rng = np.random.default_rng(1)
    B, S, d = 2, 7, 4
    q = np.zeros((B, S, 1, d), np.float32)
    k = rng.normal(size=(B, S, 1, d)).astype(np.float32)
    v = rng.normal(size=(B, S, 1, d)).astype(np.float32)
    o, lse, *_ = oracle.attention(q, k, v)
    for t in range(S):
        np.testing.assert_allclose(o[:, t, 0], v[:, :t + 1, 0].mean(axis=1), rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(lse[:, 0, t], np.log(t + 1), rtol=1e-6)


def test_attention_two_keys_softmax_scale():
    """Two positions, d=4: o_1 = softmax([q.k0, q.k1]/2) . [v0, v1] (scale 1/sqrt(4))."""
    q = np.zeros((1, 2, 1, 4), np.float32)
    k = np.zeros((1, 2, 1, 4), np.float32)
    v = np.zeros((1, 2, 1, 4), np.float32)
    q[0, 1, 0, 0] = 2.0
    k[0, 0, 0, 0] = 1.0
    k[0, 1, 0, 0] = -1.0
    v[0, 0, 0, :] = [1, 0, 0, 0]
    v[0, 1, 0, :] = [0, 1, 0, 0]
    o, *_ = oracle.attention(q, k, v)
    # scores 1 and -1 -> weights e/(e+1/e), (1/e)/(e+1/e)
    w0 = math.e / (math.e + 1 / math.e)
    np.testing.assert_allclose(o[0, 1, 0], [w0, 1 - w0, 0, 0], rtol=1e-6)


def test_attention_backward_fd():
    rng = np.random.default_rng(2)
    B, S, nq, nkv, d = 1, 5, 4, 2, 4
    q, k, v = (rng.normal(size=(B, S, n, d)) for n in (nq, nkv, nkv))
    w = rng.normal(size=(B, S, nq, d))
    o, _, dq, dk, dv = oracle.attention(q, k, v, w)
    eps = 1e-3

    def f(qq, kk, vv):
        return float((oracle.attention(qq, kk, vv)[0].astype(np.float64) * w).sum())

    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        for _ in range(4):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            args1 = [q, k, v]
            args2 = [q, k, v]
            args1[which], args2[which] = a1, a2
            fd = (f(*args1) - f(*args2)) / (2 * eps)
            assert abs(fd - grad[idx]) < 2e-3 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_rope_position_zero_is_identity_and_norm_preserving():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(2, 9, 3, 16)).astype(np.float32)
    y = oracle.rope(x, 1e4)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    # per-pair norms (i, i + d/2) are preserved
    n_x = x[..., :8] ** 2 + x[..., 8:] ** 2
    n_y = y[..., :8] ** 2 + y[..., 8:] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-5)
    # backward is the inverse rotation
    np.testing.assert_allclose(oracle.rope(y, 1e4, -1), x, rtol=1e-5, atol=1e-6)


def test_rope_half_split_pairs_and_frequencies():
    """Unit vector e_i at position p goes to cos(p f_i) e_i + sin(p f_i) e_{i+d/2},
    f_i = theta^(-2i/d)."""
    d, theta, p = 8, 100.0, 3
    for i in range(d // 2):
        x = np.zeros((1, p + 1, 1, d), np.float32)
        x[0, p, 0, i] = 1.0
        y = oracle.rope(x, theta)[0, p, 0]
        ang = p * theta ** (-2.0 * i / d)
        expect = np.zeros(d)
        expect[i] = math.cos(ang)
        expect[i + d // 2] = math.sin(ang)
        np.testing.assert_allclose(y, expect, atol=1e-6)


def test_rmsnorm_unit_gain_rms_and_eps():
    rng = np.random.default_rng(4)
    x = (rng.normal(size=(5, 64)) * 0.01).astype(np.float32)
    eps = 1e-5
    y, r = oracle.rmsnorm_fwd(x, np.ones(64, np.float32), eps)
    ms = (x.astype(np.float64) ** 2).mean(axis=1)
    rms_y = np.sqrt((y.astype(np.float64) ** 2).mean(axis=1))
    np.testing.assert_allclose(rms_y, np.sqrt(ms / (ms + eps)), rtol=1e-5)
    np.testing.assert_allclose(r, 1 / np.sqrt(ms + eps), rtol=1e-5)


def test_rmsnorm_backward_fd():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(3, 16))
    w = rng.normal(size=16)
    gy = rng.normal(size=(3, 16))
    dx, dw = oracle.rmsnorm_bwd(x, w, gy, 1e-5)
    eps = 1e-3

    def f(xx, ww):
        return float((oracle.rmsnorm_fwd(xx, ww, 1e-5)[0].astype(np.float64) * gy).sum())

    for _ in range(5):
        i, j = rng.integers(0, 3), rng.integers(0, 16)
        a, b = x.copy(), x.copy()
        a[i, j] += eps
        b[i, j] -= eps
        assert abs((f(a, w) - f(b, w)) / (2 * eps) - dx[i, j]) < 1e-3
        wa, wb = w.copy(), w.copy()
        wa[j] += eps
        wb[j] -= eps
        assert abs((f(x, wa) - f(x, wb)) / (2 * eps) - dw[j]) < 1e-3


def test_swiglu_values_and_derivative_at_zero():
    g = _golden("closed_forms.json")["swiglu"]
    a, dg, du = oracle.swiglu(np.array([0.0, 1.0, 2.0], np.float32), np.array([5.0, 2.0, 1.0], np.float32),
                              np.ones(3, np.float32))
    np.testing.assert_allclose(a, g["a"], rtol=1e-6)
    # d/dg [silu(g) u] at g=0 is silu'(0) u = 0.5 u; d/du is silu(g)
    assert abs(dg[0] - 0.5 * 5.0) < 1e-6
    np.testing.assert_allclose(du, g["silu"], rtol=1e-6)


def test_matmul_modes_against_numpy():
    rng = np.random.default_rng(6)
    A = rng.normal(size=(7, 5)).astype(np.float32)
    Bnt = rng.normal(size=(6, 5)).astype(np.float32)
    Bnn = rng.normal(size=(5, 6)).astype(np.float32)
    Atn = rng.normal(size=(5, 7)).astype(np.float32)
    np.testing.assert_allclose(oracle.matmul("nt", A, Bnt), A.astype(np.float64) @ Bnt.T, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(oracle.matmul("nn", A, Bnn), A.astype(np.float64) @ Bnn, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(oracle.matmul("tn", Atn, Bnn), Atn.T.astype(np.float64) @ Bnn, rtol=1e-5,
                               atol=1e-6)
    s = oracle.matmul_sampled("nt", A, Bnt, [0, 6, 3], [5, 0, 2])
    np.testing.assert_allclose(s, [(A[0] @ Bnt[5]), A[6] @ Bnt[0], A[3] @ Bnt[2]], rtol=1e-6)


# --------------------------------------------------------------------------
# Model-level special cases
# --------------------------------------------------------------------------
def _np_rmsnorm(x, w, eps):
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * w


def _np_ce(z, lab):
    m = z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
    return float((lse - z[np.arange(len(lab)), lab]).mean())


def test_residual_path_with_zero_output_projections():
    """With Wo = Wd = 0 every layer is the identity on the residual stream, so the
    loss is CE(RMSNorm(E[tok]; w_f) W_out^T) and every layer's weight gradient
    except the two output projections' is zero."""
    cfg = TINY
    packed = make_params(cfg, 11)
    V = oracle.unpack(cfg, packed)
    for l in range(cfg.n_layers):
        V[f"layer{l}.wo"][...] = 0
        V[f"layer{l}.wd"][...] = 0
    tok, lab = make_tokens(cfg, 2, 32, 12)
    loss, g = oracle.forward_backward(cfg, packed, tok, lab)
    x = V["embed"][tok.ravel()].astype(np.float64)
    z = _np_rmsnorm(x, V["w_final_norm"].astype(np.float64), cfg.norm_eps) @ V["w_out"].T.astype(np.float64)
    assert abs(loss - _np_ce(z, lab.ravel())) < 1e-5
    G = oracle.unpack(cfg, g)
    for l in range(cfg.n_layers):
        for nm in ("wq", "wk", "wv", "wg", "wu", "w_attn_norm", "w_ffn_norm"):
            assert np.abs(G[f"layer{l}.{nm}"]).max() == 0.0, nm
        assert np.abs(G[f"layer{l}.wo"]).max() > 0


def test_one_layer_single_token_closed_form():
    """S = 1: attention returns v, so one layer is
    h1 = h0 + (RMSNorm(h0) Wv^T) Wo^T;  h2 = h1 + (silu(m Wg^T) * (m Wu^T)) Wd^T, m = RMSNorm(h1)."""
    cfg = oracle.Config(n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=48, vocab=50)
    packed = make_params(cfg, 13, std=0.2)
    V = {k: v.astype(np.float64) for k, v in oracle.unpack(cfg, packed).items()}
    tok, lab = make_tokens(cfg, 3, 1, 14)
    loss, _ = oracle.forward_backward(cfg, packed, tok, lab)
    e = cfg.norm_eps
    h0 = V["embed"][tok.ravel()]
    a = _np_rmsnorm(h0, V["layer0.w_attn_norm"], e)
    v = a @ V["layer0.wv"].T                      # [T, nkv*d]
    o = np.concatenate([v[:, :16], v[:, :16], v[:, 16:], v[:, 16:]], axis=1)  # q heads 0,1->kv0; 2,3->kv1
    h1 = h0 + o @ V["layer0.wo"].T
    m = _np_rmsnorm(h1, V["layer0.w_ffn_norm"], e)
    gg, uu = m @ V["layer0.wg"].T, m @ V["layer0.wu"].T
    h2 = h1 + (gg / (1 + np.exp(-gg)) * uu) @ V["layer0.wd"].T
    z = _np_rmsnorm(h2, V["w_final_norm"], e) @ V["w_out"].T
    assert abs(loss - _np_ce(z, lab.ravel())) < 1e-5


def test_gqa_equals_mha_with_repeated_kv_heads():
    gq = TINY_GQA
    mh = TINY
    pg = make_params(gq, 15)
    pm = make_params(mh, 16)
    G, M = oracle.unpack(gq, pg), oracle.unpack(mh, pm)
    grp = gq.n_heads // gq.n_kv_heads
    d = gq.head_dim
    for name in G:
        if name.endswith(".wk") or name.endswith(".wv"):
            src = G[name].reshape(gq.n_kv_heads, d, gq.hidden)
            M[name][...] = np.repeat(src, grp, axis=0).reshape(M[name].shape)  # q head j -> kv head j // grp
        else:
            M[name][...] = G[name]
    tok, lab = make_tokens(gq, 2, 32, 17)
    lg, gg = oracle.forward_backward(gq, pg, tok, lab)
    lm, gm = oracle.forward_backward(mh, pm, tok, lab)
    assert abs(lg - lm) < 1e-6
    Gg, Gm = oracle.unpack(gq, gg), oracle.unpack(mh, gm)
    for name in Gg:
        if name.endswith(".wk") or name.endswith(".wv"):
            summed = Gm[name].reshape(gq.n_kv_heads, grp, d, gq.hidden).sum(axis=1).reshape(Gg[name].shape)
            np.testing.assert_allclose(Gg[name], summed, rtol=1e-4, atol=1e-7)
        else:
            np.testing.assert_allclose(Gg[name], Gm[name], rtol=1e-4, atol=1e-7)


def test_unused_embedding_rows_have_exactly_zero_gradient():
    cfg = TINY
    packed = make_params(cfg, 18)
    tok, lab = make_tokens(cfg, 2, 32, 19)
    _, g = oracle.forward_backward(cfg, packed, tok, lab)
    dE = oracle.unpack(cfg, g)["embed"]
    used = np.zeros(cfg.vocab, bool)
    used[tok.ravel()] = True
    assert np.all(dE[~used] == 0.0)
    assert np.all(np.abs(dE[used]).max(axis=1) > 0)


def test_causality_later_token_does_not_change_earlier_losses():
    """The CE term at position p depends only on tokens 0..p: changing the
    tokens from position t on leaves the terms before t unchanged (and equal
    to those of the prefix alone), and changes later ones."""
    cfg = TINY_GQA
    packed = make_params(cfg, 20)
    tok, lab = make_tokens(cfg, 2, 32, 21)
    t = 20
    tok2 = tok.copy()
    tok2[:, t:] = (tok2[:, t:] + 17) % cfg.vocab
    _, _, l1 = oracle.forward_backward(cfg, packed, tok, lab, token_losses=True)
    _, _, l2 = oracle.forward_backward(cfg, packed, tok2, lab, token_losses=True)
    _, _, lp = oracle.forward_backward(cfg, packed, tok[:, :t], lab[:, :t], token_losses=True)
    np.testing.assert_array_equal(l1[:, :t], l2[:, :t])
    np.testing.assert_allclose(l1[:, :t], lp, rtol=1e-5, atol=1e-6)
    assert np.all(np.abs(l1[:, t:] - l2[:, t:]).max(axis=1) > 1e-4)
