"""Pins of the oracle's mixture-of-experts FFN (no GPU).

The MoE layer (router softmax over E experts, top-k selection with ties to
the lower index, renormalised weights, SwiGLU experts) is pinned against:
  - central finite differences of the whole model in fp64, with the
    selection held at the one the oracle made (the loss is smooth there);
  - a closed form: one-hot inputs and experts built so that each expert
    outputs a known basis vector, which exposes the selection and the
    weights directly;
  - one expert with k = 1 equals the dense decoder (gate rows first in the
    packed expert matrix), and its router gradient is exactly zero;
  - E identical experts equal the dense decoder for any router (the weights
    sum to one), the experts' gradients sum to the dense ones and the
    router gradient vanishes;
  - relabelling the experts permutes every output consistently.
A dropped renormalisation, swapped gate/up rows, a wrong tie rule, a slot
reading another expert's weights or a wrong router backward each fail one.
"""
import math

import numpy as np
import pytest

import oracle
from tests.common import make_params, make_tokens, params_f64, rel_l2

DENSE = oracle.Config(n_layers=2, hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=24, vocab=64,
                      rope_theta=1e4, norm_eps=1e-5)


def moe_cfg(base, E, k, Fe):
    d = dict(base.__dict__)
    d.update(ffn_dim=0, n_experts=E, top_k=k, expert_ffn=Fe)
    return oracle.Config(**d)


TINY_MOE = moe_cfg(DENSE, 8, 2, 24)


def _views64(cfg, p64):
    """Named float64 views into a packed fp64 parameter vector."""
    out = {}
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, False)
        out[name] = p64[off // 4:(off + nb) // 4].reshape(shape)
    return out


def test_moe_layout():
    cfg = moe_cfg(DENSE, 8, 2, 24)
    names = [n for _, _, n, _, _ in oracle.tensor_list(cfg)]
    assert "layer0.w_router" in names and "layer1.w_experts_down" in names and "layer0.wg" not in names
    prev_end, prev_unit = 0, -1
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, False)
        assert off % 256 == 0 and off >= prev_end
        if unit != prev_unit:
            assert off % 4096 == 0
            prev_unit = unit
        assert nb == 4 * int(np.prod(shape))
        prev_end = off + nb
    h, E, Fe = cfg.hidden, 8, 24
    assert oracle.tensor_offset(cfg, 1, 6)[1] == 4 * E * h
    assert oracle.tensor_offset(cfg, 1, 7)[1] == 4 * E * 2 * Fe * h
    assert oracle.tensor_offset(cfg, 1, 8)[1] == 4 * E * h * Fe


def test_moe_whole_model_finite_differences():
    cfg = TINY_MOE
    B, S = 2, 16
    packed = make_params(cfg, 71)
    p64 = params_f64(cfg, packed)
    tok, lab = make_tokens(cfg, B, S, 72)
    loss, g, route = oracle.forward_backward_f64(cfg, p64, tok, lab, want_route=True)
    # forcing the selection the oracle made changes nothing
    loss2, g2 = oracle.forward_backward_f64(cfg, p64, tok, lab, route_in=route)
    assert loss2 == loss and np.array_equal(g2, g)
    assert np.all(np.sort(route, axis=2)[..., 1:] != np.sort(route, axis=2)[..., :-1])
    rng = np.random.default_rng(73)
    eps = 1e-5
    used = np.unique(tok)
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, False)
        base, n = off // 4, nb // 4
        if name == "embed":
            idx = rng.choice(used, 4) * cfg.hidden + rng.integers(0, cfg.hidden, 4)
        else:
            idx = rng.integers(0, n, 6)
        for i in idx:
            p = p64.copy()
            p[base + i] += eps
            lp, _ = oracle.forward_backward_f64(cfg, p, tok, lab, route_in=route)
            p[base + i] -= 2 * eps
            lm, _ = oracle.forward_backward_f64(cfg, p, tok, lab, route_in=route)
            fd = (lp - lm) / (2 * eps)
            an = g[base + i]
            assert abs(fd - an) <= 1e-5 * max(abs(fd), abs(an)) + 1e-10, (name, int(i), fd, an)


def test_moe_selection_and_weights_closed_form():
    """m_t = e_t (one-hot), so the router logits of token t are column t of
    Wr, chosen here (ties included). Every expert has Fe = 1 with gate 30 and
    up 1/30 on every input (silu(30)/30 = 1 - 9.4e-14) and down = e_e, so
    expert e outputs the basis vector e_e and out_t[e] is the weight of e."""
    T, h, E, k = 5, 8, 6, 3
    logits = np.array([[0.5, -1.0, 2.0, 0.1, 1.5, -0.3],   # distinct: 2, 4, 0
                       [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],     # all equal: 0, 1, 2
                       [1.0, 3.0, 3.0, 0.0, 3.0, 2.0],     # three-way tie on top: 1, 2, 4
                       [-1.0, 5.0, 5.0, 5.0, 5.0, -2.0],   # four tied, take the lower three: 1, 2, 3
                       [0.0, 0.0, 0.0, 0.0, 0.0, 7.0]])    # one winner, then the tie: 5, 0, 1
    expect = np.array([[2, 4, 0], [0, 1, 2], [1, 2, 4], [1, 2, 3], [5, 0, 1]])
    m = np.zeros((T, h))
    m[np.arange(T), np.arange(T)] = 1.0
    wr = np.zeros((E, h))
    wr[:, :T] = logits.T
    wgu = np.zeros((E, 2, h))
    wgu[:, 0, :] = 30.0
    wgu[:, 1, :] = 1.0 / 30.0
    wd = np.zeros((E, h, 1))
    wd[np.arange(E), np.arange(E), 0] = 1.0
    # float32 inputs are exact here except 1/30; the oracle runs in double
    out, route, *_ = oracle.moe_ffn(m, wr, wgu, wd, k)
    assert np.array_equal(route, expect)
    silu30 = 30.0 / (1.0 + math.exp(-30.0))
    for t in range(T):
        sel = expect[t]
        w = np.exp(logits[t, sel] - logits[t, sel].max())
        w /= w.sum()
        want = np.zeros(h)
        want[sel] = w * silu30 * float(np.float32(1.0 / 30.0))
        assert np.max(np.abs(out[t] - want)) < 1e-6, (t, out[t], want)


def _dense_to_moe(cfg_dense, cfg_moe, dense64, rng, copies):
    """fp64 MoE parameters whose experts all equal the dense FFN."""
    moe64 = np.zeros(oracle.packed_bytes(cfg_moe, False) // 4)
    D, M = _views64(cfg_dense, dense64), _views64(cfg_moe, moe64)
    for name, v in M.items():
        if name in D:
            v[...] = D[name]
    for l in range(cfg_dense.n_layers):
        p = f"layer{l}."
        M[p + "w_router"][...] = rng.normal(0.0, 0.5, M[p + "w_router"].shape)
        for e in range(copies):
            M[p + "w_experts_gu"][e] = np.concatenate([D[p + "wg"], D[p + "wu"]], axis=0)
            M[p + "w_experts_down"][e] = D[p + "wd"]
    return moe64


def test_single_expert_is_the_dense_layer():
    cfg_m = moe_cfg(DENSE, 1, 1, DENSE.ffn_dim)
    dense64 = params_f64(DENSE, make_params(DENSE, 81))
    moe64 = _dense_to_moe(DENSE, cfg_m, dense64, np.random.default_rng(82), 1)
    tok, lab = make_tokens(DENSE, 2, 16, 83)
    ld, gd = oracle.forward_backward_f64(DENSE, dense64, tok, lab)
    lm, gm = oracle.forward_backward_f64(cfg_m, moe64, tok, lab)
    assert abs(lm - ld) <= 1e-12 * abs(ld)
    GD, GM = _views64(DENSE, gd), _views64(cfg_m, gm)
    for name, g in GM.items():
        if name in GD:
            assert rel_l2(g, GD[name]) < 1e-10, name
    for l in range(DENSE.n_layers):
        p = f"layer{l}."
        assert not np.any(GM[p + "w_router"])
        assert rel_l2(GM[p + "w_experts_gu"][0], np.concatenate([GD[p + "wg"], GD[p + "wu"]])) < 1e-10
        assert rel_l2(GM[p + "w_experts_down"][0], GD[p + "wd"]) < 1e-10


def test_identical_experts_are_the_dense_layer():
    E = 4
    cfg_m = moe_cfg(DENSE, E, 2, DENSE.ffn_dim)
    dense64 = params_f64(DENSE, make_params(DENSE, 91))
    moe64 = _dense_to_moe(DENSE, cfg_m, dense64, np.random.default_rng(92), E)
    tok, lab = make_tokens(DENSE, 2, 16, 93)
    ld, gd = oracle.forward_backward_f64(DENSE, dense64, tok, lab)
    lm, gm = oracle.forward_backward_f64(cfg_m, moe64, tok, lab)
    assert abs(lm - ld) <= 1e-11 * abs(ld)
    GD, GM = _views64(DENSE, gd), _views64(cfg_m, gm)
    for name, g in GM.items():
        if name in GD:
            assert rel_l2(g, GD[name]) < 1e-9, name
    for l in range(DENSE.n_layers):
        p = f"layer{l}."
        gu_sum = GM[p + "w_experts_gu"].sum(axis=0)
        assert rel_l2(gu_sum, np.concatenate([GD[p + "wg"], GD[p + "wu"]])) < 1e-9
        assert rel_l2(GM[p + "w_experts_down"].sum(axis=0), GD[p + "wd"]) < 1e-9
        assert np.max(np.abs(GM[p + "w_router"])) < 1e-12 * np.max(np.abs(GD[p + "wd"]))


def test_relabelling_experts_permutes_everything():
    rng = np.random.default_rng(101)
    T, h, E, k, Fe = 40, 16, 6, 2, 12
    m = rng.normal(size=(T, h))
    wr = rng.normal(0, 0.5, (E, h))
    wgu = rng.normal(0, 0.3, (E, 2 * Fe, h))
    wd = rng.normal(0, 0.3, (E, h, Fe))
    dout = rng.normal(size=(T, h))
    out, route, dm, dwr, dwgu, dwd = oracle.moe_ffn(m, wr, wgu, wd, k, dout)
    perm = rng.permutation(E)  # new expert i is old expert perm[i]
    inv = np.argsort(perm)
    out2, route2, dm2, dwr2, dwgu2, dwd2 = oracle.moe_ffn(m, wr[perm], wgu[perm], wd[perm], k, dout)
    assert np.array_equal(perm[route2], route)
    for a, b in ((out2, out), (dm2, dm), (dwr2, dwr[perm]), (dwgu2, dwgu[perm]), (dwd2, dwd[perm])):
        assert rel_l2(a, b) < 1e-6
    assert inv.shape == (E,)


def test_routing_arguments_validated():
    cfg = TINY_MOE
    packed = make_params(cfg, 5)
    tok, lab = make_tokens(cfg, 1, 4, 6)
    bad = np.zeros((cfg.n_layers, 4, cfg.top_k), np.int32)  # expert 0 twice
    with pytest.raises(ValueError):
        oracle.forward_backward(cfg, packed, tok, lab, route_in=bad)
    bad[..., 1] = cfg.n_experts  # out of range
    with pytest.raises(ValueError):
        oracle.forward_backward(cfg, packed, tok, lab, route_in=bad)
    with pytest.raises(ValueError):
        oracle.forward_backward(DENSE, make_params(DENSE, 5), tok, lab, want_route=True)


def test_exported_router_logits_decide_the_selection():
    """The router logits the oracle exports are the ones its selection is
    made from: every layer's chosen experts are the k largest exported logits
    (ties to the lower index). A layer's logits depend on the routing of the
    layers below it only: forcing another routing in the first layer leaves
    its logits unchanged and changes the second layer's. A dense model has
    no logits to export."""
    cfg = TINY_MOE
    packed = make_params(cfg, 61)
    tok, lab = make_tokens(cfg, 2, 16, 62)
    loss, _, route, logits = oracle.forward_backward(cfg, packed, tok, lab, want_route=True, want_logits=True)
    L, T, k = route.shape
    assert logits.shape == (L, T, cfg.n_experts)
    for l in range(L):
        order = np.argsort(-logits[l].astype(np.float64), axis=1, kind="stable")[:, :k]
        assert np.array_equal(np.sort(order, axis=1), np.sort(route[l], axis=1)), l
    forced = route.copy()
    forced[0] = (route[0] + 1) % cfg.n_experts
    _, _, logits2 = oracle.forward_backward(cfg, packed, tok, lab, route_in=forced, want_logits=True)
    assert np.array_equal(logits2[0], logits[0])
    assert not np.array_equal(logits2[1], logits[1])
    with pytest.raises(ValueError):
        oracle.forward_backward(DENSE, make_params(DENSE, 63), tok, lab, want_logits=True)
