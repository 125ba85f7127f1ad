"""The mixture-of-experts layer on the GPU against the oracle.

The router's top-k choice is decided from bf16-operand, fp32-accumulated
logits on the GPU and from fp32 arithmetic in the oracle, so near-ties can
go different ways. The test therefore (1) runs the oracle with the GPU's
choices forced and compares loss and every gradient at the stated bar (loss
within 1e-2 relative, rel-L2 <= 2e-2 and cosine >= 0.999 per tensor), and
(2) checks every (layer, token) choice against the router logits the oracle
computes on that same path: each chosen expert's logit is at least the
largest unchosen logit minus ROUTER_DELTA's bound, and the k choices are
distinct.
"""
import math

import numpy as np
import pytest

import oracle
from tests.common import TINY_MOE, bf16_bits_to_f32, make_params, make_tokens, with_layers
from tests.gpu_util import need_gpu
from tests.test_gpu_e2e import compare

pytestmark = pytest.mark.gpu


def moe_session(mt, cfg, B, S, max_K):
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps, cfg.n_experts, cfg.top_k, cfg.expert_ffn)
    return mt.Session(shape, B, S, max_K, mt.MT_BF16)


def run_moe(cfg, B, S, K, seed_w, seed_t):
    torch, mt = need_gpu()
    tok, lab = make_tokens(cfg, B, S, seed_t)
    packed = make_params(cfg, seed_w, bf16=True)
    with moe_session(mt, cfg, B, S, K) as s:
        s.params[:] = packed
        loss = s.step(tok, lab, K)
        grads = s.grads.copy()
        route = s.routing(B * S)
    assert mt.mt_op_device_error() == 0
    return tok, lab, packed, loss, grads, route


# Relative error allowed in the GPU's FFN input m (the router's input): one
# bf16 rounding (2^-9) plus the drift of the bf16-computed residual stream,
# taken generously at 1e-2.
EPS_M = 1e-2


def router_delta(wr: np.ndarray, gain: np.ndarray) -> float:
    """Bound on how far apart the GPU's and the oracle's difference of two
    router logits may be. The FFN input m_t = g * x / rms(x) has
    ||m_t|| <= sqrt(h) max|g|; an error of relative size EPS_M spread over
    its h coordinates moves logit e = <m_t, Wr_e> by a sum of h terms with
    standard deviation EPS_M ||m_t|| ||Wr_e|| / sqrt(h) <= EPS_M max|g|
    ||Wr_e||; a difference of two logits has at most sqrt(2) times that, and
    six standard deviations are allowed."""
    return 6.0 * math.sqrt(2.0) * EPS_M * float(np.abs(gain).max()) * float(np.linalg.norm(wr, axis=1).max())


def check_routing_valid(cfg, packed, route, logits):
    """Every (layer, token): k distinct experts in range, and every chosen
    logit >= the largest unchosen logit - router_delta (the oracle's own
    logits on the path with this routing)."""
    L, T, k = route.shape
    assert (L, T, k) == (cfg.n_layers, logits.shape[1], cfg.top_k)
    assert route.min() >= 0 and route.max() < cfg.n_experts
    srt = np.sort(route, axis=2)
    assert np.all(srt[..., 1:] != srt[..., :-1]), "an expert chosen twice"
    W = oracle.unpack(cfg, packed, bf16=True)
    worst = -np.inf
    for l in range(L):
        delta = router_delta(bf16_bits_to_f32(W[f"layer{l}.w_router"]), bf16_bits_to_f32(W[f"layer{l}.w_ffn_norm"]))
        if k == cfg.n_experts:
            continue
        r = logits[l].astype(np.float64)
        chosen = np.zeros(r.shape, bool)
        chosen[np.arange(T)[:, None], route[l]] = True
        min_chosen = np.where(chosen, r, np.inf).min(axis=1)
        max_other = np.where(chosen, -np.inf, r).max(axis=1)
        short = max_other - min_chosen  # > 0 where an unchosen expert scored higher
        worst = max(worst, float(short.max() / delta))
        bad = np.nonzero(short > delta)[0]
        assert bad.size == 0, (l, bad[:8], short[bad[:8]], delta)
    return worst


def check_against_oracle(cfg, tok, lab, packed, loss, grads, route):
    l_ref, g_ref, logits = oracle.forward_backward(cfg, packed, tok, lab, bf16=True, route_in=route,
                                                   want_logits=True)
    check_routing_valid(cfg, packed, route, logits)
    return compare(cfg, grads, g_ref, tok, loss, l_ref)


@pytest.mark.parametrize("K", [1, 2])
def test_tiny_moe_matches_oracle(K):
    cfg = TINY_MOE
    tok, lab, packed, loss, grads, route = run_moe(cfg, 2, 32, K, 201, 202)
    check_against_oracle(cfg, tok, lab, packed, loss, grads, route)


def test_moe_wider_layer_gqa16_matches_oracle():
    """Hidden 512, 16 query heads over 1 KV head (the Qwen3-MoE group of 16;
    q width 1024 != hidden), 16 experts of width 128, top-4, ragged tokens."""
    cfg = oracle.Config(n_layers=2, hidden=512, n_heads=16, n_kv_heads=1, head_dim=64, ffn_dim=0, vocab=1000,
                        rope_theta=1e6, norm_eps=1e-6, n_experts=16, top_k=4, expert_ffn=128)
    tok, lab, packed, loss, grads, route = run_moe(cfg, 1, 77, 2, 211, 212)
    check_against_oracle(cfg, tok, lab, packed, loss, grads, route)


def test_moe_single_token_routes_k_experts():
    cfg = TINY_MOE
    tok, lab, packed, loss, grads, route = run_moe(cfg, 1, 1, 1, 221, 222)
    check_against_oracle(cfg, tok, lab, packed, loss, grads, route)
    # experts that received no token have exactly zero gradients
    G = oracle.unpack(cfg, grads)
    for l in range(cfg.n_layers):
        chosen = set(route[l, 0].tolist())
        for e in range(cfg.n_experts):
            if e not in chosen:
                assert not np.any(G[f"layer{l}.w_experts_gu"][e]) and not np.any(G[f"layer{l}.w_experts_down"][e])


def test_moe_bitwise_identical_across_K():
    torch, mt = need_gpu()
    cfg = with_layers(TINY_MOE, 4)
    tok, lab = make_tokens(cfg, 2, 32, 231)
    packed = make_params(cfg, 232, bf16=True)
    out = []
    with moe_session(mt, cfg, 2, 32, 4) as s:
        s.params[:] = packed
        for K in (1, 2, 3, 4, 1):
            loss = s.step(tok, lab, K)
            out.append((K, loss, s.grads.copy(), s.routing(64)))
    _, l0, g0, r0 = out[0]
    for K, loss, g, r in out[1:]:
        assert loss == l0, K
        assert np.array_equal(g.view(np.uint32), g0.view(np.uint32)), K
        assert np.array_equal(r, r0), K


def test_routing_query_errors():
    torch, mt = need_gpu()
    cfg = TINY_MOE
    with moe_session(mt, cfg, 1, 8, 1) as s:
        with pytest.raises(mt.MtError):
            s.routing(8)  # no step yet
        tok, lab = make_tokens(cfg, 1, 8, 1)
        s.params[:] = make_params(cfg, 2, bf16=True)
        s.step(tok, lab, 1)
        with pytest.raises(mt.MtError):
            s.routing(9)  # wrong size
        assert s.routing(8).shape == (cfg.n_layers, 8, cfg.top_k)


def test_qwen3_moe_shape_full_batch_properties():
    """Two layers of the Qwen3-235B-style MoE shape (hidden 4096, 64 q / 4 kv
    heads x 128, 128 experts x 1536, top-8, vocab 151936) at the benchmark's
    batch (B=1, S=4096: 32768 routed rows), in the step's own launch
    configuration. Properties that hold at any size: every token routes to 8
    distinct experts; K=2 and K=1 give bitwise-identical gradients and
    routing; with W_out = 0 the loss is ln(V) and every gradient except the
    head's is exactly zero (nothing flows back from the head)."""
    from tests.common import QWEN3_MOE
    torch, mt = need_gpu()
    cfg = with_layers(QWEN3_MOE, 2)
    B, S = 1, 4096
    tok, lab = make_tokens(cfg, B, S, 241)
    with moe_session(mt, cfg, B, S, 2) as s:
        s.params[:] = make_params(cfg, 242, bf16=True)
        loss2 = s.step(tok, lab, 2)
        g2 = s.grads.copy()
        r2 = s.routing(B * S)
        srt = np.sort(r2, axis=2)
        assert np.all(srt[..., 1:] != srt[..., :-1]) and r2.min() >= 0 and r2.max() < cfg.n_experts
        loss1 = s.step(tok, lab, 1)
        assert loss1 == loss2
        assert np.array_equal(s.grads.view(np.uint32), g2.view(np.uint32))
        assert np.array_equal(s.routing(B * S), r2)
        del g2
        assert math.isfinite(loss2) and 0.5 * math.log(cfg.vocab) < loss2 < 2.0 * math.log(cfg.vocab)
        off, nb = oracle.tensor_offset(cfg, cfg.n_layers + 1, 1, True)
        s.params[off:off + nb] = 0
        loss0 = s.step(tok, lab, 2)
        assert abs(loss0 - math.log(cfg.vocab)) < 1e-4 * math.log(cfg.vocab)
        goff, gnb = oracle.tensor_offset(cfg, cfg.n_layers + 1, 1, False)
        g = s.grads
        assert not np.any(g[:goff // 4] != 0) and not np.any(g[(goff + gnb) // 4:] != 0)
        assert np.any(g[goff // 4:(goff + gnb) // 4] != 0)
    assert mt.mt_op_device_error() == 0


@pytest.mark.parametrize("E,k", [(8, 1), (8, 8), (16, 3)], ids=["top1", "all_experts", "top3_of_16"])
def test_moe_routing_degenerate_cases(E, k):
    """Top-1 routing; every expert chosen by every token (the mixture is then
    the full softmax mixture and no row is padded away from any expert); an
    odd k. Same comparison against the oracle."""
    cfg = oracle.Config(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=0, vocab=256,
                        rope_theta=1e4, norm_eps=1e-5, n_experts=E, top_k=k, expert_ffn=32)
    tok, lab, packed, loss, grads, route = run_moe(cfg, 2, 24, 2, 251 + E + k, 252)
    check_against_oracle(cfg, tok, lab, packed, loss, grads, route)
    if k == E:
        assert np.all(np.sort(route, axis=2) == np.arange(E))


def _moe_op(torch, mt, m, wr, wgu, wd, k):
    """Run mt_op_moe_ffn_fwd on device bf16 tensors; returns (out, route)."""
    T, h = m.shape
    E, Fe = wr.shape[0], wd.shape[2]
    resid = torch.zeros((T, h), dtype=torch.float32, device="cuda")
    out = torch.empty((T, h), dtype=torch.float32, device="cuda")
    route = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(mt.mt_op_moe_workspace(T, h, E, k, Fe), dtype=torch.uint8, device="cuda")
    mt.mt_op_moe_ffn_fwd(m, wr, wgu, wd, resid, out, route, ws, T, h, E, k, Fe)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    return out.cpu().numpy(), route.cpu().numpy()


def _bf16_dev(torch, shape, gen, std):
    return (torch.randn(shape, generator=gen, device="cuda") * std).to(torch.bfloat16)


def _host(t):
    return t.float().cpu().numpy()


def test_moe_op_matches_oracle():
    """The layer's MoE forward as one entry point (router, routing, grouped
    expert GEMMs, combine), ragged tokens, against the oracle with the GPU's
    choices forced; the choices must be the oracle's own."""
    torch, mt = need_gpu()
    T, h, E, k, Fe = 77, 128, 16, 4, 64
    gen = torch.Generator(device="cuda").manual_seed(261)
    m = _bf16_dev(torch, (T, h), gen, 1.0)
    wr, wgu, wd = (_bf16_dev(torch, s, gen, 0.05) for s in ((E, h), (E, 2 * Fe, h), (E, h, Fe)))
    out, route = _moe_op(torch, mt, m, wr, wgu, wd, k)
    ref, own, *_ = oracle.moe_ffn(_host(m), _host(wr), _host(wgu), _host(wd), k)
    assert np.array_equal(np.sort(route, axis=1), np.sort(own, axis=1))
    ref_forced, *_ = oracle.moe_ffn(_host(m), _host(wr), _host(wgu), _host(wd), k, route_in=route)
    from tests.common import rel_l2
    assert rel_l2(out, ref_forced) < 1.5e-2


def test_moe_op_sampled_at_qwen3_shape():
    """The MoE forward at the Qwen3-style layer's full size (T=4096 tokens,
    hidden 4096, 128 experts x 1536, top-8: 32768 routed rows), checked on
    sampled tokens: their chosen experts are the top-8 of their logits
    (recomputed in double), and their outputs match the oracle run on just
    those tokens and the experts they use (the renormalised weights depend
    only on the chosen logits, so dropping the other experts changes
    nothing). The routing itself is checked for every token."""
    torch, mt = need_gpu()
    T, h, E, k, Fe = 4096, 4096, 128, 8, 1536
    gen = torch.Generator(device="cuda").manual_seed(271)
    m = _bf16_dev(torch, (T, h), gen, 1.0)
    wr, wgu, wd = (_bf16_dev(torch, s, gen, 0.02) for s in ((E, h), (E, 2 * Fe, h), (E, h, Fe)))
    out, route = _moe_op(torch, mt, m, wr, wgu, wd, k)
    # every token's choice: k distinct experts whose logits (recomputed in
    # double from the same bf16 inputs) are the k largest, up to the fp32
    # accumulation error of the GPU's logits (1e-4 of the token's largest)
    r64 = _host(m).astype(np.float64) @ _host(wr).astype(np.float64).T
    chosen = np.zeros((T, E), bool)
    chosen[np.arange(T)[:, None], route] = True
    assert np.all(chosen.sum(axis=1) == k)
    min_chosen = np.where(chosen, r64, np.inf).min(axis=1)
    max_other = np.where(chosen, -np.inf, r64).max(axis=1)
    assert np.all(min_chosen >= max_other - 1e-4 * np.abs(r64).max(axis=1))
    rng = np.random.default_rng(272)
    tok = np.sort(rng.choice(T, 6, replace=False))
    m_s = _host(m[torch.as_tensor(tok, device="cuda")]).astype(np.float64)
    used = np.unique(route[tok])
    idx = torch.as_tensor(used, device="cuda")
    remap = {e: j for j, e in enumerate(used)}
    route_sub = np.vectorize(remap.get)(route[tok]).astype(np.int32)
    ref, *_ = oracle.moe_ffn(m_s.astype(np.float32), _host(wr[idx]), _host(wgu[idx]), _host(wd[idx]), k,
                             route_in=route_sub)
    from tests.common import rel_l2
    assert rel_l2(out[tok], ref) < 1.5e-2


def _moe_op_bwd(torch, mt, m, wr, wgu, wd, dout, k):
    T, h = m.shape
    E, Fe = wr.shape[0], wd.shape[2]
    dm = torch.empty((T, h), dtype=torch.float32, device="cuda")
    dwr = torch.empty((E, h), dtype=torch.float32, device="cuda")
    dwgu = torch.empty((E, 2 * Fe, h), dtype=torch.float32, device="cuda")
    dwd = torch.empty((E, h, Fe), dtype=torch.float32, device="cuda")
    route = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(mt.mt_op_moe_bwd_workspace(T, h, E, k, Fe), dtype=torch.uint8, device="cuda")
    mt.mt_op_moe_ffn_bwd(m, wr, wgu, wd, dout, dm, dwr, dwgu, dwd, route, ws, T, h, E, k, Fe)
    torch.cuda.synchronize()
    assert mt.mt_op_device_error() == 0
    return dm, dwr, dwgu, dwd, route.cpu().numpy()


def test_moe_op_backward_matches_oracle():
    """The MoE backward entry point (forward recomputed inside, grouped expert
    products, router backward) against the oracle with the same routing."""
    from tests.common import rel_l2
    torch, mt = need_gpu()
    T, h, E, k, Fe = 77, 128, 16, 4, 64
    gen = torch.Generator(device="cuda").manual_seed(281)
    m = _bf16_dev(torch, (T, h), gen, 1.0)
    wr, wgu, wd = (_bf16_dev(torch, s, gen, 0.05) for s in ((E, h), (E, 2 * Fe, h), (E, h, Fe)))
    dout = torch.randn((T, h), generator=gen, device="cuda")
    dm, dwr, dwgu, dwd, route = _moe_op_bwd(torch, mt, m, wr, wgu, wd, dout, k)
    _, _, rdm, rdwr, rdwgu, rdwd = oracle.moe_ffn(_host(m), _host(wr), _host(wgu), _host(wd), k,
                                                  dout.cpu().numpy(), route_in=route)
    for got, ref in ((dm, rdm), (dwr, rdwr), (dwgu, rdwgu), (dwd, rdwd)):
        assert rel_l2(got.cpu().numpy(), ref) < 2e-2


def test_moe_op_backward_at_qwen3_shape_sparse_dout():
    """The MoE backward at the Qwen3-style layer's full size (T=4096, hidden
    4096, 128 experts x 1536, top-8) with dL/d(out) nonzero on six sampled
    tokens only: every gradient then comes from those tokens alone, so the
    oracle run on just them and the experts they use must reproduce the
    experts' and router's gradients of those experts and the tokens' dm rows,
    and every other gradient must vanish."""
    from tests.common import rel_l2
    torch, mt = need_gpu()
    T, h, E, k, Fe = 4096, 4096, 128, 8, 1536
    gen = torch.Generator(device="cuda").manual_seed(291)
    m = _bf16_dev(torch, (T, h), gen, 1.0)
    wr, wgu, wd = (_bf16_dev(torch, s, gen, 0.02) for s in ((E, h), (E, 2 * Fe, h), (E, h, Fe)))
    rng = np.random.default_rng(292)
    tok = np.sort(rng.choice(T, 6, replace=False))
    tok_d = torch.as_tensor(tok, device="cuda")
    dout = torch.zeros((T, h), device="cuda")
    dout[tok_d] = torch.randn((len(tok), h), generator=gen, device="cuda")
    dm, dwr, dwgu, dwd, route = _moe_op_bwd(torch, mt, m, wr, wgu, wd, dout, k)
    used = np.unique(route[tok])
    idx = torch.as_tensor(used, device="cuda")
    remap = {e: j for j, e in enumerate(used)}
    route_sub = np.vectorize(remap.get)(route[tok]).astype(np.int32)
    _, _, rdm, rdwr, rdwgu, rdwd = oracle.moe_ffn(_host(m[tok_d]), _host(wr[idx]), _host(wgu[idx]), _host(wd[idx]),
                                                  k, dout[tok_d].cpu().numpy(), route_in=route_sub)
    assert rel_l2(dm[tok_d].cpu().numpy(), rdm) < 2e-2
    assert rel_l2(dwr[idx].cpu().numpy(), rdwr) < 2e-2
    assert rel_l2(dwgu[idx].cpu().numpy(), rdwgu) < 2e-2
    assert rel_l2(dwd[idx].cpu().numpy(), rdwd) < 2e-2
    others = torch.ones(E, dtype=torch.bool, device="cuda")
    others[idx] = False
    rest = torch.ones(T, dtype=torch.bool, device="cuda")
    rest[tok_d] = False
    for t in (dwr[others], dwgu[others], dwd[others], dm[rest]):
        assert not torch.any(t != 0).item()
