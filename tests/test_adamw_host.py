"""The host AdamW of the C ABI (mt_adamw_update) against the optimizer
oracle (oracle/adamw.py, float64), over the packed layout. Host logic only:
no GPU is used."""
import numpy as np
import pytest

import layer_streamed_gb300 as mt
from oracle.adamw import AdamW, adamw_step
from tests.common import TINY, bf16_round


def _cfg(c):
    return mt.make_cfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab)


def _units(c):
    return [(0, 1)] + [(u, 9) for u in range(1, c.n_layers + 1)] + [(c.n_layers + 1, 2)]


def _tensor_mask(cfg, c, dtype, esz, units=None):
    """Boolean mask of the packed elements (element size esz) that belong to tensors of the given units."""
    n = mt.mt_packed_bytes(cfg, dtype) // esz
    mask = np.zeros(n, bool)
    for u, nt in _units(c):
        if units is not None and u not in units:
            continue
        for t in range(nt):
            off, nb = mt.mt_tensor_offset(cfg, dtype, u, t)
            mask[off // esz:(off + nb) // esz] = True
    return mask


def _state(cfg, c, seed):
    rng = np.random.default_rng(seed)
    mask = _tensor_mask(cfg, c, mt.MT_F32, 4)
    n = mask.size
    master = np.where(mask, rng.normal(0, 0.02, n), 0).astype(np.float32)
    m = np.where(mask, rng.normal(0, 1e-3, n), 0).astype(np.float32)
    v = np.where(mask, rng.uniform(0, 1e-5, n), 0).astype(np.float32)
    g = np.where(mask, rng.normal(0, 1e-2, n), 0).astype(np.float32)
    return master, m, v, g, mask


def _params_of(cfg, c, master, dtype):
    """The streamed copy: master values moved into the params layout (and rounded for bf16)."""
    esz = 2 if dtype == mt.MT_BF16 else 4
    out = np.zeros(mt.mt_packed_bytes(cfg, dtype) // esz, np.uint16 if esz == 2 else np.float32)
    for u, nt in _units(c):
        for t in range(nt):
            o32, nb32 = mt.mt_tensor_offset(cfg, mt.MT_F32, u, t)
            op, nbp = mt.mt_tensor_offset(cfg, dtype, u, t)
            vals = master[o32 // 4:(o32 + nb32) // 4]
            if esz == 2:
                out[op // 2:(op + nbp) // 2] = (bf16_round(vals).view(np.uint32) >> 16).astype(np.uint16)
            else:
                out[op // 4:(op + nbp) // 4] = vals
    return out


@pytest.mark.parametrize("dtype", [mt.MT_F32, mt.MT_BF16])
def test_host_adamw_matches_oracle(dtype):
    c = TINY
    cfg = _cfg(c)
    # the ABI takes the hyper-parameters as float32; the oracle gets those same values
    f32 = lambda x: float(np.float32(x))
    opt = AdamW(lr=f32(1e-3), beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8), weight_decay=f32(0.01))
    master, m, v, g, mask = _state(cfg, c, 5)
    params = _params_of(cfg, c, master, dtype)
    step = 3
    m0, v0 = m.copy(), v.copy()
    th_ref, m_ref, v_ref = adamw_step(opt, step, master, m, v, g)
    mt.mt_adamw_update(cfg, mt.adamw_cfg(opt.lr, opt.beta1, opt.beta2, opt.eps, opt.weight_decay), step, 0,
                       c.n_layers + 2, master.ctypes.data, m.ctypes.data, v.ctypes.data, g.ctypes.data,
                       params.ctypes.data, dtype, 3)
    # fp32 rounding of beta1 m + (1 - beta1) g is relative to the terms, which may cancel
    m_scale = opt.beta1 * np.abs(m0.astype(np.float64)) + (1 - opt.beta1) * np.abs(g.astype(np.float64))
    assert np.all(np.abs(m - m_ref) <= 4 * 2.0 ** -24 * m_scale + 1e-30)
    assert np.allclose(v, v_ref, rtol=4 * 2.0 ** -24, atol=1e-30)  # both terms >= 0: no cancellation
    assert np.all(v0 >= 0)
    # fp32 arithmetic against float64: the step itself is ~lr, so compare the moves
    moved = master.astype(np.float64) - _state(cfg, c, 5)[0]
    moved_ref = th_ref - _state(cfg, c, 5)[0]
    assert np.max(np.abs(moved - moved_ref)) <= 1e-3 * opt.lr
    assert np.all(master[~mask] == 0)  # padding untouched
    # the streamed copy is the updated master in the params dtype (bf16: round to nearest even)
    assert np.array_equal(params, _params_of(cfg, c, master, dtype))


def test_unit_range_updates_only_those_units():
    c = TINY
    cfg = _cfg(c)
    opt = mt.adamw_cfg(1e-2)
    master, m, v, g, mask = _state(cfg, c, 9)
    before = master.copy()
    params = _params_of(cfg, c, master, mt.MT_F32)
    mt.mt_adamw_update(cfg, opt, 1, 1, 2, master.ctypes.data, m.ctypes.data, v.ctypes.data, g.ctypes.data,
                       params.ctypes.data, mt.MT_F32, 0)
    in_layer1 = _tensor_mask(cfg, c, mt.MT_F32, 4, units={1})
    assert not np.array_equal(master[in_layer1], before[in_layer1])
    assert np.array_equal(master[~in_layer1], before[~in_layer1])


def test_adamw_argument_errors():
    c = TINY
    cfg = _cfg(c)
    a = np.zeros(mt.mt_packed_bytes(cfg, mt.MT_F32) // 4, np.float32)
    for step, u0, u1 in ((0, 0, 1), (1, -1, 1), (1, 0, c.n_layers + 3), (1, 2, 1)):
        with pytest.raises(mt.MtError) as e:
            mt.mt_adamw_update(cfg, mt.adamw_cfg(), step, u0, u1, a.ctypes.data, a.ctypes.data, a.ctypes.data,
                               a.ctypes.data, a.ctypes.data, mt.MT_F32, 1)
        assert e.value.code == mt.MT_ERR_ARG


def test_host_adamw_mixture_of_experts_layout():
    """The update runs over every tensor of a mixture-of-experts model's
    layout (router, experts' gate|up and down matrices) exactly as over a
    dense one: the same element-wise rule against the oracle."""
    from tests.common import TINY_MOE
    c = TINY_MOE
    cfg = mt.make_cfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab,
                      param_dtype=mt.MT_BF16, n_experts=c.n_experts, top_k=c.top_k, expert_ffn=c.expert_ffn)
    f32 = lambda x: float(np.float32(x))
    opt = AdamW(lr=f32(1e-3), beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-8), weight_decay=f32(0.01))
    master, m, v, g, mask = _state(cfg, c, 7)
    params = _params_of(cfg, c, master, mt.MT_BF16)
    th_ref, _, _ = adamw_step(opt, 2, master, m, v, g)
    mt.mt_adamw_update(cfg, mt.adamw_cfg(opt.lr, opt.beta1, opt.beta2, opt.eps, opt.weight_decay), 2, 0,
                       c.n_layers + 2, master.ctypes.data, m.ctypes.data, v.ctypes.data, g.ctypes.data,
                       params.ctypes.data, mt.MT_BF16, 2)
    start = _state(cfg, c, 7)[0]
    assert np.max(np.abs((master.astype(np.float64) - start) - (th_ref - start))) <= 1e-3 * opt.lr
    assert np.array_equal(params, _params_of(cfg, c, master, mt.MT_BF16))
    # the router and expert tensors moved
    for t in (6, 7, 8):
        off, nb = mt.mt_tensor_offset(cfg, mt.MT_F32, 1, t)
        assert np.any(master[off // 4:(off + nb) // 4] != start[off // 4:(off + nb) // 4])


def test_host_adamw_refuses_bf16_gradients():
    c = TINY
    cfg = mt.make_cfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab,
                      grad_dtype=mt.MT_BF16)
    a = np.zeros(mt.mt_packed_bytes(cfg, mt.MT_F32) // 4, np.float32)
    with pytest.raises(mt.MtError) as e:
        mt.mt_adamw_update(cfg, mt.adamw_cfg(), 1, 0, 1, a.ctypes.data, a.ctypes.data, a.ctypes.data,
                           a.ctypes.data, a.ctypes.data, mt.MT_F32, 1)
    assert e.value.code == mt.MT_ERR_UNSUPPORTED
