"""bf16 gradient streaming (grad_dtype = MT_BF16): the device rounds every
gradient to bf16 (nearest even) before it streams back.

Every gradient is produced in fp32 and rounded once, so the bf16 buffer must
equal the fp32 buffer of the same step rounded to bf16, bit for bit (the
accumulation order does not depend on the output type). Against the oracle
the bf16 gradients meet the same bar as fp32 ones (one more rounding of
2^-9 relative is far inside rel-L2 2e-2).
"""
import numpy as np
import pytest

import oracle
from tests.common import TINY, TINY_GQA, TINY_MOE, bf16_bits_to_f32, f32_to_bf16_bits, make_params, make_tokens, \
    with_layers
from tests.gpu_util import need_gpu
from tests.test_gpu_e2e import compare

pytestmark = pytest.mark.gpu


def session(mt, cfg, B, S, max_K, bf16_params, grad_dtype):
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps, cfg.n_experts, cfg.top_k, cfg.expert_ffn)
    return mt.Session(shape, B, S, max_K, mt.MT_BF16 if bf16_params else mt.MT_F32, grad_dtype=grad_dtype)


def to_f32_layout(cfg, g16):
    """bf16 gradient buffer (bf16 packed layout) -> fp32 packed layout."""
    out = np.zeros(oracle.packed_bytes(cfg, False) // 4, np.float32)
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        o16, n16 = oracle.tensor_offset(cfg, unit, t, True)
        o32, _ = oracle.tensor_offset(cfg, unit, t, False)
        out[o32 // 4:o32 // 4 + n16 // 2] = bf16_bits_to_f32(g16[o16 // 2:(o16 + n16) // 2])
    return out


def both(cfg, B, S, K, seed_w, seed_t, bf16_params):
    torch, mt = need_gpu()
    tok, lab = make_tokens(cfg, B, S, seed_t)
    packed = make_params(cfg, seed_w, bf16=bf16_params)
    res = {}
    for gd in (mt.MT_F32, mt.MT_BF16):
        with session(mt, cfg, B, S, K, bf16_params, gd) as s:
            s.params[:] = packed
            res[gd] = (s.step(tok, lab, K), s.grads.copy())
    assert mt.mt_op_device_error() == 0
    return mt, tok, lab, packed, res


@pytest.mark.parametrize("cfg,bf16_params", [(TINY, False), (with_layers(TINY_GQA, 3), False),
                                             (TINY_MOE, True)], ids=["tiny", "tiny_gqa_3l", "tiny_moe"])
def test_bf16_gradients_are_the_rounded_fp32_gradients(cfg, bf16_params):
    mt, tok, lab, packed, res = both(cfg, 2, 32, 2, 301, 302, bf16_params)
    (l32, g32), (l16, g16) = res[mt.MT_F32], res[mt.MT_BF16]
    assert l16 == l32
    assert g16.dtype == np.uint16 and g16.nbytes == oracle.packed_bytes(cfg, True)
    want = np.zeros_like(g16)
    for unit, t, name, shape, _ in oracle.tensor_list(cfg):
        o16, n16 = oracle.tensor_offset(cfg, unit, t, True)
        o32, _ = oracle.tensor_offset(cfg, unit, t, False)
        want[o16 // 2:(o16 + n16) // 2] = f32_to_bf16_bits(g32[o32 // 4:o32 // 4 + n16 // 2])
    assert np.array_equal(g16, want)


def test_bf16_gradients_match_oracle():
    cfg = TINY_GQA
    mt, tok, lab, packed, res = both(cfg, 2, 32, 1, 311, 312, False)
    l16, g16 = res[mt.MT_BF16]
    l_ref, g_ref = oracle.forward_backward(cfg, packed, tok, lab)
    compare(cfg, to_f32_layout(cfg, g16), g_ref, tok, l16, l_ref)


def test_host_optimizer_needs_fp32_gradients():
    torch, mt = need_gpu()
    cfg = TINY
    with session(mt, cfg, 1, 8, 1, False, mt.MT_BF16) as s:
        n32 = oracle.packed_bytes(cfg, False) // 4
        with pytest.raises(mt.MtError):
            s.bind_optimizer(mt.adamw_cfg(1e-3, 0.9, 0.999, 1e-8, 0.0), np.zeros(n32, np.float32))
