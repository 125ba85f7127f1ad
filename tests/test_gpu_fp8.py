"""FP8 weight streaming (param_dtype MT_FP8) on the GPU.

The step computes with the dequantised weights bf16(e4m3(code) * row scale).
So (1) its gradients equal, bit for bit, those of the bf16 step run on a
bf16 model holding exactly those weights (same kernels on the same operand
values: the device dequantisation is exact to the definition), and (2) it
meets the oracle bar against the oracle run on the dequantised weights
(decoded in numpy from the format's definition)."""
import numpy as np
import pytest

import oracle
from tests.common import bf16_bits_to_f32, make_params, make_tokens, with_layers
from tests.fp8_ref import dequant_rows_bf16_bits, fp8_tensor
from tests.gpu_util import need_gpu
from tests.test_gpu_e2e import compare

pytestmark = pytest.mark.gpu

TINY176 = oracle.Config(n_layers=3, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=176, vocab=256,
                        rope_theta=1e4, norm_eps=1e-5)


def _shape(mt, c):
    return mt.ModelShape(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab, c.rope_theta,
                         c.norm_eps, c.n_experts, c.top_k, c.expert_ffn)


def _fp8_and_bf16_models(mt, cfg, seed, B, S, K):
    """(FP8 packed params, the bf16 packed model of its dequantised weights)."""
    src = make_params(cfg, seed, bf16=True)
    lcfg = mt.make_cfg(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim, cfg.vocab,
                       cfg.rope_theta, cfg.norm_eps, B, S, K, mt.MT_FP8, cfg.n_experts, cfg.top_k, cfg.expert_ffn)
    fp8 = np.zeros(mt.mt_packed_bytes(lcfg, mt.MT_FP8), np.uint8)
    mt.mt_quantize_params_fp8(lcfg, src.ctypes.data, mt.MT_BF16, fp8.ctypes.data, 0)
    deq = np.zeros(oracle.packed_bytes(cfg, True), np.uint8)
    for unit, t, name, shape, is_gain in oracle.tensor_list(cfg):
        off8, _ = mt.mt_tensor_offset(lcfg, mt.MT_FP8, unit, t)
        off16, nb16 = oracle.tensor_offset(cfg, unit, t, True)
        if is_gain:  # fp32 gains (1.0 here: exact in bf16)
            g = fp8[off8:off8 + 4 * shape[0]].view(np.float32)
            assert np.all(bf16_bits_to_f32((g.view(np.uint32) >> 16).astype(np.uint16)) == g)
            deq[off16:off16 + nb16] = ((g.view(np.uint32) >> 16).astype(np.uint16)).view(np.uint8)
        else:  # matrices; an expert tensor [E, rows, cols] is E * rows rows
            codes, scales = fp8_tensor(fp8, off8, int(np.prod(shape[:-1])), shape[-1])
            deq[off16:off16 + nb16] = dequant_rows_bf16_bits(codes, scales).view(np.uint8).ravel()
    return fp8, deq


def _step(mt, cfg, dtype, params, tok, lab, K, max_K):
    with mt.Session(_shape(mt, cfg), tok.shape[0], tok.shape[1], max_K, dtype) as s:
        s.params[:] = params
        loss = s.step(tok, lab, K)
        return loss, s.grads.copy()


@pytest.mark.parametrize("cfg,B,S,K", [(TINY176, 2, 32, 2), (oracle.Config(n_layers=2, hidden=1024, n_heads=16,
                                                                            n_kv_heads=16, head_dim=64,
                                                                            ffn_dim=2816, vocab=32000,
                                                                            rope_theta=1e4, norm_eps=1e-5), 1, 96, 1)],
                         ids=["tiny", "small_widths"])
def test_fp8_step_equals_bf16_step_on_dequantised_weights(cfg, B, S, K):
    torch, mt = need_gpu()
    fp8, deq = _fp8_and_bf16_models(mt, cfg, 71, B, S, K)
    tok, lab = make_tokens(cfg, B, S, 72)
    l8, g8 = _step(mt, cfg, mt.MT_FP8, fp8, tok, lab, K, K)
    lb, gb = _step(mt, cfg, mt.MT_BF16, deq, tok, lab, K, K)
    assert l8 == lb
    assert np.array_equal(g8.view(np.uint32), gb.view(np.uint32))
    assert mt.mt_op_device_error() == 0


def test_fp8_mixture_of_experts_step_equals_bf16_step_on_dequantised_weights():
    """Router and expert matrices streamed as FP8 (one scale per row of each
    expert's matrices): same gradients and routing, bit for bit, as the bf16
    step on the dequantised weights."""
    torch, mt = need_gpu()
    from tests.common import TINY_MOE
    cfg = with_layers(TINY_MOE, 3)
    fp8, deq = _fp8_and_bf16_models(mt, cfg, 91, 2, 32, 2)
    tok, lab = make_tokens(cfg, 2, 32, 92)
    out = []
    for dtype, params in ((mt.MT_FP8, fp8), (mt.MT_BF16, deq)):
        with mt.Session(_shape(mt, cfg), 2, 32, 2, dtype) as s:
            s.params[:] = params
            loss = s.step(tok, lab, 2)
            out.append((loss, s.grads.copy(), s.routing(64)))
    assert out[0][0] == out[1][0]
    assert np.array_equal(out[0][1].view(np.uint32), out[1][1].view(np.uint32))
    assert np.array_equal(out[0][2], out[1][2])
    assert mt.mt_op_device_error() == 0


def test_fp8_step_matches_oracle_on_dequantised_weights_and_is_K_invariant():
    torch, mt = need_gpu()
    cfg = TINY176
    fp8, deq = _fp8_and_bf16_models(mt, cfg, 81, 2, 32, 3)
    tok, lab = make_tokens(cfg, 2, 32, 82)
    l1, g1 = _step(mt, cfg, mt.MT_FP8, fp8, tok, lab, 1, 3)
    l3, g3 = _step(mt, cfg, mt.MT_FP8, fp8, tok, lab, 3, 3)
    assert l1 == l3 and np.array_equal(g1.view(np.uint32), g3.view(np.uint32))
    l_ref, g_ref = oracle.forward_backward(cfg, deq, tok, lab, bf16=True)
    compare(cfg, g1, g_ref, tok, l1, l_ref)


def test_fp8_rejected_where_unsupported():
    torch, mt = need_gpu()
    cfg = oracle.Config(n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=172, vocab=256)
    with pytest.raises(mt.MtError):  # ffn_dim % 16 != 0
        mt.Session(_shape(mt, cfg), 1, 8, 1, mt.MT_FP8)
    with mt.Session(_shape(mt, TINY176), 1, 8, 1, mt.MT_FP8) as s:
        with pytest.raises(mt.MtError) as e:  # the host optimizer does not publish FP8
            s.bind_optimizer(mt.adamw_cfg(1e-3, 0.9, 0.95, 1e-8, 0.0),
                             np.zeros(mt.mt_packed_bytes(s.cfg, mt.MT_F32) // 4, np.float32))
        assert e.value.code == mt.MT_ERR_UNSUPPORTED
