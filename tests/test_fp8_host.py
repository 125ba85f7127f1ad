"""The FP8 packed layout and the host quantiser (no GPU): codes are the
nearest E4M3 values of w / scale with scale = row max / 448 (checked by
brute force over every code, ties to the even mantissa, saturation at 448),
offsets and sizes follow the layout, and the gains stay fp32."""
import numpy as np
import pytest

import oracle
from tests.common import bf16_bits_to_f32, f32_to_bf16_bits, make_params
from tests.fp8_ref import e4m3_table, fp8_tensor, nearest_e4m3

CFG = oracle.Config(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=176, vocab=256,
                    rope_theta=1e4, norm_eps=1e-5)


def _lib():
    import layer_streamed_gb300 as mt
    mt.build()
    mt.lib()
    return mt


def _cfg(mt, c, dtype):
    return mt.make_cfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab, c.rope_theta,
                       c.norm_eps, 2, 32, 2, dtype)


def _rows_cols(c, unit, t, shape):
    return shape[0] if len(shape) == 2 else 1, shape[-1]


def test_e4m3_table_from_the_definition():
    tab = e4m3_table()
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0 and np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6 and tab[0x38] == 1.0 and tab[0x39] == 1.125
    fin = tab[np.isfinite(tab)]
    assert np.unique(fin).size == 253  # +-0 share a value; two NaNs excluded


def test_fp8_layout_offsets_and_sizes():
    mt = _lib()
    cfg = _cfg(mt, CFG, mt.MT_FP8)
    prev_end, prev_unit = 0, -1
    for unit, t, name, shape, is_gain in oracle.tensor_list(CFG):
        off, nb = mt.mt_tensor_offset(cfg, mt.MT_FP8, unit, t)
        assert off % 256 == 0 and off >= prev_end
        if unit != prev_unit:
            assert off % 4096 == 0
            prev_unit = unit
        if is_gain:
            assert nb == 4 * shape[0]
        else:
            rows, cols = shape
            assert nb == (rows * cols + 15) // 16 * 16 + 4 * rows
        prev_end = off + nb
    assert mt.mt_packed_bytes(cfg, mt.MT_FP8) >= prev_end


def test_quantiser_is_nearest_e4m3_of_row_scaled_weights():
    mt = _lib()
    src = make_params(CFG, 5, bf16=True)
    W = oracle.unpack(CFG, src, bf16=True)
    # one row with exact midpoints between E4M3 values (row max 448: scale 1)
    wq = bf16_bits_to_f32(W["layer0.wq"][0]).copy()
    special = np.array([448.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -10), 0.0, 11.0, 12.5,
                        208.0, 232.0], np.float32)
    wq[:special.size] = special
    W["layer0.wq"][0] = f32_to_bf16_bits(wq)
    cfg = _cfg(mt, CFG, mt.MT_FP8)
    dst = np.zeros(mt.mt_packed_bytes(cfg, mt.MT_FP8), np.uint8)
    mt.mt_quantize_params_fp8(cfg, src.ctypes.data, mt.MT_BF16, dst.ctypes.data, 3)
    tab = e4m3_table()
    for unit, t, name, shape, is_gain in oracle.tensor_list(CFG):
        off, nb = mt.mt_tensor_offset(cfg, mt.MT_FP8, unit, t)
        w = bf16_bits_to_f32(W[name]).reshape(-1 if is_gain else shape[0], shape[-1]) if not is_gain else None
        if is_gain:
            np.testing.assert_array_equal(dst[off:off + nb].view(np.float32), bf16_bits_to_f32(W[name]))
            continue
        codes, scales = fp8_tensor(dst, off, *shape)
        amax = np.abs(w).max(axis=1).astype(np.float32)
        exp_scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        np.testing.assert_array_equal(scales, exp_scale)
        x = (w / exp_scale[:, None]).astype(np.float32)
        np.testing.assert_array_equal(tab[codes], nearest_e4m3(x).reshape(x.shape), err_msg=name)
    # the midpoints went to the even mantissa
    codes, _ = fp8_tensor(dst, mt.mt_tensor_offset(cfg, mt.MT_FP8, 1, 1)[0], CFG.n_heads * CFG.head_dim, CFG.hidden)
    got = tab[codes[0, :special.size]]
    np.testing.assert_array_equal(got, np.array([448, 1.0, 1.25, -1.0, 0.0, 2.0 ** -8, -0.0, 0.0, 11.0, 12.0, 208.0,
                                                 224.0], np.float32))


def test_quantiser_rejects_non_finite_weights():
    mt = _lib()
    src = make_params(CFG, 6, bf16=False)
    off, _ = oracle.tensor_offset(CFG, 1, 6, False)
    src[off:off + 4] = np.frombuffer(np.float32(np.inf).tobytes(), np.uint8)
    cfg = _cfg(mt, CFG, mt.MT_FP8)
    dst = np.zeros(mt.mt_packed_bytes(cfg, mt.MT_FP8), np.uint8)
    with pytest.raises(mt.MtError):
        mt.mt_quantize_params_fp8(cfg, src.ctypes.data, mt.MT_F32, dst.ctypes.data, 2)
