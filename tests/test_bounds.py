"""CPU checks of the element-wise bound helpers used by the GPU parity tests:
the magnitudes agree with the oracle run on absolute values, and the check
rejects one planted error and NaN."""
import numpy as np
import pytest

import oracle
from tests.bounds import U16, acc, attention_magnitudes, check, pair_sum


def _rng_attn(seed=3, B=1, S=33, nq=4, nkv=2, d=16):
    rng = np.random.default_rng(seed)
    q, do = (rng.normal(size=(B, S, nq, d)).astype(np.float32) for _ in range(2))
    k, v = (rng.normal(size=(B, S, nkv, d)).astype(np.float32) for _ in range(2))
    return q, k, v, do


def test_attention_magnitudes_match_the_oracle_on_absolute_values():
    q, k, v, do = _rng_attn()
    o_abs, dq_abs, dk_abs, dv_abs = attention_magnitudes(q, k, v, do)
    # sum_j P_ij |v_j| is the oracle's attention output with |v| as values;
    # sum_i P_ij |do_i| is its dV with |do| as the output gradient
    o_ref = oracle.attention(q, k, np.abs(v))[0]
    dv_ref = oracle.attention(q, k, v, np.abs(do))[4]
    assert np.allclose(o_abs, o_ref, rtol=1e-5, atol=1e-6)
    assert np.allclose(dv_abs, dv_ref, rtol=1e-5, atol=1e-6)
    # the gradient magnitudes bound the oracle's gradients themselves
    _, _, dq, dk, _ = oracle.attention(q, k, v, do)
    assert np.all(np.abs(dq) <= dq_abs * (1 + 1e-5) + 1e-6)
    assert np.all(np.abs(dk) <= dk_abs * (1 + 1e-5) + 1e-6)


def test_check_rejects_one_bad_element_and_nan():
    ref = np.linspace(-1, 1, 1000).reshape(10, 100)
    got = ref * (1 + 0.5 * U16)
    assert check(got, ref, U16 * np.abs(ref)) <= 0.5 + 1e-9
    bad = got.copy()
    bad[3, 7] += 4 * U16
    with pytest.raises(AssertionError):
        check(bad, ref, U16 * np.abs(ref) + 1e-3 * U16)
    bad = got.copy()
    bad[9, 99] = np.nan
    with pytest.raises(AssertionError):
        check(bad, ref, 1.0)


def test_pair_sum_and_acc():
    x = np.arange(8.0)
    assert np.array_equal(pair_sum(x), np.array([4, 6, 8, 10, 4, 6, 8, 10.0]))
    assert acc(4096) == pytest.approx(8 * 64 * 2.0 ** -24)
