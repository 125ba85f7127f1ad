"""Pins of the optimizer oracle (oracle/adamw.py) against closed forms that
follow from the update rule by hand, not by re-running the rule."""
import numpy as np
import pytest

from oracle.adamw import AdamW, adamw_step


def test_first_step_moves_by_lr_times_sign():
    # t = 1 from zero moments: m^ = g and v^ = g^2, so the step is lr g / (|g| + eps)
    opt = AdamW(lr=0.01, eps=1e-8)
    g = np.array([3.0, -0.5, 1e-3, -2e4])
    theta, m, v = adamw_step(opt, 1, np.zeros(4), np.zeros(4), np.zeros(4), g)
    assert np.allclose(theta, -0.01 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=0)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


def test_constant_gradient_takes_equal_steps():
    # with g fixed, the bias corrections are exact: m^ = g and v^ = g^2 at every t
    opt = AdamW(lr=0.003, beta1=0.8, beta2=0.95, eps=1e-8)
    g = np.array([0.7, -1.3])
    theta, m, v = np.array([1.0, 2.0]), np.zeros(2), np.zeros(2)
    for t in range(1, 8):
        theta, m, v = adamw_step(opt, t, theta, m, v, g)
    assert np.allclose(theta, np.array([1.0, 2.0]) - 7 * 0.003 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=0)


def test_weight_decay_is_decoupled():
    # zero gradient: the moments stay 0 and only the decay acts, theta (1 - lr wd)
    opt = AdamW(lr=0.1, weight_decay=0.01)
    theta, m, v = adamw_step(opt, 1, np.array([2.0, -4.0]), np.zeros(2), np.zeros(2), np.zeros(2))
    assert np.allclose(theta, np.array([2.0, -4.0]) * (1 - 0.1 * 0.01), rtol=1e-15, atol=0)


def test_two_steps_worked_by_hand():
    # g = +1 then -1, beta1 0.9, beta2 0.999, lr 1:
    # m1 = 0.1, v1 = 0.001; m2 = 0.09 - 0.1 = -0.01, v2 = 0.000999 + 0.001 = 0.001999
    # m^2 = -0.01 / 0.19, v^2 = 0.001999 / (1 - 0.998001) = 1, step = m^2 / (1 + eps)
    opt = AdamW(lr=1.0, beta1=0.9, beta2=0.999, eps=1e-8)
    th, m, v = adamw_step(opt, 1, np.zeros(1), np.zeros(1), np.zeros(1), np.ones(1))
    th2, m2, v2 = adamw_step(opt, 2, np.zeros(1), m, v, -np.ones(1))
    assert m2[0] == pytest.approx(-0.01, rel=1e-12) and v2[0] == pytest.approx(0.001999, rel=1e-12)
    assert th2[0] == pytest.approx(0.01 / 0.19 / (1 + 1e-8), rel=1e-12)


def test_step_numbers_start_at_one():
    with pytest.raises(ValueError):
        adamw_step(AdamW(), 0, np.zeros(1), np.zeros(1), np.zeros(1), np.zeros(1))
