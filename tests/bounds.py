"""Per-element error bounds for the GPU parity tests, derived from the
arithmetic the kernels perform.

  U16  bf16 keeps 8 significant bits: rounding x to nearest even moves it by
       at most half a unit in the last place, U16 = 2^-8 of |x|.
  U32  the same for fp32: 2^-24.
  acc(K)  fp32 accumulation of K products a_i b_i. Each addition rounds by
       at most U32 of the running sum; the rounding errors of a long sum
       behave like a random walk, so 8 sqrt(K) U32 times sum_i |a_i b_i| is a
       bound far beyond eight standard deviations (the worst case K U32 is
       never approached by round-to-nearest sums of mixed-sign terms).

Every bound is |got - ref| <= (terms built from these and from magnitudes
that the oracle computes on absolute values of the same operands), checked
element by element: one wrong element fails however many right ones
surround it.
"""
from __future__ import annotations

import math

import numpy as np

U16 = 2.0 ** -8
U32 = 2.0 ** -24


def acc(K: int) -> float:
    return 8.0 * math.sqrt(max(int(K), 1)) * U32


def check(got, ref, bound, what: str = "") -> float:
    """Assert |got - ref| <= bound element by element (NaN fails); returns
    the largest ratio |got - ref| / bound, for reporting."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.broadcast_to(np.asarray(bound, dtype=np.float64), ref.shape)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements outside the bound; first at {idx}: "
                             f"got {got[idx]!r}, ref {ref[idx]!r}, bound {bound[idx]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / bound, 0.0)
    return float(r.max()) if r.size else 0.0


def pair_sum(x: np.ndarray) -> np.ndarray:
    """b_i + b_{partner(i)} over the last axis (RoPE's half-split pairs
    (i, i + d/2)): the bound of a value after a rotation that mixes each
    pair with coefficients of magnitude <= 1."""
    d = x.shape[-1]
    h = d // 2
    out = x.copy()
    out[..., :h] += x[..., h:]
    out[..., h:] += x[..., :h]
    return out


def silu_parts(g: np.ndarray):
    """sigmoid(g), silu(g), and the magnitude sigma(1 + |g|(1 - sigma)) that
    bounds |silu'(g)| term by term (silu' itself can cancel to zero)."""
    g = np.asarray(g, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-g))
    return s, g * s, s * (1.0 + np.abs(g) * (1.0 - s))


def attention_magnitudes(q, k, v, do):
    """Per-element magnitudes of causal GQA attention and its gradients,
    q/do [B,S,nq,d], k/v [B,S,nkv,d] (fp64 numpy):
      o_abs  = sum_j P_ij |v_j|
      dq_abs = sum_j P_ij (|dP_ij| + Dm_i) |k_j| / sqrt(d)
      dk_abs = sum over the group's heads and i of P_ij (|dP_ij| + Dm_i) |q_i| / sqrt(d)
      dv_abs = sum over the group's heads and i of P_ij |do_i|
    with dP = do v^T and Dm_i = sum_c |do_ic| o_abs_ic, which bounds
    D_i = <do_i, o_i> and its error when o carries the forward's bf16
    rounding errors. A bf16 rounding of P, of dS = P (dP - D), of the
    forward output o or of the result perturbs each term by at most a few
    U16 of these magnitudes."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, S, nq, d = q.shape
    nkv = k.shape[2]
    grp = nq // nkv
    o_abs = np.zeros_like(q)
    dq_abs = np.zeros_like(q)
    dk_abs = np.zeros_like(k)
    dv_abs = np.zeros_like(v)
    mask = np.tril(np.ones((S, S), dtype=bool))
    sc = 1.0 / math.sqrt(d)
    for b in range(B):
        for hq in range(nq):
            g = hq // grp
            s = (q[b, :, hq] @ k[b, :, g].T) * sc
            s = np.where(mask, s, -np.inf)
            s -= s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            o_abs[b, :, hq] = p @ np.abs(v[b, :, g])
            dp = do[b, :, hq] @ v[b, :, g].T
            Dm = np.sum(np.abs(do[b, :, hq]) * o_abs[b, :, hq], axis=1)
            m = p * (np.abs(dp) + Dm[:, None])
            dq_abs[b, :, hq] = m @ np.abs(k[b, :, g]) * sc
            dk_abs[b, :, g] += m.T @ np.abs(q[b, :, hq]) * sc
            dv_abs[b, :, g] += p.T @ np.abs(do[b, :, hq])
    return o_abs, dq_abs, dk_abs, dv_abs
