"""The allocation-free RMSNorm backward (mt_op_rmsnorm_bwd_noalloc) against
the regular entry point that takes a caller workspace.

Some callers cannot allocate device memory where they call the library; this
variant takes its scratch from a fixed array inside the library instead. The
test calls it twice in a row (the array keeps the previous call's contents,
so the second call checks that nothing stale leaks in) and compares each
result with mt_op_rmsnorm_bwd on the same inputs, with the tolerance the
kernel tests use for fp32 outputs, and with the oracle's RMSNorm backward
element by element. This file is collected last so that a run stopping at
the first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
import seedgen
from tests.bounds import U16, U32, acc, check
from tests.common import rel_l2
from tests.gpu_util import from_dev, need_gpu, to_dev_f32

pytestmark = pytest.mark.gpu


def _normal(shape, seed):
    return seedgen.normal(int(np.prod(shape)), seed, 9).reshape(shape)


def _call_both(torch, mt, T, h, seed):
    x, dy, res = _normal((T, h), seed), _normal((T, h), seed + 1), _normal((T, h), seed + 2)
    w = 1.0 + 0.1 * _normal((h,), seed + 3)
    X, W, DY, RES = (to_dev_f32(torch, a) for a in (x, w, dy, res))
    Y = torch.empty((T, h), dtype=torch.bfloat16, device="cuda")
    R = torch.empty(T, device="cuda")
    mt.mt_op_rmsnorm_fwd(X, W, Y, R, T, h, 1e-5)
    out = []
    for noalloc in (False, True):
        DX = torch.full((T, h), float("nan"), device="cuda")
        DXb = torch.zeros((T, h), dtype=torch.bfloat16, device="cuda")
        DW = torch.full((h,), float("nan"), device="cuda")
        if noalloc:
            mt.mt_op_rmsnorm_bwd_noalloc(X, W, R, DY, RES, DX, DXb, DW, T, h)
        else:
            ws = torch.empty(mt.mt_op_rmsnorm_bwd_workspace(T, h), device="cuda")
            mt.mt_op_rmsnorm_bwd(X, W, R, DY, RES, DX, DXb, DW, ws, T, h)
        torch.cuda.synchronize()
        out.append((from_dev(DX), from_dev(DXb), from_dev(DW)))
    return out, (x, w, dy, res, from_dev(R))


def _check_against_oracle(T, h, inputs, got):
    """The oracle's RMSNorm backward plus the residual, element by element
    (the bounds of the kernel parity tests: the rstd the kernel was given,
    an fp32 row sum of h terms and a few fp32 operations per element)."""
    x, w, dy, res, r = inputs
    dx, dxb, dw = got
    dx_ref, dw_ref = oracle.rmsnorm_bwd(x, w, dy, 1e-5)
    r64 = r.astype(np.float64)[:, None]
    e_r = acc(h) + 4 * U32
    t1 = r64 * np.abs(w * dy)
    t2 = np.abs(x) * r64 ** 3 * np.mean(np.abs(w * dy * x), axis=1, keepdims=True)
    e_dx = (3 * e_r + acc(h) + 8 * U32) * (t1 + t2) + 2 * U32 * (np.abs(dx_ref + res) + np.abs(res))
    check(dx, dx_ref + res, e_dx, "dx")
    check(dxb, dx_ref + res, U16 * np.abs(dx_ref + res) + (1 + U16) * e_dx, "dx bf16")
    check(dw, dw_ref, (e_r + acc(T) + 4 * U32) * np.sum(np.abs(dy * x) * r64, axis=0), "dw")
    assert rel_l2(dx, dx_ref + res) < 1e-5 and rel_l2(dw, dw_ref) < 1e-5


def test_noalloc_matches_workspace_variant_on_consecutive_calls():
    torch, mt = need_gpu()
    # first call: many rows (large partial buffer); second: fewer rows and a
    # different width, so stale partials from the first call would show up
    for T, h, seed in ((1000, 512, 70), (77, 320, 80)):
        ((dx_a, dxb_a, dw_a), (dx_b, dxb_b, dw_b)), inputs = _call_both(torch, mt, T, h, seed)
        assert rel_l2(dx_b, dx_a) < 1e-5
        assert rel_l2(dxb_b, dxb_a) < 6e-3
        assert rel_l2(dw_b, dw_a) < 1e-5
        assert np.all(np.isfinite(dw_b))
        _check_against_oracle(T, h, inputs, (dx_b, dxb_b, dw_b))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch, mt = need_gpu()
    T, h = 32 * 300, 4096  # 300 * 4096 partial sums > 1,048,576
    X = torch.zeros((1, 4), device="cuda")  # never touched: the size check comes first
    with pytest.raises(mt.MtError) as e:
        mt.mt_op_rmsnorm_bwd_noalloc(X, X, X, X, None, X, None, X, T, h)
    assert e.value.code == mt.MT_ERR_BUDGET
