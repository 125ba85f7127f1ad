"""The allocation-free RMSNorm backward (mt_op_rmsnorm_bwd_noalloc) against
the regular entry point that takes a caller workspace.

Some callers cannot allocate device memory where they call the library; this
variant takes its scratch from a fixed array inside the library instead. The
test calls it twice in a row (the array keeps the previous call's contents,
so the second call checks that nothing stale leaks in) and compares each
result with mt_op_rmsnorm_bwd on the same inputs, with the tolerance the
kernel tests use for fp32 outputs. This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import seedgen
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
    return out


def test_noalloc_matches_workspace_variant_on_consecutive_calls():
    torch, mt = need_gpu()
    # first call: many rows (large partial buffer); second: fewer rows and a
    # different width, so stale partials from the first call would show up
    for T, h, seed in ((1000, 512, 70), (77, 320, 80)):
        (dx_a, dxb_a, dw_a), (dx_b, dxb_b, dw_b) = _call_both(torch, mt, T, h, seed)
        assert rel_l2(dx_b, dx_a) < 1e-5
        assert rel_l2(dxb_b, dxb_a) < 6e-3
        assert rel_l2(dw_b, dw_a) < 1e-5
        assert np.all(np.isfinite(dw_b))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch, mt = need_gpu()
    T, h = 32 * 300, 4096  # 300 * 4096 partial sums > 1,048,576
    X = torch.zeros((1, 4), device="cuda")  # never touched: the size check comes first
    with pytest.raises(mt.MtError) as e:
        mt.mt_op_rmsnorm_bwd_noalloc(X, X, X, X, None, X, None, X, T, h)
    assert e.value.code == mt.MT_ERR_BUDGET
