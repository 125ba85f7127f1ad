"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, and its packed layout and budget plan
agree with the definition (restated independently by the oracle)."""
import os
import re

import numpy as np
import pytest

import oracle
from tests.common import LLAMA8B, QWEN3_MOE, SMALL, TINY, TINY_GQA, TINY_MOE

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mt():
    import layer_streamed_gb300 as m
    m.build()
    m.lib()
    return m


def _cfg(mt, c, bf16=False, **kw):
    return mt.make_cfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.vocab, c.rope_theta,
                       c.norm_eps, kw.get("max_batch", 2), kw.get("max_seq", 32), kw.get("max_K", 2),
                       mt.MT_BF16 if bf16 else mt.MT_F32, c.n_experts, c.top_k, c.expert_ffn)


def test_header_symbols_are_exported(mt):
    hdr = open(os.path.join(ROOT, "include", "mt.h")).read()
    declared = set(re.findall(r"\b(mt_[a-z_0-9]+)\s*\(", hdr))
    declared -= {"mt_layer_cfg", "mt_stats", "mt_memory_plan"}
    assert declared == set(mt.EXPORTS), declared ^ set(mt.EXPORTS)
    L = mt.lib()
    for name in declared:
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {mt.LIB_PATH}").read()
    for name in declared:
        assert re.search(rf"\bT {name}$", out, re.M), name


@pytest.mark.parametrize("c", [TINY, TINY_GQA, SMALL, LLAMA8B], ids=["tiny", "tiny_gqa", "small", "llama8b"])
@pytest.mark.parametrize("bf16", [False, True])
def test_layout_matches_definition(mt, c, bf16):
    cfg = _cfg(mt, c, bf16)
    assert mt.mt_packed_bytes(cfg, mt.MT_BF16 if bf16 else mt.MT_F32) == oracle.packed_bytes(c, bf16)
    for unit, t, name, shape, _ in oracle.tensor_list(c):
        assert mt.mt_tensor_offset(cfg, mt.MT_BF16 if bf16 else mt.MT_F32, unit, t) == \
            oracle.tensor_offset(c, unit, t, bf16), name


def test_layout_rejects_unknown_tensor(mt):
    cfg = _cfg(mt, TINY)
    with pytest.raises(mt.MtError):
        mt.mt_tensor_offset(cfg, mt.MT_F32, 1, 9)
    with pytest.raises(mt.MtError):
        mt.mt_tensor_offset(cfg, mt.MT_F32, TINY.n_layers + 2, 0)


def test_budget_covers_two_layers_and_one_block(mt):
    """The device plan holds two weight buffers, two gradient buffers, one
    block of activations and the checkpoints; it grows with max_K and tokens."""
    c = LLAMA8B
    cfg4 = _cfg(mt, c, True, max_batch=2, max_seq=4096, max_K=4)
    cfg8 = _cfg(mt, c, True, max_batch=2, max_seq=4096, max_K=8)
    b4, b8 = mt.mt_required_budget(cfg4), mt.mt_required_budget(cfg8)
    layer_bf16 = oracle.tensor_offset(c, 2, 0, True)[0] - oracle.tensor_offset(c, 1, 0, True)[0]
    assert b4 > 4 * layer_bf16          # 2 weight buffers + 2 fp32 gradient buffers
    assert b8 > b4
    assert b4 < 40 * 2**30              # far below the 8B model's 16 GB of weights + 32 GB of grads + activations


def test_invalid_configs_rejected(mt):
    bad = [
        dict(hidden=96),       # not a multiple of 64
        dict(head_dim=48),     # unsupported head_dim
        dict(n_kv_heads=3),    # n_heads % n_kv_heads != 0
    ]
    for kw in bad:
        d = dict(TINY.__dict__)
        d.update(kw)
        c = oracle.Config(**d)
        assert mt.mt_required_budget(_cfg(mt, c)) == 0, kw
    # bf16 params need ffn % 8 == 0 (172 is not)
    assert mt.mt_required_budget(_cfg(mt, TINY, bf16=True)) == 0
    assert mt.mt_required_budget(_cfg(mt, TINY, bf16=False)) > 0


def test_create_without_gpu_fails_cleanly(mt):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(mt.MtError) as e:
        mt.mt_create(_cfg(mt, TINY), 1 << 40)
    assert e.value.code in (mt.MT_ERR_CUDA, mt.MT_ERR_BUDGET)


@pytest.mark.parametrize("c", [TINY_MOE, QWEN3_MOE], ids=["tiny_moe", "qwen3_moe"])
def test_moe_layout_matches_definition(mt, c):
    cfg = _cfg(mt, c, True)
    assert mt.mt_packed_bytes(cfg, mt.MT_BF16) == oracle.packed_bytes(c, True)
    assert mt.mt_packed_bytes(cfg, mt.MT_F32) == oracle.packed_bytes(c, False)
    for unit, t, name, shape, _ in oracle.tensor_list(c):
        for bf16 in (False, True):
            assert mt.mt_tensor_offset(cfg, mt.MT_BF16 if bf16 else mt.MT_F32, unit, t) == \
                oracle.tensor_offset(c, unit, t, bf16), name


def test_moe_budget_and_validation(mt):
    """The Qwen3-style MoE layer (4.97 GB of bf16 weights) fits two weight
    slots, two fp32 gradient slots and one block of routed activations well
    inside the device; invalid expert settings are rejected."""
    c = QWEN3_MOE
    cfg = _cfg(mt, c, True, max_batch=1, max_seq=4096, max_K=2)
    b = mt.mt_required_budget(cfg)
    layer_bf16 = oracle.tensor_offset(c, 2, 0, True)[0] - oracle.tensor_offset(c, 1, 0, True)[0]
    assert 6 * layer_bf16 < b < 6 * layer_bf16 + 12 * 2**30
    assert mt.mt_required_budget(_cfg(mt, c, False, max_batch=1, max_seq=4096, max_K=2)) == 0  # fp32 params
    import dataclasses
    for kw in (dict(n_experts=12), dict(top_k=0), dict(top_k=9, n_experts=8), dict(expert_ffn=20),
               dict(ffn_dim=1024)):
        bad = dataclasses.replace(TINY_MOE, **kw)
        assert mt.mt_required_budget(_cfg(mt, bad, True)) == 0, kw


def test_moe_op_workspace_and_argument_checks(mt):
    """Host-side checks of the kernel-level MoE entry points (no GPU work)."""
    assert mt.mt_op_moe_workspace(4096, 4096, 128, 8, 1536) > 0
    assert mt.mt_op_moe_bwd_workspace(4096, 4096, 128, 8, 1536) > mt.mt_op_moe_workspace(4096, 4096, 128, 8, 1536)
    for bad in ((0, 4096, 128, 8, 1536), (8, 100, 128, 8, 1536), (8, 4096, 12, 8, 1536), (8, 4096, 8, 9, 1536),
                (8, 4096, 128, 8, 1000)):
        assert mt.mt_op_moe_workspace(*bad) == 0 and mt.mt_op_moe_bwd_workspace(*bad) == 0
    L = mt.lib()
    assert L.mt_op_moe_ffn_fwd(None, None, None, None, None, None, None, None, 8, 4096, 128, 8, 1536, None) == \
        mt.MT_ERR_ARG
    assert L.mt_op_moe_ffn_bwd(*([None] * 11), 8, 4096, 128, 8, 1536, None) == mt.MT_ERR_ARG
