"""mt_train_step: the streamed step with the host AdamW applied to each unit
as its gradients land. Its result must be exactly that of mt_forward_backward
followed by mt_adamw_update over all units (the overlap changes only when
the updates run), and the loss on a fixed batch must fall."""
import numpy as np
import pytest

import oracle
from tests.common import TINY_GQA, bf16_bits_to_f32, make_params, make_tokens, with_layers
from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _master_f32(cfg, packed, bf16):
    """fp32 master copy (fp32 packed layout) holding the values of the packed params."""
    out = np.zeros(oracle.packed_bytes(cfg, False) // 4, np.float32)
    for unit, t, name, shape, is_gain in oracle.tensor_list(cfg):
        o32, nb32 = oracle.tensor_offset(cfg, unit, t, False)
        op, nbp = oracle.tensor_offset(cfg, unit, t, bf16)
        if bf16:
            vals = bf16_bits_to_f32(packed[op:op + nbp].view(np.uint16))
        else:
            vals = packed[op:op + nbp].view(np.float32)
        out[o32 // 4:(o32 + nb32) // 4] = vals
    return out


@pytest.mark.parametrize("bf16", [False, True])
def test_train_step_is_step_then_update(bf16):
    torch, mt = need_gpu()
    cfg = with_layers(TINY_GQA, 3)
    if bf16:  # bf16 host parameters need an FFN width that is a multiple of 8
        cfg = oracle.Config(**{**cfg.__dict__, "ffn_dim": 176})
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps)
    dt = mt.MT_BF16 if bf16 else mt.MT_F32
    tok, lab = make_tokens(cfg, 2, 32, 31)
    packed = make_params(cfg, 32, bf16=bf16)
    opt = mt.adamw_cfg(2e-3, 0.9, 0.999, 1e-8, 0.01)
    units = cfg.n_layers + 2
    runs = {}
    with mt.Session(shape, 2, 32, 2, dt) as s:
        s.params[:] = packed
        s.bind_optimizer(opt, _master_f32(cfg, packed, bf16), n_threads=3)
        for i in range(2):
            loss = s.train_step(tok, lab, 2)
            st = s.stats()
            assert st["optimizer_ms"] > 0 and st["optimizer_exposed_ms"] >= 0
            runs[i] = (loss, s.grads.copy(), s.params.copy(), s.opt_master.copy(), s.opt_m.copy(), s.opt_v.copy())
    with mt.Session(shape, 2, 32, 2, dt) as s:
        s.params[:] = packed
        master = _master_f32(cfg, packed, bf16)
        m = np.zeros_like(master)
        v = np.zeros_like(master)
        for i in range(2):
            loss = s.step(tok, lab, 2)
            mt.mt_adamw_update(s.cfg, opt, i + 1, 0, units, master.ctypes.data, m.ctypes.data, v.ctypes.data,
                               s.grads_ptr, s.params_ptr, dt, 2)
            l_a, g_a, p_a, w_a, m_a, v_a = runs[i]
            assert loss == l_a
            assert np.array_equal(s.grads.view(np.uint32), g_a.view(np.uint32))
            assert np.array_equal(s.params, p_a)
            for x, y in ((master, w_a), (m, m_a), (v, v_a)):
                assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert runs[1][0] < runs[0][0]  # one AdamW step on the same batch lowers its loss


def test_train_step_mixture_of_experts():
    """The same equality for a mixture-of-experts model (router and expert
    tensors are updated like any other), and the loss falls."""
    from tests.common import TINY_MOE
    torch, mt = need_gpu()
    cfg = TINY_MOE
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps, cfg.n_experts, cfg.top_k, cfg.expert_ffn)
    tok, lab = make_tokens(cfg, 2, 32, 33)
    packed = make_params(cfg, 34, bf16=True)
    opt = mt.adamw_cfg(2e-3, 0.9, 0.999, 1e-8, 0.01)
    units = cfg.n_layers + 2
    losses = []
    with mt.Session(shape, 2, 32, 2, mt.MT_BF16) as s:
        s.params[:] = packed
        s.bind_optimizer(opt, _master_f32(cfg, packed, True), n_threads=3)
        for i in range(2):
            losses.append(s.train_step(tok, lab, 2))
        p_train = s.params.copy()
    with mt.Session(shape, 2, 32, 2, mt.MT_BF16) as s:
        s.params[:] = packed
        master = _master_f32(cfg, packed, True)
        m = np.zeros_like(master)
        v = np.zeros_like(master)
        for i in range(2):
            assert s.step(tok, lab, 2) == losses[i]
            mt.mt_adamw_update(s.cfg, opt, i + 1, 0, units, master.ctypes.data, m.ctypes.data, v.ctypes.data,
                               s.grads_ptr, s.params_ptr, mt.MT_BF16, 2)
        assert np.array_equal(s.params, p_train)
    assert losses[1] < losses[0]


def test_train_step_needs_an_optimizer():
    torch, mt = need_gpu()
    cfg = TINY_GQA
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps)
    tok, lab = make_tokens(cfg, 2, 32, 33)
    with mt.Session(shape, 2, 32, 1, mt.MT_F32) as s:
        s.params[:] = make_params(cfg, 34)
        with pytest.raises(mt.MtError) as e:
            s.train_step(tok, lab, 1)
        assert e.value.code == mt.MT_ERR_STATE
        with pytest.raises(mt.MtError) as e:
            mt.mt_bind_optimizer(s.ctx, mt.adamw_cfg(1e-3, 1.5), s.grads_ptr, s.grads_ptr, s.grads_ptr)
        assert e.value.code == mt.MT_ERR_ARG


def test_async_steps_follow_the_staleness_one_schedule():
    """Three asynchronous steps and a flush equal the staggered schedule run
    with the synchronous pieces: step k uses the parameters through k-2."""
    torch, mt = need_gpu()
    cfg = with_layers(TINY_GQA, 3)
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps)
    batches = [make_tokens(cfg, 2, 32, 40 + k) for k in range(3)]
    packed = make_params(cfg, 44)
    opt = mt.adamw_cfg(3e-3, 0.9, 0.999, 1e-8, 0.01)
    units = cfg.n_layers + 2
    with mt.Session(shape, 2, 32, 2, mt.MT_F32) as s:
        s.params[:] = packed
        s.bind_optimizer(opt, _master_f32(cfg, packed, False), n_threads=3)
        got = []
        for tok, lab in batches:
            got.append((s.train_step_async(tok, lab, 2), s.grads.copy()))
        with pytest.raises(mt.MtError) as e:  # a pending update blocks the synchronous form
            s.train_step(*batches[0], 2)
        assert e.value.code == mt.MT_ERR_STATE
        s.optimizer_flush()
        final = (s.params.copy(), s.opt_master.copy(), s.opt_m.copy(), s.opt_v.copy())
    with mt.Session(shape, 2, 32, 2, mt.MT_F32) as s:
        s.params[:] = packed
        master = _master_f32(cfg, packed, False)
        m, v = np.zeros_like(master), np.zeros_like(master)
        grads = []

        def update(k, g):
            mt.mt_adamw_update(s.cfg, opt, k, 0, units, master.ctypes.data, m.ctypes.data, v.ctypes.data,
                               g.ctypes.data, s.params_ptr, mt.MT_F32, 2)

        for k, (tok, lab) in enumerate(batches):
            loss = s.step(tok, lab, 2)  # step k+1 with the parameters through k-1
            assert loss == got[k][0]
            assert np.array_equal(s.grads.view(np.uint32), got[k][1].view(np.uint32))
            grads.append(s.grads.copy())
            if k >= 1:
                update(k, grads[k - 1])
        update(3, grads[2])
        for x, y in zip((s.params, master, m, v), final):
            assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))


@pytest.mark.parametrize("kind,nth", [(1, 3), (2, 1)], ids=["copy_issue_fails", "final_wait_times_out"])
def test_failed_async_step_applies_the_pending_update_once(kind, nth):
    """An asynchronous step that fails part-way (a host-side injected fault:
    the third weight-copy issue fails, or the final wait times out while the
    GPU and the publisher are still working) leaves its pending update
    pending; the flush that follows completes it, and every unit's update is
    applied exactly once: master, moments and streamed parameters equal one
    mt_adamw_update of the first step's gradients."""
    torch, mt = need_gpu()
    cfg = with_layers(TINY_GQA, 3)
    shape = mt.ModelShape(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, cfg.rope_theta, cfg.norm_eps)
    tok0, lab0 = make_tokens(cfg, 2, 32, 60)
    tok1, lab1 = make_tokens(cfg, 2, 32, 61)
    packed = make_params(cfg, 62)
    opt = mt.adamw_cfg(3e-3, 0.9, 0.999, 1e-8, 0.01)
    units = cfg.n_layers + 2
    with mt.Session(shape, 2, 32, 2, mt.MT_F32) as s:
        s.params[:] = packed
        s.bind_optimizer(opt, _master_f32(cfg, packed, False), n_threads=3)
        s.train_step_async(tok0, lab0, 2)
        g0 = s.grads.copy()
        mt.mt_debug_inject_fault(s.ctx, kind, nth)
        with pytest.raises(mt.MtError):
            s.train_step_async(tok1, lab1, 2)
        mt.mt_debug_inject_fault(s.ctx, 0, 0)
        s.optimizer_flush()
        got = (s.params.copy(), s.opt_master.copy(), s.opt_m.copy(), s.opt_v.copy())
    master = _master_f32(cfg, packed, False)
    m, v = np.zeros_like(master), np.zeros_like(master)
    params = packed.copy()
    mt.mt_adamw_update(s.cfg, opt, 1, 0, units, master.ctypes.data, m.ctypes.data, v.ctypes.data, g0.ctypes.data,
                       params.ctypes.data, mt.MT_F32, 2)
    for x, y in zip((params, master, m, v), got):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))
