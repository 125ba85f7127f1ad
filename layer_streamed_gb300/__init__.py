"""Python binding of libmt.so: layer-streamed decoder training on one GPU.

Argument marshalling only: every step of the training path runs in the CUDA
library (``csrc/``); this module loads it with ctypes, exposes its C entry
points under the same names, and offers a small ``Session`` helper that owns
the pinned host buffers. There is no CPU fallback: if the compiled library is
missing, importing a function raises.

The method ("MegaTrain: Full Precision Training of 100B+ Parameter Large
Language Models on a Single GPU"): parameters and gradients live in pinned
host memory; each decoder layer's packed weights stream host-to-device into
one of two ping-pong buffers while the previous layer computes; the residual
stream is checkpointed every K layers; the backward pass recomputes each
K-block and back-propagates it layer by layer, streaming each layer's
gradients back to host on a separate stream.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmt.so")

MT_OK, MT_ERR_ARG, MT_ERR_BUDGET, MT_ERR_NOT_PINNED, MT_ERR_ALIGN = 0, -1, -2, -3, -4
MT_ERR_CUDA, MT_ERR_TIMEOUT, MT_ERR_STATE, MT_ERR_UNSUPPORTED, MT_ERR_DEVICE = -5, -6, -7, -8, -9
MT_F32, MT_BF16, MT_FP8 = 0, 1, 2
MT_GEMM_NT, MT_GEMM_NN, MT_GEMM_TN = 0, 1, 2
MT_EPI_BF16, MT_EPI_F32, MT_EPI_F32_ADD = 0, 1, 2

STATUS_NAMES = {0: "MT_OK", -1: "MT_ERR_ARG", -2: "MT_ERR_BUDGET", -3: "MT_ERR_NOT_PINNED", -4: "MT_ERR_ALIGN",
                -5: "MT_ERR_CUDA", -6: "MT_ERR_TIMEOUT", -7: "MT_ERR_STATE", -8: "MT_ERR_UNSUPPORTED",
                -9: "MT_ERR_DEVICE"}

# Every symbol include/mt.h declares.
EXPORTS = ("mt_packed_bytes", "mt_tensor_offset", "mt_required_budget", "mt_create", "mt_create_ex",
           "mt_bind_host_params", "mt_forward_backward", "mt_get_stats", "mt_set_tracing", "mt_get_memory_plan",
           "mt_last_error",
           "mt_destroy", "mt_host_alloc", "mt_host_free", "mt_debug_inject_fault", "mt_op_gemm",
           "mt_op_rmsnorm_fwd", "mt_op_rmsnorm_bwd_workspace", "mt_op_rmsnorm_bwd", "mt_op_rmsnorm_bwd_noalloc",
           "mt_op_rope", "mt_op_gemm_rope", "mt_op_attention_bwd_rope", "mt_op_gemm_swiglu", "mt_op_gemm_swiglu_bwd",
           "mt_op_attention_fwd", "mt_op_attention_bwd_workspace", "mt_op_attention_bwd", "mt_op_swiglu_fwd",
           "mt_op_swiglu_bwd", "mt_op_lmhead_ce_workspace", "mt_op_lmhead_ce", "mt_op_device_error",
           "mt_adamw_update", "mt_bind_optimizer", "mt_train_step", "mt_train_step_async", "mt_optimizer_flush",
           "mt_get_routing", "mt_replay_weight_stream", "mt_quantize_params_fp8", "mt_op_moe_workspace", "mt_op_moe_ffn_fwd", "mt_op_moe_bwd_workspace",
           "mt_op_moe_ffn_bwd")


class MtError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class mt_layer_cfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float),
                ("max_batch", ctypes.c_int32), ("max_seq", ctypes.c_int32), ("max_K", ctypes.c_int32),
                ("param_dtype", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("expert_ffn", ctypes.c_int32), ("grad_dtype", ctypes.c_int32)]


class mt_stats(ctypes.Structure):
    _fields_ = [("step_ms", ctypes.c_double), ("compute_busy_ms", ctypes.c_double), ("h2d_ms", ctypes.c_double),
                ("d2h_ms", ctypes.c_double), ("h2d_bytes", ctypes.c_double), ("d2h_bytes", ctypes.c_double),
                ("h2d_hidden_frac", ctypes.c_double), ("d2h_hidden_frac", ctypes.c_double),
                ("n_h2d", ctypes.c_int32), ("n_d2h", ctypes.c_int32), ("n_units", ctypes.c_int32),
                ("timing_enabled", ctypes.c_int32), ("gemm_ms", ctypes.c_double), ("gemm_flop", ctypes.c_double),
                ("attn_ms", ctypes.c_double), ("attn_flop", ctypes.c_double), ("n_gemm", ctypes.c_int32),
                ("n_attn", ctypes.c_int32), ("n_launches", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("optimizer_ms", ctypes.c_double), ("optimizer_exposed_ms", ctypes.c_double),
                ("h2d_phase_bytes", ctypes.c_double * 4), ("h2d_phase_ms", ctypes.c_double * 4),
                ("d2h_phase_bytes", ctypes.c_double * 4), ("d2h_phase_ms", ctypes.c_double * 4),
                ("h2d_copy_gbs_min", ctypes.c_double), ("h2d_copy_gbs_p10", ctypes.c_double),
                ("h2d_copy_gbs_p50", ctypes.c_double), ("h2d_copy_gbs_p90", ctypes.c_double),
                ("page_touch_ms", ctypes.c_double)]


class mt_replay_result(ctypes.Structure):
    _fields_ = [("n_copies", ctypes.c_int32), ("reserved", ctypes.c_int32), ("bytes", ctypes.c_double),
                ("ms", ctypes.c_double), ("host_numa_node", ctypes.c_int32), ("reserved2", ctypes.c_int32),
                ("touch_ms", ctypes.c_double)]


class mt_adamw_cfg(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class mt_memory_plan(ctypes.Structure):
    _fields_ = [("total", ctypes.c_size_t), ("weight_buffers", ctypes.c_size_t), ("grad_buffers", ctypes.c_size_t),
                ("checkpoints", ctypes.c_size_t), ("block_activations", ctypes.c_size_t),
                ("workspace", ctypes.c_size_t)]


_lib = None


def build(verbose: bool = False) -> str:
    from . import buildlib
    return buildlib.build(verbose=verbose)


def lib() -> ctypes.CDLL:
    """Load libmt.so. Raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library {LIB_PATH} is not built; call layer_streamed_gb300.build()")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    cfgp = P(mt_layer_cfg)
    sig = {
        "mt_packed_bytes": (sz, [cfgp, i32]),
        "mt_tensor_offset": (i32, [cfgp, i32, i32, i32, P(sz), P(sz)]),
        "mt_required_budget": (sz, [cfgp]),
        "mt_create": (i32, [cfgp, sz, P(vp)]),
        "mt_create_ex": (i32, [cfgp, sz, vp, P(vp), P(vp)]),
        "mt_bind_host_params": (i32, [vp, vp, i32]),
        "mt_forward_backward": (i32, [vp, vp, vp, i32, i32, i32, vp, P(f32)]),
        "mt_train_step": (i32, [vp, vp, vp, i32, i32, i32, vp, P(f32)]),
        "mt_train_step_async": (i32, [vp, vp, vp, i32, i32, i32, vp, P(f32)]),
        "mt_optimizer_flush": (i32, [vp]),
        "mt_bind_optimizer": (i32, [vp, P(mt_adamw_cfg), vp, vp, vp, i32]),
        "mt_adamw_update": (i32, [cfgp, P(mt_adamw_cfg), ctypes.c_int64, i32, i32, vp, vp, vp, vp, vp, i32, i32]),
        "mt_get_stats": (i32, [vp, P(mt_stats)]),
        "mt_get_routing": (i32, [vp, vp, sz]),
        "mt_replay_weight_stream": (i32, [vp, i32, i32, vp, i32, P(mt_replay_result)]),
        "mt_quantize_params_fp8": (i32, [cfgp, vp, i32, vp, i32]),
        "mt_set_tracing": (i32, [vp, i32, i32]),
        "mt_get_memory_plan": (i32, [vp, P(mt_memory_plan)]),
        "mt_last_error": (ctypes.c_char_p, [vp]),
        "mt_destroy": (None, [vp]),
        "mt_host_alloc": (vp, [sz]),
        "mt_host_free": (None, [vp]),
        "mt_debug_inject_fault": (i32, [vp, i32, i32]),
        "mt_op_gemm": (i32, [i32, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
        "mt_op_rmsnorm_fwd": (i32, [vp, vp, vp, vp, i32, i32, f32, vp]),
        "mt_op_rmsnorm_bwd_workspace": (sz, [i32, i32]),
        "mt_op_rmsnorm_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp]),
        "mt_op_rmsnorm_bwd_noalloc": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp]),
        "mt_op_rope": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]),
        "mt_op_gemm_rope": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, i32, f32, i32, vp]),
        "mt_op_attention_bwd_rope": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                           i32, vp, f32, vp]),
        "mt_op_gemm_swiglu": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
        "mt_op_gemm_swiglu_bwd": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
        "mt_op_attention_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp]),
        "mt_op_attention_bwd_workspace": (sz, [i32, i32, i32]),
        "mt_op_attention_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                      i32, vp]),
        "mt_op_swiglu_fwd": (i32, [vp, vp, i32, i32, i32, vp]),
        "mt_op_swiglu_bwd": (i32, [vp, vp, i32, i32, i32, vp]),
        "mt_op_lmhead_ce_workspace": (sz, [i32, i32, i32]),
        "mt_op_lmhead_ce": (i32, [vp, vp, vp, f32, vp, vp, vp, vp, i32, i32, i32, vp]),
        "mt_op_device_error": (i32, []),
        "mt_op_moe_workspace": (sz, [i32, i32, i32, i32, i32]),
        "mt_op_moe_ffn_fwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "mt_op_moe_bwd_workspace": (sz, [i32, i32, i32, i32, i32]),
        "mt_op_moe_ffn_bwd": (i32, [vp] * 11 + [i32, i32, i32, i32, i32, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(rc: int, ctx=None):
    if rc != MT_OK:
        msg = ""
        if ctx:
            m = lib().mt_last_error(ctx)
            msg = m.decode() if m else ""
        raise MtError(rc, msg)


# ---------------------------------------------------------------------------
# C entry points under their own names
# ---------------------------------------------------------------------------
def make_cfg(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, rope_theta=1e4, norm_eps=1e-5,
             max_batch=1, max_seq=1, max_K=1, param_dtype=MT_F32, n_experts=0, top_k=0,
             expert_ffn=0, grad_dtype=MT_F32) -> mt_layer_cfg:
    return mt_layer_cfg(n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, rope_theta, norm_eps,
                        max_batch, max_seq, max_K, param_dtype, n_experts, top_k, expert_ffn, grad_dtype)


def mt_packed_bytes(cfg: mt_layer_cfg, dtype: int) -> int:
    return lib().mt_packed_bytes(ctypes.byref(cfg), dtype)


def mt_tensor_offset(cfg: mt_layer_cfg, dtype: int, unit: int, tensor: int) -> tuple[int, int]:
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().mt_tensor_offset(ctypes.byref(cfg), dtype, unit, tensor, ctypes.byref(off), ctypes.byref(nb)))
    return off.value, nb.value


def mt_required_budget(cfg: mt_layer_cfg) -> int:
    return lib().mt_required_budget(ctypes.byref(cfg))


def mt_create(cfg: mt_layer_cfg, device_budget_bytes: int):
    out = ctypes.c_void_p()
    _check(lib().mt_create(ctypes.byref(cfg), device_budget_bytes, ctypes.byref(out)))
    return out


def mt_create_ex(cfg: mt_layer_cfg, device_budget_bytes: int, device_arena: int, streams=None):
    out = ctypes.c_void_p()
    arr = None
    if streams is not None:
        arr = (ctypes.c_void_p * 3)(*[int(s) for s in streams])
    _check(lib().mt_create_ex(ctypes.byref(cfg), device_budget_bytes, device_arena, arr, ctypes.byref(out)))
    return out


def mt_bind_host_params(ctx, host_params: int, dtype: int) -> None:
    _check(lib().mt_bind_host_params(ctx, host_params, dtype), ctx)


def mt_forward_backward(ctx, tokens: np.ndarray, labels: np.ndarray, K: int, host_grad_out: int) -> float:
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    B, S = tokens.shape
    loss = ctypes.c_float()
    _check(lib().mt_forward_backward(ctx, tokens.ctypes.data, labels.ctypes.data, B, S, K, host_grad_out,
                                     ctypes.byref(loss)), ctx)
    return loss.value


def mt_train_step(ctx, tokens: np.ndarray, labels: np.ndarray, K: int, host_grad_out: int) -> float:
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    B, S = tokens.shape
    loss = ctypes.c_float()
    _check(lib().mt_train_step(ctx, tokens.ctypes.data, labels.ctypes.data, B, S, K, host_grad_out,
                               ctypes.byref(loss)), ctx)
    return loss.value


def mt_train_step_async(ctx, tokens: np.ndarray, labels: np.ndarray, K: int, host_grad_out: int) -> float:
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    B, S = tokens.shape
    loss = ctypes.c_float()
    _check(lib().mt_train_step_async(ctx, tokens.ctypes.data, labels.ctypes.data, B, S, K, host_grad_out,
                                     ctypes.byref(loss)), ctx)
    return loss.value


def mt_optimizer_flush(ctx) -> None:
    _check(lib().mt_optimizer_flush(ctx), ctx)


def adamw_cfg(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0) -> mt_adamw_cfg:
    return mt_adamw_cfg(lr, beta1, beta2, eps, weight_decay)


def mt_bind_optimizer(ctx, opt: mt_adamw_cfg, master: int, m: int, v: int, n_threads: int = 0) -> None:
    _check(lib().mt_bind_optimizer(ctx, ctypes.byref(opt), master, m, v, n_threads), ctx)


def mt_adamw_update(cfg, opt: mt_adamw_cfg, step: int, unit_begin: int, unit_end: int, master: int, m: int, v: int,
                    grads: int, params: int, params_dtype: int, n_threads: int = 0) -> None:
    _check(lib().mt_adamw_update(ctypes.byref(cfg), ctypes.byref(opt), step, unit_begin, unit_end, master, m, v,
                                 grads, params, params_dtype, n_threads))


def mt_get_stats(ctx) -> dict:
    s = mt_stats()
    _check(lib().mt_get_stats(ctx, ctypes.byref(s)), ctx)
    out = {}
    for f, _ in mt_stats._fields_:
        v = getattr(s, f)
        out[f] = list(v) if isinstance(v, ctypes.Array) else v
    return out


MT_REPLAY_TOUCH = 1


def mt_quantize_params_fp8(cfg, src: int, src_dtype: int, dst: int, n_threads: int = 0) -> None:
    """Quantise a packed fp32/bf16 model at host address src into the FP8
    layout at dst (mt_packed_bytes(cfg, MT_FP8) bytes); see include/mt.h."""
    _check(lib().mt_quantize_params_fp8(ctypes.byref(cfg), src, src_dtype, dst, n_threads))


def mt_replay_weight_stream(ctx, K: int, flags: int = 0, max_copies: int = 4096) -> dict:
    """Copy-only replay of the step's weight stream (see include/mt.h):
    totals, the host NUMA node of the device and every copy's GB/s."""
    r = mt_replay_result()
    rates = np.zeros(max_copies, dtype=np.float32)
    _check(lib().mt_replay_weight_stream(ctx, K, flags, rates.ctypes.data, max_copies, ctypes.byref(r)), ctx)
    n = min(r.n_copies, max_copies)
    return {"n_copies": r.n_copies, "bytes": r.bytes, "ms": r.ms, "host_numa_node": r.host_numa_node,
            "touch_ms": r.touch_ms, "copy_gbs": rates[:n].astype(float).tolist()}


def mt_get_routing(ctx, n_layers: int, T: int, top_k: int) -> np.ndarray:
    """Experts chosen in the last step: [n_layers, T, top_k] int32."""
    out = np.zeros((n_layers, T, top_k), dtype=np.int32)
    _check(lib().mt_get_routing(ctx, out.ctypes.data, out.size), ctx)
    return out


def mt_set_tracing(ctx, level: int, sample: int = 16) -> None:
    _check(lib().mt_set_tracing(ctx, level, sample), ctx)


def mt_get_memory_plan(ctx) -> dict:
    s = mt_memory_plan()
    _check(lib().mt_get_memory_plan(ctx, ctypes.byref(s)), ctx)
    return {f: getattr(s, f) for f, _ in mt_memory_plan._fields_}


def mt_last_error(ctx) -> str:
    m = lib().mt_last_error(ctx)
    return m.decode() if m else ""


def mt_destroy(ctx) -> None:
    lib().mt_destroy(ctx)


def mt_host_alloc(nbytes: int) -> int:
    p = lib().mt_host_alloc(nbytes)
    if not p:
        raise MemoryError(f"mt_host_alloc({nbytes}) failed")
    return p


def mt_host_free(p: int) -> None:
    lib().mt_host_free(p)


def mt_debug_inject_fault(ctx, kind: int, nth: int) -> None:
    _check(lib().mt_debug_inject_fault(ctx, kind, nth), ctx)


def host_array(ptr: int, nbytes: int, dtype=np.uint8) -> np.ndarray:
    """numpy view of nbytes of host memory at ptr (no copy)."""
    buf = (ctypes.c_uint8 * nbytes).from_address(ptr)
    return np.frombuffer(buf, dtype=np.uint8).view(dtype)


# ---------------------------------------------------------------------------
# Convenience: a context plus its pinned host parameter and gradient buffers
# ---------------------------------------------------------------------------
@dataclass
class ModelShape:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 1e4
    norm_eps: float = 1e-5
    n_experts: int = 0  # > 0: mixture-of-experts FFN in every layer
    top_k: int = 0
    expert_ffn: int = 0


class Session:
    """One mt_ctx with pinned host params (layout of mt_tensor_offset) and grads.

    params/grads are numpy views of the pinned buffers; fill params before
    calling step(). Use close() (or a with-block) to free everything.
    """

    def __init__(self, shape: ModelShape, max_batch: int, max_seq: int, max_K: int, param_dtype: int = MT_F32,
                 device_budget: int | None = None, device_arena: int | None = None, streams=None,
                 grad_dtype: int = MT_F32):
        self.cfg = make_cfg(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                            shape.ffn_dim, shape.vocab, shape.rope_theta, shape.norm_eps, max_batch, max_seq,
                            max_K, param_dtype, shape.n_experts, shape.top_k, shape.expert_ffn, grad_dtype)
        self.grad_dtype = grad_dtype
        self._gnp = np.float32 if grad_dtype == MT_F32 else np.uint16  # bf16 gradients as bit patterns
        self.shape = shape
        self.param_dtype = param_dtype
        need = mt_required_budget(self.cfg)
        if need == 0:
            raise MtError(MT_ERR_ARG, "invalid configuration")
        self.budget = need if device_budget is None else device_budget
        self.ctx = None
        self._pp = self._gp = None
        if device_arena is not None:
            self.ctx = mt_create_ex(self.cfg, self.budget, device_arena, streams)
        else:
            self.ctx = mt_create(self.cfg, self.budget)
        self.param_bytes = mt_packed_bytes(self.cfg, param_dtype)
        self.grad_bytes = mt_packed_bytes(self.cfg, grad_dtype)
        self._pp = mt_host_alloc(self.param_bytes)
        self._gp = mt_host_alloc(self.grad_bytes)
        self.params = host_array(self._pp, self.param_bytes)
        self.grads = host_array(self._gp, self.grad_bytes, self._gnp)
        mt_bind_host_params(self.ctx, self._pp, param_dtype)

    @property
    def params_ptr(self) -> int:
        return self._pp

    @property
    def grads_ptr(self) -> int:
        return self._gp

    def offset(self, unit: int, tensor: int, dtype: int | None = None) -> tuple[int, int]:
        return mt_tensor_offset(self.cfg, self.param_dtype if dtype is None else dtype, unit, tensor)

    def step(self, tokens: np.ndarray, labels: np.ndarray, K: int) -> float:
        return mt_forward_backward(self.ctx, tokens, labels, K, self._gp)

    def bind_optimizer(self, opt: mt_adamw_cfg, master: np.ndarray, n_threads: int = 0) -> None:
        """Attach AdamW state: `master` is the fp32 packed copy of the
        parameters (mt_packed_bytes(cfg, MT_F32) bytes as float32); the
        moments start at zero. The arrays are kept by the session."""
        n = mt_packed_bytes(self.cfg, MT_F32) // 4
        self.opt_master = np.ascontiguousarray(master, dtype=np.float32).reshape(-1).copy()
        if self.opt_master.size != n:
            raise MtError(MT_ERR_ARG, "master copy has the wrong size")
        self.opt_m = np.zeros(n, np.float32)
        self.opt_v = np.zeros(n, np.float32)
        mt_bind_optimizer(self.ctx, opt, self.opt_master.ctypes.data, self.opt_m.ctypes.data, self.opt_v.ctypes.data,
                          n_threads)

    def train_step(self, tokens: np.ndarray, labels: np.ndarray, K: int) -> float:
        return mt_train_step(self.ctx, tokens, labels, K, self._gp)

    def train_step_async(self, tokens: np.ndarray, labels: np.ndarray, K: int) -> float:
        """Staleness-1 step; gradients land in two pinned buffers in turn
        (self.grads is the one this call wrote)."""
        if not hasattr(self, "_gp2"):
            self._gp2 = mt_host_alloc(self.grad_bytes)
            self._gbufs = [self._gp, self._gp2]
            self._gturn = 0
        ptr = self._gbufs[self._gturn]
        self._gturn ^= 1
        loss = mt_train_step_async(self.ctx, tokens, labels, K, ptr)
        self.grads = host_array(ptr, self.grad_bytes, self._gnp)
        return loss

    def optimizer_flush(self) -> None:
        mt_optimizer_flush(self.ctx)

    def stats(self) -> dict:
        return mt_get_stats(self.ctx)

    def replay_weight_stream(self, K: int, flags: int = 0) -> dict:
        return mt_replay_weight_stream(self.ctx, K, flags)

    def routing(self, T: int) -> np.ndarray:
        """[n_layers, T, top_k] experts chosen in the last step of T tokens."""
        return mt_get_routing(self.ctx, self.shape.n_layers, T, self.shape.top_k)

    def set_tracing(self, level: int, sample: int = 16) -> None:
        mt_set_tracing(self.ctx, level, sample)

    def memory_plan(self) -> dict:
        return mt_get_memory_plan(self.ctx)

    def close(self) -> None:
        if self.ctx is not None:
            mt_destroy(self.ctx)
            self.ctx = None
        self.params = self.grads = None
        if self._pp:
            mt_host_free(self._pp)
            self._pp = None
        if self._gp:
            mt_host_free(self._gp)
            self._gp = None
        if getattr(self, "_gp2", None):
            mt_host_free(self._gp2)
            self._gp2 = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


# ---------------------------------------------------------------------------
# Kernel-level entry points on torch CUDA tensors (pointer marshalling only)
# ---------------------------------------------------------------------------
def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream)


def mt_op_gemm(mode, epi, A, B, C, addend, M, N, K, lda, ldb, ldc, stream=None):
    _check(lib().mt_op_gemm(mode, epi, _ptr(A), _ptr(B), _ptr(C), _ptr(addend), M, N, K, lda, ldb, ldc,
                            _stream(stream)))


def mt_op_rmsnorm_fwd(x, w, y, rstd, T, h, eps, stream=None):
    _check(lib().mt_op_rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), T, h, eps, _stream(stream)))


def mt_op_rmsnorm_bwd_workspace(T, h) -> int:
    return lib().mt_op_rmsnorm_bwd_workspace(T, h)


def mt_op_rmsnorm_bwd(x, w, rstd, dy, resid, dx, dx_bf16, dw, workspace, T, h, stream=None):
    _check(lib().mt_op_rmsnorm_bwd(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dy), _ptr(resid), _ptr(dx), _ptr(dx_bf16),
                                   _ptr(dw), _ptr(workspace), T, h, _stream(stream)))


def mt_op_rmsnorm_bwd_noalloc(x, w, rstd, dy, resid, dx, dx_bf16, dw, T, h, stream=None):
    """RMSNorm backward without a workspace argument: for callers that cannot
    allocate device memory at the call site (see include/mt.h for the limit
    and the sharing rules of its fixed scratch array)."""
    _check(lib().mt_op_rmsnorm_bwd_noalloc(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dy), _ptr(resid), _ptr(dx),
                                           _ptr(dx_bf16), _ptr(dw), T, h, _stream(stream)))


def mt_op_rope(x, table, B, S, row_stride, head0, n_heads, d, theta, direction, stream=None):
    _check(lib().mt_op_rope(_ptr(x), _ptr(table), B, S, row_stride, head0, n_heads, d, theta, direction,
                            _stream(stream)))


def mt_op_gemm_rope(A, W, C, M, N, K, lda, ldb, ldc, table, S, d, theta, rope_cols, stream=None):
    _check(lib().mt_op_gemm_rope(_ptr(A), _ptr(W), _ptr(C), M, N, K, lda, ldb, ldc, _ptr(table), S, d, theta,
                                 rope_cols, _stream(stream)))


def mt_op_attention_bwd_rope(q, k, v, o, do, lse, dq, dk, dv, workspace, B, S, nq, nkv, d, ldq, ldkv, ldo, table,
                             theta, stream=None):
    _check(lib().mt_op_attention_bwd_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                          _ptr(dk), _ptr(dv), _ptr(workspace), B, S, nq, nkv, d, ldq, ldkv, ldo,
                                          _ptr(table), theta, _stream(stream)))


def mt_op_gemm_swiglu(X, W, gu, act, M, F, K, lda, ldb, u_off, stream=None):
    _check(lib().mt_op_gemm_swiglu(_ptr(X), _ptr(W), _ptr(gu), _ptr(act), M, F, K, lda, ldb, u_off,
                                   _stream(stream)))


def mt_op_gemm_swiglu_bwd(dY, Wd, gu, M, F, K, lda, ldb, u_off, stream=None):
    _check(lib().mt_op_gemm_swiglu_bwd(_ptr(dY), _ptr(Wd), _ptr(gu), M, F, K, lda, ldb, u_off, _stream(stream)))


def mt_op_attention_fwd(q, k, v, o, lse, B, S, nq, nkv, d, ldq, ldkv, ldo, stream=None):
    _check(lib().mt_op_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S, nq, nkv, d, ldq, ldkv, ldo,
                                     _stream(stream)))


def mt_op_attention_bwd_workspace(B, S, nq) -> int:
    return lib().mt_op_attention_bwd_workspace(B, S, nq)


def mt_op_attention_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, B, S, nq, nkv, d, ldq, ldkv, ldo, stream=None):
    _check(lib().mt_op_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(workspace), B, S, nq, nkv, d, ldq, ldkv, ldo, _stream(stream)))


def mt_op_swiglu_fwd(gu, act, T, F, ld, stream=None):
    _check(lib().mt_op_swiglu_fwd(_ptr(gu), _ptr(act), T, F, ld, _stream(stream)))


def mt_op_swiglu_bwd(gu, dact, T, F, ld, stream=None):
    _check(lib().mt_op_swiglu_bwd(_ptr(gu), _ptr(dact), T, F, ld, _stream(stream)))


def mt_op_moe_workspace(T, h, E, top_k, Fe) -> int:
    return lib().mt_op_moe_workspace(T, h, E, top_k, Fe)


def mt_op_moe_ffn_fwd(m, Wr, Wgu, Wd, resid, out, route, workspace, T, h, E, top_k, Fe, stream=None):
    _check(lib().mt_op_moe_ffn_fwd(_ptr(m), _ptr(Wr), _ptr(Wgu), _ptr(Wd), _ptr(resid), _ptr(out), _ptr(route),
                                   _ptr(workspace), T, h, E, top_k, Fe, _stream(stream)))


def mt_op_moe_bwd_workspace(T, h, E, top_k, Fe) -> int:
    return lib().mt_op_moe_bwd_workspace(T, h, E, top_k, Fe)


def mt_op_moe_ffn_bwd(m, Wr, Wgu, Wd, dout, dm, dWr, dWgu, dWd, route, workspace, T, h, E, top_k, Fe, stream=None):
    _check(lib().mt_op_moe_ffn_bwd(_ptr(m), _ptr(Wr), _ptr(Wgu), _ptr(Wd), _ptr(dout), _ptr(dm), _ptr(dWr),
                                   _ptr(dWgu), _ptr(dWd), _ptr(route), _ptr(workspace), T, h, E, top_k, Fe,
                                   _stream(stream)))


def mt_op_lmhead_ce_workspace(T, V, h) -> int:
    return lib().mt_op_lmhead_ce_workspace(T, V, h)


def mt_op_lmhead_ce(X, W, labels, scale, dX, dW, loss, workspace, T, V, h, stream=None):
    _check(lib().mt_op_lmhead_ce(_ptr(X), _ptr(W), _ptr(labels), scale, _ptr(dX), _ptr(dW), _ptr(loss),
                                 _ptr(workspace), T, V, h, _stream(stream)))


def mt_op_device_error() -> int:
    return lib().mt_op_device_error()
