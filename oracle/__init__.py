"""CPU oracle: the plain, slow, single-threaded definition of one training step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with ``layer_streamed_gb300`` and never imports it: the packed layout is
computed by ``oracle.cpp`` from its own restatement of the definition.

``oracle.cpp`` follows "MegaTrain: Full Precision Training of 100B+ Parameter
Large Language Models on a Single GPU", section 方法步骤详情 (stages 1-3: streamed
forward, loss anchor, backward), computing the same function with every
activation materialised and no recompute.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build_command() -> list[str]:
    # Portable flags only: the same source builds on x86-64 and aarch64.
    return ["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-o", _LIB_PATH,
            os.path.join(_HERE, "oracle.cpp")]


def build() -> None:
    subprocess.run(build_command(), check=True)


class _Cfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_double), ("norm_eps", ctypes.c_double),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("expert_ffn", ctypes.c_int32)]


@dataclass(frozen=True)
class Config:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 1e4
    norm_eps: float = 1e-5
    n_experts: int = 0   # > 0: every layer's FFN is a mixture of experts
    top_k: int = 0
    expert_ffn: int = 0

    def c(self) -> _Cfg:
        return _Cfg(self.n_layers, self.hidden, self.n_heads, self.n_kv_heads, self.head_dim, self.ffn_dim,
                    self.vocab, self.rope_theta, self.norm_eps, self.n_experts, self.top_k, self.expert_ffn)


# Tensor names inside a unit, in packed order.
LAYER_TENSORS = ("w_attn_norm", "wq", "wk", "wv", "wo", "w_ffn_norm", "wg", "wu", "wd")
MOE_LAYER_TENSORS = ("w_attn_norm", "wq", "wk", "wv", "wo", "w_ffn_norm", "w_router", "w_experts_gu",
                     "w_experts_down")
HEAD_TENSORS = ("w_final_norm", "w_out")


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER
        vp, i32, dbl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        L.oracle_packed_bytes.argtypes = [P(_Cfg), i32]
        L.oracle_packed_bytes.restype = sz
        L.oracle_tensor_offset.argtypes = [P(_Cfg), i32, i32, i32, P(sz), P(sz)]
        L.oracle_forward_backward_f32.argtypes = [P(_Cfg), vp, i32, vp, vp, i32, i32, dbl, vp, P(dbl), vp, vp, vp, vp]
        L.oracle_forward_backward_f64.argtypes = [P(_Cfg), vp, vp, vp, i32, i32, dbl, vp, P(dbl), vp, vp]
        L.oracle_matmul.argtypes = [i32, i32, vp, vp, vp, i32, i32, i32]
        L.oracle_matmul_sampled.argtypes = [i32, vp, vp, i32, i32, i32, vp, vp, ctypes.c_int64, vp]
        L.oracle_rmsnorm_fwd.argtypes = [i32, vp, vp, i32, i32, dbl, vp, vp]
        L.oracle_rmsnorm_bwd.argtypes = [i32, vp, vp, vp, i32, i32, dbl, vp, vp]
        L.oracle_rope.argtypes = [i32, vp, i32, i32, i32, i32, dbl, i32]
        L.oracle_attention.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_swiglu.argtypes = [i32, vp, vp, vp, sz, vp, vp, vp]
        L.oracle_cross_entropy.argtypes = [i32, vp, vp, i32, i32, dbl, P(dbl), vp]
        L.oracle_moe_ffn.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def packed_bytes(cfg: Config, bf16: bool = False) -> int:
    c = cfg.c()
    return lib().oracle_packed_bytes(ctypes.byref(c), 1 if bf16 else 0)


def tensor_offset(cfg: Config, unit: int, tensor: int, bf16: bool = False) -> tuple[int, int]:
    """(byte offset, byte size) of tensor `tensor` of unit `unit`."""
    c = cfg.c()
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    rc = lib().oracle_tensor_offset(ctypes.byref(c), 1 if bf16 else 0, unit, tensor, ctypes.byref(off),
                                    ctypes.byref(nb))
    if rc != 0:
        raise IndexError((unit, tensor))
    return off.value, nb.value


def tensor_list(cfg: Config):
    """[(unit, tensor, name, shape, is_gain)] in packed order."""
    h, qd, kd, F, V = cfg.hidden, cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.ffn_dim, cfg.vocab
    out = [(0, 0, "embed", (V, h), False)]
    shapes = [(h,), (qd, h), (kd, h), (kd, h), (h, qd), (h,), (F, h), (F, h), (h, F)]
    names = LAYER_TENSORS
    if cfg.n_experts:
        E, Fe = cfg.n_experts, cfg.expert_ffn
        shapes[6:] = [(E, h), (E, 2 * Fe, h), (E, h, Fe)]
        names = MOE_LAYER_TENSORS
    for l in range(cfg.n_layers):
        for t, (name, shp) in enumerate(zip(names, shapes)):
            out.append((l + 1, t, f"layer{l}.{name}", shp, name.endswith("norm")))
    out.append((cfg.n_layers + 1, 0, "w_final_norm", (h,), True))
    out.append((cfg.n_layers + 1, 1, "w_out", (V, h), False))
    return out


def unpack(cfg: Config, packed: np.ndarray, bf16: bool = False) -> dict[str, np.ndarray]:
    """Split a packed byte/element buffer into named views (fp32 or bf16 bits)."""
    raw = packed.view(np.uint8)
    out = {}
    for unit, t, name, shape, _ in tensor_list(cfg):
        off, nb = tensor_offset(cfg, unit, t, bf16)
        out[name] = raw[off:off + nb].view(np.uint16 if bf16 else np.float32).reshape(shape)
    return out


def _routing(cfg: Config, T: int, route_in, want_route: bool):
    """(route_in array or None, route_out array or None), each [L, T, top_k] int32."""
    shape = (cfg.n_layers, T, cfg.top_k)
    rin = None
    if route_in is not None:
        rin = np.ascontiguousarray(route_in, dtype=np.int32)
        if rin.shape != shape:
            raise ValueError(f"route_in must have shape {shape}")
    rout = np.zeros(shape, dtype=np.int32) if want_route else None
    return rin, rout


def forward_backward(cfg: Config, params: np.ndarray, tokens: np.ndarray, labels: np.ndarray, bf16: bool = False,
                     scale: float | None = None, token_losses: bool = False, route_in=None,
                     want_route: bool = False, want_logits: bool = False):
    """fp32 step. params: packed bytes (fp32 or bf16 layout).

    Returns (loss, packed fp32 grads), plus the per-position CE terms [B, S]
    when token_losses is set, plus the experts selected in every layer
    ([L, B*S, top_k]) when want_route is set, plus every layer's router
    logits ([L, B*S, n_experts]) when want_logits is set. route_in forces
    that selection (mixture-of-experts layers only)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    B, S = tokens.shape
    if scale is None:
        scale = 1.0 / (B * S)
    grads = np.zeros(packed_bytes(cfg, False) // 4, dtype=np.float32)
    loss = ctypes.c_double()
    c = cfg.c()
    tl = np.empty((B, S), dtype=np.float32) if token_losses else None
    rin, rout = _routing(cfg, B * S, route_in, want_route)
    logits = np.zeros((cfg.n_layers, B * S, cfg.n_experts), dtype=np.float32) if want_logits else None
    rc = lib().oracle_forward_backward_f32(ctypes.byref(c), _p(params), 1 if bf16 else 0, _p(tokens), _p(labels),
                                           B, S, scale, _p(grads), ctypes.byref(loss), _p(tl), _p(rin), _p(rout),
                                           _p(logits))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    out = (loss.value, grads)
    if token_losses:
        out += (tl,)
    if want_route:
        out += (rout,)
    if want_logits:
        out += (logits,)
    return out


def forward_backward_f64(cfg: Config, params64: np.ndarray, tokens: np.ndarray, labels: np.ndarray,
                         scale: float | None = None, route_in=None, want_route: bool = False):
    """fp64 step; params64 are doubles at the fp32 layout's element offsets."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    B, S = tokens.shape
    if scale is None:
        scale = 1.0 / (B * S)
    params64 = np.ascontiguousarray(params64, dtype=np.float64)
    grads = np.zeros(packed_bytes(cfg, False) // 4, dtype=np.float64)
    loss = ctypes.c_double()
    c = cfg.c()
    rin, rout = _routing(cfg, B * S, route_in, want_route)
    rc = lib().oracle_forward_backward_f64(ctypes.byref(c), _p(params64), _p(tokens), _p(labels), B, S, scale,
                                           _p(grads), ctypes.byref(loss), _p(rin), _p(rout))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    if want_route:
        return loss.value, grads, rout
    return loss.value, grads


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def matmul(mode: str, A: np.ndarray, B: np.ndarray, f64: bool = True) -> np.ndarray:
    """mode 'nt': A[M,K] B[N,K]^T; 'nn': A[M,K] B[K,N]; 'tn': A[K,M]^T B[K,N]."""
    A, B = _f32(A), _f32(B)
    if mode == "nt":
        (M, K), N = A.shape, B.shape[0]
    elif mode == "nn":
        (M, K), N = A.shape, B.shape[1]
    else:
        (K, M), N = A.shape, B.shape[1]
    Y = np.empty((M, N), dtype=np.float32)
    lib().oracle_matmul({"nt": 0, "nn": 1, "tn": 2}[mode], int(f64), _p(A), _p(B), _p(Y), M, N, K)
    return Y


def matmul_sampled(mode: str, A: np.ndarray, B: np.ndarray, rows, cols) -> np.ndarray:
    A, B = _f32(A), _f32(B)
    if mode == "nt":
        (M, K), N = A.shape, B.shape[0]
    elif mode == "nn":
        (M, K), N = A.shape, B.shape[1]
    else:
        (K, M), N = A.shape, B.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.size, dtype=np.float64)
    rc = lib().oracle_matmul_sampled({"nt": 0, "nn": 1, "tn": 2}[mode], _p(A), _p(B), M, N, K, _p(rows), _p(cols),
                                     rows.size, _p(out))
    if rc != 0:
        raise IndexError("sample out of range")
    return out


def rmsnorm_fwd(x, w, eps, f64=True):
    x, w = _f32(x), _f32(w)
    T, h = x.shape
    y = np.empty_like(x)
    r = np.empty(T, dtype=np.float32)
    lib().oracle_rmsnorm_fwd(int(f64), _p(x), _p(w), T, h, eps, _p(y), _p(r))
    return y, r


def rmsnorm_bwd(x, w, dy, eps, f64=True):
    x, w, dy = _f32(x), _f32(w), _f32(dy)
    T, h = x.shape
    dx = np.empty_like(x)
    dw = np.empty(h, dtype=np.float32)
    lib().oracle_rmsnorm_bwd(int(f64), _p(x), _p(w), _p(dy), T, h, eps, _p(dx), _p(dw))
    return dx, dw


def rope(x, theta, direction=1, f64=True):
    """x [B, S, nh, d] -> rotated copy."""
    y = _f32(x).copy()
    B, S, nh, d = y.shape
    rc = lib().oracle_rope(int(f64), _p(y), B, S, nh, d, theta, direction)
    if rc != 0:
        raise ValueError("bad rope arguments")
    return y


def attention(q, k, v, dout=None, f64=True):
    """q [B,S,nq,d], k/v [B,S,nkv,d] -> (o, lse [B,nq,S], dq, dk, dv)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, S, nq, d = q.shape
    nkv = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, nq, S), dtype=np.float32)
    dq = dk = dv = None
    if dout is not None:
        dout = _f32(dout)
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    rc = lib().oracle_attention(int(f64), _p(q), _p(k), _p(v), _p(dout), B, S, nq, nkv, d, _p(o), _p(lse), _p(dq),
                                _p(dk), _p(dv))
    if rc != 0:
        raise ValueError("bad attention arguments")
    return o, lse, dq, dk, dv


def swiglu(g, u, da=None, f64=True):
    g, u = _f32(g), _f32(u)
    a = np.empty_like(g)
    dg = du = None
    if da is not None:
        da = _f32(da)
        dg, du = np.empty_like(g), np.empty_like(g)
    lib().oracle_swiglu(int(f64), _p(g), _p(u), _p(da), g.size, _p(a), _p(dg), _p(du))
    return a, dg, du


def cross_entropy(z, labels, scale=None, want_grad=True, f64=True):
    z = _f32(z)
    T, V = z.shape
    labels = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
    if scale is None:
        scale = 1.0 / T
    loss = ctypes.c_double()
    dz = np.empty_like(z) if want_grad else None
    rc = lib().oracle_cross_entropy(int(f64), _p(z), _p(labels), T, V, scale, ctypes.byref(loss), _p(dz))
    if rc != 0:
        raise ValueError("label out of range")
    return loss.value, dz


def moe_ffn(m, w_router, w_experts_gu, w_experts_down, top_k, dout=None, route_in=None, f64=True):
    """Mixture-of-experts FFN on m [T, h]: w_router [E, h], w_experts_gu
    [E, 2Fe, h] (gate rows, then up rows), w_experts_down [E, h, Fe].

    Returns (out [T, h], route [T, top_k], dm, dw_router, dw_experts_gu,
    dw_experts_down); the gradients are None unless dout is given."""
    m, wr, wgu, wd = _f32(m), _f32(w_router), _f32(w_experts_gu), _f32(w_experts_down)
    T, h = m.shape
    E, Fe = wr.shape[0], wd.shape[2]
    out = np.empty_like(m)
    route = np.zeros((T, top_k), dtype=np.int32)
    rin = None if route_in is None else np.ascontiguousarray(route_in, dtype=np.int32).reshape(T, top_k)
    dm = dwr = dwgu = dwd = None
    if dout is not None:
        dout = _f32(dout)
        dm, dwr, dwgu, dwd = np.empty_like(m), np.empty_like(wr), np.empty_like(wgu), np.empty_like(wd)
    rc = lib().oracle_moe_ffn(int(f64), _p(m), _p(wr), _p(wgu), _p(wd), T, h, E, top_k, Fe, _p(rin), _p(route),
                              _p(out), _p(dout), _p(dm), _p(dwr), _p(dwgu), _p(dwd))
    if rc != 0:
        raise ValueError("bad mixture-of-experts arguments")
    return out, route, dm, dwr, dwgu, dwd
