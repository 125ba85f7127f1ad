"""Seeded synthetic inputs (weights, token ids) for the tests and the benchmark.

Counter-based SplitMix64 bits and Box-Muller normals, written in C
(``seedgen.c``) so that filling billions of parameters takes seconds. The
module holds none of the training step's arithmetic; the same arrays are fed
to the CUDA library and to the CPU oracle.

Input recipe (the workloads of the pages, with random weights in place of
pretrained checkpoints): every matrix ~ N(0, 0.02); RMSNorm gains = 1.0;
tokens uniform in [0, V); each sequence draws S+1 ids, the first S are the
inputs and the last S the next-token labels.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libseedgen.so")
_lib = None


def build_command() -> list[str]:
    return ["gcc", "-O3", "-fPIC", "-shared", "-std=c11", "-o", _LIB_PATH,
            os.path.join(_HERE, "seedgen.c"), "-lm", "-lpthread"]


def build() -> None:
    subprocess.run(build_command(), check=True)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, vp, dbl, i32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int32
        L.seedgen_normal_f32.argtypes = [vp, u64, u64, u64, dbl, dbl, ctypes.c_int]
        L.seedgen_normal_bf16.argtypes = [vp, u64, u64, u64, dbl, dbl, ctypes.c_int]
        L.seedgen_fill_f32.argtypes = [vp, u64, ctypes.c_float]
        L.seedgen_fill_bf16.argtypes = [vp, u64, ctypes.c_float]
        L.seedgen_tokens.argtypes = [vp, u64, u64, u64, i32]
        L.seedgen_bits.argtypes = [vp, u64, u64, u64]
        for f in (L.seedgen_normal_f32, L.seedgen_normal_bf16, L.seedgen_fill_f32, L.seedgen_fill_bf16,
                  L.seedgen_tokens, L.seedgen_bits):
            f.restype = None
        _lib = L
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_into(addr: int, n: int, bf16: bool, seed: int, stream: int, std: float = 0.02,
                mean: float = 0.0) -> None:
    """Write n normal deviates (mean, std) to host address addr."""
    f = lib().seedgen_normal_bf16 if bf16 else lib().seedgen_normal_f32
    f(addr, n, seed, stream, mean, std, _threads())


def fill_into(addr: int, n: int, bf16: bool, value: float) -> None:
    f = lib().seedgen_fill_bf16 if bf16 else lib().seedgen_fill_f32
    f(addr, n, value)


def normal(n: int, seed: int, stream: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    normal_into(out.ctypes.data, n, False, seed, stream, std, mean)
    return out


def bits(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().seedgen_bits(out.ctypes.data, n, seed, stream)
    return out


def tokens_and_labels(B: int, S: int, V: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """Per sequence draw S+1 ids: inputs = ids[0:S], labels = ids[1:S+1]."""
    ids = np.empty(B * (S + 1), dtype=np.int32)
    lib().seedgen_tokens(ids.ctypes.data, ids.size, seed, 0, V)
    ids = ids.reshape(B, S + 1)
    return np.ascontiguousarray(ids[:, :S]), np.ascontiguousarray(ids[:, 1:])


def fill_packed_params(addr: int, offsets, bf16: bool, seed: int, std: float = 0.02) -> None:
    """Fill a packed parameter block.

    offsets: iterable of (unit, tensor, byte_offset, n_elems, is_gain). Gains
    (RMSNorm weights) are set to 1.0, every matrix to N(0, std) drawn from its
    own stream (unit * 64 + tensor), so values do not depend on the layout.
    """
    for unit, tensor, off, n, is_gain in offsets:
        if is_gain:
            fill_into(addr + off, n, bf16, 1.0)
        else:
            normal_into(addr + off, n, bf16, seed, 1 + unit * 64 + tensor, std)
