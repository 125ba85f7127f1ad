"""Helpers for the GPU tests: build/load the CUDA library once, move
bf16-rounded numpy arrays to the device and back."""
from __future__ import annotations

import numpy as np
import pytest

from tests.common import bf16_bits_to_f32, f32_to_bf16_bits


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_streamed_gb300 as mt
    mt.build()
    mt.lib()
    return torch, mt


def to_dev_bf16(torch, x: np.ndarray):
    """(device bf16 tensor, the exact fp32 values it holds)."""
    bits = f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    t = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return t, bf16_bits_to_f32(bits).reshape(np.shape(x))


def to_dev_f32(torch, x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def from_dev(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.float().cpu().numpy()
