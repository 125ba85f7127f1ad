"""Shared test workloads and input builders (seeded, synthetic).

Workloads follow the decoder configurations the method is exercised on:
  tiny      2 layers, hidden 64, 4 heads x 16 (MHA), FFN 172, vocab 256, seq 32, batch 2, fp32 host
  tiny_gqa  the same with 2 KV heads
  small     8 layers, hidden 1024, 16 x 64, FFN 2816, vocab 32000, seq 2048, batch 4, fp32 host master
  llama8b   32 layers, hidden 4096, 32 q / 8 kv heads x 128, FFN 14336, vocab 128256, theta 5e5,
            seq 4096, batch 2, bf16 host weights
Weights N(0, 0.02) from a seed, RMSNorm gains 1.0, tokens uniform in [0, V),
labels = next token.
"""
from __future__ import annotations

import numpy as np

import oracle
import seedgen

TINY = oracle.Config(n_layers=2, hidden=64, n_heads=4, n_kv_heads=4, head_dim=16, ffn_dim=172, vocab=256,
                     rope_theta=1e4, norm_eps=1e-5)
TINY_GQA = oracle.Config(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=172, vocab=256,
                         rope_theta=1e4, norm_eps=1e-5)
SMALL = oracle.Config(n_layers=8, hidden=1024, n_heads=16, n_kv_heads=16, head_dim=64, ffn_dim=2816, vocab=32000,
                      rope_theta=1e4, norm_eps=1e-5)
LLAMA8B = oracle.Config(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=14336,
                        vocab=128256, rope_theta=5e5, norm_eps=1e-5)


# Mixture-of-experts workloads. The Qwen3-235B-style layer: hidden 4096, 64 q / 4 kv heads x 128, 128 experts,
# top-8, expert FFN 1536, vocab 151936 (RoPE theta 1e6 and RMSNorm eps 1e-6 as in Qwen3; the pages give neither).
QWEN3_MOE = oracle.Config(n_layers=8, hidden=4096, n_heads=64, n_kv_heads=4, head_dim=128, ffn_dim=0, vocab=151936,
                          rope_theta=1e6, norm_eps=1e-6, n_experts=128, top_k=8, expert_ffn=1536)
TINY_MOE = oracle.Config(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=0, vocab=256,
                         rope_theta=1e4, norm_eps=1e-5, n_experts=8, top_k=2, expert_ffn=32)


def with_layers(cfg: oracle.Config, n_layers: int) -> oracle.Config:
    d = dict(cfg.__dict__)
    d["n_layers"] = n_layers
    return oracle.Config(**d)


def make_params(cfg: oracle.Config, seed: int, bf16: bool = False, std: float = 0.02) -> np.ndarray:
    """Packed host parameter block (oracle's layout), uint8 array."""
    buf = np.zeros(oracle.packed_bytes(cfg, bf16), dtype=np.uint8)
    offs = []
    for unit, t, name, shape, is_gain in oracle.tensor_list(cfg):
        off, nb = oracle.tensor_offset(cfg, unit, t, bf16)
        offs.append((unit, t, off, int(np.prod(shape)), is_gain))
    seedgen.fill_packed_params(buf.ctypes.data, offs, bf16, seed, std)
    return buf


def make_tokens(cfg: oracle.Config, B: int, S: int, seed: int):
    return seedgen.tokens_and_labels(B, S, cfg.vocab, seed)


def params_f64(cfg: oracle.Config, packed_f32: np.ndarray) -> np.ndarray:
    return packed_f32.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))
