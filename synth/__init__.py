"""Seeded synthetic inputs, shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays them out in the input formats;
it holds none of the arithmetic of the method (no quantization, no decoding,
no products). Both the CPU oracle and the GPU library consume exactly the
bytes it returns.

Distributions follow the workloads the pages describe:
  * affine weights W ~ N(0, 0.02) in float32, [N, K] (quantized afterwards);
  * activations x ~ N(0, 1), stored in the activation dtype (bf16/f16 rounded
    to nearest-even from float32, or float32);
  * Q8_0 blocks: int8 codes uniform in [-127, 127], scale d ~ U(1e-4, 1e-2)
    stored as f16 in the low half of word 0 (high half zero), 9 words/block;
  * Q4_K super-blocks: d, dmin ~ U(1e-4, 1e-2) stored as f16, 12 scale bytes
    and 128 qs bytes uniform random, 144 bytes/block.
  * GGUF's own 34-byte Q8_0 blocks: the Q8_0 distributions above, f16 scale in
    bytes 0..1, the 32 codes in bytes 2..33.
  * Q6_K super-blocks: 128 ql and 64 qh bytes uniform random, 16 int8 scales
    uniform in [-128, 127], d ~ U(1e-4, 1e-2) stored as f16 in bytes 208..209,
    210 bytes/block.

f16/bf16 arrays are returned as numpy uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np
import torch


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def affine_weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """float32 [N, K] ~ N(0, std)."""
    return (rng(seed).standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(
        np.float32)


def _round_to_storage(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32))
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(M: int, K: int, dtype: str, seed: int) -> np.ndarray:
    """x [M, K] ~ N(0, 1) in the storage dtype (uint16 bits for bf16/f16)."""
    x = rng(seed).standard_normal((M, K), dtype=np.float32)
    return _round_to_storage(x, dtype)


def q8_0_blocks(N: int, K: int, seed: int) -> np.ndarray:
    """uint32 [N, K/32, 9] packed Q8_0 blocks."""
    assert K % 32 == 0
    r = rng(seed)
    nb = K // 32
    d = r.uniform(1e-4, 1e-2, size=(N, nb)).astype(np.float32).astype(np.float16)
    q = r.integers(-127, 128, size=(N, nb, 32), dtype=np.int64).astype(np.int8)
    blocks = np.zeros((N, nb, 9), dtype=np.uint32)
    blocks[:, :, 0] = d.view(np.uint16).astype(np.uint32)
    blocks[:, :, 1:] = q.view(np.uint8).reshape(N, nb, 32).copy().view("<u4").reshape(N, nb, 8)
    return blocks


def q4_k_blocks(N: int, K: int, seed: int) -> np.ndarray:
    """uint8 [N, K/256, 144] Q4_K super-blocks."""
    assert K % 256 == 0
    r = rng(seed)
    nb = K // 256
    blocks = r.integers(0, 256, size=(N, nb, 144), dtype=np.int64).astype(np.uint8)
    d = r.uniform(1e-4, 1e-2, size=(N, nb)).astype(np.float32).astype(np.float16)
    dmin = r.uniform(1e-4, 1e-2, size=(N, nb)).astype(np.float32).astype(np.float16)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:4] = dmin.view(np.uint8).reshape(N, nb, 2)
    return blocks


def q8_0_34b_blocks(N: int, K: int, seed: int) -> np.ndarray:
    """uint8 [N, K/32, 34] GGUF Q8_0 blocks (f16 scale, then 32 int8 codes)."""
    assert K % 32 == 0
    r = rng(seed)
    nb = K // 32
    d = r.uniform(1e-4, 1e-2, size=(N, nb)).astype(np.float32).astype(np.float16)
    q = r.integers(-127, 128, size=(N, nb, 32), dtype=np.int64).astype(np.int8)
    blocks = np.empty((N, nb, 34), dtype=np.uint8)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = q.view(np.uint8)
    return blocks


def q6_k_blocks(N: int, K: int, seed: int) -> np.ndarray:
    """uint8 [N, K/256, 210] Q6_K super-blocks."""
    assert K % 256 == 0
    r = rng(seed)
    nb = K // 256
    blocks = r.integers(0, 256, size=(N, nb, 210), dtype=np.int64).astype(np.uint8)
    d = r.uniform(1e-4, 1e-2, size=(N, nb)).astype(np.float32).astype(np.float16)
    blocks[:, :, 208:210] = d.view(np.uint8).reshape(N, nb, 2)
    return blocks


def f32_vector(K: int, seed: int) -> np.ndarray:
    """float32 [K] ~ N(0, 1) (activations of the block-quantized GEMVs)."""
    return rng(seed).standard_normal(K, dtype=np.float32)
