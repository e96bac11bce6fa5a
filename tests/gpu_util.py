"""Helpers of the GPU parity tests: move oracle-format numpy arrays to and from
CUDA tensors, and build seeded affine test problems with the oracle."""
import numpy as np
import torch

import oracle
import synth

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy storage array -> CUDA tensor (uint16 bits become bf16/f16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16).copy()).view(TORCH_DTYPE[dtype])
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32).copy())
    else:
        t = torch.from_numpy(a.copy())
    return t.cuda()


def to_host_f64(t: torch.Tensor, dtype: str) -> np.ndarray:
    """CUDA tensor of dtype T -> float64 values (decoded by the oracle's tables)."""
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy().astype(np.float64)
    return oracle.to_f64(t.view(torch.int16).numpy().view(np.uint16), dtype)


def affine_problem(N: int, K: int, M: int, bits: int, gs: int, dtype: str, seed: int):
    """Seeded problem: W ~ N(0, 0.02) quantized by the ORACLE, x ~ N(0, 1) in T."""
    W = synth.affine_weights(N, K, seed)
    packed, s, b = oracle.quantize(W, bits, gs, dtype)
    x = synth.activations(M, K, dtype, seed + 7919)
    return W, packed, s, b, x


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    r = np.random.default_rng(seed)
    rows = set([0, N - 1]) | set(r.integers(0, N, size=count).tolist())
    return np.array(sorted(rows), dtype=np.int64)
