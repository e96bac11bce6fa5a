"""CPU oracle for the affine group-quantized GEMV/GEMM and the Q8_0 / Q4_K
(and 34-byte Q8_0 / Q6_K) GEMVs.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the GPU library and imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, binary64 results), compiled with
gcc into ``liboracle.so`` next to this file; this module only marshals numpy
arrays into it. Storage dtypes are given as the strings ``"f32"``, ``"f16"``,
``"bf16"``; f16/bf16 arrays are numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_f32_to_f16_rne.argtypes = [ctypes.c_float]
        L.orc_f32_to_f16_rne.restype = ctypes.c_uint16
        L.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.orc_unpack.argtypes = [P, I, I64, I64, P]
        L.orc_pack.argtypes = [P, I, I64, I64, P]
        L.orc_quantize.argtypes = [P, I64, I64, I, I, I, P, P, P]
        L.orc_dequantize.argtypes = [P, P, P, I, I, I, I64, I64, P]
        L.orc_qmm.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, P, I64, P, P]
        L.orc_q8_0_dequant_block.argtypes = [P, P]
        L.orc_q8_0_gemv.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_q4_k_scale_min.argtypes = [P, I, ctypes.POINTER(I), ctypes.POINTER(I)]
        L.orc_q4_k_scale_min.restype = None
        L.orc_q4_k_dequant_block.argtypes = [P, P]
        L.orc_q4_k_gemv.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_quantize_x_q8.argtypes = [P, I64, P, P]
        L.orc_q8_0_block_dot_i8.argtypes = [P, P]
        L.orc_q8_0_block_dot_i8.restype = ctypes.c_int64
        L.orc_q8_0_gemv_i8.argtypes = [P, P, P, I64, I64, P, I64, P, P]
        L.orc_q8_0_34b_dequant_block.argtypes = [P, P]
        L.orc_q8_0_34b_gemv.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_q6_k_code.argtypes = [P, I]
        L.orc_q6_k_dequant_block.argtypes = [P, P]
        L.orc_q6_k_gemv.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_qmm_f32loop.argtypes = [P, P, P, P, I, I, I, I64, I64, I64, P, I64, P]
        L.orc_q8_0_gemv_f32loop.argtypes = [P, P, I64, I64, P, I64, P]
        L.orc_q4_k_gemv_f32loop.argtypes = [P, P, I64, I64, P, I64, P]
        for name in ("orc_unpack", "orc_pack", "orc_quantize", "orc_dequantize", "orc_qmm",
                     "orc_q8_0_dequant_block", "orc_q8_0_gemv", "orc_q4_k_dequant_block",
                     "orc_q4_k_gemv", "orc_q8_0_34b_dequant_block", "orc_q8_0_34b_gemv", "orc_q6_k_code",
                     "orc_q6_k_dequant_block", "orc_q6_k_gemv", "orc_qmm_f32loop", "orc_q8_0_gemv_f32loop",
                     "orc_q4_k_gemv_f32loop"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle: {what} rejected its arguments (status {rc})")


def _sb_np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


# --- storage formats --------------------------------------------------------

def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(int(h))


def bf16_to_f64(h: int) -> float:
    return lib().orc_bf16_to_f64(int(h))


def f32_to_f16_bits(f: float) -> int:
    return int(lib().orc_f32_to_f16_rne(float(np.float32(f))))


def f32_to_bf16_bits(f: float) -> int:
    return int(lib().orc_f32_to_bf16_rne(float(np.float32(f))))


_TABLES: dict = {}


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Decode an f32 array or an f16/bf16 bit-pattern array to float64."""
    a = np.ascontiguousarray(a)
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype not in _TABLES:
        f = lib().orc_f16_to_f64 if dtype == "f16" else lib().orc_bf16_to_f64
        _TABLES[dtype] = np.array([f(h) for h in range(65536)], dtype=np.float64)
    return _TABLES[dtype][a.reshape(-1).astype(np.int64)].reshape(a.shape)


# --- affine group quantization ----------------------------------------------

def quantize(W: np.ndarray, bits: int, group_size: int, dtype: str):
    """Affine group quantize W [N, K] (float32) -> (packed u32 [N, K*bits/32],
    scales [N, K/gs], biases [N, K/gs]) with scales/biases stored in `dtype`."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    packed = np.zeros((N, K * bits // 32), dtype=np.uint32)
    G = K // group_size if group_size else 0
    sd = _sb_np_dtype(dtype)
    scales = np.zeros((N, max(G, 0)), dtype=sd)
    biases = np.zeros((N, max(G, 0)), dtype=sd)
    _check(lib().orc_quantize(_p(W), N, K, bits, group_size, DTYPES[dtype], _p(packed),
                              _p(scales), _p(biases)), "quantize")
    return packed, scales, biases


def unpack(packed: np.ndarray, bits: int, K: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    N = packed.shape[0]
    q = np.zeros((N, K), dtype=np.uint8)
    _check(lib().orc_unpack(_p(packed), bits, N, K, _p(q)), "unpack")
    return q


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    packed = np.zeros((N, K * bits // 32), dtype=np.uint32)
    _check(lib().orc_pack(_p(q), bits, N, K, _p(packed)), "pack")
    return packed


def dequantize(packed, scales, biases, bits: int, group_size: int, dtype: str, K: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    scales = np.ascontiguousarray(scales)
    biases = np.ascontiguousarray(biases)
    N = packed.shape[0]
    out = np.zeros((N, K), dtype=np.float64)
    _check(lib().orc_dequantize(_p(packed), _p(scales), _p(biases), DTYPES[dtype], bits,
                                group_size, N, K, _p(out)), "dequantize")
    return out


def qmm(packed, scales, biases, x, bits: int, group_size: int, dtype: str, rows=None):
    """out[m, j] = sum_k what[rows[j], k] * x[m, k] in float64, plus the
    per-output sum of |what * x| (for the tolerance). x is [M, K] (or [K])."""
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    scales = np.ascontiguousarray(scales)
    biases = np.ascontiguousarray(biases)
    x = np.ascontiguousarray(x)
    squeeze = x.ndim == 1
    if squeeze:
        x = x.reshape(1, -1)
    M, K = x.shape
    N = packed.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros((M, nr), dtype=np.float64)
    absdot = np.zeros((M, nr), dtype=np.float64)
    _check(lib().orc_qmm(_p(packed), _p(scales), _p(biases), _p(x), DTYPES[dtype], bits,
                         group_size, M, N, K, _p(r), nr, _p(out), _p(absdot)), "qmm")
    if squeeze:
        return out[0], absdot[0]
    return out, absdot


# --- Q8_0 / Q4_K ------------------------------------------------------------

def q8_0_dequant_block(block9: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block9, dtype=np.uint32).reshape(9)
    out = np.zeros(32, dtype=np.float64)
    _check(lib().orc_q8_0_dequant_block(_p(b), _p(out)), "q8_0_dequant_block")
    return out


def q8_0_gemv(blocks: np.ndarray, x: np.ndarray, rows=None):
    """blocks u32 [N, K/32, 9], x f32 [K] -> (out f64, absdot f64)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N = blocks.shape[0]
    K = x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float64)
    absdot = np.zeros(nr, dtype=np.float64)
    _check(lib().orc_q8_0_gemv(_p(blocks), _p(x), N, K, _p(r), nr, _p(out), _p(absdot)),
           "q8_0_gemv")
    return out, absdot


def quantize_x_q8(x: np.ndarray):
    """x f32 [K] (K % 32 == 0) -> (xq int8 [K], xd f32 [K/32]): per 32-element
    block d = amax / 127 and q = rint(x / d) in binary32 (q = 0 when d = 0)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    K = x.shape[0]
    xq = np.zeros(K, dtype=np.int8)
    xd = np.zeros(K // 32, dtype=np.float32)
    _check(lib().orc_quantize_x_q8(_p(x), K, _p(xq), _p(xd)), "quantize_x_q8")
    return xq, xd


def q8_0_block_dot_i8(block9: np.ndarray, xq32: np.ndarray) -> int:
    b = np.ascontiguousarray(block9, dtype=np.uint32).reshape(9)
    q = np.ascontiguousarray(xq32, dtype=np.int8).reshape(32)
    return int(lib().orc_q8_0_block_dot_i8(_p(b), _p(q)))


def q8_0_gemv_i8(blocks: np.ndarray, xq: np.ndarray, xd: np.ndarray, rows=None):
    """blocks u32 [N, K/32, 9], xq int8 [K], xd f32 [K/32] -> (out f64, absdot f64):
    out[n] = sum_b d_w[n, b] * xd[b] * (exact integer dot of the block's codes)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint32)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    N = blocks.shape[0]
    K = xq.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float64)
    absdot = np.zeros(nr, dtype=np.float64)
    _check(lib().orc_q8_0_gemv_i8(_p(blocks), _p(xq), _p(xd), N, K, _p(r), nr, _p(out), _p(absdot)),
           "q8_0_gemv_i8")
    return out, absdot


def q4_k_scale_min(sc12, j: int):
    b = np.ascontiguousarray(np.asarray(sc12, dtype=np.uint8).reshape(12))
    sc = ctypes.c_int()
    m = ctypes.c_int()
    lib().orc_q4_k_scale_min(_p(b), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def q4_k_dequant_block(block144: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block144, dtype=np.uint8).reshape(144)
    out = np.zeros(256, dtype=np.float64)
    _check(lib().orc_q4_k_dequant_block(_p(b), _p(out)), "q4_k_dequant_block")
    return out


def q4_k_gemv(blocks: np.ndarray, x: np.ndarray, rows=None):
    """blocks u8 [N, K/256, 144], x f32 [K] -> (out f64, absdot f64)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N = blocks.shape[0]
    K = x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float64)
    absdot = np.zeros(nr, dtype=np.float64)
    _check(lib().orc_q4_k_gemv(_p(blocks), _p(x), N, K, _p(r), nr, _p(out), _p(absdot)),
           "q4_k_gemv")
    return out, absdot


def q8_0_34b_dequant_block(block34: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block34, dtype=np.uint8).reshape(34)
    out = np.zeros(32, dtype=np.float64)
    _check(lib().orc_q8_0_34b_dequant_block(_p(b), _p(out)), "q8_0_34b_dequant_block")
    return out


def q8_0_34b_gemv(blocks: np.ndarray, x: np.ndarray, rows=None):
    """blocks u8 [N, K/32, 34] (GGUF's own Q8_0 block), x f32 [K] -> (out f64, absdot f64)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N = blocks.shape[0]
    K = x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float64)
    absdot = np.zeros(nr, dtype=np.float64)
    _check(lib().orc_q8_0_34b_gemv(_p(blocks), _p(x), N, K, _p(r), nr, _p(out), _p(absdot)),
           "q8_0_34b_gemv")
    return out, absdot


def q6_k_codes(block210: np.ndarray) -> np.ndarray:
    """The 256 signed 6-bit codes (-32..31) of one Q6_K super-block."""
    b = np.ascontiguousarray(block210, dtype=np.uint8).reshape(210)
    return np.array([lib().orc_q6_k_code(_p(b), e) for e in range(256)], dtype=np.int64)


def q6_k_dequant_block(block210: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(block210, dtype=np.uint8).reshape(210)
    out = np.zeros(256, dtype=np.float64)
    _check(lib().orc_q6_k_dequant_block(_p(b), _p(out)), "q6_k_dequant_block")
    return out


def q6_k_gemv(blocks: np.ndarray, x: np.ndarray, rows=None):
    """blocks u8 [N, K/256, 210], x f32 [K] -> (out f64, absdot f64)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N = blocks.shape[0]
    K = x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float64)
    absdot = np.zeros(nr, dtype=np.float64)
    _check(lib().orc_q6_k_gemv(_p(blocks), _p(x), N, K, _p(r), nr, _p(out), _p(absdot)), "q6_k_gemv")
    return out, absdot


# Plain binary32 loops: a CPU timing baseline (the "reasonable CPU" number
# timed beside the oracle), not a reference; no test takes them as expected.

def qmm_f32loop(packed, scales, biases, x, bits: int, group_size: int, dtype: str, rows=None):
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    scales = np.ascontiguousarray(scales)
    biases = np.ascontiguousarray(biases)
    x = np.ascontiguousarray(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    M, K = x.shape
    N = packed.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros((M, nr), dtype=np.float32)
    _check(lib().orc_qmm_f32loop(_p(packed), _p(scales), _p(biases), _p(x), DTYPES[dtype], bits, group_size, M, N,
                                 K, _p(r), nr, _p(out)), "qmm_f32loop")
    return out


def q8_0_gemv_f32loop(blocks, x, rows=None):
    blocks = np.ascontiguousarray(blocks, dtype=np.uint32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N, K = blocks.shape[0], x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float32)
    _check(lib().orc_q8_0_gemv_f32loop(_p(blocks), _p(x), N, K, _p(r), nr, _p(out)), "q8_0_gemv_f32loop")
    return out


def q4_k_gemv_f32loop(blocks, x, rows=None):
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    N, K = blocks.shape[0], x.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = N if r is None else r.shape[0]
    out = np.zeros(nr, dtype=np.float32)
    _check(lib().orc_q4_k_gemv_f32loop(_p(blocks), _p(x), N, K, _p(r), nr, _p(out)), "q4_k_gemv_f32loop")
    return out
