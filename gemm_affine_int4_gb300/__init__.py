"""Python binding of libgai4.so, the GB300 (sm_103a) affine group-quantized
GEMV / small-M GEMM library. Argument marshalling only: every function here
calls the C entry point of the same name (include/gai4.h) with device pointers
of PyTorch tensors and the current CUDA stream; all arithmetic runs in the
library's CUDA kernels. There is no fallback: if libgai4.so is not built, or a
tensor is not on a CUDA device, the call raises.

Tensor conventions (row-major, contiguous, on one CUDA device):
  w_packed  int32/uint32 [N, K*bits/32]      scales, biases  T [N, K/group_size]
  x         T [K] (qmv) or [M, K] (qmm_t)    out             T [N] or [M, N]
with T = torch.bfloat16, torch.float16 or torch.float32.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgai4.so")

GAI4_OK = 0
GAI4_ERR_INVALID_ARG = 1
GAI4_ERR_UNSUPPORTED = 2
GAI4_ERR_MISALIGNED = 3
GAI4_ERR_WORKSPACE = 4
GAI4_ERR_CUDA = 5
GAI4_ERR_TIMEOUT = 6

_DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# name -> (argtypes, restype) of every exported entry point
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
SIGNATURES = {
    "gai4_version": ([], _I),
    "gai4_status_string": ([_I], ctypes.c_char_p),
    "gai4_quantize": ([_P, _P, _P, _P, _I, _I, _I, _I64, _I64, _P], _I),
    "gai4_unpack": ([_P, _P, _I, _I64, _I64, _P], _I),
    "gai4_dequantize": ([_P, _P, _P, _P, _I, _I, _I, _I64, _I64, _P], _I),
    "gai4_qmv": ([_P, _P, _P, _P, _P, _I, _I, _I, _I64, _I64, _P], _I),
    "gai4_qmm_t": ([_P, _P, _P, _P, _P, _I, _I, _I, _I64, _I64, _I64, _I, _P, ctypes.c_size_t, _P], _I),
    "gai4_qmm_t_workspace_bytes": ([_I64, _I64, _I64, _I, _I, _I, _I], ctypes.c_size_t),
    "gai4_qmm_t_plan": ([_I64, _I64, _I64, _I, _I, _I, _I, ctypes.c_size_t, ctypes.POINTER(_I),
                         ctypes.POINTER(_I)], _I),
    "gai4_qmm_t_noalloc": ([_P, _P, _P, _P, _P, _I, _I, _I, _I64, _I64, _I64, _I, _P], _I),
    "gai4_qmm_t_batched": ([_P, _P, _P, _I, _P, _I64, _I64, _P, _I, _I, _I, _I64, _I64, _I64, _I64, _I, _P,
                            ctypes.c_size_t, _P], _I),
    "gai4_qmm_t_batched_workspace_bytes": ([_I64, _I64, _I64, _I64, _I, _I, _I, _I], ctypes.c_size_t),
    "gai4_q8_0_gemv": ([_P, _P, _P, _I64, _I64, _P], _I),
    "gai4_q4_k_gemv": ([_P, _P, _P, _I64, _I64, _P], _I),
    "gai4_q4_k_dequantize": ([_P, _P, _I64, _I64, _I, _P], _I),
    "gai4_quantize_x_q8": ([_P, _P, _P, _I64, _P], _I),
    "gai4_q8_0_gemv_i8": ([_P, _P, _P, _P, _I64, _I64, _P], _I),
    "gai4_last_device_status": ([_P], _I),
    "gai4_check_bounded_wait": ([_I, _I64, _P, _P], _I),
    "gai4_q8_0_34b_gemv": ([_P, _P, _P, _I64, _I64, _P], _I),
    "gai4_q6_k_gemv": ([_P, _P, _P, _I64, _I64, _P], _I),
}


class Gai4Error(RuntimeError):
    def __init__(self, name: str, status: int):
        self.status = status
        super().__init__(f"{name}: {gai4_status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libgai4.so (built in-tree by __graft_entry__.build() or
    `python -m gemm_affine_int4_gb300.build`)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m gemm_affine_int4_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (argtypes, restype) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("gai4: tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("gai4: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_strided(t: torch.Tensor):
    """Device address of a strided view's first element (the strides travel
    as separate arguments)."""
    if not t.is_cuda:
        raise ValueError("gai4: tensors must live on a CUDA device")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(name: str, st: int):
    if st != GAI4_OK:
        raise Gai4Error(name, st)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE:
        raise ValueError(f"gai4: unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def gai4_version() -> int:
    return lib().gai4_version()


def gai4_status_string(status: int) -> str:
    return lib().gai4_status_string(int(status)).decode()


def gai4_quantize(w: torch.Tensor, bits: int = 4, group_size: int = 64, dtype=torch.bfloat16,
                  w_packed=None, scales=None, biases=None, stream=None):
    """Affine group quantize w [N, K] float32 -> (w_packed, scales, biases)."""
    N, K = w.shape
    if w_packed is None:
        w_packed = torch.empty((N, K * bits // 32), dtype=torch.int32, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // group_size), dtype=dtype, device=w.device)
    if biases is None:
        biases = torch.empty((N, K // group_size), dtype=dtype, device=w.device)
    _check("gai4_quantize", lib().gai4_quantize(_ptr(w), _ptr(w_packed), _ptr(scales), _ptr(biases),
                                                _dtype(scales), bits, group_size, N, K, _stream(stream)))
    return w_packed, scales, biases


def gai4_unpack(w_packed: torch.Tensor, bits: int, K: int, q_out=None, stream=None) -> torch.Tensor:
    N = w_packed.shape[0]
    if q_out is None:
        q_out = torch.empty((N, K), dtype=torch.uint8, device=w_packed.device)
    _check("gai4_unpack", lib().gai4_unpack(_ptr(w_packed), _ptr(q_out), bits, N, K, _stream(stream)))
    return q_out


def gai4_dequantize(w_packed, scales, biases, bits: int = 4, group_size: int = 64, out=None, stream=None):
    N = w_packed.shape[0]
    K = w_packed.shape[1] * 32 // bits
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=w_packed.device)
    _check("gai4_dequantize", lib().gai4_dequantize(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(out),
                                                    _dtype(scales), bits, group_size, N, K, _stream(stream)))
    return out


def gai4_qmv(w_packed, scales, biases, x, out=None, bits: int = 4, group_size: int = 64, stream=None):
    """out[n] = sum_k (s q + b)[n, k] x[k]."""
    N = w_packed.shape[0]
    K = x.shape[-1]
    if out is None:
        out = torch.empty((N,), dtype=x.dtype, device=x.device)
    _check("gai4_qmv", lib().gai4_qmv(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(x), _ptr(out),
                                      _dtype(x), bits, group_size, N, K, _stream(stream)))
    return out


def gai4_qmm_t_workspace_bytes(M: int, N: int, K: int, bits: int, group_size: int, dtype, split_k: int = 0) -> int:
    return int(lib().gai4_qmm_t_workspace_bytes(M, N, K, bits, group_size, _DTYPE[dtype], split_k))


def gai4_qmm_t_plan(M: int, N: int, K: int, bits: int, group_size: int, dtype, split_k: int = 0,
                    workspace_bytes: int = 0):
    """(path, splits): path 0 = CUDA-core kernel, 1 = tensor core."""
    path = ctypes.c_int()
    splits = ctypes.c_int()
    _check("gai4_qmm_t_plan", lib().gai4_qmm_t_plan(M, N, K, bits, group_size, _DTYPE[dtype], split_k,
                                                    workspace_bytes, ctypes.byref(path), ctypes.byref(splits)))
    return path.value, splits.value


def gai4_qmm_t(w_packed, scales, biases, x, out=None, bits: int = 4, group_size: int = 64, split_k: int = 0,
               workspace=None, stream=None):
    """out[m, n] = sum_k x[m, k] (s q + b)[n, k]. `workspace` (any dtype,
    device) holds the fp32 split-K partials; without one no split is used
    unless split_k forces it, in which case one is allocated here."""
    M, K = x.shape
    N = w_packed.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if workspace is None and split_k > 1:
        nbytes = gai4_qmm_t_workspace_bytes(M, N, K, bits, group_size, x.dtype, split_k)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("gai4_qmm_t", lib().gai4_qmm_t(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(x), _ptr(out),
                                          _dtype(x), bits, group_size, M, N, K, split_k, _ptr(workspace),
                                          ws_bytes, _stream(stream)))
    return out


def gai4_qmm_t_batched_workspace_bytes(batch, M, N, K, bits, group_size, dtype, split_k=0) -> int:
    return int(lib().gai4_qmm_t_batched_workspace_bytes(batch, M, N, K, bits, group_size, _DTYPE[dtype], split_k))


def gai4_qmm_t_batched(w_packed, scales, biases, x, out=None, bits: int = 4, group_size: int = 64, split_k: int = 0,
                       workspace=None, stream=None):
    """out[b, m, n] = sum_k x[b, m, k] (s q + b)[e(b), n, k] for x [B, M, K]
    (any batch / row strides, unit column stride, any element offset) and
    weights [N, ...] (one matrix for every batch) or [B, N, ...] (stacked).
    A workspace for the activation gather and the split-K partials is
    allocated here when none is given."""
    B, M, K = x.shape
    if x.stride(2) != 1:
        raise ValueError("gai4_qmm_t_batched: x needs unit column stride")
    w_batched = 1 if w_packed.dim() == 3 else 0
    N = w_packed.shape[-2]
    if out is None:
        out = torch.empty((B, M, N), dtype=x.dtype, device=x.device)
    if workspace is None:
        nbytes = gai4_qmm_t_batched_workspace_bytes(B, M, N, K, bits, group_size, x.dtype, split_k)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("gai4_qmm_t_batched",
           lib().gai4_qmm_t_batched(_ptr(w_packed), _ptr(scales), _ptr(biases), w_batched, _ptr_strided(x), x.stride(0),
                                    x.stride(1), _ptr(out), _dtype(x), bits, group_size, B, M, N, K, split_k,
                                    _ptr(workspace), ws_bytes, _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 8 << 20


def gai4_qmm_t_noalloc(w_packed, scales, biases, x, out, bits: int = 4, group_size: int = 64, split_k: int = 0,
                       stream=None):
    """gai4_qmm_t without a workspace argument: the split-K partials use the
    library's fixed 8 MiB device array (for callers that cannot allocate
    device memory; `out` must be given). Calls that overlap on the GPU race
    on that array."""
    M, K = x.shape
    N = w_packed.shape[0]
    _check("gai4_qmm_t_noalloc", lib().gai4_qmm_t_noalloc(_ptr(w_packed), _ptr(scales), _ptr(biases), _ptr(x),
                                                          _ptr(out), _dtype(x), bits, group_size, M, N, K, split_k,
                                                          _stream(stream)))
    return out


def gai4_q8_0_gemv(blocks, x, out=None, stream=None):
    """blocks [N, K/32, 9] int32/uint32, x [K] float32 -> out [N] float32."""
    N = blocks.shape[0]
    K = x.shape[-1]
    if out is None:
        out = torch.empty((N,), dtype=torch.float32, device=x.device)
    _check("gai4_q8_0_gemv", lib().gai4_q8_0_gemv(_ptr(blocks), _ptr(x), _ptr(out), N, K, _stream(stream)))
    return out


def gai4_quantize_x_q8(x, xq=None, xd=None, stream=None):
    """x [K] float32 -> (xq [K] int8, xd [K/32] float32): per 32-element
    block d = amax / 127, q = rint(x / d) clamped to +-127."""
    K = x.shape[-1]
    if xq is None:
        xq = torch.empty(K, dtype=torch.int8, device=x.device)
    if xd is None:
        xd = torch.empty(K // 32, dtype=torch.float32, device=x.device)
    _check("gai4_quantize_x_q8", lib().gai4_quantize_x_q8(_ptr(x), _ptr(xq), _ptr(xd), K, _stream(stream)))
    return xq, xd


def gai4_q8_0_gemv_i8(blocks, xq, xd, out=None, stream=None):
    """blocks [N, K/32, 9] int32/uint32, xq [K] int8, xd [K/32] float32 ->
    out [N] float32 (block dots exact in integers)."""
    N = blocks.shape[0]
    K = xq.shape[-1]
    if out is None:
        out = torch.empty(N, dtype=torch.float32, device=xq.device)
    _check("gai4_q8_0_gemv_i8", lib().gai4_q8_0_gemv_i8(_ptr(blocks), _ptr(xq), _ptr(xd), _ptr(out), N, K,
                                                        _stream(stream)))
    return out


def gai4_q4_k_gemv(blocks, x, out=None, stream=None):
    """blocks [N, K/256, 144] uint8, x [K] float32 -> out [N] float32."""
    N = blocks.shape[0]
    K = x.shape[-1]
    if out is None:
        out = torch.empty((N,), dtype=torch.float32, device=x.device)
    _check("gai4_q4_k_gemv", lib().gai4_q4_k_gemv(_ptr(blocks), _ptr(x), _ptr(out), N, K, _stream(stream)))
    return out


def gai4_q4_k_dequantize(blocks, decoder: int = 0, out=None, stream=None):
    """blocks [N, K/256, 144] uint8 -> weights [N, K] float32 with the (sc, m)
    decoder of the TMA-staged GEMV kernel (decoder 0) or the general one (1)."""
    N = blocks.shape[0]
    K = blocks.shape[1] * 256
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=blocks.device)
    _check("gai4_q4_k_dequantize", lib().gai4_q4_k_dequantize(_ptr(blocks), _ptr(out), N, K, decoder,
                                                              _stream(stream)))
    return out


def gai4_q8_0_34b_gemv(blocks, x, out=None, stream=None):
    """blocks [N, K/32, 34] uint8 (GGUF's 34-byte Q8_0 block), x [K] float32 -> out [N] float32."""
    N = blocks.shape[0]
    K = x.shape[-1]
    if out is None:
        out = torch.empty((N,), dtype=torch.float32, device=x.device)
    _check("gai4_q8_0_34b_gemv", lib().gai4_q8_0_34b_gemv(_ptr(blocks), _ptr(x), _ptr(out), N, K,
                                                          _stream(stream)))
    return out


def gai4_q6_k_gemv(blocks, x, out=None, stream=None):
    """blocks [N, K/256, 210] uint8 (Q6_K super-blocks), x [K] float32 -> out [N] float32."""
    N = blocks.shape[0]
    K = x.shape[-1]
    if out is None:
        out = torch.empty((N,), dtype=torch.float32, device=x.device)
    _check("gai4_q6_k_gemv", lib().gai4_q6_k_gemv(_ptr(blocks), _ptr(x), _ptr(out), N, K, _stream(stream)))
    return out


def gai4_last_device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status word."""
    return int(lib().gai4_last_device_status(_stream(stream)))


def gai4_check_bounded_wait(arrive: bool, limit_cycles: int, status: torch.Tensor | None = None, stream=None) -> int:
    """Run the library's bounded mbarrier wait on a barrier that completes
    (arrive=True) or that nothing completes (arrive=False); returns the value
    of the device status word `status` (int32 [1], zeroed here when not given)
    after the stream has finished: 0, or GAI4_ERR_TIMEOUT when the wait gave up."""
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=torch.cuda.current_device())
    _check("gai4_check_bounded_wait", lib().gai4_check_bounded_wait(1 if arrive else 0, int(limit_cycles),
                                                                   _ptr(status), _stream(stream)))
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return int(status.item())
