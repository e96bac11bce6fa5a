"""gai4_qmm_t_noalloc: the split-K matmul for callers that cannot allocate
device memory (its fp32 partials live in the library's fixed 8 MiB device
array).

Called through the C ABI on two calls in a row with different shapes, so the
second call runs on the array as the first left it. Each output must equal
gai4_qmm_t with a caller-provided workspace of the array's size (hence the
same automatic split) bit for bit, since a fixed split sums in a fixed order,
and must meet the oracle bound. Collected last (file name) so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
from gpu_util import affine_problem, to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def _noalloc_c(packed, s, b, x, out, split_k):
    """The raw C entry point (no Python-side allocation either)."""
    L = g4.lib()
    M, K = x.shape
    N = packed.shape[0]
    st = L.gai4_qmm_t_noalloc(ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(s.data_ptr()),
                              ctypes.c_void_p(b.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                              ctypes.c_void_p(out.data_ptr()), 2, 4, 64, M, N, K, split_k,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_qmm_t_two_calls():
    # (N, K, M): the second needs more partials than the first
    shapes = [(1000, 4096, 33), (2048, 10752, 85)]
    for i, (N, K, M) in enumerate(shapes):
        _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=900 + i)
        P, S_, B_, X = to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16")
        path, splits = g4.gai4_qmm_t_plan(M, N, K, 4, 64, torch.bfloat16, 0, g4.NOALLOC_SCRATCH_BYTES)
        assert path == 1 and splits > 1        # the scratch array is really used
        assert splits * M * N * 4 <= g4.NOALLOC_SCRATCH_BYTES
        assert g4.gai4_qmm_t_workspace_bytes(M, N, K, 4, 64, torch.bfloat16, splits) > 0
        out_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc_c(P, S_, B_, X, out_na, 0) == 0
        # the same automatic plan: a caller workspace as large as the array
        ws = torch.empty(g4.NOALLOC_SCRATCH_BYTES // 4, dtype=torch.float32, device="cuda")
        out_ref = g4.gai4_qmm_t(P, S_, B_, X, bits=4, group_size=64, split_k=0, workspace=ws)
        assert g4.gai4_last_device_status() == 0
        assert torch.equal(out_na, out_ref), f"noalloc call {i + 1} differs from gai4_qmm_t"
        ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16")
        assert_within(to_host_f64(out_na, "bf16"), ref, absdot, "bf16", f"noalloc call {i + 1} vs oracle")


def test_noalloc_rejects_oversized_split():
    N, K, M = 4096, 4096, 512                           # 4 * 512 * 4096 * 4 B = 32 MiB > 8 MiB
    P = torch.zeros((N, K // 8), dtype=torch.int32, device="cuda")
    S_ = torch.zeros((N, K // 64), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_c(P, S_, S_, X, out, 4) == g4.GAI4_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0        # nothing was written
