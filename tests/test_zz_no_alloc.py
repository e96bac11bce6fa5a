"""gai4_qmm_t_noalloc: the split-K matmul for callers that cannot allocate
device memory (its partials live in the library's fixed 8 MiB device array).

Called through the C ABI and checked against gai4_qmm_t (caller-provided
workspace) on two calls in a row with different shapes, so the second call
runs on the array as the first left it. Collected last (file name) so that a
run stopping at the first failure has already run every other test.
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
    shapes = [(1000, 4096, 33), (2048, 10752, 85)]    # (N, K, M): the second needs more partials
    for i, (N, K, M) in enumerate(shapes):
        _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=900 + i)
        P, S_, B_, X = to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16")
        path, splits = g4.gai4_qmm_t_plan(M, N, K, 4, 64, torch.bfloat16, 0, g4.NOALLOC_SCRATCH_BYTES)
        assert path == 1 and splits > 1        # the scratch array is really used
        out_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc_c(P, S_, B_, X, out_na, 0) == 0
        ws = torch.empty(splits * M * N, dtype=torch.float32, device="cuda")
        out_ref = g4.gai4_qmm_t(P, S_, B_, X, bits=4, group_size=64, split_k=splits, workspace=ws)
        assert g4.gai4_last_device_status() == 0
        _, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16")
        got = to_host_f64(out_na, "bf16")
        assert np.all(np.isfinite(got))
        assert_within(got, to_host_f64(out_ref, "bf16"), absdot, "bf16", f"noalloc call {i + 1}")


def test_noalloc_rejects_oversized_split():
    N, K, M = 4096, 4096, 512                           # 4 * 512 * 4096 * 4 B = 32 MiB > 8 MiB
    P = torch.zeros((N, K // 8), dtype=torch.int32, device="cuda")
    S_ = torch.zeros((N, K // 64), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_c(P, S_, S_, X, out, 4) == g4.GAI4_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0        # nothing was written
