"""GPU Q8_0 with integer activations against the oracle: the activation
quantizer bit for bit, the GEMV (TMA-staged and general kernels) within the
fp32 bound, and repeatability."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import sample_rows, to_dev
from tolerance import assert_within

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,seed", [(32, 1), (96, 2), (4096, 3), (5120, 4), (14336, 5)])
def test_quantize_x_q8_bit_exact(K, seed):
    x = synth.f32_vector(K, seed) * np.float32(4.0)
    x[:32] = 0.0                                   # a zero block
    if K >= 96:
        x[64:96] = np.float32(1e-30)               # tiny values: d far below 1
        x[40] = np.float32(-3e4)                   # a large outlier
    xq, xd = g4.gai4_quantize_x_q8(to_dev(x))
    want_q, want_d = oracle.quantize_x_q8(x)
    np.testing.assert_array_equal(xq.cpu().numpy(), want_q)
    np.testing.assert_array_equal(xd.cpu().numpy().view(np.uint32), want_d.view(np.uint32))


# 16-byte rows (K % 128 == 0) take the TMA-staged kernel, others the general one;
# K = 65536 does not fit the staged activations
@pytest.mark.parametrize("N,K", [(1, 128), (7, 96), (67, 1056), (129, 4096), (1000, 5120), (33, 14336 + 256),
                                 (3, 65536), (4099, 3072)])
def test_q8_0_gemv_i8(N, K):
    blocks = synth.q8_0_blocks(N, K, seed=N + K + 7)
    xq, xd = oracle.quantize_x_q8(synth.f32_vector(K, seed=K + 3))
    ref, absdot = oracle.q8_0_gemv_i8(blocks, xq, xd)
    got = g4.gai4_q8_0_gemv_i8(to_dev(blocks), to_dev(xq), to_dev(xd)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q8_0 i8 N={N} K={K}")


@pytest.mark.parametrize("N,K,seed", [(4096, 4096, 400), (14336, 5120, 401)])
def test_q8_0_gemv_i8_full_size_sampled(N, K, seed):
    blocks = synth.q8_0_blocks(N, K, seed)
    x = synth.f32_vector(K, seed + 1)
    xq_d, xd_d = g4.gai4_quantize_x_q8(to_dev(x))
    got = g4.gai4_q8_0_gemv_i8(to_dev(blocks), xq_d, xd_d).cpu().numpy().astype(np.float64)
    rows = sample_rows(N, 128, seed)
    xq, xd = oracle.quantize_x_q8(x)
    ref, absdot = oracle.q8_0_gemv_i8(blocks, xq, xd, rows=rows)
    assert_within(got[rows], ref, absdot, "f32", f"q8_0 i8 {N}x{K}")
    assert np.all(np.isfinite(got))
    for _ in range(3):   # fixed summation order
        again = g4.gai4_q8_0_gemv_i8(to_dev(blocks), xq_d, xd_d).cpu().numpy().astype(np.float64)
        assert np.array_equal(again, got)
