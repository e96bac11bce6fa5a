"""The plain binary32 CPU loops timed beside the oracle (the "reasonable CPU"
baseline of the benchmark) compute the same products: within the acceptance
bound of the binary64 oracle on the benchmark's kinds of calls."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import assert_within


@pytest.mark.parametrize("M,N,K", [(1, 64, 1024), (8, 33, 2048), (56, 17, 512)])
def test_affine_f32_loop(M, N, K):
    W = synth.affine_weights(N, K, M + N)
    packed, s, b = oracle.quantize(W, 4, 64, "bf16")
    x = synth.activations(M, K, "bf16", 3)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16")
    got = oracle.qmm_f32loop(packed, s, b, x, 4, 64, "bf16")
    assert_within(got.astype(np.float64), ref, absdot, "f32", "affine f32 loop")
    rows = np.array([0, N - 1, N // 2], dtype=np.int64)
    sub = oracle.qmm_f32loop(packed, s, b, x, 4, 64, "bf16", rows=rows)
    assert np.array_equal(sub, got[:, rows])


def test_block_f32_loops():
    N, K = 9, 1024
    x = synth.f32_vector(K, 4)
    b8 = synth.q8_0_blocks(N, K, 5)
    ref, absdot = oracle.q8_0_gemv(b8, x)
    assert_within(oracle.q8_0_gemv_f32loop(b8, x).astype(np.float64), ref, absdot, "f32", "q8_0 f32 loop")
    b4 = synth.q4_k_blocks(N, K, 6)
    ref, absdot = oracle.q4_k_gemv(b4, x)
    assert_within(oracle.q4_k_gemv_f32loop(b4, x).astype(np.float64), ref, absdot, "f32", "q4_k f32 loop")
