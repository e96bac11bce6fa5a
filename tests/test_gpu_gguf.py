"""GPU GEMVs over GGUF's 34-byte Q8_0 block and the Q6_K super-block against
the oracle: ragged and tail shapes (slabs shorter than a full one, buffers
whose size is not a multiple of 16 bytes), the benchmark's full sizes on
sampled rows, repeatability, and argument errors."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import sample_rows, to_dev
from tolerance import assert_within

pytestmark = pytest.mark.gpu

FORMATS = {
    "q8_0_34b": (synth.q8_0_34b_blocks, oracle.q8_0_34b_gemv, g4.gai4_q8_0_34b_gemv, 32),
    "q6_k": (synth.q6_k_blocks, oracle.q6_k_gemv, g4.gai4_q6_k_gemv, 256),
}


def _run(fmt, N, K, seed, rows=None):
    gen, ref_fn, gpu_fn, bk = FORMATS[fmt]
    blocks = gen(N, K, seed)
    x = synth.f32_vector(K, seed + 1)
    got = gpu_fn(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    ref, absdot = ref_fn(blocks, x, rows=rows)
    assert_within(got, ref, absdot, "f32", f"{fmt} N={N} K={K}")


# K up to 24576 stages x in shared memory; (3, 24576) is the largest such K,
# (2, 32768) reads x through the read-only cache
@pytest.mark.parametrize("N,K", [(1, 32), (3, 96), (7, 1024), (9, 1056), (129, 4096), (1000, 5120), (33, 14336),
                                 (4099, 3072), (5, 32 * 33), (3, 24576), (2, 32768)])
def test_q8_0_34b_gemv(N, K):
    _run("q8_0_34b", N, K, N + K)


@pytest.mark.parametrize("N,K", [(1, 256), (3, 768), (7, 2048), (9, 2304), (129, 4096), (1000, 5120),
                                 (33, 14336), (4099, 3072), (3, 256 * 17), (3, 24576), (2, 32768)])
def test_q6_k_gemv(N, K):
    _run("q6_k", N, K, 2 * N + K)


@pytest.mark.parametrize("fmt", list(FORMATS))
@pytest.mark.parametrize("N,K", [(4096, 4096), (14336, 5120)])
def test_full_size_sampled(fmt, N, K):
    _run(fmt, N, K, 11, rows=sample_rows(N, 48, seed=N))


@pytest.mark.parametrize("fmt", list(FORMATS))
def test_repeatable(fmt):
    gen, _, gpu_fn, _ = FORMATS[fmt]
    blocks = to_dev(gen(777, 5120, 5))
    x = to_dev(synth.f32_vector(5120, 6))
    a = gpu_fn(blocks, x)
    b = gpu_fn(blocks, x)
    assert torch.equal(a, b)
    assert g4.gai4_last_device_status() == g4.GAI4_OK


def test_misaligned_x_rejected():
    blocks = to_dev(synth.q6_k_blocks(4, 512, 1))
    xbuf = torch.zeros(513, dtype=torch.float32, device="cuda")
    with pytest.raises(g4.Gai4Error) as e:
        g4.gai4_q6_k_gemv(blocks, xbuf[1:])
    assert e.value.status == g4.GAI4_ERR_MISALIGNED
