"""GPU Q8_0 / Q4_K GEMVs against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import sample_rows, to_dev
from tolerance import assert_within

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(1, 32), (5, 96), (67, 1024 + 32), (129, 4096), (33, 14336 + 256)])
def test_q8_0_small(N, K):
    blocks = synth.q8_0_blocks(N, K, seed=N + K)
    x = synth.f32_vector(K, seed=K)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q8_0 N={N} K={K}")


def test_q8_0_extreme_codes_and_scales():
    """All 256 byte values, and f16 scales that are subnormal, large or zero."""
    N, K = 16, 256
    blocks = synth.q8_0_blocks(N, K, seed=1)
    allbytes = np.arange(256, dtype=np.uint8).reshape(8, 32)
    blocks[:8, :, 1:] = allbytes.copy().view("<u4").reshape(8, 1, 8)
    blocks[8, :, 0] = 0x0001          # smallest f16 subnormal
    blocks[9, :, 0] = 0x7BFF          # largest finite f16
    blocks[10, :, 0] = 0x0000         # zero scale
    blocks[11, :, 0] |= 0xFFFF0000    # junk in the unused high half
    x = synth.f32_vector(K, seed=2)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", "q8_0 extremes")


def test_q8_0_closed_form():
    """q = 1 and x = 1: out = 32 * sum(d) (exact for these sizes in binary32)."""
    N, K = 8, 256
    blocks = synth.q8_0_blocks(N, K, seed=3)
    blocks[:, :, 1:] = 0x01010101
    d = oracle.to_f64((blocks[:, :, 0] & 0xFFFF).astype(np.uint16), "f16")
    got = g4.gai4_q8_0_gemv(to_dev(blocks), torch.ones(K, device="cuda")).cpu().numpy()
    np.testing.assert_allclose(got, 32 * d.sum(axis=1), rtol=1e-5)


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (67, 4096 + 256), (129, 5120)])
def test_q4_k_small(N, K):
    blocks = synth.q4_k_blocks(N, K, seed=N + K)
    x = synth.f32_vector(K, seed=K + 1)
    ref, absdot = oracle.q4_k_gemv(blocks, x)
    got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q4_k N={N} K={K}")


# Row lengths that are multiples of 16 bytes take the TMA-staged kernel (one or
# several 1152-byte chunks per row, a partial last chunk, row counts that are
# not multiples of the rows per stage); K = 65536 does not fit the staged
# activations and takes the general kernel, as do Q8_0 rows of 36 * odd bytes.
@pytest.mark.parametrize("N,K", [(1, 128), (17, 2048), (1000, 2048), (77, 5632), (1029, 3072), (3, 65536)])
def test_q8_0_staged_shapes(N, K):
    blocks = synth.q8_0_blocks(N, K, seed=N * 7 + K)
    x = synth.f32_vector(K, seed=K + 5)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q8_0 N={N} K={K}")


@pytest.mark.parametrize("N,K", [(1, 2048), (17, 2304), (1000, 4096), (77, 5376), (4099, 3072), (3, 65536)])
def test_q4_k_staged_shapes(N, K):
    blocks = synth.q4_k_blocks(N, K, seed=N * 5 + K)
    x = synth.f32_vector(K, seed=K + 9)
    ref, absdot = oracle.q4_k_gemv(blocks, x)
    got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q4_k N={N} K={K}")


def test_blockq_repeatable():
    """The per-row sums are combined in a fixed order: repeated calls agree bit for bit."""
    N, K = 3000, 5120
    for kind in ("q8_0", "q4_k"):
        blocks = synth.q8_0_blocks(N, K, 41) if kind == "q8_0" else synth.q4_k_blocks(N, K, 41)
        fn = g4.gai4_q8_0_gemv if kind == "q8_0" else g4.gai4_q4_k_gemv
        b, x = to_dev(blocks), to_dev(synth.f32_vector(K, 42))
        first = fn(b, x).cpu().numpy()
        for _ in range(5):
            assert np.array_equal(fn(b, x).cpu().numpy(), first), kind


def test_q4_k_element_order_one_hot():
    """x = e_k picks weight k of every row: checks the nibble / sub-block order."""
    N, K = 4, 256
    blocks = synth.q4_k_blocks(N, K, seed=11)
    w = np.stack([oracle.q4_k_dequant_block(blocks[n, 0]) for n in range(N)])
    for k in (0, 1, 31, 32, 63, 64, 100, 129, 175, 200, 255):
        x = np.zeros(K, np.float32)
        x[k] = 1.0
        got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got, w[:, k], rtol=2e-6, atol=1e-7, err_msg=f"k={k}")


@pytest.mark.parametrize("kind,N,K,seed", [("q8_0", 4096, 4096, 300), ("q8_0", 14336, 5120, 301),
                                           ("q4_k", 4096, 4096, 302), ("q4_k", 14336, 5120, 303)])
def test_blockq_full_size_sampled(kind, N, K, seed):
    x = synth.f32_vector(K, seed + 1)
    rows = sample_rows(N, 128, seed)
    if kind == "q8_0":
        blocks = synth.q8_0_blocks(N, K, seed)
        got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
        ref, absdot = oracle.q8_0_gemv(blocks, x, rows=rows)
    else:
        blocks = synth.q4_k_blocks(N, K, seed)
        got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
        ref, absdot = oracle.q4_k_gemv(blocks, x, rows=rows)
    assert_within(got[rows], ref, absdot, "f32", f"{kind} {N}x{K}")
    assert np.all(np.isfinite(got))


def _q4k_enumerated_blocks(seed: int) -> np.ndarray:
    """8 x 4096 super-blocks: for each sub-block j and each (sc, m) in 64 x 64,
    one block whose 12 scale bytes give pair j = (sc, m) under get_scale_min_k4
    (the other bits of those bytes random); d = dmin = 1.0 (f16), random codes."""
    r = synth.rng(seed)
    sc, m = np.meshgrid(np.arange(64), np.arange(64), indexing="ij")
    sc, m = sc.reshape(-1), m.reshape(-1)
    out = []
    for j in range(8):
        blk = r.integers(0, 256, size=(4096, 144), dtype=np.uint8)
        blk[:, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
        blk[:, 2:4] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
        s = blk[:, 4:16].astype(np.int64)
        if j < 4:
            s[:, j] = (s[:, j] & 0xC0) | sc
            s[:, j + 4] = (s[:, j + 4] & 0xC0) | m
        else:
            s[:, j + 4] = (sc & 15) | ((m & 15) << 4)
            s[:, j - 4] = (s[:, j - 4] & 0x3F) | ((sc >> 4) << 6)
            s[:, j] = (s[:, j] & 0x3F) | ((m >> 4) << 6)
        blk[:, 4:16] = s.astype(np.uint8)
        out.append(blk)
    return np.concatenate(out)


@pytest.mark.parametrize("decoder", [0, 1])
def test_q4_k_scale_min_decode_bit_exact(decoder):
    """The 6-bit (sc, m) decoding of both Q4_K kernels, through the test-aid
    dequantize that runs the kernel's own decoder: every (sc, m) pair for
    every sub-block j, then 1e5 random super-blocks; every weight must equal
    the oracle's binary64 value rounded once to binary32."""
    enum = _q4k_enumerated_blocks(500)
    rnd = synth.q4_k_blocks(100000, 256, 501).reshape(-1, 144)
    for name, blocks in (("enumerated", enum), ("random", rnd)):
        nb = blocks.shape[0]
        got = g4.gai4_q4_k_dequantize(to_dev(blocks.reshape(nb, 1, 144)), decoder).cpu().numpy()
        want = np.stack([oracle.q4_k_dequant_block(blocks[b]) for b in range(nb)]).astype(np.float32)
        assert np.all(np.isfinite(want))
        bad = np.flatnonzero(got.reshape(-1).view(np.uint32) != want.reshape(-1).view(np.uint32))
        assert bad.size == 0, (name, decoder, bad[:8], got.reshape(-1)[bad[:8]], want.reshape(-1)[bad[:8]])
    # the enumerated blocks really cover every (sc, m) of every j
    for j in range(8):
        pairs = {oracle.q4_k_scale_min(enum[b, 4:16], j) for b in range(j * 4096, (j + 1) * 4096)}
        assert len(pairs) == 4096, j


@pytest.mark.parametrize("K", [4096, 5120])   # whole chunks; a last half chunk (lanes take the second row)
def test_q4_k_x_extreme_ranges(K):
    """The Q4_K TMA kernel scales each 64-element item of x by a power of two:
    items of zeros, tiny, huge and very wide-ranged values, and binary32
    subnormals, against the oracle."""
    N = 70
    blocks = synth.q4_k_blocks(N, K, 41)
    r = np.random.default_rng(42)
    x = r.standard_normal(K).astype(np.float64)
    for c in range(K // 64):
        sl = slice(64 * c, 64 * c + 64)
        kind = c % 6
        if kind == 0:
            x[sl] = 0.0
        elif kind == 1:
            x[sl] *= 1e-30
        elif kind == 2:
            x[sl] *= 1e30
        elif kind == 3:
            x[sl] *= np.where(r.random(64) < 0.5, 1e30, 1e-30)
        elif kind == 4:
            x[sl] = r.choice([-1.0, 1.0], 64) * 1e-40 * r.integers(1, 8, 64)
    x = x.astype(np.float32)
    ref, absdot = oracle.q4_k_gemv(blocks, x)
    got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert_within(got, ref, absdot, "f32", f"q4_k x extremes K={K}")
