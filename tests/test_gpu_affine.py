"""GPU qmv / qmm_t (affine group-quantized) against the fp64 oracle.

Small shapes are compared element by element over several tiles and a ragged
tail; the full-size shapes of the benchmark are compared on sampled rows that
the oracle computes one by one, with the GPU run in the same launch
configuration the benchmark times (gai4_qmv / gai4_qmm_t with automatic plan).
"""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import TORCH_DTYPE, affine_problem, sample_rows, to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu

DTYPES = ("f32", "f16", "bf16")


def _run_qmv(packed, s, b, x, bits, gs, dtype):
    out = g4.gai4_qmv(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x.reshape(-1), dtype),
                      bits=bits, group_size=gs)
    return to_host_f64(out, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_qmv_small_sweep(bits, gs, dtype):
    for N, K in [(1, gs), (7, 2 * gs), (129, 512 + gs), (67, 2048 + 2 * gs)]:
        K = K if (K * bits) % 32 == 0 else K * 2
        _, packed, s, b, x = affine_problem(N, K, 1, bits, gs, dtype, seed=N * 31 + K)
        ref, absdot = oracle.qmm(packed, s, b, x[0], bits, gs, dtype)
        got = _run_qmv(packed, s, b, x, bits, gs, dtype)
        assert_within(got, ref, absdot, dtype, f"qmv bits={bits} gs={gs} {dtype} N={N} K={K}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_qmv_worked_example(dtype):
    """The hand-derived 4-bit example (6 and 42), exact in every dtype."""
    words = np.zeros((1, 8), dtype=np.uint32)
    words[0, 0] = 0x76543210
    vals = {"f32": lambda v: np.asarray(v, np.float32)}
    s = np.array([[0.5]], np.float32)
    b = np.array([[-1.0]], np.float32)
    if dtype != "f32":
        tdt = TORCH_DTYPE[dtype]
        conv = lambda a: torch.from_numpy(a).to(tdt).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    else:
        conv = vals["f32"]
    for xs, want in (([1] * 8, 6.0), (list(range(8)), 42.0)):
        x = np.zeros((1, 64), np.float32)
        x[0, :8] = xs
        got = _run_qmv(words, conv(s), conv(b), conv(x), 4, 64, dtype)
        assert got[0] == want


# (N, K) of the qmv shape sweep; 4096 x 4096 is the headline shape (seed 0)
FULL_SHAPES = [(4096, 4096, 0), (5120, 5120, 1), (14336, 5120, 2), (5120, 14336, 3), (27648, 5120, 4)]


@pytest.fixture(scope="module")
def full_weights():
    cache = {}

    def get(N, K, seed):
        if (N, K) not in cache:
            cache.clear()
            cache[(N, K)] = synth.affine_weights(N, K, seed)
        return cache[(N, K)]
    return get


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N,K,seed", FULL_SHAPES)
def test_qmv_full_size_sampled(N, K, seed, dtype, full_weights):
    if seed == 0 and dtype != "bf16":
        pytest.skip("the 4096 x 4096 shape is specified in bf16 only")
    W = full_weights(N, K, seed)
    packed, s, b = oracle.quantize(W, 4, 64, dtype)
    x = synth.activations(1, K, dtype, seed + 7919)
    # GPU quantizes the same W itself; the packed bytes must equal the oracle's
    tdt = TORCH_DTYPE[dtype]
    pg, sg, bg = g4.gai4_quantize(to_dev(W), 4, 64, tdt)
    assert np.array_equal(pg.cpu().view(torch.int32).numpy().view(np.uint32), packed)
    out = g4.gai4_qmv(pg, sg, bg, to_dev(x.reshape(-1), dtype), bits=4, group_size=64)
    got = to_host_f64(out, dtype)
    rows = sample_rows(N, 96, seed)
    ref, absdot = oracle.qmm(packed, s, b, x[0], 4, 64, dtype, rows=rows)
    assert_within(got[rows], ref, absdot, dtype, f"qmv {N}x{K} {dtype}")
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 17, 33])
def test_qmm_small_m(M, dtype):
    N, K, bits, gs = 131, 1024 + 64, 4, 64
    _, packed, s, b, x = affine_problem(N, K, M, bits, gs, dtype, seed=M)
    ref, absdot = oracle.qmm(packed, s, b, x, bits, gs, dtype)
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x, dtype), bits=bits,
                        group_size=gs)
    assert_within(to_host_f64(out, dtype), ref, absdot, dtype, f"qmm_t M={M} {dtype}")


@pytest.mark.parametrize("bits,gs", [(2, 32), (3, 64), (6, 128), (8, 64)])
@pytest.mark.parametrize("M", [2, 8])
def test_qmm_small_m_widths(bits, gs, M):
    N, K = 65, 512
    _, packed, s, b, x = affine_problem(N, K, M, bits, gs, "bf16", seed=bits * 7 + M)
    ref, absdot = oracle.qmm(packed, s, b, x, bits, gs, "bf16")
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16"), bits=bits,
                        group_size=gs)
    assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", f"qmm_t bits={bits} gs={gs} M={M}")


# 4-bit shapes on the prefetching qmv kernel (scale rows a multiple of 16 bytes,
# K >= 1024): K a multiple of 1024 takes one 3-D copy per stage, other K one
# 2-D copy per 1024-column iteration with a ragged last iteration
QMV4_SHAPES = [(1, 1024), (33, 1536), (300, 2560), (4099, 3072), (77, 5632), (1000, 2048)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("N,K", QMV4_SHAPES)
def test_qmv_4bit_copy_layouts(N, K, gs, dtype):
    _, packed, s, b, x = affine_problem(N, K, 1, 4, gs, dtype, seed=N + K + gs)
    ref, absdot = oracle.qmm(packed, s, b, x[0], 4, gs, dtype)
    got = _run_qmv(packed, s, b, x, 4, gs, dtype)
    assert_within(got, ref, absdot, dtype, f"qmv N={N} K={K} gs={gs} {dtype}")
    assert np.all(np.isfinite(got))


def test_qmm_m1_equals_qmv():
    """qmm_t at M = 1 runs the qmv kernel: identical bits."""
    _, packed, s, b, x = affine_problem(300, 2048, 1, 4, 64, "bf16", seed=5)
    a = g4.gai4_qmv(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x.reshape(-1), "bf16"))
    m = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16"))
    assert torch.equal(a.view(torch.int16).cpu(), m.view(torch.int16).cpu().reshape(-1))


def test_qmv_scaling_x_by_two_f32():
    """x -> 2x scales every f32 output by exactly 2 (power-of-two scaling)."""
    _, packed, s, b, x = affine_problem(64, 1024, 1, 4, 64, "f32", seed=9)
    a = _run_qmv(packed, s, b, x, 4, 64, "f32")
    c = _run_qmv(packed, s, b, (x * 2).astype(np.float32), 4, 64, "f32")
    assert np.array_equal(c, 2 * a)


def test_qmv_repeatable():
    _, packed, s, b, x = affine_problem(1000, 4096, 1, 4, 64, "bf16", seed=10)
    args = (to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x.reshape(-1), "bf16"))
    a = g4.gai4_qmv(*args)
    c = g4.gai4_qmv(*args)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 6, 8])
def test_width_sweep_full_size_sampled(bits, gs, full_weights):
    """The bit-width x group-size sweep at N = K = 4096 for M in {1, 8, 64},
    bf16, in the launch configuration the benchmark times (qmv for M = 1,
    qmm_t with automatic plan and a workspace otherwise), on sampled rows."""
    N = K = 4096
    W = full_weights(N, K, 0)
    packed, s, b = oracle.quantize(W, bits, gs, "bf16")
    pg, sg, bg = g4.gai4_quantize(to_dev(W), bits, gs, torch.bfloat16)
    assert np.array_equal(pg.cpu().view(torch.int32).numpy().view(np.uint32), packed)
    rows = sample_rows(N, 48, bits * 1000 + gs)
    for M in (1, 8, 64):
        x = synth.activations(M, K, "bf16", 4100 + M)
        xd = to_dev(x, "bf16")
        if M == 1:
            out = g4.gai4_qmv(pg, sg, bg, xd.reshape(-1), bits=bits, group_size=gs).reshape(1, N)
        else:
            nbytes = g4.gai4_qmm_t_workspace_bytes(M, N, K, bits, gs, torch.bfloat16, 0)
            ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
            out = g4.gai4_qmm_t(pg, sg, bg, xd, bits=bits, group_size=gs, split_k=0, workspace=ws)
        got = to_host_f64(out, "bf16")
        assert np.all(np.isfinite(got))
        ref, absdot = oracle.qmm(packed, s, b, x, bits, gs, "bf16", rows=rows)
        assert_within(got[:, rows], ref, absdot, "bf16", f"bits={bits} gs={gs} M={M}")


def _x_extremes(K, dtype, seed):
    """x whose 32-element chunks are: all zero, tiny, huge, spanning many
    binades, subnormal in the type, and ordinary N(0, 1)."""
    r = np.random.default_rng(seed)
    big, small, sub = (2e4, 1e-4, 3e-7) if dtype == "f16" else (1e30, 1e-30, 1e-39)
    x = r.standard_normal(K).astype(np.float64)
    for c in range(K // 32):
        sl = slice(32 * c, 32 * c + 32)
        kind = c % 6
        if kind == 0:
            x[sl] = 0.0
        elif kind == 1:
            x[sl] *= small
        elif kind == 2:
            x[sl] *= big / 4
        elif kind == 3:
            x[sl] *= np.where(r.random(32) < 0.5, big / 4, small)
        elif kind == 4:
            x[sl] = r.choice([-1.0, 1.0], 32) * sub * r.integers(1, 8, 32)
    return _bits_of(x.astype(np.float32), dtype)


def _bits_of(x32, dtype):
    if dtype == "f32":
        return x32
    t = torch.from_numpy(x32).to(TORCH_DTYPE[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("gs", [32, 64, 128])
def test_qmv_4bit_x_extreme_ranges(dtype, gs):
    """The 4-bit qmv kernel on x with zero, tiny, huge, wide-range and
    subnormal chunks (the bf16 and binary32 paths scale each chunk by a
    power of two)."""
    N, K = 96, 4096
    _, packed, s, b, _ = affine_problem(N, K, 1, 4, gs, dtype, seed=gs + 5)
    x = _x_extremes(K, dtype, gs)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, dtype)
    got = _run_qmv(packed, s, b, x, 4, gs, dtype)
    assert np.all(np.isfinite(got))
    assert_within(got, ref, absdot, dtype, f"qmv x extremes {dtype} gs={gs}")
