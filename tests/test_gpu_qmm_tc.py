"""GPU qmm_t on the tensor-core path (tcgen05) and split-K against the oracle.

The tensor-core path rounds each dequantized weight once to the 16-bit MMA
operand type (as the dequantize-then-MMA kernels of metaltile-std
quantized.rs do); the acceptance bound is the same as everywhere.
"""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
from gpu_util import TORCH_DTYPE, affine_problem, sample_rows, to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def _run(packed, s, b, x, dtype, split_k=0, bits=4, gs=64):
    M, K = x.shape
    N = packed.shape[0]
    ws_bytes = g4.gai4_qmm_t_workspace_bytes(M, N, K, bits, gs, TORCH_DTYPE[dtype], split_k)
    ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device="cuda") if ws_bytes else None
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x, dtype), bits=bits,
                        group_size=gs, split_k=split_k, workspace=ws)
    assert g4.gai4_last_device_status() == 0
    return out


CASES = [(131, 1088, 9), (256, 2048, 16), (300, 1024, 40), (129, 4096, 85), (64, 512, 256), (200, 1024, 300),
         (1000, 1536, 33)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N,K,M", CASES)
def test_tc_matches_oracle_all_splits(N, K, M, dtype):
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, dtype, seed=N + K + M)
    path, _ = g4.gai4_qmm_t_plan(M, N, K, 4, 64, TORCH_DTYPE[dtype])
    assert path == 1
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, dtype)
    for S in (1, 2, 3, 4):
        try:
            g4.gai4_qmm_t_plan(M, N, K, 4, 64, TORCH_DTYPE[dtype], split_k=S, workspace_bytes=1 << 40)
        except g4.Gai4Error:
            continue   # not a legal split of this K
        out = _run(packed, s, b, x, dtype, split_k=S)
        assert_within(to_host_f64(out, dtype), ref, absdot, dtype, f"tc N={N} K={K} M={M} S={S} {dtype}")


@pytest.mark.parametrize("gs", [32, 128])
def test_tc_group_sizes(gs):
    N, K, M = 192, 2048, 24
    _, packed, s, b, x = affine_problem(N, K, M, 4, gs, "bf16", seed=gs)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, "bf16")
    for S in (1, 2, 4):
        out = _run(packed, s, b, x, "bf16", split_k=S, gs=gs)
        assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", f"tc gs={gs} S={S}")


def test_tc_split_deterministic():
    """A fixed split gives bit-identical outputs run to run (fixed summation order)."""
    for N, K, M in ((512, 4096, 33), (128, 4096, 48), (640, 2048, 96)):
        _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=77)
        for S in (1, 2, 4):
            a = _run(packed, s, b, x, "bf16", split_k=S)
            for _ in range(8):
                c = _run(packed, s, b, x, "bf16", split_k=S)
                assert torch.equal(a.view(torch.int16), c.view(torch.int16)), (N, K, M, S)


def test_tc_rows_equal_qmv():
    """Each output row of qmm_t agrees with qmv on that x row (both within the bound)."""
    N, K, M = 256, 2048, 12
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=3)
    out = to_host_f64(_run(packed, s, b, x, "bf16", split_k=2), "bf16")
    for m in (0, 5, 11):
        v = g4.gai4_qmv(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x[m], "bf16"))
        ref, absdot = oracle.qmm(packed, s, b, x[m], 4, 64, "bf16")
        assert_within(to_host_f64(v, "bf16"), ref, absdot, "bf16", "qmv row")
        assert_within(out[m], ref, absdot, "bf16", "qmm_t row")


# (K, N, M) of the mid-M split-K shapes and the compute-bound control
FULL = [(2048, 2048, 22), (4096, 4096, 16), (10752, 2048, 85), (14336, 4096, 33), (17408, 5120, 56),
        (5120, 17408, 28), (256, 4096, 40), (4096, 4096, 512)]


@pytest.mark.parametrize("K,N,M", FULL)
def test_tc_full_size_sampled(K, N, M):
    seed = 100 + FULL.index((K, N, M))
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=seed)
    ws_bytes = g4.gai4_qmm_t_workspace_bytes(M, N, K, 4, 64, torch.bfloat16, 0)
    ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device="cuda")
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16"), bits=4,
                        group_size=64, split_k=0, workspace=ws)   # the benchmark's call
    assert g4.gai4_last_device_status() == 0
    got = to_host_f64(out, "bf16")
    rows = sample_rows(N, 48, seed)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16", rows=rows)
    assert_within(got[:, rows], ref, absdot, "bf16", f"qmm_t {K}x{N} M={M}")
    assert np.all(np.isfinite(got))


# large M (prefill): the activations span several 256-row chunks along the
# grid's z dimension, the last one ragged in the first case; the second is the
# benchmark's prefill shape beside the step
@pytest.mark.parametrize("N,K,M", [(384, 1024, 1100), (14336, 4096, 2048)])
def test_tc_large_m_sampled(N, K, M):
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=M)
    path, _ = g4.gai4_qmm_t_plan(M, N, K, 4, 64, torch.bfloat16)
    assert path == 1
    got = to_host_f64(_run(packed, s, b, x, "bf16", split_k=0), "bf16")
    rows = sample_rows(N, 24, M)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16", rows=rows)
    assert_within(got[:, rows], ref, absdot, "bf16", f"qmm_t large M {K}x{N} M={M}")


@pytest.mark.parametrize("offset", [1, 3])   # scales / biases 2 and 6 bytes past a 16-byte boundary
def test_tc_misaligned_scales_biases(offset):
    """Scale / bias pointers that are not 16-byte aligned (views into a larger
    buffer) take the global-load path of the dequantize warps: same result
    bits as with aligned copies, and within the bound of the oracle."""
    N, K, M = 256, 2048, 24
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=77 + offset)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16")
    sd, bd = to_dev(s, "bf16"), to_dev(b, "bf16")
    sbig = torch.empty(sd.numel() + 8, dtype=torch.bfloat16, device="cuda")
    bbig = torch.empty(bd.numel() + 8, dtype=torch.bfloat16, device="cuda")
    s_mis = sbig[offset:offset + sd.numel()].view(sd.shape)
    b_mis = bbig[offset:offset + bd.numel()].view(bd.shape)
    s_mis.copy_(sd)
    b_mis.copy_(bd)
    assert s_mis.data_ptr() % 16 != 0 and b_mis.data_ptr() % 16 != 0
    assert g4.gai4_qmm_t_plan(M, N, K, 4, 64, torch.bfloat16)[0] == 1
    wd, xd = to_dev(packed), to_dev(x, "bf16")
    for S in (1, 2):
        ws = torch.empty(1 << 20, dtype=torch.float32, device="cuda")
        out_a = g4.gai4_qmm_t(wd, sd, bd, xd, bits=4, group_size=64, split_k=S, workspace=ws)
        out_m = g4.gai4_qmm_t(wd, s_mis, b_mis, xd, bits=4, group_size=64, split_k=S, workspace=ws)
        assert g4.gai4_last_device_status() == 0
        assert torch.equal(out_a, out_m)
        assert_within(to_host_f64(out_m, "bf16"), ref, absdot, "bf16", f"misaligned scales S={S}")


# tensor-core path for 2-, 3-, 6- and 8-bit codes (whole 256-column stages):
# ragged tiles, several M chunks (the wider codes take smaller chunks), every
# legal split
WIDTH_CASES = [(131, 1024, 9), (256, 2048, 40), (300, 1536, 100), (129, 4096, 300)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bits,gs", [(2, 32), (3, 64), (6, 128), (8, 64)])
@pytest.mark.parametrize("N,K,M", WIDTH_CASES)
def test_tc_other_widths(N, K, M, bits, gs, dtype):
    _, packed, s, b, x = affine_problem(N, K, M, bits, gs, dtype, seed=N + K + M + bits)
    assert g4.gai4_qmm_t_plan(M, N, K, bits, gs, TORCH_DTYPE[dtype])[0] == 1
    ref, absdot = oracle.qmm(packed, s, b, x, bits, gs, dtype)
    for S in (1, 2, 3, 4):
        try:
            g4.gai4_qmm_t_plan(M, N, K, bits, gs, TORCH_DTYPE[dtype], split_k=S, workspace_bytes=1 << 40)
        except g4.Gai4Error:
            continue
        out = _run(packed, s, b, x, dtype, split_k=S, bits=bits, gs=gs)
        assert_within(to_host_f64(out, dtype), ref, absdot, dtype, f"tc {bits}-bit N={N} K={K} M={M} S={S} {dtype}")


def test_tc_8bit_every_code():
    """Every 8-bit code value, including those at and above 128 (whose 16-bit
    pattern has the exponent field 1 instead of 0), in every row."""
    N, K, M, gs = 128, 1024, 16, 64
    r = np.random.default_rng(3)
    q = np.tile(np.arange(256, dtype=np.uint32), (N, K // 256))
    q = np.stack([np.roll(q[i], 7 * i) for i in range(N)])
    packed = oracle.pack(q, 8)
    sc = r.uniform(1e-3, 1e-2, (N, K // gs)).astype(np.float32)
    bi = r.uniform(-0.5, 0.5, (N, K // gs)).astype(np.float32)
    sb = torch.from_numpy(sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bb = torch.from_numpy(bi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x = torch.randn(M, K, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    ref, absdot = oracle.qmm(packed, sb, bb, xb, 8, gs, "bf16")
    out = _run(packed, sb, bb, xb, "bf16", bits=8, gs=gs)
    assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", "tc 8-bit every code")


def test_tc_split_workspace_contents_do_not_matter():
    """The split-K partials live in the caller's workspace: any leftover
    bytes there (all ones, random, a previous call's partials) give the same
    output bits."""
    N, K, M = 384, 4096, 33
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=91)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, "bf16")
    wd, sd, bd, xd = to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16")
    nbytes = g4.gai4_qmm_t_workspace_bytes(M, N, K, 4, 64, torch.bfloat16, 4)
    ws = torch.zeros(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    outs = []
    for fill in ("zero", "ones", "random", "reuse", "reuse"):
        if fill == "ones":
            ws.view(torch.int32).fill_(-1)
        elif fill == "random":
            ws.view(torch.int32).random_()
        out = g4.gai4_qmm_t(wd, sd, bd, xd, bits=4, group_size=64, split_k=4, workspace=ws)
        assert g4.gai4_last_device_status() == 0
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert_within(to_host_f64(outs[0], "bf16"), ref, absdot, "bf16", "split workspace contents")


def test_tc_bf16_scales_on_both_decode_forms():
    """bf16 4-bit tiles decode codes as subnormals when s * 2^133 is a finite
    bf16 (exponent field 1..121) and by the offset form otherwise; rows of one
    warp take either form: small, large (>= 2^-5), zero and subnormal scales,
    interleaved row by row."""
    N, K, M, gs = 256, 2048, 24, 64
    _, packed, s, b, x = affine_problem(N, K, M, 4, gs, "bf16", seed=123)
    s32 = oracle.to_f64(s, "bf16").astype(np.float32)
    kinds = np.arange(N) % 4
    s32[kinds == 1] *= 64.0                      # >= 2^-5: the offset form
    s32[kinds == 2] = 0.0
    s32[kinds == 3] = np.float32(3.0e-39)         # a bf16 subnormal
    s = torch.from_numpy(s32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, "bf16")
    for S in (1, 2):
        out = _run(packed, s, b, x, "bf16", split_k=S)
        assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", f"tc scale forms S={S}")
