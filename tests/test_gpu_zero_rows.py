"""Rows whose dequantized weights are all (or nearly all) exactly zero.

The oracle value of such a row is exactly 0 (or tiny), where the acceptance
bound shrinks to one subnormal ulp. Every CUDA-core kernel turns a code into
its exact value before multiplying it with x (no "constant + code" offset is
ever removed through the sum of x), so zero codes add exactly zero and the
bound holds here too. Also the tensor-core path's one departure from the
bound, on a crafted row whose bf16-rounded weights err coherently against an
output that cancels (reading r2 of the design notes: the operand is the
weight rounded once to bf16)."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import TORCH_DTYPE, to_dev, to_host_f64
from tolerance import assert_within, ulp

pytestmark = pytest.mark.gpu


def _bits16(vals, dtype):
    t = torch.tensor(np.asarray(vals, np.float32), dtype=torch.float32).to(TORCH_DTYPE[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def _sb(vals, dtype):
    return np.asarray(vals, np.float32) if dtype == "f32" else _bits16(vals, dtype)


def _zero_code_problem(N, K, bits, gs, dtype, x_seed):
    """all codes 0, bias 0, scales nonzero (0.75): every weight is exactly 0"""
    packed = np.zeros((N, K * bits // 32), dtype=np.uint32)
    s = _sb(np.full((N, K // gs), 0.75, np.float32), dtype)
    b = _sb(np.zeros((N, K // gs), np.float32), dtype)
    x = synth.activations(2, K, dtype, x_seed)
    return packed, s, b, x


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("bits,K", [(4, 4096), (4, 512), (3, 1024), (8, 1024), (2, 2048), (6, 1536)])
def test_qmv_all_zero_codes(dtype, bits, K):
    """qmv on the 4-bit TMA kernel (K >= 1024) and the general kernel (other
    widths, short rows): exactly zero."""
    N, gs = 8, 64
    packed, s, b, x = _zero_code_problem(N, K, bits, gs, dtype, 3)
    ref, absdot = oracle.qmm(packed, s, b, x[0], bits, gs, dtype)
    assert np.all(ref == 0.0)
    out = g4.gai4_qmv(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x[0], dtype), bits=bits,
                      group_size=gs)
    got = to_host_f64(out, dtype)
    assert_within(got, ref, absdot, dtype, f"qmv zero rows {bits}-bit K={K} {dtype}")
    assert np.all(got == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_qmm_t_cuda_core_all_zero_codes(dtype):
    """qmm_t on the CUDA-core kernel (M = 2 with bf16; any M with f32)."""
    N, K, gs = 8, 2048, 64
    packed, s, b, x = _zero_code_problem(N, K, 4, gs, dtype, 5)
    assert g4.gai4_qmm_t_plan(2, N, K, 4, gs, TORCH_DTYPE[dtype])[0] == 0
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, dtype)
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x, dtype), bits=4, group_size=gs)
    got = to_host_f64(out, dtype)
    assert_within(got, ref, absdot, dtype, f"qmm_t zero rows {dtype}")
    assert np.all(got == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_qmv_one_code_among_zeros_large_x_elsewhere(dtype):
    """A row with a single nonzero code where x is tiny, and x large where the
    codes are zero: the value s * x_small must not be swamped by rounding of
    the large activations (an offset decode would leave ~2^-20 s sum|x|)."""
    N, K, gs = 4, 4096, 64
    packed = np.zeros((N, K // 8), dtype=np.uint32)
    packed[:, 5] = 0x00000100                      # code 1 at column 8*5 + 2 = 42 of every row
    s = _sb(np.full((N, K // gs), 0.5, np.float32), dtype)
    b = _sb(np.zeros((N, K // gs), np.float32), dtype)
    xv = np.full(K, 1000.0, np.float32)
    xv[42] = 1.0e-3
    x = xv if dtype == "f32" else _bits16(xv, dtype)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, dtype)
    out = g4.gai4_qmv(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x, dtype), bits=4, group_size=gs)
    assert_within(to_host_f64(out, dtype), ref, absdot, dtype, f"qmv single code {dtype}")


@pytest.mark.parametrize("K", [1024, 96, 65536])   # TMA kernel; rows not 16-byte aligned; x past shared memory
def test_q8_0_all_zero_codes_nonzero_scale(K):
    N = 4
    blocks = synth.q8_0_blocks(N, K, 1)
    blocks[:, :, 1:] = 0                               # every code 0, scales kept
    x = synth.f32_vector(K, 2)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    assert np.all(ref == 0.0)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q8_0 all-zero codes K={K}")
    assert np.all(got == 0.0)


def test_q8_0_one_code_among_zeros_large_x_elsewhere():
    N, K = 4, 1024
    blocks = synth.q8_0_blocks(N, K, 3)
    blocks[:, :, 1:] = 0
    blocks[:, 2, 1] = 0x00000001                       # code +1 at element 64 of every row
    x = np.full(K, 1000.0, np.float32)
    x[64] = 1.0e-3
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", "q8_0 single code")


@pytest.mark.parametrize("K", [1024, 65536])       # TMA kernel; general kernel
def test_q4_k_all_zero_codes_zero_mins(K):
    """every code 0 and every m_j 0 (sc_j nonzero, d and dmin nonzero): all
    weights are exactly 0"""
    N = 4
    blocks = synth.q4_k_blocks(N, K, 7)
    blocks[:, :, 16:] = 0                              # codes
    blocks[:, :, 4:8] = 5                              # sc_0..3 = 5, top bits 0
    blocks[:, :, 8:12] = 0                             # m_0..3 = 0 (and the top bits of sc/m 4..7)
    blocks[:, :, 12:16] = 0x07                         # sc_4..7 = 7, m_4..7 = 0
    for j in range(8):
        assert oracle.q4_k_scale_min(blocks[0, 0, 4:16], j)[1] == 0
    x = synth.f32_vector(K, 8)
    ref, absdot = oracle.q4_k_gemv(blocks, x)
    assert np.all(ref == 0.0)
    got = g4.gai4_q4_k_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", f"q4_k all-zero codes K={K}")
    assert np.all(got == 0.0)


def _coherent_rounding_problem(M):
    """Codes alternating 1, 2 along K with s = 1 + 2^-7, b = 3 * 2^-9 (both exact
    in bf16): w_1 = 1 + 7 * 2^-9 rounds up by 2^-9 in bf16 and w_2 = 2 + 11 *
    2^-9 rounds down by 3 * 2^-9. With x alternating 2, -1 every rounding error
    adds with the same sign while the output cancels to (K / 2) b."""
    N, K, gs = 128, 4096, 64
    packed = np.full((N, K // 8), 0x21212121, dtype=np.uint32)   # codes 1, 2, 1, 2, ...
    s = _bits16(np.full((N, K // gs), 1.0 + 2.0**-7, np.float32), "bf16")
    b = _bits16(np.full((N, K // gs), 3.0 * 2.0**-9, np.float32), "bf16")
    xv = np.tile(np.array([2.0, -1.0], np.float32), K // 2)
    x = _bits16(np.tile(xv, (M, 1)), "bf16")
    return N, K, gs, packed, s, b, x


def test_tc_coherent_bf16_rounding_reading():
    """Tensor-core path (reading r2): the MMA operand is each weight rounded
    once to bf16 (unit roundoff 2^-8), so the error is bounded by
    2^-8 sum|w x| plus the fp32 accumulation and the output rounding. This
    crafted row reaches that bound's order and exceeds 1e-3 sum|w x| + 1 ulp;
    on rows whose output does not cancel, the ulp of the bf16 output (at
    least 2^-8 of its value) covers the operand rounding."""
    M = 16
    N, K, gs, packed, s, b, x = _coherent_rounding_problem(M)
    assert g4.gai4_qmm_t_plan(M, N, K, 4, gs, torch.bfloat16)[0] == 1
    ref, absdot = oracle.qmm(packed, s, b, x, 4, gs, "bf16")
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16"), bits=4,
                        group_size=gs)
    got = to_host_f64(out, "bf16")
    err = np.abs(got - ref)
    r2_bound = 2.0**-8 * absdot + 1e-5 * absdot + ulp(ref, "bf16")
    assert np.all(err <= r2_bound)
    assert np.all(err > 1e-3 * absdot + ulp(ref, "bf16"))   # the departure is real on this row
    # the CUDA-core path (exact products, binary32 sums) meets the stated bound on it
    out2 = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x[:2], "bf16"), bits=4,
                         group_size=gs)
    assert g4.gai4_qmm_t_plan(2, N, K, 4, gs, torch.bfloat16)[0] == 0
    assert_within(to_host_f64(out2, "bf16"), ref[:2], absdot[:2], "bf16", "CUDA-core coherent rounding row")
