"""Known numerical limits, kept as executable expected failures (non-strict
xfail: a kernel that already meets the bound reports XPASS).

1. Offset decode on rows whose weights are all exactly zero while their
   scales are not: the "constant + code" decode removes the constant through
   the sum of the activations and leaves a rounding residue, while the exact
   answer is 0 and the bound there is one subnormal ulp. No quantizer output
   has this form (an all-equal group gets scale 0; an all-zero Q8_0 block
   gets d = 0); only hand-built blocks do.
2. The tensor-core path rounds each dequantized weight once to bf16 (up to
   2^-9 relative). A crafted row whose weights all round the same way, with
   every product of one sign, exceeds 1e-3 * sum|w x| (about 1.9e-3)."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def _bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.xfail(reason="offset decode: rounding residue on all-zero-weight rows with nonzero scales",
                   strict=False)
def test_q8_0_all_zero_codes_nonzero_scale():
    N, K = 4, 1024
    blocks = synth.q8_0_blocks(N, K, 1)
    blocks[:, :, 1:] = 0                               # every code 0, scales kept
    x = synth.f32_vector(K, 2)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    assert np.all(ref == 0.0)
    got = g4.gai4_q8_0_gemv(to_dev(blocks), to_dev(x)).cpu().numpy().astype(np.float64)
    assert_within(got, ref, absdot, "f32", "q8_0 all-zero codes")


@pytest.mark.xfail(reason="offset decode: rounding residue on all-zero-weight rows with nonzero scales",
                   strict=False)
def test_qmv_all_zero_codes_zero_bias():
    N, K = 8, 4096
    packed = np.zeros((N, K // 8), dtype=np.uint32)
    s = _bf16_bits(np.full((N, K // 64), 0.75, np.float32))
    b = _bf16_bits(np.zeros((N, K // 64), np.float32))
    x = synth.activations(1, K, "bf16", 3)
    ref, absdot = oracle.qmm(packed, s, b, x[0], 4, 64, "bf16")
    out = g4.gai4_qmv(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x[0], "bf16"))
    assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", "qmv all-zero codes")


@pytest.mark.xfail(reason="tensor-core path: one bf16 rounding per weight, crafted to round one way",
                   strict=False)
def test_tc_crafted_one_way_rounding():
    N, K, M = 128, 4096, 16
    packed = np.full((N, K // 8), 0x11111111, dtype=np.uint32)      # every code 1
    s = _bf16_bits(np.full((N, K // 64), 1.0 + 2.0**-7, np.float32))
    b = _bf16_bits(np.full((N, K // 64), 2.0**-9, np.float32))      # w = 1 + 2^-7 + 2^-9: rounds down by 2^-9 in bf16
    x = np.abs(oracle.to_f64(synth.activations(M, K, "bf16", 4), "bf16")).astype(np.float32)
    xb = _bf16_bits(x)
    ref, absdot = oracle.qmm(packed, s, b, xb, 4, 64, "bf16")
    out = g4.gai4_qmm_t(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(xb, "bf16"))
    assert g4.gai4_qmm_t_plan(M, N, K, 4, 64, torch.bfloat16)[0] == 1
    assert_within(to_host_f64(out, "bf16"), ref, absdot, "bf16", "tc crafted rounding")
