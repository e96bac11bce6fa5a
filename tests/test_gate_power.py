"""Power of the acceptance bound: plausible kernel mistakes, planted in the
oracle's inputs on the CPU, must all be rejected by the same check the GPU
tests apply (tolerance.assert_within). Each mutant is what a kernel with that
mistake would compute exactly; a gate that let one through could not tell a
correct kernel from that broken one."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import assert_within


def _affine(N=64, K=1024, M=4, dtype="bf16", seed=1):
    W = synth.affine_weights(N, K, seed)
    packed, s, b = oracle.quantize(W, 4, 64, dtype)
    x = synth.activations(M, K, dtype, seed + 1)
    ref, absdot = oracle.qmm(packed, s, b, x, 4, 64, dtype)
    return packed, s, b, x, ref, absdot


def _rejected(got, ref, absdot, dtype):
    with pytest.raises(AssertionError):
        assert_within(got, ref, absdot, dtype, "mutant")


def test_correct_result_passes():
    packed, s, b, x, ref, absdot = _affine()
    assert_within(ref, ref, absdot, "bf16")


def test_swapped_nibble_order_rejected():
    packed, s, b, x, ref, absdot = _affine()
    w = packed.astype(np.uint32)
    swapped = ((w & 0x0F0F0F0F) << 4) | ((w >> 4) & 0x0F0F0F0F)
    got, _ = oracle.qmm(swapped.astype(np.uint32), s, b, x, 4, 64, "bf16")
    _rejected(got, ref, absdot, "bf16")


def test_dropped_bias_of_one_group_rejected():
    packed, s, b, x, ref, absdot = _affine()
    b2 = b.copy()
    b2[:, 5] = 0                      # bias term of group 5 lost (bf16 +0)
    got, _ = oracle.qmm(packed, s, b2, x, 4, 64, "bf16")
    _rejected(got, ref, absdot, "bf16")


def test_scale_of_neighbouring_group_rejected():
    packed, s, b, x, ref, absdot = _affine()
    s2 = np.roll(s, 1, axis=1)        # group g decoded with the scale of g - 1
    got, _ = oracle.qmm(packed, s2, b, x, 4, 64, "bf16")
    _rejected(got, ref, absdot, "bf16")


def test_lost_split_k_piece_rejected():
    packed, s, b, x, ref, absdot = _affine()
    K = x.shape[1]
    half = K // 2                     # the second of two K pieces never added
    got, _ = oracle.qmm(packed[:, : half // 8], s[:, : half // 64], b[:, : half // 64], x[:, :half], 4, 64, "bf16")
    _rejected(got, ref, absdot, "bf16")


def test_activation_rows_swapped_rejected():
    packed, s, b, x, ref, absdot = _affine()
    got, _ = oracle.qmm(packed, s, b, x[::-1].copy(), 4, 64, "bf16")
    _rejected(got, ref, absdot, "bf16")


def test_q8_0_codes_read_unsigned_rejected():
    N, K = 16, 512
    blocks = synth.q8_0_blocks(N, K, 3)
    x = synth.f32_vector(K, 4)
    ref, absdot = oracle.q8_0_gemv(blocks, x)
    # a kernel that zero-extends the code bytes computes the block sum with
    # q + 256 for every negative code: the same as adding 256 * d * (sum of x
    # over the negative codes' positions); built here from the oracle's own
    # per-weight decode
    w = np.stack([np.concatenate([oracle.q8_0_dequant_block(blocks[n, b]) for b in range(K // 32)])
                  for n in range(N)])
    d = np.repeat(np.array([[float(np.uint16(blocks[n, b, 0] & 0xFFFF).view(np.float16))
                             for b in range(K // 32)] for n in range(N)]), 32, axis=1)
    got = ((w + 256.0 * d * (w < 0)) * x.astype(np.float64)).sum(axis=1)
    _rejected(got, ref, absdot, "f32")


def test_q4_k_sub_block_scales_swapped_rejected():
    N, K = 16, 512
    blocks = synth.q4_k_blocks(N, K, 5)
    x = synth.f32_vector(K, 6)
    ref, absdot = oracle.q4_k_gemv(blocks, x)
    # scale bytes of sub-blocks 0 and 1 exchanged: (sc, m) of sub-block 2g
    # applied to 2g + 1 for g = 0 (low 6 bits of bytes 0/1 and 4/5)
    mut = blocks.copy()
    mut[:, :, [4, 5, 8, 9]] = blocks[:, :, [5, 4, 9, 8]]
    got, _ = oracle.q4_k_gemv(mut, x)
    _rejected(got, ref, absdot, "f32")


def test_q6_k_high_bits_at_wrong_shift_rejected():
    N, K = 16, 512
    blocks = synth.q6_k_blocks(N, K, 7)
    x = synth.f32_vector(K, 8)
    ref, absdot = oracle.q6_k_gemv(blocks, x)
    # a kernel that takes the high bit pairs of quarters 1 and 2 from each
    # other's positions: exchange bit pairs 2-3 and 4-5 of every qh byte
    mut = blocks.copy()
    qh = mut[:, :, 128:192]
    mut[:, :, 128:192] = (qh & 0xC3) | ((qh & 0x0C) << 2) | ((qh & 0x30) >> 2)
    got, _ = oracle.q6_k_gemv(mut, x)
    _rejected(got, ref, absdot, "f32")


def test_q8_0_34b_scale_from_wrong_byte_pair_rejected():
    N, K = 16, 512
    blocks = synth.q8_0_34b_blocks(N, K, 9)
    x = synth.f32_vector(K, 10)
    ref, absdot = oracle.q8_0_34b_gemv(blocks, x)
    mut = blocks.copy()
    mut[:, :, [0, 1]] = blocks[:, :, [1, 0]]   # the f16 scale read big-endian
    got, _ = oracle.q8_0_34b_gemv(mut, x)
    _rejected(got, ref, absdot, "f32")


def test_legitimate_rounding_accepted():
    """What a correct kernel may do stays inside the bound: weights rounded once
    to bf16 before the product (the tensor-core operand), products summed in
    binary32 in reverse order, the result rounded to bf16."""
    import torch
    packed, s, b, x, ref, absdot = _affine()
    K = x.shape[1]
    w = oracle.dequantize(packed, s, b, 4, 64, "bf16", K)
    w16 = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    xf = oracle.to_f64(x, "bf16").astype(np.float32)
    acc = np.zeros((x.shape[0], w.shape[0]), dtype=np.float32)
    for k in range(K - 1, -1, -1):
        acc += np.outer(xf[:, k], w16[:, k]).astype(np.float32)
    out = torch.from_numpy(acc).to(torch.bfloat16).to(torch.float64).numpy()
    assert_within(out, ref, absdot, "bf16", "legitimate rounding")
