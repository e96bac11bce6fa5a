"""GPU batched / strided qmm_t (gai4_qmm_t_batched) against the fp64 oracle:
stacked and shared weights, strided and odd-offset activations, every path
(tensor core with and without split-K, the CUDA-core kernel, qmv)."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import TORCH_DTYPE, to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def _weights(E, N, K, bits, gs, dtype, seed):
    mats = [oracle.quantize(synth.affine_weights(N, K, seed + e), bits, gs, dtype) for e in range(E)]
    return [m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats]


def _strided_x(B, M, K, dtype, seed, row_pad, batch_pad, offset):
    """x [B, M, K] as a view of a larger buffer: rows K + row_pad apart,
    batches (M + batch_pad) rows apart, starting `offset` elements in."""
    xs = [synth.activations(M, K, dtype, seed + b) for b in range(B)]
    rs = K + row_pad
    total = offset + B * (M + batch_pad) * rs + 64
    if dtype == "f32":
        buf = np.zeros(total, np.float32)
    else:
        buf = np.zeros(total, np.uint16)
    for b in range(B):
        for m in range(M):
            o = offset + b * (M + batch_pad) * rs + m * rs
            buf[o:o + K] = xs[b][m]
    dev = to_dev(buf, dtype)
    view = torch.as_strided(dev, (B, M, K), ((M + batch_pad) * rs, rs, 1), offset)
    return xs, view


CASES = [
    # (dtype, bits, gs, B, M, N, K, stacked weights, row_pad, batch_pad, offset)
    ("bf16", 4, 64, 3, 33, 256, 1024, True, 8, 3, 1),     # tensor core, gathered (odd offset)
    ("bf16", 4, 64, 2, 8, 384, 2048, False, 0, 0, 0),     # tensor core, contiguous, shared weights
    ("bf16", 4, 64, 2, 40, 512, 4096, True, 24, 0, 8),    # tensor core + split-K, gathered
    ("f16", 4, 32, 2, 1, 1000, 4096, True, 0, 5, 3),      # qmv (M = 1), gathered
    ("f32", 3, 128, 2, 5, 300, 1024, True, 16, 1, 2),     # CUDA-core kernel, gathered
    ("bf16", 8, 64, 3, 17, 130, 512, False, 64, 0, 0),    # 8-bit, tensor core or CUDA core, strided rows
]


@pytest.mark.parametrize("dtype,bits,gs,B,M,N,K,stacked,row_pad,batch_pad,offset", CASES)
def test_batched_matches_oracle(dtype, bits, gs, B, M, N, K, stacked, row_pad, batch_pad, offset):
    E = B if stacked else 1
    packed, s, b = _weights(E, N, K, bits, gs, dtype, seed=500 + B * M + N)
    xs, x = _strided_x(B, M, K, dtype, 900 + M, row_pad, batch_pad, offset)
    w_dev = to_dev(np.stack(packed) if stacked else packed[0])
    s_dev = to_dev(np.stack(s) if stacked else s[0], dtype)
    b_dev = to_dev(np.stack(b) if stacked else b[0], dtype)
    out = g4.gai4_qmm_t_batched(w_dev, s_dev, b_dev, x, bits=bits, group_size=gs)
    assert g4.gai4_last_device_status() == 0
    got = to_host_f64(out, dtype)
    for bb in range(B):
        e = bb if stacked else 0
        ref, absdot = oracle.qmm(packed[e], s[e], b[e], xs[bb], bits, gs, dtype)
        assert_within(got[bb], ref, absdot, dtype, f"batch {bb} of {dtype} b{bits} gs{gs} B{B} M{M} N{N} K{K}")


@pytest.mark.parametrize("split", [1, 2])
def test_batched_equals_single_calls(split):
    """With the same split, each batch of a batched call (one tensor-core
    launch over all batches) equals gai4_qmm_t on that batch's contiguous
    activations, bit for bit."""
    dtype, bits, gs, B, M, N, K = "bf16", 4, 64, 3, 24, 512, 2048
    packed, s, b = _weights(B, N, K, bits, gs, dtype, seed=77)
    xs, x = _strided_x(B, M, K, dtype, 78, 40, 2, 5)
    w_dev, s_dev, b_dev = to_dev(np.stack(packed)), to_dev(np.stack(s), dtype), to_dev(np.stack(b), dtype)
    ws = torch.empty(g4.gai4_qmm_t_batched_workspace_bytes(B, M, N, K, bits, gs, TORCH_DTYPE[dtype], split) // 4
                     + 64, dtype=torch.float32, device="cuda")
    out = g4.gai4_qmm_t_batched(w_dev, s_dev, b_dev, x, bits=bits, group_size=gs, split_k=split, workspace=ws)
    for bb in range(B):
        single_ws = torch.empty(g4.gai4_qmm_t_workspace_bytes(M, N, K, bits, gs, TORCH_DTYPE[dtype], split) // 4
                                + 64, dtype=torch.float32, device="cuda")
        one = g4.gai4_qmm_t(w_dev[bb], s_dev[bb], b_dev[bb], to_dev(xs[bb], dtype), bits=bits, group_size=gs,
                            split_k=split, workspace=single_ws)
        assert torch.equal(out[bb], one), bb
