"""Stray-store checks: every entry point writes its outputs (and, where it has
one, its split-K workspace) into a view of a larger device buffer whose
padding on both sides holds a byte pattern; after the call the padding must be
unchanged. Shapes are ragged so that tail tiles, partial M chunks, scalar
reduce paths and the general (non-staged) kernels run. Each output is also
checked against the oracle where that is cheap."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import TORCH_DTYPE, affine_problem, to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu

PAD = 4096          # bytes of padding on each side (keeps the views 16-byte aligned)
PATTERN = 0xA5


class Canary:
    """A contiguous tensor of `shape` and `dtype` inside a padded byte buffer."""

    def __init__(self, shape, dtype):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((PAD + self.nbytes + PAD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        raw = self.raw.cpu().numpy()
        assert np.all(raw[:PAD] == PATTERN), f"{what}: a store landed before the buffer"
        assert np.all(raw[PAD + self.nbytes:] == PATTERN), f"{what}: a store landed past the buffer"


@pytest.mark.parametrize("N,K", [(131, 1088), (131, 4096), (1, 64)])
def test_qmv(N, K):
    _, packed, s, b, x = affine_problem(N, K, 1, 4, 64, "bf16", seed=N + K)
    out = Canary((N,), torch.bfloat16)
    g4.gai4_qmv(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x[0], "bf16"), out=out.t)
    out.check(f"qmv N={N} K={K}")
    ref, absdot = oracle.qmm(packed, s, b, x[0], 4, 64, "bf16")
    assert_within(to_host_f64(out.t, "bf16"), ref, absdot, "bf16", "qmv")


# (N, K, M, dtype, bits, split): tensor core with and without split-K (ragged
# N: scalar reduce; N % 8 == 0: vector reduce; M = 300: a ragged second chunk),
# the CUDA-core kernel (f32, 3-bit)
QMM_CASES = [(131, 2048, 9, "bf16", 4, 1), (131, 2048, 9, "bf16", 4, 2), (136, 2048, 9, "bf16", 4, 4),
             (131, 1024, 300, "bf16", 4, 2), (67, 1024, 5, "f32", 4, 1), (67, 1152, 2, "bf16", 3, 1)]


@pytest.mark.parametrize("N,K,M,dtype,bits,split", QMM_CASES)
def test_qmm_t_and_workspace(N, K, M, dtype, bits, split):
    _, packed, s, b, x = affine_problem(N, K, M, bits, 64, dtype, seed=N + K + M)
    T = TORCH_DTYPE[dtype]
    out = Canary((M, N), T)
    ws_bytes = g4.gai4_qmm_t_workspace_bytes(M, N, K, bits, 64, T, split)
    ws = Canary((max(ws_bytes, 16) // 4,), torch.float32)
    g4.gai4_qmm_t(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), to_dev(x, dtype), out=out.t, bits=bits,
                  group_size=64, split_k=split, workspace=ws.t)
    assert g4.gai4_last_device_status() == 0
    out.check(f"qmm_t out N={N} K={K} M={M} S={split}")
    ws.check(f"qmm_t workspace N={N} K={K} M={M} S={split}")
    ref, absdot = oracle.qmm(packed, s, b, x, bits, 64, dtype)
    assert_within(to_host_f64(out.t, dtype), ref, absdot, dtype, "qmm_t")


def test_qmm_t_noalloc():
    N, K, M = 131, 2048, 9
    _, packed, s, b, x = affine_problem(N, K, M, 4, 64, "bf16", seed=5)
    out = Canary((M, N), torch.bfloat16)
    g4.gai4_qmm_t_noalloc(to_dev(packed), to_dev(s, "bf16"), to_dev(b, "bf16"), to_dev(x, "bf16"), out.t,
                          split_k=2)
    out.check("qmm_t_noalloc")


def test_qmm_t_batched_gathered():
    Bt, M, N, K = 2, 9, 131, 1024
    mats = [oracle.quantize(synth.affine_weights(N, K, 40 + e), 4, 64, "bf16") for e in range(Bt)]
    P = to_dev(np.stack([m[0] for m in mats]))
    S = to_dev(np.stack([m[1] for m in mats]), "bf16")
    Bi = to_dev(np.stack([m[2] for m in mats]), "bf16")
    base = to_dev(synth.activations(1, Bt * M * (K + 8) + 16, "bf16", 41)[0], "bf16")
    x = torch.as_strided(base, (Bt, M, K), (M * (K + 8), K + 8, 1), 1)   # odd element offset: gathered
    out = Canary((Bt, M, N), torch.bfloat16)
    ws_bytes = g4.gai4_qmm_t_batched_workspace_bytes(Bt, M, N, K, 4, 64, torch.bfloat16, 2)
    ws = Canary((max(ws_bytes, 16) // 4,), torch.float32)
    g4.gai4_qmm_t_batched(P, S, Bi, x, out=out.t, split_k=2, workspace=ws.t)
    assert g4.gai4_last_device_status() == 0
    out.check("qmm_t_batched out")
    ws.check("qmm_t_batched workspace")


@pytest.mark.parametrize("bits", [4, 3])
def test_quantize_unpack_dequantize(bits):
    N, K, gs = 67, 1152, 64
    W = to_dev(synth.affine_weights(N, K, bits))
    p = Canary((N, K * bits // 32), torch.int32)
    s = Canary((N, K // gs), torch.bfloat16)
    b = Canary((N, K // gs), torch.bfloat16)
    g4.gai4_quantize(W, bits, gs, torch.bfloat16, w_packed=p.t, scales=s.t, biases=b.t)
    for c, what in ((p, "packed"), (s, "scales"), (b, "biases")):
        c.check(f"quantize {what} bits={bits}")
    q = Canary((N, K), torch.uint8)
    g4.gai4_unpack(p.t, bits, K, q_out=q.t)
    q.check(f"unpack bits={bits}")
    w = Canary((N, K), torch.float32)
    g4.gai4_dequantize(p.t, s.t, b.t, bits=bits, group_size=gs, out=w.t)
    w.check(f"dequantize bits={bits}")


# staged (TMA) and general kernels of the block formats
@pytest.mark.parametrize("N,K", [(67, 4096), (67, 1056), (3, 65536)])
def test_q8_0_and_int8(N, K):
    blocks = to_dev(synth.q8_0_blocks(N, K, N + K))
    x = synth.f32_vector(K, K)
    out = Canary((N,), torch.float32)
    g4.gai4_q8_0_gemv(blocks, to_dev(x), out=out.t)
    out.check(f"q8_0 N={N} K={K}")
    xq = Canary((K,), torch.int8)
    xd = Canary((K // 32,), torch.float32)
    g4.gai4_quantize_x_q8(to_dev(x), xq=xq.t, xd=xd.t)
    xq.check("quantize_x_q8 codes")
    xd.check("quantize_x_q8 scales")
    out8 = Canary((N,), torch.float32)
    g4.gai4_q8_0_gemv_i8(blocks, xq.t, xd.t, out=out8.t)
    out8.check(f"q8_0 int8 N={N} K={K}")


@pytest.mark.parametrize("N,K", [(67, 4096), (3, 65536)])
def test_q4_k(N, K):
    out = Canary((N,), torch.float32)
    g4.gai4_q4_k_gemv(to_dev(synth.q4_k_blocks(N, K, N)), to_dev(synth.f32_vector(K, 2)), out=out.t)
    out.check(f"q4_k N={N} K={K}")


@pytest.mark.parametrize("N,K", [(67, 1024), (3, 2304), (1, 256)])
def test_gguf_blocks(N, K):
    x = to_dev(synth.f32_vector(K, 3))
    out = Canary((N,), torch.float32)
    g4.gai4_q8_0_34b_gemv(to_dev(synth.q8_0_34b_blocks(N, K, N)), x, out=out.t)
    out.check(f"q8_0 34-byte N={N} K={K}")
    out6 = Canary((N,), torch.float32)
    g4.gai4_q6_k_gemv(to_dev(synth.q6_k_blocks(N, K, N)), x, out=out6.t)
    out6.check(f"q6_k N={N} K={K}")
