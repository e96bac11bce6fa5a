"""GPU quantize / unpack / dequantize against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

DTYPES = ("f32", "f16", "bf16")


def _bits_equal(t: torch.Tensor, ref: np.ndarray):
    got = t.cpu().contiguous()
    if ref.dtype == np.uint16:
        got = got.view(torch.int16).numpy().view(np.uint16)
    elif ref.dtype == np.uint32:
        got = got.view(torch.int32).numpy().view(np.uint32)
    else:
        got = got.numpy()
        return np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    return np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_quantize_bit_exact(bits, gs, dtype):
    N, K = 37, 3 * 128
    W = synth.affine_weights(N, K, seed=bits * 10 + gs)
    W[3, :gs] = 0.25                        # a constant group (scale 0)
    W[5, gs:2 * gs] = np.linspace(-1, 1, gs, dtype=np.float32)
    p_ref, s_ref, b_ref = oracle.quantize(W, bits, gs, dtype)
    p, s, b = g4.gai4_quantize(to_dev(W), bits, gs, {"f32": torch.float32, "f16": torch.float16,
                                                     "bf16": torch.bfloat16}[dtype])
    torch.cuda.synchronize()
    assert _bits_equal(p, p_ref)
    assert _bits_equal(s, s_ref)
    assert _bits_equal(b, b_ref)


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_unpack_bit_exact(bits):
    r = np.random.default_rng(bits)
    q = r.integers(0, 2**bits, size=(19, 320), dtype=np.int64).astype(np.uint8)
    packed = oracle.pack(q, bits)
    got = g4.gai4_unpack(to_dev(packed), bits, 320)
    assert np.array_equal(got.cpu().numpy(), q)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits,gs", [(4, 64), (3, 128), (8, 32)])
def test_dequantize_bit_exact(bits, gs, dtype):
    N, K = 11, 256 if bits != 3 else 384
    W = synth.affine_weights(N, K, seed=3)
    packed, s, b = oracle.quantize(W, bits, gs, dtype)
    what = oracle.dequantize(packed, s, b, bits, gs, dtype, K)   # exact in fp64
    got = g4.gai4_dequantize(to_dev(packed), to_dev(s, dtype), to_dev(b, dtype), bits, gs)
    # one rounding of the exact value to binary32 on both sides
    assert np.array_equal(got.cpu().numpy(), what.astype(np.float32))


def test_quantize_full_size_4bit():
    """The 4096 x 4096 4-bit gs64 bf16 matrix of the headline qmv shape."""
    W = synth.affine_weights(4096, 4096, seed=0)
    p_ref, s_ref, b_ref = oracle.quantize(W, 4, 64, "bf16")
    p, s, b = g4.gai4_quantize(to_dev(W), 4, 64, torch.bfloat16)
    assert _bits_equal(p, p_ref) and _bits_equal(s, s_ref) and _bits_equal(b, b_ref)
