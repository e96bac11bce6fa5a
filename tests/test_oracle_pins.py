"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle -- a wrong nibble or
bit order, a transposed operand, a dropped bias term, a wrong rounding mode, a
mis-decoded scale byte -- fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden, read_golden_rows

DTYPES = ("f32", "f16", "bf16")


def _store(vals, dtype):
    """float values -> storage array (exactly representable values only)."""
    a = np.asarray(vals, dtype=np.float32)
    if dtype == "f32":
        return a
    t = torch.from_numpy(a).to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# --------------------------------------------------------------------------
# storage formats, against numpy / torch conversions (library routines)
# --------------------------------------------------------------------------

def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.to_f64(bits, "f16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle.to_f64(bits, "bf16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _f32_samples():
    r = np.random.default_rng(7)
    rand_bits = r.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    a = [rand_bits.view(np.float32)]
    # every f16 value and the midpoints between neighbours (ties), nudged both ways
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    for v in (h, mids):
        v32 = v.astype(np.float32)
        a += [v32, -v32, np.nextafter(v32, np.float32(np.inf)), np.nextafter(v32, np.float32(0))]
    # bf16 neighbours and midpoints over a wide exponent range
    b = np.arange(0, 0x7F80, 7, dtype=np.uint32) << 16
    bv = b.view(np.float32).astype(np.float64)
    bm = ((bv[:-1] + bv[1:]) / 2).astype(np.float32)
    a += [bm, -bm, np.nextafter(bm, np.float32(np.inf))]
    a += [np.array([65504, 65519.99, 65520, 65536, 1e30, np.inf, -np.inf, 2**-24, 2**-25,
                    3 * 2**-26, 2**-14, 0.0, -0.0], dtype=np.float32)]
    out = np.concatenate(a).astype(np.float32)
    return out[~np.isnan(out)]


def test_f32_to_f16_rne_matches_numpy():
    x = _f32_samples()
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    L = oracle.lib()
    got = np.array([L.orc_f32_to_f16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_bf16_rne_matches_torch():
    x = _f32_samples()
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    L = oracle.lib()
    got = np.array([L.orc_f32_to_bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# packing order and the 4-bit worked example
# --------------------------------------------------------------------------

def _codes(spec):
    expr, rng_ = spec.split(" for i<")
    n = int(rng_)
    return [eval(expr, {"i": i}) for i in range(n)]  # noqa: S307  (fixture text, trusted)


@pytest.mark.parametrize("row", read_golden_rows("packing_widths.txt"), ids=lambda r: r[0] + "bit")
def test_packing_widths_golden(row):
    bits = int(row[0])
    codes = _codes(row[1])
    words = [int(w, 16) for w in row[2].split()]
    # independent construction: one Python integer as the row's bit stream
    stream = 0
    for i, q in enumerate(codes):
        stream |= q << (bits * i)
    assert [(stream >> (32 * j)) & 0xFFFFFFFF for j in range(len(words))] == words
    K = len(codes)
    q = np.array([codes], dtype=np.uint8)
    assert oracle.pack(q, bits).reshape(-1).tolist() == words
    assert oracle.unpack(np.array([words], dtype=np.uint32), bits, K).reshape(-1).tolist() == codes


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_pack_unpack_roundtrip_random(bits):
    r = np.random.default_rng(bits)
    q = r.integers(0, 2**bits, size=(5, 256), dtype=np.int64).astype(np.uint8)
    p = oracle.pack(q, bits)
    assert p.shape == (5, 256 * bits // 32)
    assert np.array_equal(oracle.unpack(p, bits, 256), q)
    # the stream is dense: every bit of every word belongs to exactly one code
    ones = oracle.pack(np.full((1, 256), 2**bits - 1, dtype=np.uint8), bits)
    assert np.all(ones == 0xFFFFFFFF)


@pytest.mark.parametrize("dtype", DTYPES)
def test_nibble_worked_example(dtype):
    g = read_golden("nibble_worked_example.txt")
    words = np.array([[int(w, 0) for w in g["words"].split()]], dtype=np.uint32)
    assert oracle.unpack(words, 4, 64)[0, :8].tolist() == [int(c) for c in g["codes"].split()]
    scales = _store([[float(g["scale"])]], dtype)
    biases = _store([[float(g["bias"])]], dtype)
    for case in ("a", "b"):
        xv = np.zeros(64, dtype=np.float32)
        xv[:8] = [float(v) for v in g[f"case_{case}_x"].split()]
        out, _ = oracle.qmm(words, scales, biases, _store(xv, dtype), 4, 64, dtype)
        assert out[0] == float(g[f"case_{case}_out"])


# --------------------------------------------------------------------------
# quantize: invariants and special cases
# --------------------------------------------------------------------------

def _quant_case(bits, gs, dtype, seed):
    W = synth.affine_weights(6, 4 * gs, seed)
    packed, s, b = oracle.quantize(W, bits, gs, dtype)
    q = oracle.unpack(packed, bits, W.shape[1]).astype(np.int64)
    sv = oracle.to_f64(s, dtype)
    bv = oracle.to_f64(b, dtype)
    return W, q, sv, bv


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("gs", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_quantize_roundtrip_bound(bits, gs, dtype):
    W, q, sv, bv = _quant_case(bits, gs, dtype, seed=bits * 1000 + gs)
    L = 2**bits - 1
    N, K = W.shape
    w = W.astype(np.float64).reshape(N, K // gs, gs)
    qg = q.reshape(N, K // gs, gs)
    s_ = sv[:, :, None]
    b_ = bv[:, :, None]
    what = s_ * qg + b_
    err = np.abs(w - what)
    mn = w.min(axis=2, keepdims=True)
    mx = w.max(axis=2, keepdims=True)
    s32 = ((mx - mn).astype(np.float32) / np.float32(L)).astype(np.float64)
    slack = s_ * 2.0**-14
    clamp_bound = np.maximum(s_ / 2, L * np.abs(s32 - s_) + np.abs(mn - b_))
    clamped = (qg == 0) | (qg == L)
    strict = np.broadcast_to(s_ / 2 + slack, err.shape)
    assert np.all(err[~clamped] <= strict[~clamped])
    assert np.all(err <= np.broadcast_to(clamp_bound + slack, err.shape))
    assert q.min() >= 0 and q.max() <= L
    # the group minimum and maximum are reproduced within s'/2 (plus rounding of s', b')
    assert np.all(np.abs(mn - (b_ + s_ * qg.min(axis=2, keepdims=True))) <= clamp_bound + slack)
    if dtype == "f32":
        # no rounding of s and b: the strict bound holds everywhere
        assert np.all(err <= s_ / 2 + slack)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_quantize_codes_are_nearest(bits, dtype):
    """Brute force: no other code is closer to w than the chosen one."""
    W, q, sv, bv = _quant_case(bits, 32, dtype, seed=5 + bits)
    N, K = W.shape
    L = 2**bits - 1
    codes = np.arange(L + 1, dtype=np.float64)
    s_ = np.repeat(sv, 32, axis=1)
    b_ = np.repeat(bv, 32, axis=1)
    w = W.astype(np.float64)
    dist_all = np.abs(w[:, :, None] - (s_[:, :, None] * codes + b_[:, :, None]))
    chosen = np.take_along_axis(dist_all, q[:, :, None], axis=2)[:, :, 0]
    assert np.all(chosen <= dist_all.min(axis=2) + s_ * 2.0**-14)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quantize_constant_group_and_ramp(bits, dtype):
    L = 2**bits - 1
    gs = 64
    # ramp w_i = b' + c_i * s' with codes c_i spanning 0..L and s', b' exact in every dtype
    s_exact, b_exact = 2.0**-6, -0.25
    i = np.arange(gs)
    codes = (i * L) // (gs - 1)
    ramp = (b_exact + codes * s_exact).astype(np.float32)
    const = np.full(gs, 0.0123, dtype=np.float32)
    W = np.stack([ramp, const]).astype(np.float32)
    packed, s, b = oracle.quantize(W, bits, gs, dtype)
    q = oracle.unpack(packed, bits, gs)
    sv = oracle.to_f64(s, dtype)
    bv = oracle.to_f64(b, dtype)
    assert sv[0, 0] == s_exact and bv[0, 0] == b_exact
    assert q[0].tolist() == codes.tolist()
    assert sv[1, 0] == 0.0 and np.all(q[1] == 0)
    assert bv[1, 0] == oracle.to_f64(_store([0.0123], dtype), dtype)[0]
    what = oracle.dequantize(packed, s, b, bits, gs, dtype, gs)
    assert np.all(what[1] == bv[1, 0])


# --------------------------------------------------------------------------
# qmm / qmv: the dot product against a library matmul
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("bits,gs", [(4, 64), (3, 32), (6, 128), (2, 64), (8, 32)])
def test_qmm_matches_library_matmul(bits, gs, dtype):
    N, K, M = 9, 3 * gs, 5
    W = synth.affine_weights(N, K, seed=11)
    packed, s, b = oracle.quantize(W, bits, gs, dtype)
    x = synth.activations(M, K, dtype, seed=12)
    out, absdot = oracle.qmm(packed, s, b, x, bits, gs, dtype)
    what = oracle.dequantize(packed, s, b, bits, gs, dtype, K)
    xf = oracle.to_f64(x, dtype)
    ref = torch.from_numpy(xf) @ torch.from_numpy(what).T          # [M, N] float64
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(absdot, (torch.from_numpy(xf).abs() @ torch.from_numpy(what).abs().T).numpy(),
                               rtol=1e-12, atol=1e-12)
    # the bias-hoisted form of the pages (scale * sum q*x + bias * sum x) gives the same value
    q = oracle.unpack(packed, bits, K).astype(np.float64).reshape(N, K // gs, gs)
    sv = oracle.to_f64(s, dtype)
    bv = oracle.to_f64(b, dtype)
    xg = xf.reshape(M, K // gs, gs)
    hoisted = np.einsum("ng,mng->mn", sv, np.einsum("ngi,mgi->mng", q, xg)) + \
        np.einsum("ng,mg->mn", bv, xg.sum(axis=2))
    np.testing.assert_allclose(out, hoisted, rtol=1e-11, atol=1e-12)


def test_qmm_rows_and_sampling_consistent():
    N, K, M, gs = 17, 256, 3, 64
    W = synth.affine_weights(N, K, seed=3)
    packed, s, b = oracle.quantize(W, 4, gs, "bf16")
    x = synth.activations(M, K, "bf16", seed=4)
    full, _ = oracle.qmm(packed, s, b, x, 4, gs, "bf16")
    rows = np.array([16, 0, 5], dtype=np.int64)
    part, _ = oracle.qmm(packed, s, b, x, 4, gs, "bf16", rows=rows)
    assert np.array_equal(part, full[:, rows])
    for m in range(M):
        one, _ = oracle.qmm(packed, s, b, x[m], 4, gs, "bf16")
        assert np.array_equal(one, full[m])


# --------------------------------------------------------------------------
# Q8_0
# --------------------------------------------------------------------------

def test_q8_0_worked_example():
    g = read_golden("q8_0_worked_example.txt")
    words = np.array([int(w, 0) for w in g["words"].split()], dtype=np.uint32)
    w = oracle.q8_0_dequant_block(words)
    assert w.tolist() == [0.5 * (j - 16) for j in range(32)]
    blocks = words.reshape(1, 1, 9)
    a, _ = oracle.q8_0_gemv(blocks, np.ones(32, dtype=np.float32))
    b, _ = oracle.q8_0_gemv(blocks, np.arange(32, dtype=np.float32))
    assert a[0] == float(g["case_a_out"]) and b[0] == float(g["case_b_out"])


def test_q8_0_closed_forms():
    N, K = 7, 32 * 12
    blocks = synth.q8_0_blocks(N, K, seed=9)
    d = oracle.to_f64((blocks[:, :, 0] & 0xFFFF).astype(np.uint16), "f16")
    ones = blocks.copy()
    ones[:, :, 1:] = 0x01010101                       # q == 1 everywhere
    out, _ = oracle.q8_0_gemv(ones, np.ones(K, dtype=np.float32))
    np.testing.assert_allclose(out, 32 * d.sum(axis=1), rtol=1e-14)
    ramp = blocks.copy()
    qb = (np.arange(32) - 16).astype(np.int8).view(np.uint8).view("<u4")
    ramp[:, :, 1:] = qb                               # q_j = j - 16
    out, _ = oracle.q8_0_gemv(ramp, np.ones(K, dtype=np.float32))
    np.testing.assert_allclose(out, -16 * d.sum(axis=1), rtol=1e-14)
    # the high half of word 0 is not part of the scale
    junk = blocks.copy()
    junk[:, :, 0] |= 0xABCD0000
    x = synth.f32_vector(K, seed=1)
    assert np.array_equal(oracle.q8_0_gemv(junk, x)[0], oracle.q8_0_gemv(blocks, x)[0])
    # the result is sum over blocks of d * (q . x): compare with a library matmul
    q = blocks[:, :, 1:].copy().view(np.uint8).view(np.int8).reshape(N, K).astype(np.float64)
    ref = (q * np.repeat(d, 32, axis=1)) @ x.astype(np.float64)
    np.testing.assert_allclose(oracle.q8_0_gemv(blocks, x)[0], ref, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Q4_K
# --------------------------------------------------------------------------

@pytest.mark.parametrize("row", read_golden_rows("q4k_scale_min.txt"), ids=lambda r: r[0])
def test_q4k_scale_min_table(row):
    sc12 = np.array([int(b, 16) for b in row[1].split()], dtype=np.uint8)
    want = [tuple(int(v) for v in p.split(",")) for p in row[2].split()]
    assert [oracle.q4_k_scale_min(sc12, j) for j in range(8)] == want


def _encode_scale_min(sc, m):
    """Pack eight 6-bit (scale, min) pairs into 12 bytes following the byte
    placement the decode implies (written from the layout, not from the
    decode): bytes 0-3 low 6 bits = sc0..3, bytes 4-7 low 6 bits = m0..3,
    bytes 8-11 = sc4..7 low nibble | m4..7 low nibble << 4, and the top two
    bits of bytes 0-3 / 4-7 carry bits 4-5 of sc4..7 / m4..7."""
    b = [0] * 12
    for j in range(4):
        b[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return np.array(b, dtype=np.uint8)


def test_q4k_scale_min_bijection():
    r = np.random.default_rng(21)
    for _ in range(3000):
        sc = r.integers(0, 64, size=8).tolist()
        m = r.integers(0, 64, size=8).tolist()
        got = [oracle.q4_k_scale_min(_encode_scale_min(sc, m), j) for j in range(8)]
        assert got == list(zip(sc, m))


def test_q4k_element_order():
    g = read_golden("q4k_element_order.txt")
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([int(g["d_bits"], 0)], dtype="<u2").view(np.uint8)
    blk[2:4] = np.array([int(g["dmin_bits"], 0)], dtype="<u2").view(np.uint8)
    blk[4:16] = [int(b, 16) for b in g["scales"].split()]
    blk[16:] = np.arange(128, dtype=np.uint8)
    w = oracle.q4_k_dequant_block(blk)
    for item in g["expect"].split():
        e, v = item.split(":")
        assert w[int(e)] == float(v), e


def test_q4k_gemv_matches_library_matmul():
    N, K = 5, 512
    blocks = synth.q4_k_blocks(N, K, seed=2)
    x = synth.f32_vector(K, seed=3)
    what = np.stack([np.concatenate([oracle.q4_k_dequant_block(blocks[n, b]) for b in range(K // 256)])
                     for n in range(N)])
    out, absdot = oracle.q4_k_gemv(blocks, x)
    np.testing.assert_allclose(out, what @ x.astype(np.float64), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(absdot, np.abs(what) @ np.abs(x.astype(np.float64)), rtol=1e-12)
    rows = np.array([4, 1], dtype=np.int64)
    assert np.array_equal(oracle.q4_k_gemv(blocks, x, rows=rows)[0], out[rows])


def test_oracle_rejects_bad_shapes():
    W = np.zeros((2, 96), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.quantize(W, 4, 64, "bf16")          # K not a multiple of the group size
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 64), np.float32), 5, 64, "bf16")   # unsupported width
    with pytest.raises(ValueError):
        oracle.q4_k_gemv(np.zeros((1, 1, 144), np.uint8), np.zeros(100, np.float32))


# --- Q8_0 with integer activations (hanzo-kernel quant.rs, dp4a matvecs) -------

def test_quantize_x_q8_invariants():
    """Per 32-element block: |q| <= 127, the largest |x| maps to +-127, every
    element is within d/2 of d*q, and an all-zero block gives q = 0, d = 0."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(32 * 6).astype(np.float32) * np.float32(3.0)
    x[32:64] = 0.0                      # an all-zero block
    x[64:96] = 0.0
    x[70] = np.float32(-0.75)           # a block with one non-zero element
    xq, xd = oracle.quantize_x_q8(x)
    for b in range(6):
        xb, qb, d = x[32 * b:32 * b + 32], xq[32 * b:32 * b + 32].astype(np.int64), float(xd[b])
        assert np.all(np.abs(qb) <= 127)
        if b == 1:
            assert d == 0.0 and np.all(qb == 0)
            continue
        i = int(np.argmax(np.abs(xb)))
        assert abs(int(qb[i])) == 127 and np.sign(qb[i]) == np.sign(xb[i])
        err = np.abs(xb.astype(np.float64) - d * qb)
        assert np.all(err <= d / 2 * (1 + 2.0 ** -20)), (b, err.max(), d)
    assert xq[70] == -127 and np.count_nonzero(xq[64:96]) == 1


def test_q8_0_block_dot_i8_brute_force():
    """The integer dot against a second decoding route: the 8 code words
    viewed as 32 little-endian signed bytes, summed with Python integers."""
    rng = np.random.default_rng(6)
    blocks = synth.q8_0_blocks(4, 32 * 5, 7)
    for n in range(4):
        for b in range(5):
            blk = blocks[n, b]
            xq = rng.integers(-128, 128, size=32).astype(np.int8)
            codes = np.frombuffer(blk[1:9].astype("<u4").tobytes(), dtype=np.int8)
            want = sum(int(c) * int(v) for c, v in zip(codes, xq))
            assert oracle.q8_0_block_dot_i8(blk, xq) == want


def test_q8_0_gemv_i8_exact_rational():
    """Tiny case in exact rational arithmetic: d_w (f16), xd (f32) and the
    integer dots are exact rationals; the oracle's binary64 sum is within a few
    ulps of the exact value."""
    from fractions import Fraction
    N, K = 3, 96
    blocks = synth.q8_0_blocks(N, K, 11)
    x = synth.f32_vector(K, 12)
    xq, xd = oracle.quantize_x_q8(x)
    got, _ = oracle.q8_0_gemv_i8(blocks, xq, xd)
    for n in range(N):
        total = Fraction(0)
        for b in range(K // 32):
            blk = blocks[n, b]
            dw = Fraction(float(np.array([blk[0] & 0xFFFF], dtype=np.uint16).view(np.float16)[0]))
            codes = np.frombuffer(blk[1:9].astype("<u4").tobytes(), dtype=np.int8)
            dot = sum(int(c) * int(v) for c, v in zip(codes, xq[32 * b:32 * b + 32]))
            total += dw * Fraction(float(xd[b])) * dot
        assert abs(got[n] - float(total)) <= 8 * np.spacing(abs(float(total))) + 1e-300


def test_q8_0_gemv_i8_agrees_with_the_float_path():
    """Against the a7 oracle on the dequantized activations x = xd * xq (f32):
    the two differ only by the f32 rounding of xd * xq."""
    N, K = 7, 32 * 12
    blocks = synth.q8_0_blocks(N, K, 21)
    xq, xd = oracle.quantize_x_q8(synth.f32_vector(K, 22))
    x_deq = (xq.astype(np.float32).reshape(-1, 32) * xd[:, None]).reshape(-1)
    a, absdot = oracle.q8_0_gemv_i8(blocks, xq, xd)
    b, _ = oracle.q8_0_gemv(blocks, x_deq)
    assert np.all(np.abs(a - b) <= 2.0 ** -22 * absdot)


def test_q8_0_gemv_i8_closed_form():
    """q_w = 1 and q_x = 1 everywhere: out[n] = 32 * sum_b d_w[n, b] * xd[b]."""
    N, K = 4, 32 * 3
    blocks = synth.q8_0_blocks(N, K, 31)
    blocks[:, :, 1:] = 0x01010101
    xq = np.ones(K, dtype=np.int8)
    xd = np.array([0.5, 0.25, 2.0], dtype=np.float32)
    got, _ = oracle.q8_0_gemv_i8(blocks, xq, xd)
    dw = (blocks[:, :, 0] & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, 32 * (dw * xd.astype(np.float64)).sum(axis=1))


# --------------------------------------------------------------------------
# GGUF block layouts beyond the pages (34-byte Q8_0, Q6_K). The layouts are a
# reading (the GGUF format's published block definitions); these pins tie the
# oracle to that reading through a second, byte-oriented formulation.
# --------------------------------------------------------------------------

def _q8_0_34b_from_words(blocks9):
    """the same (d, q) as a nine-word Q8_0 block, in the 34-byte layout"""
    N, nb, _ = blocks9.shape
    out = np.empty((N, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = (blocks9[:, :, 0] & 0xFFFF).astype(np.uint16).view(np.uint8).reshape(N, nb, 2)
    out[:, :, 2:] = np.ascontiguousarray(blocks9[:, :, 1:]).view(np.uint8).reshape(N, nb, 32)
    return out


def test_q8_0_34b_equals_nine_word_layout():
    N, K = 7, 320
    b9 = synth.q8_0_blocks(N, K, 71)
    b34 = _q8_0_34b_from_words(b9)
    x = synth.f32_vector(K, 72)
    want, wabs = oracle.q8_0_gemv(b9, x)
    got, gabs = oracle.q8_0_34b_gemv(b34, x)
    assert np.array_equal(got, want) and np.array_equal(gabs, wabs)


def test_q8_0_34b_block_decode_by_numpy():
    b = synth.q8_0_34b_blocks(3, 64, 73)
    for blk in b.reshape(-1, 34):
        d = float(blk[0:2].copy().view(np.float16)[0])
        q = blk[2:].view(np.int8).astype(np.float64)
        assert np.array_equal(oracle.q8_0_34b_dequant_block(blk), d * q)


def _q6_k_encode(u, sc, d_f16):
    """Q6_K super-block from unsigned codes u = q + 32 (0..63), 16 int8 scales
    and an f16 d, built byte by byte: ql byte i of half h (i = 64h + r) holds
    element 128h + r in its low nibble and element 128h + 64 + r in its high
    nibble; qh byte 32h + l holds the top two bits of elements 128h + l,
    128h + 32 + l, 128h + 64 + l, 128h + 96 + l at bits 0-1, 2-3, 4-5, 6-7."""
    u = [int(v) for v in u]
    blk = bytearray(210)
    for i in range(128):
        h, r = divmod(i, 64)
        blk[i] = (u[128 * h + r] & 15) | ((u[128 * h + 64 + r] & 15) << 4)
    for i in range(64):
        h, l = divmod(i, 32)
        v = 0
        for k in range(4):
            v |= ((u[128 * h + 32 * k + l] >> 4) & 3) << (2 * k)
        blk[128 + i] = v
    blk[192:208] = np.asarray(sc, dtype=np.int8).tobytes()
    blk[208:210] = np.asarray([d_f16], dtype=np.float16).tobytes()
    return np.frombuffer(bytes(blk), dtype=np.uint8).copy()


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_q6_k_round_trip_through_encoder(seed):
    r = np.random.default_rng(seed)
    q = r.integers(-32, 32, size=256)
    sc = r.integers(-128, 128, size=16)
    d = np.float16(r.uniform(1e-3, 1e-1))
    blk = _q6_k_encode(q + 32, sc, d)
    assert np.array_equal(oracle.q6_k_codes(blk), q)
    want = float(d) * sc[np.arange(256) // 16].astype(np.float64) * q.astype(np.float64)
    assert np.array_equal(oracle.q6_k_dequant_block(blk), want)


def test_q6_k_every_code_value_and_range():
    blk = _q6_k_encode(np.arange(256) % 64, np.ones(16, dtype=np.int64), np.float16(1.0))
    codes = oracle.q6_k_codes(blk)
    assert np.array_equal(codes, np.arange(256) % 64 - 32)
    rnd = synth.q6_k_blocks(4, 1024, 74).reshape(-1, 210)
    allc = np.concatenate([oracle.q6_k_codes(b) for b in rnd])
    assert allc.min() == -32 and allc.max() == 31 and len(np.unique(allc)) == 64


def test_q6_k_zero_bytes_closed_form():
    """ql = qh = 0: every code is -32, so w_e = -32 * d * sc[e // 16]."""
    sc = np.arange(-8, 8, dtype=np.int64) * 9
    blk = _q6_k_encode(np.zeros(256, dtype=np.int64), sc, np.float16(0.5))
    assert np.array_equal(oracle.q6_k_dequant_block(blk), -16.0 * sc[np.arange(256) // 16].astype(np.float64))


def test_q6_k_single_bit_moves_one_code():
    """Each of the 1536 code bits (ql, qh) changes exactly one element's code, by
    the bit's weight (1, 2, 4, 8 for ql nibble bits, 16 or 32 for qh bits), and
    all 256 elements x 6 bits are reached exactly once."""
    base = np.zeros(210, dtype=np.uint8)
    base[192:208] = 1
    base[208:210] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    q0 = oracle.q6_k_codes(base)
    seen = {}
    for byte in range(192):
        for bit in range(8):
            blk = base.copy()
            blk[byte] = 1 << bit
            diff = oracle.q6_k_codes(blk) - q0
            nz = np.flatnonzero(diff)
            assert len(nz) == 1, (byte, bit)
            e = int(nz[0])
            step = int(diff[e])
            if byte < 128:
                assert step == 1 << (bit % 4)
            else:
                assert step == 16 << (bit % 2)
            key = (e, step)
            assert key not in seen
            seen[key] = (byte, bit)
    assert len(seen) == 256 * 6


def test_q6_k_gemv_exact_rational():
    from fractions import Fraction
    r = np.random.default_rng(5)
    N, K = 3, 512
    q = r.integers(-32, 32, size=(N, K // 256, 256))
    sc = r.integers(-128, 128, size=(N, K // 256, 16))
    d = r.uniform(1e-3, 1e-1, size=(N, K // 256)).astype(np.float16)
    blocks = np.stack([np.stack([_q6_k_encode(q[n, b] + 32, sc[n, b], d[n, b]) for b in range(K // 256)])
                       for n in range(N)])
    x = synth.f32_vector(K, 75)
    got, _ = oracle.q6_k_gemv(blocks, x)
    for n in range(N):
        exact, mag = Fraction(0), Fraction(0)
        for k in range(K):
            b, e = divmod(k, 256)
            t = Fraction(float(d[n, b])) * int(sc[n, b, e // 16]) * int(q[n, b, e]) * Fraction(float(x[k]))
            exact += t
            mag += abs(t)
        # K binary64 additions: |error| <= K * 2^-53 * sum |terms|
        assert abs(Fraction(got[n]) - exact) <= mag * K / Fraction(2 ** 53)
