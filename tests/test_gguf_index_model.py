"""CPU model of the address arithmetic of gguf_gemv.cu (GGUF 34-byte Q8_0 and
Q6_K GEMVs): for many shapes, every 16-byte copy starts inside the weight
buffer and lands inside its shared-memory stage, every shared read of the
decode stays inside the stage, every activation read inside x, and every row
is written exactly once; on small shapes the modelled lanes' decode, taken in
binary64, equals the oracle. The kernel's constants are read from its source."""
import os
import re

import numpy as np
import pytest

import oracle
import synth

SRC = os.path.join(os.path.dirname(__file__), "..", "gemm_affine_int4_gb300", "csrc", "gguf_gemv.cu")


def _consts():
    text = open(SRC).read()
    out = {}
    for fmt in (0, 1):
        m = re.search(r"struct GgufFmt<%d> \{[^}]*?static constexpr int ([^;]*);" % fmt, text, re.S)
        out[fmt] = {k.strip(): int(v) for k, v in (kv.split("=") for kv in m.group(1).split(","))}
    out["warps"] = int(re.search(r"constexpr int kWarps = (\d+);", text).group(1))
    m = re.search(r"std::min<int64_t>\((\d+), \(int64_t\)\((\d+) \* 1024\) / \(int64_t\)\(smem \+ (\d+)\)\)", text)
    out["ctas_per_sm_max"], out["smem_kb"], out["smem_slack"] = (int(g) for g in m.groups())
    out["max_smem_x"] = int(re.search(r"constexpr int64_t kMaxSmemX = (\d+);", text).group(1))
    return out


def _grid(fmt, N, K, sms):
    """The launcher's grid: CTAs of kWarps warps, as many per SM as the shared
    memory (stage ring, plus x when it is staged) allows, up to the cap."""
    F = C[fmt]
    ring = C["warps"] * F["kStages"] * F["kCPL"] * 512
    smem = ring + (4 * K if K <= C["max_smem_x"] else 0)
    per_sm = max(1, min(C["ctas_per_sm_max"], (C["smem_kb"] * 1024) // (smem + C["smem_slack"])))
    return min((N + C["warps"] - 1) // C["warps"], per_sm * sms), smem


C = _consts()


def _u32_at(buf, o):
    a = o & ~3
    w = int.from_bytes(bytes(buf[a:a + 8]), "little")
    return (w >> ((o & 3) * 8)) & 0xFFFFFFFF


def _model(fmt, N, K, sms=152, flat=None, x=None):
    """Walk every warp's items as the kernel does; returns the modelled output
    (binary64) when `flat` and `x` are given, else only checks bounds."""
    F = C[fmt]
    BB, BK, SB, CPL = F["kBB"], F["kBK"], F["kSB"], F["kCPL"]
    stage = CPL * 512
    nb = K // BK
    total = N * nb * BB
    RB = nb * BB
    nslab = (nb + SB - 1) // SB
    warps = C["warps"]
    grid, smem = _grid(fmt, N, K, sms)
    assert smem <= C["smem_kb"] * 1024
    wstride = grid * warps
    out = np.full(N, np.nan)
    written = np.zeros(N, dtype=np.int64)
    for w in range(grid * warps):
        n_items = ((N - 1 - w) // wstride + 1) * nslab if w < N else 0
        acc = 0.0
        for t in range(n_items):
            r = w + (t // nslab) * wstride
            s = t % nslab
            nbs = min(SB, nb - s * SB)
            start = r * RB + s * SB * BB
            a0 = start & ~15
            mis = start - a0
            nch = (mis + nbs * BB + 15) >> 4
            assert nch <= CPL * 32                                   # chunks fit the lanes' share of a stage
            g_first, g_last = a0, a0 + 16 * (nch - 1)
            assert 0 <= g_first and g_last < total                  # every copy starts inside the weights
            assert 16 * nch <= stage
            # decode reads: the highest shared byte touched (aligned word pair of the last re-aligned load)
            if fmt == 0:
                o_max = mis + 34 * (nbs - 1) + 2 + 28
                x_max = (s * SB + nbs - 1) * 32 + 28 + 4
            else:
                o_max = mis + 210 * (nbs - 1) + 128 + 32 + 28
                o_max = max(o_max, mis + 210 * (nbs - 1) + 208 + 1)
                x_max = (s * SB + nbs - 1) * 256 + 128 + 60 + 64 + 4
            assert (o_max & ~3) + 8 <= stage
            assert x_max <= K
            if flat is not None:
                buf = np.zeros(stage + 8, dtype=np.uint8)
                for c in range(nch):
                    g = a0 + 16 * c
                    n = min(16, total - g)
                    buf[16 * c:16 * c + n] = flat[g:g + n]
                acc += _decode(fmt, buf, mis, x, s * SB, nbs)
            if s == nslab - 1:
                written[r] += 1
                out[r] = acc
                acc = 0.0
    assert np.all(written == 1)
    return out


def _decode(fmt, buf, m, x, b0, nbs):
    acc = 0.0
    for lane in range(32):
        if fmt == 0:
            e4 = (lane & 7) * 4
            for jb in range(lane >> 3, nbs, 4):
                o = m + 34 * jb
                d = float(buf[o:o + 2].copy().view(np.float16)[0])
                w = _u32_at(buf, o + 2 + e4) ^ 0x80808080
                xi = (b0 + jb) * 32 + e4
                acc += d * sum((((w >> (8 * k)) & 0xFF) - 128) * float(x[xi + k]) for k in range(4))
        else:
            h, r = lane >> 4, (lane & 15) * 4
            for jb in range(nbs):
                o = m + 210 * jb
                qlw = _u32_at(buf, o + 4 * lane)
                q2 = _u32_at(buf, o + 128 + 32 * h + (r & 31)) >> ((r >> 5) * 2)
                sl = int(np.int8(buf[o + 192 + 8 * h + (r >> 4)]))
                sh = int(np.int8(buf[o + 196 + 8 * h + (r >> 4)]))
                d = float(buf[o + 208:o + 210].copy().view(np.float16)[0])
                xb = (b0 + jb) * 256 + 128 * h + r
                lo = (qlw & 0x0F0F0F0F) | ((q2 << 4) & 0x30303030)
                hi = ((qlw >> 4) & 0x0F0F0F0F) | (q2 & 0x30303030)
                a = sum((((lo >> (8 * k)) & 0xFF) - 32) * float(x[xb + k]) for k in range(4))
                b = sum((((hi >> (8 * k)) & 0xFF) - 32) * float(x[xb + 64 + k]) for k in range(4))
                acc += d * (sl * a + sh * b)
    return acc


@pytest.mark.parametrize("fmt,N,K,sms", [(0, 3, 32, 152), (0, 9, 1088, 152), (0, 17, 2080, 1), (0, 5, 32 * 33, 152),
                                         (1, 3, 256, 152), (1, 9, 2304, 1), (1, 7, 256 * 17, 152), (1, 1, 256, 152)])
def test_modelled_decode_equals_oracle(fmt, N, K, sms):
    gen, ref_fn = (synth.q8_0_34b_blocks, oracle.q8_0_34b_gemv) if fmt == 0 else (synth.q6_k_blocks, oracle.q6_k_gemv)
    blocks = gen(N, K, N + K)
    x = synth.f32_vector(K, 3)
    got = _model(fmt, N, K, sms, blocks.reshape(-1), x)
    ref, absdot = ref_fn(blocks, x)
    assert np.all(np.abs(got - ref) <= 1e-12 * absdot)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (4096, 4096), (4099, 3072), (14336, 5120), (33, 14336),
                                 (1000, 65536)])
def test_addresses_in_bounds(fmt, N, K):
    _model(fmt, N, K, sms=152 if N < 5000 else 4)   # few SMs on the large shapes: many rows per warp
