// gguf_gemv.cu -- matrix-vector products over two GGUF block layouts that
// hanzo-kernel quant.rs names but does not write out (read from the GGUF
// format's published block definitions):
//   Q8_0, 34 bytes per 32 weights: bytes 0..1 the f16 scale d, bytes 2..33
//     the int8 codes; w_j = d * q_j (the same block as the nine-word Q8_0
//     layout of gai4_q8_0_gemv, without its padding).
//   Q6_K, 210 bytes per 256 weights: ql[128] low nibbles, qh[64] high bit
//     pairs, sc[16] int8 scales, f16 d. Element e = 128h + 32c + l (h < 2,
//     c < 4, l < 32) has code q = nibble c/2 of ql[64h + 32(c%2) + l]
//     + 16 * bits 2c..2c+1 of qh[32h + l] - 32, and w_e = d * sc[e/16] * q.
//
// Neither block size is a multiple of four bytes, so a block cannot be read in
// place with aligned word loads. Each warp owns one output row at a time and
// walks it in slabs of whole blocks (one contiguous run of the row's bytes).
// A slab is fetched with 16-byte streaming loads starting at the 16-byte
// boundary at or below it, into registers one slab ahead of the decode; it is
// then written to a warp-private shared-memory buffer, from which words at
// 2-byte-aligned offsets are read as two aligned words and a funnel shift.
// A code c becomes a float through the mantissa of 2^23: a byte permute puts
// c under the exponent byte 0x4B, and one subtraction removes 2^23 and the
// code's offset (128 for Q8_0 bytes with the sign bit flipped, 32 for Q6_K)
// exactly. Products and sums are binary32; the block scale is applied once
// per block (Q8_0) or once per 4-weight run of one 16-weight scale group
// (Q6_K), and a warp-shuffle sum finishes each row.
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace gai4 {
namespace {

constexpr int kWarps = 8;   // warps per CTA

template <int FMT>
struct GgufFmt;
template <>
struct GgufFmt<0> {   // Q8_0, 34-byte blocks
    static constexpr int kBB = 34, kBK = 32, kSB = 32, kCPL = 3;
};
template <>
struct GgufFmt<1> {   // Q6_K, 210-byte super-blocks
    static constexpr int kBB = 210, kBK = 256, kSB = 8, kCPL = 4;
};
// a slab of kSB blocks plus up to 15 leading bytes fits the kCPL x 32 16-byte
// chunks the lanes hold, and leaves room for the one-word overread of a
// re-aligned load past the slab's last byte
static_assert(32 * 34 + 15 + 4 <= 3 * 32 * 16, "Q8_0 slab");
static_assert(8 * 210 + 15 + 4 <= 4 * 32 * 16, "Q6_K slab");

// the 32-bit word at a 2-byte-aligned shared-memory offset
__device__ __forceinline__ uint32_t lds_u32_at(const uint8_t* buf, int o) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(buf + (o & ~3));
    return __funnelshift_r(w[0], w[1], (o & 3) * 8);
}

// byte k of v as the float 2^23 + byte, minus `off`
template <int k>
__device__ __forceinline__ float code_f(uint32_t v, float off) {
    return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7650 | k)) - off;
}

// bytes [g, g + 16) of the buffer, those at or past `total` read as zero
__device__ __noinline__ uint4 tail_chunk(const uint8_t* p, int64_t g, int64_t total) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int b = 0; b < 16; ++b)
        if (g + b < total) w[b >> 2] |= (uint32_t)p[g + b] << (8 * (b & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// sum over slab `slab` of one Q8_0 row: 8 lanes per block (4 codes each), 4
// blocks per pass
__device__ __forceinline__ float decode_q8_0_34(const uint8_t* buf, int m, const float* __restrict__ x,
                                                int64_t slab, int64_t nb, int lane) {
    const int64_t b0 = slab * GgufFmt<0>::kSB;
    const int nbs = (int)min((int64_t)GgufFmt<0>::kSB, nb - b0);
    const int e4 = (lane & 7) * 4;
    const float off = 8388736.0f;   // 2^23 + 128
    float acc = 0.f;
#pragma unroll 2
    for (int jb = lane >> 3; jb < nbs; jb += 4) {
        const int o = m + 34 * jb;
        const float d = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(buf + o));
        const uint32_t w = lds_u32_at(buf, o + 2 + e4) ^ 0x80808080u;
        const float4 xv = __ldg(reinterpret_cast<const float4*>(x + (b0 + jb) * 32 + e4));
        float s = code_f<0>(w, off) * xv.x;
        s = fmaf(code_f<1>(w, off), xv.y, s);
        s = fmaf(code_f<2>(w, off), xv.z, s);
        s = fmaf(code_f<3>(w, off), xv.w, s);
        acc = fmaf(d, s, acc);
    }
    return acc;
}

// sum over slab `slab` of one Q6_K row. Lane l takes ql bytes 4l..4l+3 of
// each super-block: with h = l / 16 and r = 4 (l % 16), their low nibbles are
// elements 128h + r + k and their high nibbles elements 128h + 64 + r + k
// (k < 4); the high bit pairs of both sit in qh bytes 32h + r % 32 + k, at
// bits 2c and 2c + 4 (c = r / 32); the scales are sc[8h + r/16] and
// sc[8h + 4 + r/16].
__device__ __forceinline__ float decode_q6_k(const uint8_t* buf, int m, const float* __restrict__ x,
                                             int64_t slab, int64_t nb, int lane) {
    const int64_t b0 = slab * GgufFmt<1>::kSB;
    const int nbs = (int)min((int64_t)GgufFmt<1>::kSB, nb - b0);
    const int h = lane >> 4, r = (lane & 15) * 4;
    const int csh = (r >> 5) * 2;
    const float off = 8388640.0f;   // 2^23 + 32
    float acc = 0.f;
#pragma unroll 2
    for (int jb = 0; jb < nbs; ++jb) {
        const int o = m + 210 * jb;
        const uint32_t qlw = lds_u32_at(buf, o + 4 * lane);
        const uint32_t q2 = lds_u32_at(buf, o + 128 + 32 * h + (r & 31)) >> csh;
        const float sl = (float)(int8_t)buf[o + 192 + 8 * h + (r >> 4)];
        const float sh = (float)(int8_t)buf[o + 196 + 8 * h + (r >> 4)];
        const float d = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(buf + o + 208));
        const float* xb = x + (b0 + jb) * 256 + 128 * h + r;
        const float4 xl = __ldg(reinterpret_cast<const float4*>(xb));
        const float4 xh = __ldg(reinterpret_cast<const float4*>(xb + 64));
        const uint32_t lo = (qlw & 0x0F0F0F0Fu) | ((q2 << 4) & 0x30303030u);
        const uint32_t hi = ((qlw >> 4) & 0x0F0F0F0Fu) | (q2 & 0x30303030u);
        float a = code_f<0>(lo, off) * xl.x;
        a = fmaf(code_f<1>(lo, off), xl.y, a);
        a = fmaf(code_f<2>(lo, off), xl.z, a);
        a = fmaf(code_f<3>(lo, off), xl.w, a);
        float b = code_f<0>(hi, off) * xh.x;
        b = fmaf(code_f<1>(hi, off), xh.y, b);
        b = fmaf(code_f<2>(hi, off), xh.z, b);
        b = fmaf(code_f<3>(hi, off), xh.w, b);
        acc = fmaf(d, fmaf(sl, a, sh * b), acc);
    }
    return acc;
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32) gguf_gemv_kernel(const uint8_t* __restrict__ blocks,
                                                                const float* __restrict__ x, float* __restrict__ out,
                                                                int64_t N, int64_t nb, int64_t total) {
    using F = GgufFmt<FMT>;
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    __shared__ __align__(16) uint8_t sbuf[kWarps][F::kCPL * 512];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* buf = sbuf[warp];
    const int64_t nslab = (nb + F::kSB - 1) / F::kSB;
    const int64_t wstride = (int64_t)gridDim.x * kWarps;
    const int64_t RB = nb * F::kBB;

    uint4 reg[F::kCPL];
    int mis = 0;
    // 16-byte chunks of item (r, s) -- slab s of row r -- into reg; mis = the
    // slab's offset from the 16-byte boundary below it
    auto fetch = [&](int64_t r, int64_t s) {
        const int64_t b0 = s * F::kSB;
        const int64_t nbs = min((int64_t)F::kSB, nb - b0);
        const int64_t start = r * RB + b0 * F::kBB;
        const int64_t a0 = start & ~(int64_t)15;
        mis = (int)(start - a0);
        const int nch = (int)((mis + nbs * F::kBB + 15) >> 4);
#pragma unroll
        for (int i = 0; i < F::kCPL; ++i) {
            const int c = i * 32 + lane;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (c < nch) {
                const int64_t g = a0 + 16 * (int64_t)c;
                v = g + 16 <= total ? ld_stream_v4(blocks + g) : tail_chunk(blocks, g, total);
            }
            reg[i] = v;
        }
    };

    int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    int64_t slab = 0;
    if (row < N) fetch(row, 0);
    float acc = 0.f;
    while (row < N) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < F::kCPL; ++i) reinterpret_cast<uint4*>(buf)[i * 32 + lane] = reg[i];
        __syncwarp();
        const int m = mis;
        const int64_t cur_row = row, cur_slab = slab;
        if (++slab == nslab) {
            slab = 0;
            row += wstride;
        }
        if (row < N) fetch(row, slab);   // in flight during the decode below
        if constexpr (FMT == 0)
            acc += decode_q8_0_34(buf, m, x, cur_slab, nb, lane);
        else
            acc += decode_q6_k(buf, m, x, cur_slab, nb, lane);
        if (cur_slab == nslab - 1) {
            const float v = warp_sum(acc);
            if (lane == 0) out[cur_row] = v;
            acc = 0.f;
        }
    }
}

template <int FMT>
cudaError_t launch_gguf_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                             cudaStream_t s) {
    using F = GgufFmt<FMT>;
    const int64_t nb = K / F::kBK;
    const int64_t total = N * nb * F::kBB;
    const int64_t want = (N + kWarps - 1) / kWarps;
    const int64_t cap = 4LL * num_sms();   // 4 CTAs of 8 warps per SM
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    return launch_pdl(gguf_gemv_kernel<FMT>, dim3(grid), dim3(kWarps * 32), 0, s, blocks, x, out, N, nb, total);
}

}  // namespace
}  // namespace gai4

extern "C" {

gai4_status gai4_q8_0_34b_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                               void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 32 != 0) return GAI4_ERR_INVALID_ARG;
    if (((uintptr_t)blocks & 15u) != 0 || ((uintptr_t)x & 15u) != 0) return GAI4_ERR_MISALIGNED;
    return gai4::launch_gguf_gemv<0>(blocks, x, out, N, K, (cudaStream_t)stream) == cudaSuccess ? GAI4_OK
                                                                                                : GAI4_ERR_CUDA;
}

gai4_status gai4_q6_k_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K, void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 256 != 0) return GAI4_ERR_INVALID_ARG;
    if (((uintptr_t)blocks & 15u) != 0 || ((uintptr_t)x & 15u) != 0) return GAI4_ERR_MISALIGNED;
    return gai4::launch_gguf_gemv<1>(blocks, x, out, N, K, (cudaStream_t)stream) == cudaSuccess ? GAI4_OK
                                                                                                : GAI4_ERR_CUDA;
}

}  // extern "C"
