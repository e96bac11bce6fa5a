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
// x is staged once per CTA in shared memory when it fits (K up to 24576),
// otherwise read through the read-only cache; the first slabs of the blocks
// are requested before the kernels this one overlaps complete (they never
// write blocks), x only after.
// A slab is copied by 16-byte asynchronous copies (cp.async, L2-only), starting
// at the 16-byte boundary at or below it, into a warp-private ring of
// shared-memory stages kStages - 1 slabs ahead of the decode (the copy that
// reaches past the end of the weights reads only the bytes before it and
// zero-fills the rest); words at 2-byte-aligned offsets are then read from the
// stage as two aligned words and a funnel shift.
// A code c becomes a float through the mantissa of 2^23: a byte permute puts
// c under the exponent byte 0x4B, and one packed subtraction per pair of codes
// (add.rn.f32x2) removes 2^23 and the codes' offset (128 for Q8_0 bytes with
// the sign bit flipped, 32 for Q6_K) exactly; one fma.rn.f32x2 adds both
// products. Products and sums are binary32; the block scale is applied once
// per block (Q8_0) or once per 4-weight run of one 16-weight scale group
// (Q6_K), and a warp-shuffle sum finishes each row.
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace gai4 {
namespace {

constexpr int kWarps = 8;   // warps per CTA

template <int FMT>
struct GgufFmt;
// kBB bytes per block of kBK weights, kSB blocks per slab, stages of
// kCPL x 32 16-byte chunks, kStages stages per warp (8 warps x kStages stages
// fit the 48 KB of static shared memory)
template <>
struct GgufFmt<0> {   // Q8_0, 34-byte blocks
    static constexpr int kBB = 34, kBK = 32, kSB = 32, kCPL = 3, kStages = 4;
};
template <>
struct GgufFmt<1> {   // Q6_K, 210-byte super-blocks
    static constexpr int kBB = 210, kBK = 256, kSB = 8, kCPL = 4, kStages = 3;
};
// a slab of kSB blocks plus up to 15 leading bytes fits a stage, which leaves
// room for the one-word overread of a re-aligned load past the slab's last byte
static_assert(32 * 34 + 15 + 4 <= 3 * 32 * 16, "Q8_0 slab");
static_assert(8 * 210 + 15 + 4 <= 4 * 32 * 16, "Q6_K slab");
static_assert(kWarps * 4 * 3 * 512 <= 48 * 1024 && kWarps * 3 * 4 * 512 <= 48 * 1024, "ring of stages");
constexpr int64_t kMaxSmemX = 24576;   // largest K whose binary32 x is staged in shared memory

// 16 bytes of x: from shared memory (staged) or through the read-only cache
template <bool XSM>
__device__ __forceinline__ float4 ld_x4(const float* p) {
    if constexpr (XSM)
        return *reinterpret_cast<const float4*>(p);
    else
        return __ldg(reinterpret_cast<const float4*>(p));
}

// the 32-bit word at a 2-byte-aligned shared-memory offset
__device__ __forceinline__ uint32_t lds_u32_at(const uint8_t* buf, int o) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(buf + (o & ~3));
    return __funnelshift_r(w[0], w[1], (o & 3) * 8);
}

// byte k of v under the exponent of 2^23: the float 2^23 + byte (bits)
template <int k>
__device__ __forceinline__ uint32_t code_bits(uint32_t v) {
    return __byte_perm(v, 0x4B000000u, 0x7650 | k);
}
// bytes k, k + 1 of v as the exact pair (byte - off'): one packed subtract of
// (2^23 + off') from (2^23 + byte_k, 2^23 + byte_{k+1}); noff = -(2^23 + off')
template <int k>
__device__ __forceinline__ float2 code_pair(uint32_t v, float noff) {
    float2 d;
    asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n add.rn.f32x2 d, a, b;\n"
        " mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(code_bits<k>(v)), "r"(code_bits<k + 1>(v)), "f"(noff));
    return d;
}
// (c.x + a.x b.x, c.y + a.y b.y) in one instruction (fma.rn.f32x2)
__device__ __forceinline__ float2 ffma2(float2 a, float bx, float by, float2 c) {
    float2 d;
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
        " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(bx), "f"(by), "f"(c.x), "f"(c.y));
    return d;
}

// 16-byte asynchronous copy global -> shared that reads `src_bytes` (1..16)
// bytes and zero-fills the rest of the 16
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// sum over slab `slab` of one Q8_0 row: 8 lanes per block (4 codes each), 4
// blocks per pass
template <bool XSM>
__device__ __forceinline__ float decode_q8_0_34(const uint8_t* buf, int m, const float* __restrict__ x, int slab,
                                                int nb, int lane) {
    const int b0 = slab * GgufFmt<0>::kSB;
    const int nbs = min(GgufFmt<0>::kSB, nb - b0);
    const int e4 = (lane & 7) * 4;
    const float noff = -8388736.0f;   // -(2^23 + 128)
    float acc = 0.f;
#pragma unroll 2
    for (int jb = lane >> 3; jb < nbs; jb += 4) {
        const int o = m + 34 * jb;
        const float d = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(buf + o));
        const uint32_t w = lds_u32_at(buf, o + 2 + e4) ^ 0x80808080u;   // codes + 128, as bytes
        const float4 xv = ld_x4<XSM>(x + (b0 + jb) * 32 + e4);
        float2 s2 = ffma2(code_pair<0>(w, noff), xv.x, xv.y, make_float2(0.f, 0.f));
        s2 = ffma2(code_pair<2>(w, noff), xv.z, xv.w, s2);
        acc = fmaf(d, s2.x + s2.y, acc);
    }
    return acc;
}

// sum over slab `slab` of one Q6_K row. Lane l takes ql bytes 4l..4l+3 of
// each super-block: with h = l / 16 and r = 4 (l % 16), their low nibbles are
// elements 128h + r + k and their high nibbles elements 128h + 64 + r + k
// (k < 4); the high bit pairs of both sit in qh bytes 32h + r % 32 + k, at
// bits 2c and 2c + 4 (c = r / 32); the scales are sc[8h + r/16] and
// sc[8h + 4 + r/16].
template <bool XSM>
__device__ __forceinline__ float decode_q6_k(const uint8_t* buf, int m, const float* __restrict__ x, int slab,
                                             int nb, int lane) {
    const int b0 = slab * GgufFmt<1>::kSB;
    const int nbs = min(GgufFmt<1>::kSB, nb - b0);
    const int h = lane >> 4, r = (lane & 15) * 4;
    const int csh = (r >> 5) * 2;
    const float noff = -8388640.0f;   // -(2^23 + 32)
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
        const float4 xl = ld_x4<XSM>(xb);
        const float4 xh = ld_x4<XSM>(xb + 64);
        const uint32_t lo = (qlw & 0x0F0F0F0Fu) | ((q2 << 4) & 0x30303030u);
        const uint32_t hi = ((qlw >> 4) & 0x0F0F0F0Fu) | (q2 & 0x30303030u);
        float2 a2 = ffma2(code_pair<0>(lo, noff), xl.x, xl.y, make_float2(0.f, 0.f));
        a2 = ffma2(code_pair<2>(lo, noff), xl.z, xl.w, a2);
        float2 b2 = ffma2(code_pair<0>(hi, noff), xh.x, xh.y, make_float2(0.f, 0.f));
        b2 = ffma2(code_pair<2>(hi, noff), xh.z, xh.w, b2);
        acc = fmaf(d, fmaf(sl, a2.x + a2.y, sh * (b2.x + b2.y)), acc);
    }
    return acc;
}

template <int FMT, bool XSM>
__global__ void __launch_bounds__(kWarps * 32) gguf_gemv_kernel(const uint8_t* __restrict__ blocks,
                                                                const float* __restrict__ x, float* __restrict__ out,
                                                                int64_t N, int64_t nb, int64_t total) {
    using F = GgufFmt<FMT>;
    constexpr int kStageBytes = F::kCPL * 512;
    extern __shared__ __align__(16) uint8_t gg_smem[];
    pdl_launch_dependents();
    // [kWarps][kStages][kStageBytes] ring, then (XSM) x [K] binary32
    uint8_t (*sbuf)[F::kStages][kStageBytes] = reinterpret_cast<uint8_t (*)[F::kStages][kStageBytes]>(gg_smem);
    float* xs = reinterpret_cast<float*>(gg_smem + (size_t)kWarps * F::kStages * kStageBytes);
    const int64_t K = nb * F::kBK;
    if (XSM && threadIdx.x == 0) pipe::bulk_prefetch_l2(x, (uint32_t)(K * 4));   // x to the head of the DRAM queue
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nslab = (int)((nb + F::kSB - 1) / F::kSB);
    const int64_t wstride = (int64_t)gridDim.x * kWarps;
    const int64_t RB = nb * F::kBB;
    const int64_t row0 = (int64_t)blockIdx.x * kWarps + warp;
    // this warp's items: slabs 0 .. nslab - 1 of rows row0, row0 + wstride, ...
    // walked by two cursors (row, slab): the next item to copy, the next to decode

    int64_t ir = row0;   // copy cursor
    int is = 0, islot = 0;
    auto issue = [&]() {
        if (ir < N) {
            const int nbs = (int)min((int64_t)F::kSB, nb - (int64_t)is * F::kSB);
            const int64_t start = ir * RB + (int64_t)is * (F::kSB * F::kBB);
            const int64_t a0 = start & ~(int64_t)15;
            const int nch = ((int)(start - a0) + nbs * F::kBB + 15) >> 4;
            uint8_t* st = sbuf[warp][islot];
#pragma unroll
            for (int i = 0; i < F::kCPL; ++i) {
                const int c = i * 32 + lane;
                if (c < nch) {
                    const int64_t g = a0 + 16 * (int64_t)c;   // g < total: the chunk starts inside the slab
                    cp_async16(st + 16 * c, blocks + g, (int)min((int64_t)16, total - g));
                }
            }
            if (++is == nslab) {
                is = 0;
                ir += wstride;
            }
        }
        cp_async_commit();   // one group per item (empty past the end) keeps the counting uniform
        if (++islot == F::kStages) islot = 0;
    };

#pragma unroll
    for (int t = 0; t < F::kStages - 1; ++t) issue();   // blocks: before the wait
    pdl_wait();   // the kernels before this one are complete: x may be read, out written
    const float* xr = x;
    if constexpr (XSM) {
        const float4* xg4 = reinterpret_cast<const float4*>(x);
        float4* xs4 = reinterpret_cast<float4*>(xs);
        for (int64_t i = threadIdx.x; i < K / 4; i += kWarps * 32) xs4[i] = __ldg(xg4 + i);
        __syncthreads();
        xr = xs;
    }
    float acc = 0.f;
    int cslot = 0;
    for (int64_t cr = row0, cs = 0; cr < N;) {   // decode cursor
        __syncwarp();                  // every lane is done with the stage the previous item used
        issue();                       // ... which the item kStages - 1 ahead now refills
        cp_async_wait<F::kStages - 1>();
        __syncwarp();                  // this item's chunks from every lane have landed
        const uint8_t* buf = sbuf[warp][cslot];
        const int m = (int)((cr * RB + cs * (F::kSB * F::kBB)) & 15);
        if constexpr (FMT == 0)
            acc += decode_q8_0_34<XSM>(buf, m, xr, (int)cs, (int)nb, lane);
        else
            acc += decode_q6_k<XSM>(buf, m, xr, (int)cs, (int)nb, lane);
        if (++cslot == F::kStages) cslot = 0;
        if (++cs == nslab) {
            const float v = warp_sum(acc);
            if (lane == 0) out[cr] = v;
            acc = 0.f;
            cs = 0;
            cr += wstride;
        }
    }
    cp_async_wait<0>();   // no copy outlives the warp (the trailing groups are empty)
}

template <int FMT>
cudaError_t launch_gguf_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                             cudaStream_t s) {
    using F = GgufFmt<FMT>;
    const int64_t nb = K / F::kBK;
    const int64_t total = N * nb * F::kBB;
    const int64_t want = (N + kWarps - 1) / kWarps;
    const size_t ring = (size_t)kWarps * F::kStages * F::kCPL * 512;
    const bool xsm = K <= kMaxSmemX;
    const size_t smem = ring + (xsm ? (size_t)K * 4 : 0);
    // CTAs of 8 warps per SM: up to 4, as many as the shared memory holds
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(4, (int64_t)(227 * 1024) / (int64_t)(smem + 1024)));
    const int64_t cap = per_sm * num_sms();
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (!xsm) return launch_pdl(gguf_gemv_kernel<FMT, false>, dim3(grid), dim3(kWarps * 32), smem, s, blocks, x, out, N, nb, total);
    static unsigned long long configured = 0ull;   // bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(configured & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(gguf_gemv_kernel<FMT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(ring + kMaxSmemX * 4));
        if (e != cudaSuccess) return e;
        if (dev < 64) configured |= 1ull << dev;
    }
    return launch_pdl(gguf_gemv_kernel<FMT, true>, dim3(grid), dim3(kWarps * 32), smem, s, blocks, x, out, N, nb, total);
}

}  // namespace
}  // namespace gai4

extern "C" {

gai4_status gai4_q8_0_34b_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                               void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 32 != 0 || K >= (1LL << 31)) return GAI4_ERR_INVALID_ARG;
    if (((uintptr_t)blocks & 15u) != 0 || ((uintptr_t)x & 15u) != 0) return GAI4_ERR_MISALIGNED;
    return gai4::launch_gguf_gemv<0>(blocks, x, out, N, K, (cudaStream_t)stream) == cudaSuccess ? GAI4_OK
                                                                                                : GAI4_ERR_CUDA;
}

gai4_status gai4_q6_k_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K, void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 256 != 0 || K >= (1LL << 31)) return GAI4_ERR_INVALID_ARG;
    if (((uintptr_t)blocks & 15u) != 0 || ((uintptr_t)x & 15u) != 0) return GAI4_ERR_MISALIGNED;
    return gai4::launch_gguf_gemv<1>(blocks, x, out, N, K, (cudaStream_t)stream) == cudaSuccess ? GAI4_OK
                                                                                                : GAI4_ERR_CUDA;
}

}  // extern "C"
