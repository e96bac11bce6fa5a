// blockq_tma.cu -- Q8_0 and Q4_K matrix-vector products with TMA-staged
// weight rows (sm_103a, CUDA cores; the work is HBM-bound).
//
// Formats (hanzo-kernel quant.rs, "Q8_0 PACKED matvec" and the Q4_K section):
//  * Q8_0: a 36-byte block per 32 weights -- f16 scale d in the low half of
//    word 0, then 32 signed int8 codes, four per word, byte 0 first;
//    out[n] = sum_b d_b * sum_j q_j x_{32b+j}.
//  * Q4_K: a 144-byte super-block per 256 weights -- d, dmin (f16), 12 bytes of
//    eight 6-bit (sc, m) pairs (get_scale_min_k4), 128 bytes of codes; byte
//    32g + i holds weight 64g + i (low nibble, sub-block 2g) and weight
//    64g + 32 + i (high nibble, sub-block 2g + 1); a weight is d*sc*q - dmin*m.
//
// Design (one CTA per SM, persistent over row groups):
//  * A row is cut into 1152-byte chunks: 32 Q8_0 blocks (1024 weights) or 8
//    Q4_K super-blocks (2048 weights). A producer warp brings stages of
//    rows x C chunks into a ring in shared memory with 2-D TMA boxes of
//    rows x 1152 bytes (rows past N and bytes past the row end are filled
//    with zeros, which decode to zero weights).
//  * 16 consumer warps share every stage of 32 rows x 1 chunk (a warp two rows,
//    a lane one item of the chunk: a Q8_0 block, or one 64-weight group g of a
//    Q4_K super-block with its 16-byte header and 32 code bytes); a lane's
//    activations are loaded once per chunk and serve both rows. (The code
//    keeps the general form of S sets of G warps splitting K; the plan uses
//    S = 1: a K split leaves sets idle when a row is a few chunks long.)
//  * The activations are staged once per CTA in shared memory in an order in
//    which the 32 lanes of a warp read consecutive 16-byte pieces, with the
//    sum of every 32-element run.
//  * Every product q x is exact before it is summed: a block of zero codes
//    adds exactly 0. Q8_0: one shift and one three-input logic op place byte
//    b of a word in the mantissa of 256 as 384 + q (mantissa bits 15..22 =
//    q + 128 = byte ^ 0x80), one packed fp32 fma gives q = f - 384, another
//    adds q x. Q4_K: a nibble masked in place in a code word is a binary32
//    subnormal, q * 2^(its bit position) * 2^-149 (bit 23, the exponent's
//    lowest, continues the mantissa seamlessly); byte 3 is shifted down
//    first. The staged activations carry the inverse power of two of their
//    nibble's position and a per-item power of two that keeps the products
//    binary32 normals (down to 2^-103 of the item's largest magnitude), so
//    one packed fma per byte adds (q_lo x_i, q_hi x_{i+32}): 1 shift, 8 ANDs
//    and 4 packed fmas per 8 codes; the item's sums are scaled back once.
//  * Per-row results of a set are held in a small shared buffer and combined
//    over the sets in a fixed order every F row groups (one consumer barrier
//    per flush, double-buffered): the result does not depend on timing.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace gai4 {

namespace {

using namespace pipe;

constexpr int kCW = 16;                        // consumer warps
constexpr int kThreads = 32 * (kCW + 1);       // + one producer warp
constexpr uint32_t kChunkBytes = 1152;         // one row chunk
constexpr int kChunkU64 = kChunkBytes / 8;     // TMA box width in 8-byte elements
constexpr int kMaxDepth = 16;
constexpr int kFlush = 8;                      // row groups per flush
constexpr int kR = 2;                          // rows per consumer warp

struct BqArgs {
    int N;
    int chunks;            // chunks per row (the last one may be partial)
    int G, S, C;           // warps per set (kR rows each), consumer sets, chunks per stage
    int cps, kss;          // chunks per set, stages per set and row group
    int depth;
    int n_groups;          // row groups = ceil(N / (kR G))
    uint32_t stage_bytes;  // C * kR * G * 1152
    uint32_t x_off, sum_off, pend_off, bar_off;   // shared-memory layout
    const float* x;        // binary32 activations (Q8_0, Q4_K)
    const int8_t* xq;      // int8 activations and their per-block scales (Q8_0 with integer activations)
    const float* xd;
    float* out;
    int K;
    int last_half;         // Q4_K: the last chunk holds at most 4 super-blocks
    int* status;
    long long spin_limit;
};

// (a & b) ^ c as one three-input logic instruction
__device__ __forceinline__ uint32_t lop3_andxor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// (acc.x + a_lo * b_lo, acc.y + a_hi * b_hi): two binary32 fmas in one instruction
__device__ __forceinline__ float2 ffma2(uint32_t a_lo, uint32_t a_hi, float b_lo, float b_hi, float2 c) {
    float2 d;
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
        " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(a_lo), "r"(a_hi), "f"(b_lo), "f"(b_hi), "f"(c.x), "f"(c.y));
    return d;
}
// (m_lo * f_lo + c_lo, m_hi * f_hi + c_hi) with every operand a register: the
// exact codes of a decoded pair
__device__ __forceinline__ float2 codes2(uint32_t f_lo, uint32_t f_hi, uint32_t m_lo, uint32_t m_hi, uint32_t c_lo,
                                         uint32_t c_hi) {
    float2 d;
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
        " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(f_lo), "r"(f_hi), "r"(m_lo), "r"(m_hi), "r"(c_lo), "r"(c_hi));
    return d;
}
__device__ __forceinline__ float2 fma2q(float2 q, float b_lo, float b_hi, float2 c) {
    return ffma2(__float_as_uint(q.x), __float_as_uint(q.y), b_lo, b_hi, c);
}

// Q4_K: one code word (bytes k = 0..3: low nibble = element 4t + k of the
// low sub-block, high nibble = of the high one) against its staged,
// position-scaled activations. A code masked in place is a binary32
// subnormal (exponent field 0, or 1 for the nibble holding bit 23), i.e.
// exactly q * 2^(bit position) * 2^-149; byte 3 is moved down first. Each
// packed fma adds (q_lo x'_lo, q_hi x'_hi) with exact products.
__device__ __forceinline__ float2 q4k_word(uint32_t w, float4 p0, float4 p1, float2 acc) {
    const uint32_t h3 = w >> 24;
    acc = ffma2(w & 0xFu, w & 0xF0u, p0.x, p0.y, acc);
    acc = ffma2(w & 0xF00u, w & 0xF000u, p0.z, p0.w, acc);
    acc = ffma2(w & 0xF0000u, w & 0xF00000u, p1.x, p1.y, acc);
    return ffma2(h3 & 0xFu, h3 & 0xF0u, p1.z, p1.w, acc);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    const uint4 v = lds128(a);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory"); }

// (sc, m) of sub-blocks j = 2g and 2g + 1 (get_scale_min_k4) from the 12
// scale bytes held in three words b0 (bytes 0..3), b1 (4..7), b2 (8..11).
// With t_i = b_i >> (8 (j & 3)), byte 0 of t_i belongs to sub-block 2g and
// byte 1 to 2g + 1. For j < 4: sc = byte(b0) & 63, m = byte(b1) & 63; for
// j >= 4: sc = (byte(b2) & 15) | (byte(b0) >> 6) << 4, m = (byte(b2) >> 4) |
// (byte(b1) >> 6) << 4. Both forms are computed and one is selected (g is
// fixed per lane, so there is no divergent branch).
__device__ __forceinline__ void scale_min_pair(uint32_t b0, uint32_t b1, uint32_t b2, int g, float& sc0, float& m0,
                                               float& sc1, float& m1) {
    const int sh = 16 * (g & 1);
    const uint32_t t0 = b0 >> sh, t1 = b1 >> sh, t2 = b2 >> sh;
    const bool hi = g >= 2;
    const uint32_t s0 = hi ? (t2 & 15u) | ((t0 >> 2) & 0x30u) : t0 & 63u;
    const uint32_t s1 = hi ? ((t2 >> 8) & 15u) | ((t0 >> 10) & 0x30u) : (t0 >> 8) & 63u;
    const uint32_t n0 = hi ? ((t2 >> 4) & 15u) | ((t1 >> 2) & 0x30u) : t1 & 63u;
    const uint32_t n1 = hi ? ((t2 >> 12) & 15u) | ((t1 >> 10) & 0x30u) : (t1 >> 8) & 63u;
    sc0 = (float)s0;
    sc1 = (float)s1;
    m0 = (float)n0;
    m1 = (float)n1;
}

// ---------------------------------------------------------------------------
// activation staging: x (f32, K) -> shared memory in lane order, zero past K
// ---------------------------------------------------------------------------
// Q8_0: chunk ch, block b (lane), piece j (4 elements): float4 index
// (ch * 8 + j) * 32 + b; sums[32 ch + b] = sum of the block's 32 elements.
// Q4_K: chunk ch, item u = 4 sb + g (lane), pair quad q (elements i = 2q,
// 2q + 1 of both runs): float4 index (ch * 16 + q) * 32 + u holding
// (x_lo[2q], x_hi[2q], x_lo[2q+1], x_hi[2q+1]); sums[8 (8 ch + sb) + j] = sum
// of sub-block j (= sums[2 (32 ch + u)] and sums[2 (32 ch + u) + 1]).
// One pass by the consumer threads: a thread takes 8 consecutive elements
// of a 32-element run (Q8_0) or of both runs of a Q4_K item; the 4 threads of
// a run sit in adjacent lanes and add their partial sums with shuffles.
template <int FMT>
__device__ void stage_x(const BqArgs& a, uint8_t* smem) {
    float4* xs = reinterpret_cast<float4*>(smem + a.x_off);
    float* sums = reinterpret_cast<float*>(smem + a.sum_off);
    if constexpr (FMT == BQ_Q8_0_I8) {
        // chunk ch, block b (lane), half j: 16 code bytes at uint4 index
        // (ch * 2 + j) * 32 + b; sums[32 ch + b] = the block's activation scale
        uint4* xs4 = reinterpret_cast<uint4*>(smem + a.x_off);
        const int nblk = a.K / 32;
        for (int p = threadIdx.x; p < a.chunks * 64; p += kCW * 32) {
            const int ch = p >> 6, j = (p >> 5) & 1, b = p & 31, g = ch * 32 + b;
            xs4[(ch * 2 + j) * 32 + b] =
                g < nblk ? *reinterpret_cast<const uint4*>(a.xq + 32 * (int64_t)g + 16 * j) : make_uint4(0, 0, 0, 0);
        }
        for (int r = threadIdx.x; r < a.chunks * 32; r += kCW * 32) sums[r] = r < nblk ? a.xd[r] : 0.f;
        return;
    }
    const int total = a.chunks * 128;   // a multiple of 32: whole warps in the shuffles
    for (int v = threadIdx.x; v < total; v += kCW * 32) {
        const int c = v >> 2, qq = v & 3;   // run (Q8_0 block) or item (Q4_K), quarter
        const int ch = c >> 5, ln = c & 31;
        if constexpr (FMT == BQ_Q8_0) {
            const int k0 = 32 * c + 8 * qq;
            float4 f0 = make_float4(0.f, 0.f, 0.f, 0.f), f1 = f0;
            if (k0 < a.K) {   // K is a multiple of 32: a run is all in or all out
                f0 = *reinterpret_cast<const float4*>(a.x + k0);
                f1 = *reinterpret_cast<const float4*>(a.x + k0 + 4);
            }
            xs[(ch * 8 + 2 * qq) * 32 + ln] = f0;
            xs[(ch * 8 + 2 * qq + 1) * 32 + ln] = f1;
            float t = ((f0.x + f0.y) + (f0.z + f0.w)) + ((f1.x + f1.y) + (f1.z + f1.w));
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            if (qq == 0) sums[c] = t;
        } else {
            // item ln = 4 sb + g of chunk ch: runs at base (low) and base + 32 (high)
            const int base = ch * 2048 + 64 * ln, i0 = 8 * qq;
            float lo[8], hi[8];
            if (base < a.K) {   // K is a multiple of 256: an item is all in or all out
                const float4 l0 = *reinterpret_cast<const float4*>(a.x + base + i0);
                const float4 l1 = *reinterpret_cast<const float4*>(a.x + base + i0 + 4);
                const float4 h0 = *reinterpret_cast<const float4*>(a.x + base + 32 + i0);
                const float4 h1 = *reinterpret_cast<const float4*>(a.x + base + 32 + i0 + 4);
                lo[0] = l0.x; lo[1] = l0.y; lo[2] = l0.z; lo[3] = l0.w;
                lo[4] = l1.x; lo[5] = l1.y; lo[6] = l1.z; lo[7] = l1.w;
                hi[0] = h0.x; hi[1] = h0.y; hi[2] = h0.z; hi[3] = h0.w;
                hi[4] = h1.x; hi[5] = h1.y; hi[6] = h1.z; hi[7] = h1.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) lo[j] = hi[j] = 0.f;
            }
            // the item's scale 2^kc: its largest magnitude's exponent field E -> kc = 253 - E
            uint32_t eb = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                eb = max(eb, max(__float_as_uint(lo[j]) & 0x7F800000u, __float_as_uint(hi[j]) & 0x7F800000u));
            eb = max(eb, __shfl_xor_sync(0xffffffffu, eb, 1));
            eb = max(eb, __shfl_xor_sync(0xffffffffu, eb, 2));
            const int E = max((int)(eb >> 23), 1);
            const int kc = max(253 - E, -2);
            // element i (byte i % 4 of its code word): low nibble at bit 8 (i % 4)
            // (bit 0 for byte 3, after the shift by 24), high nibble 4 bits above;
            // x staged times 2^(kc - that bit), in two exact power-of-two steps
            auto scaled = [&](float v, int sh) {
                const int e = kc - sh;
                const int ea = e / 2, eb2 = e - e / 2;
                return (v * __uint_as_float((uint32_t)(127 + ea) << 23)) * __uint_as_float((uint32_t)(127 + eb2) << 23);
            };
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // pair quad 4 qq + q: elements i0 + 2q, i0 + 2q + 1
                const int k0 = (i0 + 2 * q) & 3, k1 = (i0 + 2 * q + 1) & 3;
                const int s0 = k0 == 3 ? 0 : 8 * k0, s1 = k1 == 3 ? 0 : 8 * k1;
                xs[(ch * 16 + 4 * qq + q) * 32 + ln] =
                    make_float4(scaled(lo[2 * q], s0), scaled(hi[2 * q], s0 + 4), scaled(lo[2 * q + 1], s1),
                                scaled(hi[2 * q + 1], s1 + 4));
            }
            float sl = ((lo[0] + lo[1]) + (lo[2] + lo[3])) + ((lo[4] + lo[5]) + (lo[6] + lo[7]));
            float sh = ((hi[0] + hi[1]) + (hi[2] + hi[3])) + ((hi[4] + hi[5]) + (hi[6] + hi[7]));
            sl += __shfl_xor_sync(0xffffffffu, sl, 1);
            sh += __shfl_xor_sync(0xffffffffu, sh, 1);
            sl += __shfl_xor_sync(0xffffffffu, sl, 2);
            sh += __shfl_xor_sync(0xffffffffu, sh, 2);
            if (qq == 0) {
                sums[2 * c] = sl;       // sub-block 2g of super-block 8 ch + sb
                sums[2 * c + 1] = sh;   // sub-block 2g + 1
                // the item's code sums come out times 2^(kc - 149): back by 2^p, p = 149 - kc
                const int pp = 149 - kc;
                sums[2 * a.chunks * 32 + 2 * c] = __uint_as_float((uint32_t)(127 + pp / 2) << 23);
                sums[2 * a.chunks * 32 + 2 * c + 1] = __uint_as_float((uint32_t)(127 + pp - pp / 2) << 23);
            }
        }
    }
}

template <int FMT>
__device__ __forceinline__ void bq_tma_body(const CUtensorMap& wmap, const BqArgs& a) {
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* empty = full + kMaxDepth;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxDepth);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.depth, S = a.S, G = a.G, C = a.C;

    if (threadIdx.x == 0) {
        for (int i = 0; i < D; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], G);   // the G warps of the set that owns the slot
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // valid chunks of stage (set s, stage ks of the set): [c0, c0 + n)
    auto stage_chunks = [&](int s, int ks, int& c0) {
        c0 = s * a.cps + ks * C;
        const int lim = min((s + 1) * a.cps, a.chunks);
        return max(0, min(C, lim - c0));
    };
    // Warm L2 with x first (at the head of the DRAM queue) and fetch the
    // tensor map while the barriers are set up
    if (warp == kCW && lane == 0) {
        // K % 32 == 0: whole 16-byte units (int8 codes or binary32 x)
        if constexpr (FMT == BQ_Q8_0_I8)
            bulk_prefetch_l2(a.xq, (uint32_t)a.K);
        else
            bulk_prefetch_l2(a.x, (uint32_t)a.K * 4u);
        asm volatile("prefetch.tensormap [%0];" ::"l"(&wmap) : "memory");
    }
    __syncthreads();   // barriers initialised: the producer starts while the consumers stage x
    Ctl ctl{a.status, a.spin_limit, abort_flag};

    if (warp == kCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            // The blocks are not written by the kernels this one may overlap
            // (programmatic launch): the first ring-full of stages is
            // requested at once, before those kernels complete. Only the
            // activations wait for them.
            int slot = 0, ph = 0, issued = 0;
            bool ok = true;
            for (int rg = blockIdx.x; rg < a.n_groups && ok; rg += gridDim.x) {
                for (int ks = 0; ks < a.kss && ok; ++ks) {
                    for (int s = 0; s < S; ++s) {
                        if (!mbar_wait(&empty[slot], (uint32_t)(ph ^ 1), ctl)) {
                            ok = false;
                            break;
                        }
                        int c0;
                        const int n = stage_chunks(s, ks, c0);
                        mbar_arrive_expect_tx(&full[slot], (uint32_t)n * (uint32_t)(kR * G) * kChunkBytes);
                        uint8_t* dst = smem + (size_t)slot * a.stage_bytes;
                        for (int c = 0; c < n; ++c)
                            tma_load_2d(dst + (size_t)c * (kR * G) * kChunkBytes, &wmap, &full[slot],
                                        (c0 + c) * kChunkU64, rg * (kR * G));
                        ++issued;
                        if (++slot == D) {
                            slot = 0;
                            ph ^= 1;
                        }
                    }
                }
            }
            // every issued copy has landed before the CTA may exit
            for (int i = (issued > D ? issued - D : 0); i < issued; ++i)
                mbar_wait_drain(&full[i % D], (uint32_t)((i / D) & 1), a.spin_limit, a.status);
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    stage_x<FMT>(a, smem);
    consumer_bar();
    // warp wg of set s: rows kR * wg .. kR * wg + kR - 1 of every stage of the
    // set; a lane's activations are loaded once per chunk and serve kR rows
    const int s = warp / G, wg = warp % G;
    const int RS = G * kR;
    const uint32_t xs_base = smem_u32(smem + a.x_off);
    const float* sums = reinterpret_cast<const float*>(smem + a.sum_off);
    float* pend = reinterpret_cast<float*>(smem + a.pend_off);   // [2][kFlush][S][RS]
    const uint32_t ring = smem_u32(smem);
    // loop-invariant logic-op operands, held in registers
    const uint32_t c_mask = pin_reg(FMT == BQ_Q8_0 ? 0x007F8000u : 0x00078000u);
    const uint32_t c_const = pin_reg(FMT == BQ_Q8_0 ? 0x43C00000u : 0x3F800000u);
    // code recovery q = m f + c: Q8_0 (1, 1) f + (-384, -384); Q4_K (256, 16) f + (-256, -16)
    const uint32_t r_m_lo = pin_reg(FMT == BQ_Q8_0 ? 0x3F800000u : 0x43800000u);
    const uint32_t r_m_hi = pin_reg(FMT == BQ_Q8_0 ? 0x3F800000u : 0x41800000u);
    const uint32_t r_c_lo = pin_reg(FMT == BQ_Q8_0 ? 0xC3C00000u : 0xC3800000u);
    const uint32_t r_c_hi = pin_reg(FMT == BQ_Q8_0 ? 0xC3C00000u : 0xC1800000u);
    int slot = s, ph = 0;   // this set's slots: s, s + S, ... (the depth is a multiple of S)
    int buf = 0, fi = 0;
    bool ok = true;
    for (int rg = blockIdx.x; rg < a.n_groups; rg += gridDim.x) {
        float part[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) part[r] = 0.f;
        for (int ks = 0; ks < a.kss; ++ks) {
            if (ok && !warp_wait(&full[slot], (uint32_t)ph, ctl)) ok = false;
            int c0;
            const int n = ok ? stage_chunks(s, ks, c0) : 0;
            const uint32_t st = ring + (uint32_t)slot * a.stage_bytes + (uint32_t)(wg * kR) * kChunkBytes;
            for (int c = 0; c < n; ++c) {
                const uint32_t rows = st + (uint32_t)c * (uint32_t)RS * kChunkBytes;   // row kR * wg of chunk c
                const int ch = c0 + c;
                if constexpr (FMT == BQ_Q8_0_I8) {
                    // block `lane`: its 32 activation codes (two 16-byte pieces),
                    // then per row the exact integer dot of the codes (dp4a)
                    const uint32_t xp = xs_base + (uint32_t)(ch * 2 * 32 + lane) * 16u;
                    const uint4 xa = lds128(xp), xb = lds128(xp + 32u * 16u);
                    const int xw[8] = {(int)xa.x, (int)xa.y, (int)xa.z, (int)xa.w,
                                       (int)xb.x, (int)xb.y, (int)xb.z, (int)xb.w};
                    const float dx = sums[ch * 32 + lane];
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        const uint32_t bp = rows + (uint32_t)r * kChunkBytes + 36u * (uint32_t)lane;
                        const uint32_t hdr = lds32(bp);
                        int dot = 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) dot = __dp4a((int)lds32(bp + 4u + 4u * (uint32_t)i), xw[i], dot);
                        part[r] = fmaf(f16_bits_to_f32(hdr) * dx, (float)dot, part[r]);   // |dot| < 2^24: exact
                    }
                } else if constexpr (FMT == BQ_Q8_0) {
                    // block `lane` of the chunk: 9 words at 36 * lane (odd word
                    // stride: no bank conflicts)
                    const uint32_t xp = xs_base + (uint32_t)(ch * 8 * 32 + lane) * 16u;
                    float4 xv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) xv[i] = lds128f(xp + (uint32_t)i * 32u * 16u);
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        const uint32_t bp = rows + (uint32_t)r * kChunkBytes + 36u * (uint32_t)lane;
                        const uint32_t hdr = lds32(bp);
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t w = lds32(bp + 4u + 4u * (uint32_t)i);
                            const uint32_t u0 = w << 15, u1 = w << 7, u2 = w >> 1, u3 = w >> 9;
                            acc = fma2q(codes2(lop3_andxor(u0, c_mask, c_const), lop3_andxor(u1, c_mask, c_const),
                                               r_m_lo, r_m_hi, r_c_lo, r_c_hi),
                                        xv[i].x, xv[i].y, acc);
                            acc = fma2q(codes2(lop3_andxor(u2, c_mask, c_const), lop3_andxor(u3, c_mask, c_const),
                                               r_m_lo, r_m_hi, r_c_lo, r_c_hi),
                                        xv[i].z, xv[i].w, acc);
                        }
                        part[r] = fmaf(f16_bits_to_f32(hdr), acc.x + acc.y, part[r]);
                    }
                } else if (ch == a.chunks - 1 && a.last_half) {
                    // A last chunk of at most 4 super-blocks (16 items): lanes
                    // 16..31 take the warp's second row instead of zero-filled items.
                    const int it = lane & 15, rr = lane >> 4;
                    const int sb = it >> 2, g = it & 3;
                    const int sub = 8 * (ch * 8 + sb) + 2 * g;
                    const float sx_lo = sums[sub], sx_hi = sums[sub + 1];
                    float2 acc = make_float2(0.f, 0.f);
                    const uint32_t xp = xs_base + (uint32_t)(ch * 16 * 32 + it) * 16u;
                    const uint32_t rowa = rows + (uint32_t)rr * kChunkBytes;
                    const uint32_t qoff = 144u * (uint32_t)sb + 16u + 32u * (uint32_t)g;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 qv = lds128(rowa + qoff + 16u * (uint32_t)h);
                        const uint32_t wv[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float4 p0 = lds128f(xp + (uint32_t)(8 * h + 2 * t) * 32u * 16u);
                            const float4 p1 = lds128f(xp + (uint32_t)(8 * h + 2 * t + 1) * 32u * 16u);
                            acc = q4k_word(wv[t], p0, p1, acc);
                        }
                    }
                    const uint4 hdr = lds128(rowa + 144u * (uint32_t)sb);
                    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
                    float sc_lo, m_lo, sc_hi, m_hi;
                    scale_min_pair(hdr.y, hdr.z, hdr.w, g, sc_lo, m_lo, sc_hi, m_hi);
                    const float* scl = sums + 2 * a.chunks * 32;   // the item's scale-back factors
                    const int itm = ch * 32 + 4 * sb + g;
                    acc.x = (acc.x * scl[2 * itm]) * scl[2 * itm + 1];
                    acc.y = (acc.y * scl[2 * itm]) * scl[2 * itm + 1];
                    float v = 0.f;
                    v = fmaf(d * sc_lo, acc.x, v);
                    v = fmaf(-(dmin * m_lo), sx_lo, v);
                    v = fmaf(d * sc_hi, acc.y, v);
                    v = fmaf(-(dmin * m_hi), sx_hi, v);
                    static_assert(kR == 2, "the half-chunk mapping pairs the warp's two rows");
                    part[0] += rr == 0 ? v : 0.f;
                    part[1] += rr == 1 ? v : 0.f;
                } else {
                    // item lane = 4 sb + g: header of super-block sb, code bytes 32 g .. 32 g + 31
                    const int sb = lane >> 2, g = lane & 3;
                    const int sub = 8 * (ch * 8 + sb) + 2 * g;   // global sub-block of the low nibbles
                    const float sx_lo = sums[sub], sx_hi = sums[sub + 1];
                    float2 acc[kR];
#pragma unroll
                    for (int r = 0; r < kR; ++r) acc[r] = make_float2(0.f, 0.f);
                    const uint32_t xp = xs_base + (uint32_t)(ch * 16 * 32 + lane) * 16u;
                    const uint32_t qoff = 144u * (uint32_t)sb + 16u + 32u * (uint32_t)g;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // code words 4h .. 4h + 3 (bytes i = 16h .. 16h + 15 of the run),
                        // activation pairs (x_lo_i, x_hi_i) in pair quads 8h .. 8h + 7
                        float4 xv[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) xv[q] = lds128f(xp + (uint32_t)(8 * h + q) * 32u * 16u);
#pragma unroll
                        for (int r = 0; r < kR; ++r) {
                            const uint4 qv = lds128(rows + (uint32_t)r * kChunkBytes + qoff + 16u * (uint32_t)h);
                            const uint32_t wv[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                acc[r] = q4k_word(wv[t], xv[2 * t], xv[2 * t + 1], acc[r]);
                            }
                        }
                    }
                    const float* scl = sums + 2 * a.chunks * 32;   // this item's scale-back factors
                    const float sk1 = scl[2 * (ch * 32 + lane)], sk2 = scl[2 * (ch * 32 + lane) + 1];
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        acc[r].x = (acc[r].x * sk1) * sk2;
                        acc[r].y = (acc[r].y * sk1) * sk2;
                        const uint4 hdr = lds128(rows + (uint32_t)r * kChunkBytes + 144u * (uint32_t)sb);
                        const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
                        float sc_lo, m_lo, sc_hi, m_hi;
                        scale_min_pair(hdr.y, hdr.z, hdr.w, g, sc_lo, m_lo, sc_hi, m_hi);
                        float v = part[r];
                        v = fmaf(d * sc_lo, acc[r].x, v);
                        v = fmaf(-(dmin * m_lo), sx_lo, v);
                        v = fmaf(d * sc_hi, acc[r].y, v);
                        v = fmaf(-(dmin * m_hi), sx_hi, v);
                        part[r] = v;
                    }
                }
            }
            // the slot is refilled by TMA (async proxy): order these reads first, then release it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            slot += S;
            if (slot >= D) {
                slot -= D;
                ph ^= 1;
            }
        }
        // this set's sums for the warp's rows of the group, held until the next flush
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const float v = warp_sum(part[r]);
            if (lane == 0) pend[((buf * kFlush + fi) * S + s) * RS + wg * kR + r] = v;
        }
        const bool last = rg + (int)gridDim.x >= a.n_groups;
        if (++fi == kFlush || last) {
            consumer_bar();
            // rows of the flushed groups: sets added in order s = 0, 1, ...
            const int nrows = fi * RS;
            for (int t = threadIdx.x; t < nrows; t += kCW * 32) {
                const int f = t / RS, r = t - f * RS;
                float v = 0.f;
                for (int ss = 0; ss < S; ++ss) v += pend[((buf * kFlush + f) * S + ss) * RS + r];
                const int grp = rg - (fi - 1 - f) * (int)gridDim.x;
                const int64_t n = (int64_t)grp * RS + r;
                if (n < a.N) a.out[n] = v;
            }
            buf ^= 1;
            fi = 0;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) q8_0_tma_kernel(const __grid_constant__ CUtensorMap wmap, const BqArgs a) {
    bq_tma_body<BQ_Q8_0>(wmap, a);
}
__global__ void __launch_bounds__(kThreads, 1) q4_k_tma_kernel(const __grid_constant__ CUtensorMap wmap, const BqArgs a) {
    bq_tma_body<BQ_Q4_K>(wmap, a);
}
__global__ void __launch_bounds__(kThreads, 1) q8_0_i8_tma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                  const BqArgs a) {
    bq_tma_body<BQ_Q8_0_I8>(wmap, a);
}

int num_sms_cached() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return sms;
}

// chooses G (rows per stage) by rounds x chunks per set, then C and the depth
bool plan_bq(int64_t N, int chunks, int K, int fmt, BqArgs& a, size_t& smem) {
    const int sms = num_sms_cached();
    // One set of all consumer warps: every stage is a whole chunk of kR * 16
    // rows (a K split between sets leaves sets idle when a row is a few
    // chunks long, and halves the bytes in flight per set).
    (void)sms;
    const int bestG = kCW;
    a.G = bestG;
    a.S = kCW / bestG;
    a.cps = (chunks + a.S - 1) / a.S;
    a.C = std::min(a.cps, std::max(1, 8 / bestG));
    a.kss = (a.cps + a.C - 1) / a.C;
    a.chunks = chunks;
    a.N = (int)N;
    a.K = K;
    const int sb_last = (K / 256) % 8;
    a.last_half = fmt == BQ_Q4_K && sb_last != 0 && sb_last <= 4;
    a.n_groups = (int)((N + kR * a.G - 1) / (kR * a.G));
    a.stage_bytes = (uint32_t)a.C * (uint32_t)(kR * a.G) * kChunkBytes;
    const size_t x_bytes = (size_t)chunks * (fmt == BQ_Q4_K ? 2048 * 4 : (fmt == BQ_Q8_0 ? 1024 * 4 : 1024));
    const size_t sum_bytes = (size_t)chunks * 32 * (fmt == BQ_Q4_K ? 4 : 1) * 4;   // Q4_K: two sums, two scale factors
    const size_t pend_bytes = (size_t)2 * kFlush * kCW * kR * 4;
    const size_t bar_bytes = 2 * kMaxDepth * 8 + 16;
    const size_t fixed = 128 + x_bytes + sum_bytes + pend_bytes + bar_bytes;
    const size_t cap = 227 * 1024;
    if (fixed + 2 * (size_t)a.S * a.stage_bytes > cap) return false;
    int D = (int)((cap - fixed) / a.stage_bytes);
    D = std::min(D, kMaxDepth);
    D -= D % a.S;   // slot s is always read by set s % S
    if (D < 2 * a.S) return false;
    a.depth = D;
    size_t off = (size_t)D * a.stage_bytes;   // ring first (128-byte aligned base)
    a.x_off = (uint32_t)off;
    off += x_bytes;
    a.sum_off = (uint32_t)off;
    off += sum_bytes;
    a.pend_off = (uint32_t)off;
    off += pend_bytes;
    off = (off + 7) & ~(size_t)7;
    a.bar_off = (uint32_t)off;
    off += bar_bytes;
    smem = off + 128;
    return smem <= cap;
}

template <int FMT>
cudaError_t launch_bq(const void* blocks, const float* x, const int8_t* xq, const float* xd, float* out, int64_t N,
                      int64_t K, size_t row_bytes, int* status, long long spin_limit, cudaStream_t stream) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int chunks = (int)((row_bytes + kChunkBytes - 1) / kChunkBytes);
    BqArgs a;
    size_t smem = 0;
    if (!plan_bq(N, chunks, (int)K, FMT, a, smem)) return cudaErrorNotSupported;
    CUtensorMap wmap;
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)kChunkU64, (cuuint32_t)(kR * a.G)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(blocks), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    a.x = x;
    a.xq = xq;
    a.xd = xd;
    a.out = out;
    a.status = status;
    a.spin_limit = spin_limit;
    if (!a.status) return cudaErrorInvalidValue;
    using KernFn = void (*)(const CUtensorMap, const BqArgs);
    const KernFn kern = FMT == BQ_Q8_0 ? q8_0_tma_kernel : (FMT == BQ_Q4_K ? q4_k_tma_kernel : q8_0_i8_tma_kernel);
    static unsigned long long configured = 0ull;   // bit (3 * device + format)
    int dev = 0;
    cudaGetDevice(&dev);
    const int bit = 3 * dev + FMT;
    if (bit >= 64 || !(configured & (1ull << bit))) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        if (bit < 64) configured |= 1ull << bit;
    }
    const int grid = (int)std::min<int64_t>(a.n_groups, num_sms_cached());
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, wmap, a);
}

// Test aid: one thread per (super-block, 64-weight group g) writes the group's
// 64 weights w = d * sc * q - dmin * m (one rounding: d * sc * q and dmin * m
// are exact in binary32) with the (sc, m) of sub-blocks 2g and 2g + 1 from
// scale_min_pair, the decoder of q4_k_tma_kernel, reading the 16-byte header
// as that kernel does.
__global__ void q4_k_dequant_tma_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out, int64_t nblk) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nblk * 4) return;
    const int64_t b = t >> 2;
    const int g = (int)(t & 3);
    const uint8_t* blk = blocks + b * 144;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    float sc_lo, m_lo, sc_hi, m_hi;
    scale_min_pair(hdr.y, hdr.z, hdr.w, g, sc_lo, m_lo, sc_hi, m_hi);
    float* o = out + b * 256 + 64 * g;
    for (int i = 0; i < 32; ++i) {
        const uint32_t qb = blk[16 + 32 * g + i];
        o[i] = fmaf(d * sc_lo, (float)(qb & 15u), -(dmin * m_lo));
        o[32 + i] = fmaf(d * sc_hi, (float)(qb >> 4), -(dmin * m_hi));
    }
}

}  // namespace

cudaError_t launch_q4_k_dequant_tma(const uint8_t* blocks, float* out, int64_t nblk, cudaStream_t s) {
    const int64_t threads = nblk * 4;
    q4_k_dequant_tma_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(blocks, out, nblk);
    return cudaGetLastError();
}

// Rows must start on 16-byte boundaries (TMA) and the staged activations must
// fit in shared memory next to a ring of at least two stages per set.
bool bq_tma_supported(int fmt, int64_t N, int64_t K, const void* blocks, const void* x) {
    if (N <= 0 || N > (int64_t)1 << 30 || K <= 0 || K > (int64_t)1 << 20) return false;
    if (((uintptr_t)blocks & 15u) || ((uintptr_t)x & 15u)) return false;
    const size_t row_bytes = fmt == BQ_Q4_K ? (size_t)K / 256 * 144 : (size_t)K / 32 * 36;
    if (row_bytes % 16 != 0) return false;
    if (!encode_fn()) return false;
    BqArgs a;
    size_t smem = 0;
    const int chunks = (int)((row_bytes + kChunkBytes - 1) / kChunkBytes);
    return plan_bq(N, chunks, (int)K, fmt, a, smem);
}

cudaError_t launch_q8_0_gemv_tma(const uint32_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                                 int* status, long long spin_limit, cudaStream_t s) {
    return launch_bq<BQ_Q8_0>(blocks, x, nullptr, nullptr, out, N, K, (size_t)K / 32 * 36, status, spin_limit, s);
}
cudaError_t launch_q4_k_gemv_tma(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                                 int* status, long long spin_limit, cudaStream_t s) {
    return launch_bq<BQ_Q4_K>(blocks, x, nullptr, nullptr, out, N, K, (size_t)K / 256 * 144, status, spin_limit, s);
}
cudaError_t launch_q8_0_i8_gemv_tma(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out, int64_t N,
                                    int64_t K, int* status, long long spin_limit, cudaStream_t s) {
    return launch_bq<BQ_Q8_0_I8>(blocks, nullptr, xq, xd, out, N, K, (size_t)K / 32 * 36, status, spin_limit, s);
}

}  // namespace gai4
