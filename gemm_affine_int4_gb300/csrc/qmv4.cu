// qmv4.cu -- CUDA-core qmv (M = 1) for 4-bit codes, group size 32/64/128,
// bf16 / f16 / f32 activations, binary32 accumulation.
//
// out[n] = sum_g ( s[n,g] * sum_{k in g} q[n,k] x[k] + b[n,g] * sum_{k in g} x[k] )
// (metaltile-std quantized.rs, mt_qmv: the bias-hoist split of the affine dot
// product; coalesced 128-bit weight reads, x reused across rows, warp-shuffle
// reduction.)
//
// GB300 design:
//  * One CTA per SM, persistent over blocks of BR = (24 / S) * R rows: 24
//    consumer warps and one producer warp. A consumer warp owns R rows of a
//    block; S warps split the 1024-column iterations of a row group when rows
//    alone would leave SMs idle. A lane owns 32 consecutive codes (16 bytes)
//    of each of its rows per iteration.
//  * The producer's elected thread streams each stage -- S iterations of the
//    block's packed weights, scales and biases -- into a ring of shared-memory
//    stages (full / empty mbarriers, zero fill past N). When K is a multiple
//    of 1024 the tensors are viewed as [rows][iterations][columns] and one
//    3-D TMA box per tensor brings a whole stage; otherwise one 2-D box per
//    iteration (zero fill past K). Consumer lanes issue no copies and no
//    global loads in the loop.
//  * x is staged once per CTA, permuted so that a warp's 16-byte reads are
//    contiguous, with per-chunk sums for the bias term: 16-bit activations
//    as pairs (x_j, x_{j+4}) of the same type, binary32 ones scaled per
//    element (below).
//  * Every product q x is exact before it is summed, so a chunk whose codes
//    are all zero adds exactly zero (no offset is ever subtracted).
//    16-bit activations: a 16-bit value whose exponent field is 0 or 1 is
//    its low 8 bits times the smallest subnormal (2^-133 in bf16, 2^-24 in
//    f16), so one AND of a word with 0x000F000F gives the pair
//    (q_0, q_4) * 2^-e and one with 0x00F000F0 the pair (q_1, q_5) * 2^-e * 16,
//    exactly, and the same on the word shifted by 8 gives codes 2, 6 and 3, 7.
//    Each half feeds one mixed-precision fma (binary32 += a * b, both factors
//    16-bit, the product exact) into one of two accumulators per row (codes
//    in bits 0..3 or 4..7 of a half), joined as a + b / 16. Per word
//    of 8 codes: 1 shift, 4 ANDs, 8 fmas. The f16 products (at least 2^-48 in
//    magnitude) are
//    binary32 normals; for bf16 each 32-element chunk of x is scaled by a
//    power of two 2^k that puts its largest magnitude in [2^127, 2^128), so
//    the products are binary32 normals down to 2^-120 of that magnitude, and
//    the chunk's code sum is scaled back by 2^(133-k).
//    binary32 activations: a binary32 whose bits above bit 23 are clear is
//    those bits times 2^-149 (bit 23 joins the exponent seamlessly), so code
//    j of a word, masked in place at bits 4j.. (j < 6) or at bits 4 (j - 6)..
//    of the word shifted by 24, is exactly q_j * 2^(bit - 149). x_j is staged
//    times 2^(kc - bit), kc chosen per 32-element chunk so that its largest
//    magnitude lands just below 2^127; a packed fma (fma.rn.f32x2) adds the
//    exact product q_j x_j 2^(kc - 149), and the chunk's code sum is scaled
//    back by 2^(149 - kc). Per word: 1 shift, 8 ANDs, 4 packed fmas.
#include <algorithm>
#include <initializer_list>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace gai4 {

namespace {

using namespace pipe;

#ifndef QMV4_CWARPS
#define QMV4_CWARPS 24
#endif
constexpr int kCWarps = QMV4_CWARPS;               // consumer warps
constexpr int kThreads = 32 * (kCWarps + 1);       // + one producer warp
constexpr int kItCols = 1024;                      // columns of one warp iteration (32 lanes x 32 codes)
constexpr int kMaxDepth = 8;

struct Qmv4Args {
    const void* x;
    void* out;
    int64_t N, K;
    int gs_log2;
    int S;                  // warps splitting the iterations of one row group
    int n_it;               // iterations per row: ceil(K / 1024)
    int n_st;               // stages per block: ceil(n_it / S)
    int depth;              // ring depth
    int64_t n_blocks;       // row blocks
    int sbg;                // groups per iteration: 1024 / group_size
    uint32_t w_slice;       // bytes of one iteration's packed weights in a stage: BR * 512
    uint32_t sb_slice;      // bytes of one iteration's scales (or biases), padded to 128
    uint32_t stage_bytes;   // S * (w_slice + 2 * sb_slice)
    int box3;               // 1: one 3-D box per tensor and stage, layout [row][iteration][...]
    uint32_t w_rs, w_is;    // byte strides of a row and of an iteration in a stage's packed weights
    uint32_t sb_rs, sb_is;  // element strides of a row and of an iteration in a stage's scales / biases
    int flush;              // row blocks whose partial sums are held in shared memory between flushes
    int* status;
    long long spin_limit;
};

// (acc.x + a_lo * b_lo, acc.y + a_hi * b_hi): two binary32 fmas in one instruction
__device__ __forceinline__ float2 ffma2(uint32_t a_lo, uint32_t a_hi, float b_lo, float b_hi, float2 c) {
    float2 d;
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
        " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "r"(a_lo), "r"(a_hi), "f"(b_lo), "f"(b_hi), "f"(c.x), "f"(c.y));
    return d;
}

// acc + q.lo * x.lo + q.hi * x.hi: a binary32 accumulator, 16-bit factors
// (mixed-precision fma: each product exact, one rounding per fma)
template <bool BF>
__device__ __forceinline__ void mfma2(uint32_t q2, uint32_t x2, float& acc) {
    if constexpr (BF)
        asm("{\n .reg .b16 ql, qh, xl, xh;\n mov.b32 {ql, qh}, %1;\n mov.b32 {xl, xh}, %2;\n"
            " fma.rn.f32.bf16 %0, ql, xl, %0;\n fma.rn.f32.bf16 %0, qh, xh, %0;\n}"
            : "+f"(acc)
            : "r"(q2), "r"(x2));
    else
        asm("{\n .reg .b16 ql, qh, xl, xh;\n mov.b32 {ql, qh}, %1;\n mov.b32 {xl, xh}, %2;\n"
            " fma.rn.f32.f16 %0, ql, xl, %0;\n fma.rn.f32.f16 %0, qh, xh, %0;\n}"
            : "+f"(acc)
            : "r"(q2), "r"(x2));
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory"); }

template <typename T, int R>
__global__ void __launch_bounds__(kThreads, 1)
    qmv4_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                const __grid_constant__ CUtensorMap bmap, const Qmv4Args a) {
    using St = typename T::storage;
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();
    // 128-byte aligned base (TMA destinations); pointer arithmetic on the
    // shared array keeps the accesses below in the shared state space
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int n_it = a.n_it, D = a.depth, S = a.S, n_st = a.n_st;
    const int G = kCWarps / S, BR = G * R;
    constexpr int kXP = T::kBytes == 4 ? 8 : 4;                       // 16-byte x pieces per lane and iteration
    uint4* xs = reinterpret_cast<uint4*>(smem);                       // [n_it][kXP][32] permuted x
    float4* cs = reinterpret_cast<float4*>(xs + (size_t)n_it * kXP * 32);   // [n_it * 32] (sum x, 2^a, 2^b, 0)
    uint8_t* ring = reinterpret_cast<uint8_t*>(cs + (size_t)n_it * 32);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)D * a.stage_bytes);
    uint64_t* empty = full + kMaxDepth;
    float* pend = reinterpret_cast<float*>(empty + kMaxDepth);        // [flush][kCWarps * R] partial sums
    volatile int* abort_flag = reinterpret_cast<volatile int*>(pend + (size_t)a.flush * kCWarps * R);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t my_blocks =
        a.n_blocks > (int64_t)blockIdx.x ? (a.n_blocks - 1 - (int64_t)blockIdx.x) / gridDim.x + 1 : 0;

    Ctl ctl{a.status, a.spin_limit, abort_flag};

    if (warp == kCWarps) {
        // ---------------- producer ----------------
        // stage q of this CTA (block q / n_st, iterations S (q % n_st) ..)
        // into ring slot q % D
        auto issue = [&](int64_t q) {
            const int64_t b = q / n_st;
            const int j = (int)(q - b * n_st), slot = (int)(q % D);
            const int row0 = (int)(((int64_t)blockIdx.x + b * gridDim.x) * BR);
            const int it0 = j * S;
            const int nsl = min(S, n_it - it0);   // iterations present in this stage
            // a 3-D box always lands whole (iterations past the row are zero-filled)
            const uint32_t n_its = a.box3 ? (uint32_t)S : (uint32_t)nsl;
            mbar_arrive_expect_tx(&full[slot],
                                  n_its * (a.w_slice + 2u * (uint32_t)BR * (uint32_t)a.sbg * (uint32_t)sizeof(St)));
            uint8_t* st = ring + (size_t)slot * a.stage_bytes;
            if (a.box3) {
                tma_load_3d(st, &wmap, &full[slot], 0, it0, row0);
                uint8_t* sbs = st + (size_t)S * a.w_slice;
                tma_load_3d(sbs, &smap, &full[slot], 0, it0, row0);
                tma_load_3d(sbs + (size_t)S * a.sb_slice, &bmap, &full[slot], 0, it0, row0);
            } else for (int ss = 0; ss < nsl; ++ss) {
                const int it = it0 + ss;
                tma_load_2d(st + ss * a.w_slice, &wmap, &full[slot], it * (kItCols / 8), row0);
                uint8_t* sbs = st + (size_t)S * a.w_slice + (size_t)ss * a.sb_slice;
                tma_load_2d(sbs, &smap, &full[slot], it * a.sbg, row0);
                tma_load_2d(sbs + (size_t)S * a.sb_slice, &bmap, &full[slot], it * a.sbg, row0);
            }
        };
        const int64_t total = my_blocks * n_st;
        int64_t issued = 0;
        if (lane == 0) {
            // x first into L2 (at the head of the DRAM queue), then the tensor maps
            bulk_prefetch_l2(a.x, (uint32_t)(a.K * (int64_t)sizeof(St)));   // K % 32 == 0: whole 16-byte units
            asm volatile("prefetch.tensormap [%0];" ::"l"(&wmap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&smap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&bmap) : "memory");
            for (int i = 0; i < D; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], kCWarps);   // one arrive per consumer warp
            }
            *abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the barriers, as the copies see them
            // The packed weights, scales and biases are not written by the
            // kernels this one may overlap (programmatic launch): the first
            // stage is requested at once, before those kernels complete (the
            // rest of the ring follows once the CTA is set up: requested
            // alone, the first stage lands sooner). Only the activations wait
            // for those kernels.
            if (total > 0) issue(issued++);
        }
        __syncwarp();
        __syncthreads();   // the barriers are initialised (and the consumers have staged x)
        if (lane == 0) {
            for (; issued < total; ++issued) {
                if (!mbar_wait(&empty[issued % D], (uint32_t)(((issued / D) & 1) ^ 1), ctl)) break;
                issue(issued);
            }
            // every issued copy has landed before the CTA may exit
            for (int64_t q = (issued > D ? issued - D : 0); q < issued; ++q)
                mbar_wait_drain(&full[q % D], (uint32_t)((q / D) & 1), a.spin_limit, a.status);
        }
        return;
    }

    pdl_wait();   // the kernels before this one are complete: global memory may be read

    // ---------------- consumers: stage x once ----------------
    // a thread takes 8 consecutive elements (word qq of a 32-element chunk);
    // the 4 words of a chunk sit in 4 adjacent lanes and add their sums with
    // shuffles
    const St* xg = static_cast<const St*>(a.x);
    const int64_t K = a.K;
    for (int u = threadIdx.x; u < n_it * 128; u += kCWarps * 32) {   // n_it * 128 is a multiple of 32
        const int c = u >> 2, qq = u & 3;
        const int64_t k0 = (int64_t)u * 8;
        float v[8];
        if constexpr (T::kBytes == 4) {
            float4 f0 = make_float4(0.f, 0.f, 0.f, 0.f), f1 = f0;
            if (k0 < K) {   // K is a multiple of 32: a chunk is all in or all out
                f0 = *reinterpret_cast<const float4*>(xg + k0);
                f1 = *reinterpret_cast<const float4*>(xg + k0 + 4);
            }
            v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
            v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
            // chunk scale 2^kc: the largest magnitude's exponent field E -> kc = 253 - E
            uint32_t eb = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) eb = max(eb, __float_as_uint(v[j]) & 0x7F800000u);
            eb = max(eb, __shfl_xor_sync(0xffffffffu, eb, 1));
            eb = max(eb, __shfl_xor_sync(0xffffffffu, eb, 2));
            const int E = max((int)(eb >> 23), 1);   // subnormal or zero chunk: as E = 1
            const int kc = max(253 - E, -2);          // Inf / NaN: kept as they are
            // code j of a word is read in place at bit 4j (j < 6) or, after a shift
            // by 24, at bit 4 (j - 6): x_j is staged times 2^(kc - that bit), in two
            // exact power-of-two steps
            uint32_t xb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = kc - (j < 6 ? 4 * j : 4 * (j - 6));
                const int ea = e / 2, eb2 = e - e / 2;
                xb[j] = __float_as_uint((v[j] * __uint_as_float((uint32_t)(127 + ea) << 23)) *
                                        __uint_as_float((uint32_t)(127 + eb2) << 23));
            }
            xs[((c >> 5) * 8 + 2 * qq) * 32 + (c & 31)] = make_uint4(xb[0], xb[1], xb[2], xb[3]);
            xs[((c >> 5) * 8 + 2 * qq + 1) * 32 + (c & 31)] = make_uint4(xb[4], xb[5], xb[6], xb[7]);
            if (qq == 0) {
                // code sums come out times 2^(kc - 149): back by 2^p, p = 149 - kc
                const int p = 149 - kc;
                cs[c].y = __uint_as_float((uint32_t)(127 + p / 2) << 23);
                cs[c].z = __uint_as_float((uint32_t)(127 + p - p / 2) << 23);
            }
        } else {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (k0 < K) q = *reinterpret_cast<const uint4*>(xg + k0);
            uint32_t uu[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[2 * h] = T::to_f32((uint16_t)(uu[h] & 0xFFFFu));
                v[2 * h + 1] = T::to_f32((uint16_t)(uu[h] >> 16));
            }
            if constexpr (T::kIsBF16) {
                // chunk scale 2^k: the largest magnitude's exponent field E -> 254
                uint32_t mb = 0u;
#pragma unroll
                for (int h = 0; h < 4; ++h) mb = max(mb, max(uu[h] & 0x7FFFu, (uu[h] >> 16) & 0x7FFFu));
                mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
                mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
                const int E = max((int)(mb >> 7), 1);                // subnormal or zero chunk: as E = 1
                const int k = max(254 - E, 0);                        // Inf / NaN: no scaling
                const float s1 = __uint_as_float((uint32_t)(127 + (k >> 1)) << 23);
                const float s2 = __uint_as_float((uint32_t)(127 + k - (k >> 1)) << 23);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn((v[2 * h] * s1) * s2));
                    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn((v[2 * h + 1] * s1) * s2));
                    uu[h] = lo | (hi << 16);
                }
                if (qq == 0) {
                    const int p = 133 - k;                            // the code sum is scaled back by 2^p
                    cs[c].y = __uint_as_float((uint32_t)(127 + (p >> 1)) << 23);
                    cs[c].z = __uint_as_float((uint32_t)(127 + p - (p >> 1)) << 23);
                }
            } else if (qq == 0) {
                cs[c].y = 16777216.f;   // 2^24
                cs[c].z = 1.f;
            }
            // pairs (x_j, x_{j+4}), j = 0..3, the order of the decoded code pairs
            xs[((c >> 5) * 4 + qq) * 32 + (c & 31)] =
                make_uint4(__byte_perm(uu[0], uu[2], 0x5410), __byte_perm(uu[0], uu[2], 0x7632),
                           __byte_perm(uu[1], uu[3], 0x5410), __byte_perm(uu[1], uu[3], 0x7632));
        }
        // chunk sum (unscaled x) in a fixed order
        float xsum = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
        if (qq == 0) {
            cs[c].x = xsum;
            cs[c].w = 0.f;
        }
    }
    __syncthreads();   // x staged; the ring's barriers are initialised

    // ---------------- consumers: main loop ----------------
    const int g = warp / S, sl = warp % S;
    // operands of the logic ops and exact subtractions, kept in registers
    constexpr bool kBF = T::kBytes == 2 && T::kIsBF16;
    const uint32_t m2 = pin_reg(0x000F000Fu), mh2 = pin_reg(0x00F000F0u);
    // binary32: masks of code bits 0.., 4.., .., 20..; a masked code is an exact
    // subnormal, code * 2^(bit - 149)
    const uint32_t f0 = pin_reg(0xFu), f1 = pin_reg(0xF0u), f2 = pin_reg(0xF00u), f3 = pin_reg(0xF000u),
                   f4 = pin_reg(0xF0000u), f5 = pin_reg(0xF00000u);
    const int grp_off = (lane * 32) >> a.gs_log2;   // this lane's group within an iteration
    St* out = static_cast<St*>(a.out);
    int slot = 0, ph = 0;
    for (int64_t b = 0; b < my_blocks; ++b) {
        float part[R];
#pragma unroll
        for (int r = 0; r < R; ++r) part[r] = 0.f;
        for (int j = 0; j < n_st; ++j) {
            const int it = j * S + sl;
            const bool ok = warp_wait(&full[slot], (uint32_t)ph, ctl);
            if (ok && it < n_it) {
                const uint8_t* st = ring + (size_t)slot * a.stage_bytes;
                const uint8_t* wsl = st + (size_t)sl * a.w_is + (size_t)(g * R) * a.w_rs + lane * 16;
                const St* ssl = reinterpret_cast<const St*>(st + (size_t)S * a.w_slice) + sl * a.sb_is +
                                (g * R) * a.sb_rs + grp_off;
                const St* bsl = ssl + (size_t)S * a.sb_slice / sizeof(St);
                uint4 wv[R];
                float sc[R], bc[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    wv[r] = *reinterpret_cast<const uint4*>(wsl + r * a.w_rs);
                    sc[r] = T::to_f32(ssl[r * a.sb_rs]);
                    bc[r] = T::to_f32(bsl[r * a.sb_rs]);
                }
                // the slot is refilled by TMA (async proxy): order these reads first, then release it
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);

                const float4 cst = cs[it * 32 + lane];   // (sum x, 2^a, 2^b): sum q x = code sum * 2^a * 2^b
                float2 acc[R];   // per row: codes in bits 0..3 (x) and 4..7 (y) of a half
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int tw = 0; tw < 4; ++tw) {
                    if constexpr (T::kBytes == 2) {
                        const uint4 xp = xs[(it * 4 + tw) * 32 + lane];   // (x_j, x_{j+4}), j = 0..3
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t w = tw == 0 ? wv[r].x : (tw == 1 ? wv[r].y : (tw == 2 ? wv[r].z : wv[r].w));
                            const uint32_t w8 = w >> 8;
                            mfma2<kBF>(w & m2, xp.x, acc[r].x);    // codes 0, 4
                            mfma2<kBF>(w & mh2, xp.y, acc[r].y);   // codes 1, 5 (times 16)
                            mfma2<kBF>(w8 & m2, xp.z, acc[r].x);   // codes 2, 6
                            mfma2<kBF>(w8 & mh2, xp.w, acc[r].y);  // codes 3, 7 (times 16)
                        }
                    } else {
                        const uint4 p0 = xs[(it * 8 + 2 * tw) * 32 + lane];
                        const uint4 p1 = xs[(it * 8 + 2 * tw + 1) * 32 + lane];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t w = tw == 0 ? wv[r].x : (tw == 1 ? wv[r].y : (tw == 2 ? wv[r].z : wv[r].w));
                            const uint32_t h = w >> 24;   // codes 6, 7 at bits 0.., 4..
                            float2 a2 = acc[r];
                            a2 = ffma2(w & f0, w & f1, __uint_as_float(p0.x), __uint_as_float(p0.y), a2);
                            a2 = ffma2(w & f2, w & f3, __uint_as_float(p0.z), __uint_as_float(p0.w), a2);
                            a2 = ffma2(w & f4, w & f5, __uint_as_float(p1.x), __uint_as_float(p1.y), a2);
                            a2 = ffma2(h & f0, h & f1, __uint_as_float(p1.z), __uint_as_float(p1.w), a2);
                            acc[r] = a2;
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float qx;   // sum q x of the chunk
                    if constexpr (T::kBytes == 2)
                        qx = (fmaf(0.0625f, acc[r].y, acc[r].x) * cst.y) * cst.z;
                    else
                        qx = ((acc[r].x + acc[r].y) * cst.y) * cst.z;
                    part[r] = fmaf(sc[r], qx, fmaf(bc[r], cst.x, part[r]));
                }
            } else {
                // nothing to read (an iteration past K, or a wait that gave up): release the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            if (++slot == D) {
                slot = 0;
                ph ^= 1;
            }
        }
        // the warp's row sums, held until the next flush; a flush adds the S
        // warps of each row group in a fixed order and writes the rows (no
        // barrier or global store inside the stage loop: a store would make
        // the next mbarrier arrive wait for it)
        const int bl = (int)(b % a.flush);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v = warp_sum(part[r]);
            if (lane == 0) pend[(size_t)bl * (kCWarps * R) + warp * R + r] = v;
        }
        if (bl == a.flush - 1 || b == my_blocks - 1) {
            consumer_bar();
            const int64_t b0 = b - bl;
            for (int t = threadIdx.x; t < (bl + 1) * BR; t += kCWarps * 32) {
                const int bb = t / BR, rr = t - bb * BR;
                const int gg = rr / R, r = rr - gg * R;
                const float* pb = pend + (size_t)bb * (kCWarps * R);
                float v = 0.f;
                for (int ss = 0; ss < S; ++ss) v += pb[(gg * S + ss) * R + r];
                const int64_t row = ((int64_t)blockIdx.x + (b0 + bb) * gridDim.x) * BR + rr;
                if (row < a.N) out[row] = T::from_f32(v);
            }
            consumer_bar();
        }
    }
}

// (R, S): per stage a CTA spends about max(producer issue, one iteration of R
// rows per warp) -- roughly max(800, 400 R) cycles -- so the busiest SM takes
// ceil(blocks / SMs) * ceil(n_it / S) * max(2, R) units; ties go to more rows
// per warp, then to fewer K splits
struct Qmv4Plan {
    int R, S, depth, flush;
    int64_t n_blocks;
    uint32_t w_slice, sb_slice, stage_bytes;
    size_t smem;
};

bool plan_qmv4(int64_t N, int64_t K, int gs, int tbytes, Qmv4Plan* out) {
    const int sms = num_sms();
    const int n_it = (int)((K + kItCols - 1) / kItCols);
    const int sbg = kItCols / gs;
    const size_t fixed = (size_t)n_it * ((tbytes == 4 ? 8 : 4) * 32 * 16 + 32 * 16);   // x pieces + chunk constants
    const size_t cap = 227 * 1024;
    bool found = false;
    int64_t best = 0;
    for (int R : {4, 2, 1}) {
        for (int S : {1, 2, 3, 4, 6, 8, 12, 16, 24}) {
            if (kCWarps % S != 0) continue;
            const int BR = (kCWarps / S) * R;
            const uint32_t w_slice = (uint32_t)BR * 512;
            const uint32_t sb_slice = ((uint32_t)BR * sbg * tbytes + 127) / 128 * 128;
            const uint32_t stage = (uint32_t)S * (w_slice + 2 * sb_slice);
            const int64_t nb = (N + BR - 1) / BR;
            const int64_t per_cta = (nb + sms - 1) / sms;
            // pending partial sums: all of a CTA's blocks if they fit in 16 KB
            const int64_t pend_row = (int64_t)kCWarps * R * 4;
            const int flush = (int)std::max<int64_t>(1, std::min<int64_t>(per_cta, (16 * 1024) / pend_row));
            const size_t tail = 2 * kMaxDepth * 8 + (size_t)flush * pend_row + 16 + 128;   // + alignment
            if (fixed + tail + 2 * (size_t)stage > cap) continue;
            const int depth = (int)std::min<size_t>(kMaxDepth, (cap - fixed - tail) / stage);
            const int64_t cost = per_cta * ((n_it + S - 1) / S) * std::max(2, R);
            if (!found || cost < best) {
                found = true;
                best = cost;
                out->R = R;
                out->S = S;
                out->depth = depth;
                out->flush = flush;
                out->n_blocks = nb;
                out->w_slice = w_slice;
                out->sb_slice = sb_slice;
                out->stage_bytes = stage;
                out->smem = fixed + (size_t)depth * stage + tail;
            }
        }
    }
    return found;
}

template <typename T, int R>
cudaError_t launch_t(const CUtensorMap& wm, const CUtensorMap& sm, const CUtensorMap& bm, const Qmv4Args& a,
                     size_t smem, cudaStream_t s) {
    static unsigned long long configured = 0ull;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(configured & (1ull << dev))) {
        cudaError_t e =
            cudaFuncSetAttribute(qmv4_kernel<T, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured |= 1ull << dev;
    }
    const int64_t grid = std::min<int64_t>(a.n_blocks, num_sms());
    return launch_pdl(qmv4_kernel<T, R>, dim3((unsigned)grid), dim3(kThreads), smem, s, wm, sm, bm, a);
}

template <typename T>
cudaError_t launch_r(const CUtensorMap& wm, const CUtensorMap& sm, const CUtensorMap& bm, const Qmv4Args& a,
                     int R, size_t smem, cudaStream_t s) {
    switch (R) {
    case 4: return launch_t<T, 4>(wm, sm, bm, a, smem, s);
    case 2: return launch_t<T, 2>(wm, sm, bm, a, smem, s);
    default: return launch_t<T, 1>(wm, sm, bm, a, smem, s);
    }
}

}  // namespace

int qmv4_supported(const void* scales, const void* biases, int dtype, int bits, int gs, int64_t N, int64_t K) {
    if (bits != 4 || (gs != 32 && gs != 64 && gs != 128)) return 0;
    if (K < kItCols) return 0;   // tensor extents at least one box wide
    // TMA: 16-byte aligned bases and row strides (K / group_size scales per row)
    if ((reinterpret_cast<uintptr_t>(scales) & 15) || (reinterpret_cast<uintptr_t>(biases) & 15)) return 0;
    const int tbytes = dtype == GAI4_F32 ? 4 : 2;
    if (((K / gs) * tbytes) % 16 != 0) return 0;
    if (N > (int64_t)INT32_MAX || K / 8 > (int64_t)INT32_MAX) return 0;   // TMA coordinates are 32-bit
    if (!encode_fn()) return 0;
    Qmv4Plan p;
    return plan_qmv4(N, K, gs, tbytes, &p) ? 1 : 0;
}

cudaError_t launch_qmv4(const uint32_t* w, const void* scales, const void* biases, const void* x, void* out,
                        int dtype, int gs, int64_t N, int64_t K, int* status, long long spin_limit,
                        cudaStream_t s) {
    const int tbytes = dtype == GAI4_F32 ? 4 : 2;
    Qmv4Plan p;
    if (!plan_qmv4(N, K, gs, tbytes, &p)) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int BR = (kCWarps / p.S) * p.R;
    const int sbg = kItCols / gs;
    const int n_it = (int)((K + kItCols - 1) / kItCols);
    const bool box3 = K % kItCols == 0;
    CUtensorMap wm, sm, bm;
    if (box3) {
        // [N][n_it][128 words] and [N][n_it][sbg] views; one box = one stage
        const CUtensorMapDataType dt = tbytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        cuuint64_t wd[3] = {(cuuint64_t)(kItCols / 8), (cuuint64_t)n_it, (cuuint64_t)N};
        cuuint64_t wst[2] = {(cuuint64_t)(kItCols / 2), (cuuint64_t)(K / 2)};
        cuuint32_t wbox[3] = {(cuuint32_t)(kItCols / 8), (cuuint32_t)p.S, (cuuint32_t)BR};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&wm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(w), wd, wst, wbox, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cuuint64_t sd[3] = {(cuuint64_t)sbg, (cuuint64_t)n_it, (cuuint64_t)N};
        cuuint64_t sst[2] = {(cuuint64_t)(sbg * tbytes), (cuuint64_t)((K / gs) * tbytes)};
        cuuint32_t sbox[3] = {(cuuint32_t)sbg, (cuuint32_t)p.S, (cuuint32_t)BR};
        if (enc(&sm, dt, 3, const_cast<void*>(scales), sd, sst, sbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (enc(&bm, dt, 3, const_cast<void*>(biases), sd, sst, sbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
    {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
        cuuint32_t box[2] = {(cuuint32_t)(kItCols / 8), (cuuint32_t)BR};
        cuuint32_t es[2] = {1, 1};
        if (enc(&wm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)(K / gs), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)((K / gs) * tbytes)};
        cuuint32_t box[2] = {(cuuint32_t)sbg, (cuuint32_t)BR};
        cuuint32_t es[2] = {1, 1};
        const CUtensorMapDataType dt = tbytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        if (enc(&sm, dt, 2, const_cast<void*>(scales), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (enc(&bm, dt, 2, const_cast<void*>(biases), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    }
    Qmv4Args a;
    a.x = x;
    a.out = out;
    a.N = N;
    a.K = K;
    int lg = 0;
    while ((1 << lg) < gs) ++lg;
    a.gs_log2 = lg;
    a.S = p.S;
    a.n_it = (int)((K + kItCols - 1) / kItCols);
    a.n_st = (a.n_it + p.S - 1) / p.S;
    a.depth = p.depth;
    a.n_blocks = p.n_blocks;
    a.sbg = sbg;
    a.w_slice = p.w_slice;
    a.sb_slice = p.sb_slice;
    a.stage_bytes = p.stage_bytes;
    a.box3 = box3 ? 1 : 0;
    a.flush = p.flush;
    if (box3) {   // [row][iteration][...]
        a.w_rs = (uint32_t)p.S * 512u;
        a.w_is = 512u;
        a.sb_rs = (uint32_t)(p.S * sbg);
        a.sb_is = (uint32_t)sbg;
    } else {      // [iteration][row][...]
        a.w_rs = 512u;
        a.w_is = p.w_slice;
        a.sb_rs = (uint32_t)sbg;
        a.sb_is = p.sb_slice / (uint32_t)tbytes;
    }
    a.status = status;
    a.spin_limit = spin_limit;
    switch (dtype) {
    case GAI4_F16: return launch_r<F16>(wm, sm, bm, a, p.R, p.smem, s);
    case GAI4_F32: return launch_r<F32>(wm, sm, bm, a, p.R, p.smem, s);
    default: return launch_r<BF16>(wm, sm, bm, a, p.R, p.smem, s);
    }
}

}  // namespace gai4
