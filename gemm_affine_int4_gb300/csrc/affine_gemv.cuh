// affine_gemv.cuh -- CUDA-core affine group-quantized GEMV (qmv, M = 1) and
// register-tiled small-M GEMM (qmm_t, M <= 8 per CTA row of the grid).
//
// Computes out[m, n] = sum_g ( s[n,g] * sum_{k in g} q[n,k] x[m,k]
//                               + b[n,g] * sum_{k in g} x[m,k] )
// (metaltile-std quantized.rs, mt_qmv: the "bias hoist" split of the affine
// dot product; mt_qmm_bm2 / mt_qmm_bm4: one decode of each weight reused for
// several activation rows). Accumulation is binary32.
//
// Work decomposition (sm_103a):
//  * A lane owns a "chunk" of E consecutive K elements of a row (E = 32 for
//    2/3/4-bit codes, 16 for 6/8-bit), i.e. CW = E*bits/32 packed words: one
//    16-byte load for 4 and 8 bits, 8 bytes for 2 bits, three words for 3/6.
//    Consecutive lanes own consecutive chunks, so a warp reads one contiguous
//    span of every row it works on (coalesced 16-byte loads, streamed past L1).
//    E divides every legal group size, so a chunk lies in one group and needs
//    one (scale, bias) pair: bias hoist per chunk.
//  * A warp works on R rows at once, reusing each lane's activation fragment
//    across the R rows; a CTA of NW warps covers (NW/S)*R rows, the S warps of
//    a row group splitting the K iterations round-robin. Partial sums meet in
//    shared memory at the end.
//  * The activations of the CTA's x rows are staged once per K slab in shared
//    memory, permuted so that lane l's 16-byte pieces of its chunk are
//    contiguous across the warp (conflict-free 16-byte shared loads), together
//    with the binary32 sum of every chunk (the sum_{k} x[m,k] of the bias term).
//
// Code -> number without an int->float conversion: a code q placed in the low
// mantissa bits of a constant C gives the number C + q exactly (C = 128 for
// bf16 with q < 128, 1024 for f16, 2^bits for binary32 with q in the top
// mantissa bits). The accumulator then holds sum (C + q) x; the chunk's
// sum_{k} q x is that minus C * sum_k x. For bf16/f16 activations the
// multiply-add is the sm_100 mixed-precision fma.rn.f32.{bf16,f16}: both
// 16-bit operands are exact, the product is exact in binary32, and the sum is
// binary32. Pairs of codes are extracted by one mask (two 16-bit halves of a
// register at once).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace gai4 {

template <int BITS> struct ChunkGeom;
template <> struct ChunkGeom<2> { static constexpr int E = 32, CW = 2; };
template <> struct ChunkGeom<3> { static constexpr int E = 32, CW = 3; };
template <> struct ChunkGeom<4> { static constexpr int E = 32, CW = 4; };
template <> struct ChunkGeom<6> { static constexpr int E = 16, CW = 3; };
template <> struct ChunkGeom<8> { static constexpr int E = 16, CW = 4; };

// load the CW packed words of one chunk (row stride and chunk offsets are
// multiples of the load width for every legal K)
template <int CW>
__device__ __forceinline__ void load_chunk(const uint32_t* p, uint32_t (&w)[CW]) {
    if constexpr (CW == 4) {
        uint4 v = ld_stream_v4(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (CW == 2) {
        uint2 v = ld_stream_v2(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < CW; ++i) w[i] = ld_stream_u32(p + i);
    }
}

// ---------------------------------------------------------------------------
// Decode paths. Each turns a chunk's CW words into NP 32-bit operand registers
// holding the exact codes q_e (decode: a code is first placed under the
// exponent of a constant C, giving C + q exactly, and C is then subtracted,
// also exactly), and adds sum_e q_e x_e into an accumulator (dot). Every
// product q x is exact before it is summed, so codes that are all zero add
// exactly zero. x fragments: 16-bit activations as E/2 registers (pairs,
// natural order), binary32 activations as E registers.
// ---------------------------------------------------------------------------

// (a - b) on 16-bit pairs of type T (exact here: both operands are C + q and C)
template <typename T>
__device__ __forceinline__ uint32_t sub_pair(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (T::kIsBF16)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// kind 0: 16-bit activations, 2/4-bit codes (and 8-bit codes with f16):
// one mask extracts codes e and e + 16/BITS (one per 16-bit half).
template <typename T, int BITS>
struct PathPair16 {
    using G = ChunkGeom<BITS>;
    static constexpr int E = G::E, CW = G::CW;
    static constexpr int EPH = 16 / BITS;          // codes per 16-bit half
    static constexpr int NP = E / 2;
    static constexpr uint32_t kMask = ((1u << BITS) - 1u) * 0x00010001u;
    static constexpr uint32_t kMagic = T::kMagic16 * 0x00010001u;

    __device__ __forceinline__ static void decode(const uint32_t (&w)[CW], uint32_t (&P)[NP]) {
#pragma unroll
        for (int i = 0; i < CW; ++i)
#pragma unroll
            for (int j = 0; j < EPH; ++j)
                P[i * EPH + j] = sub_pair<T>(((w[i] >> (BITS * j)) & kMask) | kMagic, kMagic);
    }
    __device__ __forceinline__ static float dot(const uint32_t (&P)[NP], const uint32_t* xr, float acc) {
#pragma unroll
        for (int i = 0; i < CW; ++i)
#pragma unroll
            for (int j = 0; j < EPH; ++j) {
                const int a = i * (32 / BITS) + j;   // element in the low half
                const int b = a + EPH;               // element in the high half
                if (j % 2 == 0) {
                    acc = fma_mix<T, 0, 0>(P[i * EPH + j], xr[a / 2], acc);
                    acc = fma_mix<T, 1, 0>(P[i * EPH + j], xr[b / 2], acc);
                } else {
                    acc = fma_mix<T, 0, 1>(P[i * EPH + j], xr[a / 2], acc);
                    acc = fma_mix<T, 1, 1>(P[i * EPH + j], xr[b / 2], acc);
                }
            }
        return acc;
    }
};

// kind 1: bf16 activations, 8-bit codes (bf16 holds 128 + q exactly only for
// q < 128): split each code into its low and high nibble planes,
// sum q x = sum lo x + 16 sum hi x (both sums of exact products).
template <typename T>
struct PathBf16Byte {
    using G = ChunkGeom<8>;
    static constexpr int E = G::E, CW = G::CW;
    static constexpr int NP = E;                   // E/2 low-nibble pairs, E/2 high
    static constexpr uint32_t kMask = 0x000F000Fu;
    static constexpr uint32_t kMagic = 0x43004300u;

    __device__ __forceinline__ static void decode(const uint32_t (&w)[CW], uint32_t (&P)[NP]) {
#pragma unroll
        for (int i = 0; i < CW; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                P[i * 2 + j] = sub_pair<T>(((w[i] >> (8 * j)) & kMask) | kMagic, kMagic);              // low
                P[E / 2 + i * 2 + j] = sub_pair<T>(((w[i] >> (8 * j + 4)) & kMask) | kMagic, kMagic);  // high
            }
    }
    __device__ __forceinline__ static float dot(const uint32_t (&P)[NP], const uint32_t* xr, float acc) {
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int i = 0; i < CW; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // pair (i, j) covers elements 4i + j (low half) and 4i + j + 2 (high half)
                const int a = 4 * i + j, b = a + 2;
                if (j == 0) {
                    lo = fma_mix<T, 0, 0>(P[i * 2 + j], xr[a / 2], lo);
                    lo = fma_mix<T, 1, 0>(P[i * 2 + j], xr[b / 2], lo);
                    hi = fma_mix<T, 0, 0>(P[E / 2 + i * 2 + j], xr[a / 2], hi);
                    hi = fma_mix<T, 1, 0>(P[E / 2 + i * 2 + j], xr[b / 2], hi);
                } else {
                    lo = fma_mix<T, 0, 1>(P[i * 2 + j], xr[a / 2], lo);
                    lo = fma_mix<T, 1, 1>(P[i * 2 + j], xr[b / 2], lo);
                    hi = fma_mix<T, 0, 1>(P[E / 2 + i * 2 + j], xr[a / 2], hi);
                    hi = fma_mix<T, 1, 1>(P[E / 2 + i * 2 + j], xr[b / 2], hi);
                }
            }
        return acc + fmaf(16.0f, hi, lo);
    }
};

// extract code e (bit offset e*BITS in the chunk's word stream) aligned so that
// its lowest bit lands at bit `dst` of the result (other bits unspecified)
template <int BITS, int CW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[CW], int e, int dst) {
    const int o = e * BITS, i = o / 32, sh = o % 32;
    if (sh + BITS <= 32) {
        const int d = dst - sh;
        return d >= 0 ? (w[i] << d) : (w[i] >> (-d));
    }
    // straddles words i and i+1: funnel shift of the 64-bit pair
    return __funnelshift_r(w[i], w[i + 1], sh - dst);
}

// kind 2: 16-bit activations, 3/6-bit codes: one code per register (low half)
template <typename T, int BITS>
struct PathSingle16 {
    using G = ChunkGeom<BITS>;
    static constexpr int E = G::E, CW = G::CW;
    static constexpr int NP = E;
    static constexpr uint32_t kMask = (1u << BITS) - 1u;

    __device__ __forceinline__ static void decode(const uint32_t (&w)[CW], uint32_t (&P)[NP]) {
#pragma unroll
        for (int e = 0; e < E; ++e) P[e] = sub_pair<T>((code_at<BITS, CW>(w, e, 0) & kMask) | T::kMagic16, T::kMagic16);
    }
    __device__ __forceinline__ static float dot(const uint32_t (&P)[NP], const uint32_t* xr, float acc) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (e % 2 == 0) acc = fma_mix<T, 0, 0>(P[e], xr[e / 2], acc);
            else            acc = fma_mix<T, 0, 1>(P[e], xr[e / 2], acc);
        }
        return acc;
    }
};

// kind 3: binary32 activations, any width: the code goes into the top BITS
// mantissa bits of 2^BITS, giving the float 2^BITS + q exactly; subtracting
// 2^BITS gives q exactly.
template <int BITS>
struct PathF32 {
    using G = ChunkGeom<BITS>;
    static constexpr int E = G::E, CW = G::CW;
    static constexpr int NP = E;
    static constexpr int kDst = 23 - BITS;
    static constexpr uint32_t kMask = ((1u << BITS) - 1u) << kDst;
    static constexpr uint32_t kExp = (uint32_t)(127 + BITS) << 23;

    __device__ __forceinline__ static void decode(const uint32_t (&w)[CW], uint32_t (&P)[NP]) {
#pragma unroll
        for (int e = 0; e < E; ++e)
            P[e] = __float_as_uint(__uint_as_float((code_at<BITS, CW>(w, e, kDst) & kMask) | kExp) -
                                   (float)(1 << BITS));
    }
    __device__ __forceinline__ static float dot(const uint32_t (&P)[NP], const uint32_t* xr, float acc) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(__uint_as_float(P[e]), __uint_as_float(xr[e]), acc);
        return acc;
    }
};

template <typename T, int BITS>
struct PathFor {
    using type = PathPair16<T, BITS>;
};
template <typename T> struct PathFor<T, 3> { using type = PathSingle16<T, 3>; };
template <typename T> struct PathFor<T, 6> { using type = PathSingle16<T, 6>; };
template <> struct PathFor<BF16, 8> { using type = PathBf16Byte<BF16>; };
template <int BITS> struct PathFor<F32, BITS> { using type = PathF32<BITS>; };
template <> struct PathFor<F32, 3> { using type = PathF32<3>; };
template <> struct PathFor<F32, 6> { using type = PathF32<6>; };

struct AffineKernelArgs {
    const uint32_t* w;
    const void* scales;
    const void* biases;
    const void* x;
    void* out;
    int64_t M, N, K;
    int64_t wpr;      // packed words per row
    int64_t groups;   // K / group_size
    int gs_shift;     // log2(group_size / E)
    int S;            // warps of a row group (K split inside the CTA)
    int KS;           // K slab length staged in shared memory
    int KSP;          // KS rounded up to whole warp iterations (32 chunks): staged layout size
};

template <typename T, int BITS, int R, int MB, int NW>
__global__ void __launch_bounds__(NW * 32) affine_gemv_kernel(const AffineKernelArgs a) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    using Path = typename PathFor<T, BITS>::type;
    using St = typename T::storage;
    constexpr int E = Path::E, CW = Path::CW, NP = Path::NP;
    constexpr int EPP = 16 / T::kBytes;       // activation elements per 16-byte piece
    constexpr int PPC = E / EPP;              // pieces per chunk
    constexpr int XR = E * T::kBytes / 4;     // 32-bit registers of one x fragment

    extern __shared__ uint4 smem[];
    const int S = a.S, KS = a.KS, KSP = a.KSP;
    const int Gw = NW / S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp / S, s = warp % S;
    const int64_t row0 = (int64_t)blockIdx.x * (Gw * R) + (int64_t)g * R;
    const int64_t m0 = (int64_t)blockIdx.y * MB;
    const int64_t M = a.M, N = a.N, K = a.K;

    // staged layout: per x row, whole warp iterations of 32 chunks x PPC pieces
    const int pieces_per_m = KSP / EPP;
    const int chunks_per_m = KSP / E;
    uint4* x_sm = smem;
    float* xsum_sm = reinterpret_cast<float*>(smem + MB * pieces_per_m);
    float* red_sm = xsum_sm + MB * chunks_per_m;

    const St* xg = static_cast<const St*>(a.x);
    const St* sg = static_cast<const St*>(a.scales);
    const St* bg = static_cast<const St*>(a.biases);

    float part[R][MB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) part[r][m] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += KS) {
        const int kslab = (int)min((int64_t)KS, K - k0);
        const int nch = kslab / E;
        const int npieces = kslab / EPP;
        __syncthreads();
        for (int idx = threadIdx.x; idx < MB * npieces; idx += NW * 32) {
            const int m = idx / npieces, p = idx - m * npieces;
            const int c = p / PPC, j = p - c * PPC;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m0 + m < M) v = *reinterpret_cast<const uint4*>(xg + (m0 + m) * K + k0 + (int64_t)p * EPP);
            x_sm[m * pieces_per_m + ((c >> 5) * PPC + j) * 32 + (c & 31)] = v;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < MB * nch; idx += NW * 32) {
            const int m = idx / nch, c = idx - m * nch;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < PPC; ++j) {
                const uint4 v = x_sm[m * pieces_per_m + ((c >> 5) * PPC + j) * 32 + (c & 31)];
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    if constexpr (T::kBytes == 2) {
                        sum += T::to_f32((uint16_t)(u[t] & 0xffffu));
                        sum += T::to_f32((uint16_t)(u[t] >> 16));
                    } else {
                        sum += __uint_as_float(u[t]);
                    }
                }
            }
            xsum_sm[m * chunks_per_m + c] = sum;
        }
        __syncthreads();

        const int its = (nch + 31) >> 5;
        const int64_t gc0 = k0 / E;   // first chunk index of the slab within a row

        uint32_t wn[R][CW];
        float sn[R], bn[R];
        auto load_it = [&](int it) {
            const int c = it * 32 + lane;
            const bool valid = c < nch;
            const int64_t gc = gc0 + c;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (valid && row < N) {
                    load_chunk<CW>(a.w + row * a.wpr + gc * CW, wn[r]);
                    const int64_t gi = row * a.groups + (gc >> a.gs_shift);
                    sn[r] = T::to_f32(sg[gi]);
                    bn[r] = T::to_f32(bg[gi]);
                } else {
#pragma unroll
                    for (int i = 0; i < CW; ++i) wn[r][i] = 0u;
                    sn[r] = 0.f;
                    bn[r] = 0.f;
                }
            }
        };

        if (s < its) load_it(s);
        for (int it = s; it < its; it += S) {
            uint32_t wc[R][CW];
            float sc[R], bc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int i = 0; i < CW; ++i) wc[r][i] = wn[r][i];
                sc[r] = sn[r];
                bc[r] = bn[r];
            }
            if (it + S < its) load_it(it + S);
            const int c = it * 32 + lane;
            if (c < nch) {
                uint32_t P[R][NP];
#pragma unroll
                for (int r = 0; r < R; ++r) Path::decode(wc[r], P[r]);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    uint32_t xr[XR];
#pragma unroll
                    for (int j = 0; j < PPC; ++j) {
                        const uint4 v = x_sm[m * pieces_per_m + (it * PPC + j) * 32 + lane];
                        xr[4 * j + 0] = v.x;
                        xr[4 * j + 1] = v.y;
                        xr[4 * j + 2] = v.z;
                        xr[4 * j + 3] = v.w;
                    }
                    const float xs = xsum_sm[m * chunks_per_m + c];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float qx = Path::dot(P[r], xr, 0.f);      // sum q x of the chunk
                        part[r][m] = fmaf(sc[r], qx, fmaf(bc[r], xs, part[r][m]));
                    }
                }
            }
        }
    }

    // reduce the lanes, then the S warps of each row group
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const float v = warp_sum(part[r][m]);
            if (lane == 0) red_sm[(warp * R + r) * MB + m] = v;
        }
    __syncthreads();
    for (int t = threadIdx.x; t < Gw * R * MB; t += NW * 32) {
        const int gg = t / (R * MB), rem = t - gg * (R * MB);
        const int r = rem / MB, m = rem - r * MB;
        float v = 0.f;
        for (int ss = 0; ss < S; ++ss) v += red_sm[((gg * S + ss) * R + r) * MB + m];
        const int64_t row = (int64_t)blockIdx.x * (Gw * R) + (int64_t)gg * R + r;
        if (row < N && m0 + m < M) static_cast<St*>(a.out)[(m0 + m) * N + row] = T::from_f32(v);
    }
}

// ---------------------------------------------------------------------------
// host side: pick the slab, set the shared-memory limit once, launch
// ---------------------------------------------------------------------------
template <typename T, int BITS, int R, int MB, int NW>
cudaError_t launch_affine_gemv_t(const AffineGemvLaunch& L, cudaStream_t stream) {
    constexpr int E = ChunkGeom<BITS>::E;
    constexpr int kXBudget = 64 * 1024;   // bytes of staged activations per CTA
    int64_t ks_max = kXBudget / (MB * T::kBytes);
    ks_max -= ks_max % (32 * E);
    const int KS = (int)(L.K <= ks_max ? L.K : ks_max);
    const int KSP = (KS + 32 * E - 1) / (32 * E) * (32 * E);
    const size_t smem = (size_t)MB * KSP * T::kBytes + (size_t)MB * (KSP / E) * 4 + (size_t)NW * R * MB * 4;
    // the shared-memory limit is a per-function, per-device attribute
    static unsigned long long configured = 0ull;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(configured & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(affine_gemv_kernel<T, BITS, R, MB, NW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured |= 1ull << dev;
    }
    AffineKernelArgs a;
    a.w = L.w;
    a.scales = L.scales;
    a.biases = L.biases;
    a.x = L.x;
    a.out = L.out;
    a.M = L.M;
    a.N = L.N;
    a.K = L.K;
    a.wpr = L.K * BITS / 32;
    a.groups = L.K / L.group_size;
    int sh = 0;
    while ((E << sh) < L.group_size) ++sh;
    a.gs_shift = sh;
    a.S = L.ksplit;
    a.KS = KS;
    a.KSP = KSP;
    const int rows_per_cta = (NW / L.ksplit) * R;
    dim3 grid((unsigned)((L.N + rows_per_cta - 1) / rows_per_cta), (unsigned)((L.M + MB - 1) / MB));
    return launch_pdl(affine_gemv_kernel<T, BITS, R, MB, NW>, grid, dim3(NW * 32), smem, stream, a);
}

// dispatch over (rows per warp, x rows per CTA) for one (T, BITS)
template <typename T, int BITS>
cudaError_t launch_affine_gemv_bits(const AffineGemvLaunch& L, cudaStream_t s) {
    constexpr int NW = 8;
    switch (L.mb) {
    case 1: return L.rows_per_warp == 2 ? launch_affine_gemv_t<T, BITS, 2, 1, NW>(L, s)
                                        : launch_affine_gemv_t<T, BITS, 4, 1, NW>(L, s);
    case 2: return launch_affine_gemv_t<T, BITS, 2, 2, NW>(L, s);
    case 4: return launch_affine_gemv_t<T, BITS, 2, 4, NW>(L, s);
    default: return launch_affine_gemv_t<T, BITS, 1, 8, NW>(L, s);
    }
}

template <typename T>
cudaError_t launch_affine_gemv_dtype(const AffineGemvLaunch& L, cudaStream_t s) {
    switch (L.bits) {
    case 2: return launch_affine_gemv_bits<T, 2>(L, s);
    case 3: return launch_affine_gemv_bits<T, 3>(L, s);
    case 4: return launch_affine_gemv_bits<T, 4>(L, s);
    case 6: return launch_affine_gemv_bits<T, 6>(L, s);
    default: return launch_affine_gemv_bits<T, 8>(L, s);
    }
}

}  // namespace gai4
