// qmm_tc.cu -- tensor-core qmm_t (sm_103a: TMA, mbarrier, tcgen05 / TMEM) and
// the split-K reduce.
//
// out[m, n] = sum_k x[m, k] * w_hat[n, k], w_hat = s * q + b (MLX PR "[Metal]
// Add staged affine_qmm_t_nax kernels with split-k": transposed affine
// quantized_matmul, split-K with fp32 partials and a separate accumulate
// kernel; metaltile-std quantized.rs, mt_qmm_mma: dequantize the weight tile
// once, then run the matrix unit on it).
//
// Mapping ("swap AB"): the 128 rows of a weight tile are the MMA M dimension,
// the x rows (tokens, padded to a multiple of 16) are the MMA N dimension, so a
// few tokens still make a legal tcgen05 shape and the accumulator
// D[128 x Mt] (fp32) lives in tensor memory.
//
// One CTA = one 128-row weight tile x one K range (split) x one chunk of at
// most 256 x rows, one CTA per SM. The K range is walked in 256-column weight
// stages, each split into two 128-column A stages (= activation stages).
// Warp roles:
//   warp 0      TMA producer of the packed-weight stages (ring of even depth)
//   warp 1      TMA producer of the activation stages, 128-byte swizzled =
//               the canonical K-major UMMA layout
//   warps 2-3   MMA issuers: tcgen05.mma kind::f16, A operand from tensor
//               memory, B operand (activations) from shared memory. The whole
//               warp runs the issue loop (warp-uniform control flow) and
//               elect.sync picks the lane that issues: a converged warp issues
//               MMAs about twice as fast as one divergent lane. Issuer j takes
//               the A stages i == j (mod 2) into its own accumulator; the
//               epilogue adds the two accumulators in a fixed order.
//   warps 4-19  dequantize, as four groups of four warps (one warp per
//               tensor-memory lane quadrant). Group g takes the A stages
//               i == g (mod 4): thread t of the group's warp in quadrant q owns
//               weight row 32q + t and decodes its 128 columns of the stage
//               (one half of a weight stage), computes w_hat = fma(q, s, b) in
//               bf16x2/f16x2 (one rounding of the exact value) and stores the
//               row slice straight into tensor memory with tcgen05.st (the A
//               ring of 64-column slots), so the weights never pass through
//               shared memory a second time. The groups run on different
//               stages, so they do not meet on one barrier per stage.
//               After the K loop the same warps read the accumulator
//               (tcgen05.ld) and write fp32 partials or the rounded output.
// Every ring slot is always waited on by the same role, phase after phase
// (mbarrier.try_wait.parity reports a phase two ahead as complete); the host
// sizes the rings for that (even depths, at least four A slots).
// Scales and biases of a stage arrive by TMA with its packed weights (same
// barrier) when the row length K / group_size is a multiple of 8; otherwise
// the dequantize warps read them from global memory. Keeping global loads out
// of the dequantize warps matters: every mbarrier arrive (a release) waits
// for all of the thread's outstanding loads.
// Every wait on an mbarrier is bounded; on time-out the kernel records
// GAI4_ERR_TIMEOUT in the device status word, lets the other roles drain, frees
// its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace gai4 {

// ---------------------------------------------------------------------------
// split-K reduce: out[m, n] = T(sum_{s < S} P[s, m, n]), summed in s order and
// rounded once (MLX PR, Correctness: fp32 partials, one rounding after the sum)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void splitk_reduce_kernel(const float* __restrict__ P, typename T::storage* __restrict__ out, int64_t M,
                                     int64_t N, SplitPlan plan) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t MN = M * N;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= MN) return;
    const int64_t n = i % N;
    const int tile = (int)(n / 128);
    const int s_t = plan.s_base + (tile < plan.n_extra ? 1 : 0);
    float acc = P[i];
    for (int s = 1; s < s_t; ++s) acc += P[(int64_t)s * MN + i];
    out[i] = T::from_f32(acc);
}

// 8 consecutive outputs of one row per thread (N % 8 == 0, 16-byte aligned
// partials and output): two 16-byte loads per partial slot, one store
template <typename T>
__global__ void splitk_reduce8_kernel(const float* __restrict__ P, typename T::storage* __restrict__ out, int64_t M,
                                      int64_t N, SplitPlan plan) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t MN = M * N;
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // chunk of 8 outputs
    if (c >= MN / 8) return;
    const int64_t i = c * 8;
    const int64_t n = i % N;
    const int tile = (int)(n / 128);   // 8 | 128: the chunk lies in one tile
    const int s_t = plan.s_base + (tile < plan.n_extra ? 1 : 0);
    float4 a = __ldcs(reinterpret_cast<const float4*>(P + i));
    float4 b = __ldcs(reinterpret_cast<const float4*>(P + i + 4));
    for (int s = 1; s < s_t; ++s) {
        const float4 u = __ldcs(reinterpret_cast<const float4*>(P + (int64_t)s * MN + i));
        const float4 v = __ldcs(reinterpret_cast<const float4*>(P + (int64_t)s * MN + i + 4));
        a.x += u.x; a.y += u.y; a.z += u.z; a.w += u.w;
        b.x += v.x; b.y += v.y; b.z += v.z; b.w += v.w;
    }
    if constexpr (sizeof(typename T::storage) == 4) {
        reinterpret_cast<float4*>(out + i)[0] = a;
        reinterpret_cast<float4*>(out + i)[1] = b;
    } else {
        uint4 o;
        o.x = (uint32_t)T::from_f32(a.x) | ((uint32_t)T::from_f32(a.y) << 16);
        o.y = (uint32_t)T::from_f32(a.z) | ((uint32_t)T::from_f32(a.w) << 16);
        o.z = (uint32_t)T::from_f32(b.x) | ((uint32_t)T::from_f32(b.y) << 16);
        o.w = (uint32_t)T::from_f32(b.z) | ((uint32_t)T::from_f32(b.w) << 16);
        *reinterpret_cast<uint4*>(out + i) = o;
    }
}

template <typename T>
static cudaError_t reduce_launch(const float* partials, void* out, int64_t M, int64_t N, const SplitPlan& plan,
                                 cudaStream_t s) {
    auto* o = static_cast<typename T::storage*>(out);
    const int64_t MN = M * N;
    const bool vec = N % 8 == 0 && (reinterpret_cast<uintptr_t>(partials) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    if (vec) {
        const unsigned blocks = (unsigned)((MN / 8 + 255) / 256);
        return launch_pdl(splitk_reduce8_kernel<T>, dim3(blocks), dim3(256), 0, s, partials, o, M, N, plan);
    }
    const unsigned blocks = (unsigned)((MN + 255) / 256);
    return launch_pdl(splitk_reduce_kernel<T>, dim3(blocks), dim3(256), 0, s, partials, o, M, N, plan);
}

cudaError_t launch_splitk_reduce(const float* partials, void* out, int64_t M, int64_t N, const SplitPlan& plan,
                                 int dtype, cudaStream_t s) {
    switch (dtype) {
    case GAI4_F16: return reduce_launch<F16>(partials, out, M, N, plan, s);
    case GAI4_F32: return reduce_launch<F32>(partials, out, M, N, plan, s);
    default: return reduce_launch<BF16>(partials, out, M, N, plan, s);
    }
}

// ---------------------------------------------------------------------------
// K-split planning (MLX PR: at most 4 pieces of >= 256 columns, K < 512 not
// split). Pieces of one tile may differ in length by one unit, so that the
// number of CTAs can match the number of SMs instead of spilling into a
// second, mostly idle wave.
// ---------------------------------------------------------------------------
int max_pieces(int64_t K, int unit) {
    if (K < 512) return 1;
    const int64_t KU = K / unit;
    int best = 1;
    for (int S = 2; S <= 4; ++S)
        if ((KU / S) * unit >= 256) best = S;
    return best;
}

bool uniform_plan(int64_t N, int64_t K, int gs, int S, SplitPlan* out) {
    SplitPlan p;
    p.tiles = (int)((N + 127) / 128);
    p.unit = gs > 64 ? gs : 64;
    p.n_extra = 0;
    p.s_base = S;
    if (S < 1 || S > 4 || K % p.unit != 0) return false;
    if (S > 1 && (K < 512 || K % ((int64_t)S * p.unit) != 0 || K / S < 256)) return false;
    *out = p;
    return true;
}

SplitPlan auto_plan(int64_t M, int64_t N, int64_t K, int gs, int max_slots, int64_t batch) {
    SplitPlan p;
    p.tiles = (int)((N + 127) / 128);
    // 256-column cuts when K allows: every stage of the tensor-core kernel then
    // starts on a 256-column boundary, so a stage's groups lie in one aligned
    // 8-group box of scales / biases
    p.unit = (K % 256 == 0 && gs <= 256) ? 256 : (gs > 64 ? gs : 64);
    p.s_base = 1;
    p.n_extra = 0;
    const int cap = std::min(max_pieces(K, p.unit), std::max(1, max_slots));
    const int64_t mchunks = (M + 255) / 256;
    const int64_t avail = std::max<int64_t>(1, num_sms() / (mchunks * batch));   // CTAs per M chunk and batch in one wave
    const int64_t KU = K / p.unit;
    const int64_t T = p.tiles;
    // candidate 1: uniform S in waves
    int64_t best_cost = -1;
    for (int S = 1; S <= cap; ++S) {
        const int64_t waves = (T * S + avail - 1) / avail;
        const int64_t cost = waves * ((KU + S - 1) / S);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            p.s_base = S;
            p.n_extra = 0;
        }
    }
    // candidate 2: one wave with s_base or s_base + 1 pieces per tile
    if (T <= avail) {
        const int sb = (int)std::min<int64_t>(cap, avail / T);
        const int ne = sb < cap ? (int)std::min<int64_t>(T, avail - T * sb) : 0;
        const int64_t cost = (KU + sb - 1) / sb;
        if (cost < best_cost) {
            best_cost = cost;
            p.s_base = sb;
            p.n_extra = ne;
        }
    }
    // Large M: when 128-row M chunks fill at most one wave unsplit, they beat
    // 256-row chunks whose K splits write M x N fp32 partials per piece and
    // need the reduce (measured at 4096^2, M = 512: 19.2 against 22.3 us). With
    // more than one wave the larger chunks' fewer MMA instructions win.
    if (M > 256 && T * ((M + 127) / 128) * batch <= num_sms()) {
        p.s_base = 1;
        p.n_extra = 0;
        p.mcap = 128;
    }
    return p;
}

// ---------------------------------------------------------------------------
// tensor-core kernel
// ---------------------------------------------------------------------------
namespace tc {

using namespace pipe;

constexpr int kTileN = 128;      // weight rows per CTA (MMA M)
constexpr int kBK = 256;         // K columns per weight stage
constexpr int kAK = 128;         // K columns per A stage = per activation stage
constexpr int kXBK = kAK;        // (two 64-column swizzle atoms)
constexpr uint32_t kAStageCols = kAK / 2;   // tensor-memory columns of one A stage (bf16 pairs)
constexpr int kMaxWStages = 12;  // packed-weight ring (runtime depth <= this, even)
constexpr int kMaxAStages = 8;   // tensor-memory A ring (runtime depth 4..8)
constexpr int kMaxXStages = 8;   // activation ring (runtime depth <= this)
constexpr int kMaxMt = 256;      // x rows per CTA (MMA N <= 256)
constexpr int kTmemCols = 512;   // one CTA per SM owns all of tensor memory
constexpr int kMaxIssuers = 2;   // MMA issuer warps (2 and 3), one accumulator each
constexpr int kDequantWarps = 16;   // 4 groups of 4 (one warp per tensor-memory lane quadrant)
constexpr int kDequantWarp0 = 4;
constexpr int kThreads = 32 * (kDequantWarp0 + kDequantWarps);
constexpr uint32_t kSbBox = 8 * kTileN * 2;    // one TMA box of scales or biases: 8 groups x 128 rows, u16

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major, 128-byte swizzled shared-memory operand descriptor (sm_100 UMMA):
// start address >> 4, leading byte offset (unused for this layout) = 1,
// stride byte offset = 1024 (8 rows x 128 B), descriptor version 1, layout
// SWIZZLE_128B (2).
// Low word: start address and leading byte offset; high word: stride byte
// offset, version and layout (the same for every operand of this kernel).
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr) { return ((saddr >> 4) & 0x3FFFu) | (1u << 16); }
constexpr uint32_t kSw128DescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));

// instruction descriptor, kind::f16: fp32 accumulate, A/B bf16 (1) or f16 (0),
// both K-major, N = mt, M = 128
__host__ __device__ constexpr uint32_t make_idesc(int is_bf16, int mt) {
    return (1u << 4) | ((uint32_t)is_bf16 << 7) | ((uint32_t)is_bf16 << 10) | ((uint32_t)(mt >> 3) << 17) |
           ((uint32_t)(kTileN >> 4) << 24);
}

// the same two operations executed by a converged warp: one elected lane
// issues; the activation descriptor is given by its low word (the high word is
// kSw128DescHi)
__device__ __forceinline__ void mma_f16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_desc_lo,
                                                    uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p, e;\n .reg .b32 r;\n .reg .b64 d;\n elect.sync r|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
        " mov.b64 d, {%2, %5};\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], d, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_desc_lo), "r"(idesc), "r"(accumulate), "r"(kSw128DescHi)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// loads addressed in the shared state space (32-bit addresses); volatile with a
// memory clobber so that they stay after the mbarrier wait that publishes the data
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
    return (uint32_t)v;
}

// packed 16-bit pair arithmetic (one rounding per result)
template <bool BF>
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (BF)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
template <bool BF>
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    if constexpr (BF)
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    else
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct Params {
    const uint16_t* scales;
    const uint16_t* biases;
    void* out;            // [M, N] T (one piece per tile)
    float* partials;      // [slots, M, N] fp32 (several pieces)
    int64_t M, N, K;
    int64_t groups;       // K / group_size
    int gs_log2;          // log2(group_size)
    SplitPlan plan;
    int mt;               // MMA N: x rows of this CTA rounded up to 16 (<= 256)
    int x_stages;
    int w_stages;
    int a_stages;
    int n_issuers;        // MMA issuer warps = accumulators (1 or 2)
    int sb_boxes;         // 8-group boxes per stage and tensor reserved in shared memory (1 or 2)
    int mchunk;           // x rows per M chunk (blockIdx.z)
    int64_t w_rows_b;     // weight / scale rows between batches (N stacked, 0 shared); batch = blockIdx.y
    uint32_t nib_mask;    // code mask in both halves (0x000F000F for 4-bit codes)
    uint32_t magic;       // bit pattern of C (128 for bf16, 1024 for f16) in both halves
    int* status;
    long long spin_limit;
};

// piece blockIdx.x of the plan -> tile, piece index, K range
__device__ __forceinline__ void piece_of(const SplitPlan& pl, int64_t K, int p, int& tile, int& j, int& s_t,
                                         int64_t& k0, int64_t& k1) {
    const int big = pl.n_extra * (pl.s_base + 1);
    if (p < big) {
        tile = p / (pl.s_base + 1);
        j = p - tile * (pl.s_base + 1);
        s_t = pl.s_base + 1;
    } else {
        const int q = p - big;
        tile = pl.n_extra + q / pl.s_base;
        j = q - (tile - pl.n_extra) * pl.s_base;
        s_t = pl.s_base;
    }
    const int64_t KU = K / pl.unit;
    k0 = (j * KU / s_t) * pl.unit;
    k1 = ((j + 1) * KU / s_t) * pl.unit;
}

// ---------------------------------------------------------------------------
// 4-bit codes: one 32-bit word (8 codes, low nibble first) -> 4 registers of
// w_hat pairs (k, k+1) in 16-bit format T.
// ---------------------------------------------------------------------------
// (a & b) | c as one three-input logic instruction (b, c in registers: a
// logic op takes at most one immediate operand)
__device__ __forceinline__ uint32_t lop3_andor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// nib_mask = 0x000F000F and magic = C in both halves, passed in registers
template <bool BF>
__device__ __forceinline__ void dequant_word4(uint32_t w, uint32_t s2, uint32_t b2, uint32_t nib_mask,
                                              uint32_t magic, uint32_t* o) {
    constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;   // 128.0 / 1024.0 in both halves
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t p = lop3_andor(w >> (4 * j), nib_mask, magic);  // (C + q_j, C + q_{j+4})
        const uint32_t q = hsub2<BF>(p, kMagic);                       // (q_j, q_{j+4}) exact
        r[j] = hfma2<BF>(q, s2, b2);                                   // (w_j, w_{j+4})
    }
    o[0] = __byte_perm(r[0], r[1], 0x5410);   // (w0, w1)
    o[1] = __byte_perm(r[2], r[3], 0x5410);   // (w2, w3)
    o[2] = __byte_perm(r[0], r[1], 0x7632);   // (w4, w5)
    o[3] = __byte_perm(r[2], r[3], 0x7632);   // (w6, w7)
}

template <bool BF>
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (BF)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bits [P, P + 32) of the 96-bit little-endian value (u0, u1, u2), P a
// compile-time constant below 96
template <int P>
__device__ __forceinline__ uint32_t win96(uint32_t u0, uint32_t u1, uint32_t u2) {
    if constexpr (P == 0) return u0;
    else if constexpr (P < 32) return __funnelshift_r(u0, u1, P);
    else if constexpr (P == 32) return u1;
    else if constexpr (P < 64) return __funnelshift_r(u1, u2, P - 32);
    else if constexpr (P == 64) return u2;
    else return u2 >> (P - 64);
}

// eight w_hat pairs (j, j + H) -> the eight pairs (k, k + 1) of 2H codes
template <int H>
__device__ __forceinline__ void pairs_from_halves(const uint32_t* r, uint32_t* o) {
#pragma unroll
    for (int i = 0; i < H / 2; ++i) {
        o[i] = __byte_perm(r[2 * i], r[2 * i + 1], 0x5410);           // codes 2i, 2i + 1
        o[H / 2 + i] = __byte_perm(r[2 * i], r[2 * i + 1], 0x7632);   // codes H + 2i, H + 2i + 1
    }
}

// 2-bit codes: one word (code j at bits 2j) -> 8 pairs (k, k + 1)
template <bool BF>
__device__ __forceinline__ void dequant16_b2(uint32_t w, uint32_t s2, uint32_t b2, uint32_t mask, uint32_t magic,
                                             uint32_t* o) {
    constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;
    uint32_t r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t p = lop3_andor(w >> (2 * j), mask, magic);   // (C + q_j, C + q_{j+8})
        r[j] = hfma2<BF>(hsub2<BF>(p, kMagic), s2, b2);
    }
    pairs_from_halves<8>(r, o);
}

// 6-bit codes: 96 bits (code j at bits 6j) -> 8 pairs (k, k + 1)
template <bool BF, int J = 0>
__device__ __forceinline__ void b6_pair(uint32_t u0, uint32_t u1, uint32_t u2, uint32_t s2, uint32_t b2,
                                        uint32_t mask, uint32_t magic, uint32_t* r) {
    if constexpr (J < 8) {
        constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;
        // code J at bits 0..5 of the first window, code J + 8 at bits 16..21 of the second
        const uint32_t a = win96<6 * J>(u0, u1, u2), b = win96<6 * J + 32>(u0, u1, u2);
        const uint32_t p = lop3_andor(__byte_perm(a, b, 0x7610), mask, magic);
        r[J] = hfma2<BF>(hsub2<BF>(p, kMagic), s2, b2);
        b6_pair<BF, J + 1>(u0, u1, u2, s2, b2, mask, magic, r);
    }
}
template <bool BF>
__device__ __forceinline__ void dequant16_b6(uint32_t u0, uint32_t u1, uint32_t u2, uint32_t s2, uint32_t b2,
                                             uint32_t mask, uint32_t magic, uint32_t* o) {
    uint32_t r[8];
    b6_pair<BF>(u0, u1, u2, s2, b2, mask, magic, r);
    pairs_from_halves<8>(r, o);
}

// 3-bit codes: 96 bits (code j at bits 3j) -> 16 pairs (k, k + 1)
template <bool BF, int J = 0>
__device__ __forceinline__ void b3_pair(uint32_t u0, uint32_t u1, uint32_t u2, uint32_t s2, uint32_t b2,
                                        uint32_t mask, uint32_t magic, uint32_t* r) {
    if constexpr (J < 16) {
        constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;
        // code J at bits 0..2 of the first window, code J + 16 at bits 16..18 of the second
        const uint32_t a = win96<3 * J>(u0, u1, u2), b = win96<3 * J + 32>(u0, u1, u2);
        const uint32_t p = lop3_andor(__byte_perm(a, b, 0x7610), mask, magic);
        r[J] = hfma2<BF>(hsub2<BF>(p, kMagic), s2, b2);
        b3_pair<BF, J + 1>(u0, u1, u2, s2, b2, mask, magic, r);
    }
}
template <bool BF>
__device__ __forceinline__ void dequant32_b3(uint32_t u0, uint32_t u1, uint32_t u2, uint32_t s2, uint32_t b2,
                                             uint32_t mask, uint32_t magic, uint32_t (&o0)[8], uint32_t (&o1)[8]) {
    uint32_t r[16];
    b3_pair<BF>(u0, u1, u2, s2, b2, mask, magic, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o0[i] = __byte_perm(r[2 * i], r[2 * i + 1], 0x5410);   // codes 2i, 2i + 1
        o1[i] = __byte_perm(r[2 * i], r[2 * i + 1], 0x7632);   // codes 16 + 2i, 17 + 2i
    }
}

// 8-bit codes: 4 words (16 codes) -> 8 pairs (k, k + 1). A byte placed in the
// low bits of a 16-bit half is that byte times the smallest subnormal (the
// exponent field is 0 or 1); two exact power-of-two products (k1 * k2 =
// 2^133 for bf16, 2^24 for f16) make it the code.
template <bool BF>
__device__ __forceinline__ void dequant16_b8(const uint32_t* u, uint32_t s2, uint32_t b2, uint32_t k1, uint32_t k2,
                                             uint32_t* o) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t lo = __byte_perm(u[m], 0u, 0x4140), hi = __byte_perm(u[m], 0u, 0x4342);
        o[2 * m] = hfma2<BF>(hmul2<BF>(hmul2<BF>(lo, k1), k2), s2, b2);
        o[2 * m + 1] = hfma2<BF>(hmul2<BF>(hmul2<BF>(hi, k1), k2), s2, b2);
    }
}

// bf16, 4-bit codes, scale s with exponent field 1..121: the codes masked
// straight into bf16 subnormals, (q_j, q_{j+4}) * 2^-133 (bits 0..3 of the
// halves) or (q_j, q_{j+4}) * 2^-129 (bits 4..7), times s * 2^133 resp.
// s * 2^129 (exact, exponent-field adds) plus b: the fma sees the same exact
// s * q + b as the offset form and rounds it the same way. 1 shift, 4 ANDs,
// 4 fmas and 4 permutes per word.
__device__ __forceinline__ void dequant_word4_sub(uint32_t w, uint32_t s133, uint32_t s129, uint32_t b2, uint32_t* o) {
    const uint32_t w8 = w >> 8;
    const uint32_t r0 = hfma2<true>(w & 0x000F000Fu, s133, b2);    // (w0, w4)
    const uint32_t r1 = hfma2<true>(w & 0x00F000F0u, s129, b2);    // (w1, w5)
    const uint32_t r2 = hfma2<true>(w8 & 0x000F000Fu, s133, b2);   // (w2, w6)
    const uint32_t r3 = hfma2<true>(w8 & 0x00F000F0u, s129, b2);   // (w3, w7)
    o[0] = __byte_perm(r0, r1, 0x5410);
    o[1] = __byte_perm(r2, r3, 0x5410);
    o[2] = __byte_perm(r0, r1, 0x7632);
    o[3] = __byte_perm(r2, r3, 0x7632);
}

// stage i's groups [g_first, g_last] lie in one or two 8-group TMA boxes
// starting at group x0 (a multiple of 8: 16-byte aligned box origin)
__device__ __forceinline__ void stage_groups(int64_t kst, int ncols, int lg, int& x0, int& nbox) {
    const int g_first = (int)(kst >> lg);
    const int g_last = (int)((kst + ncols - 1) >> lg);
    x0 = g_first & ~7;
    nbox = (g_last - x0) / 8 + 1;
}

template <int BITS, bool BF, bool SBT>
__global__ void __launch_bounds__(kThreads, 1)
    qmm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap bmap,
                   const Params p) {
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();
    // 1024-byte aligned base (128-byte swizzle atoms)
    // pointer arithmetic on the shared array keeps accesses in the shared state space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int mt = p.mt;
    const int XS = p.x_stages, WS = p.w_stages, AS = p.a_stages;
    const uint32_t x_stage_bytes = (uint32_t)mt * kXBK * 2;    // two 64-column swizzle atoms
    const uint32_t w_stage_bytes = kTileN * kBK * BITS / 8;    // 32 * BITS bytes per row (two boxes for 6, 8 bits)
    uint8_t* xbuf = smem;
    uint8_t* wbuf = xbuf + (size_t)XS * x_stage_bytes;
    const uint32_t sb_stage_bytes = 2u * kSbBox * (uint32_t)p.sb_boxes;
    uint8_t* sbbuf = wbuf + (size_t)WS * w_stage_bytes;       // SBT: per W stage, scales then biases
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbbuf + (SBT ? (size_t)WS * sb_stage_bytes : 0));
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + kMaxWStages;
    uint64_t* x_full = w_empty + kMaxWStages;
    uint64_t* x_empty = x_full + kMaxXStages;
    uint64_t* a_full = x_empty + kMaxXStages;
    uint64_t* a_empty = a_full + kMaxAStages;
    uint64_t* acc_full = a_empty + kMaxAStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int tile, piece, s_t;
    int64_t k_begin, k_end;
    piece_of(p.plan, p.K, blockIdx.x, tile, piece, s_t, k_begin, k_end);
    const int64_t n0 = (int64_t)tile * kTileN;                 // first weight row of the tile within its batch
    const int64_t m0 = (int64_t)blockIdx.z * p.mchunk;         // first x row of the chunk within its batch
    const int64_t nw0 = (int64_t)blockIdx.y * p.w_rows_b + n0;   // the tile's first row in the weight / scale tensors
    const int64_t mb0 = (int64_t)blockIdx.y * p.M;              // the batch's first row of x / out
    const int nk64 = (int)((k_end - k_begin) / 64);            // 64-column units in this piece
    const int nst = (nk64 + 3) / 4;                            // 256-column weight / A stages
    const int nxs = (nk64 + 1) / 2;                            // 128-column activation stages
    const int nas = nxs;                                       // = A stages

    // the copy of weight stage i (and its scales / biases) into ring slot i % WS
    auto issue_w = [&](int i) {
        const int s = i % WS;
        const int64_t kst = k_begin + (int64_t)kBK * i;
        int x0 = 0, nbox = 0;
        if constexpr (SBT) stage_groups(kst, (int)min((int64_t)kBK, k_end - kst), p.gs_log2, x0, nbox);
        mbar_arrive_expect_tx(&w_full[s], w_stage_bytes + 2u * kSbBox * (uint32_t)nbox);
        // x coordinate in 32-bit words: (k_begin + 256 i) * BITS / 32; 6- and
        // 8-bit stages come as two 128-column boxes
        tma_load_2d(wbuf + (size_t)s * w_stage_bytes, &wmap, &w_full[s], (int)(kst * BITS / 32), (int)nw0);
        if constexpr (BITS == 6 || BITS == 8)
            tma_load_2d(wbuf + (size_t)s * w_stage_bytes + w_stage_bytes / 2, &wmap, &w_full[s],
                        (int)(kst * BITS / 32) + 4 * BITS, (int)nw0);
        if constexpr (SBT) {
            uint8_t* sb = sbbuf + (size_t)s * sb_stage_bytes;
            for (int bx = 0; bx < nbox; ++bx) {
                tma_load_2d(sb + bx * kSbBox, &smap, &w_full[s], x0 + 8 * bx, (int)nw0);
                tma_load_2d(sb + (uint32_t)p.sb_boxes * kSbBox + bx * kSbBox, &bmap, &w_full[s], x0 + 8 * bx,
                            (int)nw0);
            }
        }
    };

    if (warp == 1 && lane == 0) {   // (warp 0 allocates tensor memory meanwhile)
        for (int i = 0; i < WS; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], 8);   // both halves: one arrive per warp of two groups
        }
        for (int i = 0; i < XS; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);               // tcgen05.commit
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(&a_full[i], 4);              // the 4 warps of one group
            mbar_init(&a_empty[i], 1);             // the commit of the stage's issuer
        }
        mbar_init(acc_full, p.n_issuers);         // one commit per issuer
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the barriers, as the copies see them
        // Programmatic launch: this kernel may start while the kernels before
        // it finish. The packed weights, scales and biases are not written by
        // them, so the first weight stage is requested now, before the
        // tensor-memory set-up (the rest of the ring follows after it:
        // requested alone, the first stage lands sooner); the activation
        // copies and every global store wait for those kernels to complete.
        if (nst > 0) issue_w(0);
    }
    if (warp == 0) {   // tensor-memory allocation (whole warp)
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t acc_col = 0;   // accumulator of issuer j: columns [j * mt, (j + 1) * mt)
    const int NI = p.n_issuers;
    const uint32_t a_col0 = (uint32_t)kTmemCols - kAStageCols * (uint32_t)AS;   // A ring at the top
    Ctl ctl{p.status, p.spin_limit, abort_flag};

    if (warp == 0) {
        // ---------------- packed-weight producer ----------------
        if (lane == 0) {
            int issued = min(nst, 1);   // the first stage went out before the set-up
            for (int i = issued; i < nst; ++i) {
                if (!mbar_wait(&w_empty[i % WS], ((i / WS) & 1) ^ 1, ctl)) break;
                issue_w(i);
                ++issued;
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int i = (issued > WS ? issued - WS : 0); i < issued; ++i)
                mbar_wait_drain(&w_full[i % WS], (i / WS) & 1, p.spin_limit, p.status);
        }
    } else if (warp == 1) {
        // ---------------- activation producer ----------------
        if (lane == 0) {
            pdl_wait();   // the kernels before this one are complete: x may be read
            int issued = 0;
            for (int j = 0; j < nxs; ++j) {
                const int s = j % XS;
                if (!mbar_wait(&x_empty[s], ((j / XS) & 1) ^ 1, ctl)) break;
                mbar_arrive_expect_tx(&x_full[s], x_stage_bytes);
                uint8_t* dst = xbuf + (size_t)s * x_stage_bytes;
                const int kx = (int)(k_begin + kXBK * j);
                tma_load_2d(dst, &xmap, &x_full[s], kx, (int)(mb0 + m0));
                tma_load_2d(dst + (size_t)mt * 128, &xmap, &x_full[s], kx + 64, (int)(mb0 + m0));
                ++issued;
            }
            for (int j = (issued > XS ? issued - XS : 0); j < issued; ++j)
                mbar_wait_drain(&x_full[j % XS], (j / XS) & 1, p.spin_limit, p.status);
        }
    } else if (warp == 2 || warp == 3) {
        // ---------------- MMA issuers (whole warps) ----------------
        // issuer jw takes the A stages i == jw (mod NI), each with its
        // activation stage i, into its own accumulator
        const int jw = warp - 2;
        if (jw < NI) {
            const uint32_t idesc = make_idesc(BF ? 1 : 0, mt);
            const uint32_t acc_tm = tmem_base + acc_col + (uint32_t)(jw * mt);
            uint32_t acc_flag = 0;
            const uint32_t xs_base = smem_u32(xbuf);
            const uint32_t atom_step = (uint32_t)mt * 8u;   // one 64-column swizzle atom (mt x 128 B) >> 4
            const uint32_t a_tm0 = tmem_base + a_col0;
            int sa = jw, pa = 0, sx = jw, px = 0;   // slots / parities of stage i (both rings have even depth with two issuers)
            for (int i = jw; i < nas; i += NI) {
                if (!warp_wait(&a_full[sa], (uint32_t)pa, ctl)) break;
                if (!warp_wait(&x_full[sx], (uint32_t)px, ctl)) break;
                fence_after();
                const int kk_end = (2 * i + 1 < nk64) ? 8 : 4;   // the last stage may hold one 64-column unit
                // descriptor of the stage's first 16 columns; the next ones
                // advance the 14-bit start-address field (no carry: shared
                // addresses are below 2^18)
                const uint32_t d0 = sw128_desc_lo(xs_base + (uint32_t)sx * x_stage_bytes);
                const uint32_t a_t0 = a_tm0 + (uint32_t)sa * kAStageCols;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    if (kk < kk_end) {
                        mma_f16_tmem_a_warp(acc_tm, a_t0 + (uint32_t)kk * 8u,
                                            d0 + (uint32_t)(kk >> 2) * atom_step + (uint32_t)(kk & 3) * 2u, idesc,
                                            acc_flag);
                        acc_flag = 1;
                    }
                }
                mma_commit_warp(&x_empty[sx]);
                mma_commit_warp(&a_empty[sa]);
                sx += NI;
                if (sx >= XS) {
                    sx -= XS;
                    px ^= 1;
                }
                sa += NI;
                if (sa >= AS) {
                    sa -= AS;
                    pa ^= 1;
                }
            }
            mma_commit_warp(acc_full);   // completes when every MMA of every issuer has finished
            // no MMA may still run when tensor memory is freed
            if (lane == 0) mbar_wait_drain(acc_full, 0, p.spin_limit, p.status);
            __syncwarp();
        }
    } else {
        // ---------------- dequantize, then epilogue ----------------
        // Warp group grp (4 warps, one per tensor-memory lane quadrant) takes
        // the A stages i == grp (mod 4): 128 columns, i.e. the half (i & 1) =
        // (grp & 1) of weight stage i / 2, for the 32 rows of its quadrant.
        const int dw = warp - kDequantWarp0;        // 0..15
        const int quad = warp & 3;                  // TMEM lane quadrant of this warp
        const int grp = dw >> 2;
        const int hw = grp & 1;                     // half of every weight stage this group reads
        const int r = quad * 32 + lane;             // weight row within the tile
        const int64_t row = n0 + r;
        const bool row_ok = row < p.N;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int lg = p.gs_log2;
        const uint32_t nibm = pin_reg(p.nib_mask), magic = pin_reg(p.magic);
        // shared addresses of this thread's four 16-byte chunks (4 hw .. 4 hw + 3)
        // of its row in ring slot 0: 128-byte rows, 128-byte TMA swizzle
        // (16-byte chunk c of row r at chunk c ^ (r & 7))
        const uint32_t wrow_s = smem_u32(wbuf) + (uint32_t)r * 128u;
        uint32_t wc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wc[c] = wrow_s + 16u * (uint32_t)((4 * hw + c) ^ (r & 7));
        // other widths: the BITS 16-byte granules of this thread's 128 columns
        // (2 bits: 64-byte rows, 64-byte swizzle; 3 bits: 96-byte rows; 6 bits:
        // two boxes of 96-byte rows; 8 bits: two boxes of 128-byte rows,
        // 128-byte swizzle)
        uint32_t wg[BITS];
#pragma unroll
        for (int c = 0; c < BITS; ++c) {
            uint32_t lin;
            if constexpr (BITS == 2) {
                lin = (uint32_t)r * 64u + (uint32_t)hw * 32u + 16u * c;
                lin ^= ((lin >> 7) & 3u) << 4;
            } else if constexpr (BITS == 3) {
                lin = (uint32_t)r * 96u + (uint32_t)hw * 48u + 16u * c;
            } else if constexpr (BITS == 6) {
                lin = (uint32_t)hw * (kTileN * 96u) + (uint32_t)r * 96u + 16u * c;
            } else {
                lin = (uint32_t)hw * (kTileN * 128u) + (uint32_t)r * 128u + 16u * c;
                lin ^= ((lin >> 7) & 7u) << 4;
            }
            wg[c] = smem_u32(wbuf) + lin;
        }
        // 8-bit codes: the two power-of-two factors that make a subnormal byte the code
        const uint32_t k1 = pin_reg(BF ? 0x7F007F00u : 0x6C006C00u), k2 = pin_reg(BF ? 0x42804280u : 0x6C006C00u);
        const uint32_t ta0 = tmem_base + lane_base + a_col0;
        // TMA-staged scales / biases: row r of each 8-group box, in slot 0
        const uint32_t sb0 = smem_u32(sbbuf) + (uint32_t)r * 16u;
        const uint32_t bias_off = (uint32_t)p.sb_boxes * kSbBox;
        // group offsets of the four 32-column quarters within the weight
        // stage; every piece starts on a group boundary and gs divides the
        // 256-column stage
        int cq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cq[q] = (128 * hw + 32 * q) >> lg;
        const int gstep2 = 2 * (kBK >> lg);
        int g = (int)(k_begin >> lg) + (grp >> 1) * (kBK >> lg);   // first group of weight stage i / 2

        const uint16_t* srow = p.scales + (row_ok ? (int64_t)blockIdx.y * p.w_rows_b + row : 0) * p.groups;
        const uint16_t* brow = p.biases + (row_ok ? (int64_t)blockIdx.y * p.w_rows_b + row : 0) * p.groups;
        // scale / bias of the four quarters of A stage i, from global memory
        // (when they do not come by TMA), one of this group's stages ahead
        auto load_sb = [&](int i, uint32_t (&sv)[4], uint32_t (&bv)[4]) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sv[q] = 0u;
                bv[q] = 0u;
                if (i < nas && 2 * i + (q >> 1) < nk64 && row_ok) {
                    const int64_t gg = (k_begin + (int64_t)kAK * i + 32 * q) >> lg;
                    sv[q] = __ldg(srow + gg);
                    bv[q] = __ldg(brow + gg);
                }
            }
        };
        uint32_t s1[4] = {0u, 0u, 0u, 0u}, b1[4] = {0u, 0u, 0u, 0u};
        if constexpr (!SBT) load_sb(grp, s1, b1);

        // weight stage v = i / 2 advances by 2 per iteration (even ring depth:
        // this group always meets the same slots); A stage i advances by 4
        int sw = grp >> 1, pw = 0, sa = grp, pa = 0;   // (WS >= 4, AS >= 4)
        uint32_t w_off = (uint32_t)sw * w_stage_bytes, sb_off = (uint32_t)sw * sb_stage_bytes;
        for (int i = grp; i < nas; i += 4) {
            const bool hi_active = 2 * i + 1 < nk64;   // the last stage may hold one 64-column unit
            uint32_t sc[4], bc[4];
            if constexpr (!SBT) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sc[q] = s1[q];
                    bc[q] = b1[q];
                }
                load_sb(i + 4, s1, b1);
            }
            if (!warp_wait(&w_full[sw], (uint32_t)pw, ctl)) break;
            uint4 v[BITS];
            if constexpr (BITS == 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = lds128(wc[c] + w_off);
            } else {
#pragma unroll
                for (int c = 0; c < BITS; ++c) v[c] = lds128(wg[c] + w_off);
            }
            if constexpr (SBT) {
                // group of each quarter relative to the slot's first box origin
                // (g rounded down to a multiple of 8): box (idx >> 3), column
                // (idx & 7); a quarter past the piece reads column 0 (in bounds, unused)
                const int rel = g & 7;
                const uint32_t sbs = sb0 + sb_off;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int idx = (q < 2 || hi_active) ? rel + cq[q] : 0;
                    const uint32_t o = (uint32_t)(idx >> 3) * kSbBox + 2u * (uint32_t)(idx & 7);
                    sc[q] = lds16(sbs + o);
                    bc[q] = lds16(sbs + bias_off + o);
                }
            }
            // the stage is refilled by TMA (async proxy): order these generic
            // reads before that write, then release this half of the stage
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[sw]);

            if (!warp_wait(&a_empty[sa], (uint32_t)(pa ^ 1), ctl)) break;
            fence_after();
            const uint32_t ta = ta0 + (uint32_t)sa * kAStageCols;
            // one 8-column store per word pair (a quarter past the piece is
            // decoded from whatever the slot holds; its columns are not read)
            uint32_t s2[4], b2[4];   // scale / bias of each 32-column quarter in both halves
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                s2[c] = __byte_perm(sc[c], 0u, 0x1010);
                b2[c] = __byte_perm(bc[c], 0u, 0x1010);
            }
            if constexpr (BITS == 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // the subnormal form when s * 2^133 is a finite bf16 (this
                    // row's scale: lanes may differ; the stores below run converged)
                    uint32_t o8[8], o8b[8];
                    const uint32_t e = (sc[c] >> 7) & 0xFFu;
                    if (BF && e >= 1u && e <= 121u) {
                        const uint32_t s133 = s2[c] + 0x42804280u, s129 = s2[c] + 0x40804080u;
                        dequant_word4_sub(v[c].x, s133, s129, b2[c], &o8[0]);
                        dequant_word4_sub(v[c].y, s133, s129, b2[c], &o8[4]);
                        dequant_word4_sub(v[c].z, s133, s129, b2[c], &o8b[0]);
                        dequant_word4_sub(v[c].w, s133, s129, b2[c], &o8b[4]);
                    } else {
                        dequant_word4<BF>(v[c].x, s2[c], b2[c], nibm, magic, &o8[0]);
                        dequant_word4<BF>(v[c].y, s2[c], b2[c], nibm, magic, &o8[4]);
                        dequant_word4<BF>(v[c].z, s2[c], b2[c], nibm, magic, &o8b[0]);
                        dequant_word4<BF>(v[c].w, s2[c], b2[c], nibm, magic, &o8b[4]);
                    }
                    __syncwarp();
                    tmem_st8(ta + 16u * c, o8);
                    tmem_st8(ta + 16u * c + 8u, o8b);
                }
            } else {
                const uint32_t* u = reinterpret_cast<const uint32_t*>(v);   // 4 * BITS words, 128 codes
                if constexpr (BITS == 2) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) {   // 16 codes per word
                        uint32_t o8[8];
                        dequant16_b2<BF>(u[m], s2[m >> 1], b2[m >> 1], nibm, magic, o8);
                        tmem_st8(ta + 8u * m, o8);
                    }
                } else if constexpr (BITS == 3) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {   // 32 codes per 3 words
                        uint32_t o0[8], o1[8];
                        dequant32_b3<BF>(u[3 * m], u[3 * m + 1], u[3 * m + 2], s2[m], b2[m], nibm, magic, o0, o1);
                        tmem_st8(ta + 16u * m, o0);
                        tmem_st8(ta + 16u * m + 8u, o1);
                    }
                } else if constexpr (BITS == 6) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) {   // 16 codes per 3 words
                        uint32_t o8[8];
                        dequant16_b6<BF>(u[3 * m], u[3 * m + 1], u[3 * m + 2], s2[m >> 1], b2[m >> 1], nibm, magic,
                                         o8);
                        tmem_st8(ta + 8u * m, o8);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 8; ++m) {   // 16 codes per 4 words
                        uint32_t o8[8];
                        dequant16_b8<BF>(&u[4 * m], s2[m >> 1], b2[m >> 1], k1, k2, o8);
                        tmem_st8(ta + 8u * m, o8);
                    }
                }
            }
            tmem_st_wait();
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[sa]);
            g += gstep2;
            sw += 2;
            w_off += 2u * w_stage_bytes;
            sb_off += 2u * sb_stage_bytes;
            if (sw >= WS) {
                sw -= WS;
                pw ^= 1;
                w_off -= (uint32_t)WS * w_stage_bytes;
                sb_off -= (uint32_t)WS * sb_stage_bytes;
            }
            sa += 4;
            if (sa >= AS) {
                sa -= AS;
                pa ^= 1;
            }
        }

        // epilogue: accumulator rows -> fp32 partials or T output; the 4 warps
        // of a quadrant take 8-column chunks in turn
        pdl_wait();   // the kernels before this one are complete: the output and partials may be written
        const bool ok = warp_wait(acc_full, 0, ctl);
        fence_after();
        if (ok) {
            const int64_t mrows = min((int64_t)mt, p.M - m0);
            const bool split = p.plan.slots() > 1;
            float* pslot = p.partials + (int64_t)piece * gridDim.y * p.M * p.N;   // slots of [batch * M, N]
            const int nacc = nxs < NI ? nxs : NI;   // accumulators that received MMAs
            for (int c = 8 * grp; c < mt; c += 32) {
                uint32_t v[8];
                __syncwarp();
                tmem_ld8(tmem_base + lane_base + acc_col + (uint32_t)c, v);
                tmem_ld_wait();
                if (nacc > 1) {   // issuer 1's partial sum, added after issuer 0's
                    uint32_t v1[8];
                    tmem_ld8(tmem_base + lane_base + acc_col + (uint32_t)(mt + c), v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                }
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int64_t m = c + j;
                        if (m < mrows) {
                            const float f = __uint_as_float(v[j]);
                            const int64_t idx = (mb0 + m0 + m) * p.N + row;
                            if (split) {
                                pslot[idx] = f;
                            } else if (BF) {
                                static_cast<uint16_t*>(p.out)[idx] = BF16::from_f32(f);
                            } else {
                                static_cast<uint16_t*>(p.out)[idx] = F16::from_f32(f);
                            }
                        }
                    }
                }
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using tc::kBK;
using tc::kMaxAStages;
using tc::kMaxMt;
using tc::kMaxWStages;
using tc::kMaxXStages;
using tc::kThreads;
using tc::kTileN;
using tc::kTmemCols;

int qmm_tc_supported(int64_t M, int64_t N, int64_t K, int bits, int gs) {
    (void)M;
    (void)N;
    if (bits != 2 && bits != 3 && bits != 4 && bits != 6 && bits != 8) return 0;
    if (K % 64 != 0 || gs < 32) return 0;   // 64-column halves, whole groups
    if (K > (int64_t)1 << 30) return 0;       // column offsets are kept in 32-bit registers
    // other widths: whole 256-column stages (every piece starts on one) and
    // packed rows a multiple of 16 bytes (TMA row stride)
    if (bits != 4 && (K % 256 != 0 || (K * bits / 8) % 16 != 0)) return 0;
    return 1;
}

// Ring depths for x rows padded to mt and the given code width; false when
// they do not fit. One CTA per SM: a second co-resident CTA of this kernel
// could run warps whose tensor-memory lane quadrant differs from
// (warp index % 4), which the dequantize and epilogue roles rely on; the
// kernel also takes all 512 tensor-memory columns. The shared-memory request
// is kept above half of the SM's capacity.
// Two issuers (two accumulators) while they leave room for four A stages
// (one per dequantize group). Ring depths and slot ownership: a ring slot
// must always be waited on by the same role, phase after phase, because
// mbarrier.try_wait.parity reports a phase two ahead of the barrier as
// complete. Hence, with two issuers taking alternate stages, the A and
// activation rings have even depth; the weight ring has even depth (two of
// the four dequantize groups read the even weight stages, two the odd ones);
// and the A ring holds at least the four stages of the four groups.
// The weight ring gets the shared memory first: its stages stream from DRAM
// and the bytes in flight per SM set the bandwidth; activation tiles are L2
// hits and need only a short ring (at least 3 stages, 2 for the widest tiles).
static bool size_rings(int mt, int bits, int sb_boxes, int* ni_out, int* as_out, int* ws_out, int* xs_out,
                       size_t* smem_out) {
    const int ni = (tc::kMaxIssuers * mt + 4 * (int)tc::kAStageCols <= kTmemCols) ? tc::kMaxIssuers : 1;
    int as = (kTmemCols - ni * mt) / (int)tc::kAStageCols;
    as = as > kMaxAStages ? kMaxAStages : as;
    if (ni == 2) as &= ~1;
    if (as < 4) return false;
    const size_t kBars = 512;
    const size_t x_stage = (size_t)mt * tc::kXBK * 2;
    const size_t w_stage = (size_t)kTileN * kBK * bits / 8 + 2u * tc::kSbBox * (size_t)sb_boxes;
    const size_t budget = 224 * 1024 - 1024 - kBars;
    const int xs_min = mt > 128 ? 2 : (ni == 2 ? 4 : 3);
    if ((size_t)xs_min * x_stage + 4 * w_stage > budget) return false;
    int ws = (int)((budget - (size_t)xs_min * x_stage) / w_stage);
    ws = ws > kMaxWStages ? kMaxWStages : ws;
    ws &= ~1;
    int xs = (int)((budget - (size_t)ws * w_stage) / x_stage);
    xs = xs > kMaxXStages ? kMaxXStages : xs;
    if (ni == 2) xs &= ~1;
    if (ws < 4 || xs < xs_min) return false;
    size_t smem = 1024 + (size_t)xs * x_stage + (size_t)ws * w_stage + kBars;
    if (smem < 120 * 1024) smem = 120 * 1024;
    if (smem > 227 * 1024) return false;
    static_assert((2 * kMaxWStages + 2 * kMaxXStages + 2 * kMaxAStages + 1) * 8 + 8 <= 512, "barrier area");
    *ni_out = ni;
    *as_out = as;
    *ws_out = ws;
    *xs_out = xs;
    *smem_out = smem;
    return true;
}

cudaError_t launch_qmm_tc(const QmmTcLaunch& L, cudaStream_t stream) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t M = L.M, N = L.N, K = L.K;
    const int64_t B = L.batch > 0 ? L.batch : 1;
    const int64_t NW = L.w_batched ? B * N : N;   // weight / scale rows in the tensors
    const int bits = L.bits;
    if (!qmm_tc_supported(M, N, K, bits, L.group_size)) return cudaErrorInvalidValue;

    // packed weights: u32 [N, K * bits / 32], one box of 256 columns x 128 rows
    // per stage (two of 128 columns for 6 and 8 bits): 4 bits 128-byte rows and
    // 2 bits 64-byte rows, swizzled at their width; 3 and 6 bits 96-byte rows
    // (16-byte reads of rows 96 bytes apart already spread over the banks);
    // 8 bits 128-byte rows, 128-byte swizzle
    CUtensorMap wmap, xmap, smap, bmap;
    {
        cuuint64_t dims[2] = {(cuuint64_t)(K * bits / 32), (cuuint64_t)NW};
        cuuint64_t strides[1] = {(cuuint64_t)(K * bits / 8)};
        const cuuint32_t bw = (bits == 6 || bits == 8) ? (cuuint32_t)(4 * bits) : (cuuint32_t)(8 * bits);
        cuuint32_t box[2] = {bw, 128};
        cuuint32_t es[2] = {1, 1};
        const CUtensorMapSwizzle sw = bits == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                      : (bits == 4 || bits == 8) ? CU_TENSOR_MAP_SWIZZLE_128B
                                                                 : CU_TENSOR_MAP_SWIZZLE_NONE;
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(L.w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // x rows per M chunk: the largest multiple of 16 (at most 256) whose rings
    // fit in shared memory next to this width's weight stages
    int mchunk = 0, mt = 0, ni = 0, as = 0, ws = 0, xs = 0, sb_boxes = 0;
    size_t smem = 0;
    const int64_t groups = K / L.group_size;
    const bool sbt = groups % 8 == 0 && (reinterpret_cast<uintptr_t>(L.scales) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(L.biases) & 15u) == 0;
    // one box of scales / biases per stage suffices when every piece starts on
    // a 256-column boundary (then so does every stage)
    if (sbt) {
        bool aligned = true;
        const int64_t KU = K / L.plan.unit;
        for (int st = L.plan.s_base; st <= L.plan.s_base + (L.plan.n_extra > 0 ? 1 : 0); ++st)
            for (int j = 0; j < st; ++j)
                if (((j * KU / st) * L.plan.unit) % 256 != 0) aligned = false;
        sb_boxes = aligned ? 1 : 2;
    }
    for (int cap = std::min(L.plan.mcap, kMaxMt); cap >= 16 && mchunk == 0; cap -= 16) {
        const int64_t mrows = M < cap ? M : cap;
        const int mt_c = (int)((mrows + 15) / 16 * 16);
        int ni_c, as_c, ws_c, xs_c;
        size_t smem_c;
        if (size_rings(mt_c, bits, sb_boxes, &ni_c, &as_c, &ws_c, &xs_c, &smem_c)) {
            mchunk = cap;
            mt = mt_c;
            ni = ni_c;
            as = as_c;
            ws = ws_c;
            xs = xs_c;
            smem = smem_c;
        }
    }
    if (mchunk == 0) return cudaErrorInvalidValue;
    const int64_t mchunks = (M + mchunk - 1) / mchunk;

    // activations: 16-bit [M, K], box {64 columns, mt rows}, 128-byte swizzle
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(B * M)};
        cuuint64_t strides[1] = {(cuuint64_t)(K * 2)};
        cuuint32_t box[2] = {64, (cuuint32_t)mt};
        cuuint32_t es[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(L.x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    // scales / biases: 16-bit [N, K / group_size], box {8 groups, 128 rows}
    // (16-byte rows, no swizzle); the row stride and both base addresses must
    // be multiples of 16 bytes, otherwise the dequantize warps load them from
    // global memory
    memset(&smap, 0, sizeof(smap));
    memset(&bmap, 0, sizeof(bmap));
    if (sbt) {
        cuuint64_t dims[2] = {(cuuint64_t)groups, (cuuint64_t)NW};
        cuuint64_t strides[1] = {(cuuint64_t)(groups * 2)};
        cuuint32_t box[2] = {8, 128};
        cuuint32_t es[2] = {1, 1};
        CUtensorMap* maps[2] = {&smap, &bmap};
        const void* srcs[2] = {L.scales, L.biases};
        for (int t = 0; t < 2; ++t)
            if (enc(maps[t], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(srcs[t]), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
    }

    tc::Params p;
    p.scales = static_cast<const uint16_t*>(L.scales);
    p.biases = static_cast<const uint16_t*>(L.biases);
    p.out = L.out;
    p.partials = L.partials;
    p.M = M;
    p.w_rows_b = L.w_batched ? N : 0;
    p.N = N;
    p.K = K;
    p.groups = K / L.group_size;
    int lg = 0;
    while ((1 << lg) < L.group_size) ++lg;
    p.gs_log2 = lg;
    p.plan = L.plan;
    p.mt = mt;
    p.mchunk = mchunk;
    p.x_stages = xs;
    p.w_stages = ws;
    p.a_stages = as;
    if ((ni == 2 && ((xs | as) & 1)) || (ws & 1) || ws < 4) return cudaErrorInvalidValue;   // ring invariants above
    p.n_issuers = ni;
    p.sb_boxes = sb_boxes > 0 ? sb_boxes : 1;
    p.nib_mask = bits == 2 ? 0x00030003u : bits == 3 ? 0x00070007u : bits == 6 ? 0x003F003Fu : 0x000F000Fu;
    p.magic = L.is_bf16 ? 0x43004300u : 0x64006400u;
    p.status = L.status;
    p.spin_limit = L.spin_limit;

    using KernFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const tc::Params);
#define GAI4_TC_KERNELS(B)                                                                                  \
    tc::qmm_tc_kernel<B, false, false>, tc::qmm_tc_kernel<B, true, false>, tc::qmm_tc_kernel<B, false, true>, \
        tc::qmm_tc_kernel<B, true, true>
    static const KernFn kernels[20] = {GAI4_TC_KERNELS(2), GAI4_TC_KERNELS(3), GAI4_TC_KERNELS(4), GAI4_TC_KERNELS(6),
                                       GAI4_TC_KERNELS(8)};
#undef GAI4_TC_KERNELS
    const int wi = bits == 2 ? 0 : bits == 3 ? 1 : bits == 4 ? 2 : bits == 6 ? 3 : 4;
    const int which = 4 * wi + (L.is_bf16 ? 1 : 0) + (sbt ? 2 : 0);
    const KernFn kern = kernels[which];
    static unsigned long long configured[20] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(configured[which] & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[which] |= 1ull << dev;
    }
    if (B > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)L.plan.pieces(), (unsigned)B, (unsigned)mchunks);
    return launch_pdl(kern, grid, dim3(kThreads), smem, stream, wmap, xmap, smap, bmap, p);
}

}  // namespace gai4
