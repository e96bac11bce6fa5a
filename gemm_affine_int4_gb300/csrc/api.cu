// api.cu -- the C ABI of libgai4.so (declared in include/gai4.h): argument
// validation, planning (kernel choice, K split) and launch. No allocation.
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gai4 {

// Device status word: kernels with bounded waits record GAI4_ERR_TIMEOUT here.
__device__ int g_device_status;

static int* status_ptr() {
    static int* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 148;
    if (!cache[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cache[dev] = v;
    }
    return cache[dev];
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool valid_bits(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 6 || bits == 8; }
static bool valid_gs(int gs) { return gs == 32 || gs == 64 || gs == 128; }
static bool valid_dtype(int d) { return d == GAI4_F32 || d == GAI4_F16 || d == GAI4_BF16; }

// common checks of the affine entry points (shape part)
static gai4_status check_affine_shape(int dtype, int bits, int gs, int64_t N, int64_t K) {
    if (!valid_dtype(dtype) || !valid_bits(bits) || !valid_gs(gs)) return GAI4_ERR_UNSUPPORTED;
    if (N <= 0 || K <= 0 || K % gs != 0 || (K * bits) % 32 != 0) return GAI4_ERR_INVALID_ARG;
    return GAI4_OK;
}

static gai4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GAI4_OK : GAI4_ERR_CUDA; }

// CUDA-core affine kernel: choose x rows per CTA, rows per warp and K split
static AffineGemvLaunch plan_affine(const uint32_t* w, const void* sc, const void* bi, const void* x, void* out,
                                    int bits, int gs, int64_t M, int64_t N, int64_t K) {
    AffineGemvLaunch L;
    L.w = w;
    L.scales = sc;
    L.biases = bi;
    L.x = x;
    L.out = out;
    L.M = M;
    L.N = N;
    L.K = K;
    L.bits = bits;
    L.group_size = gs;
    L.mb = M == 1 ? 1 : (M == 2 ? 2 : (M <= 4 ? 4 : 8));
    L.rows_per_warp = L.mb == 1 ? 4 : (L.mb == 8 ? 1 : 2);
    const int E = (bits == 6 || bits == 8) ? 16 : 32;
    const int64_t its_total = (K / E + 31) / 32;   // warp iterations per row
    const int64_t mblocks = (M + L.mb - 1) / L.mb;
    const int64_t target = 4LL * num_sms();
    int S = 1;
    while (S < 8 && 2 * S <= its_total) {
        const int64_t rows_per_cta = (8 / S) * L.rows_per_warp;
        if (((N + rows_per_cta - 1) / rows_per_cta) * mblocks >= target) break;
        S *= 2;
    }
    L.ksplit = S;
    return L;
}

static cudaError_t launch_affine(const AffineGemvLaunch& L, int dtype, cudaStream_t s) {
    switch (dtype) {
    case GAI4_F32: return launch_affine_gemv_f32(L, s);
    case GAI4_F16: return launch_affine_gemv_f16(L, s);
    default: return launch_affine_gemv_bf16(L, s);
    }
}

// M = 1: the prefetching 4-bit kernel where it applies, else the general one
static cudaError_t run_qmv(const uint32_t* w, const void* sc, const void* bi, const void* x, void* out, int dtype,
                           int bits, int gs, int64_t N, int64_t K, cudaStream_t s) {
    if (qmv4_supported(sc, bi, dtype, bits, gs, N, K)) {
        int* st = status_ptr();
        if (!st) return cudaErrorMemoryAllocation;
        return launch_qmv4(w, sc, bi, x, out, dtype, gs, N, K, st, 2000000000LL, s);
    }
    const AffineGemvLaunch L = plan_affine(w, sc, bi, x, out, bits, gs, 1, N, K);
    return launch_affine(L, dtype, s);
}

// ---------------------------------------------------------------------------
// qmm_t planning: path (CUDA-core / tensor core) and K split
// ---------------------------------------------------------------------------
static const int64_t kTcMinM = 3;   // tensor-core path from this many x rows up (bf16/f16; measured crossover)

static gai4_status plan_qmm(int64_t M, int64_t N, int64_t K, int bits, int gs, int dtype, int split_k,
                            size_t ws_bytes, bool unlimited_ws, int* path, SplitPlan* plan, int64_t batch = 1) {
    gai4_status st = check_affine_shape(dtype, bits, gs, N, K);
    if (st != GAI4_OK) return st;
    if (M <= 0) return GAI4_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > 4) return GAI4_ERR_UNSUPPORTED;
    const bool tc = dtype != GAI4_F32 && M >= kTcMinM && qmm_tc_supported(M, N, K, bits, gs);
    SplitPlan p;
    if (split_k == 0) {
        if (tc) {
            const size_t per_slot = (size_t)batch * (size_t)M * (size_t)N * sizeof(float);
            const int max_slots = unlimited_ws ? 4 : (int)std::min<size_t>(4, ws_bytes / per_slot);
            p = auto_plan(M, N, K, gs, max_slots, batch);
        } else {
            uniform_plan(N, K, gs, 1, &p);
        }
    } else {
        // forced: K cut into split_k equal ranges (multiples of 64 and of the
        // group size, >= 256 columns; K < 512 is never split)
        if (!uniform_plan(N, K, gs, split_k, &p)) return GAI4_ERR_UNSUPPORTED;
        if (split_k > 1 && !tc) return GAI4_ERR_UNSUPPORTED;   // only the tensor-core path splits K
        // codes other than 4-bit are staged in whole 256-column stages
        if (split_k > 1 && bits != 4 && (K / split_k) % 256 != 0) return GAI4_ERR_UNSUPPORTED;
    }
    *path = tc ? 1 : 0;
    *plan = p;
    return GAI4_OK;
}

}  // namespace gai4

using namespace gai4;

extern "C" {

int gai4_version(void) { return 100; }

const char* gai4_status_string(int status) {
    switch (status) {
    case GAI4_OK: return "ok";
    case GAI4_ERR_INVALID_ARG: return "invalid argument";
    case GAI4_ERR_UNSUPPORTED: return "unsupported bits/group_size/dtype/split";
    case GAI4_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case GAI4_ERR_WORKSPACE: return "split-K workspace missing or too small";
    case GAI4_ERR_CUDA: return "CUDA error";
    case GAI4_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    default: return "unknown status";
    }
}

gai4_status gai4_quantize(const float* w, uint32_t* w_packed, void* scales, void* biases, gai4_dtype dtype,
                          int bits, int group_size, int64_t N, int64_t K, void* stream) {
    gai4_status st = check_affine_shape(dtype, bits, group_size, N, K);
    if (st != GAI4_OK) return st;
    if (!w || !w_packed || !scales || !biases) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(w_packed)) return GAI4_ERR_MISALIGNED;
    return from_cuda(launch_quantize(w, w_packed, scales, biases, dtype, bits, group_size, N, K,
                                     (cudaStream_t)stream));
}

gai4_status gai4_unpack(const uint32_t* w_packed, uint8_t* q_out, int bits, int64_t N, int64_t K, void* stream) {
    if (!valid_bits(bits)) return GAI4_ERR_UNSUPPORTED;
    if (!w_packed || !q_out || N <= 0 || K <= 0 || (K * bits) % 32 != 0) return GAI4_ERR_INVALID_ARG;
    return from_cuda(launch_unpack(w_packed, q_out, bits, N, K, (cudaStream_t)stream));
}

gai4_status gai4_dequantize(const uint32_t* w_packed, const void* scales, const void* biases, float* w_out,
                            gai4_dtype dtype, int bits, int group_size, int64_t N, int64_t K, void* stream) {
    gai4_status st = check_affine_shape(dtype, bits, group_size, N, K);
    if (st != GAI4_OK) return st;
    if (!w_packed || !scales || !biases || !w_out) return GAI4_ERR_INVALID_ARG;
    return from_cuda(launch_dequantize(w_packed, scales, biases, w_out, dtype, bits, group_size, N, K,
                                       (cudaStream_t)stream));
}

gai4_status gai4_qmv(const uint32_t* w_packed, const void* scales, const void* biases, const void* x, void* out,
                     gai4_dtype dtype, int bits, int group_size, int64_t N, int64_t K, void* stream) {
    gai4_status st = check_affine_shape(dtype, bits, group_size, N, K);
    if (st != GAI4_OK) return st;
    if (!w_packed || !scales || !biases || !x || !out) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(w_packed) || !aligned16(x)) return GAI4_ERR_MISALIGNED;
    return from_cuda(run_qmv(w_packed, scales, biases, x, out, dtype, bits, group_size, N, K, (cudaStream_t)stream));
}

size_t gai4_qmm_t_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits, int group_size, gai4_dtype dtype,
                                  int split_k) {
    int path = 0;
    SplitPlan plan;
    if (plan_qmm(M, N, K, bits, group_size, dtype, split_k, 0, true, &path, &plan) != GAI4_OK) return 0;
    return plan.slots() > 1 ? (size_t)plan.slots() * (size_t)M * (size_t)N * sizeof(float) : 0;
}

gai4_status gai4_qmm_t_plan(int64_t M, int64_t N, int64_t K, int bits, int group_size, gai4_dtype dtype,
                            int split_k, size_t workspace_bytes, int* path, int* splits) {
    if (!path || !splits) return GAI4_ERR_INVALID_ARG;
    SplitPlan plan;
    gai4_status st = plan_qmm(M, N, K, bits, group_size, dtype, split_k, workspace_bytes, false, path, &plan);
    if (st == GAI4_OK) *splits = plan.slots();
    return st;
}

gai4_status gai4_qmm_t(const uint32_t* w_packed, const void* scales, const void* biases, const void* x, void* out,
                       gai4_dtype dtype, int bits, int group_size, int64_t M, int64_t N, int64_t K, int split_k,
                       void* workspace, size_t workspace_bytes, void* stream) {
    int path = 0;
    SplitPlan plan;
    gai4_status st = plan_qmm(M, N, K, bits, group_size, dtype, split_k, workspace ? workspace_bytes : 0, false,
                              &path, &plan);
    if (st != GAI4_OK) return st;
    if (!w_packed || !scales || !biases || !x || !out) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(w_packed) || !aligned16(x)) return GAI4_ERR_MISALIGNED;
    const int splits = plan.slots();
    if (splits > 1) {
        if (!workspace || workspace_bytes < (size_t)splits * (size_t)M * (size_t)N * sizeof(float))
            return GAI4_ERR_WORKSPACE;
        if (!aligned16(workspace)) return GAI4_ERR_MISALIGNED;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (path == 0) {
        if (M == 1) return from_cuda(run_qmv(w_packed, scales, biases, x, out, dtype, bits, group_size, N, K, s));
        const AffineGemvLaunch L = plan_affine(w_packed, scales, biases, x, out, bits, group_size, M, N, K);
        return from_cuda(launch_affine(L, dtype, s));
    }
    QmmTcLaunch T;
    T.w = w_packed;
    T.scales = scales;
    T.biases = biases;
    T.x = x;
    T.out = out;
    T.partials = splits > 1 ? static_cast<float*>(workspace) : nullptr;
    T.M = M;
    T.N = N;
    T.K = K;
    T.bits = bits;
    T.group_size = group_size;
    T.plan = plan;
    T.is_bf16 = dtype == GAI4_BF16;
    T.status = status_ptr();
    T.spin_limit = 2000000000LL;   // ~1 s of SM clock per wait
    if (!T.status) return GAI4_ERR_CUDA;
    cudaError_t e = launch_qmm_tc(T, s);
    if (e != cudaSuccess) return GAI4_ERR_CUDA;
    if (splits > 1) e = launch_splitk_reduce(T.partials, out, M, N, plan, dtype, s);
    return from_cuda(e);
}

gai4_status gai4_q8_0_gemv(const uint32_t* blocks, const float* x, float* out, int64_t N, int64_t K, void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 32 != 0) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(x)) return GAI4_ERR_MISALIGNED;
    if (bq_tma_supported(BQ_Q8_0, N, K, blocks, x)) {
        int* st = status_ptr();
        if (!st) return GAI4_ERR_CUDA;
        return from_cuda(launch_q8_0_gemv_tma(blocks, x, out, N, K, st, 2000000000LL, (cudaStream_t)stream));
    }
    return from_cuda(launch_q8_0_gemv(blocks, x, out, N, K, (cudaStream_t)stream));
}

gai4_status gai4_q4_k_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K, void* stream) {
    if (!blocks || !x || !out || N <= 0 || K <= 0 || K % 256 != 0) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(x)) return GAI4_ERR_MISALIGNED;
    if (bq_tma_supported(BQ_Q4_K, N, K, blocks, x)) {
        int* st = status_ptr();
        if (!st) return GAI4_ERR_CUDA;
        return from_cuda(launch_q4_k_gemv_tma(blocks, x, out, N, K, st, 2000000000LL, (cudaStream_t)stream));
    }
    return from_cuda(launch_q4_k_gemv(blocks, x, out, N, K, (cudaStream_t)stream));
}

gai4_status gai4_q4_k_dequantize(const uint8_t* blocks, float* w_out, int64_t N, int64_t K, int decoder,
                                 void* stream) {
    if (!blocks || !w_out || N <= 0 || K <= 0 || K % 256 != 0) return GAI4_ERR_INVALID_ARG;
    if (decoder != 0 && decoder != 1) return GAI4_ERR_UNSUPPORTED;
    if (!aligned16(blocks) || ((uintptr_t)w_out & 3u) != 0) return GAI4_ERR_MISALIGNED;
    const int64_t nblk = N * (K / 256);
    cudaStream_t s = (cudaStream_t)stream;
    return from_cuda(decoder == 0 ? launch_q4_k_dequant_tma(blocks, w_out, nblk, s)
                                  : launch_q4_k_dequant_general(blocks, w_out, nblk, s));
}

gai4_status gai4_quantize_x_q8(const float* x, int8_t* xq, float* xd, int64_t K, void* stream) {
    if (!x || !xq || !xd || K <= 0 || K % 32 != 0) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || ((uintptr_t)xd & 3u) != 0) return GAI4_ERR_MISALIGNED;
    return from_cuda(launch_quantize_x_q8(x, xq, xd, K, (cudaStream_t)stream));
}

gai4_status gai4_q8_0_gemv_i8(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out, int64_t N,
                              int64_t K, void* stream) {
    if (!blocks || !xq || !xd || !out || N <= 0 || K <= 0 || K % 32 != 0) return GAI4_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(xq) || ((uintptr_t)xd & 3u) != 0) return GAI4_ERR_MISALIGNED;
    if (bq_tma_supported(BQ_Q8_0_I8, N, K, blocks, xq)) {
        int* st = status_ptr();
        if (!st) return GAI4_ERR_CUDA;
        return from_cuda(launch_q8_0_i8_gemv_tma(blocks, xq, xd, out, N, K, st, 2000000000LL, (cudaStream_t)stream));
    }
    return from_cuda(launch_q8_0_i8_gemv(blocks, xq, xd, out, N, K, (cudaStream_t)stream));
}

gai4_status gai4_last_device_status(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GAI4_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return GAI4_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return GAI4_ERR_CUDA;
    }
    return v == 0 ? GAI4_OK : (gai4_status)v;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gai4_qmm_t_noalloc: gai4_qmm_t with the split-K partials in a fixed device
// array of this library, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace gai4 {

static __device__ __align__(256) float g_noalloc_scratch[GAI4_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of the array for the current device. In host code
// g_noalloc_scratch names a host-side stand-in, not device memory, so the
// address is looked up once per device (that device current) and cached.
static float* noalloc_scratch() {
    static float* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<float*>(p);
    }
    return ptrs[dev];
}

}  // namespace gai4

extern "C" gai4_status gai4_qmm_t_noalloc(const uint32_t* w_packed, const void* scales, const void* biases,
                                          const void* x, void* out, gai4_dtype dtype, int bits, int group_size,
                                          int64_t M, int64_t N, int64_t K, int split_k, void* stream) {
    float* scratch = gai4::noalloc_scratch();
    if (!scratch) return GAI4_ERR_CUDA;
    return gai4_qmm_t(w_packed, scales, biases, x, out, dtype, bits, group_size, M, N, K, split_k, scratch,
                      (size_t)GAI4_NOALLOC_SCRATCH_BYTES, stream);
}

// ---------------------------------------------------------------------------
// batched / strided qmm_t: gather the activations when they are not
// contiguous rows on 16-byte boundaries, then one gai4_qmm_t per batch
// ---------------------------------------------------------------------------
namespace gai4 {
static size_t round256(size_t n) { return (n + 255) / 256 * 256; }
static int dtype_bytes(gai4_dtype d) { return d == GAI4_F32 ? 4 : 2; }
}  // namespace gai4

extern "C" size_t gai4_qmm_t_batched_workspace_bytes(int64_t batch, int64_t M, int64_t N, int64_t K, int bits,
                                                     int group_size, gai4_dtype dtype, int split_k) {
    using namespace gai4;
    if (batch < 1 || M < 1 || K < 1) return 0;
    const size_t gather = round256((size_t)batch * (size_t)M * (size_t)K * (size_t)dtype_bytes(dtype));
    int path = 0;
    SplitPlan plan;
    if (plan_qmm(M, N, K, bits, group_size, dtype, split_k, 0, true, &path, &plan, batch) != GAI4_OK) return 0;
    if (path == 1)   // one tensor-core launch over all batches: partials [S, batch * M, N]
        return gather + (plan.slots() > 1 ? (size_t)plan.slots() * (size_t)batch * (size_t)M * (size_t)N * 4 : 0);
    return gather + gai4_qmm_t_workspace_bytes(M, N, K, bits, group_size, dtype, split_k);
}

extern "C" gai4_status gai4_qmm_t_batched(const uint32_t* w_packed, const void* scales, const void* biases,
                                          int w_batched, const void* x, int64_t x_batch_stride,
                                          int64_t x_row_stride, void* out, gai4_dtype dtype, int bits,
                                          int group_size, int64_t batch, int64_t M, int64_t N, int64_t K,
                                          int split_k, void* workspace, size_t workspace_bytes, void* stream) {
    using namespace gai4;
    if (batch < 1 || M < 1 || N < 1 || K < 1) return GAI4_ERR_INVALID_ARG;
    if (!w_packed || !scales || !biases || !x || !out) return GAI4_ERR_INVALID_ARG;
    if (x_row_stride < K || x_batch_stride < 0) return GAI4_ERR_INVALID_ARG;
    if (dtype != GAI4_F32 && dtype != GAI4_F16 && dtype != GAI4_BF16) return GAI4_ERR_UNSUPPORTED;
    if (bits < 1 || bits > 8 || group_size <= 0 || K % group_size != 0) return GAI4_ERR_INVALID_ARG;
    const int tb = dtype_bytes(dtype);
    if (((uintptr_t)x % (uintptr_t)tb) != 0 || ((uintptr_t)out % (uintptr_t)tb) != 0) return GAI4_ERR_MISALIGNED;
    cudaStream_t s = (cudaStream_t)stream;
    // weights of matrix e: w_packed + e * N * (K * bits / 32) words, scales and
    // biases + e * N * (K / group_size) elements
    const int64_t w_words = N * (K * bits / 32);
    const int64_t sb_elems = N * (K / group_size);
    const bool contiguous = x_row_stride == K && ((uintptr_t)x & 15u) == 0 &&
                            (batch == 1 || ((x_batch_stride * tb) % 16) == 0);
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    int64_t xbs = x_batch_stride;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    size_t ws_left = workspace ? workspace_bytes : 0;
    if (!contiguous) {
        const size_t need = round256((size_t)batch * (size_t)M * (size_t)K * (size_t)tb);
        if (!workspace || workspace_bytes < need) return GAI4_ERR_WORKSPACE;
        if (((uintptr_t)workspace & 15u) != 0) return GAI4_ERR_MISALIGNED;
        cudaError_t e = launch_gather_rows(x, workspace, tb, batch, M, K, x_batch_stride, x_row_stride, s);
        if (e != cudaSuccess) return GAI4_ERR_CUDA;
        xb = ws;
        xbs = M * K;
        ws += need;
        ws_left -= need;
    }
    // tensor-core path: one launch over all batches (grid y = batch), the
    // activations viewed as [batch * M, K] and the output as [batch * M, N]
    {
        int path = 0;
        SplitPlan plan;
        const gai4_status pst = plan_qmm(M, N, K, bits, group_size, dtype, split_k, ws_left, false, &path, &plan, batch);
        if (pst != GAI4_OK) return pst;
        if (path == 1 && xbs == M * K && batch <= 65535) {
            const int splits = plan.slots();
            if (splits > 1) {
                if (!ws_left || ws_left < (size_t)splits * (size_t)batch * (size_t)M * (size_t)N * 4)
                    return GAI4_ERR_WORKSPACE;
                if (((uintptr_t)ws & 15u) != 0) return GAI4_ERR_MISALIGNED;
            }
            if (((uintptr_t)w_packed & 15u) != 0 || ((uintptr_t)xb & 15u) != 0) return GAI4_ERR_MISALIGNED;
            QmmTcLaunch T;
            T.w = w_packed;
            T.scales = scales;
            T.biases = biases;
            T.x = xb;
            T.out = out;
            T.partials = splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
            T.M = M;
            T.N = N;
            T.K = K;
            T.batch = batch;
            T.w_batched = w_batched ? 1 : 0;
            T.bits = bits;
            T.group_size = group_size;
            T.plan = plan;
            T.is_bf16 = dtype == GAI4_BF16;
            T.status = status_ptr();
            T.spin_limit = 2000000000LL;
            if (!T.status) return GAI4_ERR_CUDA;
            cudaError_t e = launch_qmm_tc(T, s);
            if (e != cudaSuccess) return GAI4_ERR_CUDA;
            if (splits > 1) e = launch_splitk_reduce(T.partials, out, batch * M, N, plan, dtype, s);
            return from_cuda(e);
        }
    }
    for (int64_t b = 0; b < batch; ++b) {
        const int64_t e = w_batched ? b : 0;
        const uint32_t* wb = w_packed + e * w_words;
        const uint8_t* sbp = static_cast<const uint8_t*>(scales) + (size_t)(e * sb_elems) * tb;
        const uint8_t* bbp = static_cast<const uint8_t*>(biases) + (size_t)(e * sb_elems) * tb;
        const void* xp = xb + (size_t)(b * xbs) * tb;
        void* op = static_cast<uint8_t*>(out) + (size_t)(b * M * N) * tb;
        const gai4_status st = gai4_qmm_t(wb, sbp, bbp, xp, op, dtype, bits, group_size, M, N, K, split_k,
                                          ws_left ? ws : nullptr, ws_left, stream);
        if (st != GAI4_OK) return st;
    }
    return GAI4_OK;
}
