// internal.h -- launcher interfaces between the C ABI (api.cu) and the kernel
// translation units. Host-only declarations; no CUDA types beyond cudaStream_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gai4.h"

namespace gai4 {

// CUDA-core affine GEMV / small-M GEMM (affine_gemv_*.cu)
struct AffineGemvLaunch {
    const uint32_t* w;
    const void* scales;
    const void* biases;
    const void* x;      // [M, K]
    void* out;          // [M, N]
    int64_t M, N, K;
    int bits, group_size;
    int ksplit;         // warps of one CTA sharing a row group along K (1, 2, 4 or 8)
    int rows_per_warp;  // chosen by the launcher
    int mb;             // x rows per CTA (1, 2, 4, 8)
};
cudaError_t launch_affine_gemv_bf16(const AffineGemvLaunch& L, cudaStream_t s);
cudaError_t launch_affine_gemv_f16(const AffineGemvLaunch& L, cudaStream_t s);
cudaError_t launch_affine_gemv_f32(const AffineGemvLaunch& L, cudaStream_t s);

// CUDA-core qmv for 4-bit codes with per-lane asynchronous prefetch (qmv4.cu)
int qmv4_supported(const void* scales, const void* biases, int dtype, int bits, int gs, int64_t N, int64_t K);
cudaError_t launch_qmv4(const uint32_t* w, const void* scales, const void* biases, const void* x, void* out,
                        int dtype, int gs, int64_t N, int64_t K, int* status, long long spin_limit,
                        cudaStream_t s);

// K-split plan of the tensor-core qmm_t. The N axis is cut into 128-row
// tiles; tile t is cut along K into s_t pieces (s_t = s_base + 1 for the first
// n_extra tiles, s_base for the rest), piece j of s_t covering K columns
// [(j*KU/s_t)*unit, ((j+1)*KU/s_t)*unit), KU = K/unit. Piece j of every tile
// writes fp32 partial slot j. A uniform split S is {S, 0}.
struct SplitPlan {
    int tiles;
    int s_base;
    int n_extra;
    int unit;        // K granularity of the cuts: max(64, group_size)
    int mcap = 256;  // most x rows per M chunk of the tensor-core kernel
    __host__ __device__ int slots() const { return s_base + (n_extra > 0 ? 1 : 0); }
    __host__ __device__ int64_t pieces() const { return (int64_t)n_extra * (s_base + 1) + (int64_t)(tiles - n_extra) * s_base; }
};
// piece counts per tile legal for K (pieces >= 256 columns; K < 512 unsplit), at most 4
int max_pieces(int64_t K, int unit);
// uniform split S (1..4) if legal
bool uniform_plan(int64_t N, int64_t K, int gs, int S, SplitPlan* out);
// balanced automatic plan for the device's SM count, limited to max_slots partial slots
SplitPlan auto_plan(int64_t M, int64_t N, int64_t K, int gs, int max_slots, int64_t batch = 1);

// tensor-core qmm_t (qmm_tc.cu)
struct QmmTcLaunch {
    const uint32_t* w;
    const void* scales;
    const void* biases;
    const void* x;      // [M, K] bf16/f16
    void* out;          // [M, N]
    float* partials;    // [slots, batch * M, N] fp32 when plan.slots() > 1
    int64_t M, N, K;    // per batch
    int64_t batch = 1;  // problems in one launch: x [batch * M, K], out [batch * M, N]
    int w_batched = 0;  // weights / scales / biases stacked [batch * N, ...] (else shared)
    int bits, group_size;
    SplitPlan plan;
    int is_bf16;
    int* status;        // device status word
    long long spin_limit;
};
cudaError_t launch_qmm_tc(const QmmTcLaunch& L, cudaStream_t s);
int qmm_tc_supported(int64_t M, int64_t N, int64_t K, int bits, int group_size);

// quantize / unpack / dequantize (quant.cu)
cudaError_t launch_quantize(const float* w, uint32_t* packed, void* scales, void* biases,
                            int dtype, int bits, int gs, int64_t N, int64_t K, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* packed, uint8_t* q, int bits, int64_t N, int64_t K,
                          cudaStream_t s);
cudaError_t launch_dequantize(const uint32_t* packed, const void* scales, const void* biases,
                              float* out, int dtype, int bits, int gs, int64_t N, int64_t K,
                              cudaStream_t s);

// split-K reduce (qmm_tc.cu): out[m, n] = T(sum_{j < s_t} partials[j, m, n]),
// s_t the piece count of n's tile
cudaError_t launch_splitk_reduce(const float* partials, void* out, int64_t M, int64_t N,
                                 const SplitPlan& plan, int dtype, cudaStream_t s);

// strided activations into contiguous rows (gather.cu):
// dst[(b * M + m) * K + k] = src[b * batch_stride + m * row_stride + k]
cudaError_t launch_gather_rows(const void* src, void* dst, int elem_bytes, int64_t B, int64_t M, int64_t K,
                               int64_t batch_stride, int64_t row_stride, cudaStream_t s);

// block-quantized GEMVs with TMA-staged rows (blockq_tma.cu): supported when
// rows start on 16-byte boundaries and the activations fit in shared memory
enum { BQ_Q8_0 = 0, BQ_Q4_K = 1, BQ_Q8_0_I8 = 2 };
bool bq_tma_supported(int fmt, int64_t N, int64_t K, const void* blocks, const void* x);
cudaError_t launch_q8_0_gemv_tma(const uint32_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                                 int* status, long long spin_limit, cudaStream_t s);
cudaError_t launch_q4_k_gemv_tma(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                                 int* status, long long spin_limit, cudaStream_t s);
cudaError_t launch_q8_0_i8_gemv_tma(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out, int64_t N,
                                    int64_t K, int* status, long long spin_limit, cudaStream_t s);

// Q8_0 with integer activations, general case, and the activation quantizer (q8_act.cu)
cudaError_t launch_q8_0_i8_gemv(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out, int64_t N,
                                int64_t K, cudaStream_t s);
cudaError_t launch_quantize_x_q8(const float* x, int8_t* xq, float* xd, int64_t K, cudaStream_t s);

// Q4_K weights w[b][256] of nblk super-blocks with the (sc, m) decoder of the
// TMA-staged kernel (blockq_tma.cu) or of the general kernel (blockq.cu): test aid
cudaError_t launch_q4_k_dequant_tma(const uint8_t* blocks, float* out, int64_t nblk, cudaStream_t s);
cudaError_t launch_q4_k_dequant_general(const uint8_t* blocks, float* out, int64_t nblk, cudaStream_t s);

// block-quantized GEMVs, general case (blockq.cu)
cudaError_t launch_q8_0_gemv(const uint32_t* blocks, const float* x, float* out, int64_t N,
                             int64_t K, cudaStream_t s);
cudaError_t launch_q4_k_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N,
                             int64_t K, cudaStream_t s);

int num_sms();  // SM count of the current device (cached)

}  // namespace gai4
