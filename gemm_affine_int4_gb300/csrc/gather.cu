// gather.cu -- strided activations into contiguous rows (internal): the copy
// that gai4_qmm_t_batched runs before the matmul when the activations are not
// contiguous rows on 16-byte boundaries (the MLX PR's route copies activations
// at unaligned offsets first).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gai4 {

namespace {

// dst[(b * M + m) * K + k] = src[b * sb + m * sr + k]; elements of E bytes
template <typename E>
__global__ void gather_rows_kernel(const E* __restrict__ src, E* __restrict__ dst, int64_t B, int64_t M, int64_t K,
                                   int64_t sb, int64_t sr) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    const int64_t total = B * M * K;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = i % K, r = i / K;
        const int64_t m = r % M, b = r / M;
        dst[i] = src[b * sb + m * sr + k];
    }
}

}  // namespace

cudaError_t launch_gather_rows(const void* src, void* dst, int elem_bytes, int64_t B, int64_t M, int64_t K,
                               int64_t batch_stride, int64_t row_stride, cudaStream_t s) {
    const int64_t total = B * M * K;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 8 * 152);
    if (elem_bytes == 4)
        return launch_pdl(gather_rows_kernel<uint32_t>, dim3((unsigned)blocks), dim3(256), 0, s,
                          static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), B, M, K, batch_stride,
                          row_stride);
    return launch_pdl(gather_rows_kernel<uint16_t>, dim3((unsigned)blocks), dim3(256), 0, s,
                      static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), B, M, K, batch_stride,
                      row_stride);
}

}  // namespace gai4
