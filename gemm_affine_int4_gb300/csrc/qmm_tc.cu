// qmm_tc.cu -- tensor-core qmm_t and the split-K reduce (sm_103a).
#include "common.cuh"
#include "internal.h"

namespace gai4 {

// ---------------------------------------------------------------------------
// split-K reduce: out[m, n] = T(sum_{s < S} P[s, m, n]), summed in s order and
// rounded once (MLX PR, Correctness: fp32 partials, one rounding after the sum)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void splitk_reduce_kernel(const float* __restrict__ P, typename T::storage* __restrict__ out,
                                     int64_t MN, int S) {
    const int64_t i4 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i4 >= MN) return;
    if (i4 + 4 <= MN && (MN & 3) == 0) {
        float4 acc = *reinterpret_cast<const float4*>(P + i4);
        for (int s = 1; s < S; ++s) {
            const float4 v = *reinterpret_cast<const float4*>(P + (int64_t)s * MN + i4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        out[i4 + 0] = T::from_f32(acc.x);
        out[i4 + 1] = T::from_f32(acc.y);
        out[i4 + 2] = T::from_f32(acc.z);
        out[i4 + 3] = T::from_f32(acc.w);
    } else {
        for (int64_t i = i4; i < i4 + 4 && i < MN; ++i) {
            float acc = P[i];
            for (int s = 1; s < S; ++s) acc += P[(int64_t)s * MN + i];
            out[i] = T::from_f32(acc);
        }
    }
}

cudaError_t launch_splitk_reduce(const float* partials, void* out, int64_t M, int64_t N, int splits, int dtype,
                                 cudaStream_t s) {
    const int64_t MN = M * N;
    const unsigned blocks = (unsigned)(((MN + 3) / 4 + 255) / 256);
    switch (dtype) {
    case GAI4_F16:
        splitk_reduce_kernel<F16><<<blocks, 256, 0, s>>>(partials, static_cast<uint16_t*>(out), MN, splits);
        break;
    case GAI4_F32:
        splitk_reduce_kernel<F32><<<blocks, 256, 0, s>>>(partials, static_cast<float*>(out), MN, splits);
        break;
    default:
        splitk_reduce_kernel<BF16><<<blocks, 256, 0, s>>>(partials, static_cast<uint16_t*>(out), MN, splits);
        break;
    }
    return cudaGetLastError();
}

int qmm_tc_supported(int64_t, int64_t, int64_t, int, int) { return 0; }

cudaError_t launch_qmm_tc(const QmmTcLaunch&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gai4
