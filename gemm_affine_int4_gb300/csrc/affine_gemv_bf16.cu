// affine_gemv_bf16.cu -- instantiations of the CUDA-core affine GEMV for bf16 activations.
#include "affine_gemv.cuh"

namespace gai4 {
cudaError_t launch_affine_gemv_bf16(const AffineGemvLaunch& L, cudaStream_t s) {
    return launch_affine_gemv_dtype<BF16>(L, s);
}
}  // namespace gai4
