// affine_gemv_f16.cu -- instantiations of the CUDA-core affine GEMV for f16 activations.
#include "affine_gemv.cuh"

namespace gai4 {
cudaError_t launch_affine_gemv_f16(const AffineGemvLaunch& L, cudaStream_t s) {
    return launch_affine_gemv_dtype<F16>(L, s);
}
}  // namespace gai4
