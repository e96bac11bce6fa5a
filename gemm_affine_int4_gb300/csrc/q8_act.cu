// q8_act.cu -- Q8_0 with integer activations (internal): the per-block int8
// activation quantizer and the general-case GEMV (the TMA-staged kernel in
// blockq_tma.cu takes rows that start on 16-byte boundaries).
//
// hanzo-kernel quant.rs, "dp4a matvec" / "PACKED dp4a matvec": int8 weights
// and int8 activations, the inner sum an exact integer dot product (dp4a),
// out[row] = sum_block wd * dot(qw, xq). The activations are quantized per
// 32-element block: d = amax / 127, q = rint(x / d) clamped to +-127, in
// binary32 (IEEE division, round to nearest even), q = 0 for a zero block;
// out[n] = sum_b d_w[n, b] * d_x[b] * dot_b.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gai4 {

namespace {

// one thread per 32-element block
__global__ void quantize_x_q8_kernel(const float* __restrict__ x, int8_t* __restrict__ xq, float* __restrict__ xd,
                                     int64_t nblk) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblk) return;
    const float4* xb = reinterpret_cast<const float4*>(x + 32 * b);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = xb[i];
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.0f);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t word = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            int q = 0;
            if (d != 0.f) q = max(-127, min(127, __float2int_rn(__fdiv_rn(v[4 * j + t], d))));
            word |= (uint32_t)(q & 0xff) << (8 * t);
        }
        w[j] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(xq + 32 * b);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    xd[b] = d;
}

// general case: one warp per row, lanes over the row's blocks; per block the
// exact integer dot of the 32 codes (8 dp4a), scaled by d_w * d_x
constexpr int kWarps = 8;
__global__ void __launch_bounds__(kWarps * 32) q8_0_i8_gemv_kernel(const uint32_t* __restrict__ blocks,
                                                                   const int8_t* __restrict__ xq,
                                                                   const float* __restrict__ xd,
                                                                   float* __restrict__ out, int64_t N, int64_t K) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= N) return;
    const int64_t nb = K / 32;
    float acc = 0.f;
    for (int64_t b = lane; b < nb; b += 32) {
        const uint32_t* blk = blocks + (row * nb + b) * 9;
        const int* xw = reinterpret_cast<const int*>(xq + 32 * b);
        int dot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = __dp4a((int)__ldg(blk + 1 + i), __ldg(xw + i), dot);
        acc = fmaf(f16_bits_to_f32(__ldg(blk)) * __ldg(xd + b), (float)dot, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) out[row] = acc;
}

}  // namespace

cudaError_t launch_quantize_x_q8(const float* x, int8_t* xq, float* xd, int64_t K, cudaStream_t s) {
    const int64_t nblk = K / 32;
    if (nblk == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((nblk + 127) / 128);
    return launch_pdl(quantize_x_q8_kernel, dim3(grid), dim3(128), 0, s, x, xq, xd, nblk);
}

cudaError_t launch_q8_0_i8_gemv(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out, int64_t N,
                                int64_t K, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((N + kWarps - 1) / kWarps);
    return launch_pdl(q8_0_i8_gemv_kernel, dim3(grid), dim3(kWarps * 32), 0, s, blocks, xq, xd, out, N, K);
}

}  // namespace gai4
