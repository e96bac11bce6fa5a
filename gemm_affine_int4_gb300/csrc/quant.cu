// quant.cu -- affine group quantize/pack, unpack and dequantize (sm_103a).
//
// Quantization (MLX PR "[Metal] Add staged affine_qmm_t_nax kernels with
// split-k", reproduction script mx.quantize(w, group_size, bits); bias = min,
// scale = (max - min) / (2^bits - 1)): one thread per (row, group). The binary32
// steps are IEEE-rounded (__fsub_rn / __fdiv_rn, rintf = round-half-even) and
// the codes are computed from the stored, T-rounded scale and bias, so the
// packed words are identical to any other correct binary32 implementation.
// Packing: the row is a little-endian bit stream, bit j of code k at stream
// bit k*bits + j (metaltile-std quantized.rs, mt_qmv: low nibble first).
// A group covers group_size*bits bits, a multiple of 32, so each thread owns
// whole words and no two threads write the same word.
#include "common.cuh"
#include "internal.h"

namespace gai4 {

template <typename T>
__device__ __forceinline__ float store_rounded(void* p, int64_t i, float v) {
    using St = typename T::storage;
    const St h = T::from_f32(v);
    static_cast<St*>(p)[i] = h;
    return T::to_f32(h);
}

template <typename T, int BITS, int GS>
__global__ void __launch_bounds__(128) quantize_kernel(const float* __restrict__ w, uint32_t* __restrict__ packed,
                                                       void* scales, void* biases, int64_t N, int64_t K) {
    constexpr unsigned L = (1u << BITS) - 1u;
    constexpr int WPG = GS * BITS / 32;   // words per group
    const int64_t G = K / GS;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N * G) return;
    const int64_t n = t / G, g = t - n * G;
    const float* wg = w + n * K + g * GS;

    float mn = wg[0], mx = wg[0];
    for (int i = 1; i < GS; ++i) {
        const float v = wg[i];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)L);
    const float s_st = store_rounded<T>(scales, t, s);
    const float b_st = store_rounded<T>(biases, t, mn);

    uint32_t words[WPG];
#pragma unroll
    for (int i = 0; i < WPG; ++i) words[i] = 0u;
#pragma unroll
    for (int i = 0; i < GS; ++i) {
        unsigned q = 0u;
        if (s_st != 0.0f) {
            const float r = rintf(__fdiv_rn(__fsub_rn(wg[i], b_st), s_st));
            q = r <= 0.0f ? 0u : (r >= (float)L ? L : (unsigned)r);
        }
        const int o = i * BITS, wi = o >> 5, sh = o & 31;
        words[wi] |= q << sh;
        if (sh + BITS > 32) words[wi + 1] |= q >> (32 - sh);
    }
    uint32_t* dst = packed + n * (K * BITS / 32) + g * WPG;
#pragma unroll
    for (int i = 0; i < WPG; ++i) dst[i] = words[i];
}

template <typename T, int BITS>
static cudaError_t launch_quantize_bits(const float* w, uint32_t* packed, void* scales, void* biases, int gs,
                                        int64_t N, int64_t K, cudaStream_t s) {
    const int64_t threads = N * (K / gs);
    const unsigned blocks = (unsigned)((threads + 127) / 128);
    switch (gs) {
    case 32: quantize_kernel<T, BITS, 32><<<blocks, 128, 0, s>>>(w, packed, scales, biases, N, K); break;
    case 64: quantize_kernel<T, BITS, 64><<<blocks, 128, 0, s>>>(w, packed, scales, biases, N, K); break;
    default: quantize_kernel<T, BITS, 128><<<blocks, 128, 0, s>>>(w, packed, scales, biases, N, K); break;
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_quantize_t(const float* w, uint32_t* packed, void* scales, void* biases, int bits,
                                     int gs, int64_t N, int64_t K, cudaStream_t s) {
    switch (bits) {
    case 2: return launch_quantize_bits<T, 2>(w, packed, scales, biases, gs, N, K, s);
    case 3: return launch_quantize_bits<T, 3>(w, packed, scales, biases, gs, N, K, s);
    case 4: return launch_quantize_bits<T, 4>(w, packed, scales, biases, gs, N, K, s);
    case 6: return launch_quantize_bits<T, 6>(w, packed, scales, biases, gs, N, K, s);
    default: return launch_quantize_bits<T, 8>(w, packed, scales, biases, gs, N, K, s);
    }
}

cudaError_t launch_quantize(const float* w, uint32_t* packed, void* scales, void* biases, int dtype, int bits,
                            int gs, int64_t N, int64_t K, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    switch (dtype) {
    case GAI4_F32: return launch_quantize_t<F32>(w, packed, scales, biases, bits, gs, N, K, s);
    case GAI4_F16: return launch_quantize_t<F16>(w, packed, scales, biases, bits, gs, N, K, s);
    default: return launch_quantize_t<BF16>(w, packed, scales, biases, bits, gs, N, K, s);
    }
}

// code k of a row (bit stream)
__device__ __forceinline__ unsigned code_of(const uint32_t* row, int64_t k, int bits) {
    const int64_t o = k * bits;
    const int64_t wi = o >> 5;
    const int sh = (int)(o & 31);
    uint32_t v = row[wi] >> sh;
    if (sh + bits > 32) v |= row[wi + 1] << (32 - sh);
    return v & ((1u << bits) - 1u);
}

__global__ void unpack_kernel(const uint32_t* __restrict__ packed, uint8_t* __restrict__ q, int bits, int64_t N,
                              int64_t K) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N * K) return;
    const int64_t n = t / K, k = t - n * K;
    q[t] = (uint8_t)code_of(packed + n * (K * bits / 32), k, bits);
}

cudaError_t launch_unpack(const uint32_t* packed, uint8_t* q, int bits, int64_t N, int64_t K, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((N * K + 255) / 256);
    unpack_kernel<<<blocks, 256, 0, s>>>(packed, q, bits, N, K);
    return cudaGetLastError();
}

template <typename T>
__global__ void dequantize_kernel(const uint32_t* __restrict__ packed, const typename T::storage* __restrict__ sc,
                                  const typename T::storage* __restrict__ bi, float* __restrict__ out, int bits,
                                  int gs, int64_t N, int64_t K) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N * K) return;
    const int64_t n = t / K, k = t - n * K;
    const int64_t gi = n * (K / gs) + k / gs;
    const float q = (float)code_of(packed + n * (K * bits / 32), k, bits);
    out[t] = fmaf(T::to_f32(sc[gi]), q, T::to_f32(bi[gi]));   // one rounding of s*q + b
}

cudaError_t launch_dequantize(const uint32_t* packed, const void* scales, const void* biases, float* out,
                              int dtype, int bits, int gs, int64_t N, int64_t K, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((N * K + 255) / 256);
    switch (dtype) {
    case GAI4_F32:
        dequantize_kernel<F32><<<blocks, 256, 0, s>>>(packed, (const float*)scales, (const float*)biases, out, bits,
                                                      gs, N, K);
        break;
    case GAI4_F16:
        dequantize_kernel<F16><<<blocks, 256, 0, s>>>(packed, (const uint16_t*)scales, (const uint16_t*)biases, out,
                                                      bits, gs, N, K);
        break;
    default:
        dequantize_kernel<BF16><<<blocks, 256, 0, s>>>(packed, (const uint16_t*)scales, (const uint16_t*)biases,
                                                       out, bits, gs, N, K);
        break;
    }
    return cudaGetLastError();
}

}  // namespace gai4
