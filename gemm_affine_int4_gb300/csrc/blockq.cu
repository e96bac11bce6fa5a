// blockq.cu -- Q8_0 and Q4_K block-quantized matrix-vector products (sm_103a,
// CUDA cores; the work is HBM-bound, so no tensor-core reshaping).
//
// Q8_0 (hanzo-kernel quant.rs, matvec_q8 and "Q8_0 PACKED matvec"): a block is
// 9 words -- f16 scale d in the low half of word 0, then 32 signed int8 codes,
// four per word, byte 0 first; out[n] = sum_b d_b * sum_j q_j x_{32b+j}.
// Q4_K (hanzo-kernel quant.rs, Q4_K section, matvec_q4k, get_scale_min_k4):
// a 144-byte super-block of 256 weights -- d, dmin (f16), 12 bytes of eight
// 6-bit (sc, m) pairs, 128 bytes of 4-bit codes; for g < 4, i < 32 and
// qb = qs[32g + i], weight 64g + i is d*sc_{2g}*(qb & 15) - dmin*m_{2g} and
// weight 64g + 32 + i is d*sc_{2g+1}*(qb >> 4) - dmin*m_{2g+1}.
//
// Both kernels share the structure of the affine GEMV: a lane owns one
// 32-weight chunk per iteration (a Q8_0 block; a quarter of a Q4_K group:
// 16 low and 16 high nibbles of one 16-byte run of qs), a warp works on R rows
// with one activation fragment, the binary32 activations are staged once per
// K slab in shared memory in a lane-interleaved order together with per-chunk
// sums, and the per-chunk scale is applied to sum q x recovered from the
// "constant + code" trick (a code placed in the mantissa of a power of two).
#include "common.cuh"
#include "internal.h"

namespace gai4 {

namespace {

constexpr int kNW = 8;              // warps per CTA
constexpr int kXBudget = 64 * 1024; // bytes of staged activations per CTA

// ---------------------------------------------------------------------------
// Q8_0
// ---------------------------------------------------------------------------

// byte t of w (two's complement code q) -> the float q, exactly: first
// 384 + q (exponent of 256, mantissa bits 15..22 = q + 128 = byte ^ 0x80),
// then 384 subtracted (exact). Every product q x is exact before it is summed.
template <int t>
__device__ __forceinline__ float q8_val(uint32_t w) {
    constexpr int d = 15 - 8 * t;
    const uint32_t v = d >= 0 ? (w << (d >= 0 ? d : 0)) : (w >> (d < 0 ? -d : 0));
    return __uint_as_float((v & 0x007F8000u) ^ 0x43C00000u) - 384.0f;
}

template <int R>
__global__ void __launch_bounds__(kNW * 32) q8_0_gemv_kernel(const uint32_t* __restrict__ blocks,
                                                             const float* __restrict__ x, float* __restrict__ out,
                                                             int64_t N, int64_t K, int S, int KS) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    constexpr int PPC = 8;   // 16-byte pieces of activations per 32-element chunk
    const int KSP = (KS + 1023) / 1024 * 1024;   // whole warp iterations (32 chunks)
    extern __shared__ uint4 smem[];
    const int Gw = kNW / S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp / S, s = warp % S;
    const int64_t row0 = (int64_t)blockIdx.x * (Gw * R) + (int64_t)g * R;
    const int64_t nb = K / 32;
    uint4* x_sm = smem;
    float* xsum_sm = reinterpret_cast<float*>(smem + KSP / 4);
    float* red_sm = xsum_sm + KSP / 32;

    float part[R];
#pragma unroll
    for (int r = 0; r < R; ++r) part[r] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += KS) {
        const int kslab = (int)min((int64_t)KS, K - k0);
        const int nch = kslab / 32, npieces = kslab / 4;
        __syncthreads();
        for (int p = threadIdx.x; p < npieces; p += kNW * 32) {
            const int c = p / PPC, j = p - c * PPC;
            x_sm[((c >> 5) * PPC + j) * 32 + (c & 31)] = *reinterpret_cast<const uint4*>(x + k0 + 4 * (int64_t)p);
        }
        __syncthreads();
        for (int c = threadIdx.x; c < nch; c += kNW * 32) {
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < PPC; ++j) {
                const uint4 v = x_sm[((c >> 5) * PPC + j) * 32 + (c & 31)];
                sum += __uint_as_float(v.x) + __uint_as_float(v.y) + __uint_as_float(v.z) + __uint_as_float(v.w);
            }
            xsum_sm[c] = sum;
        }
        __syncthreads();

        const int its = (nch + 31) >> 5;
        const int64_t gc0 = k0 / 32;
        uint32_t wn[R][9];
        auto load_it = [&](int it) {
            const int c = it * 32 + lane;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (c < nch && row < N) {
                    const uint32_t* b = blocks + (row * nb + gc0 + c) * 9;
#pragma unroll
                    for (int i = 0; i < 9; ++i) wn[r][i] = __ldg(b + i);
                } else {
#pragma unroll
                    for (int i = 0; i < 9; ++i) wn[r][i] = 0u;
                }
            }
        };
        if (s < its) load_it(s);
        for (int it = s; it < its; it += S) {
            uint32_t wc[R][9];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int i = 0; i < 9; ++i) wc[r][i] = wn[r][i];
            if (it + S < its) load_it(it + S);
            const int c = it * 32 + lane;
            if (c < nch) {
                float xr[32];
#pragma unroll
                for (int j = 0; j < PPC; ++j) {
                    const uint4 v = x_sm[(it * PPC + j) * 32 + lane];
                    xr[4 * j + 0] = __uint_as_float(v.x);
                    xr[4 * j + 1] = __uint_as_float(v.y);
                    xr[4 * j + 2] = __uint_as_float(v.z);
                    xr[4 * j + 3] = __uint_as_float(v.w);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t w = wc[r][1 + i];
                        acc = fmaf(q8_val<0>(w), xr[4 * i + 0], acc);
                        acc = fmaf(q8_val<1>(w), xr[4 * i + 1], acc);
                        acc = fmaf(q8_val<2>(w), xr[4 * i + 2], acc);
                        acc = fmaf(q8_val<3>(w), xr[4 * i + 3], acc);
                    }
                    const float d = f16_bits_to_f32(wc[r][0]);
                    part[r] = fmaf(d, acc, part[r]);
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float v = warp_sum(part[r]);
        if (lane == 0) red_sm[warp * R + r] = v;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < Gw * R; t += kNW * 32) {
        const int gg = t / R, r = t - gg * R;
        float v = 0.f;
        for (int ss = 0; ss < S; ++ss) v += red_sm[(gg * S + ss) * R + r];
        const int64_t row = (int64_t)blockIdx.x * (Gw * R) + (int64_t)gg * R + r;
        if (row < N) out[row] = v;
    }
}

// ---------------------------------------------------------------------------
// Q4_K
// ---------------------------------------------------------------------------

// nibble at bits [p, p+4) of w -> the float q, exactly: first 16 + q
// (exponent of 16, code in mantissa bits 19..22), then 16 subtracted (exact)
template <int p>
__device__ __forceinline__ float q4_val(uint32_t w) {
    constexpr int d = 19 - p;
    const uint32_t v = d >= 0 ? (w << (d >= 0 ? d : 0)) : (w >> (d < 0 ? -d : 0));
    return __uint_as_float((v & 0x00780000u) | 0x41800000u) - 16.0f;
}

__device__ __forceinline__ uint32_t byte_of(uint32_t b0, uint32_t b1, uint32_t b2, int i) {
    const uint32_t w = i < 4 ? b0 : (i < 8 ? b1 : b2);
    return (w >> (8 * (i & 3))) & 0xffu;
}

// (sc, m) of sub-block j from the 12 scale bytes (held in three words)
__device__ __forceinline__ void q4k_scale_min(uint32_t b0, uint32_t b1, uint32_t b2, int j, float& sc, float& m) {
    uint32_t s_, m_;
    if (j < 4) {
        s_ = byte_of(b0, b1, b2, j) & 63u;
        m_ = byte_of(b0, b1, b2, j + 4) & 63u;
    } else {
        const uint32_t hi = byte_of(b0, b1, b2, j + 4);
        s_ = (hi & 15u) | ((byte_of(b0, b1, b2, j - 4) >> 6) << 4);
        m_ = (hi >> 4) | ((byte_of(b0, b1, b2, j) >> 6) << 4);
    }
    sc = (float)s_;
    m = (float)m_;
}

// Activation permutation: chunk c = 8*block + u (u = 2g + h) owns the 16 low
// nibbles (weights 64g + 16h + t) and the 16 high nibbles (64g + 32 + 16h + t),
// t < 16, of qs bytes [32g + 16h, 32g + 16h + 16). Piece j < 4 of the chunk
// holds low-run elements 4j..4j+3, piece 4 + j the high-run ones.
__device__ __forceinline__ void q4k_piece_slot(int p, int& c, int& j) {
    const int k = 4 * p;
    const int blk = k >> 8, e = k & 255;
    const int g = e >> 6, r = e & 63;
    const int hi = r >> 5, t = r & 31;
    const int h = t >> 4, tt = t & 15;
    c = blk * 8 + 2 * g + h;
    j = hi * 4 + (tt >> 2);
}

template <int R>
__global__ void __launch_bounds__(kNW * 32) q4_k_gemv_kernel(const uint8_t* __restrict__ blocks,
                                                             const float* __restrict__ x, float* __restrict__ out,
                                                             int64_t N, int64_t K, int S, int KS) {
    pdl_launch_dependents();
    pdl_wait();   // the kernels before this one are complete: global memory may be read
    constexpr int PPC = 8;
    const int KSP = (KS + 1023) / 1024 * 1024;   // whole warp iterations (32 chunks)
    extern __shared__ uint4 smem[];
    const int Gw = kNW / S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp / S, s = warp % S;
    const int64_t row0 = (int64_t)blockIdx.x * (Gw * R) + (int64_t)g * R;
    const int64_t nb = K / 256;
    uint4* x_sm = smem;
    float* xlo_sm = reinterpret_cast<float*>(smem + KSP / 4);
    float* xhi_sm = xlo_sm + KSP / 32;
    float* red_sm = xhi_sm + KSP / 32;

    float part[R];
#pragma unroll
    for (int r = 0; r < R; ++r) part[r] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += KS) {
        const int kslab = (int)min((int64_t)KS, K - k0);
        const int nch = kslab / 32, npieces = kslab / 4;
        __syncthreads();
        for (int p = threadIdx.x; p < npieces; p += kNW * 32) {
            int c, j;
            q4k_piece_slot(p, c, j);
            x_sm[((c >> 5) * PPC + j) * 32 + (c & 31)] = *reinterpret_cast<const uint4*>(x + k0 + 4 * (int64_t)p);
        }
        __syncthreads();
        for (int c = threadIdx.x; c < nch; c += kNW * 32) {
            float lo = 0.f, hi = 0.f;
#pragma unroll
            for (int j = 0; j < PPC; ++j) {
                const uint4 v = x_sm[((c >> 5) * PPC + j) * 32 + (c & 31)];
                const float t = __uint_as_float(v.x) + __uint_as_float(v.y) + __uint_as_float(v.z) +
                                __uint_as_float(v.w);
                if (j < 4) lo += t;
                else hi += t;
            }
            xlo_sm[c] = lo;
            xhi_sm[c] = hi;
        }
        __syncthreads();

        const int its = (nch + 31) >> 5;
        const int64_t gc0 = k0 / 32;
        uint4 hn[R], qn[R];
        auto load_it = [&](int it) {
            const int c = it * 32 + lane;
            const int64_t gc = gc0 + c;
            const int64_t blk = gc >> 3;
            const int u = (int)(gc & 7);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = row0 + r;
                if (c < nch && row < N) {
                    const uint8_t* b = blocks + (row * nb + blk) * 144;
                    hn[r] = __ldg(reinterpret_cast<const uint4*>(b));
                    qn[r] = ld_stream_v4(b + 16 + 16 * u);
                } else {
                    hn[r] = make_uint4(0u, 0u, 0u, 0u);
                    qn[r] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        };
        if (s < its) load_it(s);
        for (int it = s; it < its; it += S) {
            uint4 hc[R], qc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                hc[r] = hn[r];
                qc[r] = qn[r];
            }
            if (it + S < its) load_it(it + S);
            const int c = it * 32 + lane;
            if (c < nch) {
                const int u = (int)((gc0 + c) & 7);
                const int j_lo = 2 * (u >> 1);   // sub-block of the low nibbles: 2g
                float xr[32];
#pragma unroll
                for (int j = 0; j < PPC; ++j) {
                    const uint4 v = x_sm[(it * PPC + j) * 32 + lane];
                    xr[4 * j + 0] = __uint_as_float(v.x);
                    xr[4 * j + 1] = __uint_as_float(v.y);
                    xr[4 * j + 2] = __uint_as_float(v.z);
                    xr[4 * j + 3] = __uint_as_float(v.w);
                }
                const float xlo = xlo_sm[c], xhi = xhi_sm[c];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t q[4] = {qc[r].x, qc[r].y, qc[r].z, qc[r].w};
                    float alo = 0.f, ahi = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        alo = fmaf(q4_val<0>(q[i]), xr[4 * i + 0], alo);
                        alo = fmaf(q4_val<8>(q[i]), xr[4 * i + 1], alo);
                        alo = fmaf(q4_val<16>(q[i]), xr[4 * i + 2], alo);
                        alo = fmaf(q4_val<24>(q[i]), xr[4 * i + 3], alo);
                        ahi = fmaf(q4_val<4>(q[i]), xr[16 + 4 * i + 0], ahi);
                        ahi = fmaf(q4_val<12>(q[i]), xr[16 + 4 * i + 1], ahi);
                        ahi = fmaf(q4_val<20>(q[i]), xr[16 + 4 * i + 2], ahi);
                        ahi = fmaf(q4_val<28>(q[i]), xr[16 + 4 * i + 3], ahi);
                    }
                    const float d = f16_bits_to_f32(hc[r].x);
                    const float dmin = f16_bits_to_f32(hc[r].x >> 16);
                    float sc_lo, m_lo, sc_hi, m_hi;
                    q4k_scale_min(hc[r].y, hc[r].z, hc[r].w, j_lo, sc_lo, m_lo);
                    q4k_scale_min(hc[r].y, hc[r].z, hc[r].w, j_lo + 1, sc_hi, m_hi);
                    const float qx_lo = alo, qx_hi = ahi;   // sums of exact products q x
                    float v = part[r];
                    v = fmaf(d * sc_lo, qx_lo, v);
                    v = fmaf(-(dmin * m_lo), xlo, v);
                    v = fmaf(d * sc_hi, qx_hi, v);
                    v = fmaf(-(dmin * m_hi), xhi, v);
                    part[r] = v;
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float v = warp_sum(part[r]);
        if (lane == 0) red_sm[warp * R + r] = v;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < Gw * R; t += kNW * 32) {
        const int gg = t / R, r = t - gg * R;
        float v = 0.f;
        for (int ss = 0; ss < S; ++ss) v += red_sm[(gg * S + ss) * R + r];
        const int64_t row = (int64_t)blockIdx.x * (Gw * R) + (int64_t)gg * R + r;
        if (row < N) out[row] = v;
    }
}

constexpr int kRows = 4;   // rows per warp

int pick_ksplit(int64_t N, int64_t its_total) {
    int S = 1;
    const int64_t target = 4LL * num_sms();
    while (S < kNW && 2 * S <= its_total && (N + (kNW / S) * kRows - 1) / ((kNW / S) * kRows) < target) S *= 2;
    return S;
}

template <typename KernelT>
cudaError_t set_smem(KernelT k) {
    static unsigned long long configured = 0ull;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && (configured & (1ull << dev))) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
    if (e == cudaSuccess && dev < 64) configured |= 1ull << dev;
    return e;
}

// Test aid: as q4_k_dequant_tma_kernel, with q4k_scale_min, the decoder of
// q4_k_gemv_kernel
__global__ void q4_k_dequant_general_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ out,
                                            int64_t nblk) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nblk * 4) return;
    const int64_t b = t >> 2;
    const int g = (int)(t & 3);
    const uint8_t* blk = blocks + b * 144;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    float sc_lo, m_lo, sc_hi, m_hi;
    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g, sc_lo, m_lo);
    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g + 1, sc_hi, m_hi);
    float* o = out + b * 256 + 64 * g;
    for (int i = 0; i < 32; ++i) {
        const uint32_t qb = blk[16 + 32 * g + i];
        o[i] = fmaf(d * sc_lo, (float)(qb & 15u), -(dmin * m_lo));
        o[32 + i] = fmaf(d * sc_hi, (float)(qb >> 4), -(dmin * m_hi));
    }
}

}  // namespace

cudaError_t launch_q4_k_dequant_general(const uint8_t* blocks, float* out, int64_t nblk, cudaStream_t s) {
    const int64_t threads = nblk * 4;
    q4_k_dequant_general_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(blocks, out, nblk);
    return cudaGetLastError();
}

cudaError_t launch_q8_0_gemv(const uint32_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                             cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    int64_t ks_max = kXBudget / 4;
    ks_max -= ks_max % 1024;
    const int KS = (int)(K <= ks_max ? K : ks_max);
    const int64_t its_total = (K / 32 + 31) / 32;
    const int S = pick_ksplit(N, its_total);
    const int rows_per_cta = (kNW / S) * kRows;
    const int KSP = (KS + 1023) / 1024 * 1024;
    const size_t smem = (size_t)KSP * 4 + (size_t)(KSP / 32) * 4 + (size_t)kNW * kRows * 4;
    cudaError_t e = set_smem(q8_0_gemv_kernel<kRows>);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((N + rows_per_cta - 1) / rows_per_cta);
    return launch_pdl(q8_0_gemv_kernel<kRows>, dim3(grid), dim3(kNW * 32), smem, s, blocks, x, out, N, K, S, KS);
}

cudaError_t launch_q4_k_gemv(const uint8_t* blocks, const float* x, float* out, int64_t N, int64_t K,
                             cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    int64_t ks_max = kXBudget / 4;
    ks_max -= ks_max % 1024;
    const int KS = (int)(K <= ks_max ? K : ks_max);
    const int64_t its_total = (K / 32 + 31) / 32;
    const int S = pick_ksplit(N, its_total);
    const int rows_per_cta = (kNW / S) * kRows;
    const int KSP = (KS + 1023) / 1024 * 1024;
    const size_t smem = (size_t)KSP * 4 + (size_t)(KSP / 32) * 8 + (size_t)kNW * kRows * 4;
    cudaError_t e = set_smem(q4_k_gemv_kernel<kRows>);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((N + rows_per_cta - 1) / rows_per_cta);
    return launch_pdl(q4_k_gemv_kernel<kRows>, dim3(grid), dim3(kNW * 32), smem, s, blocks, x, out, N, K, S, KS);
}

}  // namespace gai4
