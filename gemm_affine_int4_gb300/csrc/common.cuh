// common.cuh -- shared device helpers of the sm_103a kernels (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gai4.h"

namespace gai4 {

// ---------------------------------------------------------------------------
// Programmatic dependent launch. The hot-path kernels are launched so that
// the next kernel in the stream may start (its launch and set-up: barriers,
// tensor-memory allocation) while this one finishes: every kernel lets its
// dependents be scheduled at entry, and waits for the kernels before it to
// complete -- with their memory visible -- before it reads activations or
// writes any output or workspace. The streaming GEMV / GEMM kernels read the
// packed weights (which no kernel of the library writes, and no kernel that
// does not signal programmatic launch can still be writing) before that
// wait. A kernel that reads another call's output is therefore ordered
// exactly as with plain stream order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// dtype traits: storage type, conversion to/from binary32
// ---------------------------------------------------------------------------
struct BF16 {
    using storage = uint16_t;
    static constexpr int kBytes = 2;
    static constexpr bool kIsBF16 = true;
    // 16-bit magic for the code -> value trick: bit pattern of 128.0 (bf16 has
    // 7 stored mantissa bits, so 128 + q is exact for q < 128)
    static constexpr uint32_t kMagic16 = 0x4300u;
    __device__ __forceinline__ static float to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
    __device__ __forceinline__ static uint16_t from_f32(float f) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
};

struct F16 {
    using storage = uint16_t;
    static constexpr int kBytes = 2;
    static constexpr bool kIsBF16 = false;
    // bit pattern of 1024.0 (10 stored mantissa bits: 1024 + q exact for q < 1024)
    static constexpr uint32_t kMagic16 = 0x6400u;
    __device__ __forceinline__ static float to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }
    __device__ __forceinline__ static uint16_t from_f32(float f) { return __half_as_ushort(__float2half_rn(f)); }
};

struct F32 {
    using storage = float;
    static constexpr int kBytes = 4;
    static constexpr bool kIsBF16 = false;
    __device__ __forceinline__ static float to_f32(float f) { return f; }
    __device__ __forceinline__ static float from_f32(float f) { return f; }
};

// ---------------------------------------------------------------------------
// mixed-precision multiply-add: binary32 += T16 x T16 with a half-word select
// (sm_100+ fma.rn.f32.{bf16,f16}); HA / HB pick the low (0) or high (1) half
// of each 32-bit operand.
// ---------------------------------------------------------------------------
template <typename T, int HA, int HB>
__device__ __forceinline__ float fma_mix(uint32_t a2, uint32_t b2, float c) {
    float d;
    if constexpr (T::kIsBF16) {
        if constexpr (HA == 0 && HB == 0)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.bf16 %0, a0, b0, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else if constexpr (HA == 0 && HB == 1)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.bf16 %0, a0, b1, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else if constexpr (HA == 1 && HB == 0)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.bf16 %0, a1, b0, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.bf16 %0, a1, b1, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    } else {
        if constexpr (HA == 0 && HB == 0)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.f16 %0, a0, b0, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else if constexpr (HA == 0 && HB == 1)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.f16 %0, a0, b1, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else if constexpr (HA == 1 && HB == 0)
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.f16 %0, a1, b0, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
        else
            asm("{.reg .b16 a0,a1,b0,b1; mov.b32 {a0,a1}, %1; mov.b32 {b0,b1}, %2; fma.rn.f32.f16 %0, a1, b1, %3;}"
                : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    }
    return d;
}

// ---------------------------------------------------------------------------
// streaming loads of read-only weights: no L1 allocation, 256-byte L2 prefetch
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// f16 bit pattern (low 16 bits) -> binary32, all classes
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

}  // namespace gai4
