// pipeline.cuh -- mbarrier, TMA and bounded-wait helpers shared by the
// asynchronous-copy kernels (internal).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/gai4.h"

namespace gai4 {
namespace pipe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A loop-invariant operand held in a register for the whole loop. Values that
// come from kernel parameters are otherwise re-read from the constant bank
// with one move instruction per use (a logic op takes at most one such
// operand); a warp shuffle result cannot be re-derived that way. The calling
// warp must be converged.
__device__ __forceinline__ uint32_t pin_reg(uint32_t v) { return __shfl_sync(0xffffffffu, v, 0); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

#ifndef GAI4_WAIT_HINT
#define GAI4_WAIT_HINT 1
#endif

// try_wait that may suspend the thread until the phase completes (or about
// `ns` nanoseconds pass): a waiting warp then issues almost no instructions
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

struct Ctl {
    int* status;            // device status word
    long long limit;        // clock64 cycles a single wait may take
    volatile int* abort_;   // shared flag: some role gave up
};

// bounded wait: false after `limit` cycles (or when another role gave up)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!(GAI4_WAIT_HINT ? mbar_try_wait_hint(bar, parity, 0x10000u) : mbar_try_wait(bar, parity))) {
        if (*c.abort_) return false;
        if (clock64() - t0 > c.limit) {
            *c.abort_ = 1;
            atomicExch(c.status, (int)GAI4_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// bounded wait that ignores the abort flag: used to drain copies and MMAs that
// were already issued, so that no asynchronous write lands after the CTA exits
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, long long limit, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            atomicExch(status, (int)GAI4_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// warp-uniform wait: every lane observes the phase itself (each lane's own
// acquire makes the asynchronously written data visible to it), then the warp
// reconverges (the following tcgen05 .sync.aligned instructions need every
// lane, converged) and agrees on the outcome
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Ctl& c) {
    const bool ok = mbar_wait(bar, parity, c);
    __syncwarp();
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// L2 prefetch of a contiguous byte range (16-byte aligned start, a multiple of
// 16 bytes), in pieces of at most 32 KB. It only warms the coherent L2, so it
// may be issued before the kernels this one depends on have completed; issued
// before the weight copies, it puts the activations at the head of the DRAM
// queue.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    const char* c = static_cast<const char*>(p);
    for (uint32_t o = 0; o < bytes; o += 32768u) {
        const uint32_t n = bytes - o < 32768u ? bytes - o : 32768u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"(n) : "memory");
    }
}

}  // namespace pipe

// cuTensorMapEncodeTiled from the driver, found through the runtime (no -lcuda)
static inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace gai4
