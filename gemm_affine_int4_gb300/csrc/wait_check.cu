// wait_check.cu -- gai4_check_bounded_wait: runs the bounded mbarrier wait
// that every asynchronous-copy kernel of this library uses (pipe::mbar_wait)
// on a barrier whose phase either completes (arrive != 0) or is never
// completed by anyone (arrive == 0), so that the time-out path -- give up
// after a bounded number of cycles, raise the shared abort flag, record
// GAI4_ERR_TIMEOUT in a status word, return -- can be exercised on a GPU
// without a fault, a trap or a hang. No copies are in flight in this kernel,
// so nothing has to be drained after the wait gives up.
#include <stdint.h>

#include "common.cuh"
#include "pipeline.cuh"

namespace gai4 {
namespace {

// one warp: lane 0 initialises the barrier (arrival count 1) and, when asked,
// arrives on it; every lane then waits for phase 0 with the given limit
__global__ void bounded_wait_kernel(int arrive, long long limit, int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        pipe::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) pipe::mbar_arrive(&bar);
    const pipe::Ctl c{status, limit, &abort_flag};
    (void)pipe::mbar_wait(&bar, 0, c);
    __syncthreads();
}

}  // namespace
}  // namespace gai4

extern "C" {

gai4_status gai4_check_bounded_wait(int arrive, int64_t limit_cycles, int* status, void* stream) {
    if (!status || limit_cycles <= 0 || limit_cycles > 4000000000LL) return GAI4_ERR_INVALID_ARG;
    if (((uintptr_t)status & 3u) != 0) return GAI4_ERR_MISALIGNED;
    gai4::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(arrive, (long long)limit_cycles, status);
    return cudaGetLastError() == cudaSuccess ? GAI4_OK : GAI4_ERR_CUDA;
}

}  // extern "C"
