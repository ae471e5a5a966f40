// Self-test of the bounded waits every kernel of this library relies on.
//
// Each CTA's lane 0 waits on an mbarrier that nothing arrives on.  The wait
// gives up after about 2^31 cycles (about a second) and sets
// PKV_STATUS_TIMEOUT; every other CTA sees that bit while it polls and gives
// up at once, so the launch ends in about one wait, not one per CTA.  Then the
// CTA completes its barrier's phase itself and checks that the drain wait
// (the one a kernel uses for its own copies after a timeout) returns true.
// No copy, MMA or tensor memory is involved: nothing is left in flight.
#include <cuda_runtime.h>
#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"
#include "pkv_kernels.h"
#include "tc_common.cuh"

namespace {

using namespace pkv_tc;

__global__ void selftest_bounded_wait_kernel(unsigned int* status, unsigned int* drained)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(smem_u32(&bar), 0, status)) atomicOr(status, PKV_STATUS_TIMEOUT);
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar)) : "memory");
        if (mbar_drain_wait(smem_u32(&bar), 0)) atomicAdd(drained, 1u);
    }
}

}  // namespace

extern "C" int pkv_selftest_bounded_wait(int num_ctas, unsigned int* drained, void* stream)
{
    if (num_ctas <= 0 || num_ctas > 65535)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_selftest_bounded_wait: num_ctas %d", num_ctas);
    if (!drained) return pkv_fail(PKV_ERR_NULL, "pkv_selftest_bounded_wait: NULL counter");
    unsigned int* status = pkv_status_word_ptr();
    if (!status) return pkv_fail(PKV_ERR_CUDA, "pkv_selftest_bounded_wait: no status word");
    selftest_bounded_wait_kernel<<<num_ctas, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, drained);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : pkv_fail(PKV_ERR_CUDA, "pkv_selftest_bounded_wait: %s",
                                                cudaGetErrorString(e));
}
