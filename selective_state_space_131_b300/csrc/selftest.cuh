// selftest.cuh -- a self-test of the failure detection of libm3scan: the
// bounded mbarrier wait every kernel here uses, made to run out on purpose.
// One thread waits on an mbarrier that nothing arrives at; when its cycle
// budget is spent it records a wait timeout in the device status word and
// the kernel returns, so the context stays usable.  Nothing faults, traps or
// spins without bound.
#pragma once

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace m3 {

__global__ void m3_wait_probe_kernel(long long budget_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // phase 0 never completes: no thread arrives and no copy is pending
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, budget_cycles)) set_status(kStatusWaitTimeout);
}

}  // namespace m3
