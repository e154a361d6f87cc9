// Failure-detection self-test: one CTA waits on an mbarrier that nothing ever
// arrives on, with a short limit.  The bounded wait gives up, records the
// timeout in the plan's status word (read by wf_sync_status) and the kernel
// returns normally, so the context stays usable.  This is the same bounded
// wait every kernel of the library uses on its hot path.

#include "wf_internal.h"
#include "wf_ptx.cuh"

using namespace wfptx;

namespace {

__global__ void wait_probe_kernel(uint32_t *ctl, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 never completes: no thread arrives
        mbar_wait(smem_u32(&bar), 0, &abort_flag, ctl + WF_SCRATCH_STATUS / 4,
                  ctl + WF_SCRATCH_WHERE / 4, 99u, limit_ns);
    }
    __syncthreads();
}

}  // namespace

cudaError_t wf_launch_wait_probe(void *scratch, uint64_t limit_ns, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(static_cast<uint32_t *>(scratch), limit_ns);
    return cudaGetLastError();
}
