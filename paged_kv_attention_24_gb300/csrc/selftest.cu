// Self-test of the bounded wait that every kernel of this library uses.
//
// One thread initialises an mbarrier that nothing will ever arrive at and
// waits on it with ptx::mbar_wait and a small clock budget.  The wait must
// give up and report MSGL_DEVERR_TIMEOUT in the status word; the kernel then
// returns normally, so the context stays usable.  This is how a lost arrival
// inside a real kernel surfaces (as a status bit, never a hang or a trap).
#include "kernels.h"
#include "ptx.cuh"

namespace msgl {
namespace {

__global__ void wait_timeout_kernel(uint32_t *status, long long budget) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    if (!ptx::mbar_wait(b, 0, budget)) report(status, MSGL_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace msgl

extern "C" msgl_status msgl_selftest_wait_timeout(uint32_t *status, int64_t budget_cycles,
                                                  msgl_stream_t stream) {
    if (!status || budget_cycles <= 0 || budget_cycles > 4000000000LL) {
        msgl::set_last_error("selftest: need a status word and 0 < budget_cycles <= 4e9");
        return MSGL_ERR_INVALID_ARG;
    }
    msgl::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, (long long)budget_cycles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        msgl::set_last_error(cudaGetErrorString(e));
        return MSGL_ERR_CUDA;
    }
    return MSGL_OK;
}
