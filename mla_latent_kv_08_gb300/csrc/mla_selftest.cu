// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing
// arrives on; the wait gives up after the given time, records the timeout flag
// and the kernel returns, exactly as an attention kernel's stuck wait would.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace selftest {

using namespace ptx;

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t *status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int32_t abort_flag;
    if (threadIdx.x == 0) {
        *status = 0;
        abort_flag = 0;
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, status, FLAG_TIMEOUT, timeout_ns);
    __syncwarp();
}

}  // namespace selftest
}  // namespace mla

extern "C" mla_status mla_selftest_wait_timeout(uint64_t timeout_ns, int32_t *status, void *stream) {
    if (status == nullptr || timeout_ns < 1000ull || timeout_ns > 100000000ull) return MLA_ERR_INVALID;
    mla::selftest::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
