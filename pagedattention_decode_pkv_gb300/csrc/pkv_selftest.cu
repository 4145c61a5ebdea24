// Failure detection self-test: the bounded mbarrier wait that every pipeline
// stage of the attention kernels uses, run on a barrier that nothing completes.
// The wait ends at its deadline, the kernel records PKV_ERRBIT_TIMEOUT in the
// caller's flag and returns, and the context stays usable.  Nothing faults,
// traps or spins without a bound.
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_internal.h"
#include "pkv_tma.cuh"

namespace pkv {
namespace {

constexpr uint32_t kMaxSelftestTimeoutUs = 1000000;  // one second at most

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t *err_flag, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one arrival would complete phase 0; none comes
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const uint64_t deadline = global_ns() + timeout_ns;
    const bool done = mbar_wait(b, 0, deadline);
    if (!done && threadIdx.x == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_selftest_wait_timeout(int32_t *err_flag, uint32_t timeout_us, void *stream) {
    if (!err_flag) return set_error(PKV_ERR_INVALID_ARG, "selftest: NULL err_flag");
    if (!aligned(err_flag, 4)) return set_error(PKV_ERR_INVALID_ARG, "selftest: err_flag not 4-byte aligned");
    if (timeout_us == 0 || timeout_us > kMaxSelftestTimeoutUs)
        return set_error(PKV_ERR_INVALID_ARG, "selftest: timeout must be in (0, %u] us", kMaxSelftestTimeoutUs);
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err_flag,
                                                                      static_cast<uint64_t>(timeout_us) * 1000u);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
    return ok();
}
