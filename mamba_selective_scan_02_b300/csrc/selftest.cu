// selftest.cu — the device-side failure path of the chained scans, run on its
// own: one thread waits, with the same bounded wait the chained hand-offs use
// (wait_flag), for a flag that nothing sets, and records SSM_ERR_TIMEOUT in the
// workspace status word when the poll limit runs out.  Nothing faults or
// hangs; the context stays usable.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

__global__ void flag_wait_selftest_kernel(int *status, const int *flag, int polls) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && !wait_flag(flag, 1, polls))
        record_error(status, 4 /* SSM_ERR_TIMEOUT */);
}

cudaError_t flag_wait_selftest_launch(int *status, const int *flag, int polls, cudaStream_t st) {
    flag_wait_selftest_kernel<<<1, 32, 0, st>>>(status, flag, polls);
    return cudaGetLastError();
}

}  // namespace ssm
