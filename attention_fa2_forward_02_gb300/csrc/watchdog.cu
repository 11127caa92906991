// watchdog.cu - exercises the kernels' bounded-wait path on purpose.
//
// One thread initialises an mbarrier that expects one arrival nobody makes and
// waits on it with the same time-bounded wait every pipeline wait in the
// library uses.  After the wait limit (about one second) the wait gives up,
// raises the CTA's abort flag and records the timeout in the device watchdog
// word; the kernel then returns normally.  fa2_device_status() afterwards
// reports FA2_ERR_DEVICE_TIMEOUT and clears the word.  Nothing faults, traps or
// hangs: the CUDA context stays usable.
#include "common.cuh"
#include "fa2.h"
#include "internal.h"

namespace fa2 {
namespace {

__global__ void watchdog_selftest_kernel(unsigned int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    const Watchdog wd{&abort_flag, status};
    (void)mbar_wait(smem_u32(&bar), 0, wd);  // no arrival ever comes: returns false after the limit
}

}  // namespace
}  // namespace fa2

extern "C" fa2_status fa2_watchdog_selftest(void* stream) {
    unsigned int* word = nullptr;
    if (!fa2::watchdog_word(&word)) return FA2_ERR_CUDA;
    fa2::watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word);
    return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}
