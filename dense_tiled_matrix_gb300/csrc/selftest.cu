// selftest.cu -- exercises the kernels' bounded-wait path on purpose.
//
// Every pipeline wait in the libtgemm kernels gives up after a time limit,
// records TGEMM_ERR_TIMEOUT in the device status word and lets the kernel
// finish.  tgemm_selftest_wait_timeout runs that same wait (mbar_wait from
// device.cuh) in a one-thread kernel on an mbarrier that nothing ever arrives
// at, with a short caller-chosen limit, so the timeout path can be tested
// without a hung or faulted GPU: the kernel returns after the limit, the
// context stays usable, and tgemm_get_device_status() must report the timeout.
#include "device.cuh"
#include "host.h"
#include "tgemm.h"

namespace tgemm {
namespace {

__global__ void wait_forever_kernel(uint64_t limit_ns, uint32_t* status, uint32_t* waited_out) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);            // expects one arrival; none will come
    fence_barrier_init();
    const bool ok = mbar_wait(&bar, 0, status, limit_ns);
    if (waited_out) *waited_out = ok ? 0u : 1u;
}

}  // namespace
}  // namespace tgemm

extern "C" tgemm_status tgemm_selftest_wait_timeout(int64_t limit_ns, struct CUstream_st* stream) {
    using namespace tgemm;
    clear_error();
    if (limit_ns < 1000 || limit_ns > 1000000000) {
        set_error("limit_ns must be within [1e3, 1e9] nanoseconds");
        return TGEMM_ERR_INVALID_VALUE;
    }
    Device* dev = nullptr;
    tgemm_status st = current_device(&dev);
    if (st != TGEMM_OK) return st;
    wait_forever_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_ns), dev->status, nullptr);
    count_launch();
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail("wait_forever_kernel launch", err);
    return TGEMM_OK;
}

namespace tgemm {
namespace {

__global__ void record_check_kernel(uint32_t* status) {
    if (threadIdx.x == 0 && blockIdx.x == 0) debug_fail(status, kFileSelftest, static_cast<uint32_t>(__LINE__));
}

}  // namespace
}  // namespace tgemm

extern "C" tgemm_status tgemm_selftest_debug_check(struct CUstream_st* stream) {
    using namespace tgemm;
    clear_error();
    Device* dev = nullptr;
    tgemm_status st = current_device(&dev);
    if (st != TGEMM_OK) return st;
    record_check_kernel<<<1, 32, 0, stream>>>(dev->status);
    count_launch();
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail("record_check_kernel launch", err);
    return TGEMM_OK;
}
