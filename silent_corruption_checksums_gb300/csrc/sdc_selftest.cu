// sdc_selftest.cu -- a self-test of the bounded barrier wait that every
// TMA / tensor-core kernel of this library relies on to turn a stall into an
// error status instead of a hang.
//
// One thread initialises a shared-memory mbarrier expecting one arrival and
// waits on its first phase, which nothing completes, for `polls` polls: the
// wait must give up and report it.  The thread then arrives itself and waits
// again: the wait must now succeed.  No copy, no tensor-core operation and no
// other thread is involved, and every loop is bounded, so the kernel ends in
// every case.
#include "sdc_internal.cuh"

namespace sdc {
namespace {

__global__ void bounded_wait_selftest_kernel(uint32_t polls, uint32_t *__restrict__ status) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    uint32_t st = 0;
    if (!mbar_wait(b, 0, polls)) st |= 1u;  // nothing arrived: the wait gave up
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
    if (mbar_wait(b, 0, polls)) st |= 2u;  // the phase completed: the wait succeeds
    *status = st;
}

}  // namespace
}  // namespace sdc

extern "C" sdc_status sdc_selftest_bounded_wait(uint32_t polls, uint32_t *d_status, sdc_stream_t stream) {
    if (!d_status) return sdc::fail(SDC_ERR_NULL, "NULL status");
    if (polls == 0 || polls > (1u << 24)) return sdc::fail(SDC_ERR_BAD_ARG, "polls must be 1 .. 2^24");
    int dev = -1;
    const cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return sdc::cuda_fail(de, "cudaGetDevice");
    const sdc_status st = sdc::check_device_range(d_status, 4, dev, "d_status");
    if (st != SDC_OK) return st;
    sdc::bounded_wait_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(polls, d_status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : sdc::cuda_fail(e, "sdc_selftest_bounded_wait launch");
}
