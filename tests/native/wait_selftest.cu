// Test-only kernel: the library's bounded mbarrier waits give up on a phase
// that never completes and report it, instead of hanging the GPU.
//
// One CTA: thread 0 initialises an mbarrier for one arrival that nobody makes,
// every thread of warp 0 waits on it with the library's bounded wait
// (mbar_wait_bounded, about two seconds), and the outcome lands in *status
// (1 = the wait completed, 2 = it gave up).  A second mbarrier that thread 0
// does arrive on checks the completed path.
#include "gdn_device.cuh"

namespace {

__global__ void wait_kernel(int *status)
{
    __shared__ uint64_t never, done;
    if (threadIdx.x == 0) {
        gdn::dev::mbar_init(&never, 1);
        gdn::dev::mbar_init(&done, 1);
        gdn::dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // a plain arrival completes phase 0 of `done`
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gdn::dev::smem_addr(&done))
                     : "memory");
    }
    __syncthreads();
    const bool ok_done = gdn::dev::mbar_wait_bounded(&done, 0);
    const bool ok_never = gdn::dev::mbar_wait_bounded(&never, 0);
    if (threadIdx.x == 0) {
        status[0] = ok_done ? 1 : 2;
        status[1] = ok_never ? 1 : 2;
    }
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int wait_selftest(int *status_device)
{
    wait_kernel<<<1, 32>>>(status_device);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
