// pkv_wait_check.cu -- a launch whose pipeline wait can never be satisfied,
// for testing the failure path of the kernels' bounded waits.
//
// Every wait in the library's kernels (a copy pipeline's mbarrier in the
// decode kernels, the tensor-core pipeline's barriers in the prefill) gives
// up after a bounded time, sets PKV_DEVERR_TIMEOUT in the device error word
// and lets the kernel return, so a stalled pipeline never hangs the GPU.
// This kernel runs the same two wait routines on a barrier that no thread
// arrives at and no copy feeds: nothing is in flight when it gives up.
#include <cstdint>

#include "pkv_device.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

__global__ void wait_check_kernel(unsigned int* err, int which) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none ever comes
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = which == 0 ? mbar_wait(&bar, 0) : tc::wait_spin(&bar, 0);
        if (!ok) report(err, PKV_DEVERR_TIMEOUT);
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_check_wait_timeout(int32_t which, void* stream) {
    if (which != 0 && which != 1) return PKV_ERR_INVALID;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    wait_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, which);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
