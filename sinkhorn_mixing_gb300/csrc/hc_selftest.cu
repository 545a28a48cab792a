// hc_selftest.cu -- a diagnostic for the kernels' bounded waits: one CTA
// waits, through the same wait routine the kernels use, on a barrier that
// nothing arrives on, so the wait can only run out.  It then sets bit 0 of the
// device error word and returns; the context stays usable.
#include "hc_internal.h"
#include "hc_ptx.cuh"

namespace hc {
namespace {

using namespace ptx;

__global__ void k_wait_timeout(unsigned int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        abort_word = 0;
        mbar_init(su32(&bar), 1);  // one arrival expected, none ever made
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bar<false>(su32(&bar), 0, &abort_word, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout(uint64_t limit_ns, const DeviceInfo &di, cudaStream_t s) {
    k_wait_timeout<<<1, 32, 0, s>>>(di.err_word, limit_ns);
    return launched();
}

}  // namespace hc
