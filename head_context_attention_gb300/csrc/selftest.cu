// selftest.cu -- a built-in check of the bounded-wait path: one CTA waits on
// an mbarrier that nothing arrives on, with the wait code the attention
// kernels use.  The wait gives up after the given limit, raises the CTA's
// abort flag and sets the device error word; the kernel then returns.
#include "internal.h"
#include "ptx.cuh"

namespace loong {

namespace {

__global__ void wait_probe_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // phase 0 of `bar` never completes: no thread arrives on it
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_sh, err, limit_ns);
  __syncthreads();
}

}  // namespace

int launch_wait_probe(uint32_t limit_us, cudaStream_t stream) {
  unsigned* err = device_error_word();
  if (!err) return LOONG_ERR_CUDA;
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, static_cast<unsigned long long>(limit_us) * 1000ull);
  return check_launch();
}

}  // namespace loong
