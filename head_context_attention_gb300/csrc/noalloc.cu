// noalloc.cu -- the backward pass for callers that cannot allocate device
// memory.  Some callers own no allocator: a plugin inside a framework that
// manages the whole device memory pool and hands the plugin only its input and
// output tensors, or a latency-critical loop that cannot afford the implicit
// device synchronisation of cudaMalloc/cudaFree.  For them this file keeps the
// backward's scratch (fp32 dQ, dK, dV accumulators and row statistics) in one
// file-scope device array of LOONG_NOALLOC_SCRATCH_BYTES, which every GPU that
// loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace loong {
namespace {

// In host code this name is only a host-side stand-in for the array, not its
// device address: the address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LOONG_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of the array on the current device, looked up with that
// device current on the first call there.  Only a successful lookup is kept;
// after a failure the next call looks again.
void* scratch_address(int* status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *status = cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    *status = LOONG_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      *status = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *status = LOONG_OK;
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace loong

extern "C" int loong_attn_bwd_noalloc(const loong_attn_desc* d, const void* q, const void* k, const void* v,
                                      const void* o, const void* o_res, const float* lse, const void* dout,
                                      void* dq, void* dk, void* dv, loong_stream_t stream) {
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  // the device first, so that an unsupported GPU reports LOONG_ERR_UNSUPPORTED
  // as loong_attn_bwd does, before any symbol lookup
  if ((st = loong::device_ready()) != LOONG_OK) return st;
  if (loong_attn_workspace_size(d, 1) > LOONG_NOALLOC_SCRATCH_BYTES) return LOONG_ERR_WORKSPACE;
  void* scratch = loong::scratch_address(&st);
  if (!scratch) return st;
  return loong_attn_bwd(d, q, k, v, o, o_res, lse, dout, dq, dk, dv, scratch, LOONG_NOALLOC_SCRATCH_BYTES, stream);
}
