// noalloc.cu -- the backward pass for callers that cannot allocate device
// memory.  Some callers own no allocator: a plugin inside a framework that
// manages the whole device memory pool and hands the plugin only its input and
// output tensors, or a latency-critical loop that cannot afford the implicit
// device synchronisation of cudaMalloc/cudaFree.  For them this file keeps the
// backward's scratch (fp32 dQ accumulator and row statistics) in one
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

struct ScratchSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchSlot g_scratch_slot[64];

// Device address of the array on the current device, looked up once per
// device (with that device current) on the first call there.
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
  ScratchSlot* s = &g_scratch_slot[dev];
  std::call_once(s->once, [s]() { s->err = cudaGetSymbolAddress(&s->ptr, g_noalloc_scratch); });
  if (s->err != cudaSuccess || !s->ptr) {
    *status = cuda_fail(s->err != cudaSuccess ? s->err : cudaErrorInvalidSymbol);
    return nullptr;
  }
  *status = LOONG_OK;
  return s->ptr;
}

}  // namespace
}  // namespace loong

extern "C" int loong_attn_bwd_noalloc(const loong_attn_desc* d, const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, loong_stream_t stream) {
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  if (loong_attn_workspace_size(d, 1) > LOONG_NOALLOC_SCRATCH_BYTES) return LOONG_ERR_WORKSPACE;
  void* scratch = loong::scratch_address(&st);
  if (!scratch) return st;
  return loong_attn_bwd(d, q, k, v, o, lse, dout, dq, dk, dv, scratch, LOONG_NOALLOC_SCRATCH_BYTES, stream);
}
