// exchange.cu -- side stream, events and copies of the ring exchange stand-in
// (exchange.h).
#include <mutex>

#include "exchange.h"

namespace loong {

namespace {

struct ExchangeSlot {
  std::once_flag once;
  Exchange ex;
  cudaError_t status = cudaSuccess;
};
ExchangeSlot g_ex[64];

}  // namespace

Exchange* exchange_for_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) return nullptr;
  ExchangeSlot* s = &g_ex[dev];
  std::call_once(s->once, [s]() {
    cudaError_t r = cudaEventCreateWithFlags(&s->ex.entry, cudaEventDisableTiming);
    for (int i = 0; i < 2 && r == cudaSuccess; ++i) {
      r = cudaStreamCreateWithFlags(&s->ex.side[i], cudaStreamNonBlocking);
      if (r == cudaSuccess) r = cudaEventCreateWithFlags(&s->ex.freed[i], cudaEventDisableTiming);
      for (int j = 0; j < 2 && r == cudaSuccess; ++j)
        r = cudaEventCreateWithFlags(&s->ex.ready[i][j], cudaEventDisableTiming);
    }
    s->status = r;
  });
  if (s->status != cudaSuccess) {
    cuda_fail(s->status);
    return nullptr;
  }
  return &s->ex;
}

int exchange_copies(const loong_attn_desc& d, int t, const void* src, void* recv, size_t chunk_bytes,
                    size_t offset, size_t part_bytes, size_t pitch, int rows, cudaStream_t side) {
  const auto* s = static_cast<const uint8_t*>(src);
  auto* r = static_cast<uint8_t*>(recv);
  for (int64_t b = 0; b < d.batch; ++b)
    for (int c = 0; c < d.cp; ++c) {
      const int j = ring_src(c, t, d.ring_inner, d.ring_outer);
      const size_t to = static_cast<size_t>(b * d.cp + c) * chunk_bytes + offset;
      const size_t from = static_cast<size_t>(b * d.cp + j) * chunk_bytes + offset;
      cudaError_t e = rows == 1 ? cudaMemcpyAsync(r + to, s + from, part_bytes, cudaMemcpyDeviceToDevice, side)
                                : cudaMemcpy2DAsync(r + to, pitch, s + from, pitch, part_bytes, rows,
                                                    cudaMemcpyDeviceToDevice, side);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  return LOONG_OK;
}

}  // namespace loong
