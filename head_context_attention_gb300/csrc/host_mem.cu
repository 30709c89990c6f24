// host_mem.cu -- loong_host_alloc / loong_host_free: pinned host buffers for
// loong_attn_2d_host, backed by transparent huge pages where the kernel offers
// them.
//
// The device reaches pinned host memory through translations of its pages.
// When those translations have gone cold (after a few seconds without host
// copies, or after kernels that sweep tens of GB of device memory) a copy pays
// a miss per host page.  Measured with 64 KB base pages: a 2.7 GB copy then
// took 360-380 ms instead of 12.7 ms, and splitting it over several copy
// streams did not help (the misses are served one after another).  The same
// copy from a buffer on 512 MB huge pages took 12.7 ms in that state, with
// 8192 times fewer pages to translate.
//
// A buffer is an anonymous mapping aligned to the huge-page size, advised
// MADV_HUGEPAGE, faulted in one byte per base page, collapsed into huge pages
// where the fault path fell back to base pages (MADV_COLLAPSE, which compacts
// memory for this range only; ignored by kernels without it) and registered
// with CUDA (cudaHostRegister).  Without transparent huge pages it is still
// pinned and works as before.
#include <sys/mman.h>
#include <unistd.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>

#include "internal.h"

#ifndef MADV_COLLAPSE
#define MADV_COLLAPSE 25  // Linux 6.1 and later
#endif

namespace loong {

namespace {

struct Mapping {
  void* raw;
  size_t raw_bytes;
};

std::mutex g_mu;
std::map<void*, Mapping>& mappings() {
  static std::map<void*, Mapping> m;
  return m;
}

// The transparent huge page size (bytes), or 0 if the kernel reports none.
size_t huge_page_bytes() {
  FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r");
  if (!f) return 0;
  unsigned long long v = 0;
  const int n = std::fscanf(f, "%llu", &v);
  std::fclose(f);
  return n == 1 ? static_cast<size_t>(v) : 0;
}

}  // namespace

}  // namespace loong

using namespace loong;

extern "C" {

int loong_host_alloc(size_t bytes, void** ptr) {
  if (!ptr) return LOONG_ERR_INVALID_ARG;
  *ptr = nullptr;
  if (bytes == 0) return LOONG_OK;
  const size_t page = static_cast<size_t>(sysconf(_SC_PAGESIZE));
  size_t align = huge_page_bytes();
  if (align < page) align = page;
  const size_t len = (bytes + align - 1) / align * align;
  if (len < bytes) return LOONG_ERR_INVALID_ARG;  // overflow
  const size_t raw_bytes = len + align;
  void* raw = mmap(nullptr, raw_bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED) return LOONG_ERR_CUDA;
  char* p = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(raw) + align - 1) / align * align);
  madvise(p, len, MADV_HUGEPAGE);  // advisory: without huge pages the buffer still works
  for (size_t off = 0; off < len; off += page) p[off] = 0;
  if (align > page) madvise(p, len, MADV_COLLAPSE);  // advisory, as above
  const cudaError_t e = cudaHostRegister(p, len, cudaHostRegisterDefault);
  if (e != cudaSuccess) {
    munmap(raw, raw_bytes);
    return cuda_fail(e);
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    mappings()[p] = Mapping{raw, raw_bytes};
  }
  *ptr = p;
  return LOONG_OK;
}

int loong_host_free(void* ptr) {
  if (!ptr) return LOONG_OK;
  Mapping m;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = mappings().find(ptr);
    if (it == mappings().end()) return LOONG_ERR_INVALID_ARG;
    m = it->second;
    mappings().erase(it);
  }
  const cudaError_t e = cudaHostUnregister(ptr);
  munmap(m.raw, m.raw_bytes);
  return e == cudaSuccess ? LOONG_OK : cuda_fail(e);
}

}  // extern "C"
