// api.cu -- the C ABI of include/loong_attn.h: descriptor validation,
// workspace sizing, the host ring table, tensor-map encoding, the device error
// word and dispatch to the kernel launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace loong {

namespace {

__device__ unsigned g_error_word;

thread_local char t_last_cuda_error[256] = "no CUDA error";
thread_local cudaEvent_t t_ev_start = nullptr, t_ev_stop = nullptr;

struct DeviceCache {
  std::once_flag once;
  unsigned* err = nullptr;
  int cc_major = 0, cc_minor = 0;
  cudaError_t status = cudaSuccess;
};
DeviceCache g_dev[64];

DeviceCache* device_cache() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) return nullptr;
  DeviceCache* c = &g_dev[dev];
  std::call_once(c->once, [c, dev]() {
    void* p = nullptr;
    cudaError_t e1 = cudaGetSymbolAddress(&p, g_error_word);
    if (e1 == cudaSuccess) {
      c->err = static_cast<unsigned*>(p);
      e1 = cudaMemset(p, 0, sizeof(unsigned));
    }
    cudaError_t e2 = cudaDeviceGetAttribute(&c->cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaError_t e3 = cudaDeviceGetAttribute(&c->cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    c->status = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3);
  });
  if (c->status != cudaSuccess) {
    cuda_fail(c->status);
    return nullptr;
  }
  return c;
}

bool is_pow2_ok_hd(int d) { return d == 64 || d == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Every CUDA-touching entry point checks the device first.
int device_ready() {
  DeviceCache* c = device_cache();
  if (!c) return LOONG_ERR_CUDA;
  if (!(c->cc_major == 10 && c->cc_minor == 3)) return LOONG_ERR_UNSUPPORTED;
  return LOONG_OK;
}

// Device memory of the current device (cudaMalloc'd or managed).  Host memory,
// pinned or not, is refused: a kernel could read pinned memory over the
// chip-to-chip link, but far slower, and an unregistered pointer not at all.
bool on_device(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // not sticky; keep it from a later launch check
    return false;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

// Host memory: pinned (registered) or pageable.
bool in_host_memory(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

template <typename... T>
bool all_on_device(const T*... p) {
  return (on_device(p) && ...);
}

int cuda_fail(cudaError_t e) {
  std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return LOONG_ERR_CUDA;
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LOONG_OK : cuda_fail(e);
}

void record_start(cudaStream_t s) {
  if (t_ev_start && t_ev_stop) cudaEventRecord(t_ev_start, s);
}
void record_stop(cudaStream_t s) {
  if (t_ev_start && t_ev_stop) cudaEventRecord(t_ev_stop, s);
}

unsigned* device_error_word() {
  DeviceCache* c = device_cache();
  return c ? c->err : nullptr;
}

EncodeTiledFn tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int make_head_tile_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int d) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return LOONG_ERR_CUDA;
  if (!aligned16(base)) return LOONG_ERR_INVALID_ARG;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(heads)};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return LOONG_ERR_CUDA;
  }
  return LOONG_OK;
}

int make_f32_tile_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int d) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return LOONG_ERR_CUDA;
  if (!aligned16(base)) return LOONG_ERR_INVALID_ARG;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(d) * 4 * static_cast<cuuint64_t>(heads)};
  const cuuint32_t box[3] = {32, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return LOONG_ERR_CUDA;
  }
  return LOONG_OK;
}

RingGeom ring_geom(const loong_attn_desc& d) {
  RingGeom g;
  g.cp = d.cp;
  g.inner = d.ring_inner;
  g.outer = d.ring_outer;
  g.causal = d.causal;
  g.zigzag = d.placement == LOONG_PLACEMENT_ZIGZAG;
  g.nblocks = g.zigzag ? 2 * d.cp : d.cp;
  g.blk = static_cast<int>(d.seqlen / g.nblocks);
  g.ntile = (g.blk + kTile - 1) / kTile;
  return g;
}

FwdWsLayout fwd_ws_layout(const loong_attn_desc& d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t q_elems = static_cast<size_t>(d.batch) * d.seqlen * d.hq * d.head_dim;
  const size_t kv_elems = static_cast<size_t>(d.batch) * d.seqlen * d.hkv * d.head_dim;
  FwdWsLayout L{};
  L.v16 = 0;
  L.amax = up(kv_elems * 2);
  size_t off = L.amax + 256;
  L.o_acc = off;
  if (d.mode != LOONG_MODE_FUSED) off += up(q_elems * 4);
  L.recv = off;
  if (is_copy_mode(d)) off += 4 * up(kv_elems * 2);  // two receive buffers each for K and V
  L.total = off;
  return L;
}

// The forward's scratch pointers inside a workspace of fwd_ws_layout(d).total bytes.
static FwdScratch fwd_scratch(const loong_attn_desc& d, void* ws, void* o_res) {
  const FwdWsLayout L = fwd_ws_layout(d);
  uint8_t* w = static_cast<uint8_t*>(ws);
  FwdScratch sc;
  sc.v16 = w + L.v16;
  sc.v_amax = reinterpret_cast<unsigned*>(w + L.amax);
  sc.o_acc = d.mode != LOONG_MODE_FUSED ? reinterpret_cast<float*>(w + L.o_acc) : nullptr;
  sc.kv_recv = is_copy_mode(d) ? w + L.recv : nullptr;
  sc.o_res = o_res;
  return sc;
}

Layout layout_of(const loong_attn_desc& d) {
  const RingGeom g = ring_geom(d);
  Layout l;
  l.rank_major = d.layout == LOONG_LAYOUT_RANK_MAJOR;
  l.P = d.hp;
  l.cp = d.cp;
  l.zigzag = g.zigzag;
  l.blk = g.blk;
  l.S = d.seqlen;
  l.s_rank = d.seqlen / d.cp;
  return l;
}

}  // namespace loong

using namespace loong;

extern "C" {

int loong_version(void) { return (0 << 16) | 3; }

const char* loong_status_string(int status) {
  switch (status) {
    case LOONG_OK: return "ok";
    case LOONG_ERR_INVALID_ARG: return "invalid argument";
    case LOONG_ERR_WORKSPACE: return "workspace too small";
    case LOONG_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case LOONG_ERR_CUDA: return "CUDA error";
    case LOONG_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case LOONG_ERR_DEVICE_CHECK: return "device address check failed";
    default: return "unknown status";
  }
}

const char* loong_last_cuda_error(void) { return t_last_cuda_error; }

int loong_attn_check(const loong_attn_desc* d) {
  if (!d) return LOONG_ERR_INVALID_ARG;
  if (d->batch < 1 || d->seqlen < 1 || d->hq < 1 || d->hkv < 1 || d->hp < 1 || d->cp < 1 ||
      d->ring_inner < 1 || d->ring_outer < 1)
    return LOONG_ERR_INVALID_ARG;
  if (d->hq % d->hkv || d->hkv % d->hp || d->hq % d->hp) return LOONG_ERR_INVALID_ARG;
  if (static_cast<int64_t>(d->ring_inner) * d->ring_outer != d->cp) return LOONG_ERR_INVALID_ARG;
  if (d->placement != LOONG_PLACEMENT_ZIGZAG && d->placement != LOONG_PLACEMENT_CONTIGUOUS)
    return LOONG_ERR_INVALID_ARG;
  if (d->mode < LOONG_MODE_STEPWISE || d->mode > LOONG_MODE_STEPWISE_COPY_AB) return LOONG_ERR_INVALID_ARG;
  if (d->layout != LOONG_LAYOUT_NATURAL && d->layout != LOONG_LAYOUT_RANK_MAJOR) return LOONG_ERR_INVALID_ARG;
  const int64_t nblocks = d->placement == LOONG_PLACEMENT_ZIGZAG ? 2 * static_cast<int64_t>(d->cp) : d->cp;
  if (d->seqlen % nblocks) return LOONG_ERR_INVALID_ARG;
  if ((d->seqlen / nblocks) % d->hp) return LOONG_ERR_INVALID_ARG;
  // TMA row coordinates are int32: rows of the [rows, heads, d] view
  const int64_t view_rows = d->batch * d->seqlen * (d->layout == LOONG_LAYOUT_RANK_MAJOR ? d->hp : 1);
  if (d->batch * d->seqlen > 0x7fffffffLL || view_rows > 0x7fffffffLL) return LOONG_ERR_UNSUPPORTED;
  if (!std::isfinite(d->softmax_scale)) return LOONG_ERR_INVALID_ARG;
  if (!is_pow2_ok_hd(d->head_dim)) return LOONG_ERR_UNSUPPORTED;
  if (d->causal != 0 && d->causal != 1) return LOONG_ERR_INVALID_ARG;
  // the exchange copies whole per-rank chunks: contiguous only in the rank-major layout
  if (is_copy_mode(*d) && d->layout != LOONG_LAYOUT_RANK_MAJOR) return LOONG_ERR_UNSUPPORTED;
  // two rings need two blocks per rank
  if (d->mode == LOONG_MODE_STEPWISE_COPY_AB && d->placement != LOONG_PLACEMENT_ZIGZAG) return LOONG_ERR_UNSUPPORTED;
  return LOONG_OK;
}

size_t loong_attn_workspace_size(const loong_attn_desc* d, int pass) {
  if (loong_attn_check(d) != LOONG_OK) return 0;
  const size_t q_elems = static_cast<size_t>(d->batch) * d->seqlen * d->hq * d->head_dim;
  const size_t kv_elems = static_cast<size_t>(d->batch) * d->seqlen * d->hkv * d->head_dim;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  // STEPWISE_COPY: two receive buffers each for K and V, bf16
  const size_t recv = is_copy_mode(*d) ? 4 * up(kv_elems * 2) : 0;
  if (pass == 0) return fwd_ws_layout(*d).total;
  if (pass != 1) return 0;
  const size_t stats = 2 * static_cast<size_t>(d->batch) * d->hq * stat_row_len(ring_geom(*d));
  return up(q_elems * 4) + up(stats * 4) + 2 * up(kv_elems * 4) + recv;
}

int loong_ring_schedule(int32_t inner, int32_t outer, int32_t* src) {
  if (!src || inner < 1 || outer < 1 || static_cast<int64_t>(inner) * outer > (1 << 15))
    return LOONG_ERR_INVALID_ARG;
  const int cp = inner * outer;
  for (int t = 0; t < cp; ++t)
    for (int c = 0; c < cp; ++c) src[static_cast<int64_t>(t) * cp + c] = ring_src(c, t, inner, outer);
  return LOONG_OK;
}

int loong_attn_fwd(const loong_attn_desc* d, const void* q, const void* k, const void* v, void* o,
                   float* lse, void* o_res, void* ws, size_t ws_bytes, loong_stream_t stream_) {
  NvtxRange range("loong_attn_fwd");
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  if (!q || !k || !v || !o || !lse) return LOONG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (o_res && !aligned16(o_res)))
    return LOONG_ERR_INVALID_ARG;
  const size_t need = loong_attn_workspace_size(d, 0);
  if (!ws || ws_bytes < need || !aligned16(ws)) return LOONG_ERR_WORKSPACE;
  if ((st = device_ready()) != LOONG_OK) return st;
  if (!all_on_device(q, k, v, o, lse, ws) || (o_res && !on_device(o_res))) return LOONG_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const FwdScratch sc = fwd_scratch(*d, ws, o_res);
  if (d->mode == LOONG_MODE_FUSED) return launch_fwd(*d, q, k, v, o, lse, sc, stream);
  const int64_t q_elems = d->batch * d->seqlen * d->hq * d->head_dim;
  cudaError_t e = cudaMemsetAsync(sc.o_acc, 0, static_cast<size_t>(q_elems) * 4, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((st = launch_fill_f32(lse, d->batch * d->hq * d->seqlen, -INFINITY, stream)) != LOONG_OK) return st;
  if ((st = launch_fwd(*d, q, k, v, o, lse, sc, stream)) != LOONG_OK) return st;
  return launch_f32_to_bf16(sc.o_acc, o, q_elems, stream, o_res);
}

int loong_attn_fwd_ranks(const loong_attn_desc* d, int32_t rank_begin, int32_t rank_end, const void* q,
                         const void* k, const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                         loong_stream_t stream_) {
  NvtxRange range("loong_attn_fwd_ranks");
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  if (d->mode != LOONG_MODE_FUSED) return LOONG_ERR_UNSUPPORTED;
  if (rank_begin < 0 || rank_end <= rank_begin || rank_end > d->cp) return LOONG_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return LOONG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return LOONG_ERR_INVALID_ARG;
  if (!ws || ws_bytes < loong_attn_workspace_size(d, 0) || !aligned16(ws)) return LOONG_ERR_WORKSPACE;
  if ((st = device_ready()) != LOONG_OK) return st;
  if (!all_on_device(q, k, v, o, lse, ws)) return LOONG_ERR_INVALID_ARG;
  return launch_fwd(*d, q, k, v, o, lse, fwd_scratch(*d, ws, nullptr), reinterpret_cast<cudaStream_t>(stream_),
                    rank_begin, rank_end);
}

int loong_attn_bwd(const loong_attn_desc* d, const void* q, const void* k, const void* v, const void* o,
                   const void* o_res, const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                   size_t ws_bytes, loong_stream_t stream_) {
  NvtxRange range("loong_attn_bwd");
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return LOONG_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return LOONG_ERR_INVALID_ARG;
  if (o_res && !aligned16(o_res)) return LOONG_ERR_INVALID_ARG;
  const size_t need = loong_attn_workspace_size(d, 1);
  if (!ws || ws_bytes < need || !aligned16(ws)) return LOONG_ERR_WORKSPACE;
  if ((st = device_ready()) != LOONG_OK) return st;
  for (const void* p : ptrs)
    if (!on_device(p)) return LOONG_ERR_INVALID_ARG;
  if (!on_device(ws) || (o_res && !on_device(o_res))) return LOONG_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t q_elems = static_cast<size_t>(d->batch) * d->seqlen * d->hq * d->head_dim;
  const size_t kv_elems = static_cast<size_t>(d->batch) * d->seqlen * d->hkv * d->head_dim;
  const size_t stats = 2 * static_cast<size_t>(d->batch) * d->hq * stat_row_len(ring_geom(*d));
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* dq_acc = reinterpret_cast<float*>(w);
  float* dvec = reinterpret_cast<float*>(w + up(q_elems * 4));
  float* dk_acc = reinterpret_cast<float*>(w + up(q_elems * 4) + up(stats * 4));
  float* dv_acc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dk_acc) + up(kv_elems * 4));
  void* recv = is_copy_mode(*d) ? reinterpret_cast<uint8_t*>(dv_acc) + up(kv_elems * 4) : nullptr;
  return launch_bwd(*d, q, k, v, o, o_res, lse, dout, dq, dk, dv, dq_acc, dvec, dk_acc, dv_acc, stream, recv);
}

int loong_lse_merge(int64_t rows, int32_t d, int32_t n_parts, const float* o_parts, const float* lse_parts,
                    void* o_out, float* lse_out, int out_bf16, loong_stream_t stream) {
  NvtxRange range("loong_lse_merge");
  if (rows < 0 || d < 1 || d > 1024 || d % 4 || n_parts < 1 || n_parts > 64) return LOONG_ERR_INVALID_ARG;
  if (out_bf16 != 0 && out_bf16 != 1) return LOONG_ERR_INVALID_ARG;
  if (rows == 0) return LOONG_OK;
  if (!o_parts || !lse_parts || !o_out || !lse_out) return LOONG_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o_out) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return LOONG_ERR_INVALID_ARG;
  int st = device_ready();
  if (st != LOONG_OK) return st;
  if (!all_on_device(o_parts, lse_parts, lse_out) || !on_device(o_out)) return LOONG_ERR_INVALID_ARG;
  return launch_lse_merge(rows, d, n_parts, o_parts, lse_parts, o_out, lse_out, out_bf16,
                          reinterpret_cast<cudaStream_t>(stream));
}

int loong_headctx_pack_n(int32_t n, int64_t batch, int32_t cp, int32_t P, int64_t s_local, const int32_t* heads,
                         int32_t d, int direction, int gather, const void* const* in, void* const* out,
                         loong_stream_t stream) {
  NvtxRange range("loong_headctx_pack");
  if (n < 1 || n > 4 || !heads || !in || !out) return LOONG_ERR_INVALID_ARG;
  if (batch < 0 || cp < 1 || P < 1 || s_local < 0 || d < 1) return LOONG_ERR_INVALID_ARG;
  for (int t = 0; t < n; ++t)
    if (heads[t] < 1 || heads[t] % P) return LOONG_ERR_INVALID_ARG;
  if ((d * 2) % 16) return LOONG_ERR_INVALID_ARG;
  if (direction != 0 && direction != 1) return LOONG_ERR_INVALID_ARG;
  if (gather < 0 || gather > 2) return LOONG_ERR_INVALID_ARG;
  const int64_t S = static_cast<int64_t>(cp) * P * s_local;
  if (gather == 1 && (S % (2 * cp))) return LOONG_ERR_INVALID_ARG;
  if (batch == 0 || s_local == 0) return LOONG_OK;
  for (int t = 0; t < n; ++t)
    if (!in[t] || !out[t] || !aligned16(in[t]) || !aligned16(out[t])) return LOONG_ERR_INVALID_ARG;
  int st = device_ready();
  if (st != LOONG_OK) return st;
  for (int t = 0; t < n; ++t)
    if (!on_device(in[t]) || !on_device(out[t])) return LOONG_ERR_INVALID_ARG;
  return launch_headctx_pack(n, batch, cp, P, s_local, heads, d, direction, gather, in, out,
                             reinterpret_cast<cudaStream_t>(stream));
}

int loong_headctx_pack(int64_t batch, int32_t cp, int32_t P, int64_t s_local, int32_t heads, int32_t d,
                       int direction, int gather, const void* in, void* out, loong_stream_t stream) {
  return loong_headctx_pack_n(1, batch, cp, P, s_local, &heads, d, direction, gather, &in, &out, stream);
}

int loong_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return LOONG_ERR_INVALID_ARG;
  t_ev_start = static_cast<cudaEvent_t>(start_event);
  t_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return LOONG_OK;
}

int loong_selftest_wait_timeout(uint32_t limit_us, loong_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return LOONG_ERR_INVALID_ARG;
  int st = device_ready();
  if (st != LOONG_OK) return st;
  return launch_wait_probe(limit_us, reinterpret_cast<cudaStream_t>(stream));
}

int loong_get_device_status(loong_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned* p = device_error_word();
  if (!p) return LOONG_ERR_CUDA;
  unsigned word = 0;
  e = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word) {
    e = cudaMemset(p, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
    return (word & (kErrBounds | kErrSmemAlign)) ? LOONG_ERR_DEVICE_CHECK : LOONG_ERR_DEVICE_TIMEOUT;
  }
  return LOONG_OK;
}

}  // extern "C"
