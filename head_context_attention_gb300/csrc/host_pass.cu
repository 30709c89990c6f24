// host_pass.cu -- loong_attn_2d_host: one whole 2D-attention pass from host
// memory to host memory, its copies overlapped with its kernels.
//
// Three streams per call: the caller's stream runs every kernel (repacks, ring
// forward, ring backward) in order; two library-owned copy streams carry the
// host-to-device and device-to-host copies.  Events order each copy against
// the kernels that produce or consume its buffer:
//
//   h2d:    [wait slot free] Q,K,V -> in[slot] (fwd_in)  dO -> in[slot] (bwd_in)
//   stream: [wait fwd_in] repack Q,K,V  [wait o_lse_out] forward  repack O (fwd_out)
//           [wait bwd_in] repack dO (slot free)  backward  [wait grads_out] repack dQ,dK,dV (bwd_out)
//   d2h:    [wait fwd_out] O, LSE -> host (o_lse_out)   [wait bwd_out] dQ,dK,dV -> host (grads_out)
//
// so dO arrives while the forward runs, O and LSE leave while the backward
// runs, the next call's inputs arrive while this call's kernels run (they go
// to the other slot) and this call's gradients leave while the next call's
// kernels run.  A wait on an event never recorded yet (first call) is a no-op.
#include <mutex>

#include "internal.h"

namespace loong {

namespace {

struct HostPass {
  std::mutex mu;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t slot_free[2] = {nullptr, nullptr};
  cudaEvent_t fwd_in = nullptr, bwd_in = nullptr, fwd_out = nullptr, bwd_out = nullptr;
  cudaEvent_t o_lse_out = nullptr, grads_out = nullptr;
};

struct HostPassSlot {
  std::once_flag once;
  HostPass hp;
  cudaError_t status = cudaSuccess;
};
HostPassSlot g_host_pass[64];

HostPass* host_pass_for_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) return nullptr;
  HostPassSlot* s = &g_host_pass[dev];
  std::call_once(s->once, [s]() {
    HostPass& h = s->hp;
    cudaError_t r = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking);
    if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&h.slot_free[0], &h.slot_free[1], &h.fwd_in, &h.bwd_in,
                          &h.fwd_out,      &h.bwd_out,      &h.o_lse_out, &h.grads_out};
    for (cudaEvent_t* ev : evs)
      if (r == cudaSuccess) r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    s->status = r;
  });
  if (s->status != cudaSuccess) {
    cuda_fail(s->status);
    return nullptr;
  }
  return &s->hp;
}

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of the workspace's parts.
struct HostPassLayout {
  size_t q, kv, lse;  // tensor sizes in bytes (q-shaped, kv-shaped, LSE)
  size_t in[2][4];    // slot inputs q, k, v, dO (natural layout)
  size_t out[4];      // natural outputs o, dq, dk, dv
  size_t lse_off;
  size_t ores;        // the forward's residual of O (pass 1), in the layout the kernels use
  size_t kt[8];       // RANK_MAJOR: q, k, v, dO, o, dq, dk, dv
  size_t ws_fwd, ws_bwd, ws_fwd_bytes, ws_bwd_bytes;
  size_t total;
};

HostPassLayout host_pass_layout(const loong_attn_desc& d, int pass) {
  HostPassLayout L{};
  const size_t tok = static_cast<size_t>(d.batch) * d.seqlen * d.head_dim * 2;
  L.q = tok * d.hq;
  L.kv = tok * d.hkv;
  L.lse = static_cast<size_t>(d.batch) * d.hq * d.seqlen * 4;
  const size_t shape[4] = {L.q, L.kv, L.kv, L.q};  // q, k, v, dO; o, dq share q's, dk, dv kv's
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += up256(bytes);
    return at;
  };
  for (int s = 0; s < 2; ++s)
    for (int t = 0; t < 4; ++t) L.in[s][t] = (t == 3 && pass == 0) ? 0 : take(shape[t]);
  const size_t out_shape[4] = {L.q, L.q, L.kv, L.kv};  // o, dq, dk, dv
  for (int t = 0; t < 4; ++t) L.out[t] = (t > 0 && pass == 0) ? 0 : take(out_shape[t]);
  L.lse_off = take(L.lse);
  L.ores = pass == 1 ? take(L.q) : 0;
  if (d.layout == LOONG_LAYOUT_RANK_MAJOR) {
    const size_t kt_shape[8] = {L.q, L.kv, L.kv, L.q, L.q, L.q, L.kv, L.kv};
    for (int t = 0; t < 8; ++t) L.kt[t] = ((t == 3 || t > 4) && pass == 0) ? 0 : take(kt_shape[t]);
  }
  L.ws_fwd_bytes = loong_attn_workspace_size(&d, 0);
  L.ws_fwd = take(L.ws_fwd_bytes);
  L.ws_bwd_bytes = pass == 1 ? loong_attn_workspace_size(&d, 1) : 0;
  L.ws_bwd = L.ws_bwd_bytes ? take(L.ws_bwd_bytes) : 0;
  L.total = off;
  return L;
}

}  // namespace

}  // namespace loong

using namespace loong;

extern "C" {

size_t loong_attn_2d_host_workspace_size(const loong_attn_desc* d, int pass) {
  if (loong_attn_check(d) != LOONG_OK || (pass != 0 && pass != 1)) return 0;
  return host_pass_layout(*d, pass).total;
}

int loong_attn_2d_host(const loong_attn_desc* d, int32_t slot, const void* q, const void* k, const void* v,
                       const void* dout, void* o, float* lse, void* dq, void* dk, void* dv, void* ws,
                       size_t ws_bytes, loong_stream_t stream_, void* done_event) {
  NvtxRange range("loong_attn_2d_host");
  int st = loong_attn_check(d);
  if (st != LOONG_OK) return st;
  const int pass = dout ? 1 : 0;
  if (slot != 0 && slot != 1) return LOONG_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return LOONG_ERR_INVALID_ARG;
  if (pass == 1 ? (!dq || !dk || !dv) : (dq || dk || dv)) return LOONG_ERR_INVALID_ARG;
  const HostPassLayout L = host_pass_layout(*d, pass);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return LOONG_ERR_WORKSPACE;
  if ((st = device_ready()) != LOONG_OK) return st;
  const void* host_ptrs[] = {q, k, v, dout, o, lse, dq, dk, dv};
  for (const void* p : host_ptrs)
    if (p && !in_host_memory(p)) return LOONG_ERR_INVALID_ARG;
  if (!on_device(ws)) return LOONG_ERR_INVALID_ARG;
  HostPass* hp = host_pass_for_device();
  if (!hp) return LOONG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hp->mu);

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(w + off); };
  const bool rm = d->layout == LOONG_LAYOUT_RANK_MAJOR;
  const int64_t s_local = d->seqlen / (static_cast<int64_t>(d->cp) * d->hp);
  const int gather = d->placement == LOONG_PLACEMENT_ZIGZAG ? 1 : 2;
  const int32_t heads[8] = {d->hq, d->hkv, d->hkv, d->hq, d->hq, d->hq, d->hkv, d->hkv};  // q k v dO o dq dk dv
  cudaError_t e;
#define LOONG_TRY(x)                           \
  do {                                         \
    if ((e = (x)) != cudaSuccess) return cuda_fail(e); \
  } while (0)
  auto h2d = [&](size_t dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(at(dst), src, bytes, cudaMemcpyHostToDevice, hp->h2d);
  };
  auto d2h = [&](void* dst, size_t src, size_t bytes) {
    return cudaMemcpyAsync(dst, at(src), bytes, cudaMemcpyDeviceToHost, hp->d2h);
  };
  // natural <-> rank-major repack, in one launch, of the tensors t0 .. t0+n-1 (0..7) between their natural
  // buffers nat[] and their rank-major copies
  auto repack = [&](int t0, int n, const size_t* nat, int direction) {
    const void* src[4];
    void* dst[4];
    for (int i = 0; i < n; ++i) {
      src[i] = direction == 0 ? at(nat[i]) : at(L.kt[t0 + i]);
      dst[i] = direction == 0 ? at(L.kt[t0 + i]) : at(nat[i]);
    }
    return loong_headctx_pack_n(n, d->batch, d->cp, d->hp, s_local, heads + t0, d->head_dim, direction, gather,
                                src, dst, stream_);
  };
  const size_t* in = L.in[slot];

  // ---- inputs: Q, K, V, then dO, once the slot's previous inputs are read
  LOONG_TRY(cudaStreamWaitEvent(hp->h2d, hp->slot_free[slot], 0));
  LOONG_TRY(h2d(in[0], q, L.q));
  LOONG_TRY(h2d(in[1], k, L.kv));
  LOONG_TRY(h2d(in[2], v, L.kv));
  LOONG_TRY(cudaEventRecord(hp->fwd_in, hp->h2d));
  if (pass == 1) {
    LOONG_TRY(h2d(in[3], dout, L.q));
    LOONG_TRY(cudaEventRecord(hp->bwd_in, hp->h2d));
  }

  // ---- forward; it rewrites LSE (and O in the natural layout), which the
  // previous call's output copies must have read
  LOONG_TRY(cudaStreamWaitEvent(stream, hp->fwd_in, 0));
  if (rm && (st = repack(0, 3, in, 0)) != LOONG_OK) return st;
  if (pass == 0 && rm) LOONG_TRY(cudaEventRecord(hp->slot_free[slot], stream));
  LOONG_TRY(cudaStreamWaitEvent(stream, hp->o_lse_out, 0));
  float* lse_dev = static_cast<float*>(at(L.lse_off));
  void* ws_fwd = at(L.ws_fwd);
  // the residual of O stays on the device for the backward's D
  void* o_res = pass == 1 ? at(L.ores) : nullptr;
  if (rm) {
    if ((st = loong_attn_fwd(d, at(L.kt[0]), at(L.kt[1]), at(L.kt[2]), at(L.kt[4]), lse_dev, o_res, ws_fwd,
                             L.ws_fwd_bytes, stream_)) != LOONG_OK)
      return st;
    if ((st = repack(4, 1, L.out, 1)) != LOONG_OK) return st;
  } else if ((st = loong_attn_fwd(d, at(in[0]), at(in[1]), at(in[2]), at(L.out[0]), lse_dev, o_res, ws_fwd,
                                  L.ws_fwd_bytes, stream_)) != LOONG_OK) {
    return st;
  }
  if (pass == 0 && !rm) LOONG_TRY(cudaEventRecord(hp->slot_free[slot], stream));
  LOONG_TRY(cudaEventRecord(hp->fwd_out, stream));
  // O and LSE leave while the backward runs
  LOONG_TRY(cudaStreamWaitEvent(hp->d2h, hp->fwd_out, 0));
  LOONG_TRY(d2h(o, L.out[0], L.q));
  LOONG_TRY(d2h(lse, L.lse_off, L.lse));
  LOONG_TRY(cudaEventRecord(hp->o_lse_out, hp->d2h));

  // ---- backward; its outputs are rewritten once the previous call's gradient copies are done
  if (pass == 1) {
    LOONG_TRY(cudaStreamWaitEvent(stream, hp->bwd_in, 0));
    void* ws_bwd = at(L.ws_bwd);
    if (rm) {
      if ((st = repack(3, 1, in + 3, 0)) != LOONG_OK) return st;
      LOONG_TRY(cudaEventRecord(hp->slot_free[slot], stream));
      if ((st = loong_attn_bwd(d, at(L.kt[0]), at(L.kt[1]), at(L.kt[2]), at(L.kt[4]), o_res, lse_dev, at(L.kt[3]),
                               at(L.kt[5]), at(L.kt[6]), at(L.kt[7]), ws_bwd, L.ws_bwd_bytes, stream_)) != LOONG_OK)
        return st;
      LOONG_TRY(cudaStreamWaitEvent(stream, hp->grads_out, 0));
      if ((st = repack(5, 3, L.out + 1, 1)) != LOONG_OK) return st;
    } else {
      LOONG_TRY(cudaStreamWaitEvent(stream, hp->grads_out, 0));
      if ((st = loong_attn_bwd(d, at(in[0]), at(in[1]), at(in[2]), at(L.out[0]), o_res, lse_dev, at(in[3]),
                               at(L.out[1]), at(L.out[2]), at(L.out[3]), ws_bwd, L.ws_bwd_bytes, stream_)) != LOONG_OK)
        return st;
      LOONG_TRY(cudaEventRecord(hp->slot_free[slot], stream));
    }
    LOONG_TRY(cudaEventRecord(hp->bwd_out, stream));
    LOONG_TRY(cudaStreamWaitEvent(hp->d2h, hp->bwd_out, 0));
    LOONG_TRY(d2h(dq, L.out[1], L.q));
    LOONG_TRY(d2h(dk, L.out[2], L.kv));
    LOONG_TRY(d2h(dv, L.out[3], L.kv));
    LOONG_TRY(cudaEventRecord(hp->grads_out, hp->d2h));
  }

  // ---- completion: the caller's event, or the stream itself waits for the copies
  if (done_event) {
    LOONG_TRY(cudaEventRecord(static_cast<cudaEvent_t>(done_event), hp->d2h));
  } else {
    LOONG_TRY(cudaStreamWaitEvent(stream, pass == 1 ? hp->grads_out : hp->o_lse_out, 0));
  }
#undef LOONG_TRY
  return LOONG_OK;
}

}  // extern "C"
