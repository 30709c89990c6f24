// exchange.h -- a copy-engine stand-in for the ring's K/V exchange.
//
// [G] "3. Double-Ring Asynchronous Communication Pipeline": the K/V blocks of
// the next step travel on background streams while attention runs on the
// current ones.  With every rank on one GPU, the stand-in is a device-to-device
// copy: before step t >= 1, each ring rank c receives the K/V chunk of rank
// src(c, t) into its plane of a receive buffer (the rank-major layout keeps a
// rank's chunk contiguous).  Two buffers alternate, so the copies for step t
// run on a side stream while the kernel of step t - 1 runs; step 0 reads each
// rank's own chunk in place.  With two rings (STEPWISE_COPY_AB, paired blocks)
// the chunk's block A and block B halves travel on two independent side
// streams, the guide's "two independent communication rings".
#pragma once

#include "internal.h"

namespace loong {

struct Exchange {
  cudaStream_t side[2] = {nullptr, nullptr};  // ring A (and the single ring), ring B
  cudaEvent_t entry = nullptr, freed[2] = {nullptr, nullptr};
  cudaEvent_t ready[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};  // [buffer][ring]
};

// The calling device's side stream and events, created on first use.
// nullptr (with the CUDA error recorded) if they cannot be created.
Exchange* exchange_for_device();

// Enqueue on `side` the copies of step t: recv[b*cp + c] <- src[b*cp + src(c, t)]
// for every sequence b and ring rank c, of `rows` pieces of `part_bytes`, the
// first at byte `offset` of each `chunk_bytes` chunk and the next ones `pitch`
// bytes apart (rows = 1: one contiguous piece).
int exchange_copies(const loong_attn_desc& d, int t, const void* src, void* recv, size_t chunk_bytes,
                    size_t offset, size_t part_bytes, size_t pitch, int rows, cudaStream_t side);

// Runs launch(t, buf) for the ring steps t = 0 .. cp-1 on `stream`; buf is -1
// at step 0 (K/V read in place) and else the receive buffer (0 or 1) that the
// copies of step t filled.  k, v are the rank-major inputs; rk[b], rv[b] the
// two receive buffers of each.
template <class Launch>
int run_exchanged_steps(const loong_attn_desc& d, const void* k, const void* v, void* const rk[2],
                        void* const rv[2], cudaStream_t stream, Launch launch) {
  Exchange* ex = exchange_for_device();
  if (!ex) return LOONG_ERR_CUDA;
  const size_t chunk = static_cast<size_t>(d.seqlen / d.cp) * d.hkv * d.head_dim * 2;
  // rank-major chunk [hp][S/cp][Hkv/hp][d]: block A is the first half of each
  // head rank's S/cp tokens, so the two rings move hp pieces each
  const int rings = d.mode == LOONG_MODE_STEPWISE_COPY_AB ? 2 : 1;
  cudaError_t e;
  // the side streams start once the caller's stream has produced k and v
  if ((e = cudaEventRecord(ex->entry, stream)) != cudaSuccess) return cuda_fail(e);
  for (int r = 0; r < rings; ++r)
    if ((e = cudaStreamWaitEvent(ex->side[r], ex->entry, 0)) != cudaSuccess) return cuda_fail(e);
  int st;
  for (int t = 0; t < d.cp; ++t) {
    const int buf = t & 1;
    if (t >= 1) {
      for (int r = 0; r < rings; ++r) {
        cudaStream_t side = ex->side[r];
        // the buffer was last read by the kernel of step t - 2
        if (t >= 3 && (e = cudaStreamWaitEvent(side, ex->freed[buf], 0)) != cudaSuccess) return cuda_fail(e);
        // one ring: the whole chunk; ring r of two: block r of every head rank,
        // hp pieces a head rank (two blocks) apart, as one strided copy
        const size_t blk_bytes = chunk / (2 * d.hp);
        const size_t off = rings == 1 ? 0 : r * blk_bytes;
        const size_t part = rings == 1 ? chunk : blk_bytes;
        const int rows = rings == 1 ? 1 : d.hp;
        if ((st = exchange_copies(d, t, k, rk[buf], chunk, off, part, 2 * blk_bytes, rows, side)) != LOONG_OK) return st;
        if ((st = exchange_copies(d, t, v, rv[buf], chunk, off, part, 2 * blk_bytes, rows, side)) != LOONG_OK) return st;
        if ((e = cudaEventRecord(ex->ready[buf][r], side)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(stream, ex->ready[buf][r], 0)) != cudaSuccess) return cuda_fail(e);
      }
    }
    if ((st = launch(t, t >= 1 ? buf : -1)) != LOONG_OK) return st;
    if (t >= 1 && (e = cudaEventRecord(ex->freed[buf], stream)) != cudaSuccess) return cuda_fail(e);
  }
  return LOONG_OK;
}

}  // namespace loong
