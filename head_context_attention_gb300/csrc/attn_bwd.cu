// attn_bwd.cu -- backward ring-step attention on tcgen05 tensor cores.
//
// The gradient of softmax attention, causal or not (plain chain rule; the pages
// give no backward).  One CTA owns one 128-key tile of one kv head and walks every
// (query tile, query head of the group) that attends to it, in the order the
// key/value chunk travels around the ring: step t visits ring rank
// dst(j, t), the rank that holds source j's K/V at step t.  Per iteration:
//   S^T  = K Q^T                 (keys on TMEM lanes, queries on columns)
//   dP^T = V dO^T
//   P^T  = exp2(S^T*scale*log2e - LSE*log2e),  dS^T = P^T * (dP^T - D)
//   dV  += P^T dO                (P^T from tensor memory)
//   dK  += dS^T Q                (dS^T from shared memory, K-major)
//   dQ   = dS K  -> staged in shared memory, added into the fp32 dQ
//                   accumulator by TMA bulk tensor reductions
// dK and dV stay in tensor memory and are folded into fp32 accumulators every
// kFlush iterations; the last partial is added and written as bf16 (FUSED) or
// left in the accumulators (STEPWISE, one launch per step; a step maps ranks to
// sources one to one, so no two CTAs share a tile).  The compute warps form P^T
// as soon as S^T is ready, while dP^T is still on the tensor cores, and drain
// dQ while dK is computed.  Tensors are addressed through a Layout (natural or
// rank-major, ring.cuh); in STEPWISE_COPY modes the K/V tile is read from the
// plane of the rank that holds it at the launch's step (exchange.h), while dK
// and dV go to the owner's rows.
//
// Warp roles: compute warps form four groups of four warps that each cover all
// 128 TMEM lanes (608 threads with the three below); group g
// handles query columns [GW g, GW (g+1)) of S^T/dP^T and head-dim columns
// [GD g, GD (g+1)) of dQ, and folds a share of dV (first half of the groups)
// or dK (second half).  After them, one warp issues TMA loads, one allocates
// TMEM and issues the MMAs, one issues the dQ bulk reductions (so no compute
// warp waits on their completion).
// Tensor memory (512 columns): R0 [0,128) S^T, then P^T as bf16 pairs, each
// group packing its GW queries into the first GW/2 columns of its own GW (the
// groups share lanes, so none may write where another still reads);
// R1 [128,256) dP^T then dQ; dV and dK after that (D columns each).
#include <cuda_bf16.h>

#include <cmath>

#include "exchange.h"
#include "internal.h"
#include "ptx.cuh"

namespace loong {

namespace {

template <int D>
struct BwdCfg {
  static constexpr int NS = D == 64 ? 3 : 2;      // Q / dO pipeline stages (d = 64: 3 measured fastest)
  static constexpr int ATOMS = D / 64;
  static constexpr int ATOM_BYTES = kTile * 128;  // 16 KB
  static constexpr int TILE_BYTES = kTile * D * 2;
  static constexpr int DS_BYTES = kTile * kTile * 2;  // dS^T tile, bf16 [keys][queries]
  static constexpr int NBARS = 1 + 4 * NS + 13;
  static constexpr int STAT_BYTES = 2 * kTile * 4;  // LSE*log2e and D of one query tile
  // Tiles first (1024-byte aligned, checked at run time), then the row
  // statistics stages, the barriers, the TMEM base address and the abort
  // flag, then one iteration descriptor per stage.
  static constexpr int SMEM_BYTES =
      (2 + 2 * NS) * TILE_BYTES + DS_BYTES + NS * STAT_BYTES + NBARS * 8 + 16 + NS * 16;
  // Compute groups of four warps, each covering all 128 TMEM lanes: group g
  // owns query columns [GW g, GW (g+1)) of S^T / dP^T and head-dim columns
  // [GD g, GD (g+1)) of dQ.  Four groups (four compute warps per scheduler)
  // overlap the compute warps' chain of TMEM loads, exponentials and stores
  // better than two (measured faster at d = 64 and d = 128).
#ifndef LOONG_BWD_GROUPS
#define LOONG_BWD_GROUPS 4
#endif
  static constexpr int GROUPS = LOONG_BWD_GROUPS;
  static constexpr int GW = kTile / GROUPS;  // query columns per group
  static constexpr int GCH = GW / 32;        // 32-column chunks per group
  static constexpr int GD = D / GROUPS;      // dQ head-dim columns per group
  static constexpr int ACC_COLS = 2 * D / GROUPS;  // dV / dK columns each group folds
  static constexpr int CW = 4 * GROUPS;      // compute warps; then producer, MMA, reducer
  static constexpr int THREADS = 32 * (CW + 3);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t R0 = 0, R1 = 128, RV = 256, RK = 256 + D;
  // dQ leaves through TMA bulk reductions of 32-float x 128-row boxes; the
  // boxes are staged in the Q / dO stage of the iteration they belong to.
  static constexpr int DQ_BOXES = D / 32;
  static constexpr int BOX_BYTES = kTile * 128;
  static constexpr int BOXES_PER_STAGE = TILE_BYTES / BOX_BYTES;
  // The groups whose dQ columns land in the dO half of the stage stage them at
  // once (dV(i), the last reader of that half, retired before dQ(i) exists)
  // and the reducer adds that half first; the Q half waits for dK(i).
  // Measured faster at both head dimensions with four compute groups.
  static constexpr bool EARLY_O = true;
  // groups whose dQ columns lie in the Q half of the stage (the rest: the dO half)
  static constexpr int QHALF_GROUPS = BOXES_PER_STAGE * 32 / GD;
  // the iteration descriptors (int4) after the barriers and two words
  static_assert(((2 + 2 * NS) * TILE_BYTES + DS_BYTES + NS * STAT_BYTES + NBARS * 8 + 16) % 16 == 0,
                "descriptor alignment");
};

// dK and dV build up in tensor memory; every kFlush iterations they are added
// into fp32 accumulators in global memory and the tensor-memory sums restart,
// which bounds the length of each tensor-core accumulation chain.
constexpr int kFlush = 512;

struct BwdArgs {
  int batch, S, hq, hkv, G;
  RingGeom ring;
  Layout lay;  // where Q, K, V, dO, dQ (and its accumulator), dK, dV keep (token, head)
  int kv_held;  // K, V are receive buffers (one step per launch): read the holder rank's plane
  int t_begin, t_end;
  float scale, scale_log2;
  // Row statistics, [B*Hq][stat_len] each, block b's rows at b*blk_pad:
  const float* lse2;   // LSE * log2(e)
  const float* dstat;  // D = rowsum(dO * O)
  int blk_pad, stat_len;
  float* dq_acc;      // fp32, the layout of Q
  __nv_bfloat16* dk;  // FUSED outputs
  __nv_bfloat16* dv;
  float* dk_acc;      // fp32 accumulators, the layout of K (zeroed by the launcher)
  float* dv_acc;
  unsigned* err;
};

constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool STEP>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    ring_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // uniform over the CTA; the swizzled tiles need it
    if (threadIdx.x == 0) atomicOr(a.err, kErrSmemAlign);
    return;
  }
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::TILE_BYTES;
  uint8_t* sQ = sV + C::TILE_BYTES;              // NS stages
  uint8_t* sdO = sQ + C::NS * C::TILE_BYTES;     // NS stages
  uint8_t* sdS = sdO + C::NS * C::TILE_BYTES;    // [2 query atoms][128 keys][128 B]
  float* sStat = reinterpret_cast<float*>(sdS + C::DS_BYTES);  // NS x [LSE2[128], D[128]]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sStat) + C::NS * C::STAT_BYTES);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NS;
  uint64_t* s_full = q_empty + C::NS;   // S^T(i) in R0          (MMA -> warps)
  uint64_t* dp_full = s_full + 1;       // dP^T(i) in R1         (MMA -> warps)
  uint64_t* p_full = dp_full + 1;       // P^T(i) in R0          (warps -> MMA)
  uint64_t* ds_full = p_full + 1;       // dS^T(i) in smem       (warps -> MMA)
  uint64_t* dq_full = ds_full + 1;      // dQ(i) in R1           (MMA -> warps)
  uint64_t* dq_empty = dq_full + 1;     // R1 drained            (warps -> MMA)
  uint64_t* dk_done = dq_empty + 1;     // dK(i) done: Q/dO stage free for staging
  uint64_t* acc_full = dk_done + 1;     // dK/dV ready to flush  (MMA -> warps)
  uint64_t* acc_empty = acc_full + 1;   // dK/dV flushed         (warps -> MMA)
  uint64_t* done_bar = acc_empty + 1;
  uint64_t* drain = done_bar + 1;
  // per stage, so that neither runs a phase ahead of the reducer: a stage is
  // staged into again only after the reducer has read it and it was reloaded
  uint64_t* staged_q = drain + 1;       // NS: dQ(i) columns staged in the Q half (warps -> reducer)
  uint64_t* staged_o = staged_q + C::NS;  // NS: dQ(i) columns staged in the dO half (warps -> reducer)
  uint32_t& tmem_base_sh = *reinterpret_cast<uint32_t*>(bars + C::NBARS);
  int& abort_sh = *(reinterpret_cast<int*>(bars + C::NBARS) + 1);
  volatile int* abort_flag = &abort_sh;
  // Per stage, the iteration the producer loaded into it: view row of the
  // query tile, its view head, its length, and flags (1: the causal diagonal
  // tile, 2: a dQ reduction may start there).  Written before the stage's
  // q_full arrival, so everyone who waited for the stage's data sees it; the
  // compute and reducer warps then need no walk of their own.
  int4* sInfo = reinterpret_cast<int4*>(bars + C::NBARS + 2);

  // ---- work item: (batch, kv head, key tile); early (heavy) key tiles first
  const RingGeom& g = a.ring;
  int idx = blockIdx.x;
  const int nkt = g.nblocks * g.ntile;
  const int r = idx % nkt;
  idx /= nkt;
  const int kvh = idx % a.hkv;
  const int b = idx / a.hkv;
  const int bk = r / g.ntile;
  const int kt = r % g.ntile;
  const int k0 = bk * g.blk + kt * kTile;
  const int klen = min(kTile, (bk + 1) * g.blk - k0);

  QWalk walk;
  walk.init(g, a.G, bk, kt, a.t_begin, a.t_end);
  const int n = walk.total();
  if (n == 0) return;
  const int nflush = (n - 1) / kFlush;  // flushes before the final write

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);  // the reducer, once the stage's dQ boxes are read
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, C::CW);
    mbar_init(ds_full, C::CW);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, C::CW);
    mbar_init(dk_done, 1);
    for (int st = 0; st < C::NS; ++st) {
      mbar_init(&staged_q[st], C::EARLY_O ? 4 * C::QHALF_GROUPS : C::CW);
      mbar_init(&staged_o[st], 4 * (C::GROUPS - C::QHALF_GROUPS));
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::CW);
    mbar_init(done_bar, 1);
    mbar_init(drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::CW + 1) {
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == C::CW && lane == 0) {
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmO);
    tma_prefetch_map(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_sh;

  if (warp == C::CW) {
    // ------------------------------------------------------------ TMA producer
    {  // the whole warp runs the loop; lane 0 issues
      const uint32_t leader = lane == 0;
      auto warp_wait = [&](uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, err));
      };

      mbar_expect_tx_p(leader, kv_full, 2 * C::TILE_BYTES);
      int kvc;
      // the rank that holds this key tile's chunk at the launch's (single) step
      const int holder = ring_dst(block_owner(g, bk), a.t_begin, g.inner, g.outer);
      const int64_t kr64 = a.kv_held ? a.lay.view_row_held(b, k0, kvh, a.hkv, holder, kvc)
                                     : a.lay.view_row(b, k0, kvh, a.hkv, kvc);
      // checked build: tiles start inside their tensors (TMA fills rows past the end with zeros)
      in_bounds(kr64 >= 0 && kr64 < a.lay.view_rows(a.batch) && kvc >= 0 && kvc < a.lay.view_heads(a.hkv), a.err);
      const int kr = static_cast<int>(kr64);
      for (int at = 0; at < C::ATOMS; ++at) {
        tma_load_3d_p(leader, sK + at * C::ATOM_BYTES, &tmK, kv_full, at * 64, kvc, kr);
        tma_load_3d_p(leader, sV + at * C::ATOM_BYTES, &tmV, kv_full, at * 64, kvc, kr);
      }
      int issued = 0;
      for (int i = 0; i < n; ++i, walk.advance()) {
        const int s = i % C::NS;
        const int u = i / C::NS;
        // coordinates first, off the wait's critical path
        const int head = kvh * a.G + walk.head;
        int hc;
        const int64_t qrow64 = a.lay.view_row(b, walk.q0(), head, a.hq, hc);
        in_bounds(qrow64 >= 0 && qrow64 < a.lay.view_rows(a.batch) && hc >= 0 && hc < a.lay.view_heads(a.hq), a.err);
        const int qrow = static_cast<int>(qrow64);
        // checked build: a reduction never starts outside the accumulator (skipped if it would)
        const bool red_ok =
            in_bounds(qrow64 >= 0 && qrow64 < a.lay.view_rows(a.batch) && hc >= 0 && hc < a.lay.view_heads(a.hq), a.err);
        if (i >= C::NS && !warp_wait(&q_empty[s], (u - 1) & 1, abort_flag, a.err)) break;
        if (leader) sInfo[s] = make_int4(qrow, hc, walk.qlen(), (walk.diag() ? 1 : 0) | (red_ok ? 2 : 0));
        mbar_expect_tx_p(leader, &q_full[s], 2 * C::TILE_BYTES + C::STAT_BYTES);
        for (int at = 0; at < C::ATOMS; ++at) {
          tma_load_3d_p(leader, sQ + s * C::TILE_BYTES + at * C::ATOM_BYTES, &tmQ, &q_full[s], at * 64, hc, qrow);
          tma_load_3d_p(leader, sdO + s * C::TILE_BYTES + at * C::ATOM_BYTES, &tmO, &q_full[s], at * 64, hc, qrow);
        }
        // this tile's row statistics: 16-byte aligned and in bounds by construction
        int64_t srow = (static_cast<int64_t>(b) * a.hq + head) * a.stat_len + walk.bq * a.blk_pad +
                       walk.qi * kTile;
        // checked build: a plain bulk copy must stay inside the statistics rows
        // (else it reads row 0 instead, keeping the barrier's byte count)
        if (!in_bounds(srow >= 0 && srow % 4 == 0 &&
                           srow + kTile <= (static_cast<int64_t>(b) * a.hq + head + 1) * a.stat_len,
                       a.err))
          srow = 0;
        bulk_load_p(leader, sStat + s * (2 * kTile), a.lse2 + srow, kTile * 4, &q_full[s]);
        bulk_load_p(leader, sStat + s * (2 * kTile) + kTile, a.dstat + srow, kTile * 4, &q_full[s]);
        ++issued;
      }
      mbar_drain(kv_full, 0, a.err);
      for (int s = 0; s < C::NS; ++s) {
        const int cnt = issued > s ? (issued - 1 - s) / C::NS + 1 : 0;
        if (cnt) mbar_drain(&q_full[s], (cnt - 1) & 1, a.err);
      }
    }
  } else if (warp == C::CW + 1) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the loop; one elected lane issues
      auto warp_wait = [&](uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, err));
      };
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S^T, dP^T: both K-major
      constexpr uint32_t id_dkv = idesc_bf16(128, D, false, true);   // dV, dK: B MN-major
      constexpr uint32_t id_dq = idesc_bf16(128, D, true, true);     // dQ: A and B MN-major
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), q_addr = smem_u32(sQ),
                     o_addr = smem_u32(sdO), ds_addr = smem_u32(sdS);
      // Descriptors built once: an operand's descriptor at byte offset `off`
      // is its base descriptor plus off / 16 (the 14-bit address field cannot
      // carry: every shared-memory address is below 256 KB).
      auto d16 = [](uint32_t a) { return sdesc_sw128(a, 16, 1024); };           // K-major operands
      auto dmn = [](uint32_t a) { return sdesc_sw128(a, C::ATOM_BYTES, 1024); };  // MN-major operands
      const uint64_t k16 = d16(k_addr), kmn = dmn(k_addr), v16 = d16(v_addr), ds16 = d16(ds_addr),
                     dsmn = dmn(ds_addr);
      // X^T[keys x queries] = A[keys x d] * B[queries x d]^T, both K-major
      auto mm_s = [&](uint32_t dst, uint64_t a_desc, uint64_t b_desc) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::ATOM_BYTES + (kk & 3) * 32) >> 4;
          mma_ss_w(tbase + dst, a_desc + off, b_desc + off, id_s, kk > 0);
        }
      };
      bool ok = warp_wait(kv_full, 0, abort_flag, a.err) && warp_wait(&q_full[0], 0, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        mm_s(C::R0, k16, d16(q_addr));
        mma_commit_w(s_full);
        mm_s(C::R1, v16, d16(o_addr));
        mma_commit_w(dp_full);
        bool fresh = true;  // next dV / dK start a new tensor-memory sum
        for (int i = 0; i < n; ++i) {
          const int s = i % C::NS;
          const uint64_t qmn = dmn(q_addr + s * C::TILE_BYTES), omn = dmn(o_addr + s * C::TILE_BYTES);
          if (!warp_wait(p_full, i & 1, abort_flag, a.err)) break;
          tc_fence_after();
          // dV += P^T dO: A = P^T (TMEM: each group's bf16 pairs in the first
          // columns of its own GW, 8 columns per 16 queries), B = dO MN-major
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts_w(tbase + C::RV,
                   tbase + C::R0 + (kk * 16 / C::GW) * C::GW + ((kk * 16 % C::GW) / 32) * 16 + (kk & 1) * 8,
                   omn + (kk * 2048 >> 4), id_dkv, !fresh || kk > 0);
          if (!warp_wait(ds_full, i & 1, abort_flag, a.err)) break;
          tc_fence_after();
          // dQ = dS K: A = dS (dS^T read MN-major), B = K MN-major; first, so
          // the drain of dQ overlaps the dK product
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss_w(tbase + C::R1, dsmn + (kk * 2048 >> 4), kmn + (kk * 2048 >> 4), id_dq, kk > 0);
          mma_commit_w(dq_full);
          // dK += dS^T Q: A = dS^T K-major (queries contiguous), B = Q MN-major
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::ATOM_BYTES + (kk & 3) * 32) >> 4;
            mma_ss_w(tbase + C::RK, ds16 + off, qmn + (kk * 2048 >> 4), id_dkv, !fresh || kk > 0);
          }
          mma_commit_w(dk_done);
          fresh = false;
          const bool flush = i + 1 < n && (i + 1) % kFlush == 0;
          if (flush) {
            mma_commit_w(acc_full);
            fresh = true;
          }
          if (i + 1 < n) {
            const int s1 = (i + 1) % C::NS;
            if (!warp_wait(&q_full[s1], ((i + 1) / C::NS) & 1, abort_flag, a.err)) break;
            tc_fence_after();
            mm_s(C::R0, k16, d16(q_addr + s1 * C::TILE_BYTES));  // R0's P^T was read by dV(i), issued earlier
            mma_commit_w(s_full);
            if (!warp_wait(dq_empty, i & 1, abort_flag, a.err)) break;
            tc_fence_after();
            mm_s(C::R1, v16, d16(o_addr + s1 * C::TILE_BYTES));
            mma_commit_w(dp_full);
            if (flush) {
              if (!warp_wait(acc_empty, ((i + 1) / kFlush - 1) & 1, abort_flag, a.err)) break;
              tc_fence_after();
            }
          }
        }
        mma_commit_w(done_bar);
      }
      mma_commit_w(drain);
      mbar_drain(drain, 0, a.err);
    }
  } else if (warp == C::CW + 2) {
    // ------------------------------------------------------------ dQ reducer
    // Adds each staged dQ tile into the fp32 accumulator with TMA bulk tensor
    // reductions and hands the stage back to the producer once it is read.
    {  // the whole warp runs the loop; lane 0 issues
      const uint32_t leader = lane == 0;
      auto warp_wait = [&](uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, err));
      };

      for (int i = 0; i < n; ++i) {
        const int s = i % C::NS;
        if constexpr (C::EARLY_O) {
          // the dO half first: it is staged without waiting for dK(i)
          if (!warp_wait(&staged_o[s], (i / C::NS) & 1, abort_flag, a.err)) break;
          const int4 info = sInfo[s];  // the producer wrote it before the stage's data
          const int qrow = info.x, hc = info.y;
          const bool red_ok = info.w & 2;
#pragma unroll
          for (int box = C::BOXES_PER_STAGE; box < C::DQ_BOXES; ++box)
            if (red_ok)
              tma_reduce_add_3d_p(leader, &tmDQ, sdO + s * C::TILE_BYTES + (box - C::BOXES_PER_STAGE) * C::BOX_BYTES,
                                box * 32, hc, qrow);
        }
        if (!warp_wait(&staged_q[s], (i / C::NS) & 1, abort_flag, a.err)) break;
        const int4 info = sInfo[s];
        const int qrow = info.x, hc = info.y;
        const bool red_ok = info.w & 2;
#pragma unroll
        for (int box = 0; box < (C::EARLY_O ? C::BOXES_PER_STAGE : C::DQ_BOXES); ++box) {
          const uint8_t* base = box < C::BOXES_PER_STAGE
                                    ? sQ + s * C::TILE_BYTES + box * C::BOX_BYTES
                                    : sdO + s * C::TILE_BYTES + (box - C::BOXES_PER_STAGE) * C::BOX_BYTES;
          if (red_ok) tma_reduce_add_3d_p(leader, &tmDQ, base, box * 32, hc, qrow);
        }
        bulk_commit_group_p(leader);
        bulk_wait_read_all_p(leader);
        mbar_arrive_p(leader, &q_empty[s]);
      }
      // the reductions must land before the kernel ends
      bulk_wait_all_p(leader);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;  // query columns [GW grp, GW grp + GW)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row in the pass, query row in the dQ drain
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    // checked build: this key row's dK / dV / accumulator rows lie inside their tensors
    const bool key_ok = row < klen && in_bounds(a.lay.vec(b, k0 + row, kvh, a.hkv) >= 0 &&
                                                    a.lay.vec(b, k0 + row, kvh, a.hkv) <
                                                        static_cast<int64_t>(a.batch) * a.S * a.hkv,
                                                a.err);
    const int64_t krow = a.lay.vec(b, k0 + row, kvh, a.hkv);  // this key row's d-vector in K / dK / dV
    // the first half of the groups own dV, the second dK (keys on lanes), ACC_COLS columns each
    const bool owns_dv = grp < C::GROUPS / 2;
    const int acc_part = C::GROUPS == 2 ? 0 : (owns_dv ? grp : grp - C::GROUPS / 2) * C::ACC_COLS;
    const uint32_t acc_col = (owns_dv ? C::RV : C::RK) + acc_part;
    float* acc_glob = (owns_dv ? a.dv_acc : a.dk_acc) + krow * D + acc_part;
    const float acc_mul = owns_dv ? 1.f : a.scale;
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, a.err));
    };
    for (int i = 0; i < n; ++i) {
      // row statistics of this tile, staged by the producer with Q and dO
      const float* lse_row = sStat + (i % C::NS) * (2 * kTile);
      const float* d_row = lse_row + kTile;
      // ---- P^T = exp2(S^T * scale * log2e - LSE * log2e), two 32-query chunks
      if (!warp_wait(s_full, i & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S^T(i) read Q(i): the stage's descriptor is in place
      const int4 info = sInfo[i % C::NS];
      const int qlen = info.z;
      const bool dg = info.w & 1;
      float pv[C::GCH][32];
      {
        uint32_t sv[C::GCH][32];
#pragma unroll
        for (int ch = 0; ch < C::GCH; ++ch) tmem_ld32(tbase + t_lane + C::R0 + grp * C::GW + ch * 32, sv[ch]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < C::GCH; ++ch)
#pragma unroll
          for (int e = 0; e < 32; ++e) pv[ch][e] = __uint_as_float(sv[ch][e]);
      }
      // Query columns c with lo <= c < hi are live for this key row (causal
      // diagonal, ragged query tile, key row past the block).  Interior tiles
      // have every column live and skip the per-element mask.
      const int lo = dg ? row : 0;
      const int hi = key_ok ? qlen : 0;
      const bool unmasked = __all_sync(0xffffffffu, lo == 0 && hi == kTile);
#pragma unroll
      for (int ch = 0; ch < C::GCH; ++ch) {
        const int cbase = grp * C::GW + ch * 32;  // first query column of the chunk
        uint32_t pk[16];
        if (unmasked) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            // the same query indices in every lane: broadcast shared-memory reads
            const float4 l4 = *reinterpret_cast<const float4*>(lse_row + cbase + e);
            pv[ch][e] = fast_exp2(fmaf(pv[ch][e], a.scale_log2, -l4.x));
            pv[ch][e + 1] = fast_exp2(fmaf(pv[ch][e + 1], a.scale_log2, -l4.y));
            pv[ch][e + 2] = fast_exp2(fmaf(pv[ch][e + 2], a.scale_log2, -l4.z));
            pv[ch][e + 3] = fast_exp2(fmaf(pv[ch][e + 3], a.scale_log2, -l4.w));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse_row + cbase + e);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = cbase + e + u;
              // masked columns may hold statistics of other rows or padding: select
              const float x = fast_exp2(fmaf(pv[ch][e + u], a.scale_log2, -lv[u]));
              pv[ch][e + u] = (c >= lo && c < hi) ? x : 0.f;
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) pk[e / 2] = pack_bf16(pv[ch][e], pv[ch][e + 1]);
        // P^T (bf16 pairs) into this group's own columns of R0,
        // [GW grp + 16 ch, +16): already read by this group, never read by another.
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
            "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(tbase + t_lane + C::R0 + grp * C::GW + ch * 16),
            "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]),
            "r"(pk[8]), "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
            : "memory");
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_p(lane == 0, p_full);

      // ---- dS^T = P^T * (dP^T - D) into shared memory
      if (!warp_wait(dp_full, i & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpv2[C::GCH][32];
#pragma unroll
      for (int ch = 0; ch < C::GCH; ++ch) tmem_ld32(tbase + t_lane + C::R1 + grp * C::GW + ch * 32, dpv2[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < C::GCH; ++ch) {
        const int cbase = grp * C::GW + ch * 32;
        const uint32_t(&dpv)[32] = dpv2[ch];
        uint32_t dsk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(d_row + cbase + e);
          const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float ds[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float p = pv[ch][e + u];
            const float x = p * (__uint_as_float(dpv[e + u]) - dv4[u]);
            // masked columns: p is 0 and D may be another row's or padding
            ds[u] = unmasked ? x : (p != 0.f ? x : 0.f);
          }
          dsk[e / 2] = pack_bf16(ds[0], ds[1]);
          dsk[e / 2 + 1] = pack_bf16(ds[2], ds[3]);
        }
        // dS^T row `row`, queries [cbase, cbase+32): 4 of the 8 16-byte units of
        // the row's 128-byte line in query atom cbase / 64, 128-byte swizzled
        // (written so that GW = 64 folds to constants).
        uint8_t* line = sdS + (grp * C::GW / 64) * C::ATOM_BYTES + row * 128;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const int unit = (grp * C::GW % 64) / 8 + ch * 4 + uu;
          uint4 w;
          w.x = dsk[uu * 4 + 0];
          w.y = dsk[uu * 4 + 1];
          w.z = dsk[uu * 4 + 2];
          w.w = dsk[uu * 4 + 3];
          *reinterpret_cast<uint4*>(line + ((unit ^ (row & 7)) << 4)) = w;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      mbar_arrive_p(lane == 0, ds_full);

      // ---- drain dQ (queries on lanes): TMEM -> registers, R1 released, then
      // staged (fp32, 128-byte swizzled boxes of 32 columns) into this
      // iteration's Q / dO stage once dK(i) no longer reads it, and added into
      // the fp32 accumulator by TMA bulk reductions.
      if (!warp_wait(dq_full, i & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const bool q_ok = row < qlen;
        // this group's GD columns of dQ in runs of RUN (one TMEM load each)
        constexpr int RUN = C::GD >= 32 ? 32 : 16;
        constexpr int NR = C::GD / RUN;
        uint32_t qv[NR][RUN];
#pragma unroll
        for (int cb = 0; cb < NR; ++cb) {
          if constexpr (RUN == 32)
            tmem_ld32(tbase + t_lane + C::R1 + grp * C::GD + cb * RUN, qv[cb]);
          else
            tmem_ld16(tbase + t_lane + C::R1 + grp * C::GD + cb * RUN, qv[cb]);
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_p(lane == 0, dq_empty);
        // groups staging into the Q half wait for dK(i), which may still read
        // it; the others write the dO half, whose last reader dV(i) retired
        // before dQ(i)
        const bool q_half = grp < C::QHALF_GROUPS || !C::EARLY_O;
        if (q_half && !warp_wait(dk_done, i & 1)) {
          ok = false;
          break;
        }
        const int s = i % C::NS;
#pragma unroll
        for (int cb = 0; cb < NR; ++cb) {
          const int col = grp * C::GD + cb * RUN;  // first dQ column of the run
          const int box = col / 32;
          uint8_t* base = box < C::BOXES_PER_STAGE ? sQ + s * C::TILE_BYTES + box * C::BOX_BYTES
                                                   : sdO + s * C::TILE_BYTES + (box - C::BOXES_PER_STAGE) * C::BOX_BYTES;
          uint8_t* line = base + row * 128;
#pragma unroll
          for (int c = 0; c < RUN / 4; ++c) {
            const int unit = (col % 32) / 4 + c;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q_ok)
              x = make_float4(__uint_as_float(qv[cb][c * 4]) * a.scale, __uint_as_float(qv[cb][c * 4 + 1]) * a.scale,
                              __uint_as_float(qv[cb][c * 4 + 2]) * a.scale,
                              __uint_as_float(qv[cb][c * 4 + 3]) * a.scale);
            *reinterpret_cast<float4*>(line + ((unit ^ (row & 7)) << 4)) = x;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive_p(lane == 0, q_half ? &staged_q[s] : &staged_o[s]);
      }

      // ---- every kFlush iterations: fold dV / dK into the fp32 accumulators
      if (i + 1 < n && (i + 1) % kFlush == 0) {
        if (!warp_wait(acc_full, ((i + 1) / kFlush - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < C::ACC_COLS / 32; ++cb) {
          uint32_t v[32];
          tmem_ld32(tbase + t_lane + acc_col + cb * 32, v);
          tmem_wait_ld();
          if (key_ok) {
            float4* dst = reinterpret_cast<float4*>(acc_glob + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              float4 x = dst[v4];
              x.x += __uint_as_float(v[v4 * 4 + 0]) * acc_mul;
              x.y += __uint_as_float(v[v4 * 4 + 1]) * acc_mul;
              x.z += __uint_as_float(v[v4 * 4 + 2]) * acc_mul;
              x.w += __uint_as_float(v[v4 * 4 + 3]) * acc_mul;
              dst[v4] = x;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        mbar_arrive_p(lane == 0, acc_empty);
      }
    }
    // ---------------------------------------------------------- epilogue
    if (ok) ok = warp_wait(done_bar, 0);
    if (ok) {
      tc_fence_after();
      // the accumulator holds earlier flushes (FUSED) or earlier steps (STEPWISE)
      const bool add_glob = STEP || nflush > 0;
#pragma unroll 1
      for (int cb = 0; cb < C::ACC_COLS / 32; ++cb) {
        uint32_t v[32];
        tmem_ld32(tbase + t_lane + acc_col + cb * 32, v);
        tmem_wait_ld();
        if (key_ok) {
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]) * acc_mul;
          if (add_glob) {
            const float4* src = reinterpret_cast<const float4*>(acc_glob + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              const float4 y = src[v4];
              x[v4 * 4 + 0] += y.x;
              x[v4 * 4 + 1] += y.y;
              x[v4 * 4 + 2] += y.z;
              x[v4 * 4 + 3] += y.w;
            }
          }
          if constexpr (!STEP) {
            __nv_bfloat16* dst = (owns_dv ? a.dv : a.dk) + krow * D + acc_part + cb * 32;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16(x[v4 * 8 + 0], x[v4 * 8 + 1]);
              w.y = pack_bf16(x[v4 * 8 + 2], x[v4 * 8 + 3]);
              w.z = pack_bf16(x[v4 * 8 + 4], x[v4 * 8 + 5]);
              w.w = pack_bf16(x[v4 * 8 + 6], x[v4 * 8 + 7]);
              reinterpret_cast<uint4*>(dst)[v4] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(acc_glob + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(x[v4 * 4], x[v4 * 4 + 1], x[v4 * 4 + 2], x[v4 * 4 + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::CW + 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool STEP>
int launch_bwd_t(const loong_attn_desc& d, const void* q, const void* k, const void* v, const void* dout,
                 const float* stats, float* dq_acc, void* dk, void* dv, float* dk_acc,
                 float* dv_acc, cudaStream_t stream, void* kv_recv) {
  using C = BwdCfg<D>;
  const Layout lay = layout_of(d);
  const int64_t rows = lay.view_rows(d.batch);
  const int vq = lay.view_heads(d.hq), vkv = lay.view_heads(d.hkv);
  CUtensorMap mq, mk, mv, mo;
  int st;
  if ((st = make_head_tile_map(&mq, q, rows, vq, D)) != LOONG_OK) return st;
  if ((st = make_head_tile_map(&mk, k, rows, vkv, D)) != LOONG_OK) return st;
  if ((st = make_head_tile_map(&mv, v, rows, vkv, D)) != LOONG_OK) return st;
  if ((st = make_head_tile_map(&mo, dout, rows, vq, D)) != LOONG_OK) return st;
  CUtensorMap mdq;
  if ((st = make_f32_tile_map(&mdq, dq_acc, rows, vq, D)) != LOONG_OK) return st;
  BwdArgs a;
  a.lay = lay;
  a.kv_held = 0;
  a.batch = static_cast<int>(d.batch);
  a.S = static_cast<int>(d.seqlen);
  a.hq = d.hq;
  a.hkv = d.hkv;
  a.G = d.hq / d.hkv;
  a.ring = ring_geom(d);
  a.scale = d.softmax_scale > 0.f ? d.softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  a.scale_log2 = a.scale * kLog2e;
  a.lse2 = stats;
  a.blk_pad = stat_block_pad(a.ring.blk);
  a.stat_len = static_cast<int>(stat_row_len(a.ring));
  a.dstat = stats + d.batch * d.hq * static_cast<int64_t>(a.stat_len);
  a.dq_acc = dq_acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  a.err = device_error_word();
  if (!a.err) return LOONG_ERR_CUDA;
  auto kern = ring_bwd_kernel<D, STEP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t grid = d.batch * d.hkv * static_cast<int64_t>(a.ring.nblocks) * a.ring.ntile;
  if (grid <= 0 || grid > 0x7fffffff) return LOONG_ERR_INVALID_ARG;
  const int t_first = 0, t_last = d.cp;
  if (!STEP) {
    a.t_begin = t_first;
    a.t_end = t_last;
    record_start(stream);
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, mo, mdq, a);
    record_stop(stream);
    return check_launch();
  }
  if (is_copy_mode(d)) {
    // receive buffers K0, K1, V0, V1, each the size of K (exchange.h); dK, dV
    // are accumulated at the owner's rows, so only K and V travel
    const size_t kv_bytes = static_cast<size_t>(rows) * vkv * D * 2;
    uint8_t* rb = static_cast<uint8_t*>(kv_recv);
    void* const rk[2] = {rb, rb + kv_bytes};
    void* const rv[2] = {rb + 2 * kv_bytes, rb + 3 * kv_bytes};
    CUtensorMap mkr[2], mvr[2];
    for (int i = 0; i < 2; ++i) {
      if ((st = make_head_tile_map(&mkr[i], rk[i], rows, vkv, D)) != LOONG_OK) return st;
      if ((st = make_head_tile_map(&mvr[i], rv[i], rows, vkv, D)) != LOONG_OK) return st;
    }
    record_start(stream);
    st = run_exchanged_steps(d, k, v, rk, rv, stream, [&](int t, int buf) {
      NvtxRange step("bwd ring step %d", t);
      a.t_begin = t;
      a.t_end = t + 1;
      a.kv_held = buf >= 0;
      kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(
          mq, buf >= 0 ? mkr[buf] : mk, buf >= 0 ? mvr[buf] : mv, mo, mdq, a);
      return check_launch();
    });
    record_stop(stream);
    return st;
  }
  record_start(stream);
  for (int t = t_first; t < t_last; ++t) {
    NvtxRange step("bwd ring step %d", t);
    a.t_begin = t;
    a.t_end = t + 1;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, mo, mdq, a);
    if ((st = check_launch()) != LOONG_OK) return st;
  }
  record_stop(stream);
  return LOONG_OK;
}

}  // namespace

int launch_bwd(const loong_attn_desc& d, const void* q, const void* k, const void* v, const void* o,
               const void* o_res, const float* lse, const void* dout, void* dq, void* dk, void* dv, float* dq_acc, float* dvec,
               float* dk_acc, float* dv_acc, cudaStream_t stream, void* kv_recv) {
  const int64_t q_elems = d.batch * d.seqlen * d.hq * d.head_dim;
  const int64_t kv_elems = d.batch * d.seqlen * d.hkv * d.head_dim;
  const bool step = d.mode != LOONG_MODE_FUSED;
  int st;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(q_elems) * 4, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemsetAsync(dk_acc, 0, static_cast<size_t>(kv_elems) * 4, stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(dv_acc, 0, static_cast<size_t>(kv_elems) * 4, stream)) != cudaSuccess)
    return cuda_fail(e);
  if ((st = launch_bwd_rowstats(d, o, o_res, dout, lse, dvec, stream)) != LOONG_OK) return st;
  if (d.head_dim == 128)
    st = step ? launch_bwd_t<128, true>(d, q, k, v, dout, dvec, dq_acc, dk, dv, dk_acc, dv_acc, stream, kv_recv)
              : launch_bwd_t<128, false>(d, q, k, v, dout, dvec, dq_acc, dk, dv, dk_acc, dv_acc, stream, kv_recv);
  else if (d.head_dim == 64)
    st = step ? launch_bwd_t<64, true>(d, q, k, v, dout, dvec, dq_acc, dk, dv, dk_acc, dv_acc, stream, kv_recv)
              : launch_bwd_t<64, false>(d, q, k, v, dout, dvec, dq_acc, dk, dv, dk_acc, dv_acc, stream, kv_recv);
  else
    return LOONG_ERR_UNSUPPORTED;
  if (st != LOONG_OK) return st;
  if ((st = launch_f32_to_bf16(dq_acc, dq, q_elems, stream)) != LOONG_OK) return st;
  if (step) {
    if ((st = launch_f32_to_bf16(dk_acc, dk, kv_elems, stream)) != LOONG_OK) return st;
    if ((st = launch_f32_to_bf16(dv_acc, dv, kv_elems, stream)) != LOONG_OK) return st;
  }
  return LOONG_OK;
}

}  // namespace loong
