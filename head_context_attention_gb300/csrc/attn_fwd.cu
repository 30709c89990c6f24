// attn_fwd.cu -- forward ring-step attention on tcgen05 tensor cores.
//
// One CTA owns one 128-token query tile of two query heads that share a kv
// head, and walks the key tiles that tile meets along its ring pass (ring.cuh)
// in ring order.  Per key tile j and query head h:
//   S_h = Q_h K_j^T                 tcgen05.mma, operands in shared memory
//   P_h = exp2(S_h*scale*log2e - m) softmax warps, one thread per query row
//   O_h += P_h V_j                  tcgen05.mma, P from tensor memory
// with a running row maximum m and row sum l.  The P V product takes fp16
// operands: P as fp16 (scaled by 2^7, so that the largest probability, at most
// 2^8 relative to the running maximum, sits near the top of fp16's range and
// small ones stay clear of its subnormals) and V as the fp16 copy V * 2^-e the
// launcher prepares (v16_shift); the epilogue removes both scalings exactly.
// fp16's 11 significant bits keep O within about 2^-12 of its exact value,
// which lets the backward form D = rowsum(dO * O) from O and its rounding
// residual (o_res) to that precision.  The per-step "merge" of
// [G] "Guide to LoongTrain", "Step 3" (partial results of successive ring
// steps) is the online-softmax update itself: O and l carry the reference
// maximum m, and a step whose maximum exceeds m by more than 2^8 rescales O
// and l to the new maximum, which is the log-sum-exp merge written in
// unnormalised form.  After a row's first tile the softmax forms P against the
// running maximum straight away and computes the tile's maximum only when
// some row of the warp sums to 2^15 or more: a smaller sum bounds every P of
// the row by 2^15, so no score passed m by more than 2^8.  A row whose sum
// reached the bound then takes the tile's maximum as its reference, so its
// later tiles pass the test again.  In STEPWISE mode
// the launch covers one ring step and the epilogue merges the step's
// normalised result into an fp32 accumulator by log-sum-exp.  Non-causal
// descriptors walk every key tile and mask only the ragged tail of a block.
// Q, K, V and O are addressed through a Layout (natural or rank-major,
// ring.cuh); in STEPWISE_COPY modes K and V are read from the query rank's
// plane of the receive buffers the exchange filled (exchange.h).  A launch may
// cover the query rows of a range of ring ranks.
//
// Warp roles (320 threads): warps 0-3 softmax for head slot 0, warps 4-7 for
// head slot 1 (warp w reads TMEM lanes 32*(w%4)..+31, the rows it owns),
// warp 8 issues TMA loads, warp 9 allocates TMEM and issues the MMAs.
// Tensor memory (512 columns): NSB score buffers of 128 columns, then O_0 and
// O_1 (d columns each).  The MMA jobs (key tile j, head h) run in the order
// J = 2j + h and job J's scores go to buffer J mod NSB; P overwrites the first
// 64 columns of its buffer as fp16 pairs.  Job J's Q K^T is issued right after
// job J - NSB's P V (tcgen05 operations issued by one thread execute in
// order, so the buffer is free by then).  With NSB = 2 (d = 128, where O
// takes the rest of tensor memory) a head's next scores wait for its own P V;
// with NSB = 3 (d = 64) they are computed while the softmax still works on the
// current tile, and a softmax that rescales O_h first waits for the previous
// P V into O_h.
#include <cuda_bf16.h>

#include <cmath>

#include "exchange.h"
#include "internal.h"
#include "ptx.cuh"

namespace loong {

namespace {

template <int D>
struct FwdCfg {
  static constexpr int NQ = 2;                     // query tiles (heads) per CTA
  static constexpr int NS = D == 128 ? 2 : 4;      // K and V pipeline stages
  static constexpr int ATOMS = D / 64;             // 128-byte swizzle atoms per row
  static constexpr int ATOM_BYTES = kTile * 128;   // one atom column of a tile
  static constexpr int TILE_BYTES = kTile * D * 2;
  static constexpr int NSB = D == 64 ? 3 : 2;      // score buffers in tensor memory
  static constexpr int NBARS = 1 + 4 * NS + 3 + 3 + 2 + 2;
  static constexpr int SMEM_BYTES = (NQ + 2 * NS) * TILE_BYTES + NBARS * 8 + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t S_COL(int buf) { return static_cast<uint32_t>(buf) * 128u; }
  __host__ __device__ static constexpr uint32_t O_COL(int h) { return NSB * 128u + static_cast<uint32_t>(h) * D; }
  static_assert(NSB * 128 + 2 * D <= 512, "tensor memory");
};

struct FwdArgs {
  int batch, S, hq, hkv, G, npairs;
  RingGeom ring;
  Layout lay;                  // where Q, K, V, O keep (token, head)
  int rank_begin, rank_end;    // ring ranks whose query rows this launch computes
  int kv_held;                 // K, V are receive buffers: read the query rank's plane
  int t_begin, t_end;
  float scale_log2;
  __nv_bfloat16* o;
  __nv_bfloat16* o_res;    // FUSED: bf16 rounding residual of O, or null
  float* lse;
  float* o_acc;            // STEPWISE accumulator, else null
  const unsigned* v_amax;  // bit pattern of max |V|: V was stored as V * 2^-v16_shift
  unsigned* err;
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// P is formed as exp2(x + kPBias): with the lazy rescale every probability is at
// most 2^8 relative to the running maximum, so fp16 P stays below 2^15.
constexpr float kPBias = 7.0f;
// A tile's row sum of P below this bounds each of its P by the same value:
// 2^(bias + threshold), the largest P the lazy rescale lets through.
constexpr float kSumBound = 32768.0f;
static_assert(kSumBound == float(1 << int(kPBias + kRescaleThreshold)), "sum bound = 2^(bias + threshold)");

template <int D, bool STEP>
__global__ void __launch_bounds__(320, 1)
    ring_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::NQ * C::TILE_BYTES;
  uint8_t* sV = sK + C::NS * C::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + C::NS * C::TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::NS;
  uint64_t* v_full = k_empty + C::NS;
  uint64_t* v_empty = v_full + C::NS;
  uint64_t* s_full = v_empty + C::NS;  // NSB: scores in the buffer (MMA -> softmax of its head)
  // NSB: P of the buffer's job stored (softmax -> MMA).  Per buffer, not per
  // head: a head's softmax may finish two tiles before the MMA warp takes the
  // first P, but a buffer's next P needs that buffer's next scores, issued
  // only after the MMA warp has taken this one.
  uint64_t* p_full = s_full + 3;
  uint64_t* pv_done = p_full + 3;      // 2: O_h += P V done (MMA -> softmax, before a rescale)
  uint64_t* o_final = pv_done + 2;
  uint64_t* drain = o_final + 1;
  volatile int* abort_flag = &abort_sh;

  // ---- work item: (batch, kv head, query tile, head pair); heavy tiles first.
  // The query blocks of ring ranks [rank_begin, rank_end) in decreasing order:
  // B blocks 2cp-1-c (paired placement), then A blocks c.
  const RingGeom& g = a.ring;
  int idx = blockIdx.x;
  const int hpair = idx % a.npairs;
  idx /= a.npairs;
  const int nr = a.rank_end - a.rank_begin;
  const int nqt = nr * rank_parts(g) * g.ntile;
  const int r = idx % nqt;
  idx /= nqt;
  const int kvh = idx % a.hkv;
  const int b = idx / a.hkv;
  const int jb = r / g.ntile;
  const int bq = (g.zigzag && jb < nr) ? 2 * g.cp - 1 - a.rank_begin - jb
                                       : a.rank_end - 1 - (g.zigzag ? jb - nr : jb);
  const int qi = g.ntile - 1 - r % g.ntile;
  const int q0 = bq * g.blk + qi * kTile;
  const int qlen = min(kTile, (bq + 1) * g.blk - q0);
  const int head0 = kvh * a.G + 2 * hpair;
  const bool dup = head0 + 1 >= (kvh + 1) * a.G;  // odd group: slot 1 repeats slot 0
  const int head1 = dup ? head0 : head0 + 1;

  KvWalk walk;
  walk.init(g, bq, qi, a.t_begin, a.t_end);
  const int n = walk.total();
  if (n == 0) return;  // uniform over the CTA: nothing of this tile in these steps

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int sb = 0; sb < C::NSB; ++sb) {
      mbar_init(&s_full[sb], 1);
      mbar_init(&p_full[sb], 4);
    }
    for (int h = 0; h < 2; ++h) mbar_init(&pv_done[h], 1);
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_sh;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(q_full, C::NQ * C::TILE_BYTES);
      for (int h = 0; h < C::NQ; ++h) {
        int hc;
        const int64_t qr64 = a.lay.view_row(b, q0, h ? head1 : head0, a.hq, hc);
        // checked build: the tile starts inside the tensor (TMA fills rows past its end with zeros)
        in_bounds(qr64 >= 0 && qr64 < a.lay.view_rows(a.batch) && hc >= 0 && hc < a.lay.view_heads(a.hq), a.err);
        const int qr = static_cast<int>(qr64);
        for (int at = 0; at < C::ATOMS; ++at)
          tma_load_3d(sQ + h * C::TILE_BYTES + at * C::ATOM_BYTES, &tmQ, q_full, at * 64, hc, qr);
      }
      int jk = 0, jv = 0;
      const int c_q = block_owner(g, bq);  // the query tile's ring rank
      for (int j = 0; j < n; ++j, walk.advance()) {
        const int s = j % C::NS;
        const int u = j / C::NS;
        int kvc;
        const int64_t k064 = a.kv_held ? a.lay.view_row_held(b, walk.k0(), kvh, a.hkv, c_q, kvc)
                                       : a.lay.view_row(b, walk.k0(), kvh, a.hkv, kvc);
        in_bounds(k064 >= 0 && k064 < a.lay.view_rows(a.batch) && kvc >= 0 && kvc < a.lay.view_heads(a.hkv), a.err);
        const int k0 = static_cast<int>(k064);
        if (j >= C::NS && !mbar_wait(&k_empty[s], (u - 1) & 1, abort_flag, a.err)) break;
        mbar_expect_tx(&k_full[s], C::TILE_BYTES);
        for (int at = 0; at < C::ATOMS; ++at)
          tma_load_3d(sK + s * C::TILE_BYTES + at * C::ATOM_BYTES, &tmK, &k_full[s], at * 64, kvc, k0);
        ++jk;
        if (j >= C::NS && !mbar_wait(&v_empty[s], (u - 1) & 1, abort_flag, a.err)) break;
        mbar_expect_tx(&v_full[s], C::TILE_BYTES);
        for (int at = 0; at < C::ATOMS; ++at)
          tma_load_3d(sV + s * C::TILE_BYTES + at * C::ATOM_BYTES, &tmV, &v_full[s], at * 64, kvc, k0);
        ++jv;
      }
      // Let every copy this thread issued land before the CTA can exit.
      mbar_drain(q_full, 0, a.err);
      for (int s = 0; s < C::NS; ++s) {
        const int nk = jk > s ? (jk - 1 - s) / C::NS + 1 : 0;
        const int nv = jv > s ? (jv - 1 - s) / C::NS + 1 : 0;
        if (nk) mbar_drain(&k_full[s], (nk - 1) & 1, a.err);
        if (nv) mbar_drain(&v_full[s], (nv - 1) & 1, a.err);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the loop; one elected lane issues
      auto warp_wait = [&](uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, err));
      };
      constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_f16(128, D, false, true);  // P and V in fp16
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      // Descriptors built once per tile: an operand's descriptor at byte offset
      // `off` is its base descriptor plus off / 16 (the 14-bit address field
      // cannot carry: every shared-memory address is below 256 KB).
      auto qk = [&](int h, int s, int buf) {
        const uint64_t qa = sdesc_sw128(q_addr + h * C::TILE_BYTES, 16, 1024);
        const uint64_t kb = sdesc_sw128(k_addr + s * C::TILE_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::ATOM_BYTES + (kk & 3) * 32) >> 4;
          mma_ss_w(tbase + C::S_COL(buf), qa + off, kb + off, id_qk, kk > 0);
        }
      };
      auto pv = [&](int h, int s, int buf, bool acc) {
        const uint64_t vb = sdesc_sw128(v_addr + s * C::TILE_BYTES, C::ATOM_BYTES, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts_w(tbase + C::O_COL(h), tbase + C::S_COL(buf) + kk * 8, vb + (kk * 2048 >> 4), id_pv, acc || kk > 0);
      };
      // Q K^T of job J = 2 jt + h into buffer J mod NSB; K(jt) is released
      // after its second head
      auto issue_qk = [&](int J) {
        const int jt = J >> 1, h = J & 1, st = jt % C::NS;
        if (h == 0) {
          if (!warp_wait(&k_full[st], (jt / C::NS) & 1, abort_flag, a.err)) return false;
          tc_fence_after();
        }
        qk(h, st, J % C::NSB);
        mma_commit_w(&s_full[J % C::NSB]);
        if (h == 1) mma_commit_w(&k_empty[st]);
        return true;
      };
      bool ok = warp_wait(q_full, 0, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        for (int J = 0; J < C::NSB && J < 2 * n && ok; ++J) ok = issue_qk(J);
        for (int j = 0; j < n && ok; ++j) {
          const int s = j % C::NS;
          if (!warp_wait(&v_full[s], (j / C::NS) & 1, abort_flag, a.err)) break;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int J = 2 * j + h;
            if (!warp_wait(&p_full[J % C::NSB], (J / C::NSB) & 1, abort_flag, a.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(h, s, J % C::NSB, j > 0);
            mma_commit_w(&pv_done[h]);
            if (h == 1) mma_commit_w(&v_empty[s]);
            if (J + C::NSB < 2 * n && !issue_qk(J + C::NSB)) {
              ok = false;
              break;
            }
          }
        }
        mma_commit_w(o_final);
      }
      // Every MMA this warp issued must finish before TMEM is released.
      mma_commit_w(drain);
      mbar_drain(drain, 0, a.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int h = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tbase + t_lane + C::O_COL(h);
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j, walk.advance()) {
      // Lanes leave together so the .sync.aligned TMEM accesses never diverge.
      const int J = 2 * j + h;  // this tile's MMA job and its score buffer
      const uint32_t tS = tbase + t_lane + C::S_COL(J % C::NSB);
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[J % C::NSB], (J / C::NSB) & 1, abort_flag, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
      const int klen = walk.klen();
      const bool dg = walk.diag();
      // the tile's scores, masked columns at -inf (read again by the full path)
      auto load_s = [&]() {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tmem_ld32(tS + cb * 32, sr[cb]);
        tmem_wait_ld();
        if (dg || klen < kTile) {
          const int lim = dg ? min(row, klen - 1) : klen - 1;
#pragma unroll
          for (int cb = 0; cb < 4; ++cb)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb * 32 + i > lim) sr[cb][i] = __float_as_uint(-INFINITY);
        }
      };
      load_s();
      // P = exp2(s*scale*log2e - ref + bias) for the whole tile, with the
      // columns in pairs on the paired fp32 pipe; returns this row's sum of P
      // (l carries the factor 2^bias as well)
      uint32_t pk[2][32];
      auto form_p = [&](float ref) {
        const float2 sl2v = make_float2(sl2, sl2), nref = make_float2(kPBias - ref, kPBias - ref);
        float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[cb][i]), __uint_as_float(sr[cb][i + 1])),
                                        sl2v, nref);
            const float p0 = fast_exp2(x.x);
            const float p1 = fast_exp2(x.y);
            lsum = __fadd2_rn(lsum, make_float2(p0, p1));
            pk[cb >> 1][(cb & 1) * 16 + (i >> 1)] = pack_f16(p0, p1);
          }
        return lsum.x + lsum.y;
      };
      // After the first tile, P is first formed against the running maximum.
      // A row sum below 2^(bias + threshold) bounds every P of the row by the
      // same value, so no column passed the running maximum by more than the
      // threshold: nothing to rescale, and the row maximum is not needed.
      // Otherwise (or on NaN) the warp takes the full path below.
      bool full = j == 0;
      bool over = false;  // this row's sum reached the bound
      if (!full) {
        const float ts = form_p(m_run);
        over = !(ts < kSumBound);
        full = __any_sync(0xffffffffu, over);
        if (!full) l_run += ts;
      }
      if (full) {
        if (j > 0) load_s();  // P of this tile is not stored yet: the scores are still in place
        // row maximum, two new columns per (three-input) max
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            mx0 = fmax3(mx0, __uint_as_float(sr[cb][i]), __uint_as_float(sr[cb][i + 1]));
            mx1 = fmax3(mx1, __uint_as_float(sr[cb][i + 2]), __uint_as_float(sr[cb][i + 3]));
          }
        const float m_tile = fmaxf(mx0, mx1) * sl2;
        const float m_new = fmaxf(m_run, m_tile);
        // A row whose sum reached the bound takes the new maximum even below the
        // threshold (its maximum is then above the reference): a reference
        // left low would send the warp down this path on every later tile.
        const bool rescale = j > 0 && m_new > m_run + (over ? 0.f : kRescaleThreshold);
        if (j == 0) m_run = m_new;
        // The decision is per row, but TMEM loads and stores are warp-collective:
        // the whole warp takes the branch, rows that need none scale by 1.
        if (__any_sync(0xffffffffu, rescale)) {
          // O_h must hold the previous tile's P V: with two buffers the commit
          // that signalled these scores follows it; with three, wait for it
          // (completion j - 1 of pv_done[h]; completion j needs this tile's P)
          if (C::NSB > 2 && !__all_sync(0xffffffffu, mbar_wait(&pv_done[h], (j - 1) & 1, abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? fast_exp2(m_run - m_new) : 1.f;
          l_run *= f;
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t orow[32];
            tmem_ld32(tO + cb * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * f);
            tmem_st32(tO + cb * 32, orow);
          }
          if (rescale) m_run = m_new;
        }
        l_run += form_p(m_run == -INFINITY ? 0.f : m_run);
      }
      tmem_st32(tS, pk[0]);
      tmem_st32(tS + 32, pk[1]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[J % C::NSB]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final, 0, abort_flag, a.err));
    if (ok) {
      tc_fence_after();
      const int head = h ? head1 : head0;
      const int64_t qv = a.lay.vec(b, q0 + row, head, a.hq);  // this row's d-vector in Q / O
      const int64_t lse_i = (static_cast<int64_t>(b) * a.hq + head) * a.S + (q0 + row);
      // checked build: the row's O, accumulator and LSE entries lie inside their tensors
      const bool valid = row < qlen && !(h == 1 && dup) &&
                         in_bounds(qv >= 0 && qv < static_cast<int64_t>(a.batch) * a.S * a.hq && lse_i >= 0 &&
                                       lse_i < static_cast<int64_t>(a.batch) * a.hq * a.S,
                                   a.err);
      // l_run and O carry 2^kPBias; O also carries V's 2^-e
      const float lse_p = l_run > 0.f ? (m_run + log2f(l_run) - kPBias) * kLn2 : -INFINITY;
      const float o_mul = __int_as_float((127 + v16_shift(*a.v_amax)) << 23);  // 2^e
      float* lse_ptr = a.lse + lse_i;
      if constexpr (!STEP) {
        const float inv = l_run > 0.f ? o_mul / l_run : 0.f;
        __nv_bfloat16* orow = a.o + qv * D;
        __nv_bfloat16* rrow = a.o_res ? a.o_res + qv * D : nullptr;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t ov[32];
          tmem_ld32(tO + cb * 32, ov);
          tmem_wait_ld();
          if (valid) {
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(ov[e]) * inv;
            uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16(x[v4 * 8 + 0], x[v4 * 8 + 1]);
              w.y = pack_bf16(x[v4 * 8 + 2], x[v4 * 8 + 3]);
              w.z = pack_bf16(x[v4 * 8 + 4], x[v4 * 8 + 5]);
              w.w = pack_bf16(x[v4 * 8 + 6], x[v4 * 8 + 7]);
              dst[v4] = w;
            }
            if (rrow) {
              // x - bf16(x) is exact in fp32; rounded once more to bf16 it
              // carries the next 8 bits of O
              uint4* rdst = reinterpret_cast<uint4*>(rrow + cb * 32);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                uint32_t r[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float a0 = x[v4 * 8 + 2 * u], a1 = x[v4 * 8 + 2 * u + 1];
                  r[u] = pack_bf16(a0 - __bfloat162float(__float2bfloat16_rn(a0)),
                                   a1 - __bfloat162float(__float2bfloat16_rn(a1)));
                }
                rdst[v4] = make_uint4(r[0], r[1], r[2], r[3]);
              }
            }
          }
        }
        if (valid) *lse_ptr = lse_p;
      } else {
        // Log-sum-exp merge of this step's (O_p, L_p) into (O_acc, L_acc).
        float ca = 0.f, cpart = 0.f, lse_new = -INFINITY;
        if (valid) {
          const float la = *lse_ptr;
          const float mm = fmaxf(la, lse_p);
          const float wa = la == -INFINITY ? 0.f : exp2f((la - mm) * kLog2e);
          const float wp = lse_p == -INFINITY ? 0.f : exp2f((lse_p - mm) * kLog2e);
          const float tot = wa + wp;
          if (tot > 0.f) {
            ca = wa / tot;
            cpart = wp * o_mul / (tot * l_run);
            lse_new = mm + log2f(tot) * kLn2;
          }
        }
        float* acc = a.o_acc + qv * D;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t ov[32];
          tmem_ld32(tO + cb * 32, ov);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(acc + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              float4 x = dst[v4];
              x.x = ca * x.x + cpart * __uint_as_float(ov[v4 * 4 + 0]);
              x.y = ca * x.y + cpart * __uint_as_float(ov[v4 * 4 + 1]);
              x.z = ca * x.z + cpart * __uint_as_float(ov[v4 * 4 + 2]);
              x.w = ca * x.w + cpart * __uint_as_float(ov[v4 * 4 + 3]);
              dst[v4] = x;
            }
          }
        }
        if (valid) *lse_ptr = lse_new;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool STEP>
int launch_fwd_t(const loong_attn_desc& d, const void* q, const void* k, void* o,
                 float* lse, const FwdScratch& sc, cudaStream_t stream, int rank_begin, int rank_end) {
  using C = FwdCfg<D>;
  const Layout lay = layout_of(d);
  const int64_t rows = lay.view_rows(d.batch);
  CUtensorMap mq, mk, mv;
  int st;
  // V is read as its fp16 copy (the map moves 2-byte elements either way)
  const void* v = sc.v16;
  if ((st = make_head_tile_map(&mq, q, rows, lay.view_heads(d.hq), D)) != LOONG_OK) return st;
  if ((st = make_head_tile_map(&mk, k, rows, lay.view_heads(d.hkv), D)) != LOONG_OK) return st;
  if ((st = make_head_tile_map(&mv, v, rows, lay.view_heads(d.hkv), D)) != LOONG_OK) return st;
  void* kv_recv = sc.kv_recv;

  FwdArgs a;
  a.batch = static_cast<int>(d.batch);
  a.S = static_cast<int>(d.seqlen);
  a.hq = d.hq;
  a.hkv = d.hkv;
  a.G = d.hq / d.hkv;
  a.npairs = (a.G + 1) / 2;
  a.ring = ring_geom(d);
  a.lay = lay;
  a.rank_begin = rank_begin;
  a.rank_end = rank_end;
  a.kv_held = 0;
  const float scale = d.softmax_scale > 0.f ? d.softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  a.scale_log2 = scale * kLog2e;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.o_res = static_cast<__nv_bfloat16*>(sc.o_res);
  a.lse = lse;
  a.o_acc = sc.o_acc;
  a.v_amax = sc.v_amax;
  a.err = device_error_word();
  if (!a.err) return LOONG_ERR_CUDA;

  auto kern = ring_fwd_kernel<D, STEP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t grid = d.batch * d.hkv * static_cast<int64_t>(rank_end - rank_begin) * rank_parts(a.ring) *
                       a.ring.ntile * a.npairs;
  if (grid <= 0 || grid > 0x7fffffff) return LOONG_ERR_INVALID_ARG;
  if (!STEP) {
    a.t_begin = 0;
    a.t_end = d.cp;
    record_start(stream);
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, a);
    record_stop(stream);
    return check_launch();
  }
  if (is_copy_mode(d)) {
    // receive buffers K0, K1, V0, V1, each the size of K
    const size_t kv_bytes = static_cast<size_t>(rows) * lay.view_heads(d.hkv) * D * 2;
    uint8_t* rb = static_cast<uint8_t*>(kv_recv);
    void* const rk[2] = {rb, rb + kv_bytes};
    void* const rv[2] = {rb + 2 * kv_bytes, rb + 3 * kv_bytes};
    CUtensorMap mkr[2], mvr[2];
    for (int i = 0; i < 2; ++i) {
      if ((st = make_head_tile_map(&mkr[i], rk[i], rows, lay.view_heads(d.hkv), D)) != LOONG_OK) return st;
      if ((st = make_head_tile_map(&mvr[i], rv[i], rows, lay.view_heads(d.hkv), D)) != LOONG_OK) return st;
    }
    record_start(stream);
    st = run_exchanged_steps(d, k, v, rk, rv, stream, [&](int t, int buf) {
      NvtxRange step("fwd ring step %d", t);
      a.t_begin = t;
      a.t_end = t + 1;
      a.kv_held = buf >= 0;
      kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(mq, buf >= 0 ? mkr[buf] : mk,
                                                                               buf >= 0 ? mvr[buf] : mv, a);
      return check_launch();
    });
    record_stop(stream);
    return st;
  }
  record_start(stream);
  for (int t = 0; t < d.cp; ++t) {
    NvtxRange step("fwd ring step %d", t);
    a.t_begin = t;
    a.t_end = t + 1;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, a);
    if ((st = check_launch()) != LOONG_OK) return st;
  }
  record_stop(stream);
  return LOONG_OK;
}

}  // namespace

int launch_fwd(const loong_attn_desc& d, const void* q, const void* k, const void* v, void* o,
               float* lse, const FwdScratch& sc, cudaStream_t stream, int rank_begin, int rank_end) {
  const bool step = d.mode != LOONG_MODE_FUSED;
  if (rank_end < 0) rank_end = d.cp;
  int st;
  if ((st = launch_v_to_f16(v, sc.v16, sc.v_amax, d.batch * d.seqlen * d.hkv * d.head_dim, stream)) != LOONG_OK)
    return st;
  if (d.head_dim == 128)
    return step ? launch_fwd_t<128, true>(d, q, k, o, lse, sc, stream, rank_begin, rank_end)
                : launch_fwd_t<128, false>(d, q, k, o, lse, sc, stream, rank_begin, rank_end);
  if (d.head_dim == 64)
    return step ? launch_fwd_t<64, true>(d, q, k, o, lse, sc, stream, rank_begin, rank_end)
                : launch_fwd_t<64, false>(d, q, k, o, lse, sc, stream, rank_begin, rank_end);
  return LOONG_ERR_UNSUPPORTED;
}

}  // namespace loong
