// stream_ops.cu -- bandwidth-bound kernels: the n-way log-sum-exp merge, the
// Ulysses head-context repack, the backward's D = rowsum(dO * O), fills and
// the fp32 -> bf16 conversion of accumulators.  Each thread moves 16-byte
// vectors; grids are sized in multiples of the SM count and stride over the
// work.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace loong {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

unsigned grid_for(int64_t work_items, int threads, int per_sm) {
  const int64_t want = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * per_sm;
  int64_t g = want < cap ? want : cap;
  if (g < 1) g = 1;
  return static_cast<unsigned>(g);
}

__global__ void fill_f32_kernel(float* p, int64_t n, float value) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride)
    p[i] = value;
}

__device__ __forceinline__ float bf16_residual(float x) {
  return x - __bfloat162float(__float2bfloat16_rn(x));
}

// n % 8 == 0 handled by the vector path; the tail element by element.  With
// res, also the rounding residual bf16(x - bf16(x)) (exact before its own
// rounding).
__global__ void f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                   __nv_bfloat16* __restrict__ res, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t nv = n / 8;
  const float4* in4 = reinterpret_cast<const float4*>(in);
  uint4* out4 = reinterpret_cast<uint4*>(out);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nv; i += stride) {
    const float4 a = in4[2 * i], b = in4[2 * i + 1];
    uint4 w;
    w.x = pack_bf16(a.x, a.y);
    w.y = pack_bf16(a.z, a.w);
    w.z = pack_bf16(b.x, b.y);
    w.w = pack_bf16(b.z, b.w);
    out4[i] = w;
    if (res) {
      uint4 r;
      r.x = pack_bf16(bf16_residual(a.x), bf16_residual(a.y));
      r.y = pack_bf16(bf16_residual(a.z), bf16_residual(a.w));
      r.z = pack_bf16(bf16_residual(b.x), bf16_residual(b.y));
      r.w = pack_bf16(bf16_residual(b.z), bf16_residual(b.w));
      reinterpret_cast<uint4*>(res)[i] = r;
    }
  }
  for (int64_t i = nv * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += stride) {
    out[i] = __float2bfloat16_rn(in[i]);
    if (res) res[i] = __float2bfloat16_rn(bf16_residual(in[i]));
  }
}

// max |x| over the n bf16 values of `in` (n % 8 == 0), as the bit pattern of
// a non-negative float, atomically maxed into *amax (zeroed by the caller).
// With the sign cleared, bf16 bit patterns order like the values they encode.
__global__ void absmax_bf16_kernel(const uint4* __restrict__ in, int64_t nvec, unsigned* amax) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  unsigned m = 0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec; i += stride) {
    const uint4 x = __ldg(in + i);
    const unsigned w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) m = max(m, max(w[u] & 0x7FFFu, (w[u] >> 16) & 0x7FFFu));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax, m << 16);
}

// out = fp16(in * 2^-e), e = v16_shift(*amax): the largest value lands in
// [2^14, 2^15).
__global__ void bf16_to_f16_scaled_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int64_t nvec,
                                          const unsigned* __restrict__ amax) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float f = __int_as_float((127 - v16_shift(*amax)) << 23);  // 2^-e, -100 <= e <= 114
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec; i += stride) {
    const uint4 x = __ldg(in + i);
    const unsigned w[4] = {x.x, x.y, x.z, x.w};
    unsigned y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      y[u] = pack_f16(__uint_as_float(w[u] << 16) * f, __uint_as_float(w[u] & 0xFFFF0000u) * f);
    out[i] = make_uint4(y[0], y[1], y[2], y[3]);
  }
}

// Unsigned division by a divisor fixed for the launch, n < 2^31: the
// multiply-and-shift method of Granlund and Montgomery ("Division by Invariant
// Integers using Multiplication", 1994), with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, so that n / d = (umulhi(m, n) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};

FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.l = 0;
  while ((1ull << f.l) < d) ++f.l;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
  return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(f.m, n) + n) >> f.l;
}

// One lane segment per row: L = min(32, 2^ceil(log2 vpr)) lanes, 32 / L rows
// per warp, each lane covering vectors lane, lane + L, ... of the row's
// vpr = d / 4.  NP > 0 fixes the number of parts at compile time: the n LSE
// values and the n 16-byte partial vectors are all loaded before any is used,
// so a lane has 2n loads in flight.  NP = 0 is the general loop.  An empty
// part (LSE = -inf) gets weight 0 and its partial is never combined.
template <bool OUT_BF16, int NP>
__global__ void lse_merge_kernel(int64_t rows, int d, int n_parts, int seg_log2, const float* __restrict__ o_parts,
                                 const float* __restrict__ lse_parts, void* __restrict__ o_out,
                                 float* __restrict__ lse_out) {
  const int vpr = d / 4;
  const int L = 1 << seg_log2;
  const int sub = (threadIdx.x & 31) >> seg_log2;  // row within the warp
  const int li = threadIdx.x & (L - 1);            // lane within the row
  const int rows_per_warp = 32 >> seg_log2;
  const int64_t warp_id = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int n = NP > 0 ? NP : n_parts;
  for (int64_t row = warp_id * rows_per_warp + sub; row < rows; row += nwarps * rows_per_warp) {
    float out_lse = -INFINITY;
    if constexpr (NP > 0) {
      // rows `row` and `row + step` together when a lane owns one vector per row
      // and the parts are few (more loads in flight would cost occupancy)
      const int64_t step = nwarps * rows_per_warp;
      const bool pair = NP <= 2 && vpr <= L;
      const int nr = pair && row + step < rows ? 2 : 1;
      float l[2][NP];
      float4 x[2][NP];
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < nr) {
          const int64_t rk = row + k * step;
#pragma unroll
          for (int p = 0; p < NP; ++p) l[k][p] = __ldg(lse_parts + p * rows + rk);
        }
      for (int v = li; v < vpr; v += L) {
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (k < nr) {
            const int64_t rk = row + k * step;
#pragma unroll
            for (int p = 0; p < NP; ++p)
              x[k][p] = __ldg(reinterpret_cast<const float4*>(o_parts + (p * rows + rk) * d) + v);
          }
        // weights formed after the loads are issued (lane 0 always has v = 0 and sets the LSE)
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (k < nr) {
            const int64_t rk = row + k * step;
            float mx = l[k][0];
#pragma unroll
            for (int p = 1; p < NP; ++p) mx = fmaxf(mx, l[k][p]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float lse_k = -INFINITY;
            if (mx != -INFINITY) {
              float w[NP], tot = 0.f;
#pragma unroll
              for (int p = 0; p < NP; ++p) {
                w[p] = l[k][p] == -INFINITY ? 0.f : exp2f((l[k][p] - mx) * kLog2e);
                tot += w[p];
              }
              const float inv = 1.f / tot;
#pragma unroll
              for (int p = 0; p < NP; ++p) {
                if (w[p] != 0.f) {
                  const float wp = w[p] * inv;
                  acc.x = fmaf(wp, x[k][p].x, acc.x);
                  acc.y = fmaf(wp, x[k][p].y, acc.y);
                  acc.z = fmaf(wp, x[k][p].z, acc.z);
                  acc.w = fmaf(wp, x[k][p].w, acc.w);
                }
              }
              lse_k = mx + log2f(tot) * kLn2;
            }
            if (OUT_BF16) {
              uint2 o2;
              o2.x = pack_bf16(acc.x, acc.y);
              o2.y = pack_bf16(acc.z, acc.w);
              reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + rk * d)[v] = o2;
            } else {
              reinterpret_cast<float4*>(static_cast<float*>(o_out) + rk * d)[v] = acc;
            }
            if (v == 0) lse_out[rk] = lse_k;
          }
      }
      if (nr == 2) row += step;  // the loop's own increment moves past the second row
      continue;
    } else {
      float mx = -INFINITY;
      for (int p = 0; p < n; ++p) mx = fmaxf(mx, __ldg(lse_parts + p * rows + row));
      float tot = 0.f;
      if (mx != -INFINITY)
        for (int p = 0; p < n; ++p) {
          const float l = __ldg(lse_parts + p * rows + row);
          tot += l == -INFINITY ? 0.f : exp2f((l - mx) * kLog2e);
        }
      const float inv = mx != -INFINITY ? 1.f / tot : 0.f;
      for (int v = li; v < vpr; v += L) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mx != -INFINITY) {
          for (int p = 0; p < n; ++p) {
            const float l = __ldg(lse_parts + p * rows + row);
            const float w = l == -INFINITY ? 0.f : exp2f((l - mx) * kLog2e) * inv;
            if (w != 0.f) {
              const float4 x = __ldg(reinterpret_cast<const float4*>(o_parts + (p * rows + row) * d) + v);
              acc.x = fmaf(w, x.x, acc.x);
              acc.y = fmaf(w, x.y, acc.y);
              acc.z = fmaf(w, x.z, acc.z);
              acc.w = fmaf(w, x.w, acc.w);
            }
          }
        }
        if (OUT_BF16) {
          uint2 o2;
          o2.x = pack_bf16(acc.x, acc.y);
          o2.y = pack_bf16(acc.z, acc.w);
          reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + row * d)[v] = o2;
        } else {
          reinterpret_cast<float4*>(static_cast<float*>(o_out) + row * d)[v] = acc;
        }
      }
      if (mx != -INFINITY) out_lse = mx + log2f(tot) * kLn2;
    }
    if (li == 0) lse_out[row] = out_lse;
  }
}

struct PackGeom {
  int64_t batch, s_local, seqlen, blk, s_grp;  // s_grp = P * s_local, tokens per ring rank
  int cp, P, H, Hp, vpr;  // vpr: 16-byte vectors per (token, head) row
  int gather;             // 0 rank-major, 1 paired blocks, 2 contiguous blocks
  int W;                  // 16-byte vectors per output row
  int tile_rows;          // output rows per tile
  FastDiv fW, fRv;        // division by W and by Hp * vpr
  int64_t in_vecs, out_vecs;  // sizes of the two tensors in 16-byte vectors (checked build)
  unsigned* err;
};

// Natural token of rank-local position u of ring rank c.
__device__ __forceinline__ int64_t natural_token(const PackGeom& g, int c, int64_t u) {
  if (g.gather == 1) return u < g.blk ? c * g.blk + u : (2 * g.cp - 1 - c) * g.blk + (u - g.blk);
  return c * g.s_grp + u;
}

// Rank-local (c, u) of natural token `tok`.
__device__ __forceinline__ void rank_local(const PackGeom& g, int64_t tok, int& c, int64_t& u) {
  if (g.gather == 1) {
    const int64_t blk_i = tok / g.blk;
    const int64_t off = tok - blk_i * g.blk;
    if (blk_i < g.cp) {
      c = static_cast<int>(blk_i);
      u = off;
    } else {
      c = static_cast<int>(2 * g.cp - 1 - blk_i);
      u = g.blk + off;
    }
  } else {
    c = static_cast<int>(tok / g.s_grp);
    u = tok - c * g.s_grp;
  }
}

// Both directions copy whole output rows, tile_rows at a time.  Direction 0:
// output row (n, p, u) of [N][P][S_grp][Hp] is the contiguous head range
// [p Hp, (p+1) Hp) of one input token row.  Direction 1: output token row
// (all H heads) gathers P contiguous Hp-head runs, one per head rank p.  Each
// row's source offset is formed once per tile in shared memory; the copy is
// then 16-byte vectors with U loads in flight per thread and coalesced stores
// (output rows of a tile are contiguous).
template <int DIR>
__device__ __forceinline__ int64_t pack_row_source(const PackGeom& g, int64_t row) {
  if (DIR == 0) {
    const int64_t u = row % g.s_grp;
    const int64_t np = row / g.s_grp;
    const int p = static_cast<int>(np % g.P);
    const int64_t n = np / g.P;
    int64_t tok_row;
    if (g.gather == 0) {
      tok_row = n * g.s_grp + u;  // [n][q][t] with u = q s_local + t
    } else {
      const int64_t b = n / g.cp;
      tok_row = b * g.seqlen + natural_token(g, static_cast<int>(n - b * g.cp), u);
    }
    return (tok_row * g.H + static_cast<int64_t>(p) * g.Hp) * g.vpr;
  }
  int64_t n, u;
  if (g.gather == 0) {
    n = row / g.s_grp;
    u = row - n * g.s_grp;
  } else {
    const int64_t b = row / g.seqlen;
    int c;
    rank_local(g, row - b * g.seqlen, c, u);
    n = b * g.cp + c;
  }
  return (n * g.P * g.s_grp + u) * static_cast<int64_t>(g.Hp) * g.vpr;
}

constexpr int kPackThreads = 256;
constexpr int kPackMaxRows = 256;

// Up to four tensors repacked by one launch: the same mesh and direction,
// their own head counts.  Their tiles are numbered one after the other
// (tile_begin) and the grid strides over all of them.
constexpr int kPackMaxTensors = 4;
struct PackSet {
  PackGeom g[kPackMaxTensors];
  const uint4* in[kPackMaxTensors];
  uint4* out[kPackMaxTensors];
  int64_t total_rows[kPackMaxTensors];
  int64_t tile_begin[kPackMaxTensors + 1];
  int n;
};

template <int DIR>
__global__ void __launch_bounds__(kPackThreads) pack_kernel(const __grid_constant__ PackSet set) {
  __shared__ int64_t src_row[kPackMaxRows];
  constexpr int U = 8;
  for (int64_t tile = blockIdx.x; tile < set.tile_begin[set.n]; tile += gridDim.x) {
    int t = 0;
#pragma unroll
    for (int i = 1; i < kPackMaxTensors; ++i) t += (i < set.n && tile >= set.tile_begin[i]) ? 1 : 0;
    const PackGeom& g = set.g[t];
    const uint4* __restrict__ in = set.in[t];
    uint4* __restrict__ out = set.out[t];
    const int64_t plane = g.s_grp * g.Hp * g.vpr;  // vectors per (n, p) plane of the packed layout
    const int64_t row0 = (tile - set.tile_begin[t]) * g.tile_rows;
    const int rows = static_cast<int>(min(static_cast<int64_t>(g.tile_rows), set.total_rows[t] - row0));
    __syncthreads();  // the previous tile's offsets are no longer read
    for (int r = threadIdx.x; r < rows; r += kPackThreads) src_row[r] = pack_row_source<DIR>(g, row0 + r);
    __syncthreads();
    const int nvec = rows * g.W;
    uint4* dst = out + row0 * g.W;
    for (int j0 = threadIdx.x; j0 < nvec; j0 += kPackThreads * U) {
      uint4 v[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int j = j0 + k * kPackThreads;
        if (j < nvec) {
          const uint32_t r = fdiv(static_cast<uint32_t>(j), g.fW);
          const uint32_t w = static_cast<uint32_t>(j) - r * g.W;
          int64_t off = w;
          if (DIR == 1) {
            const uint32_t p = fdiv(w, g.fRv);
            off = p * plane + (w - p * g.fRv.d);
          }
          const int64_t from = src_row[r] + off;
          // checked build: both ends of the copy lie inside their tensors
          if (in_bounds(from >= 0 && from < g.in_vecs && (row0 + r) * g.W + w < g.out_vecs, g.err))
            v[k] = __ldg(in + from);
          else
            v[k] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int j = j0 + k * kPackThreads;
        if (j < nvec && in_bounds(row0 * g.W + j < g.out_vecs, g.err)) dst[j] = v[k];
      }
    }
  }
}

// Backward row statistics (see stat_row_len): for row (b, s, h) of O and dO
// (read where `lay` keeps them), D = sum_d dO*O in fp32 and LSE*log2(e),
// written at the padded position of token s.  With o_res, O is taken as
// O + O_res (exact in fp32: the residual holds the next 8 bits).  16 threads
// per row of 128 bf16 (8 elements each), 8 for d = 64.  A block covers
// consecutive tokens of one head (blockIdx.y) of one sequence (blockIdx.z),
// so a thread finds its token and part by shifts; only the layout map and
// the block position divide (32-bit).
template <int D>
__global__ void __launch_bounds__(256) bwd_rowstats_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ o_res,
    const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse, float* __restrict__ lse2,
    float* __restrict__ dstat, int64_t rows, int S, int hq, int blk, int blk_pad, int64_t stat_len, Layout lay,
    unsigned* err) {
  constexpr int TPR = D / 8;         // threads per row
  constexpr int RPB = 256 / TPR;     // rows (tokens) per block and pass
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int part = threadIdx.x % TPR;
  const int lane_row = (threadIdx.x & 31) / TPR;  // this lane's row within its warp
  const int64_t bh = static_cast<int64_t>(b) * hq + h;
  // The loop runs per warp (lanes leave together) so the shuffles below see
  // every lane; TPR divides 32, so a row's lanes are all live or all idle.
  const int64_t step = static_cast<int64_t>(gridDim.x) * RPB;
  for (int64_t s = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / TPR; s - lane_row < S; s += step) {
    const bool live = s < S;
    float acc = 0.f;
    bool row_ok = true;
    if (live) {
      const int64_t off = lay.vec(b, s, h, hq) * D;
      // checked build: the row's O / dO vectors lie inside the tensors
      row_ok = in_bounds(off >= 0 && off + D <= rows * D, err);
      if (row_ok) {
        const uint4 ov = __ldg(reinterpret_cast<const uint4*>(o + off) + part);
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(dout + off) + part);
        const uint4 rv = o_res ? __ldg(reinterpret_cast<const uint4*>(o_res + off) + part) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
        const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&rv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(a2[e]);
          const float2 fr = __bfloat1622float2(r2[e]);
          const float2 fb = __bfloat1622float2(b2[e]);
          acc = fmaf(fa.x + fr.x, fb.x, acc);
          acc = fmaf(fa.y + fr.y, fb.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0 && row_ok) {
      const int si = static_cast<int>(s);  // s < S < 2^31
      const int blk_i = si / blk;
      const int64_t pos = bh * stat_len + static_cast<int64_t>(blk_i) * blk_pad + (si - blk_i * blk);
      if (in_bounds(pos >= 0 && pos < (bh + 1) * stat_len, err)) {
        dstat[pos] = acc;
        lse2[pos] = lse[bh * S + s] * kLog2e;
      }
    }
  }
}

}  // namespace

int launch_fill_f32(float* p, int64_t n, float value, cudaStream_t stream) {
  if (n <= 0) return LOONG_OK;
  fill_f32_kernel<<<grid_for(n, 256, 8), 256, 0, stream>>>(p, n, value);
  return check_launch();
}

int launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t stream, void* res) {
  if (n <= 0) return LOONG_OK;
  f32_to_bf16_kernel<<<grid_for(n / 8 + 1, 256, 8), 256, 0, stream>>>(in, static_cast<__nv_bfloat16*>(out),
                                                                      static_cast<__nv_bfloat16*>(res), n);
  return check_launch();
}

int launch_v_to_f16(const void* v, void* v16, unsigned* amax, int64_t n, cudaStream_t stream) {
  if (n <= 0 || n % 8) return LOONG_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t nvec = n / 8;
  absmax_bf16_kernel<<<grid_for(nvec, 256, 8), 256, 0, stream>>>(static_cast<const uint4*>(v), nvec, amax);
  int st = check_launch();
  if (st != LOONG_OK) return st;
  bf16_to_f16_scaled_kernel<<<grid_for(nvec, 256, 8), 256, 0, stream>>>(static_cast<const uint4*>(v),
                                                                        static_cast<uint4*>(v16), nvec, amax);
  return check_launch();
}

template <bool OUT_BF16>
void merge_dispatch(unsigned grid, cudaStream_t stream, int64_t rows, int d, int n_parts, int seg_log2,
                    const float* o_parts, const float* lse_parts, void* o_out, float* lse_out) {
  switch (n_parts) {
    case 1:
      lse_merge_kernel<OUT_BF16, 1><<<grid, 256, 0, stream>>>(rows, d, 1, seg_log2, o_parts, lse_parts, o_out, lse_out);
      break;
    case 2:
      lse_merge_kernel<OUT_BF16, 2><<<grid, 256, 0, stream>>>(rows, d, 2, seg_log2, o_parts, lse_parts, o_out, lse_out);
      break;
    case 3:
      lse_merge_kernel<OUT_BF16, 3><<<grid, 256, 0, stream>>>(rows, d, 3, seg_log2, o_parts, lse_parts, o_out, lse_out);
      break;
    case 4:
      lse_merge_kernel<OUT_BF16, 4><<<grid, 256, 0, stream>>>(rows, d, 4, seg_log2, o_parts, lse_parts, o_out, lse_out);
      break;
    default:
      lse_merge_kernel<OUT_BF16, 0><<<grid, 256, 0, stream>>>(rows, d, n_parts, seg_log2, o_parts, lse_parts, o_out,
                                                              lse_out);
  }
}

int launch_lse_merge(int64_t rows, int d, int n_parts, const float* o_parts, const float* lse_parts,
                     void* o_out, float* lse_out, int out_bf16, cudaStream_t stream) {
  if (rows == 0) return LOONG_OK;
  const int vpr = d / 4;
  int seg_log2 = 0;
  while ((1 << seg_log2) < vpr && seg_log2 < 5) ++seg_log2;
  const int64_t rows_per_warp = 32 >> seg_log2;
  const unsigned grid = grid_for((rows + rows_per_warp - 1) / rows_per_warp * 32, 256, 8);
  if (out_bf16)
    merge_dispatch<true>(grid, stream, rows, d, n_parts, seg_log2, o_parts, lse_parts, o_out, lse_out);
  else
    merge_dispatch<false>(grid, stream, rows, d, n_parts, seg_log2, o_parts, lse_parts, o_out, lse_out);
  return check_launch();
}

int launch_headctx_pack(int n, int64_t batch, int cp, int P, int64_t s_local, const int* heads, int d,
                        int direction, int gather, const void* const* in, void* const* out, cudaStream_t stream) {
  if (n < 1 || n > kPackMaxTensors) return LOONG_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return LOONG_ERR_CUDA;
  PackSet set{};
  set.n = n;
  set.tile_begin[0] = 0;
  for (int t = 0; t < n; ++t) {
    PackGeom& g = set.g[t];
    g.batch = batch;
    g.s_local = s_local;
    g.s_grp = static_cast<int64_t>(P) * s_local;
    g.seqlen = static_cast<int64_t>(cp) * g.s_grp;
    g.blk = gather == 1 ? g.seqlen / (2 * cp) : g.seqlen / cp;
    g.cp = cp;
    g.P = P;
    g.H = heads[t];
    g.Hp = heads[t] / P;
    g.vpr = d * 2 / 16;
    g.gather = gather;
    const int64_t total_rows = direction == 0 ? batch * cp * P * g.s_grp : batch * g.seqlen;
    const int64_t w = direction == 0 ? static_cast<int64_t>(g.Hp) * g.vpr : static_cast<int64_t>(g.H) * g.vpr;
    // a tile of about 2048 vectors (32 KB); the in-tile vector index stays in 32 bits
    if (w > (1 << 20)) return LOONG_ERR_UNSUPPORTED;
    g.W = static_cast<int>(w);
    g.tile_rows = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kPackMaxRows, 2048 / w)));
    g.fW = make_fastdiv(static_cast<uint32_t>(g.W));
    g.fRv = make_fastdiv(static_cast<uint32_t>(g.Hp * g.vpr));
    g.in_vecs = g.out_vecs = batch * g.seqlen * g.H * g.vpr;  // both directions move the whole tensor
    g.err = err;
    set.in[t] = static_cast<const uint4*>(in[t]);
    set.out[t] = static_cast<uint4*>(out[t]);
    set.total_rows[t] = total_rows;
    set.tile_begin[t + 1] = set.tile_begin[t] + (total_rows + g.tile_rows - 1) / g.tile_rows;
  }
  const int64_t ntiles = set.tile_begin[n];
  if (ntiles == 0) return LOONG_OK;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ntiles, static_cast<int64_t>(num_sms()) * 8));
  if (direction == 0)
    pack_kernel<0><<<grid, kPackThreads, 0, stream>>>(set);
  else
    pack_kernel<1><<<grid, kPackThreads, 0, stream>>>(set);
  return check_launch();
}

int launch_bwd_rowstats(const loong_attn_desc& d, const void* o, const void* o_res, const void* dout,
                        const float* lse, float* stats, cudaStream_t stream) {
  const RingGeom g = ring_geom(d);
  const int64_t rows = d.batch * d.seqlen * d.hq;
  const int64_t stat_len = stat_row_len(g);
  float* lse2 = stats;
  float* dstat = stats + d.batch * d.hq * stat_len;
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pr = static_cast<const __nv_bfloat16*>(o_res);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  const int bp = stat_block_pad(g.blk);
  unsigned* err = device_error_word();
  if (!err) return LOONG_ERR_CUDA;
  // grid: (passes over the tokens, heads, sequences); about 32 blocks of 256
  // threads per SM in all, each striding over its (head, sequence) slice
  if (d.hq > 65535 || d.batch > 65535) return LOONG_ERR_INVALID_ARG;
  const int rpb = 256 / (d.head_dim / 8);
  const int64_t slices = static_cast<int64_t>(d.hq) * d.batch;
  const int64_t want = std::max<int64_t>(1, static_cast<int64_t>(num_sms()) * 32 / slices);
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>((d.seqlen + rpb - 1) / rpb, want)),
                  static_cast<unsigned>(d.hq), static_cast<unsigned>(d.batch));
  if (d.head_dim == 128)
    bwd_rowstats_kernel<128><<<grid, 256, 0, stream>>>(po, pr, pd, lse, lse2, dstat, rows, d.seqlen, d.hq, g.blk,
                                                       bp, stat_len, layout_of(d), err);
  else if (d.head_dim == 64)
    bwd_rowstats_kernel<64><<<grid, 256, 0, stream>>>(po, pr, pd, lse, lse2, dstat, rows, d.seqlen, d.hq, g.blk,
                                                      bp, stat_len, layout_of(d), err);
  else
    return LOONG_ERR_UNSUPPORTED;
  return check_launch();
}

}  // namespace loong
