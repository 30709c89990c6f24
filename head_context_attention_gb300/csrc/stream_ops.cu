// stream_ops.cu -- bandwidth-bound kernels: the n-way log-sum-exp merge, the
// Ulysses head-context repack, the backward's D = rowsum(dO * O), fills and
// the fp32 -> bf16 conversion of accumulators.  Each thread moves 16-byte
// vectors; grids are sized in multiples of the SM count and stride over the
// work.
#include <cuda_bf16.h>

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

// n % 8 == 0 handled by the vector path; the tail element by element.
__global__ void f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                   int64_t n) {
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
  }
  for (int64_t i = nv * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += stride)
    out[i] = __float2bfloat16_rn(in[i]);
}

// One thread per (row, 4-float vector).  Every thread of a row recomputes the
// row's weights from the n LSE values (served from L1).
template <bool OUT_BF16>
__global__ void lse_merge_kernel(int64_t rows, int d, int n_parts, const float* __restrict__ o_parts,
                                 const float* __restrict__ lse_parts, void* __restrict__ o_out,
                                 float* __restrict__ lse_out) {
  const int vpr = d / 4;
  const int64_t total = rows * vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / vpr;
    const int vec = static_cast<int>(i - row * vpr);
    float mx = -INFINITY;
    for (int p = 0; p < n_parts; ++p) mx = fmaxf(mx, __ldg(lse_parts + p * rows + row));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (mx != -INFINITY) {
      float tot = 0.f;
      for (int p = 0; p < n_parts; ++p) {
        const float l = __ldg(lse_parts + p * rows + row);
        const float w = l == -INFINITY ? 0.f : exp2f((l - mx) * kLog2e);
        tot += w;
        if (w != 0.f) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(o_parts + (p * rows + row) * d) + vec);
          acc.x = fmaf(w, x.x, acc.x);
          acc.y = fmaf(w, x.y, acc.y);
          acc.z = fmaf(w, x.z, acc.z);
          acc.w = fmaf(w, x.w, acc.w);
        }
      }
      const float inv = 1.f / tot;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      lse = mx + log2f(tot) * kLn2;
    }
    if (OUT_BF16) {
      uint2 w;
      w.x = pack_bf16(acc.x, acc.y);
      w.y = pack_bf16(acc.z, acc.w);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + row * d)[vec] = w;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(o_out) + row * d)[vec] = acc;
    }
    if (vec == 0) lse_out[row] = lse;
  }
}

struct PackGeom {
  int64_t batch, s_local, seqlen, blk;
  int cp, P, H, Hp, vpr;  // vpr: 16-byte vectors per (token, head) row
  int gather;             // 0 rank-major, 1 paired blocks, 2 contiguous blocks
};

// Natural token of rank-local position u of ring rank c.
__device__ __forceinline__ int64_t natural_token(const PackGeom& g, int c, int64_t u) {
  if (g.gather == 1) return u < g.blk ? c * g.blk + u : (2 * g.cp - 1 - c) * g.blk + (u - g.blk);
  return c * (g.P * g.s_local) + u;
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
    const int64_t sl = g.P * g.s_local;
    c = static_cast<int>(tok / sl);
    u = tok - c * sl;
  }
}

// Direction 0, enumerated over output vectors (coalesced writes).
__global__ void pack_fwd_kernel(PackGeom g, const uint4* __restrict__ in, uint4* __restrict__ out) {
  const int64_t S_grp = static_cast<int64_t>(g.P) * g.s_local;  // tokens per ring rank
  const int64_t total = g.batch * g.cp * g.P * S_grp * g.Hp * g.vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
    int64_t x = i;
    const int v = static_cast<int>(x % g.vpr);
    x /= g.vpr;
    const int hh = static_cast<int>(x % g.Hp);
    x /= g.Hp;
    const int64_t u = x % S_grp;
    x /= S_grp;
    const int p = static_cast<int>(x % g.P);
    const int64_t n = x / g.P;
    const int q = static_cast<int>(u / g.s_local);
    const int64_t t = u - q * g.s_local;
    const int head = p * g.Hp + hh;
    int64_t src;
    if (g.gather == 0) {
      src = ((n * g.P + q) * g.s_local + t) * g.H + head;
    } else {
      const int64_t b = n / g.cp;
      const int c = static_cast<int>(n - b * g.cp);
      src = (b * g.seqlen + natural_token(g, c, u)) * g.H + head;
    }
    out[i] = __ldg(in + src * g.vpr + v);
  }
}

// Direction 1, enumerated over output vectors.
__global__ void pack_inv_kernel(PackGeom g, const uint4* __restrict__ in, uint4* __restrict__ out) {
  const int64_t S_grp = static_cast<int64_t>(g.P) * g.s_local;
  const int64_t total = g.batch * g.cp * S_grp * g.H * g.vpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
    int64_t x = i;
    const int v = static_cast<int>(x % g.vpr);
    x /= g.vpr;
    const int head = static_cast<int>(x % g.H);
    x /= g.H;
    int64_t n, u;
    if (g.gather == 0) {
      // out rank-major [n][q][t][H]: x = (n*P + q)*s_local + t
      const int64_t t = x % g.s_local;
      x /= g.s_local;
      const int q = static_cast<int>(x % g.P);
      n = x / g.P;
      u = q * g.s_local + t;
    } else {
      const int64_t tok = x % g.seqlen;
      const int64_t b = x / g.seqlen;
      int c;
      rank_local(g, tok, c, u);
      n = b * g.cp + c;
    }
    const int p = head / g.Hp;
    const int hh = head - p * g.Hp;
    const int64_t src = ((n * g.P + p) * S_grp + u) * g.Hp + hh;
    out[i] = __ldg(in + src * g.vpr + v);
  }
}

// Backward row statistics (see stat_row_len): for row (b, s, h) of O and dO,
// D = sum_d dO*O in fp32 and LSE*log2(e), written at the padded position of
// token s.  16 threads per row of 128 bf16 (8 elements each), 8 for d = 64.
template <int D>
__global__ void bwd_rowstats_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                    const float* __restrict__ lse, float* __restrict__ lse2,
                                    float* __restrict__ dstat, int64_t rows, int64_t S, int hq, int blk,
                                    int blk_pad, int64_t stat_len) {
  constexpr int TPR = D / 8;
  const int64_t total = rows * TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // The loop runs per warp (lanes leave together) so the shuffles below see
  // every lane; TPR divides 32, so a row's lanes are all live or all idle.
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i - static_cast<int64_t>(threadIdx.x & 31) < total; i += stride) {
    const bool live = i < total;
    const int64_t row = live ? i / TPR : 0;
    const int part = static_cast<int>(i % TPR);
    float acc = 0.f;
    if (live) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + part);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]);
        const float2 fb = __bfloat1622float2(b2[e]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0) {
      // row = (b*S + s)*hq + h
      const int64_t h = row % hq;
      const int64_t bs = row / hq;
      const int64_t b = bs / S;
      const int64_t s = bs - b * S;
      const int64_t blk_i = s / blk;
      const int64_t pos = (b * hq + h) * stat_len + blk_i * blk_pad + (s - blk_i * blk);
      dstat[pos] = acc;
      lse2[pos] = lse[(b * hq + h) * S + s] * kLog2e;
    }
  }
}

}  // namespace

int launch_fill_f32(float* p, int64_t n, float value, cudaStream_t stream) {
  if (n <= 0) return LOONG_OK;
  fill_f32_kernel<<<grid_for(n, 256, 8), 256, 0, stream>>>(p, n, value);
  return check_launch();
}

int launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t stream) {
  if (n <= 0) return LOONG_OK;
  f32_to_bf16_kernel<<<grid_for(n / 8 + 1, 256, 8), 256, 0, stream>>>(in, static_cast<__nv_bfloat16*>(out), n);
  return check_launch();
}

int launch_lse_merge(int64_t rows, int d, int n_parts, const float* o_parts, const float* lse_parts,
                     void* o_out, float* lse_out, int out_bf16, cudaStream_t stream) {
  if (rows == 0) return LOONG_OK;
  const unsigned grid = grid_for(rows * (d / 4), 256, 8);
  if (out_bf16)
    lse_merge_kernel<true><<<grid, 256, 0, stream>>>(rows, d, n_parts, o_parts, lse_parts, o_out, lse_out);
  else
    lse_merge_kernel<false><<<grid, 256, 0, stream>>>(rows, d, n_parts, o_parts, lse_parts, o_out, lse_out);
  return check_launch();
}

int launch_headctx_pack(int64_t batch, int cp, int P, int64_t s_local, int heads, int d, int direction,
                        int gather, const void* in, void* out, cudaStream_t stream) {
  PackGeom g;
  g.batch = batch;
  g.s_local = s_local;
  g.seqlen = static_cast<int64_t>(cp) * P * s_local;
  g.blk = gather == 1 ? g.seqlen / (2 * cp) : g.seqlen / cp;
  g.cp = cp;
  g.P = P;
  g.H = heads;
  g.Hp = heads / P;
  g.vpr = d * 2 / 16;
  g.gather = gather;
  const int64_t total = batch * g.seqlen * heads * g.vpr;
  if (total == 0) return LOONG_OK;
  const unsigned grid = grid_for(total, 256, 8);
  if (direction == 0)
    pack_fwd_kernel<<<grid, 256, 0, stream>>>(g, static_cast<const uint4*>(in), static_cast<uint4*>(out));
  else
    pack_inv_kernel<<<grid, 256, 0, stream>>>(g, static_cast<const uint4*>(in), static_cast<uint4*>(out));
  return check_launch();
}

int launch_bwd_rowstats(const loong_attn_desc& d, const void* o, const void* dout, const float* lse,
                        float* stats, cudaStream_t stream) {
  const RingGeom g = ring_geom(d);
  const int64_t rows = d.batch * d.seqlen * d.hq;
  const int64_t stat_len = stat_row_len(g);
  float* lse2 = stats;
  float* dstat = stats + d.batch * d.hq * stat_len;
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  const int bp = stat_block_pad(g.blk);
  if (d.head_dim == 128)
    bwd_rowstats_kernel<128><<<grid_for(rows * 16, 256, 8), 256, 0, stream>>>(po, pd, lse, lse2, dstat, rows,
                                                                               d.seqlen, d.hq, g.blk, bp, stat_len);
  else if (d.head_dim == 64)
    bwd_rowstats_kernel<64><<<grid_for(rows * 8, 256, 8), 256, 0, stream>>>(po, pd, lse, lse2, dstat, rows,
                                                                             d.seqlen, d.hq, g.blk, bp, stat_len);
  else
    return LOONG_ERR_UNSUPPORTED;
  return check_launch();
}

}  // namespace loong
