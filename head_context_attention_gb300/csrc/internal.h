// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdio>

#include "../../include/loong_attn.h"
#include "ring.cuh"

namespace loong {

// Records the CUDA error text for loong_last_cuda_error and maps to a status.
int cuda_fail(cudaError_t e);
// cudaGetLastError after a launch: LOONG_OK or LOONG_ERR_CUDA.
int check_launch();

// Optional events recorded around the main attention launches (this thread).
void record_start(cudaStream_t s);
void record_stop(cudaStream_t s);

// LOONG_OK when the current device is usable (compute capability 10.3), else
// LOONG_ERR_UNSUPPORTED or LOONG_ERR_CUDA; every CUDA-touching entry point
// checks it first.
int device_ready();
// Memory of the current device (cudaMalloc'd or managed).
bool on_device(const void* p);
// Host memory, pinned or pageable.
bool in_host_memory(const void* p);

// Device address of the library's error word on the current device.
unsigned* device_error_word();

// Lazily loaded cuTensorMapEncodeTiled; nullptr if the driver lacks it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// bf16 tensor [rows][heads][d] viewed as the 3-D tensor (d, heads, rows),
// box (64, 1, 128), 128-byte swizzle.  Returns LOONG_OK or an error status.
int make_head_tile_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int d);

// fp32 tensor [rows][heads][d] viewed as (d, heads, rows), box (32, 1, 128),
// 128-byte swizzle (one box row is 128 bytes).
int make_f32_tile_map(CUtensorMap* map, const void* base, int64_t rows, int heads, int d);

// An NVTX range (profiler timelines: one per entry point and per ring step)
// for the lifetime of the object; no cost unless a tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  NvtxRange(const char* fmt, int v) {
    char buf[48];
    std::snprintf(buf, sizeof(buf), fmt, v);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

RingGeom ring_geom(const loong_attn_desc& d);
// STEPWISE_COPY or STEPWISE_COPY_AB: the K/V exchange goes through receive buffers.
inline bool is_copy_mode(const loong_attn_desc& d) {
  return d.mode == LOONG_MODE_STEPWISE_COPY || d.mode == LOONG_MODE_STEPWISE_COPY_AB;
}
// Token/head placement of the descriptor's tensors (natural or rank-major).
Layout layout_of(const loong_attn_desc& d);

// The forward's workspace and optional outputs.
struct FwdScratch {
  void* v16 = nullptr;          // fp16 V * 2^-e, the layout of V
  unsigned* v_amax = nullptr;   // bit pattern of max |V| (v16_shift gives e)
  float* o_acc = nullptr;       // STEPWISE: fp32 O accumulator
  void* kv_recv = nullptr;      // STEPWISE_COPY: K0, K1, V0, V1 receive buffers (exchange.h)
  void* o_res = nullptr;        // bf16 rounding residual of O, or null
};
// Byte offsets of the forward workspace's parts (each on a 256-byte boundary)
// and its total size.
struct FwdWsLayout {
  size_t v16, amax, o_acc, recv, total;
};
FwdWsLayout fwd_ws_layout(const loong_attn_desc& d);

// Kernel launchers (asynchronous on `stream`).
// Query rows of ring ranks [rank_begin, rank_end) only (all of them: 0, cp).
// The forward first writes V's fp16 copy into sc.v16.
int launch_fwd(const loong_attn_desc& d, const void* q, const void* k, const void* v, void* o,
               float* lse, const FwdScratch& sc, cudaStream_t stream, int rank_begin = 0, int rank_end = -1);
// o_res: the forward's residual of O, or null (D from O alone).
int launch_bwd(const loong_attn_desc& d, const void* q, const void* k, const void* v,
               const void* o, const void* o_res, const float* lse, const void* dout, void* dq, void* dk, void* dv,
               float* dq_acc, float* dvec, float* dk_acc, float* dv_acc, cudaStream_t stream,
               void* kv_recv = nullptr);
// max |V| into *amax (two launches: the maximum, then V * 2^-e as fp16 into v16).
int launch_v_to_f16(const void* v, void* v16, unsigned* amax, int64_t n, cudaStream_t stream);

int launch_fill_f32(float* p, int64_t n, float value, cudaStream_t stream);
// One CTA whose bounded mbarrier wait has nothing to wait for (selftest.cu).
int launch_wait_probe(uint32_t limit_us, cudaStream_t stream);
// out = bf16(in); with res, also res = bf16(in - out) (the rounding residual).
int launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t stream, void* res = nullptr);
int launch_lse_merge(int64_t rows, int d, int n_parts, const float* o_parts,
                     const float* lse_parts, void* o_out, float* lse_out, int out_bf16,
                     cudaStream_t stream);
// n (1..4) tensors of the same mesh and direction, heads[t] heads each, one launch.
int launch_headctx_pack(int n, int64_t batch, int cp, int P, int64_t s_local, const int* heads, int d,
                        int direction, int gather, const void* const* in, void* const* out, cudaStream_t stream);
// Backward row statistics: for every (batch, query head, token) the values
// LSE*log2(e) and D = rowsum(dO*O), in [B*Hq][stat_row_len] arrays (LSE part
// first, then D) where block b's tokens start at b*stat_block_pad(blk), so a
// 128-row tile's statistics are 16-byte aligned and reads past a tile stay in
// bounds.
inline int stat_block_pad(int blk) { return (blk + 3) & ~3; }
inline int64_t stat_row_len(const RingGeom& g) {
  return static_cast<int64_t>(g.nblocks) * stat_block_pad(g.blk) + kTile;
}
// With o_res, D = rowsum(dO * (O + O_res)).
int launch_bwd_rowstats(const loong_attn_desc& d, const void* o, const void* o_res, const void* dout,
                        const float* lse, float* stats, cudaStream_t stream);

}  // namespace loong
