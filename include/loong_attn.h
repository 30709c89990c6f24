/*
 * loong_attn.h -- C ABI of the GB300 (sm_103a) LoongTrain 2D-Attention ring step.
 *
 * One process, one GPU.  Every emulated rank of the head-parallel x
 * context-parallel mesh lives on this device; a ring "exchange" is the choice
 * of which K/V chunk a rank reads at a step, so no bytes move between steps.
 *
 * Sources (page title, section):
 *   [G] "Guide to LoongTrain: 2D Head-Context Parallelism for LLMs"
 *   [A] "LoongTrain: Efficient Training of Long-Sequence LLMs with
 *       Head-Context Parallelism" (abstract page)
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, o, o_res, dout, dq, dk, dv, lse, ws, in, out,
 *     o_parts, lse_parts, o_out, lse_out are DEVICE pointers owned by the caller:
 *     memory of the current device, from cudaMalloc or managed.  A host
 *     pointer (pinned or not) or another device's memory is refused with
 *     LOONG_ERR_INVALID_ARG before any work is enqueued.  The
 *     library allocates no device memory, keeps no state between calls except a
 *     cached device query, a loaded tensor-map encoder, one device error word
 *     and (STEPWISE_COPY) one side stream with its events per device, and
 *     synchronises only in loong_get_device_status.
 *   - All work is enqueued asynchronously on `stream` (0 = legacy default).
 *   - Tensors are contiguous.  In the NATURAL layout Q, O, dO, dQ are bf16
 *     [B, S, Hq, d] and K, V, dK, dV bf16 [B, S, Hkv, d], natural token order.
 *     In the RANK_MAJOR layout (descriptor field `layout`) they are
 *     [B*cp, hp, S/cp, H/hp, d] with H = Hq or Hkv: ring rank c's S/cp tokens
 *     (its blocks in part order, as the placement assigns them) for head rank
 *     p's H/hp heads, which is what loong_headctx_pack (direction 0, gather 1
 *     for ZIGZAG, 2 for CONTIGUOUS) produces from the natural layout.  LSE is
 *     fp32 [B, Hq, S] in natural token order in both: the natural log of the
 *     softmax denominator of the scaled logits.
 *   - Base pointers must be 16-byte aligned.
 *   - Return value: LOONG_OK (0) or a negative loong_status.  No exception
 *     crosses the ABI; no call aborts the process or traps the GPU.
 */
#ifndef LOONG_ATTN_H
#define LOONG_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LOONG_API __attribute__((visibility("default")))
#else
#define LOONG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* loong_stream_t;

typedef enum {
  LOONG_OK = 0,
  LOONG_ERR_INVALID_ARG = -1,     /* null, misaligned or non-device pointer,
                                     bad size or divisibility                 */
  LOONG_ERR_WORKSPACE = -2,       /* ws_bytes smaller than the workspace size */
  LOONG_ERR_UNSUPPORTED = -3,     /* valid but not built: head_dim, a mode /
                                     layout pairing, device is not compute
                                     capability 10.3                          */
  LOONG_ERR_CUDA = -4,            /* a CUDA call failed; see loong_last_cuda_error */
  LOONG_ERR_DEVICE_TIMEOUT = -5,  /* a kernel's bounded wait expired; the
                                     kernel stopped early and its outputs are
                                     undefined                                  */
  LOONG_ERR_DEVICE_CHECK = -6     /* libloong_attn_checked.so: a device
                                     address check failed and the access was
                                     skipped (or shared memory was misaligned);
                                     outputs are undefined                      */
} loong_status;

enum { LOONG_PLACEMENT_CONTIGUOUS = 0, LOONG_PLACEMENT_ZIGZAG = 1 };
enum { LOONG_MODE_STEPWISE = 0, LOONG_MODE_FUSED = 1, LOONG_MODE_STEPWISE_COPY = 2, LOONG_MODE_STEPWISE_COPY_AB = 3 };
enum { LOONG_LAYOUT_NATURAL = 0, LOONG_LAYOUT_RANK_MAJOR = 1 };

/*
 * Problem descriptor.  Follows the problem statement of [G] "1. 2D Mesh
 * Topology" (P = P_head x P_seq), "2. Paired-Block Allocation for Causal Load
 * Balancing" and [A] (Double-Ring-Attention).
 *   batch, seqlen     B and S (tokens per sequence).
 *   hq, hkv           query and key/value heads, hq % hkv == 0 (grouped-query
 *                     attention, [G] "The Scalability Limits of DeepSpeed
 *                     Ulysses").
 *   head_dim          d, 64 or 128.
 *   hp                head-parallel degree P_head: hq % hp == 0 and
 *                     hkv % hp == 0 (each head rank keeps whole kv heads).
 *   cp                context-parallel (ring) degree P_seq.
 *   ring_inner/outer  double-ring shape, inner * outer == cp.  At step
 *                     t = o*inner + i ring rank c holds the K/V of rank
 *                     ((c/inner - o) mod outer)*inner + ((c%inner - i) mod inner).
 *   causal            1: query i sees key j only for j <= i ([G] "The
 *                     Communication Overhead and Causal Imbalance of Ring
 *                     Attention"); 0: every key ([G] "Step 3", is_causal off).
 *   placement         LOONG_PLACEMENT_ZIGZAG: ring rank r owns blocks r and
 *                     2cp-1-r of length S/(2cp); CONTIGUOUS: block r of length
 *                     S/cp.  The block length must be a multiple of hp.
 *   mode              LOONG_MODE_FUSED: one launch walks all ring steps and
 *                     keeps the running softmax on chip; STEPWISE: one launch
 *                     per ring step, each merging its partial result into an
 *                     fp32 accumulator by log-sum-exp.  STEPWISE_COPY
 *                     (RANK_MAJOR layout only): STEPWISE with the ring's K/V
 *                     exchange made real ([G] "3. Double-Ring Asynchronous
 *                     Communication Pipeline"): before step t >= 1 every ring
 *                     rank's incoming chunk is copied (cudaMemcpyAsync, device
 *                     to device) into its receive buffer on a side stream the
 *                     library owns, double-buffered so that the copies of step
 *                     t overlap the kernel of step t-1, and the kernels read
 *                     K/V from the receive buffers.  dK, dV are added at their
 *                     owner's rows (their return trip is not copied).  The
 *                     side stream and its events are one per device: calls in
 *                     this mode on one device must not overlap.
 *                     STEPWISE_COPY_AB (ZIGZAG placement): the same with the
 *                     guide's two rings ([G] section 3): the block A and block
 *                     B halves of every chunk travel on two independent side
 *                     streams.  Results equal STEPWISE's.
 *   softmax_scale     <= 0 selects 1/sqrt(head_dim) ([G] "Step 3",
 *                     forward_local_attention).
 *   layout            LOONG_LAYOUT_NATURAL or LOONG_LAYOUT_RANK_MAJOR (the
 *                     per-rank layout after the Ulysses exchange, [G] "The
 *                     Scalability Limits of DeepSpeed Ulysses"; see above).
 *                     RANK_MAJOR needs batch * seqlen * hp < 2^31.
 */
typedef struct {
  int64_t batch, seqlen;
  int32_t hq, hkv, head_dim;
  int32_t hp, cp, ring_inner, ring_outer;
  int32_t causal;
  int32_t placement;
  int32_t mode;
  float softmax_scale;
  int32_t layout;
} loong_attn_desc;

/* Library version, (major << 16) | minor. */
LOONG_API int loong_version(void);

/* Human-readable text for a loong_status value (static storage). */
LOONG_API const char* loong_status_string(int status);

/* Text of the last CUDA error seen by this library in this thread (static). */
LOONG_API const char* loong_last_cuda_error(void);

/*
 * Check a descriptor without touching the GPU.  Returns LOONG_OK,
 * LOONG_ERR_INVALID_ARG or LOONG_ERR_UNSUPPORTED (see loong_attn_desc).
 */
LOONG_API int loong_attn_check(const loong_attn_desc* desc);

/*
 * Device workspace, in bytes, that loong_attn_fwd (pass 0) or loong_attn_bwd
 * (pass 1) needs for `desc`; 0 for an invalid descriptor.  Host-only.
 *   fwd: the fp16 copy of V that the P V product reads (B*S*Hkv*d values of
 *        2 bytes) and one word for max |V|; STEPWISE adds the fp32 O
 *        accumulator, B*S*Hq*d values.
 *   STEPWISE_COPY adds, to both passes, four 2-byte receive buffers of
 *        B*S*Hkv*d values each (K and V, two of each).
 *   bwd: fp32 dQ accumulator (B*S*Hq*d) + fp32 row statistics (LSE*log2 e
 *        and D = rowsum(dO*O)), 2 x B x Hq x (nblocks*roundup(blk,4) + 128)
 *        values, with nblocks = 2cp (ZIGZAG) or cp and blk = S/nblocks,
 *        + fp32 dK, dV accumulators, B*S*Hkv*d values each.
 *   Each part starts on a 256-byte boundary.
 */
LOONG_API size_t loong_attn_workspace_size(const loong_attn_desc* desc, int pass);

/*
 * The ring schedule as a host table: src[t * cp + c] = ring rank whose K/V
 * ring rank c holds at step t (double-ring reading above).  src must hold
 * inner*outer*inner*outer int32.  Host-only.
 */
LOONG_API int loong_ring_schedule(int32_t ring_inner, int32_t ring_outer, int32_t* src);

/*
 * Forward ring attention ([G] "Step 3", forward_local_attention per block
 * pair, merged over the ring steps).  For every emulated rank (ring rank c,
 * head rank h), every ring step t and every query head of head group h,
 * computes causal softmax attention of rank c's query blocks against the K/V
 * blocks of rank src(c, t) and merges the step's result into the running
 * result by log-sum-exp.  The result equals causal attention over the whole
 * sequence up to rounding.  The probabilities enter the P V product as fp16
 * (V as a scaled fp16 copy in the workspace) and accumulation is fp32, so the
 * unrounded O is within about 2^-12 of exact attention.
 *   q, k, v   inputs (layouts above), read only.
 *   o         bf16 output, the layout of q.
 *   lse       fp32 output [B,Hq,S].
 *   o_res     NULL, or a bf16 output in the layout of q: the rounding
 *             residual of O, bf16(O32 - bf16(O32)) with O32 the fp32 result,
 *             so that O + o_res holds O32 to about 16 bits.  Pass it to
 *             loong_attn_bwd, which then forms D = rowsum(dO * O) from
 *             O + o_res.
 *   ws        device workspace of at least loong_attn_workspace_size(desc,0)
 *             bytes; every descriptor needs one.
 */
LOONG_API int loong_attn_fwd(const loong_attn_desc* desc, const void* q, const void* k, const void* v,
                   void* o, float* lse, void* o_res, void* ws, size_t ws_bytes, loong_stream_t stream);

/*
 * loong_attn_fwd restricted to the query rows of ring ranks
 * [rank_begin, rank_end) (all heads, all sequences of the batch): the work of
 * those emulated ranks alone, so that one rank's share of the ring pass can be
 * timed ([G] section 2 gives every rank the same work under paired blocks).
 * Rows of other ranks in o and lse are left untouched; the rows written equal
 * those of loong_attn_fwd bit for bit.  FUSED mode only (STEPWISE returns
 * LOONG_ERR_UNSUPPORTED); ws as for loong_attn_fwd.  0 <= rank_begin <
 * rank_end <= cp.
 */
LOONG_API int loong_attn_fwd_ranks(const loong_attn_desc* desc, int32_t rank_begin, int32_t rank_end,
                                   const void* q, const void* k, const void* v, void* o, float* lse,
                                   void* ws, size_t ws_bytes, loong_stream_t stream);

/*
 * Backward of loong_attn_fwd: the exact gradient of causal softmax attention
 * (the pages give no backward; this is the plain chain rule through softmax).
 * Over the same schedule: P = exp(s - LSE), dV += P^T dO, dP = dO V^T,
 * dS = P * (dP - D) with D = rowsum(dO * O), dQ += scale dS K,
 * dK += scale dS^T Q; dK and dV sum over the query heads of a kv group.
 *   o, lse    the outputs of loong_attn_fwd for the same inputs.
 *   o_res     the forward's o_res output, or NULL.  D is formed in fp32 from
 *             O + o_res, else from the bf16 O alone.  The D term of dQ and dK
 *             is -scale * D * (probability-weighted keys or queries), so an
 *             error in D is amplified where a few large keys take the
 *             probability mass; with o_res, D carries the forward's own
 *             accuracy instead of bf16's 2^-9.
 *   dout      bf16 dO, the layout of q.
 *   dq        bf16, the layout of q; dk, dv bf16, the layout of k; written,
 *             not added to.
 *   ws        at least loong_attn_workspace_size(desc,1) bytes.
 */
LOONG_API int loong_attn_bwd(const loong_attn_desc* desc, const void* q, const void* k, const void* v,
                   const void* o, const void* o_res, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                   loong_stream_t stream);

/*
 * Largest workspace, in bytes, that loong_attn_bwd_noalloc can serve: 32 MiB.
 * A problem fits when loong_attn_workspace_size(desc, 1) is at most this; in
 * FUSED and STEPWISE mode that size is at most 4*B*S*Hq*d + 8*B*S*Hkv*d +
 * 8*B*Hq*(S + 3*nblocks + 128) bytes plus 256 per part (four parts), with
 * nblocks = 2cp (ZIGZAG) or cp.  For example S = 4096 tokens, Hq = 8, Hkv = 1,
 * d = 128 needs about 20.3 MiB.
 */
#define LOONG_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * loong_attn_bwd without a workspace argument, for callers that cannot
 * allocate device memory: a plugin inside a framework that owns the whole
 * device pool and hands it only inputs and outputs, or a latency-critical loop
 * that cannot take cudaMalloc's implicit device synchronisation.  The paper
 * has no counterpart; this is an interface convenience.
 *   Same arguments, layouts and results as loong_attn_bwd, minus ws/ws_bytes.
 *   The descriptor is checked first, then the device (LOONG_ERR_UNSUPPORTED
 *   on one that is not compute capability 10.3); a problem whose workspace
 *   exceeds the array gives LOONG_ERR_WORKSPACE.
 *   Scratch lives in one static device array of LOONG_NOALLOC_SCRATCH_BYTES
 *   that every GPU loading the library holds until the process exits.  The
 *   call allocates nothing: no cudaMalloc, cudaFree or allocating library
 *   routine.  Returns LOONG_ERR_WORKSPACE when
 *   loong_attn_workspace_size(desc, 1) exceeds LOONG_NOALLOC_SCRATCH_BYTES.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  A failed lookup is not remembered: the next
 *   call tries again.
 *   Every call on a device shares the one array and it keeps the last call's
 *   contents (the parts that must start at zero are cleared by each call):
 *   calls whose work overlaps on the GPU (other streams, other host threads)
 *   race on it and must be serialised by the caller.
 */
LOONG_API int loong_attn_bwd_noalloc(const loong_attn_desc* desc, const void* q, const void* k,
                                     const void* v, const void* o, const void* o_res, const float* lse,
                                     const void* dout, void* dq, void* dk, void* dv, loong_stream_t stream);

/*
 * n-way log-sum-exp merge of partial attention results over disjoint key sets
 * (the pages leave the merge implicit; it is the rule under which softmax over
 * a union of key sets is recovered from the parts):
 *   L = ln sum_p exp(L_p),  O = sum_p exp(L_p - L) O_p.
 * A part with L_p = -inf is empty and has weight 0; if all parts are empty the
 * row gets L = -inf and O = 0.
 *   o_parts   fp32 [n_parts][rows][d];  lse_parts fp32 [n_parts][rows].
 *   o_out     fp32 [rows][d] (out_bf16 == 0) or bf16 [rows][d] (out_bf16 == 1).
 *   lse_out   fp32 [rows].
 * rows >= 0 (0 is a no-op), 1 <= d <= 1024 with d % 4 == 0, 1 <= n_parts <= 64.
 * Outputs must not overlap inputs.
 */
LOONG_API int loong_lse_merge(int64_t rows, int32_t d, int32_t n_parts,
                    const float* o_parts, const float* lse_parts,
                    void* o_out, float* lse_out, int out_bf16, loong_stream_t stream);

/*
 * Ulysses head-context repack ([G] "The Scalability Limits of DeepSpeed
 * Ulysses": all-to-all (S/P, H) -> (S, H/P) before attention and the inverse
 * after), for every ring rank's head-parallel group at once, as a bit copy of
 * 2-byte elements.
 *   direction 0:  out[n][p][q*s_local + t][h'][:] = in[n][q][t][p*H/P + h'][:]
 *   direction 1:  the inverse (out and in swap roles).
 * with n < batch*cp (group = ring rank of one sequence), p, q < P, t < s_local,
 * h' < H/P.  `gather` selects the layout of the (S/P, H) side:
 *   0  rank-major [batch*cp][P][s_local][H][d];
 *   1  natural token order [batch][S][H][d], S = cp*P*s_local, ring rank n
 *      owning the paired blocks n and 2cp-1-n ([G] section 2);
 *   2  natural token order with contiguous blocks.
 * The (S, H/P) side is always rank-major [batch*cp][P][P*s_local][H/P][d].
 * H % P == 0, d*2 bytes a multiple of 16, in and out must not overlap.
 */
LOONG_API int loong_headctx_pack(int64_t batch, int32_t cp, int32_t P, int64_t s_local, int32_t heads,
                       int32_t d, int direction, int gather, const void* in, void* out,
                       loong_stream_t stream);

/*
 * loong_headctx_pack over n tensors (1 <= n <= 4) in one launch: the same
 * batch, cp, P, s_local, d, direction and gather, their own head counts, as
 * the Q, K, V (and dO) of one pass, whose repacks are the one all-to-all the
 * guide describes.  Tensor t has heads[t] heads (each a multiple of P) and
 * moves from in[t] to out[t]; heads, in and out are host arrays of n entries.
 * The results equal n calls of loong_headctx_pack bit for bit.
 */
LOONG_API int loong_headctx_pack_n(int32_t n, int64_t batch, int32_t cp, int32_t P, int64_t s_local,
                                   const int32_t* heads, int32_t d, int direction, int gather,
                                   const void* const* in, void* const* out, loong_stream_t stream);

/*
 * Device workspace, in bytes, of loong_attn_2d_host for `desc`: pass 0 runs
 * the forward alone, pass 1 the forward and the backward; 0 for an invalid
 * descriptor.  Host-only.  It holds two sets of natural-layout inputs (the
 * slots), the natural-layout outputs and LSE, the forward's residual of O
 * (pass 1: the backward forms D from O and it), the rank-major tensors of the
 * pass (RANK_MAJOR) and the workspaces of loong_attn_fwd / loong_attn_bwd,
 * each part on a 256-byte boundary.
 */
LOONG_API size_t loong_attn_2d_host_workspace_size(const loong_attn_desc* desc, int pass);

/*
 * One whole 2D-attention pass from host memory to host memory: the inputs
 * travel to the device, the Ulysses repack moves them into every emulated
 * rank's layout ([G] "The Scalability Limits of DeepSpeed Ulysses"), the ring
 * forward (and backward) run on it, and the outputs are repacked and travel
 * back.  With a NATURAL descriptor the ring kernels read and write the
 * natural layout and there is no repack.
 *   q, k, v, dout   host inputs, natural layout [B,S,H,d] bf16.  dout == NULL
 *                   runs the forward alone (dq, dk, dv must then be NULL).
 *   o, lse          host outputs: bf16 [B,S,Hq,d] and fp32 [B,Hq,S].
 *   dq, dk, dv      host outputs, bf16, the layouts of q and k.
 *   slot            0 or 1: which of the workspace's two device input sets
 *                   this call fills.  Alternate it between consecutive calls
 *                   so that a call's inputs can arrive while the previous
 *                   call's kernels still read theirs.
 *   ws, ws_bytes    device workspace of loong_attn_2d_host_workspace_size
 *                   bytes (pass 1 when dout != NULL, else pass 0).
 *   done_event      a cudaEvent_t of the caller, or NULL.  Non-NULL: it is
 *                   recorded once every output has reached host memory, and
 *                   `stream` does not wait for the output copies, so the next
 *                   call's kernels overlap them.  NULL: `stream` waits for the
 *                   output copies before its later work.
 * Every copy runs on one of two library-owned copy streams (host to device,
 * device to host), ordered against the kernels on `stream` by events: a
 * call's input copies start when the call is made, once the slot's previous
 * inputs have been read; dO arrives while the forward runs, and O and LSE
 * leave while the backward runs.  Pinned host memory (cudaHostAlloc /
 * cudaHostRegister, or loong_host_alloc below, which also keeps the copies at
 * full speed when the device's translations of host pages have gone cold)
 * lets the copies overlap the kernels; pageable memory is accepted but
 * copies synchronously.  The caller must not change the inputs
 * or read the outputs before the call's work has finished (done_event, or
 * `stream` when done_event is NULL).  Calls on one device are serialised by
 * the library (one enqueue at a time).  Device pointers in the host
 * arguments, a slot other than 0 or 1 and null pointers give
 * LOONG_ERR_INVALID_ARG; a short workspace gives LOONG_ERR_WORKSPACE.
 */
LOONG_API int loong_attn_2d_host(const loong_attn_desc* desc, int32_t slot, const void* q, const void* k,
                                 const void* v, const void* dout, void* o, float* lse, void* dq, void* dk,
                                 void* dv, void* ws, size_t ws_bytes, loong_stream_t stream,
                                 void* done_event);

/*
 * Pinned host memory for the host arguments of loong_attn_2d_host (or any
 * host <-> device copy): `bytes` bytes at *ptr, registered with CUDA, in an
 * anonymous mapping aligned to the kernel's transparent huge page size and
 * advised to use huge pages (where the kernel offers none the buffer is
 * still pinned).  Why: the device translates every host page a copy touches,
 * and when those translations have gone cold (a few seconds without copies,
 * or after kernels that sweep much device memory) each page costs a miss.
 * Measured with 64 KB base pages, a 2.7 GB host-to-device copy then took
 * 360-380 ms from cudaHostAlloc memory and 12.7 ms from huge pages.  The
 * range is also asked to collapse into huge pages (MADV_COLLAPSE, where the
 * kernel has it).  On some hosts device writes into the buffer split part of
 * it back into base pages, and copies into it slow down again.
 *   bytes == 0 sets *ptr = NULL.  The caller owns the buffer and releases it
 *   with loong_host_free.  Returns LOONG_OK, LOONG_ERR_INVALID_ARG (null
 *   ptr), or LOONG_ERR_CUDA (mapping or registration failed; *ptr = NULL).
 */
LOONG_API int loong_host_alloc(size_t bytes, void** ptr);

/*
 * Unregister and unmap a buffer from loong_host_alloc.  NULL is a no-op; a
 * pointer that loong_host_alloc did not return gives LOONG_ERR_INVALID_ARG.
 * No copy may still use the buffer.
 */
LOONG_API int loong_host_free(void* ptr);

/*
 * Measurement aid.  When both are non-NULL, the calling thread's next
 * loong_attn_fwd / loong_attn_bwd calls record `start_event` on their stream
 * just before launching the main ring-attention kernel(s) and `stop_event`
 * just after the last of them, so the kernels' device time can be read with
 * cudaEventElapsedTime without counting the call's helper kernels.  The events
 * are cudaEvent_t handles owned by the caller; pass NULL, NULL to stop.
 */
LOONG_API int loong_set_timing_events(void* start_event, void* stop_event);

/*
 * Synchronise `stream` and report device-side failures of earlier calls:
 * LOONG_ERR_DEVICE_CHECK if an address check of the checked build failed or a
 * kernel found its shared memory misaligned, else LOONG_ERR_DEVICE_TIMEOUT if
 * a kernel's bounded wait expired (the error word is then cleared),
 * LOONG_ERR_CUDA if the stream reports a CUDA error, LOONG_OK otherwise.
 */
LOONG_API int loong_get_device_status(loong_stream_t stream);

/*
 * Self-test of the bounded-wait path (no counterpart on the pages): launches
 * one CTA on `stream` whose mbarrier wait, the same code every kernel's waits
 * use, has nothing to wait for.  It gives up after limit_us microseconds
 * (1 .. 1000000), raises the CTA's abort flag, sets the device error word and
 * returns, so the next loong_get_device_status reports
 * LOONG_ERR_DEVICE_TIMEOUT and clears the word; the context stays usable.
 * Returns LOONG_ERR_INVALID_ARG for a limit out of range (before any CUDA
 * call), else the launch status.
 */
LOONG_API int loong_selftest_wait_timeout(uint32_t limit_us, loong_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOONG_ATTN_H */
