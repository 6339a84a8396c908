/*
 * extkv.h -- C ABI of libextkv: biased grouped-query attention over an
 * external static KV cache, native to GB300 (sm_103a).
 *
 * The three operations are the three nodes of the static-cache graph the
 * pages describe ("Skill: Attention Optimization", section "In-place KV for
 * ONNX Attention via TensorScatter (static cache)"; mobius issue #366,
 * "Emit bias-aware external-KV (TensorScatter + nonpad_kv_seqlen) attention for
 * float-bias decoders"):
 *     cache' = TensorScatter(cache, new_rows, write_indices)      -> ext_kv_scatter
 *     bias   = create_static_cache_attention_bias(...)            -> build_static_cache_bias
 *     Y      = Attention(Q, K cache', V cache', bias, nonpad_kv_seqlen,
 *                        q_num_heads, kv_num_heads, is_causal=0)  -> attention_ext_kv
 *
 * Conventions shared by every entry point
 *   - Pointers named *_cache, q, y, bias, extra, status, workspace, nonpad,
 *     write_idx, q_start, spans, span_offsets are DEVICE pointers, owned by
 *     the caller.  A call allocates no device memory (the workspace is the
 *     caller's; attention_ext_kv_noalloc uses a static array of the library)
 *     and no pointer is used after the call's kernels finish, except by a
 *     recorded step (extkv_step_*), which replays its calls on the buffers it
 *     was recorded with until it is freed.  Host-side caches of encoded
 *     tensor maps are keyed by pointer values and never dereferenced.
 *     Structs passed by pointer (extkv_bias_spec) are HOST memory, read
 *     during the call only.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) and never synchronises, except
 *     extkv_read_status.
 *   - All tensors are dense, row-major, in BNSH order:
 *       q, y           (B, Hq,  S_q,     D)
 *       k/v cache      (B, Hkv, max_seq, D)
 *       k/v new rows   (B, Hkv, S_new,   D)
 *       bias, extra    (B, 1,   S_q,     max_seq)   broadcast over heads
 *       nonpad, write_idx, q_start   (B,) int64
 *     Element type of q, y, caches, new rows, bias and extra: extkv_dtype.
 *   - Return value: EXTKV_OK, or a negative extkv_status with a stable
 *     message available from extkv_last_error() (thread-local).  Argument
 *     errors are detected on the host before anything is launched.
 *   - Data-dependent errors (an out-of-range write index or nonpad value)
 *     cannot be seen on the host without a sync: the kernels skip the
 *     offending batch and OR a flag into status[0] (EXTKV_DEV_*) and add one
 *     to status[1].  `status` is NULL (no report) or 16 bytes of device
 *     memory, 4-byte aligned, zeroed by extkv_clear_status or by the caller.
 *   - Integer arithmetic on positions and lengths is signed 64-bit, so
 *     differences such as nonpad - S_q may go negative without wrapping
 *     ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 12).
 */
#ifndef EXTKV_H_
#define EXTKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { EXTKV_F32 = 0, EXTKV_BF16 = 1 } extkv_dtype;

typedef enum {
  EXTKV_OK = 0,
  EXTKV_ERR_INVALID_ARG = -1, /* a null pointer, a bad size or a misaligned pointer */
  EXTKV_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. a forced kernel that cannot run) */
  EXTKV_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  EXTKV_ERR_DEVICE = -4       /* extkv_read_status found a device-side flag */
} extkv_status;

/* Flags OR-ed into status[0] by the kernels. */
#define EXTKV_DEV_BAD_WRITE_IDX 0x1 /* write_idx[b] < 0 or write_idx[b] + S_new > max_seq */
#define EXTKV_DEV_BAD_NONPAD 0x2    /* nonpad[b] < 0 or nonpad[b] > max_seq */
#define EXTKV_DEV_TIMEOUT 0x4       /* a bounded pipeline wait gave up; the tile was abandoned */
#define EXTKV_DEV_BOUNDS 0x8        /* a library built with EXTKV_CHECKED skipped a global access whose
                                       index fell outside its buffer (device bounds checks in place
                                       of a sanitizer: no trap, no fault) */

/*
 * The bias specification of mobius issue #366 (deliverable: causal + sliding
 * window + bidirectional block overlay + padding, keyed on absolute query
 * positions, valid only where slot < nonpad_kv_seqlen[b]).
 *
 * Query position of row i of batch b: p = q_start[b] + i, or, with q_start
 * NULL, the bottom-right alignment of an external cache,
 * p = max(nonpad[b] - S_q, 0) + i ("ONNX Domain Attention (Opset 23/24) CUDA
 * Patterns", section 11).  Key slot j is allowed iff
 *     j < nonpad[b]  and  ( (causal_ok and window_ok) or same_span )
 *     causal_ok = !causal || j <= p
 *     window_ok = window <= 0 || p - j < window   (keys p-W+1 .. p; "Skill:
 *                 Attention Optimization", "GQA sliding window")
 *     same_span = some span (start, len) of batch b holds both p and j
 * An allowed slot carries extra[b,0,i,j] (or 0 when extra is NULL); any other
 * slot carries the element type's lowest finite value (the CPU reference's
 * sentinel, "ONNX Domain Attention ...", section 8).
 *
 * Spans: span_offsets (B+1,) int64 indexes rows of spans (n,2) int64 holding
 * (start, len) in absolute positions; both NULL for no spans.  All pointer
 * fields are device pointers and may be NULL.
 */
typedef struct {
  int32_t causal;
  int32_t window;
  const int64_t *span_offsets;
  const int64_t *spans;
  const void *extra;
  const int64_t *q_start;
} extkv_bias_spec;

/*
 * TensorScatter of new K/V rows into the static cache, in place
 * ("Skill: Attention Optimization", "In-place KV for ONNX Attention via
 * TensorScatter (static cache)"): for every b < B, h < Hkv, s < S_new
 *     k_cache[b,h,write_idx[b]+s,:] = k_new[b,h,s,:]   (and the same for V).
 * The scatter runs along the sequence axis of the BNSH cache.  A bit-exact
 * copy.  S_new == 0 (a KV-shared layer, which writes no K/V) is a no-op.
 * Requires D * sizeof(T) % 16 == 0 and 16-byte aligned tensors.  A batch whose
 * rows would leave [0, max_seq) is skipped and flagged EXTKV_DEV_BAD_WRITE_IDX.
 */
int ext_kv_scatter(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                   const int64_t *write_idx, int64_t B, int64_t Hkv, int64_t S_new,
                   int64_t max_seq, int64_t D, int dtype, int32_t *status, void *stream);

/*
 * Materialises the (B,1,S_q,max_seq) additive bias of `spec` (see
 * extkv_bias_spec; mobius issue #366, deliverable and acceptance criteria)
 * into `bias`.  Bit-exact: every entry is either the extra term, +0, or
 * lowest(T).  Requires max_seq * sizeof(T) % 16 == 0, max_seq <= 2^31 - 256
 * (else EXTKV_ERR_UNSUPPORTED) and a 16-byte aligned
 * `bias` (and `extra`).  A batch with nonpad outside [0, max_seq] is left
 * untouched and flagged EXTKV_DEV_BAD_NONPAD.
 */
int build_static_cache_bias(void *bias, const extkv_bias_spec *spec, const int64_t *nonpad,
                            int64_t B, int64_t S_q, int64_t max_seq, int dtype,
                            int32_t *status, void *stream);

/*
 * A boolean attention mask as the additive bias that attention_ext_kv takes
 * ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 6: the bool
 * mask is converted to an additive bias; the attention-mask skill, "Bool mask
 * vs float additive bias": both represent any pattern).  mask: (B,1,S_q,max_seq)
 * bytes, nonzero = attend; bias: (B,1,S_q,max_seq) of T, written 0 where the
 * mask is set and lowest(T) (the sentinel of build_static_cache_bias) where it
 * is not.  Bit-exact.  Both 16-byte aligned.  Slots at or beyond nonpad[b] stay
 * masked by attention_ext_kv whatever the mask says; a mask that already
 * applies causal masking must not be combined with a causal fused spec (the
 * pages warn against applying causal twice).  A maskless causal layer
 * (is_causal = 1 with nonpad, no mask) needs no bias at all: pass the fused
 * spec {causal = 1, window = 0} to attention_ext_kv.
 */
int build_bias_from_bool_mask(void *bias, const uint8_t *mask, int64_t B, int64_t S_q, int64_t max_seq,
                              int dtype, void *stream);

/*
 * Bytes of device workspace attention_ext_kv needs for these sizes on the
 * current device: enough for whichever kernel runs, chosen automatically or
 * by extkv_set_algo.  The decode path keeps its live-tile plan and the
 * partial results of units split across CTAs there; the prefill path, with a
 * materialised bias or an extra term, one 64-bit mask of attended keys per
 * (batch, 128-row query tile, 64-key tile), and for a materialised bias each
 * query row's attended keys per 128-key tile (16 bytes) with a byte per tile
 * saying whether the bias holds values other than 0 and the sentinel there;
 * for small grids, the partial rows of key splits; the generic path needs
 * none (0).
 * The caller allocates it, 256-byte aligned, and may reuse it for every call
 * on one stream; calls that can overlap on the GPU need separate workspaces.
 * Contents need no initialisation and are not preserved between calls.
 */
size_t attention_ext_kv_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q,
                                       int64_t max_seq, int64_t D, int dtype);

/*
 * Y = softmax(scale * Q K^T + bias) V over the external static cache, for
 * a prefill chunk (S_q > 1) or a decode step (S_q == 1).
 *   - Op order: scale*(Q@K^T), then + bias, then softmax, then @V
 *     ("ONNX Domain Attention (Opset 23/24) CUDA Patterns", section 4; no
 *     softcap).
 *   - Grouped-query heads: query head h reads KV head h / (Hq/Hkv), no KV
 *     replication (section 1, the reshape-Q trick).
 *   - Masking: key j of row (b,i) is masked iff j >= nonpad[b] or its bias
 *     is <= lowest(T) (the sentinel, or -inf).  A finite very negative bias
 *     is not masked.  A row with no unmasked key, and every row of a batch
 *     with nonpad[b] == 0, is written as exact zeros (section 6).  Cache slots
 *     at or beyond nonpad[b] and masked slots are never read into the result,
 *     whatever they hold (NaN included).
 *   - The bias is one of: `bias` (a materialised (B,1,S_q,max_seq) tensor,
 *     16-byte aligned), `fused` (the same specification evaluated in
 *     registers, never materialised; results equal those of
 *     build_static_cache_bias + `bias`), or neither (only nonpad masks).
 *     Passing both is EXTKV_ERR_INVALID_ARG.
 *   - A KV-shared layer ("[GQA] Support KV-shared layers with empty K/V
 *     inputs", Design) is this call on the borrowed cache with no scatter.
 *   - Accumulation is fp32; Y is rounded to T (nearest even).
 *   - Requires Hq % Hkv == 0, 8 <= D <= 512 with D % 8 == 0.  A batch with
 *     nonpad outside [0, max_seq] gets zero rows and EXTKV_DEV_BAD_NONPAD.
 * `workspace` / `ws_bytes`: at least attention_ext_kv_workspace_size(...)
 * bytes of device memory (see there); may be NULL when that size is 0.  Too
 * small a workspace is EXTKV_ERR_INVALID_ARG.
 */
int attention_ext_kv(void *y, const void *q, const void *k_cache, const void *v_cache,
                     const void *bias, const extkv_bias_spec *fused, const int64_t *nonpad,
                     float scale, int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q,
                     int64_t max_seq, int64_t D, int dtype, void *workspace, size_t ws_bytes,
                     int32_t *status, void *stream);

/*
 * attention_ext_kv with a softcap ("ONNX Domain Attention (Opset 23/24) CUDA
 * Patterns", section 4 op order): each scaled score x = scale * q.k becomes
 * softcap * tanh(x / softcap) before the bias is added, so a masked slot stays
 * masked (its V row never reaches the output).  softcap == 0 is
 * attention_ext_kv; a negative, NaN or infinite softcap is
 * EXTKV_ERR_INVALID_ARG.  Every path (decode, prefill, generic) takes it.
 */
int attention_ext_kv_softcap(void *y, const void *q, const void *k_cache, const void *v_cache,
                             const void *bias, const extkv_bias_spec *fused, const int64_t *nonpad,
                             float scale, float softcap, int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q,
                             int64_t max_seq, int64_t D, int dtype, void *workspace, size_t ws_bytes,
                             int32_t *status, void *stream);

/*
 * attention_ext_kv_softcap with value rows of another head size: q is
 * (B,Hq,S_q,Dk), k_cache (B,Hkv,max_seq,Dk), v_cache (B,Hkv,max_seq,Dv) and
 * y (B,Hq,S_q,Dv) ("Skill: Attention Optimization", "ORT CUDA Attention
 * Kernel Dispatch": head_size != v_head_size, the case of a KV-shared layer
 * borrowing the cache of a layer with another head size; the scores use the
 * Dk-long dot products and each output row is a weighted sum of Dv-long
 * value rows).  Dk == Dv is attention_ext_kv_softcap.  Both head sizes are
 * multiples of 8 in [8, 512]; everything else as attention_ext_kv_softcap.
 * The workspace is attention_ext_kv_workspace_size_dv(...) bytes.  Dk != Dv
 * with each of 128, 256, 512 runs on the tensor-core prefill kernel, or for a
 * decode step (g * S_q <= 8 rows per KV head, no softcap) on the decode
 * kernel; other asymmetric pairs run on the exact fp32 SIMT kernel.
 */
int attention_ext_kv_dv(void *y, const void *q, const void *k_cache, const void *v_cache, const void *bias,
                        const extkv_bias_spec *fused, const int64_t *nonpad, float scale, float softcap,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk,
                        int64_t Dv, int dtype, void *workspace, size_t ws_bytes, int32_t *status,
                        void *stream);

/* Workspace bytes for attention_ext_kv_dv (attention_ext_kv_workspace_size with Dk, Dv). */
size_t attention_ext_kv_workspace_size_dv(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq,
                                          int64_t Dk, int64_t Dv, int dtype);

/*
 * ext_kv_scatter followed by attention_ext_kv, in one call: the same results
 * (the caches hold the new rows afterwards, bit for bit, and y is what
 * attention_ext_kv gives over the updated caches).  The scatter is the step
 * just before the attention in the pages' decode graph ("Skill: Attention
 * Optimization", "In-place KV for ONNX Attention via TensorScatter (static
 * cache)"); fusing it saves a launch and a pass over the new rows.
 *   - k_new / v_new: (B, Hkv, S_new, D), written to slots
 *     [write_idx[b], write_idx[b] + S_new) of k_cache / v_cache (which are
 *     therefore not const here).  S_new == 0 is attention_ext_kv.
 *   - Where the decode kernel runs (see attention_ext_kv), it writes the
 *     rows itself and takes the tiles that hold them from k_new / v_new;
 *     elsewhere the scatter kernel runs first, then the attention.
 *     extkv_last_kernel() names the path ("..._scatter" when fused).
 *   - A batch whose new rows would leave [0, max_seq) is not written and is
 *     flagged EXTKV_DEV_BAD_WRITE_IDX; its attention reads the cache as it was.
 *   - Other arguments, requirements and errors as for ext_kv_scatter and
 *     attention_ext_kv; the workspace is attention_ext_kv_workspace_size(...).
 */
int attention_ext_kv_scatter(void *y, const void *q, void *k_cache, void *v_cache, const void *k_new,
                             const void *v_new, const int64_t *write_idx, int64_t S_new,
                             const void *bias, const extkv_bias_spec *fused, const int64_t *nonpad,
                             float scale, int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q,
                             int64_t max_seq, int64_t D, int dtype, void *workspace, size_t ws_bytes,
                             int32_t *status, void *stream);

/*
 * Size of the static scratch array behind attention_ext_kv_noalloc: 8 MiB of
 * device memory, held by every GPU that loads this library until exit.  The
 * decode call's scratch is its plan tables plus two fp32 partials per CTA of
 * the persistent grid, (16 + R * D) floats each, R = (Hq/Hkv) * S_q: about
 * 2.6 MB for Hq/Hkv = 2, D = 256; a D = 512 decode with 8 query rows per
 * unit over the full grid needs about 10 MB and is refused.
 */
#define EXTKV_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * attention_ext_kv for callers that cannot allocate device memory.  The pages
 * have no counterpart; it exists for code that is handed only its input and
 * output buffers -- e.g. a custom operator of an inference runtime whose
 * operator interface offers no scratch allocator, or a latency-critical path
 * where a cudaMalloc (which may synchronise the device) is not acceptable.
 *   - Same arguments and results as attention_ext_kv without the workspace:
 *     the decode path's scratch lives in a static device array of
 *     EXTKV_NOALLOC_SCRATCH_BYTES.  This call allocates nothing.
 *   - Decode shapes only (bf16, (Hq/Hkv)*S_q <= 8, D in {64,128,256,512});
 *     other shapes, and sizes whose scratch would exceed the array, return
 *     EXTKV_ERR_UNSUPPORTED with a message.
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress), and so does the first call after the device's
 *     context was rebuilt (cudaDeviceReset); make those calls outside any
 *     stream capture.
 *   - An unknown dtype returns EXTKV_ERR_INVALID_ARG; fp32 is refused as
 *     EXTKV_ERR_UNSUPPORTED (the decode kernel is bf16 only).
 *   - extkv_last_kernel() and extkv_last_launches() report this call as they
 *     do attention_ext_kv.
 *   - Every call on a device shares the one array, and it keeps the previous
 *     call's contents (the call clears what must start at zero itself).  Calls
 *     that can overlap on the GPU -- on different streams without ordering --
 *     race on it.
 */
int attention_ext_kv_noalloc(void *y, const void *q, const void *k_cache, const void *v_cache,
                             const void *bias, const extkv_bias_spec *fused,
                             const int64_t *nonpad, float scale, int64_t B, int64_t Hq,
                             int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t D, int dtype,
                             int32_t *status, void *stream);

/* Zeroes the 16-byte status word on `stream` (asynchronous). */
int extkv_clear_status(int32_t *status, void *stream);

/*
 * Synchronises `stream`, copies the status word to the host and returns
 * EXTKV_OK when no flag is set, else EXTKV_ERR_DEVICE with the flags spelled
 * out in extkv_last_error().  The word is not cleared.
 */
int extkv_read_status(const int32_t *status, void *stream);

/* Message of the calling thread's last failed call ("" if none). */
const char *extkv_last_error(void);

/*
 * Name of the kernel the calling thread's last successful attention_ext_kv
 * launched, so a test can check which path ran instead of trusting a
 * fallback ("ONNX Domain Attention ...", section 7: always verify which
 * runner a test actually hits).
 */
const char *extkv_last_kernel(void);

/*
 * Number of kernels the calling thread's last successful attention_ext_kv
 * launched (a plan kernel, the attention kernel, a merge kernel), for callers
 * and benchmarks that account for launches.  0 before any call.
 */
int extkv_last_launches(void);

/*
 * Limit, in polls, of the attention kernels' pipeline waits for the calling
 * thread's later calls: polls >= 0 sets it (0: a wait that is not already
 * complete gives up at once); a negative value restores the kernels' own
 * limit (about 4 million polls), the default.  For failure-detection tests:
 * with a tiny limit a wait runs out before its data lands, the kernel sets
 * EXTKV_DEV_TIMEOUT in the status word, waits (at the full limit) for its own
 * copies in flight, frees its tensor memory and returns; the output of that
 * call is not valid.  Returns the previous setting (negative: the default).
 * The pages state the rule this serves, not the mechanism: every launch is
 * checked and a failure never passes silently ("ONNX Domain Attention
 * (Opset 23/24) CUDA Patterns", section 5).
 */
int extkv_set_wait_polls(int polls);

/*
 * Recorded steps.  A caller that issues the same library calls over the same
 * buffers every step (a decode loop) can record them once and then start the
 * whole step with one launch, instead of one host launch per kernel (the
 * decode path of attention_ext_kv launches three).
 *   extkv_step_begin   creates a stream, starts capturing the calling thread's
 *                      work on it into a CUDA graph, and returns the stream in
 *                      *stream; the library calls that follow are issued with it.
 *   extkv_step_end     ends that capture, instantiates the graph, destroys the
 *                      stream and returns the step in *step (null on an error,
 *                      and the capture is discarded).
 *   extkv_step_launch  starts the step on `stream` (any stream of the same
 *                      device): every call of it runs again, reading and
 *                      writing the buffers it was recorded with -- their
 *                      contents may change between launches, their addresses
 *                      may not -- and the status word it was given.
 *   extkv_step_free    releases a step (null: nothing).
 * Between begin and end call nothing that synchronises (extkv_read_status),
 * and issue each call once before recording it, so that its first-use setup
 * (kernel attributes, tensor maps) stays outside the capture.  The caller owns
 * the step.  Returns EXTKV_OK, EXTKV_ERR_INVALID_ARG for a null argument, or
 * EXTKV_ERR_CUDA (message in extkv_last_error).
 */
typedef struct extkv_step extkv_step;
int extkv_step_begin(void **stream);
int extkv_step_end(void *stream, extkv_step **step);
int extkv_step_launch(const extkv_step *step, void *stream);
void extkv_step_free(extkv_step *step);

/*
 * Attention kernel selection for the calling thread.  EXTKV_ALGO_AUTO picks
 * by shape and type; the others force one kernel, and attention_ext_kv then
 * returns EXTKV_ERR_UNSUPPORTED for shapes that kernel cannot run.  Returns
 * the previous setting, or EXTKV_ERR_INVALID_ARG for an unknown value.
 */
#define EXTKV_ALGO_AUTO 0
#define EXTKV_ALGO_GENERIC 1 /* fp32 SIMT, one warp per query row: any supported shape */
#define EXTKV_ALGO_DECODE 2  /* the decode kernels: bf16, S_q <= 8, S_q*Hq/Hkv <= 64, up to 1024
                                batches, D in {64,128,256,512} (and pairs of 128, 256, 512); the
                                cluster kernel where every group of up to 8 of a KV head's query
                                rows can have 8 CTAs resident at once, stream-K otherwise */
#define EXTKV_ALGO_PREFILL 3 /* tcgen05/TMEM prefill: bf16, head sizes 64/64 or any pair of 128, 256, 512;
                                one CTA per query tile */
#define EXTKV_ALGO_PREFILL_PAIR 4 /* the same prefill on CTA pairs with 2-SM MMAs (two query heads of a
                                     KV head as one M = 256 tile) where the shape allows it: head size
                                     256/256, an even group, no split over keys; otherwise the
                                     EXTKV_ALGO_PREFILL kernel.  Opt-in: slower than one CTA per tile
                                     on the shapes measured (the pair waits on both halves' softmax
                                     before each P.V) */
#define EXTKV_ALGO_DECODE_STREAMK 5 /* the stream-K decode alone: a plan kernel (materialised bias),
                                       the decode kernel over equal slices of all live tiles, a
                                       merge kernel for units split across slices */
#define EXTKV_ALGO_DECODE_CLUSTER 6 /* the cluster decode alone: a cluster of up to 8 CTAs per
                                       (batch, KV head, group of up to 8 query rows) sharing its
                                       live tiles, combined through distributed shared memory (one
                                       kernel); with few units, up to 16 clusters per unit whose
                                       partials the stream-K merge kernel combines.  bf16, one head
                                       size in {64,128,256,512}, S_q <= 8, S_q*Hq/Hkv <= 64, all
                                       clusters resident at once; a materialised bias with
                                       S_q*max_seq <= 8192 (one copy of a batch's rows is
                                       scanned); with the fused spec, no spans when S_q > 1 */
int extkv_set_algo(int algo);

#ifdef __cplusplus
}
#endif
#endif /* EXTKV_H_ */
