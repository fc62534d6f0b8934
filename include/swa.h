/*
 * swa.h -- sliding-window grouped-query attention on GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels.  It covers Gemma-3/4-style sliding
 * layers: prefill (causal or generic mask) into a prompt-sized sliding cache,
 * compaction at first decode into an anchored buffer of W + 64 rows,
 * single-token decode under one fixed-shape runtime mask shared by all
 * sliding layers, and a roll every 64 decode tokens.
 *
 * Sources (page title, section):
 *   [SPYRE]   "Enable compact sliding-window attention for Gemma 3 and Gemma 4
 *             variants" (torch-spyre/hf-adapters pull request 496), Summary,
 *             Compilation behavior, Performance.
 *   [FASTLLM] "Add SDPA attention implementation" (ServiceNow/Fast-LLM pull
 *             request 512), Summary.
 *   [BONSAI]  "Gemma3 Local Attention Cache" (jax-ml/bonsai issue 124).
 *
 * Conventions (every call):
 *   - Device pointers belong to the caller.  The library allocates no device
 *     memory; it owns only the small host-side cache handle.
 *   - Every call that takes a stream is asynchronous on that stream.
 *   - Arguments are validated on the host before any CUDA call; a bad call
 *     returns a status and leaves device memory untouched.
 *     swa_last_error() then describes the problem (per host thread).
 *   - Device kernels never trap.  An inconsistency found on the device (a
 *     corrupted cache state, an image block that crosses a chunk end) is
 *     recorded in a device error word; swa_cache_check() / swa_plan_check()
 *     report it as SWA_EDEVICE.
 *   - bf16 tensors are raw IEEE bfloat16 bits (swa_bf16).  Every tensor
 *     pointer must be 16-byte aligned.
 *   - Layouts are row-major with the last dimension contiguous.
 *
 * Mask predicate (one sequence, padded positions q and k):
 *   allowed(q,k) = q >= vs and k >= vs and doc(q) == doc(k) and q - k < W
 *                  and (k <= q or (img(q) >= 0 and img(q) == img(k)))
 * i.e. window AND (causal OR same image block) with left padding vs
 * ([SPYRE] Summary; [FASTLLM] Summary for documents).  The window holds W keys
 * including the query.  Each image id must form one contiguous run.
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SWA_API __attribute__((visibility("default")))
#else
#define SWA_API
#endif

typedef struct CUstream_st* swa_stream_t; /* the same type as cudaStream_t */
typedef uint16_t swa_bf16;                /* raw bfloat16 bits */

typedef enum swa_status {
  SWA_OK = 0,
  SWA_EINVAL = 1,       /* invalid argument (NULL, shape, alignment, size) */
  SWA_ESTATE = 2,       /* the cache is in the wrong state for this call */
  SWA_EUNSUPPORTED = 3, /* valid but not supported (head size, group size) */
  SWA_ECUDA = 4,        /* a CUDA runtime call failed */
  SWA_ETIMEOUT = 5,     /* a bounded device wait gave up */
  SWA_EDEVICE = 6       /* an earlier kernel recorded a device-side error */
} swa_status;

enum { SWA_CACHE_PREFILL = 0, SWA_CACHE_COMPACT = 1, SWA_CACHE_RING = 2 };
enum { SWA_MODE_CAUSAL = 0, SWA_MODE_GENERIC = 1 };
enum { SWA_MASK_DECODE = 0, SWA_MASK_PREFILL = 1, SWA_MASK_DENSE_DEBUG = 2 };

/* Rows added to the window by the compact buffer, and the roll period in
 * decode tokens ([SPYRE] Summary: the compact buffer is W + 64 rows and rolls
 * every 64 decode tokens). */
#define SWA_ROLL_ROWS 64

/* ------------------------------------------------------------------------ */
/* Cache                                                                     */
/* ------------------------------------------------------------------------ */

/* Shape of a sliding cache.  One cache holds every sliding layer of a model:
 * K and V, each [layers, batch, kv_heads, rows, head_dim] bf16.
 *   kind       SWA_CACHE_PREFILL: prompt-sized, row = position ([SPYRE]
 *              Summary: prompt-sized sliding caches).
 *              SWA_CACHE_COMPACT: W + 64 rows, row r holds position origin + r.
 *              SWA_CACHE_RING: W rows, position p lives in row p % W; it never
 *              rolls ([BONSAI] Steps 1-3: smaller caches for the local layers,
 *              positions assigned with % and wrapping around, a window mask
 *              compatible with the wrap).  Decodes like a compact cache.
 *   prompt_len S, the padded prompt length (positions 0 .. S-1).
 *   rows       0 selects the default: max(S, W + 64) for a prefill cache
 *              (short prompts still get the minimum width, [SPYRE] Summary),
 *              W + 64 for a compact cache, W for a ring (the only values
 *              accepted there).
 *   window     W >= 1; a compact cache needs W >= 64. */
typedef struct swa_cache_desc {
  int32_t kind;
  int32_t layers;
  int32_t batch;
  int32_t kv_heads;
  int32_t head_dim;
  int32_t window;
  int32_t prompt_len;
  int32_t rows;
} swa_cache_desc;

/* Device-side cache state (the first 32 bytes of the cache memory).  Kernels
 * read position data only from here, so one captured graph serves every
 * decode position ([SPYRE] Compilation behavior: positions, the origin and
 * padding are device data, not constants of the compiled program). */
typedef struct swa_device_state {
  int32_t origin;     /* position held by row 0 (compact: S - W at first)   */
  int32_t next_row;   /* row the next decode step writes                    */
  int32_t cur_row;    /* row written by the current step (-1 before any)    */
  int32_t step;       /* decode steps taken                                  */
  int32_t prompt_len; /* S                                                   */
  int32_t window;     /* W                                                   */
  int32_t rows;       /* physical rows per (layer, sequence, head) slab      */
  int32_t error;      /* first device-side error code, 0 = none              */
} swa_device_state;

typedef struct swa_cache swa_cache; /* opaque host handle */

/* Bytes of device memory a cache of this shape needs (state + valid_start +
 * K + V, each part 256-byte aligned): the prompt-sized prefill cache and the
 * W + 64-row compact buffer of [SPYRE] Summary, or the W-row ring of [BONSAI].
 * Returns 0 for an invalid desc. */
SWA_API size_t swa_cache_bytes(const swa_cache_desc* desc);

/* Bind a cache to caller-owned device memory `dev_mem` (>= swa_cache_bytes,
 * 256-byte aligned), zero-fill it and write the initial state ([SPYRE]
 * Summary and Compilation behavior: the index map lives in device data):
 *   prefill cache: origin 0, next_row S;   compact cache: origin S - W,
 *   next_row W (right-aligned anchoring; rows of negative positions stay
 *   zero and are never admitted by the mask);   ring: origin 0 (unused),
 *   next_row S % W.
 * dev_valid_start: [batch] int32 device array of left-pad counts (copied),
 * or NULL for no padding.  On success *out receives a handle the caller frees
 * with swa_cache_free (which never frees dev_mem). */
SWA_API swa_status swa_cache_alloc(const swa_cache_desc* desc, void* dev_mem, size_t bytes,
                                   const int32_t* dev_valid_start, swa_stream_t stream,
                                   swa_cache** out);

/* Release the host handle only.  NULL is ignored.  (Library plumbing: the
 * pages have no counterpart.) */
SWA_API void swa_cache_free(swa_cache* cache);

/* Resolved shape and device pointers of a cache (any out pointer may be NULL):
 * K and V base pointers ([layers, batch, kv_heads, rows, head_dim] bf16) and
 * the swa_device_state.  (Library plumbing: the pages have no counterpart.) */
SWA_API swa_status swa_cache_info(const swa_cache* cache, swa_cache_desc* desc_out, void** k_out,
                                  void** v_out, void** state_out);

/* Host mirror of the index map: origin, next_row and decode steps taken
 * (the compact index of [SPYRE] Summary, kept on the host only to report
 * misuse synchronously). */
SWA_API swa_status swa_cache_position(const swa_cache* cache, int32_t* origin, int32_t* next_row,
                                      int32_t* step);

/* Advance the host mirror by `steps` decode steps whose masks were built by
 * replaying a captured CUDA graph (a replay advances only the device state;
 * one graph per fixed shape serves every position, [SPYRE] Compilation
 * behavior).  SWA_ESTATE if that would run past a due roll.  No CUDA call. */
SWA_API swa_status swa_cache_advance(swa_cache* cache, int32_t steps);

/* Synchronise `stream` and report a device-side error recorded in the cache
 * state (SWA_EDEVICE), clearing it.  (Library plumbing: the pages have no
 * counterpart.) */
SWA_API swa_status swa_cache_check(swa_cache* cache, swa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Masks                                                                     */
/* ------------------------------------------------------------------------ */

/* Description of one prefill call (one chunk of queries).
 *   batch        B sequences (cache mode), 1 for packed documents.
 *   seq_len      key positions per sequence: S (cache mode) or the total
 *                token count T (packed documents).
 *   chunk_start  first query position of this call ([SPYRE] Summary:
 *   chunk_len    chunked prefill is preserved); 0 and T for packed documents.
 *   window       W.
 *   num_docs     number of packed documents (0 in cache mode).
 *   valid_start  [B] int32 device, left-pad counts, or NULL (no padding).
 *   img_id       [B, seq_len] int32 device, -1 for text, the image-block id
 *                for image tokens, or NULL (text only).  Generic mode only.
 *                Each id must be one contiguous run inside one chunk.
 *   cu_seqlens   [num_docs + 1] int32 device document offsets (packed mode,
 *                [FASTLLM] Summary), or NULL.
 *   plan         a plan built by swa_build_mask(SWA_MASK_PREFILL) for exactly
 *                this meta; required by generic-mode prefill. */
typedef struct swa_prefill_meta {
  int32_t batch;
  int32_t seq_len;
  int32_t chunk_start;
  int32_t chunk_len;
  int32_t window;
  int32_t num_docs;
  const int32_t* valid_start;
  const int32_t* img_id;
  const int32_t* cu_seqlens;
  const void* plan;
} swa_prefill_meta;

/* Bytes of the device buffer swa_build_mask(SWA_MASK_PREFILL) fills (the
 * generic prefill plan of [SPYRE] Compilation behavior). */
SWA_API size_t swa_prefill_plan_bytes(const swa_prefill_meta* meta);

/* Build a runtime mask on the device.
 * SWA_MASK_DECODE (cache: compact, meta NULL): the per-step decode mask
 *   [batch, rows] uint8 at dev_out, shared by every sliding layer of the step
 *   ([SPYRE] Summary: one fixed-shape runtime mask per decode step).  It
 *   advances the device state: cur_row = next_row, next_row += 1, step += 1,
 *   and mask[b, r] = (r <= cur_row) and (pos_r > p - W) and
 *   (pos_r >= valid_start[b]) and (pos_r >= 0), pos_r = origin + r,
 *   p = S + step (before the increment).  SWA_ESTATE when a roll is due.
 *   Ring cache (SWA_MASK_DECODE on SWA_CACHE_RING): cur_row = p % W,
 *   next_row = (p + 1) % W, and mask[b, r] = (pos_r >= valid_start[b]) and
 *   (pos_r >= 0) with pos_r = p - ((p - r) mod W), the position row r holds
 *   (always in (p - W, p]).
 * SWA_MASK_PREFILL (cache may be NULL, meta required): the prefill plan at
 *   dev_out (swa_prefill_plan_bytes): for every query row the interval
 *   [lo, hi] of keys it attends (the predicate above reduces to one interval
 *   per row), and for every 128-row query tile the key range it touches, so
 *   the kernel skips key tiles no row needs.  Positions, padding, image
 *   blocks and documents enter only as device data.
 * SWA_MASK_DENSE_DEBUG (meta required; meta->plan or causal arithmetic when
 *   NULL): the dense mask [batch, chunk_len, seq_len] uint8 the prefill kernel
 *   applies, for tests. */
SWA_API swa_status swa_build_mask(swa_cache* cache, int32_t kind, const swa_prefill_meta* meta,
                                  void* dev_out, swa_stream_t stream);

/* Report a device-side error recorded while building `plan` (SWA_EDEVICE,
 * e.g. an image block crossing the chunk end, or recorded by the backward
 * pass that used it); synchronises `stream`.  ([SPYRE] Compilation behavior:
 * the generic plan; the error word is this library's own.) */
SWA_API swa_status swa_plan_check(const void* plan, swa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Prefill                                                                   */
/* ------------------------------------------------------------------------ */

/* Sliding-window attention for one chunk of queries.
 * Cache mode (cache = prefill cache): q [B, C, Hq, D]; k, v [B, C, Hkv, D]
 *   are this chunk's keys/values, written to cache rows
 *   [chunk_start, chunk_start + C) of `layer` first; attention then reads the
 *   cache.  k = v = NULL means the rows are already in the cache.
 * Packed mode (cache = NULL): q [T, Hq, D], k, v [T, Hkv, D]; documents from
 *   meta->cu_seqlens; mode must be SWA_MODE_GENERIC.
 * mode SWA_MODE_CAUSAL: the narrow causal plan, img_id must be NULL and no
 *   plan is needed; SWA_MODE_GENERIC: the generic plan (future same-image
 *   keys, documents) reads meta->plan ([SPYRE] Compilation behavior).
 * out [.., Hq, D] bf16 like q; lse (natural-log sum of exp of the scaled
 *   scores) [.., Hq] fp32, or NULL.  Rows with no admitted key give out = 0
 *   and lse = -inf.  scale multiplies q.k (typically 1/sqrt(D)).
 * Supported: head_dim 256 or 512, Hq a multiple of Hkv. */
SWA_API swa_status swa_prefill(swa_cache* cache, int32_t layer, int32_t mode, int32_t q_heads,
                               int32_t kv_heads, int32_t head_dim, const swa_prefill_meta* meta,
                               const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float scale,
                               swa_bf16* out, float* lse, swa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Backward (training)                                                       */
/* ------------------------------------------------------------------------ */

/* Workspace bytes swa_prefill_backward needs for this meta (whole sequences:
 * chunk_start = 0, chunk_len = seq_len) and head count; 0 with
 * swa_last_error set on invalid arguments.  The score tiles dominate it:
 * 3 x 32 KB per (sequence, query head, 128-row query tile, key tile of its
 * band), the band being 1 + ceil((W - 1) / 128) key tiles without images and
 * every key tile with them.  (The training pass of "Add SDPA attention
 * implementation", Summary; the workspace layout is this library's own.) */
SWA_API size_t swa_prefill_backward_workspace_bytes(int32_t q_heads, const swa_prefill_meta* meta);

/* Gradients of swa_prefill's output with respect to q, k and v, for training
 * ("Add SDPA attention implementation", Summary: models with head size 512
 * must train; its benchmark table times forward + backward of packed
 * documents).  With P the softmax weights of the forward pass over the keys
 * each query admits, dout = dL/dout, and delta_i = dout_i . out_i:
 *   dv_j = sum_i P_ij dout_i,   dS_ij = scale * P_ij * (dout_i . v_j - delta_i),
 *   dq_i = sum_j dS_ij k_j,     dk_j = sum_i dS_ij q_i,
 * with dk and dv summed over the query heads that share a KV head.
 * Whole sequences only (meta->chunk_start = 0, chunk_len = seq_len), with the
 * plan swa_build_mask(SWA_MASK_PREFILL) built for that meta (padding, image
 * blocks or packed documents as in swa_prefill's generic mode).
 * Layouts: q, out, dout, dq [B, S, Hq, D]; k, v, dk, dv [B, S, Hkv, D]
 * (packed documents: B = 1, S = T); lse [B, S, Hq] fp32 as swa_prefill wrote
 * it (natural log); out is swa_prefill's output.  All bf16 except lse.
 * Rows with no admitted key, and keys no query admits, get zero gradients.
 * workspace: >= swa_prefill_backward_workspace_bytes device bytes, 256-byte
 * aligned, no initialisation needed; the caller owns it.  Three kernels run
 * on `stream`; calls that overlap on the GPU need separate workspaces.
 * A device-side inconsistency (a band wider than the workspace allows, a
 * bounded wait that gave up) is recorded in the plan's error word:
 * swa_plan_check reports it.
 * Supported: head_dim 256 or 512, Hq a multiple of Hkv. */
SWA_API swa_status swa_prefill_backward(int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                                        const swa_prefill_meta* meta, const swa_bf16* q, const swa_bf16* k,
                                        const swa_bf16* v, const swa_bf16* out, const swa_bf16* dout,
                                        const float* lse, float scale, swa_bf16* dq, swa_bf16* dk,
                                        swa_bf16* dv, void* workspace, size_t ws_bytes, swa_stream_t stream);

/* Compaction at first decode ([SPYRE] Summary): rows [S - W, S) of every
 * (layer, sequence, head) slab of the prefill cache go to rows [0, W) of the
 * compact cache (same shape apart from rows, same S and W); rows of negative
 * positions are zero.  Into a ring cache, position pos goes to row pos % W
 * instead.  Bit-exact copy. */
SWA_API swa_status swa_compact(const swa_cache* prefill, swa_cache* compact, swa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Decode                                                                    */
/* ------------------------------------------------------------------------ */

/* Workspace bytes swa_decode needs for this cache and query-head count (the
 * split-K scratch of the decode of [SPYRE] Summary; the split is this
 * library's own). */
SWA_API size_t swa_decode_workspace_bytes(const swa_cache* cache, int32_t q_heads);

/* One decode token of one sliding layer, after swa_build_mask(DECODE) of the
 * step: appends k_new, v_new [B, Hkv, D] at the step's row (the new row goes
 * into the compact cache at its row index, [SPYRE] Summary), then attends
 * q [B, Hq, D] over the rows the mask [B, rows] admits (decode reads only the
 * compact buffer's rows, [SPYRE] Compilation behavior).  Split-K over rows, with the last
 * CTA of each (sequence, kv head) combining the partial results.
 * out [B, Hq, D] bf16; lse [B, Hq] fp32 or NULL.
 * workspace: >= swa_decode_workspace_bytes device bytes, zero-filled before
 * its first use; each call leaves it ready for the next.  Calls that overlap
 * on the GPU need separate workspaces.
 * KV-sharing layer ([SPYRE] Summary: layers that reuse another layer's K/V keep working):
 * k_new = v_new = NULL attends over layer `layer`'s rows without appending;
 * that layer's own swa_decode must already have appended this step's row.
 * Launch chaining: the kernel is launched with programmatic dependent launch.
 * It may start while the previous kernel of the stream is still running and
 * read this layer's cache rows then; it waits for that kernel before reading
 * q, k_new, v_new, the mask and the cache state, and before writing anything.
 * So the kernel launched just before it on the stream must not write this
 * layer's cache rows (swa_build_mask, projections and the other layers'
 * swa_decode calls do not; swa_roll and swa_compact are followed by the
 * step's swa_build_mask anyway).  A KV-sharing call reads nothing before
 * that wait.
 * Supported: head_dim 64, 128, 256 or 512; Hq / Hkv in {1, 2, 4, 8}. */
SWA_API swa_status swa_decode(swa_cache* cache, int32_t layer, int32_t q_heads, const swa_bf16* q,
                              const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask,
                              float scale, swa_bf16* out, float* lse, void* workspace,
                              size_t ws_bytes, swa_stream_t stream);

/* Flag of swa_decode_ex (below). */
#define SWA_DECODE_INPUTS_READY 1u

/* swa_decode with flags (0: exactly swa_decode; the decode itself is
 * [SPYRE] Summary's, the flag is library plumbing with no counterpart in the
 * pages).
 * SWA_DECODE_INPUTS_READY: the caller guarantees that q, k_new, v_new, the
 * mask and the cache state are complete in memory as soon as the kernel
 * enqueued immediately before this call starts running, and that this kernel
 * does not write them.  This holds for the decodes of a step's layers 1, 2, ...
 * when the queries and new rows of every layer were produced before the
 * step's swa_build_mask, each layer's call enqueued right after the previous
 * layer's: the mask kernel lets no successor start before it has finished,
 * the first layer's decode (called without the flag) waits for it, and each
 * later layer's decode starts only after the previous one has started.  The
 * kernel then reads those inputs before it waits for the previous kernel (see
 * "Launch chaining" above; its compute and writes still follow that wait),
 * which takes one round trip to global memory off each layer's critical path.
 * Ignored by a KV-sharing call (k_new = NULL) and by the batched-decode kernel
 * (many slabs).  With the flag and inputs that are not complete when the
 * previous kernel starts, results are undefined.  Other flag bits: SWA_EINVAL. */
SWA_API swa_status swa_decode_ex(swa_cache* cache, int32_t layer, int32_t q_heads, const swa_bf16* q,
                                 const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask,
                                 float scale, swa_bf16* out, float* lse, void* workspace,
                                 size_t ws_bytes, uint32_t flags, swa_stream_t stream);

/* Largest scratch area swa_decode_noalloc can use (bytes): the device image of
 * libswa.so holds one static array of this size on every GPU that loads it,
 * until the process exits.  Its first SWA_DECODE_STATIC_MAX_SLABS x 4 bytes
 * (rounded up to 256) are ticket counters, one per (sequence, KV head) slab;
 * the split statistics and partials follow. */
#define SWA_DECODE_STATIC_SCRATCH_BYTES (8u << 20)
#define SWA_DECODE_STATIC_MAX_SLABS 65536

/* swa_decode for callers that may not allocate device memory -- for example a
 * plugin running inside an inference runtime that plans every buffer up front
 * and hands the plugin only its inputs and outputs, where a cudaMalloc would
 * break the runtime's memory accounting and can synchronise the device.  The
 * pages have no counterpart to this entry point; it exists only for such
 * callers.
 * Same arguments, results and checks as swa_decode, without the workspace.
 * Only shapes whose splits merge through the workspace (several splits per
 * slab that do not form one thread-block cluster: large batches, or windows
 * longer than 16 clusters' worth of rows) use scratch; for them the ticket
 * counters and the split partials live in the static array above, and a shape
 * with more than SWA_DECODE_STATIC_MAX_SLABS slabs or partials that do not fit
 * fails with SWA_EUNSUPPORTED before any CUDA call.
 * The first call on a device does a set-up with that device current: it looks
 * up the array's device address and clears the ticket area (a synchronous
 * memset); make that first call before any stream capture.  Every decode
 * leaves its slabs' tickets at zero again (also when a bounded wait gave up),
 * so later calls need no clearing.  Every call on a device shares the one
 * array and leaves the last call's partials in it, so calls that overlap on
 * the GPU (other streams, other host threads) race: serialise them.
 * Allocates nothing. */
SWA_API swa_status swa_decode_noalloc(swa_cache* cache, int32_t layer, int32_t q_heads, const swa_bf16* q,
                                      const swa_bf16* k_new, const swa_bf16* v_new, const uint8_t* mask,
                                      float scale, swa_bf16* out, float* lse, swa_stream_t stream);

/* The roll every 64 decode tokens ([SPYRE] Summary: rows shift down by a
 * fixed offset with device-to-device copies): when next_row == rows, rows [64, rows) of every
 * slab of every layer move to rows [0, W) (an overlap-safe in-place shift),
 * origin += 64, next_row = W.  SWA_ESTATE unless the roll is due (a ring
 * cache never rolls). */
SWA_API swa_status swa_roll(swa_cache* cache, swa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/* Message of the last failed call on this host thread ("" if none).
 * (Library plumbing: the pages have no counterpart.) */
SWA_API const char* swa_last_error(void);

/* Static name of a status code.  (Library plumbing.) */
SWA_API const char* swa_status_string(swa_status status);

/* Library ABI version (major * 100 + minor).  (Library plumbing.) */
SWA_API int32_t swa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
