/*
 * rkv.h — C ABI of librkv.so: the rolling KV-cache step for unbounded
 * streaming attention, on one NVIDIA B300 (sm_103a).
 *
 * What one step does, for every active audio stream and every layer
 * (Audio8 ASR Infinite 无限长转写原理, "Rolling KV Cache 三步拆解"):
 *   1. the window is fixed; once full, the oldest tokens leave it
 *      (第 1 步; voxtral.c rolling-KV article §二 keeps the last
 *      VOX_DEC_WINDOW positions);
 *   2. the new K/V are written with RoPE at their position: either the
 *      logical position physical + kv_pos_offset, never re-encoded
 *      (voxtral.c article §二 "RoPE 逻辑位置修正", the offset-only scheme),
 *      or a window-relative position, every retained key being rotated by
 *      R(-delta) when delta positions leave the window (第 2 步, the exact
 *      re-base scheme);
 *   3. attention of the step's queries over the fixed window, so the cost
 *      per step is constant (第 3 步); one query per stream for the decoder
 *      (one text token per clock step, Edge0/Audio8-ASR-Infinite model card
 *      "亮点"), frame_len = 4 queries with a causal mask inside the step for
 *      the audio encoder's incremental step (voxtral.c article §三).
 *
 * Conventions for every function below.
 *   - Return value: RKV_OK (0) or a negative rkv_status.  Host-side
 *     validation failures return before anything is enqueued.  The message
 *     of the last failure is rkv_last_error(handle) (or rkv_last_error(NULL)
 *     for calls without a handle; per thread).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call that takes one is asynchronous on it unless
 *     stated, and may be captured into a CUDA graph.
 *   - Device buffers are owned by the caller; the library never allocates
 *     or frees device memory.  Pointers marked "device" must be device (or
 *     managed) memory of the current device; "host" pointers are read
 *     during the call only.
 *   - bf16 tensors are uint16 bit patterns of bfloat16, row-major, densely
 *     packed, 16-byte aligned.
 *   - Errors found by kernels (an index outside its table, a wait that timed
 *     out) are recorded in a device status word and reported by
 *     rkv_sync_status(); the kernel skips the offending access and returns.
 *
 * Per-step order.  rkv_begin_step opens a step; then, for every layer,
 * rkv_rebase (exact scheme only) and rkv_append_rope in either order, then
 * rkv_decode_attn (any number of times).  Calling rkv_append_rope or
 * rkv_rebase twice for a layer in one step, rkv_decode_attn before them,
 * rkv_rebase in the offset-only scheme, or opening the next step while a
 * layer lacks them returns RKV_ERR_STATE.
 *
 * Memory in HBM (pool_dev).  Regions of [L][pages][Hkv][page_size][d]
 * 16-bit elements: rotated keys (fp16), values (bf16), and in
 * RKV_SCHEME_EXACT_REBASE pre-RoPE keys (bf16); with the fp8 store
 * (RKV_KV_E4M3) byte planes of key codes and value codes of the same shape
 * and a (key, value) pair of float scales per row.  Stream s owns
 * ceil(C_s / page_size) pages, C_s = W_s + window_slack the capacity of its
 * ring; token j lives in ring slot j mod C_s, so eviction moves no data.
 * Within a row of d 16-bit elements the 16-byte chunk c sits at chunk
 * position c ^ (row offset in the page & 7), which makes a page copied
 * verbatim into shared memory bank-conflict-free for 8x8 matrix loads.
 * rkv_create zeroes the pool.
 */
#ifndef RKV_H_
#define RKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RKV_API __attribute__((visibility("default")))
#else
#define RKV_API
#endif

typedef uint16_t rkv_bf16; /* bfloat16 bits */

typedef enum {
  RKV_OK = 0,
  RKV_ERR_INVALID_ARG = -1,  /* null pointer, id out of range, duplicate id, misaligned buffer */
  RKV_ERR_CONFIG = -2,       /* configuration or clock not supported / inconsistent */
  RKV_ERR_CUDA = -3,         /* a CUDA runtime call failed (message has the CUDA error) */
  RKV_ERR_CAPACITY = -4,     /* a caller buffer is smaller than rkv_required_bytes says */
  RKV_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up */
  RKV_ERR_STATE = -6,        /* call out of order (see "Per-step order" above) */
  RKV_ERR_DEVICE_BOUNDS = -7, /* a kernel found an index outside its table */
  RKV_ERR_DEVICE_RANGE = -8   /* a rotated key did not fit fp16 (|k| >= 65520), or, in the fp8
                               * store, a value row reached |v| >= 61440 (read back in fp16) */
} rkv_status;

typedef enum {
  RKV_SCHEME_OFFSET_ONLY = 0,  /* K rotated once at P0 + j; kv_pos_offset bookkeeping only */
  RKV_SCHEME_EXACT_REBASE = 1, /* K kept at window-relative positions, re-based on every roll */
  RKV_SCHEME_EXACT_ON_READ = 2 /* the same exact positions and re-base bookkeeping, but the re-base is
                                * applied as attention reads: a key is stored once, rotated by its
                                * ring slot index j mod C (C = W + window_slack; positions stay below C
                                * however long the stream runs), and the query is rotated by its offset from the ring
                                * lap of each key, so no stored key is ever re-rotated (re-base moves
                                * no bytes) */
} rkv_scheme;

/* How the pool stores keys and values. */
typedef enum {
  RKV_KV_F16 = 0,  /* rotated keys as fp16, values as the bf16 given (the default) */
  RKV_KV_E4M3 = 1  /* keys (rotated) and values as fp8 e4m3 (round to nearest even), each row of d
                    * elements (one token, one kv head) with its own power-of-two scale 2^e, e the
                    * smallest for which max|x| / 2^e <= 448; half the bytes per token, read back
                    * exactly as code * 2^e.  Offset-only and the re-base applied on read only
                    * (a materialised re-base would round every retained key again each roll), and
                    * (n_q_heads / n_kv_heads) * q_per_step <= 8.  No page prescribes it: an
                    * optional store for more streams per GPU at lower precision. */
} rkv_kv_format;

/* Shape and policy of one handle.  All layers share it. */
typedef struct {
  int32_t n_layers;        /* L >= 1 */
  int32_t n_streams;       /* S, 1 .. RKV_MAX_STREAMS */
  int32_t n_q_heads;       /* Hq, multiple of n_kv_heads; Hq/Hkv * q_per_step <= 16 */
  int32_t n_kv_heads;      /* Hkv >= 1; q head h reads kv head h / (Hq/Hkv) */
  int32_t head_dim;        /* d: 64 or 128; RoPE pairs (x_i, x_{i+d/2}) */
  int32_t q_per_step;      /* Q: 1 (decoder) .. 8; Q > 1 is causal inside the step */
  int32_t page_size;       /* ring slots per page: 16, 32, 64 or 128 */
  int32_t scheme;          /* rkv_scheme */
  int32_t rebase_interval; /* exact scheme: re-base once this many tokens left (>= 1) */
  int32_t window_slack;    /* ring capacity beyond the window, >= 0: a stream keeps up to C_s =
                            * W_s + window_slack tokens and, at the step that would exceed C_s,
                            * evicts down to the last W_s in one batch (the oldest batch leaves
                            * together); 0 evicts exactly enough on every step (a plain sliding
                            * window of W_s) */
  int32_t kv_format;       /* rkv_kv_format; 0 (zero-initialised configs) is the fp16 store */
  int32_t reserved;        /* must be 0 */
  double rope_theta;       /* RoPE base theta > 1 (1e6 for the Qwen2.5 decoder) */
  double softmax_scale;    /* score scale; 0 selects 1/sqrt(head_dim) */
} rkv_config;

#define RKV_MAX_STREAMS 1024
#define RKV_MAX_WINDOW (1 << 20)
#define RKV_STATE_FIELDS 8

/* Clock arithmetic of the audio front end (Edge0/Audio8-ASR-Infinite README,
 * "Optimized operation points"; explainer "三档音频时钟", "可配置转写延迟"). */
typedef struct {
  int32_t clock_ms;          /* 20 ms tower frame x frame_len */
  int32_t window;            /* clock steps in the 30 s native context, rounded up */
  int32_t num_delay_tokens;  /* target_delay_ms / clock_ms */
  int32_t left_pad_tokens;   /* streaming_n_left_pad_tokens: 18 / 12 / 9 */
  int32_t samples_per_token; /* 16 kHz samples per clock step */
  int32_t post_trained;      /* 1 if (clock, delay) is in the post-trained table */
  double decisions_per_s;    /* 1000 / clock_ms */
} rkv_clock;

typedef struct rkv_handle rkv_handle;

/* Validate frame_len (4, 6 or 8) and target_delay_ms (a positive multiple of
 * the clock) and fill *out.  Host only.  RKV_ERR_CONFIG if invalid,
 * RKV_ERR_INVALID_ARG if out is NULL. */
RKV_API int rkv_clock_resolve(int32_t frame_len, int32_t target_delay_ms, rkv_clock* out);

/* Bytes of the two caller-owned device buffers a handle needs.  `window` is a
 * host array [n_streams] of per-stream windows W_s (q_per_step <= W_s <=
 * RKV_MAX_WINDOW).  The sizes depend only on the config and the windows, not
 * on how long the streams run: memory is constant (explainer 第 1 步).
 * Host only. */
RKV_API int rkv_required_bytes(const rkv_config* cfg, const int32_t* window,
                       size_t* pool_bytes, size_t* state_bytes);

/* Create a handle.
 *   window       host [S] int32: window W_s of each stream
 *   start_offset host [S] int64: logical position P0_s of each stream's first
 *                token, 0 <= P0_s < 2^52
 *   pool_dev     device buffer >= pool_bytes, 256-byte aligned: the K/V pages
 *   state_dev    device buffer >= state_bytes, 256-byte aligned: stream state,
 *                page tables, RoPE tables, status word
 * Initialises state_dev on `stream` and waits for it (synchronous).  Streams
 * start empty (n = 0).  The handle keeps the two pointers; the caller keeps
 * the buffers alive until rkv_destroy. */
RKV_API int rkv_create(const rkv_config* cfg, const int32_t* window, const int64_t* start_offset,
               void* pool_dev, size_t pool_bytes, void* state_dev, size_t state_bytes,
               void* stream, rkv_handle** out);

/* Open a step for the streams in active_ids (host [n_active], distinct ids in
 * [0, S), 1 <= n_active <= S).  On the device, for each active stream:
 * n += Q; len = min(n, W) (with window_slack > 0: len grows to C = W +
 * window_slack, then drops back to W in one batch); evicted = n - len;
 * kv_pos_offset = P0 + evicted; head_slot = evicted mod C; in the exact
 * schemes, if evicted - rope_base >=
 * rebase_interval, the step re-bases by delta = evicted - rope_base and
 * rope_base = evicted.  Then cos/sin of the new tokens' RoPE positions are
 * computed once for all layers (fp64 with error-free range reduction).
 * The id list travels in the kernel's parameters, so a captured graph
 * replays the same active set. */
RKV_API int rkv_begin_step(rkv_handle* h, const int32_t* active_ids, int32_t n_active, void* stream);

/* RoPE + append for one layer (explainer 第 2 步; voxtral.c article §二:
 * RoPE is baked into K at write time).
 *   k  device [A][Q][Hkv][d] bf16, pre-RoPE keys of the new tokens (A =
 *      n_active, rows in active_ids order)
 *   v  device [A][Q][Hkv][d] bf16
 * Writes the key rotated to its position (logical P0 + j; j - rope_base in
 * RKV_SCHEME_EXACT_REBASE; its ring slot j mod C in RKV_SCHEME_EXACT_ON_READ)
 * into ring slot (token mod C) of each stream, stored as fp16 (round to
 * nearest even; eleven significant bits, so a stored key adds ~2e-4 to a
 * unit-scale score, where bf16 would add ~1.6e-3), and v as given (bf16),
 * plus the pre-RoPE k in RKV_SCHEME_EXACT_REBASE.  With the fp8 store the
 * rotated key and the value are written as e4m3 codes with their rows'
 * scales (rkv_kv_format).  A rotated key of magnitude >= 65520 is reported
 * as RKV_ERR_DEVICE_RANGE by rkv_sync_status.  Once per layer per step. */
RKV_API int rkv_append_rope(rkv_handle* h, int32_t layer, const rkv_bf16* k, const rkv_bf16* v,
                            void* stream);

/* Exact re-base for one layer (explainer 第 2 步): every retained key of a
 * stream whose step re-bases is rotated by R(-delta), which brings the
 * stored positions back to j - rope_base inside the window.  The rotation is
 * applied to the key's pre-RoPE copy with the composite angle, so a stored
 * key carries one fp16 rounding however many times it was re-based.  Exact
 * schemes only (RKV_ERR_STATE otherwise); must be called once per layer per
 * step, before rkv_decode_attn of that layer (a no-op on the device for
 * streams that do not re-base this step).  In RKV_SCHEME_EXACT_ON_READ it
 * enqueues nothing: rkv_decode_attn rotates the query by each key's offset
 * from its ring lap instead, which gives every score the same position
 * difference. */
RKV_API int rkv_rebase(rkv_handle* h, int32_t layer, void* stream);

/* Windowed GQA attention for one layer (explainer 第 3 步), split-K over the
 * window with a log-sum-exp merge of the splits in distributed shared memory
 * (no scratch memory).
 *   q     device [A][Q][Hq][d] bf16, pre-RoPE queries of the new tokens;
 *         rotated inside the kernel in fp32 to the positions the scheme's
 *         stored keys are measured from (never rounded back to 16 bits), not
 *         modified
 *   out   device [A][Q][Hq][d] bf16: softmax(q k^T * scale) v over the window
 *   lse   device [A][Q][Hq] fp32: natural log of sum exp(scaled scores); may
 *         be NULL
 * Query token n_old + i of a stream attends its tokens j with
 * max(0, n_new - W) <= j <= n_old + i.  q may be written by the kernel
 * launched immediately before this call on `stream`: the kernel reads q only
 * after that kernel has completed (programmatic dependent launch lets this
 * kernel start early, but it waits for its predecessor before touching q,
 * the pages or out). */
RKV_API int rkv_decode_attn(rkv_handle* h, int32_t layer, const rkv_bf16* q, rkv_bf16* out,
                            float* lse, void* stream);

/* rkv_append_rope and rkv_decode_attn of one layer in one launch: a warp of
 * each attention CTA writes the step's new keys (rotated as rkv_append_rope
 * rotates them) and values into the pool while the CTA streams the window's
 * older ring stages; the stages that hold new tokens are streamed last,
 * once those rows are written, and attended over in the same pass.
 * Arguments as the two calls take them (q [A][Q][Hq][d], k and v
 * [A][Q][Hkv][d], out, lse); results as rkv_append_rope followed by
 * rkv_decode_attn.  In the exact schemes rkv_rebase of the layer must come
 * first.  Counts as the layer's append (RKV_ERR_STATE if the layer's tokens
 * were appended already).  q, k and v may be written by the kernel launched
 * just before. */
RKV_API int rkv_append_decode_attn(rkv_handle* h, int32_t layer, const rkv_bf16* q, const rkv_bf16* k,
                                   const rkv_bf16* v, rkv_bf16* out, float* lse, void* stream);

/* rkv_decode_attn for layers layer0 .. layer0 + n_layers - 1 of the open
 * step in one launch (the layers' queries must all be known, as in
 * rkv_step).  q and out are [n_layers][A][Q][Hq][d], lse [n_layers][A][Q][Hq]
 * (may be NULL); every layer in the range must have had rkv_append_rope (and
 * rkv_rebase in the exact schemes) in this step, else RKV_ERR_STATE. */
RKV_API int rkv_decode_attn_layers(rkv_handle* h, int32_t layer0, int32_t n_layers, const rkv_bf16* q,
                                   rkv_bf16* out, float* lse, void* stream);

/* The whole step for all layers: rkv_begin_step, then rkv_rebase (exact
 * re-base scheme), rkv_append_rope and rkv_decode_attn for every layer, each
 * as one launch over all layers (the layers' inputs are all given, so their
 * work is independent).  Same results as the per-layer calls.
 *   q     device [L][A][Q][Hq][d], k, v [L][A][Q][Hkv][d], all pre-RoPE bf16
 *   out   device [L][A][Q][Hq][d], lse [L][A][Q][Hq] (may be NULL) */
RKV_API int rkv_step(rkv_handle* h, const int32_t* active_ids, int32_t n_active, const rkv_bf16* q,
             const rkv_bf16* k, const rkv_bf16* v, rkv_bf16* out, float* lse, void* stream);

/* Decode attention that allocates nothing and needs no scratch from the
 * caller.  No page describes this call: it exists for callers that may not
 * allocate device memory where they run attention, such as a real-time audio
 * callback that cannot risk an allocator call synchronising the device
 * inside its 80 ms clock step, or a plug-in inside a serving engine whose
 * caching allocator already holds the free HBM.
 *
 * Same arguments and call-order rules as rkv_decode_attn.  When the windows
 * are split over several CTAs, the per-split partial results go to a fixed
 * array compiled into the library (8 MiB per device, held by every GPU that
 * loads the library until the process exits) and a second kernel merges
 * them; rkv_decode_attn merges its splits in distributed shared memory
 * instead and may split differently, so the two agree to fp32 rounding of
 * the merge, not bit for bit.  A call whose windows are not split uses no
 * part of the array.  A call that needs more than 8 MiB of partials
 * ((2 + head_dim) floats per active stream, query row and split) returns
 * RKV_ERR_CAPACITY with the sizes in the message.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current, so make that first call before any stream capture.
 * Every call on a device shares the one array, and the array keeps the last
 * call's contents; nothing in it needs to start at zero, because every
 * partial the merge reads is written earlier in the same call.  Calls that
 * overlap on the GPU (other streams, other handles, other threads) race on
 * the array: the caller must serialise them.  No cudaMalloc, cudaFree or
 * allocating library routine is called. */
RKV_API int rkv_decode_attn_static(rkv_handle* h, int32_t layer, const rkv_bf16* q, rkv_bf16* out,
                                   float* lse, void* stream);

/* Empty one stream so that its next step starts a new history: n = len =
 * evicted = rope_base = 0, kv_pos_offset = P0 = start_offset (0 <= P0 <
 * 2^52); its window and pages are kept.  This is voxtral.c's continuous-mode
 * restart (voxtral.c article §四: a hard reset of the decoder cache while the
 * audio keeps flowing), and the way a serving loop hands a stream slot to a
 * new audio stream.  Enqueued on `stream` (graph-capturable), so it takes
 * effect for the next rkv_begin_step on that stream; kernels of an open step
 * use the step's own descriptors and are not affected.  The stale keys and
 * values left in the pages are never read: a slot is attended only once the
 * new history has written it. */
RKV_API int rkv_reset_stream(rkv_handle* h, int32_t stream_id, int64_t start_offset, void* stream);

/* rkv_reset_stream for a list of stream slots held in device memory, one
 * launch for all of them: a serving loop whose streams leave and join
 * between steps writes the list (and the new start offsets) on the device,
 * so a captured graph of the step takes a new list on every replay.
 *   ids_dev  device [n] int32: stream ids, distinct; a negative id is skipped
 *   p0_dev   device [n] int64: their new start offsets
 * An entry with an id >= n_streams or a start offset outside [0, 2^52) is
 * skipped and reported as RKV_ERR_DEVICE_BOUNDS by rkv_sync_status.  Takes
 * effect for the next rkv_begin_step, as rkv_reset_stream does. */
RKV_API int rkv_reset_streams(rkv_handle* h, const int32_t* ids_dev, const int64_t* p0_dev, int32_t n,
                              void* stream);

/* Snapshot of one stream for resume: its ring state and the contents of its
 * pages in every layer (no page describes this; it is how a 24/7 serving
 * loop moves or checkpoints a live stream).  rkv_stream_snapshot_bytes gives
 * the size: a 128-byte header (configuration, window, scheme), the
 * RKV_STATE_FIELDS int64 state, then the stream's pages, region by region and
 * layer by layer.  rkv_save_stream writes it to `dst`; rkv_load_stream
 * restores it into a stream slot of a handle with the same configuration and
 * the same window for that slot (else RKV_ERR_CONFIG), after which the stream
 * continues exactly where it was saved.  dst / src may be host or device
 * memory.  Both wait for `stream` before returning (not graph-capturable) and
 * return RKV_ERR_STATE while a step is in progress (some layer of the open
 * step lacks rkv_append_rope or rkv_rebase). */
RKV_API int rkv_stream_snapshot_bytes(const rkv_handle* h, int32_t stream_id, size_t* bytes);
RKV_API int rkv_save_stream(rkv_handle* h, int32_t stream_id, void* dst, size_t bytes, void* stream);
RKV_API int rkv_load_stream(rkv_handle* h, int32_t stream_id, const void* src, size_t bytes, void* stream);

/* Check a stream state record (RKV_STATE_FIELDS int64, the order of
 * rkv_get_stream_state) against the rules every step keeps under `cfg`:
 * W_s in [q_per_step, RKV_MAX_WINDOW], 0 <= P0 < 2^52, n >= 0 a multiple of
 * q_per_step with P0 + n < 2^52, len = min(n, W) (with window_slack > 0:
 * the batched rule of rkv_begin_step), evicted = n - len,
 * kv_pos_offset = P0 + evicted, head_slot = evicted mod C, and rope_base in
 * (evicted - rebase_interval, evicted] for the exact schemes, 0 otherwise.
 * rkv_load_stream applies it to a snapshot before restoring it.  Host only:
 * RKV_OK, else RKV_ERR_CONFIG with the broken rule in rkv_last_error(NULL). */
RKV_API int rkv_check_stream_state(const rkv_config* cfg, const int64_t* state);

/* Copy one stream's device state to host `out` (RKV_STATE_FIELDS int64):
 * n, len, evicted, kv_pos_offset, rope_base, head_slot, W, P0.  Waits for
 * `stream`. */
RKV_API int rkv_get_stream_state(rkv_handle* h, int32_t stream_id, int64_t* out, void* stream);

/* Wait for `stream`, read and clear the device status word: RKV_OK,
 * RKV_ERR_DEVICE_BOUNDS, RKV_ERR_DEVICE_RANGE or RKV_ERR_TIMEOUT. */
RKV_API int rkv_sync_status(rkv_handle* h, void* stream);

/* Failure-detection test hook (no page describes it).  The attention
 * kernel's waits on its shared-memory stages are bounded: a wait gives up
 * after one second, records RKV_ERR_TIMEOUT in the status word, drains the
 * CTA's own copies in flight and returns, and later launches of the handle
 * skip their copies until rkv_sync_status has read the status.  This hook
 * lets a test drive that path without any fault: wait_ns shortens the limit
 * (1 us .. 1 s; 0 restores one second), and withhold_stage >= 0 makes each
 * attention CTA's producer skip the copy of its stage with that number
 * (counted from 0 along the CTA's walk), so the consumers' wait for it runs
 * out; -1 turns that off.  Affects launches enqueued after the call.  Host
 * only. */
RKV_API int rkv_set_wait_test(rkv_handle* h, int32_t withhold_stage, uint64_t wait_ns);

/* Message of the last failure on this handle (NULL: of the calling thread's
 * last failure without a handle).  Valid until the next call. */
RKV_API const char* rkv_last_error(const rkv_handle* h);

/* Free the host-side handle.  Device buffers stay with the caller. */
RKV_API int rkv_destroy(rkv_handle* h);

/* ---- building blocks, exposed for tests and benchmarks ---------------- */

/* cos/sin of RoPE angles: cs_dev[n][d/2][2] fp32 = (cos, sin)(pos[i] * omega_j)
 * with omega_j = theta^(-2j/d) rounded to fp64 on the host, the product
 * split exactly (FMA) and reduced modulo 2*pi with a three-part 2*pi.
 *   pos_dev device [n] int64, |pos| < 2^52. */
RKV_API int rkv_rope_cossin(const int64_t* pos_dev, int32_t n, int32_t head_dim, double theta,
                    float* cs_dev, void* stream);

/* Counter-based N(0,1)-like bf16 inputs (SplitMix64, Steele, Lea and Flood
 * 2014; twelve 12-bit fields summed, Irwin-Hall), times an fp32 scale,
 * rounded to nearest even.  out_dev[t][e] for token token0 + t, element e <
 * width of one token's [heads][head_dim] tensor. */
RKV_API int rkv_gen_tokens(uint64_t seed, uint32_t tag, int32_t stream_id, int32_t layer, int64_t token0,
                   int32_t n_tokens, int32_t width, float scale, rkv_bf16* out_dev, void* stream);

/* The same draws for the open step's new tokens of one layer, in the layout
 * rkv_append_rope takes: q [A][Q][Hq][d] (tag 1), k and v [A][Q][Hkv][d]
 * (tags 2, 3); token index = the stream's own token count. */
RKV_API int rkv_gen_step_inputs(rkv_handle* h, uint64_t seed, int32_t layer, float scale, rkv_bf16* q,
                        rkv_bf16* k, rkv_bf16* v, void* stream);

/* The same draws for the next step of the listed streams, every layer, in
 * the layout rkv_step takes: q [L][A][Q][Hq][d], k and v [L][A][Q][Hkv][d]
 * (tags 1, 2, 3; rows in active_ids order).  The token index of a stream's
 * row t is its device token count n (as it stands when the kernel runs) plus
 * t, i.e. the tokens the next rkv_begin_step or rkv_step will append. */
RKV_API int rkv_gen_next_inputs(rkv_handle* h, uint64_t seed, const int32_t* active_ids, int32_t n_active,
                                float scale, rkv_bf16* q, rkv_bf16* k, rkv_bf16* v, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H_ */
