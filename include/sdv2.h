/*
 * sdv2.h -- C ABI of the GB300 (sm_103a) streaming causal-video chunk-attention library.
 *
 * One call sequence per DiT layer and denoise step of a streamed chunk:
 *   sdv2_rope_append_kv   Causal-RoPE on the chunk's q and k, then k_rot and v written into the
 *                         layer's fixed-size KV cache (pinned sink + rolling window of frames).
 *   sdv2_chunk_attention  the chunk's queries attend to every valid cache row: sink + window,
 *                         the chunk itself included.
 * and, once per batch of input frames,
 *   sdv2_motion_l2        squared L2 distance of adjacent video frames (motion magnitude).
 *
 * Conventions shared by every entry point:
 *  - All device memory is allocated and owned by the caller.  The library never allocates
 *    device memory and keeps no per-call state on the host.  Host arrays passed in are read
 *    before the call returns.
 *  - Work is enqueued asynchronously on the caller's CUDA stream (`stream`, a cudaStream_t
 *    passed as void*; NULL = the legacy default stream).  No entry point synchronizes, except
 *    sdv2_workspace_init, sdv2_check_device_error and sdv2_noalloc_check_device_error, which
 *    say so.
 *  - Arguments are validated on the host before anything is launched; a rejected call
 *    launches nothing and returns SDV2_ERR_INVALID_ARG or SDV2_ERR_UNSUPPORTED.  A failed
 *    launch returns SDV2_ERR_CUDA.  sdv2_last_error() gives a one-line reason (per thread).
 *  - Device pointers must be 16-byte aligned.
 *  - bf16 means bfloat16: the upper 16 bits of the IEEE binary32 layout (sign, 8 exponent
 *    bits, 7 mantissa bits), stored as uint16.  Every bf16 the library writes is rounded to
 *    nearest, ties to even.
 *
 * Notation (stream configuration): B streams, H heads, D = head_dim = 128, HW = grid_h*grid_w
 * tokens per latent frame, F frames per chunk, Nq = F*HW queries per chunk, F_s sink frames,
 * W window frames (the window includes the current chunk), R refresh period in chunks.
 */
#ifndef SDV2_H
#define SDV2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDV2_OK = 0,
    SDV2_ERR_INVALID_ARG = 1,   /* a pointer, size or configuration field is invalid */
    SDV2_ERR_UNSUPPORTED = 2,   /* valid but not built for (e.g. head_dim != 128, not sm_103) */
    SDV2_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
    SDV2_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up (see check_device_error) */
} sdv2_status;

/*
 * Stream configuration, shared by all streams of a batch and by all layers.
 *
 * 3D RoPE ("Accelerating Video Generation Inference with Sequential-Parallel 3D Positional
 * Encoding Using a Global Time Index", technical summary 2(나) and 2(다)): the head dims are
 * split into consecutive segments of rope_t, rope_h and rope_w dims (t first); inside a
 * segment of d dims, pair (2j, 2j+1) turns by pos * rope_base^(-2j/d), where pos is the time
 * index t, the grid row h or the grid column w of the token.  rope_t + rope_h + rope_w must
 * equal head_dim and each must be even.
 *
 * Time index (Causal-RoPE with a global time index; RoPE refresh of "StreamDiffusionV2",
 * review page section 三): token n of chunk c of stream b lies in frame i = n / HW of the
 * chunk; its time index is t = start_frame[b] + F*(c mod R) + i, or start_frame[b] + F*c + i
 * when refresh_chunks R = 0.  Its grid position is h = (n mod HW) / grid_w, w = n mod grid_w.
 *
 * Cache (sink token + rolling KV cache, same review page section 三): frames are numbered per
 * stream, f = c*F + i.  Frame f lives in slot f if f < F_s, else in slot F_s + (f - F_s) mod W.
 * After chunk c has been appended the valid slots are exactly the prefix
 * [0, n_vis) with n = (c+1)*F and n_vis = min(F_s, n) + min(W, max(0, n - F_s)).
 */
typedef struct {
    int32_t batch;             /* B >= 1 streams                                               */
    int32_t heads;             /* H >= 1                                                       */
    int32_t head_dim;          /* D; only 128 is built                                         */
    int32_t rope_t, rope_h, rope_w;
    double rope_base;          /* > 1, e.g. 10000                                              */
    int32_t grid_h, grid_w;    /* latent tokens per frame = grid_h * grid_w                    */
    int32_t chunk_frames;      /* F >= 1                                                       */
    int32_t sink_frames;       /* F_s >= 0                                                     */
    int32_t window_frames;     /* W >= F                                                       */
    int32_t refresh_chunks;    /* R >= 0 (0 = the offset never resets)                         */
    int64_t qkv_token_stride;  /* elements between consecutive tokens of q, k, v; 0 = H*D      */
} sdv2_stream_cfg;

/* One cache slot's metadata: which frame it holds and with which RoPE time index its keys
 * were rotated.  frame_id = -1 marks an empty slot. */
typedef struct {
    int64_t frame_id;
    int64_t tpos;
} sdv2_slot_meta;

/* ---- sizes ------------------------------------------------------------------------------ */

/* Bytes of the workspace: a header with the device error word, the fp32 cos/sin tables of the
 * h and w axes (position-major for the append kernel and a pair-major copy for the fused
 * projection), and the attention's key-split scratch (per-item arrival counters, per-row
 * running max and sum, per-row unnormalised fp32 outputs for up to 4 key splits of every
 * (stream, head, 256 query rows) item).  The workspace belongs to one configuration; it may
 * be shared by all layers, but calls that use it must not overlap on the GPU (use one
 * workspace per concurrently running stream). */
size_t sdv2_workspace_bytes(const sdv2_stream_cfg* cfg);

/* Bytes of ONE of the two cache tensors (k or v) of one layer:
 * [B][H][(F_s+W)*HW][D] bf16 = B*H*(F_s+W)*HW*D*2. */
size_t sdv2_cache_bytes(const sdv2_stream_cfg* cfg);

/* Bytes of one layer's slot metadata: [B][F_s+W] sdv2_slot_meta. */
size_t sdv2_meta_bytes(const sdv2_stream_cfg* cfg);

/* Valid KV rows n_vis*HW that chunk `chunk_index` attends to (formula in the struct comment);
 * -1 on an invalid configuration or a negative chunk index. */
int64_t sdv2_visible_tokens(const sdv2_stream_cfg* cfg, int64_t chunk_index);

/* ---- set-up ----------------------------------------------------------------------------- */

/* Fill the workspace: zero it, then write the header and the fp32 cos/sin tables of the h and
 * w axes in both layouts (angles and cos/sin in fp64 on the host, rounded once to fp32).  Enqueues a memset
 * and copies on `stream` and synchronizes it before returning.
 * ws: device, sdv2_workspace_bytes(cfg) bytes. */
sdv2_status sdv2_workspace_init(const sdv2_stream_cfg* cfg, void* ws, void* stream);

/* Make one layer's cache empty: every slot's frame_id = -1, tpos = 0, and k and v zero.
 * k_cache, v_cache: device, sdv2_cache_bytes(cfg) each; meta: device, sdv2_meta_bytes(cfg). */
sdv2_status sdv2_cache_reset(const sdv2_stream_cfg* cfg, void* k_cache, void* v_cache, void* meta,
                             void* stream);

/* ---- the hot path ----------------------------------------------------------------------- */

/*
 * Causal-RoPE + cache append for chunk chunk_index[b] of every stream b.
 *
 * start_frame, chunk_index: HOST arrays of B int64, start_frame in [0, 2^50] and chunk_index in
 *   [0, 2^40]: the global start frame S_b of stream b and the chunk being appended.  Positions are derived as in the struct comment.
 * q, k, v: device bf16, token-major [B][Nq][H][D], with qkv_token_stride elements between
 *   consecutive tokens (so a packed [token][3][H][D] projection output can be passed as three
 *   pointers) and Nq*stride elements between streams.
 * q_rot: device bf16, [B][H][Nq][D] (head-major, the layout sdv2_chunk_attention reads).
 * k_cache, v_cache: device bf16 [B][H][(F_s+W)*HW][D].  The F frames of the chunk are written
 *   to their slots: k rotated, v copied.  Rows of other slots are not touched.
 * meta: device [B][F_s+W] sdv2_slot_meta; the chunk's slots get frame_id = c*F + i and tpos.
 * ws: device workspace from sdv2_workspace_init for the same configuration.
 *
 * Rounding (bit-exact contract): for each pair (x, y) with table values c, s (fp32),
 *   x' = bf16_rne(fmaf(x, c, -(y*s))),  y' = bf16_rne(fmaf(x, s, y*c)),
 * where y*s and y*c are single fp32 products.
 * Calling it again for the same chunk (the next denoise step) overwrites the same slots.
 * Limits: B*F*rope_t/2 <= 1536 (the time-axis table travels in the launch parameters).
 */
sdv2_status sdv2_rope_append_kv(const sdv2_stream_cfg* cfg, const int64_t* start_frame,
                                const int64_t* chunk_index, const void* q, const void* k,
                                const void* v, void* q_rot, void* k_cache, void* v_cache,
                                void* meta, void* ws, void* stream);

/*
 * Fused QKV projection + Causal-RoPE + cache append ("Accelerating Video Generation Inference
 * with Sequential-Parallel 3D Positional Encoding Using a Global Time Index", technical summary
 * 2(다): the QKV projection and the Causal-RoPE computation fused into one kernel).
 *
 * For every token of chunk chunk_index[b] of every stream b:
 *   [q | k | v] = W_qkv x + bias   (features: q head h dim d at h*D + d, then k, then v)
 * then q and k are rotated with the token's 3D RoPE (positions exactly as sdv2_rope_append_kv)
 * and q_rot, the cache rows of the chunk's frames and their slot metadata are written as by
 * sdv2_rope_append_kv.
 * x: device bf16 [B][Nq][C] with C = H*D, tokens x_token_stride elements apart (0 = C;
 *   a multiple of 8); streams Nq*x_token_stride apart.
 * w_qkv: device bf16 [3*H*D][C] (row = output feature); bias: device fp32 [3*H*D] or NULL.
 * q_rot, k_cache, v_cache, meta, ws: as sdv2_rope_append_kv.
 * Numerics: bf16 products with fp32 accumulation (tcgen05 tensor cores), + bias in fp32, q/k
 * pairs rotated in fp32 as (fmaf(x, c, -(y*s)), fmaf(x, s, y*c)), one bf16 RNE per output.
 * (It differs from projecting to bf16 first and calling sdv2_rope_append_kv by that one
 * rounding.)  Limits: those of sdv2_rope_append_kv.
 */
sdv2_status sdv2_qkv_rope_append(const sdv2_stream_cfg* cfg, const int64_t* start_frame,
                                 const int64_t* chunk_index, const void* x, int64_t x_token_stride,
                                 const void* w_qkv, const float* bias, void* q_rot, void* k_cache,
                                 void* v_cache, void* meta, void* ws, void* stream);

/*
 * Chunk attention: out[b][n][h][:] = sum_j softmax_j(scale * <q_rot[b][h][n], k_j>) v_j over
 * the valid cache rows j < sdv2_visible_tokens(cfg, chunk_index[b]) of stream b, head h.
 * There is no mask inside the valid rows: the chunk attends to itself in full and to every
 * retained earlier frame (chunk-causal attention of a Self-Forcing-style streaming DiT).
 *
 * chunk_index: HOST array of B int64 in [0, 2^40].
 * q_rot: device bf16 [B][H][Nq][D]; k_cache, v_cache: device bf16 [B][H][(F_s+W)*HW][D].
 * scale: softmax scale; <= 0 selects 1/sqrt(D).
 * out: device bf16 [B][Nq][H][D] (token-major, ready for the output projection).
 * lse: device fp32 [B][H][Nq] natural-log log-sum-exp of the scaled scores, or NULL.
 * ws: device workspace (error word of the bounded waits; key-split scratch).
 * Numerics: bf16 tensor-core products with fp32 accumulation, online softmax in fp32.
 * Work split: items of (stream, head, 256 query rows); the first items run whole, one CTA
 * each, in whole waves of the GPU's SMs, and the key range of every later item is cut into 1-4
 * splits (sdv2_debug_kv_schedule gives the choice); the split that finishes its keys last
 * merges the others' partial rows with its own (log-sum-exp weights, splits summed in index
 * order, so the output does not depend on which split merges) and writes the output.  The
 * result is deterministic: the same inputs give the same bits on every call.
 * Limits: B <= 16; B * H * ceil(Nq/256) * splits < 2^31; the device must be sm_103 (tcgen05
 * tensor cores).
 */
sdv2_status sdv2_chunk_attention(const sdv2_stream_cfg* cfg, const int64_t* chunk_index,
                                 const void* q_rot, const void* k_cache, const void* v_cache,
                                 float scale, void* out, float* lse, void* ws, void* stream);

/*
 * Chunk attention for callers that cannot allocate device memory.  (The pages describe no
 * counterpart: this is an interface for deployment, not a step of the method.)
 *
 * Some callers cannot call cudaMalloc at all: code running inside a memory pool it does not
 * own, plugin hosts that forbid allocation after start-up, real-time loops that must never
 * reach the allocator (an allocation can synchronize the device and stall a frame).  They
 * cannot provide the workspace sdv2_chunk_attention needs.  This entry point computes the same
 * attention with the same arguments minus `ws`; its scratch (device error word, key-split
 * arrival counters, per-row partial results of the key splits) lives in a 16 MiB file-scope
 * __device__ array inside the library, which every GPU that loads the library holds until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current) and keeps it; make that first call before any stream capture.
 * - Every call on a device shares the array, which keeps the previous call's contents; each
 *   call clears the key-split counters on `stream` (a memset) before its kernel.  Calls whose
 *   work overlaps on the GPU (other streams, graph branches) race on the array: do not
 *   overlap them.
 * - Key splits are chosen as for sdv2_chunk_attention (sdv2_debug_set_kv_splits applies here
 *   too), then reduced until their partial rows fit in the array (results stay within the same
 *   tolerance; speed may differ).  sdv2_last_kv_splits reports the count used.
 * - Sizes beyond the array's reach are rejected with SDV2_ERR_UNSUPPORTED before anything is
 *   enqueued: batch * heads * ceil(Nq / 256) must be <= 16384.
 * - Bounded device waits use the limit of sdv2_set_wait_timeout_ns.  A wait that gives up
 *   leaves this call's outputs undefined and sets the array's error word, which later calls
 *   do not clear: sdv2_noalloc_check_device_error reports it (and clears it).
 * Other arguments, layouts and numerics: as sdv2_chunk_attention.
 */
sdv2_status sdv2_chunk_attention_noalloc(const sdv2_stream_cfg* cfg, const int64_t* chunk_index,
                                         const void* q_rot, const void* k_cache,
                                         const void* v_cache, float scale, void* out, float* lse,
                                         void* stream);

/*
 * Error check of sdv2_chunk_attention_noalloc on the current device, allocation-free as well
 * (the pages have no counterpart).  Synchronizes `stream`, reads the static array's error word
 * with one cudaMemcpyAsync and returns SDV2_ERR_TIMEOUT if a bounded device wait of an earlier
 * sdv2_chunk_attention_noalloc call gave up since the last check (that call's outputs are
 * undefined), SDV2_ERR_CUDA on a CUDA error, else SDV2_OK.  After a timeout it clears the
 * error word and the key-split counters, so the next call starts clean.  Calls on the device
 * that are still running on other streams must be finished first (they share the array).
 */
sdv2_status sdv2_noalloc_check_device_error(void* stream);

/*
 * Motion magnitude of adjacent frames ("StreamDiffusionV2" review page, section 二 table and
 * section 三: L2 motion estimation between adjacent frames feeds the noise controller).
 *
 * frames: device uint8 [B][T+1][Hp][Wp][C], contiguous.
 * ssd: device uint64 [B][T]: ssd[b][t] = sum over pixels and channels of
 *   (frames[b][t+1] - frames[b][t])^2, exact.
 * m: device fp32 [B][T] or NULL: sqrt(ssd / (Hp*Wp*C)), the RMS pixel difference.
 * Requires T >= 1, B*T <= 65535 and Hp*Wp*C a multiple of 16.
 */
sdv2_status sdv2_motion_l2(const uint8_t* frames, int32_t B, int64_t T, int32_t Hp, int32_t Wp,
                           int32_t C, uint64_t* ssd, float* m, void* stream);

/* ---- refresh, sink update, noise controller ------------------------------------------- */

/*
 * RoPE refresh, second reading ("StreamDiffusionV2" review page, section 三: the positional
 * offset is reset periodically).  sdv2_rope_append_kv already restarts the time offset every R
 * chunks (t = S + F*(c mod R) + i); the keys kept in the window were rotated at the old,
 * larger positions.  This call turns them back by F*R on the time axis so that the distance
 * between the new chunk and every window frame stays what it was without the reset.
 *
 * For every stream b whose chunk_index[b] is a refresh chunk (R > 0, c > 0, c mod R == 0):
 * every WINDOW slot (slot >= F_s) holding a frame of an earlier chunk (0 <= frame_id < c*F)
 * has the time-axis pairs of its keys rotated by the angle -F*R*omega_j (same rounding as
 * sdv2_rope_append_kv, with position -F*R) and its tpos decreased by F*R.  Sink slots, values,
 * the h/w dims and streams not at a refresh chunk are untouched.  Call it once per layer at a
 * refresh chunk, BEFORE the chunk's first sdv2_rope_append_kv (not again for later denoise
 * steps of the same chunk).
 * k_cache: device [B][H][(F_s+W)*HW][D] bf16; meta: device [B][F_s+W]; chunk_index: host [B].
 * Limits: B <= 64.
 */
sdv2_status sdv2_rope_refresh_rerotate(const sdv2_stream_cfg* cfg, const int64_t* chunk_index,
                                       void* k_cache, void* meta, void* stream);

/*
 * Sink update ("StreamDiffusionV2: A Streaming System for Dynamic and Interactive Video
 * Generation", technical summary section 2, part A item 2: sink tokens follow recent visual
 * context).  Read here as: the sink is replaced by copies of the F_s most recently appended
 * frames.  For every stream b with update[b] != 0 (host int32 [B]), after chunk chunk_index[b]
 * has been appended (n = (c+1)*F frames), sink slot s (0 <= s < F_s) receives the k and v rows
 * and the metadata (frame_id, tpos) of frame n - F_s + s, which lives in the window.  Needs
 * n >= 2*F_s and W >= F_s.  The copies keep their rotation; the window keeps the originals.
 */
sdv2_status sdv2_sink_update(const sdv2_stream_cfg* cfg, const int64_t* chunk_index,
                             const int32_t* update, void* k_cache, void* v_cache, void* meta,
                             void* stream);

/* Motion-aware noise controller: a declared monotone map (the pages give no formula and
 * disagree on its direction: the StreamDiffusionV2 technical summary, section 2 part A item 3,
 * vs the review page, section 三). */
typedef struct {
    float motion_lo, motion_hi;  /* RMS motion (0..255 scale) mapped to the low / high end     */
    float rate_lo, rate_hi;      /* noise rates at the two ends (>= 0)                          */
    float ema;                   /* smoothing over frames, in [0, 1); 0 = none                  */
    int32_t more_noise_when_fast;/* 1: fast motion -> rate_hi (review page); 0: -> rate_lo      */
} sdv2_noise_ctl;

/*
 * rate[b][t] from m[b][t] (device fp32 [B][T], e.g. the RMS output of sdv2_motion_l2):
 *   u = clamp((m - motion_lo) / (motion_hi - motion_lo), 0, 1); if !more_noise_when_fast:
 *   u = 1 - u; r = fmaf(rate_hi - rate_lo, u, rate_lo);
 *   s = (first value of the stream) ? r : fmaf(ema, s - r, r);  rate[b][t] = s.
 * state: device fp32 [B] carried across calls (-1 = no history yet) or NULL (no carry-over).
 * fp32 throughout, one rounding per written operation (fmaf where written).
 */
sdv2_status sdv2_noise_from_motion(const sdv2_noise_ctl* ctl, const float* m, int32_t B, int64_t T,
                                   float* state, float* rate, void* stream);

/* ---- errors ----------------------------------------------------------------------------- */

/* Synchronizes `stream`, reads the workspace's device error word and returns SDV2_ERR_TIMEOUT
 * if a bounded device wait gave up since the last check (the outputs of the calls involved
 * are then undefined), SDV2_ERR_CUDA on a CUDA error, else SDV2_OK.  After an error it clears
 * the error word and the key-split counters, so the workspace is usable again. */
sdv2_status sdv2_check_device_error(void* ws, void* stream);

/* Upper bound of every bounded device-side wait, in nanoseconds (default 2e9).  Applies to
 * launches made after the call, from any thread. */
void sdv2_set_wait_timeout_ns(uint64_t ns);

/* Fault injection for tests of the bounded waits: when tile >= 0, the next
 * sdv2_chunk_attention launches skip the copy of KV tile `tile` (the consumers' waits then
 * run out, the kernel records SDV2_ERR_TIMEOUT and returns).  -1 turns it off. */
void sdv2_debug_drop_kv_tile(int64_t tile);

/* Key-range split count of later sdv2_chunk_attention calls: 0 = automatic (default),
 * 1..4 = forced (capped by the number of key tiles).  For tests and tuning. */
void sdv2_debug_set_kv_splits(int32_t splits);

/* Split count of the split items in this thread's most recent sdv2_chunk_attention call (1 if
 * no item was split). */
int32_t sdv2_last_kv_splits(void);

/* The automatic work schedule of sdv2_chunk_attention, for tests (host only, no GPU): for
 * `items` = B * H * ceil(Nq/256) (stream, head, 256 query rows) items whose key loops have at
 * least `min_tiles` 128-key tiles, on a GPU with `sms` SMs, returns the key-range split count of
 * the split items and sets *full_items to the number of items that run whole (the first ones,
 * in whole waves of `sms`); -1 on invalid arguments.  The schedule minimises the estimated
 * makespan: k whole waves of unsplit items, then the rest cut into s key ranges. */
int32_t sdv2_debug_kv_schedule(int64_t items, int32_t min_tiles, int32_t sms, int32_t* full_items);

const char* sdv2_status_string(sdv2_status s);
const char* sdv2_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* SDV2_H */
