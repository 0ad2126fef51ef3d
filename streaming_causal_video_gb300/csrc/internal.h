// Launch parameters and launchers shared by the library's translation units (not installed).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/sdv2.h"

namespace sdv2 {

// Bits of the device error word at the start of the workspace.
constexpr uint32_t kErrTimeout = 1u;   // a bounded mbarrier wait gave up

// ---- RoPE + cache append ----------------------------------------------------------------------

constexpr int kMaxChunkFrames = 64;     // B*F frames per append call
constexpr int kMaxTimePairs = 1536;     // B*F*(rope_t/2) fp32 cos/sin pairs per append call

// Where one frame of the chunk goes: its cache slot, its stream-relative number and its RoPE
// time index.  One entry per (stream b, frame i), index b*F + i.
struct FrameDesc {
    int64_t frame;
    int64_t tpos;
    int32_t slot;
    int32_t pad;
};

struct RopeAppendParams {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    uint16_t* q_rot;
    uint16_t* k_cache;
    uint16_t* v_cache;
    sdv2_slot_meta* meta;
    const float2* h_tab;      // [grid_h][rope_h/2] (cos, sin)
    const float2* w_tab;      // [grid_w][rope_w/2] (cos, sin)
    int64_t tok_stride;       // elements between tokens of q/k/v
    int32_t B, H, HW, grid_w, F, nslots, Nq;
    int32_t tp, hp, wp;       // rotation pairs per axis
    FrameDesc frames[kMaxChunkFrames];
    float2 tcs[kMaxTimePairs];  // [B*F][tp] (cos, sin) of the time axis
};

cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t s);

// ---- chunk attention --------------------------------------------------------------------------

constexpr int kMaxAttnStreams = 16;
constexpr int kAttnRowsPerCta = 256;     // two 128-row query tiles per CTA
constexpr int kMaxKvSplits = 4;          // key-range splits per (stream, head, query pair)

struct AttnParams {
    CUtensorMap qmap;                       // (D, Nq, B*H) over q_rot
    CUtensorMap kmap[kMaxAttnStreams];      // per stream: (D, valid rows, H) over k_cache
    CUtensorMap vmap[kMaxAttnStreams];      // per stream: (D, valid rows, H) over v_cache
    uint16_t* out;                          // [B][Nq][H][D] bf16
    float* lse;                             // [B][H][Nq] or null
    uint32_t* err;                          // device error word
    int32_t* counters;                      // [2][B*H*qpairs] split tickets, published splits (0 between calls)
    float* part_ml;                         // [split items*splits][256][2] running max (log2) and sum
    float* part_o;                          // [split items*splits][HD/4][256][4] unnormalised output
    int32_t nkv[kMaxAttnStreams];           // valid rows per stream
    int32_t B, H, Nq;
    int32_t qpairs;                         // ceil(Nq / 256)
    int32_t full_items;                     // items 0..full_items-1 run whole, one unit each
    int32_t splits;                         // key-range splits of every later item (1..kMaxKvSplits)
    float scale_log2;                       // softmax scale * log2(e)
    uint64_t timeout_ns;
    int64_t drop_tile;                      // fault injection: KV tile whose copy is skipped, or -1
};

// Encodes the tensor maps and launches; returns the CUDA error of the launch.
// Workspace pieces used by the attention call.
struct AttnScratch {
    uint32_t* err;
    int32_t* counters;
    float* part_ml;
    float* part_o;
};

// How the (stream, head, query pair) items are cut into CTAs: the first full_items items run
// whole (one CTA each; a multiple of the SM count, so whole waves), every later item is cut into
// `splits` key ranges whose partial rows are merged by the last to finish.
struct KvSchedule {
    int full_items;
    int splits;
};

// The schedule with the smallest estimated makespan on `slots` SMs for `items` items whose key
// loops have at least `min_tiles` tiles.
KvSchedule choose_kv_schedule(int64_t items, int min_tiles, int slots);

// Encodes the tensor maps, picks the schedule -- `sched` if given, else `force_splits` > 0 key
// ranges for every item, else choose_kv_schedule -- and launches; returns the CUDA error of the
// launch.  *splits_used receives the split count of the split items (1 if none is split).
cudaError_t launch_chunk_attention(const uint16_t* q_rot, const uint16_t* k_cache,
                                   const uint16_t* v_cache, int B, int H, int Nq,
                                   int64_t rows_per_head, const int32_t* nkv, float scale,
                                   uint16_t* out, float* lse, const AttnScratch& ws,
                                   uint64_t timeout_ns, int64_t drop_tile, int force_splits,
                                   const KvSchedule* sched, cudaStream_t s, int* splits_used,
                                   const char** why);

// ---- motion -----------------------------------------------------------------------------------

cudaError_t launch_motion_l2(const uint8_t* frames, int B, int64_t T, int64_t frame_bytes,
                             uint64_t* ssd, float* m, cudaStream_t s);

// ---- refresh re-rotation, sink update, noise controller ------------------------------------

constexpr int kMaxTimePairsPerAxis = 64;
constexpr int kMaxSinkFrames = 64;
constexpr int kMaxCacheStreams = 64;

struct RerotateParams {
    uint16_t* k_cache;
    sdv2_slot_meta* meta;
    int32_t B, H, HW, Fs, W, nslots;
    int32_t tp;                              // time-axis rotation pairs
    int32_t tvecs;                           // 16-byte vectors that hold time-axis dims
    int64_t shift;                           // F*R: subtracted from the slots' tpos
    int32_t active[kMaxCacheStreams];        // stream is at a refresh chunk
    int64_t limit[kMaxCacheStreams];         // frames below c*F are re-rotated
    float2 cs[kMaxTimePairsPerAxis];         // (cos, sin) of the angle -F*R*omega_j
};

struct SinkUpdateParams {
    uint16_t* k_cache;
    uint16_t* v_cache;
    sdv2_slot_meta* meta;
    int32_t B, H, HW, Fs, nslots;
    int32_t active[kMaxCacheStreams];
    int32_t src_slot[kMaxCacheStreams * kMaxSinkFrames];   // [b][s]: window slot copied into sink slot s
};

struct NoiseParams {
    const float* m;
    float* rate;
    float* state;                            // [B] or null
    int32_t B;
    int64_t T;
    float m_lo, m_hi, out_lo, out_hi, ema;
    int32_t more_noise_when_fast;
};

cudaError_t launch_rerotate(const RerotateParams& p, cudaStream_t s);
cudaError_t launch_sink_update(const SinkUpdateParams& p, cudaStream_t s);
cudaError_t launch_noise(const NoiseParams& p, cudaStream_t s);

// ---- fused QKV projection + Causal-RoPE + cache append -------------------------------------

struct QkvRopeParams {
    CUtensorMap xmap;                         // x: [M = B*Nq][C] bf16
    CUtensorMap wmap;                         // w_qkv: [3*H*D][C] bf16
    const float* bias;                        // [3*H*D] or null
    uint16_t* q_rot;
    uint16_t* k_cache;
    uint16_t* v_cache;
    sdv2_slot_meta* meta;
    const float2* h_tab;                      // pair-major: [rope_h/2][grid_h] (cos, sin)
    const float2* w_tab;                      // pair-major: [rope_w/2][grid_w]
    uint32_t* err;
    uint64_t timeout_ns;
    int32_t M, C, B, H, HW, grid_h, grid_w, F, nslots, Nq;
    int32_t tp, hp, wp;
    int32_t m_fastest;                        // tile order: token tiles fastest (weights larger than L2)
    FrameDesc frames[kMaxChunkFrames];
    float2 tcs[kMaxTimePairs];
};

// Encodes the tensor maps (x rows `x_ld` elements apart) and launches.
cudaError_t launch_qkv_rope(QkvRopeParams& p, const void* x, const void* w, int64_t x_ld, cudaStream_t s,
                            const char** why);

// Sets the per-thread message returned by sdv2_last_error().
void set_last_error(const char* msg);

// Process-wide settings of the attention entry points (sdv2_set_wait_timeout_ns,
// sdv2_debug_drop_kv_tile, sdv2_debug_set_kv_splits) and the per-thread split count that
// sdv2_last_kv_splits reports.
uint64_t wait_timeout_ns();
int64_t debug_drop_tile();
int debug_force_splits();
void set_last_kv_splits(int splits);

// Largest chunk index the entry points accept (frame numbers c*F stay far inside int64).
constexpr int64_t kMaxChunkIndex = int64_t(1) << 40;

// ---- misc kernels -----------------------------------------------------------------------------

cudaError_t launch_cache_reset(uint16_t* k, uint16_t* v, size_t cache_bytes, sdv2_slot_meta* meta,
                               int64_t nmeta, cudaStream_t s);

}  // namespace sdv2
