// C ABI of the library: argument validation, host-side RoPE tables, and dispatch to the kernels.
//
// RoPE frequencies follow the 3D rotary embedding of a Wan-style DiT with the time index of
// Causal-RoPE ("Accelerating Video Generation Inference with Sequential-Parallel 3D Positional
// Encoding Using a Global Time Index", technical summary 2(나), 2(다)): the angle of pair j of an
// axis of d dims at position pos is pos * base^(-2j/d), evaluated in fp64, and the table holds
// the fp64 cos/sin rounded once to fp32 (precomputed contiguous tables instead of a cache).
// The RoPE refresh ("StreamDiffusionV2" review page, section 三) resets the chunk offset of the
// time index every R chunks.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "internal.h"

namespace {

thread_local char g_last_error[256] = "";
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int64_t> g_drop_tile{-1};

constexpr size_t kErrBytes = 256;   // workspace header: error word and where the split counters are

// First bytes of the workspace.  The error word is what the kernels set; the counter location
// lets sdv2_check_device_error clear the split counters after an aborted launch.
struct WsHeader {
    uint32_t err;
    uint32_t pad;
    uint64_t counters_off;
    uint64_t counters_bytes;
};

sdv2_status fail(sdv2_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
sdv2_status fail(sdv2_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

sdv2_status ok()
{
    g_last_error[0] = 0;
    return SDV2_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

sdv2_status check_cfg(const sdv2_stream_cfg* c)
{
    if (!c) return fail(SDV2_ERR_INVALID_ARG, "cfg is NULL");
    if (c->batch < 1 || c->heads < 1) return fail(SDV2_ERR_INVALID_ARG, "batch and heads must be >= 1");
    if (c->rope_t < 0 || c->rope_h < 0 || c->rope_w < 0 || (c->rope_t | c->rope_h | c->rope_w) & 1)
        return fail(SDV2_ERR_INVALID_ARG, "rope_t, rope_h, rope_w must be even and >= 0");
    if (c->rope_t + c->rope_h + c->rope_w != c->head_dim)
        return fail(SDV2_ERR_INVALID_ARG, "rope_t + rope_h + rope_w (%d) != head_dim (%d)",
                    c->rope_t + c->rope_h + c->rope_w, c->head_dim);
    if (c->head_dim != 128) return fail(SDV2_ERR_UNSUPPORTED, "only head_dim 128 is built (got %d)", c->head_dim);
    if (!(c->rope_base > 1.0) || !std::isfinite(c->rope_base)) return fail(SDV2_ERR_INVALID_ARG, "rope_base must be > 1");
    if (c->grid_h < 1 || c->grid_w < 1) return fail(SDV2_ERR_INVALID_ARG, "grid_h and grid_w must be >= 1");
    if (c->chunk_frames < 1) return fail(SDV2_ERR_INVALID_ARG, "chunk_frames must be >= 1");
    if (c->sink_frames < 0) return fail(SDV2_ERR_INVALID_ARG, "sink_frames must be >= 0");
    if (c->window_frames < c->chunk_frames)
        return fail(SDV2_ERR_INVALID_ARG, "window_frames (%d) must be >= chunk_frames (%d)", c->window_frames,
                    c->chunk_frames);
    if (c->refresh_chunks < 0) return fail(SDV2_ERR_INVALID_ARG, "refresh_chunks must be >= 0");
    const int64_t hw = static_cast<int64_t>(c->grid_h) * c->grid_w;
    const int64_t rows = (static_cast<int64_t>(c->sink_frames) + c->window_frames) * hw;
    const int64_t nq = hw * c->chunk_frames;
    if (rows > (int64_t(1) << 30) || nq > (int64_t(1) << 30))
        return fail(SDV2_ERR_INVALID_ARG, "cache rows per head (%lld) or chunk tokens (%lld) exceed 2^30",
                    (long long)rows, (long long)nq);
    const int64_t stride = c->qkv_token_stride ? c->qkv_token_stride : int64_t(c->heads) * c->head_dim;
    if (stride < int64_t(c->heads) * c->head_dim || (stride & 7))
        return fail(SDV2_ERR_INVALID_ARG, "qkv_token_stride (%lld) must be >= H*D and a multiple of 8",
                    (long long)stride);
    return SDV2_OK;
}

int64_t hw_of(const sdv2_stream_cfg* c) { return static_cast<int64_t>(c->grid_h) * c->grid_w; }
int64_t slots_of(const sdv2_stream_cfg* c) { return static_cast<int64_t>(c->sink_frames) + c->window_frames; }

int64_t visible_frames(const sdv2_stream_cfg* c, int64_t chunk)
{
    const int64_t n = (chunk + 1) * c->chunk_frames;
    const int64_t fs = c->sink_frames, w = c->window_frames;
    return std::min(fs, n) + std::min(w, std::max<int64_t>(0, n - fs));
}

int64_t slot_of(const sdv2_stream_cfg* c, int64_t frame)
{
    if (frame < c->sink_frames) return frame;
    return c->sink_frames + (frame - c->sink_frames) % c->window_frames;
}

double omega(int j, int d, double base) { return std::pow(base, -static_cast<double>(2 * j) / static_cast<double>(d)); }

void cos_sin_f32(int64_t pos, int j, int d, double base, float* cs)
{
    const double th = static_cast<double>(pos) * omega(j, d, base);
    cs[0] = static_cast<float>(std::cos(th));
    cs[1] = static_cast<float>(std::sin(th));
}

// Frame descriptors (slot, stream-relative frame, time index) and the time-axis (cos, sin)
// rows of one chunk of every stream: entries b*F + i.
void fill_frames(const sdv2_stream_cfg* c, const int64_t* start_frame, const int64_t* chunk_index,
                 sdv2::FrameDesc* frames, float2* tcs)
{
    const int F = c->chunk_frames, tp = c->rope_t / 2;
    for (int b = 0; b < c->batch; ++b) {
        const int64_t cidx = chunk_index[b];
        const int64_t ceff = c->refresh_chunks > 0 ? cidx % c->refresh_chunks : cidx;
        for (int i = 0; i < F; ++i) {
            sdv2::FrameDesc& fd = frames[b * F + i];
            fd.frame = cidx * F + i;
            fd.tpos = start_frame[b] + ceff * F + i;
            fd.slot = static_cast<int32_t>(slot_of(c, fd.frame));
            for (int j = 0; j < tp; ++j) cos_sin_f32(fd.tpos, j, c->rope_t, c->rope_base, &tcs[(b * F + i) * tp + j].x);
        }
    }
}

// Checks shared by the two append entry points: host arrays, sizes of the per-call tables.
sdv2_status check_append_args(const sdv2_stream_cfg* c, const int64_t* start_frame, const int64_t* chunk_index)
{
    if (!start_frame || !chunk_index) return fail(SDV2_ERR_INVALID_ARG, "start_frame and chunk_index are required");
    const int B = c->batch, F = c->chunk_frames, tp = c->rope_t / 2;
    if (static_cast<int64_t>(B) * F > sdv2::kMaxChunkFrames || static_cast<int64_t>(B) * F * tp > sdv2::kMaxTimePairs)
        return fail(SDV2_ERR_UNSUPPORTED, "B*F (%d) must be <= %d and B*F*rope_t/2 (%d) <= %d", B * F,
                    sdv2::kMaxChunkFrames, B * F * tp, sdv2::kMaxTimePairs);
    for (int b = 0; b < B; ++b) {
        if (start_frame[b] < 0 || chunk_index[b] < 0)
            return fail(SDV2_ERR_INVALID_ARG, "start_frame[%d] and chunk_index[%d] must be >= 0", b, b);
        if (chunk_index[b] > sdv2::kMaxChunkIndex || start_frame[b] > (int64_t(1) << 50))
            return fail(SDV2_ERR_INVALID_ARG, "start_frame[%d] or chunk_index[%d] too large", b, b);
    }
    return SDV2_OK;
}

// sm_103 check, cached per device.
sdv2_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SDV2_ERR_CUDA, "cudaGetDevice failed");
    // 0 = not looked up yet, 1 = sm_103, -1 = another device; threads racing on the first
    // lookup store the same value
    static std::atomic<int8_t> known[64];
    if (dev < 0 || dev >= 64) return fail(SDV2_ERR_UNSUPPORTED, "device index %d out of range", dev);
    int8_t k = known[dev].load(std::memory_order_relaxed);
    if (k == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        k = (major == 10 && minor == 3) ? 1 : -1;
        known[dev].store(k, std::memory_order_relaxed);
    }
    if (k < 0) return fail(SDV2_ERR_UNSUPPORTED, "the library is built for sm_103a (GB300) only");
    return SDV2_OK;
}

sdv2_status cuda_status(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return ok();
    return fail(SDV2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Workspace: [error word | h table | w table | h table, pair-major | w table, pair-major |
// split counters | split (m, l) | split rows].
struct WsLayout {
    size_t htab, wtab, htab_pm, wtab_pm, counters, part_ml, part_o, total;
};

WsLayout ws_layout(const sdv2_stream_cfg* c)
{
    WsLayout L{};
    const int64_t nq = hw_of(c) * c->chunk_frames;
    const int64_t items = static_cast<int64_t>(c->batch) * c->heads *
                          ((nq + sdv2::kAttnRowsPerCta - 1) / sdv2::kAttnRowsPerCta);
    const int64_t rows = items * sdv2::kMaxKvSplits * sdv2::kAttnRowsPerCta;
    size_t off = kErrBytes;
    L.htab = off;
    off += round_up(sizeof(float2) * c->grid_h * (c->rope_h / 2), 256);
    L.wtab = off;
    off += round_up(sizeof(float2) * c->grid_w * (c->rope_w / 2), 256);
    L.htab_pm = off;
    off += round_up(sizeof(float2) * c->grid_h * (c->rope_h / 2), 256);
    L.wtab_pm = off;
    off += round_up(sizeof(float2) * c->grid_w * (c->rope_w / 2), 256);
    L.counters = off;
    off += round_up(sizeof(int32_t) * 2 * items, 256);       // tickets, published splits
    L.part_ml = off;
    off += round_up(sizeof(float) * 2 * rows, 256);
    L.part_o = off;
    off += round_up(sizeof(float) * 128 * rows, 256);
    L.total = off;
    return L;
}

std::atomic<int> g_force_splits{0};
thread_local int g_last_splits = 0;

}  // namespace

namespace sdv2 {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg ? msg : ""); }
uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }
int64_t debug_drop_tile() { return g_drop_tile.load(); }
int debug_force_splits() { return g_force_splits.load(); }
void set_last_kv_splits(int splits) { g_last_splits = splits; }
}  // namespace sdv2

extern "C" {

const char* sdv2_status_string(sdv2_status s)
{
    switch (s) {
    case SDV2_OK: return "ok";
    case SDV2_ERR_INVALID_ARG: return "invalid argument";
    case SDV2_ERR_UNSUPPORTED: return "unsupported";
    case SDV2_ERR_CUDA: return "CUDA error";
    case SDV2_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* sdv2_last_error(void) { return g_last_error; }

void sdv2_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void sdv2_debug_drop_kv_tile(int64_t tile) { g_drop_tile.store(tile < 0 ? -1 : tile); }

void sdv2_debug_set_kv_splits(int32_t splits) { g_force_splits.store(splits < 0 ? 0 : splits); }

int32_t sdv2_last_kv_splits(void) { return g_last_splits; }

int32_t sdv2_debug_kv_schedule(int64_t items, int32_t min_tiles, int32_t sms, int32_t* full_items)
{
    if (items < 1 || min_tiles < 1 || sms < 1 || !full_items) return -1;
    const sdv2::KvSchedule ks = sdv2::choose_kv_schedule(items, min_tiles, sms);
    *full_items = ks.full_items;
    return ks.splits;
}

size_t sdv2_workspace_bytes(const sdv2_stream_cfg* c)
{
    if (check_cfg(c) != SDV2_OK) return 0;
    return ws_layout(c).total;
}

size_t sdv2_cache_bytes(const sdv2_stream_cfg* c)
{
    if (check_cfg(c) != SDV2_OK) return 0;
    return static_cast<size_t>(c->batch) * c->heads * slots_of(c) * hw_of(c) * c->head_dim * 2;
}

size_t sdv2_meta_bytes(const sdv2_stream_cfg* c)
{
    if (check_cfg(c) != SDV2_OK) return 0;
    return static_cast<size_t>(c->batch) * slots_of(c) * sizeof(sdv2_slot_meta);
}

int64_t sdv2_visible_tokens(const sdv2_stream_cfg* c, int64_t chunk_index)
{
    if (check_cfg(c) != SDV2_OK || chunk_index < 0) return -1;
    return visible_frames(c, chunk_index) * hw_of(c);
}

sdv2_status sdv2_workspace_init(const sdv2_stream_cfg* c, void* ws, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if (!ws || !aligned16(ws)) return fail(SDV2_ERR_INVALID_ARG, "ws must be a non-null 16-byte aligned pointer");
    if ((s = check_device()) != SDV2_OK) return s;
    const WsLayout L = ws_layout(c);
    const int hp = c->rope_h / 2, wp = c->rope_w / 2;
    std::vector<float> htab(2 * c->grid_h * hp), wtab(2 * c->grid_w * wp);
    std::vector<float> htab_pm(htab.size()), wtab_pm(wtab.size());     // [pair][position]
    for (int y = 0; y < c->grid_h; ++y)
        for (int j = 0; j < hp; ++j) {
            cos_sin_f32(y, j, c->rope_h, c->rope_base, &htab[2 * (y * hp + j)]);
            htab_pm[2 * (j * c->grid_h + y)] = htab[2 * (y * hp + j)];
            htab_pm[2 * (j * c->grid_h + y) + 1] = htab[2 * (y * hp + j) + 1];
        }
    for (int x = 0; x < c->grid_w; ++x)
        for (int j = 0; j < wp; ++j) {
            cos_sin_f32(x, j, c->rope_w, c->rope_base, &wtab[2 * (x * wp + j)]);
            wtab_pm[2 * (j * c->grid_w + x)] = wtab[2 * (x * wp + j)];
            wtab_pm[2 * (j * c->grid_w + x) + 1] = wtab[2 * (x * wp + j) + 1];
        }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* base = static_cast<unsigned char*>(ws);
    cudaError_t e = cudaMemsetAsync(ws, 0, L.total, st);
    if (e == cudaSuccess && !htab.empty())
        e = cudaMemcpyAsync(base + L.htab, htab.data(), htab.size() * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !wtab.empty())
        e = cudaMemcpyAsync(base + L.wtab, wtab.data(), wtab.size() * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !htab_pm.empty())
        e = cudaMemcpyAsync(base + L.htab_pm, htab_pm.data(), htab_pm.size() * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !wtab_pm.empty())
        e = cudaMemcpyAsync(base + L.wtab_pm, wtab_pm.data(), wtab_pm.size() * sizeof(float), cudaMemcpyHostToDevice, st);
    WsHeader hdr{0, 0, L.counters, L.part_ml - L.counters};
    if (e == cudaSuccess) e = cudaMemcpyAsync(ws, &hdr, sizeof(hdr), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e, "workspace upload");
}

sdv2_status sdv2_cache_reset(const sdv2_stream_cfg* c, void* k_cache, void* v_cache, void* meta, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if (!k_cache || !v_cache || !meta || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta))
        return fail(SDV2_ERR_INVALID_ARG, "k_cache, v_cache and meta must be non-null and 16-byte aligned");
    if ((s = check_device()) != SDV2_OK) return s;
    cudaError_t e = sdv2::launch_cache_reset(static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
                                             sdv2_cache_bytes(c), static_cast<sdv2_slot_meta*>(meta),
                                             static_cast<int64_t>(c->batch) * slots_of(c),
                                             static_cast<cudaStream_t>(stream));
    return cuda_status(e, "cache_reset launch");
}

sdv2_status sdv2_rope_append_kv(const sdv2_stream_cfg* c, const int64_t* start_frame, const int64_t* chunk_index,
                                const void* q, const void* k, const void* v, void* q_rot, void* k_cache,
                                void* v_cache, void* meta, void* ws, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    const void* ptrs[] = {q, k, v, q_rot, k_cache, v_cache, meta, ws};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return fail(SDV2_ERR_INVALID_ARG, "device pointers must be non-null and 16-byte aligned");
    if ((s = check_append_args(c, start_frame, chunk_index)) != SDV2_OK) return s;
    const int B = c->batch, F = c->chunk_frames, tp = c->rope_t / 2;
    if ((s = check_device()) != SDV2_OK) return s;

    static thread_local sdv2::RopeAppendParams p;
    std::memset(&p, 0, sizeof(p));
    const int64_t hw = hw_of(c);
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.q_rot = static_cast<uint16_t*>(q_rot);
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.v_cache = static_cast<uint16_t*>(v_cache);
    p.meta = static_cast<sdv2_slot_meta*>(meta);
    const WsLayout L = ws_layout(c);
    p.h_tab = reinterpret_cast<const float2*>(static_cast<const unsigned char*>(ws) + L.htab);
    p.w_tab = reinterpret_cast<const float2*>(static_cast<const unsigned char*>(ws) + L.wtab);
    p.tok_stride = c->qkv_token_stride ? c->qkv_token_stride : int64_t(c->heads) * c->head_dim;
    p.B = B;
    p.H = c->heads;
    p.HW = static_cast<int32_t>(hw);
    p.grid_w = c->grid_w;
    p.F = F;
    p.nslots = static_cast<int32_t>(slots_of(c));
    p.Nq = static_cast<int32_t>(hw * F);
    p.tp = tp;
    p.hp = c->rope_h / 2;
    p.wp = c->rope_w / 2;
    fill_frames(c, start_frame, chunk_index, p.frames, p.tcs);
    return cuda_status(sdv2::launch_rope_append(p, static_cast<cudaStream_t>(stream)), "rope_append launch");
}

sdv2_status sdv2_chunk_attention(const sdv2_stream_cfg* c, const int64_t* chunk_index, const void* q_rot,
                                 const void* k_cache, const void* v_cache, float scale, void* out, float* lse,
                                 void* ws, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if (!chunk_index) return fail(SDV2_ERR_INVALID_ARG, "chunk_index is required");
    const void* ptrs[] = {q_rot, k_cache, v_cache, out, ws};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return fail(SDV2_ERR_INVALID_ARG, "device pointers must be non-null and 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SDV2_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (c->batch > sdv2::kMaxAttnStreams)
        return fail(SDV2_ERR_UNSUPPORTED, "batch (%d) > %d streams per attention call", c->batch, sdv2::kMaxAttnStreams);
    if (static_cast<int64_t>(c->heads) * c->batch > 65535) return fail(SDV2_ERR_UNSUPPORTED, "too many heads");
    if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(c->head_dim));
    if (!std::isfinite(scale)) return fail(SDV2_ERR_INVALID_ARG, "scale must be finite");
    int32_t nkv[sdv2::kMaxAttnStreams];
    for (int b = 0; b < c->batch; ++b) {
        if (chunk_index[b] < 0 || chunk_index[b] > sdv2::kMaxChunkIndex)
            return fail(SDV2_ERR_INVALID_ARG, "chunk_index[%d] must be in [0, 2^40]", b);
        nkv[b] = static_cast<int32_t>(visible_frames(c, chunk_index[b]) * hw_of(c));
    }
    if ((s = check_device()) != SDV2_OK) return s;
    const char* why = "launch";
    const WsLayout L = ws_layout(c);
    unsigned char* base = static_cast<unsigned char*>(ws);
    sdv2::AttnScratch scratch{reinterpret_cast<uint32_t*>(base), reinterpret_cast<int32_t*>(base + L.counters),
                              reinterpret_cast<float*>(base + L.part_ml), reinterpret_cast<float*>(base + L.part_o)};
    cudaError_t e = sdv2::launch_chunk_attention(
        static_cast<const uint16_t*>(q_rot), static_cast<const uint16_t*>(k_cache), static_cast<const uint16_t*>(v_cache),
        c->batch, c->heads, static_cast<int>(hw_of(c) * c->chunk_frames), slots_of(c) * hw_of(c), nkv, scale,
        static_cast<uint16_t*>(out), lse, scratch, g_timeout_ns.load(), g_drop_tile.load(), g_force_splits.load(),
        nullptr, static_cast<cudaStream_t>(stream), &g_last_splits, &why);
    return cuda_status(e, why);
}

sdv2_status sdv2_motion_l2(const uint8_t* frames, int32_t B, int64_t T, int32_t Hp, int32_t Wp, int32_t C,
                           uint64_t* ssd, float* m, void* stream)
{
    if (!frames || !ssd || !aligned16(frames) || !aligned16(ssd) || (m && !aligned16(m)))
        return fail(SDV2_ERR_INVALID_ARG, "frames and ssd (and m if given) must be non-null and 16-byte aligned");
    if (B < 1 || T < 1 || Hp < 1 || Wp < 1 || C < 1)
        return fail(SDV2_ERR_INVALID_ARG, "B, T, Hp, Wp, C must be >= 1");
    const int64_t npix = static_cast<int64_t>(Hp) * Wp * C;
    if (npix % 16) return fail(SDV2_ERR_INVALID_ARG, "Hp*Wp*C (%lld) must be a multiple of 16", (long long)npix);
    if (static_cast<int64_t>(B) * T > 65535)
        return fail(SDV2_ERR_UNSUPPORTED, "B*T must be <= 65535");
    if (npix > (int64_t(1) << 40)) return fail(SDV2_ERR_INVALID_ARG, "frame too large");
    sdv2_status s = check_device();
    if (s != SDV2_OK) return s;
    return cuda_status(sdv2::launch_motion_l2(frames, B, T, npix, ssd, m, static_cast<cudaStream_t>(stream)),
                       "motion_l2 launch");
}

sdv2_status sdv2_qkv_rope_append(const sdv2_stream_cfg* c, const int64_t* start_frame, const int64_t* chunk_index,
                                  const void* x, int64_t x_token_stride, const void* w_qkv, const float* bias,
                                  void* q_rot, void* k_cache, void* v_cache, void* meta, void* ws, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if ((s = check_append_args(c, start_frame, chunk_index)) != SDV2_OK) return s;
    const void* ptrs[] = {x, w_qkv, q_rot, k_cache, v_cache, meta, ws};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return fail(SDV2_ERR_INVALID_ARG, "device pointers must be non-null and 16-byte aligned");
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 15u)) return fail(SDV2_ERR_INVALID_ARG, "bias must be 16-byte aligned");
    const int64_t C = static_cast<int64_t>(c->heads) * c->head_dim;
    const int64_t ld = x_token_stride ? x_token_stride : C;
    if (ld < C || (ld % 8)) return fail(SDV2_ERR_INVALID_ARG, "x_token_stride must be >= H*D and a multiple of 8");
    const int64_t M = static_cast<int64_t>(c->batch) * hw_of(c) * c->chunk_frames;
    if (M > (int64_t(1) << 31) - 256) return fail(SDV2_ERR_UNSUPPORTED, "too many tokens");
    if ((s = check_device()) != SDV2_OK) return s;
    static thread_local sdv2::QkvRopeParams p;
    std::memset(&p, 0, sizeof(p));
    const WsLayout L = ws_layout(c);
    p.bias = bias;
    p.q_rot = static_cast<uint16_t*>(q_rot);
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.v_cache = static_cast<uint16_t*>(v_cache);
    p.meta = static_cast<sdv2_slot_meta*>(meta);
    p.h_tab = reinterpret_cast<const float2*>(static_cast<const unsigned char*>(ws) + L.htab_pm);
    p.w_tab = reinterpret_cast<const float2*>(static_cast<const unsigned char*>(ws) + L.wtab_pm);
    p.err = static_cast<uint32_t*>(ws);
    p.timeout_ns = g_timeout_ns.load();
    p.M = static_cast<int32_t>(M);
    p.C = static_cast<int32_t>(C);
    p.B = c->batch;
    p.H = c->heads;
    p.HW = static_cast<int32_t>(hw_of(c));
    p.grid_h = c->grid_h;
    p.grid_w = c->grid_w;
    p.F = c->chunk_frames;
    p.nslots = static_cast<int32_t>(slots_of(c));
    p.Nq = static_cast<int32_t>(hw_of(c) * c->chunk_frames);
    p.tp = c->rope_t / 2;
    p.hp = c->rope_h / 2;
    p.wp = c->rope_w / 2;
    fill_frames(c, start_frame, chunk_index, p.frames, p.tcs);
    const char* why = "launch";
    cudaError_t e = sdv2::launch_qkv_rope(p, x, w_qkv, ld, static_cast<cudaStream_t>(stream), &why);
    return cuda_status(e, why);
}

sdv2_status sdv2_rope_refresh_rerotate(const sdv2_stream_cfg* c, const int64_t* chunk_index, void* k_cache,
                                       void* meta, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if (!chunk_index) return fail(SDV2_ERR_INVALID_ARG, "chunk_index is required");
    if (!k_cache || !meta || !aligned16(k_cache) || !aligned16(meta))
        return fail(SDV2_ERR_INVALID_ARG, "k_cache and meta must be non-null and 16-byte aligned");
    if (c->batch > sdv2::kMaxCacheStreams) return fail(SDV2_ERR_UNSUPPORTED, "more than 64 streams");
    if (c->rope_t / 2 > sdv2::kMaxTimePairsPerAxis) return fail(SDV2_ERR_UNSUPPORTED, "rope_t > 128");
    for (int b = 0; b < c->batch; ++b)
        if (chunk_index[b] < 0 || chunk_index[b] > sdv2::kMaxChunkIndex)
            return fail(SDV2_ERR_INVALID_ARG, "chunk_index[%d] must be in [0, 2^40]", b);
    if ((s = check_device()) != SDV2_OK) return s;
    sdv2::RerotateParams p{};
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.meta = static_cast<sdv2_slot_meta*>(meta);
    p.B = c->batch;
    p.H = c->heads;
    p.HW = static_cast<int32_t>(hw_of(c));
    p.Fs = c->sink_frames;
    p.W = c->window_frames;
    p.nslots = static_cast<int32_t>(slots_of(c));
    p.tp = c->rope_t / 2;
    p.tvecs = (p.tp + 3) / 4;
    const int64_t R = c->refresh_chunks;
    p.shift = static_cast<int64_t>(c->chunk_frames) * R;
    bool any = false;
    for (int b = 0; b < c->batch; ++b) {
        p.active[b] = (R > 0 && chunk_index[b] > 0 && chunk_index[b] % R == 0) ? 1 : 0;
        p.limit[b] = chunk_index[b] * c->chunk_frames;
        any = any || p.active[b];
    }
    if (!any) return ok();            // with rope_t = 0 nothing rotates, but the slots' tpos still move
    for (int j = 0; j < p.tp; ++j) cos_sin_f32(-p.shift, j, c->rope_t, c->rope_base, &p.cs[j].x);
    return cuda_status(sdv2::launch_rerotate(p, static_cast<cudaStream_t>(stream)), "rerotate launch");
}

sdv2_status sdv2_sink_update(const sdv2_stream_cfg* c, const int64_t* chunk_index, const int32_t* update,
                             void* k_cache, void* v_cache, void* meta, void* stream)
{
    sdv2_status s = check_cfg(c);
    if (s != SDV2_OK) return s;
    if (!chunk_index || !update) return fail(SDV2_ERR_INVALID_ARG, "chunk_index and update are required");
    if (!k_cache || !v_cache || !meta || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(meta))
        return fail(SDV2_ERR_INVALID_ARG, "k_cache, v_cache and meta must be non-null and 16-byte aligned");
    if (c->batch > sdv2::kMaxCacheStreams) return fail(SDV2_ERR_UNSUPPORTED, "more than 64 streams");
    if (c->sink_frames > sdv2::kMaxSinkFrames) return fail(SDV2_ERR_UNSUPPORTED, "more than 64 sink frames");
    if (c->sink_frames == 0) return ok();
    if (c->window_frames < c->sink_frames)
        return fail(SDV2_ERR_INVALID_ARG, "a sink update needs window_frames >= sink_frames");
    sdv2::SinkUpdateParams p{};
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.v_cache = static_cast<uint16_t*>(v_cache);
    p.meta = static_cast<sdv2_slot_meta*>(meta);
    p.B = c->batch;
    p.H = c->heads;
    p.HW = static_cast<int32_t>(hw_of(c));
    p.Fs = c->sink_frames;
    p.nslots = static_cast<int32_t>(slots_of(c));
    bool any = false;
    for (int b = 0; b < c->batch; ++b) {
        if (chunk_index[b] < 0 || chunk_index[b] > sdv2::kMaxChunkIndex)
            return fail(SDV2_ERR_INVALID_ARG, "chunk_index[%d] must be in [0, 2^40]", b);
        p.active[b] = update[b] ? 1 : 0;
        if (!p.active[b]) continue;
        const int64_t n = (chunk_index[b] + 1) * c->chunk_frames;   // frames appended so far
        if (n < 2 * static_cast<int64_t>(c->sink_frames))
            return fail(SDV2_ERR_INVALID_ARG, "stream %d: a sink update needs at least 2*sink_frames frames", b);
        for (int i = 0; i < c->sink_frames; ++i)
            p.src_slot[b * sdv2::kMaxSinkFrames + i] = static_cast<int32_t>(slot_of(c, n - c->sink_frames + i));
        any = true;
    }
    if (!any) return ok();
    if ((s = check_device()) != SDV2_OK) return s;
    return cuda_status(sdv2::launch_sink_update(p, static_cast<cudaStream_t>(stream)), "sink update launch");
}

sdv2_status sdv2_noise_from_motion(const sdv2_noise_ctl* ctl, const float* m, int32_t B, int64_t T, float* state,
                                   float* rate, void* stream)
{
    if (!ctl || !m || !rate) return fail(SDV2_ERR_INVALID_ARG, "ctl, m and rate are required");
    if (B < 1 || T < 1) return fail(SDV2_ERR_INVALID_ARG, "B and T must be >= 1");
    if (!(ctl->motion_hi > ctl->motion_lo) || !std::isfinite(ctl->motion_lo) || !std::isfinite(ctl->motion_hi))
        return fail(SDV2_ERR_INVALID_ARG, "motion_hi must be > motion_lo (both finite)");
    if (!(ctl->rate_lo >= 0.f) || !(ctl->rate_hi >= 0.f) || !std::isfinite(ctl->rate_lo) || !std::isfinite(ctl->rate_hi))
        return fail(SDV2_ERR_INVALID_ARG, "rates must be finite and >= 0");
    if (!(ctl->ema >= 0.f && ctl->ema < 1.f)) return fail(SDV2_ERR_INVALID_ARG, "ema must be in [0, 1)");
    const void* ptrs[] = {m, rate};
    for (const void* p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 3u)) return fail(SDV2_ERR_INVALID_ARG, "m and rate must be 4-byte aligned");
    sdv2_status s = check_device();
    if (s != SDV2_OK) return s;
    sdv2::NoiseParams p{};
    p.m = m;
    p.rate = rate;
    p.state = state;
    p.B = B;
    p.T = T;
    p.m_lo = ctl->motion_lo;
    p.m_hi = ctl->motion_hi;
    p.out_lo = ctl->rate_lo;
    p.out_hi = ctl->rate_hi;
    p.ema = ctl->ema;
    p.more_noise_when_fast = ctl->more_noise_when_fast;
    return cuda_status(sdv2::launch_noise(p, static_cast<cudaStream_t>(stream)), "noise controller launch");
}

sdv2_status sdv2_check_device_error(void* ws, void* stream)
{
    if (!ws) return fail(SDV2_ERR_INVALID_ARG, "ws is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader hdr{};
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && hdr.err) {
        // An aborted launch may leave split counters mid-count: clear them with the error word.
        e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), st);
        if (e == cudaSuccess && hdr.counters_bytes)
            e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + hdr.counters_off, 0, hdr.counters_bytes, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "check_device_error");
    if (hdr.err & sdv2::kErrTimeout)
        return fail(SDV2_ERR_TIMEOUT, "a bounded device wait gave up (error word 0x%x)", hdr.err);
    return ok();
}

}  // extern "C"
