// sdv2_chunk_attention_noalloc: chunk attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all -- for example code that runs inside a memory pool
// it does not own, a plugin host that forbids allocation after start-up, or a real-time loop
// that must never hit the allocator (an allocation can synchronize the device and stall a
// frame).  Such callers cannot size and own the workspace that sdv2_chunk_attention needs.
// This variant keeps its scratch (device error word, key-split arrival counters and the
// per-row partial results of the key splits) in one file-scope __device__ array instead.
//
// The array is part of the library's module: every GPU that loads the library holds its
// kNoAllocScratchBytes until the process exits.  All calls on a device share it, and it keeps
// the previous call's contents; each call therefore clears the split counters on its stream
// before the kernel runs.  The error word is not cleared by a call: a bounded wait that gave up
// leaves it set until sdv2_noalloc_check_device_error reads it, so a later call cannot hide an
// earlier timeout.  Calls whose kernels overlap on the GPU (different streams, or graph
// branches) race on the array and must not be issued.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace sdv2 {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB per GPU
constexpr size_t kNaHeader = 256;                            // error word
constexpr int64_t kNaMaxItems = 16384;                       // (stream, head, 256 rows) items
constexpr size_t kNaCounters = kNaHeader;
constexpr size_t kNaCountersBytes = sizeof(int32_t) * 2 * kNaMaxItems;   // tickets, published splits
constexpr size_t kNaPartMl = kNaCounters + kNaCountersBytes;
// Rows of split partials that fit: 8 bytes of (max, sum) + 512 bytes of output per row,
// rounded down to whole 256-row units.
constexpr int64_t kNaRows =
    static_cast<int64_t>((kNoAllocScratchBytes - kNaPartMl - 256) / (8 + 512)) / kAttnRowsPerCta * kAttnRowsPerCta;
constexpr size_t kNaPartO = kNaPartMl + ((static_cast<size_t>(kNaRows) * 8 + 255) / 256) * 256;
static_assert(kNaPartO + static_cast<size_t>(kNaRows) * 512 <= kNoAllocScratchBytes, "no-alloc scratch layout");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_na_mutex;
unsigned char* g_na_ptr[64] = {};          // device address of the array, per device

// Device address of the array on the current device `dev`, looked up (with that device
// current) on the first call and kept.  The first lookup also clears the error word and the
// counters on `st`.  Returns null if the lookup failed.
unsigned char* scratch_base(int dev, cudaStream_t st, cudaError_t* err)
{
    std::lock_guard<std::mutex> lock(g_na_mutex);
    *err = cudaSuccess;
    if (!g_na_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
        e = cudaMemsetAsync(p, 0, kNaPartMl, st);
        if (e != cudaSuccess) {
            *err = e;
            return nullptr;
        }
        g_na_ptr[dev] = static_cast<unsigned char*>(p);
    }
    return g_na_ptr[dev];
}

sdv2_status na_fail(sdv2_status s, const char* msg)
{
    char buf[256];
    snprintf(buf, sizeof(buf), "sdv2_chunk_attention_noalloc: %s", msg);
    set_last_error(buf);     // readable through sdv2_last_error()
    return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace sdv2

extern "C" sdv2_status sdv2_chunk_attention_noalloc(const sdv2_stream_cfg* cfg, const int64_t* chunk_index,
                                                    const void* q_rot, const void* k_cache, const void* v_cache,
                                                    float scale, void* out, float* lse, void* stream)
{
    using namespace sdv2;
    // Configuration and sizes (the library's own checks run inside these size queries).
    if (!cfg || sdv2_cache_bytes(cfg) == 0) return na_fail(SDV2_ERR_INVALID_ARG, "invalid stream configuration");
    if (!chunk_index) return na_fail(SDV2_ERR_INVALID_ARG, "chunk_index is required");
    const void* ptrs[] = {q_rot, k_cache, v_cache, out};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return na_fail(SDV2_ERR_INVALID_ARG, "device pointers must be non-null and 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return na_fail(SDV2_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (cfg->batch > kMaxAttnStreams) return na_fail(SDV2_ERR_UNSUPPORTED, "more than 16 streams");
    const int64_t hw = static_cast<int64_t>(cfg->grid_h) * cfg->grid_w;
    const int nq = static_cast<int>(hw * cfg->chunk_frames);
    const int64_t qpairs = (nq + kAttnRowsPerCta - 1) / kAttnRowsPerCta;
    const int64_t items = static_cast<int64_t>(cfg->batch) * cfg->heads * qpairs;
    if (items > kNaMaxItems)
        return na_fail(SDV2_ERR_UNSUPPORTED,
                       "batch * heads * ceil(Nq/256) exceeds 16384, the size its 16 MiB static scratch serves");
    if (static_cast<int64_t>(cfg->heads) * cfg->batch > 65535) return na_fail(SDV2_ERR_UNSUPPORTED, "too many heads");
    int32_t nkv[kMaxAttnStreams];
    int min_tiles = 1 << 30;
    for (int b = 0; b < cfg->batch; ++b) {
        if (chunk_index[b] < 0 || chunk_index[b] > kMaxChunkIndex)
            return na_fail(SDV2_ERR_INVALID_ARG, "chunk_index must be in [0, 2^40]");
        nkv[b] = static_cast<int32_t>(sdv2_visible_tokens(cfg, chunk_index[b]));
        min_tiles = std::min(min_tiles, (nkv[b] + 127) / 128);
    }
    if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(cfg->head_dim));
    if (!std::isfinite(scale)) return na_fail(SDV2_ERR_INVALID_ARG, "scale must be finite");

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return na_fail(SDV2_ERR_CUDA, "cudaGetDevice failed");
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return na_fail(SDV2_ERR_UNSUPPORTED, "the library is built for sm_103a (GB300) only");
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Set-up, once per device and with that device current: the device address of the array.
    cudaError_t e = cudaSuccess;
    unsigned char* base = scratch_base(dev, st, &e);
    if (!base) return na_fail(SDV2_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");

    // Schedule: the automatic (or forced) choice, its split count reduced until the split items'
    // partial rows fit in the array (with one split nothing is stored).
    const int force = debug_force_splits();
    KvSchedule ks = force > 0 ? KvSchedule{0, std::min(force, std::min(kMaxKvSplits, min_tiles))}
                              : choose_kv_schedule(items, min_tiles, std::max(1, sms));
    while (ks.splits > 1 && (items - ks.full_items) * ks.splits * kAttnRowsPerCta > kNaRows) --ks.splits;
    if (ks.splits <= 1) ks = KvSchedule{static_cast<int>(items), 1};

    // The array keeps the previous call's contents: clear the split counters (the error word
    // stays, see above).
    e = cudaMemsetAsync(base + kNaCounters, 0, kNaCountersBytes, st);
    if (e != cudaSuccess) return na_fail(SDV2_ERR_CUDA, "clearing the static scratch failed");
    AttnScratch scratch{reinterpret_cast<uint32_t*>(base), reinterpret_cast<int32_t*>(base + kNaCounters),
                        reinterpret_cast<float*>(base + kNaPartMl), reinterpret_cast<float*>(base + kNaPartO)};
    int used = 0;
    const char* why = "launch";
    e = launch_chunk_attention(static_cast<const uint16_t*>(q_rot), static_cast<const uint16_t*>(k_cache),
                               static_cast<const uint16_t*>(v_cache), cfg->batch, cfg->heads, nq,
                               (static_cast<int64_t>(cfg->sink_frames) + cfg->window_frames) * hw, nkv, scale,
                               static_cast<uint16_t*>(out), lse, scratch, wait_timeout_ns(), debug_drop_tile(), 0,
                               &ks, st, &used, &why);
    if (e != cudaSuccess) return na_fail(SDV2_ERR_CUDA, why);
    set_last_kv_splits(used);
    set_last_error("");
    return SDV2_OK;
}

extern "C" sdv2_status sdv2_noalloc_check_device_error(void* stream)
{
    using namespace sdv2;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return na_fail(SDV2_ERR_CUDA, "cudaGetDevice failed");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    unsigned char* base = scratch_base(dev, st, &e);
    if (!base) return na_fail(SDV2_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    uint32_t word = 0;
    e = cudaMemcpyAsync(&word, base, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && word) {
        // clear the error word and the counters an aborted launch may have left mid-count
        e = cudaMemsetAsync(base, 0, kNaPartMl, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) {
        char buf[200];
        snprintf(buf, sizeof(buf), "reading the static scratch's error word: %s", cudaGetErrorString(e));
        return na_fail(SDV2_ERR_CUDA, buf);
    }
    if (word & kErrTimeout) return na_fail(SDV2_ERR_TIMEOUT, "a bounded device wait gave up");
    set_last_error("");
    return SDV2_OK;
}
