// Cache maintenance at RoPE-refresh time, and the motion-driven noise controller.
//
// * Re-rotation of the window keys (the second reading of "RoPE refresh" on the
//   "StreamDiffusionV2" review page, section 三, "periodically reset the positional-encoding
//   offset"): when the time offset resets by F*R, the keys already in the rolling window are
//   turned back by the same F*R on the time axis, so that distances between the new chunk and
//   the window stay what they were (positions stay continuous across the reset).
// * Sink update ("StreamDiffusionV2" technical summary, section 2 part A item 2: sink tokens are
//   updated from recent visual context): the sink slots receive copies of the most recently appended frames.
// * Noise controller (review page section 三 / technical summary section 2 part A item 3): a monotone map from the
//   per-frame motion magnitude to a noise rate, with optional exponential smoothing.
//
// All three are HBM- or latency-bound and tiny next to attention; they use 16-byte vectors
// where they move data.
#include <cuda_bf16.h>

#include "internal.h"

namespace sdv2 {
namespace {

__device__ __forceinline__ uint32_t rotate_pair_rr(uint32_t xy, float c, float s)
{
    const float x = __uint_as_float(xy << 16);
    const float y = __uint_as_float(xy & 0xFFFF0000u);
    const float xr = __fmaf_rn(x, c, -__fmul_rn(y, s));
    const float yr = __fmaf_rn(x, s, __fmul_rn(y, c));
    const __nv_bfloat162 o = __floats2bfloat162_rn(xr, yr);
    return *reinterpret_cast<const uint32_t*>(&o);
}

// Re-rotation.  Grid: z = stream * W + window slot, y = head, x covers the slot's rows.  Only
// the time segment of each 256-byte key row moves: its first tvecs 16-byte vectors.  The block's
// lanes are laid out as (row, vector < tvecs) -- 256 / tvecs rows per pass, every lane but the
// remainder holding a live vector -- so a warp covers consecutive rows' time segments; each
// thread takes kRerotRowsPerThread rows, all loads issued before any rotation.  A slot
// qualifies when it holds a frame of an earlier chunk (0 <= frame_id < c*F) of a stream whose
// current chunk is a refresh chunk.  The rows of one (stream, head, slot) are contiguous.
constexpr int kRerotRowsPerThread = 4;
constexpr int kRerotThreads = 256;

__global__ void __launch_bounds__(kRerotThreads) rerotate_kernel(const __grid_constant__ RerotateParams p)
{
    const int b = blockIdx.z / p.W;
    const int ws = blockIdx.z - b * p.W;                        // window slot index 0..W-1
    const int h = blockIdx.y;
    if (!p.active[b]) return;
    const int slot = p.Fs + ws;
    sdv2_slot_meta* m = p.meta + static_cast<int64_t>(b) * p.nslots + slot;
    const int64_t fid = m->frame_id;
    if (fid < 0 || fid >= p.limit[b]) return;
    // the slot's time index moves even when the time segment is empty (rope_t = 0)
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) m->tpos -= p.shift;   // frame_id, which the others read, stays
    if (p.tvecs == 0) return;
    const int rows_per_pass = kRerotThreads / p.tvecs;
    const int lrow = static_cast<int>(threadIdx.x) / p.tvecs;
    const int vec = static_cast<int>(threadIdx.x) - lrow * p.tvecs;
    if (lrow >= rows_per_pass) return;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * rows_per_pass * kRerotRowsPerThread + lrow;
    uint4* base = reinterpret_cast<uint4*>(p.k_cache + ((static_cast<int64_t>(b) * p.H + h) * p.nslots * p.HW +
                                                        static_cast<int64_t>(slot) * p.HW) * 128) + vec;
    float c[4], s[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int pr = min(vec * 4 + u, p.tp - 1);
        c[u] = p.cs[pr].x;
        s[u] = p.cs[pr].y;
    }
    uint4 v[kRerotRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRerotRowsPerThread; ++k) {
        const int64_t row = row0 + static_cast<int64_t>(k) * rows_per_pass;
        if (row < p.HW) v[k] = base[row * 16];
    }
#pragma unroll
    for (int k = 0; k < kRerotRowsPerThread; ++k) {
        const int64_t row = row0 + static_cast<int64_t>(k) * rows_per_pass;
        if (row < p.HW) {
            uint32_t* w = reinterpret_cast<uint32_t*>(&v[k]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (vec * 4 + u < p.tp) w[u] = rotate_pair_rr(w[u], c[u], s[u]);
            base[row * 16] = v[k];
        }
    }
}

// Sink update.  Grid: z = stream * F_s + sink slot, y = head, x covers the slot's HW * 16
// vectors of k and of v (contiguous for one (stream, head, slot)); each thread copies eight
// vectors of each, all sixteen loads issued before the first store.  The first thread of each slot copies
// the metadata.
constexpr int kSinkVecsPerThread = 8;
__global__ void __launch_bounds__(256) sink_update_kernel(const __grid_constant__ SinkUpdateParams p)
{
    const int b = blockIdx.z / p.Fs;
    const int s = blockIdx.z - b * p.Fs;
    const int h = blockIdx.y;
    if (!p.active[b]) return;
    const int src = p.src_slot[b * kMaxSinkFrames + s];
    const int64_t head_base = (static_cast<int64_t>(b) * p.H + h) * p.nslots * p.HW;
    const uint4* kf = reinterpret_cast<const uint4*>(p.k_cache) + (head_base + static_cast<int64_t>(src) * p.HW) * 16;
    const uint4* vf = reinterpret_cast<const uint4*>(p.v_cache) + (head_base + static_cast<int64_t>(src) * p.HW) * 16;
    uint4* kt = reinterpret_cast<uint4*>(p.k_cache) + (head_base + static_cast<int64_t>(s) * p.HW) * 16;
    uint4* vt = reinterpret_cast<uint4*>(p.v_cache) + (head_base + static_cast<int64_t>(s) * p.HW) * 16;
    const int64_t n = static_cast<int64_t>(p.HW) * 16;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (256 * kSinkVecsPerThread) + threadIdx.x;
    uint4 kv[kSinkVecsPerThread], vv[kSinkVecsPerThread];
#pragma unroll
    for (int u = 0; u < kSinkVecsPerThread; ++u) {
        const int64_t i = i0 + u * 256;
        if (i < n) {
            kv[u] = kf[i];
            vv[u] = vf[i];
        }
    }
#pragma unroll
    for (int u = 0; u < kSinkVecsPerThread; ++u) {
        const int64_t i = i0 + u * 256;
        if (i < n) {
            kt[i] = kv[u];
            vt[i] = vv[u];
        }
    }
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0)
        p.meta[static_cast<int64_t>(b) * p.nslots + s] = p.meta[static_cast<int64_t>(b) * p.nslots + src];
}

// One block per stream: the block stages up to kNoiseTile motion values in shared memory, one
// thread walks them in order (the smoothing is a sequential recurrence, kept in the oracle's
// order and rounding), and the block writes the rates back.
constexpr int kNoiseThreads = 256;
constexpr int kNoiseTile = 4096;

__global__ void __launch_bounds__(kNoiseThreads) noise_kernel(const __grid_constant__ NoiseParams p)
{
    __shared__ float buf[kNoiseTile];
    __shared__ float carry;
    const int b = blockIdx.x;
    if (threadIdx.x == 0) carry = p.state ? p.state[b] : -1.0f;
    const float* m = p.m + static_cast<int64_t>(b) * p.T;
    float* rate = p.rate + static_cast<int64_t>(b) * p.T;
    for (int64_t t0 = 0; t0 < p.T; t0 += kNoiseTile) {
        const int n = static_cast<int>((p.T - t0 < kNoiseTile) ? (p.T - t0) : kNoiseTile);
        for (int i = threadIdx.x; i < n; i += kNoiseThreads) buf[i] = m[t0 + i];
        __syncthreads();
        if (threadIdx.x == 0) {
            float state = carry;
            for (int i = 0; i < n; ++i) {
                float u = (buf[i] - p.m_lo) / (p.m_hi - p.m_lo);
                u = fminf(fmaxf(u, 0.0f), 1.0f);
                if (!p.more_noise_when_fast) u = 1.0f - u;
                const float r = __fmaf_rn(p.out_hi - p.out_lo, u, p.out_lo);
                state = (state < 0.0f) ? r : __fmaf_rn(p.ema, state - r, r);   // ema*state + (1-ema)*r
                buf[i] = state;
            }
            carry = state;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kNoiseThreads) rate[t0 + i] = buf[i];
        __syncthreads();
    }
    if (threadIdx.x == 0 && p.state) p.state[b] = carry;
}

}  // namespace

cudaError_t launch_rerotate(const RerotateParams& p, cudaStream_t s)
{
    if (p.B == 0 || p.W == 0 || p.HW == 0 || p.H == 0) return cudaSuccess;   // an empty time segment still moves tpos
    const int rows_per_block = (p.tvecs > 0 ? kRerotThreads / p.tvecs : kRerotThreads) * kRerotRowsPerThread;
    const dim3 grid(static_cast<unsigned>((p.HW + rows_per_block - 1) / rows_per_block), static_cast<unsigned>(p.H),
                    static_cast<unsigned>(p.B * p.W));
    rerotate_kernel<<<grid, kRerotThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sink_update(const SinkUpdateParams& p, cudaStream_t s)
{
    if (p.B == 0 || p.Fs == 0 || p.HW == 0 || p.H == 0) return cudaSuccess;
    const int per_block = 256 * kSinkVecsPerThread;
    const dim3 grid(static_cast<unsigned>((static_cast<int64_t>(p.HW) * 16 + per_block - 1) / per_block), static_cast<unsigned>(p.H),
                    static_cast<unsigned>(p.B * p.Fs));
    sink_update_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_noise(const NoiseParams& p, cudaStream_t s)
{
    noise_kernel<<<p.B, kNoiseThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sdv2
