// Cache maintenance at RoPE-refresh time, and the motion-driven noise controller.
//
// * Re-rotation of the window keys (the second reading of "RoPE refresh" on the
//   "StreamDiffusionV2" review page, section 三, "periodically reset the positional-encoding
//   offset"): when the time offset resets by F*R, the keys already in the rolling window are
//   turned back by the same F*R on the time axis, so that distances between the new chunk and
//   the window stay what they were (positions stay continuous across the reset).
// * Sink update ("StreamDiffusionV2" gist summary 2.A.2: sink tokens are updated from recent
//   visual context): the sink slots receive copies of the most recently appended frames.
// * Noise controller (review page section 三 / gist summary 2.A.3): a monotone map from the
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

// One thread per (stream, window slot, token of the frame, head, 16-byte vector of the time
// segment).  A slot qualifies when it holds a frame of an earlier chunk (0 <= frame_id < c*F)
// of a stream whose current chunk is a refresh chunk.
__global__ void rerotate_kernel(const __grid_constant__ RerotateParams p)
{
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t per_slot = static_cast<int64_t>(p.HW) * p.H * p.tvecs;
    const int64_t per_stream = per_slot * p.W;
    if (gid >= per_stream * p.B) return;
    const int b = static_cast<int>(gid / per_stream);
    const int64_t rem = gid - static_cast<int64_t>(b) * per_stream;
    const int ws = static_cast<int>(rem / per_slot);            // window slot index 0..W-1
    const int64_t r2 = rem - static_cast<int64_t>(ws) * per_slot;
    const int vec = static_cast<int>(r2 % p.tvecs);
    const int64_t r3 = r2 / p.tvecs;
    const int h = static_cast<int>(r3 % p.H);
    const int tok = static_cast<int>(r3 / p.H);
    if (!p.active[b]) return;
    const int slot = p.Fs + ws;
    sdv2_slot_meta* m = p.meta + static_cast<int64_t>(b) * p.nslots + slot;
    const int64_t fid = m->frame_id;
    if (fid < 0 || fid >= p.limit[b]) return;
    uint4* row = reinterpret_cast<uint4*>(
        p.k_cache + ((static_cast<int64_t>(b) * p.H + h) * p.nslots * p.HW + static_cast<int64_t>(slot) * p.HW + tok) * 128);
    uint4 v = row[vec];
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int pr = vec * 4 + u;
        if (pr < p.tp) w[u] = rotate_pair_rr(w[u], p.cs[pr].x, p.cs[pr].y);
    }
    row[vec] = v;
    if (tok == 0 && h == 0 && vec == 0) m->tpos -= p.shift;   // frame_id, which the others read, stays
}

// One thread per (stream, sink slot, token, head, 16-byte vector) copies k and v rows; the
// first thread of each slot copies the metadata.
__global__ void sink_update_kernel(const __grid_constant__ SinkUpdateParams p)
{
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t per_slot = static_cast<int64_t>(p.HW) * p.H * 16;
    const int64_t per_stream = per_slot * p.Fs;
    if (gid >= per_stream * p.B) return;
    const int b = static_cast<int>(gid / per_stream);
    if (!p.active[b]) return;
    const int64_t rem = gid - static_cast<int64_t>(b) * per_stream;
    const int s = static_cast<int>(rem / per_slot);
    const int64_t r2 = rem - static_cast<int64_t>(s) * per_slot;
    const int vec = static_cast<int>(r2 & 15);
    const int64_t r3 = r2 >> 4;
    const int h = static_cast<int>(r3 % p.H);
    const int tok = static_cast<int>(r3 / p.H);
    const int src = p.src_slot[b * kMaxSinkFrames + s];
    const int64_t head_base = (static_cast<int64_t>(b) * p.H + h) * p.nslots * p.HW;
    const int64_t from = (head_base + static_cast<int64_t>(src) * p.HW + tok) * 16 + vec;
    const int64_t to = (head_base + static_cast<int64_t>(s) * p.HW + tok) * 16 + vec;
    reinterpret_cast<uint4*>(p.k_cache)[to] = reinterpret_cast<const uint4*>(p.k_cache)[from];
    reinterpret_cast<uint4*>(p.v_cache)[to] = reinterpret_cast<const uint4*>(p.v_cache)[from];
    if (tok == 0 && h == 0 && vec == 0)
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
    const int64_t n = static_cast<int64_t>(p.B) * p.W * p.HW * p.H * p.tvecs;
    if (n == 0) return cudaSuccess;
    rerotate_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sink_update(const SinkUpdateParams& p, cudaStream_t s)
{
    const int64_t n = static_cast<int64_t>(p.B) * p.Fs * p.HW * p.H * 16;
    if (n == 0) return cudaSuccess;
    sink_update_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_noise(const NoiseParams& p, cudaStream_t s)
{
    noise_kernel<<<p.B, kNoiseThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sdv2
