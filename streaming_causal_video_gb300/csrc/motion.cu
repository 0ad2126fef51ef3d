// Motion magnitude of adjacent frames: exact squared L2 distance of uint8 frames.
//
// "StreamDiffusionV2" review page, section 二 (table of innovations: L2 motion estimate ->
// adaptive noise rate) and section 三 (motion-aware noise controller: compute the motion
// magnitude of adjacent frames).  The technical summary (section 2 part A item 3) mentions optical flow as one way of
// estimating the motion strength; the raw pixel L2 distance is the plain reading of "L2".
//
// Work split: each block owns a slab of 16-byte vectors of the frame and a run of consecutive
// frame pairs; a thread keeps its vectors of frame t in registers while it reads frame t+1, so
// every frame is read from HBM once per run (runs are as long as the grid size allows).  Per pair: |a-b| per byte (vabsdiffu4) and the
// 4-way dot product with itself (dp4a) accumulate in 32 bits, then a block reduction and one
// 64-bit atomic add per block and pair.
#include <algorithm>

#include "internal.h"

namespace sdv2 {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int kMaxFramesPerRun = 32;

__device__ __forceinline__ uint32_t ssd16(uint4 a, uint4 b, uint32_t acc)
{
    uint32_t d;
    d = __vabsdiffu4(a.x, b.x); acc = __dp4a(d, d, acc);
    d = __vabsdiffu4(a.y, b.y); acc = __dp4a(d, d, acc);
    d = __vabsdiffu4(a.z, b.z); acc = __dp4a(d, d, acc);
    d = __vabsdiffu4(a.w, b.w); acc = __dp4a(d, d, acc);
    return acc;
}

__global__ void motion_zero_kernel(uint64_t* ssd, int64_t n)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) ssd[i] = 0;
}

// grid: x = slabs of kThreads*kVecPerThread vectors, y = stream * runs + run; a run covers
// `fpr` consecutive frame pairs.
__global__ void __launch_bounds__(kThreads) motion_ssd_kernel(const uint4* __restrict__ frames, int64_t vecs,
                                                              int64_t T, int runs, int fpr, uint64_t* __restrict__ ssd)
{
    const int b = blockIdx.y / runs;
    const int run = blockIdx.y - b * runs;
    const int64_t t0 = static_cast<int64_t>(run) * fpr;
    if (t0 >= T) return;
    const int64_t t1 = min(T, t0 + fpr);
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads * kVecPerThread + threadIdx.x;
    const uint4* f = frames + static_cast<int64_t>(b) * (T + 1) * vecs;

    uint4 prev[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        const int64_t i = base + u * kThreads;
        prev[u] = (i < vecs) ? __ldcs(f + t0 * vecs + i) : make_uint4(0, 0, 0, 0);
    }
    __shared__ unsigned long long warp_sums[kThreads / 32];
    for (int64_t t = t0; t < t1; ++t) {
        uint32_t acc = 0;
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t i = base + u * kThreads;
            const uint4 cur = (i < vecs) ? __ldcs(f + (t + 1) * vecs + i) : make_uint4(0, 0, 0, 0);
            acc = ssd16(cur, prev[u], acc);
            prev[u] = cur;
        }
        // 32 lanes * 4 vectors * 16 bytes * 255^2 < 2^32: the warp sum fits in 32 bits.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long s = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) s += warp_sums[w];
            atomicAdd(reinterpret_cast<unsigned long long*>(ssd) + static_cast<int64_t>(b) * T + t, s);
        }
        __syncthreads();
    }
}

// m = sqrt(ssd / npix): an IEEE fp64 quotient and square root (both correctly rounded), then
// one rounding to fp32.
__global__ void motion_rms_kernel(const uint64_t* ssd, float* m, int64_t n, double npix)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) m[i] = static_cast<float>(sqrt(static_cast<double>(ssd[i]) / npix));
}

}  // namespace

cudaError_t launch_motion_l2(const uint8_t* frames, int B, int64_t T, int64_t frame_bytes, uint64_t* ssd,
                             float* m, cudaStream_t s)
{
    const int64_t n = static_cast<int64_t>(B) * T;
    motion_zero_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(ssd, n);
    const int64_t vecs = frame_bytes / 16;
    const int64_t slabs = (vecs + kThreads * kVecPerThread - 1) / (kThreads * kVecPerThread);
    // Frames per run: long runs read each frame once, short runs give more blocks; aim for at
    // least four blocks per SM (a run's first frame is read twice, from L2 when runs are short).
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = static_cast<int64_t>(B) * slabs * T / (4 * static_cast<int64_t>(sms));
    const int fpr = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxFramesPerRun, want)));
    const int runs = static_cast<int>((T + fpr - 1) / fpr);
    dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(B * runs));
    motion_ssd_kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(frames), vecs, T, runs, fpr, ssd);
    if (m) {
        motion_rms_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(ssd, m, n,
                                                                               static_cast<double>(frame_bytes));
    }
    return cudaGetLastError();
}

}  // namespace sdv2
