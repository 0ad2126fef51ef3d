// Causal-RoPE + sink/ring KV-cache append (one HBM pass over the chunk's q, k, v).
//
// Rotary embedding over (t, h, w) with a locally computed global time index: "Accelerating
// Video Generation Inference with Sequential-Parallel 3D Positional Encoding Using a Global Time
// Index", technical summary 2(나) (positions from each block's start frame) and 2(다) (cos/sin
// precomputed into contiguous tables, fused with the projection epilogue in the page's design).
// Cache layout and eviction: "StreamDiffusionV2" review page, section 三 (sink token guided
// rolling KV cache).
//
// Work split: one thread per (stream, token, 16-byte vector of the head) -- 8 bf16 = 4 rotation
// pairs -- looping over all heads, so that the 4 (cos, sin) pairs are looked up once and used
// 2*H times.  Reads and writes are 16-byte vectors; a warp covers two tokens' 256-byte head
// rows, so every access is a full 32-byte sector.
#include <cuda_bf16.h>

#include "internal.h"

namespace sdv2 {
namespace {

constexpr int kVecs = 16;       // 16-byte vectors per 128-dim bf16 head row
constexpr int kThreads = 256;   // 16 tokens per block
constexpr int kHeadBatch = 3;   // heads whose loads are issued together (two batches in flight)

__device__ __forceinline__ uint32_t rotate_pair(uint32_t xy, float c, float s)
{
    // Low half = element 2j (x), high half = element 2j+1 (y).
    const float x = __uint_as_float(xy << 16);
    const float y = __uint_as_float(xy & 0xFFFF0000u);
    const float xr = __fmaf_rn(x, c, -__fmul_rn(y, s));
    const float yr = __fmaf_rn(x, s, __fmul_rn(y, c));
    const __nv_bfloat162 o = __floats2bfloat162_rn(xr, yr);   // .x (low) = xr
    return *reinterpret_cast<const uint32_t*>(&o);
}

__device__ __forceinline__ uint4 rotate_vec(uint4 a, const float (&c)[4], const float (&s)[4])
{
    uint4 r;
    r.x = rotate_pair(a.x, c[0], s[0]);
    r.y = rotate_pair(a.y, c[1], s[1]);
    r.z = rotate_pair(a.z, c[2], s[2]);
    r.w = rotate_pair(a.w, c[3], s[3]);
    return r;
}

__global__ void __launch_bounds__(kThreads, 2) rope_append_kernel(const __grid_constant__ RopeAppendParams p)
{
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int vec = static_cast<int>(gid & (kVecs - 1));
    const int64_t tok = gid >> 4;                      // over B * Nq
    if (tok >= static_cast<int64_t>(p.B) * p.Nq) return;
    const int b = static_cast<int>(tok / p.Nq);
    const int n = static_cast<int>(tok - static_cast<int64_t>(b) * p.Nq);
    const int64_t src = static_cast<int64_t>(b) * p.Nq * p.tok_stride + static_cast<int64_t>(n) * p.tok_stride
                        + vec * 8;
    const uint4* __restrict__ q = reinterpret_cast<const uint4*>(p.q + src);
    const uint4* __restrict__ k = reinterpret_cast<const uint4*>(p.k + src);
    const uint4* __restrict__ v = reinterpret_cast<const uint4*>(p.v + src);

    // The first heads' loads go out before anything else, so that the table lookups below run
    // while they are in flight; afterwards each batch's loads are issued before the previous
    // batch is rotated and stored.
    uint4 qa[kHeadBatch], ka[kHeadBatch], va[kHeadBatch];
#pragma unroll
    for (int u = 0; u < kHeadBatch; ++u) {
        if (u < p.H) {
            qa[u] = __ldg(q + u * kVecs);
            ka[u] = __ldg(k + u * kVecs);
            va[u] = __ldg(v + u * kVecs);
        }
    }

    const int i = n / p.HW;                            // frame of the chunk
    const int r = n - i * p.HW;                        // token inside the frame
    const int gh = r / p.grid_w;
    const int gw = r - gh * p.grid_w;
    const int fr = b * p.F + i;
    const FrameDesc fd = p.frames[fr];

    // (cos, sin) of this thread's 4 pairs: pair index 4*vec + u across the t, h, w segments; the
    // table is picked by a select on its address, so that the 4 loads issue together.
    float c[4], s[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int pr = vec * 4 + u;
        const float2* src_t = &p.tcs[fr * p.tp + pr];
        const float2* src_h = p.h_tab + gh * p.hp + (pr - p.tp);
        const float2* src_w = p.w_tab + gw * p.wp + (pr - p.tp - p.hp);
        const float2* cs_ptr = pr < p.tp ? src_t : (pr < p.tp + p.hp ? src_h : src_w);
        const float2 cs = *cs_ptr;
        c[u] = cs.x;
        s[u] = cs.y;
    }

    const int64_t rows = static_cast<int64_t>(p.nslots) * p.HW;
    const int64_t crow = static_cast<int64_t>(fd.slot) * p.HW + r;
    for (int h0 = 0; h0 < p.H; h0 += kHeadBatch) {
        const int nh = min(kHeadBatch, p.H - h0);
        uint4 qr[kHeadBatch], kr[kHeadBatch], vr[kHeadBatch];
#pragma unroll
        for (int u = 0; u < kHeadBatch; ++u) {
            qr[u] = qa[u];
            kr[u] = ka[u];
            vr[u] = va[u];
        }
        const int h1 = h0 + kHeadBatch;                // next batch: loads issued now
#pragma unroll
        for (int u = 0; u < kHeadBatch; ++u) {
            if (h1 + u < p.H) {
                qa[u] = __ldg(q + (h1 + u) * kVecs);
                ka[u] = __ldg(k + (h1 + u) * kVecs);
                va[u] = __ldg(v + (h1 + u) * kVecs);
            }
        }
#pragma unroll
        for (int u = 0; u < kHeadBatch; ++u) {
            if (u < nh) {
                const int64_t bh = static_cast<int64_t>(b) * p.H + h0 + u;
                uint4* qo = reinterpret_cast<uint4*>(p.q_rot + (bh * p.Nq + n) * 128) + vec;
                uint4* ko = reinterpret_cast<uint4*>(p.k_cache + (bh * rows + crow) * 128) + vec;
                uint4* vo = reinterpret_cast<uint4*>(p.v_cache + (bh * rows + crow) * 128) + vec;
                *qo = rotate_vec(qr[u], c, s);
                *ko = rotate_vec(kr[u], c, s);
                *vo = vr[u];
            }
        }
    }

    if (r == 0 && vec == 0) {
        sdv2_slot_meta m;
        m.frame_id = fd.frame;
        m.tpos = fd.tpos;
        p.meta[static_cast<int64_t>(b) * p.nslots + fd.slot] = m;
    }
}

__global__ void cache_reset_kernel(uint4* k, uint4* v, int64_t nvec, sdv2_slot_meta* meta, int64_t nmeta)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        k[i] = z;
        v[i] = z;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nmeta; i += stride) {
        meta[i].frame_id = -1;
        meta[i].tpos = 0;
    }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t s)
{
    const int64_t threads = static_cast<int64_t>(p.B) * p.Nq * kVecs;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    rope_append_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cache_reset(uint16_t* k, uint16_t* v, size_t cache_bytes, sdv2_slot_meta* meta,
                               int64_t nmeta, cudaStream_t s)
{
    const int64_t nvec = static_cast<int64_t>(cache_bytes / 16);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache_reset_kernel<<<sms * 8, 256, 0, s>>>(reinterpret_cast<uint4*>(k), reinterpret_cast<uint4*>(v),
                                               nvec, meta, nmeta);
    return cudaGetLastError();
}

}  // namespace sdv2
