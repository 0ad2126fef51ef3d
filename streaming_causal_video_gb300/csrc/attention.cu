// Chunk attention on the 5th-generation tensor cores (tcgen05 + tensor memory) of sm_103a.
//
// What it computes: the chunk's queries attend, with no mask, to every valid row of the layer's
// KV cache -- the sink frames, the rolling window and the chunk itself -- which is the
// chunk-causal attention of a Self-Forcing-style autoregressive video DiT ("Accelerating Video
// Generation Inference with Sequential-Parallel 3D Positional Encoding Using a Global Time
// Index", technical summary sections 1 and 2(가): causal autoregressive generation with KV
// caching; "StreamDiffusionV2" review page, section 三: sink tokens + rolling KV cache).
//   out[b, n, h, :] = sum_j softmax_j(scale * q_rot[b, h, n, :] . k[b, h, j, :]) v[b, h, j, :]
//
// How (one CTA = one head of one stream, two 128-row query tiles and one key split):
//   warps 8, 10 (TMA): Q tiles once, then K (warp 8, 3-stage ring) and V (warp 10, 2-stage ring)
//                       tiles of 128 keys.  The CTAs of one head walk the same keys at about the
//                       same time, so most tiles come from L2 (explicit L2 prefetches measured
//                       slower).  3D tensor maps per stream clip the key range at the valid
//                       prefix, so rows past it arrive as zeros; 128-byte swizzled boxes of 64
//                       dims.
//   warp 9 (MMA)      : runs converged: every lane polls each barrier and a warp vote agrees on
//                       the outcome; an elected lane issues each tcgen05.mma.  S_t = Q_t K^T
//                       (A and B from shared memory, K-major) into tensor memory;
//                       O_t += P_t V (A = P from tensor memory, B = V from shared memory,
//                       MN-major).  Completion is signalled with tcgen05.commit on mbarriers.
//                       Descriptors are built once and advanced by constants, because the
//                       issuing warp's own instruction latency between MMAs, not the tensor core,
//                       is what limits a single MMA stream of 128x128x16 steps.
//   warps 0-3, 4-7    : one softmax warpgroup per query tile; thread = query row = TMEM lane.
//                       Online softmax in fp32 with a lazily updated running max (the output
//                       accumulator in tensor memory is rescaled only when the max grows by more
//                       than 2^8), P written back into the S columns as packed bf16.
// Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1, 128 fp32 columns each.
// The two tiles ping-pong: while one warpgroup turns S_t into P_t, the tensor core runs the
// other tile's PV and next QK^T.  Because tcgen05 operations issued by one thread complete in
// order and a commit covers all earlier ones, the arrival of S_t(j) also proves that
// O_t += P_t(j-1) V(j-1) has finished, so O_t can be rescaled without another barrier.
//
// With several key splits, each split takes a ticket when its main loop is done.  All but the
// last publish their unnormalised rows and (max, sum) to the workspace, stored as
// [dims/4][row][4] floats so that a warp moves 512 contiguous bytes, and count themselves as
// published; the last merges them with its own rows, still in tensor memory, after a bounded
// wait for that count (the splits it waits for are already running their epilogues).
//
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel records kErrTimeout in
// the workspace error word, tells the other roles to stop, drains its own copies and MMAs and
// frees its tensor memory before returning.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace sdv2 {
namespace {

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per KV tile
constexpr int HD = 128;                 // head dim
constexpr int NQT = 2;                  // query tiles per CTA
constexpr int KST = 3;                  // K stages
constexpr int VST = 2;                  // V stages
constexpr uint32_t TILE = BM * HD * 2;  // 32 KB
constexpr uint32_t HALF = TILE / 2;     // one 64-dim box: 128 rows x 128 bytes
constexpr int TMA_WARP = 4 * NQT;        // Q and K tiles
constexpr int MMA_WARP = 4 * NQT + 1;    // MMA issue (also allocates tensor memory)
constexpr int TMA_V_WARP = 4 * NQT + 2;  // V tiles
constexpr int NTHREADS = (4 * NQT + 3) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kFastSumBound = 256.0f;     // 2^kRescaleThreshold: largest row sum the optimistic pass accepts
constexpr float kLn2 = 0.6931471805599453f;

// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_KEMPTY = B_KFULL + KST;
constexpr int B_VFULL = B_KEMPTY + KST;
constexpr int B_VEMPTY = B_VFULL + VST;
constexpr int B_SFULL = B_VEMPTY + VST;
constexpr int B_PFULL = B_SFULL + NQT;
constexpr int B_OFULL = B_PFULL + NQT;
constexpr int B_MMADONE = B_OFULL + NQT;
constexpr int NBARS = B_MMADONE + 1;

constexpr uint32_t SMEM_TILES = (NQT + KST + VST) * TILE;
constexpr uint32_t SMEM_BYTES = SMEM_TILES + 1024 /* barriers, flags */ + 1024 /* alignment */;

__device__ __forceinline__ uint32_t s_col(int t) { return static_cast<uint32_t>(t * 128); }
__device__ __forceinline__ uint32_t o_col(int t) { return static_cast<uint32_t>((NQT + t) * 128); }

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, uint32_t* err)
{
    *abort_flag = 1;
    atomicOr(err, kErrTimeout);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Work unit (blockIdx.x) -> (item, key split, splits of the item).  Items are (stream, head,
// query pair) in that order; the first p.full_items run whole (one unit each, dispatched first),
// every later item is cut into p.splits key ranges.
__device__ __forceinline__ void decode_unit(const AttnParams& p, int& item, int& sp, int& nsp)
{
    const int unit = blockIdx.x;
    if (unit < p.full_items) {
        item = unit;
        sp = 0;
        nsp = 1;
    } else {
        const int u = unit - p.full_items;
        item = p.full_items + u / p.splits;
        sp = u - (u / p.splits) * p.splits;
        nsp = p.splits;
    }
}

__global__ void __launch_bounds__(NTHREADS, 1) chunk_attention_kernel(const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + NQT * TILE;
    const uint32_t sV = sK + KST * TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_TILES);
    const uint32_t bar0 = smem_u32(bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
#define BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
    const int lane = threadIdx.x & 31;
    int item_i, sp, nsp;
    decode_unit(p, item_i, sp, nsp);
    // the epilogue reads the unit back from shared memory rather than keeping it in registers
    volatile int* unit_info = reinterpret_cast<volatile int*>(tmem_slot + 4);
    if (threadIdx.x == 0) {
        unit_info[0] = item_i;
        unit_info[1] = sp;
        unit_info[2] = nsp;
    }
    const int qp = item_i % p.qpairs;               // query pair (256 rows)
    const int h = (item_i / p.qpairs) % p.H;
    const int b = item_i / (p.qpairs * p.H);
    const int nkv = p.nkv[b];
    const int tiles_all = (nkv + BN - 1) / BN;
    const int t_begin = static_cast<int>(static_cast<int64_t>(sp) * tiles_all / nsp);
    const int ntiles = static_cast<int>(static_cast<int64_t>(sp + 1) * tiles_all / nsp) - t_begin;
    const int q0 = qp * (BM * NQT);
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int i = 0; i < KST; ++i) { mbar_init(BAR(B_KFULL + i), 1); mbar_init(BAR(B_KEMPTY + i), 1); }
        for (int i = 0; i < VST; ++i) { mbar_init(BAR(B_VFULL + i), 1); mbar_init(BAR(B_VEMPTY + i), 1); }
        for (int t = 0; t < NQT; ++t) {
            mbar_init(BAR(B_SFULL + t), 1);
            mbar_init(BAR(B_PFULL + t), 128);
            mbar_init(BAR(B_OFULL + t), 1);
        }
        mbar_init(BAR(B_MMADONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == TMA_WARP || warp == TMA_V_WARP) {
        // ------------------------------------------------------------------ producers (TMA)
        // One thread loads Q and the K ring, another the V ring, so that a late K slot never
        // holds back a V load.
        if (lane == 0) {
            const bool is_k = (warp == TMA_WARP);
            const CUtensorMap* map = is_k ? &p.kmap[b] : &p.vmap[b];
            tma_prefetch_desc(map);
            const uint32_t s_ring = is_k ? sK : sV;
            const int bar_full = is_k ? B_KFULL : B_VFULL;
            const int bar_empty = is_k ? B_KEMPTY : B_VEMPTY;
            const int nst = is_k ? KST : VST;
            constexpr int NST = KST > VST ? KST : VST;
            if (is_k) {
                const CUtensorMap* qm = &p.qmap;
                tma_prefetch_desc(qm);
                const int plane = b * p.H + h;
                mbar_arrive_expect_tx(BAR(B_QFULL), NQT * TILE);
                for (int t = 0; t < NQT; ++t)
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(sQ + t * TILE + hf * HALF, qm, BAR(B_QFULL), hf * 64, q0 + t * BM, plane);
            }
            int pend[NST] = {};
            uint32_t par[NST] = {};
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % nst;
                const uint32_t ph = static_cast<uint32_t>(j / nst) & 1u;
                if (!mbar_wait_bounded(BAR(bar_empty + st), ph ^ 1u, tmo, abort_flag)) { raise_abort(abort_flag, p.err); break; }
                const int jg = t_begin + j;
                if (jg != p.drop_tile) {
                    mbar_arrive_expect_tx(BAR(bar_full + st), TILE);
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(s_ring + st * TILE + hf * HALF, map, BAR(bar_full + st), hf * 64, jg * BN, h);
                    pend[st] = 1;
                    par[st] = ph;
                }
            }
            // Drain: every copy this thread started must land before the CTA may exit.
            volatile int no_abort = 0;
            if (is_k) mbar_wait_bounded(BAR(B_QFULL), 0, tmo, &no_abort);
            for (int i = 0; i < nst; ++i)
                if (pend[i]) mbar_wait_bounded(BAR(bar_full + i), par[i], tmo, &no_abort);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop converged: every lane polls each barrier and a warp
        // vote agrees on the outcome (cheaper than one lane polling while the others wait at a
        // shuffle), and one elected lane issues each tcgen05 instruction.  Shared-memory
        // descriptors are built once: the k-th 16-wide step of a K-major 128-byte-swizzled tile
        // starts (k/4)*HALF + (k%4)*32 bytes further, and V's k-th step 16 rows (2048 bytes)
        // further, which is a constant added to the descriptor's address field.
        constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);
        constexpr uint32_t idO = idesc_bf16_f32(BM, HD, true);
        const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dK = sdesc_sw128(sK, 16, 1024);
        const uint64_t dV = sdesc_sw128(sV, HALF, 1024);
        constexpr uint64_t kTileStep = TILE >> 4;           // descriptor units (16 bytes)
        auto wait = [&](int bar_idx, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(BAR(bar_idx), parity, tmo, abort_flag);
            return __all_sync(0xffffffffu, r);
        };
        auto issue_s = [&](int t, int ks) {
            const uint64_t a0 = dQ + static_cast<uint64_t>(t) * kTileStep;
            const uint64_t b0 = dK + static_cast<uint64_t>(ks) * kTileStep;
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
                const uint64_t o = static_cast<uint64_t>(((k >> 2) * HALF + (k & 3) * 32) >> 4);
                mma_ss_warp(tmem + s_col(t), a0 + o, b0 + o, idS, k > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int t, int vs, bool acc) {
            const uint64_t b0 = dV + static_cast<uint64_t>(vs) * kTileStep;
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                mma_ts_warp(tmem + o_col(t), tmem + s_col(t) + static_cast<uint32_t>(k) * 8u,
                            b0 + static_cast<uint64_t>(k) * (2048u >> 4), idO, (acc || k > 0) ? 1u : 0u);
        };
        bool ok = wait(B_QFULL, 0) && wait(B_KFULL + 0, 0);
        if (ok) {
            tc_fence_after();
            for (int t = 0; t < NQT; ++t) {
                issue_s(t, 0);
                mma_commit_warp(BAR(B_SFULL + t));
            }
            mma_commit_warp(BAR(B_KEMPTY + 0));
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            const int vs = j % VST;
            if (!wait(B_VFULL + vs, static_cast<uint32_t>(j / VST) & 1u)) { ok = false; break; }
            const bool more = j + 1 < ntiles;
            const int ks = (j + 1) % KST;
            for (int t = 0; t < NQT; ++t) {
                if (!wait(B_PFULL + t, static_cast<uint32_t>(j) & 1u)) { ok = false; break; }
                tc_fence_after();
                issue_pv(t, vs, j > 0);
                if (!more) mma_commit_warp(BAR(B_OFULL + t));
                if (more) {
                    if (t == 0 && !wait(B_KFULL + ks, static_cast<uint32_t>((j + 1) / KST) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(t, ks);
                    mma_commit_warp(BAR(B_SFULL + t));
                }
            }
            if (!ok) break;
            mma_commit_warp(BAR(B_VEMPTY + vs));
            if (more) mma_commit_warp(BAR(B_KEMPTY + ks));
        }
        if (!ok && lane == 0) raise_abort(abort_flag, p.err);
        // Drain: all MMAs issued by this warp complete before tensor memory is freed.
        mma_commit_warp(BAR(B_MMADONE));
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait_bounded(BAR(B_MMADONE), 0, tmo, &no_abort);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_base + s_col(t);
        const uint32_t tO = tmem + lane_base + o_col(t);
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!mbar_wait_bounded(BAR(B_SFULL + t), static_cast<uint32_t>(j) & 1u, tmo, abort_flag)) { ok = false; break; }
            tc_fence_after();
            uint32_t r[128];
            tmem_ld_x128_sync(tS, r);
            const int valid = nkv - (t_begin + j) * BN;      // > 0; < BN only on the last tile
            if (valid < BN) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= valid) r[i] = 0xFF800000u;       // -inf: masked key
            }
            const uint64_t sl2x2 = f32x2_pack(sl2, sl2);
            bool done = false;
            if (j > 0) {
                // Optimistic pass: the exponentials against the running max, without this tile's
                // max.  The running max is raised only when a tile's scores exceed it by more than
                // 2^8 (lazy rescale below), which is exactly when some term of the pass would exceed
                // 2^8; a row sum of at most 2^8 rules that out, and then the terms, the packed P and
                // the sum (same four chains, same order as the pass below) are what the max pass
                // would have produced.  Otherwise S, still intact in tensor memory, is loaded again
                // for the max pass.
                const uint64_t negm2 = f32x2_pack(-m_run, -m_run);
                uint64_t sum4[4];
#pragma unroll
                for (int a2 = 0; a2 < 4; ++a2) sum4[a2] = 0;
                uint32_t pk[2][32];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = hf * 64 + 2 * i;
                        const uint64_t x = ffma2(f32x2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sl2x2, negm2);
                        float x0, x1;
                        f32x2_unpack(x, x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        sum4[i & 3] = fadd2(sum4[i & 3], f32x2_pack(p0, p1));
                        pk[hf][i] = pack_bf16x2(p0, p1);
                    }
                }
                const uint64_t s01 = fadd2(sum4[0], sum4[1]), s23 = fadd2(sum4[2], sum4[3]);
                float lo, hi;
                f32x2_unpack(fadd2(s01, s23), lo, hi);
                const float s_tile = lo + hi;
                if (__all_sync(0xffffffffu, s_tile <= kFastSumBound)) {
                    tmem_st_x32(tS, pk[0]);
                    tmem_st_x32(tS + 32, pk[1]);
                    l_run += s_tile;
                    done = true;
                } else {
                    tmem_ld_x128_sync(tS, r);
                    if (valid < BN) {
#pragma unroll
                        for (int i = 0; i < 128; ++i)
                            if (i >= valid) r[i] = 0xFF800000u;
                    }
                }
            }
            if (!done) {
                // Row max of the raw scores (scale > 0 commutes with max): 8 independent chains of
                // three-input max, each over the 16 scores i = a (mod 8).
                float mx8[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    float m = fmax3(__uint_as_float(r[a]), __uint_as_float(r[a + 8]), __uint_as_float(r[a + 16]));
#pragma unroll
                    for (int i = 24; i < 120; i += 16)
                        m = fmax3(m, __uint_as_float(r[i + a]), __uint_as_float(r[i + 8 + a]));
                    mx8[a] = fmaxf(m, __uint_as_float(r[120 + a]));
                }
                const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                const float m_new = fmaxf(m_run, mx * sl2);
                const bool grow = m_new > m_run + kRescaleThreshold;
                if (__any_sync(0xffffffffu, grow)) {
                    const float f = grow ? ex2_approx(m_run - m_new) : 1.0f;
                    if (j > 0) {
                        // O_t is stable here: S_t(j) was committed after O_t += P_t(j-1) V(j-1).
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            tmem_ld_x32_sync(tO + c * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                            tmem_st_x32(tO + c * 32, o);
                        }
                    }
                    if (grow) {
                        l_run *= f;
                        m_run = m_new;
                    }
                }
                // p = 2^(s * scale * log2(e) - m): one packed FFMA per two scores, one MUFU.EX2 per
                // score; the row sum accumulates pairs with packed adds in 4 independent chains.
                const uint64_t negm2 = f32x2_pack(-m_run, -m_run);
                uint64_t sum4[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) sum4[a] = 0;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = hf * 64 + 2 * i;
                        const uint64_t x = ffma2(f32x2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sl2x2, negm2);
                        float x0, x1;
                        f32x2_unpack(x, x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        sum4[i & 3] = fadd2(sum4[i & 3], f32x2_pack(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st_x32(tS + hf * 32, pk);
                }
                {
                    const uint64_t s01 = fadd2(sum4[0], sum4[1]), s23 = fadd2(sum4[2], sum4[3]);
                    float lo, hi;
                    f32x2_unpack(fadd2(s01, s23), lo, hi);
                    l_run += lo + hi;
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(B_PFULL + t));
        }
        item_i = unit_info[0];                               // written by thread 0 before the first __syncthreads
        sp = unit_info[1];
        nsp = unit_info[2];
        const int64_t item = item_i;
        const int eb = item_i / (p.qpairs * p.H);            // stream, head, first query row again
        const int eh = (item_i / p.qpairs) % p.H;
        const int rloc = t * BM + row;                       // row inside the CTA's 256
        const int q = (item_i % p.qpairs) * (BM * NQT) + rloc;
        const int64_t pidx = item - p.full_items;            // split items: index of the partial rows
        if (ok && !mbar_wait_bounded(BAR(B_OFULL + t), 0, tmo, abort_flag)) ok = false;
        // warp-uniform from here on: the epilogue's tensor-memory loads are warp-collective
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) raise_abort(abort_flag, p.err);
        if (ok) tc_fence_after();
        if (nsp == 1) {
            if (ok) {
                const float inv = 1.0f / l_run;
                uint16_t* dst = p.out + ((static_cast<int64_t>(eb) * p.Nq + q) * p.H + eh) * HD;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld_x32_sync(tO + c * 32, o);
                    if (q < p.Nq) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                            d4[v] = w;
                        }
                    }
                }
                if (p.lse && q < p.Nq)
                    p.lse[(static_cast<int64_t>(eb) * p.H + eh) * p.Nq + q] = (m_run + __log2f(l_run)) * kLn2;
            }
        } else {
            // Split keys.  Each split takes a ticket once its main loop is done; the split with
            // the last ticket merges.  The others publish their unnormalised rows and (max, sum)
            // -- stored as [split item][HD/4][row][4] floats, so that a warp writes 512
            // contiguous bytes -- and then count themselves as published; the merger waits
            // (bounded) for that count and merges the published rows with its own, which stay in
            // tensor memory.  Every split the merger waits for has already taken its ticket, so
            // it is running and only has its stores left.
            int32_t* tickets = p.counters;
            int32_t* published = p.counters + static_cast<int64_t>(p.B) * p.H * p.qpairs;
            if (threadIdx.x == 0) {
                int last = 0;
                if (!*abort_flag) last = (atomicAdd(tickets + item, 1) == nsp - 1) ? 1 : 0;
                *last_flag = last;
            }
            named_bar_sync(1, 32 * 4 * NQT);
            if (!*last_flag) {
                if (ok) {
                    const int64_t slot = (pidx * nsp + sp) * kAttnRowsPerCta + rloc;
                    float4* po = reinterpret_cast<float4*>(p.part_o) + (pidx * nsp + sp) * (HD / 4) * kAttnRowsPerCta + rloc;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32_sync(tO + c * 32, o);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            __stcg(po + (c * 8 + v) * kAttnRowsPerCta,
                                   make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                               __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3])));
                    }
                    __stcg(reinterpret_cast<float2*>(p.part_ml) + slot, make_float2(m_run, l_run));
                }
                __threadfence();
                named_bar_sync(1, 32 * 4 * NQT);
                if (threadIdx.x == 0 && ok && !*abort_flag) atomicAdd(published + item, 1);
            } else {
                if (threadIdx.x == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (*reinterpret_cast<volatile int32_t*>(published + item) < nsp - 1) {
                        if (*abort_flag || globaltimer_ns() - t0 > tmo) {
                            raise_abort(abort_flag, p.err);
                            break;
                        }
                        __nanosleep(64);
                    }
                    // every other split is done with both counters: ready for the next call
                    tickets[item] = 0;
                    published[item] = 0;
                }
                named_bar_sync(1, 32 * 4 * NQT);
                __threadfence();
                if (ok && !*abort_flag) {
                    float ms[kMaxKvSplits], ls[kMaxKvSplits];
                    float M = m_run;
#pragma unroll
                    for (int s2 = 0; s2 < kMaxKvSplits; ++s2) {
                        if (s2 < nsp && s2 != sp) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) +
                                                     (pidx * nsp + s2) * kAttnRowsPerCta + rloc);
                            ms[s2] = ml.x;
                            ls[s2] = ml.y;
                            M = fmaxf(M, ml.x);
                        }
                    }
                    // Sums run over the splits in index order, with this split's own rows at its
                    // own place, so that the result does not depend on which split merges.
                    ms[sp & (kMaxKvSplits - 1)] = m_run;
                    ls[sp & (kMaxKvSplits - 1)] = l_run;
                    float L = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < kMaxKvSplits; ++s2)
                        if (s2 < nsp) {
                            ms[s2] = ex2_approx(ms[s2] - M);      // weight of split s2
                            L += ls[s2] * ms[s2];
                        }
                    const float inv = 1.0f / L;
                    uint16_t* dst = p.out + ((static_cast<int64_t>(eb) * p.Nq + q) * p.H + eh) * HD;
                    // 32 dims at a time: this split's own rows from tensor memory, the eight float4
                    // loads of each other split together
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        float4 acc[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                        for (int s2 = 0; s2 < nsp; ++s2) {
                            float4 u[8];
                            if (s2 == sp) {
                                uint32_t o[32];
                                tmem_ld_x32_sync(tO + c * 32, o);
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    u[v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                                       __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
                            } else {
                                const float4* src = reinterpret_cast<const float4*>(p.part_o) +
                                                    ((pidx * nsp + s2) * (HD / 4) + c * 8) * kAttnRowsPerCta + rloc;
#pragma unroll
                                for (int v = 0; v < 8; ++v) u[v] = __ldcg(src + v * kAttnRowsPerCta);
                            }
                            const float wgt = ms[s2 & (kMaxKvSplits - 1)];
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                acc[v].x += u[v].x * wgt; acc[v].y += u[v].y * wgt;
                                acc[v].z += u[v].z * wgt; acc[v].w += u[v].w * wgt;
                            }
                        }
                        if (q < p.Nq) {
#pragma unroll
                            for (int v = 0; v < 8; v += 2) {
                                uint4 wv;
                                wv.x = pack_bf16x2(acc[v].x * inv, acc[v].y * inv);
                                wv.y = pack_bf16x2(acc[v].z * inv, acc[v].w * inv);
                                wv.z = pack_bf16x2(acc[v + 1].x * inv, acc[v + 1].y * inv);
                                wv.w = pack_bf16x2(acc[v + 1].z * inv, acc[v + 1].w * inv);
                                *reinterpret_cast<uint4*>(dst + c * 32 + v * 4) = wv;
                            }
                        }
                    }
                    if (p.lse && q < p.Nq) p.lse[(static_cast<int64_t>(eb) * p.H + eh) * p.Nq + q] = (M + __log2f(L)) * kLn2;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
#undef BAR
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once; a function-local static is initialised by
// exactly one thread, so concurrent first calls from several host threads are safe.
EncodeTiledFn get_encode_tiled()
{
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return nullptr;
    }();
    return fn;
}

// (D = 128 dims, rows, planes) bf16 tensor with row stride 256 bytes; boxes of 64 dims x 128 rows.
bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t planes, int64_t plane_stride_bytes)
{
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD * 2), static_cast<cuuint64_t>(plane_stride_bytes)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BM), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

KvSchedule choose_kv_schedule(int64_t items, int min_tiles, int slots)
{
    // Estimated makespan in units of one item's key loop on one SM: k whole waves of unsplit
    // items, then the remaining items cut into s key ranges, in ceil(units / slots) waves of 1/s
    // each (2 % added per split phase for the partial writes and the merge).  Ties go to more
    // unsplit items, then to fewer splits.
    KvSchedule best{0, 1};
    double best_t = 1e300;
    const int64_t S = std::max(1, slots);
    for (int64_t k = 0; k * S <= items; ++k) {
        const int64_t rest = items - k * S;
        for (int sp = 1; sp <= kMaxKvSplits && sp <= std::max(1, min_tiles); ++sp) {
            if (rest == 0 && sp > 1) break;
            const double waves = std::ceil(static_cast<double>(rest) * sp / S);
            const double t = static_cast<double>(k) + waves / sp * (sp > 1 ? 1.02 : 1.0);
            if (t < best_t - 1e-9 || (std::fabs(t - best_t) <= 1e-9 && k * S > best.full_items)) {
                best_t = t;
                best.full_items = static_cast<int>(k * S);
                best.splits = sp;
            }
        }
    }
    if (best.splits == 1) best.full_items = static_cast<int>(items);   // nothing is split
    return best;
}

cudaError_t launch_chunk_attention(const uint16_t* q_rot, const uint16_t* k_cache, const uint16_t* v_cache, int B,
                                   int H, int Nq, int64_t rows_per_head, const int32_t* nkv, float scale,
                                   uint16_t* out, float* lse, const AttnScratch& ws, uint64_t timeout_ns,
                                   int64_t drop_tile, int force_splits, const KvSchedule* sched, cudaStream_t s,
                                   int* splits_used, const char** why)
{
    AttnParams p{};   // about 4.4 KB; passed by value as the launch's parameter block
    if (!encode_rows_map(&p.qmap, q_rot, Nq, static_cast<int64_t>(B) * H, static_cast<int64_t>(Nq) * HD * 2)) {
        *why = "cuTensorMapEncodeTiled failed for q_rot";
        return cudaErrorInvalidValue;
    }
    int min_tiles = 1 << 30;
    for (int b = 0; b < B; ++b) {
        const int64_t off = static_cast<int64_t>(b) * H * rows_per_head * HD;
        if (!encode_rows_map(&p.kmap[b], k_cache + off, nkv[b], H, rows_per_head * HD * 2) ||
            !encode_rows_map(&p.vmap[b], v_cache + off, nkv[b], H, rows_per_head * HD * 2)) {
            *why = "cuTensorMapEncodeTiled failed for the KV cache";
            return cudaErrorInvalidValue;
        }
        p.nkv[b] = nkv[b];
        min_tiles = std::min(min_tiles, (nkv[b] + BN - 1) / BN);
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    p.qpairs = (Nq + kAttnRowsPerCta - 1) / kAttnRowsPerCta;
    const int64_t items = static_cast<int64_t>(B) * H * p.qpairs;
    KvSchedule ks;
    if (sched) ks = *sched;
    else if (force_splits > 0) ks = KvSchedule{0, std::min(force_splits, std::min(kMaxKvSplits, min_tiles))};
    else ks = choose_kv_schedule(items, min_tiles, std::max(1, sms));
    if (ks.splits <= 1) ks = KvSchedule{static_cast<int>(std::min<int64_t>(items, INT32_MAX)), 1};
    const int64_t units = ks.full_items + (items - ks.full_items) * ks.splits;
    if (ks.full_items < 0 || ks.full_items > items || units > INT32_MAX) {
        *why = "too many attention work units (batch * heads * ceil(Nq/256) * splits must be < 2^31)";
        return cudaErrorInvalidConfiguration;
    }
    p.full_items = ks.full_items;
    p.splits = ks.splits;
    *splits_used = ks.splits;
    p.out = out;
    p.lse = lse;
    p.err = ws.err;
    p.counters = ws.counters;
    p.part_ml = ws.part_ml;
    p.part_o = ws.part_o;
    p.B = B;
    p.H = H;
    p.Nq = Nq;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = timeout_ns;
    p.drop_tile = drop_tile;

    static std::atomic<uint64_t> attr_set{0};   // one bit per device
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM_BYTES));
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set.fetch_or(bit);
    }
    chunk_attention_kernel<<<static_cast<unsigned>(units), NTHREADS, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sdv2
