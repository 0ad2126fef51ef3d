// Fused QKV projection + Causal-RoPE + KV-cache append.
//
// "Accelerating Video Generation Inference with Sequential-Parallel 3D Positional Encoding
// Using a Global Time Index", technical summary 2(다): the QKV projection and the Causal-RoPE
// computation are fused into a single kernel (there in TileLang on A800), with the cos/sin
// frequencies precomputed into contiguous tables.  Here: one tcgen05 GEMM
//     [q | k | v][token] = W_qkv x[token] (+ bias),   W_qkv: [3*H*D][C],  x: [B*Nq][C]
// whose epilogue rotates q and k with the token's 3D RoPE (time index from the stream's start
// frame and chunk, as in sdv2_rope_append_kv) and writes q_rot (head-major) and k_rot, v into
// the frames' cache slots, without a round trip of q, k, v through memory.
//
// Tiling: clusters of two CTAs on the two SMs of a TPC share each MMA (tcgen05.mma.cta_group::2,
// M = 256): a pair tile is 256 tokens x 256 features; each CTA holds its 128 token rows and
// half of the 256 weight rows per hidden step, and the accumulator of its 128 rows x 256
// features lands in its own tensor memory.  Each SM stages 32 KB per hidden step of 64 (a
// 128 x 256 tile on one SM would need 48 KB) and spends 512 MMA cycles on it, more than the
// step's copies and barrier handshake cost; a 6-stage ring (192 KB) keeps enough copies in
// flight next to the epilogue's tables.  4680 x 4608 makes 19 x 18 = 342 pair tiles (4.5 per
// pair on 76 pairs), 4680 x 15360 (14B) 19 x 60 = 1140 (15 per pair).  Pairs are persistent
// (tile t, t + pairs, ..., in an order with the q/k tiles first and the v tiles last, so that
// the final tile's epilogue -- which nothing overlaps -- has no table reads or rotation); a
// CTA's fp32 accumulator fills a 256-column buffer of tensor memory, so two tiles fit: the MMA
// warp fills one buffer while the epilogues of both CTAs drain the other.  A tile may straddle
// heads and the q|k|v boundaries (the epilogue finds the type and head of each 32-feature
// chunk); rows past the last token and feature rows past 3*H*D (odd head counts) load as zeros
// and the epilogue skips them.
//   warp 0: TMA producer (both CTAs load into their own shared memory and count the bytes on
//   the leader CTA's stage barrier; the leader arms it for both); warp 1: in the leader, MMA
//   issuer (converged: every lane polls, a warp vote agrees; elect.sync issues), whose commits
//   arrive on the barriers of both CTAs; warps 2-9: epilogue, two per TMEM lane quarter (each
//   takes half of the columns), thread = token row, with the next 32-column TMEM load in flight
//   while the current chunk is rotated and stored, arriving (relaxed: the arrival orders no
//   memory) on the leader's accumulator-empty barrier when a buffer is drained.
// The epilogue is what bounded this kernel (the MMA loop alone runs at the speed of a library
// GEMM of the same shape), and its cost is the number of distinct rows each warp instruction
// touches: the t, h and w cos/sin tables are copied into shared memory once per CTA (pair-major
// h and w, so that the warp's consecutive tokens read adjacent entries; tables too large for
// the area are read from global memory), a chunk's 16 pairs are loaded back to back through a
// pointer select, each warp stages its 128 bias values per tile with coalesced loads, and the
// four lanes of each quad transpose their 64-byte row segments with two xor-shuffle steps, so
// each store instruction writes 8 whole segments instead of 16 bytes of 32 rows.
// Rounding: acc (fp32, fp32 accumulation) + bias (fp32 add); q and k pairs rotated in fp32 as
// (fmaf(x, c, -(y*s)), fmaf(x, s, y*c)); one bf16 round-to-nearest-even per output.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "ptx_pair.cuh"

namespace sdv2 {
namespace {

constexpr int PBM = 256;                       // tokens per pair tile
constexpr int PBN = 256;                       // features per pair tile
constexpr int CBM = PBM / 2;                   // token rows in each CTA
constexpr int CBN = PBN / 2;                   // weight rows in each CTA
static_assert(PBN % 64 == 0 && PBN <= 256, "N of an M = 256 pair MMA; the epilogue splits it in 32-column chunks per half");
constexpr int QBK = 64;                        // hidden elements per TMA box (128 bytes of bf16)
constexpr int KSUB = 1;                        // boxes of QBK per ring stage (one barrier handshake)
constexpr int QST = 6;                         // ring stages
constexpr uint32_t A_BYTES = CBM * QBK * 2;    // 16 KB
constexpr uint32_t B_BYTES = CBN * QBK * 2;    // 16 KB
constexpr uint32_t SUB_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t STAGE_BYTES = KSUB * SUB_BYTES;
static_assert(128 % (QBK * KSUB) == 0, "the hidden dimension (heads x 128) is a whole number of ring stages");
constexpr int QTHREADS = 10 * 32;
constexpr int QEPI_WARPS = 8;
constexpr uint32_t QACC_COLS = 256;            // accumulator buffer stride
constexpr uint32_t QTMEM_COLS = 512;           // two accumulator buffers, at columns 0 and 256
// barriers: full[QST], empty[QST], acc_full[2], acc_empty[2], mma_done
constexpr int QB_FULL = 0, QB_EMPTY = QST, QB_ACC_FULL = 2 * QST, QB_ACC_EMPTY = 2 * QST + 2,
              QB_DONE = 2 * QST + 4, QNBARS = 2 * QST + 5;
// Shared memory: [ring][cos/sin tables t | h | w, when they fit][bias of each epilogue warp's
// columns of the current tile][barriers].  The 22 KB table area holds the tables of the 1.3B and
// 14B 480p and the 720p shapes; larger tables are read from global memory.
constexpr uint32_t TAB_OFF = QST * STAGE_BYTES;
constexpr uint32_t TAB_BYTES = 22 * 1024;
constexpr uint32_t BIAS_OFF = TAB_OFF + TAB_BYTES;
constexpr uint32_t BIAS_BYTES = QEPI_WARPS * (PBN / 2) * 4;
constexpr uint32_t BAR_OFF = BIAS_OFF + BIAS_BYTES;
constexpr uint32_t QSMEM_BYTES = BAR_OFF + 256 + 1024;
constexpr uint16_t kBothCtas = 0x3;
static_assert(QNBARS * 8 + 8 <= 256, "barriers and flags fit their 256 bytes");
static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "128-byte swizzle needs 1024-byte aligned tiles");
static_assert(QSMEM_BYTES <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Starts a load of 32 consecutive 32-bit columns of this thread's TMEM lane; the registers hold
// the values only after tmem_wait_ld_tied on the same array.
__device__ __forceinline__ void tmem_ld_x32_async(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}

// Waits for this thread's TMEM loads.  The array is an in-out operand, so no use of it is
// scheduled above the wait and its registers stay reserved while the load is in flight.
__device__ __forceinline__ void tmem_wait_ld_tied(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ uint4 shfl_xor_u4(uint4 v, int mask)
{
    v.x = __shfl_xor_sync(0xffffffffu, v.x, mask);
    v.y = __shfl_xor_sync(0xffffffffu, v.y, mask);
    v.z = __shfl_xor_sync(0xffffffffu, v.z, mask);
    v.w = __shfl_xor_sync(0xffffffffu, v.w, mask);
    return v;
}

// Tile order: the q/k feature tiles (those starting before 2*H*D) of every token tile first, then
// the v tiles, so that the last tile of each pair -- whose epilogue nothing overlaps -- is one
// without table reads and rotation.  Within each part the feature tiles vary fastest, unless the
// weights do not fit in L2 (m_fastest): then the token tiles vary fastest, so that the pairs of a
// wave share a few weight slices and the token rows stay in L2 from wave to wave instead of the
// whole weight matrix streaming from DRAM once per wave.
struct TileOrder {
    int nqk, nv;                       // feature tiles per token tile: q/k (2*H*D is a multiple of
                                       // 256), v (the last one ragged for odd H)
    int mtiles;
    bool m_fastest;
    __device__ __forceinline__ void coords(int t, int& mt, int& nt) const
    {
        const int qk_tiles = mtiles * nqk;
        const bool qk = t < qk_tiles;
        const int u = qk ? t : t - qk_tiles;   // the v part is only reached when nv > 0
        const int per = qk ? nqk : nv;         // feature tiles of this part
        if (m_fastest) {
            const int j = u / mtiles;
            mt = u - j * mtiles;
            nt = j;
        } else {
            mt = u / per;
            nt = u - mt * per;
        }
        if (!qk) nt += nqk;
    }
};

__global__ void __launch_bounds__(QTHREADS, 1) qkv_rope_kernel(const __grid_constant__ QkvRopeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    const uint32_t bar0 = smem_u32(bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + QNBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
#define QBAR(i) (bar0 + 8u * static_cast<uint32_t>(i))
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();                 // 0: the leader, which issues the MMAs
    const int pair = static_cast<int>(cluster_id_x());
    const int npairs = static_cast<int>(cluster_count_x());
    const int ntn = (3 * p.H * 128 + PBN - 1) / PBN;        // feature tiles (the last may be ragged)
    TileOrder order;
    order.mtiles = (p.M + PBM - 1) / PBM;
    order.nqk = (2 * p.H * 128 + PBN - 1) / PBN;
    order.nv = ntn - order.nqk;
    order.m_fastest = p.m_fastest != 0;
    const int ntiles = order.mtiles * ntn;
    const int my_tiles = pair < ntiles ? (ntiles - 1 - pair) / npairs + 1 : 0;
    const int ksteps = p.C / (QBK * KSUB);
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < QST; ++i) {
            mbar_init(QBAR(QB_FULL + i), 1);
            mbar_init(QBAR(QB_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(QBAR(QB_ACC_FULL + i), 1);
            mbar_init(QBAR(QB_ACC_EMPTY + i), 2 * QEPI_WARPS);
        }
        mbar_init(QBAR(QB_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), QTMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // both CTAs' barriers are initialised before either signals the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&p.xmap);
            tma_prefetch_desc(&p.wmap);
            const uint32_t full_leader = map_to_rank(QBAR(QB_FULL), 0);
            uint32_t pend = 0, par = 0;                      // per stage: armed, and the parity it was armed in
            bool ok = true;
            int g = 0;                                       // k-steps issued so far, over all tiles
            for (int li = 0; ok && li < my_tiles; ++li) {
                int mt, nt;
                order.coords(pair + li * npairs, mt, nt);
                const int m0 = mt * PBM + static_cast<int>(rank) * CBM;
                const int n0 = nt * PBN + static_cast<int>(rank) * CBN;
                for (int kk = 0; kk < ksteps; ++kk, ++g) {
                    const int st = g % QST;
                    const uint32_t ph = static_cast<uint32_t>(g / QST) & 1u;
                    // the leader's commit of the stage's previous MMAs arrives on both CTAs' barrier
                    if (!mbar_wait_cluster_bounded(QBAR(QB_EMPTY + st), ph ^ 1u, tmo, abort_flag)) {
                        *abort_flag = 1;
                        atomicOr(p.err, kErrTimeout);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = s0 + st * STAGE_BYTES;
                    if (rank == 0) mbar_arrive_expect_tx(QBAR(QB_FULL + st), 2 * STAGE_BYTES);
                    const uint32_t fb = full_leader + 8u * static_cast<uint32_t>(st);
#pragma unroll
                    for (int sb = 0; sb < KSUB; ++sb) {
                        tma_load_3d_pair(sa + sb * SUB_BYTES, &p.xmap, fb, (kk * KSUB + sb) * QBK, m0, 0);
                        tma_load_3d_pair(sa + sb * SUB_BYTES + A_BYTES, &p.wmap, fb, (kk * KSUB + sb) * QBK, n0, 0);
                    }
                    pend |= 1u << st;
                    par = (par & ~(1u << st)) | (ph << st);
                }
            }
            // Drain (leader): the last copies into each stage, its own and the peer's, must land
            // before the pair may exit (earlier ones were consumed by the MMAs before the stage
            // was refilled).  The peer stays resident until then: both CTAs meet at the final
            // cluster barrier.
            if (rank == 0) {
                volatile int no_abort = 0;
                for (int i = 0; i < QST; ++i)
                    if ((pend >> i) & 1u) mbar_wait_cluster_bounded(QBAR(QB_FULL + i), (par >> i) & 1u, tmo, &no_abort);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0) {
            // -------------------------------------------------------- MMA issuer (leader)
            constexpr uint32_t idesc = idesc_bf16_f32(PBM, PBN, false);
            const uint64_t dA = sdesc_sw128(s0, 16, 1024);
            const uint64_t dB = sdesc_sw128(s0 + A_BYTES, 16, 1024);
            constexpr uint64_t kStage = STAGE_BYTES >> 4;
            auto wait = [&](int bar_idx, uint32_t parity) -> bool {
                const bool r = mbar_wait_cluster_bounded(QBAR(bar_idx), parity, tmo, abort_flag);
                return __all_sync(0xffffffffu, r);
            };
            bool ok = true;
            int g = 0;
            for (int li = 0; ok && li < my_tiles; ++li) {
                const int buf = li & 1;
                // both CTAs' epilogues have drained this buffer's previous tile (first use: passes at once)
                if (!wait(QB_ACC_EMPTY + buf, (static_cast<uint32_t>(li >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + static_cast<uint32_t>(buf) * QACC_COLS;
                for (int kk = 0; kk < ksteps; ++kk, ++g) {
                    const int st = g % QST;
                    if (!wait(QB_FULL + st, static_cast<uint32_t>(g / QST) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a = dA + static_cast<uint64_t>(st) * kStage;
                    const uint64_t b = dB + static_cast<uint64_t>(st) * kStage;
#pragma unroll
                    for (int k = 0; k < KSUB * (QBK / 16); ++k) {
                        const uint64_t off = static_cast<uint64_t>((k / (QBK / 16)) * (SUB_BYTES >> 4) + (k % (QBK / 16)) * 2);
                        mma_ss_pair_warp(dacc, a + off, b + off, idesc, (kk > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit_pair_warp(QBAR(QB_EMPTY + st), kBothCtas);
                }
                if (!ok) break;
                mma_commit_pair_warp(QBAR(QB_ACC_FULL + buf), kBothCtas);   // this tile's accumulators are complete
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
            }
            // Tensor memory of both CTAs is freed only after every MMA has completed.
            mma_commit_pair_warp(QBAR(QB_DONE), kBothCtas);
        }
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait_cluster_bounded(QBAR(QB_DONE), 0, tmo, &no_abort);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: 256 threads per CTA
        // Two warps per TMEM lane quarter (a warp reaches the lanes of quarter warp index mod 4):
        // warps 2-5 drain the first half of the columns, warps 6-9 the second; thread = token row.
        const int part = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int col0 = part * (PBN / 2);                               // first column (feature) of this thread
        constexpr int kEpiCols = PBN / 2;                                // columns one thread drains
        const int hd = p.H * 128;
        const int64_t rows = static_cast<int64_t>(p.nslots) * p.HW;
        const uint32_t acc_empty_leader = map_to_rank(QBAR(QB_ACC_EMPTY), 0);
        // The cos/sin tables go to shared memory once per CTA (while the first tile's MMAs run):
        // read there, a chunk's 16 loads neither miss in L1 nor compete with the global stores.
        const int n_t = p.B * p.F * p.tp, n_h = p.hp * p.grid_h, n_w = p.wp * p.grid_w;
        const bool tabs_staged = static_cast<int64_t>(n_t + n_h + n_w) * 8 <= TAB_BYTES;
        float2* tab_s = reinterpret_cast<float2*>(smem + TAB_OFF);
        if (tabs_staged) {
            const int et = static_cast<int>(threadIdx.x) - 64;
            for (int k = et; k < n_t; k += 32 * QEPI_WARPS) tab_s[k] = p.tcs[k];
            for (int k = et; k < n_h; k += 32 * QEPI_WARPS) tab_s[n_t + k] = p.h_tab[k];
            for (int k = et; k < n_w; k += 32 * QEPI_WARPS) tab_s[n_t + n_h + k] = p.w_tab[k];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * QEPI_WARPS) : "memory");    // the epilogue warps only
        const float2* t_base = tabs_staged ? tab_s : p.tcs;
        const float2* h_base = tabs_staged ? tab_s + n_t : p.h_tab;
        const float2* w_base = tabs_staged ? tab_s + n_t + n_h : p.w_tab;
        float* bias_w = reinterpret_cast<float*>(smem + BIAS_OFF) + (warp - 2) * (PBN / 2);
        for (int li = 0; li < my_tiles; ++li) {
            const int buf = li & 1;
            bool ok = mbar_wait_cluster_bounded(QBAR(QB_ACC_FULL + buf), static_cast<uint32_t>(li >> 1) & 1u, tmo,
                                                abort_flag) &&
                      !*abort_flag;
            ok = __all_sync(0xffffffffu, ok);               // the TMEM loads below are warp-collective
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.err, kErrTimeout);
                }
                break;
            }
            tc_fence_after();
            int mt, nt;
            order.coords(pair + li * npairs, mt, nt);
            const int m0 = mt * PBM + static_cast<int>(rank) * CBM;
            const int n0 = nt * PBN;
            const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  static_cast<uint32_t>(buf) * QACC_COLS + static_cast<uint32_t>(col0);
            const int m = m0 + row;
            const bool valid = m < p.M;
            const int mm = valid ? m : 0;
            const int b = mm / p.Nq;
            const int n = mm - b * p.Nq;
            const int i = n / p.HW;
            const int r = n - i * p.HW;
            const int gh = r / p.grid_w;
            const int gw = r - gh * p.grid_w;
            const FrameDesc fd = p.frames[b * p.F + i];
            const float2* t_row = t_base + (b * p.F + i) * p.tp;
            const float2* h_col = h_base + gh;            // pair-major tables: the warp's consecutive
            const float2* w_col = w_base + gw;            // tokens read adjacent entries of a pair's row
            if (p.bias) {                                 // this warp's columns of the tile, one coalesced load each
#pragma unroll
                for (int j = 0; j < kEpiCols / 32; ++j) {
                    const int f = n0 + col0 + j * 32 + lane;
                    bias_w[j * 32 + lane] = f < 3 * hd ? p.bias[f] : 0.0f;
                }
                __syncwarp();
            }
            // element offsets of this token's q_rot row and k/v cache row (head 0, dim 0)
            const int64_t off_q = (static_cast<int64_t>(b) * p.H * p.Nq + n) * 128;
            const int64_t off_kv = (static_cast<int64_t>(b) * p.H * rows + static_cast<int64_t>(fd.slot) * p.HW + r) * 128;
            const uint32_t valid_mask = __ballot_sync(0xffffffffu, valid);
            const int quad0 = lane & ~3;                  // first lane of this thread's lane quad
            const int qj = lane & 3;
            // the next chunk's TMEM load is in flight while this chunk is rotated and stored
            uint32_t a[2][32];
            tmem_ld_x32_async(trow, a[0]);
            tmem_wait_ld_tied(a[0]);
#pragma unroll
            for (int cchunk = 0; cchunk < kEpiCols / 32; ++cchunk) {
                uint32_t(&cur)[32] = a[cchunk & 1];
                if (cchunk + 1 < kEpiCols / 32)
                    tmem_ld_x32_async(trow + static_cast<uint32_t>((cchunk + 1) * 32), a[(cchunk + 1) & 1]);
                const int f0 = n0 + col0 + cchunk * 32;           // feature of cur[0]
                if (f0 < 3 * hd) {                                // features past 3*H*D: zero-filled weight rows
                    const int type = f0 / hd;                     // 0 = q, 1 = k, 2 = v
                    const int fl = f0 - type * hd;
                    const int head = fl >> 7;
                    const int d0 = fl & 127;                      // first dim of the chunk in its head
                    uint16_t* base = (type == 0) ? p.q_rot + static_cast<int64_t>(head) * p.Nq * 128 + d0
                                   : ((type == 1) ? p.k_cache : p.v_cache) + static_cast<int64_t>(head) * rows * 128 + d0;
                    const int64_t off = type == 0 ? off_q : off_kv;
                    float bv[32];
                    if (p.bias) {
                        const float4* b4 = reinterpret_cast<const float4*>(bias_w + cchunk * 32);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const float4 t4 = b4[v];
                            bv[4 * v] = t4.x;
                            bv[4 * v + 1] = t4.y;
                            bv[4 * v + 2] = t4.z;
                            bv[4 * v + 3] = t4.w;
                        }
                    }
                    float2 csv[16];
                    if (type < 2) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int pr = (d0 >> 1) + u;
                            const float2* src = pr < p.tp ? t_row + pr
                                              : pr < p.tp + p.hp ? h_col + (pr - p.tp) * p.grid_h
                                                                 : w_col + (pr - p.tp - p.hp) * p.grid_w;
                            csv[u] = *src;           // generic load: shared memory, or launch parameters and global
                        }
                    }
                    uint32_t o[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        float x = __uint_as_float(cur[2 * u]);
                        float y = __uint_as_float(cur[2 * u + 1]);
                        if (p.bias) {
                            x = __fadd_rn(x, bv[2 * u]);
                            y = __fadd_rn(y, bv[2 * u + 1]);
                        }
                        if (type < 2) {
                            const float2 cs = csv[u];
                            const float xr = __fmaf_rn(x, cs.x, -__fmul_rn(y, cs.y));
                            const float yr = __fmaf_rn(x, cs.y, __fmul_rn(y, cs.x));
                            x = xr;
                            y = yr;
                        }
                        o[u] = pack2(x, y);
                    }
                    // Lane quad transpose: lane j of a quad holds its token's 64-byte segment as
                    // vectors e[0..3]; afterwards it holds vector j of the quad's four tokens, so
                    // that each store below writes four whole segments (8 per warp) instead of a
                    // sixteenth of 32 rows.  Step 1 swaps 2x2 blocks between lanes j and j^2,
                    // step 2 the off-diagonal vectors of each block between lanes j and j^1.
                    uint4 e[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) e[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    {
                        const bool hi = (qj & 2) != 0;
                        const uint4 s0 = hi ? e[0] : e[2], s1 = hi ? e[1] : e[3];
                        const uint4 r0 = shfl_xor_u4(s0, 2), r1 = shfl_xor_u4(s1, 2);
                        if (hi) { e[0] = r0; e[1] = r1; } else { e[2] = r0; e[3] = r1; }
                        const bool odd = (qj & 1) != 0;
                        const uint4 t0 = odd ? e[0] : e[1], t1 = odd ? e[2] : e[3];
                        const uint4 u0 = shfl_xor_u4(t0, 1), u1 = shfl_xor_u4(t1, 1);
                        if (odd) { e[0] = u0; e[2] = u1; } else { e[1] = u0; e[3] = u1; }
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v) {                 // token quad0 + v, its vector qj
                        const int64_t ov = __shfl_sync(0xffffffffu, off, quad0 + v);
                        if ((valid_mask >> (quad0 + v)) & 1u) reinterpret_cast<uint4*>(base + ov)[qj] = e[v];
                    }
                    if (valid && type == 1 && head == 0 && d0 == 0 && r == 0) {    // one writer per (stream, frame)
                        sdv2_slot_meta md;
                        md.frame_id = fd.frame;
                        md.tpos = fd.tpos;
                        p.meta[static_cast<int64_t>(b) * p.nslots + fd.slot] = md;
                    }
                }
                if (cchunk + 1 < kEpiCols / 32) tmem_wait_ld_tied(a[(cchunk + 1) & 1]);
            }
            // Every TMEM load of this buffer has completed (tcgen05.wait::ld above): hand it back
            // to the leader's MMA warp.  The arrival orders nothing else, so it is relaxed: a
            // release would first wait for this warp's global stores to reach cluster scope.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader + 8u * static_cast<uint32_t>(buf));
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();          // no CTA leaves while the other may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, QTMEM_COLS);
    }
#undef QBAR
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once; a function-local static is initialised by
// exactly one thread, so concurrent first calls from several host threads are safe.
EncodeTiledFn encode_fn()
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

// [rows][cols] bf16 matrix with row stride `ld` elements; boxes of 64 cols x box_rows rows.
bool encode_matrix(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(rows * ld * 2)};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_qkv_rope(QkvRopeParams& p, const void* x, const void* w, int64_t x_ld, cudaStream_t s,
                            const char** why)
{
    if (!encode_matrix(&p.xmap, x, p.M, p.C, x_ld, CBM) || !encode_matrix(&p.wmap, w, 3LL * p.H * 128, p.C, p.C, CBN)) {
        *why = "cuTensorMapEncodeTiled failed for x or w_qkv";
        return cudaErrorInvalidValue;
    }
    int dev = 0;
    cudaGetDevice(&dev);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(QTHREADS, 1, 1);
    cfg.dynamicSmemBytes = QSMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Per device, once: the shared-memory limit and how many CTA pairs can be resident at once
    // (a persistent pair per TPC whose two SMs are both available).
    static std::atomic<int> resident_pairs[64];
    std::atomic<int>& slot = resident_pairs[dev & 63];
    int pairs_max = slot.load();
    if (pairs_max <= 0) {
        cudaError_t e = cudaFuncSetAttribute(qkv_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(QSMEM_BYTES));
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        e = cudaOccupancyMaxActiveClusters(&pairs_max, qkv_rope_kernel, &cfg);
        if (e != cudaSuccess || pairs_max <= 0) {
            *why = "no CTA pair of the fused projection kernel fits on this device";
            return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        }
        slot.store(pairs_max);
    }
    int l2_bytes = 0;
    cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev);
    p.m_fastest = 3LL * p.H * 128 * p.C * 2 > static_cast<int64_t>(l2_bytes) / 2 ? 1 : 0;
    const int64_t ntiles = static_cast<int64_t>((p.M + PBM - 1) / PBM) * ((3 * p.H * 128 + PBN - 1) / PBN);
    const int64_t pairs = std::max<int64_t>(1, std::min<int64_t>(ntiles, pairs_max));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cudaError_t e = cudaLaunchKernelEx(&cfg, qkv_rope_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sdv2
