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
// Tiling: persistent CTAs, one per SM, walk the tiles of 128 tokens x 192 features (tile t,
// t + gridDim.x, ...; the constants also allow two 128-row halves per tile).  A tile's fp32
// accumulator takes 256 of the 512 tensor-memory columns, so two tiles fit: the MMA warp fills
// one accumulator buffer while the epilogue drains the other, and the epilogue of a tile runs
// under the next tile's main loop.  The hidden dimension streams in steps of 64 (128-byte
// swizzled TMA boxes) through a 4-stage ring of 40 KB stages.  N = 192 MMAs read their
// operands from shared memory at 107 bytes per cycle (a 256 x 128 tile as two M = 128 halves
// needs 128, the whole shared-memory bandwidth), and 4680 x 4608 makes 888 tiles, 5.84 per SM
// (128 x 256: 666 tiles, 4.38 per SM, 5 on some).  A tile may straddle heads and the q|k|v
// boundaries (the epilogue finds the type and head of each 32-feature chunk); the last feature
// tile may be ragged (its weight rows past the end load as zeros and the epilogue skips them).
//   warp 0: TMA producer; warp 1: MMA issuer (converged: every lane polls the stage barrier and
//   a warp vote agrees on the outcome; elect.sync issues); warps 2-9: epilogue, two per TMEM lane
//   quarter (one per half), thread = token row, with the next 32-column TMEM load in flight while
//   the current chunk is rotated and stored (bias read as float4); with one 128-row half the two
//   warps of a quarter take the two halves of the columns.  A chunk's 16 cos/sin pairs
//   are loaded into registers before any is used: each pair's table (time, h or w axis) is
//   picked by a pointer select, so the 16 loads issue back to back instead of one per branch
//   of the axis test.  Barriers: full/empty per ring stage; accumulator full/empty per buffer
//   (the empty one counts the eight epilogue warps).
// Rounding: acc (fp32, fp32 accumulation) + bias (fp32 add); q and k pairs rotated in fp32 as
// (fmaf(x, c, -(y*s)), fmaf(x, s, y*c)); one bf16 round-to-nearest-even per output.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace sdv2 {
namespace {

constexpr int QBM = 128;                       // tokens per tile: 1 or 2 halves of 128 rows
constexpr int QBN = 192;                       // features per tile
constexpr int QHALVES = QBM / 128;             // 128-row accumulators per tile
static_assert((QHALVES == 1 || QHALVES == 2) && QHALVES * QBN <= 256 && QBN % 64 == 0 && QBN <= 256,
              "a tile's accumulators fit in one 256-column buffer; the epilogue splits them in 32-column chunks");
constexpr int QBK = 64;                        // hidden elements per step (128 bytes of bf16)
constexpr int QST = 4;                         // ring stages
constexpr uint32_t A_BYTES = QBM * QBK * 2;    // 32 KB
constexpr uint32_t A_HALF = A_BYTES / 2;       // rows 128..255 of the A box start here
constexpr uint32_t B_BYTES = QBN * QBK * 2;    // 16 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int QTHREADS = 10 * 32;
constexpr int QEPI_WARPS = 8;
constexpr uint32_t QACC_COLS = 256;            // accumulator buffer stride: QHALVES halves of QBN columns each
constexpr uint32_t QTMEM_COLS = 512;           // two accumulator buffers, at columns 0 and 256
// barriers: full[QST], empty[QST], acc_full[2], acc_empty[2], mma_done
constexpr int QB_FULL = 0, QB_EMPTY = QST, QB_ACC_FULL = 2 * QST, QB_ACC_EMPTY = 2 * QST + 2,
              QB_DONE = 2 * QST + 4, QNBARS = 2 * QST + 5;
constexpr uint32_t QSMEM_BYTES = QST * STAGE_BYTES + 256 + 1024;
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

__global__ void __launch_bounds__(QTHREADS, 1) qkv_rope_kernel(const __grid_constant__ QkvRopeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + QST * STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + QNBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
#define QBAR(i) (bar0 + 8u * static_cast<uint32_t>(i))
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
    const int lane = threadIdx.x & 31;
    const int ntn = (3 * p.H * 128 + QBN - 1) / QBN;        // feature tiles (the last may be ragged)
    const int ntiles = ((p.M + QBM - 1) / QBM) * ntn;
    const int my_tiles = static_cast<int>(blockIdx.x) < ntiles
                             ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1 : 0;
    const int ksteps = p.C / QBK;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < QST; ++i) {
            mbar_init(QBAR(QB_FULL + i), 1);
            mbar_init(QBAR(QB_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(QBAR(QB_ACC_FULL + i), 1);
            mbar_init(QBAR(QB_ACC_EMPTY + i), QEPI_WARPS);
        }
        mbar_init(QBAR(QB_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), QTMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&p.xmap);
            tma_prefetch_desc(&p.wmap);
            int pend[QST] = {};
            uint32_t par[QST] = {};
            bool ok = true;
            int g = 0;                                       // k-steps issued so far, over all tiles
            for (int li = 0; ok && li < my_tiles; ++li) {
                const int tile = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
                const int m0 = (tile / ntn) * QBM;
                const int n0 = (tile % ntn) * QBN;
                for (int kk = 0; kk < ksteps; ++kk, ++g) {
                    const int st = g % QST;
                    const uint32_t ph = static_cast<uint32_t>(g / QST) & 1u;
                    if (!mbar_wait_bounded(QBAR(QB_EMPTY + st), ph ^ 1u, tmo, abort_flag)) {
                        *abort_flag = 1;
                        atomicOr(p.err, kErrTimeout);
                        ok = false;
                        break;
                    }
                    const uint32_t sa = s0 + st * STAGE_BYTES;
                    mbar_arrive_expect_tx(QBAR(QB_FULL + st), STAGE_BYTES);
                    tma_load_3d(sa, &p.xmap, QBAR(QB_FULL + st), kk * QBK, m0, 0);
                    tma_load_3d(sa + A_BYTES, &p.wmap, QBAR(QB_FULL + st), kk * QBK, n0, 0);
                    pend[st] = 1;
                    par[st] = ph;
                }
            }
            // Drain: the last copy into each stage must land before the CTA may exit (earlier
            // ones were consumed by the MMA warp before the stage was refilled).
            volatile int no_abort = 0;
            for (int i = 0; i < QST; ++i)
                if (pend[i]) mbar_wait_bounded(QBAR(QB_FULL + i), par[i], tmo, &no_abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(128, QBN, false);
        const uint64_t dA = sdesc_sw128(s0, 16, 1024);
        const uint64_t dB = sdesc_sw128(s0 + A_BYTES, 16, 1024);
        constexpr uint64_t kStage = STAGE_BYTES >> 4;
        constexpr uint64_t kHalf = A_HALF >> 4;
        auto wait = [&](int bar_idx, uint32_t parity) -> bool {
            const bool r = mbar_wait_bounded(QBAR(bar_idx), parity, tmo, abort_flag);
            return __all_sync(0xffffffffu, r);
        };
        bool ok = true;
        int g = 0;
        for (int li = 0; ok && li < my_tiles; ++li) {
            const int buf = li & 1;
            // the epilogue has drained this buffer's previous tile (first use: passes at once)
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
                // both halves of the tile multiply the same weight stage
#pragma unroll
                for (int hh = 0; hh < QHALVES; ++hh)
#pragma unroll
                    for (int k = 0; k < QBK / 16; ++k)
                        mma_ss_warp(dacc + static_cast<uint32_t>(hh * QBN),
                                    a + static_cast<uint64_t>(hh) * kHalf + static_cast<uint64_t>(k * 2),
                                    b + static_cast<uint64_t>(k * 2), idesc, (kk > 0 || k > 0) ? 1u : 0u);
                mma_commit_warp(QBAR(QB_EMPTY + st));
            }
            if (!ok) break;
            mma_commit_warp(QBAR(QB_ACC_FULL + buf));        // this tile's accumulators are complete
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.err, kErrTimeout);
        }
        // Tensor memory is freed only after every MMA of this warp has completed.
        mma_commit_warp(QBAR(QB_DONE));
        if (lane == 0) {
            volatile int no_abort = 0;
            mbar_wait_bounded(QBAR(QB_DONE), 0, tmo, &no_abort);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: 256 threads
        // Two warps per TMEM lane quarter (a warp reaches the lanes of quarter warp index mod 4):
        // with two 128-row halves, warps 2-5 read rows 0..127 and warps 6-9 rows 128..255, all
        // columns; with one half, warps 2-5 read the first half of the columns, warps 6-9 the
        // second.  Either way a thread drains 128 columns of one row.
        const int part = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int row = (QHALVES == 2 ? part * 128 : 0) + quarter * 32 + lane;
        const int col0 = QHALVES == 2 ? 0 : part * (QBN / 2);          // first column (feature) of this thread
        constexpr int kEpiCols = QBN * QHALVES / 2;                    // columns one thread drains
        const int hd = p.H * 128;
        const int64_t rows = static_cast<int64_t>(p.nslots) * p.HW;
        for (int li = 0; li < my_tiles; ++li) {
            const int buf = li & 1;
            bool ok = mbar_wait_bounded(QBAR(QB_ACC_FULL + buf), static_cast<uint32_t>(li >> 1) & 1u, tmo, abort_flag) &&
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
            const int tile = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
            const int m0 = (tile / ntn) * QBM;
            const int n0 = (tile % ntn) * QBN;
            const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  static_cast<uint32_t>(buf) * QACC_COLS +
                                  static_cast<uint32_t>(QHALVES == 2 ? part * QBN : col0);
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
            const float2* t_row = p.tcs + (b * p.F + i) * p.tp;
            const float2* h_row = p.h_tab + gh * p.hp;
            const float2* w_row = p.w_tab + gw * p.wp;
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
                if (valid && f0 < 3 * hd) {                       // features past 3*H*D: zero-filled weight rows
                    const int type = f0 / hd;                     // 0 = q, 1 = k, 2 = v
                    const int fl = f0 - type * hd;
                    const int head = fl >> 7;
                    const int d0 = fl & 127;                      // first dim of the chunk in its head
                    const int64_t bh = static_cast<int64_t>(b) * p.H + head;
                    uint16_t* dst = (type == 0) ? p.q_rot + (bh * p.Nq + n) * 128 + d0
                                  : (type == 1) ? p.k_cache + (bh * rows + static_cast<int64_t>(fd.slot) * p.HW + r) * 128 + d0
                                                : p.v_cache + (bh * rows + static_cast<int64_t>(fd.slot) * p.HW + r) * 128 + d0;
                    float bv[32];
                    if (p.bias) {
                        const float4* b4 = reinterpret_cast<const float4*>(p.bias + f0);
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
                                              : pr < p.tp + p.hp ? h_row + (pr - p.tp) : w_row + (pr - p.tp - p.hp);
                            csv[u] = *src;           // generic load: t pairs live in the launch parameters
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
                    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int v = 0; v < 4; ++v) d4[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    if (type == 1 && head == 0 && d0 == 0 && r == 0) {    // one writer per (stream, frame)
                        sdv2_slot_meta md;
                        md.frame_id = fd.frame;
                        md.tpos = fd.tpos;
                        p.meta[static_cast<int64_t>(b) * p.nslots + fd.slot] = md;
                    }
                }
                if (cchunk + 1 < kEpiCols / 32) tmem_wait_ld_tied(a[(cchunk + 1) & 1]);
            }
            // every TMEM load of this buffer has completed: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(QBAR(QB_ACC_EMPTY + buf));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, QTMEM_COLS);
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
    if (!encode_matrix(&p.xmap, x, p.M, p.C, x_ld, QBM) || !encode_matrix(&p.wmap, w, 3LL * p.H * 128, p.C, p.C, QBN)) {
        *why = "cuTensorMapEncodeTiled failed for x or w_qkv";
        return cudaErrorInvalidValue;
    }
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(qkv_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(QSMEM_BYTES));
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set.fetch_or(bit);
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t ntiles = static_cast<int64_t>((p.M + QBM - 1) / QBM) * ((3 * p.H * 128 + QBN - 1) / QBN);
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(ntiles, std::max(1, sms))));
    qkv_rope_kernel<<<grid, QTHREADS, QSMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace sdv2
