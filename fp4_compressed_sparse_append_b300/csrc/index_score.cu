// a2/a4: indexer scores, score(t) = sum_h w_h * ReLU(iq_h . ik_t), with FP8
// E4M3 indexer queries and FP8 E4M3 or MXFP4 keys, on the tcgen05 tensor cores.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select" (item 3: a small side network with its own low-precision
// queries and keys scores every cached entry), and section "The hierarchical
// indexer" (Reindex layers rescore only the pool's rows).
//
// The scan is a contraction: for a tile of 128 cached rows, D[128 x N] =
// K_tile[128 x DI] * Q^T[DI x N] with N = P*HI query heads of one sequence (or
// HI heads of one (sequence, position) over a pool).  Rows are the MMA's M
// dimension, so after the MMA each epilogue thread owns one cached row in
// tensor memory and reduces sum_h w_h ReLU(.) over its own columns with no
// cross-thread traffic; the [128 x N] product never leaves the SM.
//
// Persistent, warp-specialised CTAs (two per SM when their tensor-memory
// slots fit in half of it, so that two MMA threads keep the tensor core and the
// key stream busy while either one waits on a barrier):
//   warp 0      TMA producer: each job is up to 4 consecutive 128-row key tiles
//               of one unit (or 16 pool blocks of 8 rows) in one stage of a
//               shared-memory ring; the unit's query rows.
//   warp 1      TMEM owner and MMA issuer (one thread): kind::f8f6f4, M=128 per
//               key tile, all tiles of a stage into one accumulator slot of a
//               ring in tensor memory, so one barrier round trip and one commit
//               cover a whole stage and the MMAs run ahead of the epilogue.
//   warps 2..9  epilogue, two groups of four warps (each group covers the four
//               tensor-memory lane quarters): with several key tiles per job
//               the groups split each slot's tiles, otherwise they take
//               alternate slots; tcgen05.ld, weighted ReLU sum, coalesced fp32
//               score stores.
// The stage size matters: the MMA thread's fixed cost per stage (barrier waits,
// commits) is several hundred cycles, so a single CTA with 16 KB stages caps
// near 25 GB/s; 32 KB stages with two CTAs per SM stream fastest.
// Every wait is bounded (kWaitLimitNs); a wait that runs out raises
// CSA_DEV_TIMEOUT and the CTA drains its copies and returns.
#include <cuda_fp8.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kTileRows = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// MXFP4 keys (E2M1 codes and one UE8M0 scale per 32 channels, 68 B a key)
// go to the tensor core as they are stored: the TMA reads each key's 64 code
// bytes and writes them 8 bytes to every 16 (the padded 4-bit operand layout),
// and the MMA is the block-scaled kind::mxf8f6f4 with an E2M1 A operand and
// the E4M3 queries as B.  Four scale warps copy each tile's block scales from
// shared memory to tensor memory, where the MMA applies them: a tile's scales
// take four columns, the MMA reads row r's 32-bit word (its four block
// exponents) at lane r of column r / 32, and the instruction descriptor picks
// the byte of each 32-channel step; each warp writes its 32 rows' words into
// all four columns of its lane quarter.  They take the place of the
// second epilogue group, so the CTA keeps 320 threads and two CTAs fit an SM.
constexpr int kEpiWarpsMx = 4;
constexpr int kSclWarp0 = 2 + kEpiWarpsMx;
constexpr int kSclThreads = 128;  // thread = row of a 128-row tile
static_assert(2 + kEpiWarpsMx + kSclThreads / 32 == kThreads / 32, "same block size as the E4M3 variant");
constexpr int kMxCodeRow = 64;    // E2M1 code bytes per key (d_index 128)
constexpr int kMxScaleRow = 4;    // UE8M0 scale bytes per key
constexpr int kMxPoolScaleSlot = 128;  // pool: each 8-key block's 32 scale bytes in a 128-byte-aligned TMA slot
constexpr int kSfbCols = 16;      // tensor-memory columns of the queries' block scales (all 2^0)
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;  // four UE8M0 bytes of 2^0
constexpr int kMaxStages = 8;
constexpr int kMaxCols = 512;
constexpr int kMaxAcc = 8;
constexpr int kMaxTilesPerJob = 4;
constexpr int kMaxUnitsSmem = 2048;  // units whose tile counts are prefix-summed in shared memory

struct IdxArgs {
    int B, P, HI, cap, DI;
    int units;       // full scan: B (all P positions of a sequence share one key scan); pool: B*P
    int pool_mode;
    int groups;      // query positions per unit: P (full) or 1 (pool)
    int n_real;      // query rows (MMA columns) per unit: groups * HI
    int n_sub;       // column sub-chunks per key tile
    int gps;         // groups per sub-chunk
    int sub_cols;    // MMA N of a sub-chunk (gps*HI rounded up to 16, <= 256)
    int mt;          // 128-row key tiles per job (and per stage)
    int n_acc;       // accumulator slots in tensor memory (a power of two, 2..kMaxAcc)
    int stages;
    int b_rows, b_loads, b_box_rows;
    uint32_t tmem_cols;
    int prefix_smem; // units <= kMaxUnitsSmem: per-unit job counts prefix-summed in shared memory
    int mx;          // MXFP4 keys (block-scaled MMA)
    int mx_scale_stage;  // staged scale bytes per stage: mt*128*4, or 16 slots of 128 for a pool
    int sfa_col;     // MXFP4: tensor-memory column of the keys' scales, 4 columns per (stage, tile)
    int sfb_col;     // MXFP4: tensor-memory column of the queries' scales (kSfbCols columns)
    const int32_t *lengths;
    const int32_t *pool;
    int pool_blocks;
    const float *w;
    float *scores;
    int64_t ld;
    float *bmax;     // full scan, or null: each 8-row block's best visible score, [units*P][ldb]
    int64_t ldb;
    int *status;
};

// Jobs of one unit: ceil(rows / (mt*128)) for a full scan, 16 pool blocks
// (one 128-row tile) per job for a pool.
__device__ __forceinline__ int unit_jobs_global(const IdxArgs &a, int u)
{
    if (a.pool_mode) return (a.pool_blocks + 15) / 16;
    const int len = min(a.lengths[u], a.cap);
    const int rows = a.mt * kTileRows;
    return len > 0 ? (len + rows - 1) / rows : 0;
}

struct JobIter {
    int u, job, jobs_u;
};

struct Jobs {
    const IdxArgs &a;
    const int *prefix;  // [units + 1] in shared memory, or nullptr
    __device__ __forceinline__ int count(int u) const
    {
        return prefix ? prefix[u + 1] - prefix[u] : unit_jobs_global(a, u);
    }
    __device__ __forceinline__ int64_t total() const
    {
        if (prefix) return prefix[a.units];
        int64_t t = 0;
        for (int u = 0; u < a.units; ++u) t += unit_jobs_global(a, u);
        return t;
    }
    __device__ __forceinline__ void seek(int64_t j, JobIter &it) const
    {
        if (prefix) {
            int lo = 0, hi = a.units;  // last u with prefix[u] <= j
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= j) lo = mid;
                else hi = mid;
            }
            it.u = lo;
            it.jobs_u = count(lo);
            it.job = static_cast<int>(j - prefix[lo]);
            while (it.job >= it.jobs_u && it.u < a.units - 1) {  // skip empty units
                it.job -= it.jobs_u;
                ++it.u;
                it.jobs_u = count(it.u);
            }
            return;
        }
        int64_t acc = 0;
        it.u = 0;
        while (it.u < a.units) {
            const int t = unit_jobs_global(a, it.u);
            if (acc + t > j) {
                it.jobs_u = t;
                it.job = static_cast<int>(j - acc);
                return;
            }
            acc += t;
            ++it.u;
        }
        it.jobs_u = 0;
        it.job = 0;
    }
    __device__ __forceinline__ void next(JobIter &it) const
    {
        if (++it.job < it.jobs_u) return;
        it.job = 0;
        do {
            ++it.u;
            it.jobs_u = it.u < a.units ? count(it.u) : 1;
        } while (it.u < a.units && it.jobs_u == 0);
    }
};

__device__ __forceinline__ uint32_t swizzle_mode(int di)
{
    return di == 128 ? 2u : (di == 64 ? 4u : 6u);  // 128B, 64B, 32B
}

// sum_h w[h] * ReLU(acc[h]) over one query position's HI columns (HI a multiple
// of 32), which start at tensor-memory address `taddr` of this warp's lane
// quarter; w is this warp's copy in shared memory.  ReLU one value at a time,
// the weighting two at a time (packed fp32 FMA), into four paired partial sums
// that keep the FMA chains short.
__device__ __forceinline__ float2 relu2(uint32_t a, uint32_t b)
{
    return make_float2(fmaxf(__uint_as_float(a), 0.f), fmaxf(__uint_as_float(b), 0.f));
}

__device__ __forceinline__ float weighted_relu_sum(uint32_t taddr, const float *w, int HI)
{
    float2 s0 = make_float2(0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
    if (HI == 64) {  // both loads in flight before one wait
        uint32_t r[32], t[32];
        tmem_ld32(taddr, r);
        tmem_ld32(taddr + 32, t);
        tmem_ld_wait();
        const float4 *w4 = reinterpret_cast<const float4 *>(w);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 ww = w4[k], wv = w4[k + 8];
            s0 = __ffma2_rn(make_float2(ww.x, ww.y), relu2(r[4 * k + 0], r[4 * k + 1]), s0);
            s1 = __ffma2_rn(make_float2(ww.z, ww.w), relu2(r[4 * k + 2], r[4 * k + 3]), s1);
            s2 = __ffma2_rn(make_float2(wv.x, wv.y), relu2(t[4 * k + 0], t[4 * k + 1]), s2);
            s3 = __ffma2_rn(make_float2(wv.z, wv.w), relu2(t[4 * k + 2], t[4 * k + 3]), s3);
        }
        return ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
    }
    for (int c0 = 0; c0 < HI; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait();
        const float4 *w4 = reinterpret_cast<const float4 *>(w + c0);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float4 ww = w4[k], wv = w4[k + 1];
            s0 = __ffma2_rn(make_float2(ww.x, ww.y), relu2(r[4 * k + 0], r[4 * k + 1]), s0);
            s1 = __ffma2_rn(make_float2(ww.z, ww.w), relu2(r[4 * k + 2], r[4 * k + 3]), s1);
            s2 = __ffma2_rn(make_float2(wv.x, wv.y), relu2(r[4 * k + 4], r[4 * k + 5]), s2);
            s3 = __ffma2_rn(make_float2(wv.z, wv.w), relu2(r[4 * k + 6], r[4 * k + 7]), s3);
        }
    }
    return ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
}

// Same sum for any HI: 16-column loads masked to this position's columns.
__device__ __forceinline__ float weighted_relu_sum_any(uint32_t taddr, int col, const float *w, int HI)
{
    float s = 0.f;
    for (int c0 = col & ~15; c0 < col + HI; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int c = c0 + k;
            if (c >= col && c < col + HI) s = fmaf(w[c - col], fmaxf(__uint_as_float(r[k]), 0.f), s);
        }
    }
    return s;
}

// The block-scaled MMA: D (+)= (A * 2^scale_A) * (B * 2^scale_B)^T over one
// 32-channel step; the scale words sit in tensor memory, the descriptor's
// scale ids (bits 29-30 for A, 4-5 for B) pick their byte.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of the block-scaled MMA: A E2M1 (5), B E4M3 (0),
// both K-major, UE8M0 scales (bit 23), fp32 accumulation implied.
__host__ __device__ constexpr uint32_t instr_desc_mx(uint32_t M, uint32_t N)
{
    return (5u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%1,%1,%1};" ::"r"(taddr), "r"(v) : "memory");
}

template <bool MX>
__global__ void __launch_bounds__(kThreads, 2)
    index_score_kernel(const __grid_constant__ CUtensorMap keys128, const __grid_constant__ CUtensorMap keys8,
                       const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap scl128,
                       const __grid_constant__ CUtensorMap scl8, IdxArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned carve-up (swizzle atoms need it).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int tile_bytes = kTileRows * a.DI;
    const int stage_bytes = a.mt * tile_bytes;
    uint8_t *a_smem = base;  // [stages][mt][128 rows][DI bytes] key tiles (MXFP4: padded 4-bit codes)
    // MXFP4: each stage's block scales, [mt][128][4] (or 16 pool slots of 128 bytes).
    uint8_t *stg_scales = a_smem + a.stages * stage_bytes;
    const int stg_bytes = MX ? (a.stages * a.mx_scale_stage + 1023) & ~1023 : 0;
    uint8_t *b_smem = stg_scales + stg_bytes;
    constexpr int EW = MX ? kEpiWarpsMx : kEpiWarps;  // epilogue warps (groups of four)
    float *w_smem = reinterpret_cast<float *>(b_smem + ((a.b_rows * a.DI + 1023) & ~1023));  // [EW][n_pad]
    const int n_pad = (a.n_real + 3) & ~3;
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_smem + EW * n_pad);
    uint64_t *full = bars;                       // [kMaxStages]
    uint64_t *empty = full + kMaxStages;         // [kMaxStages]
    uint64_t *bfull = empty + kMaxStages;
    uint64_t *bempty = bfull + 1;
    uint64_t *tfull = bempty + 1;                // [kMaxAcc]
    uint64_t *tempty = tfull + kMaxAcc;          // [kMaxAcc]
    uint64_t *mma_done = tempty + kMaxAcc;
    uint64_t *sready = mma_done + 1;             // [kMaxStages] MXFP4: the stage's scales are in tensor memory
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sready + kMaxStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *prefix = const_cast<int *>(reinterpret_cast<volatile int *>(tmem_slot + 2));  // [units + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            if (MX) mbar_init(&sready[s], kSclThreads);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        for (int i = 0; i < a.n_acc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], (a.mt > 1 || EW == 4) ? 32 * EW : 32 * (EW / 2));
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&keys128);
        prefetch_tensormap(&keys8);
        prefetch_tensormap(&qmap);
        if (MX) {
            prefetch_tensormap(&scl128);
            prefetch_tensormap(&scl8);
        }
    }
    // Everything above touches only this CTA; from here on the kernel reads
    // what earlier work on the stream wrote (lengths, keys, queries).
    pdl_wait();
    if (warp == 2 && a.prefix_smem) {
        int carry = 0;
        for (int u0 = 0; u0 < a.units; u0 += 32) {
            const int u = u0 + lane;
            int t = u < a.units ? unit_jobs_global(a, u) : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
                if (lane >= o) t += y;
            }
            if (u < a.units) prefix[u + 1] = carry + t;
            carry += __shfl_sync(0xFFFFFFFFu, t, 31);
        }
        if (lane == 0) prefix[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const Jobs jobs{a, a.prefix_smem ? prefix : nullptr};

    // This CTA's contiguous share of the flattened (unit, job) list.
    const int64_t total = jobs.total();
    const int64_t j0 = total * blockIdx.x / gridDim.x;
    const int64_t j1 = total * (blockIdx.x + 1) / gridDim.x;

    if (warp == 0) {
        // ------------------------------------------------------------- producer
        if (lane == 0 && j0 < j1) {
            // A full scan reads every key once: its copies are the first lines
            // the L2 gives up, so the scores and block maxima this kernel writes
            // stay there for the top-K that reads them next.
            const uint64_t stream = l2_evict_first_policy();
            JobIter it;
            jobs.seek(j0, it);
            int stage = 0;
            uint32_t phase = 0, bphase = 0;
            int cur = -1;
            uint32_t issued_mask = 0, issued_parity = 0;
            for (int64_t j = j0; j < j1; ++j, jobs.next(it)) {
                if (it.u != cur) {
                    if (cur >= 0) {
                        if (!mbar_wait<true>(bempty, bphase, abort_flag)) break;
                        bphase ^= 1;
                    }
                    mbar_arrive_expect_tx(bfull, static_cast<uint32_t>(a.b_loads * a.b_box_rows * a.DI));
                    for (int i = 0; i < a.b_loads; ++i)
                        tma_load_2d(b_smem + i * a.b_box_rows * a.DI, &qmap, bfull, 0,
                                    it.u * a.n_real + i * a.b_box_rows);
                    cur = it.u;
                }
                if (!mbar_wait<true>(&empty[stage], phase ^ 1, abort_flag)) break;
                uint8_t *dst = a_smem + stage * stage_bytes;
                if (!a.pool_mode && MX) {
                    // codes of mt tiles, padded to the MMA's layout by the copy
                    // (which counts the bytes it reads: 64 a key), and their
                    // scales as 16-byte rows of 4 keys
                    uint8_t *ds = stg_scales + stage * a.mx_scale_stage;
                    mbar_arrive_expect_tx(&full[stage],
                                          static_cast<uint32_t>(a.mt * kTileRows * (kMxCodeRow + kMxScaleRow)));
                    const int row0 = it.u * a.cap + it.job * a.mt * kTileRows;
                    for (int m = 0; m < a.mt; ++m) {
                        tma_load_2d_hint(dst + m * tile_bytes, &keys128, &full[stage], 0, row0 + m * kTileRows, stream);
                        tma_load_2d_hint(ds + m * kTileRows * kMxScaleRow, &scl128, &full[stage], 0,
                                         (row0 + m * kTileRows) / 4, stream);
                    }
                } else if (!a.pool_mode) {
                    // mt whole boxes; rows past the cache's end read as zeros
                    // and rows past the unit's length are never stored.
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(stage_bytes));
                    const int row0 = it.u * a.cap + it.job * a.mt * kTileRows;
                    for (int m = 0; m < a.mt; ++m)
                        tma_load_2d_hint(dst + m * tile_bytes, &keys128, &full[stage], 0, row0 + m * kTileRows, stream);
                } else {
                    const int b = it.u / a.P;
                    const int32_t *prow = a.pool + static_cast<int64_t>(it.u) * a.pool_blocks;
                    int nv = 0;
                    int32_t blk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int jb = it.job * 16 + k;
                        blk[k] = jb < a.pool_blocks ? prow[jb] : -1;
                        if (blk[k] >= 0 && blk[k] < (a.cap + kPoolBlock - 1) / kPoolBlock)  // no overflow
                            ++nv;
                        else
                            blk[k] = -1;
                    }
                    if (MX) {
                        uint8_t *ds = stg_scales + stage * a.mx_scale_stage;
                        mbar_arrive_expect_tx(&full[stage],
                                              static_cast<uint32_t>(nv * kPoolBlock * (kMxCodeRow + kMxScaleRow)));
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (blk[k] >= 0) {
                                tma_load_2d(dst + k * kPoolBlock * a.DI, &keys8, &full[stage], 0,
                                            b * a.cap + blk[k] * kPoolBlock);
                                tma_load_2d(ds + k * kMxPoolScaleSlot, &scl8, &full[stage], 0,
                                            (b * a.cap + blk[k] * kPoolBlock) / 4);
                            }
                    } else {
                        mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nv * kPoolBlock * a.DI));
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (blk[k] >= 0)
                                tma_load_2d(dst + k * kPoolBlock * a.DI, &keys8, &full[stage], 0,
                                            b * a.cap + blk[k] * kPoolBlock);
                    }
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (*abort_flag) {
                // Let every copy this thread issued land before the CTA exits.
                for (int s = 0; s < a.stages; ++s)
                    if (issued_mask >> s & 1) {
                        const unsigned long long t0 = global_ns();
                        while (!mbar_try_wait(&full[s], issued_parity >> s & 1) &&
                               global_ns() - t0 < kWaitLimitNs) {
                        }
                    }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0 && j0 < j1) {
            const uint32_t sw = swizzle_mode(a.DI);
            const uint32_t sbo = 8 * a.DI;  // bytes between 8-row swizzle atoms
            // Descriptors of stage 0 / query row 0; the address field is the
            // low 14 bits (in 16-byte units), so offsets are added in place.
            const uint64_t da0 = smem_desc(smem_u32(a_smem), 16, sbo, sw);
            const uint64_t db0 = smem_desc(smem_u32(b_smem), 16, sbo, sw);
            const uint32_t idesc = MX ? instr_desc_mx(128, a.sub_cols) : instr_desc(128, a.sub_cols, 0, 0, 0, 0);
            const int slot_cols = a.mt * a.sub_cols;
            const int ksteps = a.DI / 32;
            JobIter it;
            jobs.seek(j0, it);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0, bphase = 0;
            int cur = -1;
            bool ok = true;
            for (int64_t j = j0; j < j1 && ok; ++j) {
                if (it.u != cur) {
                    if (!mbar_wait<true>(bfull, bphase, abort_flag)) break;
                    bphase ^= 1;
                    cur = it.u;
                }
                if (!mbar_wait<true>(&full[stage], phase, abort_flag)) break;
                if (MX && !mbar_wait<true>(&sready[stage], phase, abort_flag)) break;
                const uint64_t da_stage = da0 + static_cast<uint64_t>((stage * stage_bytes) >> 4);
                for (int sub = 0; sub < a.n_sub; ++sub) {
                    if (!mbar_wait<true>(&tempty[acc], acc_phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t db_sub = db0 + static_cast<uint64_t>((sub * a.gps * a.HI * a.DI) >> 4);
                    const uint32_t d_slot = tmem + acc * slot_cols;
                    for (int m = 0; m < a.mt; ++m) {
                        const uint64_t da_m = da_stage + static_cast<uint64_t>((m * tile_bytes) >> 4);
                        if (MX) {
                            const uint32_t sfa = tmem + a.sfa_col + (stage * a.mt + m) * 4;
                            for (uint32_t k = 0; k < static_cast<uint32_t>(ksteps); ++k)
                                mma_mxf8f6f4(d_slot + m * a.sub_cols, da_m + 2 * k, db_sub + 2 * k,
                                             idesc | (k << 29) | (k << 4), sfa, tmem + a.sfb_col, k > 0 ? 1u : 0u);
                        } else {
                            for (int k = 0; k < ksteps; ++k)
                                mma_f8f6f4(d_slot + m * a.sub_cols, da_m + 2 * k, db_sub + 2 * k, idesc,
                                           k > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&tfull[acc]);
                    if (++acc == a.n_acc) {
                        acc = 0;
                        acc_phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&empty[stage]);
                JobIter nx = it;
                jobs.next(nx);
                if (j + 1 == j1 || nx.u != it.u) mma_commit(bempty);
                it = nx;
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // Wait for every MMA issued here before tensor memory is released.
            mma_commit(mma_done);
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(mma_done, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (MX && warp >= kSclWarp0) {
        // ------------------------------------------------------------- MXFP4 block scales
        // The warp of lane quarter q copies the scale word of rows 32q..32q+31
        // of each staged tile to tensor-memory lanes 32q..32q+31 (the same
        // word in the tile's four columns), after the queries' unit scales.
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        for (int c = 0; c < kSfbCols; c += 4) tmem_st4(tl + a.sfb_col + c, kUnitScales);
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t j = j0; j < j1; ++j) {
            if (!mbar_wait<true>(&full[stage], phase, abort_flag)) break;
            const uint8_t *ss = stg_scales + stage * a.mx_scale_stage;
            for (int m = 0; m < a.mt; ++m) {
                // pool tiles: block row >> 3 in its own 128-byte slot
                const uint32_t w = *reinterpret_cast<const uint32_t *>(
                    a.pool_mode ? ss + (row >> 3) * kMxPoolScaleSlot + (row & 7) * kMxScaleRow
                                : ss + (m * kTileRows + row) * kMxScaleRow);
                tmem_st4(tl + a.sfa_col + (stage * a.mt + m) * 4, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sready[stage]);
            if (++stage == a.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        tmem_st_wait();
    } else {
        // ------------------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int q = warp & 3;     // tensor-memory lane quarter this warp may access
        // Two groups split each slot's tiles, or take alternate slots; one
        // group (MXFP4) takes every tile of every slot.
        const int ngrp = EW / 4;
        const int grp = ew >> 2;
        const bool split_tiles = a.mt > 1 && ngrp > 1;
        const int row_in_tile = q * 32 + lane;
        const int slot_cols = a.mt * a.sub_cols;
        float *wcopy = w_smem + ew * n_pad;
        JobIter it;
        if (j0 < j1) jobs.seek(j0, it);
        uint32_t seq = 0;           // (job, sub-chunk) slots in MMA order
        int cur = -1, len_b = 0;
        for (int64_t j = j0; j < j1; ++j, jobs.next(it)) {
            if (it.u != cur) {
                __syncwarp();
                const float *wsrc = a.w + static_cast<int64_t>(it.u) * a.n_real;
                for (int i = lane; i < a.n_real; i += 32) wcopy[i] = wsrc[i];
                __syncwarp();
                len_b = a.pool_mode ? 0 : min(a.lengths[it.u], a.cap);
                cur = it.u;
            }
            bool ok = true;
            for (int sub = 0; sub < a.n_sub; ++sub, ++seq) {
                if (ngrp > 1 && !split_tiles && static_cast<int>(seq & 1u) != grp) continue;
                const int acc = static_cast<int>(seq & static_cast<uint32_t>(a.n_acc - 1));
                const uint32_t par = (seq / static_cast<uint32_t>(a.n_acc)) & 1u;
                if (!mbar_wait<true>(&tfull[acc], par, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_slot = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * slot_cols;
                const int g0 = sub * a.gps, g1 = min(a.groups, g0 + a.gps);
                for (int m = split_tiles ? grp : 0; m < a.mt; m += split_tiles ? 2 : 1) {
                    const uint32_t t_base = t_slot + m * a.sub_cols;
                    const int r = (it.job * a.mt + m) * kTileRows + row_in_tile;
                    for (int g = g0; g < g1; ++g) {
                        const int col = (g - g0) * a.HI;
                        const float s = (a.HI & 31) == 0 ? weighted_relu_sum(t_base + col, wcopy + g * a.HI, a.HI)
                                                         : weighted_relu_sum_any(t_base, col, wcopy + g * a.HI, a.HI);
                        if (!a.pool_mode) {
                            const int Lp = len_b - a.P + 1 + g;
                            if (r < Lp) a.scores[(static_cast<int64_t>(it.u) * a.P + g) * a.ld + r] = s;
                            if (a.bmax) {
                                // a block's 8 rows are 8 consecutive lanes of this warp
                                float v = r < Lp ? s : -INFINITY;
                                v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
                                v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
                                v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
                                if ((r & 7) == 0 && r < Lp)
                                    a.bmax[(static_cast<int64_t>(it.u) * a.P + g) * a.ldb + (r >> 3)] = v;
                            }
                        } else {
                            if (r < a.pool_blocks * kPoolBlock) a.scores[static_cast<int64_t>(it.u) * a.ld + r] = s;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) raise_status(a.status, CSA_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

}  // namespace

cudaError_t launch_index_score(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, float *scores, int64_t ld, int *status,
                               cudaStream_t st, float *bmax, int64_t ldb)
{
    if (c.B * P == 0) return cudaSuccess;
    IdxArgs a{};
    a.B = c.B;
    a.P = P;
    a.HI = HI;
    a.cap = c.cap;
    a.DI = c.DI;
    a.pool_mode = pool != nullptr;
    a.units = a.pool_mode ? c.B * P : c.B;
    a.groups = a.pool_mode ? 1 : P;
    a.n_real = a.groups * HI;
    if (a.n_real > kMaxCols || HI > 256) return cudaErrorInvalidValue;
    // Column sub-chunks: whole positions per chunk, at most 256 MMA columns
    // each, so that two accumulator slots always fit the 512 tensor-memory columns.
    int n_sub = 1;
    while ((((a.groups + n_sub - 1) / n_sub) * HI + 15) / 16 * 16 > 256) ++n_sub;
    a.n_sub = n_sub;
    a.gps = (a.groups + n_sub - 1) / n_sub;
    a.sub_cols = (a.gps * HI + 15) / 16 * 16;
    if (n_sub > 1 && (a.gps * HI) % 8) return cudaErrorInvalidValue;
    // Two CTAs per SM when two accumulator slots of two key tiles (or one,
    // for a pool) fit in half of tensor memory; key tiles per job: as many as
    // keep two slots within the CTA's share of tensor memory.
    a.mx = c.mx;
    const int per_sm = 2 * (a.pool_mode ? 1 : 2) * a.sub_cols <= kMaxCols / 2 ? 2 : 1;
    const int cols_cta = kMaxCols / per_sm;
    // MXFP4: tensor memory also holds the keys' scales (4 columns per tile of
    // every stage, reserved for kMaxStages) and the queries' unit scales.
    auto sf_cols = [&](int mt) { return a.mx ? kMaxStages * mt * 4 + kSfbCols : 0; };
    a.mt = 1;
    const int max_mt = kMaxTilesPerJob / per_sm;
    while (!a.pool_mode && 2 * a.mt <= max_mt && 2 * (2 * a.mt) * a.sub_cols + sf_cols(2 * a.mt) <= cols_cta)
        a.mt *= 2;
    // Accumulator slots: a power of two, two or more where they fit (one only
    // when an MXFP4 cache's scales leave room for a single slot of 256 columns).
    a.n_acc = 2 * a.mt * a.sub_cols + sf_cols(a.mt) <= cols_cta ? 2 : 1;
    while (2 * a.n_acc <= kMaxAcc && 2 * a.n_acc * a.mt * a.sub_cols + sf_cols(a.mt) <= cols_cta) a.n_acc *= 2;
    const int acc_cols = a.n_acc * a.mt * a.sub_cols;
    // Query rows staged per unit: every sub-chunk's MMA reads sub_cols rows.
    const int need_rows = (n_sub - 1) * a.gps * HI + a.sub_cols;
    a.b_loads = (need_rows + 255) / 256;
    a.b_box_rows = ((need_rows + a.b_loads - 1) / a.b_loads + 7) / 8 * 8;
    a.b_rows = a.b_loads * a.b_box_rows;
    a.prefix_smem = a.units <= kMaxUnitsSmem;
    a.lengths = c.lengths;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    a.w = w;
    a.scores = scores;
    a.ld = ld;
    a.bmax = pool ? nullptr : bmax;
    a.ldb = ldb;
    a.status = status;

    const size_t stage_bytes = static_cast<size_t>(a.mt) * kTileRows * c.DI;
    const size_t b_bytes = (static_cast<size_t>(a.b_rows) * c.DI + 1023) & ~size_t(1023);
    const size_t w_bytes = static_cast<size_t>(a.mx ? kEpiWarpsMx : kEpiWarps) * ((a.n_real + 3) & ~3) * sizeof(float);
    const size_t prefix_bytes = a.prefix_smem ? (static_cast<size_t>(a.units) + 1) * sizeof(int) : 0;
    const size_t fixed = 1024 /*align*/ + b_bytes + w_bytes + (3 * kMaxStages + 2 * kMaxAcc + 4) * 8 + 16 +
                         prefix_bytes + (a.mx ? 1024 : 0) /*scale staging round-up*/;
    const size_t budget = per_sm == 1 ? 224 * 1024 : 110 * 1024;
    // MXFP4: each stage also stages its keys' block scales.
    a.mx_scale_stage = a.pool_mode ? 16 * kMxPoolScaleSlot : a.mt * kTileRows * kMxScaleRow;
    const size_t per_stage = stage_bytes + (a.mx ? a.mx_scale_stage : 0);
    if (budget < fixed + 2 * per_stage) return cudaErrorInvalidValue;
    int stages = static_cast<int>((budget - fixed) / per_stage);
    if (stages > kMaxStages) stages = kMaxStages;
    a.stages = stages;
    const size_t smem = fixed + stages * per_stage;
    a.sfa_col = acc_cols;
    a.sfb_col = acc_cols + stages * a.mt * 4;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(a.mx ? a.sfb_col + kSfbCols : acc_cols)) cols *= 2;
    if (cols > static_cast<uint32_t>(cols_cta)) return cudaErrorInvalidValue;
    a.tmem_cols = cols;

    const CUtensorMapSwizzle sw = c.DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : c.DI == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap k128, k8, qm, s128, s8;
    const uint64_t rows = static_cast<uint64_t>(c.B) * c.cap;
    if (encode_tensor_map_2d_u8(&qm, iq, c.DI, static_cast<uint64_t>(c.B) * P * HI, c.DI, a.b_box_rows, sw) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (a.mx) {
        // codes [rows][128 four-bit values], written 8 bytes to every 16 with
        // the 128-byte swizzle; scales [rows][4] as [rows / 4][16]
        if (c.DI != 128 || c.cap % 4) return cudaErrorInvalidValue;
        if (encode_tensor_map_2d_packed4(&k128, c.ikeys, rows, kTileRows) != CUDA_SUCCESS ||
            encode_tensor_map_2d_packed4(&k8, c.ikeys, rows, kPoolBlock) != CUDA_SUCCESS ||
            encode_tensor_map_2d_u8(&s128, c.iscales, 16, rows / 4, 16, kTileRows / 4, CU_TENSOR_MAP_SWIZZLE_NONE) !=
                CUDA_SUCCESS ||
            encode_tensor_map_2d_u8(&s8, c.iscales, 16, rows / 4, 16, kPoolBlock / 4, CU_TENSOR_MAP_SWIZZLE_NONE) !=
                CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        if (encode_tensor_map_2d_u8(&k128, c.ikeys, c.DI, rows, c.DI, kTileRows, sw) != CUDA_SUCCESS ||
            encode_tensor_map_2d_u8(&k8, c.ikeys, c.DI, rows, c.DI, kPoolBlock, sw) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        s128 = k128;
        s8 = k8;
    }

    auto kernel = a.mx ? index_score_kernel<true> : index_score_kernel<false>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3(sm_count() * per_sm), dim3(kThreads), smem, st, 0, k128, k8, qm, s128, s8, a);
}

}  // namespace csa
