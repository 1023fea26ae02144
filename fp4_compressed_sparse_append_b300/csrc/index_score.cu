// a2/a4: indexer scores, score(t) = sum_h w_h * ReLU(iq_h . ik_t), with FP8
// E4M3 indexer queries and keys, on the tcgen05 tensor cores.
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
#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kTileRows = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
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
    const int32_t *lengths;
    const int32_t *pool;
    int pool_blocks;
    const float *w;
    float *scores;
    int64_t ld;
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

__global__ void __launch_bounds__(kThreads, 2)
    index_score_kernel(const __grid_constant__ CUtensorMap keys128, const __grid_constant__ CUtensorMap keys8,
                       const __grid_constant__ CUtensorMap qmap, IdxArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned carve-up (swizzle atoms need it).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int tile_bytes = kTileRows * a.DI;
    const int stage_bytes = a.mt * tile_bytes;
    uint8_t *a_smem = base;
    uint8_t *b_smem = a_smem + a.stages * stage_bytes;
    float *w_smem = reinterpret_cast<float *>(b_smem + ((a.b_rows * a.DI + 1023) & ~1023));  // [kEpiWarps][n_pad]
    const int n_pad = (a.n_real + 3) & ~3;
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_smem + kEpiWarps * n_pad);
    uint64_t *full = bars;                       // [kMaxStages]
    uint64_t *empty = full + kMaxStages;         // [kMaxStages]
    uint64_t *bfull = empty + kMaxStages;
    uint64_t *bempty = bfull + 1;
    uint64_t *tfull = bempty + 1;                // [kMaxAcc]
    uint64_t *tempty = tfull + kMaxAcc;          // [kMaxAcc]
    uint64_t *mma_done = tempty + kMaxAcc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *prefix = const_cast<int *>(reinterpret_cast<volatile int *>(tmem_slot + 2));  // [units + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        for (int i = 0; i < a.n_acc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], a.mt > 1 ? 32 * kEpiWarps : 32 * (kEpiWarps / 2));
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
            JobIter it;
            jobs.seek(j0, it);
            int stage = 0;
            uint32_t phase = 0, bphase = 0;
            int cur = -1;
            uint32_t issued_mask = 0, issued_parity = 0;
            for (int64_t j = j0; j < j1; ++j, jobs.next(it)) {
                if (it.u != cur) {
                    if (cur >= 0) {
                        if (!mbar_wait(bempty, bphase, abort_flag)) break;
                        bphase ^= 1;
                    }
                    mbar_arrive_expect_tx(bfull, static_cast<uint32_t>(a.b_loads * a.b_box_rows * a.DI));
                    for (int i = 0; i < a.b_loads; ++i)
                        tma_load_2d(b_smem + i * a.b_box_rows * a.DI, &qmap, bfull, 0,
                                    it.u * a.n_real + i * a.b_box_rows);
                    cur = it.u;
                }
                if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
                uint8_t *dst = a_smem + stage * stage_bytes;
                if (!a.pool_mode) {
                    // mt whole boxes; rows past the cache's end read as zeros
                    // and rows past the unit's length are never stored.
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(stage_bytes));
                    const int row0 = it.u * a.cap + it.job * a.mt * kTileRows;
                    for (int m = 0; m < a.mt; ++m)
                        tma_load_2d(dst + m * tile_bytes, &keys128, &full[stage], 0, row0 + m * kTileRows);
                } else {
                    const int b = it.u / a.P;
                    const int32_t *prow = a.pool + static_cast<int64_t>(it.u) * a.pool_blocks;
                    int nv = 0;
                    int32_t blk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int jb = it.job * 16 + k;
                        blk[k] = jb < a.pool_blocks ? prow[jb] : -1;
                        if (blk[k] >= 0 && blk[k] * kPoolBlock < a.cap)
                            ++nv;
                        else
                            blk[k] = -1;
                    }
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nv * kPoolBlock * a.DI));
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (blk[k] >= 0)
                            tma_load_2d(dst + k * kPoolBlock * a.DI, &keys8, &full[stage], 0,
                                        b * a.cap + blk[k] * kPoolBlock);
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
            const uint32_t idesc = instr_desc(128, a.sub_cols, 0, 0, 0, 0);
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
                    if (!mbar_wait(bfull, bphase, abort_flag)) break;
                    bphase ^= 1;
                    cur = it.u;
                }
                if (!mbar_wait(&full[stage], phase, abort_flag)) break;
                const uint64_t da_stage = da0 + static_cast<uint64_t>((stage * stage_bytes) >> 4);
                for (int sub = 0; sub < a.n_sub; ++sub) {
                    if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t db_sub = db0 + static_cast<uint64_t>((sub * a.gps * a.HI * a.DI) >> 4);
                    const uint32_t d_slot = tmem + acc * slot_cols;
                    for (int m = 0; m < a.mt; ++m) {
                        const uint64_t da_m = da_stage + static_cast<uint64_t>((m * tile_bytes) >> 4);
                        for (int k = 0; k < ksteps; ++k)
                            mma_f8f6f4(d_slot + m * a.sub_cols, da_m + 2 * k, db_sub + 2 * k, idesc, k > 0 ? 1u : 0u);
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
    } else {
        // ------------------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int q = warp & 3;     // tensor-memory lane quarter this warp may access
        const int grp = ew >> 2;    // the two groups split each slot's tiles, or take alternate slots
        const bool split_tiles = a.mt > 1;
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
                len_b = a.pool_mode ? 0 : a.lengths[it.u];
                cur = it.u;
            }
            bool ok = true;
            for (int sub = 0; sub < a.n_sub; ++sub, ++seq) {
                if (!split_tiles && static_cast<int>(seq & 1u) != grp) continue;
                const int acc = static_cast<int>(seq & static_cast<uint32_t>(a.n_acc - 1));
                const uint32_t par = (seq / static_cast<uint32_t>(a.n_acc)) & 1u;
                if (!mbar_wait(&tfull[acc], par, abort_flag)) {
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

int g_num_sms = 0;

}  // namespace

cudaError_t launch_index_score(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, float *scores, int64_t ld, int *status,
                               cudaStream_t st)
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
    const int per_sm = 2 * (a.pool_mode ? 1 : 2) * a.sub_cols <= kMaxCols / 2 ? 2 : 1;
    const int cols_cta = kMaxCols / per_sm;
    a.mt = 1;
    while (!a.pool_mode && 2 * a.mt <= kMaxTilesPerJob / per_sm && 2 * (2 * a.mt) * a.sub_cols <= cols_cta) a.mt *= 2;
    a.n_acc = 2;
    while (2 * a.n_acc <= kMaxAcc && 2 * a.n_acc * a.mt * a.sub_cols <= cols_cta) a.n_acc *= 2;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(a.n_acc * a.mt * a.sub_cols)) cols *= 2;
    a.tmem_cols = cols;
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
    a.status = status;

    const size_t stage_bytes = static_cast<size_t>(a.mt) * kTileRows * c.DI;
    const size_t b_bytes = (static_cast<size_t>(a.b_rows) * c.DI + 1023) & ~size_t(1023);
    const size_t w_bytes = static_cast<size_t>(kEpiWarps) * ((a.n_real + 3) & ~3) * sizeof(float);
    const size_t prefix_bytes = a.prefix_smem ? (static_cast<size_t>(a.units) + 1) * sizeof(int) : 0;
    const size_t fixed =
        1024 /*align*/ + b_bytes + w_bytes + (2 * kMaxStages + 2 * kMaxAcc + 4) * 8 + 16 + prefix_bytes;
    const size_t budget = per_sm == 1 ? 224 * 1024 : 110 * 1024;
    int stages = static_cast<int>((budget - fixed) / stage_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    a.stages = stages;
    const size_t smem = fixed + stages * stage_bytes;

    const CUtensorMapSwizzle sw = c.DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : c.DI == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap k128, k8, qm;
    const uint64_t rows = static_cast<uint64_t>(c.B) * c.cap;
    if (encode_tensor_map_2d_u8(&k128, c.ikeys, c.DI, rows, c.DI, kTileRows, sw) != CUDA_SUCCESS ||
        encode_tensor_map_2d_u8(&k8, c.ikeys, c.DI, rows, c.DI, kPoolBlock, sw) != CUDA_SUCCESS ||
        encode_tensor_map_2d_u8(&qm, iq, c.DI, static_cast<uint64_t>(c.B) * P * HI, c.DI, a.b_box_rows, sw) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    const cudaError_t e =
        cudaFuncSetAttribute(index_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(index_score_kernel, dim3(g_num_sms * per_sm), dim3(kThreads), smem, st, 0, k128, k8, qm,
                         a);
}

}  // namespace csa
