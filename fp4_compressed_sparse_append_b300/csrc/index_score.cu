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
// Persistent, warp-specialised CTA (one per SM):
//   warp 0      TMA producer: key tiles (128 rows, or 16 pool blocks of 8 rows)
//               into a ring of shared-memory stages; the unit's query rows.
//   warp 1      TMEM owner and MMA issuer (one thread): kind::f8f6f4, M=128,
//               fp32 accumulators double-buffered in tensor memory.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, weighted ReLU sum,
//               coalesced fp32 score stores.
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

struct IdxArgs {
    int B, P, HI, cap, DI;
    int units;       // full scan: B (all P positions of a sequence share one key scan); pool: B*P
    int pool_mode;
    int groups;      // query positions per unit: P (full) or 1 (pool)
    int n_real;      // query rows (MMA columns) per unit: groups * HI
    int n_sub;       // column sub-chunks per tile (each its own accumulator)
    int gps;         // groups per sub-chunk
    int sub_cols;    // MMA N of a sub-chunk (gps*HI rounded up to 16, <= 256)
    int stages;
    int b_rows, b_loads, b_box_rows;
    uint32_t tmem_cols;
    const int32_t *lengths;
    const int32_t *pool;
    int pool_blocks;
    const float *w;
    float *scores;
    int64_t ld;
    int *status;
};

struct JobIter {
    int u, tile, tiles_u;
};

__device__ __forceinline__ int unit_tiles(const IdxArgs &a, int u)
{
    if (a.pool_mode) return (a.pool_blocks + 15) / 16;
    const int len = min(a.lengths[u], a.cap);
    return len > 0 ? (len + kTileRows - 1) / kTileRows : 0;
}

__device__ __forceinline__ void job_seek(const IdxArgs &a, int64_t j, JobIter &it)
{
    int64_t acc = 0;
    it.u = 0;
    while (it.u < a.units) {
        const int t = unit_tiles(a, it.u);
        if (acc + t > j) {
            it.tiles_u = t;
            it.tile = static_cast<int>(j - acc);
            return;
        }
        acc += t;
        ++it.u;
    }
    it.tiles_u = 0;
    it.tile = 0;
}

__device__ __forceinline__ void job_next(const IdxArgs &a, JobIter &it)
{
    if (++it.tile < it.tiles_u) return;
    it.tile = 0;
    do {
        ++it.u;
        it.tiles_u = it.u < a.units ? unit_tiles(a, it.u) : 1;
    } while (it.u < a.units && it.tiles_u == 0);
}

__device__ __forceinline__ uint32_t swizzle_mode(int di)
{
    return di == 128 ? 2u : (di == 64 ? 4u : 6u);  // 128B, 64B, 32B
}

// sum_h w[h] * ReLU(acc[h]) over one query position's HI columns (HI a multiple
// of 32), which start at tensor-memory address `taddr` of this warp's lane
// quarter; w is this warp's copy in shared memory.  Four partial sums keep the
// FMA chains short.
__device__ __forceinline__ float weighted_relu_sum(uint32_t taddr, const float *w, int HI)
{
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int c0 = 0; c0 < HI; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait();
        const float4 *w4 = reinterpret_cast<const float4 *>(w + c0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 ww = w4[k];
            s0 = fmaf(ww.x, fmaxf(__uint_as_float(r[4 * k + 0]), 0.f), s0);
            s1 = fmaf(ww.y, fmaxf(__uint_as_float(r[4 * k + 1]), 0.f), s1);
            s2 = fmaf(ww.z, fmaxf(__uint_as_float(r[4 * k + 2]), 0.f), s2);
            s3 = fmaf(ww.w, fmaxf(__uint_as_float(r[4 * k + 3]), 0.f), s3);
        }
    }
    return (s0 + s1) + (s2 + s3);
}

__global__ void __launch_bounds__(kThreads, 1)
    index_score_kernel(const __grid_constant__ CUtensorMap keys128, const __grid_constant__ CUtensorMap keys8,
                       const __grid_constant__ CUtensorMap qmap, IdxArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned carve-up (swizzle atoms need it).
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int a_bytes = kTileRows * a.DI;
    uint8_t *a_smem = base;
    uint8_t *b_smem = a_smem + a.stages * a_bytes;
    float *w_smem = reinterpret_cast<float *>(b_smem + ((a.b_rows * a.DI + 1023) & ~1023));  // [kEpiWarps][n_pad]
    const int n_pad = (a.n_real + 3) & ~3;
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_smem + kEpiWarps * n_pad);
    uint64_t *full = bars;                       // [kMaxStages]
    uint64_t *empty = full + kMaxStages;         // [kMaxStages]
    uint64_t *bfull = empty + kMaxStages;
    uint64_t *bempty = bfull + 1;
    uint64_t *tfull = bempty + 1;                // [2]
    uint64_t *tempty = tfull + 2;                // [2]
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 32 * kEpiWarps);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // This CTA's contiguous share of the flattened (unit, tile) jobs.
    int64_t total = 0;
    for (int u = 0; u < a.units; ++u) total += unit_tiles(a, u);
    const int64_t j0 = total * blockIdx.x / gridDim.x;
    const int64_t j1 = total * (blockIdx.x + 1) / gridDim.x;

    if (warp == 0) {
        // ------------------------------------------------------------- producer
        if (lane == 0 && j0 < j1) {
            JobIter it;
            job_seek(a, j0, it);
            int stage = 0;
            uint32_t phase = 0, bphase = 0;
            int cur = -1;
            uint32_t issued_mask = 0, issued_parity = 0;
            for (int64_t j = j0; j < j1; ++j, job_next(a, it)) {
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
                uint8_t *dst = a_smem + stage * a_bytes;
                if (!a.pool_mode) {
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(a_bytes));
                    tma_load_2d(dst, &keys128, &full[stage], 0, it.u * a.cap + it.tile * kTileRows);
                } else {
                    const int b = it.u / a.P;
                    const int32_t *prow = a.pool + static_cast<int64_t>(it.u) * a.pool_blocks;
                    int nv = 0;
                    int32_t blk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int jb = it.tile * 16 + k;
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
            const uint32_t a_base = smem_u32(a_smem), b_base = smem_u32(b_smem);
            const uint32_t idesc = instr_desc(128, a.sub_cols, 0, 0, 0, 0);
            JobIter it;
            job_seek(a, j0, it);
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
                const uint32_t a_stage = a_base + stage * a_bytes;
                for (int sub = 0; sub < a.n_sub; ++sub) {
                    if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_sub = b_base + sub * a.gps * a.HI * a.DI;
                    const uint32_t d_col = tmem + acc * a.sub_cols;
                    for (int k = 0; k < a.DI / 32; ++k) {
                        const uint64_t da = smem_desc(a_stage + k * 32, 16, sbo, sw);
                        const uint64_t db = smem_desc(b_sub + k * 32, 16, sbo, sw);
                        mma_f8f6f4(d_col, da, db, idesc, k > 0 ? 1u : 0u);
                    }
                    mma_commit(&tfull[acc]);
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&empty[stage]);
                JobIter nx = it;
                job_next(a, nx);
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
        const int q = warp & 3;   // tensor-memory lane quarter this warp may access
        const int half = ew >> 2;  // the two warps of a quarter split the positions
        const int row_in_tile = q * 32 + lane;
        float *wcopy = w_smem + ew * n_pad;
        JobIter it;
        if (j0 < j1) job_seek(a, j0, it);
        int acc = 0;
        uint32_t acc_phase = 0;
        int cur = -1, len_b = 0;
        for (int64_t j = j0; j < j1; ++j, job_next(a, it)) {
            if (it.u != cur) {
                __syncwarp();
                const float *wsrc = a.w + static_cast<int64_t>(it.u) * a.n_real;
                for (int i = lane; i < a.n_real; i += 32) wcopy[i] = wsrc[i];
                __syncwarp();
                len_b = a.pool_mode ? 0 : a.lengths[it.u];
                cur = it.u;
            }
            bool ok = true;
            for (int sub = 0; sub < a.n_sub; ++sub) {
                if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * a.sub_cols;
                const int g0 = sub * a.gps, g1 = min(a.groups, g0 + a.gps);
                for (int g = g0 + half; g < g1; g += 2) {
                    const int col = (g - g0) * a.HI;
                    float s;
                    if ((a.HI & 31) == 0) {
                        s = weighted_relu_sum(t_base + col, wcopy + g * a.HI, a.HI);
                    } else {
                        // General head counts: 16-column loads, masked to this position.
                        s = 0.f;
                        for (int c0 = col & ~15; c0 < col + a.HI; c0 += 16) {
                            uint32_t r[16];
                            tmem_ld16(t_base + c0, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const int c = c0 + k;
                                if (c >= col && c < col + a.HI)
                                    s = fmaf(wcopy[g * a.HI + c - col], fmaxf(__uint_as_float(r[k]), 0.f), s);
                            }
                        }
                    }
                    if (!a.pool_mode) {
                        const int t = it.tile * kTileRows + row_in_tile;
                        const int Lp = len_b - a.P + 1 + g;
                        if (t < Lp) a.scores[(static_cast<int64_t>(it.u) * a.P + g) * a.ld + t] = s;
                    } else {
                        const int c = it.tile * kTileRows + row_in_tile;
                        if (c < a.pool_blocks * kPoolBlock) a.scores[static_cast<int64_t>(it.u) * a.ld + c] = s;
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
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
    // each, so that two accumulators always fit the 512 tensor-memory columns.
    int n_sub = 1;
    while ((((a.groups + n_sub - 1) / n_sub) * HI + 15) / 16 * 16 > 256) ++n_sub;
    a.n_sub = n_sub;
    a.gps = (a.groups + n_sub - 1) / n_sub;
    a.sub_cols = (a.gps * HI + 15) / 16 * 16;
    if (n_sub > 1 && (a.gps * HI) % 8) return cudaErrorInvalidValue;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * a.sub_cols)) cols *= 2;
    a.tmem_cols = cols;
    // Query rows staged per unit: every sub-chunk's MMA reads sub_cols rows.
    const int need_rows = (n_sub - 1) * a.gps * HI + a.sub_cols;
    a.b_loads = (need_rows + 255) / 256;
    a.b_box_rows = ((need_rows + a.b_loads - 1) / a.b_loads + 7) / 8 * 8;
    a.b_rows = a.b_loads * a.b_box_rows;
    a.lengths = c.lengths;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    a.w = w;
    a.scores = scores;
    a.ld = ld;
    a.status = status;

    const size_t a_bytes = static_cast<size_t>(kTileRows) * c.DI;
    const size_t b_bytes = (static_cast<size_t>(a.b_rows) * c.DI + 1023) & ~size_t(1023);
    const size_t w_bytes = static_cast<size_t>(kEpiWarps) * ((a.n_real + 3) & ~3) * sizeof(float);
    const size_t fixed = 1024 /*align*/ + b_bytes + w_bytes + (2 * kMaxStages + 8) * 8 + 64;
    const size_t budget = 220 * 1024;
    int stages = static_cast<int>((budget - fixed) / a_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    a.stages = stages;
    const size_t smem = fixed + stages * a_bytes;

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
    cudaError_t e =
        cudaFuncSetAttribute(index_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    index_score_kernel<<<g_num_sms, kThreads, smem, st>>>(k128, k8, qm, a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace csa
