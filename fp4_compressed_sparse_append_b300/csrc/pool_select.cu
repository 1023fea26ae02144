// a4: a Reindex layer over the hierarchical pool, scoring and selection in one
// kernel.  "G2C Brief - DeepSeek V4.1-Flash", section "The hierarchical
// indexer: making later indexers context-independent": the first Full layer
// keeps a pool of 2,048 blocks of 8 positions, and later Reindex layers score
// only the pool's 16,384 rows with their own indexer query and keep the best
// K; section "CSA2: most layers don't keep their own cache" (Reindex borrows
// the keys and selects afresh).  Score: sum_h w_h * ReLU(iq_h . ik), FP8 E4M3
// queries and keys, fp32 accumulation.
//
// One thread-block cluster per (sequence, position): CTA r of C takes a
// contiguous share of the pool's blocks (at most 128 blocks, 1,024 rows).
//   1. Each of its first 128 threads reads one block id and starts the TMA
//      copy of that block's 8 key rows into the CTA's tile of 16 blocks; the
//      indexer query arrives by TMA too.
//   2. One thread issues, per 128-row tile, the kind::f8f6f4 MMA
//      D[128 rows x HI] = K_tile . Q^T into its own tensor-memory columns.
//   3. Four warps (one per lane quarter) turn each row's HI accumulators into
//      sum_h w_h ReLU(.) and store the row's order-preserving score key (0 for
//      an empty pool slot or a row past the visible length) straight into the
//      shared memory of CTA 0, with the block ids.
//   4. After one cluster barrier CTA 0 alone selects the K largest keys of the
//      whole pool (ties: the earlier pool slot, which is the lower row id for
//      an ascending pool) with cta_select::select_keys (select_cta.cuh) and
//      writes the selected rows in pool order, then -1 padding.
// Every wait is bounded; a wait that runs out raises CSA_DEV_TIMEOUT.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "csa_internal.h"
#include "select_cta.cuh"

namespace csa {
namespace {

constexpr int kThreads = 512;
constexpr int kTileRows = 128;
constexpr int kMaxTiles = 8;                   // 1,024 rows per CTA
constexpr int kBlocksPerCta = kMaxTiles * kTileRows / kPoolBlock;  // 128
constexpr int kMaxCluster = 16;
constexpr int kMaxCand = kMaxCluster * kMaxTiles * kTileRows;     // 16,384
constexpr int kU = 4;                          // loads in flight per thread (score gathers)

struct PoolArgs {
    int P, HI, cap, DI;
    const int32_t *lengths;
    const int32_t *pool;    // [units][pool_blocks], ascending, -1 padded
    int pool_blocks;
    int bpc;                // blocks per CTA (<= 128)
    const float *w;         // [units][HI]
    int K;
    int32_t *idx;           // [units][K]
    int *status;
};

struct PoolSmem {
    uint64_t tbar[kMaxTiles];   // key tile copied
    uint64_t mbar[kMaxTiles];   // tile's MMA done
    uint64_t qbar, done;
    float w[64];
    int32_t blk[kBlocksPerCta];
    uint32_t tmem_slot;
    int abort;
};

__device__ __forceinline__ uint32_t swizzle_mode(int di)
{
    return di == 128 ? 2u : (di == 64 ? 4u : 6u);  // 128B, 64B, 32B
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

static_assert(kThreads == cta_select::kThreads && kMaxCand == cta_select::kMaxKeys, "one selection CTA shape");

// The K best of the n pool rows whose keys are in allk (at their key_slot),
// written to out as row ids in pool order (candidate c is row
// allb[c / 8] * 8 + c % 8), then -1 padding.  All threads of the CTA call it.
__device__ __forceinline__ void write_selection(uint32_t *allk, const int32_t *allb, int n, int K, int32_t *out,
                                                cta_select::Scratch &sc)
{
    int32_t *kept_c = reinterpret_cast<int32_t *>(allk);
    const int kept = cta_select::select_keys(allk, n, static_cast<uint32_t>(K), kept_c, sc);
    for (int j = threadIdx.x; j < K; j += kThreads) {
        const int c = j < kept ? kept_c[j] : -1;
        out[j] = c >= 0 ? allb[c >> 3] * kPoolBlock + (c & 7) : -1;
    }
}

template <int HT>
__global__ void __launch_bounds__(kThreads, 1)
    pool_select_kernel(const __grid_constant__ CUtensorMap keys8, const __grid_constant__ CUtensorMap qmap, PoolArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int DI = a.DI;
    uint8_t *k_s = base;                                       // [8 tiles][128 rows][DI] key tiles
    uint8_t *q_s = k_s + kMaxTiles * kTileRows * DI;           // [HT rows][DI] indexer query
    uint32_t *allk = reinterpret_cast<uint32_t *>(q_s + ((HT * DI + 1023) & ~1023));  // CTA 0: [candidates] keys
    int32_t *allb = reinterpret_cast<int32_t *>(allk + kMaxCand);                    // CTA 0: [blocks] ids
    PoolSmem &sm = *reinterpret_cast<PoolSmem *>(allb + kMaxCluster * kBlocksPerCta);
    // CTA 0, select phase: the selection's scratch over the dead key tiles
    // (at least 32 KB: 8 tiles of 128 rows of >= 32 bytes)
    cta_select::Scratch &sc = *reinterpret_cast<cta_select::Scratch *>(k_s);
    volatile int *abort_flag = &sm.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.y;
    const uint32_t rank = blockIdx.x;   // cluster rank (the cluster spans x)
    const int C = gridDim.x;
    const int n_tiles = (a.bpc * kPoolBlock + kTileRows - 1) / kTileRows;

    if (tid == 0) {
        for (int t = 0; t < kMaxTiles; ++t) {
            mbar_init(&sm.tbar[t], 16);
            mbar_init(&sm.mbar[t], 1);
        }
        mbar_init(&sm.qbar, 1);
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&keys8);
        prefetch_tensormap(&qmap);
    }
    if (warp == 4) {
        tmem_alloc(&sm.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Every CTA of the cluster has started before any stores into CTA 0.
    if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const uint32_t tmem = sm.tmem_slot;

    // Below: reads of what earlier work on the stream wrote.
    pdl_wait();
    pdl_trigger();
    const int b = unit / a.P, p = unit % a.P;
    const int Lp = min(a.lengths[b], a.cap) - a.P + 1 + p;
    const int cap_blocks = (a.cap + kPoolBlock - 1) / kPoolBlock;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.qbar, static_cast<uint32_t>(HT * DI));
        tma_load_2d(q_s, &qmap, &sm.qbar, 0, unit * a.HI);
    }
    if (tid < HT) sm.w[tid] = tid < a.HI ? a.w[static_cast<int64_t>(unit) * a.HI + tid] : 0.f;
    if (tid < n_tiles * 16) {
        // one pool block per thread: its id, and the copy of its 8 key rows
        const int j = rank * a.bpc + tid;
        int32_t blk = (tid < a.bpc && j < a.pool_blocks) ? a.pool[static_cast<int64_t>(unit) * a.pool_blocks + j] : -1;
        if (blk >= cap_blocks) blk = -1;
        sm.blk[tid] = blk;
        uint64_t *bar = &sm.tbar[tid >> 4];
        if (blk >= 0) {
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kPoolBlock * DI));
            tma_load_2d(k_s + tid * kPoolBlock * DI, &keys8, bar, 0, b * a.cap + blk * kPoolBlock);
        } else {
            mbar_arrive(bar);
        }
    }
    __syncthreads();  // block ids and weights in shared memory
    if (C > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sw = swizzle_mode(DI), sbo = 8 * DI;
            const uint64_t da0 = smem_desc(smem_u32(k_s), 16, sbo, sw);
            const uint64_t db = smem_desc(smem_u32(q_s), 16, sbo, sw);
            const uint32_t idesc = instr_desc(128, HT, 0, 0, 0, 0);
            bool ok = mbar_wait<true>(&sm.qbar, 0, abort_flag);
            for (int t = 0; t < n_tiles && ok; ++t) {
                if (!mbar_wait<true>(&sm.tbar[t], 0, abort_flag)) break;
                tc_fence_after();
                const uint64_t da = da0 + static_cast<uint64_t>((t * kTileRows * DI) >> 4);
                for (int k = 0; k < DI / 32; ++k) mma_f8f6f4(tmem + t * HT, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                mma_commit(&sm.mbar[t]);
            }
            // Before tensor memory is released and the key tiles are reused:
            // every issued MMA has completed and every key copy has landed.
            mma_commit(&sm.done);
            unsigned long long t0 = global_ns();
            while (!mbar_try_wait(&sm.done, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
            for (int t = 0; t < n_tiles; ++t) {
                t0 = global_ns();
                while (!mbar_try_wait(&sm.tbar[t], 0) && global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ scores
        const int row = warp * 32 + lane;                                  // row within a tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t dst0 = cluster_map(smem_u32(allk), 0);
        const uint32_t dstb = cluster_map(smem_u32(allb), 0) + rank * a.bpc * 4;
        if (row < a.bpc) st_cluster_u32(dstb + row * 4, static_cast<uint32_t>(sm.blk[row]));
        for (int t = 0; t < n_tiles; ++t) {
            if (!mbar_wait<true>(&sm.mbar[t], 0, abort_flag)) break;
            tc_fence_after();
            float s = 0.f;
            {
                // 32 heads' accumulators at a time (registers are few at 1,024 threads)
                constexpr int HC = HT < 32 ? HT : 32;
                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < HT; c0 += HC) {
                    uint32_t r[HC];
#pragma unroll
                    for (int c = 0; c < HC; c += 16)
                        tmem_ld16(tmem + lane_off + t * HT + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(&r[c]));
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < HC; h += 4) {
                        s0 = fmaf(sm.w[c0 + h], fmaxf(__uint_as_float(r[h]), 0.f), s0);
                        s1 = fmaf(sm.w[c0 + h + 1], fmaxf(__uint_as_float(r[h + 1]), 0.f), s1);
                        s2 = fmaf(sm.w[c0 + h + 2], fmaxf(__uint_as_float(r[h + 2]), 0.f), s2);
                        s3 = fmaf(sm.w[c0 + h + 3], fmaxf(__uint_as_float(r[h + 3]), 0.f), s3);
                    }
                }
                s = (s0 + s1) + (s2 + s3);
            }
            const int local = t * kTileRows + row;      // candidate within this CTA
            if (local < a.bpc * kPoolBlock) {
                const int32_t blk = sm.blk[local >> 3];
                const bool valid = blk >= 0 && blk * kPoolBlock + (local & 7) < Lp;
                const int cand = static_cast<int>(rank) * a.bpc * kPoolBlock + local;
                st_cluster_u32(dst0 + cta_select::key_slot(cand) * 4, valid ? score_key(s) : 0u);
            }
        }
    }

    // Every CTA's keys are in CTA 0 after this barrier.
    tc_fence_before();
    __syncthreads();
    if (C > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (*abort_flag && tid == 0) raise_status(a.status, CSA_DEV_TIMEOUT);
    if (rank != 0) return;

    write_selection(allk, allb, C * a.bpc * kPoolBlock, a.K, a.idx + static_cast<int64_t>(unit) * a.K, sc);
}

// Arrival counters of pool_spread_kernel: a library-owned array, zero when the
// library is loaded; each launch leaves its counters at 0 again (the last
// arrival wraps them).  Launches take consecutive ranges in turn, one counter
// per query, so only launches kSpreadCounters queries apart in issue order
// share a counter.  In host code this name is only a stand-in for the device
// array: the kernel gets the device address looked up below.
constexpr int kSpreadCounters = 1 << 16;
static __device__ unsigned int g_spread_counters[kSpreadCounters];

// The same Reindex layer spread over one CTA per 128-row tile of the pool
// (16 blocks), with no cluster: a cluster holds at most 16 CTAs, each of which
// must then copy 128 KB of keys at one SM's share of the L2's bandwidth.  Each
// CTA scores its tile and stores its rows' order-preserving keys to global
// memory (the caller's workspace); every thread fences its stores, and one
// thread counts the CTA's arrival with atomicInc on the query's counter.  The
// CTA that arrives last (the counter then wraps back to 0 by itself) reads
// every key of the pool from the L2 and selects, as CTA 0 of the cluster
// kernel does.  No CTA waits for another.
struct SpreadArgs {
    int P, HI, cap, DI;
    const int32_t *lengths;
    const int32_t *pool;        // [units][pool_blocks], ascending, -1 padded
    int pool_blocks;
    const float *w;             // [units][HI]
    int K;
    int32_t *idx;               // [units][K]
    uint32_t *keys;             // [units][pool_blocks * 8] (workspace)
    unsigned int *counters;     // [units] arrival counters, 0 between launches
    int *status;
};

struct SpreadSmem {
    uint64_t tbar, mbar, qbar, done;
    float w[64];
    int32_t blk[16];
    uint32_t tmem_slot;
    int abort;
    int last;
};

constexpr int kSpreadBlocks = kTileRows / kPoolBlock;  // 16 pool blocks per CTA
constexpr size_t kSpreadSmemBytes = (sizeof(SpreadSmem) + 1023) & ~size_t(1023);  // keeps the keys 1024-aligned

template <int HT>
__global__ void __launch_bounds__(kThreads, 1)
    pool_spread_kernel(const __grid_constant__ CUtensorMap keys8, const __grid_constant__ CUtensorMap qmap,
                       SpreadArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int DI = a.DI;
    uint8_t *k_s = base;                                       // [128 rows][DI] key tile
    uint8_t *q_s = k_s + kTileRows * DI;                       // [HT rows][DI] indexer query
    // the barriers first (8-byte aligned at a 1024-byte offset), then the last
    // CTA's keys, block ids and selection scratch
    SpreadSmem &sm = *reinterpret_cast<SpreadSmem *>(q_s + ((HT * DI + 1023) & ~1023));
    uint32_t *allk = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(&sm) + kSpreadSmemBytes);
    int32_t *allb = reinterpret_cast<int32_t *>(allk + kMaxCand);                    // last CTA: [blocks]
    cta_select::Scratch &sc = *reinterpret_cast<cta_select::Scratch *>(allb + kMaxCluster * kBlocksPerCta);
    volatile int *abort_flag = &sm.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.y, cta = blockIdx.x, ctas = gridDim.x;
    const int n = a.pool_blocks * kPoolBlock;
    constexpr uint32_t kCols = HT < 32 ? 32 : HT;

    if (tid == 0) {
        mbar_init(&sm.tbar, kSpreadBlocks);
        mbar_init(&sm.mbar, 1);
        mbar_init(&sm.qbar, 1);
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&keys8);
        prefetch_tensormap(&qmap);
    }
    if (warp == 4) {
        tmem_alloc(&sm.tmem_slot, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;

    // Below: reads of what earlier work on the stream wrote.
    pdl_wait();
    pdl_trigger();
    const int b = unit / a.P, p = unit % a.P;
    const int cap_blocks = (a.cap + kPoolBlock - 1) / kPoolBlock;
    // the block ids first: the key copies wait on them, the length only on the epilogue
    const int jb = cta * kSpreadBlocks + tid;
    int32_t blk = (tid < kSpreadBlocks && jb < a.pool_blocks) ? a.pool[static_cast<int64_t>(unit) * a.pool_blocks + jb] : -1;
    const int Lp = min(a.lengths[b], a.cap) - a.P + 1 + p;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.qbar, static_cast<uint32_t>(HT * DI));
        tma_load_2d(q_s, &qmap, &sm.qbar, 0, unit * a.HI);
    }
    if (tid < HT) sm.w[tid] = tid < a.HI ? a.w[static_cast<int64_t>(unit) * a.HI + tid] : 0.f;
    if (tid < kSpreadBlocks) {
        // one pool block per thread: its id, and the copy of its 8 key rows
        if (blk >= cap_blocks) blk = -1;
        sm.blk[tid] = blk;
        if (blk >= 0) {
            mbar_arrive_expect_tx(&sm.tbar, static_cast<uint32_t>(kPoolBlock * DI));
            tma_load_2d(k_s + tid * kPoolBlock * DI, &keys8, &sm.tbar, 0, b * a.cap + blk * kPoolBlock);
        } else {
            mbar_arrive(&sm.tbar);
        }
    }
    __syncthreads();  // block ids and weights in shared memory

    if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sw = swizzle_mode(DI), sbo = 8 * DI;
            const uint64_t da = smem_desc(smem_u32(k_s), 16, sbo, sw);
            const uint64_t db = smem_desc(smem_u32(q_s), 16, sbo, sw);
            const uint32_t idesc = instr_desc(128, HT, 0, 0, 0, 0);
            if (mbar_wait<true>(&sm.qbar, 0, abort_flag) && mbar_wait<true>(&sm.tbar, 0, abort_flag)) {
                tc_fence_after();
                for (int k = 0; k < DI / 32; ++k) mma_f8f6f4(tmem, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                mma_commit(&sm.mbar);
            }
            // Before tensor memory is released: every issued MMA has completed
            // and every key copy has landed.
            mma_commit(&sm.done);
            unsigned long long t0 = global_ns();
            while (!mbar_try_wait(&sm.done, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
            t0 = global_ns();
            while (!mbar_try_wait(&sm.tbar, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ scores
        const int row = warp * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const int cand = cta * kTileRows + row;
        if (mbar_wait<true>(&sm.mbar, 0, abort_flag)) {
            tc_fence_after();
            constexpr int HC = HT < 32 ? HT : 32;
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < HT; c0 += HC) {
                uint32_t r[HC];
#pragma unroll
                for (int c = 0; c < HC; c += 16)
                    tmem_ld16(tmem + lane_off + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(&r[c]));
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < HC; h += 4) {
                    s0 = fmaf(sm.w[c0 + h], fmaxf(__uint_as_float(r[h]), 0.f), s0);
                    s1 = fmaf(sm.w[c0 + h + 1], fmaxf(__uint_as_float(r[h + 1]), 0.f), s1);
                    s2 = fmaf(sm.w[c0 + h + 2], fmaxf(__uint_as_float(r[h + 2]), 0.f), s2);
                    s3 = fmaf(sm.w[c0 + h + 3], fmaxf(__uint_as_float(r[h + 3]), 0.f), s3);
                }
            }
            const float sc_row = (s0 + s1) + (s2 + s3);
            if (cand < n) {
                const int32_t blk = sm.blk[row >> 3];
                const bool valid = blk >= 0 && blk * kPoolBlock + (row & 7) < Lp;
                a.keys[static_cast<int64_t>(unit) * n + cand] = valid ? score_key(sc_row) : 0u;
            }
        } else if (cand < n) {
            a.keys[static_cast<int64_t>(unit) * n + cand] = 0u;  // timed out: no candidate
        }
        __threadfence();  // this thread's key, before the CTA's arrival is counted
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
    if (tid == 0) {
        // Every CTA arrives exactly once; the last arrival wraps the counter to 0.
        const unsigned int old = atomicInc(a.counters + unit, static_cast<unsigned int>(ctas - 1));
        sm.last = old == static_cast<unsigned int>(ctas - 1);
        if (*abort_flag) raise_status(a.status, CSA_DEV_TIMEOUT);
    }
    __syncthreads();
    if (!sm.last) return;

    // ---- the last CTA of this query: every key and block id of its pool
    __threadfence();  // the other CTAs' keys, counted before this arrival
    const uint4 *src = reinterpret_cast<const uint4 *>(a.keys + static_cast<int64_t>(unit) * n);
    const int nq = n / 4;
#pragma unroll
    for (int u = 0; u < kMaxCand / 4 / kThreads; ++u) {
        const int q = u * kThreads + tid;
        if (q < nq) *reinterpret_cast<uint4 *>(allk + cta_select::key_slot(4 * q)) = __ldcg(src + q);
    }
    {
        // the block ids (at most kMaxCluster * kBlocksPerCta): every load in
        // flight at once, beside the keys'
        constexpr int kIdLoads = kMaxCluster * kBlocksPerCta / kThreads;
        int32_t bl[kIdLoads];
#pragma unroll
        for (int u = 0; u < kIdLoads; ++u) {
            const int j = u * kThreads + tid;
            bl[u] = j < a.pool_blocks ? a.pool[static_cast<int64_t>(unit) * a.pool_blocks + j] : -1;
        }
#pragma unroll
        for (int u = 0; u < kIdLoads; ++u) {
            const int j = u * kThreads + tid;
            if (j < a.pool_blocks) allb[j] = bl[u] >= cap_blocks ? -1 : bl[u];
        }
    }
    __syncthreads();
    write_selection(allk, allb, n, a.K, a.idx + static_cast<int64_t>(unit) * a.K, sc);
}

// A Full layer that also keeps a pool of at least K blocks selects its top K
// rows among the pool's rows, from the scores the scan wrote.  This is exact:
// a block outside the pool has at least pool_keep >= K blocks ranked above it
// (best member score, then lower block id), and each of those holds a visible
// row that outranks every row of that block (a higher score, or an equal
// score at a lower row id), so none of its rows is among the top K.  One CTA
// per (sequence, position) reads the pool's rows' scores and selects.
struct RowsArgs {
    const float *scores;    // [units][ld]
    int64_t ld;
    const int32_t *lengths;
    int cap, P;
    const int32_t *pool;    // [units][pool_blocks], ascending, -1 padded
    int pool_blocks;
    int K;
    int32_t *idx;           // [units][K]
};

__global__ void __launch_bounds__(kThreads, 1) pool_rows_kernel(RowsArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint32_t *allk = reinterpret_cast<uint32_t *>(smem_raw);       // [pool rows] keys
    int32_t *allb = reinterpret_cast<int32_t *>(allk + kMaxCand);   // [pool blocks] ids
    cta_select::Scratch &sc = *reinterpret_cast<cta_select::Scratch *>(allb + kMaxCluster * kBlocksPerCta);
    const int tid = threadIdx.x;
    const int unit = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int b = unit / a.P, p = unit % a.P;
    const int Lp = min(a.lengths[b], a.cap) - a.P + 1 + p;
    const int cap_blocks = (a.cap + kPoolBlock - 1) / kPoolBlock;
    const int32_t *prow = a.pool + static_cast<int64_t>(unit) * a.pool_blocks;
    const float *srow = a.scores + static_cast<int64_t>(unit) * a.ld;
    const int n = a.pool_blocks * kPoolBlock;
    // Each block's 8 scores are two 16-byte loads (row ids are multiples of 8
    // and ld a multiple of 4); four blocks per thread are in flight at once.
    // A thread reads its blocks' ids itself (all four loads in flight), so its
    // score loads wait on those alone.
    for (int j0 = tid; j0 < a.pool_blocks; j0 += kU * kThreads) {
        float4 v[kU][2];
        int32_t blk[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = j0 + u * kThreads;
            const int32_t x = j < a.pool_blocks ? prow[j] : -1;
            blk[u] = x >= cap_blocks ? -1 : x;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = j0 + u * kThreads;
            if (j < a.pool_blocks) allb[j] = blk[u];
            const int64_t r0 = static_cast<int64_t>(blk[u] >= 0 ? blk[u] : 0) * kPoolBlock;
            if (blk[u] >= 0 && r0 + kPoolBlock <= a.ld) {
                const float4 *sp = reinterpret_cast<const float4 *>(srow + r0);
                v[u][0] = __ldg(sp);
                v[u][1] = __ldg(sp + 1);
            } else {
                // a block that reaches past the row's end (capacity not a
                // multiple of 8): its rows one by one, within the row
                float t[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) t[m] = (blk[u] >= 0 && r0 + m < a.ld) ? __ldg(srow + r0 + m) : 0.f;
                v[u][0] = make_float4(t[0], t[1], t[2], t[3]);
                v[u][1] = make_float4(t[4], t[5], t[6], t[7]);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = j0 + u * kThreads;
            if (j >= a.pool_blocks) continue;
            const float f[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
            uint32_t kq[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) kq[m] = (blk[u] >= 0 && blk[u] * kPoolBlock + m < Lp) ? score_key(f[m]) : 0u;
            // candidates 8j .. 8j+7 at their swizzled slots (cta_select::key_slot)
            uint4 *dst = reinterpret_cast<uint4 *>(allk);
            const int sw = (j >> 2) & 7;
            dst[(2 * j) ^ sw] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
            dst[(2 * j + 1) ^ sw] = make_uint4(kq[4], kq[5], kq[6], kq[7]);
        }
    }
    __syncthreads();
    write_selection(allk, allb, n, a.K, a.idx + static_cast<int64_t>(unit) * a.K, sc);
}

size_t pool_smem_bytes(int DI, int HT)
{
    return 1024 + static_cast<size_t>(kMaxTiles) * kTileRows * DI + ((static_cast<size_t>(HT) * DI + 1023) & ~size_t(1023)) +
           static_cast<size_t>(kMaxCand) * 4 + kMaxCluster * kBlocksPerCta * 4 + sizeof(PoolSmem);
}

size_t spread_smem_bytes(int DI, int HT)
{
    return 1024 + static_cast<size_t>(kTileRows) * DI + ((static_cast<size_t>(HT) * DI + 1023) & ~size_t(1023)) +
           kSpreadSmemBytes + static_cast<size_t>(kMaxCand) * 4 + kMaxCluster * kBlocksPerCta * 4 +
           sizeof(cta_select::Scratch);
}

int heads_tile(int HI) { return HI <= 16 ? 16 : (HI <= 32 ? 32 : 64); }

// The kernel's shared-memory limit is set once, to the largest request any
// call can make (128-byte keys).
template <int HT>
cudaError_t configure()
{
    static bool done = false;
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(pool_select_kernel<HT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pool_smem_bytes(128, HT)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(pool_select_kernel<HT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    done = e == cudaSuccess;
    return e;
}

}  // namespace

int pool_select_supported(const CacheView &c, int P, int HI, int pool_blocks, int K)
{
    // E4M3 keys, HI <= 64 heads (a multiple of 16 or 8 padded up), pools of
    // up to 2,048 blocks (16 CTAs of 128 blocks), K <= 16,384.
    return !c.mx && HI >= 1 && HI <= 64 && (c.DI == 32 || c.DI == 64 || c.DI == 128) && pool_blocks >= 1 &&
           pool_blocks <= kMaxCluster * kBlocksPerCta && K >= 1 && K <= kMaxCand && c.B * P >= 1;
}

int pool_rows_supported(int pool_keep, int K)
{
    return pool_keep >= K && pool_keep <= kMaxCluster * kBlocksPerCta;
}

cudaError_t launch_pool_rows(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                             int pool_blocks, int K, int32_t *idx, cudaStream_t st)
{
    if (!pool_rows_supported(pool_blocks, K)) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kMaxCand) * 4 + kMaxCluster * kBlocksPerCta * 4 + sizeof(cta_select::Scratch);
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(pool_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    RowsArgs a{};
    a.scores = scores;
    a.ld = ld;
    a.lengths = c.lengths;
    a.cap = c.cap;
    a.P = P;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    a.K = K;
    a.idx = idx;
    return launch_kernel(pool_rows_kernel, dim3(c.B * P), dim3(kThreads), smem, st, 0, a);
}

cudaError_t launch_pool_select(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, int K, int32_t *idx, int *status,
                               cudaStream_t st)
{
    if (!pool_select_supported(c, P, HI, pool_blocks, K)) return cudaErrorInvalidValue;
    const int units = c.B * P;
    const int HT = heads_tile(HI);
    // Cluster size: the smallest power of two whose CTAs hold at most 128 blocks each.
    int C = 1;
    while (C * kBlocksPerCta < pool_blocks) C *= 2;
    PoolArgs a{};
    a.P = P;
    a.HI = HI;
    a.cap = c.cap;
    a.DI = c.DI;
    a.lengths = c.lengths;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    a.bpc = (pool_blocks + C - 1) / C;
    a.w = w;
    a.K = K;
    a.idx = idx;
    a.status = status;
    const size_t smem = pool_smem_bytes(c.DI, HT);
    cudaError_t e = HT == 16 ? configure<16>() : (HT == 32 ? configure<32>() : configure<64>());
    if (e != cudaSuccess) return e;
    const CUtensorMapSwizzle sw = c.DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : c.DI == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap k8, qm;
    if (encode_tensor_map_2d_u8(&k8, c.ikeys, c.DI, static_cast<uint64_t>(c.B) * c.cap, c.DI, kPoolBlock, sw) !=
            CUDA_SUCCESS ||
        encode_tensor_map_2d_u8(&qm, iq, c.DI, static_cast<uint64_t>(units) * HI, c.DI, HT, sw) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int cl = C > 1 ? C : 0;
    if (HT == 16) return launch_kernel(pool_select_kernel<16>, dim3(C, units), dim3(kThreads), smem, st, cl, k8, qm, a);
    if (HT == 32) return launch_kernel(pool_select_kernel<32>, dim3(C, units), dim3(kThreads), smem, st, cl, k8, qm, a);
    return launch_kernel(pool_select_kernel<64>, dim3(C, units), dim3(kThreads), smem, st, cl, k8, qm, a);
}

int pool_spread_supported(const CacheView &c, int P, int HI, int pool_blocks, int K)
{
    return pool_select_supported(c, P, HI, pool_blocks, K) && c.B * P <= kSpreadCounters &&
           c.B * P <= 65535;
}

size_t pool_spread_keys_bytes(const CacheView &c, int P, int pool_blocks)
{
    return static_cast<size_t>(c.B) * P * pool_blocks * kPoolBlock * sizeof(uint32_t);
}

namespace {

constexpr int kMaxDevicesSpread = 64;
unsigned int *g_counters_ptr[kMaxDevicesSpread];
std::mutex g_counters_mu;
std::atomic<uint32_t> g_counter_next{0};

// Device address of the counters on the current device (looked up once per
// device, with that device current), and the first of `units` consecutive
// counters for this launch.
unsigned int *spread_counters(int units)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesSpread) return nullptr;
    unsigned int *base;
    {
        std::lock_guard<std::mutex> lk(g_counters_mu);
        if (!g_counters_ptr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_spread_counters) != cudaSuccess) return nullptr;
            g_counters_ptr[dev] = static_cast<unsigned int *>(p);
        }
        base = g_counters_ptr[dev];
    }
    uint32_t first = g_counter_next.fetch_add(static_cast<uint32_t>(units)) % kSpreadCounters;
    if (first + units > static_cast<uint32_t>(kSpreadCounters)) first = 0;
    return base + first;
}

template <int HT>
cudaError_t configure_spread()
{
    static bool done = false;
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(pool_spread_kernel<HT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(spread_smem_bytes(128, HT)));
    done = e == cudaSuccess;
    return e;
}

}  // namespace

cudaError_t launch_pool_spread(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, int K, int32_t *idx, uint32_t *keys,
                               int *status, cudaStream_t st)
{
    if (!pool_spread_supported(c, P, HI, pool_blocks, K) || !keys) return cudaErrorInvalidValue;
    const int units = c.B * P;
    unsigned int *counters = spread_counters(units);
    if (!counters) return cudaErrorInvalidValue;
    const int HT = heads_tile(HI);
    SpreadArgs a{};
    a.P = P;
    a.HI = HI;
    a.cap = c.cap;
    a.DI = c.DI;
    a.lengths = c.lengths;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    a.w = w;
    a.K = K;
    a.idx = idx;
    a.keys = keys;
    a.counters = counters;
    a.status = status;
    cudaError_t e = HT == 16 ? configure_spread<16>() : (HT == 32 ? configure_spread<32>() : configure_spread<64>());
    if (e != cudaSuccess) return e;
    const CUtensorMapSwizzle sw = c.DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : c.DI == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap k8, qm;
    if (encode_tensor_map_2d_u8(&k8, c.ikeys, c.DI, static_cast<uint64_t>(c.B) * c.cap, c.DI, kPoolBlock, sw) !=
            CUDA_SUCCESS ||
        encode_tensor_map_2d_u8(&qm, iq, c.DI, static_cast<uint64_t>(units) * HI, c.DI, HT, sw) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem = spread_smem_bytes(c.DI, HT);
    const dim3 grid((pool_blocks + kSpreadBlocks - 1) / kSpreadBlocks, units);
    if (HT == 16) return launch_kernel(pool_spread_kernel<16>, grid, dim3(kThreads), smem, st, 0, k8, qm, a);
    if (HT == 32) return launch_kernel(pool_spread_kernel<32>, grid, dim3(kThreads), smem, st, 0, k8, qm, a);
    return launch_kernel(pool_spread_kernel<64>, grid, dim3(kThreads), smem, st, 0, k8, qm, a);
}

}  // namespace csa
