// a3: top-K selection of row ids by indexer score, and the hierarchical pool.
// "DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section "The
// Paper": the query keeps only the top indices; "G2C Brief - DeepSeek
// V4.1-Flash", section "The hierarchical indexer": positions grouped in blocks
// of 8, each block scored by its best member, the top 2,048 blocks kept.
//
// One thread-block cluster per query row.  The row's candidates are split into
// contiguous chunks, one per CTA, and the K-th largest score is found by a
// most-significant-digit radix select over order-preserving 32-bit keys
// (digits of 11, 11 and 10 bits).  Each pass builds a per-CTA histogram in
// shared memory; the CTAs then read each other's histograms through
// distributed shared memory, so the whole selection needs no global scratch
// and no second kernel.  Chunks stay cached in shared memory between passes
// when they fit.  Ties at the threshold are resolved by lower row id: each CTA
// knows how many tied candidates precede its chunk.  Output ids are written
// in ascending order (CTA order, then chunk order), then -1 padding.
#include <cooperative_groups.h>

#include "common.cuh"
#include "csa_internal.h"

namespace cg = cooperative_groups;

namespace csa {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 2048;
constexpr int kSelCache = 12288;  // keys cached per CTA (48 KB)

struct SelArgs {
    const float *scores;
    int64_t ld;
    const int32_t *lengths;
    int P;
    const int32_t *pool;
    int pool_blocks;
    int block;  // 1: candidates are rows; 8: candidates are blocks of 8 rows (best member)
    int K;
    int32_t *out;
};

constexpr int kMaxCluster = 16;

// Per-CTA shared state.  CTAs of a cluster only ever WRITE into each other's
// shared memory (distributed shared-memory stores), and every such write is
// followed by a cluster barrier before it is read; no CTA loads from another
// CTA's shared memory.
struct SelShared {
    uint32_t hist[kBins];                 // this CTA's histogram of the current digit
    uint32_t stage[kBins];                // [src CTA][bins owned here]: pushed by every CTA
    uint32_t slice[kBins];                // summed bins owned here
    uint32_t totals[kMaxCluster];         // slice totals of every CTA (pushed)
    uint32_t valid_all[kMaxCluster];      // candidate counts of every CTA (pushed)
    uint32_t above_all[kMaxCluster];      // per-CTA count strictly above the threshold (pushed)
    uint32_t eq_all[kMaxCluster];         // per-CTA count at the threshold (pushed)
    uint32_t res_digit, res_gt, res_class;  // pushed by the CTA that owns the chosen digit
    uint32_t warp_tot[kSelWarps];
    uint32_t bcast;
};

// Candidate i of a row: its key (0 = not a candidate) and its output id.
struct RowView {
    const float *srow;
    const int32_t *prow;
    int L;
    int block;
    __device__ __forceinline__ uint32_t key(int64_t i, int32_t &id) const
    {
        if (prow) {
            const int32_t blk = prow[i >> 3];
            const int64_t row = static_cast<int64_t>(blk) * kPoolBlock + (i & 7);
            id = static_cast<int32_t>(row);
            return (blk >= 0 && row < L) ? score_key(srow[i]) : 0u;
        }
        id = static_cast<int32_t>(i);
        if (block == 1) return score_key(srow[i]);
        const int64_t r0 = i * kPoolBlock;
        float best = srow[r0];
        for (int m = 1; m < kPoolBlock; ++m)
            if (r0 + m < L) best = fmaxf(best, srow[r0 + m]);
        return score_key(best);
    }
    __device__ __forceinline__ int32_t id(int64_t i) const
    {
        if (prow) return prow[i >> 3] * kPoolBlock + static_cast<int32_t>(i & 7);
        return static_cast<int32_t>(i);
    }
};

// Block-wide exclusive scan of v (one value per thread); returns the exclusive
// prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_tot, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = lane < kSelWarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kSelWarps) warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const uint32_t before = (warp ? warp_tot[warp - 1] : 0) + x - v;
    *total = warp_tot[kSelWarps - 1];
    __syncthreads();
    return before;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t *warp_tot)
{
    uint32_t total;
    block_exclusive_scan(v, warp_tot, &total);
    return total;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(SelArgs a)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(dyn_smem);
    uint32_t *cache = reinterpret_cast<uint32_t *>(dyn_smem + sizeof(SelShared));

    const int r = blockIdx.y;
    const int b = r / a.P, p = r % a.P;
    const int L = a.lengths[b] - a.P + 1 + p;
    int64_t n;
    if (a.pool)
        n = static_cast<int64_t>(a.pool_blocks) * kPoolBlock;
    else if (L <= 0)
        n = 0;
    else
        n = a.block == 1 ? L : (L + kPoolBlock - 1) / kPoolBlock;
    RowView rv{a.scores + static_cast<int64_t>(r) * a.ld,
               a.pool ? a.pool + static_cast<int64_t>(r) * a.pool_blocks : nullptr, L, a.block};
    const int64_t chunk = (n + C - 1) / C;
    const int64_t e0 = min(n, rank * chunk), e1 = min(n, e0 + chunk);
    const int m = static_cast<int>(e1 - e0);
    const bool cached = m <= kSelCache;
    const int tid = threadIdx.x;

    const int lane = tid & 31;
    const int bpc = kBins / C;  // histogram bins owned by each CTA

    // Pass 0: count candidates, cache keys; every CTA learns every count.
    uint32_t cnt = 0;
    for (int i = tid; i < m; i += kSelThreads) {
        int32_t id;
        const uint32_t k = rv.key(e0 + i, id);
        if (cached) cache[i] = k;
        cnt += k != 0;
    }
    cnt = block_sum(cnt, sh.warp_tot);
    if (tid < C) cluster.map_shared_rank(&sh, tid)->valid_all[rank] = cnt;
    cluster.sync();
    uint32_t total_valid = 0;
    for (int q = 0; q < C; ++q) total_valid += sh.valid_all[q];

    const uint32_t K = static_cast<uint32_t>(a.K);
    uint32_t prefix = 0, above = 0, need = total_valid, local_above = 0, local_eq = cnt;
    int pbits = 0;
    if (total_valid > K) {
        for (int pass = 0; pass < 3; ++pass) {
            const int width = pass < 2 ? 11 : 10;
            const int shift = 32 - pbits - width;
            const uint32_t mask = (1u << width) - 1u;
            for (int i = tid; i < kBins; i += kSelThreads) sh.hist[i] = 0;
            if (tid == 0) {
                sh.bcast = 0;
                sh.res_gt = above;
                sh.res_class = 0;
            }
            __syncthreads();
            // Local histogram; lanes with the same digit add once (warp-aggregated).
            for (int base = 0; base < m; base += kSelThreads) {
                const int i = base + tid;
                uint32_t k = 0;
                if (i < m) {
                    if (cached) {
                        k = cache[i];
                    } else {
                        int32_t id;
                        k = rv.key(e0 + i, id);
                    }
                }
                const bool in = k != 0 && (pbits == 0 || (k >> (32 - pbits)) == prefix);
                const uint32_t digit = in ? ((k >> shift) & mask) : 0xFFFFFFFFu;
                const unsigned peers = __match_any_sync(0xFFFFFFFFu, digit);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], static_cast<uint32_t>(__popc(peers)));
            }
            __syncthreads();
            // Push each bin to the CTA that owns it.
            for (int i = tid; i < kBins; i += kSelThreads) {
                const int owner = i / bpc, j = i - owner * bpc;
                cluster.map_shared_rank(sh.stage, owner)[rank * bpc + j] = sh.hist[i];
            }
            cluster.sync();
            // Sum the owned bins over the sources; push the slice total everywhere.
            uint32_t part = 0;
            for (int j = tid; j < bpc; j += kSelThreads) {
                uint32_t g = 0;
                for (int q = 0; q < C; ++q) g += sh.stage[q * bpc + j];
                sh.slice[j] = g;
                part += g;
            }
            part = block_sum(part, sh.warp_tot);
            if (tid < C) cluster.map_shared_rank(&sh, tid)->totals[rank] = part;
            cluster.sync();
            // The slice holding the K-th largest key, scanning from the top.
            int owner = 0;
            uint32_t cum = above;
            for (int q = C - 1; q >= 0; --q) {
                if (cum + sh.totals[q] >= K) {
                    owner = q;
                    break;
                }
                cum += sh.totals[q];
            }
            if (rank == owner) {
                // Suffix sums over this slice's bins (each thread takes `per`
                // consecutive bins; threads are scanned in reverse order).
                const int per = (bpc + kSelThreads - 1) / kSelThreads;
                uint32_t s_mine = 0;
                for (int j = 0; j < per; ++j) {
                    const int bin = tid * per + j;
                    if (bin < bpc) s_mine += sh.slice[bin];
                }
                sh.hist[kSelThreads - 1 - tid] = s_mine;  // hist is free until the next pass
                __syncthreads();
                const uint32_t mirrored = sh.hist[tid];
                __syncthreads();
                uint32_t tot;
                const uint32_t excl = block_exclusive_scan(mirrored, sh.warp_tot, &tot);
                sh.hist[kSelThreads - 1 - tid] = excl;
                __syncthreads();
                uint32_t suf = cum + sh.hist[tid];  // keys in bins above my bins (whole cluster)
                for (int j = per - 1; j >= 0; --j) {
                    const int bin = tid * per + j;
                    if (bin >= bpc) continue;
                    const uint32_t gt = suf;
                    suf += sh.slice[bin];
                    if (gt < K && suf >= K) {
                        sh.bcast = static_cast<uint32_t>(owner * bpc + bin);
                        sh.res_gt = gt;
                        sh.res_class = sh.slice[bin];
                    }
                }
                __syncthreads();
                if (tid < C) {
                    SelShared *dst = cluster.map_shared_rank(&sh, tid);
                    dst->res_digit = sh.bcast;
                    dst->res_gt = sh.res_gt;
                    dst->res_class = sh.res_class;
                }
            }
            cluster.sync();
            // The local histogram was reused as scratch by the owner: recount
            // this CTA's share above and at the chosen digit from the keys.
            const uint32_t d = sh.res_digit & mask;
            const uint32_t gt = sh.res_gt;
            const uint32_t class_total = sh.res_class;
            uint32_t la = 0, le = 0;
            for (int i = tid; i < m; i += kSelThreads) {
                uint32_t k;
                if (cached) {
                    k = cache[i];
                } else {
                    int32_t id;
                    k = rv.key(e0 + i, id);
                }
                if (k != 0 && (pbits == 0 || (k >> (32 - pbits)) == prefix)) {
                    const uint32_t dg = (k >> shift) & mask;
                    la += dg > d;
                    le += dg == d;
                }
            }
            la = block_sum(la, sh.warp_tot);
            le = block_sum(le, sh.warp_tot);
            local_above += la;
            local_eq = le;
            above = gt;
            prefix = (prefix << width) | d;
            pbits += width;
            need = K - above;
            if (need == class_total) break;
        }
    }

    // Tied class: take the `need` candidates with the lowest ids.
    if (tid < C) {
        SelShared *dst = cluster.map_shared_rank(&sh, tid);
        dst->above_all[rank] = local_above;
        dst->eq_all[rank] = local_eq;
    }
    cluster.sync();  // last remote write: after this, CTAs only touch their own memory
    uint32_t tie_before = 0, out_before = 0, take = 0;
    for (int q = 0; q < C; ++q) {
        const uint32_t eq = sh.eq_all[q];
        const uint32_t tq = tie_before >= need ? 0u : min(eq, need - tie_before);
        if (q < rank) out_before += sh.above_all[q] + tq;
        if (q == rank) take = tq;
        tie_before += eq;
    }

    const uint32_t selected_total = total_valid > K ? K : total_valid;
    int32_t *orow = a.out + static_cast<int64_t>(r) * a.K;
    uint32_t run_ties = 0, run_sel = 0;
    for (int base = 0; base < m; base += kSelThreads) {
        const int i = base + tid;
        uint32_t k = 0;
        int32_t id = -1;
        if (i < m) {
            if (cached) {
                k = cache[i];
                id = rv.id(e0 + i);
            } else {
                k = rv.key(e0 + i, id);
            }
        }
        bool in_above = false, in_class = false;
        if (k != 0) {
            if (pbits == 0) {
                in_class = true;
            } else {
                const uint32_t top = k >> (32 - pbits);
                in_above = top > prefix;
                in_class = top == prefix;
            }
        }
        uint32_t tile_ties;
        const uint32_t ex_class = block_exclusive_scan(static_cast<uint32_t>(in_class), sh.warp_tot, &tile_ties);
        const bool sel = in_above || (in_class && run_ties + ex_class < take);
        uint32_t tot_sel;
        const uint32_t ex_sel = block_exclusive_scan(static_cast<uint32_t>(sel), sh.warp_tot, &tot_sel);
        if (sel) orow[out_before + run_sel + ex_sel] = id;
        run_ties += tile_ties;
        run_sel += tot_sel;
    }
    if (rank == C - 1)
        for (uint32_t j = selected_total + tid; j < K; j += kSelThreads) orow[j] = -1;
}

int g_max_cluster = 0;

}  // namespace

cudaError_t launch_select(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                          int pool_blocks, int block, int K, int32_t *out, int * /*status*/, cudaStream_t st)
{
    const int rows = c.B * P;
    if (rows == 0) return cudaSuccess;
    const size_t smem = sizeof(SelShared) + kSelCache * sizeof(uint32_t);
    if (g_max_cluster == 0) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        // Largest cluster size (power of two <= 16) that can be resident.
        g_max_cluster = 1;
        for (int cs = 16; cs >= 2; cs >>= 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cs, 1, 1);
            cfg.blockDim = dim3(kSelThreads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = cs;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, select_kernel, &cfg) == cudaSuccess && nclusters > 0) {
                g_max_cluster = cs;
                break;
            }
            cudaGetLastError();
        }
    }
    int64_t n_max = pool ? static_cast<int64_t>(pool_blocks) * kPoolBlock
                         : (block == 1 ? c.cap : (c.cap + kPoolBlock - 1) / kPoolBlock);
    int C = 1;
    while (C < g_max_cluster && ((n_max + C - 1) / C > kSelCache || static_cast<int64_t>(rows) * C < 2 * 148))
        C *= 2;
    SelArgs args{scores, ld, c.lengths, P, pool, pool_blocks, block, K, out};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, rows, 1);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, select_kernel, args);
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace csa
