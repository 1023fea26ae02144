// a3: top-K selection of row ids by indexer score, and the hierarchical pool.
// "DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section "The
// Paper": the query keeps only the top indices; "G2C Brief - DeepSeek
// V4.1-Flash", section "The hierarchical indexer": positions grouped in blocks
// of 8, each block scored by its best member, the top 2,048 blocks kept.
//
// One thread-block cluster per query row (or per segment of a very long row).
// The candidates are split into contiguous chunks, one per CTA, held in shared
// memory as order-preserving 32-bit keys.  The K-th largest key is found by a
// bucket select that adapts to the data: pass 0 finds the key range [lo, hi];
// each pass histograms the live range into at most 2048 buckets of 2^shift
// keys, so no pass wastes bins on bit patterns no score has.  The CTAs push
// their histograms to the CTA that owns each bucket range (distributed shared
// memory stores, then a cluster barrier); the owner of the bucket holding the
// K-th key broadcasts it.  At most three passes resolve a 32-bit key.  Ties at
// the threshold go to the lower row id: each CTA knows how many tied
// candidates precede its chunk.  Output ids are written in ascending order.
//
// Rows longer than 16 x 12288 candidates are split into segments: stage 1
// keeps each segment's own top K (with scores) in the workspace; stage 2
// selects the row's top K among those, which is exact because every member of
// the row's top K is in its segment's top K (the same order decides both).
#include <cooperative_groups.h>

#include "common.cuh"
#include "csa_internal.h"

namespace cg = cooperative_groups;

namespace csa {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 2048;
constexpr int kSelCache = 12288;  // keys held per CTA (48 KB)
constexpr int kMaxCluster = 16;

enum SelSource { kRows = 0, kBlocks = 1, kPoolRows = 2, kPairs = 3 };

struct SelArgs {
    int source;
    const float *scores;       // kRows/kBlocks/kPoolRows: [rows][ld];  kPairs: [rows][n_pairs]
    int64_t ld;
    const int32_t *lengths;
    int P;
    const int32_t *pool;       // kPoolRows: [rows][pool_blocks]
    int pool_blocks;
    const int32_t *pair_ids;   // kPairs: [rows][n_pairs], -1 = empty
    int n_pairs;
    int segments;              // > 1: this launch writes per-segment candidates
    int64_t seg_len;
    int K;                     // keys kept per row (or per segment)
    int32_t *out_ids;          // [rows*segments][K]
    float *out_scores;         // segments > 1: [rows*segments][K]
};

// Per-CTA shared state.  CTAs of a cluster only ever WRITE into each other's
// shared memory, and every such write is followed by a cluster barrier before
// it is read; no CTA loads from another CTA's shared memory.
struct SelShared {
    uint32_t hist[kBins];                 // this CTA's histogram of the current pass
    uint32_t stage[kBins];                // [source CTA][buckets owned here], pushed by every CTA
    uint32_t slice[kBins];                // owned buckets summed over the cluster
    uint32_t scratch[kSelThreads];
    uint32_t cnt_all[kMaxCluster];        // pass 0 counts (pushed)
    uint32_t min_all[kMaxCluster];
    uint32_t max_all[kMaxCluster];
    uint32_t totals[kMaxCluster];         // owned-slice totals (pushed)
    uint32_t sel_all[kMaxCluster];        // selected counts per CTA (pushed)
    uint32_t eq_all[kMaxCluster];         // counts at the threshold per CTA (pushed)
    uint32_t res_bucket, res_gt, res_class;
    uint32_t warp_tot[kSelWarps];
};

struct RowView {
    int source;
    const float *s;
    const int32_t *prow;
    const int32_t *ids;
    int L;
    __device__ __forceinline__ uint32_t key(int64_t i) const
    {
        switch (source) {
        case kRows: return score_key(s[i]);
        case kBlocks: {
            const int64_t r0 = i * kPoolBlock;
            float best = s[r0];
            for (int m = 1; m < kPoolBlock; ++m)
                if (r0 + m < L) best = fmaxf(best, s[r0 + m]);
            return score_key(best);
        }
        case kPoolRows: {
            const int32_t blk = prow[i >> 3];
            const int64_t row = static_cast<int64_t>(blk) * kPoolBlock + (i & 7);
            return (blk >= 0 && row < L) ? score_key(s[i]) : 0u;
        }
        default: return ids[i] >= 0 ? score_key(s[i]) : 0u;
        }
    }
    __device__ __forceinline__ int32_t id(int64_t i) const
    {
        switch (source) {
        case kPoolRows: return prow[i >> 3] * kPoolBlock + static_cast<int32_t>(i & 7);
        case kPairs: return ids[i];
        default: return static_cast<int32_t>(i);
        }
    }
};

// Inverse of score_key (for the candidates a segment hands to stage 2).
__device__ __forceinline__ float key_score(uint32_t k)
{
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

// Block-wide exclusive scan of one value per thread; *total gets the sum.
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
        if (lane < kSelWarps) warp_tot[lane] = t;
    }
    __syncthreads();
    const uint32_t before = (warp ? warp_tot[warp - 1] : 0) + x - v;
    *total = warp_tot[kSelWarps - 1];
    __syncthreads();
    return before;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t *warp_tot)
{
    uint32_t t;
    block_exclusive_scan(v, warp_tot, &t);
    return t;
}

__device__ __forceinline__ uint32_t block_min(uint32_t v, uint32_t *scratch)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = 0xFFFFFFFFu;
    for (int w = 0; w < kSelWarps; ++w) r = min(r, scratch[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t *scratch)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = 0;
    for (int w = 0; w < kSelWarps; ++w) r = max(r, scratch[w]);
    __syncthreads();
    return r;
}

enum Rule { kAll, kRange, kTies };

__device__ __forceinline__ bool selected(Rule rule, uint32_t k, uint32_t lo, uint32_t hi, uint32_t &tie_rank,
                                         uint32_t take)
{
    if (rule == kAll) return k != 0;
    if (rule == kRange) return k != 0 && k >= lo;
    if (k == lo) return tie_rank++ < take;
    return k > hi;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(SelArgs a)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(dyn_smem);
    uint32_t *cache = reinterpret_cast<uint32_t *>(dyn_smem + sizeof(SelShared));
    const int tid = threadIdx.x, lane = tid & 31;

    const int row = blockIdx.y / a.segments, seg = blockIdx.y % a.segments;
    int64_t n;
    RowView rv{a.source, nullptr, nullptr, nullptr, 0};
    if (a.source == kPairs) {
        n = a.n_pairs;
        rv.s = a.scores + static_cast<int64_t>(row) * a.n_pairs;
        rv.ids = a.pair_ids + static_cast<int64_t>(row) * a.n_pairs;
    } else {
        const int b = row / a.P, p = row % a.P;
        const int L = a.lengths[b] - a.P + 1 + p;
        rv.s = a.scores + static_cast<int64_t>(row) * a.ld;
        rv.L = L;
        if (a.source == kPoolRows) {
            n = static_cast<int64_t>(a.pool_blocks) * kPoolBlock;
            rv.prow = a.pool + static_cast<int64_t>(row) * a.pool_blocks;
        } else {
            n = L <= 0 ? 0 : (a.source == kRows ? L : (L + kPoolBlock - 1) / kPoolBlock);
        }
    }
    const int64_t s0 = min(n, seg * a.seg_len), s1 = min(n, s0 + a.seg_len);
    const int64_t chunk = (s1 - s0 + C - 1) / C;
    const int64_t e0 = min(s1, s0 + rank * chunk), e1 = min(s1, e0 + chunk);
    const int m = static_cast<int>(e1 - e0);  // <= kSelCache (the host sizes the cluster so)

    // Pass 0: keys into shared memory; count, min and max of the candidates.
    uint32_t cnt = 0, kmin = 0xFFFFFFFFu, kmax = 0;
    for (int i = tid; i < m; i += kSelThreads) {
        const uint32_t k = rv.key(e0 + i);
        cache[i] = k;
        if (k) {
            ++cnt;
            kmin = min(kmin, k);
            kmax = max(kmax, k);
        }
    }
    cnt = block_sum(cnt, sh.warp_tot);
    kmin = block_min(kmin, sh.scratch);
    kmax = block_max(kmax, sh.scratch);
    if (tid < C) {
        SelShared *dst = cluster.map_shared_rank(&sh, tid);
        dst->cnt_all[rank] = cnt;
        dst->min_all[rank] = kmin;
        dst->max_all[rank] = kmax;
    }
    cluster.sync();
    uint32_t total = 0, lo = 0xFFFFFFFFu, hi = 0;
    for (int q = 0; q < C; ++q) {
        total += sh.cnt_all[q];
        lo = min(lo, sh.min_all[q]);
        hi = max(hi, sh.max_all[q]);
    }

    const uint32_t K = static_cast<uint32_t>(a.K);
    // Selection rule after the passes:
    //   kAll  : every candidate (total <= K)
    //   kRange: every key >= lo
    //   kTies : keys > hi, plus the first `need` keys equal to lo (== hi) in id order
    Rule rule = kAll;
    uint32_t need = 0, local_above = 0, local_eq = 0;
    if (total > K) {
        uint32_t above = 0;
        rule = kRange;
        for (int pass = 0; pass < 4; ++pass) {
            if (lo == hi) {  // every live key is equal: the ties rule decides
                rule = kTies;
                need = K - above;
                uint32_t le = 0;
                for (int i = tid; i < m; i += kSelThreads) le += cache[i] == lo;
                local_eq = block_sum(le, sh.warp_tot);
                break;
            }
            const uint32_t span = hi - lo;
            const int bits = 32 - __clz(span);
            const int shift = bits > 11 ? bits - 11 : 0;
            const int nb = static_cast<int>(span >> shift) + 1;  // <= 2048 buckets
            const int bpc = (nb + C - 1) / C;                    // buckets owned per CTA
            for (int i = tid; i < kBins; i += kSelThreads) sh.hist[i] = 0;
            if (tid == 0) {
                sh.res_bucket = 0;
                sh.res_gt = above;
                sh.res_class = 0;
            }
            __syncthreads();
            for (int base = 0; base < m; base += kSelThreads) {
                const int i = base + tid;
                const uint32_t k = i < m ? cache[i] : 0u;
                const bool in = k != 0 && k >= lo && k <= hi;
                const uint32_t bkt = in ? (k - lo) >> shift : 0xFFFFFFFFu;
                const unsigned peers = __match_any_sync(0xFFFFFFFFu, bkt);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bkt], static_cast<uint32_t>(__popc(peers)));
            }
            __syncthreads();
            for (int i = tid; i < nb; i += kSelThreads) {
                const int owner = i / bpc;
                cluster.map_shared_rank(sh.stage, owner)[rank * bpc + (i - owner * bpc)] = sh.hist[i];
            }
            cluster.sync();
            uint32_t part = 0;
            const int own0 = rank * bpc, own_n = max(0, min(nb - own0, bpc));
            for (int j = tid; j < own_n; j += kSelThreads) {
                uint32_t g = 0;
                for (int q = 0; q < C; ++q) g += sh.stage[q * bpc + j];
                sh.slice[j] = g;
                part += g;
            }
            part = block_sum(part, sh.warp_tot);
            if (tid < C) cluster.map_shared_rank(&sh, tid)->totals[rank] = part;
            cluster.sync();
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
                // Suffix sums over the owned buckets, highest first: each thread
                // takes `per` consecutive buckets; threads are scanned in reverse.
                const int per = (own_n + kSelThreads - 1) / kSelThreads;
                uint32_t mine = 0;
                for (int j = 0; j < per; ++j) {
                    const int bkt = tid * per + j;
                    if (bkt < own_n) mine += sh.slice[bkt];
                }
                sh.scratch[kSelThreads - 1 - tid] = mine;
                __syncthreads();
                const uint32_t mirrored = sh.scratch[tid];
                __syncthreads();
                uint32_t t_;
                const uint32_t excl = block_exclusive_scan(mirrored, sh.warp_tot, &t_);
                sh.scratch[kSelThreads - 1 - tid] = excl;
                __syncthreads();
                uint32_t suf = cum + sh.scratch[tid];
                for (int j = per - 1; j >= 0; --j) {
                    const int bkt = tid * per + j;
                    if (bkt >= own_n) continue;
                    const uint32_t gt = suf;
                    suf += sh.slice[bkt];
                    if (gt < K && suf >= K) {
                        sh.res_bucket = static_cast<uint32_t>(own0 + bkt);
                        sh.res_gt = gt;
                        sh.res_class = sh.slice[bkt];
                    }
                }
                __syncthreads();
                if (tid < C) {
                    SelShared *dst = cluster.map_shared_rank(&sh, tid);
                    dst->res_bucket = sh.res_bucket;
                    dst->res_gt = sh.res_gt;
                    dst->res_class = sh.res_class;
                }
            }
            cluster.sync();
            const uint32_t d = sh.res_bucket;
            const uint32_t cls = sh.res_class;
            above = sh.res_gt;
            uint32_t la = 0;
            for (int i = tid; i < nb; i += kSelThreads)
                if (static_cast<uint32_t>(i) > d) la += sh.hist[i];
            local_above += block_sum(la, sh.warp_tot);
            local_eq = sh.hist[d];
            const uint32_t nlo = lo + (d << shift);
            const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << shift) - 1);
            hi = static_cast<uint32_t>(nhi < hi ? nhi : hi);
            lo = nlo;
            need = K - above;
            if (need == cls) {  // the whole bucket is selected
                rule = kRange;
                break;
            }
        }
    }

    // Per-CTA selected counts (and counts at the threshold) to every CTA.
    const uint32_t mine_sel = rule == kAll ? cnt : (rule == kRange ? local_above + local_eq : local_above);
    if (tid < C) {
        SelShared *dst = cluster.map_shared_rank(&sh, tid);
        dst->sel_all[rank] = mine_sel;
        dst->eq_all[rank] = local_eq;
    }
    cluster.sync();  // last remote write: from here on CTAs touch only their own memory
    uint32_t out_before = 0, tie_before = 0, take = 0;
    for (int q = 0; q < C; ++q) {
        uint32_t tq = 0;
        if (rule == kTies) tq = tie_before >= need ? 0u : min(sh.eq_all[q], need - tie_before);
        if (q < rank) out_before += sh.sel_all[q] + tq;
        if (q == rank) take = tq;
        tie_before += sh.eq_all[q];
    }

    // Collect: thread t owns keys [t*E, t*E+E) of the chunk, so the block scans
    // give each thread its tie rank and its output position in id order.
    const int E = (m + kSelThreads - 1) / kSelThreads;
    const int i0 = min(m, tid * E), i1 = min(m, i0 + E);
    uint32_t t_;
    uint32_t my_ties = 0;
    if (rule == kTies)
        for (int i = i0; i < i1; ++i) my_ties += cache[i] == lo;
    const uint32_t ties_before_me = rule == kTies ? block_exclusive_scan(my_ties, sh.warp_tot, &t_) : 0u;
    uint32_t my_sel = 0;
    {
        uint32_t tr = ties_before_me;
        for (int i = i0; i < i1; ++i) my_sel += selected(rule, cache[i], lo, hi, tr, take);
    }
    const uint32_t pos0 = out_before + block_exclusive_scan(my_sel, sh.warp_tot, &t_);
    const int64_t obase = static_cast<int64_t>(blockIdx.y) * a.K;
    {
        uint32_t tr = ties_before_me, pos = pos0;
        for (int i = i0; i < i1; ++i) {
            const uint32_t k = cache[i];
            if (selected(rule, k, lo, hi, tr, take)) {
                a.out_ids[obase + pos] = rv.id(e0 + i);
                if (a.out_scores) a.out_scores[obase + pos] = key_score(k);
                ++pos;
            }
        }
    }
    const uint32_t selected_total = total > K ? K : total;
    if (rank == C - 1)
        for (uint32_t j = selected_total + tid; j < K; j += kSelThreads) {
            a.out_ids[obase + j] = -1;
            if (a.out_scores) a.out_scores[obase + j] = -INFINITY;
        }
}

int g_max_cluster = 0;

cudaError_t launch(const SelArgs &args, int grid_rows, int64_t n_per_cluster, cudaStream_t st)
{
    const size_t smem = sizeof(SelShared) + kSelCache * sizeof(uint32_t);
    if (g_max_cluster == 0) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        g_max_cluster = 1;
        for (int cs = kMaxCluster; cs >= 2; cs >>= 1) {
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
    int C = 1;
    while (C < g_max_cluster &&
           ((n_per_cluster + C - 1) / C > kSelCache || static_cast<int64_t>(grid_rows) * C < 2 * 148))
        C *= 2;
    if ((n_per_cluster + C - 1) / C > kSelCache) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, grid_rows, 1);
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

struct SelPlan {
    int64_t n_max;
    int segments;
    int64_t seg_len;
    int k_seg;
};

SelPlan sel_plan(const CacheView &c, const int32_t *pool, int pool_blocks, int block, int K)
{
    SelPlan p;
    p.n_max = pool ? static_cast<int64_t>(pool_blocks) * kPoolBlock
                   : (block == 1 ? c.cap : (c.cap + kPoolBlock - 1) / kPoolBlock);
    const int64_t one_cluster = static_cast<int64_t>(kMaxCluster) * kSelCache;
    p.segments = static_cast<int>((p.n_max + one_cluster - 1) / one_cluster);
    if (p.segments < 1) p.segments = 1;
    p.seg_len = (p.n_max + p.segments - 1) / p.segments;
    p.k_seg = static_cast<int>(p.seg_len < K ? p.seg_len : K);
    return p;
}

}  // namespace

size_t select_workspace_bytes(const CacheView &c, int P, const int32_t *pool, int pool_blocks, int block, int K)
{
    const SelPlan p = sel_plan(c, pool, pool_blocks, block, K);
    if (p.segments == 1) return 0;
    const size_t n = static_cast<size_t>(c.B) * P * p.segments * p.k_seg;
    return (n * 4 + 255) / 256 * 256 + n * 4;
}

int select_supported(const CacheView &c, const int32_t *pool, int pool_blocks, int block, int K)
{
    const SelPlan p = sel_plan(c, pool, pool_blocks, block, K);
    return p.segments == 1 ||
           static_cast<int64_t>(p.segments) * p.k_seg <= static_cast<int64_t>(kMaxCluster) * kSelCache;
}

cudaError_t launch_select(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                          int pool_blocks, int block, int K, int32_t *out, void *ws, size_t ws_bytes,
                          cudaStream_t st)
{
    const int rows = c.B * P;
    if (rows == 0) return cudaSuccess;
    const SelPlan p = sel_plan(c, pool, pool_blocks, block, K);
    SelArgs a{};
    a.source = pool ? kPoolRows : (block == 1 ? kRows : kBlocks);
    a.scores = scores;
    a.ld = ld;
    a.lengths = c.lengths;
    a.P = P;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    if (p.segments == 1) {
        a.segments = 1;
        a.seg_len = p.n_max;
        a.K = K;
        a.out_ids = out;
        return launch(a, rows, p.n_max, st);
    }
    // Stage 1: each segment's own top k_seg, with scores, into the workspace.
    if (!ws || ws_bytes < select_workspace_bytes(c, P, pool, pool_blocks, block, K)) return cudaErrorInvalidValue;
    const size_t n = static_cast<size_t>(rows) * p.segments * p.k_seg;
    float *cand_s = static_cast<float *>(ws);
    int32_t *cand_i = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + (n * 4 + 255) / 256 * 256);
    a.segments = p.segments;
    a.seg_len = p.seg_len;
    a.K = p.k_seg;
    a.out_ids = cand_i;
    a.out_scores = cand_s;
    cudaError_t e = launch(a, rows * p.segments, p.seg_len, st);
    if (e != cudaSuccess) return e;
    // Stage 2: the row's top K among the segments' candidates (in id order).
    SelArgs b{};
    b.source = kPairs;
    b.scores = cand_s;
    b.pair_ids = cand_i;
    b.n_pairs = p.segments * p.k_seg;
    b.P = P;
    b.segments = 1;
    b.seg_len = b.n_pairs;
    b.K = K;
    b.out_ids = out;
    return launch(b, rows, b.n_pairs, st);
}

}  // namespace csa
