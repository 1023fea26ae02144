// a3: top-K selection of row ids by indexer score, and the hierarchical pool.
// "DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section "The
// Paper": the query keeps only the top indices; "G2C Brief - DeepSeek
// V4.1-Flash", section "The hierarchical indexer": positions grouped in blocks
// of 8, each block scored by its best member, the top 2,048 blocks kept.
//
// One thread-block cluster per query row (or per segment of a very long row).
// The candidates are split into contiguous chunks, one per CTA, held in shared
// memory as order-preserving 32-bit keys (0 = no candidate).  The K-th largest
// key is found by a most-significant-digit radix select with fixed digits of
// 12, 12 and 8 bits: each pass histograms, in shared memory, the keys whose
// higher digits equal the threshold found so far; the cluster sums the CTAs'
// histograms in distributed shared memory: each CTA owns a slice of the bins,
// every CTA adds its non-zero counts into the owners' slices (one remote
// reduction per non-zero bin), and each owner stores its summed slice into
// every CTA with 16-byte stores, so after two cluster barriers all CTAs hold
// the same histogram and find the same threshold bin.  Indexer scores crowd
// into a few coarse bins (a weighted sum over many heads varies little
// relative to its size) and then spread over many fine bins, so the exchange
// must stay cheap for sparse and dense histograms alike.  A pass stops early when the
// threshold bin is taken whole, so typical data needs one or two passes.  Ties
// at the final key go to the lower row id.  Output ids are written in ascending
// order: per (iteration, warp) counts from warp ballots, one block scan, and
// one exchange of per-CTA counts give every selected key its position.
//
// A row of 8,193 to 16,384 candidates goes to one CTA instead
// (select_one_kernel, with the selection of select_cta.cuh): no cluster
// barrier, no warp votes.  A row of at most 8,192 stays in one CTA of this
// kernel.
//
// Rows longer than one cluster holds are split into segments: stage 1 keeps
// each segment's own top K (with scores) in the workspace; stage 2 selects the
// row's top K among those, which is exact because every member of the row's
// top K is in its segment's top K (the same order decides both).
#include <cooperative_groups.h>

#include "common.cuh"
#include "csa_internal.h"
#include "select_cta.cuh"

namespace cg = cooperative_groups;

namespace csa {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kDigit0Bins = 4096;    // key bits 31..20
constexpr int kDigit1Bins = 4096;    // key bits 19..8
constexpr int kDigit2Bins = 256;     // key bits 7..0
constexpr int kSelCacheMax = 16384;  // keys held per CTA at most (64 KB): two CTAs fit one SM
constexpr int kMaxIters = kSelCacheMax / kSelThreads;
constexpr int kMaxCluster = 16;
constexpr int kMinChunk = 4096;      // a row of up to 2x this stays whole in one CTA (no cluster barrier)
constexpr int kMinChunkLong = 1024;  // a longer row is not spread thinner than this per CTA
constexpr int64_t kSegmentLen = static_cast<int64_t>(kMaxCluster) * 8192;

// kBlockMax: blocks of 8 rows whose best visible scores the scan already
// wrote (one score per block), instead of kBlocks' maximum over row scores.
enum SelSource { kRows = 0, kBlocks = 1, kPoolRows = 2, kPairs = 3, kBlockMax = 4 };

struct SelArgs {
    const float *scores;       // kRows/kBlocks/kPoolRows: [rows][ld];  kPairs: [rows][n_pairs]
    int64_t ld;
    const int32_t *lengths;    // read as min(lengths[b], cap)
    int cap;
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

// Per-CTA shared state.  Other CTAs of the cluster only ever add into acc and
// store into hist_g, cnt_above and cnt_eq, and every such write is followed by a
// cluster barrier before it is read; no CTA loads another CTA's shared memory.
struct SelShared {
    uint32_t hist_l[kDigit0Bins];  // this CTA's histogram of the current pass
    uint32_t acc[kDigit0Bins / 2]; // sums of the bins this CTA owns, at most half (other CTAs add into it)
    uint32_t hist_g[kDigit0Bins];  // cluster-wide histogram of the current pass
    uint32_t cnt_above[kMaxCluster];     // per-CTA count of keys above the threshold
    uint32_t cnt_eq[kMaxCluster];        // per-CTA count of keys at the threshold
    uint32_t jw[kMaxIters * kSelWarps];  // per (iteration, warp): above << 16 | equal
    uint32_t warp_tot[kSelWarps];
    uint32_t res_bin, res_above;
};
static_assert(kDigit1Bins <= kDigit0Bins && kDigit2Bins <= kDigit0Bins, "one histogram size serves every pass");

template <int S>
struct RowView {
    const float *s;
    const int32_t *prow;
    const int32_t *ids;
    int L;
    __device__ __forceinline__ uint32_t key(int64_t i) const
    {
        if (S == kRows || S == kBlockMax) return score_key(__ldg(s + i));
        if (S == kBlocks) {
            const int64_t r0 = i * kPoolBlock;
            if (r0 + kPoolBlock <= L) {
                // a whole block: two 16-byte loads (a row of scores starts 16-byte
                // aligned and a block at a multiple of 8 scores)
                const float4 a = __ldg(reinterpret_cast<const float4 *>(s + r0));
                const float4 b = __ldg(reinterpret_cast<const float4 *>(s + r0) + 1);
                return score_key(fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w))));
            }
            float best = __ldg(s + r0);
#pragma unroll
            for (int m = 1; m < kPoolBlock; ++m)
                if (r0 + m < L) best = fmaxf(best, __ldg(s + r0 + m));
            return score_key(best);
        }
        // Both loads are issued before either is tested, so they overlap.
        if (S == kPoolRows) {
            const int32_t blk = __ldg(prow + (i >> 3));
            const float v = __ldg(s + i);
            const int64_t row = static_cast<int64_t>(blk) * kPoolBlock + (i & 7);
            return (blk >= 0 && row < L) ? score_key(v) : 0u;
        }
        const int32_t id = __ldg(ids + i);
        const float v = __ldg(s + i);
        return id >= 0 ? score_key(v) : 0u;
    }
    // Keys of candidates 4q .. 4q+3 (4q < n) from one 16-byte score load (and
    // one block id or four pair ids): rows, pool rows and pairs whose row
    // start is 16-byte aligned (a row of scores always is: the C ABI takes
    // them 16-byte aligned with a stride that is a multiple of 4, at least the
    // row's length).  Candidates >= n get 0.
    __device__ __forceinline__ uint4 key4(int q, int n) const
    {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(s) + q);
        const int i = 4 * q;
        bool ok[4];
        if (S == kPoolRows) {
            const int32_t blk = __ldg(prow + (q >> 1));
            const int64_t r0 = static_cast<int64_t>(blk) * kPoolBlock + (i & 7);
#pragma unroll
            for (int r = 0; r < 4; ++r) ok[r] = blk >= 0 && r0 + r < L;
        } else if (S == kPairs) {
            const int4 id4 = __ldg(reinterpret_cast<const int4 *>(ids) + q);
            ok[0] = id4.x >= 0 && i < n;
            ok[1] = id4.y >= 0 && i + 1 < n;
            ok[2] = id4.z >= 0 && i + 2 < n;
            ok[3] = id4.w >= 0 && i + 3 < n;
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) ok[r] = i + r < n;
        }
        return make_uint4(ok[0] ? score_key(v.x) : 0u, ok[1] ? score_key(v.y) : 0u, ok[2] ? score_key(v.z) : 0u,
                          ok[3] ? score_key(v.w) : 0u);
    }
    __device__ __forceinline__ int32_t id(int64_t i) const
    {
        if (S == kPoolRows) return __ldg(prow + (i >> 3)) * kPoolBlock + static_cast<int32_t>(i & 7);
        if (S == kPairs) return __ldg(ids + i);
        return static_cast<int32_t>(i);
    }
};

// Inverse of score_key (for the candidates a segment hands to stage 2).
__device__ __forceinline__ float key_score(uint32_t k)
{
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

__device__ __forceinline__ uint32_t cluster_addr(const void *local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_red_add(uint32_t addr, uint32_t v)
{
    asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_store(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_barrier()
{
    cluster_arrive();
    cluster_wait();
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

__device__ __forceinline__ void cluster_store4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Sums the cluster's per-CTA histograms of nb bins: CTA r owns bins
// [r*nb/C, (r+1)*nb/C); every CTA adds its non-zero counts into the owners'
// acc; after a barrier each owner stores its slice into every CTA's hist_g and
// clears its acc for the next pass; after a second barrier every CTA holds the
// whole histogram.  Returns the histogram to search (the CTA's own when it is
// alone).
__device__ __forceinline__ const uint32_t *reduce_histogram(SelShared &sh, int nb, int C, int rank)
{
    __syncthreads();  // the local histogram is complete
    if (C == 1) return sh.hist_l;
    const int S = nb / C;  // >= 16, <= nb / 2
    for (int b = threadIdx.x; b < nb; b += kSelThreads) {
        const uint32_t v = sh.hist_l[b];
        const int owner = b / S;
        if (v) cluster_red_add(cluster_addr(&sh.acc[b - owner * S], owner), v);
    }
    cluster_barrier();
    const int nv = S / 4;
    const uint4 *mine = reinterpret_cast<const uint4 *>(sh.acc);
    for (int i = threadIdx.x; i < nv * C; i += kSelThreads) {
        const int q = i / nv, j = i - q * nv;
        cluster_store4(cluster_addr(&sh.hist_g[rank * S + 4 * j], q), mine[j]);
    }
    __syncthreads();  // every store above has read its values
    for (int j = threadIdx.x; j < S; j += kSelThreads) sh.acc[j] = 0;
    cluster_barrier();
    return sh.hist_g;
}

__device__ __forceinline__ void zero_histogram(SelShared &sh, int nb)
{
    uint4 *z = reinterpret_cast<uint4 *>(sh.hist_l);
    for (int i = threadIdx.x; i < nb / 4; i += kSelThreads) z[i] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void zero_owned(SelShared &sh)
{
    uint4 *z = reinterpret_cast<uint4 *>(sh.acc);
    for (int i = threadIdx.x; i < kDigit0Bins / 8; i += kSelThreads) z[i] = make_uint4(0, 0, 0, 0);
}

// Finds, in a cluster-wide histogram h of nb bins, the bin b holding the
// need-th largest key: fewer than `need` keys lie in the bins above b and at
// least `need` in b and above.  Thread t owns the nb/T bins just below the top
// t*nb/T ones, so an exclusive scan over threads is the count above its range.
// Returns the histogram total; sh.res_bin and sh.res_above (the count above
// the bin) are set when the total is at least `need`.
__device__ __forceinline__ uint32_t find_bin(const uint32_t *h, int nb, uint32_t need, SelShared &sh)
{
    const int tid = threadIdx.x;
    const int per = nb >= kSelThreads ? nb / kSelThreads : 1;
    const int hi = nb - tid * per;
    const int lo = hi - per;
    uint32_t s = 0;
    // each thread's bins are read in an order rotated by the thread's index
    // (per is a power of two), so the lanes of a warp hit different banks
    if (lo >= 0)
        for (int j = 0; j < per; ++j) s += h[lo + ((j + tid) & (per - 1))];
    uint32_t total;
    const uint32_t excl = block_exclusive_scan(s, sh.warp_tot, &total);
    if (lo >= 0 && s && excl < need && excl + s >= need) {
        uint32_t cum = excl;
        for (int b = hi - 1; b >= lo; --b) {
            if (cum + h[b] >= need) {
                sh.res_bin = static_cast<uint32_t>(b);
                sh.res_above = cum;
                break;
            }
            cum += h[b];
        }
    }
    __syncthreads();
    return total;
}

template <int S>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(SelArgs a)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(dyn_smem);
    uint32_t *cache = reinterpret_cast<uint32_t *>(dyn_smem + sizeof(SelShared));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    zero_histogram(sh, kDigit0Bins);
    zero_owned(sh);
    // Above: this CTA only.  Below: reads of what earlier work on the stream wrote.
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.y / a.segments, seg = blockIdx.y % a.segments;
    int64_t n;
    RowView<S> rv{nullptr, nullptr, nullptr, 0};
    if (S == kPairs) {
        n = a.n_pairs;
        rv.s = a.scores + static_cast<int64_t>(row) * a.n_pairs;
        rv.ids = a.pair_ids + static_cast<int64_t>(row) * a.n_pairs;
    } else {
        const int b = row / a.P, p = row % a.P;
        const int L = min(a.lengths[b], a.cap) - a.P + 1 + p;
        rv.s = a.scores + static_cast<int64_t>(row) * a.ld;
        rv.L = L;
        if (S == kPoolRows) {
            n = static_cast<int64_t>(a.pool_blocks) * kPoolBlock;
            rv.prow = a.pool + static_cast<int64_t>(row) * a.pool_blocks;
        } else {
            n = L <= 0 ? 0 : (S == kRows ? L : (L + kPoolBlock - 1) / kPoolBlock);
        }
    }
    const int64_t s0 = min(n, seg * a.seg_len), s1 = min(n, s0 + a.seg_len);
    const int64_t chunk = (s1 - s0 + C - 1) / C;
    const int64_t e0 = min(s1, s0 + rank * chunk), e1 = min(s1, e0 + chunk);
    const int m = static_cast<int>(e1 - e0);  // <= kSelCacheMax (the host sizes the cluster so)

    __syncthreads();   // histogram zeroed before any thread counts into it
    // Every CTA of the cluster runs before any stores into another's memory.
    // A CTA alone needs no cluster barrier anywhere (they cost ~10x a CTA barrier).
    const bool solo = C == 1;
    if (!solo) cluster_arrive();

    // Pass 0: keys into shared memory and the digit-0 histogram.  Loads are
    // issued U at a time so that their latencies overlap.
    constexpr int U = 8;
    for (int base = 0; base < m; base += U * kSelThreads) {
        uint32_t k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * kSelThreads + tid;
            k[u] = i < m ? rv.key(e0 + i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * kSelThreads + tid;
            if (i < m) {
                cache[i] = k[u];
                if (k[u]) atomicAdd(&sh.hist_l[k[u] >> 20], 1u);
            }
        }
    }
    if (!solo) cluster_wait();
    const uint32_t *h0 = reduce_histogram(sh, kDigit0Bins, C, rank);

    // Selection: every key > thr_gt, plus the first `need` keys equal to
    // thr_eq in id order.
    const uint32_t K = static_cast<uint32_t>(a.K);
    uint32_t thr_gt = 0, thr_eq = 0, need = 0;
    const uint32_t total = find_bin(h0, kDigit0Bins, K, sh);
    if (total > K) {
        // Digits of 12, 12 and 8 bits: after each, the key bits above `hi`
        // are fixed to `prefix` and `above` keys lie above them.  One loop
        // body serves the second and third digits (one copy of the code).
        uint32_t prefix = sh.res_bin, above = sh.res_above;
        const uint32_t *h = h0;
        int hi = 20;
        for (;;) {
            const uint32_t in_bin = h[sh.res_bin];
            if (in_bin == K - above) {  // the bin is taken whole
                thr_gt = prefix ? (prefix << hi) - 1u : 0u;
                break;
            }
            if (hi == 0) {  // prefix is one key value (>= 1: key 0 is never counted)
                need = K - above;  // 1 <= need < in_bin
                thr_gt = prefix;
                thr_eq = prefix;
                break;
            }
            const int d = hi > 8 ? 12 : 8, lo = hi - d, nb = 1 << d;
            __syncthreads();  // every thread has read h (the CTA's own histogram when alone)
            zero_histogram(sh, nb);
            __syncthreads();
            for (int i = tid; i < m; i += kSelThreads) {
                const uint32_t k = cache[i];
                if (k && (k >> hi) == prefix) atomicAdd(&sh.hist_l[(k >> lo) & static_cast<uint32_t>(nb - 1)], 1u);
            }
            h = reduce_histogram(sh, nb, C, rank);
            find_bin(h, nb, K - above, sh);
            prefix = (prefix << d) | sh.res_bin;
            above += sh.res_above;
            hi = lo;
        }
    }

    // Per (iteration, warp) counts of keys above the threshold and at it.
    const int J = (m + kSelThreads - 1) / kSelThreads;
    for (int j = 0; j < J; ++j) {
        const int i = j * kSelThreads + tid;
        const uint32_t k = i < m ? cache[i] : 0u;
        const unsigned ba = __ballot_sync(0xFFFFFFFFu, k > thr_gt);
        const unsigned be = __ballot_sync(0xFFFFFFFFu, need && k == thr_eq);
        if (lane == 0) sh.jw[j * kSelWarps + warp] = (static_cast<uint32_t>(__popc(ba)) << 16) | __popc(be);
    }
    __syncthreads();
    uint32_t cta_tot;
    {
        const uint32_t v = tid < J * kSelWarps ? sh.jw[tid] : 0u;
        const uint32_t ex = block_exclusive_scan(v, sh.warp_tot, &cta_tot);
        if (tid < J * kSelWarps) sh.jw[tid] = ex;
    }
    if (!solo) {
        if (tid < C) {
            cluster_store(cluster_addr(&sh.cnt_above[rank], tid), cta_tot >> 16);
            cluster_store(cluster_addr(&sh.cnt_eq[rank], tid), cta_tot & 0xFFFFu);
        }
        cluster_barrier();  // last remote write: from here on CTAs touch only their own memory
    }
    uint32_t above0 = 0, tie0 = 0;
    for (int q = 0; q < rank; ++q) {
        above0 += sh.cnt_above[q];
        tie0 += sh.cnt_eq[q];
    }

    // Output position of a selected key = selected keys with a lower id.
    const int64_t obase = static_cast<int64_t>(blockIdx.y) * a.K;
    const unsigned lt = (1u << lane) - 1u;
    // Ids that live in memory (pool rows, stage-2 pairs) are fetched eight
    // iterations at a time, so their latencies overlap instead of adding up.
    constexpr int W = (S == kPoolRows || S == kPairs) ? 8 : 1;
    for (int j0 = 0; j0 < J; j0 += W) {
        int32_t idv[W];
#pragma unroll
        for (int u = 0; u < W; ++u) {
            const int i = (j0 + u) * kSelThreads + tid;
            idv[u] = (W > 1 && j0 + u < J && i < m) ? rv.id(e0 + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < W; ++u) {
            const int j = j0 + u;
            if (j >= J) break;
            const int i = j * kSelThreads + tid;
            const uint32_t k = i < m ? cache[i] : 0u;
            const bool is_above = k > thr_gt;
            const bool is_tie = need && k == thr_eq;
            const unsigned ba = __ballot_sync(0xFFFFFFFFu, is_above);
            const unsigned be = __ballot_sync(0xFFFFFFFFu, is_tie);
            const uint32_t base = sh.jw[j * kSelWarps + warp];
            const uint32_t a_before = above0 + (base >> 16) + __popc(ba & lt);
            const uint32_t t_before = tie0 + (base & 0xFFFFu) + __popc(be & lt);
            int64_t pos = -1;
            if (is_above) pos = a_before + min(t_before, need);
            else if (is_tie && t_before < need) pos = a_before + t_before;
            if (pos >= 0) {
                a.out_ids[obase + pos] = W > 1 ? idv[u] : rv.id(e0 + i);
                if (a.out_scores) a.out_scores[obase + pos] = key_score(k);
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

// A row of at most cta_select::kMaxKeys candidates: one CTA, no cluster.  The
// keys are gathered with eight loads in flight per thread, selected by
// cta_select::select_keys, and the kept candidates' ids written in order with
// -1 padding.
template <int S>
__global__ void __launch_bounds__(cta_select::kThreads, 1) select_one_kernel(SelArgs a)
{
    namespace cs = cta_select;
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    uint32_t *keys = reinterpret_cast<uint32_t *>(dyn_smem);  // then the kept candidates
    cs::Scratch &sc = *reinterpret_cast<cs::Scratch *>(keys + cs::kMaxKeys);
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.y;
    int n;
    RowView<S> rv{nullptr, nullptr, nullptr, 0};
    if (S == kPairs) {
        n = a.n_pairs;
        rv.s = a.scores + static_cast<int64_t>(row) * a.n_pairs;
        rv.ids = a.pair_ids + static_cast<int64_t>(row) * a.n_pairs;
    } else {
        const int b = row / a.P, p = row % a.P;
        const int L = min(a.lengths[b], a.cap) - a.P + 1 + p;
        rv.s = a.scores + static_cast<int64_t>(row) * a.ld;
        rv.L = L;
        if (S == kPoolRows) {
            n = a.pool_blocks * kPoolBlock;
            rv.prow = a.pool + static_cast<int64_t>(row) * a.pool_blocks;
        } else {
            n = L <= 0 ? 0 : (S == kRows ? L : (L + kPoolBlock - 1) / kPoolBlock);
        }
    }
    n = min(n, cs::kMaxKeys);  // the host sends longer rows to the cluster kernel
    const bool vec = S != kBlocks && (S != kPairs || (a.n_pairs & 3) == 0);
    if (vec) {
        // 16-byte loads, all of a thread's in flight at once (n <= 16,384 is
        // at most 8 quads per thread)
        const int nq = (n + 3) / 4;
        uint4 k[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int q = u * cs::kThreads + tid;
            k[u] = q < nq ? rv.key4(q, n) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int q = u * cs::kThreads + tid;
            if (q < nq) *reinterpret_cast<uint4 *>(keys + cs::key_slot(4 * q)) = k[u];
        }
    }
    constexpr int U = S == kBlocks ? 2 : 8;
    for (int base = 0; !vec && base < n; base += U * cs::kThreads) {
        uint32_t k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * cs::kThreads + tid;
            k[u] = i < n ? rv.key(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * cs::kThreads + tid;
            if (i < n) keys[cs::key_slot(i)] = k[u];
        }
    }
    __syncthreads();
    int32_t *kept_c = reinterpret_cast<int32_t *>(keys);
    const int kept = cs::select_keys(keys, n, static_cast<uint32_t>(a.K), kept_c, sc);
    int32_t *out = a.out_ids + static_cast<int64_t>(row) * a.K;
    for (int j = tid; j < a.K; j += cs::kThreads) out[j] = j < kept ? rv.id(kept_c[j]) : -1;
}

size_t select_smem(int64_t chunk)
{
    return sizeof(SelShared) + static_cast<size_t>((chunk + 3) / 4 * 4) * sizeof(uint32_t);
}

template <int S>
cudaError_t launch_source(const SelArgs &args, int grid_rows, int64_t n_per_cluster, cudaStream_t st)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(select_smem(kSelCacheMax)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(select_kernel<S>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // Smallest cluster whose chunks fit shared memory, widened (down to
    // kMinChunkLong keys per CTA) while the grid is under one CTA per SM: spreading
    // a row's keys over more CTAs also spreads the contention of its shared-
    // memory histogram, which crowded indexer scores make high.
    // Rows of at most 2 * kMinChunk keys stay in one CTA: there the cluster
    // barriers cost more than the spread saves.
    const int64_t min_chunk = n_per_cluster <= 2 * kMinChunk ? kMinChunk : kMinChunkLong;
    int C = 1;
    while (C < kMaxCluster &&
           ((n_per_cluster + C - 1) / C > kSelCacheMax ||
            (static_cast<int64_t>(grid_rows) * C < sm_count() && (n_per_cluster + 2 * C - 1) / (2 * C) >= min_chunk)))
        C *= 2;
    const int64_t chunk = (n_per_cluster + C - 1) / C;
    if (chunk > kSelCacheMax) return cudaErrorInvalidValue;
    return launch_kernel(select_kernel<S>, dim3(C, grid_rows), dim3(kSelThreads), select_smem(chunk), st, C, args);
}

// Rows of 2 * kMinChunk + 1 to cta_select::kMaxKeys candidates without
// per-candidate score outputs go to one CTA each (select_one_kernel); longer
// ones to the clusters; shorter ones to select_kernel alone in one CTA, whose
// loops cover only the row's keys (select_one_kernel's cover 16,384 slots,
// which measures slower for 4,096 keys and faster for 16,384).
template <int S>
cudaError_t launch_one_or_cluster(const SelArgs &args, int grid_rows, int64_t n_per_cluster, cudaStream_t st)
{
    if (n_per_cluster <= 2 * kMinChunk || n_per_cluster > cta_select::kMaxKeys || args.segments != 1 ||
        args.out_scores)
        return launch_source<S>(args, grid_rows, n_per_cluster, st);
    constexpr size_t smem = cta_select::kMaxKeys * 4 + sizeof(cta_select::Scratch);
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(select_one_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_kernel(select_one_kernel<S>, dim3(1, grid_rows), dim3(cta_select::kThreads), smem, st, 0, args);
}

cudaError_t launch(int source, const SelArgs &args, int grid_rows, int64_t n_per_cluster, cudaStream_t st)
{
    switch (source) {
    case kRows: return launch_one_or_cluster<kRows>(args, grid_rows, n_per_cluster, st);
    case kBlocks: return launch_one_or_cluster<kBlocks>(args, grid_rows, n_per_cluster, st);
    case kPoolRows: return launch_one_or_cluster<kPoolRows>(args, grid_rows, n_per_cluster, st);
    case kBlockMax: return launch_one_or_cluster<kBlockMax>(args, grid_rows, n_per_cluster, st);
    default: return launch_one_or_cluster<kPairs>(args, grid_rows, n_per_cluster, st);
    }
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
    const int64_t one_cluster = static_cast<int64_t>(kMaxCluster) * kSelCacheMax;
    p.segments = p.n_max <= one_cluster ? 1 : static_cast<int>((p.n_max + kSegmentLen - 1) / kSegmentLen);
    p.seg_len = (p.n_max + p.segments - 1) / p.segments;
    if (p.seg_len < 1) p.seg_len = 1;
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
           static_cast<int64_t>(p.segments) * p.k_seg <= static_cast<int64_t>(kMaxCluster) * kSelCacheMax;
}

cudaError_t launch_select(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                          int pool_blocks, int block, int K, int32_t *out, void *ws, size_t ws_bytes,
                          cudaStream_t st, bool block_max)
{
    const int rows = c.B * P;
    if (rows == 0) return cudaSuccess;
    const SelPlan p = sel_plan(c, pool, pool_blocks, block, K);
    const int source = pool ? kPoolRows : (block == 1 ? kRows : (block_max ? kBlockMax : kBlocks));
    SelArgs a{};
    a.scores = scores;
    a.ld = ld;
    a.lengths = c.lengths;
    a.cap = c.cap;
    a.P = P;
    a.pool = pool;
    a.pool_blocks = pool_blocks;
    if (p.segments == 1) {
        a.segments = 1;
        a.seg_len = p.n_max;
        a.K = K;
        a.out_ids = out;
        return launch(source, a, rows, p.n_max, st);
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
    cudaError_t e = launch(source, a, rows * p.segments, p.seg_len, st);
    if (e != cudaSuccess) return e;
    // Stage 2: the row's top K among the segments' candidates (in id order).
    SelArgs b{};
    b.scores = cand_s;
    b.pair_ids = cand_i;
    b.n_pairs = p.segments * p.k_seg;
    b.P = P;
    b.segments = 1;
    b.seg_len = b.n_pairs;
    b.K = K;
    b.out_ids = out;
    return launch(kPairs, b, rows, b.n_pairs, st);
}

int select_pairs_supported(int n, int K)
{
    return n >= 1 && K >= 1 && static_cast<int64_t>(n) <= static_cast<int64_t>(kMaxCluster) * kSelCacheMax;
}

cudaError_t launch_select_pairs(int rows, int n, const float *scores, const int32_t *ids, int K, int32_t *out,
                                cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    if (!select_pairs_supported(n, K)) return cudaErrorInvalidValue;
    SelArgs b{};
    b.scores = scores;
    b.pair_ids = ids;
    b.n_pairs = n;
    b.P = 1;
    b.segments = 1;
    b.seg_len = n;
    b.K = K;
    b.out_ids = out;
    return launch(kPairs, b, rows, n, st);
}

}  // namespace csa
