// Top-K selection inside one CTA, for up to 16,384 candidates: the K largest
// order-preserving 32-bit keys (0 = no candidate), ties to the lower candidate
// index, returned as candidate indices in ascending order.  "DeepSeek V4.1
// Flash: Pushing the Limits" (talk write-up), section "The Paper": the query
// keeps only the top indices; "G2C Brief - DeepSeek V4.1-Flash", section "The
// hierarchical indexer": a Reindex layer keeps the best K of the pool's rows.
//
// One CTA of 512 threads does all the work, so the cost is the instructions
// issued per key (16 warps share four schedulers: one instruction per key is
// about 0.07 us), and the design keeps that count small:
//   - thread t owns the 32 consecutive candidates [32t, 32t + 32), held in
//     registers: what a thread keeps is counted without warp votes (a vote
//     costs tens of cycles per warp here) and output positions come from one
//     block scan of per-thread counts;
//   - one histogram pass over all keys: (key - base) over 4,096 bins that
//     span [base, maximum].  For K <= 2,048, base is a lower bound on the
//     K-th largest key: the smallest of the largest keys of the 2,048 groups
//     of 8 consecutive candidates.  When at least K groups hold a key, those
//     are at least K distinct keys, and of any K keys one is no larger than
//     the K-th largest, so no key below base is kept (otherwise base is the
//     smallest key).  Without the bound, indexer scores of exactly 0 (every
//     head's product negative) stretch the range, and the bin holding the
//     K-th largest key can hold hundreds of keys.
//     When at most 4,096 keys lie at or above base (the usual case: the
//     bound is tight), they are first moved, in candidate order, into one
//     list over the key array, 8 entries a thread, and the passes and the
//     output run over those: a shared-memory atomic costs about as much with
//     one lane active as with 32, and most of a thread's 32 keys lie below
//     base;
//   - the keys of the threshold bin are gathered, in candidate order, into a
//     list of at most 1,024 (another pass first if the bin is larger), and
//     further passes over the next lower bits run on that list only;
//   - a list of at most 32 keys is ranked exactly by one warp;
//   - every outcome is one rule: keep the keys above thr_gt, and the first
//     `need` keys equal to thr_eq in candidate order.
// The keys live in shared memory at key_slot(c): 16-byte chunks of each
// 32-key row XOR-swizzled by the row index, so that both a warp's coalesced
// writes (32 consecutive candidates, or 8 lanes of 4) and its per-thread
// 16-byte reads (one thread's 32 candidates) are free of bank conflicts.
#pragma once

#include "common.cuh"

namespace csa {
namespace cta_select {

constexpr int kThreads = 512;
constexpr int kPerThread = 32;
constexpr int kMaxKeys = kThreads * kPerThread;  // 16,384
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;
constexpr int kListMax = 1024;                   // keys of a threshold bin gathered into a list
constexpr int kRankMax = 32;                     // list length ranked exactly by one warp
constexpr int kGroup = 8;                        // keys per group of the lower bound
constexpr int kBigList = 4096;                   // keys >= the bound moved into one list, at most
constexpr int kBigPer = kBigList / kThreads;     // its entries a thread
static_assert(2 * kBigList <= kMaxKeys, "the big list's (key, candidate) pairs fit the key array");
static_assert(kBigPer % 2 == 0, "a thread's list entries load as 16-byte pairs");
constexpr int kWarps = kThreads / 32;
static_assert(kWarps <= 32, "one lane per warp in the cross-warp reductions");
static_assert(kListMax == 2 * kThreads, "list passes give each thread two entries");

struct alignas(16) Scratch {
    uint32_t hist[kBins];
    uint32_t lk[kListMax];  // gathered keys, in candidate order
    int32_t lc[kListMax];   // and their candidates
    uint32_t wa[kWarps], wb[kWarps], wc[kWarps], wd[kWarps], we[kWarps];
    uint32_t scan_buf[2][kWarps];  // per-warp sums of block_scan, used in turn
    uint32_t res_bin, res_above;
    uint32_t thr_gt, thr_eq, need;
};
// Whatever a kernel places after the scratch starts 16-byte aligned.
static_assert(sizeof(Scratch) % 16 == 0, "the scratch's size keeps what follows it aligned");

// Shared-memory index of candidate c's key.
__device__ __forceinline__ int key_slot(int c) { return c ^ (((c >> 5) & 7) << 2); }

// Exclusive block scan of one value per thread (all kThreads threads, in the
// same sequence of calls); *total gets the sum.  One CTA barrier: the per-warp
// sums alternate between two buffers (sb, the caller's index, flips), and a
// thread passes scan k+1's barrier only after its reads of scan k's buffer, so
// scan k+2 may rewrite it.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, Scratch &sc, uint32_t *total, int &sb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    uint32_t *buf = sc.scan_buf[sb];
    sb ^= 1;
    if (lane == 31) buf[warp] = x;
    __syncthreads();
    // lane i reads warp i's sum: one load and two warp reductions, not a
    // loop of kWarps dependent loads
    const uint32_t w = lane < kWarps ? buf[lane] : 0u;
    *total = __reduce_add_sync(0xFFFFFFFFu, w);
    return __reduce_add_sync(0xFFFFFFFFu, lane < warp ? w : 0u) + x - v;
}

__device__ __forceinline__ void zero_bins(Scratch &sc, int nb)
{
    uint4 *z = reinterpret_cast<uint4 *>(sc.hist);
    for (int i = threadIdx.x; i < (nb + 3) / 4; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {  // overwritten by find_bin's owner of the bin
        sc.res_bin = 0;
        sc.res_above = 0;
    }
}

// find_bin for fewer than 4,096 bins (later passes over short ranges): each
// thread sums nb/kThreads bins (or one), read in an order rotated by the
// thread so that a warp's lanes hit different banks.  Out of line: the first
// pass of a selection uses 4,096 bins.
static __device__ __noinline__ void find_bin_small(int nb, uint32_t want, Scratch &sc, int sb)
{
    const int tid = threadIdx.x;
    const int per = nb >= kThreads ? nb / kThreads : 1;
    const int bhi = nb - tid * per, blo = bhi - per;
    uint32_t ssum = 0;
    if (blo >= 0)
        for (int j = 0; j < per; ++j) ssum += sc.hist[blo + ((j + tid) & (per - 1))];
    uint32_t tot;
    const uint32_t excl = block_scan(ssum, sc, &tot, sb);
    if (blo >= 0 && ssum && excl < want && excl + ssum >= want) {
        uint32_t cum = excl;
        for (int bb = bhi - 1; bb >= blo; --bb) {
            const uint32_t hb = sc.hist[bb];
            if (cum + hb >= want) {
                sc.res_bin = static_cast<uint32_t>(bb);
                sc.res_above = cum;
                break;
            }
            cum += hb;
        }
    }
    __syncthreads();
}

// With sc.hist holding nb bins: the bin b holding the want-th largest key
// (fewer than `want` keys in the bins above b, at least `want` in b and
// above).  With 4,096 bins thread t sums bins [4096 - 8(t+1), 4096 - 8t) in
// two 16-byte loads, kept in registers for the owner's search; fewer bins go
// out of line.  Sets *bin and *above (the count in the bins above it), the
// same in every thread.
__device__ __forceinline__ void find_bin(int nb, uint32_t want, Scratch &sc, uint32_t *bin, uint32_t *above, int &sb)
{
    if (nb != kBins) {
        find_bin_small(nb, want, sc, sb);
        sb ^= 1;  // the one block scan inside
        *bin = sc.res_bin;
        *above = sc.res_above;
        return;
    }
    const int tid = threadIdx.x;
    const int blo = kBins - (tid + 1) * 8;
    uint32_t h[8];
    const uint4 a = *reinterpret_cast<const uint4 *>(&sc.hist[blo]);
    const uint4 b = *reinterpret_cast<const uint4 *>(&sc.hist[blo + 4]);
    h[0] = a.x, h[1] = a.y, h[2] = a.z, h[3] = a.w, h[4] = b.x, h[5] = b.y, h[6] = b.z, h[7] = b.w;
    const uint32_t ssum = ((h[0] + h[1]) + (h[2] + h[3])) + ((h[4] + h[5]) + (h[6] + h[7]));
    uint32_t tot;
    const uint32_t excl = block_scan(ssum, sc, &tot, sb);
    if (ssum && excl < want && excl + ssum >= want) {
        uint32_t cum = excl;
        bool found = false;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (!found && cum + h[i] >= want) {
                sc.res_bin = static_cast<uint32_t>(blo + i);
                sc.res_above = cum;
                found = true;
            }
            cum += found ? 0u : h[i];
        }
    }
    __syncthreads();
    *bin = sc.res_bin;
    *above = sc.res_above;
}

// The search for the K-th largest key over v = key - base: the bits of v
// above `hi` are fixed to `prefix`, and `above` keys lie above them (all of
// them kept).  Once done, the rule is: keep keys > thr_gt, and the first
// `need` keys == thr_eq in candidate order.
struct Cut {
    uint32_t prefix = 0, above = 0, in_bin = 0;
    int hi = 0;
    bool done = false;
    uint32_t thr_gt = 0, thr_eq = 0, need = 0;
};

// A. Histogram passes over a thread's M keys (those >= base whose bits above
// hi match the prefix), until the rule is found or the threshold bin holds at
// most kListMax keys.  The first pass's bins are zero on entry, ordered by a
// CTA barrier.
template <int M>
__device__ __forceinline__ void passes(const uint32_t (&ks)[M], uint32_t base, uint32_t K, Cut &c, Scratch &sc,
                                       int &sb)
{
    for (int pass = 0;; ++pass) {
        if (c.hi == 0) {  // one key value left
            c.thr_gt = c.thr_eq = base + c.prefix;
            c.need = K - c.above;
            c.done = true;
            return;
        }
        const int d = c.hi < kBinBits ? c.hi : kBinBits, lo = c.hi - d, nb = 1 << d;
        if (pass) {
            __syncthreads();  // every thread has read the last pass's bins
            zero_bins(sc, nb);
            __syncthreads();
        }
        const uint32_t mask = c.hi >= 32 ? 0u : (0xFFFFFFFFu << c.hi);
        const uint32_t pfx = c.hi >= 32 ? 0u : (c.prefix << c.hi);
#pragma unroll
        for (int j = 0; j < M; ++j) {
            const uint32_t v = ks[j] - base;
            if (ks[j] >= base && (v & mask) == pfx) atomicAdd(&sc.hist[(v >> lo) & (nb - 1)], 1u);
        }
        __syncthreads();
        uint32_t bin, ab;
        find_bin(nb, K - c.above, sc, &bin, &ab, sb);
        c.above += ab;
        const uint32_t in_bin = sc.hist[bin];
        const uint32_t P = (c.prefix << d) | bin;
        if (in_bin == K - c.above) {  // the bin is taken whole
            c.thr_gt = base + (P << lo) - 1u;
            c.done = true;
            return;
        }
        if (lo == 0) {  // the bin is one key value
            c.thr_gt = c.thr_eq = base + P;
            c.need = K - c.above;
            c.done = true;
            return;
        }
        c.prefix = P;
        c.hi = lo;
        c.in_bin = in_bin;
        if (in_bin <= kListMax) return;
    }
}

// B. The threshold bin's keys ((key - base) >> hi == prefix, 1 <= hi < 32)
// gathered into the list in candidate order; returns their number.
template <int M, class Cand>
__device__ __forceinline__ uint32_t gather(const uint32_t (&ks)[M], Cand cand, uint32_t base, const Cut &c,
                                           Scratch &sc, int &sb)
{
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < M; ++j) mine += (ks[j] >= base && ((ks[j] - base) >> c.hi) == c.prefix) ? 1u : 0u;
    uint32_t m;
    uint32_t off = block_scan(mine, sc, &m, sb);
#pragma unroll
    for (int j = 0; j < M; ++j)
        if (ks[j] >= base && ((ks[j] - base) >> c.hi) == c.prefix) {
            sc.lk[off] = ks[j];
            sc.lc[off] = cand(j);
            ++off;
        }
    __syncthreads();
    return m;
}

// Output: the kept candidates of a thread's M keys (key j is candidate
// cand(j); a thread's keys are consecutive in candidate order, and threads in
// order), positions from one scan of (kept, ties) counts.  Ends with a barrier.
template <int M, class Cand>
__device__ __forceinline__ void write_kept(const uint32_t (&ks)[M], Cand cand, const Cut &c, int32_t *obuf,
                                           Scratch &sc, int &sb)
{
    uint32_t sel = 0, tie = 0;
#pragma unroll
    for (int j = 0; j < M; ++j) {
        sel |= (ks[j] > c.thr_gt ? 1u : 0u) << j;
        tie |= (c.need && ks[j] == c.thr_eq ? 1u : 0u) << j;
    }
    uint32_t tot2;
    const uint32_t ex = block_scan((static_cast<uint32_t>(__popc(sel)) << 16) | static_cast<uint32_t>(__popc(tie)), sc,
                                   &tot2, sb);
    const uint32_t a_before = ex >> 16, t_before = ex & 0xFFFFu;
    if (c.need) {
        // the first `need` ties in candidate order are kept
        uint32_t take = c.need > t_before ? c.need - t_before : 0u;
        uint32_t tb = tie;
        while (take && tb) {
            sel |= tb & (~tb + 1u);
            tb &= tb - 1u;
            --take;
        }
    }
    uint32_t pos = a_before + min(t_before, c.need);
#pragma unroll
    for (int j = 0; j < M; ++j)
        if (sel & (1u << j)) obuf[pos++] = cand(j);
    __syncthreads();
}

// C. Passes over the list's next lower bits until at most kRankMax keys
// remain (or the rule is found); thread t holds entries 2t and 2t + 1.  Out
// of line: rare once the first pass spans [bound, maximum].
struct ListState {
    Cut c;
    uint32_t m, nd;
    int sb;
};
static __device__ __noinline__ ListState list_passes(ListState st, uint32_t base, Scratch &sc)
{
    const int tid = threadIdx.x;
    Cut &c = st.c;
    uint32_t &m = st.m, &nd = st.nd;
    int &sb = st.sb;
    while (static_cast<int>(m) > kRankMax) {
        if (c.hi == 0) {  // one key value left
            c.thr_gt = c.thr_eq = base + c.prefix;
            c.need = nd;
            c.done = true;
            break;
        }
        const int d = c.hi < kBinBits ? c.hi : kBinBits, lo = c.hi - d, nb = 1 << d;
        const int i0 = 2 * tid, i1 = 2 * tid + 1;
        const bool h0 = i0 < static_cast<int>(m), h1 = i1 < static_cast<int>(m);
        const uint32_t e0 = h0 ? sc.lk[i0] : 0u, e1 = h1 ? sc.lk[i1] : 0u;
        const int32_t ec0 = h0 ? sc.lc[i0] : 0, ec1 = h1 ? sc.lc[i1] : 0;
        zero_bins(sc, nb);
        __syncthreads();
        const uint32_t b0 = ((e0 - base) >> lo) & (nb - 1), b1 = ((e1 - base) >> lo) & (nb - 1);
        if (h0) atomicAdd(&sc.hist[b0], 1u);
        if (h1) atomicAdd(&sc.hist[b1], 1u);
        __syncthreads();
        uint32_t bin, ab;
        find_bin(nb, nd, sc, &bin, &ab, sb);
        nd -= ab;
        const uint32_t in_bin = sc.hist[bin];
        const uint32_t P = (c.prefix << d) | bin;
        if (in_bin == nd) {
            c.thr_gt = base + (P << lo) - 1u;
            c.need = 0;
            c.done = true;
            break;
        }
        if (lo == 0) {
            c.thr_gt = c.thr_eq = base + P;
            c.need = nd;
            c.done = true;
            break;
        }
        // keep the bin's entries, in order (each thread's entries were
        // read before the scan's first barrier)
        const bool k0 = h0 && b0 == bin, k1 = h1 && b1 == bin;
        uint32_t o = block_scan((k0 ? 1u : 0u) + (k1 ? 1u : 0u), sc, &m, sb);
        if (k0) {
            sc.lk[o] = e0;
            sc.lc[o] = ec0;
            ++o;
        }
        if (k1) {
            sc.lk[o] = e1;
            sc.lc[o] = ec1;
        }
        __syncthreads();
        c.prefix = P;
        c.hi = lo;
    }
    return st;
}

// C and D on the m keys gathered from the threshold bin (the list): passes
// over their next lower bits until at most kRankMax remain, then one warp
// ranks those.  Sets the rule in c.
__device__ __forceinline__ void list_rank(Cut &c, uint32_t m, uint32_t base, uint32_t K, Scratch &sc, int &sb)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t nd = K - c.above;  // keys still to keep, all in the list
    if (static_cast<int>(m) > kRankMax) {
        const ListState st = list_passes(ListState{c, m, nd, sb}, base, sc);
        c = st.c;
        m = st.m;
        nd = st.nd;
        sb = st.sb;
    }
    if (!c.done) {
        // D. rank the m <= 32 listed keys in one warp; the nd-th
        // largest, V, sets the rule: keys > V, and the first
        // nd - (listed keys > V) keys equal to V (every key equal to V
        // is listed)
        if (warp == 0) {
            const bool has = lane < static_cast<int>(m);
            const uint32_t key = has ? sc.lk[lane] : 0u;
            const int32_t cand = has ? sc.lc[lane] : 0;
            uint32_t r = 0;
            for (int i = 0; i < static_cast<int>(m); ++i) {
                const uint32_t o = __shfl_sync(0xFFFFFFFFu, key, i);
                const int32_t oc = __shfl_sync(0xFFFFFFFFu, cand, i);
                r += (o > key || (o == key && oc < cand)) ? 1u : 0u;
            }
            const unsigned at = __ballot_sync(0xFFFFFFFFu, has && r == nd - 1u);
            const uint32_t V = __shfl_sync(0xFFFFFFFFu, key, __ffs(static_cast<int>(at)) - 1);
            const uint32_t gt = __reduce_add_sync(0xFFFFFFFFu, (has && key > V) ? 1u : 0u);
            if (lane == 0) {
                sc.thr_gt = V;
                sc.thr_eq = V;
                sc.need = nd - gt;
            }
        }
        __syncthreads();
        c.thr_gt = sc.thr_gt;
        c.thr_eq = sc.thr_eq;
        c.need = sc.need;
    }
}

// The selection over the keys left in shared memory (keys[key_slot(c)]),
// in rolled loops: when more than kBigList keys reach the bound, or when every
// key is kept.  Out of line, so that the common path's code stays short.
// Called by all threads, after a CTA barrier; the first pass's bins are zero.
static __device__ __noinline__ int select_keys_smem(const uint32_t *keys, int n, uint32_t K, uint32_t base, uint32_t kmax,
                                             uint32_t total, int32_t *obuf, Scratch &sc, int sb)
{
    const int tid = threadIdx.x;
    const int c0 = tid * kPerThread;
    auto key = [&](int j) {
        const int cand = c0 + j;
        return cand < n ? keys[key_slot(cand)] : 0u;
    };
    Cut c;
    if (total > K) {
        const uint32_t range = kmax - base;
        c.hi = range ? 32 - __clz(static_cast<int>(range)) : 0;
        // A. passes over all keys until the threshold bin holds <= kListMax
        for (int pass = 0;; ++pass) {
            if (c.hi == 0) {  // one key value left
                c.thr_gt = c.thr_eq = base + c.prefix;
                c.need = K - c.above;
                c.done = true;
                break;
            }
            const int d = c.hi < kBinBits ? c.hi : kBinBits, lo = c.hi - d, nb = 1 << d;
            if (pass) {
                __syncthreads();  // every thread has read the last pass's bins
                zero_bins(sc, nb);
                __syncthreads();
            }
            const uint32_t mask = c.hi >= 32 ? 0u : (0xFFFFFFFFu << c.hi);
            const uint32_t pfx = c.hi >= 32 ? 0u : (c.prefix << c.hi);
#pragma unroll 1
            for (int j = 0; j < kPerThread; ++j) {
                const uint32_t k = key(j), v = k - base;
                if (k >= base && (v & mask) == pfx) atomicAdd(&sc.hist[(v >> lo) & (nb - 1)], 1u);
            }
            __syncthreads();
            uint32_t bin, ab;
            find_bin(nb, K - c.above, sc, &bin, &ab, sb);
            c.above += ab;
            const uint32_t in_bin = sc.hist[bin];
            const uint32_t P = (c.prefix << d) | bin;
            if (in_bin == K - c.above) {  // the bin is taken whole
                c.thr_gt = base + (P << lo) - 1u;
                c.done = true;
                break;
            }
            if (lo == 0) {  // the bin is one key value
                c.thr_gt = c.thr_eq = base + P;
                c.need = K - c.above;
                c.done = true;
                break;
            }
            c.prefix = P;
            c.hi = lo;
            if (in_bin <= kListMax) break;
        }
        if (!c.done) {
            // B. the bin's keys into the list, in candidate order
            uint32_t mine = 0;
#pragma unroll 1
            for (int j = 0; j < kPerThread; ++j) {
                const uint32_t k = key(j);
                mine += (k >= base && ((k - base) >> c.hi) == c.prefix) ? 1u : 0u;
            }
            uint32_t m;
            uint32_t off = block_scan(mine, sc, &m, sb);
#pragma unroll 1
            for (int j = 0; j < kPerThread; ++j) {
                const uint32_t k = key(j);
                if (k >= base && ((k - base) >> c.hi) == c.prefix) {
                    sc.lk[off] = k;
                    sc.lc[off] = c0 + j;
                    ++off;
                }
            }
            __syncthreads();
            list_rank(c, m, base, K, sc, sb);
        }
    }
    // Output (every key read before the scan's barrier, so obuf may be the
    // key array)
    uint32_t sel = 0, tie = 0;
#pragma unroll 1
    for (int j = 0; j < kPerThread; ++j) {
        const uint32_t k = key(j);
        sel |= (k > c.thr_gt ? 1u : 0u) << j;
        tie |= (c.need && k == c.thr_eq ? 1u : 0u) << j;
    }
    uint32_t tot2;
    const uint32_t ex = block_scan((static_cast<uint32_t>(__popc(sel)) << 16) | static_cast<uint32_t>(__popc(tie)), sc,
                                   &tot2, sb);
    const uint32_t a_before = ex >> 16, t_before = ex & 0xFFFFu;
    if (c.need) {
        uint32_t take = c.need > t_before ? c.need - t_before : 0u;
        uint32_t tb = tie;
        while (take && tb) {
            sel |= tb & (~tb + 1u);
            tb &= tb - 1u;
            --take;
        }
    }
    uint32_t pos = a_before + min(t_before, c.need);
    while (sel) {
        const int j = __ffs(static_cast<int>(sel)) - 1;
        obuf[pos++] = c0 + j;
        sel &= sel - 1u;
    }
    __syncthreads();
    return static_cast<int>(total > K ? K : total);
}

// The K largest of the keys of candidates [0, n), n <= kMaxKeys, read from
// keys[key_slot(c)].  Writes the kept candidates' indices in ascending order
// to obuf[0, kept) and returns kept = min(K, number of non-zero keys).  keys
// is kMaxKeys entries of shared memory that the selection may overwrite
// (every key is in registers before the first write); obuf may be the key
// array itself.  Called by all kThreads threads, after a CTA barrier that
// follows the keys' stores (and any earlier use of the scratch); ends with a
// CTA barrier (obuf is then complete).
__device__ __forceinline__ int select_keys(uint32_t *keys, int n, uint32_t K, int32_t *obuf, Scratch &sc)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = tid * kPerThread;
    uint32_t kk[kPerThread];
    {
        const uint4 *kv = reinterpret_cast<const uint4 *>(keys + c0);
#pragma unroll
        for (int m = 0; m < kPerThread / 4; ++m) {
            const uint4 v = kv[m ^ (tid & 7)];
            kk[4 * m] = c0 + 4 * m < n ? v.x : 0u;
            kk[4 * m + 1] = c0 + 4 * m + 1 < n ? v.y : 0u;
            kk[4 * m + 2] = c0 + 4 * m + 2 < n ? v.z : 0u;
            kk[4 * m + 3] = c0 + 4 * m + 3 < n ? v.w : 0u;
        }
    }
    uint32_t cnt = 0, kmin = 0xFFFFFFFFu, kmax = 0, gmin = 0xFFFFFFFFu, gcnt = 0;
#pragma unroll
    for (int g = 0; g < kPerThread / kGroup; ++g) {
        uint32_t gm = 0;  // the group's largest key (0: an empty group)
#pragma unroll
        for (int j = g * kGroup; j < (g + 1) * kGroup; ++j) {
            const uint32_t k = kk[j];
            cnt += k ? 1u : 0u;
            kmin = min(kmin, k ? k : 0xFFFFFFFFu);
            gm = max(gm, k);
        }
        kmax = max(kmax, gm);
        gmin = min(gmin, gm ? gm : 0xFFFFFFFFu);
        gcnt += gm ? 1u : 0u;
    }
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
    gmin = __reduce_min_sync(0xFFFFFFFFu, gmin);
    gcnt = __reduce_add_sync(0xFFFFFFFFu, gcnt);
    if (lane == 0) {
        sc.wa[warp] = kmin;
        sc.wb[warp] = kmax;
        sc.wc[warp] = cnt;
        sc.wd[warp] = gmin;
        sc.we[warp] = gcnt;
    }
    zero_bins(sc, kBins);  // the first pass's bins, ordered before it by the barrier below
    __syncthreads();
    // lane i reads warp i's values (kWarps <= 32)
    const bool wl = lane < kWarps;
    kmin = __reduce_min_sync(0xFFFFFFFFu, wl ? sc.wa[lane] : 0xFFFFFFFFu);
    kmax = __reduce_max_sync(0xFFFFFFFFu, wl ? sc.wb[lane] : 0u);
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, wl ? sc.wc[lane] : 0u);
    gmin = __reduce_min_sync(0xFFFFFFFFu, wl ? sc.wd[lane] : 0xFFFFFFFFu);
    gcnt = __reduce_add_sync(0xFFFFFFFFu, wl ? sc.we[lane] : 0u);
    // Keys below base are never kept; every non-zero key is >= kmin >= 1, so
    // "key >= base" also excludes the empty candidates.
    const uint32_t base = gcnt >= K ? gmin : kmin;
    int sb = 0;  // block_scan's buffer
    if (total > K) {
        // The keys >= base, if few, move into the big list in candidate order
        // (over the key array: every key is in registers), kBigPer entries a
        // thread, and the passes run over those instead of over 32 keys a
        // thread of which most lie below base.
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) mine += kk[j] >= base ? 1u : 0u;
        uint32_t nb_list;
        uint32_t off = block_scan(mine, sc, &nb_list, sb);
        if (nb_list <= static_cast<uint32_t>(kBigList)) {
            // entry i = (key, candidate) in one 8-byte store
            uint2 *bl = reinterpret_cast<uint2 *>(keys);
#pragma unroll
            for (int j = 0; j < kPerThread; ++j)
                if (kk[j] >= base) bl[off++] = make_uint2(kk[j], static_cast<uint32_t>(c0 + j));
            __syncthreads();
            uint32_t e[kBigPer];   // this thread's entries of the list
            int32_t ec[kBigPer];   // and their candidates
            const int i0 = tid * kBigPer;
#pragma unroll
            for (int q = 0; q < kBigPer / 2; ++q) {
                const uint4 v = *reinterpret_cast<const uint4 *>(bl + i0 + 2 * q);  // entries i0+2q, i0+2q+1
                const bool h0 = static_cast<uint32_t>(i0 + 2 * q) < nb_list, h1 = static_cast<uint32_t>(i0 + 2 * q + 1) < nb_list;
                e[2 * q] = h0 ? v.x : 0u;
                ec[2 * q] = h0 ? static_cast<int32_t>(v.y) : 0;
                e[2 * q + 1] = h1 ? v.z : 0u;
                ec[2 * q + 1] = h1 ? static_cast<int32_t>(v.w) : 0;
            }
            auto from_list = [&](int j) { return ec[j]; };
            Cut c;
            const uint32_t range = kmax - base;
            c.hi = range ? 32 - __clz(static_cast<int>(range)) : 0;
            passes<kBigPer>(e, base, K, c, sc, sb);
            if (!c.done) list_rank(c, gather<kBigPer>(e, from_list, base, c, sc, sb), base, K, sc, sb);
            // Output: every kept key is >= base, so the list alone holds them.
            write_kept<kBigPer>(e, from_list, c, obuf, sc, sb);
            return static_cast<int>(K);
        }
    }
    return select_keys_smem(keys, n, K, base, kmax, total, obuf, sc, sb);
}

}  // namespace cta_select
}  // namespace csa
