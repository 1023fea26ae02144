// The context split of one long sequence over several devices (row slices):
// each device scores its own slice and keeps a local top K as (score, global
// id) pairs; the pairs of every device are gathered and the global top K is
// selected among them (which is exact: a row of the global top K is in its
// slice's top K, the same order deciding both); each device attends over the
// selected rows in its slice; the partial outputs are merged by log-sum-exp.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select" (score every entry, keep the best, attend to those only) and
// "The hierarchical indexer" (blocks of 8 scored by their best member).
// The kernels here are the device steps of that split that the single-device
// path does not have: pairs from a local selection, the window of global ids
// a device owns, and the merge.
#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2ef = 1.4426950408889634f;

// Pairs of row r (one per query unit): score of the selected candidate (its
// best member's score over the visible rows for blocks of 8) and its id plus
// the slice's first global row (or block).  Empty slots give (-inf, -1).
__global__ void pairs_from_idx_kernel(const float *scores, int64_t ld, const int32_t *lengths, int cap, int P,
                                      const int32_t *idx, int n, int block, int32_t id_offset, float *pair_scores,
                                      int32_t *pair_ids)
{
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int b = row / P, p = row % P;
    const int L = min(lengths[b], cap) - P + 1 + p;
    const int32_t id = idx[static_cast<int64_t>(row) * n + j];
    float sc = -INFINITY;
    int32_t gid = -1;
    if (id >= 0) {
        const float *s = scores + static_cast<int64_t>(row) * ld;
        if (block == 1) {
            if (id < L) sc = s[id];
        } else {
            for (int m = 0; m < block; ++m) {
                const int64_t r = static_cast<int64_t>(id) * block + m;
                if (r < L) sc = fmaxf(sc, s[r]);
            }
        }
        gid = id + id_offset;
    }
    pair_scores[static_cast<int64_t>(row) * n + j] = sc;
    pair_ids[static_cast<int64_t>(row) * n + j] = gid;
}

__global__ void ids_window_kernel(const int32_t *ids, int64_t count, int32_t lo, int32_t hi, int32_t *out)
{
    pdl_wait();
    pdl_trigger();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= count) return;
    const int32_t id = ids[i];
    out[i] = (id >= lo && id < hi) ? id - lo : -1;
}

// out = sum_g 2^(m_g - M) O_g / sum_g 2^(m_g - M) (lse_g in natural log; a
// part with lse = -inf has no rows); one thread per 4 dims of a head.
__global__ void lse_merge_kernel(int parts, int units, int H, int D, const float *outs, const float *lses, float *out,
                                 float *lse)
{
    pdl_wait();
    pdl_trigger();
    const int d = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    const int h = blockIdx.y, u = blockIdx.z;
    if (d >= D) return;
    const int64_t stride_part = static_cast<int64_t>(units) * H;
    const int64_t uh = static_cast<int64_t>(u) * H + h;
    float M = -INFINITY;
    for (int g = 0; g < parts; ++g) M = fmaxf(M, lses[g * stride_part + uh] * kLog2ef);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < parts; ++g) {
        const float m = lses[g * stride_part + uh] * kLog2ef;
        if (m == -INFINITY) continue;
        const float w = exp2f(m - M);
        L += w;
        const float4 v = *reinterpret_cast<const float4 *>(outs + (g * stride_part + uh) * D + d);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<float4 *>(out + uh * D + d) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (lse && d == 0) lse[uh] = L > 0.f ? (M + log2f(L)) * kLn2f : -INFINITY;
}

}  // namespace

cudaError_t launch_pairs_from_idx(const CacheView &c, const float *scores, int64_t ld, const int32_t *idx, int n,
                                  int block, int32_t id_offset, float *pair_scores, int32_t *pair_ids, cudaStream_t st)
{
    const int rows = c.B;  // one query position per sequence
    if (rows == 0 || n == 0) return cudaSuccess;
    return launch_kernel(pairs_from_idx_kernel, dim3((n + 255) / 256, rows), dim3(256), 0, st, 0, scores, ld,
                         static_cast<const int32_t *>(c.lengths), c.cap, 1, idx, n, block, id_offset, pair_scores,
                         pair_ids);
}

cudaError_t launch_ids_window(const int32_t *ids, int64_t count, int32_t lo, int32_t hi, int32_t *out, cudaStream_t st)
{
    if (count == 0) return cudaSuccess;
    return launch_kernel(ids_window_kernel, dim3(static_cast<unsigned>((count + 255) / 256)), dim3(256), 0, st, 0, ids,
                         count, lo, hi, out);
}

cudaError_t launch_lse_merge(int parts, int units, int H, int D, const float *outs, const float *lses, float *out,
                             float *lse, cudaStream_t st)
{
    if (units == 0) return cudaSuccess;
    return launch_kernel(lse_merge_kernel, dim3((D / 4 + 127) / 128, H, units), dim3(128), 0, st, 0, parts, units, H,
                         D, outs, lses, out, lse);
}

}  // namespace csa
