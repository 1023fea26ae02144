// a5/a6: sparse attention of each query over its selected FP4 rows, split
// over the selection (flash-decode) with a merge pass.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select": the query attends to only the selected entries; one shared
// 512-dim latent per entry serves every query head.  "DeepSeek V4.1 Flash:
// Pushing the Limits", section "The Paper": a single W_KV, so keys and values
// are the same vector.
//
// First version: CUDA cores.  Each CTA takes one (sequence, position) and a
// contiguous share of its selection, walks it in tiles of kTile rows with an
// online softmax, and writes an unnormalised partial (O, m, l) per head.  The
// merge kernel combines the partials of a query.
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kTile = 32;
constexpr int kAttThreads = 256;

struct AttArgs {
    CacheView c;
    int P, H, K;
    const uint16_t *q;
    float scale;
    const int32_t *idx;
    int nsplit, keys_per_split;
    float *part_o;     // [units][nsplit][H][D]
    float2 *part_ml;   // [units][nsplit][H]
    int *status;
};

__device__ __forceinline__ float e2m1_value(uint32_t code)
{
    const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
    const float v = mag[code & 7];
    return (code & 8) ? -v : v;
}

__device__ __forceinline__ float e4m3_value(uint32_t byte)
{
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3)));
}

__global__ void __launch_bounds__(kAttThreads, 1) attend_simple_kernel(AttArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int D = a.c.D, H = a.H;
    uint16_t *qs = reinterpret_cast<uint16_t *>(smem);                        // [H][D] bf16 bits
    float *vs = reinterpret_cast<float *>(smem + static_cast<size_t>(H) * D * 2);  // [kTile][D]
    float *ss = vs + kTile * D;                                               // [H][kTile]
    float *mh = ss + H * kTile;                                               // [H] running max
    float *lh = mh + H;                                                       // [H] running sum
    float *fh = lh + H;                                                       // [H] rescale factor
    int *valid = reinterpret_cast<int *>(fh + H);                             // [kTile]

    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / a.P;
    const int len = a.c.lengths[b];
    const int tid = threadIdx.x;
    const int n_out = H * D;
    const int per_thread = (n_out + kAttThreads - 1) / kAttThreads;  // <= 128

    for (int i = tid; i < H * D / 8; i += kAttThreads)
        reinterpret_cast<uint4 *>(qs)[i] =
            reinterpret_cast<const uint4 *>(a.q + static_cast<int64_t>(unit) * H * D)[i];
    for (int h = tid; h < H; h += kAttThreads) {
        mh[h] = -INFINITY;
        lh[h] = 0.f;
    }
    float acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0.f;

    const int j0 = split * a.keys_per_split;
    const int j1 = min(a.K, j0 + a.keys_per_split);
    const int32_t *irow = a.idx + static_cast<int64_t>(unit) * a.K;
    for (int t0 = j0; t0 < j1; t0 += kTile) {
        __syncthreads();
        // dequantise the tile's rows into fp32
        for (int e = tid; e < kTile * D; e += kAttThreads) {
            const int j = e / D, d = e % D;
            int32_t row = (t0 + j < j1) ? irow[t0 + j] : -1;
            if (row >= len) {
                if (d == 0) raise_status(a.status, CSA_DEV_BAD_INDEX);
                row = -1;
            }
            float v = 0.f;
            if (row >= 0) {
                const int64_t g = static_cast<int64_t>(b) * a.c.cap + row;
                const uint32_t byte = a.c.codes[g * (D / 2) + d / 2];
                v = e2m1_value((d & 1) ? (byte >> 4) : (byte & 0xF)) * e4m3_value(a.c.scales[g * (D / 16) + d / 16]);
            }
            vs[e] = v;
            if (d == 0) valid[j] = row >= 0;
        }
        __syncthreads();
        // logits
        for (int e = tid; e < H * kTile; e += kAttThreads) {
            const int h = e / kTile, j = e % kTile;
            float dot = 0.f;
            for (int d = 0; d < D; ++d)
                dot = fmaf(__uint_as_float(static_cast<uint32_t>(qs[h * D + d]) << 16), vs[j * D + d], dot);
            ss[e] = valid[j] ? a.scale * dot : -INFINITY;
        }
        __syncthreads();
        // online softmax statistics per head
        for (int h = tid; h < H; h += kAttThreads) {
            float mt = -INFINITY;
            for (int j = 0; j < kTile; ++j) mt = fmaxf(mt, ss[h * kTile + j]);
            const float mnew = fmaxf(mh[h], mt);
            const float f = (mnew == -INFINITY) ? 1.f : __expf(mh[h] - mnew);
            float l = lh[h] * f;
            for (int j = 0; j < kTile; ++j) {
                const float pj = (mnew == -INFINITY) ? 0.f : __expf(ss[h * kTile + j] - mnew);
                ss[h * kTile + j] = pj;
                l += pj;
            }
            mh[h] = mnew;
            lh[h] = l;
            fh[h] = f;
        }
        __syncthreads();
#pragma unroll 4
        for (int i = 0; i < per_thread; ++i) {
            const int o = tid + i * kAttThreads;
            if (o < n_out) {
                const int h = o / D, d = o % D;
                float s = acc[i] * fh[h];
                for (int j = 0; j < kTile; ++j) s = fmaf(ss[h * kTile + j], vs[j * D + d], s);
                acc[i] = s;
            }
        }
    }
    __syncthreads();
    float *po = a.part_o + (static_cast<int64_t>(unit) * a.nsplit + split) * n_out;
    for (int i = 0; i < per_thread; ++i) {
        const int o = tid + i * kAttThreads;
        if (o < n_out) po[o] = acc[i];
    }
    for (int h = tid; h < H; h += kAttThreads)
        a.part_ml[(static_cast<int64_t>(unit) * a.nsplit + split) * H + h] = make_float2(mh[h], lh[h]);
}

// Combines the split partials of one (query, head): out = sum_s e^{m_s-M} O_s / sum_s e^{m_s-M} l_s.
__global__ void attend_merge_kernel(int D, int H, int nsplit, const float *__restrict__ part_o,
                                    const float2 *__restrict__ part_ml, float *__restrict__ out,
                                    float *__restrict__ lse)
{
    extern __shared__ float wsh[];  // [nsplit] weights
    const int unit = blockIdx.y, h = blockIdx.x;
    __shared__ float inv_l, lse_v;
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[(static_cast<int64_t>(unit) * nsplit + s) * H + h].x);
        float L = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float2 ml = part_ml[(static_cast<int64_t>(unit) * nsplit + s) * H + h];
            const float wgt = (M == -INFINITY || ml.x == -INFINITY) ? 0.f : __expf(ml.x - M);
            wsh[s] = wgt;
            L += wgt * ml.y;
        }
        inv_l = L > 0.f ? 1.f / L : 0.f;
        lse_v = L > 0.f ? M + __logf(L) : -INFINITY;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < nsplit; ++s)
            acc = fmaf(wsh[s], part_o[((static_cast<int64_t>(unit) * nsplit + s) * H + h) * D + d], acc);
        out[(static_cast<int64_t>(unit) * H + h) * D + d] = acc * inv_l;
    }
    if (lse && threadIdx.x == 0) lse[static_cast<int64_t>(unit) * H + h] = lse_v;
}

void plan(const CacheView &c, int P, int H, int K, int &nsplit, int &kps)
{
    const int units = c.B * P;
    int want = (2 * 148 + units - 1) / units;
    const int max_split = (K + kTile - 1) / kTile;
    if (want > max_split) want = max_split;
    if (want < 1) want = 1;
    kps = (K + want - 1) / want;
    kps = (kps + kTile - 1) / kTile * kTile;
    nsplit = (K + kps - 1) / kps;
}

}  // namespace

size_t attend_workspace_bytes(const CacheView &c, int P, int H, int K)
{
    int nsplit, kps;
    plan(c, P, H, K, nsplit, kps);
    const size_t units = static_cast<size_t>(c.B) * P;
    size_t o = units * nsplit * H * c.D * sizeof(float);
    o = (o + 255) / 256 * 256;
    return o + units * nsplit * H * sizeof(float2);
}

cudaError_t launch_attend(const CacheView &c, int P, int H, const uint16_t *q, float scale, const int32_t *idx,
                          int K, float *out, float *lse, void *ws, size_t ws_bytes, int *status, cudaStream_t st)
{
    const int units = c.B * P;
    if (units == 0) return cudaSuccess;
    int nsplit, kps;
    plan(c, P, H, K, nsplit, kps);
    if (ws_bytes < attend_workspace_bytes(c, P, H, K)) return cudaErrorInvalidValue;
    size_t o_bytes = static_cast<size_t>(units) * nsplit * H * c.D * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    AttArgs a{c, P, H, K, q, scale, idx, nsplit, kps, static_cast<float *>(ws),
              reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + o_bytes), status};
    const size_t smem = static_cast<size_t>(H) * c.D * 2 + static_cast<size_t>(kTile) * c.D * 4 +
                        static_cast<size_t>(H) * kTile * 4 + 3 * H * 4 + kTile * 4;
    cudaError_t e =
        cudaFuncSetAttribute(attend_simple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attend_simple_kernel<<<dim3(nsplit, units), kAttThreads, smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
    attend_merge_kernel<<<dim3(H, units), 128, nsplit * sizeof(float), st>>>(c.D, H, nsplit, a.part_o, a.part_ml, out,
                                                                           lse);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace csa
