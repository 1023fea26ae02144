// a2/a4: indexer scores, score(t) = sum_h w_h * ReLU(iq_h . ik_t), with FP8
// E4M3 indexer queries and keys.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select" (item 3: a small side network with its own low-precision
// queries and keys scores every cached entry), and section "The hierarchical
// indexer" (Reindex layers rescore only the pool's rows).
//
// First version: CUDA cores.  One thread per candidate row, the query heads
// decoded once per CTA into shared memory.
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

__device__ __forceinline__ float e4m3_to_float(uint32_t byte)
{
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3)));
}

__global__ void __launch_bounds__(128) index_score_simple_kernel(CacheView c, int P, int HI,
                                                                 const uint8_t *__restrict__ iq,
                                                                 const float *__restrict__ w,
                                                                 const int32_t *__restrict__ pool, int pool_blocks,
                                                                 float *__restrict__ scores, int64_t ld)
{
    extern __shared__ float qs[];  // [HI][DI] then w[HI]
    const int r = blockIdx.y;
    const int b = r / P, p = r % P;
    const int L = c.lengths[b] - P + 1 + p;
    const int DI = c.DI;
    for (int i = threadIdx.x; i < HI * DI; i += blockDim.x)
        qs[i] = e4m3_to_float(iq[static_cast<int64_t>(r) * HI * DI + i]);
    for (int h = threadIdx.x; h < HI; h += blockDim.x) qs[HI * DI + h] = w[static_cast<int64_t>(r) * HI + h];
    __syncthreads();
    const int64_t n = pool ? static_cast<int64_t>(pool_blocks) * kPoolBlock : (L > 0 ? L : 0);
    const int32_t *prow = pool ? pool + static_cast<int64_t>(r) * pool_blocks : nullptr;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t row = i;
        if (prow) {
            const int32_t blk = prow[i >> 3];
            row = static_cast<int64_t>(blk) * kPoolBlock + (i & 7);
            if (blk < 0 || row >= L) continue;
        }
        const uint8_t *kr = c.ikeys + (static_cast<int64_t>(b) * c.cap + row) * DI;
        float kf[128];
#pragma unroll
        for (int d = 0; d < 128; ++d)
            if (d < DI) kf[d] = e4m3_to_float(kr[d]);
        float acc = 0.f;
        for (int h = 0; h < HI; ++h) {
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < 128; ++d)
                if (d < DI) dot = fmaf(qs[h * DI + d], kf[d], dot);
            acc = fmaf(qs[HI * DI + h], fmaxf(dot, 0.f), acc);
        }
        scores[static_cast<int64_t>(r) * ld + i] = acc;
    }
}

}  // namespace

cudaError_t launch_index_score(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, float *scores, int64_t ld, int * /*status*/,
                               cudaStream_t st)
{
    const int rows = c.B * P;
    if (rows == 0) return cudaSuccess;
    const int64_t n = pool ? static_cast<int64_t>(pool_blocks) * kPoolBlock : c.cap;
    int64_t bx = (n + 127) / 128;
    if (bx > 65535) bx = 65535;
    const size_t smem = (static_cast<size_t>(HI) * c.DI + HI) * sizeof(float);
    cudaFuncSetAttribute(index_score_simple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    index_score_simple_kernel<<<dim3(static_cast<unsigned>(bx), rows), 128, smem, st>>>(c, P, HI, iq, w, pool,
                                                                                         pool_blocks, scores, ld);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace csa
