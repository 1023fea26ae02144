// a1: quantise new latent rows to FP4 (E2M1 codes + one E4M3 scale per 16
// channels) and append them to the global cache.
// "G2C Brief - DeepSeek V4.1-Flash", section "FP4 cache entries, and why
// they're safe": main cache entries are E2M1 with one E4M3 scale per group of
// 16 channels (NVFP4 without its second-level global scale).
//
// Layout of the work: two threads per 16-channel group.  Each thread issues one
// 128-bit load (8 bf16 channels), the pair exchanges its partial |max| with one
// warp shuffle, and each thread writes its 8 codes as one packed 32-bit store;
// the even thread of the pair writes the scale byte.  Consecutive threads cover
// consecutive channels, so loads and stores are fully coalesced.
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

// E2M1 magnitude code of a = |x| against scale s > 0, by comparison with the
// midpoints between grid values (0, .5, 1, 1.5, 2, 3, 4, 6) times s.  The
// products t*s are exact in fp32 (3 + 4 significant bits), so this is exact
// round-to-nearest; at a midpoint the even code wins: crossing from an even
// code needs a strictly greater value, crossing from an odd code does not.
__device__ __forceinline__ uint32_t e2m1_code(float a, float s)
{
    return (a > 0.25f * s) + (a >= 0.75f * s) + (a > 1.25f * s) + (a >= 1.75f * s) + (a > 2.5f * s) +
           (a >= 3.5f * s) + (a > 5.0f * s);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

__global__ void __launch_bounds__(256) quantize_append_kernel(CacheView c, const uint16_t *__restrict__ rows,
                                                              const uint8_t *__restrict__ ikeys_new, int n_new,
                                                              int *status)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const int len0 = c.lengths[b];
    if (len0 < 0 || len0 + n_new > c.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, CSA_DEV_CAPACITY);
        return;
    }
    const int64_t halves_per_row = c.D / 8;  // 8 channels per thread
    const int64_t total = static_cast<int64_t>(n_new) * halves_per_row;
    const int64_t base_row = static_cast<int64_t>(b) * c.cap + len0;
    // Warp-uniform trip count: every lane of a warp reaches the shuffle in every
    // iteration, and the pair (i, i^1) always shares a warp.
    const int lane = threadIdx.x & 31;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
         base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = base + lane;
        const bool live = i < total;
        const int64_t j = live ? i / halves_per_row : 0;
        const int h = live ? static_cast<int>(i % halves_per_row) : 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (live)
            v = *reinterpret_cast<const uint4 *>(rows + (static_cast<int64_t>(b) * n_new + j) * c.D + h * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[k] & 0xFFFFu)));
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[k] >> 16)));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        if (!live) continue;
        // scale = E4M3 round-to-nearest-even(amax / 6), saturating at 448.
        // amax/6 is a correctly rounded fp32 quotient of a bf16, which is never
        // within an fp32 half-ulp of an E4M3 rounding midpoint unless equal to
        // it, so rounding it again gives the same byte as rounding the exact quotient.
        const __nv_fp8_storage_t sbyte = __nv_cvt_float_to_fp8(amax / 6.0f, __NV_SATFINITE, __NV_E4M3);
        const float s = __half2float(__half(__nv_cvt_fp8_to_halfraw(sbyte, __NV_E4M3)));
        uint32_t packed = 0;
        if (s > 0.f) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t bits = (w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu;
                const uint32_t code = e2m1_code(fabsf(bf16_bits_to_float(bits)), s) | ((bits >> 12) & 0x8u);
                packed |= code << (4 * k);
            }
        }
        const int64_t row = base_row + j;
        *reinterpret_cast<uint32_t *>(c.codes + row * (c.D / 2) + h * 4) = packed;
        if ((h & 1) == 0) c.scales[row * (c.D / 16) + h / 2] = static_cast<uint8_t>(sbyte);
    }
    if (ikeys_new) {
        const int64_t vec_per_row = c.DI / 16;
        const int64_t total_k = static_cast<int64_t>(n_new) * vec_per_row;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_k;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int64_t j = i / vec_per_row, v = i % vec_per_row;
            const uint4 x =
                *reinterpret_cast<const uint4 *>(ikeys_new + (static_cast<int64_t>(b) * n_new + j) * c.DI + v * 16);
            *reinterpret_cast<uint4 *>(c.ikeys + (base_row + j) * c.DI + v * 16) = x;
        }
    }
}

__global__ void advance_lengths_kernel(int32_t *lengths, int B, int cap, int n_new)
{
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        const int len0 = lengths[b];
        if (len0 >= 0 && len0 + n_new <= cap) lengths[b] = len0 + n_new;
    }
}

}  // namespace

cudaError_t launch_quantize_append(const CacheView &c, const uint16_t *rows, const uint8_t *ikeys_new, int n_new,
                                   int *status, cudaStream_t st)
{
    if (n_new <= 0) return cudaSuccess;
    const int64_t work = static_cast<int64_t>(n_new) * (c.D / 8);
    int64_t blocks_x = (work + 255) / 256;
    const int64_t want = (4 * 148 + c.B - 1) / c.B;  // enough CTAs to cover the GPU for tiny appends too
    if (blocks_x > want * 8) blocks_x = want * 8;
    if (blocks_x < 1) blocks_x = 1;
    dim3 grid(static_cast<unsigned>(blocks_x), c.B);
    const cudaError_t e = launch_kernel(quantize_append_kernel, grid, dim3(256), 0, st, 0, c, rows, ikeys_new, n_new,
                                        status);
    if (e != cudaSuccess) return e;
    return launch_kernel(advance_lengths_kernel, dim3((c.B + 127) / 128), dim3(128), 0, st, 0, c.lengths, c.B, c.cap,
                         n_new);
}

}  // namespace csa
