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
    if (ikeys_new && c.mx) {
        // packed MXFP4 rows (codes then scales), 4-byte words: DI/8 of codes, DI/128 of scales
        const int64_t wpr = c.DI / 8 + c.DI / 128;
        const int64_t total_k = static_cast<int64_t>(n_new) * wpr;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_k;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int64_t j = i / wpr, k = i % wpr;
            const uint32_t x = *reinterpret_cast<const uint32_t *>(ikeys_new + (static_cast<int64_t>(b) * n_new + j) *
                                                                                   (wpr * 4) + k * 4);
            if (k < c.DI / 8)
                *reinterpret_cast<uint32_t *>(c.ikeys + (base_row + j) * (c.DI / 2) + k * 4) = x;
            else
                *reinterpret_cast<uint32_t *>(c.iscales + (base_row + j) * (c.DI / 32) + (k - c.DI / 8) * 4) = x;
        }
    } else if (ikeys_new) {
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

// Indexer keys projected from the just-stored main cache entries.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select": the indexer's keys are a projection of the main cache
// entries rather than a separately computed cache.
//     ik[j] = E4M3( sum_c v[c] * w[c][j] ),  v = E2M1(code) * E4M3(scale)
// One CTA per (up to kProjRows new rows, sequence, kProjCols key channels);
// runs after the append kernel, before the lengths advance, and reads the rows
// it stored (from L2).  The dequantised rows are exact in fp32 and held in
// shared memory as [channel][row]; thread (channel slice, row half, group of 4
// key channels) accumulates 4 rows x 4 key channels over its slice in fp32
// (w read as 4 bf16 at a time, coalesced along the key channels); the slices
// are summed, and each sum is rounded once to E4M3 (nearest, ties to even,
// saturating at 448).
constexpr int kProjThreads = 256;
constexpr int kProjRows = 8;
constexpr int kProjCols = 32;                                 // key channels per CTA
constexpr int kProjGroups = kProjCols / 4;                    // groups of 4 key channels
constexpr int kProjSlices = kProjThreads / (2 * kProjGroups);  // channel slices (16)

__device__ __forceinline__ float e4m3_byte_to_float(uint8_t byte)
{
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3)));
}

__device__ __forceinline__ float2 e2m1_pair(uint8_t byte)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(uint32_t(byte)));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

__global__ void __launch_bounds__(kProjThreads) project_ikeys_kernel(CacheView c, const uint16_t *__restrict__ w,
                                                                     int n_new)
{
    extern __shared__ __align__(16) float psm[];
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, tid = threadIdx.x;
    const int len0 = c.lengths[b];
    if (len0 < 0 || len0 + n_new > c.cap) return;  // left unchanged (and flagged) by the append kernel
    const int D = c.D, DI = c.DI;
    const int j0 = blockIdx.x * kProjRows, col0 = blockIdx.z * kProjCols;
    const int nr = min(kProjRows, n_new - j0);
    const int64_t row0 = static_cast<int64_t>(b) * c.cap + len0 + j0;
    float *v = psm;                                // [D][kProjRows]
    float *part = psm + D * kProjRows;             // [kProjSlices][kProjRows][kProjCols]
    // Dequantise: thread (code byte, row), rows fastest; the loads of all its
    // iterations are issued before any is used.
    constexpr int kDq = 8;
    for (int i0 = 0; i0 < kProjRows * (D / 2); i0 += kDq * kProjThreads) {
        uint8_t cb8[kDq], sb8[kDq];
#pragma unroll
        for (int u = 0; u < kDq; ++u) {
            const int i = i0 + u * kProjThreads + tid;
            const int r = i % kProjRows, cb = i / kProjRows;
            const bool live = i < kProjRows * (D / 2) && r < nr;
            cb8[u] = live ? c.codes[(row0 + r) * (D / 2) + cb] : 0;
            sb8[u] = live ? c.scales[(row0 + r) * (D / 16) + cb / 8] : 0;
        }
#pragma unroll
        for (int u = 0; u < kDq; ++u) {
            const int i = i0 + u * kProjThreads + tid;
            if (i >= kProjRows * (D / 2)) break;
            const int r = i % kProjRows, cb = i / kProjRows;
            const float s = e4m3_byte_to_float(sb8[u]);
            const float2 x = e2m1_pair(cb8[u]);
            v[(2 * cb) * kProjRows + r] = x.x * s;
            v[(2 * cb + 1) * kProjRows + r] = x.y * s;
        }
    }
    __syncthreads();
    const int ks = tid / (2 * kProjGroups), rh = (tid / kProjGroups) & 1, jg = tid % kProjGroups;
    const int cpk = D / kProjSlices;
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
    const uint16_t *wp = w + static_cast<int64_t>(ks * cpk) * DI + col0 + jg * 4;
    const float *vp = v + ks * cpk * kProjRows + rh * 4;
    // w comes from L2: sixteen channels' loads are issued before their use.
    constexpr int kBatch = 16;
    for (int cc0 = 0; cc0 < cpk; cc0 += kBatch) {
        uint2 wb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            wb[u] = cc0 + u < cpk ? __ldg(reinterpret_cast<const uint2 *>(wp + static_cast<int64_t>(cc0 + u) * DI))
                                  : make_uint2(0u, 0u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (cc0 + u >= cpk) break;
            const float4 vv = *reinterpret_cast<const float4 *>(vp + (cc0 + u) * kProjRows);
            const float wq[4] = {__uint_as_float(wb[u].x << 16), __uint_as_float(wb[u].x & 0xFFFF0000u),
                                 __uint_as_float(wb[u].y << 16), __uint_as_float(wb[u].y & 0xFFFF0000u)};
            const float vr[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(vr[r], wq[q], acc[r][q]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4 *>(part + (ks * kProjRows + rh * 4 + r) * kProjCols + jg * 4) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    __syncthreads();
    // One warp per row (nr * 32 <= kProjThreads): lane j sums key channel col0 + j.
    for (int i = tid; i < nr * kProjCols; i += kProjThreads) {
        const int r = i / kProjCols, j = i - r * kProjCols;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kProjSlices; ++q) sum += part[(q * kProjRows + r) * kProjCols + j];
        if (!c.mx) {
            c.ikeys[(row0 + r) * DI + col0 + j] =
                static_cast<uint8_t>(__nv_cvt_float_to_fp8(sum, __NV_SATFINITE, __NV_E4M3));
            continue;
        }
        // MXFP4: the 32 channels of this CTA are one block.  X = floor(log2
        // amax) - 2 clamped to [-8, 6] (amax's exponent field; -8 for zero or
        // a subnormal), codes from |sum| * 2^-X (exact) against the E2M1
        // midpoints, ties to the even code, 6 beyond.
        float amax = fabsf(sum);
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
        const int X = ex == 0 ? -8 : min(6, max(-8, ex - 127 - 2));
        const float q = fabsf(sum) * __uint_as_float(static_cast<uint32_t>(127 - X) << 23);
        const uint32_t code = ((q > 0.25f) + (q >= 0.75f) + (q > 1.25f) + (q >= 1.75f) + (q > 2.5f) + (q >= 3.5f) +
                               (q > 5.0f)) |
                              (__float_as_uint(sum) >> 28 & 0x8u);
        const uint32_t pair = code | (__shfl_down_sync(0xFFFFFFFFu, code, 1) << 4);
        if ((j & 1) == 0) c.ikeys[(row0 + r) * (DI / 2) + (col0 + j) / 2] = static_cast<uint8_t>(pair);
        if (j == 0) c.iscales[(row0 + r) * (DI / 32) + col0 / 32] = static_cast<uint8_t>(X + 127);
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

size_t project_smem_bytes(const CacheView &c)
{
    return static_cast<size_t>(c.D) * kProjRows * sizeof(float) +
           static_cast<size_t>(kProjSlices) * kProjRows * kProjCols * sizeof(float);
}

cudaError_t launch_quantize_append(const CacheView &c, const uint16_t *rows, const uint8_t *ikeys_new, int n_new,
                                   int *status, cudaStream_t st, const uint16_t *w_ik)
{
    if (n_new <= 0) return cudaSuccess;
    const int64_t work = static_cast<int64_t>(n_new) * (c.D / 8);
    int64_t blocks_x = (work + 255) / 256;
    const int64_t want = (4 * static_cast<int64_t>(sm_count()) + c.B - 1) / c.B;  // cover the GPU for tiny appends too
    if (blocks_x > want * 8) blocks_x = want * 8;
    if (blocks_x < 1) blocks_x = 1;
    dim3 grid(static_cast<unsigned>(blocks_x), c.B);
    cudaError_t e = launch_kernel(quantize_append_kernel, grid, dim3(256), 0, st, 0, c, rows, ikeys_new, n_new,
                                  status);
    if (e != cudaSuccess) return e;
    if (w_ik) {
        if (c.DI != 32 && c.DI != 64 && c.DI != 128) return cudaErrorInvalidValue;
        const size_t smem = project_smem_bytes(c);
        e = cudaFuncSetAttribute(project_ikeys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_kernel(project_ikeys_kernel, dim3((n_new + kProjRows - 1) / kProjRows, c.B, c.DI / kProjCols),
                          dim3(kProjThreads), smem, st, 0, c, w_ik, n_new);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(advance_lengths_kernel, dim3((c.B + 127) / 128), dim3(128), 0, st, 0, c.lengths, c.B, c.cap,
                         n_new);
}

}  // namespace csa
