// Persistent cache records: rows of the global cache written out as records,
// and records appended back.  "G2C Brief - DeepSeek V4.1-Flash", section "FP4
// cache entries, and why they're safe" (the derivation of the 890 bytes per
// token: a main entry of 288 B and an MXFP4 indexer entry of 68 B, 356 B an
// entry).  A record holds the main entry's code bytes, its scale bytes, then
// the indexer entry's bytes (E4M3: d_index bytes; MXFP4: d_index/2 code bytes,
// then d_index/32 scale bytes).
//
// Both directions only move bytes, so they are bound by memory bandwidth (the
// device's, or the host link's when the records live in pinned host memory).
// Every field is a whole number of 4-byte words; a record is not always a
// whole number of 16-byte words (356 B).  A CTA takes a tile of kTile
// consecutive rows of one sequence and stages them in shared memory in record
// order: on the cache side each field of the tile is one contiguous run, read
// or written word by word by consecutive threads; on the record side the tile
// is one contiguous block.  Every thread keeps several independent loads in
// flight in each phase.
#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kThreads = 256;

struct Fields {
    int cw, sw, kw, xw;  // words of codes, scales, key codes, key scales
    __host__ __device__ int words() const { return cw + sw + kw + xw; }
};

Fields fields_of(const CacheView &c)
{
    Fields f;
    f.cw = c.D / 2 / 4;
    f.sw = c.D / 16 / 4;
    f.kw = (c.mx ? c.DI / 2 : c.DI) / 4;
    f.xw = c.mx ? c.DI / 32 / 4 : 0;
    return f;
}

constexpr int kTile = 64;  // rows (records) per CTA

// Field f of rows [r, r + kTile) of row-major array `base` (fw words a row) is
// the contiguous run base + r * fw; word j of it belongs to record j / fw.
struct FieldRun {
    uint32_t *base;
    int fw, off;  // words a row, word offset in the record
};

// j / fw for j < 2^16 and 1 < fw < 2^16 by a multiply-high with
// m = floor((2^32 - 1) / fw) + 1 (exact there: the error term
// j * (fw * m - 2^32) stays below 2^32); fw = 1 is marked by m = 0.
__device__ __forceinline__ uint32_t div_magic(int fw)
{
    return fw == 1 ? 0u : 0xFFFFFFFFu / static_cast<uint32_t>(fw) + 1u;
}
__device__ __forceinline__ int div_by(int j, uint32_t m)
{
    return m ? static_cast<int>(__umulhi(static_cast<uint32_t>(j), m)) : j;
}

__device__ __forceinline__ FieldRun field_run(const CacheView &c, const Fields &f, int k)
{
    if (k == 0) return {reinterpret_cast<uint32_t *>(c.codes), f.cw, 0};
    if (k == 1) return {reinterpret_cast<uint32_t *>(c.scales), f.sw, f.cw};
    if (k == 2) return {reinterpret_cast<uint32_t *>(c.ikeys), f.kw, f.cw + f.sw};
    return {reinterpret_cast<uint32_t *>(c.iscales), f.xw, f.cw + f.sw + f.kw};
}

// Records of rows [row0, row0 + n) of every sequence into out [B][n][record];
// rows at or past the sequence's length become zero records.
// Grid: (tiles of kTile rows, B).
__global__ void __launch_bounds__(kThreads) spill_kernel(CacheView c, Fields f, int row0, int n, uint32_t *out)
{
    extern __shared__ uint32_t tile[];  // [kTile][record words]
    pdl_wait();
    const int b = blockIdx.y;
    const int i0 = blockIdx.x * kTile;
    const int rows = min(kTile, n - i0);
    const int rw = f.words();
    const int valid = max(0, min(rows, c.lengths[b] - (row0 + i0)));  // rows below the length
    const int64_t row = static_cast<int64_t>(b) * c.cap + row0 + i0;
    for (int k = 0; k < 4; ++k) {
        const FieldRun fr = field_run(c, f, k);
        if (fr.fw == 0) continue;
        const uint32_t *src = fr.base + row * fr.fw;
        const int words = rows * fr.fw;
        const uint32_t m = div_magic(fr.fw);
        for (int j = threadIdx.x; j < words; j += kThreads) {
            const int rec = div_by(j, m);
            tile[rec * rw + fr.off + (j - rec * fr.fw)] = rec < valid ? src[j] : 0u;
        }
    }
    __syncthreads();
    uint32_t *dst = out + (static_cast<int64_t>(b) * n + i0) * rw;
    for (int j = threadIdx.x; j < rows * rw; j += kThreads) dst[j] = tile[j];
    pdl_trigger();
}

// Records in[B][n][record] appended at rows lengths[b] .. lengths[b] + n - 1;
// a sequence that would pass capacity is left as it is and raises
// CSA_DEV_CAPACITY.  The lengths advance in a second kernel.
// Grid: (tiles of kTile records, B).
__global__ void __launch_bounds__(kThreads) reload_kernel(CacheView c, Fields f, int n, const uint32_t *in,
                                                           int *status)
{
    extern __shared__ uint32_t tile[];  // [kTile][record words]
    pdl_wait();
    const int b = blockIdx.y;
    const int i0 = blockIdx.x * kTile;
    const int rows = min(kTile, n - i0);
    const int rw = f.words();
    const int len0 = c.lengths[b];
    if (len0 < 0 || len0 + n > c.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, CSA_DEV_CAPACITY);
        pdl_trigger();
        return;
    }
    const uint32_t *src = in + (static_cast<int64_t>(b) * n + i0) * rw;
    for (int j = threadIdx.x; j < rows * rw; j += kThreads) tile[j] = src[j];
    __syncthreads();
    const int64_t row = static_cast<int64_t>(b) * c.cap + len0 + i0;
    for (int k = 0; k < 4; ++k) {
        const FieldRun fr = field_run(c, f, k);
        if (fr.fw == 0) continue;
        uint32_t *dst = fr.base + row * fr.fw;
        const int words = rows * fr.fw;
        const uint32_t m = div_magic(fr.fw);
        for (int j = threadIdx.x; j < words; j += kThreads) {
            const int rec = div_by(j, m);
            dst[j] = tile[rec * rw + fr.off + (j - rec * fr.fw)];
        }
    }
    pdl_trigger();
}

__global__ void reload_lengths_kernel(int32_t *lengths, int B, int cap, int n)
{
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        const int len0 = lengths[b];
        if (len0 >= 0 && len0 + n <= cap) lengths[b] = len0 + n;
    }
}

}  // namespace

size_t record_bytes(const CacheView &c) { return static_cast<size_t>(fields_of(c).words()) * 4; }

cudaError_t launch_spill(const CacheView &c, int row0, int n, uint8_t *out, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    const Fields f = fields_of(c);
    const size_t smem = static_cast<size_t>(kTile) * f.words() * 4;
    return launch_kernel(spill_kernel, dim3((n + kTile - 1) / kTile, c.B), dim3(kThreads), smem, st, 0, c, f, row0, n,
                         reinterpret_cast<uint32_t *>(out));
}

cudaError_t launch_reload(const CacheView &c, const uint8_t *in, int n, int *status, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    const Fields f = fields_of(c);
    const size_t smem = static_cast<size_t>(kTile) * f.words() * 4;
    const cudaError_t e = launch_kernel(reload_kernel, dim3((n + kTile - 1) / kTile, c.B), dim3(kThreads), smem, st,
                                        0, c, f, n, reinterpret_cast<const uint32_t *>(in), status);
    if (e != cudaSuccess) return e;
    return launch_kernel(reload_lengths_kernel, dim3((c.B + 127) / 128), dim3(128), 0, st, 0, c.lengths, c.B, c.cap,
                         n);
}

}  // namespace csa
