// Internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace csa {

struct CacheView {
    int B, cap, D, DI;
    uint8_t *codes, *scales, *ikeys;
    int32_t *lengths;
    int mx;            // MXFP4 indexer keys: ikeys holds DI/2 code bytes per row, iscales DI/32
    uint8_t *iscales;
};

// a1
// w_ik (optional): [D][DI] bf16; the appended rows' indexer keys are then
// projected from their stored entries instead of copied from ikeys_new.
cudaError_t launch_quantize_append(const CacheView &c, const uint16_t *rows, const uint8_t *ikeys_new, int n_new,
                                   int *status, cudaStream_t st, const uint16_t *w_ik = nullptr);

// a2/a4
// bmax (full scan only, or null): each 8-row block's best visible score,
// [B*P][ldb], beside the row scores.
cudaError_t launch_index_score(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, float *scores, int64_t ld, int *status,
                               cudaStream_t st, float *bmax = nullptr, int64_t ldb = 0);

// a3 (and the pool): `block` = 1 selects rows, 8 selects blocks of 8 rows by their best member.
size_t select_workspace_bytes(const CacheView &c, int P, const int32_t *pool, int pool_blocks, int block, int K);
int select_supported(const CacheView &c, const int32_t *pool, int pool_blocks, int block, int K);
// block_max (with block = 8): scores holds each block's best visible score
// ([B*P][ld], from launch_index_score's bmax) instead of the rows' scores.
cudaError_t launch_select(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                          int pool_blocks, int block, int K, int32_t *out, void *ws, size_t ws_bytes,
                          cudaStream_t st, bool block_max = false);

// a4 over a pool in one kernel (scores stay on chip; E4M3 keys, HI <= 64,
// pools of up to 2,048 blocks).
int pool_select_supported(const CacheView &c, int P, int HI, int pool_blocks, int K);
cudaError_t launch_pool_select(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, int K, int32_t *idx, int *status,
                               cudaStream_t st);
// A Reindex layer over the pool spread over one CTA per 128-row tile, the last
// CTA of each query selecting; keys: [B*P][pool_blocks * 8] words of scratch
// (pool_spread_keys_bytes).  Uses library-owned arrival counters.
int pool_spread_supported(const CacheView &c, int P, int HI, int pool_blocks, int K);
size_t pool_spread_keys_bytes(const CacheView &c, int P, int pool_blocks);
cudaError_t launch_pool_spread(const CacheView &c, int P, int HI, const uint8_t *iq, const float *w,
                               const int32_t *pool, int pool_blocks, int K, int32_t *idx, uint32_t *keys,
                               int *status, cudaStream_t st);

// Full layer with a pool of pool_keep >= K blocks: the top K rows from the
// pool's rows (exact, see pool_select.cu), given the scan's scores.
int pool_rows_supported(int pool_keep, int K);
cudaError_t launch_pool_rows(const CacheView &c, int P, const float *scores, int64_t ld, const int32_t *pool,
                             int pool_blocks, int K, int32_t *idx, cudaStream_t st);

// a3 over candidate pairs: the K best of n (score, id) pairs per row (id -1 =
// empty; ties to the earlier pair), ids written in pair order, -1 padded.
int select_pairs_supported(int n, int K);
cudaError_t launch_select_pairs(int rows, int n, const float *scores, const int32_t *ids, int K, int32_t *out,
                                cudaStream_t st);

// The context split of one sequence's rows over several devices (split.cu).
cudaError_t launch_pairs_from_idx(const CacheView &c, const float *scores, int64_t ld, const int32_t *idx, int n,
                                  int block, int32_t id_offset, float *pair_scores, int32_t *pair_ids, cudaStream_t st);
cudaError_t launch_ids_window(const int32_t *ids, int64_t count, int32_t lo, int32_t hi, int32_t *out, cudaStream_t st);
cudaError_t launch_lse_merge(int parts, int units, int H, int D, const float *outs, const float *lses, float *out,
                             float *lse, cudaStream_t st);

// a5/a6, and the local window of the joint softmax (rows [B][n][D] FP8 E4M3).
struct SwaView {
    const uint8_t *rows;
    const int32_t *lengths;  // [B] local rows per sequence, or null: n each
    int n, window;
};
size_t attend_workspace_bytes(const CacheView &c, int P, int H, int K, const SwaView *swa = nullptr);
cudaError_t launch_attend(const CacheView &c, int P, int H, const uint16_t *q, float scale, const int32_t *idx,
                          int K, float *out, float *lse, void *ws, size_t ws_bytes, int *status, cudaStream_t st,
                          const SwaView *swa = nullptr);

// Persistent records of cache rows (main entry codes, scales, indexer entry).
size_t record_bytes(const CacheView &c);
cudaError_t launch_spill(const CacheView &c, int row0, int n, uint8_t *out, cudaStream_t st);
cudaError_t launch_reload(const CacheView &c, const uint8_t *in, int n, int *status, cudaStream_t st);

// Host-side count of kernel launches issued by the library (csa_kernel_launches).
void count_launch(int n = 1);

// Streaming multiprocessors of the current device (queried once per device;
// 148, a B300's count, when no device can be queried).  Grid and split plans
// size themselves by it.
int sm_count();

// Launches `kernel` with programmatic stream serialization (it may begin while
// the previous kernel on the stream finishes; the kernel calls pdl_wait()
// before reading anything earlier work wrote) and, if cluster_x > 0, with
// thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          int cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) count_launch();
    return e;
}

// Driver entry point for tensor-map encoding (resolved once through the runtime).
CUresult encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                                 uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);
// Rows of 128 packed 4-bit values (64 bytes): a box of box_rows rows lands in
// shared memory as 128-byte rows, each 16-byte chunk holding 8 code bytes then
// 8 untouched bytes, with the 128-byte swizzle; the copy completes 64 bytes a
// row on its barrier.  base must be 32-byte aligned.
CUresult encode_tensor_map_2d_packed4(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows);

}  // namespace csa
