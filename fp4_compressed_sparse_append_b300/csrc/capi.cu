// The C ABI (include/csa.h): argument checks, workspace layout, and the
// per-layer composition of the kernels for the Full / Reindex / Reuse modes
// ("G2C Brief - DeepSeek V4.1-Flash", section "CSA2: most layers don't keep
// their own cache").  Every check here runs before any launch.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "csa_internal.h"

namespace {

// One status word per device (see csa_device_status).
__device__ int g_csa_status;

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

int *status_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_csa_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa_status check_cache(const csa_cache *c)
{
    if (!c || !c->codes || !c->scales || !c->ikeys || !c->lengths) return CSA_ERR_INVALID_ARG;
    if (c->batch < 1 || c->capacity < 1) return CSA_ERR_INVALID_ARG;
    // Row coordinates of the TMA tensor maps and the scan's row arithmetic are
    // 32-bit: batch x capacity rows must stay below 2^31 (far beyond any cache
    // that fits the device).
    if (static_cast<int64_t>(c->batch) * c->capacity >= (int64_t(1) << 31)) return CSA_ERR_UNSUPPORTED;
    if (!aligned16(c->codes) || !aligned16(c->scales) || !aligned16(c->ikeys) ||
        (reinterpret_cast<uintptr_t>(c->lengths) & 3u))
        return CSA_ERR_INVALID_ARG;
    if (c->d_latent <= 0 || c->d_latent % 16) return CSA_ERR_INVALID_ARG;
    if (c->d_index <= 0 || c->d_index % 16) return CSA_ERR_INVALID_ARG;
    if (c->d_latent % 128 || c->d_latent > 512) return CSA_ERR_UNSUPPORTED;
    if (c->d_index != 32 && c->d_index != 64 && c->d_index != 128) return CSA_ERR_UNSUPPORTED;
    if (c->ikey_format != CSA_IKEY_E4M3 && c->ikey_format != CSA_IKEY_MXFP4) return CSA_ERR_INVALID_ARG;
    if (c->ikey_format == CSA_IKEY_MXFP4) {
        // the packed key copy reads from a 32-byte-aligned base
        if (!c->iscales || !aligned16(c->iscales) || (reinterpret_cast<uintptr_t>(c->ikeys) & 31u))
            return CSA_ERR_INVALID_ARG;
        if (c->d_index != 128 || c->capacity % 4) return CSA_ERR_UNSUPPORTED;
    }
    return CSA_OK;
}

csa::CacheView view(const csa_cache *c)
{
    return csa::CacheView{c->batch,  c->capacity, c->d_latent, c->d_index,
                          c->codes,  c->scales,   c->ikeys,    c->lengths,
                          c->ikey_format == CSA_IKEY_MXFP4 ? 1 : 0, c->iscales};
}

csa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

csa_status check_index_args(const csa_cache *c, int P, int HI, const uint8_t *iq, const float *w,
                            const int32_t *pool, int pool_blocks, const void *scores, int64_t ld)
{
    if (P < 1 || HI < 1 || !iq || !w || !scores) return CSA_ERR_INVALID_ARG;
    if (!aligned16(iq) || !aligned16(w) || !aligned16(scores)) return CSA_ERR_INVALID_ARG;
    if (pool) {
        if (pool_blocks < 1 || !aligned16(pool)) return CSA_ERR_INVALID_ARG;
        if (ld < static_cast<int64_t>(pool_blocks) * CSA_POOL_BLOCK) return CSA_ERR_INVALID_ARG;
    } else if (ld < c->capacity) {
        return CSA_ERR_INVALID_ARG;
    }
    if (ld % 4) return CSA_ERR_INVALID_ARG;
    if (HI * P > 512 || HI > 256) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

}  // namespace

namespace csa {
std::atomic<uint64_t> &launch_counter();
}

extern "C" {

const char *csa_status_string(csa_status s)
{
    switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_DEVICE: return "device-side fault recorded in the status word";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

csa_status csa_quantize_append(const csa_cache *cache, const uint16_t *rows, const uint8_t *ikeys_new,
                               int32_t n_new, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (n_new < 0) return CSA_ERR_INVALID_ARG;
    if (n_new == 0) return CSA_OK;
    if (!rows || !aligned16(rows) || (ikeys_new && !aligned16(ikeys_new))) return CSA_ERR_INVALID_ARG;
    if (n_new > cache->capacity) return CSA_ERR_INVALID_ARG;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_quantize_append(view(cache), rows, ikeys_new, n_new, st, stream));
}

size_t csa_cache_record_bytes(const csa_cache *cache)
{
    if (check_cache(cache) != CSA_OK) return 0;
    return csa::record_bytes(view(cache));
}

csa_status csa_cache_spill(const csa_cache *cache, int32_t row0, int32_t n, uint8_t *records, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (row0 < 0 || n < 0 || static_cast<int64_t>(row0) + n > cache->capacity) return CSA_ERR_INVALID_ARG;
    if (n == 0) return CSA_OK;
    if (!records || (reinterpret_cast<uintptr_t>(records) & 3u)) return CSA_ERR_INVALID_ARG;
    return from_cuda(csa::launch_spill(view(cache), row0, n, records, stream));
}

csa_status csa_cache_reload(const csa_cache *cache, const uint8_t *records, int32_t n, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (n < 0 || n > cache->capacity) return CSA_ERR_INVALID_ARG;
    if (n == 0) return CSA_OK;
    if (!records || (reinterpret_cast<uintptr_t>(records) & 3u)) return CSA_ERR_INVALID_ARG;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_reload(view(cache), records, n, st, stream));
}

csa_status csa_quantize_append_project(const csa_cache *cache, const uint16_t *rows, const uint16_t *w_ik,
                                       int32_t n_new, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (n_new < 0 || !w_ik || !aligned16(w_ik)) return CSA_ERR_INVALID_ARG;
    if (cache->d_index != 32 && cache->d_index != 64 && cache->d_index != 128) return CSA_ERR_UNSUPPORTED;
    if (n_new == 0) return CSA_OK;
    if (!rows || !aligned16(rows)) return CSA_ERR_INVALID_ARG;
    if (n_new > cache->capacity) return CSA_ERR_INVALID_ARG;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_quantize_append(view(cache), rows, nullptr, n_new, st, stream, w_ik));
}

// Block maxima beside a full scan's scores: one fp32 per 8 rows of capacity.
static bool block_max_ok(const csa_cache *c, const float *block_max, int64_t ldb)
{
    const int64_t blocks = (static_cast<int64_t>(c->capacity) + CSA_POOL_BLOCK - 1) / CSA_POOL_BLOCK;
    return block_max && aligned16(block_max) && ldb >= blocks && ldb % 4 == 0;
}

csa_status csa_index_score(const csa_cache *cache, int32_t P, int32_t HI, const uint8_t *iq, const float *w,
                           const int32_t *pool, int32_t pool_blocks, float *scores, int64_t ld, float *block_max,
                           int64_t ldb, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    s = check_index_args(cache, P, HI, iq, w, pool, pool_blocks, scores, ld);
    if (s != CSA_OK) return s;
    if (block_max && (pool || !block_max_ok(cache, block_max, ldb))) return CSA_ERR_INVALID_ARG;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_index_score(view(cache), P, HI, iq, w, pool, pool ? pool_blocks : 0, scores, ld, st,
                                             stream, block_max, block_max ? ldb : 0));
}

static csa_status check_topk(const csa_cache *cache, int32_t P, int32_t pool_blocks, int has_pool, int32_t K,
                             int32_t pool_keep, int has_pool_out)
{
    if (P < 1 || K < 1 || K > 16384) return CSA_ERR_INVALID_ARG;
    if (has_pool && pool_blocks < 1) return CSA_ERR_INVALID_ARG;
    if (has_pool && has_pool_out) return CSA_ERR_INVALID_ARG;
    if (has_pool_out && (pool_keep < 1 || pool_keep > 16384)) return CSA_ERR_INVALID_ARG;
    const csa::CacheView v = view(cache);
    const int32_t *fake_pool = has_pool ? reinterpret_cast<const int32_t *>(16) : nullptr;
    if (!csa::select_supported(v, fake_pool, pool_blocks, 1, K)) return CSA_ERR_UNSUPPORTED;
    if (has_pool_out && !csa::select_supported(v, nullptr, 0, CSA_POOL_BLOCK, pool_keep)) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

static size_t topk_ws(const csa_cache *cache, int32_t P, int32_t pool_blocks, int has_pool, int32_t K,
                      int32_t pool_keep, int has_pool_out)
{
    const csa::CacheView v = view(cache);
    const int32_t *fake_pool = has_pool ? reinterpret_cast<const int32_t *>(16) : nullptr;
    size_t a = csa::select_workspace_bytes(v, P, fake_pool, pool_blocks, 1, K);
    if (has_pool_out) {
        const size_t b = csa::select_workspace_bytes(v, P, nullptr, 0, CSA_POOL_BLOCK, pool_keep);
        if (b > a) a = b;
    }
    return a;
}

csa_status csa_topk_workspace_size(const csa_cache *cache, int32_t P, int32_t pool_blocks, int32_t K,
                                   int32_t pool_keep, size_t *bytes)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!bytes) return CSA_ERR_INVALID_ARG;
    s = check_topk(cache, P, pool_blocks, pool_blocks > 0, K, pool_keep, pool_keep > 0);
    if (s != CSA_OK) return s;
    *bytes = topk_ws(cache, P, pool_blocks, pool_blocks > 0, K, pool_keep, pool_keep > 0);
    return CSA_OK;
}

csa_status csa_topk(const csa_cache *cache, int32_t P, const float *scores, int64_t ld, const int32_t *pool,
                    int32_t pool_blocks, int32_t K, int32_t *idx, int32_t pool_keep, int32_t *pool_out,
                    const float *block_max, int64_t ldb, void *workspace, size_t workspace_bytes,
                    csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!scores || !idx) return CSA_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(idx) || ld % 4) return CSA_ERR_INVALID_ARG;
    if (pool && !aligned16(pool)) return CSA_ERR_INVALID_ARG;
    if (pool_out && !aligned16(pool_out)) return CSA_ERR_INVALID_ARG;
    if (block_max && (!pool_out || !block_max_ok(cache, block_max, ldb))) return CSA_ERR_INVALID_ARG;
    s = check_topk(cache, P, pool_blocks, pool != nullptr, K, pool_keep, pool_out != nullptr);
    if (s != CSA_OK) return s;
    if (pool ? ld < static_cast<int64_t>(pool_blocks) * CSA_POOL_BLOCK : ld < cache->capacity)
        return CSA_ERR_INVALID_ARG;
    const size_t need = topk_ws(cache, P, pool_blocks, pool != nullptr, K, pool_keep, pool_out != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return CSA_ERR_WORKSPACE;
    const csa::CacheView v = view(cache);
    // the pool's blocks, from the block maxima when the scan wrote them
    const float *bsrc = block_max ? block_max : scores;
    const int64_t bld = block_max ? ldb : ld;
    if (pool_out && csa::pool_rows_supported(pool_keep, K)) {
        // the pool first; the top K rows then lie in the pool's blocks
        cudaError_t e = csa::launch_select(v, P, bsrc, bld, nullptr, 0, CSA_POOL_BLOCK, pool_keep, pool_out,
                                           workspace, workspace_bytes, stream, block_max != nullptr);
        if (e == cudaSuccess) e = csa::launch_pool_rows(v, P, scores, ld, pool_out, pool_keep, K, idx, stream);
        return from_cuda(e);
    }
    cudaError_t e =
        csa::launch_select(v, P, scores, ld, pool, pool ? pool_blocks : 0, 1, K, idx, workspace, workspace_bytes, stream);
    if (e == cudaSuccess && pool_out)
        e = csa::launch_select(v, P, bsrc, bld, nullptr, 0, CSA_POOL_BLOCK, pool_keep, pool_out, workspace,
                               workspace_bytes, stream, block_max != nullptr);
    return from_cuda(e);
}

csa_status csa_pool_topk(const csa_cache *cache, int32_t P, int32_t HI, const uint8_t *iq, const float *w,
                         const int32_t *pool, int32_t pool_blocks, int32_t K, int32_t *idx, void *workspace,
                         size_t workspace_bytes, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (P < 1 || HI < 1 || K < 1 || K > 16384 || !iq || !w || !pool || !idx || pool_blocks < 1) return CSA_ERR_INVALID_ARG;
    if (!aligned16(iq) || !aligned16(w) || !aligned16(pool) || !aligned16(idx)) return CSA_ERR_INVALID_ARG;
    const csa::CacheView v = view(cache);
    if (!csa::pool_select_supported(v, P, HI, pool_blocks, K)) return CSA_ERR_UNSUPPORTED;
    if (workspace) {
        if (!csa::pool_spread_supported(v, P, HI, pool_blocks, K)) return CSA_ERR_UNSUPPORTED;
        if (!aligned16(workspace) || workspace_bytes < csa::pool_spread_keys_bytes(v, P, pool_blocks))
            return CSA_ERR_WORKSPACE;
    }
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    if (!workspace) return from_cuda(csa::launch_pool_select(v, P, HI, iq, w, pool, pool_blocks, K, idx, st, stream));
    return from_cuda(csa::launch_pool_spread(v, P, HI, iq, w, pool, pool_blocks, K, idx,
                                             static_cast<uint32_t *>(workspace), st, stream));
}

csa_status csa_pool_topk_workspace_size(const csa_cache *cache, int32_t P, int32_t pool_blocks, size_t *bytes)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!bytes || P < 1 || pool_blocks < 1) return CSA_ERR_INVALID_ARG;
    *bytes = csa::pool_spread_keys_bytes(view(cache), P, pool_blocks);
    return CSA_OK;
}

csa_status csa_select_pairs(const csa_cache *cache, const float *scores, int64_t ld, const int32_t *idx, int32_t n,
                            int32_t block, int32_t id_offset, float *pair_scores, int32_t *pair_ids,
                            csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!scores || !idx || !pair_scores || !pair_ids || n < 1 || (block != 1 && block != CSA_POOL_BLOCK))
        return CSA_ERR_INVALID_ARG;
    if (ld < cache->capacity || ld % 4) return CSA_ERR_INVALID_ARG;
    return from_cuda(csa::launch_pairs_from_idx(view(cache), scores, ld, idx, n, block, id_offset, pair_scores, pair_ids,
                                                stream));
}

csa_status csa_topk_pairs(int32_t rows, int32_t n, const float *pair_scores, const int32_t *pair_ids, int32_t K,
                          int32_t *idx, csa_stream_t stream)
{
    if (rows < 1 || n < 1 || K < 1 || K > 16384 || !pair_scores || !pair_ids || !idx) return CSA_ERR_INVALID_ARG;
    if (!aligned16(pair_scores) || !aligned16(pair_ids) || !aligned16(idx)) return CSA_ERR_INVALID_ARG;
    if (!csa::select_pairs_supported(n, K)) return CSA_ERR_UNSUPPORTED;
    return from_cuda(csa::launch_select_pairs(rows, n, pair_scores, pair_ids, K, idx, stream));
}

csa_status csa_ids_window(const int32_t *ids, int64_t count, int32_t lo, int32_t hi, int32_t *out, csa_stream_t stream)
{
    if (count < 0 || !ids || !out || hi < lo) return CSA_ERR_INVALID_ARG;
    return from_cuda(csa::launch_ids_window(ids, count, lo, hi, out, stream));
}

csa_status csa_lse_merge(int32_t parts, int32_t units, int32_t H, int32_t D, const float *outs, const float *lses,
                         float *out, float *lse, csa_stream_t stream)
{
    if (parts < 1 || units < 1 || H < 1 || D < 4 || D % 4 || !outs || !lses || !out) return CSA_ERR_INVALID_ARG;
    if (!aligned16(outs) || !aligned16(out) || (lse && !aligned16(lse))) return CSA_ERR_INVALID_ARG;
    if (H > 65535 || units > 65535) return CSA_ERR_UNSUPPORTED;
    return from_cuda(csa::launch_lse_merge(parts, units, H, D, outs, lses, out, lse, stream));
}

csa_status csa_attend_workspace_size(const csa_cache *cache, int32_t P, int32_t H, int32_t K, size_t *bytes)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!bytes || P < 1 || H < 1 || K < 1) return CSA_ERR_INVALID_ARG;
    if (H > 64) return CSA_ERR_UNSUPPORTED;
    *bytes = csa::attend_workspace_bytes(view(cache), P, H, K);
    return CSA_OK;
}

csa_status csa_sparse_attend(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q, float scale,
                             const int32_t *idx, int32_t K, float *out, float *lse, void *workspace,
                             size_t workspace_bytes, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (P < 1 || H < 1 || K < 1 || !q || !idx || !out) return CSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse))) return CSA_ERR_INVALID_ARG;
    if (H > 64) return CSA_ERR_UNSUPPORTED;
    const csa::CacheView v = view(cache);
    const size_t need = csa::attend_workspace_bytes(v, P, H, K);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return CSA_ERR_WORKSPACE;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_attend(v, P, H, q, scale, idx, K, out, lse, workspace, workspace_bytes, st, stream));
}

// The local window descriptor: rows 16-byte aligned, n >= P, 1 <= window <= 1024.
static csa_status check_swa(const csa_swa *swa, int32_t P)
{
    if (!swa) return CSA_OK;
    if (!swa->rows || !aligned16(swa->rows) || swa->n < P || swa->window < 1 || swa->window > 1024)
        return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

static csa::SwaView swa_view(const csa_swa *swa)
{
    return csa::SwaView{swa->rows, swa->lengths, swa->n, swa->window};
}

csa_status csa_attend_swa_workspace_size(const csa_cache *cache, int32_t P, int32_t H, int32_t K, const csa_swa *swa,
                                         size_t *bytes)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!bytes || P < 1 || H < 1 || K < 1) return CSA_ERR_INVALID_ARG;
    if (H > 64) return CSA_ERR_UNSUPPORTED;
    if ((s = check_swa(swa, P)) != CSA_OK) return s;
    const csa::SwaView sv = swa ? swa_view(swa) : csa::SwaView{};
    *bytes = csa::attend_workspace_bytes(view(cache), P, H, K, swa ? &sv : nullptr);
    return CSA_OK;
}

csa_status csa_sparse_attend_swa(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q, float scale,
                                 const int32_t *idx, int32_t K, const csa_swa *swa, float *out, float *lse,
                                 void *workspace, size_t workspace_bytes, csa_stream_t stream)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (P < 1 || H < 1 || K < 1 || !q || !idx || !out) return CSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse))) return CSA_ERR_INVALID_ARG;
    if (H > 64) return CSA_ERR_UNSUPPORTED;
    if ((s = check_swa(swa, P)) != CSA_OK) return s;
    const csa::CacheView v = view(cache);
    const csa::SwaView sv = swa ? swa_view(swa) : csa::SwaView{};
    const csa::SwaView *svp = swa ? &sv : nullptr;
    const size_t need = csa::attend_workspace_bytes(v, P, H, K, svp);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return CSA_ERR_WORKSPACE;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    return from_cuda(
        csa::launch_attend(v, P, H, q, scale, idx, K, out, lse, workspace, workspace_bytes, st, stream, svp));
}

static size_t layer_scores_ld(const csa_cache *cache, const csa_layer_args *a)
{
    if (a->mode == CSA_REINDEX && a->pool_in) return round_up(static_cast<size_t>(a->pool_blocks) * CSA_POOL_BLOCK, 4);
    return round_up(static_cast<size_t>(cache->capacity), 4);
}

// A Full layer that builds the pool: the scan also writes each 8-row block's
// best visible score, [B*P][ld] with ld = ceil(capacity / 8) rounded up to 4.
static size_t layer_bmax_ld(const csa_cache *cache, const csa_layer_args *a)
{
    if (a->mode != CSA_FULL || !a->pool_out) return 0;
    return round_up((static_cast<size_t>(cache->capacity) + CSA_POOL_BLOCK - 1) / CSA_POOL_BLOCK, 4);
}

static csa_status check_layer(const csa_cache *cache, const csa_layer_args *a)
{
    csa_status s = check_cache(cache);
    if (s != CSA_OK) return s;
    if (!a) return CSA_ERR_INVALID_ARG;
    if (a->mode != CSA_FULL && a->mode != CSA_REINDEX && a->mode != CSA_REUSE) return CSA_ERR_INVALID_ARG;
    if (a->P < 1 || a->H < 1 || a->K < 1 || a->K > 16384 || !a->q || !a->idx || !a->out) return CSA_ERR_INVALID_ARG;
    if (a->H > 64) return CSA_ERR_UNSUPPORTED;
    if (a->mode != CSA_REUSE) {
        if (!a->iq || !a->w || a->HI < 1) return CSA_ERR_INVALID_ARG;
        if (a->HI * a->P > 512 || a->HI > 256) return CSA_ERR_UNSUPPORTED;
    }
    if (a->n_new < 0 || (a->n_new > 0 && (a->mode != CSA_FULL || !a->rows_new))) return CSA_ERR_INVALID_ARG;
    if (a->w_ik && (a->ikeys_new || !aligned16(a->w_ik))) return CSA_ERR_INVALID_ARG;
    if (a->w_ik && a->n_new > 0 && cache->d_index != 32 && cache->d_index != 64 && cache->d_index != 128)
        return CSA_ERR_UNSUPPORTED;
    if ((a->pool_in || a->pool_out) && (a->pool_blocks < 1 || a->pool_blocks > 16384)) return CSA_ERR_INVALID_ARG;
    if (a->pool_in && a->mode != CSA_REINDEX) return CSA_ERR_INVALID_ARG;
    if (a->pool_out && a->mode != CSA_FULL) return CSA_ERR_INVALID_ARG;
    if ((s = check_swa(a->swa, a->P)) != CSA_OK) return s;
    if (a->mode != CSA_REUSE) {
        const int has_pool = a->mode == CSA_REINDEX && a->pool_in != nullptr;
        const int has_pool_out = a->mode == CSA_FULL && a->pool_out != nullptr;
        s = check_topk(cache, a->P, a->pool_blocks, has_pool, a->K, a->pool_blocks, has_pool_out);
        if (s != CSA_OK) return s;
    }
    return CSA_OK;
}

static size_t layer_select_ws(const csa_cache *cache, const csa_layer_args *a)
{
    if (a->mode == CSA_REUSE) return 0;
    const int has_pool = a->mode == CSA_REINDEX && a->pool_in != nullptr;
    const int has_pool_out = a->mode == CSA_FULL && a->pool_out != nullptr;
    return topk_ws(cache, a->P, a->pool_blocks, has_pool, a->K, a->pool_blocks, has_pool_out);
}

csa_status csa_layer_workspace_size(const csa_cache *cache, const csa_layer_args *a, size_t *bytes)
{
    csa_status s = check_layer(cache, a);
    if (s != CSA_OK) return s;
    if (!bytes) return CSA_ERR_INVALID_ARG;
    const csa::CacheView v = view(cache);
    size_t total = 0;
    if (a->mode != CSA_REUSE) {
        total += round_up(static_cast<size_t>(cache->batch) * a->P * layer_scores_ld(cache, a) * sizeof(float), 256);
        total += round_up(layer_select_ws(cache, a), 256);
        total += round_up(static_cast<size_t>(cache->batch) * a->P * layer_bmax_ld(cache, a) * sizeof(float), 256);
    }
    const csa::SwaView sv = a->swa ? swa_view(a->swa) : csa::SwaView{};
    total += round_up(csa::attend_workspace_bytes(v, a->P, a->H, a->K, a->swa ? &sv : nullptr), 256);
    *bytes = total;
    return CSA_OK;
}

csa_status csa_layer_step(const csa_cache *cache, const csa_layer_args *a, csa_stream_t stream)
{
    csa_status s = check_layer(cache, a);
    if (s != CSA_OK) return s;
    size_t need = 0;
    csa_layer_workspace_size(cache, a, &need);
    if (need > 0 && (!a->workspace || a->workspace_bytes < need || !aligned16(a->workspace))) return CSA_ERR_WORKSPACE;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    const csa::CacheView v = view(cache);
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);
    cudaError_t e = cudaSuccess;
    if (a->mode != CSA_REUSE) {
        const int64_t ld = static_cast<int64_t>(layer_scores_ld(cache, a));
        float *scores = reinterpret_cast<float *>(ws);
        ws += round_up(static_cast<size_t>(cache->batch) * a->P * ld * sizeof(float), 256);
        void *sel_ws = ws;
        const size_t sel_bytes = layer_select_ws(cache, a);
        ws += round_up(sel_bytes, 256);
        const int64_t ldb = static_cast<int64_t>(layer_bmax_ld(cache, a));
        float *bmax = ldb ? reinterpret_cast<float *>(ws) : nullptr;
        ws += round_up(static_cast<size_t>(cache->batch) * a->P * ldb * sizeof(float), 256);
        if (a->n_new > 0) {
            e = csa::launch_quantize_append(v, a->rows_new, a->ikeys_new, a->n_new, st, stream, a->w_ik);
            if (e != cudaSuccess) return CSA_ERR_CUDA;
        }
        const int32_t *pool = a->mode == CSA_REINDEX ? a->pool_in : nullptr;
        const int pool_blocks = pool ? a->pool_blocks : 0;
        const bool make_pool = a->mode == CSA_FULL && a->pool_out;
        if (pool && csa::pool_spread_supported(v, a->P, a->HI, pool_blocks, a->K)) {
            // a Reindex layer over the pool: scores and selection in one kernel,
            // the keys through the scores' workspace
            e = csa::launch_pool_spread(v, a->P, a->HI, a->iq, a->w, pool, pool_blocks, a->K, a->idx,
                                        reinterpret_cast<uint32_t *>(scores), st, stream);
        } else if (pool && csa::pool_select_supported(v, a->P, a->HI, pool_blocks, a->K)) {
            e = csa::launch_pool_select(v, a->P, a->HI, a->iq, a->w, pool, pool_blocks, a->K, a->idx, st, stream);
        } else {
            e = csa::launch_index_score(v, a->P, a->HI, a->iq, a->w, pool, pool_blocks, scores, ld, st, stream, bmax,
                                        ldb);
            if (make_pool && csa::pool_rows_supported(a->pool_blocks, a->K)) {
                // the pool first (from the blocks' best scores the scan wrote); the
                // top K rows then lie in the pool's blocks
                if (e == cudaSuccess)
                    e = csa::launch_select(v, a->P, bmax, ldb, nullptr, 0, CSA_POOL_BLOCK, a->pool_blocks,
                                           a->pool_out, sel_ws, sel_bytes, stream, true);
                if (e == cudaSuccess)
                    e = csa::launch_pool_rows(v, a->P, scores, ld, a->pool_out, a->pool_blocks, a->K, a->idx, stream);
            } else {
                if (e == cudaSuccess)
                    e = csa::launch_select(v, a->P, scores, ld, pool, pool_blocks, 1, a->K, a->idx, sel_ws, sel_bytes,
                                           stream);
                if (e == cudaSuccess && make_pool)
                    e = csa::launch_select(v, a->P, bmax, ldb, nullptr, 0, CSA_POOL_BLOCK, a->pool_blocks,
                                           a->pool_out, sel_ws, sel_bytes, stream, true);
            }
        }
        if (e != cudaSuccess) return CSA_ERR_CUDA;
    }
    const csa::SwaView sv = a->swa ? swa_view(a->swa) : csa::SwaView{};
    const csa::SwaView *svp = a->swa ? &sv : nullptr;
    const size_t att = csa::attend_workspace_bytes(v, a->P, a->H, a->K, svp);
    e = csa::launch_attend(v, a->P, a->H, a->q, a->scale, a->idx, a->K, a->out, a->lse, ws, att, st, stream, svp);
    return from_cuda(e);
}

uint64_t csa_kernel_launches(void) { return csa::launch_counter().load(); }

csa_status csa_device_status(int32_t *bits, int32_t clear, csa_stream_t stream)
{
    if (!bits) return CSA_ERR_INVALID_ARG;
    int *st = status_word();
    if (!st) return CSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, st, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return CSA_ERR_CUDA;
    if (clear && cudaMemsetAsync(st, 0, sizeof(int), stream) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
    *bits = v;
    return v ? CSA_ERR_DEVICE : CSA_OK;
}

}  // extern "C"

namespace csa {

std::atomic<uint64_t> &launch_counter()
{
    static std::atomic<uint64_t> n{0};
    return n;
}

void count_launch(int n) { launch_counter() += static_cast<uint64_t>(n); }

int sm_count()
{
    static int counts[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();  // no device here: clear the error and plan for a B300
        return 148;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        counts[dev] = n;
    }
    return counts[dev];
}

namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

}  // namespace

CUresult encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                                 uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    const EncodeFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {inner_bytes, rows};
    const cuuint64_t strides[1] = {inner_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tensor_map_2d_packed4(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows)
{
    const EncodeFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {128, rows};  // in 4-bit values
    const cuuint64_t strides[1] = {64};      // bytes per row
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace csa
