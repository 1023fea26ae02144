/*
 * csa.h - C ABI of the CSA2 sparse-attention decode step over an FP4 global
 * KV cache, for NVIDIA B300 (sm_103a).
 *
 * The step, as the pages on DeepSeek-V4.1-Flash describe it:
 *  - "G2C Brief - DeepSeek V4.1-Flash: a model designed around its KV cache",
 *    section "The global branch: compress, index, select": a learned indexer
 *    scores every cached entry for the query with low-precision queries and
 *    keys, the query keeps the best entries (top-k) and attends to only those.
 *    One shared latent per cached position serves every query head.
 *  - same page, section "FP4 cache entries, and why they're safe": main cache
 *    entries are E2M1 4-bit floats with one E4M3 scale per 16 channels
 *    (288 bytes for a 512-dim entry).
 *  - same page, section "CSA2: most layers don't keep their own cache": each
 *    layer is Full (own KV, own indexer keys, own selection), Reindex (borrows
 *    the KV and indexer keys, re-scores with its own indexer query) or Reuse
 *    (borrows the KV and the last selection); every layer has its own query.
 *  - same page, section "The hierarchical indexer": the first Full layer also
 *    groups positions into blocks of 8, scores each block by its best member
 *    and keeps the top 2,048 blocks; later Reindex layers search only that pool.
 * The indexer score is sum_h w_h * ReLU(q_h . k) with FP8 E4M3 indexer queries
 * and keys (the pages give no formula; this is the workload statement's).
 *
 * Conventions for every call:
 *  - Pointers named in the argument lists are DEVICE pointers, owned by the
 *    caller; the library never allocates, frees or retains them.  Every
 *    device pointer must be 16-byte aligned (cache lengths: 4-byte).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  No call synchronises the host, except csa_device_status.
 *  - Kernels are launched with programmatic dependent launch: each may start
 *    while the kernel before it on the stream finishes, and waits for it
 *    before reading anything that kernel could have written.  One exception:
 *    the attention kernels fetch the main query q before that wait, so q
 *    must not be written by a kernel that lets its dependents start early
 *    (griddepcontrol.launch_dependents) and runs immediately before the call.
 *    Kernels that do not use that instruction, copies and the library's own
 *    kernels are all safe producers of q.
 *  - Argument errors return CSA_ERR_INVALID_ARG / CSA_ERR_UNSUPPORTED before
 *    anything is launched.  Launch failures return CSA_ERR_CUDA.
 *  - Faults found on the device (a row index outside [0, length), an append
 *    past capacity, a pipeline wait that ran out) do not trap: the kernel
 *    skips the access, ORs a bit into a per-device status word and carries on.
 *    csa_device_status reads (and optionally clears) that word.
 *  - Sequence b holds valid rows [0, lengths[b]).  Kernels read lengths[b] as
 *    min(lengths[b], capacity), so no row at or past the capacity is read or
 *    written whatever the array holds.  With P query positions per
 *    sequence, the last P rows are the step's own positions and position p
 *    (0 <= p < P) sees rows [0, lengths[b] - P + 1 + p).
 *  - Index lists (top-K selections, pools) are written in ascending order
 *    followed by -1 padding; an index of -1 is always skipped on read.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *csa_stream_t;

typedef enum csa_status {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, bad mode */
    CSA_ERR_UNSUPPORTED = 2,  /* valid but outside the shapes this library handles */
    CSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    CSA_ERR_DEVICE = 4,       /* csa_device_status: a device-side fault bit is set */
    CSA_ERR_WORKSPACE = 5     /* workspace missing or smaller than the size query said */
} csa_status;

/* Bits of the device status word. */
#define CSA_DEV_BAD_INDEX 0x1   /* a selected row id was >= min(lengths[b], capacity) (row skipped) */
#define CSA_DEV_CAPACITY  0x2   /* an append would pass capacity (sequence left unchanged) */
#define CSA_DEV_TIMEOUT   0x4   /* a pipeline wait ran past its limit (kernel returned early) */

typedef enum csa_mode { CSA_FULL = 0, CSA_REINDEX = 1, CSA_REUSE = 2 } csa_mode;

#define CSA_POOL_BLOCK 8        /* rows per hierarchical-pool block */

/*
 * The global cache shared by the layers of one chain (one "Full" owner).
 *   codes   : [batch][capacity][d_latent/2]  two E2M1 codes per byte, the even
 *             channel in the low nibble, sign in bit 3 of each nibble
 *   scales  : [batch][capacity][d_latent/16] one E4M3 scale per 16 channels
 *   ikeys   : CSA_IKEY_E4M3:  [batch][capacity][d_index]    FP8 E4M3 indexer key per row
 *             CSA_IKEY_MXFP4: [batch][capacity][d_index/2]  E2M1 codes of the key
 *                             (even channel in the low nibble)
 *   iscales : CSA_IKEY_MXFP4: [batch][capacity][d_index/32] UE8M0 block scales
 *             (2^(byte - 127) per 32 channels); unused (may be NULL) for E4M3
 *   lengths : [batch] int32                  valid rows per sequence
 * d_latent is 128, 256, 384 or 512; d_index is 32, 64 or 128; capacity >= 1;
 * batch x capacity < 2^31 (row ids are 32-bit), else CSA_ERR_UNSUPPORTED.
 * MXFP4 keys ("G2C Brief", section "FP4 cache entries, and why they're safe":
 * 128 values x 4 bits + one 8-bit scale per 32 values = 68 B, the OCP MXFP4
 * format the pages assume) need d_index = 128 and capacity a multiple of 4.
 * Their rule, where the library writes them (csa_quantize_append_project): per
 * block of 32 channels, X = floor(log2 amax) - 2 clamped to [-8, 6] (-8 for an
 * all-zero block), scale byte X + 127, codes the E2M1 values nearest to
 * x / 2^X (ties to even, 6 beyond) with the sign of x.  A key given by the
 * caller may carry any scale byte but 255 (NaN in the OCP format, which gives
 * unspecified scores): the scan applies 2^(byte - 127) exactly in the tensor
 * core's block-scaled product, accumulating in fp32.  The ikeys base must be
 * 32-byte aligned (the scan's 4-bit copy requires it).
 */
#define CSA_IKEY_E4M3 0
#define CSA_IKEY_MXFP4 1

typedef struct csa_cache {
    int32_t batch;
    int32_t capacity;
    int32_t d_latent;
    int32_t d_index;
    uint8_t *codes;
    uint8_t *scales;
    uint8_t *ikeys;
    int32_t *lengths;
    int32_t ikey_format;          /* CSA_IKEY_E4M3 (0) or CSA_IKEY_MXFP4 */
    uint8_t *iscales;             /* CSA_IKEY_MXFP4 only */
} csa_cache;

/*
 * a1: quantise new latent rows to FP4 and append them.
 * ("G2C Brief", section "FP4 cache entries, and why they're safe".)
 *   rows      : [batch][n_new][d_latent] bf16 bits
 *   ikeys_new : [batch][n_new][d_index] E4M3 bytes (MXFP4 cache: [batch][n_new]
 *               [d_index/2 + d_index/32], each row's codes then its scales),
 *               copied as given; or NULL to leave the keys as they are
 * Per 16-channel group: scale = E4M3 round-to-nearest-even(amax / 6), saturating
 * at 448; each channel's code is the E2M1 value nearest to x / scale (ties to
 * the even code, beyond 6 clamped to 6) with the sign of x kept; a group whose
 * scale rounds to 0 stores zero codes.  Rows go to positions lengths[b] ..
 * lengths[b] + n_new - 1, then lengths[b] += n_new.  A sequence that would
 * pass capacity is left unchanged and sets CSA_DEV_CAPACITY.
 * Inputs must be finite (non-finite inputs give unspecified codes).
 */
CSA_API csa_status csa_quantize_append(const csa_cache *cache, const uint16_t *rows,
                               const uint8_t *ikeys_new, int32_t n_new, csa_stream_t stream);

/*
 * a1 with indexer keys projected from the stored rows.  ("G2C Brief", section
 * "The global branch: compress, index, select": the indexer's keys are a
 * projection of the main cache entries rather than a separately computed
 * cache.)  Appends rows as csa_quantize_append does, then writes each appended
 * row's indexer key
 *     ik[j] = E4M3( sum_c v[c] * w_ik[c][j] ),  j < d_index,
 * from its stored entry v = E2M1(code) * E4M3(scale) (exact), summed in fp32
 * and rounded once: nearest, ties to even, saturating at 448 (a zero sum is
 * +0); for an MXFP4 cache each block of 32 sums is quantised by the MXFP4
 * rule above instead.  The sum's order differs from an exact one, so a key can
 * differ by one code (or a block by its exponent) from the exactly rounded
 * product where that product lies within fp32 rounding of a rounding boundary.
 *   w_ik : [d_latent][d_index] bf16 bits, device, 16-byte aligned (read only)
 * d_index must be 32, 64 or 128 (else CSA_ERR_UNSUPPORTED).
 */
CSA_API csa_status csa_quantize_append_project(const csa_cache *cache, const uint16_t *rows, const uint16_t *w_ik,
                                               int32_t n_new, csa_stream_t stream);

/*
 * Persistent records of cache entries, to spill a cache out of device memory
 * (to host memory or storage) and reload it.  ("G2C Brief", section "FP4
 * cache entries, and why they're safe": an entry is its 288-byte main entry
 * and its 68-byte MXFP4 indexer entry, 356 B; a cache layer with compression
 * m keeps one entry per m tokens, which makes the 890 bytes per token of three
 * m = 2 layers and one m = 1 layer.)
 * A record is, in this order: the row's d_latent/2 code bytes, its
 * d_latent/16 scale bytes, then its indexer entry (E4M3 cache: d_index bytes;
 * MXFP4 cache: d_index/2 code bytes, then d_index/32 scale bytes).
 * csa_cache_record_bytes returns that size (0 for an invalid cache).
 */
CSA_API size_t csa_cache_record_bytes(const csa_cache *cache);

/*
 * Spill (persistent records, "G2C Brief", section "FP4 cache entries, and why
 * they're safe", as above): the records of rows row0 .. row0 + n - 1 of every
 * sequence into
 *   records : [batch][n][record bytes], device memory or pinned host memory
 *             the device can address (4-byte aligned; written only)
 * A row at or past the sequence's length (read on the device) gives a record
 * of zeros.  The cache is not changed.  row0 + n must not pass capacity
 * (else CSA_ERR_INVALID_ARG).
 */
CSA_API csa_status csa_cache_spill(const csa_cache *cache, int32_t row0, int32_t n, uint8_t *records,
                                   csa_stream_t stream);

/*
 * Reload (persistent records, "G2C Brief", section "FP4 cache entries, and why
 * they're safe", as above): appends n records per sequence,
 *   records : [batch][n][record bytes] as csa_cache_spill writes them, device
 *             memory or device-addressable pinned host memory (4-byte aligned)
 * at rows lengths[b] .. lengths[b] + n - 1, then lengths[b] += n (the append
 * rule of csa_quantize_append: a sequence that would pass capacity is left
 * unchanged and sets CSA_DEV_CAPACITY).  Spilling rows 0 .. L - 1 and
 * reloading them into an empty cache of the same shape and key format gives
 * back the same rows.
 */
CSA_API csa_status csa_cache_reload(const csa_cache *cache, const uint8_t *records, int32_t n, csa_stream_t stream);

/*
 * a2/a4: indexer scores for B*P queries.
 * ("G2C Brief", sections "The global branch" and "The hierarchical indexer".)
 *   iq     : [batch][P][HI][d_index] E4M3 indexer queries
 *   w      : [batch][P][HI] fp32 per-head weights
 *   pool   : NULL   -> score rows t < L_p = lengths[b] - P + 1 + p;
 *                      scores[(b*P+p)*ld + t]
 *            [batch][P][pool_blocks] block ids (ascending, -1 padded)
 *                   -> score candidate c = 8*j + m, row pool[j]*8 + m;
 *                      scores[(b*P+p)*ld + c]
 *   scores : fp32, row stride ld (>= capacity, or >= 8*pool_blocks with a pool)
 *   block_max : NULL, or (only with pool == NULL) fp32 with row stride ldb
 *            (>= ceil(capacity / 8), a multiple of 4; 16-byte aligned):
 *            block_max[(b*P+p)*ldb + j] = the largest score of rows
 *            8j .. 8j+7 below L_p, for j < ceil(L_p / 8) ("The hierarchical
 *            indexer": a block of 8 is ranked by its best member); csa_topk
 *            builds its pool from these instead of the row scores
 * score = sum_h w[h] * ReLU(sum_d iq[h][d] * ik[row][d]), fp32.  Entries for
 * rows past L_p or empty pool slots, and block maxima past ceil(L_p / 8), are
 * left unspecified.
 * Supported: HI*P <= 512, HI % 16 == 0 (or HI*P % 16 == 0).
 */
CSA_API csa_status csa_index_score(const csa_cache *cache, int32_t P, int32_t HI,
                           const uint8_t *iq, const float *w,
                           const int32_t *pool, int32_t pool_blocks,
                           float *scores, int64_t ld, float *block_max, int64_t ldb,
                           csa_stream_t stream);

/*
 * a3: top-K selection (and the hierarchical block pool) from scores.
 * ("Pushing the Limits" talk write-up, "The Paper": keep the best indices;
 *  "G2C Brief", "The hierarchical indexer": blocks of 8 scored by their best
 *  member, keep the top blocks.)
 *   scores, ld, pool, pool_blocks : as produced by csa_index_score
 *   idx      : [batch][P][K] int32 row ids of the K largest scores among the
 *              candidates (ties: lower row id), ascending, then -1 padding
 *   pool_out : NULL, or (only with pool == NULL) [batch][P][pool_keep] ids of
 *              the pool_keep blocks of 8 rows (block j = rows 8j..8j+7 < L_p)
 *              with the largest best-member score (ties: lower id), ascending,
 *              then -1 padding
 *   block_max, ldb : NULL, or (only with pool_out) the block maxima that
 *              csa_index_score wrote beside these scores; the pool is then
 *              selected from them (ceil(L_p / 8) reads instead of L_p), with
 *              the same result
 *   workspace: csa_topk_workspace_size bytes (zero for rows of at most 196,608
 *              candidates; longer rows are selected in two stages through it)
 * 1 <= K <= 16384; pool_keep <= 16384.
 */
CSA_API csa_status csa_topk(const csa_cache *cache, int32_t P, const float *scores, int64_t ld,
                    const int32_t *pool, int32_t pool_blocks, int32_t K, int32_t *idx,
                    int32_t pool_keep, int32_t *pool_out, const float *block_max, int64_t ldb,
                    void *workspace, size_t workspace_bytes, csa_stream_t stream);

/*
 * a4 over the hierarchical pool in one call: csa_index_score of the pool's
 * rows followed by csa_topk of those scores, with the scores kept on chip.
 * ("G2C Brief", section "The hierarchical indexer": later Reindex layers
 * score only the pool's rows with their own indexer query and keep the best;
 * section "CSA2: most layers don't keep their own cache": Reindex borrows the
 * keys and selects afresh.)
 *   iq, w          : as csa_index_score
 *   pool           : [batch][P][pool_blocks] block ids, ascending, -1 padded
 *   idx            : [batch][P][K] ids of the K best-scoring pool rows among
 *                    rows < L_p (ties: the earlier pool slot), ascending, then
 *                    -1 padding
 *   workspace      : NULL, or csa_pool_topk_workspace_size bytes of device
 *                    scratch (16-byte aligned)
 * The same result as csa_index_score + csa_topk (up to the fp32 summation
 * order of the scores), in one launch.  Without a workspace, one cluster of up
 * to 16 CTAs scores the pool and selects on chip.  With one, one CTA per 128
 * pool rows scores its rows into the workspace and the last CTA of each query
 * to finish selects (faster: the key copies spread over more SMs); its
 * arrival counters come from a library-owned array of 65,536, taken in turn,
 * so calls whose counters coincide (65,536 query units of such calls apart in
 * issue order) must not run at the same time.  csa_layer_step takes the
 * workspace form for Reindex layers over a pool.
 * Supported: E4M3 keys, HI <= 64, pool_blocks <= 2048, K <= 16384; otherwise
 * CSA_ERR_UNSUPPORTED (use the two calls instead).
 */
CSA_API csa_status csa_pool_topk(const csa_cache *cache, int32_t P, int32_t HI, const uint8_t *iq, const float *w,
                                 const int32_t *pool, int32_t pool_blocks, int32_t K, int32_t *idx, void *workspace,
                                 size_t workspace_bytes, csa_stream_t stream);

/* Workspace query of csa_pool_topk's spread form.  No counterpart on the
 * pages: B * P * pool_blocks * 8 four-byte keys. */
CSA_API csa_status csa_pool_topk_workspace_size(const csa_cache *cache, int32_t P, int32_t pool_blocks,
                                                size_t *bytes);

/* Workspace query of csa_topk.  No counterpart on the pages: the library
 * allocates nothing, so the caller supplies the scratch of the two-stage
 * select of long rows.  pool_blocks > 0: the scores are over a pool of that
 * many blocks; pool_keep > 0: a pool of that many blocks is also built. */
CSA_API csa_status csa_topk_workspace_size(const csa_cache *cache, int32_t P, int32_t pool_blocks, int32_t K,
                                           int32_t pool_keep, size_t *bytes);

/*
 * a5/a6: sparse attention of each query over its selected FP4 rows.
 * ("G2C Brief", "The global branch": the query attends to only the selected
 *  entries; "Pushing the Limits", "The Paper": one W_KV, so K and V are equal.)
 *   q     : [batch][P][H][d_latent] bf16 bits
 *   idx   : [batch][P][K] row ids (-1 = skip; an id >= min(lengths[b], capacity)
 *           sets CSA_DEV_BAD_INDEX and is skipped)
 *   out   : [batch][P][H][d_latent] fp32 = sum_j softmax_j(scale * q.v_j) v_j
 *   lse   : [batch][P][H] fp32 log-sum-exp of the logits, or NULL
 *   workspace : device scratch of csa_attend_workspace_size bytes
 * A query with no valid row gets out = 0, lse = -inf.  1 <= H <= 64.
 */
CSA_API csa_status csa_sparse_attend(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q,
                             float scale, const int32_t *idx, int32_t K, float *out, float *lse,
                             void *workspace, size_t workspace_bytes, csa_stream_t stream);

/* Workspace query of csa_sparse_attend.  No counterpart on the pages: the bytes
 * of split partials the call keeps in the caller's workspace (0 when every
 * query's splits merge on chip). */
CSA_API csa_status csa_attend_workspace_size(const csa_cache *cache, int32_t P, int32_t H, int32_t K,
                                     size_t *bytes);

/*
 * The local branch and the joint softmax.  ("G2C Brief", "Two attention
 * paths in every layer": besides the selected global entries every query sees
 * a sliding window of the 128 most recent tokens; "FP4 cache entries, and why
 * they're safe": that local cache stays in FP8; "Pushing the Limits", "The
 * Paper": the selected entries are joined to the window's KV for one attention.)
 * Plain reading: one softmax over the union of the selected FP4 rows and the
 * window rows, with K == V for both.
 *   rows    : [batch][n][d_latent] FP8 E4M3 bytes (device, 16-byte aligned),
 *             the sequence's local rows in token order; position p of P is
 *             the row L - P + p of a sequence with L local rows.
 *   lengths : [batch] int32 device array of L per sequence, or NULL (L = n for
 *             every sequence).  L outside [P, n] sets CSA_DEV_BAD_INDEX in the
 *             status word and that sequence's windows are left empty.
 *   n       : row capacity per sequence (the stride of rows), n >= P.
 *   window  : rows attended per query, 1..1024: local rows
 *             [max(0, own - window + 1), own] of a query whose own row is own.
 * The caller owns the window array and fills it (e.g. the last `window`
 * tokens' latent rows converted to E4M3); the library only reads it.
 */
typedef struct csa_swa {
    const uint8_t *rows;
    const int32_t *lengths;
    int32_t n;
    int32_t window;
} csa_swa;

/*
 * csa_sparse_attend with the local window ("G2C Brief", "Two attention paths
 * in every layer"; "Pushing the Limits", "The Paper"; the reading above): out
 * and lse are those of the joint
 * softmax over the selected rows of idx and the window rows of swa (NULL swa:
 * exactly csa_sparse_attend).  workspace: csa_attend_swa_workspace_size bytes.
 */
CSA_API csa_status csa_sparse_attend_swa(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q,
                                         float scale, const int32_t *idx, int32_t K, const csa_swa *swa, float *out,
                                         float *lse, void *workspace, size_t workspace_bytes, csa_stream_t stream);

/* Workspace query of csa_sparse_attend_swa (no counterpart on the pages; the
 * window adds one split to each query). */
CSA_API csa_status csa_attend_swa_workspace_size(const csa_cache *cache, int32_t P, int32_t H, int32_t K,
                                                 const csa_swa *swa, size_t *bytes);

/*
 * csa_sparse_attend without a workspace argument and without any allocation.
 * The pages describe no counterpart of this call; it exists for callers that
 * cannot allocate device memory themselves: code running under a framework
 * that owns the GPU's memory (its own caching allocator, or one arena sized at
 * start-up, where a direct cudaMalloc would go around its accounting or fail
 * once the arena is full), and serving loops that cannot afford an allocation,
 * which may synchronise the device, in the middle of a step.
 *
 * Same arguments and results as csa_sparse_attend.  The split partials go to
 * one array of CSA_NOALLOC_SCRATCH_BYTES bytes that the library places in
 * device memory when it is loaded; every GPU that loads the library keeps that
 * array until the process exits.
 *  - Calls whose csa_attend_workspace_size exceeds CSA_NOALLOC_SCRATCH_BYTES
 *    return CSA_ERR_WORKSPACE without launching anything.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and remembers it; make that first call before any
 *    stream capture.
 *  - All calls share the one array per device.  Calls that can run at the same
 *    time on the GPU (different streams, no ordering between them) overwrite
 *    each other's partials: order them on one stream or with events.
 *  - The array keeps whatever the last call left in it; nothing in it has to
 *    start at zero, because each call writes every partial it later reads.
 *  - A call needs partials in memory only when its plan splits each query
 *    over more CTAs than a thread-block cluster holds (more than 8): at most
 *    16 queries (batch x P) on a 148-SM GPU, and K above 512.  Whether they
 *    fit depends on batch x P, H, d_latent and K together, and not
 *    monotonically on the number of queries: at 64 heads x 512 dims and
 *    K = 2048, 1 to 8 and 10 to 12 queries fit, 9 and 13 do not.  The exact
 *    test is csa_attend_workspace_size(cache, P, H, K, &n) with
 *    n <= CSA_NOALLOC_SCRATCH_BYTES: a call that passes it is never refused
 *    for size.
 */
#define CSA_NOALLOC_SCRATCH_BYTES (17u << 20)

CSA_API csa_status csa_sparse_attend_noalloc(const csa_cache *cache, int32_t P, int32_t H, const uint16_t *q,
                                             float scale, const int32_t *idx, int32_t K, float *out, float *lse,
                                             csa_stream_t stream);

/*
 * a7: one CSA2 layer for B*P queries.  ("G2C Brief", section "CSA2: most
 * layers don't keep their own cache": Full layers own the KV, the indexer keys
 * and the selection, Reindex layers borrow the KV and keys and select afresh
 * with their own indexer query, Reuse layers borrow the last selection; every
 * layer has its own query.  Section "The hierarchical indexer": the first Full
 * layer's pool, which later Reindex layers search.)
 *   FULL    : [append rows_new/ikeys_new if n_new > 0] -> scores over every
 *             visible row -> idx (top K) [-> pool_out] -> attention
 *   REINDEX : scores over every visible row, or over pool_in's rows when
 *             pool_in != NULL -> idx (fresh top K) -> attention
 *   REUSE   : attention over the given idx
 * idx is written by FULL/REINDEX and read by REUSE.  With swa set, every mode's
 * attention is the joint softmax of csa_sparse_attend_swa.  All arrays are
 * laid out as in the calls above.  workspace: csa_layer_workspace_size bytes.
 */
typedef struct csa_layer_args {
    csa_mode mode;
    int32_t P;                   /* query positions per sequence */
    int32_t H;                   /* main query heads */
    int32_t HI;                  /* indexer heads (FULL/REINDEX) */
    int32_t K;                   /* top-K */
    float scale;                 /* softmax scale, e.g. 1/sqrt(d_latent) */
    const uint16_t *q;           /* [batch][P][H][d_latent] bf16 bits */
    const uint8_t *iq;           /* [batch][P][HI][d_index] (FULL/REINDEX) */
    const float *w;              /* [batch][P][HI] (FULL/REINDEX) */
    const uint16_t *rows_new;    /* FULL only: [batch][n_new][d_latent] bf16 bits, or NULL */
    const uint8_t *ikeys_new;    /* FULL only: [batch][n_new][d_index], or NULL */
    int32_t n_new;               /* rows appended before scoring (FULL), else 0 */
    int32_t pool_blocks;         /* pool size in blocks (pool_in / pool_out) */
    const int32_t *pool_in;      /* REINDEX: [batch][P][pool_blocks] or NULL */
    int32_t *pool_out;           /* FULL: [batch][P][pool_blocks] or NULL */
    int32_t *idx;                /* [batch][P][K] */
    float *out;                  /* [batch][P][H][d_latent] fp32 */
    float *lse;                  /* [batch][P][H] fp32 or NULL */
    void *workspace;
    size_t workspace_bytes;
    const csa_swa *swa;          /* local window joined to the softmax, or NULL */
    const uint16_t *w_ik;        /* FULL with n_new > 0: project the new rows' indexer keys
                                    ([d_latent][d_index] bf16, as csa_quantize_append_project)
                                    instead of copying ikeys_new (which must then be NULL); or NULL */
} csa_layer_args;

/* One layer of the CSA2 mode chain ("G2C Brief", section "CSA2: most layers
 * don't keep their own cache"), as described above csa_layer_args. */
CSA_API csa_status csa_layer_step(const csa_cache *cache, const csa_layer_args *args, csa_stream_t stream);

/* Workspace query of csa_layer_step (no counterpart on the pages): scores,
 * selection scratch and attention partials of one layer. */
CSA_API csa_status csa_layer_workspace_size(const csa_cache *cache, const csa_layer_args *args, size_t *bytes);

/*
 * The context split: one sequence's cached rows split into contiguous slices
 * over G devices (each slice a csa_cache of its own, one query position per
 * sequence).  ("G2C Brief", section "The global branch: compress, index,
 * select": every entry is scored, the best are kept and attended to; section
 * "The hierarchical indexer": blocks of 8 scored by their best member.)  Each
 * device selects its slice's top K, turns it into (score, global id) pairs
 * (csa_select_pairs), the pairs of every device are gathered (by the caller's
 * collective), the global top K is taken among them (csa_topk_pairs; exact,
 * since a member of the global top K is in its own slice's top K), each
 * device attends over the selected ids in its slice (csa_ids_window, then
 * csa_sparse_attend), and the partial outputs are merged (csa_lse_merge).
 *
 * csa_select_pairs: for each sequence b of the slice's cache,
 *   idx         : [batch][n] local ids selected from scores (-1 = empty),
 *                 rows (block = 1) or blocks of 8 rows (block = 8)
 *   pair_scores : [batch][n] the score of each id (for a block: its best
 *                 member among the visible rows), -inf for an empty slot
 *   pair_ids    : [batch][n] id + id_offset (the slice's first global row, or
 *                 block), -1 for an empty slot
 */
CSA_API csa_status csa_select_pairs(const csa_cache *cache, const float *scores, int64_t ld, const int32_t *idx,
                                    int32_t n, int32_t block, int32_t id_offset, float *pair_scores,
                                    int32_t *pair_ids, csa_stream_t stream);

/* The context split's global selection ("G2C Brief", "The global branch"):
 * for each of `rows` rows, the ids of the K best of n (score, id) pairs
 * (ties: the earlier pair; id -1 = empty), in pair order then -1 padding;
 * pairs given in ascending id order (the devices' lists in slice order) give
 * ascending ids.  n <= 262144, 1 <= K <= 16384. */
CSA_API csa_status csa_topk_pairs(int32_t rows, int32_t n, const float *pair_scores, const int32_t *pair_ids,
                                  int32_t K, int32_t *idx, csa_stream_t stream);

/* No counterpart on the pages (the context split's bookkeeping): out[i] =
 * ids[i] - lo for lo <= ids[i] < hi, else -1 (the global ids a device owns, as
 * its local ids). */
CSA_API csa_status csa_ids_window(const int32_t *ids, int64_t count, int32_t lo, int32_t hi, int32_t *out,
                                  csa_stream_t stream);

/* The context split's merge ("G2C Brief", "The global branch": one softmax
 * over all the selected entries): parts partial results of the same queries,
 *   outs : [parts][units][H][D] fp32, each normalised over its own rows
 *   lses : [parts][units][H] fp32 (natural log; -inf = no rows)
 * -> out [units][H][D] = sum_g e^(lse_g - L) outs_g with L = ln sum_g e^lse_g,
 *    lse [units][H] = L (or NULL).  D a multiple of 4, all pointers 16-byte
 *    aligned. */
CSA_API csa_status csa_lse_merge(int32_t parts, int32_t units, int32_t H, int32_t D, const float *outs,
                                 const float *lses, float *out, float *lse, csa_stream_t stream);

/*
 * No counterpart on the pages (error reporting of this library).
 * Waits for `stream`, then copies the device status word of the current
 * device into *bits (0 = no fault) and, if clear != 0, resets it.
 * Returns CSA_ERR_DEVICE when a bit is set, else CSA_OK.
 */
CSA_API csa_status csa_device_status(int32_t *bits, int32_t clear, csa_stream_t stream);

/* No counterpart on the pages.  Number of kernels this library has launched in
 * the calling process (a host counter, for accounting in benchmarks; no device
 * work). */
CSA_API uint64_t csa_kernel_launches(void);

/* No counterpart on the pages.  Static description of a status code. */
CSA_API const char *csa_status_string(csa_status status);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
