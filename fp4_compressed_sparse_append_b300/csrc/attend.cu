// a5/a6: sparse attention of each query over its selected FP4 rows, on the
// tcgen05 tensor cores, split over the selection (flash-decode) with a merge pass.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select": the query attends to only the selected entries; one shared
// latent per entry serves every query head.  "DeepSeek V4.1 Flash: Pushing
// the Limits", section "The Paper": a single W_KV, so keys and values are the
// same vector.
//
// One CTA = one (sequence, position) query and a contiguous share of its
// selection, in tiles of 64 selected rows, as a warp-specialised pipeline:
//   gather warps   fetch one tile ahead: each thread holds a quarter of one FP4
//                  row (D/8 code bytes + D/64 scale bytes) in registers, then
//                  dequantises it to fp16 (E2M1 x E4M3 is exact in fp16) into a
//                  K-major 128B-swizzled tile V[64 rows][D] (two buffers);
//   MMA thread     S = Q . V^T (M = 64 heads, N = 64 rows, K = D; Q staged once
//                  per CTA as fp16 scaled per head by a power of two, safe from
//                  fp16 overflow and exact for every entry that lands in fp16's
//                  normal range, i.e. for heads whose entries span fewer than
//                  about 28 binades; smaller entries round to fp16 subnormals),
//                  and O^T += V^T . P^T with
//                  P split into fp16 high and low parts (two MMAs into one fp32
//                  accumulator keep P's precision near fp32); V^T is read from
//                  the same tile through an MN-major descriptor.  S of tile t+1
//                  is issued before O^T of tile t, so the tensor core works
//                  while the softmax runs;
//   softmax warps  one thread per head: the head's 64 logits come out of tensor
//                  memory as one row, so max, exp2 and sums need no cross-thread
//                  traffic; the running maximum is rescaled lazily (only when
//                  it grows by more than 2^8).
// The accumulator O^T [D x heads] stays in tensor memory across the CTA's tiles.
// At the end the softmax warps write the final output (one split).  With
// several splits of one query launched as a thread-block cluster, each split
// copies its unnormalised O, m and l into its own shared memory and, after a
// cluster barrier, each CTA combines one slice of the dims over every split by
// distributed-shared-memory loads and writes it; with more splits than a
// cluster holds, the partials go through global memory to the merge kernel.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kRows = 64;           // selected rows per tile (MMA N of S, K of O^T)
constexpr int kSoftWarps = 4;       // one per tensor-memory lane quarter
constexpr int kGatherWarps = 8;     // four threads per selected row
constexpr int kParts = kGatherWarps * 32 / 64;  // row parts (threads per row)
constexpr int kMaxPieces = 512 / (32 * kParts); // 16-byte code pieces per part at D = 512
constexpr int kThreads = 32 * (kSoftWarps + kGatherWarps + 1);  // + the MMA warp
constexpr int kMaxHeads = 64;       // S uses M = 64 (heads, zero-padded)
constexpr float kRescaleLog2 = 8.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxClusterSplit = 8;  // portable cluster size

struct AttArgs {
    CacheView c;
    int P, H, K;      // H: heads per CTA (one head group)
    int G;            // head groups per query: CTA row y is query y / G, heads (y % G) * H ..
    int NH;           // heads rounded up to 16 (MMA N of O^T)
    const uint16_t *q;
    float scale;
    const int32_t *idx;
    int nsplit, tiles_per_split, tiles_total;
    int cluster;      // 1: the nsplit CTAs of a query form a cluster and merge in shared memory
    // Local branch: split swa_split (the last) attends to the window of the
    // FP8 local rows [batch][swa_n][D] instead of selected FP4 rows; -1: none.
    const uint8_t *swa;
    const int32_t *swa_len;  // local rows per sequence, or null: swa_n each
    int swa_n, swa_window, swa_split;
    float *part_o;    // [units][nsplit][H][D]   (nsplit > 1)
    float2 *part_ml;  // [units][nsplit][H] (m in log2 units, l)
    float *out;       // [units][H][D]           (nsplit == 1)
    float *lse;       // [units][H] or null      (nsplit == 1)
    uint32_t tmem_cols;
    int *status;
};

// Byte offset of element (row, col) in a K-major, 128B-swizzled fp16 tile
// with `rows` rows: 64-column blocks of rows x 128 B; 8-row atoms of 1024 B;
// the 16-byte chunk index is XORed with (row % 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int col, int rows)
{
    const int kb = col >> 6, c = (col >> 3) & 7;
    return static_cast<uint32_t>(kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4) +
                                 (col & 7) * 2);
}

// Two E2M1 codes (one byte, even channel in the low nibble) times an fp16 scale.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t byte, uint32_t scale_h2)
{
    uint32_t v;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(v) : "r"(byte));
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(scale_h2));
    return r;
}

// Two E4M3 bytes (low byte = first value) -> two fp16 values, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t pair)
{
    uint32_t v;
    const uint16_t p16 = static_cast<uint16_t>(pair);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(v) : "h"(p16));
    return v;
}

// E4M3 byte -> fp16 value replicated in both halves.
__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t byte)
{
    uint32_t v;
    const uint16_t pair = static_cast<uint16_t>(byte | (byte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(v) : "h"(pair));
    return v;
}

// 8 bf16 (one uint4) * 2^e -> 8 fp16 (exact unless below fp16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float sc)
{
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t r4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(w4[k] << 16) * sc;
        const float hi = __uint_as_float(w4[k] & 0xFFFF0000u) * sc;
        const __half2 h = __floats2half2_rn(lo, hi);  // one conversion for the pair; lo in the low half
        r4[k] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(r4[0], r4[1], r4[2], r4[3]);
}

struct AttSmem {
    uint64_t vfull[2], vempty[2], sfull[2], sempty[2], pfull[2], pempty[2], xbar, done, qbar;
    uint32_t valid[2][2];     // row-valid bits of each V buffer
    float fac[2][kMaxHeads];  // rescale factor per head, by tile parity
    float cfac[kMaxHeads];    // scale * log2(e) * 2^-e per head (e: power of two applied to Q)
    float l_fin[kMaxHeads];   // final softmax sums (for the epilogue)
    float m_fin[kMaxHeads];
    int flag[2];              // == tile + 1 when some head rescales at that tile (by parity)
    uint32_t tmem_slot;
    int abort;
};

// SWA: one split attends to the local window; CLUSTER: the splits of a query
// form a cluster and merge on chip; ONE: every split holds at most one tile
// (no rescale of O, no next-tile gather).  Each combination is its own
// kernel, so the others' code is not in it: a CTA runs its code once, and
// code it carries but does not run still costs instruction fetches.
template <bool SWA, bool CLUSTER, bool ONE>
__global__ void __launch_bounds__(kThreads, 1) attend_kernel(const __grid_constant__ CUtensorMap qmap, AttArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int D = a.c.D, NH = a.NH, H = a.H;
    uint8_t *q_s = base;                                    // [64 heads][D] fp16, K-major SW128
    uint8_t *v_s = q_s + kMaxHeads * D * 2;                 // 2 x [64 rows][D]
    uint8_t *p_s = v_s + 2 * kRows * D * 2;                 // 2 x {hi, lo} x [NH heads][64 rows]
    const int p_bytes = NH * kRows * 2;                     // one P tile
    AttSmem &sm = *reinterpret_cast<AttSmem *>(p_s + 4 * p_bytes);
    volatile int *abort_flag = &sm.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // vunit: a query's head group (its q, out, lse and partials); unit: the
    // query (its selection, sequence and window)
    const int vunit = blockIdx.y, unit = vunit / a.G, split = blockIdx.x;
    const int b = unit / a.P;
    int len = 0;
    const bool win = SWA && split == a.swa_split;
    const int32_t *irow = a.idx + static_cast<int64_t>(unit) * a.K;
    const int mma_warp = kSoftWarps + kGatherWarps;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.vfull[i], 32 * kGatherWarps);
            mbar_init(&sm.vempty[i], 1);
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], 32 * kSoftWarps);
            sm.flag[i] = 0;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.pfull[i], 32 * kSoftWarps);
            mbar_init(&sm.pempty[i], 1);
        }
        mbar_init(&sm.xbar, 32 * kSoftWarps);
        mbar_init(&sm.done, 1);
        mbar_init(&sm.qbar, 1);
        sm.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&qmap);
    }
    if (warp == mma_warp) {
        tmem_alloc(&sm.tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    __syncthreads();  // barrier initialisation visible to every waiting thread
    // The query block [64 head rows][D] bf16 arrives by TMA, 128B-swizzled in
    // 64-dim boxes, in the second V buffer (free until the first tile is done).
    // The query is an input of the step, never written by this library's
    // kernels, so it is fetched before waiting on the previous kernel.
    uint8_t *q_stage = v_s + kRows * D * 2;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.qbar, static_cast<uint32_t>(NH * D * 2));
        for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(q_stage + kb * kMaxHeads * 128, &qmap, &sm.qbar, kb * 128, vunit * H);
    }
    // Q staged once as fp16 * 2^e per head, max|q| * 2^e < 2^15 (exact while
    // an entry stays within fp16's normal range, about 28 binades below the
    // head's largest; smaller ones round to fp16 subnormals), before the
    // wait on the previous kernel (q is an input of the step): thread (head
    // qh, quarter qq) of the first 256 threads converts dims [qq*D/4, (qq+1)*D/4)
    // from the bf16 block in shared memory.
    if (!mbar_wait(&sm.qbar, 0, abort_flag)) {
        // timed out: the status bit is raised at the end; the CTA drains below
    } else if (tid < 4 * kMaxHeads) {
        // Two passes over this thread's 16-byte chunks, both unrolled with
        // independent work per chunk: the exponent scan (four max chains), then
        // the conversion, re-reading shared memory.  Lane = 8 * quarter + head
        // (mod 8): each 8-lane phase of a 16-byte access covers 8 heads, whose
        // swizzled chunks fall in 8 different bank groups.
        const int qh = warp * 8 + (lane & 7), qq = lane >> 3, qn = D / 32;
        const uint32_t qst = smem_u32(q_stage), qs = smem_u32(q_s);
        auto chunk = [&](int i) -> uint4 {
            // 16-byte chunk i of this quarter: dims qq*D/4 + 8i .. +8
            const int dim = qq * (D / 4) + i * 8;
            const int kb = dim >> 6, c = (dim >> 3) & 7;
            return ld_shared_v4(qst + kb * kMaxHeads * 128 + qh * 128 + ((c ^ (qh & 7)) << 4));
        };
        constexpr uint32_t kExp = 0x7F807F80u;  // the exponent fields of two bf16
        uint32_t m4[4] = {0u, 0u, 0u, 0u};
        if (qh < H) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i < qn) {
                    const uint4 v = chunk(i);
                    m4[i & 3] = __vmaxu2(m4[i & 3], __vmaxu2(__vmaxu2(v.x & kExp, v.y & kExp),
                                                             __vmaxu2(v.z & kExp, v.w & kExp)));
                }
            }
        }
        const uint32_t m2 = __vmaxu2(__vmaxu2(m4[0], m4[1]), __vmaxu2(m4[2], m4[3]));
        uint32_t emax = max((m2 >> 7) & 0xFFu, m2 >> 23);
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 8));
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 16));
        const float e = emax > 0 ? 14.f - (static_cast<float>(emax) - 127.f) : 0.f;
        const float qscale = exp2f(e);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < qn)
                st_shared_v4(qs + sw128_off(qh, qq * (D / 4) + i * 8, kMaxHeads),
                             qh < H ? bf16x8_to_f16x8(chunk(i), qscale) : make_uint4(0, 0, 0, 0));
        if (qq == 0) sm.cfac[qh] = a.scale * kLog2e * exp2f(-e);
    }
    // Below: reads of what earlier kernels on the stream wrote (lengths, indices, cache).
    pdl_wait();
    // A gather thread's row id in the first tile of a selection split, loaded
    // beside the sequence length (the two loads are independent).
    int32_t first_id = -1;
    {
        const int j0 = (split * a.tiles_per_split) * kRows + ((tid - 32 * kSoftWarps) & (kRows - 1));
        if (!win && warp >= kSoftWarps && warp < mma_warp && split * a.tiles_per_split < a.tiles_total && j0 < a.K)
            first_id = irow[j0];
    }
    len = min(a.c.lengths[b], a.c.cap);
    // The window split's rows: [w_lo, w_hi) of the sequence's local rows, the
    // window of tokens that ends at this position's own row (L - P + p for a
    // sequence of L local rows).  A length outside [P, swa_n] is a caller
    // error: flagged, and the window left empty.
    int w_lo = 0, w_hi = 0;
    if (win) {
        const int L = a.swa_len ? a.swa_len[b] : a.swa_n;
        if (L < a.P || L > a.swa_n) {
            if (tid == 0) raise_status(a.status, CSA_DEV_BAD_INDEX);
        } else {
            w_hi = L - a.P + unit % a.P + 1;
            w_lo = max(0, w_hi - a.swa_window);
        }
    }
    const int t_first = win ? 0 : split * a.tiles_per_split;
    const int t_last = win ? (w_hi - w_lo + kRows - 1) / kRows : min(a.tiles_total, t_first + a.tiles_per_split);
    const int n_tiles = ONE ? min(1, max(0, t_last - t_first)) : max(0, t_last - t_first);

    // Gather-warp state: the rows of tile i+1 are loaded while tile i is used;
    // thread (row gr, part gp) holds D/kParts channels of one FP4 row: nc
    // 16-byte code pieces (32 channels each) and their two scale bytes each.
    const bool is_gather = warp >= kSoftWarps && warp < mma_warp;
    const int gt = tid - 32 * kSoftWarps;
    const int gr = gt & (kRows - 1), gp = gt >> 6;
    const int nc = D / (32 * kParts);
    int32_t nrow = -1;
    uint4 ncw[2 * kMaxPieces];  // FP4: nc pieces; FP8 window rows: 2 nc pieces (16 channels each)
    uint32_t nsw[kMaxPieces];   // two scale bytes per FP4 code piece
    auto prefetch = [&](int tile) {
        if (win) {
            const int row = w_lo + tile * kRows + gr;
            nrow = row < w_hi ? row : -1;
            const uint4 *wp = reinterpret_cast<const uint4 *>(
                                  a.swa + (static_cast<int64_t>(b) * a.swa_n + (nrow >= 0 ? row : 0)) * D) +
                              gp * 2 * nc;
#pragma unroll
            for (int i = 0; i < 2 * kMaxPieces; ++i) ncw[i] = (nrow >= 0 && i < 2 * nc) ? wp[i] : make_uint4(0, 0, 0, 0);
            return;
        }
        const int j = tile * kRows + gr;
        int32_t row = tile == t_first ? first_id : (j < a.K ? irow[j] : -1);
        if (row >= len) {
            if (gp == 0) raise_status(a.status, CSA_DEV_BAD_INDEX);
            row = -1;
        }
        nrow = row;
        const int64_t g = static_cast<int64_t>(b) * a.c.cap + (row >= 0 ? row : 0);
        const uint4 *cp = reinterpret_cast<const uint4 *>(a.c.codes + g * (D / 2)) + gp * nc;
        const uint16_t *sp = reinterpret_cast<const uint16_t *>(a.c.scales + g * (D / 16)) + gp * nc;
#pragma unroll
        for (int i = 0; i < kMaxPieces; ++i) ncw[i] = (row >= 0 && i < nc) ? cp[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < kMaxPieces; ++i) nsw[i] = (row >= 0 && i < nc) ? sp[i] : 0u;
    };
    if (is_gather && n_tiles > 0) prefetch(t_first);

    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t t_s = tmem;                 // S: 2 buffers x 64 columns (rows of the tile)
    const uint32_t t_o = tmem + 2 * kRows;     // O^T: (D/128) blocks of NH columns

    if (warp == mma_warp) {
        // ------------------------------------------------------------ MMA thread
        if (lane == 0 && n_tiles > 0) {
            const uint32_t v_bytes = kRows * D * 2;
            const uint32_t idesc_s = instr_desc(64, kRows, 0, 0, 0, 0);  // K-major Q, K-major V
            const uint32_t idesc_o = instr_desc(128, NH, 0, 0, 1, 0);    // MN-major V^T, K-major P
            // Descriptors are built once; an MMA's operand is the base plus a
            // byte offset added to the start-address field (>> 4).
            const uint64_t dq = smem_desc(smem_u32(q_s), 16, 1024, 2);
            const uint64_t dv = smem_desc(smem_u32(v_s), 16, 1024, 2);
            const uint64_t dvt = smem_desc(smem_u32(v_s), kRows * 128 /*next 64 dims*/, 1024 /*next 8 rows*/, 2);
            const uint64_t dp = smem_desc(smem_u32(p_s), 16, 1024, 2);
            auto issue_s = [&](int i) {
                tc_fence_after();
                const uint64_t vb = dv + (((i & 1) * v_bytes) >> 4);
                for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(t_s + (i & 1) * kRows, dq + ((kb * kMaxHeads * 128 + ks * 32) >> 4),
                                vb + ((kb * kRows * 128 + ks * 32) >> 4), idesc_s, (kb > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&sm.sfull[i & 1]);
            };
            auto issue_pv = [&](int i) {
                tc_fence_after();
                const uint64_t vb = dvt + (((i & 1) * v_bytes) >> 4);
                for (int mt = 0; mt < D / 128; ++mt)
                    for (int hl = 0; hl < 2; ++hl) {
                        const uint64_t pb = dp + ((((i & 1) * 2 + hl) * p_bytes) >> 4);
#pragma unroll
                        for (int ks = 0; ks < kRows / 16; ++ks)
                            mma_f16(t_o + mt * NH, vb + ((2 * mt * kRows * 128 + ks * 2048) >> 4), pb + ((ks * 32) >> 4),
                                    idesc_o, (i > 0 || hl > 0 || ks > 0) ? 1u : 0u);
                    }
                mma_commit(&sm.pempty[i & 1]);
                mma_commit(&sm.vempty[i & 1]);
            };
            // Issue in order of readiness: O^T of tile i as soon as its P is
            // written (which also frees its V buffer for the gather sooner),
            // S of tile i+1 as soon as its V is gathered and its S buffer is
            // free.  Polling is non-blocking so neither waits behind the other.
            int ns = 0, npv = 0;
            unsigned long long t_idle = global_ns();
            while (npv < n_tiles) {
                if (npv < ns && mbar_test(&sm.pfull[npv & 1], (npv >> 1) & 1)) {
                    issue_pv(npv++);
                    t_idle = global_ns();
                } else if (ns < n_tiles && ns < npv + 2 && mbar_test(&sm.vfull[ns & 1], (ns >> 1) & 1) &&
                           mbar_test(&sm.sempty[ns & 1], ((ns >> 1) & 1) ^ 1)) {
                    issue_s(ns++);
                    t_idle = global_ns();
                } else if (*abort_flag) {
                    break;
                } else if (global_ns() - t_idle > kWaitLimitNs) {
                    *abort_flag = 1;
                    break;
                }
            }
            mma_commit(&sm.done);
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(&sm.done, 0) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (is_gather) {
        // ------------------------------------------------------------ gather warps
        for (int i = 0; i < n_tiles; ++i) {
            if (!mbar_wait(&sm.vempty[i & 1], ((i >> 1) & 1) ^ 1, abort_flag)) break;
            const uint32_t vb = smem_u32(v_s) + (i & 1) * kRows * D * 2;
            const unsigned vbits = __ballot_sync(0xFFFFFFFFu, nrow >= 0);
            if (gp == 0 && lane == 0) sm.valid[i & 1][gr >> 5] = vbits;
            if (win) {
                // FP8 E4M3 window rows: exact in fp16, two channels per conversion.
#pragma unroll
                for (int c = 0; c < 2 * kMaxPieces; ++c) {
                    if (c >= 2 * nc) break;
                    const uint32_t words[4] = {ncw[c].x, ncw[c].y, ncw[c].z, ncw[c].w};
                    const int ch0 = gp * (D / kParts) + c * 16;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 o;
                        o.x = e4m3x2_to_h2(words[2 * h] & 0xFFFF);
                        o.y = e4m3x2_to_h2(words[2 * h] >> 16);
                        o.z = e4m3x2_to_h2(words[2 * h + 1] & 0xFFFF);
                        o.w = e4m3x2_to_h2(words[2 * h + 1] >> 16);
                        st_shared_v4(vb + sw128_off(gr, ch0 + h * 8, kRows), o);
                    }
                }
                fence_async_smem();
                mbar_arrive(&sm.vfull[i & 1]);
                if (!ONE && i + 1 < n_tiles) prefetch(t_first + i + 1);
                continue;
            }
#pragma unroll
            for (int c16 = 0; c16 < kMaxPieces; ++c16) {
                if (c16 >= nc) break;
                const uint32_t sc = nsw[c16];  // the scales of this piece's two 16-channel groups
                const uint32_t s0 = e4m3_to_h2(sc & 0xFF), s1 = e4m3_to_h2(sc >> 8);
                const uint32_t words[4] = {ncw[c16].x, ncw[c16].y, ncw[c16].z, ncw[c16].w};
                const int ch0 = gp * (D / kParts) + c16 * 32;
#pragma unroll
                for (int h8 = 0; h8 < 4; ++h8) {
                    const uint32_t sv = h8 < 2 ? s0 : s1;
                    const uint32_t wd = words[h8];
                    uint4 o;
                    o.x = dequant_pair(wd & 0xFF, sv);
                    o.y = dequant_pair((wd >> 8) & 0xFF, sv);
                    o.z = dequant_pair((wd >> 16) & 0xFF, sv);
                    o.w = dequant_pair(wd >> 24, sv);
                    st_shared_v4(vb + sw128_off(gr, ch0 + h8 * 8, kRows), o);
                }
            }
            fence_async_smem();
            mbar_arrive(&sm.vfull[i & 1]);
            if (!ONE && i + 1 < n_tiles) prefetch(t_first + i + 1);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        // Head h = 16*warp + (lane & 15) is tensor-memory lane 32*warp + (lane & 15)
        // of S; lane < 16 takes the tile's rows 0..31, lane + 16 rows 32..63.
        const int h = warp * 16 + (lane & 15), ch = lane >> 4;
        const bool active = h < H;
        const float cf = sm.cfac[h];
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            const uint32_t par = (i >> 1) & 1;
            ok = mbar_wait(&sm.sfull[i & 1], par, abort_flag) && mbar_wait(&sm.vfull[i & 1], par, abort_flag);
            if (!ok) break;
            tc_fence_after();
            uint32_t z[32];
            asm volatile(
                "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
                "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], 32;"
                : "=r"(z[0]), "=r"(z[1]), "=r"(z[2]), "=r"(z[3]), "=r"(z[4]), "=r"(z[5]), "=r"(z[6]), "=r"(z[7]),
                  "=r"(z[8]), "=r"(z[9]), "=r"(z[10]), "=r"(z[11]), "=r"(z[12]), "=r"(z[13]), "=r"(z[14]),
                  "=r"(z[15]), "=r"(z[16]), "=r"(z[17]), "=r"(z[18]), "=r"(z[19]), "=r"(z[20]), "=r"(z[21]),
                  "=r"(z[22]), "=r"(z[23]), "=r"(z[24]), "=r"(z[25]), "=r"(z[26]), "=r"(z[27]), "=r"(z[28]),
                  "=r"(z[29]), "=r"(z[30]), "=r"(z[31])
                : "r"(t_s + (i & 1) * kRows + lane_off));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&sm.sempty[i & 1]);
            const uint32_t vbits = sm.valid[i & 1][ch];
            float tmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float zz = (vbits >> k & 1) ? __uint_as_float(z[k]) * cf : -INFINITY;
                z[k] = __float_as_uint(zz);
                tmax = fmaxf(tmax, zz);
            }
            tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 16));
            float f = 1.f;
            if (active && tmax > -INFINITY && (m_run == -INFINITY || tmax > m_run + kRescaleLog2)) {
                f = m_run == -INFINITY ? 0.f : fast_exp2(m_run - tmax);
                m_run = tmax;
            }
            if (!ONE) {
                // Every softmax thread sees every head's factor and the flag
                // (one tile: nothing is rescaled)
                if (lane < 16) sm.fac[i & 1][h] = f;
                const bool mine = i > 0 && f != 1.f;
                if (__any_sync(0xFFFFFFFFu, mine) && lane == 0) sm.flag[i & 1] = i + 1;
                mbar_arrive(&sm.xbar);
                ok = mbar_wait(&sm.xbar, i & 1, abort_flag);
            }
            // the P buffer of this tile is free once O^T of tile i-2 is done
            ok = ok && mbar_wait(&sm.pempty[i & 1], ((i >> 1) & 1) ^ 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            if (!ONE && sm.flag[i & 1] == i + 1) {
                // Rescale O^T: wait for O^T of tile i-1, then this warp's quarter of
                // the lanes (dims) of every 128-dim block, all head columns.
                if (!mbar_wait(&sm.pempty[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int mt = 0; mt < D / 128; ++mt)
                    for (int c0 = 0; c0 < NH; c0 += 16) {
                        uint32_t r16[16];
                        const uint32_t ta = t_o + mt * NH + lane_off + c0;
                        tmem_ld16(ta, r16);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            r16[k] = __float_as_uint(__uint_as_float(r16[k]) * sm.fac[i & 1][c0 + k]);
                        tmem_st16(ta, r16);
                    }
                tmem_st_wait();
            }
            l_run *= f;
            float lsum = 0.f;
            if (h < NH) {
                const uint32_t ph_s = smem_u32(p_s) + (i & 1) * 2 * p_bytes, pl_s = ph_s + p_bytes;
#pragma unroll
                for (int k8 = 0; k8 < 4; ++k8) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        // p = hi + lo: hi keeps p's leading 11 significant bits
                        // (exact in fp16 for p >= 2^-14), lo the exact fp32
                        // remainder rounded to fp16; one conversion per pair each.
                        float hf[2], lf[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float zz = __uint_as_float(z[k8 * 8 + k2 * 2 + e]);
                            const float pv = (active && zz > -INFINITY) ? fast_exp2(zz - m_run) : 0.f;
                            lsum += pv;
                            hf[e] = __uint_as_float(__float_as_uint(pv) & 0xFFFFE000u);
                            lf[e] = pv - hf[e];
                        }
                        const __half2 h2 = __floats2half2_rn(hf[0], hf[1]), l2 = __floats2half2_rn(lf[0], lf[1]);
                        hw[k2] = *reinterpret_cast<const uint32_t *>(&h2);
                        lw[k2] = *reinterpret_cast<const uint32_t *>(&l2);
                    }
                    const uint32_t off = sw128_off(h, ch * 32 + k8 * 8, NH);
                    st_shared_v4(ph_s + off, make_uint4(hw[0], hw[1], hw[2], hw[3]));
                    st_shared_v4(pl_s + off, make_uint4(lw[0], lw[1], lw[2], lw[3]));
                }
            }
            lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 16);
            l_run += lsum;
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.pfull[i & 1]);
        }
        // ---- the last O^T update done: final (m, l) per head
        if (ok && n_tiles > 0) ok = mbar_wait(&sm.pempty[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, abort_flag);
        if (lane < 16) {
            sm.l_fin[h] = l_run;
            sm.m_fin[h] = m_run;
        }
        if (lane < 16 && active && !CLUSTER) {
            if (a.nsplit == 1) {
                if (a.lse)
                    a.lse[static_cast<int64_t>(vunit) * H + h] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            } else {
                a.part_ml[(static_cast<int64_t>(vunit) * a.nsplit + split) * H + h] = make_float2(m_run, l_run);
            }
        }
    }

    // ---- epilogue over all softmax and gather warps: O^T from tensor memory
    // (warp w reads lane quadrant w % 4, i.e. 32 dims of each 128-dim block)
    // to the split partial in global memory, to the final output (one split),
    // or to shared memory [H][D] over the V buffers for the cluster merge.
    // Work items are (dim block, 16 heads); the three warps of a quadrant
    // take every third item.
    if (warp < mma_warp) {
        named_barrier_sync(1, 32 * mma_warp);  // the softmax warps have seen the last O^T update
        tc_fence_after();
        if (!*abort_flag) {
            const int q4 = warp & 3, grp = warp >> 2, ngrp = mma_warp / 4;
            const uint32_t loff = static_cast<uint32_t>(q4 * 32) << 16;
            const int nc16 = NH / 16, items = (D / 128) * nc16;
            const bool final_out = a.nsplit == 1 && !CLUSTER;
            float *obuf = reinterpret_cast<float *>(v_s);
            float *obase = final_out ? a.out + static_cast<int64_t>(vunit) * H * D
                                     : a.part_o + (static_cast<int64_t>(vunit) * a.nsplit + split) * H * D;
            for (int it = grp; it < items; it += ngrp) {
                const int mt = it / nc16, c0 = (it - mt * nc16) * 16;
                const int d = mt * 128 + q4 * 32 + lane;
                uint32_t r[16];
                tmem_ld16(t_o + mt * NH + loff + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int hh = c0 + k;
                    if (hh >= H) break;
                    float v = n_tiles > 0 ? __uint_as_float(r[k]) : 0.f;
                    if (CLUSTER) {
                        obuf[hh * D + d] = v;
                    } else {
                        if (final_out) {
                            const float lh = sm.l_fin[hh];
                            v = lh > 0.f ? v * __frcp_rn(lh) : 0.f;
                        }
                        obase[static_cast<int64_t>(hh) * D + d] = v;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (CLUSTER) {
        // Every split's O, m and l are in its shared memory after this barrier;
        // each CTA merges dims [d0, d1) of every head over the splits.
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int C = a.nsplit, rank = static_cast<int>(cluster.block_rank());
        const int slice = ((D + C - 1) / C + 3) & ~3;  // C slices of a multiple of 4 dims cover D
        const int d0 = min(D, rank * slice), d1 = min(D, d0 + slice);
        float *wq = reinterpret_cast<float *>(p_s);  // [split][head] normalised weights (P buffers are free)
        if (tid < H) {
            float mq[kMaxClusterSplit], lq[kMaxClusterSplit];
            float M = -INFINITY;
            for (int q = 0; q < C; ++q) {
                const AttSmem *rs = cluster.map_shared_rank(&sm, q);
                mq[q] = rs->m_fin[tid];
                lq[q] = rs->l_fin[tid];
                if (lq[q] > 0.f) M = fmaxf(M, mq[q]);
            }
            float L = 0.f;
            for (int q = 0; q < C; ++q) {
                mq[q] = lq[q] > 0.f ? exp2f(mq[q] - M) : 0.f;
                L = fmaf(mq[q], lq[q], L);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            for (int q = 0; q < C; ++q) wq[q * kMaxHeads + tid] = mq[q] * inv;
            if (rank == 0 && a.lse)
                a.lse[static_cast<int64_t>(vunit) * H + tid] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        __syncthreads();
        const int nd4 = (d1 - d0) / 4;
        const float *obuf = reinterpret_cast<const float *>(v_s);
        for (int w = tid; w < H * nd4; w += kThreads) {
            const int hh = w / nd4, d = d0 + 4 * (w - hh * nd4);
            // All the splits' loads are issued before any is used.
            float4 v[kMaxClusterSplit];
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q)
                if (q < C) v[q] = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(obuf, q) + hh * D + d);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxClusterSplit; ++q) {
                if (q >= C) break;
                const float wgt = wq[q * kMaxHeads + hh];
                acc.x = fmaf(wgt, v[q].x, acc.x);
                acc.y = fmaf(wgt, v[q].y, acc.y);
                acc.z = fmaf(wgt, v[q].z, acc.z);
                acc.w = fmaf(wgt, v[q].w, acc.w);
            }
            *reinterpret_cast<float4 *>(a.out + (static_cast<int64_t>(vunit) * H + hh) * D + d) = acc;
        }
        cluster.sync();  // no CTA leaves while another still reads its shared memory
    }
    // The next kernel (the split merge) is released only now: its CTAs are
    // small enough to share this CTA's SM, and waiting there they slow it.
    pdl_trigger();
    if (*abort_flag && tid == 0) raise_status(a.status, CSA_DEV_TIMEOUT);
    if (warp == mma_warp) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// Combines the split partials: block = one warp over (128 dims, head, query),
// so that even one query's merge spreads over more CTAs than there are SMs
// (each SM's share of the partials is what bounds it); each lane loads its 4
// dims (one 16-byte load) from every split at once.
// out = sum_s 2^(m_s - M) O_s / L, L = sum_s 2^(m_s - M) l_s,
// lse = ln 2 * (M + log2 L).
constexpr int kMaxSplit = 32;  // one warp holds every split's (m, l) in the merge
constexpr int kMergeDims = 128;

template <int MS>
__global__ void __launch_bounds__(32) attend_merge_kernel(int D, int H, int nsplit, const float *__restrict__ part_o,
                                                         const float2 *__restrict__ part_ml, float *__restrict__ out,
                                                         float *__restrict__ lse)
{
    pdl_wait();
    __shared__ float wsh[MS];
    const int lane = threadIdx.x;
    const int d = blockIdx.x * kMergeDims + lane * 4, h = blockIdx.y, unit = blockIdx.z;
    float4 pv[MS];
#pragma unroll
    for (int s = 0; s < MS; ++s)
        pv[s] = (s < nsplit && d < D) ? *reinterpret_cast<const float4 *>(
                                            part_o + ((static_cast<int64_t>(unit) * nsplit + s) * H + h) * D + d)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < nsplit) ml = part_ml[(static_cast<int64_t>(unit) * nsplit + lane) * H + h];
    float M = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    const float w = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
    float L = w * ml.y;
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
    if (lane < MS) wsh[lane] = w;
    if (lse && blockIdx.x == 0 && lane == 0)
        lse[static_cast<int64_t>(unit) * H + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    __syncwarp();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < MS; ++s) {
        const float ws = wsh[s];
        acc.x = fmaf(ws, pv[s].x, acc.x);
        acc.y = fmaf(ws, pv[s].y, acc.y);
        acc.z = fmaf(ws, pv[s].z, acc.z);
        acc.w = fmaf(ws, pv[s].w, acc.w);
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    if (d < D)
        *reinterpret_cast<float4 *>(out + (static_cast<int64_t>(unit) * H + h) * D + d) =
            make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
}

struct Plan {
    int nsplit, tiles_per_split, tiles_total, cluster;
    int swa_split;  // index of the local-window split, or -1
    int G;          // head groups per query
};

// Splits of one query's selection: at most one wave of CTAs.  Up to
// kMaxClusterSplit splits form a cluster and merge on chip; more (only for
// very few queries) merge through global memory, which measures faster than a
// cluster of 16 for them.  With a local window, one more split per query
// attends to the window and is merged like the others.
// When a query's splits still leave SMs idle, its heads are split into G
// groups of at least 16 (the heads' softmaxes are independent), each group a
// CTA row of its own over the same selection: a CTA then converts only its
// group's query rows and writes only its group's share of the output or
// partial (a quarter of the 128 KB partial for one query of 64 heads split 4
// ways).  The partials and the workspace keep their total size.
Plan plan(const CacheView &c, int P, int H, int K, const SwaView *swa)
{
    const int units = c.B * P;
    const int extra = swa ? 1 : 0;
    const int tiles = (K + kRows - 1) / kRows;
    int want = sm_count() / units - extra;  // splits x queries within one wave of CTAs (one per SM)
    if (want > tiles) want = tiles;
    if (want > kMaxSplit - extra) want = kMaxSplit - extra;
    if (want < 1) want = 1;
    Plan p;
    if (tiles == 0) {  // nothing selected: one split
        p.tiles_total = 0;
        p.tiles_per_split = 1;
        p.nsplit = 1 + extra;
        p.swa_split = swa ? 1 : -1;
        p.cluster = p.nsplit > 1;
        p.G = 1;
        return p;
    }
    p.tiles_total = tiles;
    p.tiles_per_split = (tiles + want - 1) / want;
    const int main_splits = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    p.nsplit = main_splits + extra;
    p.swa_split = swa ? main_splits : -1;
    p.cluster = p.nsplit > 1 && p.nsplit <= kMaxClusterSplit;
    p.G = 1;
    while (H % (2 * p.G) == 0 && H / (2 * p.G) >= 16 &&
           static_cast<int64_t>(units) * p.nsplit * 2 * p.G <= sm_count())
        p.G *= 2;
    return p;
}

size_t smem_bytes(int D, int NH)
{
    return 1024 + static_cast<size_t>(kMaxHeads) * D * 2 + 2 * static_cast<size_t>(kRows) * D * 2 +
           4 * static_cast<size_t>(NH) * kRows * 2 + sizeof(AttSmem);
}

}  // namespace

size_t attend_workspace_bytes(const CacheView &c, int P, int H, int K, const SwaView *swa)
{
    const Plan p = plan(c, P, H, K, swa);
    if (p.nsplit == 1 || p.cluster) return 0;
    const size_t units = static_cast<size_t>(c.B) * P;
    size_t o = units * p.nsplit * H * c.D * sizeof(float);
    o = (o + 255) / 256 * 256;
    return o + units * p.nsplit * H * sizeof(float2);
}

cudaError_t launch_attend(const CacheView &c, int P, int H, const uint16_t *q, float scale, const int32_t *idx,
                          int K, float *out, float *lse, void *ws, size_t ws_bytes, int *status, cudaStream_t st,
                          const SwaView *swa)
{
    const int units = c.B * P;
    if (units == 0) return cudaSuccess;
    if (H > kMaxHeads || c.D % 128 || c.D > 512) return cudaErrorInvalidValue;
    if (swa && (!swa->rows || swa->n < P || swa->window < 1)) return cudaErrorInvalidValue;
    const Plan p = plan(c, P, H, K, swa);
    const int Hg = H / p.G;  // heads per CTA
    const size_t smem = smem_bytes(c.D, (Hg + 15) / 16 * 16);
    const bool one = !swa && p.tiles_per_split == 1;
    auto kernel = swa ? (p.cluster ? attend_kernel<true, true, false> : attend_kernel<true, false, false>)
                      : one ? (p.cluster ? attend_kernel<false, true, true> : attend_kernel<false, false, true>)
                            : (p.cluster ? attend_kernel<false, true, false> : attend_kernel<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (ws_bytes < attend_workspace_bytes(c, P, H, K, swa)) return cudaErrorInvalidValue;
    AttArgs a{};
    a.c = c;
    a.P = P;
    a.H = Hg;
    a.G = p.G;
    a.K = K;
    a.NH = (Hg + 15) / 16 * 16;
    a.q = q;
    a.scale = scale;
    a.idx = idx;
    a.nsplit = p.nsplit;
    a.tiles_per_split = p.tiles_per_split;
    a.tiles_total = p.tiles_total;
    a.cluster = p.cluster;
    a.swa = swa ? swa->rows : nullptr;
    a.swa_len = swa ? swa->lengths : nullptr;
    a.swa_n = swa ? swa->n : 0;
    a.swa_window = swa ? swa->window : 0;
    a.swa_split = p.swa_split;
    size_t o_bytes = static_cast<size_t>(units) * p.nsplit * H * c.D * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    a.part_o = static_cast<float *>(ws);
    a.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + o_bytes);
    a.out = out;
    a.lse = lse;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * kRows + (c.D / 128) * a.NH)) cols *= 2;
    a.tmem_cols = cols;
    a.status = status;
    // Query rows [units*H][D] bf16 as bytes: 64-dim (128-byte) boxes of NH rows
    // (one head group, rounded up to 16).
    CUtensorMap qm;
    if (encode_tensor_map_2d_u8(&qm, q, static_cast<uint64_t>(c.D) * 2, static_cast<uint64_t>(units) * H, 128,
                                a.NH, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    e = launch_kernel(kernel, dim3(p.nsplit, units * p.G), dim3(kThreads), smem, st, p.cluster ? p.nsplit : 0,
                      qm, a);
    if (e != cudaSuccess || p.nsplit == 1 || p.cluster) return e;
    // The merge loads every split's value at once: 16 or 32 registers.
    auto merge = p.nsplit <= 16 ? attend_merge_kernel<16> : attend_merge_kernel<kMaxSplit>;
    return launch_kernel(merge, dim3((c.D + kMergeDims - 1) / kMergeDims, Hg, units * p.G), dim3(32), 0, st, 0, c.D, Hg,
                         p.nsplit,
                         static_cast<const float *>(a.part_o), static_cast<const float2 *>(a.part_ml), out, lse);
}

}  // namespace csa
