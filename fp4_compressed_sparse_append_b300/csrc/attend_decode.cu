// a5/a6 for few queries: sparse attention over the selected FP4 rows, one
// thread-block cluster per query.  "G2C Brief - DeepSeek V4.1-Flash", section
// "The global branch: compress, index, select": the query attends to only the
// selected entries; one shared latent per entry serves every query head.
// "DeepSeek V4.1 Flash: Pushing the Limits", section "The Paper": one W_KV, so
// keys and values are the same vector.
//
// A decode step has a handful of queries and thousands of selected rows per
// query, so the rows, not the heads, fill the tensor core's M dimension.  One
// CTA takes a contiguous share of one query's selection, in tiles of 128 rows:
//   worker warps   (8) two threads per selected row.  Each loads half of its
//                  row's FP4 codes and E4M3 scales, dequantises them exactly to
//                  fp16 and stores them into V[128 rows][D] (K-major, 128-byte
//                  swizzle); the next tile's rows are loaded while the tensor
//                  core works on the current one.  Then each runs the softmax
//                  of its row for half of the heads (below);
//   MMA thread     S^T = V . Q^T   (M = 128 rows, N = heads, K = D) into tensor
//                  memory, then O^T += V^T . P^T (M = 128 dims per chunk,
//                  N = heads, K = 128 rows), V^T read from the same tile
//                  through an MN-major descriptor;
//   softmax        the row's logits for its heads come out of tensor memory
//                  in one load; per-head maxima and sums over the tile's rows
//                  are butterfly reductions across the warp plus one exchange
//                  between the four warps of a head half; P is written as two
//                  fp16 parts (hi + lo); the running maximum is rescaled lazily
//                  (when it grows by 2^8).  Nine warps leave each thread 168
//                  registers (thirteen would cap it at 128, with spills).
// O^T stays in tensor memory.  Q is staged once per CTA as fp16 scaled per
// head by a power of two: exact for every entry within fp16's normal range,
// i.e. for heads whose entries span fewer than about 28 binades (smaller
// entries round to fp16 subnormals).
//
// The CTAs of one query form a cluster, so all of them run at once: each
// stores its unnormalised O and its (max, sum) per head in the caller's
// workspace, and after one cluster barrier each combines one slice of the dims
// over the splits with the log-sum-exp weights and writes it.  (Exchanging
// the partials through distributed shared memory measured several times
// slower: 4-byte remote stores of 128 KB per CTA took about 7 us.)
#include <cuda_fp16.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kTRows = 128;                     // selected rows per tile
constexpr int kWorkWarps = 8;                   // two threads per selected row (gather, softmax)
constexpr int kWorkers = 32 * kWorkWarps;
constexpr int kThreads = kWorkers + 32;         // + the MMA warp
constexpr int kMmaWarp = kWorkWarps;
constexpr int kMaxHeads = 64;
constexpr int kMaxSplit = 16;                   // splits of one query (cluster size), a power of two
constexpr float kRescaleLog2 = 8.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecArgs {
    CacheView c;
    int P, H, K;
    float scale;
    const int32_t *idx;
    int nsplit, tiles_per_split;
    float *part_o;    // nsplit > 1: [units][nsplit][H][D] unnormalised split outputs (workspace)
    float2 *part_ml;  // nsplit > 1: [units][nsplit][H] (max in log2 units, sum) per split
    float *out;       // [units][H][D]
    float *lse;       // [units][H] or null
    uint32_t tmem_cols;
    int *status;
};

struct DecSmem {
    uint64_t vfull, vempty, sfull[2], sempty[2], pfull, pempty, done, qbar, rbar;
    uint32_t valid[4];                  // row-valid bits of the V tile
    __align__(16) float cf[kMaxHeads];                // scale * log2(e) * 2^-e per head (e: power of two applied to Q)
    float m_run[kMaxHeads];             // running maximum per head (log2 units)
    float l_run[kMaxHeads];             // running sum per head
    float fac[kMaxHeads];               // rescale factor of the current tile
    float redm[4][kMaxHeads];           // per lane-quarter tile maxima
    float reds[4][kMaxHeads];           // per lane-quarter tile sums
    float wq[kMaxSplit][kMaxHeads];     // merge weight of every split, per head
    int flag;                           // == tile + 1 when some head rescales at that tile
    uint32_t tmem_slot;
    int abort;
};

__device__ __forceinline__ uint32_t sw128_off(int row, int col, int rows)
{
    const int kb = col >> 6, c = (col >> 3) & 7;
    return static_cast<uint32_t>(kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4) +
                                 (col & 7) * 2);
}

// Two E2M1 codes (one byte, even channel in the low nibble) times an fp16 scale
// (exact: 3 significant bits times 4).
__device__ __forceinline__ uint32_t dequant_pair(uint32_t byte, uint32_t scale_h2)
{
    uint32_t v;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(v) : "r"(byte));
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(scale_h2));
    return r;
}

__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t byte)
{
    uint32_t v;
    const uint16_t pair = static_cast<uint16_t>(byte | (byte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(v) : "h"(pair));
    return v;
}

// 8 bf16 (one uint4) * 2^e -> 8 fp16.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, float sc)
{
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t r4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w4[k] << 16) * sc, __uint_as_float(w4[k] & 0xFFFF0000u) * sc);
        r4[k] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(r4[0], r4[1], r4[2], r4[3]);
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from shared to global memory,
// committed as a group; the waits block until the group has completed.
__device__ __forceinline__ void bulk_store(void *gdst, uint32_t ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders the async proxy's global writes (bulk copies) before later generic
// memory operations of this thread.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Reduction of N per-head values across the 32 lanes of a warp, halving the
// values a lane keeps at every step (offsets 16, 8, 4, 2, 1): afterwards lane
// l holds in v[j] the reduction for head l*N/32 + j (N >= 32), or for head
// l / (32/N) (N < 32, held by all 32/N lanes of that group).
template <int N, int O, bool Max>
__device__ __forceinline__ void head_reduce(float *v, int lane)
{
    if constexpr (N == 1) {
        const float r = __shfl_xor_sync(0xFFFFFFFFu, v[0], O);
        v[0] = Max ? fmaxf(v[0], r) : v[0] + r;
    } else {
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const float lo = v[j], hi = v[j + N / 2];
            const float r = __shfl_xor_sync(0xFFFFFFFFu, up ? lo : hi, O);
            const float k = up ? hi : lo;
            v[j] = Max ? fmaxf(k, r) : k + r;
        }
    }
    if constexpr (O > 1) head_reduce<(N > 1 ? N / 2 : 1), O / 2, Max>(v, lane);
}

// Stores this lane's share of a per-head warp reduction into dst[head]: for
// N < 32 the 32 / N lanes that hold a head's value are consecutive, and the
// first of them stores it.
template <int N>
__device__ __forceinline__ void store_reduced(float *dst, const float *v, int lane)
{
    if constexpr (N >= 32) {
#pragma unroll
        for (int j = 0; j < N / 32; ++j) dst[lane * (N / 32) + j] = v[j];
    } else {
        constexpr int kLanes = 32 / N;
        if (lane % kLanes == 0) dst[lane / kLanes] = v[0];
    }
}

// 32 lanes x NH consecutive 32-bit columns of tensor memory into r[0..NH).
template <int NH>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[NH])
{
#pragma unroll
    for (int c = 0; c < NH; c += 16) tmem_ld16(taddr + c, *reinterpret_cast<uint32_t(*)[16]>(&r[c]));
}

template <int NH>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&r)[NH])
{
#pragma unroll
    for (int c = 0; c < NH; c += 16) tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(&r[c]));
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1) attend_decode_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap pmap, DecArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int D = a.c.D, H = a.H;
    uint8_t *q_s = base;                           // [64 heads][D] fp16, K-major SW128 (64-dim blocks of 64 rows)
    uint8_t *v_s = q_s + kMaxHeads * D * 2;        // [128 rows][D] fp16, K-major SW128 (64-dim blocks of 128 rows)
    uint8_t *p_s = v_s + kTRows * D * 2;           // [NH heads][128 rows] fp16, K-major SW128 (two 64-row blocks)
    DecSmem &sm = *reinterpret_cast<DecSmem *>(p_s + NH * kTRows * 2);
    volatile int *abort_flag = &sm.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.y, split = blockIdx.x;  // the nsplit CTAs of a query form one cluster
    const int b = unit / a.P;

    if (tid == 0) {
        mbar_init(&sm.vfull, kWorkers);
        mbar_init(&sm.vempty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], kWorkers);
        }
        mbar_init(&sm.pfull, kWorkers);
        mbar_init(&sm.pempty, 1);
        mbar_init(&sm.done, 1);
        mbar_init(&sm.qbar, 1);
        mbar_init(&sm.rbar, 1);
        sm.abort = 0;
        sm.flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&qmap);
        if (a.nsplit > 1) prefetch_tensormap(&pmap);
    }
    if (tid < kMaxHeads) {
        sm.m_run[tid] = -INFINITY;
        sm.l_run[tid] = 0.f;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    __syncthreads();

    // The query block [64 head rows][D] bf16 arrives by TMA (128-byte swizzled
    // 64-dim boxes) in the V buffer, which is free until the first gather.  The
    // query is an input of the step, fetched before the wait on the previous
    // kernel; the first 256 threads convert it to fp16 * 2^e per head.
    uint8_t *q_stage = v_s;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.qbar, static_cast<uint32_t>(kMaxHeads * D * 2));
        for (int kb = 0; kb < D / 64; ++kb)
            tma_load_2d(q_stage + kb * kMaxHeads * 128, &qmap, &sm.qbar, kb * 128, unit * H);
    }
    if (tid < 4 * kMaxHeads && mbar_wait(&sm.qbar, 0, abort_flag)) {
        // thread = (head qh, quarter qq of the dims); lane = 8 * quarter + head % 8
        const int qh = warp * 8 + (lane & 7), qq = lane >> 3, qn = D / 32;
        const uint32_t qst = smem_u32(q_stage), qs = smem_u32(q_s);
        auto chunk = [&](int i) -> uint4 {
            const int dim = qq * (D / 4) + i * 8;
            const int kb = dim >> 6, c = (dim >> 3) & 7;
            return ld_shared_v4(qst + kb * kMaxHeads * 128 + qh * 128 + ((c ^ (qh & 7)) << 4));
        };
        constexpr uint32_t kExp = 0x7F807F80u;  // exponent fields of two bf16
        uint32_t m4[4] = {0u, 0u, 0u, 0u};
        if (qh < H) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i < qn) {
                    const uint4 v = chunk(i);
                    m4[i & 3] = __vmaxu2(m4[i & 3], __vmaxu2(__vmaxu2(v.x & kExp, v.y & kExp), __vmaxu2(v.z & kExp, v.w & kExp)));
                }
        }
        const uint32_t m2 = __vmaxu2(__vmaxu2(m4[0], m4[1]), __vmaxu2(m4[2], m4[3]));
        uint32_t emax = max((m2 >> 7) & 0xFFu, m2 >> 23);
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 8));
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 16));
        // max|q| * 2^e < 2^15: no fp16 overflow in Q, and Q.v stays finite in fp32
        const float e = emax > 0 ? 14.f - (static_cast<float>(emax) - 127.f) : 0.f;
        const float qscale = exp2f(e);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < qn)
                st_shared_v4(qs + sw128_off(qh, qq * (D / 4) + i * 8, kMaxHeads),
                             qh < H ? bf16x8_to_f16x8(chunk(i), qscale) : make_uint4(0, 0, 0, 0));
        if (qq == 0) sm.cf[qh] = a.scale * kLog2e * exp2f(-e);
    }
    // Below: reads of what earlier kernels on the stream wrote (lengths, indices, cache).
    pdl_wait();
    pdl_trigger();
    const int len = min(a.c.lengths[b], a.c.cap);
    const int ntile_all = (a.K + kTRows - 1) / kTRows;
    const int t_first = split * a.tiles_per_split;
    const int n_tiles = max(0, min(ntile_all, t_first + a.tiles_per_split) - t_first);
    const int32_t *irow = a.idx + static_cast<int64_t>(unit) * a.K;

    // Gather-warp state: thread (row gr, half gp) holds D/2 channels of one FP4
    // row of the next tile: D/64 16-byte code pieces and D/128 scale words.
    const bool is_worker = warp < kMmaWarp;
    const int gr = tid & (kTRows - 1), gp = tid >> 7;  // worker: row and half of it
    const int npc = D / 64;
    int32_t nrow = -1;
    uint4 pc[8];
    uint32_t ps[4];
    auto fetch = [&](int tile) {
        const int j = (t_first + tile) * kTRows + gr;
        int32_t row = j < a.K ? __ldg(irow + j) : -1;
        if (row >= len) {
            if (gp == 0) raise_status(a.status, CSA_DEV_BAD_INDEX);
            row = -1;
        }
        nrow = row;
        const int64_t g = static_cast<int64_t>(b) * a.c.cap + (row >= 0 ? row : 0);
        const uint4 *cp = reinterpret_cast<const uint4 *>(a.c.codes + g * (D / 2)) + gp * npc;
        const uint32_t *sp = reinterpret_cast<const uint32_t *>(a.c.scales + g * (D / 16)) + gp * (D / 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) pc[i] = (row >= 0 && i < npc) ? __ldg(cp + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) ps[i] = (row >= 0 && i < D / 128) ? __ldg(sp + i) : 0u;
    };
    if (is_worker && n_tiles > 0) fetch(0);

    fence_async_smem();  // the fp16 Q written above is read by the tensor core
    tc_fence_before();
    __syncthreads();     // Q converted (its staging area is free), tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t t_s = tmem;            // S^T: 2 buffers x NH columns
    const uint32_t t_o = tmem + 2 * NH;   // O^T: D/128 chunks x NH columns

    if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA thread
        if (lane == 0 && n_tiles > 0) {
            const uint32_t idesc_s = instr_desc(128, NH, 0, 0, 0, 0);  // V and Q both K-major
            const uint32_t idesc_o = instr_desc(128, NH, 0, 0, 1, 0);  // V^T MN-major, P K-major
            const uint64_t dq = smem_desc(smem_u32(q_s), 16, 1024, 2);
            const uint64_t dv = smem_desc(smem_u32(v_s), 16, 1024, 2);
            const uint64_t dvt = smem_desc(smem_u32(v_s), kTRows * 128 /*next 64 dims*/, 1024 /*next 8 rows*/, 2);
            const uint64_t dp = smem_desc(smem_u32(p_s), 16, 1024, 2);
            for (int i = 0; i < n_tiles; ++i) {
                if (!mbar_wait(&sm.vfull, i & 1, abort_flag)) break;
                if (!mbar_wait(&sm.sempty[i & 1], ((i >> 1) & 1) ^ 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t ts = t_s + (i & 1) * NH;
                for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(ts, dv + ((kb * kTRows * 128 + ks * 32) >> 4), dq + ((kb * kMaxHeads * 128 + ks * 32) >> 4),
                                idesc_s, (kb > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&sm.sfull[i & 1]);
                // O^T += V^T . P^T with P in two fp16 parts that the softmax
                // writes one after the other into the one P buffer: its high
                // part (phase 2i of pfull/pempty), then the remainder (2i + 1).
                bool ok = true;
                for (int part = 0; part < 2 && ok; ++part) {
                    if (!(ok = mbar_wait(&sm.pfull, part, abort_flag))) break;
                    tc_fence_after();
                    for (int mt = 0; mt < D / 128; ++mt)
#pragma unroll
                        for (int ks = 0; ks < kTRows / 16; ++ks)
                            mma_f16(t_o + mt * NH, dvt + ((2 * mt * kTRows * 128 + ks * 2048) >> 4),
                                    dp + ((((ks >> 2) * NH * 128) + (ks & 3) * 32) >> 4), idesc_o,
                                    (i > 0 || part > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&sm.pempty);
                }
                if (!ok) break;
                mma_commit(&sm.vempty);
            }
            mma_commit(&sm.done);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ worker warps
        const bool gath = true, soft = true;
        const int sq = warp & 3, shalf = warp >> 2;  // softmax: lane quarter (rows) and head half
        constexpr int HS = NH / 2;                    // heads per softmax thread
        const uint32_t lane_off = static_cast<uint32_t>(sq * 32) << 16;
        const int r = sq * 32 + lane, rr = r & 63;
        const uint32_t pb = smem_u32(p_s) + (r >> 6) * NH * 128;  // the P block of this row
        const uint32_t vb = smem_u32(v_s);
        bool ok = true;
        for (int i = 0; i < n_tiles; ++i) {
            if (gath) {
                ok = ok && mbar_wait(&sm.vempty, (i & 1) ^ 1, abort_flag);
                const unsigned vbits = __ballot_sync(0xFFFFFFFFu, nrow >= 0);
                if (gp == 0 && lane == 0) sm.valid[gr >> 5] = vbits;
                if (ok) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (k >= npc) break;
                        const uint32_t sw = ps[k >> 1] >> (16 * (k & 1));  // scales of this piece's two 16-channel groups
                        const uint32_t s0 = e4m3_to_h2(sw & 0xFF), s1 = e4m3_to_h2((sw >> 8) & 0xFF);
                        const uint32_t words[4] = {pc[k].x, pc[k].y, pc[k].z, pc[k].w};
                        const int ch0 = gp * (D / 2) + k * 32;
#pragma unroll
                        for (int h8 = 0; h8 < 4; ++h8) {
                            const uint32_t sv = h8 < 2 ? s0 : s1;
                            const uint32_t wd = words[h8];
                            uint4 o;
                            o.x = dequant_pair(wd & 0xFF, sv);
                            o.y = dequant_pair((wd >> 8) & 0xFF, sv);
                            o.z = dequant_pair((wd >> 16) & 0xFF, sv);
                            o.w = dequant_pair(wd >> 24, sv);
                            st_shared_v4(vb + sw128_off(gr, ch0 + h8 * 8, kTRows), o);
                        }
                    }
                }
                fence_async_smem();
                mbar_arrive(&sm.vfull);
            }
            if (soft) {
                // Thread = tile row r (tensor-memory lane r of S^T) and half of
                // the heads.  The eight warps meet at a named barrier twice per
                // tile; every warp runs every tile and every barrier (a wait
                // that ran out only skips the work), so none is left alone.
                ok = ok && mbar_wait(&sm.sfull[i & 1], (i >> 1) & 1, abort_flag) && mbar_wait(&sm.vfull, i & 1, abort_flag);
                tc_fence_after();
                const uint32_t ts = t_s + (i & 1) * NH + shalf * HS + lane_off;
                const bool valid = ok && ((sm.valid[sq] >> lane) & 1u);
                {
                    // per-head maximum of the tile's raw logits (cf > 0 is applied after)
                    uint32_t z[HS];
                    tmem_ld_row<HS>(ts, z);
                    tmem_ld_wait();
                    float x[HS];
#pragma unroll
                    for (int h = 0; h < HS; ++h) x[h] = valid ? __uint_as_float(z[h]) : -INFINITY;
                    head_reduce<HS, 16, true>(x, lane);
                    store_reduced<HS>(sm.redm[sq] + shalf * HS, x, lane);
                }
                named_barrier_sync(1, kWorkers);
                if (tid < NH) {
                    // the previous tile's sum, then this tile's running maximum (log2 units)
                    if (i > 0)
                        sm.l_run[tid] = sm.l_run[tid] * sm.fac[tid] +
                                        ((sm.reds[0][tid] + sm.reds[1][tid]) + (sm.reds[2][tid] + sm.reds[3][tid]));
                    const float zmax = fmaxf(fmaxf(sm.redm[0][tid], sm.redm[1][tid]), fmaxf(sm.redm[2][tid], sm.redm[3][tid]));
                    const float tmax = zmax * sm.cf[tid];
                    const float mo = sm.m_run[tid];
                    float f = 1.f;
                    if (tmax > -INFINITY && (mo == -INFINITY || tmax > mo + kRescaleLog2)) {
                        f = mo == -INFINITY ? 0.f : fast_exp2(mo - tmax);
                        sm.m_run[tid] = tmax;
                    }
                    sm.fac[tid] = f;
                    if (i > 0 && f != 1.f) sm.flag = i + 1;
                }
                named_barrier_sync(1, kWorkers);
                // P of this row as two fp16 parts, p = hi + lo: hi keeps p's
                // leading 11 significant bits (exact in fp16 for p >= 2^-14),
                // lo is the exact fp32 remainder rounded to fp16, so P.V keeps
                // about 22 bits of P (one fp16 P would err by 2^-12 of each
                // weight, which the output's outlier channels magnify past the
                // tolerance).  The per-head sums use P in fp32.  The last PV of
                // the previous tile has completed before P and O^T are touched
                // (phase 2i - 1 of pempty).
                ok = ok && mbar_wait(&sm.pempty, 1, abort_flag);
                tc_fence_after();
                if (ok && sm.flag == i + 1) {
                    // Rescale O^T: this thread's dim of every 128-dim chunk, its heads.
                    for (int mt = 0; mt < D / 128; ++mt) {
                        uint32_t o[HS];
                        const uint32_t ta = t_o + mt * NH + shalf * HS + lane_off;
                        tmem_ld_row<HS>(ta, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int h = 0; h < HS; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * sm.fac[shalf * HS + h]);
                        tmem_st_row<HS>(ta, o);
                    }
                    tmem_st_wait();
                }
                uint32_t lo2[HS / 2];
                {
                    uint32_t z[HS];
                    tmem_ld_row<HS>(ts, z);
                    tmem_ld_wait();
                    float p[HS];
#pragma unroll
                    for (int j = 0; j < HS; j += 2) {
                        const int h = shalf * HS + j, h1 = h + 1;
                        const float p0 = valid ? fast_exp2(fmaf(__uint_as_float(z[j]), sm.cf[h], -sm.m_run[h])) : 0.f;
                        const float p1 = valid ? fast_exp2(fmaf(__uint_as_float(z[j + 1]), sm.cf[h1], -sm.m_run[h1])) : 0.f;
                        const float hi0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
                        const float hi1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
                        const __half2 h2 = __floats2half2_rn(hi0, hi1), l2 = __floats2half2_rn(p0 - hi0, p1 - hi1);
                        const uint32_t hw = *reinterpret_cast<const uint32_t *>(&h2);
                        lo2[j / 2] = *reinterpret_cast<const uint32_t *>(&l2);
                        if (ok) {
                            st_shared_b16(pb + (h >> 3) * 1024 + (h & 7) * 128 + (((rr >> 3) ^ (h & 7)) << 4) + (rr & 7) * 2,
                                          static_cast<uint16_t>(hw & 0xFFFFu));
                            st_shared_b16(pb + (h1 >> 3) * 1024 + (h1 & 7) * 128 + (((rr >> 3) ^ (h1 & 7)) << 4) + (rr & 7) * 2,
                                          static_cast<uint16_t>(hw >> 16));
                        }
                        p[j] = p0;
                        p[j + 1] = p1;
                    }
                    head_reduce<HS, 16, false>(p, lane);
                    store_reduced<HS>(sm.reds[sq] + shalf * HS, p, lane);
                }
                tc_fence_before();
                mbar_arrive(&sm.sempty[i & 1]);
                fence_async_smem();
                mbar_arrive(&sm.pfull);  // the high part
                // the remainder, once the high part's MMAs have read the buffer
                ok = ok && mbar_wait(&sm.pempty, 0, abort_flag);
                if (ok) {
#pragma unroll
                    for (int j = 0; j < HS; j += 2) {
                        const int h = shalf * HS + j, h1 = h + 1;
                        st_shared_b16(pb + (h >> 3) * 1024 + (h & 7) * 128 + (((rr >> 3) ^ (h & 7)) << 4) + (rr & 7) * 2,
                                      static_cast<uint16_t>(lo2[j / 2] & 0xFFFFu));
                        st_shared_b16(pb + (h1 >> 3) * 1024 + (h1 & 7) * 128 + (((rr >> 3) ^ (h1 & 7)) << 4) + (rr & 7) * 2,
                                      static_cast<uint16_t>(lo2[j / 2] >> 16));
                    }
                }
                fence_async_smem();
                mbar_arrive(&sm.pfull);  // the remainder
                if (gath && i + 1 < n_tiles) fetch(i + 1);
            }
        }
        if (soft) {
            // the last tile's sum
            named_barrier_sync(1, kWorkers);
            if (tid < NH && n_tiles > 0)
                sm.l_run[tid] = sm.l_run[tid] * sm.fac[tid] + ((sm.reds[0][tid] + sm.reds[1][tid]) + (sm.reds[2][tid] + sm.reds[3][tid]));
            // the last O^T update is complete before the epilogue reads it
            if (ok && n_tiles > 0) {
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(&sm.done, 0)) {
                    if (*abort_flag) break;
                    if (global_ns() - t0 > kWaitLimitNs) {
                        *abort_flag = 1;
                        break;
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ epilogue
    tc_fence_before();
    __syncthreads();  // final (m, l) per head in shared memory; O^T complete in tensor memory
    tc_fence_after();
    const bool live = !*abort_flag && n_tiles > 0;
    // O^T leaves tensor memory through the eight worker warps into stage
    // [H][D] fp32 over the V buffer (free once the last PV is done): warp w
    // reads lane quarter w % 4 (32 dims of each 128-dim chunk), the two warps
    // of a quarter take alternate (chunk, 16 heads) items, four items' loads
    // in flight at once; lane = dim, so the stores are conflict-free.  One
    // bulk copy then moves the whole block to global memory.
    float *stage = reinterpret_cast<float *>(v_s);
    const bool single = a.nsplit == 1;
    if (live && warp < kMmaWarp) {
        const int q4 = warp & 3, g = warp >> 2;
        const uint32_t loff = static_cast<uint32_t>(q4 * 32) << 16;
        const int nc16 = NH / 16, items = (D / 128) * nc16;
        constexpr int kIt = 4;
        for (int it0 = g; it0 < items; it0 += 2 * kIt) {
            uint32_t r16[kIt][16];
#pragma unroll
            for (int u = 0; u < kIt; ++u) {
                const int it = it0 + 2 * u;
                if (it < items) {
                    const int mt = it / nc16, c0 = (it - mt * nc16) * 16;
                    tmem_ld16(t_o + mt * NH + loff + c0, r16[u]);
                }
            }
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < kIt; ++u) {
                const int it = it0 + 2 * u;
                if (it >= items) break;
                const int mt = it / nc16, c0 = (it - mt * nc16) * 16;
                const int d = mt * 128 + q4 * 32 + lane;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int h = c0 + k;
                    if (h >= H) break;
                    float v = __uint_as_float(r16[u][k]);
                    if (single) {
                        const float l = sm.l_run[h];
                        v = l > 0.f ? v / l : 0.f;
                    }
                    stage[h * D + d] = v;
                }
            }
        }
    }
    fence_async_smem();
    __syncthreads();
    const uint32_t block_bytes = static_cast<uint32_t>(H * D * 4);
    if (single) {
        if (tid == 0 && live) {
            bulk_store(a.out + static_cast<int64_t>(unit) * H * D, smem_u32(stage), block_bytes);
            bulk_commit();
            bulk_wait_all();
        }
        if (tid < H && a.lse) {
            const float l = live ? sm.l_run[tid] : 0.f;
            a.lse[static_cast<int64_t>(unit) * H + tid] = l > 0.f ? (sm.m_run[tid] + log2f(l)) * kLn2 : -INFINITY;
        }
    } else {
        // Split merge through the workspace: every split stores its
        // unnormalised O [H][D] and its (m, l) per head; after one cluster
        // barrier (the splits of a query run at once, as one cluster) split r
        // fetches dims [r*S, (r+1)*S) of every head from every split by TMA
        // and combines them with the log-sum-exp weights.
        const int C = a.nsplit;
        const int rank = split;  // x is the cluster dimension: rank = blockIdx.x
        const int S = D / C;
        const int64_t pbase = static_cast<int64_t>(unit) * C;
        if (tid == 0 && live) {
            bulk_store(a.part_o + (pbase + rank) * H * D, smem_u32(stage), block_bytes);
            bulk_commit();
            bulk_wait_all();
            fence_proxy_async_global();
        }
        if (tid < H)
            __stcg(a.part_ml + (pbase + rank) * H + tid,
                   live ? make_float2(sm.m_run[tid], sm.l_run[tid]) : make_float2(-INFINITY, 0.f));
        __threadfence();
        cluster_sync_all();  // every split's partial is in the workspace
        if (tid == 0) {
            // slice q of every split -> stage[q][H][S] (the stage was read out above)
            mbar_arrive_expect_tx(&sm.rbar, static_cast<uint32_t>(C * H * S * 4));
            for (int q = 0; q < C; ++q)
                tma_load_2d(stage + q * H * S, &pmap, &sm.rbar, rank * S, static_cast<int>((pbase + q) * H));
        }
        if (tid < H) {
            // the merge weights of this head over the splits (while the slices arrive)
            float2 ml[kMaxSplit];
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
                ml[q] = q < C ? __ldcg(a.part_ml + (pbase + q) * H + tid) : make_float2(-INFINITY, 0.f);
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
                if (ml[q].y > 0.f) M = fmaxf(M, ml[q].x);
            float L = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q) {
                ml[q].x = ml[q].y > 0.f ? exp2f(ml[q].x - M) : 0.f;
                L = fmaf(ml[q].x, ml[q].y, L);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
                if (q < C) sm.wq[q][tid] = ml[q].x * inv;
            if (rank == 0 && a.lse) a.lse[static_cast<int64_t>(unit) * H + tid] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        const bool got = mbar_wait(&sm.rbar, 0, abort_flag);
        __syncthreads();  // the weights are in shared memory
        if (got && !*abort_flag) {
            const int nd4 = S / 4;
            for (int it = tid; it < H * nd4; it += kThreads) {
                const int h = it / nd4, d4 = it - h * nd4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < kMaxSplit; ++q) {
                    if (q >= C) break;
                    const float wgt = sm.wq[q][h];
                    if (wgt == 0.f) continue;  // a split without rows wrote no O
                    const float4 v = *reinterpret_cast<const float4 *>(stage + (q * H + h) * S + 4 * d4);
                    acc.x = fmaf(wgt, v.x, acc.x);
                    acc.y = fmaf(wgt, v.y, acc.y);
                    acc.z = fmaf(wgt, v.z, acc.z);
                    acc.w = fmaf(wgt, v.w, acc.w);
                }
                *reinterpret_cast<float4 *>(a.out + (static_cast<int64_t>(unit) * H + h) * D + rank * S + 4 * d4) = acc;
            }
        }
    }
    if (*abort_flag && tid == 0) raise_status(a.status, CSA_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

size_t decode_smem_bytes(int D, int NH)
{
    return 1024 + static_cast<size_t>(kMaxHeads) * D * 2 + static_cast<size_t>(kTRows) * D * 2 +
           static_cast<size_t>(NH) * kTRows * 2 + sizeof(DecSmem);
}

int heads_tile(int H) { return H <= 16 ? 16 : (H <= 32 ? 32 : 64); }

// The kernel's shared-memory limit is set once, to the largest request any
// call can make (D = 512).
template <int NH>
cudaError_t configure()
{
    static bool done = false;
    if (done) return cudaSuccess;
    size_t smem = decode_smem_bytes(512, NH);
    if (smem < 120 * 1024) smem = 120 * 1024;
    cudaError_t e = cudaFuncSetAttribute(attend_decode_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attend_decode_kernel<NH>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    done = e == cudaSuccess;
    return e;
}

// Clusters of `ns` CTAs of this kernel that the device can hold at once
// (queried once per cluster size and shared-memory size).
template <int NH>
int active_clusters(int ns, size_t smem)
{
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, int> known;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(ns, smem);
    const auto it = known.find(key);
    if (it != known.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(ns);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attend_decode_kernel<NH>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    known[key] = n;
    return n;
}

}  // namespace

// The few-query path takes every query whose splits fit one wave of CTAs (one
// per SM): at most one CTA per SM per query, and units <= SMs.
int decode_supported(const CacheView &c, int P, int H, int K)
{
    const int units = c.B * P;
    return units >= 1 && units <= sm_count() && H >= 1 && H <= kMaxHeads && K >= 1 && c.D % 128 == 0 && c.D <= 512;
}

// The most splits per query: a power of two, at most 16, at most one per tile,
// D / splits >= 8, and every query's splits within one wave of CTAs.  The
// launch takes fewer when the device cannot hold that many clusters at once.
static int max_splits(const CacheView &c, int P, int K)
{
    const int units = c.B * P;
    const int tiles = (K + kTRows - 1) / kTRows;
    int ns = kMaxSplit;
    while (ns > 1 && (ns > tiles || c.D / ns < 8 || static_cast<int64_t>(units) * ns > sm_count())) ns /= 2;
    return ns;
}

static size_t part_o_bytes(const CacheView &c, int P, int H, int ns)
{
    const size_t o = static_cast<size_t>(c.B) * P * ns * H * c.D * sizeof(float);
    return (o + 255) / 256 * 256;
}

size_t decode_workspace_bytes(const CacheView &c, int P, int H, int K)
{
    const int ns = max_splits(c, P, K);
    if (ns == 1) return 0;
    return part_o_bytes(c, P, H, ns) + static_cast<size_t>(c.B) * P * ns * H * sizeof(float2);
}

cudaError_t launch_attend_decode(const CacheView &c, int P, int H, const uint16_t *q, float scale,
                                 const int32_t *idx, int K, float *out, float *lse, void *ws, size_t ws_bytes,
                                 int *status, cudaStream_t st)
{
    const int units = c.B * P;
    if (!decode_supported(c, P, H, K)) return cudaErrorInvalidValue;
    if (ws_bytes < decode_workspace_bytes(c, P, H, K)) return cudaErrorInvalidValue;
    const int NH = heads_tile(H);
    // Tensor memory: S^T (two buffers) and O^T, NH columns each per 128 dims.
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>((2 + c.D / 128) * NH)) cols *= 2;
    // CTAs that share an SM must fit their tensor memory together (an
    // allocation waits for free columns): with more than half of it, ask for
    // enough shared memory that a second CTA cannot be resident.
    size_t smem = decode_smem_bytes(c.D, NH);
    if (cols > 256 && smem < 120 * 1024) smem = 120 * 1024;
    cudaError_t e = NH == 16 ? configure<16>() : (NH == 32 ? configure<32>() : configure<64>());
    if (e != cudaSuccess) return e;
    const int tiles = (K + kTRows - 1) / kTRows;
    // Splits per query: the most (max_splits) whose clusters the device holds at once.
    int ns = max_splits(c, P, K);
    while (ns > 1) {
        const int fit = NH == 16 ? active_clusters<16>(ns, smem)
                                 : (NH == 32 ? active_clusters<32>(ns, smem) : active_clusters<64>(ns, smem));
        if (fit >= units) break;
        ns /= 2;
    }
    DecArgs a{};
    a.c = c;
    a.P = P;
    a.H = H;
    a.K = K;
    a.scale = scale;
    a.idx = idx;
    a.nsplit = ns;
    a.tiles_per_split = (tiles + ns - 1) / ns;
    a.part_o = static_cast<float *>(ws);
    a.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + part_o_bytes(c, P, H, ns));
    a.out = out;
    a.lse = lse;
    a.tmem_cols = cols;
    a.status = status;
    // Query rows [units*H][D] bf16 as bytes: 64-dim (128-byte) boxes of 64 rows.
    CUtensorMap qm;
    if (encode_tensor_map_2d_u8(&qm, q, static_cast<uint64_t>(c.D) * 2, static_cast<uint64_t>(units) * H, 128,
                                kMaxHeads, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // Split partials [units * ns * H rows][D] fp32, fetched in boxes of
    // D / ns dims x H heads (one split's slice).
    CUtensorMap pm = qm;
    if (ns > 1 && encode_tensor_map_2d_f32(&pm, ws, static_cast<uint64_t>(c.D), static_cast<uint64_t>(units) * ns * H,
                                           static_cast<uint32_t>(c.D / ns), static_cast<uint32_t>(H)) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int cl = ns > 1 ? ns : 0;
    if (NH == 16)
        return launch_kernel(attend_decode_kernel<16>, dim3(ns, units), dim3(kThreads), smem, st, cl, qm, pm, a);
    if (NH == 32)
        return launch_kernel(attend_decode_kernel<32>, dim3(ns, units), dim3(kThreads), smem, st, cl, qm, pm, a);
    return launch_kernel(attend_decode_kernel<64>, dim3(ns, units), dim3(kThreads), smem, st, cl, qm, pm, a);
}

}  // namespace csa
