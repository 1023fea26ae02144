// a5/a6: sparse attention of each query over its selected FP4 rows, on the
// tcgen05 tensor cores, split over the selection (flash-decode) with a merge pass.
// "G2C Brief - DeepSeek V4.1-Flash", section "The global branch: compress,
// index, select": the query attends to only the selected entries; one shared
// latent per entry serves every query head.  "DeepSeek V4.1 Flash: Pushing
// the Limits", section "The Paper": a single W_KV, so keys and values are the
// same vector.
//
// One CTA = one (sequence, position) query and a contiguous share of its
// selection, in tiles of 128 selected rows.  Per tile:
//   1. each thread gathers one selected FP4 row (D/2 code bytes + D/16 scale
//      bytes) and dequantises it to fp16 in registers (E2M1 x E4M3 is exact in
//      fp16) into a K-major 128B-swizzled tile V[128 rows][D];
//   2. S^T = V . Q^T on the tensor cores (M = 128 rows, N = heads, K = D), with
//      Q staged 256 dims at a time as fp16 scaled per head by a power of two
//      (exact for bf16 queries, and safe from fp16 overflow);
//   3. S^T goes through shared memory so that each thread owns one head's
//      logits; softmax statistics with a lazily rescaled running maximum;
//   4. O^T += V^T . P^T with P split into fp16 high and low parts (two MMAs
//      into the same fp32 accumulator), which keeps P's precision near fp32.
//      V^T is read from the same tile through an MN-major descriptor.
// The accumulator O^T [D x heads] stays in tensor memory across the CTA's tiles;
// at the end the CTA writes either the final output (one split) or a partial
// (O, m, l) that the merge kernel combines.
#include <cuda_fp16.h>

#include "common.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kRows = 128;         // selected rows per tile (MMA M for S^T)
constexpr int kThreads = 256;      // 8 warps: two per tensor-memory lane quarter
constexpr int kMaxHeads = 64;
constexpr float kRescaleLog2 = 8.f;  // rescale only when the running max grows by more than 2^8
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttArgs {
    CacheView c;
    int P, H, K;
    int NH;           // heads rounded up to 16 (MMA N)
    const uint16_t *q;
    float scale;
    const int32_t *idx;
    int nsplit, tiles_per_split, tiles_total;
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

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi)
{
    return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
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
        r4[k] = pack_half2(__float2half_rn(lo), __float2half_rn(hi));
    }
    return make_uint4(r4[0], r4[1], r4[2], r4[3]);
}

// Every thread waits for the MMAs committed to `bar`; the verdict is read after a
// CTA barrier so that all threads agree on it even if one wait ran out.
__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, volatile int *abort_flag)
{
    mbar_wait(bar, phase, abort_flag);
    phase ^= 1;
    __syncthreads();
    tc_fence_after();
    return *abort_flag == 0;
}

__global__ void __launch_bounds__(kThreads, 1) attend_kernel(AttArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int D = a.c.D, NH = a.NH, H = a.H;
    const int v_bytes = kRows * D * 2;
    const int qh_bytes = NH * 256 * 2;        // one 256-dim chunk of Q
    const int sst_bytes = kRows * (NH + 1) * 4;
    const int qs_bytes = qh_bytes > sst_bytes ? qh_bytes : sst_bytes;
    const int p_bytes = NH * kRows * 2;
    uint8_t *v_s = base;
    uint8_t *q_s = v_s + v_bytes;                               // Q chunk, then S^T staging
    uint8_t *p_hi = q_s + ((qs_bytes + 1023) & ~1023);
    uint8_t *p_lo = p_hi + p_bytes;
    float *st = reinterpret_cast<float *>(p_lo + p_bytes);     // per-head state
    float *m_run = st;                 // running max (log2 units)
    float *l_run = m_run + kMaxHeads;  // running sum
    float *fac = l_run + kMaxHeads;    // rescale factor this tile
    float *cfac = fac + kMaxHeads;     // scale * log2(e) * 2^-e (e: power of two applied to Q)
    uint32_t *valid = reinterpret_cast<uint32_t *>(cfac + kMaxHeads);  // [kRows/32] bit masks
    uint64_t *mma_bar = reinterpret_cast<uint64_t *>(valid + kRows / 32);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_bar + 1);
    int *flags = reinterpret_cast<int *>(tmem_slot + 1);  // [0] rescale needed, [1] abort
    volatile int *abort_flag = flags + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, whalf = warp >> 2;  // tensor-memory lane quarter; column half
    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / a.P;
    const int len = a.c.lengths[b];
    const int t_first = split * a.tiles_per_split;
    const int t_last = min(a.tiles_total, t_first + a.tiles_per_split);
    const int32_t *irow = a.idx + static_cast<int64_t>(unit) * a.K;

    if (tid == 0) {
        mbar_init(mma_bar, 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }

    // The selected rows of a tile are fetched one tile ahead: thread (row r,
    // half rh) holds half of one FP4 row (D/4 code bytes, D/32 scale bytes).
    const int gr = tid & (kRows - 1), grh = tid >> 7;
    const int nc = D / 64;  // 16-byte code pieces per half row (32 channels each)
    int32_t nrow = -1;
    uint4 ncw[8];
    uint32_t nsw[4];
    auto prefetch = [&](int tile) {
        const int j = tile * kRows + gr;
        int32_t row = j < a.K ? irow[j] : -1;
        if (row >= len) {
            raise_status(a.status, CSA_DEV_BAD_INDEX);
            row = -1;
        }
        nrow = row;
        const int64_t g = static_cast<int64_t>(b) * a.c.cap + (row >= 0 ? row : 0);
        const uint4 *cp = reinterpret_cast<const uint4 *>(a.c.codes + g * (D / 2)) + grh * nc;
        const uint32_t *sp = reinterpret_cast<const uint32_t *>(a.c.scales + g * (D / 16)) + grh * (D / 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) ncw[i] = (row >= 0 && i < nc) ? cp[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) nsw[i] = (row >= 0 && i < D / 128) ? sp[i] : 0u;
    };
    if (t_first < t_last) prefetch(t_first);

    // Q lives in registers for the whole CTA, as fp16 scaled per head by a power
    // of two: thread (head qh, quarter qq) holds dims [qq*D/4, (qq+1)*D/4).
    const int qh = tid >> 2, qq = tid & 3;
    const int qn = D / 32;  // 16-byte pieces per thread
    uint4 qreg[16];
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + (static_cast<int64_t>(unit) * H + qh) * D) + qq * qn;
#pragma unroll
        for (int i = 0; i < 16; ++i) qreg[i] = (qh < H && i < qn) ? src[i] : make_uint4(0, 0, 0, 0);
    }
    // Per-head power of two e with max|q| * 2^e < 2^15 (fp16-safe, exact for bf16).
    {
        uint32_t emax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t w4[4] = {qreg[i].x, qreg[i].y, qreg[i].z, qreg[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) emax = max(emax, max((w4[k] >> 7) & 0xFFu, (w4[k] >> 23) & 0xFFu));
        }
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 1));
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 2));
        const float e = emax > 0 ? 14.f - (static_cast<float>(emax) - 127.f) : 0.f;
        const float qscale = exp2f(e);
#pragma unroll
        for (int i = 0; i < 16; ++i) qreg[i] = bf16x8_to_f16x8(qreg[i], qscale);
        if (qq == 0) {
            cfac[qh] = a.scale * kLog2e * exp2f(-e);
            m_run[qh] = -INFINITY;
            l_run[qh] = 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s = tmem;             // S^T: NH columns
    const uint32_t t_o = tmem + NH;        // O^T: (D/128) blocks of NH columns
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t v_base = smem_u32(v_s), q_base = smem_u32(q_s);
    const uint32_t phi_base = smem_u32(p_hi), plo_base = smem_u32(p_lo);
    uint32_t mma_phase = 0;
    bool o_started = false;
    bool ok = true;
    const uint32_t idesc_s = instr_desc(128, NH, 0, 0, 0, 0);   // K-major V, K-major Q
    const uint32_t idesc_o = instr_desc(128, NH, 0, 0, 1, 0);   // MN-major V^T, K-major P

    for (int tile = t_first; tile < t_last && ok; ++tile) {
        // ---- 1. dequantise the prefetched rows into the fp16 tile V
        {
            const unsigned vb = __ballot_sync(0xFFFFFFFFu, nrow >= 0);
            if (grh == 0 && lane == 0) valid[gr >> 5] = vb;
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                if (c16 >= nc) break;
                const uint32_t sc = (nsw[c16 >> 1] >> (16 * (c16 & 1))) & 0xFFFF;  // the 2 scales of 32 channels
                const uint32_t s0 = e4m3_to_h2(sc & 0xFF), s1 = e4m3_to_h2(sc >> 8);
                const uint32_t words[4] = {ncw[c16].x, ncw[c16].y, ncw[c16].z, ncw[c16].w};
                const int ch0 = grh * (D / 2) + c16 * 32;
#pragma unroll
                for (int h8 = 0; h8 < 4; ++h8) {  // 8 channels = 4 code bytes -> one 16-byte chunk
                    const uint32_t sv = h8 < 2 ? s0 : s1;
                    const uint32_t wd = words[h8];
                    uint4 o;
                    o.x = dequant_pair(wd & 0xFF, sv);
                    o.y = dequant_pair((wd >> 8) & 0xFF, sv);
                    o.z = dequant_pair((wd >> 16) & 0xFF, sv);
                    o.w = dequant_pair(wd >> 24, sv);
                    *reinterpret_cast<uint4 *>(v_s + sw128_off(gr, ch0 + h8 * 8, kRows)) = o;
                }
            }
        }
        // ---- 2. S^T = V . Q^T, Q staged in 256-dim chunks from registers
        for (int d0 = 0; d0 < D && ok; d0 += 256) {
            const int dn = min(256, D - d0);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int dim = qq * (D / 4) + i * 8;
                if (i < qn && qh < NH && dim >= d0 && dim < d0 + dn)
                    *reinterpret_cast<uint4 *>(q_s + sw128_off(qh, dim - d0, NH)) = qreg[i];
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                for (int kb = 0; kb < dn / 64; ++kb)
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t da =
                            smem_desc(v_base + ((d0 / 64) + kb) * kRows * 128 + ks * 32, 16, 1024, 2);
                        const uint64_t db = smem_desc(q_base + kb * NH * 128 + ks * 32, 16, 1024, 2);
                        mma_f16(t_s, da, db, idesc_s, (d0 > 0 || kb > 0 || ks > 0) ? 1u : 0u);
                    }
                mma_commit(mma_bar);
            }
            __syncwarp();
            ok = wait_mma(mma_bar, mma_phase, abort_flag);
        }
        if (!ok) break;
        if (tile + 1 < t_last) prefetch(tile + 1);  // in flight during softmax and PV
        // ---- 3. logits via shared memory (thread = row, then thread quad = head)
        float *sst = reinterpret_cast<float *>(q_s);  // [kRows][NH+1]
        {
            const int row = quarter * 32 + lane;
            for (int c0 = whalf * 16; c0 < NH; c0 += 32) {  // 16-column groups alternate between the warp halves
                uint32_t r16[16];
                tmem_ld16(t_s + lane_off + c0, r16);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) sst[row * (NH + 1) + c0 + k] = __uint_as_float(r16[k]);
            }
        }
        __syncthreads();
        {
            const int h = tid >> 2, part = tid & 3;  // 64 heads x 4 parts of 32 rows
            const float cf = h < H ? cfac[h] : 0.f;
            const uint32_t vbits = valid[part];
            float z[32];
#pragma unroll
            for (int k = 0; k < 32; ++k)
                z[k] = (h < H && (vbits >> k & 1)) ? sst[(part * 32 + k) * (NH + 1) + h] * cf : -INFINITY;
            float tmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; ++k) tmax = fmaxf(tmax, z[k]);
            tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 1));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 2));
            float mu = h < kMaxHeads ? m_run[h] : -INFINITY;
            float f = 1.f;
            if (h < H && tmax > -INFINITY && (mu == -INFINITY || tmax > mu + kRescaleLog2)) {
                f = mu == -INFINITY ? 0.f : fast_exp2(mu - tmax);
                mu = tmax;
            }
            float lsum = 0.f;
            if (h < NH) {
#pragma unroll
                for (int k8 = 0; k8 < 4; ++k8) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        __half ph[2], pl[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float zz = z[k8 * 8 + k2 * 2 + e];
                            const float p = (zz > -INFINITY && mu > -INFINITY) ? fast_exp2(zz - mu) : 0.f;
                            lsum += p;
                            ph[e] = __float2half_rn(p);
                            pl[e] = __float2half_rn(p - __half2float(ph[e]));
                        }
                        hw[k2] = pack_half2(ph[0], ph[1]);
                        lw[k2] = pack_half2(pl[0], pl[1]);
                    }
                    const uint32_t off = sw128_off(h, part * 32 + k8 * 8, NH);
                    *reinterpret_cast<uint4 *>(p_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(p_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
            lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
            if (part == 0 && h < kMaxHeads) {
                fac[h] = f;
                if (f != 1.f) flags[0] = 1;
                m_run[h] = mu;
                l_run[h] = l_run[h] * f + lsum;
            }
        }
        __syncthreads();
        // ---- rescale O^T when some head's running max moved by more than 2^8 (rare)
        if (flags[0] && o_started) {
            for (int mt = whalf; mt < D / 128; mt += 2)
                for (int c0 = 0; c0 < NH; c0 += 16) {
                    uint32_t r16[16];
                    const uint32_t ta = t_o + mt * NH + lane_off + c0;
                    tmem_ld16(ta, r16);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k) r16[k] = __float_as_uint(__uint_as_float(r16[k]) * fac[c0 + k]);
                    tmem_st16(ta, r16);
                }
            tmem_st_wait();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) flags[0] = 0;
        // ---- 4. O^T += V^T . P_hi^T + V^T . P_lo^T
        if (tid == 0) {
            tc_fence_after();
            for (int mt = 0; mt < D / 128; ++mt)
                for (int hl = 0; hl < 2; ++hl) {
                    const uint32_t pb = hl ? plo_base : phi_base;
                    for (int ks = 0; ks < kRows / 16; ++ks) {
                        const uint64_t da = smem_desc(v_base + (2 * mt) * kRows * 128 + ks * 2048,
                                                      kRows * 128 /*next 64 dims*/, 1024 /*next 8 rows*/, 2);
                        const uint64_t db = smem_desc(pb + (ks >> 2) * NH * 128 + (ks & 3) * 32, 16, 1024, 2);
                        mma_f16(t_o + mt * NH, da, db, idesc_o, (o_started || hl > 0 || ks > 0) ? 1u : 0u);
                    }
                }
            mma_commit(mma_bar);
        }
        __syncwarp();
        ok = wait_mma(mma_bar, mma_phase, abort_flag);
        o_started = true;
    }

    // ---- the result (one split) or this split's partial (merged by the next kernel)
    if (ok) {
        __syncthreads();
        const bool final_out = a.nsplit == 1;
        float *obase = final_out ? a.out + static_cast<int64_t>(unit) * H * D
                                 : a.part_o + (static_cast<int64_t>(unit) * a.nsplit + split) * H * D;
        for (int mt = whalf; mt < D / 128; mt += 2) {  // thread = one dim of a 128-dim block
            const int d = mt * 128 + quarter * 32 + lane;
            uint32_t r[kMaxHeads];
#pragma unroll
            for (int c0 = 0; c0 < kMaxHeads; c0 += 16)
                if (c0 < NH) tmem_ld16(t_o + mt * NH + lane_off + c0, *reinterpret_cast<uint32_t(*)[16]>(r + c0));
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < kMaxHeads; ++h) {
                if (h >= H) break;
                float v = o_started ? __uint_as_float(r[h]) : 0.f;
                if (final_out) v = l_run[h] > 0.f ? v * __frcp_rn(l_run[h]) : 0.f;
                obase[static_cast<int64_t>(h) * D + d] = v;
            }
        }
        if (tid < H) {
            if (final_out) {
                if (a.lse)
                    a.lse[static_cast<int64_t>(unit) * H + tid] =
                        l_run[tid] > 0.f ? (m_run[tid] + log2f(l_run[tid])) * kLn2 : -INFINITY;
            } else {
                a.part_ml[(static_cast<int64_t>(unit) * a.nsplit + split) * H + tid] =
                    make_float2(m_run[tid], l_run[tid]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) raise_status(a.status, CSA_DEV_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// Combines the split partials: block = (128 dims, head, query); each thread
// loads its dim from every split at once.  out = sum_s 2^(m_s - M) O_s / L,
// L = sum_s 2^(m_s - M) l_s, lse = ln 2 * (M + log2 L).
constexpr int kMaxSplit = 16;

__global__ void __launch_bounds__(128) attend_merge_kernel(int D, int H, int nsplit, const float *__restrict__ part_o,
                                                          const float2 *__restrict__ part_ml, float *__restrict__ out,
                                                          float *__restrict__ lse)
{
    __shared__ float wsh[kMaxSplit];
    __shared__ float inv_l;
    const int d = blockIdx.x * 128 + threadIdx.x, h = blockIdx.y, unit = blockIdx.z;
    float pv[kMaxSplit];
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
        pv[s] = (s < nsplit && d < D) ? part_o[((static_cast<int64_t>(unit) * nsplit + s) * H + h) * D + d] : 0.f;
    if (threadIdx.x < 32) {
        const int s = threadIdx.x;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (s < nsplit) ml = part_ml[(static_cast<int64_t>(unit) * nsplit + s) * H + h];
        float M = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        const float w = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
        float L = w * ml.y;
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        if (s < kMaxSplit) wsh[s] = w;
        if (s == 0) {
            inv_l = L > 0.f ? 1.f / L : 0.f;
            if (lse && blockIdx.x == 0) lse[static_cast<int64_t>(unit) * H + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
    __syncthreads();
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) acc = fmaf(wsh[s], pv[s], acc);
    if (d < D) out[(static_cast<int64_t>(unit) * H + h) * D + d] = acc * inv_l;
}

struct Plan {
    int nsplit, tiles_per_split, tiles_total;
};

// Splits of one query's selection: about one wave of CTAs, at most kMaxSplit.
Plan plan(const CacheView &c, int P, int K)
{
    const int units = c.B * P;
    const int tiles = (K + kRows - 1) / kRows;
    int want = (148 + units - 1) / units;
    if (want > tiles) want = tiles;
    if (want > kMaxSplit) want = kMaxSplit;
    if (want < 1) want = 1;
    Plan p;
    p.tiles_total = tiles;
    p.tiles_per_split = (tiles + want - 1) / want;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    return p;
}

size_t smem_bytes(int D, int NH)
{
    const size_t v = static_cast<size_t>(kRows) * D * 2;
    const size_t qh = static_cast<size_t>(NH) * 256 * 2, sst = static_cast<size_t>(kRows) * (NH + 1) * 4;
    const size_t qs = ((qh > sst ? qh : sst) + 1023) & ~size_t(1023);
    const size_t p = 2 * static_cast<size_t>(NH) * kRows * 2;
    return 1024 + v + qs + p + 4 * kMaxHeads * 4 + kRows * 4 + 64;
}

}  // namespace

size_t attend_workspace_bytes(const CacheView &c, int P, int H, int K)
{
    const Plan p = plan(c, P, K);
    if (p.nsplit == 1) return 0;
    const size_t units = static_cast<size_t>(c.B) * P;
    size_t o = units * p.nsplit * H * c.D * sizeof(float);
    o = (o + 255) / 256 * 256;
    return o + units * p.nsplit * H * sizeof(float2);
}

cudaError_t launch_attend(const CacheView &c, int P, int H, const uint16_t *q, float scale, const int32_t *idx,
                          int K, float *out, float *lse, void *ws, size_t ws_bytes, int *status, cudaStream_t st)
{
    const int units = c.B * P;
    if (units == 0) return cudaSuccess;
    if (H > kMaxHeads || c.D % 128 || c.D > 512) return cudaErrorInvalidValue;
    const Plan p = plan(c, P, K);
    if (ws_bytes < attend_workspace_bytes(c, P, H, K)) return cudaErrorInvalidValue;
    AttArgs a{};
    a.c = c;
    a.P = P;
    a.H = H;
    a.K = K;
    a.NH = (H + 15) / 16 * 16;
    a.q = q;
    a.scale = scale;
    a.idx = idx;
    a.nsplit = p.nsplit;
    a.tiles_per_split = p.tiles_per_split;
    a.tiles_total = p.tiles_total;
    size_t o_bytes = static_cast<size_t>(units) * p.nsplit * H * c.D * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    a.part_o = static_cast<float *>(ws);
    a.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + o_bytes);
    a.out = out;
    a.lse = lse;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(a.NH + (c.D / 128) * a.NH)) cols *= 2;
    a.tmem_cols = cols;
    a.status = status;
    const size_t smem = smem_bytes(c.D, a.NH);
    cudaError_t e =
        cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attend_kernel<<<dim3(p.nsplit, units), kThreads, smem, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
    if (p.nsplit > 1) {
        attend_merge_kernel<<<dim3((c.D + 127) / 128, H, units), 128, 0, st>>>(c.D, H, p.nsplit, a.part_o, a.part_ml,
                                                                               out, lse);
        e = cudaGetLastError();
        if (e == cudaSuccess) count_launch();
    }
    return e;
}

}  // namespace csa
