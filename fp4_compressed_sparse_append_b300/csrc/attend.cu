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
constexpr int kThreads = 128;
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
    float *qexp = fac + kMaxHeads;     // per-head log2 scale applied to Q
    float *cfac = qexp + kMaxHeads;    // scale * log2(e) * 2^-qexp
    int *valid = reinterpret_cast<int *>(cfac + kMaxHeads);  // [kRows]
    uint64_t *mma_bar = reinterpret_cast<uint64_t *>(valid + kRows);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_bar + 1);
    int *flags = reinterpret_cast<int *>(tmem_slot + 1);  // [0] rescale needed, [1] abort
    volatile int *abort_flag = flags + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / a.P;
    const int len = a.c.lengths[b];
    const int t_first = split * a.tiles_per_split;
    const int t_last = min(a.tiles_total, t_first + a.tiles_per_split);

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
    // Per-head power-of-two scale for the fp16 copy of Q (max|q| * 2^e < 2^15),
    // and the softmax factor; two threads per head, 16-byte loads.
    {
        const int h = tid >> 1, half = tid & 1;
        uint32_t emax = 0;
        if (h < H) {
            const uint4 *qh = reinterpret_cast<const uint4 *>(a.q + (static_cast<int64_t>(unit) * H + h) * D) +
                              half * (D / 16);
            uint4 v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = i < D / 16 ? qh[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    emax = max(emax, max((w4[k] >> 7) & 0xFFu, (w4[k] >> 23) & 0xFFu));
            }
        }
        emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, 1));
        if (half == 0 && h < kMaxHeads) {
            const float e = emax > 0 ? 14.f - (static_cast<float>(emax) - 127.f) : 0.f;
            qexp[h] = e;
            cfac[h] = a.scale * kLog2e * exp2f(-e);
            m_run[h] = -INFINITY;
            l_run[h] = 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_s = tmem;             // S^T: NH columns
    const uint32_t t_o = tmem + NH;        // O^T: (D/128) blocks of NH columns
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t v_base = smem_u32(v_s), q_base = smem_u32(q_s);
    const uint32_t phi_base = smem_u32(p_hi), plo_base = smem_u32(p_lo);
    uint32_t mma_phase = 0;
    bool o_started = false;
    bool ok = true;
    const int32_t *irow = a.idx + static_cast<int64_t>(unit) * a.K;
    const uint32_t idesc_s = instr_desc(128, NH, 0, 0, 0, 0);   // K-major V, K-major Q
    const uint32_t idesc_o = instr_desc(128, NH, 0, 0, 1, 0);   // MN-major V^T, K-major P

    for (int tile = t_first; tile < t_last && ok; ++tile) {
        // ---- 1. gather + dequantise one selected row per thread
        {
            const int j = tile * kRows + tid;
            int32_t row = j < a.K ? irow[j] : -1;
            if (row >= len) {
                raise_status(a.status, CSA_DEV_BAD_INDEX);
                row = -1;
            }
            valid[tid] = row >= 0;
            const int64_t g = static_cast<int64_t>(b) * a.c.cap + (row >= 0 ? row : 0);
            const uint4 *cp = reinterpret_cast<const uint4 *>(a.c.codes + g * (D / 2));
            const uint2 *sp = reinterpret_cast<const uint2 *>(a.c.scales + g * (D / 16));
            // Issue every load of the row before using any (up to 288 bytes in flight per thread).
            uint4 cw[16];
            uint2 s8[4];
#pragma unroll
            for (int i = 0; i < 16; ++i) cw[i] = (row >= 0 && i < D / 32) ? cp[i] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 4; ++i) s8[i] = (row >= 0 && i < D / 128) ? sp[i] : make_uint2(0, 0);
#pragma unroll
            for (int c16 = 0; c16 < 16; ++c16) {             // 32 channels per 16 code bytes
                if (c16 >= D / 32) break;
                const uint32_t sw = (c16 >> 1) & 1 ? s8[c16 >> 2].y : s8[c16 >> 2].x;
                const uint32_t sc = (sw >> (16 * (c16 & 1))) & 0xFFFF;  // the two scales of these 32 channels
                const uint32_t s0 = e4m3_to_h2(sc & 0xFF), s1 = e4m3_to_h2(sc >> 8);
                const uint32_t words[4] = {cw[c16].x, cw[c16].y, cw[c16].z, cw[c16].w};
#pragma unroll
                for (int h8 = 0; h8 < 4; ++h8) {             // 8 channels = 4 code bytes -> one 16-B chunk
                    const uint32_t sv = h8 < 2 ? s0 : s1;
                    const uint32_t wd = words[h8];
                    uint4 o;
                    o.x = dequant_pair(wd & 0xFF, sv);
                    o.y = dequant_pair((wd >> 8) & 0xFF, sv);
                    o.z = dequant_pair((wd >> 16) & 0xFF, sv);
                    o.w = dequant_pair(wd >> 24, sv);
                    *reinterpret_cast<uint4 *>(v_s + sw128_off(tid, c16 * 32 + h8 * 8, kRows)) = o;
                }
            }
        }
        // ---- 2. S^T = V . Q^T, Q staged in 256-dim chunks
        for (int d0 = 0; d0 < D && ok; d0 += 256) {
            const int dn = min(256, D - d0);
            // stage Q[:, d0:d0+dn] as fp16 * 2^qexp (thread pairs per head)
            {
                // NH*dn/8 16-byte pieces, at most 16 per thread: load them all, then convert.
                constexpr int kPer = kMaxHeads * 256 / 8 / kThreads;
                const int n_e = NH * (dn / 8);
                uint4 raw8[kPer];
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = tid + i * kThreads;
                    const int h = e / (dn / 8), c8 = e % (dn / 8);
                    raw8[i] = (e < n_e && h < H) ? *reinterpret_cast<const uint4 *>(
                                                       a.q + (static_cast<int64_t>(unit) * H + h) * D + d0 + c8 * 8)
                                                 : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = tid + i * kThreads;
                    if (e >= n_e) break;
                    const int h = e / (dn / 8), c8 = e % (dn / 8);
                    const float sc = h < H ? exp2f(qexp[h]) : 0.f;
                    const uint32_t w4[4] = {raw8[i].x, raw8[i].y, raw8[i].z, raw8[i].w};
                    uint32_t r4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = __uint_as_float(w4[k] << 16) * sc;
                        const float hi = __uint_as_float(w4[k] & 0xFFFF0000u) * sc;
                        r4[k] = pack_half2(__float2half_rn(lo), __float2half_rn(hi));
                    }
                    *reinterpret_cast<uint4 *>(q_s + sw128_off(h, c8 * 8, NH)) = make_uint4(r4[0], r4[1], r4[2], r4[3]);
                }
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
            ok = mbar_wait(mma_bar, mma_phase, abort_flag);
            mma_phase ^= 1;
            tc_fence_after();
        }
        if (!ok) break;
        // ---- 3. logits through shared memory: thread = row -> thread pair = head
        float *sst = reinterpret_cast<float *>(q_s);  // [kRows][NH+1]
        for (int c0 = 0; c0 < NH; c0 += 16) {
            uint32_t r[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                  "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                  "=r"(r[14]), "=r"(r[15])
                : "r"(t_s + lane_off + c0));
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 16; ++k) sst[tid * (NH + 1) + c0 + k] = __uint_as_float(r[k]);
        }
        __syncthreads();
        {
            const int h = tid >> 1, half = tid & 1;  // 64 heads x 2 halves of 64 rows
            float tmax = -INFINITY;
            if (h < H)
                for (int k = 0; k < 64; ++k) {
                    const int rr = half * 64 + k;
                    if (valid[rr]) tmax = fmaxf(tmax, sst[rr * (NH + 1) + h] * cfac[h]);
                }
            tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 1));
            float mu = h < kMaxHeads ? m_run[h] : -INFINITY;
            float f = 1.f;
            if (h < H && tmax > -INFINITY && (mu == -INFINITY || tmax > mu + kRescaleLog2)) {
                f = mu == -INFINITY ? 0.f : fast_exp2(mu - tmax);
                mu = tmax;
            }
            float lsum = 0.f;
            if (h < NH) {
#pragma unroll 4
                for (int k8 = 0; k8 < 8; ++k8) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        __half ph[2], pl[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int rr = half * 64 + k8 * 8 + k2 * 2 + e;
                            float p = 0.f;
                            if (h < H && valid[rr] && mu > -INFINITY)
                                p = fast_exp2(sst[rr * (NH + 1) + h] * cfac[h] - mu);
                            lsum += p;
                            ph[e] = __float2half_rn(p);
                            pl[e] = __float2half_rn(p - __half2float(ph[e]));
                        }
                        hw[k2] = pack_half2(ph[0], ph[1]);
                        lw[k2] = pack_half2(pl[0], pl[1]);
                    }
                    const uint32_t off = sw128_off(h, half * 64 + k8 * 8, NH);
                    *reinterpret_cast<uint4 *>(p_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(p_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
            __syncwarp();
            if (half == 0 && h < kMaxHeads) {
                fac[h] = f;
                if (f != 1.f) flags[0] = 1;
                m_run[h] = mu;
                l_run[h] = l_run[h] * f + lsum;
            }
        }
        __syncthreads();
        // ---- rescale O^T when some head's running max moved (rare)
        if (flags[0] && o_started) {
            for (int mt = 0; mt < D / 128; ++mt)
                for (int c0 = 0; c0 < NH; c0 += 32) {
                    uint32_t r[32];
                    const uint32_t ta = t_o + mt * NH + lane_off + c0;
                    if (c0 + 32 <= NH) {
                        tmem_ld32(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * fac[c0 + k]);
                        tmem_st32(ta, r);
                    } else {
                        uint32_t r16[16];
                        asm volatile(
                            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                            : "=r"(r16[0]), "=r"(r16[1]), "=r"(r16[2]), "=r"(r16[3]), "=r"(r16[4]), "=r"(r16[5]),
                              "=r"(r16[6]), "=r"(r16[7]), "=r"(r16[8]), "=r"(r16[9]), "=r"(r16[10]), "=r"(r16[11]),
                              "=r"(r16[12]), "=r"(r16[13]), "=r"(r16[14]), "=r"(r16[15])
                            : "r"(ta));
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            r16[k] = __float_as_uint(__uint_as_float(r16[k]) * fac[c0 + k]);
                        asm volatile(
                            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                            "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(ta),
                            "r"(r16[0]), "r"(r16[1]), "r"(r16[2]), "r"(r16[3]), "r"(r16[4]), "r"(r16[5]),
                            "r"(r16[6]), "r"(r16[7]), "r"(r16[8]), "r"(r16[9]), "r"(r16[10]), "r"(r16[11]),
                            "r"(r16[12]), "r"(r16[13]), "r"(r16[14]), "r"(r16[15])
                            : "memory");
                    }
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
                for (int part = 0; part < 2; ++part) {
                    const uint32_t pb = part ? plo_base : phi_base;
                    for (int ks = 0; ks < kRows / 16; ++ks) {
                        const uint64_t da = smem_desc(v_base + (2 * mt) * kRows * 128 + ks * 2048,
                                                      kRows * 128 /*next 64 dims*/, 1024 /*next 8 rows*/, 2);
                        const uint64_t db = smem_desc(pb + (ks >> 2) * NH * 128 + (ks & 3) * 32, 16, 1024, 2);
                        mma_f16(t_o + mt * NH, da, db, idesc_o, (o_started || part > 0 || ks > 0) ? 1u : 0u);
                    }
                }
            mma_commit(mma_bar);
        }
        __syncwarp();
        ok = mbar_wait(mma_bar, mma_phase, abort_flag);
        mma_phase ^= 1;
        tc_fence_after();
        o_started = true;
    }

    // ---- write the result (or the split partial): thread = one dim of each 128-dim block
    if (ok) {
        __syncthreads();
        const bool final_out = a.nsplit == 1;
        float *obase = final_out ? a.out + static_cast<int64_t>(unit) * H * D
                                 : a.part_o + (static_cast<int64_t>(unit) * a.nsplit + split) * H * D;
        for (int mt = 0; mt < D / 128; ++mt) {
            const int d = mt * 128 + warp * 32 + lane;
            for (int c0 = 0; c0 < NH; c0 += 16) {
                uint32_t r[16];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                    "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                    : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                      "=r"(r[14]), "=r"(r[15])
                    : "r"(t_o + mt * NH + lane_off + c0));
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int h = c0 + k;
                    if (h >= H) continue;
                    float v = o_started ? __uint_as_float(r[k]) : 0.f;
                    if (final_out) v = l_run[h] > 0.f ? v / l_run[h] : 0.f;
                    obase[static_cast<int64_t>(h) * D + d] = v;
                }
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

// Combines the split partials of one (query, head):
// out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, lse = ln 2 * (M + log2 sum).
__global__ void __launch_bounds__(128) attend_merge_kernel(int D, int H, int nsplit, const float *__restrict__ part_o,
                                                          const float2 *__restrict__ part_ml, float *__restrict__ out,
                                                          float *__restrict__ lse)
{
    __shared__ float wsh[32];
    __shared__ float inv_l, lse_v;
    const int unit = blockIdx.y, h = blockIdx.x;
    if (threadIdx.x < 32) {
        const int s = threadIdx.x;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (s < nsplit) ml = part_ml[(static_cast<int64_t>(unit) * nsplit + s) * H + h];
        float M = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        const float wgt = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
        float L = wgt * ml.y;
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        wsh[s] = wgt;
        if (s == 0) {
            inv_l = L > 0.f ? 1.f / L : 0.f;
            lse_v = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float v[32];
#pragma unroll
        for (int s = 0; s < 32; ++s)
            v[s] = (s < nsplit && wsh[s] != 0.f) ? part_o[((static_cast<int64_t>(unit) * nsplit + s) * H + h) * D + d]
                                                 : 0.f;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < 32; ++s) acc = fmaf(wsh[s], v[s], acc);
        out[(static_cast<int64_t>(unit) * H + h) * D + d] = acc * inv_l;
    }
    if (lse && threadIdx.x == 0) lse[static_cast<int64_t>(unit) * H + h] = lse_v;
}

struct Plan {
    int nsplit, tiles_per_split, tiles_total;
};

Plan plan(const CacheView &c, int P, int K)
{
    const int units = c.B * P;
    const int tiles = (K + kRows - 1) / kRows;
    int want = (148 + units - 1) / units;  // about one wave of CTAs
    if (want > tiles) want = tiles;
    if (want < 1) want = 1;
    Plan p;
    p.tiles_total = tiles;
    p.tiles_per_split = (tiles + want - 1) / want;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    while (p.nsplit > 32) {  // the merge combines at most 32 partials
        ++p.tiles_per_split;
        p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    }
    return p;
}

size_t smem_bytes(int D, int NH)
{
    const size_t v = static_cast<size_t>(kRows) * D * 2;
    const size_t qh = static_cast<size_t>(NH) * 256 * 2, sst = static_cast<size_t>(kRows) * (NH + 1) * 4;
    const size_t qs = ((qh > sst ? qh : sst) + 1023) & ~size_t(1023);
    const size_t p = 2 * static_cast<size_t>(NH) * kRows * 2;
    return 1024 + v + qs + p + 5 * kMaxHeads * 4 + kRows * 4 + 64;
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
        attend_merge_kernel<<<dim3(H, units), 128, 0, st>>>(c.D, H, p.nsplit, a.part_o, a.part_ml, out, lse);
        e = cudaGetLastError();
        if (e == cudaSuccess) count_launch();
    }
    return e;
}

}  // namespace csa
