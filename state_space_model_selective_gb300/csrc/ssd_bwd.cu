// ssd_bwd.cu -- gradient of the chunked SSD (ssd_chunked_bwd) on tcgen05 tensor
// cores, GB300 / sm_103a.
//
// The forward operation is ssd_chunked_fwd's ("Mamba-3 NKI Kernels for AWS
// Neuron", section "Kernel details", mamba3_siso_ssd_kernel: the Mamba-2 SSD
// structure, equivalent to the step recurrence S = exp(dt A) S + dt B x^T,
// y = C S).  Its reverse-mode derivative, for the loss sum(dy y) +
// sum(dfinal final_state), is evaluated block by block in reverse, with the
// adjoint state dS = dL/dS carried between blocks.  For a block of Q = 128
// steps with cs_i = sum_{j<=i} dt_j A (inside the block), input weights w
// (w = dt for ssd_chunked_bwd; the Mamba-3 gradient passes its scale weights),
// L[i,j] = exp(cs_i - cs_j) for j <= i (else 0), S_in / S_out the states
// entering / leaving the block and dS_out the adjoint leaving it:
//   T       = dY X^T                      (Q x Q; (L o T) includes w_j)
//   dC      = diag(e^cs) dY S_in + (L o T w) B
//   dB      = diag(w e^(cs_last - cs)) X dS_out + (L o T w)^T C
//   bracket = diag(e^(cs_last - cs)) B dS_out^T + (L o C B^T)^T dY,  dX = diag(w) bracket
//   dS_in   = e^cs_last dS_out + (e^cs o dY)^T C
//   d cs_i  = C_i . dC_i - B_i . dB_i  (+ <dS_out, S_out> at the block's last row)
//   dw_k    = x_k . bracket_k,  ddt_k = (dw_k if w = dt) + A sum_{i >= k} d cs_i,
//   dA     += sum_k dt_k sum_{i >= k} d cs_i
// (the C . dC - B . dB form of the log-decay gradient: every term of y_i and
// of S_out depends on cs only through factors e^(cs_i - cs_j)).
//
// GB300 mapping.  One CTA of 256 threads per (batch, head): two warpgroups,
// thread (r, part) owning TMEM lane r (block row r) and half of each row's
// columns (part 0 the first half); C, B, x and dy arrive by TMA in the 128-byte-
// swizzled layout the MMAs read; S_in, dS_out and e^cs o dY are split into
// bf16 hi + lo pairs and written by the threads.  Eleven products per block,
// all M = 128 tcgen05 MMAs with fp32 accumulators in the CTA's 512 TMEM
// columns, issued in six groups between which the threads mask, scale and
// split (the masked Q x Q products go back into TMEM as bf16 hi/lo operands).
// The states entering each block come from the forward kernel run in its
// checkpoint mode.  dB and dC are per-head partials summed over a group's heads
// by a second kernel, in a fixed order.
#include <algorithm>
#include <functional>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace {

using namespace ssm;
using namespace ssd_detail;

constexpr int kWorkers = 256;              // two warpgroups: thread (row, half of the row)
constexpr int kThreads = kWorkers + 32;   // + the issuing warp (TMA loads, MMAs)

// Shared memory (offsets from the 1024-aligned base)
constexpr uint32_t kSC = 0;         // C tile [128 i][128 n] (two 64-n boxes, 16 KB apart)
constexpr uint32_t kSB = 32768;     // B tile [128 j][128 n]
constexpr uint32_t kSX = 65536;     // x tile [128 j][64 p]
constexpr uint32_t kSDY = 81920;    // dy tile [128 i][64 p]
constexpr uint32_t kSS = 98304;     // S_in hi | lo [128 n][64 p]
constexpr uint32_t kSDS = 131072;   // dS_out hi | lo [128 n][64 p]
constexpr uint32_t kSE = 163840;    // (e^cs o dY) hi | lo [128 i][64 p]
constexpr uint32_t kMisc = 196608;  // cs2[128], q2[128], sums, mbarriers, TMEM address
constexpr int kNumBars = 18;
constexpr uint32_t kMiscBytes = (2 * 128 + 32 + 3 * 128) * 4 + kNumBars * 8 + 16;
constexpr uint32_t kSmemAlloc = kMisc + kMiscBytes + 1024;  // + realignment slack

// TMEM columns (one CTA per SM: all 512)
constexpr uint32_t kTmT = 0;     // T = dY X^T -> (L o T w) hi/lo; then T^T -> (L o T w)^T hi/lo
constexpr uint32_t kTmP = 128;   // P = dY S_in -> dC
constexpr uint32_t kTmGT = 256;  // G^T = B C^T -> (L o G)^T hi/lo
constexpr uint32_t kTmR = 384;   // R = B dS_out^T -> bracket (64); then Q -> dB (128)
constexpr uint32_t kTmDS = 448;  // dS_in^T (64)
constexpr uint32_t kTmQ = 384;
constexpr uint32_t kTmemCols = 512;

struct BwdArgs {
    const float* dt;       // (batch, seqlen, nheads)
    // input weights w (batch, seqlen, nheads), or NULL for w = dt.  With w
    // given, ddt receives only the log-decay part A sum_{i >= k} d cs_i and dw
    // the input-weight part x_k . bracket_k.
    const float* w;
    float* dw;
    const float* A;        // (nheads,)
    const float* bstates;  // [batch * nheads][nblocks + 1][64][128]
    const float* dfinal;   // (batch, nheads, 64, 128) or NULL
    float* dx;             // (batch, seqlen, nheads, 64)
    float* ddt;            // (batch, seqlen, nheads)
    float* dh0;            // (batch, nheads, 64, 128) or NULL
    float* pB;             // [nheads][batch][128][seqlen] per-head dB
    float* pC;             // [nheads][batch][128][seqlen] per-head dC
    float* pA;             // [batch * nheads]
    uint32_t* status;
    int batch, seqlen, nheads, ngroups;
    // Mamba-3's diagonal correction of dx, applied as dx is written (NULL:
    // none): dx_{t,r'} -= c_t sum_r G_t[r][r'] dy_{t,r}, c_t = dt_{t+1} (1 -
    // lambda_{t+1}) (0 at the last step), G_t[r][r'] = C_{t,r} . B_{t,r'}
    // ([step][group][RK][RK]); dt, lambda per step (batch, steps, nheads)
    const float* corr_g;
    const float* corr_dt;
    const float* corr_lam;
    int corr_steps;
};

// One 32-column chunk of a masked, decayed Q x Q row, split into bf16 hi/lo:
// m_k = g_k 2^(base + col2[k]) for columns k inside [lo, hi] (relative to the
// chunk), 0 outside.
__device__ __forceinline__ void masked_chunk(const float* gv, const float* col2, float base,
                                             int lo, int hi, uint32_t* hp, uint32_t* lp) {
#pragma unroll
    for (int q = 0; q < 32; q += 4) {
        const float4 cc = *reinterpret_cast<const float4*>(col2 + q);
        const float cv[4] = {cc.x, cc.y, cc.z, cc.w};
        float m[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m[k] = gv[q + k] * ex2_approx(base + cv[k]);
            if (q + k < lo || q + k > hi) m[k] = 0.0f;
        }
        split2_bf16(m[0], m[1], hp[q >> 1], lp[q >> 1]);
        split2_bf16(m[2], m[3], hp[(q >> 1) + 1], lp[(q >> 1) + 1]);
    }
}

// This warpgroup's half (columns 64 part .. + 63) of row r of a TMEM Q x Q
// product, turned into its masked, decayed bf16 hi/lo operand in place: column
// k kept for k in [kmin, kmax] with factor 2^(base + col2[k]).
__device__ __forceinline__ void mask_row_half(uint32_t taddr, const float* col2, float base,
                                              int kmin, int kmax, int part) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 64 * part + 32 * hh;
        uint32_t hp[16], lp[16];
        if (c0 + 31 < kmin || c0 > kmax) {
#pragma unroll
            for (int q = 0; q < 16; ++q) hp[q] = lp[q] = 0u;
        } else {
            float gv[32];
            tmem_ld32(taddr + c0, gv);
            tmem_wait_ld();
            masked_chunk(gv, col2 + c0, base, kmin - c0, kmax - c0, hp, lp);
        }
        tmem_st16(taddr + c0, hp);
        tmem_st16(taddr + c0 + 16, lp);
    }
}

// This warpgroup's half of row j of G^T and of T^T (two TMEM products with the
// same mask and decay), each turned into its bf16 hi/lo operand in place:
// columns i >= j kept, G^T with factor e^(cs_i - cs_j) = 2^(cs2[i] - cs2_j),
// T^T with that factor times the input weight w_j.  One exp2 per element
// serves both.
__device__ __forceinline__ void mask_pair_half(uint32_t tg, uint32_t tt, const float* cs2,
                                               float cs2_j, float w_j, int j, int part) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 64 * part + 32 * hh;
        uint32_t gh[16], gl[16], th[16], tl[16];
        if (c0 + 31 < j) {
#pragma unroll
            for (int q = 0; q < 16; ++q) gh[q] = gl[q] = th[q] = tl[q] = 0u;
        } else {
            float gv[32], tv[32];
            tmem_ld32(tg + c0, gv);
            tmem_ld32(tt + c0, tv);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
                float f0 = ex2_approx(cs2[c0 + q] - cs2_j), f1 = ex2_approx(cs2[c0 + q + 1] - cs2_j);
                if (c0 + q < j) f0 = 0.0f;
                if (c0 + q + 1 < j) f1 = 0.0f;
                split2_bf16(gv[q] * f0, gv[q + 1] * f1, gh[q >> 1], gl[q >> 1]);
                split2_bf16(tv[q] * (f0 * w_j), tv[q + 1] * (f1 * w_j), th[q >> 1], tl[q >> 1]);
            }
        }
        tmem_st16(tg + c0, gh);
        tmem_st16(tg + c0 + 16, gl);
        tmem_st16(tt + c0, th);
        tmem_st16(tt + c0 + 16, tl);
    }
}

// 32 fp32 values (this warpgroup's p range 32 part .. + 31) of one [n][p] or
// [i][p] row, written as bf16 hi and lo into a 128-byte-swizzled tile pair
// (lo 16 KB after hi).
__device__ __forceinline__ void store_split_half(uint8_t* tile, int row, int part, const float* v) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t hp[4], lp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2_bf16(v[8 * c + 2 * e], v[8 * c + 2 * e + 1], hp[e], lp[e]);
        const int cc = 4 * part + c;
        const uint32_t off = (uint32_t)(row * 128 + ((cc ^ (row & 7)) << 4));
        *reinterpret_cast<uint4*>(tile + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
        *reinterpret_cast<uint4*>(tile + 16384 + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
    }
}

// The 32 bf16 of row r, columns 32 part .. + 31, of a TMA tile [128][64] in the
// 128-byte swizzle, as fp32.
__device__ __forceinline__ void load_tile_half(const uint8_t* tile, int row, int part, float* v) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int cc = 4 * part + c;
        const uint4 w = *reinterpret_cast<const uint4*>(tile + row * 128 + ((cc ^ (row & 7)) << 4));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[8 * c + 2 * e] = bf16lo(ww[e]);
            v[8 * c + 2 * e + 1] = bf16hi(ww[e]);
        }
    }
}

// This warpgroup's half of a dot product: row r of a TMA tile [128][128] (two
// 64-wide boxes 16 KB apart; box `part` holds columns 64 part .. + 63) against
// the same 64 fp32 columns of TMEM row r, 32 at a time; optionally the 64
// values are also stored, column n at dst[n * stride] (the rows of a warp are
// consecutive in dst, so each store is coalesced).
__device__ __forceinline__ float dot_half_tmem(const uint8_t* tile, int row, int part,
                                               uint32_t taddr, float* dst, long long stride) {
    const uint8_t* box = tile + part * 16384 + row * 128;
    float acc = 0.0f;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32(taddr + 64 * part + 32 * hh, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int cc = 4 * hh + c;
            const uint4 w = *reinterpret_cast<const uint4*>(box + ((cc ^ (row & 7)) << 4));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc = fmaf(bf16lo(ww[e]), v[8 * c + 2 * e],
                           fmaf(bf16hi(ww[e]), v[8 * c + 2 * e + 1], acc));
        }
        if (dst) {
            float* d = dst + (64 * part + 32 * hh) * stride;
#pragma unroll
            for (int q = 0; q < 32; ++q) d[q * stride] = v[q];
        }
    }
    return acc;
}

// This warpgroup's 64 columns of TMEM row r scaled by f in place, 32 at a time.
__device__ __forceinline__ void scale_half(uint32_t taddr, int part, float f) {
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32(taddr + 64 * part + 32 * hh, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] *= f;
        tmem_st32f(taddr + 64 * part + 32 * hh, v);
    }
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// RK > 1 (Mamba-3 MIMO): rows are sub-tokens, RK consecutive rows one step
// that see one another fully (the mask is block-lower-triangular); the step's
// dt sits on its first row (0 on the others) and its weight on every row.
// CORR: Mamba-3's diagonal correction is applied to dx as it is written
// (BwdArgs::corr_*); without it the plain SSD gradient's dx write is unchanged.
template <int RK, bool CORR>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_bwd_kernel(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
                   const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                   const BwdArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    float* s_cs2 = reinterpret_cast<float*>(smem + kMisc);  // log2-scaled cs of each row
    float* s_q2 = s_cs2 + kQ;                               // log2(w_j) - cs2_j
    float* s_wsum = s_q2 + kQ;                              // [2][4] warp totals (cs scan)
    float* s_rsum = s_wsum + 8;                             // [4] warp totals (d cs suffix scan)
    float* s_dot = s_rsum + 8;                              // [8] <dS_out, S_out> per warp
    float* s_da = s_dot + 8;                                // [4] dA per warp
    float* s_pd = s_da + 8;                                 // [3][128] the second half's dots
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_pd + 3 * kQ);
    uint64_t* bar_cb = bars + 0;   // TMA: C, B in
    uint64_t* bar_s = bars + 1;    // bulk: S_in, S_out in
    uint64_t* bar_xy = bars + 2;   // TMA: x, dy in
    uint64_t* bar_fin = bars + 3;  // issuer: every MMA done (at exit)
    uint64_t* m_tp = bars + 4;     // MMA done: T, P
    uint64_t* m_rs = bars + 5;     // MMA done: R, dS_in^T
    uint64_t* m_gt = bars + 6;     // MMA done: G^T
    uint64_t* m_dc = bars + 7;     // MMA done: dC
    uint64_t* m_br = bars + 8;     // MMA done: bracket
    uint64_t* m_q = bars + 9;      // MMA done: Q = X dS_out
    uint64_t* m_tt = bars + 10;    // MMA done: T^T
    uint64_t* m_db = bars + 11;    // MMA done: dB
    uint64_t* r_op = bars + 12;    // workers: the block's shared-memory operands written
    uint64_t* r_dc = bars + 13;    // workers: (L o T w) and e^cs P in TMEM
    uint64_t* r_br = bars + 14;    // workers: (L o G)^T and the scaled R in TMEM
    uint64_t* r_db = bars + 15;    // workers: (L o T w)^T and the scaled Q in TMEM
    uint64_t* r_x = bars + 16;     // workers: done reading the x tile
    uint64_t* r_cb = bars + 17;    // workers: done reading the C and B tiles
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile uint32_t* s_abort = s_tmem + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x;
    const int h = item % a.nheads, b = item / a.nheads;
    const int g = h / (a.nheads / a.ngroups);
    const int L = a.seqlen;
    const int nblocks = (L + kQ - 1) / kQ;
    const float* bs_item = a.bstates + (long long)item * (nblocks + 1) * kP * kNs;

    if (warp == 0) tmem_alloc(s_tmem, kTmemCols);
    if (tid == 0) {
        for (int k = 0; k < 12; ++k) mbar_init(bars + k, 1);
        for (int k = 12; k < kNumBars; ++k) mbar_init(bars + k, kWorkers);
        *s_abort = 0u;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == kWorkers / 32) {
        // ================= issuing warp: TMA loads and MMAs (one lane)
        if (lane == 0) {
            prefetch_tensormap(&tm_C);
            prefetch_tensormap(&tm_B);
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_dy);
            auto load_cb = [&](int blk) {
                mbar_arrive_expect_tx(bar_cb, 2 * 32768);
                tma_load_4d(smem + kSC, &tm_C, bar_cb, 0, g, blk * kQ, b);
                tma_load_4d(smem + kSC + 16384, &tm_C, bar_cb, 64, g, blk * kQ, b);
                tma_load_4d(smem + kSB, &tm_B, bar_cb, 0, g, blk * kQ, b);
                tma_load_4d(smem + kSB + 16384, &tm_B, bar_cb, 64, g, blk * kQ, b);
            };
            auto load_s = [&](int blk) {
                mbar_arrive_expect_tx(bar_s, 2 * 32768);
                bulk_load(smem + kSE, bs_item + (long long)blk * kP * kNs, 32768, bar_s);
                bulk_load(smem + kSDS, bs_item + (long long)(blk + 1) * kP * kNs, 32768, bar_s);
            };
            auto load_xy = [&](int blk) {
                mbar_arrive_expect_tx(bar_xy, 2 * 16384);
                tma_load_3d(smem + kSX, &tm_x, bar_xy, h * kP, blk * kQ, b);
                tma_load_3d(smem + kSDY, &tm_dy, bar_xy, h * kP, blk * kQ, b);
            };
            // pending load phases (parity), -1 when none
            int p_cb = -1, p_s = -1, p_xy = -1;
            if (nblocks > 0) {
                load_cb(nblocks - 1);
                load_s(nblocks - 1);
                load_xy(nblocks - 1);
                p_cb = p_s = p_xy = 0;
            }
            uint32_t ph = 0;
            constexpr uint32_t id128 = idesc_bf16_f32(128, 128);
            constexpr uint32_t id128b = idesc_bf16_f32(128, 128) | kIdescBMN;
            constexpr uint32_t id64b = idesc_bf16_f32(128, 64) | kIdescBMN;
            constexpr uint32_t id64ab = idesc_bf16_f32(128, 64) | kIdescAMN | kIdescBMN;
            for (int blk = nblocks - 1; blk >= 0; --blk, ph ^= 1u) {
                auto W = [&](uint64_t* bar) {
                    if (*s_abort) return false;
                    if (!mbar_wait(bar, ph, a.status)) {
                        *s_abort = 1u;
                        return false;
                    }
                    return true;
                };
                if (!W(bar_cb) || !W(bar_s) || !W(bar_xy)) break;
                p_cb = p_s = p_xy = -1;
                if (!W(r_op)) break;
                tc_fence_after();
                // T = dY X^T, P = dY S_in (hi + lo)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kTmT, kdesc<kQ>(sbase + kSDY, kk), kdesc<kQ>(sbase + kSX, kk),
                             id128, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + kTmP, kdesc<kQ>(sbase + kSDY, kk & 3),
                             kdesc<kQ>(sbase + kSS + (kk >> 2) * 16384, kk & 3), id128, kk > 0);
                mma_commit(m_tp);
                // R = B dS_out^T (hi + lo), dS_in^T = C^T (e^cs o dY) (hi + lo)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16(tmem + kTmR, kdesc<kQ>(sbase + kSB, kk), mdesc(sbase + kSDS, kk, 16384),
                             id64b, kk > 0);
                    mma_bf16(tmem + kTmR, kdesc<kQ>(sbase + kSB, kk),
                             mdesc(sbase + kSDS + 16384, kk, 16384), id64b, 1);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16(tmem + kTmDS, mdesc(sbase + kSC, kk, 16384),
                             mdesc(sbase + kSE, kk, 16384), id64ab, kk > 0);
                    mma_bf16(tmem + kTmDS, mdesc(sbase + kSC, kk, 16384),
                             mdesc(sbase + kSE + 16384, kk, 16384), id64ab, 1);
                }
                mma_commit(m_rs);
                // G^T = B C^T
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + kTmGT, kdesc<kQ>(sbase + kSB, kk), kdesc<kQ>(sbase + kSC, kk),
                             id128, kk > 0);
                mma_commit(m_gt);
                // dC = e^cs o P + (L o T w) B
                if (!W(r_dc)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16_ta(tmem + kTmP, tmem + kTmT + mcol_hi(kk), mdesc(sbase + kSB, kk, 16384),
                                id128b, 1);
                    mma_bf16_ta(tmem + kTmP, tmem + kTmT + mcol_hi(kk) + 16,
                                mdesc(sbase + kSB, kk, 16384), id128b, 1);
                }
                mma_commit(m_dc);
                // T^T = X dY^T into the consumed (L o T w) columns
                if (!W(m_dc)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kTmT, kdesc<kQ>(sbase + kSX, kk), kdesc<kQ>(sbase + kSDY, kk),
                             id128, kk > 0);
                mma_commit(m_tt);
                // bracket = e^(cs_last - cs) o R + (L o G)^T dY
                if (!W(r_br)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16_ta(tmem + kTmR, tmem + kTmGT + mcol_hi(kk), mdesc(sbase + kSDY, kk, 16384),
                                id64b, 1);
                    mma_bf16_ta(tmem + kTmR, tmem + kTmGT + mcol_hi(kk) + 16,
                                mdesc(sbase + kSDY, kk, 16384), id64b, 1);
                }
                mma_commit(m_br);
                // Q = X dS_out (hi + lo) into the bracket's and dS_in's columns, once
                // the workers have read both
                if (!W(r_x)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + kTmQ, kdesc<kQ>(sbase + kSX, kk & 3),
                             kdesc<kQ>(sbase + kSDS + (kk >> 2) * 16384, kk & 3), id128, kk > 0);
                mma_commit(m_q);
                if (blk > 0) {
                    // the states' regions and x, dy are free once Q, their last
                    // reader, is done (the workers' x reads are behind r_x)
                    if (!W(m_q)) break;
                    load_s(blk - 1);
                    p_s = (int)(ph ^ 1u);
                    load_xy(blk - 1);
                    p_xy = (int)(ph ^ 1u);
                }
                // dB = w e^(cs_last - cs) o Q + (L o T w)^T C
                if (!W(r_db)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16_ta(tmem + kTmQ, tmem + kTmT + mcol_hi(kk), mdesc(sbase + kSC, kk, 16384),
                                id128b, 1);
                    mma_bf16_ta(tmem + kTmQ, tmem + kTmT + mcol_hi(kk) + 16,
                                mdesc(sbase + kSC, kk, 16384), id128b, 1);
                }
                mma_commit(m_db);
                if (blk > 0) {
                    // C and B once dB and the workers' dC, dB dots are done
                    if (!W(m_db) || !W(r_cb)) break;
                    load_cb(blk - 1);
                    p_cb = (int)(ph ^ 1u);
                }
            }
            // never leave with an MMA or a load in flight (bounded waits)
            mma_commit(bar_fin);
            (void)mbar_wait(bar_fin, 0, nullptr);
            if (p_cb >= 0) (void)mbar_wait(bar_cb, (uint32_t)p_cb, nullptr);
            if (p_s >= 0) (void)mbar_wait(bar_s, (uint32_t)p_s, nullptr);
            if (p_xy >= 0) (void)mbar_wait(bar_xy, (uint32_t)p_xy, nullptr);
        }
    } else {
        // ================= worker warpgroups: thread (row, part)
        const int quarter = warp & 3;         // TMEM lane quarter this warp may access
        const int part = warp >> 2;           // which half of each row's columns it takes
        const int row = quarter * 32 + lane;  // TMEM lane and block row
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const float Ah = a.A[h];
        // the adjoint state dS_out[p = 32 part + q][n = row], carried from block to block
        float dS[32];
#pragma unroll
        for (int q = 0; q < 32; ++q)
            dS[q] = a.dfinal ? a.dfinal[((long long)item * kP + 32 * part + q) * kNs + row] : 0.0f;
        float dA_acc = 0.0f;
        bool ok = true;
        uint32_t ph = 0;
        auto dt_of = [&](int blk) {
            const int t = blk * kQ + row;
            return t < L ? a.dt[((long long)b * L + t) * a.nheads + h] : 0.0f;
        };
        const float* wsrc = a.w ? a.w : a.dt;
        auto w_of = [&](int blk) {
            const int t = blk * kQ + row;
            return t < L ? wsrc[((long long)b * L + t) * a.nheads + h] : 0.0f;
        };
        float dt_next = nblocks > 0 ? dt_of(nblocks - 1) : 0.0f;
        float w_next = nblocks > 0 ? w_of(nblocks - 1) : 0.0f;
        // per-head dB, dC partials: [h][b][n][t], t contiguous (coalesced across a warp's rows)
        const long long pofs = ((long long)h * a.batch + b) * kNs * L;

        for (int blk = nblocks - 1; blk >= 0; --blk, ph ^= 1u) {
            // bounded wait on `bar`, agreed by all workers (all leave together)
            auto Wc = [&](uint64_t* bar) {
                bool got = !*s_abort && mbar_wait(bar, ph, a.status);
                if (!got) *s_abort = 1u;
                return named_bar_and(1, kWorkers, got);
            };
            const int t = blk * kQ + row;
            const float dtr = dt_next;  // this row's step: log-decay dt A
            const float wr = w_next;    // and input weight
            if (blk > 0) {
                dt_next = dt_of(blk - 1);
                w_next = w_of(blk - 1);
            }

            // ---- cumulative log-decay within the block
            float v = dtr * Ah;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane == 31) s_wsum[part * 4 + quarter] = v;
            if (!Wc(bar_cb) || !Wc(bar_s) || !Wc(bar_xy)) { ok = false; break; }
            float cs_last = 0.0f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float ws = s_wsum[part * 4 + w];
                if (w < quarter) v += ws;
                cs_last += ws;
            }
            const float cs2 = v * kLog2e, cs2_last = cs_last * kLog2e;
            float lg;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(wr));
            const float q2 = lg - cs2;
            if (part == 0) {
                s_cs2[row] = cs2;
                s_q2[row] = q2;
            }
            const float e_r = ex2_approx(cs2);
            const float eL_r = ex2_approx(cs2_last - cs2);
            const float u_r = wr * eL_r;
            const float e_last = ex2_approx(cs2_last);

            // ---- S_in split [n = row][p]; <dS_out, S_out>; then dS_out and
            // e^cs o dY split over the fp32 states' regions
            {
                const float* sin = reinterpret_cast<const float*>(smem + kSE) + 32 * part * kNs + row;
                const float* sout = reinterpret_cast<const float*>(smem + kSDS) + 32 * part * kNs + row;
                float sv[32];
                float dot = 0.0f;
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    sv[q] = sin[q * kNs];
                    dot = fmaf(dS[q], sout[q * kNs], dot);
                }
                store_split_half(smem + kSS, row, part, sv);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (lane == 0) s_dot[warp] = dot;
            }
            named_bar_sync(1, kWorkers);  // the fp32 states are read; s_dot, s_cs2 visible
            store_split_half(smem + kSDS, row, part, dS);
            {
                float dyv[32];
                load_tile_half(smem + kSDY, row, part, dyv);
#pragma unroll
                for (int q = 0; q < 32; ++q) dyv[q] *= e_r;
                store_split_half(smem + kSE, row, part, dyv);
            }
            float sdot = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sdot += s_dot[w];
            fence_proxy_async_smem();
            mbar_arrive(r_op);

            // ---- (L o T w) and e^cs P, for dC
            if (!Wc(m_tp)) { ok = false; break; }
            tc_fence_after();
            // (L o T w) row i = row: columns j <= i, factor e^(cs_i - cs_j) w_j
            mask_row_half(t_lane + kTmT, s_q2, cs2, 0, RK * (row / RK) + RK - 1, part);
            scale_half(t_lane + kTmP, part, e_r);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(r_dc);
            // ---- R scaled by e^(cs_last - cs_j); the adjoint entering the block:
            // dS_in[p][n = row] = e^cs_last dS_out + (C^T (e^cs o dY))[n][p]
            if (!Wc(m_rs)) { ok = false; break; }
            tc_fence_after();
            {
                float rv[32], sv[32];
                tmem_ld32(t_lane + kTmR + 32 * part, rv);
                tmem_ld32(t_lane + kTmDS + 32 * part, sv);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    rv[q] *= eL_r;
                    dS[q] = fmaf(e_last, dS[q], sv[q]);
                }
                tmem_st32f(t_lane + kTmR + 32 * part, rv);
            }
            // ---- (L o G)^T and (L o T w)^T, row j = row: columns i >= j
            if (!Wc(m_gt) || !Wc(m_tt)) { ok = false; break; }
            tc_fence_after();
            mask_pair_half(t_lane + kTmGT, t_lane + kTmT, s_cs2, cs2, wr, RK * (row / RK), part);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(r_br);
            // ---- dX_j = w_j bracket_j; the input-weight gradient is x_j . bracket_j
            if (!Wc(m_br)) { ok = false; break; }
            tc_fence_after();
            float dw = 0.0f;
            {
                float xv[32], br[32];
                load_tile_half(smem + kSX, row, part, xv);
                tmem_ld32(t_lane + kTmR + 32 * part, br);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) dw = fmaf(xv[q], br[q], dw);
                if (!CORR && t < L) {
                    float* dxr = a.dx + (((long long)b * L + t) * a.nheads + h) * kP + 32 * part;
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(dxr + q) = make_float4(
                            wr * br[q], wr * br[q + 1], wr * br[q + 2], wr * br[q + 3]);
                }
                if (CORR && t < L) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) br[q] *= wr;
                    {
                        // the step's RK rows of dy: tile rows row - rp .. row - rp + RK - 1
                        const int ts = t / RK, rp = t - ts * RK;
                        const long long bt = (long long)b * a.corr_steps + ts;
                        const float c = ts + 1 < a.corr_steps
                                            ? a.corr_dt[(bt + 1) * a.nheads + h] *
                                                  (1.0f - a.corr_lam[(bt + 1) * a.nheads + h])
                                            : 0.0f;
                        const float* Gp = a.corr_g + (bt * a.ngroups + g) * (RK * RK);
#pragma unroll
                        for (int r = 0; r < RK; ++r) {
                            const float coef = c * Gp[r * RK + rp];
                            float dyv[32];
                            load_tile_half(smem + kSDY, row - rp + r, part, dyv);
#pragma unroll
                            for (int q = 0; q < 32; ++q) br[q] = fmaf(-coef, dyv[q], br[q]);
                        }
                    }
                    float* dxr = a.dx + (((long long)b * L + t) * a.nheads + h) * kP + 32 * part;
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(dxr + q) =
                            make_float4(br[q], br[q + 1], br[q + 2], br[q + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(r_x);
            // ---- Q row j scaled by w_j e^(cs_last - cs_j)
            if (!Wc(m_q)) { ok = false; break; }
            tc_fence_after();
            scale_half(t_lane + kTmQ, part, u_r);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(r_db);
            // ---- dC row i: its log-decay term C_i . dC_i (this half) and its
            // partial (while dB runs)
            const float dcs_c =
                dot_half_tmem(smem + kSC, row, part, t_lane + kTmP, t < L ? a.pC + pofs + t : nullptr, L);
            // ---- dB row j: its log-decay term B_j . dB_j (this half) and its partial
            if (!Wc(m_db)) { ok = false; break; }
            tc_fence_after();
            const float dcs_b =
                dot_half_tmem(smem + kSB, row, part, t_lane + kTmQ, t < L ? a.pB + pofs + t : nullptr, L);
            mbar_arrive(r_cb);

            // ---- log-decay gradient of each row, its suffix sums over the block,
            // ddt and dA (first warpgroup)
            if (part == 1) {
                s_pd[row] = dcs_c;
                s_pd[kQ + row] = dcs_b;
                s_pd[2 * kQ + row] = dw;
            }
            named_bar_sync(1, kWorkers);
            if (part == 0) {
                float dcs = (dcs_c + s_pd[row]) - (dcs_b + s_pd[kQ + row]) +
                            (row == kQ - 1 ? sdot : 0.0f);
                const float dw_all = dw + s_pd[2 * kQ + row];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_down_sync(0xffffffffu, dcs, o);
                    if (lane + o < 32) dcs += u;
                }
                if (lane == 0) s_rsum[quarter] = dcs;
                named_bar_sync(2, kWorkers / 2);  // the first warpgroup only
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    if (w > quarter) dcs += s_rsum[w];
                if (t < L) {
                    const long long o = ((long long)b * L + t) * a.nheads + h;
                    if (a.dw) {
                        a.ddt[o] = Ah * dcs;
                        a.dw[o] = dw_all;
                    } else {
                        a.ddt[o] = fmaf(Ah, dcs, dw_all);
                    }
                }
                dA_acc = fmaf(dtr, dcs, dA_acc);
            }
            named_bar_sync(1, kWorkers);  // s_* are rewritten by the next block
        }
        if (ok) {
            if (a.dh0) {
#pragma unroll
                for (int q = 0; q < 32; ++q)
                    a.dh0[((long long)item * kP + 32 * part + q) * kNs + row] = dS[q];
            }
            if (part == 0) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, o);
                if (lane == 0) s_da[quarter] = dA_acc;
            }
            named_bar_sync(1, kWorkers);
            if (tid == 0) a.pA[item] = s_da[0] + s_da[1] + s_da[2] + s_da[3];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// dB, dC = the per-head partials ([h][b][n][t]) summed over each group's heads,
// in head order, and written as (batch, seqlen, ngroups, dstate): a 128 x 32
// (t, n) tile per block, each thread adding four consecutive steps of four
// rows with 16-byte loads, transposed through shared memory so that both the
// reads (t contiguous) and the writes (n contiguous) are coalesced.  seqlen is
// a multiple of 4 (of the chunk).
__global__ void ssd_bwd_reduce_bc_kernel(const float* __restrict__ pB, const float* __restrict__ pC,
                                         float* __restrict__ dB, float* __restrict__ dC, int batch,
                                         int seqlen, int nheads, int ngroups) {
    __shared__ float tile[32][129];
    const int hpg = nheads / ngroups;
    const int t0 = blockIdx.x * 128, n0 = blockIdx.y * 32;
    const long long L = seqlen;
    for (int z = blockIdx.z; z < 2 * batch * ngroups; z += gridDim.z) {
        const bool isC = z & 1;
        const int bg = z >> 1, bb = bg / ngroups, gg = bg % ngroups;
        const float* src = isC ? pC : pB;
        {
            // rows n0 + threadIdx.y + 8 k, k < 4; steps t .. t + 3
            const int t = t0 + 4 * threadIdx.x;
            float4 acc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (t < seqlen) {
#pragma unroll 2
                for (int hh = gg * hpg; hh < (gg + 1) * hpg; ++hh) {
                    const float* p0 =
                        src + (((long long)hh * batch + bb) * kNs + n0 + threadIdx.y) * L + t;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 v = *reinterpret_cast<const float4*>(p0 + 8 * k * L);
                        acc[k].x += v.x; acc[k].y += v.y; acc[k].z += v.z; acc[k].w += v.w;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float* row = &tile[threadIdx.y + 8 * k][4 * threadIdx.x];
                row[0] = acc[k].x; row[1] = acc[k].y; row[2] = acc[k].z; row[3] = acc[k].w;
            }
        }
        __syncthreads();
        float* dst = isC ? dC : dB;
        for (int r = threadIdx.y; r < 128; r += blockDim.y) {
            const int t = t0 + r, n = n0 + threadIdx.x;
            if (t < seqlen) dst[(((long long)bb * L + t) * ngroups + gg) * kNs + n] = tile[threadIdx.x][r];
        }
        __syncthreads();
    }
}

// dA = the per-(batch, head) sums added over the batch, in batch order.
__global__ void ssd_bwd_reduce_a_kernel(const float* __restrict__ pA, float* __restrict__ dA,
                                        int batch, int nheads) {
    for (int hh = blockIdx.x * blockDim.x + threadIdx.x; hh < nheads; hh += gridDim.x * blockDim.x) {
        float acc = 0.0f;
        for (int bb = 0; bb < batch; ++bb) acc += pA[(long long)bb * nheads + hh];
        dA[hh] = acc;
    }
}

struct BwdWs {
    size_t header, bstates, pb, pc, pa, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

BwdWs bwd_workspace(int batch, int seqlen, int nheads) {
    BwdWs w{};
    const size_t items = (size_t)batch * nheads;
    const size_t nblocks = ((size_t)seqlen + kQ - 1) / kQ;
    w.header = 256;
    w.bstates = round256(items * (nblocks + 1) * kP * kNs * 4);
    w.pb = round256((size_t)nheads * batch * seqlen * kNs * 4);
    w.pc = w.pb;
    w.pa = round256(items * 4);
    w.total = w.header + w.bstates + w.pb + w.pc + w.pa;
    return w;
}

using MakeStates = std::function<ssm_status_t(float*)>;

// Steps 1-3 of the gradient, after validation: block states (from
// `block_states`, else by `make_states` when given, else by the Mamba-2
// forward), the reverse block walk with input weights `wts` (NULL: dt; with
// weights, `dw` receives their gradient and ddt only the log-decay part), and
// the fixed-order sums.  The workspace holds bwd_workspace(...).total bytes.

// Mamba-3's diagonal correction of dx (BwdArgs::corr_*); g = NULL: none.
struct DxCorr {
    const float* g = nullptr;
    const float* dt = nullptr;
    const float* lam = nullptr;
    int steps = 0;
};

ssm_status_t run_bwd(const void* x, const float* dt, const float* wts, const float* A_head,
                     const void* B, const void* C, const float* initial_state, const void* dy,
                     const float* dfinal_state, const float* block_states,
                     const MakeStates& make_states, float* dx, float* ddt, float* dw,
                     float* dA_head, float* dB, float* dC, float* dinitial_state, int batch,
                     int seqlen, int nheads, int ngroups, void* workspace, cudaStream_t s,
                     int rank = 1, const DxCorr& corr = DxCorr{}) {
    const size_t items = (size_t)batch * nheads;
    const BwdWs w = bwd_workspace(batch, seqlen, nheads);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (cudaMemsetAsync(ws, 0, w.header, s) != cudaSuccess) return SSM_ERR_CUDA;
    float* bstates = reinterpret_cast<float*>(ws + w.header);
    BwdArgs a{};
    a.dt = dt;
    a.w = wts;
    a.dw = dw;
    a.A = A_head;
    a.bstates = block_states ? block_states : bstates;
    a.dfinal = dfinal_state;
    a.dx = dx;
    a.ddt = ddt;
    a.dh0 = dinitial_state;
    a.pB = reinterpret_cast<float*>(ws + w.header + w.bstates);
    a.pC = reinterpret_cast<float*>(ws + w.header + w.bstates + w.pb);
    a.pA = reinterpret_cast<float*>(ws + w.header + w.bstates + w.pb + w.pc);
    a.status = reinterpret_cast<uint32_t*>(ws + 4);  // the header's status word
    a.batch = batch;
    a.seqlen = seqlen;
    a.nheads = nheads;
    a.ngroups = ngroups;
    a.corr_g = corr.g;
    a.corr_dt = corr.dt;
    a.corr_lam = corr.lam;
    a.corr_steps = corr.steps;

    // 1. the state entering every block (and the final state), unless the
    // forward kept them
    if (!block_states) {
        const ssm_status_t rc =
            make_states ? make_states(bstates)
                        : ssd_internal::ssd_forward_block_states(x, dt, A_head, B, C, initial_state,
                                                                 bstates, batch, seqlen, nheads,
                                                                 ngroups, s);
        if (rc != SSM_OK) return rc;
    }
    // 2. the blocks in reverse, one CTA per (batch, head)
    CUtensorMap mc, mb, mx, mdy;
    if (!ssd_host::make_bc_map(&mc, C, batch, seqlen, ngroups) ||
        !ssd_host::make_bc_map(&mb, B, batch, seqlen, ngroups) ||
        !ssd_host::make_x_map(&mx, x, batch, seqlen, nheads) ||
        !ssd_host::make_x_map(&mdy, dy, batch, seqlen, nheads))
        return SSM_ERR_CUDA;
    auto kern = rank == 4   ? ssd_bwd_kernel<4, true>
                : rank == 2 ? ssd_bwd_kernel<2, true>
                : corr.g    ? ssd_bwd_kernel<1, true>
                            : ssd_bwd_kernel<1, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    kern<<<(unsigned)items, kThreads, kSmemAlloc, s>>>(mc, mb, mx, mdy, a);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    // 3. sums over a group's heads and over the batch
    {
        const dim3 grid((unsigned)((seqlen + 127) / 128), kNs / 32,
                        (unsigned)std::min<long long>(2LL * batch * ngroups, 65535));
        ssd_bwd_reduce_bc_kernel<<<grid, dim3(32, 8), 0, s>>>(a.pB, a.pC, dB, dC, batch, seqlen,
                                                             nheads, ngroups);
        if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
        ssd_bwd_reduce_a_kernel<<<(unsigned)((nheads + 127) / 128), 128, 0, s>>>(a.pA, dA_head,
                                                                                batch, nheads);
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" size_t ssd_chunked_bwd_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                                  int dstate, int ngroups) {
    if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups < 1 || headdim != kP || dstate != kNs ||
        nheads % ngroups != 0)
        return 0;
    return bwd_workspace(batch, seqlen, nheads).total;
}

extern "C" ssm_status_t ssd_chunked_bwd(const void* x, const float* dt, const float* A_head,
                                        const void* B, const void* C, int chunk,
                                        const float* initial_state, const void* dy,
                                        const float* dfinal_state, const float* block_states,
                                        float* dx, float* ddt,
                                        float* dA_head, float* dB, float* dC,
                                        float* dinitial_state, int batch, int seqlen, int nheads,
                                        int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype)) return SSM_ERR_DTYPE;
    if (chunk != 64 || headdim != kP || dstate != kNs || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    if ((size_t)batch * nheads > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    const size_t items = (size_t)batch * nheads;
    const size_t steps = (size_t)batch * seqlen;
    const size_t sb = items * headdim * dstate * 4;
    if (nheads > 0 && !dA_head) return SSM_ERR_NULL;
    const bool work = items > 0 && seqlen > 0;
    if (work && (!x || !dt || !A_head || !B || !C || !dy || !dx || !ddt || !dB || !dC))
        return SSM_ERR_NULL;
    if (work && !workspace) return SSM_ERR_WORKSPACE;
    const void* ptrs[] = {x, dt, A_head, B, C, initial_state, dy, dfinal_state, block_states, dx,
                          ddt, dA_head, dB, dC, dinitial_state, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = steps * nheads * headdim * 2, bcb = steps * ngroups * dstate * 2;
    struct R { const void* p; size_t n; };
    const R ins[] = {{x, xb}, {dt, steps * nheads * 4}, {A_head, (size_t)nheads * 4}, {B, bcb},
                     {C, bcb}, {initial_state, initial_state ? sb : 0}, {dy, xb},
                     {dfinal_state, dfinal_state ? sb : 0},
                     {block_states,
                      block_states ? sb * (((size_t)seqlen + kQ - 1) / kQ + 1) : 0}};
    const R outs[] = {{dx, steps * nheads * headdim * 4}, {ddt, steps * nheads * 4},
                      {dA_head, (size_t)nheads * 4}, {dB, bcb * 2}, {dC, bcb * 2},
                      {dinitial_state, dinitial_state ? sb : 0}};
    constexpr int kOuts = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < kOuts; ++i) {
        for (const R& r : ins)
            if (overlaps(outs[i].p, outs[i].n, r.p, r.n)) return SSM_ERR_ALIAS;
        for (int j = i + 1; j < kOuts; ++j)
            if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_ALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!work) {
        // no step: dA = 0 and the adjoint passes through to the initial state
        if (nheads > 0 && cudaMemsetAsync(dA_head, 0, (size_t)nheads * 4, s) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (dinitial_state && sb) {
            const cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, sb,
                                                                 cudaMemcpyDeviceToDevice, s)
                                               : cudaMemsetAsync(dinitial_state, 0, sb, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const BwdWs w = bwd_workspace(batch, seqlen, nheads);
    if (workspace_bytes < w.total) return SSM_ERR_WORKSPACE;
    for (const R& r : ins)
        if (overlaps(workspace, w.total, r.p, r.n)) return SSM_ERR_ALIAS;
    for (const R& r : outs)
        if (overlaps(workspace, w.total, r.p, r.n)) return SSM_ERR_ALIAS;

    return run_bwd(x, dt, nullptr, A_head, B, C, initial_state, dy, dfinal_state, block_states,
                   MakeStates(), dx, ddt, nullptr, dA_head, dB, dC, dinitial_state, batch, seqlen,
                   nheads, ngroups, workspace, s);
}

// ------------------------------------------------ Mamba-3 SISO gradient
//
// The three-term recurrence of "Mamba-3 NKI Kernels for AWS Neuron" (section
// "How it works", Eq. 9), h_t = alpha_t h_{t-1} + beta_t u_{t-1} + gamma_t u_t
// with u_t = B_t (x) x_t, is the Mamba-2 SSD recurrence of
//   s_t = h_t + c_t u_t,   c_t = dt_{t+1} (1 - lambda_{t+1})  (0 at the last step):
//   s_t = alpha_t s_{t-1} + w_t u_t,   w_t = gamma_t + c_t  (the page's "scale"),
//   y_t = C_t . s_t - c_t (C_t . B_t) x_t  (its diagonal correction),
//   s_{-1} = h_init + c_{-1} prev_B (x) prev_x,  c_{-1} = dt_0 (1 - lambda_0),
//   and s_{L-1} = h_{L-1}.
// So the gradient is the SSD gradient with input weights w, from the block
// states the Mamba-3 forward carries (which are s), plus the correction
// term's, taken through w, c and s_{-1} back to dt, lambda, x, B, C and the
// previous token:
//   dc_t      = dw_t - (C_t . B_t)(x_t . dy_t),   dc_{-1} = <dS_init, prev_B (x) prev_x>
//   ddt_t     = A sum_{i >= t} d cs_i + lambda_t dw_t + (1 - lambda_t) dc_{t-1}
//   dlambda_t = dt_t dw_t - dt_t dc_{t-1}
//   dx_t     -= c_t (C_t . B_t) dy_t
//   dB_t     -= (sum_h c_t x_t . dy_t) C_t,   dC_t -= (sum_h c_t x_t . dy_t) B_t
//   dh_init = dS_init, dprev_x = c_{-1} dS_init prev_B, dprev_B = sum_h c_{-1} dS_init^T prev_x.

namespace {

// w[b,t,h] = lambda_t dt_t + dt_{t+1} (1 - lambda_{t+1}), the second term 0 at
// the last step.
__global__ void m3_weights_kernel(const float* __restrict__ dt, const float* __restrict__ lam,
                                  float* __restrict__ w, int batch, int seqlen, int nheads) {
    const long long n = (long long)batch * seqlen * nheads;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)((i / nheads) % seqlen);
        float v = lam[i] * dt[i];
        if (t + 1 < seqlen) v = fmaf(dt[i + nheads], 1.0f - lam[i + nheads], v);
        w[i] = v;
    }
}

__device__ __forceinline__ void unpack8(uint4 w, float (&v)[8]) {
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

// The per-step rank dots: for every (step, head) the R x R products
// XD[r'][r] = x_{t,r'} . dy_{t,r} over headdim, and for every (step, group)
// G[r][r'] = C_{t,r} . B_{t,r'} over dstate.  Eight lanes take one item, each
// a 16-byte vector of every row (x, dy: 8 of 64 elements; B, C: 16 of 128 in
// two passes); the R^2 partial dots are reduce-scattered over the 8 lanes
// (rank 4: 14 shuffles, each lane stores 2 of them; rank 2: 4 shuffles, one
// lane of each pair stores; rank 1, the single-input gradient's x.dy and
// C.B: 3 shuffles, one lane of the 8 stores).
template <int RK>
__global__ void m3m_dots_kernel(const __nv_bfloat16* __restrict__ x,
                                const __nv_bfloat16* __restrict__ dy,
                                const __nv_bfloat16* __restrict__ B,
                                const __nv_bfloat16* __restrict__ C, float* __restrict__ XD,
                                float* __restrict__ G, int batch, int seqlen, int nheads,
                                int ngroups) {
    constexpr int R2 = RK * RK;
    static_assert(R2 == 1 || R2 == 4 || R2 == 16, "ranks 1, 2, 4");
    constexpr int kLanes = 8;
    const long long steps = (long long)batch * seqlen;
    const long long nx = steps * nheads, nb = steps * ngroups;
    const int sub = threadIdx.x & (kLanes - 1);  // lane within the item
    // whole warps step together (4 items each), so every shuffle has all lanes
    const long long wstride = ((long long)gridDim.x * blockDim.x) / 32 * 4;
    const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32 * 4;
    for (long long qw = w0; qw < nx + nb; qw += wstride) {
        const long long q = qw + (threadIdx.x & 31) / kLanes;
        float acc[R2];
#pragma unroll
        for (int k = 0; k < R2; ++k) acc[k] = 0.0f;
        if (q >= nx + nb) {
            // past the last item: zeros through the shuffles, nothing stored
        } else if (q < nx) {
            const long long bt = q / nheads;
            const int h = (int)(q % nheads);
            float a[RK][8], d[RK][8];
#pragma unroll
            for (int r = 0; r < RK; ++r) {
                const long long row = ((bt * RK + r) * nheads + h) * kP + 8 * sub;
                unpack8(__ldg(reinterpret_cast<const uint4*>(x + row)), a[r]);
                unpack8(__ldg(reinterpret_cast<const uint4*>(dy + row)), d[r]);
            }
#pragma unroll
            for (int rp = 0; rp < RK; ++rp)
#pragma unroll
                for (int r = 0; r < RK; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[rp * RK + r] = fmaf(a[rp][e], d[r][e], acc[rp * RK + r]);
        } else {
            const long long q2 = q - nx;
            const long long bt = q2 / ngroups;
            const int g = (int)(q2 % ngroups);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float bw[RK][8], cw[RK][8];
#pragma unroll
                for (int r = 0; r < RK; ++r) {
                    const long long row = ((bt * RK + r) * ngroups + g) * kNs + 64 * half + 8 * sub;
                    unpack8(__ldg(reinterpret_cast<const uint4*>(B + row)), bw[r]);
                    unpack8(__ldg(reinterpret_cast<const uint4*>(C + row)), cw[r]);
                }
#pragma unroll
                for (int r = 0; r < RK; ++r)
#pragma unroll
                    for (int rp = 0; rp < RK; ++rp)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[r * RK + rp] = fmaf(cw[r][e], bw[rp][e], acc[r * RK + rp]);
            }
        }
        // reduce-scatter over the item's 8 lanes (lane bits 2, 1, 0): afterwards
        // a lane holds the totals of R2 / 8 values from index base (R2 >= 8), or
        // of value base, shared by 8 / R2 lanes of which the lowest stores it
        int base = 0;
        int n = R2;
#pragma unroll
        for (int m = 4; m >= 1; m >>= 1) {
            if (n == 1) {
                acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], m);
                continue;
            }
            n >>= 1;
            const bool hi = sub & m;
#pragma unroll
            for (int k = 0; k < R2 / 2; ++k) {
                if (k < n) {
                    const float send = hi ? acc[k] : acc[k + n];
                    const float keep = hi ? acc[k + n] : acc[k];
                    acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            if (hi) base += n;
        }
        if (q >= nx + nb) continue;
        float* out = q < nx ? XD + q * R2 : G + (q - nx) * R2;
        if constexpr (R2 >= 8) {
            constexpr int per = R2 / 8;
#pragma unroll
            for (int k = 0; k < per; ++k) out[base + k] = acc[k];
        } else {
            if ((sub & (8 / R2 - 1)) == 0) out[base] = acc[0];
        }
    }
}

// The previous token, per (b, h), from dS = dL/ds_{-1} [64 p][128 n] and
// c0 = dt_0 (1 - lambda_0), all RK ranks in one pass over dS (RK = 1: the
// single-input gradient):
//   dprev_x[b,r,h,p] = c0 sum_n dS[p,n] prev_B[b,r,g,n],
//   pprevB[b,h,r,n]  = c0 sum_p dS[p,n] prev_x[b,r,h,p] (summed over the group next),
//   dc0[b,h]         = sum_r sum_p prev_x[b,r,h,p] sum_n dS[p,n] prev_B[b,r,g,n].
// 128 threads: dS staged in shared memory, thread n for the column sums, a
// thread pair per row for the row sums.
template <int RK>
__global__ void __launch_bounds__(kNs) m3m_prev_kernel(const float* __restrict__ dS,
                                                     const __nv_bfloat16* __restrict__ prev_B,
                                                     const __nv_bfloat16* __restrict__ prev_x,
                                                     const float* __restrict__ dt,
                                                     const float* __restrict__ lam,
                                                     float* __restrict__ dprev_x,
                                                     float* __restrict__ pprevB,
                                                     float* __restrict__ dc0, int batch,
                                                     int seqlen, int nheads, int ngroups) {
    // dS[p][n] staged with rows of kNs + 2 floats: the column pass (thread n)
    // and the row pass (a thread pair per row p, split by the parity of n)
    // both read distinct banks
    constexpr int kRow = kNs + 2;
    __shared__ float Ss[kP * kRow];
    __shared__ float pb[RK][kNs], px[RK][kP], red[kNs / 32];
    const int item = blockIdx.x, b = item / nheads, h = item % nheads;
    const int g = h / (nheads / ngroups);
    const int tid = threadIdx.x;
    const long long i0 = (long long)b * seqlen * nheads + h;
    const float c0 = dt[i0] * (1.0f - lam[i0]);
    {
        const float4* S4 = reinterpret_cast<const float4*>(dS + (long long)item * kP * kNs);
        constexpr int kVec = kP * kNs / 4 / kNs;  // float4 loads per thread
        float4 v[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) v[j] = __ldg(S4 + tid + j * kNs);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int e = (tid + j * kNs) * 4, pp = e / kNs, n = e % kNs;
            float* d = Ss + pp * kRow + n;
            d[0] = v[j].x; d[1] = v[j].y; d[2] = v[j].z; d[3] = v[j].w;
        }
    }
#pragma unroll
    for (int r = 0; r < RK; ++r) {
        pb[r][tid] = __bfloat162float(prev_B[(((long long)b * RK + r) * ngroups + g) * kNs + tid]);
        if (tid < kP) px[r][tid] = __bfloat162float(prev_x[(((long long)b * RK + r) * nheads + h) * kP + tid]);
    }
    __syncthreads();
    // pprevB[r][n] = c0 sum_p dS[p][n] prev_x[r][p]
    {
        float col[RK];
#pragma unroll
        for (int r = 0; r < RK; ++r) col[r] = 0.0f;
#pragma unroll 8
        for (int pp = 0; pp < kP; ++pp) {
            const float sv = Ss[pp * kRow + tid];
#pragma unroll
            for (int r = 0; r < RK; ++r) col[r] = fmaf(sv, px[r][pp], col[r]);
        }
#pragma unroll
        for (int r = 0; r < RK; ++r) pprevB[((long long)item * RK + r) * kNs + tid] = c0 * col[r];
    }
    // dprev_x[r][p] = c0 sum_n dS[p][n] prev_B[r][n]: row p = tid / 2, n of
    // parity tid % 2, the pair combined by one shuffle
    {
        const int pp = tid >> 1, par = tid & 1;
        float row[RK];
#pragma unroll
        for (int r = 0; r < RK; ++r) row[r] = 0.0f;
        const float* Sp = Ss + pp * kRow + par;
#pragma unroll 8
        for (int m = 0; m < kNs / 2; ++m) {
            const float sv = Sp[2 * m];
#pragma unroll
            for (int r = 0; r < RK; ++r) row[r] = fmaf(sv, pb[r][2 * m + par], row[r]);
        }
        float part = 0.0f;
#pragma unroll
        for (int r = 0; r < RK; ++r) {
            row[r] += __shfl_xor_sync(0xffffffffu, row[r], 1);
            if (par == 0) dprev_x[(((long long)b * RK + r) * nheads + h) * kP + pp] = c0 * row[r];
            part = fmaf(px[r][pp], row[r], part);
        }
        if (par) part = 0.0f;  // each row once
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((tid & 31) == 0) red[tid >> 5] = part;
    }
    __syncthreads();
    if (tid == 0) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kNs / 32; ++w) sum += red[w];
        dc0[item] = sum;
    }
}

// dprev_B[b,g,n] = the group's heads' pprevB, added in head order.
__global__ void m3_prev_b_kernel(const float* __restrict__ pprevB, float* __restrict__ dprev_B,
                                 int batch, int nheads, int ngroups) {
    const int hpg = nheads / ngroups;
    const long long n = (long long)batch * ngroups * kNs;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int nn = (int)(i % kNs);
        const long long bg = i / kNs;
        const int b = (int)(bg / ngroups), g = (int)(bg % ngroups);
        float acc = 0.0f;
        for (int h = g * hpg; h < (g + 1) * hpg; ++h)
            acc += pprevB[((long long)b * nheads + h) * kNs + nn];
        dprev_B[i] = acc;
    }
}

// One CTA per (b, t): ddt (holding the log-decay part on entry) and dlambda of
// every head, then dB, dC -= (sum over the group's heads of c_t x_t . dy_t)
// C_t, B_t.  (dx's term -c_t (C_t . B_t) dy_t is applied by the gradient
// kernel as it writes dx.)  Shared memory: nheads floats.
__global__ void m3_post_kernel(const float* __restrict__ dt, const float* __restrict__ lam,
                               const float* __restrict__ dw, const float* __restrict__ xd,
                               const float* __restrict__ cb, const float* __restrict__ dc0,
                               const __nv_bfloat16* __restrict__ B,
                               const __nv_bfloat16* __restrict__ C, float* __restrict__ ddt,
                               float* __restrict__ dlam, float* __restrict__ dB,
                               float* __restrict__ dC, int batch, int seqlen, int nheads,
                               int ngroups) {
    extern __shared__ float sm[];
    float* cx = sm;  // c_t (x_t . dy_t) per head
    const int hpg = nheads / ngroups;
    for (long long row = blockIdx.x; row < (long long)batch * seqlen; row += gridDim.x) {
        const int t = (int)(row % seqlen);
        const int b = (int)(row / seqlen);
        for (int h = threadIdx.x; h < nheads; h += blockDim.x) {
            const long long i = row * nheads + h;
            const int g = h / hpg;
            const float c = t + 1 < seqlen ? dt[i + nheads] * (1.0f - lam[i + nheads]) : 0.0f;
            float dcp = 0.0f;  // dL/dc_{t-1}
            if (t > 0) dcp = dw[i - nheads] - cb[(row - 1) * ngroups + g] * xd[i - nheads];
            else if (dc0) dcp = dc0[(long long)b * nheads + h];
            const float dwt = dw[i], l = lam[i], d = dt[i];
            ddt[i] = ddt[i] + l * dwt + (1.0f - l) * dcp;
            dlam[i] = d * dwt - d * dcp;
            cx[h] = c * xd[i];
        }
        __syncthreads();
        const long long bo = row * ngroups * kNs;
        for (int idx = threadIdx.x; idx < ngroups * kNs; idx += blockDim.x) {
            const int g = idx / kNs;
            float s = 0.0f;
            for (int h = g * hpg; h < (g + 1) * hpg; ++h) s += cx[h];
            dB[bo + idx] -= s * __bfloat162float(C[bo + idx]);
            dC[bo + idx] -= s * __bfloat162float(B[bo + idx]);
        }
        __syncthreads();
    }
}

struct M3Ws {
    size_t ssd, w, dw, xd, cb, ds, dc0, ppb, total;
};

M3Ws m3_workspace(int batch, int seqlen, int nheads, int ngroups) {
    M3Ws m{};
    const size_t steps = (size_t)batch * seqlen, items = (size_t)batch * nheads;
    m.ssd = bwd_workspace(batch, seqlen, nheads).total;
    m.w = round256(steps * nheads * 4);
    m.dw = m.w;
    m.xd = m.w;
    m.cb = round256(steps * ngroups * 4);
    m.ds = round256(items * kP * kNs * 4);
    m.dc0 = round256(items * 4);
    m.ppb = round256(items * kNs * 4);
    m.total = m.ssd + m.w + m.dw + m.xd + m.cb + m.ds + m.dc0 + m.ppb;
    return m;
}

unsigned grid_for(long long n, int threads) {
    return (unsigned)std::max<long long>(1, std::min<long long>((n + threads - 1) / threads, 65535));
}

}  // namespace

extern "C" size_t ssd_mamba3_bwd_workspace_bytes(int batch, int seqlen, int nheads, int headdim,
                                                 int dstate, int ngroups) {
    if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups < 1 || headdim != kP || dstate != kNs ||
        nheads % ngroups != 0)
        return 0;
    return m3_workspace(batch, seqlen, nheads, ngroups).total;
}

extern "C" ssm_status_t ssd_mamba3_bwd(const void* x, const float* dt, const float* lam,
                                       const float* A_head, const void* B, const void* C,
                                       int chunk, const float* initial_state, const void* prev_B,
                                       const void* prev_x, const void* dy,
                                       const float* dfinal_state, const float* block_states,
                                       float* dx, float* ddt,
                                       float* dlam, float* dA_head, float* dB, float* dC,
                                       float* dinitial_state, float* dprev_B, float* dprev_x,
                                       int batch, int seqlen, int nheads, int headdim,
                                       int dstate, int ngroups, ssm_dtype_t in_dtype,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype)) return SSM_ERR_DTYPE;
    if (chunk != 64 || headdim != kP || dstate != kNs || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    if ((size_t)batch * nheads > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    // the per-step kernel keeps two floats per head in shared memory (48 KB)
    if ((size_t)nheads * 2 * sizeof(float) > 48 * 1024) return SSM_ERR_UNSUPPORTED;
    if ((prev_B == nullptr) != (prev_x == nullptr)) return SSM_ERR_NULL;
    const bool has_prev = prev_B != nullptr;
    const size_t items = (size_t)batch * nheads;
    const size_t steps = (size_t)batch * seqlen;
    const size_t sb = items * headdim * dstate * 4;
    if (nheads > 0 && !dA_head) return SSM_ERR_NULL;
    if (has_prev && items > 0 && (!dprev_B || !dprev_x)) return SSM_ERR_NULL;
    const bool work = items > 0 && seqlen > 0;
    if (work && (!x || !dt || !lam || !A_head || !B || !C || !dy || !dx || !ddt || !dlam ||
                 !dB || !dC))
        return SSM_ERR_NULL;
    if (work && !workspace) return SSM_ERR_WORKSPACE;
    const void* ptrs[] = {x, dt, lam, A_head, B, C, initial_state, prev_B, prev_x, dy,
                          dfinal_state, block_states, dx, ddt, dlam, dA_head, dB, dC,
                          dinitial_state, dprev_B, dprev_x, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = steps * nheads * headdim * 2, bcb = steps * ngroups * dstate * 2;
    const size_t pbb = (size_t)batch * ngroups * dstate, pxb = items * headdim;
    const size_t bsb = block_states ? sb * (((size_t)seqlen + kQ - 1) / kQ + 1) : 0;
    struct R { const void* p; size_t n; };
    const R ins[] = {{x, xb}, {dt, steps * nheads * 4}, {lam, steps * nheads * 4},
                     {A_head, (size_t)nheads * 4}, {B, bcb}, {C, bcb},
                     {initial_state, initial_state ? sb : 0}, {prev_B, has_prev ? pbb * 2 : 0},
                     {prev_x, has_prev ? pxb * 2 : 0}, {dy, xb},
                     {dfinal_state, dfinal_state ? sb : 0}, {block_states, bsb}};
    const R outs[] = {{dx, steps * nheads * headdim * 4}, {ddt, steps * nheads * 4},
                      {dlam, steps * nheads * 4}, {dA_head, (size_t)nheads * 4},
                      {dB, bcb * 2}, {dC, bcb * 2}, {dinitial_state, dinitial_state ? sb : 0},
                      {dprev_B, has_prev ? pbb * 4 : 0}, {dprev_x, has_prev ? pxb * 4 : 0}};
    constexpr int kOuts = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < kOuts; ++i) {
        for (const R& r : ins)
            if (overlaps(outs[i].p, outs[i].n, r.p, r.n)) return SSM_ERR_ALIAS;
        for (int j = i + 1; j < kOuts; ++j)
            if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_ALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!work) {
        // no step: dA = 0, the adjoint passes through to the initial state and
        // the previous token never enters
        if (nheads > 0 && cudaMemsetAsync(dA_head, 0, (size_t)nheads * 4, s) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (dinitial_state && sb) {
            const cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, sb,
                                                                 cudaMemcpyDeviceToDevice, s)
                                               : cudaMemsetAsync(dinitial_state, 0, sb, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        if (has_prev && items > 0) {
            if (cudaMemsetAsync(dprev_B, 0, pbb * 4, s) != cudaSuccess ||
                cudaMemsetAsync(dprev_x, 0, pxb * 4, s) != cudaSuccess)
                return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const M3Ws m = m3_workspace(batch, seqlen, nheads, ngroups);
    if (workspace_bytes < m.total) return SSM_ERR_WORKSPACE;
    for (const R& r : ins)
        if (overlaps(workspace, m.total, r.p, r.n)) return SSM_ERR_ALIAS;
    for (const R& r : outs)
        if (overlaps(workspace, m.total, r.p, r.n)) return SSM_ERR_ALIAS;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* w = reinterpret_cast<float*>(ws + m.ssd);
    float* dw = reinterpret_cast<float*>(ws + m.ssd + m.w);
    float* xd = reinterpret_cast<float*>(ws + m.ssd + m.w + m.dw);
    float* cb = reinterpret_cast<float*>(ws + m.ssd + m.w + m.dw + m.xd);
    float* dS = reinterpret_cast<float*>(ws + m.ssd + m.w + m.dw + m.xd + m.cb);
    float* dc0 = reinterpret_cast<float*>(ws + m.ssd + m.w + m.dw + m.xd + m.cb + m.ds);
    float* ppb = reinterpret_cast<float*>(ws + m.ssd + m.w + m.dw + m.xd + m.cb + m.ds + m.dc0);
    float* dS_out = dinitial_state ? dinitial_state : (has_prev ? dS : nullptr);

    // 1. the input weights w = gamma + c
    const long long nw = (long long)steps * nheads;
    m3_weights_kernel<<<grid_for(nw, 256), 256, 0, s>>>(dt, lam, w, batch, seqlen, nheads);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    const MakeStates states = [&](float* bs) {
        return ssd_internal::ssd_mamba3_forward_block_states(x, dt, lam, A_head, B, C,
                                                             initial_state, prev_B, prev_x, bs,
                                                             batch, seqlen, nheads, ngroups, s);
    };
    // 2. x . dy per head and C . B per group, every step (inputs only; C . B
    // feeds the diagonal correction the gradient kernel applies to dx)
    const long long nrows = (long long)steps * (nheads + ngroups);
    m3m_dots_kernel<1><<<grid_for(nrows * 8, 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(dy),
        static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), xd, cb,
        batch, seqlen, nheads, ngroups);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    // 3. the SSD gradient with weights w from the Mamba-3 forward's block states
    DxCorr corr;
    corr.g = cb;
    corr.dt = dt;
    corr.lam = lam;
    corr.steps = seqlen;
    ssm_status_t rc = run_bwd(x, dt, w, A_head, B, C, initial_state, dy, dfinal_state,
                              block_states, states, dx, ddt, dw, dA_head, dB, dC, dS_out, batch,
                              seqlen, nheads, ngroups, workspace, s, 1, corr);
    if (rc != SSM_OK) return rc;
    // 4. the previous token's gradients and dL/dc_{-1}
    if (has_prev) {
        m3m_prev_kernel<1><<<(unsigned)items, kNs, 0, s>>>(
            dS_out, static_cast<const __nv_bfloat16*>(prev_B),
            static_cast<const __nv_bfloat16*>(prev_x), dt, lam, dprev_x, ppb, dc0, batch, seqlen,
            nheads, ngroups);
        if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
        m3_prev_b_kernel<<<grid_for((long long)pbb, 256), 256, 0, s>>>(ppb, dprev_B, batch,
                                                                       nheads, ngroups);
        if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    }
    // 5. ddt, dlambda and the diagonal correction's terms
    m3_post_kernel<<<(unsigned)std::min<long long>((long long)steps, 65535), 256,
                     nheads * sizeof(float), s>>>(
        dt, lam, dw, xd, cb, has_prev ? dc0 : nullptr, static_cast<const __nv_bfloat16*>(B),
        static_cast<const __nv_bfloat16*>(C), ddt, dlam, dB, dC, batch, seqlen, nheads, ngroups);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// ------------------------------------------------ Mamba-3 MIMO gradient
//
// The rank-R recurrence (section "Kernel details", mamba3_mimo_ssd_kernel:
// BX_t = sum_r B_{t,r} (x) x_{t,r}, S = alpha_t S + beta_t BX_{t-1} + gamma_t BX_t,
// y_{t,r} = C_{t,r} . S) is taken the same way over sub-tokens (t, r): s_t =
// h_t + c_t BX_t is the SSD state of the sub-token sequence with the step's dt
// on its first sub-token (0 on the others), the weight w_t on every one and a
// block-lower-triangular mask (a sub-token sees its whole step), and
//   y_{t,r} = C_{t,r} . s_t - c_t sum_r' (C_{t,r} . B_{t,r'}) x_{t,r'},
//   s_{-1} = h_init + c_{-1} sum_r prev_B_r (x) prev_x_r.
// With G_{rr'} = C_{t,r} . B_{t,r'} (per group) and XD_{r'r} = x_{t,r'} . dy_{t,r}
// (per head), the correction adds
//   dx_{t,r'} -= c_t sum_r G_{rr'} dy_{t,r},  dB_{t,r'} -= c_t sum_h sum_r XD_{r'r} C_{t,r},
//   dC_{t,r} -= c_t sum_h sum_r' XD_{r'r} B_{t,r'},  dc_t -= sum_{r,r'} G_{rr'} XD_{r'r};
// dw_t is the sum of its sub-tokens' weight gradients, and ddt, dlambda follow
// as for SISO.

namespace {

// Per sub-token row (b, t R + r, h): the step's dt on r = 0 (0 otherwise) and
// its weight w_t = lambda_t dt_t + dt_{t+1} (1 - lambda_{t+1}) on every rank.
__global__ void m3m_expand_kernel(const float* __restrict__ dt, const float* __restrict__ lam,
                                  float* __restrict__ dts, float* __restrict__ wts, int batch,
                                  int seqlen, int rank, int nheads) {
    const long long n = (long long)batch * seqlen * rank * nheads;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int h = (int)(i % nheads);
        const int r = (int)((i / nheads) % rank);
        const long long bt = i / ((long long)nheads * rank);
        const int t = (int)(bt % seqlen);
        const long long src = bt * nheads + h;
        float w = lam[src] * dt[src];
        if (t + 1 < seqlen) w = fmaf(dt[src + nheads], 1.0f - lam[src + nheads], w);
        dts[i] = r == 0 ? dt[src] : 0.0f;
        wts[i] = w;
    }
}

// XD[bt][h][r'][r] = x_{t,r'} . dy_{t,r} (over p) and G[bt][g][r][r'] =
// C_{t,r} . B_{t,r'} (over n): one warp per (step, head) or (step, group) row
// reads its RK x (or C) and RK dy (or B) rows once and forms all RK^2 dots,
// each summed over the lanes by a fixed butterfly.

// dprev_B[b,r,g,n] = the group's heads' pprevB, added in head order.
__global__ void m3m_prev_b_kernel(const float* __restrict__ pprevB, float* __restrict__ dprev_B,
                                  int batch, int rank, int nheads, int ngroups) {
    const int hpg = nheads / ngroups;
    const long long n = (long long)batch * rank * ngroups * kNs;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int nn = (int)(i % kNs);
        const int g = (int)((i / kNs) % ngroups);
        const int r = (int)((i / ((long long)kNs * ngroups)) % rank);
        const int b = (int)(i / ((long long)kNs * ngroups * rank));
        float acc = 0.0f;
        for (int h = g * hpg; h < (g + 1) * hpg; ++h)
            acc += pprevB[(((long long)b * nheads + h) * rank + r) * kNs + nn];
        dprev_B[i] = acc;
    }
}

// One CTA per (b, t): ddt and dlambda of every head (the step's log-decay part
// from its first sub-token row, dw summed over its ranks), then the
// correction's terms in dB and dC (c XD summed over the group's heads first,
// in head order).  The correction's term in dx is applied by the gradient
// kernel as it writes dx.  Shared memory: (nheads + ngroups) R^2 floats.
template <int RK>
__global__ void m3m_post_kernel(const float* __restrict__ dt, const float* __restrict__ lam,
                                const float* __restrict__ dw_rows,
                                const float* __restrict__ ddec_rows, const float* __restrict__ XD,
                                const float* __restrict__ G, const float* __restrict__ dc0,
                                const __nv_bfloat16* __restrict__ B,
                                const __nv_bfloat16* __restrict__ C, float* __restrict__ ddt,
                                float* __restrict__ dlam, float* __restrict__ dB,
                                float* __restrict__ dC, int batch, int seqlen, int nheads,
                                int ngroups) {
    extern __shared__ float sm[];
    constexpr int R2 = RK * RK;
    float* cX = sm;                // [h][r'][r] c_t XD_{r'r}
    float* sX = sm + nheads * R2;  // [g][r'][r] sum over the group's heads of cX
    const int hpg = nheads / ngroups;
    for (long long bt = blockIdx.x; bt < (long long)batch * seqlen; bt += gridDim.x) {
        const int t = (int)(bt % seqlen);
        const int b = (int)(bt / seqlen);
        for (int h = threadIdx.x; h < nheads; h += blockDim.x) {
            const long long i = bt * nheads + h;
            const int g = h / hpg;
            const float c = t + 1 < seqlen ? dt[i + nheads] * (1.0f - lam[i + nheads]) : 0.0f;
            float dwt = 0.0f, dwp = 0.0f;
#pragma unroll
            for (int r = 0; r < RK; ++r) {
                dwt += dw_rows[(bt * RK + r) * nheads + h];
                if (t > 0) dwp += dw_rows[((bt - 1) * RK + r) * nheads + h];
            }
            float dcp = 0.0f;  // dL/dc_{t-1}
            if (t > 0) {
                const float* Gp = G + ((bt - 1) * ngroups + g) * R2;
                const float* Xp = XD + ((bt - 1) * nheads + h) * R2;
                float corr = 0.0f;
#pragma unroll
                for (int r = 0; r < RK; ++r)
#pragma unroll
                    for (int rp = 0; rp < RK; ++rp)
                        corr = fmaf(Gp[r * RK + rp], Xp[rp * RK + r], corr);
                dcp = dwp - corr;
            } else if (dc0) {
                dcp = dc0[(long long)b * nheads + h];
            }
            const float l = lam[i], d = dt[i];
            ddt[i] = ddec_rows[(bt * RK) * nheads + h] + l * dwt + (1.0f - l) * dcp;
            dlam[i] = d * dwt - d * dcp;
            const float* Xp = XD + (bt * nheads + h) * R2;
#pragma unroll
            for (int k = 0; k < R2; ++k) cX[h * R2 + k] = c * Xp[k];
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < ngroups * R2; idx += blockDim.x) {
            const int g = idx / R2, k = idx % R2;
            float acc = 0.0f;
            for (int h = g * hpg; h < (g + 1) * hpg; ++h) acc += cX[h * R2 + k];
            sX[idx] = acc;
        }
        __syncthreads();
        // dB_{t,r'} -= sum_r sX_{r'r} C_{t,r};  dC_{t,r} -= sum_r' sX_{r'r} B_{t,r'}
        for (int idx = threadIdx.x; idx < RK * ngroups * kNs; idx += blockDim.x) {
            const int n = idx % kNs, g = (idx / kNs) % ngroups, ra = idx / (kNs * ngroups);
            float accB = 0.0f, accC = 0.0f;
#pragma unroll
            for (int r = 0; r < RK; ++r) {
                accB = fmaf(sX[g * R2 + ra * RK + r],
                            __bfloat162float(C[((bt * RK + r) * ngroups + g) * kNs + n]), accB);
                accC = fmaf(sX[g * R2 + r * RK + ra],
                            __bfloat162float(B[((bt * RK + r) * ngroups + g) * kNs + n]), accC);
            }
            dB[((bt * RK + ra) * ngroups + g) * kNs + n] -= accB;
            dC[((bt * RK + ra) * ngroups + g) * kNs + n] -= accC;
        }
        __syncthreads();
    }
}

struct M3mWs {
    size_t ssd, dts, wts, dw, ddec, xd, g, ds, dc0, ppb, total;
};

M3mWs m3m_workspace(int batch, int seqlen, int rank, int nheads, int ngroups) {
    M3mWs m{};
    const size_t steps = (size_t)batch * seqlen, items = (size_t)batch * nheads;
    m.ssd = bwd_workspace(batch, seqlen * rank, nheads).total;
    m.dts = round256(steps * rank * nheads * 4);
    m.wts = m.dts;
    m.dw = m.dts;
    m.ddec = m.dts;
    m.xd = round256(steps * nheads * rank * rank * 4);
    m.g = round256(steps * ngroups * rank * rank * 4);
    m.ds = round256(items * kP * kNs * 4);
    m.dc0 = round256(items * 4);
    m.ppb = round256(items * rank * kNs * 4);
    m.total = m.ssd + m.dts + m.wts + m.dw + m.ddec + m.xd + m.g + m.ds + m.dc0 + m.ppb;
    return m;
}

// Step 3 of the MIMO gradient for rank RK: the per-step rank dots x . dy and
// C . B (inputs only, so they run before the gradient kernel, which applies
// the diagonal correction to dx from them).
template <int RK>
ssm_status_t m3m_dots(const void* x, const void* B, const void* C, const void* dy, float* XD,
                      float* Gd, int batch, int seqlen, int nheads, int ngroups, cudaStream_t s) {
    const long long nrows = (long long)batch * seqlen * (nheads + ngroups);
    m3m_dots_kernel<RK><<<grid_for(nrows * 8, 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(dy),
        static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), XD, Gd,
        batch, seqlen, nheads, ngroups);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Steps 4-5 of the MIMO gradient for rank RK.
template <int RK>
ssm_status_t m3m_tail(const float* dt, const float* lam, const void* B, const void* C,
                      bool has_prev, const void* prev_B, const void* prev_x, const float* dS,
                      const float* dw, const float* ddec, const float* XD, const float* Gd,
                      float* dc0, float* ppb, float* ddt, float* dlam, float* dB, float* dC,
                      float* dprev_B, float* dprev_x, int batch, int seqlen, int nheads,
                      int ngroups, cudaStream_t s) {
    const long long steps = (long long)batch * seqlen;
    if (has_prev) {
        m3m_prev_kernel<RK><<<(unsigned)((long long)batch * nheads), kNs, 0, s>>>(
            dS, static_cast<const __nv_bfloat16*>(prev_B),
            static_cast<const __nv_bfloat16*>(prev_x), dt, lam, dprev_x, ppb, dc0, batch, seqlen,
            nheads, ngroups);
        if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
        m3m_prev_b_kernel<<<grid_for((long long)batch * RK * ngroups * kNs, 256), 256, 0, s>>>(
            ppb, dprev_B, batch, RK, nheads, ngroups);
        if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    }
    m3m_post_kernel<RK><<<(unsigned)std::min<long long>(steps, 65535), 256,
                          (nheads + ngroups) * RK * RK * sizeof(float), s>>>(
        dt, lam, dw, ddec, XD, Gd, has_prev ? dc0 : nullptr, static_cast<const __nv_bfloat16*>(B),
        static_cast<const __nv_bfloat16*>(C), ddt, dlam, dB, dC, batch, seqlen, nheads, ngroups);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" size_t ssd_mamba3_mimo_bwd_workspace_bytes(int batch, int seqlen, int rank, int nheads,
                                                      int headdim, int dstate, int ngroups) {
    if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups < 1 || headdim != kP || dstate != kNs ||
        nheads % ngroups != 0 || (rank != 1 && rank != 2 && rank != 4))
        return 0;
    return m3m_workspace(batch, seqlen, rank, nheads, ngroups).total;
}

extern "C" ssm_status_t ssd_mamba3_mimo_bwd(
    const void* x, const float* dt, const float* lam, const float* A_head, const void* B,
    const void* C, int chunk, int rank, const float* initial_state, const void* prev_B,
    const void* prev_x, const void* dy, const float* dfinal_state, const float* block_states,
    float* dx, float* ddt, float* dlam, float* dA_head, float* dB, float* dC,
    float* dinitial_state, float* dprev_B,
    float* dprev_x, int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups,
    ssm_dtype_t in_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1 || rank < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype)) return SSM_ERR_DTYPE;
    if ((rank != 1 && rank != 2 && rank != 4) || chunk * rank != 64 || headdim != kP ||
        dstate != kNs || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    if ((size_t)batch * nheads > (size_t)INT32_MAX ||
        (size_t)seqlen * rank > (size_t)INT32_MAX)
        return SSM_ERR_UNSUPPORTED;
    // the per-step kernel keeps (2 nheads + ngroups) rank^2 floats in shared memory (48 KB)
    if ((size_t)(2 * nheads + ngroups) * rank * rank * sizeof(float) > 48 * 1024)
        return SSM_ERR_UNSUPPORTED;
    if ((prev_B == nullptr) != (prev_x == nullptr)) return SSM_ERR_NULL;
    const bool has_prev = prev_B != nullptr;
    const size_t items = (size_t)batch * nheads;
    const size_t steps = (size_t)batch * seqlen, subs = steps * rank;
    const size_t sb = items * headdim * dstate * 4;
    if (nheads > 0 && !dA_head) return SSM_ERR_NULL;
    if (has_prev && items > 0 && (!dprev_B || !dprev_x)) return SSM_ERR_NULL;
    const bool work = items > 0 && seqlen > 0;
    if (work && (!x || !dt || !lam || !A_head || !B || !C || !dy || !dx || !ddt || !dlam ||
                 !dB || !dC))
        return SSM_ERR_NULL;
    if (work && !workspace) return SSM_ERR_WORKSPACE;
    const void* ptrs[] = {x, dt, lam, A_head, B, C, initial_state, prev_B, prev_x, dy,
                          dfinal_state, block_states, dx, ddt, dlam, dA_head, dB, dC,
                          dinitial_state, dprev_B, dprev_x, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = subs * nheads * headdim * 2, bcb = subs * ngroups * dstate * 2;
    const size_t bsb = block_states ? sb * (((size_t)seqlen * rank + kQ - 1) / kQ + 1) : 0;
    const size_t pbb = (size_t)batch * rank * ngroups * dstate,
                 pxb = (size_t)batch * rank * nheads * headdim;
    struct R { const void* p; size_t n; };
    const R ins[] = {{x, xb}, {dt, steps * nheads * 4}, {lam, steps * nheads * 4},
                     {A_head, (size_t)nheads * 4}, {B, bcb}, {C, bcb},
                     {initial_state, initial_state ? sb : 0}, {prev_B, has_prev ? pbb * 2 : 0},
                     {prev_x, has_prev ? pxb * 2 : 0}, {dy, xb},
                     {dfinal_state, dfinal_state ? sb : 0}, {block_states, bsb}};
    const R outs[] = {{dx, subs * nheads * headdim * 4}, {ddt, steps * nheads * 4},
                      {dlam, steps * nheads * 4}, {dA_head, (size_t)nheads * 4},
                      {dB, bcb * 2}, {dC, bcb * 2}, {dinitial_state, dinitial_state ? sb : 0},
                      {dprev_B, has_prev ? pbb * 4 : 0}, {dprev_x, has_prev ? pxb * 4 : 0}};
    constexpr int kOuts = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < kOuts; ++i) {
        for (const R& r : ins)
            if (overlaps(outs[i].p, outs[i].n, r.p, r.n)) return SSM_ERR_ALIAS;
        for (int j = i + 1; j < kOuts; ++j)
            if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_ALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!work) {
        if (nheads > 0 && cudaMemsetAsync(dA_head, 0, (size_t)nheads * 4, s) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (dinitial_state && sb) {
            const cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, sb,
                                                                 cudaMemcpyDeviceToDevice, s)
                                               : cudaMemsetAsync(dinitial_state, 0, sb, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        if (has_prev && items > 0) {
            if (cudaMemsetAsync(dprev_B, 0, pbb * 4, s) != cudaSuccess ||
                cudaMemsetAsync(dprev_x, 0, pxb * 4, s) != cudaSuccess)
                return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const M3mWs m = m3m_workspace(batch, seqlen, rank, nheads, ngroups);
    if (workspace_bytes < m.total) return SSM_ERR_WORKSPACE;
    for (const R& r : ins)
        if (overlaps(workspace, m.total, r.p, r.n)) return SSM_ERR_ALIAS;
    for (const R& r : outs)
        if (overlaps(workspace, m.total, r.p, r.n)) return SSM_ERR_ALIAS;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    size_t o = m.ssd;
    auto take = [&](size_t bytes) { float* p = reinterpret_cast<float*>(ws + o); o += bytes; return p; };
    float* dts = take(m.dts);
    float* wts = take(m.wts);
    float* dw = take(m.dw);
    float* ddec = take(m.ddec);
    float* XD = take(m.xd);
    float* Gd = take(m.g);
    float* dS = take(m.ds);
    float* dc0 = take(m.dc0);
    float* ppb = take(m.ppb);
    float* dS_out = dinitial_state ? dinitial_state : (has_prev ? dS : nullptr);

    // 1. per sub-token: the step's dt on its first row and its weight on every row
    m3m_expand_kernel<<<grid_for((long long)subs * nheads, 256), 256, 0, s>>>(
        dt, lam, dts, wts, batch, seqlen, rank, nheads);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    const MakeStates states = [&](float* bs) {
        return ssd_internal::ssd_mamba3_forward_block_states(x, dt, lam, A_head, B, C,
                                                             initial_state, prev_B, prev_x, bs,
                                                             batch, seqlen, nheads, ngroups, s,
                                                             rank);
    };
    // 2. the per-step rank dots (they feed the gradient kernel's dx correction)
    auto dots = rank == 1 ? m3m_dots<1> : rank == 2 ? m3m_dots<2> : m3m_dots<4>;
    ssm_status_t rc = dots(x, B, C, dy, XD, Gd, batch, seqlen, nheads, ngroups, s);
    if (rc != SSM_OK) return rc;
    // 3. the SSD gradient over the sub-tokens (block-lower-triangular mask)
    DxCorr corr;
    corr.g = Gd;
    corr.dt = dt;
    corr.lam = lam;
    corr.steps = seqlen;
    rc = run_bwd(x, dts, wts, A_head, B, C, initial_state, dy, dfinal_state, block_states,
                 states, dx, ddec, dw, dA_head, dB, dC, dS_out, batch, seqlen * rank, nheads,
                 ngroups, workspace, s, rank, corr);
    if (rc != SSM_OK) return rc;
    // 4.-5. the previous token and the per-step terms
    auto tail = rank == 1 ? m3m_tail<1> : rank == 2 ? m3m_tail<2> : m3m_tail<4>;
    rc = tail(dt, lam, B, C, has_prev, prev_B, prev_x, dS_out, dw, ddec, XD, Gd, dc0, ppb, ddt,
              dlam, dB, dC, dprev_B, dprev_x, batch, seqlen, nheads, ngroups, s);
    return rc;
}
