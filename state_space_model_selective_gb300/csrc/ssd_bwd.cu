// ssd_bwd.cu -- gradient of the chunked SSD (ssd_chunked_bwd) on tcgen05 tensor
// cores, GB300 / sm_103a.
//
// The forward operation is ssd_chunked_fwd's ("Mamba-3 NKI Kernels for AWS
// Neuron", section "Kernel details", mamba3_siso_ssd_kernel: the Mamba-2 SSD
// structure, equivalent to the step recurrence S = exp(dt A) S + dt B x^T,
// y = C S).  Its reverse-mode derivative, for the loss sum(dy y) +
// sum(dfinal final_state), is evaluated block by block in reverse, with the
// adjoint state dS = dL/dS carried between blocks.  For a block of Q = 128
// steps with cs_i = sum_{j<=i} dt_j A (inside the block), w = dt,
// L[i,j] = exp(cs_i - cs_j) for j <= i (else 0), S_in / S_out the states
// entering / leaving the block and dS_out the adjoint leaving it:
//   T       = dY X^T                      (Q x Q; (L o T) includes w_j)
//   dC      = diag(e^cs) dY S_in + (L o T w) B
//   dB      = diag(w e^(cs_last - cs)) X dS_out + (L o T w)^T C
//   bracket = diag(e^(cs_last - cs)) B dS_out^T + (L o C B^T)^T dY,  dX = diag(w) bracket
//   dS_in   = e^cs_last dS_out + (e^cs o dY)^T C
//   d cs_i  = C_i . dC_i - B_i . dB_i  (+ <dS_out, S_out> at the block's last row)
//   ddt_k   = x_k . bracket_k + A sum_{i >= k} d cs_i,   dA += sum_k dt_k sum_{i >= k} d cs_i
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

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace {

using namespace ssm;
using namespace ssd_detail;

constexpr int kThreads = 256;  // two warpgroups, each taking half of every row

// Shared memory (offsets from the 1024-aligned base)
constexpr uint32_t kSC = 0;         // C tile [128 i][128 n] (two 64-n boxes, 16 KB apart)
constexpr uint32_t kSB = 32768;     // B tile [128 j][128 n]
constexpr uint32_t kSX = 65536;     // x tile [128 j][64 p]
constexpr uint32_t kSDY = 81920;    // dy tile [128 i][64 p]
constexpr uint32_t kSS = 98304;     // S_in hi | lo [128 n][64 p]
constexpr uint32_t kSDS = 131072;   // dS_out hi | lo [128 n][64 p]
constexpr uint32_t kSE = 163840;    // (e^cs o dY) hi | lo [128 i][64 p]
constexpr uint32_t kMisc = 196608;  // cs2[128], q2[128], sums, mbarriers, TMEM address
constexpr uint32_t kMiscBytes = (2 * 128 + 32 + 3 * 128) * 4 + 9 * 8 + 16;
constexpr uint32_t kSmemAlloc = kMisc + kMiscBytes + 1024;  // + realignment slack

// TMEM columns (one CTA per SM: all 512)
constexpr uint32_t kTmGT = 0;    // G^T = B C^T -> (L o G)^T hi/lo
constexpr uint32_t kTmT = 128;   // T = dY X^T -> (L o T w) hi/lo; then dB
constexpr uint32_t kTmTT = 256;  // T^T -> (L o T w)^T hi/lo; then bracket (64) | dS_in^T (64)
constexpr uint32_t kTmR = 256;
constexpr uint32_t kTmDS = 320;
constexpr uint32_t kTmP = 384;   // dY S_in -> dC
constexpr uint32_t kTmemCols = 512;

struct BwdArgs {
    const float* dt;       // (batch, seqlen, nheads)
    const float* A;        // (nheads,)
    const float* bstates;  // [batch * nheads][nblocks + 1][64][128]
    const float* dfinal;   // (batch, nheads, 64, 128) or NULL
    float* dx;             // (batch, seqlen, nheads, 64)
    float* ddt;            // (batch, seqlen, nheads)
    float* dh0;            // (batch, nheads, 64, 128) or NULL
    float* pB;             // [nheads][batch][seqlen][128] per-head dB
    float* pC;             // [nheads][batch][seqlen][128] per-head dC
    float* pA;             // [batch * nheads]
    uint32_t* status;
    int batch, seqlen, nheads, ngroups;
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
// values are also stored to dst (global, 16-byte aligned).
__device__ __forceinline__ float dot_half_tmem(const uint8_t* tile, int row, int part,
                                               uint32_t taddr, float* dst) {
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
#pragma unroll
            for (int q = 0; q < 32; q += 4)
                *reinterpret_cast<float4*>(dst + 64 * part + 32 * hh + q) =
                    make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
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

__global__ void __launch_bounds__(kThreads, 1)
    ssd_bwd_kernel(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
                   const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                   const BwdArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    float* s_cs2 = reinterpret_cast<float*>(smem + kMisc);  // log2-scaled cs of each row
    float* s_q2 = s_cs2 + kQ;                               // log2(dt_j) - cs2_j
    float* s_wsum = s_q2 + kQ;                              // [2][4] warp totals (cs scan)
    float* s_rsum = s_wsum + 8;                             // [4] warp totals (d cs suffix scan)
    float* s_dot = s_rsum + 8;                              // [8] <dS_out, S_out> per warp
    float* s_da = s_dot + 8;                                // [4] dA per warp
    float* s_pd = s_da + 8;                                 // [3][128] the second half's dots
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(s_pd + 3 * kQ);  // C, B, S_in, S_out in
    uint64_t* bar_ld2 = bar_ld + 1;                                  // x, dy in
    uint64_t* bar_mma = bar_ld + 2;  // [6] one per MMA group
    uint64_t* bar_fin = bar_ld + 8;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_ld + 9);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int part = warp >> 2;            // which half of each row's columns it takes
    const int row = quarter * 32 + lane;   // TMEM lane and block row
    const int item = blockIdx.x;
    const int h = item % a.nheads, b = item / a.nheads;
    const int g = h / (a.nheads / a.ngroups);
    const int L = a.seqlen;
    const int nblocks = (L + kQ - 1) / kQ;
    const float Ah = a.A[h];
    const float* bs_item = a.bstates + (long long)item * (nblocks + 1) * kP * kNs;

    // Loads of block blk (thread 0): C, B and the states entering and leaving it
    // (fp32 [p][n], into the regions their split forms replace), then x and dy.
    auto load_cbs = [&](int blk) {
        mbar_arrive_expect_tx(bar_ld, 4 * 32768);
        tma_load_4d(smem + kSC, &tm_C, bar_ld, 0, g, blk * kQ, b);
        tma_load_4d(smem + kSC + 16384, &tm_C, bar_ld, 64, g, blk * kQ, b);
        tma_load_4d(smem + kSB, &tm_B, bar_ld, 0, g, blk * kQ, b);
        tma_load_4d(smem + kSB + 16384, &tm_B, bar_ld, 64, g, blk * kQ, b);
        bulk_load(smem + kSE, bs_item + (long long)blk * kP * kNs, 32768, bar_ld);
        bulk_load(smem + kSDS, bs_item + (long long)(blk + 1) * kP * kNs, 32768, bar_ld);
    };
    auto load_xdy = [&](int blk) {
        mbar_arrive_expect_tx(bar_ld2, 2 * 16384);
        tma_load_3d(smem + kSX, &tm_x, bar_ld2, h * kP, blk * kQ, b);
        tma_load_3d(smem + kSDY, &tm_dy, bar_ld2, h * kP, blk * kQ, b);
    };

    if (warp == 0) tmem_alloc(s_tmem, kTmemCols);
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_ld2, 1);
        for (int k = 0; k < 6; ++k) mbar_init(bar_mma + k, 1);
        mbar_init(bar_fin, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_dy);
        if (nblocks > 0) {
            load_cbs(nblocks - 1);
            load_xdy(nblocks - 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ld_pending = nblocks > 0, ld2_pending = nblocks > 0;
    uint32_t ld_par = 0, ld2_par = 0;  // phase parity of the pending loads

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
    float dt_next = nblocks > 0 ? dt_of(nblocks - 1) : 0.0f;

    for (int blk = nblocks - 1; blk >= 0; --blk, ph ^= 1u) {
        const int t0 = blk * kQ;
        const int t = t0 + row;
        const float dtr = dt_next;
        if (blk > 0) dt_next = dt_of(blk - 1);

        // ---- cumulative log-decay within the block (warp part)
        float v = dtr * Ah;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) s_wsum[part * 4 + quarter] = v;
        // ---- S_in as the split operand [n = row][p]; <dS_out, S_out> for the
        // log-decay gradient of the block's last row
        {
            const bool got = mbar_wait(bar_ld, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
            ld_pending = false;
        }
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
        __syncthreads();  // S_out read out of its region; warp sums visible
        store_split_half(smem + kSDS, row, part, dS);  // dS_out over S_out
        float cs_last = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float ws = s_wsum[part * 4 + w];
            if (w < quarter) v += ws;
            cs_last += ws;
        }
        const float cs2 = v * kLog2e, cs2_last = cs_last * kLog2e;
        float lg;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(dtr));
        const float q2 = lg - cs2;
        if (part == 0) {
            s_cs2[row] = cs2;
            s_q2[row] = q2;
        }
        const float e_r = ex2_approx(cs2);
        const float eL_r = ex2_approx(cs2_last - cs2);
        const float u_r = dtr * eL_r;
        const float e_last = ex2_approx(cs2_last);
        float sdot = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sdot += s_dot[w];
        fence_proxy_async_smem();
        tc_fence_before();

        // ---- group 1: G^T = B C^T, T = dY X^T, T^T = X dY^T, P = dY S_in
        {
            const bool got = mbar_wait(bar_ld2, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
            ld2_pending = false;
        }
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id128 = idesc_bf16_f32(128, 128);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + kTmGT, kdesc<kQ>(sbase + kSB, kk), kdesc<kQ>(sbase + kSC, kk), id128,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(tmem + kTmT, kdesc<kQ>(sbase + kSDY, kk), kdesc<kQ>(sbase + kSX, kk), id128,
                         kk > 0);
                mma_bf16(tmem + kTmTT, kdesc<kQ>(sbase + kSX, kk), kdesc<kQ>(sbase + kSDY, kk), id128,
                         kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + kTmP, kdesc<kQ>(sbase + kSDY, kk), kdesc<kQ>(sbase + kSS, kk), id128,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + kTmP, kdesc<kQ>(sbase + kSDY, kk),
                         kdesc<kQ>(sbase + kSS + 16384, kk), id128, 1);
            mma_commit(bar_mma + 0);
        }
        // e^cs o dY as the split MN-major operand of dS_in^T (rows i, p
        // contiguous), over the S_in region (read above)
        {
            float dyv[32];
            load_tile_half(smem + kSDY, row, part, dyv);
#pragma unroll
            for (int q = 0; q < 32; ++q) dyv[q] *= e_r;
            store_split_half(smem + kSE, row, part, dyv);
        }
        {
            const bool got = mbar_wait(bar_mma + 0, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // (L o G)^T row j = row: columns i >= j, factor e^(cs_i - cs_j)
        mask_row_half(t_lane + kTmGT, s_cs2, -cs2, row, kQ - 1, part);
        // (L o T w) row i = row: columns j <= i, factor e^(cs_i - cs_j) dt_j
        mask_row_half(t_lane + kTmT, s_q2, cs2, 0, row, part);
        // (L o T w)^T row j = row: columns i >= j, factor e^(cs_i - cs_j) dt_j
        mask_row_half(t_lane + kTmTT, s_cs2, q2, row, kQ - 1, part);
        // dY S_in scaled by e^cs_i
        scale_half(t_lane + kTmP, part, e_r);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- group 2: dC = e^cs o (dY S_in) + (L o T w) B
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t idC = idesc_bf16_f32(128, 128) | kIdescBMN;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16_ta(tmem + kTmP, tmem + kTmT + mcol_hi(kk), mdesc(sbase + kSB, kk, 16384),
                            idC, 1);
                mma_bf16_ta(tmem + kTmP, tmem + kTmT + mcol_hi(kk) + 16,
                            mdesc(sbase + kSB, kk, 16384), idC, 1);
            }
            mma_commit(bar_mma + 1);
        }
        {
            const bool got = mbar_wait(bar_mma + 1, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // ---- group 3 (the (L o T w) operand is consumed): Q = X dS_out into its place
        if (tid == 0) {
            constexpr uint32_t id128 = idesc_bf16_f32(128, 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + kTmT, kdesc<kQ>(sbase + kSX, kk), kdesc<kQ>(sbase + kSDS, kk), id128,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + kTmT, kdesc<kQ>(sbase + kSX, kk),
                         kdesc<kQ>(sbase + kSDS + 16384, kk), id128, 1);
            mma_commit(bar_mma + 2);
        }
        // dC row i: its log-decay term C_i . dC_i (this half) and its per-head partial
        const float dcs_c = dot_half_tmem(
            smem + kSC, row, part, t_lane + kTmP,
            t < L ? a.pC + (((long long)h * a.batch + b) * L + t) * kNs : nullptr);
        {
            const bool got = mbar_wait(bar_mma + 2, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // X dS_out row j scaled by dt_j e^(cs_last - cs_j)
        scale_half(t_lane + kTmT, part, u_r);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();

        // ---- group 4: dB = dt e^(cs_last - cs) o (X dS_out) + (L o T w)^T C
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t idB = idesc_bf16_f32(128, 128) | kIdescBMN;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16_ta(tmem + kTmT, tmem + kTmTT + mcol_hi(kk), mdesc(sbase + kSC, kk, 16384),
                            idB, 1);
                mma_bf16_ta(tmem + kTmT, tmem + kTmTT + mcol_hi(kk) + 16,
                            mdesc(sbase + kSC, kk, 16384), idB, 1);
            }
            mma_commit(bar_mma + 3);
        }
        {
            const bool got = mbar_wait(bar_mma + 3, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // ---- group 5 (the (L o T w)^T operand is consumed): R = B dS_out^T and
        // dS_in^T = C^T (e^cs o dY) into its place, N = 64 each
        if (tid == 0) {
            constexpr uint32_t idR = idesc_bf16_f32(128, 64) | kIdescBMN;
            constexpr uint32_t idS = idesc_bf16_f32(128, 64) | kIdescAMN | kIdescBMN;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16(tmem + kTmR, kdesc<kQ>(sbase + kSB, kk), mdesc(sbase + kSDS, kk, 16384),
                         idR, kk > 0);
                mma_bf16(tmem + kTmR, kdesc<kQ>(sbase + kSB, kk),
                         mdesc(sbase + kSDS + 16384, kk, 16384), idR, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16(tmem + kTmDS, mdesc(sbase + kSC, kk, 16384), mdesc(sbase + kSE, kk, 16384),
                         idS, kk > 0);
                mma_bf16(tmem + kTmDS, mdesc(sbase + kSC, kk, 16384),
                         mdesc(sbase + kSE + 16384, kk, 16384), idS, 1);
            }
            mma_commit(bar_mma + 4);
        }
        // dB row j: its log-decay term B_j . dB_j (this half) and its per-head partial
        const float dcs_b = dot_half_tmem(
            smem + kSB, row, part, t_lane + kTmT,
            t < L ? a.pB + (((long long)h * a.batch + b) * L + t) * kNs : nullptr);
        {
            const bool got = mbar_wait(bar_mma + 4, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // C, B, S_in's and S_out's regions are free (group 5 was their last
        // reader): the previous block's loads start now
        if (tid == 0 && blk > 0) load_cbs(blk - 1);
        if (blk > 0) {
            ld_pending = true;
            ld_par = ph ^ 1u;
        }
        // B dS_out^T row j scaled by e^(cs_last - cs_j); the adjoint entering
        // the block: dS_in[p][n = row] = e^cs_last dS_out + (C^T (e^cs o dY))[n][p]
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
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();

        // ---- group 6: bracket = e^(cs_last - cs) o (B dS_out^T) + (L o G)^T dY
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t idX = idesc_bf16_f32(128, 64) | kIdescBMN;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16_ta(tmem + kTmR, tmem + kTmGT + mcol_hi(kk), mdesc(sbase + kSDY, kk, 16384),
                            idX, 1);
                mma_bf16_ta(tmem + kTmR, tmem + kTmGT + mcol_hi(kk) + 16,
                            mdesc(sbase + kSDY, kk, 16384), idX, 1);
            }
            mma_commit(bar_mma + 5);
        }
        {
            const bool got = mbar_wait(bar_mma + 5, ph, a.status);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
        // dX_j = dt_j bracket_j; the input-weight part of ddt_j is x_j . bracket_j
        float dw = 0.0f;
        {
            float xv[32], br[32];
            load_tile_half(smem + kSX, row, part, xv);
            tmem_ld32(t_lane + kTmR + 32 * part, br);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) dw = fmaf(xv[q], br[q], dw);
            if (t < L) {
                float* dxr = a.dx + (((long long)b * L + t) * a.nheads + h) * kP + 32 * part;
#pragma unroll
                for (int q = 0; q < 32; q += 4)
                    *reinterpret_cast<float4*>(dxr + q) =
                        make_float4(dtr * br[q], dtr * br[q + 1], dtr * br[q + 2], dtr * br[q + 3]);
            }
        }
        // ---- log-decay gradient of each row (both halves' dots), its suffix
        // sums over the block, ddt and dA (first warpgroup)
        if (part == 1) {
            s_pd[row] = dcs_c;
            s_pd[kQ + row] = dcs_b;
            s_pd[2 * kQ + row] = dw;
        }
        tc_fence_before();
        __syncthreads();  // also: every read of this block's tiles and TMEM is done
        float dcs = 0.0f, dw_all = 0.0f;
        if (part == 0) {
            dcs = (dcs_c + s_pd[row]) - (dcs_b + s_pd[kQ + row]) + (row == kQ - 1 ? sdot : 0.0f);
            dw_all = dw + s_pd[2 * kQ + row];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_down_sync(0xffffffffu, dcs, o);
                if (lane + o < 32) dcs += u;
            }
            if (lane == 0) s_rsum[quarter] = dcs;
        }
        __syncthreads();
        if (part == 0) {
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (w > quarter) dcs += s_rsum[w];
            if (t < L) a.ddt[((long long)b * L + t) * a.nheads + h] = fmaf(Ah, dcs, dw_all);
            dA_acc = fmaf(dtr, dcs, dA_acc);
        }
        __syncthreads();  // s_rsum, s_wsum, s_dot, s_pd are rewritten by the next block
        if (tid == 0 && blk > 0) load_xdy(blk - 1);  // x was read above, dy by group 6
        if (blk > 0) {
            ld2_pending = true;
            ld2_par = ph ^ 1u;
        }
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
        __syncthreads();
        if (tid == 0) a.pA[item] = s_da[0] + s_da[1] + s_da[2] + s_da[3];
    } else if (tid == 0) {
        // a wait ran out: let every issued MMA and load finish before leaving
        mma_commit(bar_fin);
        (void)mbar_wait(bar_fin, 0, nullptr);
        if (ld_pending) (void)mbar_wait(bar_ld, ld_par, nullptr);
        if (ld2_pending) (void)mbar_wait(bar_ld2, ld2_par, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// dB, dC = the per-head partials summed over each group's heads; dA = the
// per-(batch, head) sums added over the batch.  Fixed order: deterministic.
__global__ void ssd_bwd_reduce_kernel(const float* __restrict__ pB, const float* __restrict__ pC,
                                      const float* __restrict__ pA, float* __restrict__ dB,
                                      float* __restrict__ dC, float* __restrict__ dA, int batch,
                                      int seqlen, int nheads, int ngroups) {
    const int hpg = nheads / ngroups;
    const long long rows = (long long)batch * seqlen;          // (b, t)
    const long long nbc = rows * ngroups * kNs;                // one of dB, dC
    const long long head_stride = rows * kNs;                  // pB[h] block
    const long long total = 2 * nbc + nheads;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        if (i < 2 * nbc) {
            const bool isC = i >= nbc;
            const long long e = isC ? i - nbc : i;  // ((b t) g) n
            const long long n = e % kNs, gi = (e / kNs) % ngroups, bt = e / (kNs * ngroups);
            const float* src = (isC ? pC : pB) + bt * kNs + n;
            float s = 0.0f;
            for (int hh = (int)gi * hpg; hh < ((int)gi + 1) * hpg; ++hh) s += src[hh * head_stride];
            (isC ? dC : dB)[e] = s;
        } else {
            const int hh = (int)(i - 2 * nbc);
            float s = 0.0f;
            for (int bb = 0; bb < batch; ++bb) s += pA[(long long)bb * nheads + hh];
            dA[hh] = s;
        }
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
                                        const float* dfinal_state, float* dx, float* ddt,
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
    const void* ptrs[] = {x, dt, A_head, B, C, initial_state, dy, dfinal_state, dx, ddt,
                          dA_head, dB, dC, dinitial_state, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = steps * nheads * headdim * 2, bcb = steps * ngroups * dstate * 2;
    struct R { const void* p; size_t n; };
    const R ins[] = {{x, xb}, {dt, steps * nheads * 4}, {A_head, (size_t)nheads * 4}, {B, bcb},
                     {C, bcb}, {initial_state, initial_state ? sb : 0}, {dy, xb},
                     {dfinal_state, dfinal_state ? sb : 0}};
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

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (cudaMemsetAsync(ws, 0, w.header, s) != cudaSuccess) return SSM_ERR_CUDA;
    float* bstates = reinterpret_cast<float*>(ws + w.header);
    BwdArgs a{};
    a.dt = dt;
    a.A = A_head;
    a.bstates = bstates;
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

    // 1. the state entering every block (and the final state)
    ssm_status_t rc = ssd_internal::ssd_forward_block_states(
        x, dt, A_head, B, C, initial_state, bstates, batch, seqlen, nheads, ngroups, s);
    if (rc != SSM_OK) return rc;
    // 2. the blocks in reverse, one CTA per (batch, head)
    CUtensorMap mc, mb, mx, mdy;
    if (!ssd_host::make_bc_map(&mc, C, batch, seqlen, ngroups) ||
        !ssd_host::make_bc_map(&mb, B, batch, seqlen, ngroups) ||
        !ssd_host::make_x_map(&mx, x, batch, seqlen, nheads) ||
        !ssd_host::make_x_map(&mdy, dy, batch, seqlen, nheads))
        return SSM_ERR_CUDA;
    if (cudaFuncSetAttribute(ssd_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess)
        return SSM_ERR_CUDA;
    ssd_bwd_kernel<<<(unsigned)items, kThreads, kSmemAlloc, s>>>(mc, mb, mx, mdy, a);
    if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
    // 3. sums over a group's heads and over the batch
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = 2LL * (long long)steps * ngroups * kNs + nheads;
    const unsigned rgrid =
        (unsigned)std::max<long long>(1, std::min<long long>((total + 255) / 256, 8LL * sms));
    ssd_bwd_reduce_kernel<<<rgrid, 256, 0, s>>>(a.pB, a.pC, a.pA, dB, dC, dA_head, batch, seqlen,
                                                nheads, ngroups);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
