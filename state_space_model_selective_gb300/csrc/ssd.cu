// ssd.cu -- chunked SSD forward (ssd_chunked_fwd) on tcgen05 tensor cores,
// GB300 / sm_103a.
//
// "Mamba-3 NKI Kernels for AWS Neuron", section "Kernel details"
// (mamba3_siso_ssd_kernel: the Mamba-2 SSD structure, chunk 64, equivalent to
// the step-by-step recurrence) and section "Configuration constraints"
// (seqlen divisible by the chunk size).  Scalar A per head; dt is taken as
// given.  For every block of Q steps (cs_i = sum_{j<=i} dt_j A_h inside the
// block):
//   G        = C B^T                                      (Q x Q, K = N)
//   M'[i,j]  = G[i,j] exp(cs_i - cs_j) dt_j  (j <= i)      causal, decayed
//   Y        = M' X + diag(exp(cs)) (C S_prev^T)           (Q x P)
//   S_chunk  = B^T (w o X),  w_j = exp(cs_last - cs_j) dt_j (N x P)
//   S_prev   = exp(cs_last) S_prev + S_chunk
//
// GB300 mapping.  One CTA per (batch, head), 128 threads; the chunked form is
// exact for any block length, and the kernel evaluates it in Q = 128-step
// blocks so that every product is a 128-row tcgen05 MMA (M = 128, K = 16 per
// instruction, fp32 accumulators in tensor memory):
//   G (N=128), C S^T (N=64), B^T X' (N=64), M' X (N=64).
// C and B tiles arrive by 4-D TMA in the 128-byte-swizzled K-major layout
// the MMA reads directly; the remaining operands are written to shared memory
// by the threads in the same layout (X^T, the weighted X'^T, B^T, M', S).
// Operands that are fp32 intermediates (M', X', S) are split into a bf16
// high part and a bf16 remainder (v = hi + lo, about 16 significant bits) and
// enter the MMA twice; C, B and X are exact in bf16.  Each thread owns one
// TMEM lane: row i of G / Y, and row n of S_chunk^T with the running state
// S_prev[n, :] kept in its registers.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace {

using namespace ssm;
using namespace ssd_detail;
using ssd_host::make_bc_map;
using ssd_host::make_x_map;
using ssd_host::make_y_map;
constexpr int kThreads = 256;  // two warpgroups; each per-row phase splits a row's columns
constexpr int kHalf = 32;      // columns of a 64-wide row per warpgroup

// Shared memory (offsets from the 1024-aligned dynamic base).  The total stays
// under half of an SM's shared memory so that two CTAs share an SM.
constexpr uint32_t kRC = 0;        // C tile [128 i][128 n], K-major -> X' hi | X' lo [128 j][64 p]
constexpr uint32_t kRB = 32768;    // B tile [128 j][128 n]: G's B (K-major), S_chunk's A (MN-major)
constexpr uint32_t kRX = 65536;    // x tile [128 j][64 p]: Y_diag's B (MN-major)
constexpr uint32_t kRS = 81920;    // S_prev hi | lo [128 n][64 p]: Y_off's B (MN-major)
constexpr uint32_t kMisc = 114688; // q2[128], warp sums [2][4], 6 mbarriers, TMEM address
constexpr uint32_t kSmemBytes = kMisc + kQ * 4 + 32 + 48 + 8;
// TMEM columns
constexpr uint32_t kTmG = 0;    // G = C B^T (fp32), overwritten in place by M' hi/lo (bf16 pairs)
constexpr uint32_t kTmY = 128;  // C S_hi^T | C S_lo^T (128 columns), then exp(cs_i) Y_off + Y_diag (64)
constexpr uint32_t kTmS = 192;  // S_chunk^T [n][p], once the C S_lo^T half has been read
constexpr uint32_t kTmemCols = 256;

struct SsdArgs {
    const __nv_bfloat16* x;
    const float* dt;
    const float* A;
    const float* h0;  // initial state (batch, nheads, headdim, dstate) or NULL
    // Mamba-3 only: lambda (batch, seqlen, nheads); the token before the first,
    // prev_B (batch, ngroups, dstate) and prev_x (batch, nheads, headdim), or NULL
    const float* lam;
    const __nv_bfloat16* prev_B;
    const __nv_bfloat16* prev_x;
    void* y;
    float* final_state;
    // optional: the state entering every block and the final state,
    // [batch * nheads][nblocks + 1][headdim][dstate] (the backward pass reads it)
    float* bstates;
    int batch, seqlen, nheads, ngroups;
};

// One 32-column chunk of M' for row i: m_j = G[i][j] 2^(cs2_i + q2_j), with
// columns past jmax zeroed when MASK (the chunk holding row i's own step; jmax
// = its last column relative to the chunk).  With DIAG (Mamba-3) the entries
// of row i's own step, columns jd0 .. jmax, are G[i][j] diag_w instead (one
// entry for SISO, the step's R sub-tokens for MIMO).
template <bool MASK, bool DIAG>
__device__ __forceinline__ void mprime_chunk(const float* gv, const float* q2c, float cs2_i, int jmax,
                                             int jd0, float diag_w, uint32_t* hp, uint32_t* lp) {
#pragma unroll
    for (int q = 0; q < 32; q += 4) {
        const float4 qq = *reinterpret_cast<const float4*>(q2c + q);
        const float qv[4] = {qq.x, qq.y, qq.z, qq.w};
        float m[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m[k] = gv[q + k] * ex2_approx(cs2_i + qv[k]);
            if (MASK && DIAG && q + k >= jd0) m[k] = gv[q + k] * diag_w;
            if (MASK && q + k > jmax) m[k] = 0.0f;
        }
        split2_bf16(m[0], m[1], hp[q >> 1], lp[q >> 1]);
        split2_bf16(m[2], m[3], hp[(q >> 1) + 1], lp[(q >> 1) + 1]);
    }
}

// M3 = false: Mamba-2 (the input weight of step j is dt_j).  M3 = true:
// Mamba-3 SISO single-SSD form, "Mamba-3 NKI Kernels for AWS Neuron",
// "Kernel details", mamba3_siso_ssd_kernel: the weight is
// scale_j = gamma_j + dt_{j+1} (1 - lambda_{j+1}) (gamma = lambda dt; 0 past
// the last step), the diagonal of M' takes gamma_i, and the previous token's
// B (x) x enters the state as dt_0 (1 - lambda_0) prev_B (x) prev_x.
// RK > 1 (Mamba-3 MIMO, "Kernel details", mamba3_mimo_ssd_kernel): the rank
// is flattened into the sequence -- x, y, B, C hold RK sub-tokens per step,
// row u of a block is sub-token u % RK of step u / RK -- and sub-tokens share
// their step's decay and weights; a sub-token sees every sub-token of its own
// step (the block-diagonal part, weight gamma) and of earlier steps.
// BS: also write the state entering every block and the final state to
// a.bstates (the backward pass's checkpoints): 1 with y as well (y optional),
// 2 states only -- no C tile, no G, M', Y_off or Y_diag products and no y; a
// block is then cs, X' and S_chunk^T = B^T X' only.
template <typename Tout, bool M3, int RK, int BS = 0>
__global__ void __launch_bounds__(kThreads, 2)
    ssd_fwd_kernel(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
                   const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_y, const SsdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr bool SO = BS == 2;  // states only
    const uint32_t sbase = smem_u32(smem);
    float* s_q2 = reinterpret_cast<float*>(smem + kMisc);
    float* s_wsum = s_q2 + kQ;  // [2][4] per-warpgroup warp totals
    uint64_t* bar_cb = reinterpret_cast<uint64_t*>(smem + kMisc + kQ * 4 + 32);  // C, B tiles in
    uint64_t* bar_x = bar_cb + 1;      // x tile in
    uint64_t* bar_g = bar_cb + 2;      // G = C B^T done
    uint64_t* bar_yoff = bar_cb + 3;   // Y_off done (committed every step, empty on block 0)
    uint64_t* bar_s = bar_cb + 4;      // S_chunk done: the B and X' (C) regions are free
    uint64_t* bar_mma2 = bar_cb + 5;   // Y_diag done: the x region is free
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_cb + 6);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int part = warp >> 2;    // which half of a row's columns this warpgroup takes
    const int row = quarter * 32 + lane;  // TMEM lane: row i of G / Y, state n of S
    // Work items are (batch, head) pairs blockIdx.x, blockIdx.x + gridDim.x, ...;
    // each is nblocks steps of kQ time steps, run in order.
    const int nsub = a.seqlen * RK;  // sub-tokens (rows) per sequence
    const int nblocks = (nsub + kQ - 1) / kQ;
    const int nitems = a.batch * a.nheads;
    const int my_items = ((int)blockIdx.x < nitems) ? (nitems - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nsteps = my_items * nblocks;
    const int hpg = a.nheads / a.ngroups;

    if (sbase & 1023u) {
        // The swizzled tiles need a 1024-byte-aligned base and there is no
        // room to realign: make the failure visible instead of computing.
        const float nanv = __int_as_float(0x7fc00000);
        for (int it = 0; it < my_items; ++it) {
            const int item = (int)blockIdx.x + it * (int)gridDim.x;
            const int hh = item % a.nheads, bb = item / a.nheads;
            if constexpr (BS != 0) {
                float* bs = a.bstates + (long long)item * (nblocks + 1) * kP * kNs;
                for (int e = tid; e < (nblocks + 1) * kP * kNs; e += kThreads) bs[e] = nanv;
                if (!a.y) continue;
            }
            for (int t = tid; t < nsub; t += kThreads) {
                Tout* yr = reinterpret_cast<Tout*>(a.y) +
                           (((long long)bb * nsub + t) * a.nheads + hh) * kP;
                for (int p = 0; p < kP; ++p) yr[p] = from_f32<Tout>(nanv);
            }
        }
        return;
    }

    if (warp == 0) tmem_alloc(s_tmem, kTmemCols);
    if (tid == 0) {
        mbar_init(bar_cb, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_yoff, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_mma2, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_x);
        if (a.y) prefetch_tensormap(&tm_y);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane base

    float S[kHalf];  // S_prev[n = row][32 part + q] of the current item
#pragma unroll
    for (int q = 0; q < kHalf; ++q) S[q] = 0.0f;
    const bool has_h0 = a.h0 != nullptr;

    // Loads are issued by thread kLoader: C and B of step st as soon as the
    // previous step's S_chunk MMAs are done, x once its Y_diag MMAs are.  At
    // most one load per barrier is ever outstanding.
    constexpr int kLoader = 32;
    int cb_issued = 0, x_issued = 0;  // (loader) loads issued so far
    auto step_coords = [&](int st, int& hn, int& bn, int& gn, int& tn) {
        const int item = (int)blockIdx.x + (st / nblocks) * (int)gridDim.x;
        hn = item % a.nheads;
        bn = item / a.nheads;
        gn = hn / hpg;
        tn = (st % nblocks) * kQ;
    };
    auto load_cb = [&](int st) {
        int hn, bn, gn, tn;
        step_coords(st, hn, bn, gn, tn);
        mbar_arrive_expect_tx(bar_cb, SO ? 32768 : 2 * 32768);
        if constexpr (!SO) {  // states only: no C (the region holds X')
            tma_load_4d(smem + kRC, &tm_C, bar_cb, 0, gn, tn, bn);
            tma_load_4d(smem + kRC + 16384, &tm_C, bar_cb, 64, gn, tn, bn);
        }
        tma_load_4d(smem + kRB, &tm_B, bar_cb, 0, gn, tn, bn);
        tma_load_4d(smem + kRB + 16384, &tm_B, bar_cb, 64, gn, tn, bn);
        ++cb_issued;
    };
    auto load_x = [&](int st) {
        int hn, bn, gn, tn;
        step_coords(st, hn, bn, gn, tn);
        mbar_arrive_expect_tx(bar_x, 16384);
        tma_load_3d(smem + kRX, &tm_x, bar_x, hn * kP, tn, bn);
        ++x_issued;
    };
    // per-step inputs of this thread's row for step st, 0 past the sequence
    // end: dt, A_h, and (Mamba-3) lambda, dt and lambda of the next step
    struct StepIn { float dt, A, lam, dt1, lam1; };
    auto load_step = [&](int st, StepIn& v) {
        const int item = (int)blockIdx.x + (st / nblocks) * (int)gridDim.x;
        const int hn = item % a.nheads, bn = item / a.nheads;
        const int t = ((st % nblocks) * kQ + row) / RK;  // the row's step
        const long long i0 = ((long long)bn * a.seqlen + t) * a.nheads + hn;
        v.dt = t < a.seqlen ? a.dt[i0] : 0.0f;
        v.A = a.A[hn];
        if constexpr (M3) {
            v.lam = t < a.seqlen ? a.lam[i0] : 0.0f;
            v.dt1 = t + 1 < a.seqlen ? a.dt[i0 + a.nheads] : 0.0f;
            v.lam1 = t + 1 < a.seqlen ? a.lam[i0 + a.nheads] : 0.0f;
        }
    };
    bool ok = true;
    if (tid == kLoader && nsteps > 0) {
        load_cb(0);
        load_x(0);
    }
    StepIn in_next{0.f, 0.f, 0.f, 0.f, 0.f};  // loaded one step ahead
    if (nsteps > 0) load_step(0, in_next);
    const bool has_prev = M3 && a.prev_B != nullptr && a.prev_x != nullptr;

    for (int st = 0; st < nsteps; ++st) {
        const int item = (int)blockIdx.x + (st / nblocks) * (int)gridDim.x;
        const int blk = st % nblocks;
        const int h = item % a.nheads, b = item / a.nheads;
        const int t0 = blk * kQ;
        const uint32_t ph = (uint32_t)(st & 1);
        // a state enters this block: carried from the previous block, or given
        const bool carry = blk > 0 || has_h0 || has_prev;
        if (blk == 0 && has_h0) {
            const float* ip = a.h0 + ((long long)(b * a.nheads + h) * kP + kHalf * part) * kNs + row;
#pragma unroll
            for (int q = 0; q < kHalf; ++q) S[q] = ip[q * kNs];
        }
        if (blk == 0 && has_prev) {
            // the previous token's beta term, pending: dt_0 (1 - lambda_0) prev_B (x) prev_x
            const long long i0 = (long long)b * a.seqlen * a.nheads + h;
            const float pw = a.seqlen > 0 ? a.dt[i0] * (1.0f - a.lam[i0]) : 0.0f;
            const int g = h / hpg;
#pragma unroll 1
            for (int r = 0; r < RK; ++r) {  // sum over the previous token's ranks
                const float pb =
                    pw * __bfloat162float(a.prev_B[(((long long)b * RK + r) * a.ngroups + g) * kNs + row]);
                const uint4* px = reinterpret_cast<const uint4*>(
                    a.prev_x + (((long long)b * RK + r) * a.nheads + h) * kP + kHalf * part);
#pragma unroll
                for (int c = 0; c < kHalf / 8; ++c) {
                    const uint4 w = px[c];
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        S[8 * c + 2 * e] = fmaf(pb, bf16lo(ww[e]), S[8 * c + 2 * e]);
                        S[8 * c + 2 * e + 1] = fmaf(pb, bf16hi(ww[e]), S[8 * c + 2 * e + 1]);
                    }
                }
            }
        }

        if constexpr (BS != 0) {
            float* bs = a.bstates +
                        (((long long)item * (nblocks + 1) + blk) * kP + kHalf * part) * kNs + row;
#pragma unroll
            for (int q = 0; q < kHalf; ++q) bs[q * kNs] = S[q];
        }

        // ---- G = C B^T as soon as the C and B tiles are in (thread 0)
        if (!SO && tid == 0) {
            const bool got = mbar_wait(bar_cb, ph, nullptr);
            tc_fence_after();
            if (got) {
                constexpr uint32_t id128 = idesc_bf16_f32(128, 128);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + kTmG, kdesc<kQ>(sbase + kRC, kk), kdesc<kQ>(sbase + kRB, kk),
                             id128, kk > 0);
                mma_commit(bar_g);
            }
        }

        // ---- cumulative log-decay cs_i = sum_{j<=i} dt_j A (padding: dt = 0),
        // computed by both warpgroups for their own rows
        const StepIn in = in_next;
        if (st + 1 < nsteps) load_step(st + 1, in_next);
        const float dti = in.dt;
        // input weight of this row's step (Mamba-2: dt; Mamba-3: scale) and, for
        // Mamba-3, the diagonal weight gamma
        // (every product below is rounded on its own, __fmul_rn, so that no
        // instance of this kernel -- with y, or states only -- contracts it
        // into a neighbouring add: all of them carry the same states, bit for bit)
        float w_i = dti, gamma_i = 0.0f;
        if constexpr (M3) {
            gamma_i = __fmul_rn(in.lam, dti);
            w_i = __fadd_rn(gamma_i, __fmul_rn(in.dt1, 1.0f - in.lam1));
        }
        // the step's log-decay enters the running sum once, at its first sub-token
        float v = (RK == 1 || row % RK == 0) ? __fmul_rn(dti, in.A) : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) s_wsum[part * 4 + quarter] = v;
        // the previous step's y tile (in the S region) has been read by its
        // TMA store before anyone rewrites the region
        if (tid == kLoader) bulk_wait_read_all();
        __syncthreads();
        float cs_last = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float ws = s_wsum[part * 4 + w];
            if (w < quarter) v += ws;
            cs_last += ws;
        }
        const float cs2_i = __fmul_rn(v, kLog2e);  // log2-scaled cs_i
        const float cs2_last = __fmul_rn(cs_last, kLog2e);
        // q2_j = log2(w_j) - cs_j log2(e): exp(cs_i - cs_j) w_j = 2^(cs2_i + q2_j)
        if (part == 0) {
            float lg;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(w_i));
            s_q2[row] = lg - cs2_i;
        }
        const float e_i = ex2_approx(cs2_i);
        const float a_blk = ex2_approx(cs2_last);

        // ---- S_prev as the hi/lo operand of Y_off (row n, p contiguous)
        if (!SO && carry) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t hp[4], lp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split2_bf16(S[8 * c4 + 2 * e], S[8 * c4 + 2 * e + 1], hp[e], lp[e]);
                const uint32_t off = (uint32_t)(row * 128 + (((part * 4 + c4) ^ (row & 7)) << 4));
                *reinterpret_cast<uint4*>(smem + kRS + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
                *reinterpret_cast<uint4*>(smem + kRS + 16384 + off) =
                    make_uint4(lp[0], lp[1], lp[2], lp[3]);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();  // S operand and q2 visible

        // ---- Y_off = C S_prev^T: N = 128, S_hi in columns 0..63, S_lo in 64..127
        // (none when no state enters the block)
        if (!SO && tid == 0) {
            tc_fence_after();
            if (carry) {
                constexpr uint32_t id128n = idesc_bf16_f32(128, 128) | kIdescBMN;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + kTmY, kdesc<kQ>(sbase + kRC, kk), mdesc(sbase + kRS, kk, 16384),
                             id128n, kk > 0);
            }
            mma_commit(bar_yoff);
        }

        // ---- M'[i][j] = G[i][j] exp(cs_i - cs_j) dt_j for j <= i, else 0,
        // split hi/lo and written back over G in TMEM (row i = this lane).
        // 32-column chunk k of this warpgroup is wholly above the diagonal for
        // k > quarter, on it for k == quarter, below it otherwise.
        if constexpr (!SO) {
            {
                const bool got = mbar_wait(bar_g, ph, nullptr);
                if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int ck = 2 * part + half;
                const int c0 = 32 * ck;
                uint32_t hp[16], lp[16];
                if (ck > quarter) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) hp[q] = lp[q] = 0u;
                } else {
                    float gv[32];
                    tmem_ld32(t_lane + kTmG + c0, gv);
                    tmem_wait_ld();
                    if (ck == quarter)
                        mprime_chunk<true, M3>(gv, s_q2 + c0, cs2_i, RK * (lane / RK) + RK - 1,
                                               RK * (lane / RK), gamma_i, hp, lp);
                    else
                        mprime_chunk<false, M3>(gv, s_q2 + c0, cs2_i, 31, 0, gamma_i, hp, lp);
                }
                tmem_st16(t_lane + kTmG + c0, hp);
                tmem_st16(t_lane + kTmG + c0 + 16, lp);
            }
        }

        // ---- Y_off done (the C region is free):  X' = w o X (w_j = exp(cs_last -
        // cs_j) dt_j), hi and lo, into the C region in the x tile's own MN-major
        // layout; Y_off summed over its hi/lo halves and scaled by exp(cs_i)
        {
            const bool got =
                (SO || mbar_wait(bar_yoff, ph, nullptr)) && mbar_wait(bar_x, ph, nullptr);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int it = tid + kThreads * r;
            const int j = it >> 3, c = it & 7;
            const uint32_t off = (uint32_t)(j * 128 + ((c ^ (j & 7)) << 4));
            const uint4 xv = *reinterpret_cast<const uint4*>(smem + kRX + off);
            const float w = ex2_approx(cs2_last + s_q2[j]);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            uint32_t hp[4], lp[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                split2_bf16(__fmul_rn(bf16lo(xw[e]), w), __fmul_rn(bf16hi(xw[e]), w), hp[e], lp[e]);
            *reinterpret_cast<uint4*>(smem + kRC + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
            *reinterpret_cast<uint4*>(smem + kRC + 16384 + off) =
                make_uint4(lp[0], lp[1], lp[2], lp[3]);
        }
        if (!SO && carry) {
            float yo[kHalf], yl[kHalf];
            tmem_ld32(t_lane + kTmY + kHalf * part, yo);
            tmem_ld32(t_lane + kTmY + kP + kHalf * part, yl);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < kHalf; ++q) yo[q] = (yo[q] + yl[q]) * e_i;
            tmem_st32f(t_lane + kTmY + kHalf * part, yo);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA batch 2: S_chunk^T = B^T X' (hi + lo), committed on its own;
        // then Y += M' X (hi + lo)
        if (tid == 0) {
            tc_fence_after();
            // states only: the B tile (no G product waited for it)
            const bool go = !SO || mbar_wait(bar_cb, ph, nullptr);
            if (SO) tc_fence_after();
            constexpr uint32_t idS = idesc_bf16_f32(128, 64) | kIdescAMN | kIdescBMN;
            constexpr uint32_t idY = idesc_bf16_f32(128, 64) | kIdescBMN;
            if (go) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_bf16(tmem + kTmS, mdesc(sbase + kRB, kk, 16384),
                             mdesc(sbase + kRC, kk, 16384), idS, kk > 0);
                    mma_bf16(tmem + kTmS, mdesc(sbase + kRB, kk, 16384),
                             mdesc(sbase + kRC + 16384, kk, 16384), idS, 1);
                }
                mma_commit(bar_s);
                if constexpr (!SO) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        mma_bf16_ta(tmem + kTmY, tmem + kTmG + mcol_hi(kk),
                                    mdesc(sbase + kRX, kk, 16384), idY,
                                    (carry || kk > 0) ? 1u : 0u);
                        mma_bf16_ta(tmem + kTmY, tmem + kTmG + mcol_hi(kk) + 16,
                                    mdesc(sbase + kRX, kk, 16384), idY, 1);
                    }
                }
                mma_commit(bar_mma2);
            }
        }
        // ---- next step's loads (the next block, or the next item's first):
        // C and B once S_chunk has read the B and X' regions, x after Y_diag
        bool got2 = true;
        if (tid == kLoader && st + 1 < nsteps) {
            got2 = mbar_wait(bar_s, ph, nullptr);
            if (got2) load_cb(st + 1);
        }
        got2 = mbar_wait(bar_mma2, ph, nullptr) && got2;
        if (!named_bar_and(1, kThreads, got2)) { ok = false; break; }
        tc_fence_after();
        if (tid == kLoader && st + 1 < nsteps) load_x(st + 1);

        // ---- rows of Y and of S_chunk^T out of tensor memory; the y tile is
        // staged in the S region (128-byte rows, 16-byte chunks XOR-swizzled by
        // row mod 8): fp32 as two [128 t][32 p] halves, bf16 as one [128 t][64 p]
        float sc[kHalf];
        if constexpr (SO) {
            tmem_ld32(t_lane + kTmS + kHalf * part, sc);
            tmem_wait_ld();
        } else {
            float yv[kHalf];
            tmem_ld32(t_lane + kTmY + kHalf * part, yv);
            tmem_ld32(t_lane + kTmS + kHalf * part, sc);
            tmem_wait_ld();
            if constexpr (sizeof(Tout) == 4) {
                uint8_t* box = smem + kRS + part * 16384 + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(box + ((c ^ (row & 7)) << 4)) =
                        make_float4(yv[4 * c], yv[4 * c + 1], yv[4 * c + 2], yv[4 * c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(smem + kRS + row * 128 +
                                              (((part * 4 + c) ^ (row & 7)) << 4)) =
                        make_uint4(pack_bf16(yv[8 * c], yv[8 * c + 1]),
                                   pack_bf16(yv[8 * c + 2], yv[8 * c + 3]),
                                   pack_bf16(yv[8 * c + 4], yv[8 * c + 5]),
                                   pack_bf16(yv[8 * c + 6], yv[8 * c + 7]));
            }
        }
        fence_proxy_async_smem();  // the staged tile is read by the TMA store
        tc_fence_before();  // every TMEM read of the step precedes the next step's MMAs
        __syncthreads();
        if (tid == 0) tc_fence_after();

        // ---- y out of the staged tile by TMA stores (one thread; rows past
        // the sequence end are clipped by the map)
        if ((BS == 0 || a.y != nullptr) && tid == kLoader) {
            if constexpr (sizeof(Tout) == 4) {
                tma_store_3d(&tm_y, smem + kRS, h * kP, t0, b);
                tma_store_3d(&tm_y, smem + kRS + 16384, h * kP + kHalf, t0, b);
            } else {
                tma_store_3d(&tm_y, smem + kRS, h * kP, t0, b);
            }
            bulk_commit();
        }

        // ---- state: S_prev[n = row][32 part + :] = exp(cs_last) S_prev + S_chunk^T;
        // at the item's last block, its final state [b][h][p = 32 part + :][n = row]
#pragma unroll
        for (int q = 0; q < kHalf; ++q) S[q] = fmaf(a_blk, S[q], sc[q]);
        if (blk == nblocks - 1) {
            if constexpr (BS != 0) {
                float* bs = a.bstates + (((long long)item * (nblocks + 1) + nblocks) * kP +
                                         kHalf * part) * kNs + row;
#pragma unroll
                for (int q = 0; q < kHalf; ++q) bs[q * kNs] = S[q];
            }
            if (a.final_state) {
                float* fs =
                    a.final_state + ((long long)(b * a.nheads + h) * kP + kHalf * part) * kNs + row;
#pragma unroll
                for (int q = 0; q < kHalf; ++q) fs[q * kNs] = S[q];
            }
#pragma unroll
            for (int q = 0; q < kHalf; ++q) S[q] = 0.0f;
        }
    }
    (void)ok;

    if (tid == kLoader) {
        bulk_wait_all();  // every y store has completed
        // never leave with a load still landing in shared memory: wait (bounded)
        // for the phase of the last load issued on each barrier
        if (cb_issued > 0) (void)mbar_wait(bar_cb, (uint32_t)((cb_issued - 1) & 1), nullptr);
        if (x_issued > 0) (void)mbar_wait(bar_x, (uint32_t)((x_issued - 1) & 1), nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <typename Tout, bool M3, int RK, int BS = 0>
ssm_status_t launch(const CUtensorMap& mc, const CUtensorMap& mb, const CUtensorMap& mx,
                    const CUtensorMap& my, const SsdArgs& a, cudaStream_t s) {
    auto kern = ssd_fwd_kernel<Tout, M3, RK, BS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    // persistent: two CTAs per SM (shared memory and tensor memory are sized
    // for two), each looping over (batch, head) items
    static std::mutex m;
    static int cached_dev = -1, sms = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(m);
        if (dev != cached_dev) {
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                sms <= 0)
                return SSM_ERR_CUDA;
            cached_dev = dev;
        }
    }
    const long long items = (long long)a.batch * a.nheads;
    const unsigned grid = (unsigned)std::min<long long>(items, 2LL * sms);
    kern<<<grid, kThreads, kSmemBytes, s>>>(mc, mb, mx, my, a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// Validation and launch shared by the Mamba-2 (m3 = false), Mamba-3 SISO
// (m3, rank 1) and Mamba-3 MIMO (m3, rank > 1) entry points.  seqlen counts
// steps; x, y, B, C hold `rank` sub-tokens per step.
ssm_status_t ssd_entry(const void* x, const float* dt, const float* lam, const float* A_head,
                       const void* B, const void* C, int chunk, int rank,
                       const float* initial_state, const void* prev_B, const void* prev_x,
                       void* y, float* final_state, float* bstates, int batch, int seqlen,
                       int nheads, int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
                       ssm_dtype_t out_dtype, bool m3, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1 || rank < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    // ranks 1, 2, 4 with chunk * rank = 64 sub-tokens (the pages: chunk 64 for
    // SISO, 16 for MIMO rank 4)
    if ((rank != 1 && rank != 2 && rank != 4) || chunk * rank != 64 || headdim != kP ||
        dstate != kNs || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    if ((long long)seqlen * rank > (long long)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * seqlen * rank;   // sub-token rows
    const size_t steps = (size_t)batch * seqlen;
    if (batch == 0 || nheads == 0) return SSM_OK;
    if ((size_t)batch * nheads > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    if (m3 && ((prev_B == nullptr) != (prev_x == nullptr))) return SSM_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sb = (size_t)batch * nheads * headdim * dstate * 4;  // one state tensor
    if (seqlen == 0) {  // empty sequence: the state passes through unchanged
        if (final_state && !aligned16(final_state)) return SSM_ERR_ALIGN;
        if (initial_state && !aligned16(initial_state)) return SSM_ERR_ALIGN;
        if (final_state && initial_state != final_state) {
            if (initial_state && overlaps(final_state, sb, initial_state, sb)) return SSM_ERR_ALIAS;
            const cudaError_t e =
                initial_state ? cudaMemcpyAsync(final_state, initial_state, sb,
                                                cudaMemcpyDeviceToDevice, s)
                              : cudaMemsetAsync(final_state, 0, sb, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    if (!x || !dt || !A_head || !B || !C || (!y && !bstates)) return SSM_ERR_NULL;
    if (m3 && !lam) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A_head, B, C, y, final_state, initial_state, lam, prev_B, prev_x};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = rows * nheads * headdim * 2;
    const size_t yb = rows * nheads * headdim * dtype_size(out_dtype);
    const size_t bcb = rows * ngroups * dstate * 2;
    const size_t fb = final_state ? sb : 0;
    // initial_state may be final_state itself (each (batch, head) state is read
    // before it is written, by the same threads), but no other overlap
    const size_t ib = (initial_state && initial_state != final_state) ? sb : 0;
    struct R { const void* p; size_t n; } ins[] = {
        {x, xb}, {dt, steps * nheads * 4}, {A_head, (size_t)nheads * 4}, {B, bcb}, {C, bcb},
        {initial_state, ib}, {lam, m3 ? steps * nheads * 4 : 0},
        {prev_B, m3 && prev_B ? (size_t)batch * rank * ngroups * dstate * 2 : 0},
        {prev_x, m3 && prev_x ? (size_t)batch * rank * nheads * headdim * 2 : 0}};
    for (const R& r : ins)
        if (overlaps(y, yb, r.p, r.n) || overlaps(final_state, fb, r.p, r.n)) return SSM_ERR_ALIAS;
    if (overlaps(y, yb, final_state, fb)) return SSM_ERR_ALIAS;
    if (initial_state && overlaps(y, yb, initial_state, sb)) return SSM_ERR_ALIAS;
    if (bstates) {
        if (!aligned16(bstates)) return SSM_ERR_ALIGN;
        const size_t bsb =
            (size_t)batch * nheads * (((size_t)seqlen * rank + kQ - 1) / kQ + 1) * kP * kNs * 4;
        for (const R& r : ins)
            if (overlaps(bstates, bsb, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(bstates, bsb, y, yb) || overlaps(bstates, bsb, final_state, fb) ||
            (initial_state && overlaps(bstates, bsb, initial_state, sb)))
            return SSM_ERR_ALIAS;
    }

    CUtensorMap mc, mb, mx, my;
    const int nsub = seqlen * rank;
    if (!make_bc_map(&mc, C, batch, nsub, ngroups) || !make_bc_map(&mb, B, batch, nsub, ngroups) ||
        !make_x_map(&mx, x, batch, nsub, nheads))
        return SSM_ERR_CUDA;
    memset(&my, 0, sizeof(my));
    if (y && !make_y_map(&my, y, batch, nsub, nheads, out_dtype)) return SSM_ERR_CUDA;
    SsdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dt = dt;
    a.A = A_head;
    a.h0 = initial_state;
    a.lam = lam;
    a.prev_B = static_cast<const __nv_bfloat16*>(prev_B);
    a.prev_x = static_cast<const __nv_bfloat16*>(prev_x);
    a.y = y;
    a.final_state = final_state;
    a.batch = batch;
    a.seqlen = seqlen;
    a.nheads = nheads;
    a.ngroups = ngroups;
    const bool bf = out_dtype == SSM_BF16;
    if (bstates) {  // the states the gradients start from, kept by the forward
        a.bstates = bstates;
        if (!m3)
            return bf ? launch<__nv_bfloat16, false, 1, 1>(mc, mb, mx, my, a, s)
                      : launch<float, false, 1, 1>(mc, mb, mx, my, a, s);
        switch (rank) {
            case 1: return bf ? launch<__nv_bfloat16, true, 1, 1>(mc, mb, mx, my, a, s)
                              : launch<float, true, 1, 1>(mc, mb, mx, my, a, s);
            case 2: return bf ? launch<__nv_bfloat16, true, 2, 1>(mc, mb, mx, my, a, s)
                              : launch<float, true, 2, 1>(mc, mb, mx, my, a, s);
            default: return bf ? launch<__nv_bfloat16, true, 4, 1>(mc, mb, mx, my, a, s)
                               : launch<float, true, 4, 1>(mc, mb, mx, my, a, s);
        }
    }
    if (!m3) return bf ? launch<__nv_bfloat16, false, 1>(mc, mb, mx, my, a, s)
                       : launch<float, false, 1>(mc, mb, mx, my, a, s);
    switch (rank) {
        case 1: return bf ? launch<__nv_bfloat16, true, 1>(mc, mb, mx, my, a, s)
                          : launch<float, true, 1>(mc, mb, mx, my, a, s);
        case 2: return bf ? launch<__nv_bfloat16, true, 2>(mc, mb, mx, my, a, s)
                          : launch<float, true, 2>(mc, mb, mx, my, a, s);
        default: return bf ? launch<__nv_bfloat16, true, 4>(mc, mb, mx, my, a, s)
                           : launch<float, true, 4>(mc, mb, mx, my, a, s);
    }
}

}  // namespace

namespace ssd_internal {

ssm_status_t ssd_forward_block_states(const void* x, const float* dt, const float* A_head,
                                      const void* B, const void* C, const float* initial_state,
                                      float* bstates, int batch, int seqlen, int nheads,
                                      int ngroups, cudaStream_t stream) {
    CUtensorMap mc, mb, mx, my;
    if (!make_bc_map(&mc, C, batch, seqlen, ngroups) || !make_bc_map(&mb, B, batch, seqlen, ngroups) ||
        !make_x_map(&mx, x, batch, seqlen, nheads))
        return SSM_ERR_CUDA;
    memset(&my, 0, sizeof(my));  // no y is written
    SsdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dt = dt;
    a.A = A_head;
    a.h0 = initial_state;
    a.y = nullptr;
    a.final_state = nullptr;
    a.bstates = bstates;
    a.batch = batch;
    a.seqlen = seqlen;
    a.nheads = nheads;
    a.ngroups = ngroups;
    return launch<float, false, 1, 2>(mc, mb, mx, my, a, stream);
}

// The Mamba-3 forward (SISO, or MIMO of rank 2 or 4 over 128-row blocks of
// sub-tokens) writing only the states its chunked form carries between blocks
// (bstates [batch * nheads][nblocks + 1][64][128]): the state entering each
// block including the pending term dt_{t+1} (1 - lambda_{t+1}) BX_t of the
// block's last step, and the final state.  Arguments are validated by the
// caller.
ssm_status_t ssd_mamba3_forward_block_states(const void* x, const float* dt, const float* lam,
                                             const float* A_head, const void* B, const void* C,
                                             const float* initial_state, const void* prev_B,
                                             const void* prev_x, float* bstates, int batch,
                                             int seqlen, int nheads, int ngroups,
                                             cudaStream_t stream, int rank) {
    const int nsub = seqlen * rank;
    CUtensorMap mc, mb, mx, my;
    if (!make_bc_map(&mc, C, batch, nsub, ngroups) || !make_bc_map(&mb, B, batch, nsub, ngroups) ||
        !make_x_map(&mx, x, batch, nsub, nheads))
        return SSM_ERR_CUDA;
    memset(&my, 0, sizeof(my));  // no y is written
    SsdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dt = dt;
    a.lam = lam;
    a.A = A_head;
    a.h0 = initial_state;
    a.prev_B = static_cast<const __nv_bfloat16*>(prev_B);
    a.prev_x = static_cast<const __nv_bfloat16*>(prev_x);
    a.y = nullptr;
    a.final_state = nullptr;
    a.bstates = bstates;
    a.batch = batch;
    a.seqlen = seqlen;
    a.nheads = nheads;
    a.ngroups = ngroups;
    switch (rank) {
        case 1: return launch<float, true, 1, 2>(mc, mb, mx, my, a, stream);
        case 2: return launch<float, true, 2, 2>(mc, mb, mx, my, a, stream);
        case 4: return launch<float, true, 4, 2>(mc, mb, mx, my, a, stream);
    }
    return SSM_ERR_UNSUPPORTED;
}

}  // namespace ssd_internal

extern "C" ssm_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A_head,
                                        const void* B, const void* C, int chunk,
                                        const float* initial_state, void* y,
                                        float* final_state, int batch, int seqlen, int nheads,
                                        int headdim, int dstate, int ngroups,
                                        ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                        void* stream) {
    return ssd_entry(x, dt, nullptr, A_head, B, C, chunk, 1, initial_state, nullptr, nullptr, y,
                     final_state, nullptr, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, false, stream);
}

extern "C" size_t ssd_chunked_checkpoint_bytes(int batch, int seqlen, int nheads, int headdim,
                                               int dstate) {
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim != kP || dstate != kNs) return 0;
    const size_t nblocks = ((size_t)seqlen + kQ - 1) / kQ;
    return (size_t)batch * nheads * (nblocks + 1) * kP * kNs * sizeof(float);
}

extern "C" ssm_status_t ssd_chunked_fwd_ckpt(const void* x, const float* dt, const float* A_head,
                                             const void* B, const void* C, int chunk,
                                             const float* initial_state, void* y,
                                             float* final_state, float* block_states, int batch,
                                             int seqlen, int nheads, int headdim, int dstate,
                                             int ngroups, ssm_dtype_t in_dtype,
                                             ssm_dtype_t out_dtype, void* stream) {
    if (!block_states && batch > 0 && nheads > 0 && seqlen > 0) return SSM_ERR_NULL;
    return ssd_entry(x, dt, nullptr, A_head, B, C, chunk, 1, initial_state, nullptr, nullptr, y,
                     final_state, block_states, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, false, stream);
}

extern "C" ssm_status_t ssd_mamba3_fwd_ckpt(const void* x, const float* dt, const float* lam,
                                            const float* A_head, const void* B, const void* C,
                                            int chunk, const float* initial_state,
                                            const void* prev_B, const void* prev_x, void* y,
                                            float* final_state, float* block_states, int batch,
                                            int seqlen, int nheads, int headdim, int dstate,
                                            int ngroups, ssm_dtype_t in_dtype,
                                            ssm_dtype_t out_dtype, void* stream) {
    if (!block_states && batch > 0 && nheads > 0 && seqlen > 0) return SSM_ERR_NULL;
    return ssd_entry(x, dt, lam, A_head, B, C, chunk, 1, initial_state, prev_B, prev_x, y,
                     final_state, block_states, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, true, stream);
}

extern "C" ssm_status_t ssd_mamba3_mimo_fwd_ckpt(
    const void* x, const float* dt, const float* lam, const float* A_head, const void* B,
    const void* C, int chunk, int rank, const float* initial_state, const void* prev_B,
    const void* prev_x, void* y, float* final_state, float* block_states, int batch, int seqlen,
    int nheads, int headdim, int dstate, int ngroups, ssm_dtype_t in_dtype,
    ssm_dtype_t out_dtype, void* stream) {
    if (!block_states && batch > 0 && nheads > 0 && seqlen > 0) return SSM_ERR_NULL;
    return ssd_entry(x, dt, lam, A_head, B, C, chunk, rank, initial_state, prev_B, prev_x, y,
                     final_state, block_states, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, true, stream);
}

extern "C" ssm_status_t ssd_mamba3_fwd(const void* x, const float* dt, const float* lam,
                                       const float* A_head, const void* B, const void* C,
                                       int chunk, const float* initial_state, const void* prev_B,
                                       const void* prev_x, void* y, float* final_state,
                                       int batch, int seqlen, int nheads, int headdim,
                                       int dstate, int ngroups, ssm_dtype_t in_dtype,
                                       ssm_dtype_t out_dtype, void* stream) {
    return ssd_entry(x, dt, lam, A_head, B, C, chunk, 1, initial_state, prev_B, prev_x, y,
                     final_state, nullptr, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, true, stream);
}

extern "C" ssm_status_t ssd_mamba3_mimo_fwd(const void* x, const float* dt, const float* lam,
                                            const float* A_head, const void* B, const void* C,
                                            int chunk, int rank, const float* initial_state,
                                            const void* prev_B, const void* prev_x, void* y,
                                            float* final_state, int batch, int seqlen,
                                            int nheads, int headdim, int dstate, int ngroups,
                                            ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                            void* stream) {
    return ssd_entry(x, dt, lam, A_head, B, C, chunk, rank, initial_state, prev_B, prev_x, y,
                     final_state, nullptr, batch, seqlen, nheads, headdim, dstate, ngroups,
                     in_dtype, out_dtype, true, stream);
}
