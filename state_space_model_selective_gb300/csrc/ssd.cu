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
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace {

using namespace ssm;

constexpr int kQ = 128;   // steps per block (MMA M)
constexpr int kP = 64;    // headdim
constexpr int kNs = 128;  // dstate
constexpr int kGroups = 4;                // warpgroups; each per-row phase splits the columns
constexpr int kThreads = 128 * kGroups;
constexpr int kPart = kP / kGroups;       // columns of a 64-wide row per warpgroup

// shared-memory regions (offsets from a 1024-aligned base)
constexpr uint32_t kRC = 0;            // C tile [128 t][128 n]  -> later M' hi
constexpr uint32_t kRB = 32768;        // B tile [128 j][128 n]  -> later M' lo
constexpr uint32_t kRBT = 65536;       // x tile [128 j][64 p] -> B^T [128 n][128 j] -> S staging
constexpr uint32_t kRX = 98304;        // X^T [64 p][128 j]
constexpr uint32_t kRXP = 114688;      // X'^T hi [64][128] | lo [64][128]
constexpr uint32_t kRS = 147456;       // S hi [64 p][128 n] | lo [64][128]
constexpr uint32_t kMisc = 180224;     // cs, dt, w arrays, warp sums, barriers
constexpr uint32_t kSmemBytes = kMisc + 3 * kQ * 4 + 64 + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
constexpr uint32_t kTmemCols = 256;    // G / Y_diag: 0..127, Y_off: 128..191, S^T: 192..255

struct SsdArgs {
    const __nv_bfloat16* x;
    const float* dt;
    const float* A;
    void* y;
    float* final_state;
    int batch, seqlen, nheads, ngroups;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi); returns (hi, lo) as floats
__device__ __forceinline__ void split_bf16(float v, float& hi, float& lo) {
    hi = __bfloat162float(__float2bfloat16_rn(v));
    lo = v - hi;
}

// K-major operand descriptor for k-step kk (16 bf16) of a tile with R rows.
template <int R>
__device__ __forceinline__ uint64_t kdesc(uint32_t tile_saddr, int kk) {
    return smem_desc_k128(tile_saddr + (uint32_t)((kk >> 2) * (R * 128) + (kk & 3) * 32));
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_fwd_kernel(const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_B,
                   const __grid_constant__ CUtensorMap tm_x, const SsdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(smem);
    float* s_cs = reinterpret_cast<float*>(smem + kMisc);
    float* s_dt = s_cs + kQ;
    float* s_w = s_dt + kQ;
    float* s_wsum = s_w + kQ;  // [4] warp totals
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + kMisc + 3 * kQ * 4 + 32);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_mma + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int part = warp >> 2;     // which part of a row's columns this warp takes
    const int row = quarter * 32 + lane;  // the TMEM lane (row i, or state n) of this thread
    const int h = blockIdx.x % a.nheads;
    const int b = blockIdx.x / a.nheads;
    const int g = h / (a.nheads / a.ngroups);
    const float Ah = a.A[h];

    if (warp == 0) tmem_alloc(s_tmem, kTmemCols);
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_C);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_x);
    }
    // S_prev = 0: zero both halves of the S operand tile
    for (int i = tid; i < 32768 / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kRS)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane base

    float S[kPart];  // S_prev[n = row][part * kPart + p]
#pragma unroll
    for (int p = 0; p < kPart; ++p) S[p] = 0.0f;

    const int nblocks = (a.seqlen + kQ - 1) / kQ;
    const long long xrow0 = (long long)b * a.seqlen;
    bool ok = true;
    uint32_t tma_phase = 0;
    // dt of this block's step tid, loaded one block ahead
    float dt_next = (tid < kQ && tid < a.seqlen) ? a.dt[(xrow0 + tid) * a.nheads + h] : 0.0f;

    for (int blk = 0; blk < nblocks && ok; ++blk) {
        const int t0 = blk * kQ;
        const int nv = min(kQ, a.seqlen - t0);

        if (tid == 0) {
            mbar_arrive_expect_tx(bar_tma, 5 * 16384);
            tma_load_4d(smem + kRC, &tm_C, bar_tma, 0, g, t0, b);
            tma_load_4d(smem + kRC + 16384, &tm_C, bar_tma, 64, g, t0, b);
            tma_load_4d(smem + kRB, &tm_B, bar_tma, 0, g, t0, b);
            tma_load_4d(smem + kRB + 16384, &tm_B, bar_tma, 64, g, t0, b);
            tma_load_3d(smem + kRBT, &tm_x, bar_tma, h * kP, t0, b);
        }

        // ---- cumulative log-decay of the block (padding steps: dt = 0); the
        // first warpgroup holds one step per thread
        const float dti = dt_next;
        dt_next = (tid < kQ && t0 + kQ + tid < a.seqlen)
                      ? a.dt[(xrow0 + t0 + kQ + tid) * a.nheads + h]
                      : 0.0f;  // padding steps of a partial last block: dt = 0
        float v = dti * Ah;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31 && warp < 4) s_wsum[warp] = v;
        __syncthreads();
        if (tid < kQ) {
            for (int w = 0; w < warp; ++w) v += s_wsum[w];
            s_cs[tid] = v;
            s_dt[tid] = dti;
        }
        __syncthreads();
        const float cs_last = s_cs[kQ - 1];
        if (tid < kQ) s_w[tid] = ex2_approx((cs_last - v) * kLog2e) * dti;
        const float e_i = ex2_approx(s_cs[row] * kLog2e);
        const float a_blk = ex2_approx(cs_last * kLog2e);
        __syncthreads();

        // ---- C, B tiles landed?  Then B^T [128 n][128 j] (exact)
        {
            const bool got = mbar_wait(bar_tma, tma_phase, nullptr);
            tma_phase ^= 1;
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        // ---- X^T (exact) and X'^T = (w o X)^T split hi/lo, [64 p][128 j],
        // from the x tile [128 j][64 p] that TMA put in the B^T region
        for (int item = tid; item < kP * (kQ / 8); item += kThreads) {
            const int p = item % kP, jg = item / kP;
            float xv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                xv[q] = bf16lo(*reinterpret_cast<const uint16_t*>(
                    smem + kRBT + kmaj_off<kQ>(jg * 8 + q, p)));
            float hi[8], lo[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) split_bf16(s_w[jg * 8 + q] * xv[q], hi[q], lo[q]);
            const uint4 wx = make_uint4(pack_bf16(xv[0], xv[1]), pack_bf16(xv[2], xv[3]),
                                        pack_bf16(xv[4], xv[5]), pack_bf16(xv[6], xv[7]));
            const uint4 wh = make_uint4(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]),
                                        pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7]));
            const uint4 wl = make_uint4(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]),
                                        pack_bf16(lo[4], lo[5]), pack_bf16(lo[6], lo[7]));
            const uint32_t off = kmaj_off<kP>(p, jg * 8);
            *reinterpret_cast<uint4*>(smem + kRX + off) = wx;
            *reinterpret_cast<uint4*>(smem + kRXP + off) = wh;
            *reinterpret_cast<uint4*>(smem + kRXP + 16384 + off) = wl;
        }
        __syncthreads();  // the x tile is read; B^T overwrites it
        for (int item = tid; item < kNs * (kQ / 8); item += kThreads) {
            const int n = item % kNs, jg = item / kNs;
            uint16_t e[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                e[q] = *reinterpret_cast<const uint16_t*>(smem + kRB + kmaj_off<kQ>(jg * 8 + q, n));
            const uint4 w4 = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                                        e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
            *reinterpret_cast<uint4*>(smem + kRBT + kmaj_off<kNs>(n, jg * 8)) = w4;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA batch 1: G = C B^T, Y_off = C S^T (hi + lo), S_chunk^T = B^T X'^T^T (hi + lo)
        if (tid == 0) {
            constexpr uint32_t id128 = idesc_bf16_f32(128, 128);
            constexpr uint32_t id64 = idesc_bf16_f32(128, 64);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 0, kdesc<kQ>(sbase + kRC, kk), kdesc<kQ>(sbase + kRB, kk), id128,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 128, kdesc<kQ>(sbase + kRC, kk), kdesc<kP>(sbase + kRS, kk), id64,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 128, kdesc<kQ>(sbase + kRC, kk),
                         kdesc<kP>(sbase + kRS + 16384, kk), id64, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 192, kdesc<kNs>(sbase + kRBT, kk), kdesc<kP>(sbase + kRXP, kk),
                         id64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 192, kdesc<kNs>(sbase + kRBT, kk),
                         kdesc<kP>(sbase + kRXP + 16384, kk), id64, 1);
            mma_commit(bar_mma);
        }
        {
            const bool got = mbar_wait(bar_mma, 0, nullptr);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();

        // ---- M' row i = row from G (TMEM cols 0..127) -> hi into RC, lo into RB;
        // warpgroup `part` takes columns 32 part .. 32 part + 31.  Chunks wholly
        // above the causal diagonal (all j > i for the warp's rows) are zero.
        {
            const float csi = s_cs[row];
            const int c = part;
            if (c > quarter) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    const uint32_t off = kmaj_off<kQ>(row, c * 32 + q8 * 8);
                    *reinterpret_cast<uint4*>(smem + kRC + off) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(smem + kRB + off) = make_uint4(0, 0, 0, 0);
                }
            } else {
                float gv[32];
                tmem_ld32(t_lane + c * 32, gv);
                tmem_wait_ld();
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int j = c * 32 + q8 * 8 + q;
                        float m = 0.0f;
                        if (j <= row) m = gv[q8 * 8 + q] * ex2_approx((csi - s_cs[j]) * kLog2e) * s_dt[j];
                        split_bf16(m, hi[q], lo[q]);
                    }
                    const uint32_t off = kmaj_off<kQ>(row, c * 32 + q8 * 8);
                    *reinterpret_cast<uint4*>(smem + kRC + off) =
                        make_uint4(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]),
                                   pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7]));
                    *reinterpret_cast<uint4*>(smem + kRB + off) =
                        make_uint4(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]),
                                   pack_bf16(lo[4], lo[5]), pack_bf16(lo[6], lo[7]));
                }
            }
        }
        // ---- state: S_prev[n = row][part * kPart + :] = exp(cs_last) S_prev + S_chunk^T;
        // staged as fp32 rows (16-byte chunks XOR-swizzled by n mod 8) in RBT
        {
            float sc[kPart];
            tmem_ld16(t_lane + 192 + part * kPart, sc);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < kPart; ++q) S[q] = fmaf(a_blk, S[q], sc[q]);
            float* st = reinterpret_cast<float*>(smem + kRBT) + row * kP;
#pragma unroll
            for (int c4 = 0; c4 < kPart / 4; ++c4)
                reinterpret_cast<float4*>(st)[(part * (kPart / 4) + c4) ^ (row & 7)] =
                    make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- MMA batch 2: Y_diag = M' X (hi + lo) into TMEM cols 0..63
        if (tid == 0) {
            constexpr uint32_t id64 = idesc_bf16_f32(128, 64);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 0, kdesc<kQ>(sbase + kRC, kk), kdesc<kP>(sbase + kRX, kk), id64,
                         kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + 0, kdesc<kQ>(sbase + kRB, kk), kdesc<kP>(sbase + kRX, kk), id64, 1);
            mma_commit(bar_mma);
        }

        // ---- S operand for the next block: [64 p][128 n] hi/lo from the staging
        for (int item = tid; item < kP * (kNs / 8); item += kThreads) {
            const int p = item % kP, ng = item / kP;
            float hi[8], lo[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int n = ng * 8 + q;
                const float* st = reinterpret_cast<const float*>(smem + kRBT) + n * kP;
                const float sv = st[(((p >> 2) ^ (n & 7)) << 2) | (p & 3)];
                split_bf16(sv, hi[q], lo[q]);
            }
            const uint32_t off = kmaj_off<kP>(p, ng * 8);
            *reinterpret_cast<uint4*>(smem + kRS + off) =
                make_uint4(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]),
                           pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7]));
            *reinterpret_cast<uint4*>(smem + kRS + 16384 + off) =
                make_uint4(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]),
                           pack_bf16(lo[4], lo[5]), pack_bf16(lo[6], lo[7]));
        }

        {
            const bool got = mbar_wait(bar_mma, 1, nullptr);
            if (!named_bar_and(1, kThreads, got)) { ok = false; break; }
        }
        tc_fence_after();

        // ---- y[i = row][part * kPart + :] = Y_diag + exp(cs_i) Y_off
        {
            float yd[kPart], yo[kPart];
            Tout* yrow = reinterpret_cast<Tout*>(a.y) + ((xrow0 + t0 + row) * a.nheads + h) * kP;
            {
                const int c = part;
                tmem_ld16(t_lane + c * kPart, yd);
                tmem_ld16(t_lane + 128 + c * kPart, yo);
                tmem_wait_ld();
                if (row < nv) {
                    if constexpr (sizeof(Tout) == 4) {
#pragma unroll
                        for (int q = 0; q < kPart; q += 4)
                            *reinterpret_cast<float4*>(reinterpret_cast<float*>(yrow) + c * kPart + q) =
                                make_float4(fmaf(e_i, yo[q], yd[q]), fmaf(e_i, yo[q + 1], yd[q + 1]),
                                            fmaf(e_i, yo[q + 2], yd[q + 2]),
                                            fmaf(e_i, yo[q + 3], yd[q + 3]));
                    } else {
#pragma unroll
                        for (int q = 0; q < kPart; q += 8)
                            *reinterpret_cast<uint4*>(yrow + c * kPart + q) = make_uint4(
                                pack_bf16(fmaf(e_i, yo[q], yd[q]), fmaf(e_i, yo[q + 1], yd[q + 1])),
                                pack_bf16(fmaf(e_i, yo[q + 2], yd[q + 2]),
                                          fmaf(e_i, yo[q + 3], yd[q + 3])),
                                pack_bf16(fmaf(e_i, yo[q + 4], yd[q + 4]),
                                          fmaf(e_i, yo[q + 5], yd[q + 5])),
                                pack_bf16(fmaf(e_i, yo[q + 6], yd[q + 6]),
                                          fmaf(e_i, yo[q + 7], yd[q + 7])));
                    }
                }
            }
        }
        fence_proxy_async_smem();  // generic reads/writes before the next block's TMA
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // ---- final state [b][h][p = part * kPart + :][n = row]
    if (ok && a.final_state) {
        float* fs = a.final_state + ((long long)(b * a.nheads + h) * kP + part * kPart) * kNs + row;
#pragma unroll
        for (int p = 0; p < kPart; ++p) fs[p * kNs] = S[p];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool make_bc_map(CUtensorMap* map, const void* base, int batch, int seqlen, int ngroups) {
    ssm_host::EncodeTiledFn fn = ssm_host::encode_tiled_fn();
    if (!fn) return false;
    // (batch, seqlen, ngroups, dstate) as 4-D {dstate, ngroups, seqlen, batch}
    const cuuint64_t dims[4] = {(cuuint64_t)kNs, (cuuint64_t)ngroups, (cuuint64_t)seqlen,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)kNs * 2, (cuuint64_t)ngroups * kNs * 2,
                                   (cuuint64_t)seqlen * ngroups * kNs * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_x_map(CUtensorMap* map, const void* base, int batch, int seqlen, int nheads) {
    ssm_host::EncodeTiledFn fn = ssm_host::encode_tiled_fn();
    if (!fn) return false;
    // (batch, seqlen, nheads, headdim) as 3-D {nheads * headdim, seqlen, batch}
    const cuuint64_t dims[3] = {(cuuint64_t)nheads * kP, (cuuint64_t)seqlen, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)nheads * kP * 2,
                                   (cuuint64_t)seqlen * nheads * kP * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kP, (cuuint32_t)kQ, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <typename Tout>
ssm_status_t launch(const CUtensorMap& mc, const CUtensorMap& mb, const CUtensorMap& mx,
                    const SsdArgs& a, cudaStream_t s) {
    auto kern = ssd_fwd_kernel<Tout>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    const unsigned grid = (unsigned)(a.batch * a.nheads);
    kern<<<grid, kThreads, kSmemAlloc, s>>>(mc, mb, mx, a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" ssm_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A_head,
                                        const void* B, const void* C, int chunk, void* y,
                                        float* final_state, int batch, int seqlen, int nheads,
                                        int headdim, int dstate, int ngroups,
                                        ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                        void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    if (chunk != 64 || headdim != kP || dstate != kNs || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * seqlen;
    if (batch == 0 || nheads == 0) return SSM_OK;
    if ((size_t)batch * nheads > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (seqlen == 0) {  // empty sequence: the state stays zero
        const size_t fb0 = (size_t)batch * nheads * headdim * dstate * 4;
        if (final_state && !aligned16(final_state)) return SSM_ERR_ALIGN;
        if (final_state && cudaMemsetAsync(final_state, 0, fb0, s) != cudaSuccess)
            return SSM_ERR_CUDA;
        return SSM_OK;
    }
    if (!x || !dt || !A_head || !B || !C || !y) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A_head, B, C, y, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = rows * nheads * headdim * 2;
    const size_t yb = rows * nheads * headdim * dtype_size(out_dtype);
    const size_t bcb = rows * ngroups * dstate * 2;
    const size_t fb = final_state ? (size_t)batch * nheads * headdim * dstate * 4 : 0;
    struct R { const void* p; size_t n; } ins[] = {
        {x, xb}, {dt, rows * nheads * 4}, {A_head, (size_t)nheads * 4}, {B, bcb}, {C, bcb}};
    for (const R& r : ins)
        if (overlaps(y, yb, r.p, r.n) || overlaps(final_state, fb, r.p, r.n)) return SSM_ERR_ALIAS;
    if (overlaps(y, yb, final_state, fb)) return SSM_ERR_ALIAS;

    CUtensorMap mc, mb, mx;
    if (!make_bc_map(&mc, C, batch, seqlen, ngroups) || !make_bc_map(&mb, B, batch, seqlen, ngroups) ||
        !make_x_map(&mx, x, batch, seqlen, nheads))
        return SSM_ERR_CUDA;
    SsdArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.dt = dt;
    a.A = A_head;
    a.y = y;
    a.final_state = final_state;
    a.batch = batch;
    a.seqlen = seqlen;
    a.nheads = nheads;
    a.ngroups = ngroups;
    return out_dtype == SSM_BF16 ? launch<__nv_bfloat16>(mc, mb, mx, a, s)
                                 : launch<float>(mc, mb, mx, a, s);
}
