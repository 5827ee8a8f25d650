// scan_bwd.cu -- gradient of the selective scan (ssm_scan_bwd) for GB300 /
// sm_103a.
//
// What it computes: the reverse-mode derivative of ssm_scan_fwd's recurrence
// ("We brought Mamba to Trainium -- and mapped where custom kernels actually
// help", section "Mamba: bringing an unsupported model to the chip, and
// writing its missing kernel"; discretisation, D skip and gate as in
// "Mamba-3 NKI Kernels for AWS Neuron", section "How it works") for the loss
// sum(dy y) + sum(dfinal final_state):
//   lambda_t = dL/dh_t = dy0_t C_t + a_{t+1} lambda_{t+1},  dy0_t = dy_t silu(z_t)
//   dC_t += dy0_t h_t,  dB_t += lambda_t dl_t u_t,  dA += lambda_t h_{t-1} a_t dl_t
//   du_t = dy0_t D + sum_n lambda_t dl_t B_t,  ddelta_t = softplus'(.) sum_n
//   lambda_t (h_{t-1} A a_t + B_t u_t),  dz_t = dy_t y0_t silu'(z_t)
//
// How (three launches):
//  1. the forward kernel re-runs and writes only the state entering every
//     16-step segment (checkpoints);
//  2. scan_bwd_kernel: a CTA owns one (batch, group, 32-channel block) and
//     walks its 32-step tiles in reverse, with the forward kernel's lane map
//     (4 lanes per channel, 4 states each).  While a tile is computed, the
//     raw inputs of the tile before it (u, delta, dy, z, B, C and the two
//     checkpoints) stream into shared memory with 16-byte cp.async copies.
//     Per tile the per-step terms (dl, dl*u, dy0, u; softplus', dy silu')
//     are formed once per (channel, step); per 16-step segment the states
//     are recomputed from the checkpoint into registers, then the adjoint
//     recurrence runs backwards.  Sums over states (du, ddelta, the gate's
//     y0) are reduce-scattered over the channel's 4 lanes; sums over
//     channels (dB, dC) are reduce-scattered over a warp's 8 channels, then
//     the 4 warps' sums are added in warp order into a per-tile shared
//     buffer, which is written out as this channel block's partial;
//  3. scan_bwd_reduce_kernel adds the partials: dB, dC over channel blocks,
//     dA, dD, dbias over the batch (a fixed order, so results are
//     deterministic).
#include <algorithm>

#include "common.cuh"
#include "scan_internal.h"

namespace {

using namespace ssm;

constexpr int kN = 16;        // dstate
constexpr int kCH = 32;       // channels per CTA
constexpr int kThreads = 128; // 4 lanes x 32 channels
constexpr int kTL = 32;       // steps per tile
constexpr int kSeg = 16;      // steps per recomputed segment (one checkpoint)
constexpr int kSegPerTile = kTL / kSeg;
constexpr int kRecA = kTL * 16 + 16;  // bytes per channel row of recA (float4 per step, padded)
constexpr int kRecB = kTL * 8 + 16;   // bytes per channel row of recB (float2 per step, padded)
constexpr int kSumT = kN + 1;          // floats per step row of the tile's dB, dC sums (padded)
constexpr int kSegT = kSeg * kN + 16;  // floats per (warp, dB or dC) block of a segment (padded)

struct BwdArgs {
    const void* u;
    const void* delta;
    const void* z;
    const void* dy;
    const float* A;
    const float* Dskip;
    const float* bias;
    const void* Bm;
    const void* Cm;
    const float* ckpt;    // [ceil(L/16)][batch * dim][16]
    const float* dfinal;  // (batch, dim, 16) or NULL
    float* du;
    float* ddelta;
    float* dz;            // NULL when z is
    float* dh0;           // (batch, dim, 16) or NULL
    float* pBC;           // [bpg][batch][ngroups][2][16][L] partial dB, dC
    float* pA;            // [batch][dim][16]
    float* pD;            // [batch][dim]
    float* pbias;         // [batch][dim]
    int batch, dim, seqlen, ngroups, dpg, bpg, softplus;
};

// Shared memory (bytes from the base).  The raw tile holds one tile's inputs
// as they are in global memory: 4 activation arrays x 32 channel rows, B and
// C x 16 state rows (each row kTL elements, padded by 16 bytes), then the
// tile's two checkpoints [seg][channel][16] fp32.
template <typename T>
struct Lay {
    static constexpr int ES = sizeof(T);
    static constexpr int ROW = kTL * ES + 16;
    static constexpr int CHUNKS = kTL * ES / 16;  // 16-byte chunks per row
    static constexpr int ACT = 4 * kCH * ROW;     // u, delta, dy, z
    static constexpr int BCR = 2 * kN * ROW;      // B, C
    static constexpr int CK = kSegPerTile * kCH * kN * 4;
    static constexpr int RAW = ACT + BCR + CK;
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_RECA = OFF_RAW + RAW;
    static constexpr int OFF_RECB = OFF_RECA + kCH * kRecA;
    static constexpr int OFF_BC = OFF_RECB + kCH * kRecB;    // fp32 B [t][16] then C [t][16]
    static constexpr int OFF_SUM = OFF_BC + 2 * kTL * kN * 4;     // fp32 dB, dC [type][t][kSumT]
    static constexpr int OFF_SEG = OFF_SUM + 2 * kTL * kSumT * 4; // per warp: a segment's dB, dC
    static constexpr int OFF_CK = OFF_SEG + 4 * 2 * kSegT * 4;     // the checkpoints, copied
    static constexpr int SMEM = OFF_CK + CK;
    static_assert(OFF_RECA % 16 == 0 && OFF_BC % 16 == 0 && ROW % 16 == 0, "16-byte alignment");
};

__device__ __forceinline__ float sigmoid_f(float x) {
    return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// 16-byte asynchronous global -> shared copy; src_bytes < 16 zero-fills the
// rest (0: nothing is read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Starts (VEC: cp.async) or performs (plain loads) the copy of tile `tile`'s
// raw inputs into the raw area.  VEC requires rows of 16-byte multiples
// (seqlen * sizeof(T) % 16 == 0); then a 16-byte chunk is either wholly
// inside the sequence or wholly past it (zero-filled).  Channels past the
// group's end read nothing and hold zeros.
template <typename T, bool VEC>
__device__ __forceinline__ void fetch_tile(const BwdArgs& a, uint8_t* smem, int tile,
                                           long long row0, int cvalid, long long bcrow0,
                                           int tid) {
    using Y = Lay<T>;
    uint8_t* raw = smem + Y::OFF_RAW;
    const int t0 = tile * kTL;
    const long long L = a.seqlen;
    auto act = [&](int arr) -> const void* {
        return arr == 0 ? a.u : arr == 1 ? a.delta : arr == 2 ? a.dy : a.z;
    };
    if constexpr (VEC) {
        // activations and B, C: (4 * 32 + 2 * 16) rows x CHUNKS chunks
        constexpr int NCH = (4 * kCH + 2 * kN) * Y::CHUNKS;
        for (int i = tid; i < NCH; i += kThreads) {
            const int r = i / Y::CHUNKS, c = i % Y::CHUNKS;
            const int tc = t0 + c * (16 / Y::ES);  // first step of the chunk
            const char* src;
            bool ok;
            if (r < 4 * kCH) {
                const int arr = r / kCH, ch = r % kCH;
                ok = ch < cvalid && tc < a.seqlen && act(arr) != nullptr;
                src = static_cast<const char*>(ok ? act(arr) : a.u) +
                      (ok ? ((row0 + ch) * L + tc) * Y::ES : 0);
            } else {
                const int arr = (r - 4 * kCH) / kN, n = (r - 4 * kCH) % kN;
                ok = tc < a.seqlen;
                src = static_cast<const char*>(arr ? a.Cm : a.Bm) +
                      (ok ? ((bcrow0 + n) * L + tc) * Y::ES : 0);
            }
            cp_async16(raw + r * Y::ROW + c * 16, src, ok ? 16u : 0u);
        }
    } else {
        for (int i = tid; i < (4 * kCH + 2 * kN) * kTL; i += kThreads) {
            const int r = i / kTL, t = i % kTL;
            const int tg = t0 + t;
            T v = from_f32<T>(0.0f);
            if (r < 4 * kCH) {
                const int arr = r / kCH, ch = r % kCH;
                if (ch < cvalid && tg < a.seqlen && act(arr) != nullptr)
                    v = static_cast<const T*>(act(arr))[(row0 + ch) * L + tg];
            } else {
                const int arr = (r - 4 * kCH) / kN, n = (r - 4 * kCH) % kN;
                if (tg < a.seqlen)
                    v = static_cast<const T*>(arr ? a.Cm : a.Bm)[(bcrow0 + n) * L + tg];
            }
            reinterpret_cast<T*>(raw + r * Y::ROW)[t] = v;
        }
    }
    // checkpoints of the tile's segments: [seg][channel][16] fp32, 4 chunks each
    {
        const long long BD = (long long)a.batch * a.dim;
        const int nseg_total = (a.seqlen + kSeg - 1) / kSeg;
        float* ck = reinterpret_cast<float*>(raw + Y::ACT + Y::BCR);
        for (int i = tid; i < kSegPerTile * kCH * 4; i += kThreads) {
            const int s = i / (kCH * 4), ch = (i / 4) % kCH, c = i % 4;
            const long long seg = (long long)tile * kSegPerTile + s;
            const bool ok = seg < nseg_total && ch < cvalid;
            const float* src = a.ckpt + (ok ? (seg * BD + row0 + ch) * kN + c * 4 : 0);
            cp_async16(ck + (s * kCH + ch) * kN + c * 4, src, ok ? 16u : 0u);
        }
    }
    cp_async_commit();
}

// 8 consecutive elements of a raw row as fp32.
template <typename T>
__device__ __forceinline__ void load8(const uint8_t* p, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16lo(ws[i]);
            v[2 * i + 1] = bf16hi(ws[i]);
        }
    } else {
        const float4 a = *reinterpret_cast<const float4*>(p);
        const float4 b = *reinterpret_cast<const float4*>(p + 16);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// Per-step terms of one tile from the raw area, once per (channel, step):
// thread -> channel tid % 32, steps 8 (tid / 32) .. + 7.  Steps past the
// sequence end (tn = the tile's steps) and channels past the group get
// dl = 0 and dy = 0 (zero-filled): an identity step that contributes
// nothing.  Also converts B, C to fp32 [t][n].
template <typename T>
__device__ __forceinline__ void prep_tile(const BwdArgs& a, uint8_t* smem, float bias_p,
                                          bool pvalid, int tn, bool has_z, int tid) {
    using Y = Lay<T>;
    const uint8_t* raw = smem + Y::OFF_RAW;
    {
        const int pc = tid % kCH, pq = tid / kCH;
        float u[8], dl_[8], dy[8], zz[8];
        const int off = pq * 8 * Y::ES;
        load8<T>(raw + (0 * kCH + pc) * Y::ROW + off, u);
        load8<T>(raw + (1 * kCH + pc) * Y::ROW + off, dl_);
        load8<T>(raw + (2 * kCH + pc) * Y::ROW + off, dy);
        if (has_z) load8<T>(raw + (3 * kCH + pc) * Y::ROW + off, zz);
        float4* ra = reinterpret_cast<float4*>(smem + Y::OFF_RECA + pc * kRecA) + pq * 8;
        float2* rb = reinterpret_cast<float2*>(smem + Y::OFF_RECB + pc * kRecB) + pq * 8;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float x = dl_[j] + bias_p;
            const float dl = a.softplus ? softplus_f(x) : x;
            const float spd = a.softplus ? sigmoid_f(x) : 1.0f;
            float dy0 = dy[j], dygd = 0.0f;
            if (has_z) {
                const float sg = sigmoid_f(zz[j]);
                dy0 = dy[j] * zz[j] * sg;
                dygd = dy[j] * sg * fmaf(zz[j], 1.0f - sg, 1.0f);
            }
            // a step past the end must be the identity whatever the bias
            const bool live = pvalid && pq * 8 + j < tn;
            ra[j] = make_float4(live ? dl : 0.0f, live ? dl * u[j] : 0.0f, dy0, u[j]);
            rb[j] = make_float2(spd, dygd);
        }
    }
    {
        // a warp holds 16 states x one even and one odd q; odd q store their
        // steps pairwise swapped, so the two halves hit different banks
        const int arr = tid / 64, n = tid % kN, q = (tid / kN) % 4;
        float v[8];
        load8<T>(raw + (4 * kCH + arr * kN + n) * Y::ROW + q * 8 * Y::ES, v);
        float* bcf = reinterpret_cast<float*>(smem + Y::OFF_BC) + arr * kTL * kN;
        const bool odd = q & 1;
#pragma unroll
        for (int j = 0; j < 8; ++j) bcf[(q * 8 + (j ^ (int)odd)) * kN + n] = odd ? v[j ^ 1] : v[j];
    }
    // the checkpoints leave the raw area, which the next tile's copies reuse
    {
        const float4* src = reinterpret_cast<const float4*>(raw + Y::ACT + Y::BCR);
        float4* dst = reinterpret_cast<float4*>(smem + Y::OFF_CK);
#pragma unroll
        for (int i = tid; i < Y::CK / 16; i += kThreads) dst[i] = src[i];
    }
}

// v[8] -> one value summed over the 8 lanes that share lane bits 0-1 (a warp's
// 8 channels of one 4-state group): halve over lane bits 4, 3, 2.  The lane
// ends with v[4 bit4 + 2 bit3 + bit2] summed.
__device__ __forceinline__ float reduce_scatter8_channels(const float* v, int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w[4], w2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[i + 4];
        const float keep = b4 ? v[i + 4] : v[i];
        w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? w[i] : w[i + 2];
        const float keep = b3 ? w[i + 2] : w[i];
        w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? w2[0] : w2[1];
    const float keep = b2 ? w2[1] : w2[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 4);
}

template <typename T, bool VEC, bool Z>
__global__ void __launch_bounds__(kThreads, 3) scan_bwd_kernel(const BwdArgs a) {
    using Y = Lay<T>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cb = blockIdx.x % a.bpg, bg = blockIdx.x / a.bpg;
    const int g = bg % a.ngroups, b = bg / a.ngroups;
    const int d0 = g * a.dpg + cb * kCH;
    const int cvalid = min(kCH, a.dpg - cb * kCH);  // channels of this block in the group
    const long long row0 = (long long)b * a.dim + d0;
    const long long bcrow0 = (long long)bg * kN;
    const int cl = warp * 8 + (lane >> 2), ng = lane & 3, n0 = ng * 4;
    const int d = d0 + cl;
    const bool valid = cl < cvalid;
    const long long drow = row0 + cl;
    const long long L = a.seqlen;
    const float bias_p = (a.bias && tid % kCH < cvalid) ? a.bias[d0 + tid % kCH] : 0.0f;

    float A2[4], An[4], lam[4], dA[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        An[k] = valid ? a.A[(long long)d * kN + n0 + k] : 0.0f;
        A2[k] = An[k] * kLog2e;
        dA[k] = 0.0f;
        lam[k] = (valid && a.dfinal) ? a.dfinal[drow * kN + n0 + k] : 0.0f;
    }
    const float Dd = (a.Dskip && valid) ? a.Dskip[d] : 0.0f;
    float accD = 0.0f, accBias = 0.0f;
    const float4* recA = reinterpret_cast<const float4*>(smem + Y::OFF_RECA + cl * kRecA);
    const float2* recB = reinterpret_cast<const float2*>(smem + Y::OFF_RECB + cl * kRecB);
    const float* Bt = reinterpret_cast<const float*>(smem + Y::OFF_BC);
    const float* Ct = Bt + kTL * kN;
    float* sum = reinterpret_cast<float*>(smem + Y::OFF_SUM);  // [2][kTL][kSumT]
    float* segw = reinterpret_cast<float*>(smem + Y::OFF_SEG);  // [warp][2][kSegT]
    const float* ckp = reinterpret_cast<const float*>(smem + Y::OFF_CK);  // [seg][ch][16]
    const int ntiles = (a.seqlen + kTL - 1) / kTL;

    fetch_tile<T, VEC>(a, smem, ntiles - 1, row0, cvalid, bcrow0, tid);
    for (int tile = ntiles - 1; tile >= 0; --tile) {
        const int t0 = tile * kTL, tn = min(kTL, a.seqlen - t0);
        cp_async_wait_all();
        __syncthreads();  // every thread's copies of this tile have landed
        prep_tile<T>(a, smem, bias_p, tid % kCH < cvalid, tn, Z, tid);
        __syncthreads();  // per-step terms ready; the raw area is free
        if (tile > 0) fetch_tile<T, VEC>(a, smem, tile - 1, row0, cvalid, bcrow0, tid);
        const int nseg = (tn + kSeg - 1) / kSeg;
#pragma unroll 1
        for (int s = nseg - 1; s >= 0; --s) {
            const int ts0 = s * kSeg;
            const float4 hv = *reinterpret_cast<const float4*>(ckp + (s * kCH + cl) * kN + n0);
            const float hs[4] = {hv.x, hv.y, hv.z, hv.w};
            // ---- recompute the segment's states from its checkpoint
            float H[kSeg][4], ys[kSeg];
            {
                float h[4] = {hs[0], hs[1], hs[2], hs[3]};
#pragma unroll
                for (int i = 0; i < kSeg; ++i) {
                    const int t = ts0 + i;
                    const float4 ra = recA[t];
                    const float4 bq = *reinterpret_cast<const float4*>(Bt + t * kN + n0);
                    h[0] = fmaf(ex2_approx(ra.x * A2[0]), h[0], ra.y * bq.x);
                    h[1] = fmaf(ex2_approx(ra.x * A2[1]), h[1], ra.y * bq.y);
                    h[2] = fmaf(ex2_approx(ra.x * A2[2]), h[2], ra.y * bq.z);
                    h[3] = fmaf(ex2_approx(ra.x * A2[3]), h[3], ra.y * bq.w);
#pragma unroll
                    for (int k = 0; k < 4; ++k) H[i][k] = h[k];
                    if constexpr (Z) {
                        const float4 cq = *reinterpret_cast<const float4*>(Ct + t * kN + n0);
                        ys[i] = fmaf(cq.w, h[3], fmaf(cq.z, h[2], fmaf(cq.y, h[1], cq.x * h[0])));
                    }
                }
            }
            // ---- the gate's derivative needs y0 = sum_n C h + D u: reduce-scatter
            // the 16 steps' partial sums over the channel's 4 lanes (lane ng ends
            // with steps 4 ng .. 4 ng + 3)
            if constexpr (Z) {
                const bool b1 = lane & 2, b0 = lane & 1;
                float w8[8], w4[4];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float send = b1 ? ys[i] : ys[i + 8];
                    const float keep = b1 ? ys[i + 8] : ys[i];
                    w8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = b0 ? w8[i] : w8[i + 4];
                    const float keep = b0 ? w8[i + 4] : w8[i];
                    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = ts0 + 4 * ng + q;
                    if (valid && t < tn) {
                        const float y0 = fmaf(Dd, recA[t].w, w4[q]);
                        a.dz[drow * L + t0 + t] = recB[t].y * y0;
                    }
                }
            }
            // ---- the adjoint recurrence, last step first
            float pdu[4], pdl[4];
#pragma unroll
            for (int i = kSeg - 1; i >= 0; --i) {
                const int t = ts0 + i;
                const float4 ra = recA[t];  // dl, dl u, dy0, u
                const float4 bq = *reinterpret_cast<const float4*>(Bt + t * kN + n0);
                const float4 cq = *reinterpret_cast<const float4*>(Ct + t * kN + n0);
                const float bb[4] = {bq.x, bq.y, bq.z, bq.w}, cc[4] = {cq.x, cq.y, cq.z, cq.w};
                float v[8];
                float sdu = 0.0f, sdl = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float av = ex2_approx(ra.x * A2[k]);
                    const float hp = i > 0 ? H[i - 1][k] : hs[k];
                    lam[k] = fmaf(ra.z, cc[k], lam[k]);
                    v[4 + k] = ra.z * H[i][k];  // dC
                    v[k] = lam[k] * ra.y;       // dB
                    const float t1 = lam[k] * hp * av;
                    dA[k] = fmaf(t1, ra.x, dA[k]);
                    const float lb = lam[k] * bb[k];
                    sdl = fmaf(t1, An[k], fmaf(lb, ra.w, sdl));
                    sdu = fmaf(lb, ra.x, sdu);
                    lam[k] *= av;
                }
                pdu[i & 3] = sdu;
                pdl[i & 3] = sdl;
                // dB, dC of step t summed over the warp's 8 channels
                {
                    const float r = reduce_scatter8_channels(v, lane);
                    const int type = (lane >> 4) & 1, kk = (lane >> 2) & 3;
                    segw[(warp * 2 + type) * kSegT + i * kN + n0 + kk] = r;
                }
                if ((i & 3) == 0) {
                    // (du, d dl) of steps i .. i + 3 over the channel's 4 lanes:
                    // lane ng ends with step i + ng
                    const bool b1 = lane & 2, b0 = lane & 1;
                    float w4[4], w2[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // values of steps (j, j + 2)
                        const float su = b1 ? pdu[j] : pdu[j + 2];
                        const float ku = b1 ? pdu[j + 2] : pdu[j];
                        const float sl = b1 ? pdl[j] : pdl[j + 2];
                        const float kl = b1 ? pdl[j + 2] : pdl[j];
                        w4[2 * j] = ku + __shfl_xor_sync(0xffffffffu, su, 2);
                        w4[2 * j + 1] = kl + __shfl_xor_sync(0xffffffffu, sl, 2);
                    }
                    // w4 = (du, dl) of steps (2 b1, 2 b1 + 1)
                    {
                        const float su = b0 ? w4[0] : w4[2];
                        const float ku = b0 ? w4[2] : w4[0];
                        const float sl = b0 ? w4[1] : w4[3];
                        const float kl = b0 ? w4[3] : w4[1];
                        w2[0] = ku + __shfl_xor_sync(0xffffffffu, su, 1);
                        w2[1] = kl + __shfl_xor_sync(0xffffffffu, sl, 1);
                    }
                    const int to = ts0 + i + ng;  // this lane's step
                    if (valid && to < tn) {
                        const float4 ro = recA[to];
                        const float dd = w2[1] * recB[to].x;
                        a.du[drow * L + t0 + to] = fmaf(ro.z, Dd, w2[0]);
                        a.ddelta[drow * L + t0 + to] = dd;
                        accD = fmaf(ro.z, ro.w, accD);
                        accBias += dd;
                    }
                }
            }
            // the four warps' sums, added in warp order (the same bits on every run)
            __syncthreads();
            for (int e = tid; e < 2 * kSeg * kN; e += kThreads) {
                const int type = e / (kSeg * kN), rem = e % (kSeg * kN);  // rem = i * 16 + n
                float acc = segw[(0 * 2 + type) * kSegT + rem];
#pragma unroll
                for (int w = 1; w < 4; ++w) acc += segw[(w * 2 + type) * kSegT + rem];
                sum[(type * kTL + ts0 + rem / kN) * kSumT + rem % kN] = acc;
            }
            __syncthreads();
        }
        // this channel block's dB, dC of the tile: pBC [cb][b][g][type][n][t]
        {
            const long long base = (long long)cb * a.batch * a.ngroups * 2 * kN * L +
                                   (long long)bg * 2 * kN * L;
            for (int i = tid; i < 2 * kN * kTL; i += kThreads) {
                const int tn_i = i % kTL, rest = i / kTL;  // rest = type * 16 + n
                if (tn_i < tn)
                    a.pBC[base + rest * L + t0 + tn_i] =
                        sum[((rest >> 4) * kTL + tn_i) * kSumT + (rest & 15)];
            }
        }
    }

    // ---- per-channel sums: dA (this batch row), dD, dbias, and dh0
    if (valid) {
        *reinterpret_cast<float4*>(a.pA + drow * kN + n0) = make_float4(dA[0], dA[1], dA[2], dA[3]);
        if (a.dh0)
            *reinterpret_cast<float4*>(a.dh0 + drow * kN + n0) =
                make_float4(lam[0], lam[1], lam[2], lam[3]);
    }
    accD += __shfl_xor_sync(0xffffffffu, accD, 1);
    accD += __shfl_xor_sync(0xffffffffu, accD, 2);
    accBias += __shfl_xor_sync(0xffffffffu, accBias, 1);
    accBias += __shfl_xor_sync(0xffffffffu, accBias, 2);
    if (valid && ng == 0) {
        a.pD[drow] = accD;
        a.pbias[drow] = accBias;
    }
}

// dB, dC = sums of the channel blocks' partials; dA, dD, dbias = sums over the
// batch.  One output per thread, partials added in a fixed order.
__global__ void scan_bwd_reduce_kernel(const float* __restrict__ pBC, const float* __restrict__ pA,
                                       const float* __restrict__ pD,
                                       const float* __restrict__ pbias, float* __restrict__ dB,
                                       float* __restrict__ dC, float* __restrict__ dA,
                                       float* __restrict__ dD, float* __restrict__ dbias,
                                       int batch, int dim, int seqlen, int ngroups, int bpg) {
    const long long L = seqlen;
    const long long nbc = (long long)batch * ngroups * 2 * kN * L;  // one channel block's partial
    const long long total = nbc + (long long)dim * kN + 2LL * dim;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        if (i < nbc) {
            float s = 0.0f;
            for (int c = 0; c < bpg; ++c) s += pBC[c * nbc + i];
            // i = ((bg * 2 + type) * 16 + n) * L + t
            const long long t = i % L, rest = i / L;
            const long long n = rest % kN, type = (rest / kN) % 2, bgi = rest / (2 * kN);
            float* out = type ? dC : dB;
            out[(bgi * kN + n) * L + t] = s;
        } else if (i < nbc + (long long)dim * kN) {
            const long long j = i - nbc;  // d * 16 + n
            float s = 0.0f;
            for (int b = 0; b < batch; ++b) s += pA[(long long)b * dim * kN + j];
            dA[j] = s;
        } else {
            const long long j = i - nbc - (long long)dim * kN;  // [0, 2 dim)
            const bool is_bias = j >= dim;
            const long long dd = is_bias ? j - dim : j;
            float* out = is_bias ? dbias : dD;
            if (!out) continue;
            const float* src = is_bias ? pbias : pD;
            float s = 0.0f;
            for (int b = 0; b < batch; ++b) s += src[(long long)b * dim + dd];
            out[dd] = s;
        }
    }
}

template <typename T, bool VEC, bool Z>
ssm_status_t launch_bwd_one(const BwdArgs& a, unsigned grid, cudaStream_t s) {
    auto kern = scan_bwd_kernel<T, VEC, Z>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<T>::SMEM) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    kern<<<grid, kThreads, Lay<T>::SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T>
ssm_status_t launch_bwd(const BwdArgs& a, bool vec, bool z, unsigned grid, cudaStream_t s) {
    if (vec) return z ? launch_bwd_one<T, true, true>(a, grid, s)
                      : launch_bwd_one<T, true, false>(a, grid, s);
    return z ? launch_bwd_one<T, false, true>(a, grid, s) : launch_bwd_one<T, false, false>(a, grid, s);
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct BwdWs {
    size_t fwd, ckpt, pbc, pa, pd, pbias, total;
};

BwdWs bwd_workspace(int batch, int dim, int seqlen, int ngroups) {
    BwdWs w{};
    const size_t rows = (size_t)batch * dim;
    const size_t segs = ((size_t)seqlen + kSeg - 1) / kSeg;
    const size_t dpg = (size_t)dim / ngroups;
    const size_t bpg = (dpg + kCH - 1) / kCH;
    w.fwd = round256(ssm_internal::scan_forward_workspace_bytes(batch, dim, seqlen, ngroups));
    w.ckpt = round256(segs * rows * kN * 4);
    w.pbc = round256(bpg * (size_t)batch * ngroups * 2 * kN * (size_t)seqlen * 4);
    w.pa = round256(rows * kN * 4);
    w.pd = round256(rows * 4);
    w.pbias = round256(rows * 4);
    w.total = w.fwd + w.ckpt + w.pbc + w.pa + w.pd + w.pbias;
    return w;
}

}  // namespace

extern "C" size_t ssm_scan_bwd_workspace_bytes(int batch, int dim, int seqlen, int dstate,
                                               int ngroups) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate != kN || ngroups < 1 || dim % ngroups)
        return 0;
    return bwd_workspace(batch, dim, seqlen, ngroups).total;
}

extern "C" ssm_status_t ssm_scan_bwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* initial_state, const void* dy, const float* dfinal_state,
    const float* checkpoints, float* du,
    float* ddelta, float* dA, float* dB, float* dC, float* dD, float* dz, float* ddelta_bias,
    float* dinitial_state, int batch, int dim, int seqlen, int dstate, int ngroups,
    ssm_dtype_t in_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || dim < 0 || seqlen < 0 || ngroups < 1 || dstate < 1) return SSM_ERR_SHAPE;
    if (dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype)) return SSM_ERR_DTYPE;
    if (dstate != kN) return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * dim;
    if (rows > (size_t)INT32_MAX || (size_t)batch * ngroups * kN > (size_t)INT32_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (dim > 0 && !dA) return SSM_ERR_NULL;
    if (rows > 0 && seqlen > 0 &&
        (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dB || !dC))
        return SSM_ERR_NULL;
    if (rows > 0 && seqlen > 0 && z && !dz) return SSM_ERR_NULL;
    if (rows > 0 && seqlen > 0 && !workspace) return SSM_ERR_WORKSPACE;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, initial_state, dy, dfinal_state,
                          checkpoints, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                          dinitial_state, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;

    const size_t es = dtype_size(in_dtype);
    const size_t act = rows * (size_t)seqlen * es, act32 = rows * (size_t)seqlen * 4;
    const size_t bc = (size_t)batch * ngroups * kN * (size_t)seqlen * es;
    const size_t bc32 = (size_t)batch * ngroups * kN * (size_t)seqlen * 4;
    const size_t st = rows * kN * 4;
    struct R { const void* p; size_t n; };
    const R ins[] = {{u, act}, {delta, act}, {z, z ? act : 0}, {B, bc}, {C, bc},
                     {A, (size_t)dim * kN * 4}, {D, D ? (size_t)dim * 4 : 0},
                     {delta_bias, delta_bias ? (size_t)dim * 4 : 0},
                     {initial_state, initial_state ? st : 0}, {dy, act},
                     {dfinal_state, dfinal_state ? st : 0},
                     {checkpoints, checkpoints ? ((size_t)seqlen + kSeg - 1) / kSeg * st : 0}};
    const R outs[] = {{du, act32}, {ddelta, act32}, {dz, z ? act32 : 0},
                      {dB, bc32}, {dC, bc32}, {dA, (size_t)dim * kN * 4},
                      {dD, dD ? (size_t)dim * 4 : 0},
                      {ddelta_bias, ddelta_bias ? (size_t)dim * 4 : 0},
                      {dinitial_state, dinitial_state ? st : 0}};
    constexpr int kOuts = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < kOuts; ++i) {
        for (const R& r : ins)
            if (overlaps(outs[i].p, outs[i].n, r.p, r.n)) return SSM_ERR_ALIAS;
        for (int j = i + 1; j < kOuts; ++j)
            if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return SSM_ERR_ALIAS;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0 || seqlen == 0) {
        // No step: every parameter gradient is zero and dinitial_state = dfinal.
        auto zero = [&](void* p, size_t n) {
            return !p || n == 0 || cudaMemsetAsync(p, 0, n, s) == cudaSuccess;
        };
        bool ok = zero(dA, (size_t)dim * kN * 4) && zero(dD, (size_t)dim * 4) &&
                  zero(ddelta_bias, (size_t)dim * 4);
        if (ok && dinitial_state && st)
            ok = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, st,
                                                cudaMemcpyDeviceToDevice, s) == cudaSuccess
                              : zero(dinitial_state, st);
        return ok ? SSM_OK : SSM_ERR_CUDA;
    }

    const BwdWs w = bwd_workspace(batch, dim, seqlen, ngroups);
    if (workspace_bytes < w.total) return SSM_ERR_WORKSPACE;
    for (const R& r : ins)
        if (overlaps(workspace, w.total, r.p, r.n)) return SSM_ERR_ALIAS;
    for (const R& r : outs)
        if (overlaps(workspace, w.total, r.p, r.n)) return SSM_ERR_ALIAS;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    BwdArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.dy = dy; a.A = A; a.Dskip = D; a.bias = delta_bias;
    a.Bm = B; a.Cm = C;
    float* ckpt = reinterpret_cast<float*>(ws + w.fwd);
    a.ckpt = checkpoints ? checkpoints : ckpt;
    a.dfinal = dfinal_state;
    a.du = du; a.ddelta = ddelta; a.dz = z ? dz : nullptr; a.dh0 = dinitial_state;
    a.pBC = reinterpret_cast<float*>(ws + w.fwd + w.ckpt);
    a.pA = reinterpret_cast<float*>(ws + w.fwd + w.ckpt + w.pbc);
    a.pD = reinterpret_cast<float*>(ws + w.fwd + w.ckpt + w.pbc + w.pa);
    a.pbias = reinterpret_cast<float*>(ws + w.fwd + w.ckpt + w.pbc + w.pa + w.pd);
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.ngroups = ngroups;
    a.dpg = dim / ngroups; a.bpg = (a.dpg + kCH - 1) / kCH;
    a.softplus = delta_softplus ? 1 : 0;

    // 1. states entering every 16-step segment (unless the forward kept them)
    ssm_status_t rc = SSM_OK;
    if (!checkpoints) {
        rc = ssm_internal::scan_forward_checkpoints(u, delta, A, B, C, delta_bias, delta_softplus,
                                                    initial_state, ckpt, batch, dim, seqlen,
                                                    ngroups, in_dtype, workspace, s);
        if (rc != SSM_OK) return rc;
    } else if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) {
        return SSM_ERR_CUDA;  // a clean status word for ssm_last_device_status
    }

    // 2. the adjoint sweep, one CTA per (batch, group, channel block)
    const long long grid = (long long)batch * ngroups * a.bpg;
    if (grid > INT32_MAX) return SSM_ERR_UNSUPPORTED;
    // 16-byte copies need rows of whole 16-byte chunks (bases are checked above)
    const bool vec = ((size_t)seqlen * es) % 16 == 0;
    rc = in_dtype == SSM_BF16 ? launch_bwd<__nv_bfloat16>(a, vec, z != nullptr, (unsigned)grid, s)
                              : launch_bwd<float>(a, vec, z != nullptr, (unsigned)grid, s);
    if (rc != SSM_OK) return rc;

    // 3. sums of the partials
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)batch * ngroups * 2 * kN * seqlen + (long long)dim * kN +
                            2LL * dim;
    const long long want = (total + 255) / 256;
    const unsigned rgrid = (unsigned)std::max<long long>(1, std::min<long long>(want, 8LL * sms));
    scan_bwd_reduce_kernel<<<rgrid, 256, 0, s>>>(a.pBC, a.pA, a.pD, a.pbias, dB, dC, dA, dD,
                                                ddelta_bias, batch, dim, seqlen, ngroups, a.bpg);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
