// scan_seg.cu -- sequence-parallel selective scan (ssm_scan_fwd's path for
// problems with too few channels to fill the GPU one channel per lane group).
//
// What it computes is ssm_scan_fwd's recurrence ("We brought Mamba to
// Trainium -- and mapped where custom kernels actually help", section "Mamba:
// bringing an unsupported model to the chip, and writing its missing kernel";
// discretisation and epilogue from "Mamba-3 NKI Kernels for AWS Neuron",
// section "How it works", Phases 0 and 5).  How it splits the sequence rests
// on the associativity of the recurrence, the point of the first page's
// section "We built the parallel scan -- and it taught us something sharper":
// a span of steps acts on the state as h -> P h + q, with P = prod a (per
// state) and q the state the span reaches from zero, and two spans compose by
//     (P1, q1) o (P2, q2) = (P1 P2, P2 q1 + q2)      (first span 1, then 2).
//
// Layout of the work:
//  * A lane owns one (channel, time segment of SEGL steps) and all 16 states
//    of that channel in registers, so the read-out sum over states needs no
//    cross-lane reduction.  TS consecutive lanes hold the TS consecutive
//    segments of one channel: a warp covers 32 / TS channels over a chunk of
//    TS * SEGL = 128 steps.  A CTA (4 warps) covers 4 * 32 / TS channels of one
//    (batch, group) over one chunk.
//  * Pass A: each lane scans its segment from the zero state, keeping q (its
//    end state) and P = 2^(A log2e * sum dl).
//  * In-warp combine: an inclusive scan of the (P, q) pairs over the TS lanes
//    of a channel with __shfl_up_sync, log2(TS) levels; then shifted by one
//    lane to get the exclusive prefix (the map from the chunk's entry state to
//    the state entering the lane's segment).
//  * Across CTAs (chunks of one channel block), a decoupled look-back: each
//    chunk publishes its aggregate (P, q) as soon as pass A and the combine are
//    done, then looks back over its predecessors' flags, composing aggregates
//    until it reaches a published inclusive state; it then publishes its own
//    inclusive state (before its pass C, so successors need not wait for it).
//    Chunks are handed out in order by a ticket, so a predecessor is always
//    running or done, and every wait is bounded (SSM_ERR_TIMEOUT).
//  * Pass C: each lane replays its segment from its entry state, forming
//    y = (sum_n C h + D u) * silu(z), and the last chunk's last lane writes the
//    final state.
// Every element costs two exps instead of one (passes A and C): the price of
// the sequence parallelism, which pays when the channels alone leave most of
// the GPU idle.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "scan_internal.h"

namespace {

using namespace ssm;

constexpr int kN = 16;        // dstate
constexpr int kChunk = 128;   // steps per CTA chunk (TS * SEGL)
constexpr int kWarps = 4;     // warps per CTA
constexpr int kThreads = kWarps * 32;

enum : uint32_t { kFlagNone = 0, kFlagAgg = 1, kFlagInc = 2 };

struct alignas(16) SegHeader {
    uint32_t ticket;
    uint32_t status;
    uint32_t pad[62];
};
static_assert(sizeof(SegHeader) == 256, "workspace header is 256 bytes");

struct SegArgs {
    const void* u;
    const void* delta;
    const void* z;
    const float* A;
    const float* Dskip;
    const float* bias;
    const float* h0;
    void* y;
    float* final_state;
    const void* Bm;
    const void* Cm;
    uint32_t* ticket;  // NULL when there is one chunk
    uint32_t* status;
    uint32_t* flags;   // [nchunks][nblocks]
    float* agg;        // [nchunks][batch * dim][2][16]  (P, q)
    float* inc;        // [nchunks][batch * dim][16]     inclusive state
    int batch, dim, seqlen, ngroups;
    int dpg, bpg, nblocks, nchunks;
    int softplus;
    uint32_t flag_spin_limit;
    int keep_status;         // the status word holds an earlier call's result to keep
    int drop_first_publish;  // test hook: chunk 0 never publishes its inclusive state
};

// K consecutive values of row `row` from step t0 (t0 % 4 == 0, K % 4 == 0),
// as fp32; steps at or past L read as 0.  16- or 8-byte loads when the row
// length is a multiple of 4 steps (base pointers are 16-byte aligned), else
// element loads.
template <typename T, int K>
__device__ __forceinline__ void load_steps(const T* base, long long row, int t0, int L, bool vec,
                                           float* v) {
    const T* p = base + row * (long long)L + t0;
    if (vec && t0 + K <= L) {
#pragma unroll
        for (int k = 0; k < K; k += 4) {
            if constexpr (sizeof(T) == 2) {
                const uint2 w = __ldg(reinterpret_cast<const uint2*>(p + k));
                v[k + 0] = bf16lo(w.x); v[k + 1] = bf16hi(w.x);
                v[k + 2] = bf16lo(w.y); v[k + 3] = bf16hi(w.y);
            } else {
                const float4 w = __ldg(reinterpret_cast<const float4*>(p + k));
                v[k + 0] = w.x; v[k + 1] = w.y; v[k + 2] = w.z; v[k + 3] = w.w;
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] = (t0 + k < L) ? to_f32(p[k]) : 0.0f;
    }
}

// 4 consecutive values of row `row` from step t0 (t0 % 4 == 0); steps at or
// past L are not written.
template <typename T>
__device__ __forceinline__ void store4(T* base, long long row, int t0, int L, bool vec,
                                       const float* v) {
    T* p = base + row * (long long)L + t0;
    if (vec && t0 + 4 <= L) {
        if constexpr (sizeof(T) == 2) {
            __nv_bfloat162 lo, hi;
            lo.x = __float2bfloat16_rn(v[0]); lo.y = __float2bfloat16_rn(v[1]);
            hi.x = __float2bfloat16_rn(v[2]); hi.y = __float2bfloat16_rn(v[3]);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t*>(&lo);
            w.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(p) = w;
        } else {
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (t0 + k < L) p[k] = from_f32<T>(v[k]);
    }
}

// Shared memory of one CTA: B and C of the chunk as fp32 rows of 144 bytes
// per step (B[16], C[16], 16 bytes of padding, so that writes of one state
// for consecutive steps spread over the banks); segment s starts 16*s bytes
// further on than its steps alone would put it, so that the TS lanes of a
// channel (different segments, same step offset) read different bank groups.
template <int TS, int SEGL>
struct SegSmem {
    static constexpr int kRow = 144;
    static constexpr int kSegBytes = SEGL * kRow + 16;
    static constexpr int kBC = TS * kSegBytes;
    static constexpr int kBytes = kBC + 64;  // + look-back result
    __device__ static constexpr int off(int t) { return (t / SEGL) * kSegBytes + (t % SEGL) * kRow; }
};

template <typename Tin, typename Tout, int TS>
__global__ void __launch_bounds__(kThreads, 4)
    scan_seg_kernel(const SegArgs a) {
    constexpr int SEGL = kChunk / TS;
    constexpr int CHW = 32 / TS;       // channels per warp
    constexpr int CH = kWarps * CHW;   // channels per CTA
    using SM = SegSmem<TS, SEGL>;
    static_assert(SEGL % 4 == 0, "segments are whole groups of 4 steps");

    __shared__ __align__(16) uint8_t smem[SM::kBytes];
    __shared__ int s_ticket;
    int* s_look = reinterpret_cast<int*>(smem + SM::kBC);  // [0] newest inclusive, [1] ok

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int seg = lane % TS;        // time segment within the chunk
    const int cw = lane / TS;         // channel within the warp

    int ticket = blockIdx.x;
    if (a.ticket) {
        if (tid == 0) s_ticket = static_cast<int>(atomicAdd(a.ticket, 1u));
        __syncthreads();
        ticket = s_ticket;
    } else if (blockIdx.x == 0 && tid == 0 && !a.keep_status) {
        *a.status = 0;  // one chunk: no waits, so nothing else writes the status
    }
    const int chunk = ticket / a.nblocks;
    const int blk = ticket % a.nblocks;
    const int cb = blk % a.bpg;
    const int bg = blk / a.bpg;  // b * ngroups + g
    const int g = bg % a.ngroups;
    const int b = bg / a.ngroups;
    const int c0 = chunk * kChunk;  // first step of the chunk
    const bool vec = (a.seqlen & 3) == 0;

    const int cl = warp * CHW + cw;  // channel within the CTA
    const bool valid = cb * CH + cl < a.dpg;
    const int d = g * a.dpg + cb * CH + cl;
    const long long row = valid ? (long long)b * a.dim + d : 0;
    const int t0 = c0 + seg * SEGL;
    const bool has_z = a.z != nullptr;

    // ---- the lane's delta, u and z, loaded first so that their latency
    // overlaps the staging of B and C (one round trip for all of them)
    float dl[SEGL], uv[SEGL], zv[SEGL];
#pragma unroll
    for (int k0 = 0; k0 < SEGL; k0 += 4) {
        load_steps<Tin, 4>(reinterpret_cast<const Tin*>(a.delta), row, t0 + k0, a.seqlen, vec,
                           dl + k0);
        load_steps<Tin, 4>(reinterpret_cast<const Tin*>(a.u), row, t0 + k0, a.seqlen, vec,
                           uv + k0);
        if (has_z)
            load_steps<Tin, 4>(reinterpret_cast<const Tin*>(a.z), row, t0 + k0, a.seqlen, vec,
                               zv + k0);
    }

    // ---- B and C of the chunk into shared memory as fp32 [t][n]: thread
    // (state n, 4-step group) reads 4 steps of B and of C, every load of the
    // thread issued before its first store (one round trip, not four)
    {
        constexpr int kIters = kN * (kChunk / 4) / kThreads;
        static_assert(kN * (kChunk / 4) % kThreads == 0, "whole staging rounds");
        float vb[kIters][4], vc[kIters][4];
#pragma unroll
        for (int r = 0; r < kIters; ++r) {
            const int i = tid + r * kThreads;
            const int n = i % kN, t = (i / kN) * 4;
            load_steps<Tin, 4>(reinterpret_cast<const Tin*>(a.Bm), (long long)bg * kN + n, c0 + t,
                               a.seqlen, vec, vb[r]);
            load_steps<Tin, 4>(reinterpret_cast<const Tin*>(a.Cm), (long long)bg * kN + n, c0 + t,
                               a.seqlen, vec, vc[r]);
        }
#pragma unroll
        for (int r = 0; r < kIters; ++r) {
            const int i = tid + r * kThreads;
            const int n = i % kN, t = (i / kN) * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float* row = reinterpret_cast<float*>(smem + SM::off(t + k));
                row[n] = vb[r][k];
                row[kN + n] = vc[r][k];
            }
        }
    }
    __syncthreads();

    const uint8_t* segBC = smem + seg * SM::kSegBytes;

    // ---- prep: dl = softplus(delta + bias) (or delta + bias) and dl * u;
    // steps past the sequence get dl = 0, the identity step
    float dlu[SEGL];
    {
        const float bias = (a.bias && valid) ? a.bias[d] : 0.0f;
#pragma unroll
        for (int k = 0; k < SEGL; ++k) {
            const float x = dl[k] + bias;
            float v = a.softplus ? softplus_f(x) : x;
            if (t0 + k >= a.seqlen || !valid) v = 0.0f;
            dl[k] = v;
            dlu[k] = v * uv[k];
        }
    }

    // ---- pass A: the segment from the zero state; P = 2^(A log2e sum dl)
    float q[kN], P[kN];
    {
        float A2[kN];
#pragma unroll
        for (int n = 0; n < kN; ++n) A2[n] = valid ? a.A[(long long)d * kN + n] * kLog2e : 0.0f;
        float dsum = 0.0f;
#pragma unroll
        for (int n = 0; n < kN; ++n) q[n] = 0.0f;
#pragma unroll
        for (int k = 0; k < SEGL; ++k) {
            const float4* bc = reinterpret_cast<const float4*>(segBC + k * SM::kRow);
            dsum += dl[k];
#pragma unroll
            for (int j = 0; j < kN / 4; ++j) {
                const float4 bv = bc[j];
                q[4 * j + 0] = fmaf(ex2_approx(dl[k] * A2[4 * j + 0]), q[4 * j + 0], dlu[k] * bv.x);
                q[4 * j + 1] = fmaf(ex2_approx(dl[k] * A2[4 * j + 1]), q[4 * j + 1], dlu[k] * bv.y);
                q[4 * j + 2] = fmaf(ex2_approx(dl[k] * A2[4 * j + 2]), q[4 * j + 2], dlu[k] * bv.z);
                q[4 * j + 3] = fmaf(ex2_approx(dl[k] * A2[4 * j + 3]), q[4 * j + 3], dlu[k] * bv.w);
            }
        }
#pragma unroll
        for (int n = 0; n < kN; ++n) P[n] = ex2_approx(A2[n] * dsum);
    }

    // ---- in-warp combine: inclusive scan of (P, q) over the channel's TS
    // lanes: (earlier) o (this) = (P' P, P q' + q)
#pragma unroll
    for (int o = 1; o < TS; o <<= 1) {
#pragma unroll
        for (int n = 0; n < kN; ++n) {
            const float Pp = __shfl_up_sync(0xffffffffu, P[n], o, TS);
            const float qp = __shfl_up_sync(0xffffffffu, q[n], o, TS);
            if (seg >= o) {
                q[n] = fmaf(P[n], qp, q[n]);
                P[n] *= Pp;
            }
        }
    }
    // the channel's last lane now holds the chunk's aggregate

    // ---- the chunk's entry state hc (every lane of the channel)
    float hc[kN];
    if (chunk == 0) {
        if (a.h0 && valid) {
            const float4* src = reinterpret_cast<const float4*>(a.h0 + row * kN);
#pragma unroll
            for (int j = 0; j < kN / 4; ++j) {
                const float4 v = src[j];
                hc[4 * j] = v.x; hc[4 * j + 1] = v.y; hc[4 * j + 2] = v.z; hc[4 * j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int n = 0; n < kN; ++n) hc[n] = 0.0f;
        }
    } else {
        const size_t stride = (size_t)a.batch * a.dim;
        // publish the aggregate, then look back
        if (seg == TS - 1 && valid) {
            float4* dst = reinterpret_cast<float4*>(a.agg + ((size_t)chunk * stride + row) * 2 * kN);
#pragma unroll
            for (int j = 0; j < kN / 4; ++j) {
                __stcg(dst + j, make_float4(P[4 * j], P[4 * j + 1], P[4 * j + 2], P[4 * j + 3]));
                __stcg(dst + kN / 4 + j,
                       make_float4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]));
            }
        }
        // the barrier orders every thread's stores before thread 0's release
        // (release is cumulative over what the barrier made visible to it)
        __syncthreads();
        if (tid == 0) st_release_gpu(a.flags + (size_t)chunk * a.nblocks + blk, kFlagAgg);

        // warp 0 finds the newest predecessor with a published inclusive
        // state such that every chunk after it has published its aggregate;
        // lane i examines chunk j_hi - i, 32 chunks per round
        if (warp == 0) {
            int j_hi = chunk - 1;
            int j_inc = -1;
            bool ok = true;
            uint32_t polls = 0, ns = 32;
            while (true) {
                const int j = j_hi - lane;
                uint32_t f = kFlagNone;
                if (j >= 0) f = ld_acquire_gpu(a.flags + (size_t)j * a.nblocks + blk);
                const uint32_t inc_mask = __ballot_sync(0xffffffffu, f == kFlagInc);
                const uint32_t none_mask = __ballot_sync(0xffffffffu, f == kFlagNone);
                const int first_inc = inc_mask ? __ffs(inc_mask) - 1 : 32;
                const uint32_t below = first_inc >= 32 ? 0xffffffffu : ((1u << first_inc) - 1u);
                if ((none_mask & below) == 0) {
                    if (first_inc < 32) { j_inc = j_hi - first_inc; break; }
                    j_hi -= 32;  // 32 aggregates and no inclusive state: further back
                    continue;
                }
                if (++polls >= a.flag_spin_limit) { ok = false; break; }
                __nanosleep(ns);
                ns = ns < 256 ? ns * 2 : 256;
            }
            if (lane == 0) {
                s_look[0] = j_inc;
                s_look[1] = ok ? 1 : 0;
                if (!ok) record_status(a.status, SSM_ERR_TIMEOUT);
            }
        }
        __syncthreads();
        const int j_inc = s_look[0];
        const bool ok = s_look[1] != 0;
#pragma unroll
        for (int n = 0; n < kN; ++n) hc[n] = 0.0f;
        // warp 0 read every flag it relied on with acquire; the barrier above
        // orders this thread's reads after those
        if (ok && valid) {
            const float4* src =
                reinterpret_cast<const float4*>(a.inc + ((size_t)j_inc * stride + row) * kN);
#pragma unroll
            for (int j = 0; j < kN / 4; ++j) {
                const float4 v = __ldcg(src + j);
                hc[4 * j] = v.x; hc[4 * j + 1] = v.y; hc[4 * j + 2] = v.z; hc[4 * j + 3] = v.w;
            }
            // compose the aggregates of chunks j_inc + 1 .. chunk - 1 in order
            for (int j = j_inc + 1; j < chunk; ++j) {
                const float4* ag =
                    reinterpret_cast<const float4*>(a.agg + ((size_t)j * stride + row) * 2 * kN);
#pragma unroll
                for (int i = 0; i < kN / 4; ++i) {
                    const float4 pv = __ldcg(ag + i);
                    const float4 qv = __ldcg(ag + kN / 4 + i);
                    hc[4 * i + 0] = fmaf(pv.x, hc[4 * i + 0], qv.x);
                    hc[4 * i + 1] = fmaf(pv.y, hc[4 * i + 1], qv.y);
                    hc[4 * i + 2] = fmaf(pv.z, hc[4 * i + 2], qv.z);
                    hc[4 * i + 3] = fmaf(pv.w, hc[4 * i + 3], qv.w);
                }
            }
        }
    }

    // ---- each lane's end state from the chunk's entry state; the last
    // lane's is the chunk's inclusive state, published for the successors
    float h[kN];
#pragma unroll
    for (int n = 0; n < kN; ++n) h[n] = fmaf(P[n], hc[n], q[n]);
    // final state: the last lane of the last chunk, the same composition a
    // successor chunk would take as its entry state, so that a sequence
    // scanned in pieces (each resumed from the last one's final state, cut at
    // multiples of 128 steps) gives the bits of the whole scan
    if (chunk == a.nchunks - 1 && seg == TS - 1 && valid && a.final_state) {
        float4* dst = reinterpret_cast<float4*>(a.final_state + row * kN);
#pragma unroll
        for (int j = 0; j < kN / 4; ++j)
            dst[j] = make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
    }
    if (a.ticket && chunk < a.nchunks - 1) {
        if (seg == TS - 1 && valid) {
            float4* dst = reinterpret_cast<float4*>(
                a.inc + ((size_t)chunk * a.batch * a.dim + (size_t)row) * kN);
#pragma unroll
            for (int j = 0; j < kN / 4; ++j)
                __stcg(dst + j, make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]));
        }
        __syncthreads();
        if (tid == 0 && !(a.drop_first_publish && chunk == 0))
            st_release_gpu(a.flags + (size_t)chunk * a.nblocks + blk, kFlagInc);
    }
    // the state entering each lane's segment: its left neighbour's end state
#pragma unroll
    for (int n = 0; n < kN; ++n) {
        const float e = __shfl_up_sync(0xffffffffu, h[n], 1, TS);
        h[n] = seg ? e : hc[n];
    }

    // ---- pass C: replay the segment from its entry state, with the read-out
    {
        float A2[kN];
#pragma unroll
        for (int n = 0; n < kN; ++n) A2[n] = valid ? a.A[(long long)d * kN + n] * kLog2e : 0.0f;
        const float Dd = (a.Dskip && valid) ? a.Dskip[d] : 0.0f;
#pragma unroll
        for (int k0 = 0; k0 < SEGL; k0 += 4) {
            float yv[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = k0 + kk;
                const float4* bc = reinterpret_cast<const float4*>(segBC + k * SM::kRow);
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < kN / 4; ++j) {
                    const float4 bv = bc[j];
                    const float4 cv = bc[kN / 4 + j];
                    h[4 * j + 0] =
                        fmaf(ex2_approx(dl[k] * A2[4 * j + 0]), h[4 * j + 0], dlu[k] * bv.x);
                    h[4 * j + 1] =
                        fmaf(ex2_approx(dl[k] * A2[4 * j + 1]), h[4 * j + 1], dlu[k] * bv.y);
                    h[4 * j + 2] =
                        fmaf(ex2_approx(dl[k] * A2[4 * j + 2]), h[4 * j + 2], dlu[k] * bv.z);
                    h[4 * j + 3] =
                        fmaf(ex2_approx(dl[k] * A2[4 * j + 3]), h[4 * j + 3], dlu[k] * bv.w);
                    acc = fmaf(cv.x, h[4 * j + 0], acc);
                    acc = fmaf(cv.y, h[4 * j + 1], acc);
                    acc = fmaf(cv.z, h[4 * j + 2], acc);
                    acc = fmaf(cv.w, h[4 * j + 3], acc);
                }
                const float gate = has_z ? silu_f(zv[k]) : 1.0f;
                yv[kk] = fmaf(Dd, uv[k], acc) * gate;
            }
            if (valid)
                store4<Tout>(reinterpret_cast<Tout*>(a.y), row, t0 + k0, a.seqlen, vec, yv);
        }
    }

}

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

int sm_count() {
    static std::mutex m;
    static int cached_dev = -1, sms = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(m);
    if (dev != cached_dev) {
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
        cached_dev = dev;
    }
    return sms;
}

std::atomic<int> g_seg_ts{0};  // test hook: forced segments per chunk (0: planned)

int channels_per_cta(int ts) { return kWarps * 32 / ts; }

}  // namespace

namespace ssm_internal {

bool scan_seg_eligible(long long batch, long long dim) {
    return batch * dim <= kScanSegMaxChannels;
}

size_t scan_seg_workspace_bytes(int batch, int dim, int seqlen, int ngroups) {
    const long long rows = (long long)batch * dim;
    const long long nchunks = (seqlen + kChunk - 1) / kChunk;
    if (nchunks <= 1) return sizeof(SegHeader);
    // the most channel blocks any plan makes: the smallest CTA (TS = 32)
    const long long dpg = dim / ngroups;
    const long long max_blocks = (long long)batch * ngroups * ((dpg + channels_per_cta(32) - 1) /
                                                               channels_per_cta(32));
    size_t bytes = sizeof(SegHeader);
    bytes += r256(sizeof(uint32_t) * (size_t)nchunks * (size_t)max_blocks);
    bytes += r256((size_t)nchunks * rows * 2 * kN * sizeof(float));
    bytes += r256((size_t)nchunks * rows * kN * sizeof(float));
    return bytes;
}

int scan_seg_plan_ts(long long batch, long long dim, int seqlen) {
    const int forced = g_seg_ts.load(std::memory_order_relaxed);
    if (forced == 8 || forced == 16 || forced == 32) return forced;
    // the longest segments whose warps still give every SM sub-partition
    // about two to work on
    const long long nchunks = (seqlen + kChunk - 1) / kChunk;
    const long long want = 2LL * 4 * sm_count();
    for (int ts : {8, 16}) {
        const long long warps = batch * dim * ts / 32 * nchunks;
        if (warps >= want) return ts;
    }
    return 32;
}

template <typename Tin, typename Tout, int TS>
static ssm_status_t seg_launch(SegArgs a, cudaStream_t stream) {
    const int ch = channels_per_cta(TS);
    a.bpg = (a.dpg + ch - 1) / ch;
    a.nblocks = a.batch * a.ngroups * a.bpg;
    const unsigned grid = (unsigned)a.nblocks * (unsigned)a.nchunks;
    scan_seg_kernel<Tin, Tout, TS><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename Tin, typename Tout>
static ssm_status_t seg_dispatch(SegArgs& a, int ts, cudaStream_t stream) {
    switch (ts) {
        case 8: return seg_launch<Tin, Tout, 8>(a, stream);
        case 16: return seg_launch<Tin, Tout, 16>(a, stream);
        default: return seg_launch<Tin, Tout, 32>(a, stream);
    }
}

ssm_status_t scan_seg_forward(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int delta_softplus,
                              const float* initial_state, void* y, float* final_state, int batch,
                              int dim, int seqlen, int ngroups, ssm_dtype_t in_dtype,
                              ssm_dtype_t out_dtype, void* workspace, uint32_t spin_limit,
                              int drop_first_publish, int ts, bool keep_status,
                              cudaStream_t stream) {
    SegArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.A = A; a.Dskip = D; a.bias = delta_bias;
    a.h0 = initial_state; a.y = y; a.final_state = final_state; a.Bm = B; a.Cm = C;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.ngroups = ngroups;
    a.dpg = dim / ngroups; a.softplus = delta_softplus ? 1 : 0;
    a.nchunks = (seqlen + kChunk - 1) / kChunk;
    a.flag_spin_limit = spin_limit;
    a.drop_first_publish = drop_first_publish;
    a.keep_status = keep_status ? 1 : 0;
    if (ts != 8 && ts != 16 && ts != 32) ts = scan_seg_plan_ts(batch, dim, seqlen);

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SegHeader* hdr = reinterpret_cast<SegHeader*>(ws);
    a.status = &hdr->status;
    if (a.nchunks > 1) {
        const int ch = channels_per_cta(ts);
        const size_t nblocks = (size_t)batch * ngroups * ((a.dpg + ch - 1) / ch);
        const size_t rows = (size_t)batch * dim;
        a.ticket = &hdr->ticket;
        a.flags = reinterpret_cast<uint32_t*>(ws + sizeof(SegHeader));
        const size_t flag_bytes = r256(sizeof(uint32_t) * (size_t)a.nchunks * nblocks);
        a.agg = reinterpret_cast<float*>(ws + sizeof(SegHeader) + flag_bytes);
        a.inc = a.agg + r256((size_t)a.nchunks * rows * 2 * kN * sizeof(float)) / sizeof(float);
        // the ticket, the status word (unless an earlier call's status is
        // being accumulated) and the flags start at zero
        if (keep_status) {
            if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream) != cudaSuccess ||
                cudaMemsetAsync(ws + 2 * sizeof(uint32_t), 0,
                                sizeof(SegHeader) - 2 * sizeof(uint32_t) + flag_bytes,
                                stream) != cudaSuccess)
                return SSM_ERR_CUDA;
        } else if (cudaMemsetAsync(ws, 0, sizeof(SegHeader) + flag_bytes, stream) !=
                   cudaSuccess) {
            return SSM_ERR_CUDA;
        }
    }
    // one chunk: no carry between CTAs and no waits; the kernel clears the
    // status word itself, so nothing is enqueued before it
    if (in_dtype == SSM_BF16)
        return out_dtype == SSM_BF16 ? seg_dispatch<__nv_bfloat16, __nv_bfloat16>(a, ts, stream)
                                     : seg_dispatch<__nv_bfloat16, float>(a, ts, stream);
    return out_dtype == SSM_BF16 ? seg_dispatch<float, __nv_bfloat16>(a, ts, stream)
                                 : seg_dispatch<float, float>(a, ts, stream);
}

void scan_seg_debug_force_ts(int ts) { g_seg_ts.store(ts, std::memory_order_relaxed); }

}  // namespace ssm_internal
