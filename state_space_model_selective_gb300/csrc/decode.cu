// decode.cu -- single-token decode step (ssm_decode_step) for GB300 / sm_103a.
//
// "Mamba-3 NKI Kernels for AWS Neuron", section "How it works" (decode via
// step(), Eq. 9; at lambda = 1: h = alpha h + dt B (x) x, y = C^T h) and
// section "Kernel details" (mamba3_siso_decode_state_kernel: state update
// and output contraction for all heads at once), plus Phase 5 (D skip, silu
// gate).
//
// The step is one streaming read-modify-write of the fp32 state
// (batch, nheads, headdim, dstate), so it is bound by HBM bandwidth.
//  * dstate 128 (decode_bulk_kernel): the state streams through shared
//    memory in tiles of up to 64 rows (32 KB, contiguous per (b, h)) by bulk
//    asynchronous copies -- one load and one store per tile, issued by a
//    producer warp, two tiles in flight per CTA, persistent CTAs -- and four
//    compute warps update each tile in place (lane = 4 consecutive states).
//  * other dstate (decode_kernel): each (b, h, p) row of dstate floats is
//    owned by dstate/16 lanes holding 16 consecutive states each (16-byte
//    loads with evict-first cache hints, two rows' loads in flight per lane).
// In both, the C^T h contraction is an intra-warp shuffle reduction.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace {

using namespace ssm;

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16lo(w[i]);
            v[2 * i + 1] = bf16hi(w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p) + i);
            v[4 * i] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
        }
    }
}

// One CTA per (batch, head): alpha = exp(dt A) and the head's B and C vectors
// (in shared memory, fp32) are loaded once and reused for every headdim row.
// A row of dstate floats is split over LPR = dstate / 16 lanes (16 states,
// four 16-byte loads each); the CTA's 256 threads cover 256 / LPR rows at a
// time, and each thread handles up to RPT rows with all their loads issued
// before any arithmetic.
// Mamba-3 SISO inputs of a decode step (M3 kernels only): lambda (batch,
// nheads) fp32 and the previous token's B (batch, ngroups, dstate) and x
// (batch, nheads, headdim).
template <typename T>
struct M3In {
    const float* lam;
    const T* prev_B;
    const T* prev_x;
};

template <typename T, int LPR, bool M3>
__global__ void __launch_bounds__(256, 3)
    decode_kernel(float* __restrict__ state, const T* __restrict__ x,
                  const float* __restrict__ dt, const float* __restrict__ A,
                  const T* __restrict__ Bm, const T* __restrict__ Cm,
                  const float* __restrict__ Dskip, const T* __restrict__ z, T* __restrict__ y,
                  int nheads, int headdim, int ngroups, M3In<T> m3) {
    constexpr int kDstate = LPR * 16;
    constexpr int kRowsPerPass = 256 / LPR;
    constexpr int RPT = 2;
    const int h = blockIdx.x % nheads;
    const long long b = blockIdx.x / nheads;
    const int g = h / (nheads / ngroups);
    const int part = threadIdx.x % LPR;
    const int r0 = threadIdx.x / LPR;

    __shared__ __align__(16) float sB[kDstate], sC[kDstate], sBp[M3 ? kDstate : 4];
    const long long row_base = (b * nheads + h) * (long long)headdim;
    const long long bc0 = (b * ngroups + g) * kDstate;
    const float4* sB4 = reinterpret_cast<const float4*>(sB + part * 16);
    const float4* sC4 = reinterpret_cast<const float4*>(sC + part * 16);
    const float4* sBp4 = reinterpret_cast<const float4*>(sBp + (M3 ? part * 16 : 0));
    // input weight of B (x) x (Mamba-2: dt; Mamba-3: gamma) and of the
    // previous token's term (Mamba-3: beta)
    float wx = 0.0f, wp = 0.0f, alpha = 0.0f, Dh = 0.0f;

    for (int p0 = 0; p0 < headdim; p0 += kRowsPerPass * RPT) {
        float s[RPT][16];
        float xv[RPT], zv[RPT], xpv[RPT];
        bool act[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = p0 + r * kRowsPerPass + r0;
            act[r] = p < headdim;
            const long long row = row_base + (act[r] ? p : 0);
            const float4* sp = reinterpret_cast<const float4*>(state + row * kDstate + part * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = act[r] ? __ldcs(sp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                s[r][4 * i] = v.x; s[r][4 * i + 1] = v.y; s[r][4 * i + 2] = v.z; s[r][4 * i + 3] = v.w;
            }
            xv[r] = act[r] ? to_f32(x[row]) : 0.0f;
            zv[r] = (act[r] && z) ? to_f32(z[row]) : 0.0f;
            xpv[r] = (M3 && act[r]) ? to_f32(m3.prev_x[row]) : 0.0f;
        }
        if (p0 == 0) {
            // B, C, alpha: after the first rows' loads are in flight
            for (int i = threadIdx.x; i < kDstate; i += 256) {
                sB[i] = to_f32(Bm[bc0 + i]);
                sC[i] = to_f32(Cm[bc0 + i]);
                if constexpr (M3) sBp[i] = to_f32(m3.prev_B[bc0 + i]);
            }
            const float dtv = dt[b * nheads + h];
            alpha = expf(dtv * A[h]);
            wx = dtv;
            if constexpr (M3) {
                wx = m3.lam[b * nheads + h] * dtv;  // gamma
                wp = (dtv - wx) * alpha;            // beta
            }
            Dh = Dskip ? Dskip[h] : 0.0f;
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = p0 + r * kRowsPerPass + r0;
            const long long row = row_base + (act[r] ? p : 0);
            const float dbx = wx * xv[r], pbx = wp * xpv[r];
            float acc = 0.0f;
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const float4 bq = sB4[i4], cq = sC4[i4];
                const float bb[4] = {bq.x, bq.y, bq.z, bq.w}, cc[4] = {cq.x, cq.y, cq.z, cq.w};
                float pp[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (M3) {
                    const float4 pq = sBp4[i4];
                    pp[0] = pq.x; pp[1] = pq.y; pp[2] = pq.z; pp[3] = pq.w;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float in = M3 ? fmaf(dbx, bb[k], pbx * pp[k]) : dbx * bb[k];
                    s[r][4 * i4 + k] = fmaf(alpha, s[r][4 * i4 + k], in);
                    acc = fmaf(cc[k], s[r][4 * i4 + k], acc);
                }
            }
            if (act[r]) {
                float4* sp = reinterpret_cast<float4*>(state + row * kDstate + part * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    __stcs(sp + i, make_float4(s[r][4 * i], s[r][4 * i + 1], s[r][4 * i + 2],
                                               s[r][4 * i + 3]));
            }
            // whole rows share a warp (LPR divides 32), so the row's lanes
            // reduce among themselves; every lane takes part in the shuffles
#pragma unroll
            for (int o = LPR / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (act[r] && part == 0) {
                float out = acc + Dh * xv[r];
                if (z) out *= silu_f(zv[r]);
                y[row] = from_f32<T>(out);
            }
        }
    }
}

template <typename T, int LPR, bool M3>
ssm_status_t launch(float* state, const void* x, const float* dt, const float* A, const void* B,
                    const void* C, const float* D, const void* z, void* y, long long rows,
                    int nheads, int headdim, int ngroups, M3In<T> m3, cudaStream_t s) {
    const long long grid = rows / headdim;  // batch * nheads
    decode_kernel<T, LPR, M3><<<(unsigned)grid, 256, 0, s>>>(
        state, static_cast<const T*>(x), dt, A, static_cast<const T*>(B),
        static_cast<const T*>(C), D, static_cast<const T*>(z), static_cast<T*>(y), nheads,
        headdim, ngroups, m3);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

// 4 consecutive values as fp32 (8-byte bf16 or 16-byte fp32 load)
template <typename T>
__device__ __forceinline__ void load4(const T* p, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    } else {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
}

// ------------------------------------------------------- dstate 128, bulk copies

constexpr int kBulkRows = 64;                    // rows per tile
constexpr int kBulkN = 128;                      // dstate
constexpr int kTileBytes = kBulkRows * kBulkN * 4;
constexpr int kBulkCompute = 128;                // 4 compute warps
constexpr int kBulkThreads = kBulkCompute + 32;  // + 1 producer warp
constexpr int kBulkSmem = 2 * kTileBytes + 64;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Producer loop of the bulk decode kernels (one thread): load the CTA's
// first two tiles, then for each tile i wait until the compute warps have
// updated it (empty), store it, and reuse the stage for tile i + 2 once the
// store has read it.  `tile(i, bh, p0, nr)` gives tile i's (b, h) pair, first
// row and row count.
template <typename TileFn>
__device__ __forceinline__ void bulk_producer(float* state, uint8_t* dsm, uint64_t* full,
                                              uint64_t* empty, long long my, int headdim,
                                              TileFn tile) {
    for (long long i = 0; i < 2 && i < my; ++i) {
        long long bh; int p0, nr;
        tile(i, bh, p0, nr);
        mbar_arrive_expect_tx(&full[i], (uint32_t)nr * kBulkN * 4);
        bulk_load(dsm + i * kTileBytes, state + (bh * headdim + p0) * kBulkN,
                  (uint32_t)nr * kBulkN * 4, &full[i]);
    }
    for (long long i = 0; i < my; ++i) {
        const int s = (int)(i & 1);
        if (!mbar_wait(&empty[s], (uint32_t)((i >> 1) & 1), nullptr)) break;
        long long bh; int p0, nr;
        tile(i, bh, p0, nr);
        bulk_store(state + (bh * headdim + p0) * kBulkN, dsm + s * kTileBytes,
                   (uint32_t)nr * kBulkN * 4);
        bulk_commit_group();
        if (i + 2 < my) {
            bulk_wait_read_all();  // the stage has been read out
            tile(i + 2, bh, p0, nr);
            mbar_arrive_expect_tx(&full[s], (uint32_t)nr * kBulkN * 4);
            bulk_load(dsm + s * kTileBytes, state + (bh * headdim + p0) * kBulkN,
                      (uint32_t)nr * kBulkN * 4, &full[s]);
        }
    }
    bulk_wait_all();
}

// Tiles are (b, h, chunk of up to 64 rows); CTA k takes tiles k, k + grid, ...
// Stage s of the two shared-memory stages holds the CTA's tiles s, s + 2, ...:
// full[s] completes when a tile has landed, empty[s] when the compute warps
// have updated it in place (then the producer stores it and reuses the stage).
template <typename T, bool M3>
__global__ void __launch_bounds__(kBulkThreads)
    decode_bulk_kernel(float* __restrict__ state, const T* __restrict__ x,
                       const float* __restrict__ dt, const float* __restrict__ A,
                       const T* __restrict__ Bm, const T* __restrict__ Cm,
                       const float* __restrict__ Dskip, const T* __restrict__ z,
                       T* __restrict__ y, int batch, int nheads, int headdim, int ngroups,
                       M3In<T> m3) {
    extern __shared__ __align__(128) uint8_t dsm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(dsm + 2 * kTileBytes);
    uint64_t* empty = full + 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunks = (headdim + kBulkRows - 1) / kBulkRows;
    const long long ntiles = (long long)batch * nheads * nchunks;
    const long long my = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkCompute / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // tile i of this CTA: (b, h) pair bh, first row p0, rows nr
    auto tile = [&](long long i, long long& bh, int& p0, int& nr) {
        const long long t = blockIdx.x + i * gridDim.x;
        bh = t / nchunks;
        p0 = (int)(t % nchunks) * kBulkRows;
        nr = min(kBulkRows, headdim - p0);
    };

    if (warp == kBulkCompute / 32) {  // ------------------------------ producer
        if (lane == 0) bulk_producer(state, dsm, full, empty, my, headdim, tile);
        return;
    }

    // ------------------------------------------------------------- compute
    for (long long i = 0; i < my; ++i) {
        const int s = (int)(i & 1);
        long long bh; int p0, nr;
        tile(i, bh, p0, nr);
        const int h = (int)(bh % nheads);
        const long long b = bh / nheads;
        const int g = h / (nheads / ngroups);
        // per-tile inputs, loaded before waiting for the state
        const long long bc = (b * ngroups + g) * kBulkN + 4 * lane;
        float bv[4], cv[4], bp[4] = {0.f, 0.f, 0.f, 0.f};
        load4<T>(Bm + bc, bv);
        load4<T>(Cm + bc, cv);
        if constexpr (M3) load4<T>(m3.prev_B + bc, bp);
        const float dtv = dt[bh];
        const float alpha = expf(dtv * A[h]);
        // input weights: Mamba-2 dt; Mamba-3 gamma = lambda dt and, for the
        // previous token, beta = (dt - gamma) alpha
        float wx = dtv, wp = 0.0f;
        if constexpr (M3) {
            wx = m3.lam[bh] * dtv;
            wp = (dtv - wx) * alpha;
        }
        const long long row0 = bh * headdim + p0;  // (b, h, p0) row index
        float dbx[16], pbx[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int p = warp + 4 * r;
            dbx[r] = p < nr ? wx * to_f32(x[row0 + p]) : 0.0f;
            pbx[r] = (M3 && p < nr) ? wp * to_f32(m3.prev_x[row0 + p]) : 0.0f;
        }
        // the output row this lane finishes (lanes 2k, 2k + 1: warp-local row
        // k), its x, gate and D loaded now, before the wait for the state
        const int pe = warp + 4 * (lane >> 1);
        const bool oute = (lane & 1) == 0 && pe < nr;
        const float xe = oute ? to_f32(x[row0 + pe]) : 0.0f;
        const float ze = (oute && z) ? to_f32(z[row0 + pe]) : 0.0f;
        const float De = Dskip ? Dskip[h] : 0.0f;
        if (!mbar_wait(&full[s], (uint32_t)((i >> 1) & 1), nullptr)) break;

        // rows warp, warp + 4, ...: state (in place) and the C^T h partial sums
        float* st = reinterpret_cast<float*>(dsm + s * kTileBytes);
        float acc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int p = warp + 4 * r;
            acc[r] = 0.0f;
            if (p < nr) {
                float4* q = reinterpret_cast<float4*>(st + p * kBulkN) + lane;
                const float4 v = *q;
                float in[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    in[k] = M3 ? fmaf(dbx[r], bv[k], pbx[r] * bp[k]) : dbx[r] * bv[k];
                const float n0 = fmaf(alpha, v.x, in[0]);
                const float n1 = fmaf(alpha, v.y, in[1]);
                const float n2 = fmaf(alpha, v.z, in[2]);
                const float n3 = fmaf(alpha, v.w, in[3]);
                *q = make_float4(n0, n1, n2, n3);
                acc[r] = fmaf(cv[3], n3, fmaf(cv[2], n2, fmaf(cv[1], n1, cv[0] * n0)));
            }
        }
        fence_proxy_async_smem();  // the updated tile is read by the bulk store
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // reduce-scatter the 16 rows' sums over the warp: afterwards lanes
        // 2k and 2k + 1 hold the total of warp-local row k
#pragma unroll
        for (int m = 16, n = 8; m >= 2; m >>= 1, n >>= 1) {
            const bool hi = lane & m;
#pragma unroll
            for (int k = 0; k < n; ++k) {
                const float send = hi ? acc[k] : acc[k + n];
                const float keep = hi ? acc[k + n] : acc[k];
                acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
        if (oute) {
            float out = acc[0] + De * xe;
            if (z) out *= silu_f(ze);
            y[row0 + pe] = from_f32<T>(out);
        }
    }
}

// Mamba-3 MIMO decode, rank RK ("Mamba-3 NKI Kernels for AWS Neuron",
// "Kernel details", mamba3_mimo_decode_kernel): the same tile stream as
// decode_bulk_kernel, with the rank-R input terms
//   state = alpha state + beta sum_r prev_B[r] (x) prev_x[r] + gamma sum_r B[r] (x) x[r]
// and RK read-outs per row, y[r][p] = sum_n C[r][n] state[p][n] (+ D x[r][p],
// gate), each reduce-scattered over the warp like the single one.
// x, z, y, prev_x: (batch, RK, nheads, headdim); B, C, prev_B: (batch, RK,
// ngroups, 128).
template <typename T, int RK>
__global__ void __launch_bounds__(kBulkThreads)
    decode_bulk_mimo_kernel(float* __restrict__ state, const T* __restrict__ x,
                            const float* __restrict__ dt, const float* __restrict__ A,
                            const T* __restrict__ Bm, const T* __restrict__ Cm,
                            const float* __restrict__ Dskip, const T* __restrict__ z,
                            T* __restrict__ y, int batch, int nheads, int headdim, int ngroups,
                            M3In<T> m3) {
    extern __shared__ __align__(128) uint8_t dsm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(dsm + 2 * kTileBytes);
    uint64_t* empty = full + 2;
    // the tile's weighted inputs, gamma x[r][p] and beta prev_x[r][p], fp32
    float* sx = reinterpret_cast<float*>(dsm + 2 * kTileBytes + 64);
    float* sxp = sx + RK * kBulkRows;
    float* sxr = sxp + RK * kBulkRows;  // x itself (the skip term), and z (the gate)
    float* szr = sxr + RK * kBulkRows;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunks = (headdim + kBulkRows - 1) / kBulkRows;
    const long long ntiles = (long long)batch * nheads * nchunks;
    // CTA k takes an equal contiguous range of tiles: consecutive heads of one
    // batch share their group's B, prev_B and C, which then stay in registers.
    // (Measured against the strided order, CTA k taking tiles k, k + grid, ...:
    // 106 against 114 us on batch 256, 32 heads, rank 4; runs of 2-16
    // consecutive tiles, strided, balance worse.)
    const long long t_begin = ntiles * blockIdx.x / gridDim.x;
    const long long my = ntiles * (blockIdx.x + 1) / gridDim.x - t_begin;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkCompute / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    auto tile = [&](long long i, long long& bh, int& p0, int& nr) {
        const long long t = t_begin + i;
        bh = t / nchunks;
        p0 = (int)(t % nchunks) * kBulkRows;
        nr = min(kBulkRows, headdim - p0);
    };

    if (warp == kBulkCompute / 32) {
        if (lane == 0) bulk_producer(state, dsm, full, empty, my, headdim, tile);
        return;
    }

    const long long rstride_x = (long long)nheads * headdim;  // between ranks of x
    const long long rstride_b = (long long)ngroups * kBulkN;  // between ranks of B
    // the tile's per-head inputs (dt, lambda, A, this thread's share of the x and
    // prev_x values the tile stages) are loaded one tile ahead, so that their
    // latency hides behind the previous tile's work
    constexpr int kStageVals = RK * kBulkRows / kBulkCompute;
    static_assert(kStageVals * kBulkCompute == RK * kBulkRows, "staging split");
    struct HeadIn {
        float dtv, lam, A, D;
        float xs[kStageVals], xps[kStageVals], zs[kStageVals];
    };
    auto load_head = [&](long long i, HeadIn& t) {
        long long bh; int p0, nr;
        tile(i, bh, p0, nr);
        const int h = (int)(bh % nheads);
        const long long b = bh / nheads;
        t.dtv = dt[bh];
        t.lam = m3.lam[bh];
        t.A = A[h];
        t.D = Dskip ? Dskip[h] : 0.0f;
        const long long xrow0 = (b * RK * nheads + h) * (long long)headdim + p0;  // rank 0
#pragma unroll
        for (int j = 0; j < kStageVals; ++j) {
            const int k = tid + j * kBulkCompute;
            const int r = k / kBulkRows, p = k % kBulkRows;
            const bool v = p < nr;
            t.xs[j] = v ? to_f32(x[xrow0 + r * rstride_x + p]) : 0.0f;
            t.xps[j] = v ? to_f32(m3.prev_x[xrow0 + r * rstride_x + p]) : 0.0f;
            t.zs[j] = (v && z) ? to_f32(z[xrow0 + r * rstride_x + p]) : 0.0f;
        }
    };
    HeadIn nxt;
    if (my > 0) load_head(0, nxt);
    float bv[RK][4], bp[RK][4], cv[RK][4];  // the group's rows, while (b, g) stays
    long long cur_bg = -1;
    for (long long i = 0; i < my; ++i) {
        const int s = (int)(i & 1);
        const HeadIn cur = nxt;
        long long bh; int p0, nr;
        tile(i, bh, p0, nr);
        const int h = (int)(bh % nheads);
        const long long b = bh / nheads;
        const int g = h / (nheads / ngroups);
        if (b * ngroups + g != cur_bg) {
            cur_bg = b * ngroups + g;
            const long long bc = ((b * RK) * ngroups + g) * kBulkN + 4 * lane;
#pragma unroll
            for (int r = 0; r < RK; ++r) {
                load4<T>(Bm + bc + r * rstride_b, bv[r]);
                load4<T>(m3.prev_B + bc + r * rstride_b, bp[r]);
                load4<T>(Cm + bc + r * rstride_b, cv[r]);
            }
        }
        const float dtv = cur.dtv;
        const float alpha = expf(dtv * cur.A);
        const float gam = cur.lam * dtv;
        const float bet = (dtv - gam) * alpha;
        const long long xrow0 = (b * RK * nheads + h) * (long long)headdim + p0;  // rank 0
        // stage gamma x and beta prev_x of the tile's rows (the previous tile's
        // reads are finished: named barrier at the end of each tile)
#pragma unroll
        for (int j = 0; j < kStageVals; ++j) {
            const int k = tid + j * kBulkCompute;
            sx[k] = gam * cur.xs[j];
            sxp[k] = bet * cur.xps[j];
            sxr[k] = cur.xs[j];
            szr[k] = cur.zs[j];
        }
        if (i + 1 < my) load_head(i + 1, nxt);
        // every compute warp takes the same branch: a timed-out wait ends all of
        // them here, before the barrier at the end of the tile
        const bool got = mbar_wait(&full[s], (uint32_t)((i >> 1) & 1), nullptr);
        if (!named_bar_and(1, kBulkCompute, got)) break;
        float* st = reinterpret_cast<float*>(dsm + s * kTileBytes);

        // state update of rows warp, warp + 4, ... (in place), four rows at a time,
        // each row's RK read-outs taken from the updated values in registers; the
        // 4 RK partial sums of a group are reduce-scattered over the warp
        constexpr int V = 4 * RK;  // values per group: (row k4, rank r) at k4 * RK + r
#pragma unroll 1
        for (int g4 = 0; g4 < 4; ++g4) {
            float acc[V];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int p = warp + 4 * (4 * g4 + k4);
#pragma unroll
                for (int r = 0; r < RK; ++r) acc[k4 * RK + r] = 0.0f;
                if (p < nr) {
                    float in[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int r = 0; r < RK; ++r) {
                        const float xg = sx[r * kBulkRows + p], xb = sxp[r * kBulkRows + p];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            in[k] = fmaf(xg, bv[r][k], fmaf(xb, bp[r][k], in[k]));
                    }
                    float4* q = reinterpret_cast<float4*>(st + p * kBulkN) + lane;
                    const float4 v = *q;
                    const float4 nv = make_float4(fmaf(alpha, v.x, in[0]), fmaf(alpha, v.y, in[1]),
                                                  fmaf(alpha, v.z, in[2]), fmaf(alpha, v.w, in[3]));
                    *q = nv;
#pragma unroll
                    for (int r = 0; r < RK; ++r)
                        acc[k4 * RK + r] = fmaf(cv[r][3], nv.w, fmaf(cv[r][2], nv.z,
                                               fmaf(cv[r][1], nv.y, cv[r][0] * nv.x)));
                }
            }
            // reduce-scatter over lane bits 4, 3, ...: value index = sum of the
            // halves kept; the remaining low lane bits are summed outright
            int idx = 0;
#pragma unroll
            for (int m = 16, n = V / 2; n >= 1; m >>= 1, n >>= 1) {
                const bool hi = lane & m;
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const float send = hi ? acc[k] : acc[k + n];
                    const float keep = hi ? acc[k + n] : acc[k];
                    acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
                if (hi) idx += n;
            }
            constexpr int kLow = 32 / V;  // lanes still holding parts of one value
#pragma unroll
            for (int m = kLow / 2; m >= 1; m >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], m);
            const int k4 = idx / RK, r = idx % RK;
            const int p = warp + 4 * (4 * g4 + k4);
            if ((lane & (kLow - 1)) == 0 && p < nr) {
                const long long row = xrow0 + r * rstride_x + p;
                float out = acc[0] + cur.D * sxr[r * kBulkRows + p];
                if (z) out *= silu_f(szr[r * kBulkRows + p]);
                y[row] = from_f32<T>(out);
            }
        }
        fence_proxy_async_smem();  // the updated tile is read by the bulk store
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        named_bar_sync(1, kBulkCompute);  // sx, sxp, sxr, szr are rewritten for the next tile
    }
}

template <typename T, bool M3>
ssm_status_t launch_bulk(float* state, const void* x, const float* dt, const float* A,
                         const void* B, const void* C, const float* D, const void* z, void* y,
                         int batch, int nheads, int headdim, int ngroups, M3In<T> m3,
                         cudaStream_t s) {
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
            if (cudaFuncSetAttribute(decode_bulk_kernel<T, M3>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kBulkSmem) != cudaSuccess)
                return SSM_ERR_CUDA;
            cached_dev = dev;
        }
    }
    const long long tiles =
        (long long)batch * nheads * ((headdim + kBulkRows - 1) / kBulkRows);
    const unsigned grid = (unsigned)std::min<long long>(tiles, 3LL * sms);
    decode_bulk_kernel<T, M3><<<grid, kBulkThreads, kBulkSmem, s>>>(
        state, static_cast<const T*>(x), dt, A, static_cast<const T*>(B),
        static_cast<const T*>(C), D, static_cast<const T*>(z), static_cast<T*>(y), batch, nheads,
        headdim, ngroups, m3);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, int RK>
ssm_status_t launch_bulk_mimo(float* state, const void* x, const float* dt, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              void* y, int batch, int nheads, int headdim, int ngroups,
                              M3In<T> m3, cudaStream_t s) {
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
            if (cudaFuncSetAttribute(decode_bulk_mimo_kernel<T, RK>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kBulkSmem + 4 * RK * kBulkRows * 4) != cudaSuccess)
                return SSM_ERR_CUDA;
            cached_dev = dev;
        }
    }
    const long long tiles =
        (long long)batch * nheads * ((headdim + kBulkRows - 1) / kBulkRows);
    const unsigned grid = (unsigned)std::min<long long>(tiles, 3LL * sms);
    decode_bulk_mimo_kernel<T, RK><<<grid, kBulkThreads, kBulkSmem + 4 * RK * kBulkRows * 4, s>>>(
        state, static_cast<const T*>(x), dt, A, static_cast<const T*>(B),
        static_cast<const T*>(C), D, static_cast<const T*>(z), static_cast<T*>(y), batch, nheads,
        headdim, ngroups, m3);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T, bool M3>
ssm_status_t by_dstate(int dstate, float* state, const void* x, const float* dt, const float* A,
                       const void* B, const void* C, const float* D, const void* z, void* y,
                       long long rows, int nheads, int headdim, int ngroups, M3In<T> m3,
                       cudaStream_t s) {
    switch (dstate) {
        case 16:
            return launch<T, 1, M3>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups,
                                    m3, s);
        case 32:
            return launch<T, 2, M3>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups,
                                    m3, s);
        case 64:
            return launch<T, 4, M3>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups,
                                    m3, s);
        case 128:
            return launch_bulk<T, M3>(state, x, dt, A, B, C, D, z, y,
                                      (int)(rows / headdim / nheads), nheads, headdim, ngroups, m3,
                                      s);
        case 256:
            return launch<T, 16, M3>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim,
                                     ngroups, m3, s);
    }
    return SSM_ERR_UNSUPPORTED;
}

// Validation and dispatch shared by the Mamba-2 (m3 = false) and Mamba-3 SISO
// (m3 = true) decode entry points.
ssm_status_t decode_entry(float* state, const void* x, const float* dt, const float* lam,
                          const float* A, const void* B, const void* C, const float* D,
                          const void* z, const void* prev_B, const void* prev_x, void* y,
                          int batch, int nheads, int headdim, int dstate, int ngroups,
                          ssm_dtype_t dtype, bool m3, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || nheads < 0 || headdim < 0 || dstate < 1 || ngroups < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(dtype)) return SSM_ERR_DTYPE;
    if (dstate != 16 && dstate != 32 && dstate != 64 && dstate != 128 && dstate != 256)
        return SSM_ERR_UNSUPPORTED;
    const long long rows = (long long)batch * nheads * headdim;
    if (rows == 0) return SSM_OK;
    if (!state || !x || !dt || !A || !B || !C || !y) return SSM_ERR_NULL;
    if (m3 && (!lam || !prev_B || !prev_x)) return SSM_ERR_NULL;
    const void* ptrs[] = {state, x, dt, A, B, C, D, z, y, lam, prev_B, prev_x};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const size_t sbytes = (size_t)rows * dstate * 4, rbytes = (size_t)rows * es;
    const size_t bcbytes = (size_t)batch * ngroups * dstate * es;
    struct R { const void* p; size_t n; } ins[] = {
        {x, rbytes}, {dt, (size_t)batch * nheads * 4}, {A, (size_t)nheads * 4},
        {B, bcbytes}, {C, bcbytes}, {D, D ? (size_t)nheads * 4 : 0}, {z, z ? rbytes : 0},
        {lam, m3 ? (size_t)batch * nheads * 4 : 0}, {prev_B, m3 ? bcbytes : 0},
        {prev_x, m3 ? rbytes : 0}};
    for (const R& r : ins) {
        if (overlaps(state, sbytes, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(y, rbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, rbytes, state, sbytes)) return SSM_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SSM_BF16) {
        using T = __nv_bfloat16;
        const M3In<T> m{lam, static_cast<const T*>(prev_B), static_cast<const T*>(prev_x)};
        return m3 ? by_dstate<T, true>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads,
                                       headdim, ngroups, m, s)
                  : by_dstate<T, false>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads,
                                        headdim, ngroups, m, s);
    }
    const M3In<float> m{lam, static_cast<const float*>(prev_B), static_cast<const float*>(prev_x)};
    return m3 ? by_dstate<float, true>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads,
                                       headdim, ngroups, m, s)
              : by_dstate<float, false>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads,
                                        headdim, ngroups, m, s);
}

}  // namespace

extern "C" ssm_status_t ssm_decode_step(float* state, const void* x, const float* dt,
                                        const float* A, const void* B, const void* C,
                                        const float* D, const void* z, void* y, int batch,
                                        int nheads, int headdim, int dstate, int ngroups,
                                        ssm_dtype_t dtype, void* stream) {
    return decode_entry(state, x, dt, nullptr, A, B, C, D, z, nullptr, nullptr, y, batch, nheads,
                        headdim, dstate, ngroups, dtype, false, stream);
}

extern "C" ssm_status_t ssm_decode_step_mamba3(float* state, const void* prev_B,
                                               const void* prev_x, const void* x,
                                               const float* dt, const float* lam,
                                               const float* A, const void* B, const void* C,
                                               const float* D, const void* z, void* y, int batch,
                                               int nheads, int headdim, int dstate, int ngroups,
                                               ssm_dtype_t dtype, void* stream) {
    return decode_entry(state, x, dt, lam, A, B, C, D, z, prev_B, prev_x, y, batch, nheads,
                        headdim, dstate, ngroups, dtype, true, stream);
}

extern "C" ssm_status_t ssm_decode_step_mamba3_mimo(float* state, const void* prev_B,
                                                    const void* prev_x, const void* x,
                                                    const float* dt, const float* lam,
                                                    const float* A, const void* B, const void* C,
                                                    const float* D, const void* z, void* y,
                                                    int batch, int rank, int nheads, int headdim,
                                                    int dstate, int ngroups, ssm_dtype_t dtype,
                                                    void* stream) {
    using namespace ssm_host;
    if (rank < 1 || batch < 0 || nheads < 0 || headdim < 0 || dstate < 1 || ngroups < 1)
        return SSM_ERR_SHAPE;
    if (rank == 1)  // the (batch, 1, ...) layouts are the single-input ones
        return ssm_decode_step_mamba3(state, prev_B, prev_x, x, dt, lam, A, B, C, D, z, y, batch,
                                      nheads, headdim, dstate, ngroups, dtype, stream);
    if (nheads % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(dtype)) return SSM_ERR_DTYPE;
    if ((rank != 2 && rank != 4) || dstate != kBulkN) return SSM_ERR_UNSUPPORTED;
    const long long rows = (long long)batch * nheads * headdim;
    if (rows == 0) return SSM_OK;
    if (!state || !x || !dt || !A || !B || !C || !y || !lam || !prev_B || !prev_x)
        return SSM_ERR_NULL;
    const void* ptrs[] = {state, x, dt, A, B, C, D, z, y, lam, prev_B, prev_x};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const size_t sbytes = (size_t)rows * dstate * 4, rbytes = (size_t)rows * rank * es;
    const size_t bcbytes = (size_t)batch * rank * ngroups * dstate * es;
    struct R { const void* p; size_t n; } ins[] = {
        {x, rbytes}, {dt, (size_t)batch * nheads * 4}, {A, (size_t)nheads * 4},
        {B, bcbytes}, {C, bcbytes}, {D, D ? (size_t)nheads * 4 : 0}, {z, z ? rbytes : 0},
        {lam, (size_t)batch * nheads * 4}, {prev_B, bcbytes}, {prev_x, rbytes}};
    for (const R& r : ins) {
        if (overlaps(state, sbytes, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(y, rbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, rbytes, state, sbytes)) return SSM_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SSM_BF16) {
        using T = __nv_bfloat16;
        const M3In<T> m{lam, static_cast<const T*>(prev_B), static_cast<const T*>(prev_x)};
        return rank == 2 ? launch_bulk_mimo<T, 2>(state, x, dt, A, B, C, D, z, y, batch, nheads,
                                                  headdim, ngroups, m, s)
                         : launch_bulk_mimo<T, 4>(state, x, dt, A, B, C, D, z, y, batch, nheads,
                                                  headdim, ngroups, m, s);
    }
    const M3In<float> m{lam, static_cast<const float*>(prev_B), static_cast<const float*>(prev_x)};
    return rank == 2 ? launch_bulk_mimo<float, 2>(state, x, dt, A, B, C, D, z, y, batch, nheads,
                                                  headdim, ngroups, m, s)
                     : launch_bulk_mimo<float, 4>(state, x, dt, A, B, C, D, z, y, batch, nheads,
                                                  headdim, ngroups, m, s);
}
