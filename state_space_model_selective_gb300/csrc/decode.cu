// decode.cu -- single-token decode step (ssm_decode_step) for GB300 / sm_103a.
//
// "Mamba-3 NKI Kernels for AWS Neuron", section "How it works" (decode via
// step(), Eq. 9; at lambda = 1: h = alpha h + dt B (x) x, y = C^T h) and
// section "Kernel details" (mamba3_siso_decode_state_kernel: state update
// and output contraction for all heads at once), plus Phase 5 (D skip, silu
// gate).
//
// The step is one streaming read-modify-write of the fp32 state
// (batch, nheads, headdim, dstate), so it is bound by HBM bandwidth: each
// (b, h, p) row of dstate floats is owned by dstate/16 lanes holding 16
// consecutive states each (16-byte loads with evict-first cache hints, two
// rows' loads in flight per lane), the C^T h contraction is an intra-warp
// shuffle reduction, and the row's first lane writes y.
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
template <typename T, int LPR>
__global__ void __launch_bounds__(256, 3)
    decode_kernel(float* __restrict__ state, const T* __restrict__ x,
                  const float* __restrict__ dt, const float* __restrict__ A,
                  const T* __restrict__ Bm, const T* __restrict__ Cm,
                  const float* __restrict__ Dskip, const T* __restrict__ z, T* __restrict__ y,
                  int nheads, int headdim, int ngroups) {
    constexpr int kDstate = LPR * 16;
    constexpr int kRowsPerPass = 256 / LPR;
    constexpr int RPT = 2;
    const int h = blockIdx.x % nheads;
    const long long b = blockIdx.x / nheads;
    const int g = h / (nheads / ngroups);
    const int part = threadIdx.x % LPR;
    const int r0 = threadIdx.x / LPR;

    __shared__ __align__(16) float sB[kDstate], sC[kDstate];
    const long long row_base = (b * nheads + h) * (long long)headdim;
    const long long bc0 = (b * ngroups + g) * kDstate;
    const float4* sB4 = reinterpret_cast<const float4*>(sB + part * 16);
    const float4* sC4 = reinterpret_cast<const float4*>(sC + part * 16);
    float dtv = 0.0f, alpha = 0.0f, Dh = 0.0f;

    for (int p0 = 0; p0 < headdim; p0 += kRowsPerPass * RPT) {
        float s[RPT][16];
        float xv[RPT], zv[RPT];
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
        }
        if (p0 == 0) {
            // B, C, alpha: after the first rows' loads are in flight
            for (int i = threadIdx.x; i < kDstate; i += 256) {
                sB[i] = to_f32(Bm[bc0 + i]);
                sC[i] = to_f32(Cm[bc0 + i]);
            }
            dtv = dt[b * nheads + h];
            alpha = expf(dtv * A[h]);
            Dh = Dskip ? Dskip[h] : 0.0f;
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = p0 + r * kRowsPerPass + r0;
            const long long row = row_base + (act[r] ? p : 0);
            const float dbx = dtv * xv[r];
            float acc = 0.0f;
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const float4 bq = sB4[i4], cq = sC4[i4];
                const float bb[4] = {bq.x, bq.y, bq.z, bq.w}, cc[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    s[r][4 * i4 + k] = fmaf(alpha, s[r][4 * i4 + k], dbx * bb[k]);
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

template <typename T, int LPR>
ssm_status_t launch(float* state, const void* x, const float* dt, const float* A, const void* B,
                    const void* C, const float* D, const void* z, void* y, long long rows,
                    int nheads, int headdim, int ngroups, cudaStream_t s) {
    const long long grid = rows / headdim;  // batch * nheads
    decode_kernel<T, LPR><<<(unsigned)grid, 256, 0, s>>>(
        state, static_cast<const T*>(x), dt, A, static_cast<const T*>(B),
        static_cast<const T*>(C), D, static_cast<const T*>(z), static_cast<T*>(y), nheads,
        headdim, ngroups);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename T>
ssm_status_t by_dstate(int dstate, float* state, const void* x, const float* dt, const float* A,
                       const void* B, const void* C, const float* D, const void* z, void* y,
                       long long rows, int nheads, int headdim, int ngroups, cudaStream_t s) {
    switch (dstate) {
        case 16: return launch<T, 1>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups, s);
        case 32: return launch<T, 2>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups, s);
        case 64: return launch<T, 4>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups, s);
        case 128: return launch<T, 8>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups, s);
        case 256: return launch<T, 16>(state, x, dt, A, B, C, D, z, y, rows, nheads, headdim, ngroups, s);
    }
    return SSM_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" ssm_status_t ssm_decode_step(float* state, const void* x, const float* dt,
                                        const float* A, const void* B, const void* C,
                                        const float* D, const void* z, void* y, int batch,
                                        int nheads, int headdim, int dstate, int ngroups,
                                        ssm_dtype_t dtype, void* stream) {
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
    const void* ptrs[] = {state, x, dt, A, B, C, D, z, y};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const size_t sbytes = (size_t)rows * dstate * 4, rbytes = (size_t)rows * es;
    const size_t bcbytes = (size_t)batch * ngroups * dstate * es;
    struct R { const void* p; size_t n; } ins[] = {
        {x, rbytes}, {dt, (size_t)batch * nheads * 4}, {A, (size_t)nheads * 4},
        {B, bcbytes}, {C, bcbytes}, {D, D ? (size_t)nheads * 4 : 0}, {z, z ? rbytes : 0}};
    for (const R& r : ins) {
        if (overlaps(state, sbytes, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(y, rbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, rbytes, state, sbytes)) return SSM_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == SSM_BF16
               ? by_dstate<__nv_bfloat16>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads,
                                          headdim, ngroups, s)
               : by_dstate<float>(dstate, state, x, dt, A, B, C, D, z, y, rows, nheads, headdim,
                                  ngroups, s);
}
