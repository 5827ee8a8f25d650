// bench_peaks.cu -- throughput probes for the arithmetic units the selective
// scan uses (multi-function-unit ex2, fp32 FMA, packed fp32x2 FMA, broadcast
// shared loads, and how they share the issue slots when mixed), so that the
// scan's roofline is set against measured per-clock rates on this GPU.
// A measurement tool of bench.py (`python bench.py --peaks`), built into its
// own library under _build/; not part of the library or its ABI.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;

__global__ void probe_ex2(float* out, int iters) {
    float x[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) x[k] = 0.001f * (threadIdx.x + k);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k)
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[k]) : "f"(-x[k]));
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += x[k];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void probe_ffma(float* out, int iters, float a, float b) {
    float x[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) x[k] = 0.001f * (threadIdx.x + k);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k)
            asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[k]) : "f"(a), "f"(b));
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += x[k];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void probe_ffma2(float* out, int iters, float a, float b) {
    uint64_t x[kChains];
    const float2 av = make_float2(a, a), bv = make_float2(b, b);
    const uint64_t ar = *reinterpret_cast<const uint64_t*>(&av);
    const uint64_t br = *reinterpret_cast<const uint64_t*>(&bv);
#pragma unroll
    for (int k = 0; k < kChains; ++k) {
        const float2 v = make_float2(0.001f * (threadIdx.x + k), 0.002f * k);
        x[k] = *reinterpret_cast<const uint64_t*>(&v);
    }
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kChains; ++k)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[k]) : "l"(ar), "l"(br));
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) {
        const float2 v = *reinterpret_cast<const float2*>(&x[k]);
        s += v.x + v.y;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Latency probes: one warp runs a chain of dependent operations (16 per loop
// iteration, unrolled); thread 0 writes the elapsed SM clocks per operation.
template <int KIND>
__global__ void latency_probe(float* out, int iters) {
    __shared__ float sm[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm[i] = 0.0f;
    __syncthreads();
    float x = 0.001f * (threadIdx.x + 1);
    const float2 av = make_float2(0.999f, 0.999f), bv = make_float2(0.001f, 0.001f);
    const uint64_t ar = *reinterpret_cast<const uint64_t*>(&av);
    const uint64_t br = *reinterpret_cast<const uint64_t*>(&bv);
    const float2 xv = make_float2(x, x);
    uint64_t v = *reinterpret_cast<const uint64_t*>(&xv);
    unsigned addr = (unsigned)__cvta_generic_to_shared(sm) + 4 * (threadIdx.x & 7);
    __syncwarp();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if constexpr (KIND == 0) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x) : "f"(-x));
            if constexpr (KIND == 1) asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(x) : "f"(x));
            if constexpr (KIND == 2)
                asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x) : "f"(0.999f), "f"(0.001f));
            if constexpr (KIND == 3)
                asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v) : "l"(ar), "l"(br));
            if constexpr (KIND == 4) {  // the loaded value (0) is added to the next address
                unsigned w;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(addr));
                addr += w;
            }
        }
    }
    const long long t1 = clock64();
    if (threadIdx.x == 0) out[0] = (float)(t1 - t0) / (16.0f * iters);
    if (threadIdx.x == 1) out[1] = x + (float)(v & 1) + (float)(addr & 1);
}

// The selective scan's per-step arithmetic for NS states of one channel, from
// registers only: exponent products, NS ex2, state update and read-out, in
// scalar fp32.  y is accumulated so the work is not dead.  Timed by the host.
template <int NS>
__global__ void scan_mix_probe(float* out, int steps) {
    float h[NS], A[NS], Bv[NS], Cv[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        h[k] = 0.0f;
        A[k] = -1.4427f * (k + 1);
        Bv[k] = 0.01f * (k + threadIdx.x % 7);
        Cv[k] = 0.02f * (k - 3);
    }
    float ysum = 0.0f;
    float dl = 0.01f + 1e-5f * threadIdx.x, du = 0.003f;
    for (int t = 0; t < steps; ++t) {
        dl = fmaf(dl, 0.9999f, 1e-6f);  // a fresh step value
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            float e;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(dl * A[k]));
            h[k] = fmaf(e, h[k], du * Bv[k]);
            acc[k & 3] = fmaf(Cv[k], h[k], acc[k & 3]);
        }
        ysum += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = ysum + h[0] + h[NS - 1];
}

// Shared-memory load throughput by access pattern: each thread issues
// `iters` x 8 loads (volatile, so none is merged or hoisted).  WIDTH = 4, 8 or
// 16 bytes; PATTERN 0: every lane of the warp reads the same address; 1: 4
// distinct addresses (lane % 4); 2: 4 distinct addresses (lane / 8, one per
// quarter-warp); 3: 32 distinct consecutive addresses.
template <int WIDTH, int PATTERN>
__global__ void lds_probe(float* out, int iters) {
    __shared__ __align__(16) float sm[4096];
    for (int i = threadIdx.x; i < 4096; i += blockDim.x) sm[i] = 0.001f * i;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    int slot = 0;
    if (PATTERN == 1) slot = lane & 3;
    if (PATTERN == 2) slot = lane >> 3;
    if (PATTERN == 3) slot = lane;
    const unsigned base = (unsigned)__cvta_generic_to_shared(sm) + slot * WIDTH;
    float acc = 0.0f;
    for (int i = 0; i < iters; ++i) {
        // 8 loads 128 bytes apart in one of 8 1-KB rows (all below 9 KB)
        const unsigned row = base + ((unsigned)i & 7u) * 1024u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const unsigned q = row + u * 128u;
            float v0, v1, v2, v3;
            if constexpr (WIDTH == 4) {
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v0) : "r"(q));
            } else if constexpr (WIDTH == 8) {
                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v0), "=f"(v1) : "r"(q));
            } else {
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(v0), "=f"(v1), "=f"(v2), "=f"(v3)
                             : "r"(q));
            }
            acc += v0;  // one add per load keeps the issue cost per load low
        }
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// The scan's full per-element arithmetic (dl*A, ex2, du*B, state FMA,
// read-out FMA) for NS states of one channel, from registers, with dl and
// du changing every step.  PACKED = 1 does the four fp32 operations on pairs
// of states with the fp32x2 instructions (mul/fma .f32x2).
template <int NS, int PACKED>
__global__ void scan_mix2_probe(float* out, int steps) {
    float h[NS], A[NS], Bv[NS], Cv[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        h[k] = 0.0f;
        A[k] = -1.4427f * (k + 1);
        Bv[k] = 0.01f * (k + threadIdx.x % 7);
        Cv[k] = 0.02f * (k - 3);
    }
    float ysum = 0.0f;
    float dl = 0.01f + 1e-5f * threadIdx.x, du = 0.003f;
    for (int t = 0; t < steps; ++t) {
        dl = fmaf(dl, 0.9999f, 1e-6f);
        du = fmaf(du, 0.9999f, 1e-6f);
        if constexpr (PACKED) {
            uint64_t acc2 = 0;
            const float2 dd = make_float2(dl, dl), uu = make_float2(du, du);
            const uint64_t dl2 = *reinterpret_cast<const uint64_t*>(&dd);
            const uint64_t du2 = *reinterpret_cast<const uint64_t*>(&uu);
#pragma unroll
            for (int k = 0; k < NS; k += 2) {
                const float2 ap = make_float2(A[k], A[k + 1]);
                const float2 bp = make_float2(Bv[k], Bv[k + 1]);
                const float2 cp = make_float2(Cv[k], Cv[k + 1]);
                float2 hp = make_float2(h[k], h[k + 1]);
                uint64_t arg, bx, hh = *reinterpret_cast<uint64_t*>(&hp);
                asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(arg) : "l"(dl2),
                    "l"(*reinterpret_cast<const uint64_t*>(&ap)));
                asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(bx) : "l"(du2),
                    "l"(*reinterpret_cast<const uint64_t*>(&bp)));
                float2 av = *reinterpret_cast<float2*>(&arg);
                float e0, e1;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(av.x));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(av.y));
                const float2 ep = make_float2(e0, e1);
                asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(hh)
                    : "l"(*reinterpret_cast<const uint64_t*>(&ep)), "l"(bx));
                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2)
                    : "l"(*reinterpret_cast<const uint64_t*>(&cp)), "l"(hh));
                hp = *reinterpret_cast<float2*>(&hh);
                h[k] = hp.x;
                h[k + 1] = hp.y;
            }
            const float2 a = *reinterpret_cast<float2*>(&acc2);
            ysum += a.x + a.y;
        } else {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                float e;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(dl * A[k]));
                h[k] = fmaf(e, h[k], du * Bv[k]);
                acc[k & 3] = fmaf(Cv[k], h[k], acc[k & 3]);
            }
            ysum += (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = ysum + h[0] + h[NS - 1];
}

}  // namespace

// Shared-memory load probe (see lds_probe); returns warp-level loads issued.
extern "C" double ssm_lds_probe(int width, int pattern, int blocks, int threads, int iters,
                                float* out, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define LDS_CASE(W, P) \
    if (width == W && pattern == P) lds_probe<W, P><<<blocks, threads, 0, s>>>(out, iters);
    LDS_CASE(4, 0) LDS_CASE(4, 1) LDS_CASE(4, 2) LDS_CASE(4, 3)
    LDS_CASE(8, 0) LDS_CASE(8, 1) LDS_CASE(8, 2) LDS_CASE(8, 3)
    LDS_CASE(16, 0) LDS_CASE(16, 1) LDS_CASE(16, 2) LDS_CASE(16, 3)
#undef LDS_CASE
    if (cudaGetLastError() != cudaSuccess) return -1.0;
    return (double)blocks * (threads / 32) * iters * 8;
}

// Full per-element scan arithmetic (scan_mix2_probe), scalar or packed;
// returns the number of steps x threads executed, or -1.
extern "C" double ssm_scan_mix2_probe(int ns, int packed, int blocks, int threads, int steps,
                                      float* out, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define MIX2_CASE(N, P) \
    if (ns == N && packed == P) scan_mix2_probe<N, P><<<blocks, threads, 0, s>>>(out, steps);
    MIX2_CASE(4, 0) MIX2_CASE(4, 1) MIX2_CASE(8, 0) MIX2_CASE(8, 1) MIX2_CASE(16, 0)
    MIX2_CASE(16, 1)
#undef MIX2_CASE
    if (cudaGetLastError() != cudaSuccess) return -1.0;
    return (double)blocks * threads * steps;
}

// Per-step arithmetic of the scan with `ns` (4, 8 or 16) states per thread;
// returns the number of steps x threads executed, or -1.
extern "C" double ssm_scan_mix_probe(int ns, int blocks, int threads, int steps, float* out,
                                     void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (ns) {
        case 4: scan_mix_probe<4><<<blocks, threads, 0, s>>>(out, steps); break;
        case 8: scan_mix_probe<8><<<blocks, threads, 0, s>>>(out, steps); break;
        case 16: scan_mix_probe<16><<<blocks, threads, 0, s>>>(out, steps); break;
        default: return -1.0;
    }
    if (cudaGetLastError() != cudaSuccess) return -1.0;
    return (double)blocks * threads * steps;
}

// Cycles per dependent operation for kind 0 ex2, 1 rcp, 2 fp32 FMA,
// 3 fp32x2 FMA, 4 shared-memory load; one warp, `iters` operations.
extern "C" float ssm_latency_probe(int kind, int iters, float* out, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (kind) {
        case 0: latency_probe<0><<<1, 32, 0, s>>>(out, iters); break;
        case 1: latency_probe<1><<<1, 32, 0, s>>>(out, iters); break;
        case 2: latency_probe<2><<<1, 32, 0, s>>>(out, iters); break;
        case 3: latency_probe<3><<<1, 32, 0, s>>>(out, iters); break;
        case 4: latency_probe<4><<<1, 32, 0, s>>>(out, iters); break;
        default: return -1.0f;
    }
    float h[2] = {0, 0};
    if (cudaMemcpyAsync(h, out, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1.0f;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1.0f;
    return h[0];
}

// kind 0: ex2 (one MUFU op per lane per instruction)
// kind 1: fp32 FMA; kind 2: packed fp32x2 FMA (two FMAs per lane per instruction)
// Returns the number of per-lane results the launch computes, or -1.
extern "C" double ssm_peak_probe(int kind, int blocks, int threads, int iters, float* out,
                                 void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const double lanes = (double)blocks * threads;
    switch (kind) {
        case 0: probe_ex2<<<blocks, threads, 0, s>>>(out, iters); break;
        case 1: probe_ffma<<<blocks, threads, 0, s>>>(out, iters, 0.999f, 0.001f); break;
        case 2: probe_ffma2<<<blocks, threads, 0, s>>>(out, iters, 0.999f, 0.001f); break;
        default: return -1.0;
    }
    if (cudaGetLastError() != cudaSuccess) return -1.0;
    return lanes * iters * kChains * (kind == 2 ? 2.0 : 1.0);
}

// ---------------------------------------------------------------- overlap
//
// How the MUFU, the FP32 pipe and broadcast shared loads share a warp
// scheduler's issue slots.  Per "step" each thread runs, by mode bit:
//   1: 8 x (FMUL + MUFU ex2) on 8 independent chains
//   2: NF scalar FFMAs on 16 independent accumulators
//   4: NF packed fp32x2 FMAs on 8 independent accumulator pairs
// plus NL warp-uniform (broadcast) 16-byte shared loads.  Returns the SM
// clocks of the slowest CTA; the caller divides by warp-steps per
// sub-partition.
namespace {

__device__ __forceinline__ unsigned long long pk2(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

template <int MODE, int NF, int NL>
__global__ void __launch_bounds__(128) overlap_probe(float* out, int iters, long long* cyc,
                                                     float k) {
    __shared__ float4 sm[64];
    const int tid = threadIdx.x;
    if (tid < 64) sm[tid] = make_float4(tid * 0.01f, 0.5f, 0.25f, 0.125f);
    __syncthreads();
    const long long c0 = clock64();
    float m[8], f[16];
    unsigned long long pv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { m[i] = 0.1f * i + tid * 1e-4f; pv[i] = pk2(0.01f * i, 0.02f * i); }
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = 0.01f * i;
    float acc = 0.0f;
    const unsigned long long k2 = pk2(0.999f, 0.998f), c2 = pk2(1e-3f, 2e-3f);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            if (MODE & 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(m[i]) : "f"(m[i] * k));
            }
            if (MODE & 2) {
#pragma unroll
                for (int j = 0; j < NF; ++j) f[j & 15] = fmaf(f[j & 15], 0.999f, 1e-3f);
            }
            if (MODE & 4) {
#pragma unroll
                for (int j = 0; j < NF; ++j)
                    asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(pv[j & 7]) : "l"(k2), "l"(c2));
            }
#pragma unroll
            for (int l = 0; l < NL; ++l) acc += sm[(s * NL + l) & 63].x;
        }
    }
    const long long c1 = clock64();
    float r = acc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float a, b;
        asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(pv[i]));
        r += m[i] + a + b;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) r += f[i];
    out[blockIdx.x * blockDim.x + tid] = r;
    if (tid == 0) cyc[blockIdx.x] = c1 - c0;
}

}  // namespace

// case: 0 MUFU only, 1 FFMA only, 2 FFMA2 only, 3 broadcast loads only,
// 4 MUFU + 24 FFMA, 5 MUFU + 12 FFMA2, 6 MUFU + 24 FFMA + 4 loads,
// 7 MUFU + 12 FFMA2 + 8 loads.  blocks: 4 warps each; out: blocks * 128
// floats; cyc: blocks int64.  Returns 0 on a launch error, else 1.
extern "C" int ssm_overlap_probe(int which, int blocks, int iters, float* out, long long* cyc,
                                 void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (which) {
        case 0: overlap_probe<1, 0, 0><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 1: overlap_probe<2, 32, 0><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 2: overlap_probe<4, 16, 0><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 3: overlap_probe<0, 0, 8><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 4: overlap_probe<3, 24, 0><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 5: overlap_probe<5, 12, 0><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        case 6: overlap_probe<3, 24, 4><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
        default: overlap_probe<5, 12, 8><<<blocks, 128, 0, s>>>(out, iters, cyc, 0.5f); break;
    }
    return cudaGetLastError() == cudaSuccess ? 1 : 0;
}
