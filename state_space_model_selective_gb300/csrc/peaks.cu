// peaks.cu -- throughput probes for the arithmetic units the selective scan
// uses (multi-function-unit ex2, fp32 FMA, packed fp32x2 FMA), so that the
// scan's roofline is set against measured per-clock rates on this GPU.
// Built into its own library (libssm_peaks.so); not part of the ssm.h ABI.
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

}  // namespace

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
