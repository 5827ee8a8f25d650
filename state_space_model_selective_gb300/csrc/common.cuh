// common.cuh -- small device and host helpers shared by the kernels of the
// GB300 selective-scan library (inline PTX for sm_103a: mbarrier, TMA,
// MUFU approximations, acquire/release flags, named barriers).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm.h"

namespace ssm {

// ------------------------------------------------------------------ types

template <typename T> struct DType;
template <> struct DType<float> { static constexpr ssm_dtype_t code = SSM_F32; };
template <> struct DType<__nv_bfloat16> { static constexpr ssm_dtype_t code = SSM_BF16; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// bf16 pair packed in a 32-bit word -> two floats (exact: a bf16 is the top
// half of an fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------- MUFU math

// 2^x on the multi-function unit (relative error about 2 ulp; flushes
// denormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// 1/x on the multi-function unit (at most 1 ulp).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

constexpr float kLog2e = 1.4426950408889634f;

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^-|x|), accurate to a few
// ulp in fp32 including far into the negative tail (where 1 + e^x would round
// away e^x).  log1p(t) for t = e^-|x| in (0, 1] is evaluated as
// 2 atanh(s) = 2 s f(s^2), s = t / (2 + t) in (0, 1/3], with f(w) =
// atanh(sqrt(w)) / sqrt(w) replaced by a degree-4 polynomial fitted for
// minimum relative error on [0, 1/9] (csrc/fit_softplus_poly.py: 4e-9, about
// 1 ulp once evaluated in fp32).  2 MUFU ops + ~11 FP32 ops.
__device__ __forceinline__ float softplus_f(float x) {
    const float t = ex2_approx(-fabsf(x) * kLog2e);
    const float s = t * rcp_approx(2.0f + t);
    const float w = s * s;
    float p = 0.1408916562795639f;
    p = fmaf(p, w, 0.13980305194854736f);
    p = fmaf(p, w, 0.20012454688549042f);
    p = fmaf(p, w, 0.3333315849304199f);
    p = fmaf(p, w, 1.0f);
    return fmaf(s + s, p, fmaxf(x, 0.0f));
}

// silu(z) = z / (1 + e^-z); -> -0 for z -> -inf, z for z -> +inf.
__device__ __forceinline__ float silu_f(float z) {
    return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
}

// ------------------------------------------------------- bounded waiting

// Spin limits.  A wait that runs out records SSM_ERR_TIMEOUT and gives up;
// the kernel then finishes without touching the data it waited for.
constexpr uint32_t kMbarSpinLimit = 1u << 22;   // try_wait rounds of <= 1 us each
constexpr uint32_t kFlagSpinLimit = 1u << 22;   // look-back polls (~seconds)

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t code) {
    if (status) atomicCAS(status, 0u, code);
}

// --------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Wait until the phase with the given parity has completed.  Returns false
// if the wait ran out (after recording SSM_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < kMbarSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity), "r"(1000u)
            : "memory");
        if (done) return true;
    }
    record_status(status, SSM_ERR_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------- TMA

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on
// `bar`.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy accesses (TMA writes, tcgen05.mma operand reads) that follow
// the next synchronisation.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ barriers

// Named barrier over `nthreads` threads (a multiple of 32).  Id 0 is
// __syncthreads().
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads,
// so that every thread takes the same branch after it.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// --------------------------------------------------- acquire / release

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

}  // namespace ssm

// --------------------------------------------------------------- host side

namespace ssm_host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [lo, lo + bytes) and [lo2, lo2 + bytes2) overlap?
inline bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

inline size_t dtype_size(ssm_dtype_t t) { return t == SSM_BF16 ? 2 : 4; }

inline bool dtype_ok(ssm_dtype_t t) { return t == SSM_F32 || t == SSM_BF16; }

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library has no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Row-major 2-D tensor (rows x cols, cols contiguous) with a box of
// box_rows x box_cols, 128-byte swizzle (or none), zero fill out of bounds.
bool make_tmap_2d(CUtensorMap* map, const void* base, ssm_dtype_t dtype, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols, bool swizzle = true);

}  // namespace ssm_host
