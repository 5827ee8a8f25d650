// rope.cu -- Mamba-3's data-dependent rotation of B and C (ssm_mamba3_rope).
//
// What it computes: "Mamba-3 NKI Kernels for AWS Neuron", section "How it
// works", Phase 1: the angle cumsum cum_angles = -cumsum(dt * theta) along
// the sequence, then RoPE applied to B and C (the page's "complex-valued
// state via data-dependent RoPE": rotating state pair k of B_t and C_t by the
// running angle turns the real recurrence into one with complex eigenvalues
// exp(dt (A + i theta))).  The rotated B and C feed ssd_mamba3_fwd,
// ssd_mamba3_mimo_fwd and, one step at a time, the decode steps.
//
// How: one thread per (batch, head, state pair k) walks the sequence; per
// step it adds -dt * theta to its angle (Kahan-compensated fp32 sum, so the
// angle's error stays near one rounding of its value instead of growing with
// the sequence), takes sincos of it, and rotates pair (2k, 2k + 1) of the
// group's B and C for every rank of the step into the head's rows.  Adjacent
// threads own adjacent pairs, so every load and store of a warp is one
// contiguous span.
#include "common.cuh"

namespace {

using namespace ssm;

template <typename T> struct Pair;
template <> struct Pair<float> {
    using V = float2;
    __device__ static float2 load(const float* p) { return *reinterpret_cast<const float2*>(p); }
    __device__ static void store(float* p, float a, float b) {
        *reinterpret_cast<float2*>(p) = make_float2(a, b);
    }
    __device__ static float lo(float2 v) { return v.x; }
    __device__ static float hi(float2 v) { return v.y; }
};
template <> struct Pair<__nv_bfloat16> {
    using V = __nv_bfloat162;
    __device__ static __nv_bfloat162 load(const __nv_bfloat16* p) {
        return *reinterpret_cast<const __nv_bfloat162*>(p);
    }
    __device__ static void store(__nv_bfloat16* p, float a, float b) {
        __nv_bfloat162 v;
        v.x = __float2bfloat16_rn(a);
        v.y = __float2bfloat16_rn(b);
        *reinterpret_cast<__nv_bfloat162*>(p) = v;
    }
    __device__ static float lo(__nv_bfloat162 v) { return __bfloat162float(v.x); }
    __device__ static float hi(__nv_bfloat162 v) { return __bfloat162float(v.y); }
};

struct RopeArgs {
    const void* B;
    const void* C;
    const float* dt;
    const float* theta;
    const float* angle0;
    void* Brot;
    void* Crot;
    float* angle_out;
    int batch, seqlen, rank, nheads, ngroups, dstate;
};

template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(const RopeArgs a) {
    using P = Pair<T>;
    const int half = a.dstate / 2;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)a.batch * a.nheads * half;
    if (idx >= total) return;
    const int k = (int)(idx % half);
    const int h = (int)((idx / half) % a.nheads);
    const int b = (int)(idx / ((long long)half * a.nheads));
    const int g = h / (a.nheads / a.ngroups);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    T* Br = static_cast<T*>(a.Brot);
    T* Cr = static_cast<T*>(a.Crot);

    float angle = a.angle0 ? a.angle0[idx] : 0.0f;
    float comp = 0.0f;  // Kahan compensation of the running sum
    for (int t = 0; t < a.seqlen; ++t) {
        const long long bt = (long long)b * a.seqlen + t;
        const float w = -a.dt[bt * a.nheads + h] * a.theta[(bt * a.nheads + h) * half + k];
        const float yk = w - comp;
        const float sum = angle + yk;
        comp = (sum - angle) - yk;
        angle = sum;
        float sn, cs;
        sincosf(angle, &sn, &cs);
        for (int r = 0; r < a.rank; ++r) {
            const long long src = ((bt * a.rank + r) * a.ngroups + g) * a.dstate + 2 * k;
            const long long dst = ((bt * a.rank + r) * a.nheads + h) * a.dstate + 2 * k;
            const typename P::V bv = P::load(Bm + src);
            const typename P::V cv = P::load(Cm + src);
            P::store(Br + dst, P::lo(bv) * cs - P::hi(bv) * sn, P::lo(bv) * sn + P::hi(bv) * cs);
            P::store(Cr + dst, P::lo(cv) * cs - P::hi(cv) * sn, P::lo(cv) * sn + P::hi(cv) * cs);
        }
    }
    if (a.angle_out) a.angle_out[idx] = angle - comp;
}

}  // namespace

extern "C" ssm_status_t ssm_mamba3_rope(const void* B, const void* C, const float* dt,
                                        const float* theta, const float* angle0, void* B_rot,
                                        void* C_rot, float* angle_out, int batch, int seqlen,
                                        int rank, int nheads, int ngroups, int dstate,
                                        ssm_dtype_t dtype, void* stream) {
    using namespace ssm_host;
    if (batch < 0 || seqlen < 0 || rank < 1 || nheads < 0 || ngroups < 1 || dstate < 2)
        return SSM_ERR_SHAPE;
    if (dstate % 2 != 0 || nheads % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(dtype)) return SSM_ERR_DTYPE;
    const size_t half = (size_t)dstate / 2;
    const size_t nang = (size_t)batch * nheads * half;
    if (nang == 0) return SSM_OK;
    if (nang > (size_t)INT32_MAX * 256) return SSM_ERR_UNSUPPORTED;
    if (seqlen > 0 && (!B || !C || !dt || !theta || !B_rot || !C_rot)) return SSM_ERR_NULL;
    const void* ptrs[] = {B, C, dt, theta, angle0, B_rot, C_rot, angle_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const size_t steps = (size_t)batch * seqlen;
    const size_t bc = steps * rank * ngroups * dstate * es;
    const size_t rot = steps * rank * nheads * dstate * es;
    const size_t dtb = steps * nheads * 4, thb = steps * nheads * half * 4, angb = nang * 4;
    struct R { const void* p; size_t n; } ins[] = {
        {B, bc}, {C, bc}, {dt, dtb}, {theta, thb}, {angle0, angle0 ? angb : 0}};
    struct O { const void* p; size_t n; } outs[] = {
        {B_rot, seqlen ? rot : 0}, {C_rot, seqlen ? rot : 0}, {angle_out, angle_out ? angb : 0}};
    for (const O& o : outs) {
        for (const R& r : ins) {
            // the final angle may be written over the initial one (in place)
            if (o.p == angle_out && r.p == angle0 && angle_out == angle0) continue;
            if (overlaps(o.p, o.n, r.p, r.n)) return SSM_ERR_ALIAS;
        }
    }
    if (overlaps(B_rot, outs[0].n, C_rot, outs[1].n) ||
        overlaps(B_rot, outs[0].n, angle_out, outs[2].n) ||
        overlaps(C_rot, outs[1].n, angle_out, outs[2].n))
        return SSM_ERR_ALIAS;

    RopeArgs a{B, C, dt, theta, angle0, B_rot, C_rot, angle_out,
               batch, seqlen, rank, nheads, ngroups, dstate};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned grid = (unsigned)((nang + 255) / 256);
    if (dtype == SSM_BF16) rope_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else rope_kernel<float><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
