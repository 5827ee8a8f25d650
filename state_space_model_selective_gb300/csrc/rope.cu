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
// How: one CTA per (batch, head, block of up to 64 state pairs) walks the
// sequence in tiles of 2048 (step, pair) angles.  Per tile it
//   1. stages w = -dt * theta in shared memory (rows of theta fetched into
//      registers one tile ahead);
//   2. scans w along the steps: the tile's steps are cut into segments of 8,
//      one thread per (pair, segment) sums its segment with compensation,
//      composes the segment sums before its own onto the carried angle, walks
//      its segment again from there and writes cos and sin of each step's
//      angle to shared memory.  Angles are carried as float-float pairs
//      (hi + lo: compensated steps, TwoSum composition), so their error stays
//      near one rounding of their value instead of growing with the sequence;
//   3. rotates every (step, rank, pair) of the tile with 16-byte loads and
//      stores spread over all threads (the first two units of each thread
//      loaded before the scan), so whole rows move per warp instruction.
#include <type_traits>

#include "common.cuh"

namespace {

using namespace ssm;

constexpr int kThreads = 256;
constexpr int kSegSteps = 8;                 // steps one thread scans per tile
constexpr int kTile = kThreads * kSegSteps;  // (step, pair) angles per tile
constexpr int kMaxPairsLog2 = 6;             // at most 64 state pairs per CTA

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
    int kp_log2;  // log2 of the pairs one CTA covers
    int kblocks;  // CTAs per (batch, head)
};

// one compensated step: (hi, lo) += w, the rounding error of the add kept in lo
__device__ __forceinline__ void comp_add(float& hi, float& lo, float w) {
    const float y = w + lo;
    const float t = hi + y;
    lo = y - (t - hi);
    hi = t;
}

// float-float sum (hi, lo) += (bh, bl): TwoSum of the high parts, the error
// and both low parts folded in, then renormalised
__device__ __forceinline__ void ff_add(float& hi, float& lo, float bh, float bl) {
    const float s = hi + bh;
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (bh - bb);
    const float l = e + lo + bl;
    hi = s + l;
    lo = l - (hi - s);
}

// sin and cos of the float-float angle hi + lo, to fp32 accuracy.  Reduction
// by multiples of pi/2 (Cody and Waite: pi/2 split into two floats, each
// product k * part taken exactly inside an FMA; the residue of the split is
// below 2e-15 per multiple), the low part of the angle added to the reduced
// argument, then the Taylor polynomials of sin and cos on [-pi/4, pi/4]
// (truncated after the x^9 and x^10 terms: below 2e-9 there) and the
// quadrant applied by swapping and negating.  The absolute error stays near
// 1e-7 for angles up to about 1e6.
__device__ __forceinline__ void sincos_ff(float hi, float lo, float& s_out, float& c_out) {
    constexpr float kTwoOverPi = 0.636619772f;
    constexpr float kPio2A = 1.57079637050628662109375f;  // the float nearest pi/2
    constexpr float kPio2B = -4.37113882867379e-08f;      // pi/2 - kPio2A
    const float k = rintf(hi * kTwoOverPi);
    float r = fmaf(-k, kPio2A, hi);
    r = fmaf(-k, kPio2B, r) + lo;
    const float r2 = r * r;
    float ps = fmaf(r2, 1.0f / 362880.0f, -1.0f / 5040.0f);
    ps = fmaf(r2, ps, 1.0f / 120.0f);
    ps = fmaf(r2, ps, -1.0f / 6.0f);
    const float sn = fmaf(r * r2, ps, r);
    float pc = fmaf(r2, -1.0f / 3628800.0f, 1.0f / 40320.0f);
    pc = fmaf(r2, pc, -1.0f / 720.0f);
    pc = fmaf(r2, pc, 1.0f / 24.0f);
    pc = fmaf(r2, pc, -0.5f);
    const float cs = fmaf(r2, pc, 1.0f);
    // angle = k pi/2 + r: quadrant q = k mod 4 (two's complement keeps it for k < 0)
    const int q = (int)k & 3;
    const float s = (q & 1) ? cs : sn;
    const float c = (q & 1) ? sn : cs;
    s_out = (q & 2) ? -s : s;
    c_out = ((q + 1) & 2) ? -c : c;
}

// sin and cos of hi + lo where the outputs are bf16: reduction by multiples of
// 2 pi (Cody and Waite again, 2 pi split into two floats), the low part added,
// then the hardware sine and cosine on [-pi, pi], whose documented absolute
// error there is below 2^-21 -- thousands of times below one bf16 step.
__device__ __forceinline__ void sincos_hw(float hi, float lo, float& s_out, float& c_out) {
    constexpr float kInv2Pi = 0.159154943f;
    constexpr float k2PiA = 6.28318548202514648438f;   // the float nearest 2 pi
    constexpr float k2PiB = -1.7484555314695172e-07f;  // 2 pi - k2PiA
    const float k = rintf(hi * kInv2Pi);
    float r = fmaf(-k, k2PiA, hi);
    r = fmaf(-k, k2PiB, r) + lo;
    __sincosf(r, &s_out, &c_out);
}

template <typename T> struct Trig;
template <> struct Trig<float> {
    __device__ static void sincos(float hi, float lo, float& s, float& c) { sincos_ff(hi, lo, s, c); }
};
template <> struct Trig<__nv_bfloat16> {
    __device__ static void sincos(float hi, float lo, float& s, float& c) { sincos_hw(hi, lo, s, c); }
};

// the PPV (cos, sin) pairs at rot (16-byte aligned when PPV > 1)
template <int PPV>
__device__ __forceinline__ void load_rot(const float2* rot, float2 (&r)[PPV]) {
    if constexpr (PPV == 1) {
        r[0] = rot[0];
    } else {
#pragma unroll
        for (int p = 0; p < PPV; p += 2) {
            const float4 v = reinterpret_cast<const float4*>(rot)[p / 2];
            r[p] = make_float2(v.x, v.y);
            r[p + 1] = make_float2(v.z, v.w);
        }
    }
}

// 2 * PPV consecutive elements (PPV state pairs) as one load or store
template <typename T, int PPV> struct Pairs;

template <int PPV>
struct Pairs<float, PPV> {
    using W = typename std::conditional<PPV == 2, float4, float2>::type;
    __device__ static W load(const float* p) { return __ldg(reinterpret_cast<const W*>(p)); }
    // the pairs of b and c rotated by the (cos, sin) pairs at rot, stored at ob and oc
    __device__ static void rotate_store(W b, W c, const float2* rot, float* ob, float* oc) {
        float2 r[PPV];
        load_rot<PPV>(rot, r);
        const float* bv = reinterpret_cast<const float*>(&b);
        const float* cv = reinterpret_cast<const float*>(&c);
        W rb, rc;
        float* bo = reinterpret_cast<float*>(&rb);
        float* co = reinterpret_cast<float*>(&rc);
#pragma unroll
        for (int p = 0; p < PPV; ++p) {
            bo[2 * p] = bv[2 * p] * r[p].x - bv[2 * p + 1] * r[p].y;
            bo[2 * p + 1] = bv[2 * p] * r[p].y + bv[2 * p + 1] * r[p].x;
            co[2 * p] = cv[2 * p] * r[p].x - cv[2 * p + 1] * r[p].y;
            co[2 * p + 1] = cv[2 * p] * r[p].y + cv[2 * p + 1] * r[p].x;
        }
        *reinterpret_cast<W*>(ob) = rb;
        *reinterpret_cast<W*>(oc) = rc;
    }
};

// bf16: one pair per 32-bit word (element 2k in the low half)
template <int PPV>
struct Pairs<__nv_bfloat16, PPV> {
    using W = typename std::conditional<PPV == 4, uint4, unsigned int>::type;
    __device__ static W load(const __nv_bfloat16* p) {
        return __ldg(reinterpret_cast<const W*>(p));
    }
    __device__ static unsigned int rot_word(unsigned int v, float2 r) {
        const float x = bf16lo(v), y = bf16hi(v);
        const __nv_bfloat162 o = __floats2bfloat162_rn(x * r.x - y * r.y, x * r.y + y * r.x);
        return *reinterpret_cast<const unsigned int*>(&o);
    }
    __device__ static void rotate_store(W b, W c, const float2* rot, __nv_bfloat16* ob,
                                        __nv_bfloat16* oc) {
        float2 r[PPV];
        load_rot<PPV>(rot, r);
        const unsigned int* bw = reinterpret_cast<const unsigned int*>(&b);
        const unsigned int* cw = reinterpret_cast<const unsigned int*>(&c);
        W rb, rc;
        unsigned int* bo = reinterpret_cast<unsigned int*>(&rb);
        unsigned int* co = reinterpret_cast<unsigned int*>(&rc);
#pragma unroll
        for (int p = 0; p < PPV; ++p) {
            bo[p] = rot_word(bw[p], r[p]);
            co[p] = rot_word(cw[p], r[p]);
        }
        *reinterpret_cast<W*>(ob) = rb;
        *reinterpret_cast<W*>(oc) = rc;
    }
};

// theta (and dt) of one tile, fetched into registers a tile ahead: 2048
// values, 2 float4 per thread when rows allow it (TV4), else 8 floats.  The
// (step, pair) a thread fetches within a tile is the same every tile, so its
// offsets are taken once.
template <bool TV4>
struct ThetaRegs {
    static constexpr int N = TV4 ? 2 : 8;
    static constexpr int W = TV4 ? 4 : 1;
    float v[N][W];
    float d[N];
    int step[N];     // step within the tile, or a large value for a pair out of range
    int off_th[N];   // theta offset from the tile's first (step, head) row
    int off_dt[N];

    __device__ void init(const RopeArgs& a, int k0, int half, int tid) {
        const int kp_log2 = a.kp_log2, kp = 1 << kp_log2;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const int e = tid + j * kThreads;
            const int i = TV4 ? e >> (kp_log2 - 2) : e >> kp_log2;
            const int q = TV4 ? (e & ((kp >> 2) - 1)) * 4 : e & (kp - 1);
            step[j] = k0 + q < half ? i : 1 << 30;
            off_th[j] = i * a.nheads * half + q;
            off_dt[j] = i * a.nheads;
        }
    }
    // base_th, base_dt: offsets of (step t0, head h, pair k0) and (step t0, head h)
    __device__ void fetch(const RopeArgs& a, long long base_th, long long base_dt, int tn) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
#pragma unroll
            for (int c = 0; c < W; ++c) v[j][c] = 0.0f;
            d[j] = 0.0f;
            if (step[j] < tn) {
                d[j] = __ldg(a.dt + base_dt + off_dt[j]);
                const float* src = a.theta + base_th + off_th[j];
                if constexpr (TV4) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
                    v[j][0] = x.x;
                    v[j][1] = x.y;
                    v[j][2] = x.z;
                    v[j][3] = x.w;
                } else {
                    v[j][0] = __ldg(src);
                }
            }
        }
    }
    // w = -dt * theta into the tile's [step][pair] array
    __device__ void put(float* w_s, int tid) const {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const int e = tid + j * kThreads;
            if constexpr (TV4) {
                reinterpret_cast<float4*>(w_s)[e] =
                    make_float4(-d[j] * v[j][0], -d[j] * v[j][1], -d[j] * v[j][2], -d[j] * v[j][3]);
            } else {
                w_s[e] = -d[j] * v[j][0];
            }
        }
    }
};

template <typename T, int PPV, bool TV4>
__global__ void __launch_bounds__(kThreads, 3) rope_kernel(const RopeArgs a) {
    using V = Pairs<T, PPV>;
    constexpr int PF = 2;  // B/C units a thread loads ahead of the scan per tile
    constexpr int kPpvLog2 = PPV == 4 ? 2 : PPV == 2 ? 1 : 0;
    __shared__ __align__(16) float w_s[kTile];      // [step in tile][pair]
    __shared__ __align__(16) float2 rot_s[kTile];   // (cos, sin) [step in tile][pair]
    __shared__ float2 agg_s[kThreads];              // segment sums (hi, lo) [segment][pair]
    __shared__ float2 carry_s[1 << kMaxPairsLog2];  // angle (hi, lo) before the tile [pair]

    const int tid = threadIdx.x;
    const int kp = 1 << a.kp_log2;           // pairs per CTA
    const int nseg = kThreads >> a.kp_log2;  // segments per tile
    const int tile_steps = nseg * kSegSteps;
    const int half = a.dstate / 2;
    const int kb = blockIdx.x % a.kblocks;
    const int h = (blockIdx.x / a.kblocks) % a.nheads;
    const int b = blockIdx.x / (a.kblocks * a.nheads);
    const int g = h / (a.nheads / a.ngroups);
    const int k0 = kb * kp;
    const int kk = tid & (kp - 1);  // this thread's pair in the scan
    const int seg = tid >> a.kp_log2;
    const bool kvalid = k0 + kk < half;
    const T* __restrict__ Bm = static_cast<const T*>(a.B);
    const T* __restrict__ Cm = static_cast<const T*>(a.C);
    T* __restrict__ Br = static_cast<T*>(a.Brot);
    T* __restrict__ Cr = static_cast<T*>(a.Crot);
    const long long ang_idx = ((long long)b * a.nheads + h) * half + k0 + kk;
    const int upr_log2 = a.kp_log2 - kPpvLog2;  // vector units per (step, rank) row
    const int gn = a.ngroups * a.dstate, hn = a.nheads * a.dstate;  // one (step, rank) row

    // A unit is PPV pairs of one (step, rank) row of the tile; with row =
    // step * rank + r its B / C offset is row * gn + 2 q from the tile's base
    // and its rotated offset row * hn + 2 q, so no division by rank is needed
    // except for the step index of its (cos, sin).
    struct Unit {
        int row, q, rot, ob, od;
    };
    auto unit = [&](int u) {
        Unit x;
        x.row = u >> upr_log2;
        x.q = (u & ((1 << upr_log2) - 1)) << kPpvLog2;
        const int i = a.rank == 1 ? x.row : x.row / a.rank;
        x.rot = i * kp + x.q;
        x.ob = x.row * gn + 2 * x.q;
        x.od = x.row * hn + 2 * x.q;
        return x;
    };
    Unit pu[PF];
#pragma unroll
    for (int j = 0; j < PF; ++j) pu[j] = unit(tid + j * kThreads);

    // offsets of the current tile's first row: B / C (group g), rotated (head
    // h), theta (head h, pair k0) and dt (head h)
    const long long bt0 = (long long)b * a.seqlen;
    long long base_bc = bt0 * a.rank * gn + (long long)g * a.dstate + 2 * k0;
    long long base_out = bt0 * a.rank * hn + (long long)h * a.dstate + 2 * k0;
    long long base_th = (bt0 * a.nheads + h) * half + k0;
    long long base_dt = bt0 * a.nheads + h;
    const long long step_bc = (long long)tile_steps * a.rank * gn;
    const long long step_out = (long long)tile_steps * a.rank * hn;
    const long long step_th = (long long)tile_steps * a.nheads * half;
    const long long step_dt = (long long)tile_steps * a.nheads;

    if (tid < kp) carry_s[tid] = make_float2((a.angle0 && kvalid) ? a.angle0[ang_idx] : 0.0f, 0.0f);
    ThetaRegs<TV4> th;
    th.init(a, k0, half, tid);
    th.fetch(a, base_th, base_dt, min(tile_steps, a.seqlen));
    th.put(w_s, tid);

    for (int t0 = 0; t0 < a.seqlen; t0 += tile_steps) {
        const int tn = min(tile_steps, a.seqlen - t0);
        const int nrows = tn * a.rank;
        // loads issued ahead: this tile's first B / C units, the next tile's theta
        typename V::W pb[PF], pc[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            if (pu[j].row < nrows && k0 + pu[j].q < half) {
                pb[j] = V::load(Bm + base_bc + pu[j].ob);
                pc[j] = V::load(Cm + base_bc + pu[j].ob);
            }
        }
        const bool more = t0 + tile_steps < a.seqlen;
        if (more)
            th.fetch(a, base_th + step_th, base_dt + step_dt,
                     min(tile_steps, a.seqlen - t0 - tile_steps));
        __syncthreads();  // the tile's w and carry are in shared memory

        // segmented compensated cumsum of w along the steps
        const float* wcol = w_s + seg * kSegSteps * kp + kk;
        float wv[kSegSteps];
#pragma unroll
        for (int j = 0; j < kSegSteps; ++j) wv[j] = wcol[j * kp];
        float shi = 0.0f, slo = 0.0f;
#pragma unroll
        for (int j = 0; j < kSegSteps; ++j) comp_add(shi, slo, wv[j]);
        agg_s[tid] = make_float2(shi, slo);
        const float2 cin = carry_s[kk];
        __syncthreads();
        float phi = cin.x, plo = cin.y;  // the angle before this thread's segment
        for (int s2 = 0; s2 < seg; ++s2) {
            const float2 ag = agg_s[(s2 << a.kp_log2) + kk];
            ff_add(phi, plo, ag.x, ag.y);
        }
        float2* rcol = rot_s + seg * kSegSteps * kp + kk;
#pragma unroll
        for (int j = 0; j < kSegSteps; ++j) {
            comp_add(phi, plo, wv[j]);
            float sn, cs;
            Trig<T>::sincos(phi, plo, sn, cs);
            rcol[j * kp] = make_float2(cs, sn);
        }
        // the last segment's walk ends at the next tile's carry
        if (seg == nseg - 1) carry_s[kk] = make_float2(phi, plo);
        __syncthreads();  // cos / sin complete; w free for the next tile

        // rotate the tile's rows of B and C
#pragma unroll
        for (int j = 0; j < PF; ++j)
            if (pu[j].row < nrows && k0 + pu[j].q < half)
                V::rotate_store(pb[j], pc[j], rot_s + pu[j].rot, Br + base_out + pu[j].od,
                                Cr + base_out + pu[j].od);
        const int nunits = nrows << upr_log2;
        for (int u = tid + PF * kThreads; u < nunits; u += kThreads) {
            const Unit x = unit(u);
            if (k0 + x.q >= half) continue;
            V::rotate_store(V::load(Bm + base_bc + x.ob), V::load(Cm + base_bc + x.ob),
                            rot_s + x.rot, Br + base_out + x.od, Cr + base_out + x.od);
        }
        if (more) th.put(w_s, tid);
        base_bc += step_bc;
        base_out += step_out;
        base_th += step_th;
        base_dt += step_dt;
        __syncthreads();  // rot_s read, the next tile's w written
    }
    if (a.angle_out && kvalid && tid < kp) {
        const float2 c = carry_s[kk];
        a.angle_out[ang_idx] = c.x + c.y;
    }
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

    // pairs per CTA: the smallest power of two covering the state pairs, at most 64
    int kp_log2 = 0;
    while ((1 << kp_log2) < (int)half && kp_log2 < kMaxPairsLog2) ++kp_log2;
    const int kblocks = (int)((half + (1u << kp_log2) - 1) >> kp_log2);
    const size_t blocks = (size_t)batch * nheads * kblocks;
    if (blocks > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    // offsets within one tile are kept in int
    const size_t tile_steps = (size_t)(kThreads >> kp_log2) * kSegSteps;
    if (tile_steps * rank * nheads * dstate > (size_t)INT32_MAX) return SSM_ERR_UNSUPPORTED;
    // 16-byte units of B and C when a row holds whole units (the base pointers
    // are 16-byte aligned above), and float4 rows of theta likewise
    const size_t ppv = 16 / (2 * es);
    const bool vec = half % ppv == 0;
    const bool theta_v4 = half % 4 == 0;
    RopeArgs a{B, C, dt, theta, angle0, B_rot, C_rot, angle_out,
               batch, seqlen, rank, nheads, ngroups, dstate, kp_log2, kblocks};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned grid = (unsigned)blocks;
    auto launch = [&](auto kernel) { kernel<<<grid, kThreads, 0, s>>>(a); };
    if (dtype == SSM_BF16) {
        if (vec) theta_v4 ? launch(rope_kernel<__nv_bfloat16, 4, true>)
                          : launch(rope_kernel<__nv_bfloat16, 4, false>);
        else theta_v4 ? launch(rope_kernel<__nv_bfloat16, 1, true>)
                      : launch(rope_kernel<__nv_bfloat16, 1, false>);
    } else {
        if (vec) theta_v4 ? launch(rope_kernel<float, 2, true>)
                          : launch(rope_kernel<float, 2, false>);
        else theta_v4 ? launch(rope_kernel<float, 1, true>)
                      : launch(rope_kernel<float, 1, false>);
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
