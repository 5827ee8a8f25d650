// scan.cu -- selective scan forward (ssm_scan_fwd) for GB300 / sm_103a.
//
// What it computes: "We brought Mamba to Trainium -- and mapped where custom
// kernels actually help", section "Mamba: bringing an unsupported model to the
// chip, and writing its missing kernel" (h_t = A_t h_{t-1} + B_t x_t,
// y_t = sum_n C_t h_t, state kept on chip for the whole sequence), with the
// discretisation and epilogue of "Mamba-3 NKI Kernels for AWS Neuron",
// section "How it works" (Phase 0: dt = softplus(dt + dt_bias),
// alpha = exp(dt A); Phase 5: D skip, then silu gate).
//
// How (work-efficient: every (b, l, d, n) element costs one exp and four
// fp32 operations, nothing is recomputed):
//  * A CTA owns one (batch, group, block of CH channels) and one L-chunk.
//    Four lanes share a channel; each holds 4 of the 16 states in registers
//    and walks the chunk's time steps in order.
//  * A producer warp streams 64-step tiles of u, delta, z, B and C into a
//    ring of shared-memory stages with 2-D TMA (128-byte swizzle), tracked
//    by mbarriers.  The compute warps first "prep" each group of 16 or 64
//    steps of a tile once per (channel, step) -- dl = softplus(delta + bias)
//    and dl*u -- then run the group's recurrence, reading B and C from the
//    tile's fp32 [t][state group] rows.
//  * y partial sums over the 4 lanes' states are reduce-scattered with warp
//    shuffles; each lane then finishes 2 of every 8 steps (D skip, silu gate)
//    and stores them.
//  * Consecutive L-chunks of one channel block are chained across CTAs: CTA
//    order is a ticket taken at start (chunk-major), and a CTA reads its
//    carried-in state from the predecessor chunk's published inclusive state
//    (bounded wait, acquire/release flags).  A predecessor always holds an
//    earlier ticket, so it is running or finished: the wait always ends.
//    The associativity of the recurrence ("We built the parallel scan"
//    section of the first page) is what makes the chunk split exact.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "scan_internal.h"

namespace {

using namespace ssm;

constexpr int kN = 16;          // dstate
constexpr int kSPT = 4;         // states per thread
constexpr int kNG = kN / kSPT;  // threads per channel
constexpr int kTL = 64;         // time steps per tile
constexpr int kMaxChunks = 32;  // upper bound on L-chunks per channel block
// Steps prepped at a time (PS): 16 (a quarter of a tile, so that four CTAs'
// shared memory fits on an SM) or 64 (the whole tile, three CTAs).
__host__ __device__ constexpr int prep_stride(int ps) { return ps * 8 + 16; }  // bytes per channel row

struct alignas(16) WsHeader {
    uint32_t ticket;
    uint32_t status;
    uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

struct ScanArgs {
    const void* u;
    const void* delta;
    const void* z;
    const float* A;
    const float* Dskip;
    const float* bias;
    const float* h0;
    void* y;
    float* final_state;
    uint32_t* ticket;
    uint32_t* status;
    uint32_t* flags;  // [nchunks - 1][nblocks]
    float* carry;     // [nchunks - 1][batch * dim][kN]
    const void* Bm;
    const void* Cm;
    // checkpoint mode (kernel flag CK = 1, or 2 without the read-out): the
    // state entering every 16-step segment, [seg][batch * dim][kN] (the
    // backward pass recomputes from these); y is then optional
    float* ckpt;
    int batch, dim, seqlen, ngroups;
    int dpg;          // channels per group
    int bpg;          // channel blocks per group
    int nblocks;      // batch * ngroups * bpg
    int nchunks;
    int chunk_tiles;  // tiles per chunk
    int softplus;
    uint32_t flag_spin_limit;  // look-back polls before SSM_ERR_TIMEOUT
    int drop_first_publish;    // test hook: chunk 0 never publishes its carry
};

// Byte offset of (row r, step t) in a tile of ROWS rows x kTL steps laid out
// as the 128-byte-swizzled TMA boxes: boxes of 128 bytes per row along time,
// the 16-byte chunk index XORed with (row mod 8).
template <typename T, int ROWS>
__device__ __forceinline__ int tile_off(int r, int t) {
    constexpr int E = sizeof(T);
    constexpr int TPB = 128 / E;
    const int box = t / TPB;
    const int byte = (t % TPB) * E;
    return box * (ROWS * 128) + r * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15));
}

// Byte offset of (row r, step t) in the same boxes without the swizzle (the
// B and C tiles: every lane of a quarter-warp reads one address, so there
// are no bank conflicts to spread, and the offsets stay affine in t).
template <typename T, int ROWS>
__device__ __forceinline__ int tile_off_lin(int r, int t) {
    constexpr int E = sizeof(T);
    constexpr int TPB = 128 / E;
    return (t / TPB) * (ROWS * 128) + r * 128 + (t % TPB) * E;
}

// 8 consecutive steps t0..t0+7 (t0 % 8 == 0) of row r, as fp32.
template <typename T, int ROWS>
__device__ __forceinline__ void load8(const uint8_t* tile, int r, int t0, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(tile + tile_off<T, ROWS>(r, t0));
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
    } else {
        const float4 a = *reinterpret_cast<const float4*>(tile + tile_off<T, ROWS>(r, t0));
        const float4 b = *reinterpret_cast<const float4*>(tile + tile_off<T, ROWS>(r, t0 + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// 4 consecutive steps t0..t0+3 (t0 % 4 == 0) of row r, as fp32.
template <typename T, int ROWS>
__device__ __forceinline__ void load4s(const uint8_t* tile, int r, int t0, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(tile + tile_off<T, ROWS>(r, t0));
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    } else {
        const float4 a = *reinterpret_cast<const float4*>(tile + tile_off<T, ROWS>(r, t0));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
}

// 8 consecutive steps t0..t0+7 (t0 % 8 == 0) of row n of an unswizzled
// B or C tile, as fp32.
template <typename T>
__device__ __forceinline__ void row8_lin(const uint8_t* tile, int n, int t0, float* v) {
    if constexpr (sizeof(T) == 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(tile + tile_off_lin<T, kN>(n, t0));
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
    } else {
        const float4 x = *reinterpret_cast<const float4*>(tile + tile_off_lin<T, kN>(n, t0));
        const float4 y = *reinterpret_cast<const float4*>(tile + tile_off_lin<T, kN>(n, t0 + 4));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    }
}

// In-place conversion, by one warp (lane pl), of a stage's B and C tiles
// ([n][t] in the input type, B then C from the region's start) into fp32 rows
// [t][group g][B[4g..4g+3], C[4g..4g+3]] of 128 bytes per step.  Every lane
// reads its values before any lane writes.
template <typename T>
__device__ __forceinline__ void convert_bc(uint8_t* region, int pl) {
    constexpr int BC_TILE = kN * kTL * (int)sizeof(T);
    const int g = pl & 3, blk = pl >> 2;  // states 4g..4g+3, steps 8 blk..8 blk+7
    float vb[4][8], vc[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        row8_lin<T>(region, 4 * g + k, 8 * blk, vb[k]);
        row8_lin<T>(region + BC_TILE, 4 * g + k, 8 * blk, vc[k]);
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        float4* dst = reinterpret_cast<float4*>(region + (8 * blk + s) * 128 + g * 32);
        dst[0] = make_float4(vb[0][s], vb[1][s], vb[2][s], vb[3][s]);
        dst[1] = make_float4(vc[0][s], vc[1][s], vc[2][s], vc[3][s]);
    }
}

// B and C of one tile straight into the fp32 [t][group] rows, with plain
// loads and bounds checks (rows not 16-byte aligned for TMA).
template <typename T>
__device__ __forceinline__ void stage_bc_plain(uint8_t* region, const T* Bm, const T* Cm,
                                               long long row0, int L, int t0, int tid,
                                               int nthreads) {
    for (int i = tid; i < kN * kTL; i += nthreads) {
        const int n = i / kTL, t = i % kTL;
        const int tg = t0 + t;
        float vb = 0.0f, vc = 0.0f;
        if (tg < L) {
            vb = to_f32(Bm[(row0 + n) * (long long)L + tg]);
            vc = to_f32(Cm[(row0 + n) * (long long)L + tg]);
        }
        float* dst = reinterpret_cast<float*>(region + t * 128 + (n / 4) * 32) + (n % 4);
        dst[0] = vb;
        dst[4] = vc;
    }
}

// Fallback staging when the rows are not 16-byte aligned for TMA: plain
// loads with bounds checks into the same swizzled layout.
template <typename T, int ROWS>
__device__ __forceinline__ void stage_plain(uint8_t* tile, const T* src, long long row0,
                                            long long rows_total, int L, int t0, int tid,
                                            int nthreads) {
    for (int i = tid; i < ROWS * kTL; i += nthreads) {
        const int r = i / kTL, t = i % kTL;
        const long long row = row0 + r;
        const int tg = t0 + t;
        T v = from_f32<T>(0.0f);
        if (row < rows_total && tg < L) v = src[row * (long long)L + tg];
        *reinterpret_cast<T*>(tile + tile_off<T, ROWS>(r, t)) = v;
    }
}

template <typename T>
__device__ __forceinline__ void store_y2(T* p, float a, float b, bool ok0, bool ok1, bool vec) {
    if (vec && ok1) {
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float2*>(p) = make_float2(a, b);
        } else {
            __nv_bfloat162 v;
            v.x = __float2bfloat16_rn(a);
            v.y = __float2bfloat16_rn(b);
            *reinterpret_cast<__nv_bfloat162*>(p) = v;
        }
    } else {
        if (ok0) p[0] = from_f32<T>(a);
        if (ok1) p[1] = from_f32<T>(b);
    }
}

template <typename Tin>
struct Geom {
    static constexpr int E = sizeof(Tin);
    static constexpr int TPB = 128 / E;       // steps per 128-byte box row
    static constexpr int NBOX = kTL / TPB;    // boxes per tile along time
    static constexpr int kStages = 2;
};

template <typename Tin, int CH, bool TMA, int PS>
struct Smem {
    static constexpr int E = sizeof(Tin);
    static constexpr int IN_TILE = CH * kTL * E;
    static constexpr int BC_TILE = kN * kTL * E;
    // B and C of a tile as fp32 [t][4 state groups][B 4 states, C 4 states];
    // the TMA tiles of B and C land in its front half and are converted in place
    static constexpr int BCF = kTL * kN * 2 * 4;
    static_assert(2 * BC_TILE <= BCF, "the B/C tiles fit the converted region");
    static constexpr int STAGE = 3 * IN_TILE + BCF;
    static constexpr int NSTAGE = TMA ? Geom<Tin>::kStages : 1;
    static constexpr int PREP = 2 * CH * prep_stride(PS);  // (dl, dl*u) and (u, silu(z))
    static constexpr int BARS = 3 * NSTAGE * 8 + 16;
    static constexpr int BYTES = NSTAGE * STAGE + PREP + BARS;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
};

template <typename Tin, typename Tout, int CH, bool TMA, int CK, int PS>
__global__ void __launch_bounds__(CH * kNG + 32, PS == 16 ? 4 : 3)
    scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_d,
                    const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_C, const ScanArgs a) {
    using S = Smem<Tin, CH, TMA, PS>;
    using G = Geom<Tin>;
    constexpr int NCOMP = CH * kNG;
    constexpr int kPrepStride = prep_stride(PS);
    constexpr int LPS = PS / 4;  // steps a lane preps per group
    static_assert(PS == 16 || PS == 64, "prep groups of 16 or 64 steps");
    constexpr int NSTAGE = S::NSTAGE;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* stages = smem;
    uint8_t* prep = stages + NSTAGE * S::STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(prep + S::PREP);  // TMA bytes landed
    uint64_t* ready = full + NSTAGE;   // B/C converted: the tile can be used
    uint64_t* empty = ready + NSTAGE;  // the compute warps are done with the stage
    int* s_ticket = reinterpret_cast<int*>(empty + NSTAGE);

    const int tid = threadIdx.x;
    if (tid == 0) {
        *s_ticket = static_cast<int>(atomicAdd(a.ticket, 1u));
        if constexpr (TMA) {
            for (int s = 0; s < NSTAGE; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&ready[s], 1);
                mbar_init(&empty[s], NCOMP / 32);
            }
            fence_mbar_init();
        }
    }
    __syncthreads();

    const int ticket = *s_ticket;
    const int chunk = ticket / a.nblocks;
    const int blk = ticket % a.nblocks;
    const int cb = blk % a.bpg;
    const int bg = blk / a.bpg;  // b * ngroups + g
    const int g = bg % a.ngroups;
    const int b = bg / a.ngroups;
    const int d0 = g * a.dpg + cb * CH;
    const long long row0 = static_cast<long long>(b) * a.dim + d0;
    const long long bcrow0 = static_cast<long long>(bg) * kN;
    const int t_begin = chunk * a.chunk_tiles * kTL;
    const int t_end = min(a.seqlen, t_begin + a.chunk_tiles * kTL);
    const int ntiles = (t_end - t_begin + kTL - 1) / kTL;
    const bool has_z = a.z != nullptr;

    // ------------------------------------------------------------ producer
    // One warp: lane 0 issues the TMA loads of each tile; once a tile has
    // landed the whole warp converts its B and C to the fp32 [t][n] layout
    // the recurrence reads (while the compute warps work on the previous
    // tile), then releases it on `ready`.
    if (tid >= NCOMP) {
        if constexpr (TMA) {
            const int pl = tid - NCOMP;
            if (pl == 0) {
                prefetch_tensormap(&tm_u);
                prefetch_tensormap(&tm_d);
                if (has_z) prefetch_tensormap(&tm_z);
                prefetch_tensormap(&tm_B);
                prefetch_tensormap(&tm_C);
            }
            const uint32_t bytes = (has_z ? 3 : 2) * S::IN_TILE + 2 * S::BC_TILE;
            auto issue = [&](int k) {
                const int s = k % NSTAGE;
                mbar_arrive_expect_tx(&full[s], bytes);
                uint8_t* st = stages + s * S::STAGE;
                const int t0 = t_begin + k * kTL;
#pragma unroll
                for (int bx = 0; bx < G::NBOX; ++bx) {
                    const int tc = t0 + bx * G::TPB;
                    tma_load_2d(st + bx * CH * 128, &tm_u, &full[s], tc, (int)row0);
                    tma_load_2d(st + S::IN_TILE + bx * CH * 128, &tm_d, &full[s], tc, (int)row0);
                    if (has_z)
                        tma_load_2d(st + 2 * S::IN_TILE + bx * CH * 128, &tm_z, &full[s], tc,
                                    (int)row0);
                    tma_load_2d(st + 3 * S::IN_TILE + bx * kN * 128, &tm_B, &full[s], tc,
                                (int)bcrow0);
                    tma_load_2d(st + 3 * S::IN_TILE + S::BC_TILE + bx * kN * 128, &tm_C,
                                &full[s], tc, (int)bcrow0);
                }
            };
            // tile k lands, is converted and published; its stage is reloaded
            // with tile k + NSTAGE once the compute warps have released it.
            auto land = [&](int k) -> bool {
                const int s = k % NSTAGE;
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / NSTAGE) & 1, a.status)))
                    return false;
                convert_bc<Tin>(stages + s * S::STAGE + 3 * S::IN_TILE, pl);
                fence_proxy_async_smem();  // before the stage's next TMA writes
                __syncwarp();
                if (pl == 0) mbar_arrive(&ready[s]);
                return true;
            };
            const int pro = min(NSTAGE, ntiles);
            if (pl == 0)
                for (int k = 0; k < pro; ++k) issue(k);
            int issued = pro, landed = 0;
            bool alive = ntiles > 0 && land(0);
            if (alive) landed = 1;
            for (int k = 0; alive && k < ntiles; ++k) {
                if (k + 1 < ntiles) {
                    if (!(alive = land(k + 1))) break;
                    landed = k + 2;
                }
                const int kn = k + NSTAGE;
                if (kn < ntiles) {
                    const int s = k % NSTAGE;
                    if (!(alive = __all_sync(0xffffffffu,
                                             mbar_wait(&empty[s], ((kn / NSTAGE) & 1) ^ 1,
                                                       a.status))))
                        break;
                    if (pl == 0) issue(kn);
                    issued = kn + 1;
                }
            }
            // Never leave the CTA with copies still landing in its shared
            // memory: wait (bounded) for every stage issued but not waited on.
            for (int k = landed; k < issued; ++k)
                mbar_wait(&full[k % NSTAGE], (k / NSTAGE) & 1, a.status);
        }
        return;
    }

    // ------------------------------------------------------------- compute
    const int warp = tid >> 5, lane = tid & 31;
    // lanes l, l + 8, l + 16, l + 24 share a channel; a quarter-warp (the
    // unit a 16-byte shared load serves at once) holds 8 channels with the
    // same four states, so every B/C load it makes is one broadcast address
    const int cl = warp * 8 + (lane & 7);  // channel within the block
    const int ng = lane >> 3;              // which 4 of the 16 states
    const int n0 = ng * kSPT;
    const int d = d0 + cl;
    const bool valid = (cb * CH + cl) < a.dpg;
    const long long drow = static_cast<long long>(b) * a.dim + d;

    float A2[kSPT], h[kSPT];
#pragma unroll
    for (int k = 0; k < kSPT; ++k) {
        A2[k] = valid ? a.A[static_cast<long long>(d) * kN + n0 + k] * kLog2e : 0.0f;
        h[k] = 0.0f;
    }

    // prep mapping: each warp preps its own 8 channels (lane: channel cl,
    // steps 16 pq .. 16 pq + 15), so a tile needs no barrier across warps
    const int pq = ng;
    const float pbias = (a.bias && valid) ? a.bias[d] : 0.0f;
    const float pD = (a.Dskip && valid) ? a.Dskip[d] : 0.0f;

    // prep tile rows: [CH][kTL] (dl, dl*u) pairs, then [CH][kTL] (u, g)
    // pairs, g = silu(z) (1 without a gate)
    const float* prow = reinterpret_cast<const float*>(prep + cl * kPrepStride);
    const float* prow2 = reinterpret_cast<const float*>(prep + (CH + cl) * kPrepStride);
    Tout* yrow = reinterpret_cast<Tout*>(a.y) + drow * a.seqlen;
    // vector stores need the row start aligned to 2 elements; TMA implies it
    const bool vec_store = TMA;

    bool ok = true;
    for (int k = 0; k < ntiles; ++k) {
        const int s = k % NSTAGE;
        uint8_t* st = stages + s * S::STAGE;
        const int t0 = t_begin + k * kTL;

        if constexpr (TMA) {
            const bool got = mbar_wait(&full[s], (k / NSTAGE) & 1, a.status);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        } else {
            stage_plain<Tin, CH>(st, reinterpret_cast<const Tin*>(a.u), row0,
                                 (long long)a.batch * a.dim, a.seqlen, t0, tid, NCOMP);
            stage_plain<Tin, CH>(st + S::IN_TILE, reinterpret_cast<const Tin*>(a.delta), row0,
                                 (long long)a.batch * a.dim, a.seqlen, t0, tid, NCOMP);
            if (has_z)
                stage_plain<Tin, CH>(st + 2 * S::IN_TILE, reinterpret_cast<const Tin*>(a.z),
                                     row0, (long long)a.batch * a.dim, a.seqlen, t0, tid, NCOMP);
            stage_bc_plain<Tin>(st + 3 * S::IN_TILE, reinterpret_cast<const Tin*>(a.Bm),
                                reinterpret_cast<const Tin*>(a.Cm), bcrow0, a.seqlen, t0, tid,
                                NCOMP);
            named_bar_sync(1, NCOMP);
        }

        // The tile runs in groups of PS steps: each warp preps its own 8
        // channels for the group (lane: channel cl, steps LPS pq .. LPS pq +
        // LPS - 1), then runs the group's 8-step recurrence blocks.  Only one
        // group's prep rows are held at a time.
        const uint8_t* tBC = st + 3 * S::IN_TILE + ng * 32;
        for (int qt = 0; qt < kTL / PS && ok; ++qt) {
            // ---- prep, once per (channel, step): dl = softplus(delta + bias)
            // (or delta + bias), dl * u, and the read-out's u and silu(z);
            // steps past the chunk end get dl = 0, an exact identity step
            // (exp(0) = 1, input term 0).
            constexpr int CS = LPS >= 8 ? 8 : 4;  // steps per chunk (one 16- or 8-byte load)
#pragma unroll
            for (int c = 0; c < LPS / CS; ++c) {
                const int tq = pq * LPS + c * CS;  // step within the group
                const int tl = qt * PS + tq;       // step within the tile
                float uv[CS], dv[CS], zv[CS];
                if constexpr (CS == 8) {
                    load8<Tin, CH>(st, cl, tl, uv);
                    load8<Tin, CH>(st + S::IN_TILE, cl, tl, dv);
                    if (has_z) load8<Tin, CH>(st + 2 * S::IN_TILE, cl, tl, zv);
                } else {
                    load4s<Tin, CH>(st, cl, tl, uv);
                    load4s<Tin, CH>(st + S::IN_TILE, cl, tl, dv);
                    if (has_z) load4s<Tin, CH>(st + 2 * S::IN_TILE, cl, tl, zv);
                }
                float o[2 * CS], e[2 * CS];
#pragma unroll
                for (int j = 0; j < CS; ++j) {
                    const float x = dv[j] + pbias;
                    const float dl = a.softplus ? softplus_f(x) : x;
                    o[2 * j] = dl;
                    o[2 * j + 1] = dl * uv[j];
                    if constexpr (CK != 2) {
                        e[2 * j] = uv[j];  // the read-out adds D u with one FMA
                        e[2 * j + 1] = has_z ? silu_f(zv[j]) : 1.0f;
                    }
                }
                // only the tile that runs past the sequence end (uniform over
                // the CTA) has steps to neutralise
                if (t0 + kTL > t_end) {
#pragma unroll
                    for (int j = 0; j < CS; ++j)
                        if (t0 + tl + j >= t_end) o[2 * j] = o[2 * j + 1] = 0.0f;
                }
                float4* dst = reinterpret_cast<float4*>(prep + cl * kPrepStride + tq * 8);
                float4* dst2 = reinterpret_cast<float4*>(prep + (CH + cl) * kPrepStride + tq * 8);
#pragma unroll
                for (int j = 0; j < CS / 2; ++j) {
                    dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                    if constexpr (CK != 2)
                        dst2[j] = make_float4(e[4 * j], e[4 * j + 1], e[4 * j + 2], e[4 * j + 3]);
                }
            }
            __syncwarp();

            if (qt == 0) {
                // ---- carried-in state, once per CTA, after the first prep
                if (k == 0) {
                    if (chunk == 0) {
                        if (a.h0 && valid) {
                            const float4 v =
                                *reinterpret_cast<const float4*>(a.h0 + drow * kN + n0);
                            h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
                        }
                    } else {
                        const uint32_t* flag = a.flags + (size_t)(chunk - 1) * a.nblocks + blk;
                        if (lane == 0) {
                            bool seen = false;
                            uint32_t ns = 32;
                            for (uint32_t it = 0; it < a.flag_spin_limit; ++it) {
                                if (ld_acquire_gpu(flag)) { seen = true; break; }
                                __nanosleep(ns);
                                ns = ns < 256 ? ns * 2 : 256;
                            }
                            if (!seen) record_status(a.status, SSM_ERR_TIMEOUT);
                        }
                        __syncwarp();
                        (void)ld_acquire_gpu(flag);  // order this thread's reads after the flag
                        if (valid) {
                            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                a.carry + ((size_t)(chunk - 1) * a.batch * a.dim + drow) * kN + n0));
                            h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
                        }
                    }
                }
                // ---- B and C from the stage's fp32 [t][state group] rows (one
                // broadcast address per quarter-warp), once the producer has
                // converted them
                if constexpr (TMA) {
                    const bool got = mbar_wait(&ready[s], (k / NSTAGE) & 1, a.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                }
            }

            // ---- the recurrence over the group, 8 steps per block (unrolled by
            // 4 blocks at most: further unrolling measured slower)
            constexpr int kUnroll = PS / 8 < 4 ? PS / 8 : 4;
#pragma unroll kUnroll
            for (int jj = 0; jj < PS / 8; ++jj) {
                const int j = qt * (PS / 8) + jj;  // 8-step block within the tile
                if (CK != 0 && (j & 1) == 0 && valid && t0 + j * 8 < a.seqlen) {
                    const long long seg = (t0 + j * 8) / 16;
                    __stcg(reinterpret_cast<float4*>(
                               a.ckpt + (seg * a.batch * a.dim + drow) * kN + n0),
                           make_float4(h[0], h[1], h[2], h[3]));
                }
                float yp[8];
#pragma unroll
                for (int q = 0; q < 8; q += 2) {
                    const float4 pp = *reinterpret_cast<const float4*>(prow + (jj * 8 + q) * 2);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int t = j * 8 + q + r;
                        const float dl = r ? pp.z : pp.x;
                        const float du = r ? pp.w : pp.y;
                        const float4 bv = *reinterpret_cast<const float4*>(tBC + t * 128);
                        h[0] = fmaf(ex2_approx(dl * A2[0]), h[0], du * bv.x);
                        h[1] = fmaf(ex2_approx(dl * A2[1]), h[1], du * bv.y);
                        h[2] = fmaf(ex2_approx(dl * A2[2]), h[2], du * bv.z);
                        h[3] = fmaf(ex2_approx(dl * A2[3]), h[3], du * bv.w);
                        if constexpr (CK != 2) {
                            const float4 cv = *reinterpret_cast<const float4*>(tBC + t * 128 + 16);
                            float acc = cv.x * h[0];
                            acc = fmaf(cv.y, h[1], acc);
                            acc = fmaf(cv.z, h[2], acc);
                            acc = fmaf(cv.w, h[3], acc);
                            yp[q + r] = acc;
                        }
                    }
                }
                if constexpr (CK == 2) continue;  // states only: no read-out
                // reduce-scatter the 8 partial sums over the 4 lanes of the channel
                // (lane bits 3 and 4): afterwards lane ng holds the full sums of
                // steps 2ng and 2ng+1, added as (p0 + p2) + (p1 + p3).
                float f[2];
                const bool hi2 = ng & 2, hi1 = ng & 1;
                float k4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = hi2 ? yp[i] : yp[i + 4];
                    const float keep = hi2 ? yp[i + 4] : yp[i];
                    k4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = hi1 ? k4[i] : k4[i + 2];
                    const float keep = hi1 ? k4[i + 2] : k4[i];
                    f[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                const int tq = jj * 8 + 2 * ng;  // step within the group
                const int tg = t0 + j * 8 + 2 * ng;
                const float4 eg = *reinterpret_cast<const float4*>(prow2 + tq * 2);
                const float o0 = fmaf(pD, eg.x, f[0]) * eg.y;
                const float o1 = fmaf(pD, eg.z, f[1]) * eg.w;
                if ((CK == 0 || a.y) && valid && tg < t_end)
                    store_y2<Tout>(yrow + tg, o0, o1, true, tg + 1 < t_end, vec_store);
            }
            __syncwarp();  // this warp's prep rows are rewritten by the next group
        }
        if (!ok) break;

        if constexpr (TMA) {
            if (lane == 0) mbar_arrive(&empty[s]);
        } else {
            named_bar_sync(1, NCOMP);  // the single stage is restaged next
        }
    }

    // ---- outgoing state: final_state for the last chunk, else the carry
    if (valid && ok) {
        const float4 v = make_float4(h[0], h[1], h[2], h[3]);
        if (chunk == a.nchunks - 1) {
            if (a.final_state)
                *reinterpret_cast<float4*>(a.final_state + drow * kN + n0) = v;
        } else {
            __stcg(reinterpret_cast<float4*>(
                       a.carry + ((size_t)chunk * a.batch * a.dim + drow) * kN + n0),
                   v);
        }
    }
    if (chunk < a.nchunks - 1) {
        __threadfence();
        named_bar_sync(1, NCOMP);
        if (tid == 0 && !(a.drop_first_publish && chunk == 0))
            st_release_gpu(a.flags + (size_t)chunk * a.nblocks + blk, 1u);
    }
}

// ------------------------------------------------------------------ host

// Look-back settings of every scan launch, set by ssm_debug_set_lookback:
// the poll limit (0: kFlagSpinLimit) and whether chunk 0 withholds its
// publish, so that a test can watch the bounded wait run out.
std::atomic<uint32_t> g_flag_spin_limit{0};
std::atomic<int> g_drop_first_publish{0};

struct Plan {
    int CH;
    int ps;  // steps prepped at a time: 16 (four CTAs per SM) or 64 (three)
    int bpg, nblocks, nchunks, chunk_tiles;
    bool tma;
};

struct DevInfo {
    int sms = 0;
};

DevInfo dev_info() {
    static std::mutex m;
    static int cached_dev = -1;
    static DevInfo info;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(m);
    if (dev != cached_dev) {
        cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
        if (info.sms <= 0) info.sms = 1;
        cached_dev = dev;
    }
    return info;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace is sized for the largest plan any device could pick, so that
// ssm_scan_workspace_bytes is a pure function of the problem.
size_t chained_workspace_bound(long long batch, long long dim, int seqlen, int ngroups) {
    const long long dpg = dim / ngroups;
    const long long max_blocks = batch * ngroups * ((dpg + 15) / 16);
    const long long tiles = (seqlen + kTL - 1) / kTL;
    const long long max_chunks = std::min<long long>(kMaxChunks, std::max<long long>(1, tiles));
    size_t bytes = sizeof(WsHeader);
    bytes += round256(sizeof(uint32_t) * (size_t)(max_chunks - 1) * (size_t)max_blocks);
    bytes += (size_t)(max_chunks - 1) * (size_t)batch * (size_t)dim * kN * sizeof(float);
    return round256(bytes);
}

// Which forward path runs (ssm_debug_set_scan_path): 0 planned, 1 the chained
// scan, 2 the sequence-parallel scan (only for problems eligible for it).
std::atomic<int> g_scan_path{0};

bool use_seg_path(long long batch, long long dim) {
    if (!ssm_internal::scan_seg_eligible(batch, dim)) return false;
    return g_scan_path.load(std::memory_order_relaxed) != 1;
}

size_t workspace_bound(long long batch, long long dim, int seqlen, int ngroups) {
    size_t bytes = chained_workspace_bound(batch, dim, seqlen, ngroups);
    if (ssm_internal::scan_seg_eligible(batch, dim))
        bytes = std::max(bytes, ssm_internal::scan_seg_workspace_bytes(
                                    (int)batch, (int)dim, seqlen, ngroups));
    return bytes;
}

template <typename Tin, typename Tout, int CH, bool TMA, int CK, int PS>
int occupancy_blocks() {
    using S = Smem<Tin, CH, TMA, PS>;
    static int cached = -1;
    if (cached < 0) {
        auto kern = scan_fwd_kernel<Tin, Tout, CH, TMA, CK, PS>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
        int nb = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, CH * kNG + 32, S::ALLOC);
        cached = std::max(nb, 1);
    }
    return cached;
}

template <typename Tin, typename Tout, int CH, bool TMA, int CK, int PS>
ssm_status_t launch(const ScanArgs& base, const Plan& p, const CUtensorMap* maps,
                    cudaStream_t stream) {
    using S = Smem<Tin, CH, TMA, PS>;
    auto kern = scan_fwd_kernel<Tin, Tout, CH, TMA, CK, PS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    ScanArgs a = base;
    const uint32_t lim = g_flag_spin_limit.load(std::memory_order_relaxed);
    a.flag_spin_limit = lim ? lim : kFlagSpinLimit;
    a.drop_first_publish = g_drop_first_publish.load(std::memory_order_relaxed);
    a.bpg = p.bpg;
    a.nblocks = p.nblocks;
    a.nchunks = p.nchunks;
    a.chunk_tiles = p.chunk_tiles;
    const unsigned grid = (unsigned)p.nblocks * (unsigned)p.nchunks;
    kern<<<grid, CH * kNG + 32, S::ALLOC, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                     a);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

template <typename Tin, typename Tout, int CH, bool TMA, int CK, int PS>
void plan_for(const ScanArgs& a, Plan& p) {
    p.CH = CH;
    p.ps = PS;
    p.tma = TMA;
    p.bpg = (a.dpg + CH - 1) / CH;
    p.nblocks = a.batch * a.ngroups * p.bpg;
    const int tiles = (a.seqlen + kTL - 1) / kTL;
    const long long slots =
        (long long)occupancy_blocks<Tin, Tout, CH, TMA, CK, PS>() * dev_info().sms;
    int nchunks = 1;
    if (p.nblocks >= slots) {
        // Enough independent channel blocks to fill the GPU: cut L into
        // chained chunks so that about 8 waves of CTAs balance the SMs.
        const long long want = (8 * slots + p.nblocks - 1) / p.nblocks;
        nchunks = (int)std::min<long long>(std::min<long long>(want, kMaxChunks), tiles);
        nchunks = std::max(nchunks, 1);
    }
    p.chunk_tiles = (tiles + nchunks - 1) / nchunks;
    p.nchunks = (tiles + p.chunk_tiles - 1) / p.chunk_tiles;
}

// The variant with 16-step prep groups holds four CTAs per SM; it runs when the
// channel blocks fill four on every SM (the larger problems, where the extra
// warps hide latency: batch 4, L 16384, 5120 channels in 1.84 ms against 1.92
// with the whole-tile prep).  Otherwise the whole-tile prep at three CTAs per
// SM, which does less work per step (batch 8, L 2048, 1536 channels: 176 us
// against 180 with 16-step groups).
template <typename Tin, typename Tout, bool TMA, int CK>
void choose_plan_tma(const ScanArgs& a, Plan& p) {
    plan_for<Tin, Tout, 32, TMA, CK, 16>(a, p);
    const long long slots16 =
        (long long)occupancy_blocks<Tin, Tout, 32, TMA, CK, 16>() * dev_info().sms;
    if (p.nblocks < slots16) plan_for<Tin, Tout, 32, TMA, CK, 64>(a, p);
}

template <typename Tin, typename Tout, int CK>
void choose_plan(const ScanArgs& a, bool tma, Plan& p) {
    if (tma) choose_plan_tma<Tin, Tout, true, CK>(a, p);
    else choose_plan_tma<Tin, Tout, false, CK>(a, p);
}

template <typename Tin, typename Tout, int CK = 0>
ssm_status_t dispatch(ScanArgs& a, ssm_dtype_t in_dtype, bool tma, cudaStream_t stream,
                      void* workspace, bool keep_status = false) {
    Plan p{};
    choose_plan<Tin, Tout, CK>(a, tma, p);

    // workspace: header | flags | carry
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    a.ticket = &hdr->ticket;
    a.status = &hdr->status;
    a.flags = reinterpret_cast<uint32_t*>(ws + sizeof(WsHeader));
    const size_t flag_bytes = round256(sizeof(uint32_t) * (size_t)(p.nchunks - 1) * p.nblocks);
    a.carry = reinterpret_cast<float*>(ws + sizeof(WsHeader) + flag_bytes);
    // the ticket, the status word (unless an earlier call's status is being
    // accumulated) and the flags start at zero
    if (keep_status) {
        if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream) != cudaSuccess ||
            cudaMemsetAsync(ws + 2 * sizeof(uint32_t), 0,
                            sizeof(WsHeader) - 2 * sizeof(uint32_t) + flag_bytes,
                            stream) != cudaSuccess)
            return SSM_ERR_CUDA;
    } else if (cudaMemsetAsync(ws, 0, sizeof(WsHeader) + flag_bytes, stream) != cudaSuccess) {
        return SSM_ERR_CUDA;
    }

    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (tma) {
        const uint64_t rows = (uint64_t)a.batch * a.dim;
        const uint64_t bcrows = (uint64_t)a.batch * a.ngroups * kN;
        const uint32_t tpb = Geom<Tin>::TPB;
        bool okm = ssm_host::make_tmap_2d(&maps[0], a.u, in_dtype, rows, a.seqlen, 32, tpb) &&
                   ssm_host::make_tmap_2d(&maps[1], a.delta, in_dtype, rows, a.seqlen, 32, tpb) &&
                   ssm_host::make_tmap_2d(&maps[3], a.Bm, in_dtype, bcrows, a.seqlen, kN, tpb,
                                          false) &&
                   ssm_host::make_tmap_2d(&maps[4], a.Cm, in_dtype, bcrows, a.seqlen, kN, tpb,
                                          false);
        if (okm && a.z)
            okm = ssm_host::make_tmap_2d(&maps[2], a.z, in_dtype, rows, a.seqlen, 32, tpb);
        if (!okm) return SSM_ERR_CUDA;
        return p.ps == 16 ? launch<Tin, Tout, 32, true, CK, 16>(a, p, maps, stream)
                          : launch<Tin, Tout, 32, true, CK, 64>(a, p, maps, stream);
    }
    return p.ps == 16 ? launch<Tin, Tout, 32, false, CK, 16>(a, p, maps, stream)
                      : launch<Tin, Tout, 32, false, CK, 64>(a, p, maps, stream);
}

}  // namespace

namespace ssm_internal {

size_t scan_forward_workspace_bytes(int batch, int dim, int seqlen, int ngroups) {
    return workspace_bound(batch, dim, seqlen, ngroups);
}

// The forward recurrence writing only the state entering every 16-step
// segment (ckpt [ceil(seqlen/16)][batch * dim][16]); no y, no final state.
// Arguments are validated by the caller; workspace holds
// scan_forward_workspace_bytes.
ssm_status_t scan_forward_checkpoints(const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, const float* delta_bias,
                                      int delta_softplus, const float* h0, float* ckpt,
                                      int batch, int dim, int seqlen, int ngroups,
                                      ssm_dtype_t in_dtype, void* workspace,
                                      cudaStream_t stream) {
    ScanArgs a{};
    a.u = u; a.delta = delta; a.z = nullptr; a.A = A; a.Dskip = nullptr; a.bias = delta_bias;
    a.h0 = h0; a.y = nullptr; a.final_state = nullptr; a.Bm = B; a.Cm = C; a.ckpt = ckpt;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.ngroups = ngroups;
    a.dpg = dim / ngroups; a.softplus = delta_softplus ? 1 : 0;
    const size_t es = in_dtype == SSM_BF16 ? 2 : 4;
    const bool tma = ((size_t)seqlen * es) % 16 == 0;
    if (in_dtype == SSM_BF16)
        return dispatch<__nv_bfloat16, float, 2>(a, in_dtype, tma, stream, workspace);
    return dispatch<float, float, 2>(a, in_dtype, tma, stream, workspace);
}

}  // namespace ssm_internal

extern "C" size_t ssm_scan_workspace_bytes(int batch, int dim, int seqlen, int dstate,
                                           int ngroups) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate != kN || ngroups < 1 || dim % ngroups)
        return 0;
    return workspace_bound(batch, dim, seqlen, ngroups);
}

namespace {

// ssm_scan_fwd, and with ckpt != NULL ssm_scan_fwd_ckpt: validation and launch.
ssm_status_t scan_fwd_entry(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z, const float* delta_bias,
                            int delta_softplus, const float* initial_state, void* y,
                            float* final_state, float* ckpt, int batch, int dim, int seqlen,
                            int dstate, int ngroups, ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                            void* workspace, size_t workspace_bytes, void* stream,
                            int seg_ts = 0, bool keep_status = false, int force_path = 0) {
    using namespace ssm_host;
    if (batch < 0 || dim < 0 || seqlen < 0 || ngroups < 1 || dstate < 1) return SSM_ERR_SHAPE;
    if (dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    if (dstate != kN) return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * dim;
    if (rows == 0) return SSM_OK;
    // TMA coordinates and CTA counts are 32-bit
    if (rows > (size_t)INT32_MAX || (size_t)batch * ngroups * kN > (size_t)INT32_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y || !A)) return SSM_ERR_NULL;
    if (seqlen > 0 && !workspace) return SSM_ERR_WORKSPACE;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state,
                          workspace, ckpt};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;

    const size_t es = dtype_size(in_dtype), eo = dtype_size(out_dtype);
    const size_t act = rows * (size_t)seqlen * es;
    const size_t bc = (size_t)batch * ngroups * kN * (size_t)seqlen * es;
    struct R { const void* p; size_t n; } ins[] = {
        {u, act}, {delta, act}, {z, z ? act : 0}, {B, bc}, {C, bc}, {A, (size_t)dim * kN * 4},
        {D, D ? (size_t)dim * 4 : 0}, {delta_bias, delta_bias ? (size_t)dim * 4 : 0},
        {initial_state, initial_state ? rows * kN * 4 : 0}};
    const size_t ybytes = rows * (size_t)seqlen * eo;
    const size_t fbytes = final_state ? rows * kN * 4 : 0;
    for (const R& r : ins) {
        if (overlaps(y, ybytes, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(final_state, fbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, ybytes, final_state, fbytes)) return SSM_ERR_ALIAS;
    const size_t cbytes = ckpt ? ((size_t)seqlen + 15) / 16 * rows * kN * 4 : 0;
    for (const R& r : ins)
        if (overlaps(ckpt, cbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    if (overlaps(ckpt, cbytes, y, ybytes) || overlaps(ckpt, cbytes, final_state, fbytes))
        return SSM_ERR_ALIAS;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (seqlen == 0) {
        if (final_state) {
            cudaError_t e = initial_state
                                ? cudaMemcpyAsync(final_state, initial_state, rows * kN * 4,
                                                  cudaMemcpyDeviceToDevice, s)
                                : cudaMemsetAsync(final_state, 0, rows * kN * 4, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const size_t need = workspace_bound(batch, dim, seqlen, ngroups);
    if (workspace_bytes < need) return SSM_ERR_WORKSPACE;
    if (overlaps(workspace, need, y, ybytes) || overlaps(workspace, need, final_state, fbytes) ||
        overlaps(workspace, need, ckpt, cbytes))
        return SSM_ERR_ALIAS;
    for (const R& r : ins)
        if (overlaps(workspace, need, r.p, r.n)) return SSM_ERR_ALIAS;

    if (force_path == 2 && !ssm_internal::scan_seg_eligible(batch, dim)) return SSM_ERR_UNSUPPORTED;
    const bool seg = force_path == 2 || (force_path == 0 && use_seg_path(batch, dim));
    if (seg) {
        const uint32_t lim = g_flag_spin_limit.load(std::memory_order_relaxed);
        const ssm_status_t st = ssm_internal::scan_seg_forward(
            u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state, y, final_state,
            batch, dim, seqlen, ngroups, in_dtype, out_dtype, workspace,
            lim ? lim : kFlagSpinLimit, g_drop_first_publish.load(std::memory_order_relaxed),
            seg_ts, keep_status, s);
        if (st != SSM_OK || !ckpt) return st;
        // the checkpoints from the chained scan's states-only pass; y and
        // final_state stay the sequence-parallel scan's, as ssm_scan_fwd gives
        ScanArgs c{};
        c.u = u; c.delta = delta; c.z = nullptr; c.A = A; c.Dskip = nullptr; c.bias = delta_bias;
        c.h0 = initial_state; c.y = nullptr; c.final_state = nullptr; c.Bm = B; c.Cm = C;
        c.ckpt = ckpt; c.batch = batch; c.dim = dim; c.seqlen = seqlen; c.ngroups = ngroups;
        c.dpg = dim / ngroups; c.softplus = delta_softplus ? 1 : 0;
        const bool tma_c = ((size_t)seqlen * es) % 16 == 0;
        return in_dtype == SSM_BF16
                   ? dispatch<__nv_bfloat16, float, 2>(c, in_dtype, tma_c, s, workspace, true)
                   : dispatch<float, float, 2>(c, in_dtype, tma_c, s, workspace, true);
    }

    ScanArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.A = A; a.Dskip = D; a.bias = delta_bias;
    a.h0 = initial_state; a.y = y; a.final_state = final_state; a.Bm = B; a.Cm = C; a.ckpt = ckpt;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.ngroups = ngroups;
    a.dpg = dim / ngroups; a.softplus = delta_softplus ? 1 : 0;

    // TMA needs 16-byte row strides (base alignment is already checked).
    const bool tma = ((size_t)seqlen * es) % 16 == 0;
    if (in_dtype == SSM_BF16) {
        return out_dtype == SSM_BF16
                   ? (ckpt ? dispatch<__nv_bfloat16, __nv_bfloat16, true>(a, in_dtype, tma, s, workspace, keep_status)
                           : dispatch<__nv_bfloat16, __nv_bfloat16>(a, in_dtype, tma, s, workspace, keep_status))
                   : (ckpt ? dispatch<__nv_bfloat16, float, true>(a, in_dtype, tma, s, workspace, keep_status)
                           : dispatch<__nv_bfloat16, float>(a, in_dtype, tma, s, workspace, keep_status));
    }
    if (out_dtype == SSM_BF16)
        return ckpt ? dispatch<float, __nv_bfloat16, true>(a, in_dtype, tma, s, workspace, keep_status)
                    : dispatch<float, __nv_bfloat16>(a, in_dtype, tma, s, workspace, keep_status);
    return ckpt ? dispatch<float, float, true>(a, in_dtype, tma, s, workspace, keep_status)
                : dispatch<float, float>(a, in_dtype, tma, s, workspace, keep_status);
}

}  // namespace

namespace ssm_internal {

ssm_status_t scan_forward_segment(const void* u, const void* delta, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus,
                                  const float* initial_state, void* y, float* final_state,
                                  int batch, int dim, int seqlen, int ngroups,
                                  ssm_dtype_t in_dtype, ssm_dtype_t out_dtype, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream, int seg_ts,
                                  bool keep_status, int path) {
    return scan_fwd_entry(u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state, y,
                          final_state, nullptr, batch, dim, seqlen, kN, ngroups, in_dtype,
                          out_dtype, workspace, workspace_bytes, stream, seg_ts, keep_status,
                          path);
}

bool scan_uses_seg_path(long long batch, long long dim) { return use_seg_path(batch, dim); }

}  // namespace ssm_internal

extern "C" ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     const float* delta_bias, int delta_softplus,
                                     const float* initial_state, void* y, float* final_state,
                                     int batch, int dim, int seqlen, int dstate, int ngroups,
                                     ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    return scan_fwd_entry(u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state, y,
                          final_state, nullptr, batch, dim, seqlen, dstate, ngroups, in_dtype,
                          out_dtype, workspace, workspace_bytes, stream);
}

extern "C" size_t ssm_scan_checkpoint_bytes(int batch, int dim, int seqlen, int dstate) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate != kN) return 0;
    return ((size_t)seqlen + 15) / 16 * (size_t)batch * dim * kN * sizeof(float);
}

extern "C" ssm_status_t ssm_scan_fwd_ckpt(const void* u, const void* delta, const float* A,
                                          const void* B, const void* C, const float* D,
                                          const void* z, const float* delta_bias,
                                          int delta_softplus, const float* initial_state, void* y,
                                          float* final_state, float* checkpoints, int batch,
                                          int dim, int seqlen, int dstate, int ngroups,
                                          ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                          void* workspace, size_t workspace_bytes, void* stream) {
    if (!checkpoints && batch > 0 && dim > 0 && seqlen > 0) return SSM_ERR_NULL;
    return scan_fwd_entry(u, delta, A, B, C, D, z, delta_bias, delta_softplus, initial_state, y,
                          final_state, checkpoints, batch, dim, seqlen, dstate, ngroups, in_dtype,
                          out_dtype, workspace, workspace_bytes, stream);
}

// ------------------------------------------------ allocation-free variant
//
// ssm_scan_fwd_noalloc: the same scan kernel, with its look-back scratch
// (ticket, status word, per-chunk flags and carried states) taken from a
// fixed array in the library's device image instead of a caller-supplied
// workspace.  Every GPU that loads the library holds this array until the
// process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// cuCtxGetCurrent, fetched from the driver through the runtime (the library
// has no link-time dependency on libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol names a host-side shadow, not device memory, so the address is
// looked up with the device current (cudaGetSymbolAddress) and cached per
// device.  The cache is keyed by the device's current context too: after a
// cudaDeviceReset the device gets a new context, the library's module is
// loaded again at a new address, and the first call in the new context looks
// the address up again.
void* noalloc_scratch_address() {
    static std::mutex m;
    static void* addr[128] = {};
    static CUcontext ctx_of[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    CtxGetCurrentFn get = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lk(m);
    if (!ctx || !addr[dev] || ctx_of[dev] != ctx) {
        // the look-up also makes the device's primary context current when no
        // context was yet; the context is read again after it
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    return addr[dev];
}

// Scratch bytes the plan for this problem uses: header | flags | carry,
// exactly as dispatch() lays it out.
template <typename Tin, typename Tout>
size_t planned_scratch_bytes(const ScanArgs& a, bool tma) {
    Plan p{};
    choose_plan<Tin, Tout, 0>(a, tma, p);
    return sizeof(WsHeader) + round256(sizeof(uint32_t) * (size_t)(p.nchunks - 1) * p.nblocks) +
           (size_t)(p.nchunks - 1) * (size_t)a.batch * a.dim * kN * sizeof(float);
}

}  // namespace

extern "C" ssm_status_t ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                             const void* B, const void* C, const float* D,
                                             const void* z, const float* delta_bias,
                                             int delta_softplus, const float* initial_state,
                                             void* y, float* final_state, int batch, int dim,
                                             int seqlen, int dstate, int ngroups,
                                             ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                             void* stream) {
    using namespace ssm_host;
    if (batch < 0 || dim < 0 || seqlen < 0 || ngroups < 1 || dstate < 1) return SSM_ERR_SHAPE;
    if (dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    if (dstate != kN) return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * dim;
    if (rows == 0) return SSM_OK;
    if (rows > (size_t)INT32_MAX || (size_t)batch * ngroups * kN > (size_t)INT32_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y || !A)) return SSM_ERR_NULL;
    const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(in_dtype), eo = dtype_size(out_dtype);
    const size_t act = rows * (size_t)seqlen * es;
    const size_t bc = (size_t)batch * ngroups * kN * (size_t)seqlen * es;
    struct R { const void* p; size_t n; } ins[] = {
        {u, act}, {delta, act}, {z, z ? act : 0}, {B, bc}, {C, bc}, {A, (size_t)dim * kN * 4},
        {D, D ? (size_t)dim * 4 : 0}, {delta_bias, delta_bias ? (size_t)dim * 4 : 0},
        {initial_state, initial_state ? rows * kN * 4 : 0}};
    const size_t ybytes = rows * (size_t)seqlen * eo;
    const size_t fbytes = final_state ? rows * kN * 4 : 0;
    for (const R& r : ins) {
        if (overlaps(y, ybytes, r.p, r.n)) return SSM_ERR_ALIAS;
        if (overlaps(final_state, fbytes, r.p, r.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, ybytes, final_state, fbytes)) return SSM_ERR_ALIAS;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (seqlen == 0) {
        if (final_state) {
            cudaError_t e = initial_state
                                ? cudaMemcpyAsync(final_state, initial_state, rows * kN * 4,
                                                  cudaMemcpyDeviceToDevice, s)
                                : cudaMemsetAsync(final_state, 0, rows * kN * 4, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    void* scratch = noalloc_scratch_address();
    if (!scratch) return SSM_ERR_CUDA;

    if (use_seg_path(batch, dim)) {
        if (ssm_internal::scan_seg_workspace_bytes(batch, dim, seqlen, ngroups) >
            kNoAllocScratchBytes)
            return SSM_ERR_WORKSPACE;
        const uint32_t lim = g_flag_spin_limit.load(std::memory_order_relaxed);
        return ssm_internal::scan_seg_forward(u, delta, A, B, C, D, z, delta_bias,
                                              delta_softplus, initial_state, y, final_state,
                                              batch, dim, seqlen, ngroups, in_dtype, out_dtype,
                                              scratch, lim ? lim : kFlagSpinLimit,
                                              g_drop_first_publish.load(std::memory_order_relaxed),
                                              0, false, s);
    }

    ScanArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.A = A; a.Dskip = D; a.bias = delta_bias;
    a.h0 = initial_state; a.y = y; a.final_state = final_state; a.Bm = B; a.Cm = C;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.ngroups = ngroups;
    a.dpg = dim / ngroups; a.softplus = delta_softplus ? 1 : 0;
    const bool tma = ((size_t)seqlen * es) % 16 == 0;

    size_t need;
    if (in_dtype == SSM_BF16)
        need = out_dtype == SSM_BF16 ? planned_scratch_bytes<__nv_bfloat16, __nv_bfloat16>(a, tma)
                                     : planned_scratch_bytes<__nv_bfloat16, float>(a, tma);
    else
        need = out_dtype == SSM_BF16 ? planned_scratch_bytes<float, __nv_bfloat16>(a, tma)
                                     : planned_scratch_bytes<float, float>(a, tma);
    if (need > kNoAllocScratchBytes) return SSM_ERR_WORKSPACE;

    // dispatch() clears the header and flags on the stream before the launch;
    // the carried states need no clearing (each is written before it is read).
    if (in_dtype == SSM_BF16) {
        return out_dtype == SSM_BF16
                   ? dispatch<__nv_bfloat16, __nv_bfloat16>(a, in_dtype, tma, s, scratch)
                   : dispatch<__nv_bfloat16, float>(a, in_dtype, tma, s, scratch);
    }
    return out_dtype == SSM_BF16 ? dispatch<float, __nv_bfloat16>(a, in_dtype, tma, s, scratch)
                                 : dispatch<float, float>(a, in_dtype, tma, s, scratch);
}

extern "C" ssm_status_t ssm_noalloc_last_status(void* stream) {
    void* scratch = noalloc_scratch_address();
    if (!scratch) return SSM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word is the second 32-bit word of the scratch header, in
    // both scan paths' layouts; read into the host's stack (pageable)
    uint32_t hdr[2] = {0, 0};
    if (cudaMemcpyAsync(hdr, scratch, sizeof(hdr), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
    return hdr[1] == 0 ? SSM_OK : static_cast<ssm_status_t>(hdr[1]);
}

extern "C" ssm_status_t ssm_debug_set_scan_path(int path, int segments) {
    if (path < 0 || path > 2) return SSM_ERR_SHAPE;
    if (segments != 0 && segments != 8 && segments != 16 && segments != 32) return SSM_ERR_SHAPE;
    g_scan_path.store(path, std::memory_order_relaxed);
    ssm_internal::scan_seg_debug_force_ts(segments);
    return SSM_OK;
}

extern "C" ssm_status_t ssm_debug_set_lookback(int drop_first_publish, unsigned int spin_limit) {
    g_flag_spin_limit.store(spin_limit, std::memory_order_relaxed);
    g_drop_first_publish.store(drop_first_publish ? 1 : 0, std::memory_order_relaxed);
    return SSM_OK;
}
