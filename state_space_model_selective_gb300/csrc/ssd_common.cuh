// ssd_common.cuh -- pieces shared by the chunked SSD's forward (ssd.cu) and
// backward (ssd_bwd.cu) kernels: bf16 hi/lo splitting of fp32 operands,
// operand descriptors of the 128-byte-swizzled tiles, the TMEM column map of a
// split operand, and the TMA maps of the (batch, seqlen, ...) tensors.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace ssd_detail {

using namespace ssm;

constexpr int kQ = 128;   // steps per block (MMA M)
constexpr int kP = 64;    // headdim
constexpr int kNs = 128;  // dstate

// Two fp32 values rounded to nearest-even bf16 and packed (a in the low half),
// one conversion instruction.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// (a, b) = hi + lo with hi = bf16(v), lo = bf16(v - hi) (about 16 significant
// bits in all), returned as the packed hi pair and the packed lo pair.
__device__ __forceinline__ void split2_bf16(float a, float b, uint32_t& hp, uint32_t& lp) {
    hp = pack_bf16(a, b);
    lp = pack_bf16(a - bf16lo(hp), b - bf16hi(hp));
}

// K-major operand descriptor for k-step kk (16 bf16) of a tile with R rows.
template <int R>
__device__ __forceinline__ uint64_t kdesc(uint32_t tile_saddr, int kk) {
    return smem_desc_k128(tile_saddr + (uint32_t)((kk >> 2) * (R * 128) + (kk & 3) * 32));
}

// MN-major operand descriptor for k-step kk of a tile of 128-byte rows (one
// row per k); 64-wide MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t mdesc(uint32_t tile_saddr, int kk, uint32_t lbo) {
    return smem_desc_mn128(tile_saddr + (uint32_t)kk * 2048u, lbo);
}

// TMEM column of a split operand (hi part) for k-step kk: a row's 32-column
// chunk c is held as 16 packed hi columns followed by 16 lo columns, in place
// of the 32 fp32 columns it was computed from.
__device__ __forceinline__ uint32_t mcol_hi(int kk) {
    return (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1));
}

}  // namespace ssd_detail

namespace ssd_host {

// (batch, seqlen, ngroups, dstate) bf16 as a 4-D map {dstate, ngroups, seqlen,
// batch} with 64 x 1 x 128 x 1 boxes (128-byte swizzle).
inline bool make_bc_map(CUtensorMap* map, const void* base, int batch, int seqlen, int ngroups) {
    using ssd_detail::kNs;
    using ssd_detail::kQ;
    ssm_host::EncodeTiledFn fn = ssm_host::encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kNs, (cuuint64_t)ngroups, (cuuint64_t)seqlen,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)kNs * 2, (cuuint64_t)ngroups * kNs * 2,
                                   (cuuint64_t)seqlen * ngroups * kNs * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// (batch, seqlen, nheads, headdim) bf16 as a 3-D map {nheads * headdim,
// seqlen, batch} with 64 x 128 x 1 boxes (128-byte swizzle).
inline bool make_x_map(CUtensorMap* map, const void* base, int batch, int seqlen, int nheads) {
    using ssd_detail::kP;
    using ssd_detail::kQ;
    ssm_host::EncodeTiledFn fn = ssm_host::encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)nheads * kP, (cuuint64_t)seqlen, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)nheads * kP * 2,
                                   (cuuint64_t)seqlen * nheads * kP * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kP, (cuuint32_t)kQ, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// y (batch, seqlen, nheads, headdim) in fp32 or bf16 as a 3-D map {nheads *
// headdim, seqlen, batch} whose boxes are one 128-byte row span (32 fp32 or 64
// bf16 columns) x 128 steps x 1 (128-byte swizzle), the layout the forward
// kernel stages y in; stores clip at the sequence end.
inline bool make_y_map(CUtensorMap* map, void* base, int batch, int seqlen, int nheads,
                       ssm_dtype_t dtype) {
    using ssd_detail::kP;
    using ssd_detail::kQ;
    ssm_host::EncodeTiledFn fn = ssm_host::encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t es = dtype == SSM_BF16 ? 2 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)nheads * kP, (cuuint64_t)seqlen, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)nheads * kP * es,
                                   (cuuint64_t)seqlen * nheads * kP * es};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)kQ, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
              3, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ssd_host
