// api.cu -- entry points of the C ABI that are not tied to one kernel:
// version, status strings, the device-status read-back, and the host-side
// tensor-map encoder used by the TMA kernels.
#include <mutex>

#include "common.cuh"

namespace ssm_host {

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, ssm_dtype_t dtype, uint64_t rows,
                  uint64_t cols, uint32_t box_rows, uint32_t box_cols, bool swizzle) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * dtype_size(dtype)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace ssm_host

extern "C" int ssm_abi_version(void) { return 4; }

extern "C" const char* ssm_status_string(ssm_status_t s) {
    switch (s) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "required pointer is NULL";
        case SSM_ERR_SHAPE: return "invalid or inconsistent size";
        case SSM_ERR_ALIGN: return "pointer not 16-byte aligned";
        case SSM_ERR_DTYPE: return "unknown dtype";
        case SSM_ERR_UNSUPPORTED: return "size not implemented by this library";
        case SSM_ERR_WORKSPACE: return "workspace missing or too small";
        case SSM_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case SSM_ERR_CUDA: return "CUDA runtime error";
        case SSM_ERR_ALIAS: return "an output overlaps an input";
    }
    return "unknown status";
}

// The scan workspace starts with this header (see scan.cu).
extern "C" ssm_status_t ssm_last_device_status(const void* workspace, void* stream) {
    if (!workspace) return SSM_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t hdr[2] = {0, 0};
    if (cudaMemcpyAsync(hdr, workspace, sizeof(hdr), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
    return hdr[1] == 0 ? SSM_OK : static_cast<ssm_status_t>(hdr[1]);
}
