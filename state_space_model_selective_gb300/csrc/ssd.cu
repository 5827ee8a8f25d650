// ssd.cu -- chunked SSD forward (ssd_chunked_fwd) for GB300 / sm_103a.
#include "common.cuh"

extern "C" ssm_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A_head,
                                        const void* B, const void* C, int chunk, void* y,
                                        float* final_state, int batch, int seqlen, int nheads,
                                        int headdim, int dstate, int ngroups,
                                        ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                        void* stream) {
    using namespace ssm_host;
    (void)stream;
    if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1 || ngroups < 1 ||
        chunk < 1)
        return SSM_ERR_SHAPE;
    if (nheads % ngroups != 0 || seqlen % chunk != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    if (chunk != 64 || headdim != 64 || dstate != 128 || in_dtype != SSM_BF16)
        return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * seqlen;
    if (rows == 0 || nheads == 0) return SSM_OK;
    if (!x || !dt || !A_head || !B || !C || !y) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A_head, B, C, y, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t xb = rows * nheads * headdim * 2, yb = rows * nheads * headdim * dtype_size(out_dtype);
    const size_t bcb = rows * ngroups * dstate * 2;
    const size_t fb = final_state ? (size_t)batch * nheads * headdim * dstate * 4 : 0;
    struct R { const void* p; size_t n; } ins[] = {
        {x, xb}, {dt, rows * nheads * 4}, {A_head, (size_t)nheads * 4}, {B, bcb}, {C, bcb}};
    for (const R& r : ins)
        if (overlaps(y, yb, r.p, r.n) || overlaps(final_state, fb, r.p, r.n)) return SSM_ERR_ALIAS;
    if (overlaps(y, yb, final_state, fb)) return SSM_ERR_ALIAS;
    return SSM_ERR_UNSUPPORTED;  // kernel not built yet
}
