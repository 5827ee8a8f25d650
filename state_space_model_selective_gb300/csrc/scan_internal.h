// scan_internal.h -- entry points shared between the library's translation
// units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "ssm.h"

namespace ssm_internal {

// Workspace of one forward scan (look-back flags and carried states).
size_t scan_forward_workspace_bytes(int batch, int dim, int seqlen, int ngroups);

// The forward recurrence writing only the state entering every 16-step
// segment: ckpt [ceil(seqlen / 16)][batch * dim][16] fp32.  No y, no final
// state.  Arguments are validated by the caller.
ssm_status_t scan_forward_checkpoints(const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, const float* delta_bias,
                                      int delta_softplus, const float* h0, float* ckpt,
                                      int batch, int dim, int seqlen, int ngroups,
                                      ssm_dtype_t in_dtype, void* workspace,
                                      cudaStream_t stream);

}  // namespace ssm_internal
