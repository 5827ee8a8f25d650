// ssd_internal.h -- entry points shared between the library's translation
// units for the chunked SSD (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "ssm.h"

namespace ssd_internal {

// The chunked SSD forward writing only the state entering every 128-step
// block and the final state: bstates [batch * nheads][ceil(seqlen / 128) + 1]
// [64][128] fp32 (headdim 64, dstate 128, bf16 x, B, C).  No y.  Arguments are
// validated by the caller.
ssm_status_t ssd_forward_block_states(const void* x, const float* dt, const float* A_head,
                                      const void* B, const void* C, const float* initial_state,
                                      float* bstates, int batch, int seqlen, int nheads,
                                      int ngroups, cudaStream_t stream);

// The Mamba-3 forward (rank 1, 2 or 4; MIMO blocks are 128 rows of
// sub-tokens) writing only the states its chunked form carries between
// blocks: the state entering each block (with the pending dt_{t+1} (1 -
// lambda_{t+1}) BX_t of the step before, and the previous token's term in block
// 0) and the final state, laid out as above.  prev_B, prev_x (bf16) may both be
// NULL.  Arguments are validated by the caller.
ssm_status_t ssd_mamba3_forward_block_states(const void* x, const float* dt, const float* lam,
                                             const float* A_head, const void* B, const void* C,
                                             const float* initial_state, const void* prev_B,
                                             const void* prev_x, float* bstates, int batch,
                                             int seqlen, int nheads, int ngroups,
                                             cudaStream_t stream, int rank = 1);

}  // namespace ssd_internal
