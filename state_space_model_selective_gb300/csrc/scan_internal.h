// scan_internal.h -- entry points shared between the library's translation
// units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

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

// ssm_scan_fwd (validation included) for one piece of a problem scanned in
// pieces (a range of its channels): path forces the kernel (0: planned for
// this piece, 1: the chained scan, 2: the sequence-parallel scan) and seg_ts
// the sequence-parallel path's segments per chunk (0: planned), so that every
// piece runs exactly as it would inside the whole problem's call; keep_status
// leaves the workspace's status word as the previous piece left it, so that a
// timeout in any piece stays visible.
ssm_status_t scan_forward_segment(const void* u, const void* delta, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* delta_bias, int delta_softplus,
                                  const float* initial_state, void* y, float* final_state,
                                  int batch, int dim, int seqlen, int ngroups,
                                  ssm_dtype_t in_dtype, ssm_dtype_t out_dtype, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream, int seg_ts,
                                  bool keep_status, int path);

// Whether ssm_scan_fwd takes the sequence-parallel path for this many channels.
bool scan_uses_seg_path(long long batch, long long dim);

// ---- the sequence-parallel path (scan_seg.cu)

// Problems with at most this many channels (batch * dim) may take the
// sequence-parallel path: split into 128-step chunks and in-warp segments,
// combined with the associative operator and a decoupled look-back.  Above
// it the channels fill the GPU and the work-efficient chained scan is used.
constexpr long long kScanSegMaxChannels = 3072;

bool scan_seg_eligible(long long batch, long long dim);

// Workspace of the sequence-parallel path (header, flags, aggregates and
// inclusive states of every chunk).
size_t scan_seg_workspace_bytes(int batch, int dim, int seqlen, int ngroups);

// Segments per 128-step chunk the sequence-parallel path would use (8, 16 or
// 32) on the current device.
int scan_seg_plan_ts(long long batch, long long dim, int seqlen);

// The sequence-parallel forward.  Arguments are validated by the caller;
// workspace holds scan_seg_workspace_bytes; spin_limit bounds each look-back;
// drop_first_publish (a test hook) makes chunk 0 withhold its inclusive state;
// ts: segments per chunk (8, 16, 32; anything else: planned); keep_status:
// leave the workspace's status word as an earlier call left it.
ssm_status_t scan_seg_forward(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int delta_softplus,
                              const float* initial_state, void* y, float* final_state, int batch,
                              int dim, int seqlen, int ngroups, ssm_dtype_t in_dtype,
                              ssm_dtype_t out_dtype, void* workspace, uint32_t spin_limit,
                              int drop_first_publish, int ts, bool keep_status,
                              cudaStream_t stream);

// Test hook: force the segments per chunk (8, 16 or 32; 0 = planned).
void scan_seg_debug_force_ts(int ts);

}  // namespace ssm_internal
