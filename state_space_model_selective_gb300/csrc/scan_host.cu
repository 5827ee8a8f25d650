// scan_host.cu -- the selective scan on host-resident activations
// (ssm_scan_fwd_host): host -> device copies, the scan and device -> host copies
// pipelined over segments of the sequence.
//
// What it computes is exactly ssm_scan_fwd's ("We brought Mamba to Trainium --
// and mapped where custom kernels actually help", section "Mamba: bringing an
// unsupported model to the chip, and writing its missing kernel"), with the
// sequence cut into segments that chain through the state: scanning [t0, t1)
// from the state after t0 equals the whole scan restricted to [t0, t1) (the
// associativity of the recurrence, section "We built the parallel scan -- and
// it taught us something sharper").
//
// How: segment k's rows of u, delta, z, B, C (strided in the host layout) are
// copied with 2-D DMA copies on a copy stream into one of two device slots; the
// caller's stream runs ssm_scan_fwd on the slot with the previous segment's
// final state; a second copy stream brings y's rows back.  Copies in both
// directions run on the copy engines while the SMs scan the neighbouring
// segments.  The two copy streams and the events are created once per device
// and kept for the life of the process.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "scan_internal.h"

namespace {

using namespace ssm_host;

constexpr int kN = 16;
constexpr int kSlots = 2;

struct Plan {
    int seg;       // steps per segment (all but the last)
    int nseg;      // segments
    size_t act_in, bc_in, act_out;  // bytes of one slot's u (and delta, z), B (and C), y
    size_t state;                   // bytes of one state (batch * dim * 16 fp32)
    size_t scan_ws;                 // bytes of ssm_scan_fwd's workspace (one segment)
    size_t slot, total;
};

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

Plan plan_for(int batch, int dim, int seqlen, int ngroups, size_t es, size_t eo) {
    Plan p{};
    // about eight segments, each a multiple of 128 steps (16-byte rows for
    // TMA, and the sequence-parallel scan's chunk boundaries where the whole
    // sequence's scan has them)
    const int want = (seqlen + 7) / 8;
    p.seg = std::max(128, (want + 127) / 128 * 128);
    p.seg = std::min(p.seg, std::max(seqlen, 1));
    p.nseg = seqlen > 0 ? (seqlen + p.seg - 1) / p.seg : 0;
    const size_t rows = (size_t)batch * dim, bcrows = (size_t)batch * ngroups * kN;
    p.act_in = r256(rows * p.seg * es);
    p.bc_in = r256(bcrows * p.seg * es);
    p.act_out = r256(rows * p.seg * eo);
    p.state = r256(rows * kN * 4);
    p.scan_ws = r256(ssm_scan_workspace_bytes(batch, dim, p.seg, kN, ngroups));
    p.slot = 3 * p.act_in + 2 * p.bc_in + p.act_out;
    // scan workspace first (ssm_last_device_status reads its header), then the
    // two slots and the two states (a segment's initial and final state)
    p.total = p.scan_ws + kSlots * p.slot + 2 * p.state;
    return p;
}

struct DeviceQueues {
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t ev_in[kSlots], ev_comp[kSlots], ev_out[kSlots], ev_done;
    bool ok = false;
};

// Copy streams and events of the current device, created on first use.
DeviceQueues* queues(std::mutex*& lock) {
    static std::mutex m;
    static DeviceQueues q[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    lock = &m;
    std::lock_guard<std::mutex> lk(m);
    DeviceQueues& d = q[dev];
    if (!d.ok) {
        bool good = cudaStreamCreateWithFlags(&d.copy_in, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&d.copy_out, cudaStreamNonBlocking) == cudaSuccess;
        for (int s = 0; good && s < kSlots; ++s)
            good = cudaEventCreateWithFlags(&d.ev_in[s], cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventCreateWithFlags(&d.ev_comp[s], cudaEventDisableTiming) == cudaSuccess &&
                   cudaEventCreateWithFlags(&d.ev_out[s], cudaEventDisableTiming) == cudaSuccess;
        good = good && cudaEventCreateWithFlags(&d.ev_done, cudaEventDisableTiming) == cudaSuccess;
        if (!good) return nullptr;
        d.ok = true;
    }
    return &d;
}

// Host memory the copy engines can reach asynchronously: page-locked (pinned)
// or registered with CUDA.
bool is_pinned(const void* p) {
    if (!p) return true;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

bool is_device(const void* p) {
    if (!p) return true;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" size_t ssm_scan_fwd_host_workspace_bytes(int batch, int dim, int seqlen, int dstate,
                                                    int ngroups, ssm_dtype_t in_dtype,
                                                    ssm_dtype_t out_dtype) {
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate != kN || ngroups < 1 || dim % ngroups ||
        !dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return 0;
    return plan_for(batch, dim, seqlen, ngroups, dtype_size(in_dtype), dtype_size(out_dtype)).total;
}

extern "C" ssm_status_t ssm_scan_fwd_host(const void* u, const void* delta, const float* A,
                                          const void* B, const void* C, const float* D,
                                          const void* z, const float* delta_bias,
                                          int delta_softplus, const float* initial_state,
                                          void* y, float* final_state, int batch, int dim,
                                          int seqlen, int dstate, int ngroups,
                                          ssm_dtype_t in_dtype, ssm_dtype_t out_dtype,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream) {
    if (batch < 0 || dim < 0 || seqlen < 0 || ngroups < 1 || dstate < 1) return SSM_ERR_SHAPE;
    if (dim % ngroups != 0) return SSM_ERR_SHAPE;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return SSM_ERR_DTYPE;
    if (dstate != kN) return SSM_ERR_UNSUPPORTED;
    const size_t rows = (size_t)batch * dim;
    if (rows == 0) return SSM_OK;
    if (rows > (size_t)INT32_MAX || (size_t)batch * ngroups * kN > (size_t)INT32_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (!A || !workspace) return !A ? SSM_ERR_NULL : SSM_ERR_WORKSPACE;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return SSM_ERR_NULL;
    const void* dev_ptrs[] = {A, D, delta_bias, workspace};
    for (const void* p : dev_ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    const size_t es = dtype_size(in_dtype), eo = dtype_size(out_dtype);
    const Plan pl = plan_for(batch, dim, seqlen, ngroups, es, eo);
    if (workspace_bytes < pl.total) return SSM_ERR_WORKSPACE;
    // where each pointer lives: activations and results on the host (page-locked),
    // parameters and workspace on the device
    const void* host_ptrs[] = {u, delta, z, B, C, initial_state, y, final_state};
    for (const void* p : host_ptrs)
        if (!is_pinned(p)) return SSM_ERR_UNSUPPORTED;
    for (const void* p : dev_ptrs)
        if (!is_device(p)) return SSM_ERR_UNSUPPORTED;

    std::mutex* lock = nullptr;
    DeviceQueues* q = queues(lock);
    if (!q) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(*lock);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* scan_ws = ws;
    auto slot_base = [&](int k) { return ws + pl.scan_ws + (size_t)(k % kSlots) * pl.slot; };
    float* fsb[2] = {reinterpret_cast<float*>(ws + pl.scan_ws + kSlots * pl.slot),
                     reinterpret_cast<float*>(ws + pl.scan_ws + kSlots * pl.slot + pl.state)};
    const size_t sbytes = rows * kN * 4;
    bool ok = true;
    auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };

    // the copy streams start after the caller's earlier work (which may still use
    // this workspace)
    chk(cudaEventRecord(q->ev_done, s));
    chk(cudaStreamWaitEvent(q->copy_in, q->ev_done, 0));
    chk(cudaStreamWaitEvent(q->copy_out, q->ev_done, 0));
    if (initial_state) chk(cudaMemcpyAsync(fsb[1], initial_state, sbytes, cudaMemcpyHostToDevice, s));
    if (seqlen == 0) {
        if (final_state) {
            if (!initial_state) chk(cudaMemsetAsync(fsb[1], 0, sbytes, s));
            chk(cudaMemcpyAsync(final_state, fsb[1], sbytes, cudaMemcpyDeviceToHost, s));
        }
        return ok ? SSM_OK : SSM_ERR_CUDA;
    }
    const size_t L = (size_t)seqlen, bcrows = (size_t)batch * ngroups * kN;
    const int seg_ts = ssm_internal::scan_seg_plan_ts(batch, dim, seqlen);
    ssm_status_t rc = SSM_OK;
    for (int k = 0; k < pl.nseg && ok && rc == SSM_OK; ++k) {
        const int sl = k % kSlots;
        const size_t t0 = (size_t)k * pl.seg;
        const size_t Lk = std::min((size_t)pl.seg, L - t0);
        uint8_t* base = slot_base(k);
        uint8_t* du = base;
        uint8_t* dd = du + pl.act_in;
        uint8_t* dz = dd + pl.act_in;
        uint8_t* dB = dz + pl.act_in;
        uint8_t* dC = dB + pl.bc_in;
        uint8_t* dy = dC + pl.bc_in;
        // segment k's inputs into the slot, once the scan two segments back is done with it
        if (k >= kSlots) chk(cudaStreamWaitEvent(q->copy_in, q->ev_comp[sl], 0));
        auto in2d = [&](void* dst, const void* src, size_t nrows) {
            chk(cudaMemcpy2DAsync(dst, Lk * es, static_cast<const uint8_t*>(src) + t0 * es, L * es,
                                  Lk * es, nrows, cudaMemcpyHostToDevice, q->copy_in));
        };
        in2d(du, u, rows);
        in2d(dd, delta, rows);
        if (z) in2d(dz, z, rows);
        in2d(dB, B, bcrows);
        in2d(dC, C, bcrows);
        chk(cudaEventRecord(q->ev_in[sl], q->copy_in));
        // the scan of segment k on the caller's stream, from the previous state
        chk(cudaStreamWaitEvent(s, q->ev_in[sl], 0));
        if (k >= kSlots) chk(cudaStreamWaitEvent(s, q->ev_out[sl], 0));
        if (!ok) break;
        const float* st_in = k == 0 ? (initial_state ? fsb[1] : nullptr) : fsb[(k - 1) % 2];
        // every segment with the whole sequence's plan; the status word keeps
        // the first timeout of any segment
        rc = ssm_internal::scan_forward_segment(
            du, dd, A, dB, dC, D, z ? dz : nullptr, delta_bias, delta_softplus, st_in, dy,
            fsb[k % 2], batch, dim, (int)Lk, ngroups, in_dtype, out_dtype, scan_ws, pl.scan_ws, s,
            seg_ts, k > 0);
        chk(cudaEventRecord(q->ev_comp[sl], s));
        // segment k's y back to the host
        chk(cudaStreamWaitEvent(q->copy_out, q->ev_comp[sl], 0));
        chk(cudaMemcpy2DAsync(static_cast<uint8_t*>(y) + t0 * eo, L * eo, dy, Lk * eo, Lk * eo, rows,
                              cudaMemcpyDeviceToHost, q->copy_out));
        chk(cudaEventRecord(q->ev_out[sl], q->copy_out));
    }
    if (ok && rc == SSM_OK && final_state)
        chk(cudaMemcpyAsync(final_state, fsb[(pl.nseg - 1) % 2], sbytes, cudaMemcpyDeviceToHost,
                            q->copy_out));
    // the caller's stream completes after every copy of this call
    chk(cudaEventRecord(q->ev_done, q->copy_out));
    chk(cudaStreamWaitEvent(s, q->ev_done, 0));
    chk(cudaEventRecord(q->ev_in[0], q->copy_in));
    chk(cudaStreamWaitEvent(s, q->ev_in[0], 0));
    if (rc != SSM_OK) return rc;
    return ok ? SSM_OK : SSM_ERR_CUDA;
}
