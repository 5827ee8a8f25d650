// scan_host.cu -- the selective scan on host-resident activations
// (ssm_scan_fwd_host): host -> device copies, the scan and device -> host copies
// pipelined over segments of the problem's channels.
//
// What it computes is exactly ssm_scan_fwd's ("We brought Mamba to Trainium --
// and mapped where custom kernels actually help", section "Mamba: bringing an
// unsupported model to the chip, and writing its missing kernel"): every
// channel's recurrence is independent of the others, so a range of channels is
// a problem of its own.
//
// How: the (batch, channel) rows are cut into about eight segments, each a
// contiguous range of rows -- whole batches, whole B/C groups of one batch, or
// part of one group; the first and the last are cut smaller, since nothing
// overlaps the first one's input copy or the last one's scan and output copy --
// so that every array of a segment (u, delta, z, y, the
// states, and its groups' B and C) is one contiguous block of host memory,
// moved by a single 1-D copy at the link's full rate (2-D copies of short rows
// run well below it).  Segment k's inputs are copied on a copy stream into one
// of four device slots, the caller's stream scans the slot, and a second copy
// stream brings y and the final state back.  Four slots let the input copies
// run up to three segments ahead of the scans.  Copies in both directions run
// on the copy engines while the SMs scan the neighbouring segments.  The two
// copy streams and the events are created once per device and kept for the
// life of the process.
//
// Which kernel scans a segment: a segment of a few thousand channels leaves
// most SMs idle in the chained scan, whose CTAs each walk the whole sequence
// (about 0.8 ms for any segment of a 16 k-step problem), and the last
// segment's scan is on the critical path.  So when every segment fits the
// sequence-parallel scan, all segments take it, with one segments-per-chunk
// count, and its time shrinks with the segment (on long sequences the
// segments are capped to fit it).  A channel's arithmetic depends only on the
// kernel and that count, so the result is bit-equal to ssm_scan_fwd of any
// channel subset the sequence-parallel scan takes with the same count.  Other
// problems (those ssm_scan_fwd itself gives to the sequence-parallel scan,
// and short sequences with segments too large for it) run every segment with
// the whole problem's kernel and plan: bit-equal to ssm_scan_fwd.
#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "scan_internal.h"

namespace {

using namespace ssm_host;

constexpr int kN = 16;
constexpr int kSlots = 4;
constexpr long long kTargetSegments = 8;
// Input and output bytes a segment capped to the sequence-parallel scan's size
// must still move for the cap to apply.
constexpr size_t kMinCappedSegmentBytes = size_t(32) << 20;

// One segment: batches [b0, b0 + nb), channels [c0, c0 + nc) of each, which lie
// in groups [g0, g0 + ng).  Either whole batches (c0 = 0, nc = dim), or one
// batch with whole groups, or one batch with part of one group; in each case
// its rows of u, delta, z, y and of the states, and its rows of B and C, are
// contiguous.
struct Seg {
    int b0, nb, c0, nc, g0, ng;
};

struct Plan {
    std::vector<Seg> segs;
    long long max_rows = 0, max_bcrows = 0, max_nc = 0;
    size_t act_in = 0, bc_in = 0, act_out = 0, state = 0, par = 0;  // one slot's regions
    size_t scan_ws = 0;  // bytes of ssm_scan_fwd's workspace for the largest segment
    size_t slot = 0, total = 0;
};

size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

Plan plan_for(int batch, int dim, int seqlen, int ngroups, size_t es, size_t eo) {
    Plan p{};
    const long long rows = (long long)batch * dim;
    const int cg = dim / ngroups;  // channels per group
    long long target = std::max(1LL, (rows + kTargetSegments - 1) / kTargetSegments);
    // on long sequences, segments small enough for the sequence-parallel scan
    // (their copies still far outweigh a segment's fixed launch and copy costs)
    const long long cap = ssm_internal::kScanSegMaxChannels;
    if (target > cap && (size_t)cap * seqlen * (3 * es + eo) >= kMinCappedSegmentBytes)
        target = cap;
    if (target >= dim) {
        const int per = (int)std::min<long long>(target / dim, batch);
        for (int b = 0; b < batch; b += per)
            p.segs.push_back({b, std::min(per, batch - b), 0, dim, 0, ngroups});
    } else if (target >= cg) {
        const int per = (int)(target / cg);
        for (int b = 0; b < batch; ++b)
            for (int g = 0; g < ngroups; g += per) {
                const int ng = std::min(per, ngroups - g);
                p.segs.push_back({b, 1, g * cg, ng * cg, g, ng});
            }
    } else {
        const int pieces = (int)((cg + target - 1) / target);
        const int pc = (cg + pieces - 1) / pieces;
        for (int b = 0; b < batch; ++b)
            for (int g = 0; g < ngroups; ++g)
                for (int c = 0; c < cg; c += pc)
                    p.segs.push_back({b, 1, g * cg + c, std::min(pc, cg - c), g, 1});
    }
    // The first segment's input copy runs before anything can overlap it, and the
    // last segment's scan and output copy after: the end segments are halved.
    // (Halving them again gained nothing on a 16 k-step problem: with the
    // chained scan each extra segment's scan, about 0.8 ms whatever its size,
    // no longer hid behind the copies; with the sequence-parallel scan the
    // copies alone set the time.)
    auto halve = [&](const Seg& sg, std::vector<Seg>& out) {
        if (sg.nb > 1) {  // whole batches
            const int h = sg.nb / 2;
            out.push_back({sg.b0, h, 0, dim, 0, ngroups});
            out.push_back({sg.b0 + h, sg.nb - h, 0, dim, 0, ngroups});
        } else if (sg.ng > 1) {  // whole groups
            const int h = sg.ng / 2;
            out.push_back({sg.b0, 1, sg.c0, h * cg, sg.g0, h});
            out.push_back({sg.b0, 1, sg.c0 + h * cg, (sg.ng - h) * cg, sg.g0 + h, sg.ng - h});
        } else if (sg.nc > 1) {  // part of one group
            const int h = sg.nc / 2;
            out.push_back({sg.b0, 1, sg.c0, h, sg.g0, 1});
            out.push_back({sg.b0, 1, sg.c0 + h, sg.nc - h, sg.g0, 1});
        } else {
            out.push_back(sg);
        }
    };
    if (p.segs.size() >= 2) {
        std::vector<Seg> cut;
        const size_t n = p.segs.size();
        for (size_t i = 0; i < n; ++i) {
            if (i == 0 || i == n - 1) halve(p.segs[i], cut);
            else cut.push_back(p.segs[i]);
        }
        p.segs.swap(cut);
    }
    for (const Seg& sg : p.segs) {
        p.max_rows = std::max(p.max_rows, (long long)sg.nb * sg.nc);
        p.max_bcrows = std::max(p.max_bcrows, (long long)sg.nb * sg.ng * kN);
        p.max_nc = std::max(p.max_nc, (long long)sg.nc);
        p.scan_ws = std::max(p.scan_ws, ssm_scan_workspace_bytes(sg.nb, sg.nc, seqlen, kN, sg.ng));
    }
    const size_t L = (size_t)seqlen;
    p.act_in = r256((size_t)p.max_rows * L * es);
    p.bc_in = r256((size_t)p.max_bcrows * L * es);
    p.act_out = r256((size_t)p.max_rows * L * eo);
    p.state = r256((size_t)p.max_rows * kN * 4);
    p.par = r256((size_t)p.max_nc * 4);
    p.scan_ws = r256(p.scan_ws);
    // per slot: u, delta, z, B, C in; y out; the initial and final state; D
    // and delta_bias slices that need realigning
    p.slot = 3 * p.act_in + 2 * p.bc_in + p.act_out + 2 * p.state + 2 * p.par;
    // scan workspace first (ssm_last_device_status reads its header)
    p.total = p.scan_ws + kSlots * p.slot;
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
    // (arrays of no bytes -- the activations when seqlen is 0 -- are never touched)
    const void* host_ptrs[] = {seqlen ? u : nullptr, seqlen ? delta : nullptr,
                               seqlen ? z : nullptr,  seqlen ? B : nullptr,
                               seqlen ? C : nullptr,  initial_state,
                               seqlen ? y : nullptr,  final_state};
    for (const void* p : host_ptrs)
        if (!is_pinned(p)) return SSM_ERR_UNSUPPORTED;
    for (const void* p : dev_ptrs)
        if (!is_device(p)) return SSM_ERR_UNSUPPORTED;

    // every segment's arrays fit its slot's regions (the plan's own invariant,
    // checked before anything is enqueued)
    for (const Seg& sg : pl.segs) {
        const size_t nrows = (size_t)sg.nb * sg.nc, nbc = (size_t)sg.nb * sg.ng * kN;
        if (nrows * seqlen * es > pl.act_in || nbc * seqlen * es > pl.bc_in ||
            nrows * seqlen * eo > pl.act_out || nrows * kN * 4 > pl.state ||
            (size_t)sg.nc * 4 > pl.par ||
            ssm_scan_workspace_bytes(sg.nb, sg.nc, seqlen, kN, sg.ng) > pl.scan_ws)
            return SSM_ERR_WORKSPACE;
    }

    std::mutex* lock = nullptr;
    DeviceQueues* q = queues(lock);
    if (!q) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(*lock);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* scan_ws = ws;
    bool ok = true;
    auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };

    // the copy streams start after the caller's earlier work (which may still use
    // this workspace)
    chk(cudaEventRecord(q->ev_done, s));
    chk(cudaStreamWaitEvent(q->copy_in, q->ev_done, 0));
    chk(cudaStreamWaitEvent(q->copy_out, q->ev_done, 0));
    const size_t L = (size_t)seqlen;
    // the kernel (path) and sequence-parallel segments per chunk of every segment
    int path, seg_ts;
    if (ssm_internal::scan_seg_eligible(batch, dim) ||
        !ssm_internal::scan_seg_eligible(1, pl.max_rows)) {
        // the whole problem's kernel and plan
        path = ssm_internal::scan_uses_seg_path(batch, dim) ? 2 : 1;
        seg_ts = ssm_internal::scan_seg_plan_ts(batch, dim, seqlen);
    } else {
        // every segment fits the sequence-parallel scan: one count for all
        path = ssm_internal::scan_uses_seg_path(1, pl.max_rows) ? 2 : 1;
        seg_ts = ssm_internal::scan_seg_plan_ts(1, pl.max_rows, seqlen);
    }
    ssm_status_t rc = SSM_OK;
    for (size_t k = 0; k < pl.segs.size() && ok && rc == SSM_OK; ++k) {
        const Seg& sg = pl.segs[k];
        const int sl = (int)(k % kSlots);
        const size_t r0 = (size_t)sg.b0 * dim + sg.c0;            // first row
        const size_t nrows = (size_t)sg.nb * sg.nc;
        const size_t bc0 = ((size_t)sg.b0 * ngroups + sg.g0) * kN;  // first B/C row
        const size_t nbc = (size_t)sg.nb * sg.ng * kN;
        uint8_t* du = ws + pl.scan_ws + (size_t)sl * pl.slot;
        uint8_t* dd = du + pl.act_in;
        uint8_t* dz = dd + pl.act_in;
        uint8_t* dB = dz + pl.act_in;
        uint8_t* dC = dB + pl.bc_in;
        uint8_t* dy = dC + pl.bc_in;
        float* dh0 = reinterpret_cast<float*>(dy + pl.act_out);
        float* dfs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dh0) + pl.state);
        float* dD = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dfs) + pl.state);
        float* dbias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dD) + pl.par);
        // segment k's inputs into the slot, once the scan two segments back is done with it
        if (k >= (size_t)kSlots) chk(cudaStreamWaitEvent(q->copy_in, q->ev_comp[sl], 0));
        auto in1d = [&](void* dst, const void* src, size_t off, size_t bytes) {
            chk(cudaMemcpyAsync(dst, static_cast<const uint8_t*>(src) + off, bytes,
                                cudaMemcpyHostToDevice, q->copy_in));
        };
        if (L > 0) {
            in1d(du, u, r0 * L * es, nrows * L * es);
            in1d(dd, delta, r0 * L * es, nrows * L * es);
            if (z) in1d(dz, z, r0 * L * es, nrows * L * es);
            in1d(dB, B, bc0 * L * es, nbc * L * es);
            in1d(dC, C, bc0 * L * es, nbc * L * es);
        }
        if (initial_state) in1d(dh0, initial_state, r0 * kN * 4, nrows * kN * 4);
        chk(cudaEventRecord(q->ev_in[sl], q->copy_in));
        // the scan of segment k on the caller's stream
        chk(cudaStreamWaitEvent(s, q->ev_in[sl], 0));
        if (k >= (size_t)kSlots) chk(cudaStreamWaitEvent(s, q->ev_out[sl], 0));
        if (!ok) break;
        // per-channel parameters of the segment: A's rows are 64 bytes (always
        // 16-byte aligned); D and delta_bias slices are copied when their
        // offset is not
        const float* pD = D ? D + sg.c0 : nullptr;
        const float* pbias = delta_bias ? delta_bias + sg.c0 : nullptr;
        if (sg.c0 % 4 != 0) {
            if (D) chk(cudaMemcpyAsync(dD, pD, (size_t)sg.nc * 4, cudaMemcpyDeviceToDevice, s));
            if (delta_bias)
                chk(cudaMemcpyAsync(dbias, pbias, (size_t)sg.nc * 4, cudaMemcpyDeviceToDevice, s));
            pD = D ? dD : nullptr;
            pbias = delta_bias ? dbias : nullptr;
        }
        rc = ssm_internal::scan_forward_segment(
            du, dd, A + (size_t)sg.c0 * kN, dB, dC, pD, z ? dz : nullptr, pbias, delta_softplus,
            initial_state ? dh0 : nullptr, dy, final_state ? dfs : nullptr, sg.nb, sg.nc,
            seqlen, sg.ng, in_dtype, out_dtype, scan_ws, pl.scan_ws, s, seg_ts, k > 0, path);
        chk(cudaEventRecord(q->ev_comp[sl], s));
        // segment k's y and final state back to the host
        chk(cudaStreamWaitEvent(q->copy_out, q->ev_comp[sl], 0));
        if (L > 0)
            chk(cudaMemcpyAsync(static_cast<uint8_t*>(y) + r0 * L * eo, dy, nrows * L * eo,
                                cudaMemcpyDeviceToHost, q->copy_out));
        if (final_state)
            chk(cudaMemcpyAsync(final_state + r0 * kN, dfs, nrows * kN * 4, cudaMemcpyDeviceToHost,
                                q->copy_out));
        chk(cudaEventRecord(q->ev_out[sl], q->copy_out));
    }
    // the caller's stream completes after every copy of this call
    chk(cudaEventRecord(q->ev_done, q->copy_out));
    chk(cudaStreamWaitEvent(s, q->ev_done, 0));
    chk(cudaEventRecord(q->ev_in[0], q->copy_in));
    chk(cudaStreamWaitEvent(s, q->ev_in[0], 0));
    if (rc != SSM_OK) return rc;
    return ok ? SSM_OK : SSM_ERR_CUDA;
}
