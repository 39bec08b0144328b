// host_pipe.cpp -- add_rms_fwd_host: the fused residual add + RMSNorm on
// tensors that live in host memory, streamed through the device in chunks of
// rows so that the three stages overlap:
//
//   copy stream  (host -> device)   x, residual of chunk k+1
//   caller's stream (compute)        add_rms_fwd of chunk k
//   copy stream  (device -> host)   residual_out, y of chunk k-1
//
// Host->device and device->host copies run on the GPU's two copy directions
// at once, and the kernel of a chunk takes a few microseconds against the
// copies' hundreds, so a call costs about the time of moving its bytes over
// the host link.  Device staging is the caller's workspace: kSlots slots of
// (x, residual, residual_out, y) for one chunk each; slot reuse is ordered by
// events (a slot's inputs are overwritten only after the kernel that read
// them, its outputs only after the copy that read them back).  The call
// returns once everything is enqueued; the caller's stream waits for the
// last copies, so completion of `stream` means the host outputs are written.
// The copy streams and events are created once per device; calls on one
// device are serialized on a mutex while they enqueue.
#include <cuda_runtime_api.h>

#include <cstdint>
#include <mutex>

#include "nrm.h"
#include "nrm_internal.h"

namespace {

// Three slots of 4 MB per tensor: measured on GB300 at 4096 x 4096 bf16
// (0.55 ms per call); 2 MB chunks were slower (0.84 ms), 8 MB chunks or two or
// four slots no faster.
constexpr int kSlots = 3;
constexpr int kTensors = 4;                        // x, residual, residual_out, y
constexpr int64_t kChunkBytes = (int64_t)4 << 20;  // per tensor per chunk
constexpr int kMaxDev = 64;

struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t e_in[kSlots] = {}, e_comp[kSlots] = {}, e_out[kSlots] = {};
    bool ok = false;
};
HostPipe g_pipe[kMaxDev];
std::once_flag g_pipe_once[kMaxDev];
std::mutex g_pipe_mu[kMaxDev];

bool pipe_init(HostPipe &p) {
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int i = 0; i < kSlots; ++i) {
        if (cudaEventCreateWithFlags(&p.e_in[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.e_comp[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.e_out[i], cudaEventDisableTiming) != cudaSuccess)
            return false;
    }
    return true;
}

int64_t chunk_rows(int64_t N, size_t es) {
    const int64_t r = kChunkBytes / (N * (int64_t)es);
    return r < 1 ? 1 : r;
}

}  // namespace

extern "C" {

size_t add_rms_fwd_host_workspace_size(int64_t N, int dtype) {
    if (N < 1 || (dtype != NRM_F32 && dtype != NRM_F16 && dtype != NRM_BF16)) return 0;
    const size_t es = dtype == NRM_F32 ? 4 : 2;
    const int64_t R = chunk_rows(N, es);
    if ((uint64_t)R > (uint64_t)INT64_MAX / (uint64_t)N / es / (kSlots * kTensors)) return 0;
    // each staging tensor starts on a 256-byte boundary
    const size_t tensor = (((size_t)R * (size_t)N * es) + 255) / 256 * 256;
    return tensor * kSlots * kTensors;
}

int add_rms_fwd_host(const void *x, const void *residual, const void *w, void *residual_out,
                     void *y, float *rstd, int64_t rows, int64_t N, float eps, int dtype,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (dtype != NRM_F32 && dtype != NRM_F16 && dtype != NRM_BF16) return NRM_ERR_DTYPE;
    if (rows < 0 || N < 1) return NRM_ERR_SHAPE;
    const size_t es = dtype == NRM_F32 ? 4 : 2;
    if (rows > 0 && (uint64_t)N > (uint64_t)INT64_MAX / (uint64_t)rows / es) return NRM_ERR_SHAPE;
    if (rows == 0) return NRM_OK;
    if (!x || !residual || !residual_out || !y) return NRM_ERR_NULL;
    const size_t need = add_rms_fwd_host_workspace_size(N, dtype);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return NRM_ERR_WORKSPACE;
    // host buffers: outputs must not overlap inputs, except residual_out == residual
    const size_t tb = (size_t)rows * (size_t)N * es;
    auto ov = [tb](const void *a, const void *b) {
        const uintptr_t p = reinterpret_cast<uintptr_t>(a), q = reinterpret_cast<uintptr_t>(b);
        return p < q + tb && q < p + tb;
    };
    if (ov(y, x) || ov(y, residual) || ov(y, residual_out) || ov(residual_out, x) ||
        (residual_out != residual && ov(residual_out, residual)))
        return NRM_ERR_ALIAS;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    std::call_once(g_pipe_once[dev], [dev]() { g_pipe[dev].ok = pipe_init(g_pipe[dev]); });
    HostPipe &P = g_pipe[dev];
    if (!P.ok) return NRM_ERR_DEVICE;

    const int64_t R = chunk_rows(N, es);
    const size_t tensor = (((size_t)R * (size_t)N * es) + 255) / 256 * 256;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    auto slot_ptr = [&](int slot, int t) { return ws + ((size_t)slot * kTensors + t) * tensor; };
    const unsigned char *hx = static_cast<const unsigned char *>(x);
    const unsigned char *hr = static_cast<const unsigned char *>(residual);
    unsigned char *hro = static_cast<unsigned char *>(residual_out);
    unsigned char *hy = static_cast<unsigned char *>(y);
    const int64_t chunks = (rows + R - 1) / R;

    std::lock_guard<std::mutex> lock(g_pipe_mu[dev]);
    // the copies start after the work already on the caller's stream
    if (cudaEventRecord(P.e_comp[0], stream) != cudaSuccess ||
        cudaStreamWaitEvent(P.in, P.e_comp[0], 0) != cudaSuccess)
        return NRM_ERR_LAUNCH;
    for (int64_t k = 0; k < chunks; ++k) {
        const int s = (int)(k % kSlots);
        const int64_t r0 = k * R, nr = (rows - r0) < R ? (rows - r0) : R;
        const size_t off = (size_t)r0 * (size_t)N * es, bytes = (size_t)nr * (size_t)N * es;
        // inputs of slot s: after the kernel that last read them
        if (k >= kSlots && cudaStreamWaitEvent(P.in, P.e_comp[s], 0) != cudaSuccess)
            return NRM_ERR_LAUNCH;
        if (cudaMemcpyAsync(slot_ptr(s, 0), hx + off, bytes, cudaMemcpyHostToDevice, P.in) !=
                cudaSuccess ||
            cudaMemcpyAsync(slot_ptr(s, 1), hr + off, bytes, cudaMemcpyHostToDevice, P.in) !=
                cudaSuccess ||
            cudaEventRecord(P.e_in[s], P.in) != cudaSuccess)
            return NRM_ERR_LAUNCH;
        // compute: after the inputs arrive and the slot's outputs were copied back
        if (cudaStreamWaitEvent(stream, P.e_in[s], 0) != cudaSuccess) return NRM_ERR_LAUNCH;
        if (k >= kSlots && cudaStreamWaitEvent(stream, P.e_out[s], 0) != cudaSuccess)
            return NRM_ERR_LAUNCH;
        const int st = add_rms_fwd(slot_ptr(s, 0), slot_ptr(s, 1), w, slot_ptr(s, 2),
                                   slot_ptr(s, 3), rstd ? rstd + r0 : nullptr, nr, N, eps, dtype,
                                   stream);
        if (st != NRM_OK) return st;
        if (cudaEventRecord(P.e_comp[s], stream) != cudaSuccess) return NRM_ERR_LAUNCH;
        // outputs back to the host
        if (cudaStreamWaitEvent(P.out, P.e_comp[s], 0) != cudaSuccess ||
            cudaMemcpyAsync(hro + off, slot_ptr(s, 2), bytes, cudaMemcpyDeviceToHost, P.out) !=
                cudaSuccess ||
            cudaMemcpyAsync(hy + off, slot_ptr(s, 3), bytes, cudaMemcpyDeviceToHost, P.out) !=
                cudaSuccess ||
            cudaEventRecord(P.e_out[s], P.out) != cudaSuccess)
            return NRM_ERR_LAUNCH;
    }
    // the caller's stream completes after the last copy back
    if (cudaStreamWaitEvent(stream, P.e_out[(chunks - 1) % kSlots], 0) != cudaSuccess)
        return NRM_ERR_LAUNCH;
    return NRM_OK;
}

}  // extern "C"
