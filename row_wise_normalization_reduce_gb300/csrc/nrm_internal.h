// nrm_internal.h -- host-side declarations shared by the C ABI (api.cpp) and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace nrm {

enum Op { OP_LN = 0, OP_RMS = 1, OP_ADD_RMS = 2, OP_SOFTMAX = 3 };
enum DType { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };
enum PlanKind {
    PLAN_AUTO = 0,
    PLAN_GENERIC = 1,
    PLAN_WARP = 2,
    PLAN_CTA = 3,
    PLAN_TMA = 4,
    PLAN_PERSIST = 5,
    PLAN_WRAW = 6,
    PLAN_CLUSTER = 7
};

// Bits of the device fault word (see fault.cu).
enum FaultBits : unsigned {
    FAULT_WAIT = 1u,    // a kernel gave up waiting for a bulk copy
    FAULT_DRAIN = 2u    // ... and then for its copies still in flight
};

// Largest number of shared-memory stages of the bulk-copy row pipeline, and
// the dynamic shared memory a CTA may use (static arrays take the rest of the
// 227 KB).
constexpr int kMaxStages = 16;
constexpr int kSmemMax = 224 * 1024;

// Everything a row kernel needs.  Pointers are device pointers; unused ones
// are NULL.  p0 = gamma (LayerNorm) or w (RMS ops); p1 = beta.
struct RowArgs {
    const void *x;
    const void *res;      // add+RMS only
    const void *p0;
    const void *p1;
    void *res_out;        // add+RMS only
    void *y;
    float *mean;          // LayerNorm: row mean; softmax: row max
    float *rstd;          // norms: 1/sqrt(...); softmax: row sum of exp(x - max)
    int64_t rows;
    int64_t N;
    float eps;
    unsigned *fault;      // device fault word of the current device
    unsigned wait_limit;  // tries per bounded wait (0: give up at once)
    float fN;             // (float)N, and its correctly rounded reciprocal,
    float invN;           // computed once on the host
    int64_t ldx, ldr, ldro, ldy;  // row strides (elements) of x, res, res_out, y
};

struct Plan {
    int kind;      // PlanKind
    int threads;   // CTA size
    int packs;     // 16-byte packs per thread (WARP: per lane)
    int stages;    // TMA: shared-memory row stages per group
    int groups;    // TMA: row groups per CTA
    int smem_params;  // TMA: parameters widened to binary32 in shared memory
    int sms;       // SMs of the device
    int64_t grid;  // CTAs launched (TMA: set at launch from occupancy)
    int prefetch;  // CTA: L2 prefetch distance in waves of resident CTAs (0: off)
};

// Resident CTAs per SM of `kernel` (a __global__ function) on the current
// device at `threads` threads and `smem` bytes of dynamic shared memory; the
// kernel's dynamic shared-memory limit is raised to `smem` when needed.  Asked
// once per device, kernel, block size and shared-memory size.  occupancy.cpp.
cudaError_t resident_ctas(const void *kernel, int threads, size_t smem, int *per_sm);

// Address of the current device's fault word (set up once per device), or
// NULL if it cannot be obtained.  fault.cu.
unsigned *fault_word();

// Launch a row operator with a fully specified plan.  Returns a cudaError_t
// from the launch (cudaSuccess or the launch error), or
// cudaErrorInvalidConfiguration when the template set has no such plan.
// One instance per operator and storage type (rows_<op>_<type>.cu).
#define NRM_ROW_LAUNCHERS(op)                                                          \
    cudaError_t launch_##op##_f32(const RowArgs &a, const Plan &p, cudaStream_t s);    \
    cudaError_t launch_##op##_f16(const RowArgs &a, const Plan &p, cudaStream_t s);    \
    cudaError_t launch_##op##_bf16(const RowArgs &a, const Plan &p, cudaStream_t s);   \
    inline cudaError_t launch_##op(const RowArgs &a, const Plan &p, int dtype, cudaStream_t s) { \
        switch (dtype) {                                                               \
        case DT_F32: return launch_##op##_f32(a, p, s);                                \
        case DT_F16: return launch_##op##_f16(a, p, s);                                \
        case DT_BF16: return launch_##op##_bf16(a, p, s);                              \
        default: return cudaErrorInvalidValue;                                         \
        }                                                                              \
    }
NRM_ROW_LAUNCHERS(ln)
NRM_ROW_LAUNCHERS(rms)
NRM_ROW_LAUNCHERS(add_rms)
#undef NRM_ROW_LAUNCHERS
// Row softmax (softmax.cu): PLAN_CTA (row in registers) or PLAN_GENERIC.
cudaError_t launch_softmax(const RowArgs &a, const Plan &p, int dtype, cudaStream_t s);

// BatchNorm training forward.  x, gamma, beta, y are stored in the call's
// dtype; statistics are binary32.  ws holds batch*C float2 partials.
struct BnArgs {
    const void *x;
    const void *gamma;
    const void *beta;
    void *y;
    float *save_mean;
    float *save_rstd;
    float *running_mean;
    float *running_var;
    int64_t batch, C, HW;
    float eps, momentum;
    void *ws;             // two-kernel plans: batch * C float2 partials
    unsigned *fault;      // device fault word (cluster and one-pass plans), or NULL
    unsigned wait_limit;  // tries per bounded wait
    int bn_plan;          // BnPlan
    size_t ws_bytes = 0;  // bytes at ws (the one-pass plan runs only if it fits)
    int prefetch = 0;     // one-pass plan's L2 prefetch: 0 auto, 1 off, s >= 2: s - 1 rounds ahead
    int packs = 0;        // one-pass plan's packs per thread: 0 auto, 4 or 8
    int cluster_size = 0; // cluster plan: CTAs per cluster (0: 8), a measurement hook
    int max_clusters = 0; // cluster plan: at most this many clusters (0: one per channel
                          // when they all fit at once), a measurement hook
    double *stats_out = nullptr;  // cluster plan: write each channel's binary64
                                  // (count, mean, M2) at [3c] instead of normalizing
};

// BatchNorm plans: automatic, streaming two kernels (registers + dependent
// launch), one cluster of CTAs per channel (shared memory + DSMEM), and the
// scalar two-kernel plan (any layout).
// BN_PLAN_NO_STREAM: automatic choice without the streaming plan (whose
// per-chunk partials may not fit a fixed partials array).  BN_PLAN_FLOW: the
// one-pass plan (bn_flow.cu): statistics and normalization in one kernel,
// each channel normalized a few channels after its statistics, its second
// read served by L2.
enum BnPlan {
    BN_PLAN_AUTO = 0,
    BN_PLAN_STREAM = 1,
    BN_PLAN_CLUSTER = 2,
    BN_PLAN_SCALAR = 3,
    BN_PLAN_NO_STREAM = 4,
    BN_PLAN_FLOW = 5
};

// Packs (16 bytes) per work unit of the streaming BatchNorm plans: a unit is
// a chunk of at most this many packs of one plane; the workspace holds one
// float2 per unit.
constexpr int kBnChunkPacks = 1024;

// Capacity of the library's fixed partials array used by
// bn_fwd_train_noalloc: batch * C planes (one float2 each, 512 KB).
constexpr int64_t kBnFixedPlanes = 65536;

// The current device's address and size of that array (bn.cu), looked up
// once per device with the device current; an NRM status.
int bn_fixed_workspace(void **ws, size_t *bytes);

// Workspace bytes of the one-pass plans for C channels and `units` chunks in
// all: the per-chunk 8-byte partials (padded to 16 bytes), then 24 bytes per
// channel (folded statistics and control words).
inline size_t bn_flow_ws_bytes(int64_t C, int64_t units) {
    return (((size_t)units * 8 + 15) & ~(size_t)15) + (size_t)C * 24;
}

// The launchers report the plan they ran through *used as a PlanKind
// (cluster: PLAN_TMA, streaming: PLAN_CTA, scalar: PLAN_GENERIC, one-pass:
// PLAN_PERSIST).
cudaError_t launch_bn_train(const BnArgs &a, int dtype, int num_sms, cudaStream_t s, int *used);

// BatchNorm inference forward: y = (x - running_mean) * rsqrt(running_var +
// eps) * gamma + beta, per channel.
struct BnInferArgs {
    const void *x;
    const void *gamma;
    const void *beta;
    void *y;
    const float *running_mean;
    const float *running_var;
    int64_t batch, C, HW;
    float eps;
    int bn_plan;          // BN_PLAN_SCALAR forces the element-wise scalar kernel
};
cudaError_t launch_bn_infer(const BnInferArgs &a, int dtype, int num_sms, cudaStream_t s,
                            int *used);

// BatchNorm training backward.  dy, x, gamma, dx are stored in the call's
// dtype; mean/rstd (the saved statistics), dgamma and dbeta are binary32.
// ws holds batch*C float2 per-plane partial sums (sum dy, sum dy*(x-mean)).
struct BnBwdArgs {
    const void *dy;
    const void *x;
    const void *gamma;
    const float *mean;
    const float *rstd;
    void *dx;
    float *dgamma;
    float *dbeta;
    int64_t batch, C, HW;
    void *ws;
    int bn_plan;          // BN_PLAN_AUTO / STREAM / SCALAR / FLOW
    unsigned *fault = nullptr;  // device fault word (one-pass plan), or NULL
    unsigned wait_limit = 0;    // tries per bounded wait
    size_t ws_bytes = 0;        // bytes at ws (the one-pass plan runs only if it fits)
    int prefetch = 0;           // one-pass plan's L2 prefetch, as BnArgs::prefetch
};
// The one-pass backward (bn_flow_bwd.cu) for 16-byte aligned planes of whole
// packs; *launched tells whether it ran.
cudaError_t launch_bn_bwd_flow(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                               bool *launched);
cudaError_t launch_bn_bwd(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                          int *used);

// Stage 1 alone, per (n, c) plane into a.ws (scalar plans, any layout):
// (mean, M2) of d = x - x[0, c, 0] for the forward; (sum dy, sum dy*(x - mean))
// for the backward.
cudaError_t launch_bn_plane_stats(const BnArgs &a, int dtype, int num_sms, cudaStream_t s);
// Stage 1 per unit (chunks of at most kBnChunkPacks packs; planes of 16-byte
// aligned packs, fewer than kBnUnitPlaneLimit packs): the unit layout is
// returned as chunks per plane, packs per chunk, packs per plane.
constexpr int64_t kBnUnitPlaneLimit = (int64_t)1 << 20;
cudaError_t launch_bn_unit_stats_host(const BnArgs &a, int dtype, int num_sms, cudaStream_t s,
                                      int *nch, int *cpk, int *q);
cudaError_t launch_bn_bwd_unit_sums_host(const BnBwdArgs &a, int dtype, int num_sms,
                                         cudaStream_t s, int *nch);
cudaError_t launch_bn_bwd_plane_sums(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s);

// Synchronized BatchNorm pieces (bn_sync.cu).
struct BnSyncArgs {
    const void *x;       // forward: x; backward: x
    const void *dy;      // backward only
    const void *gamma;
    const void *beta;
    void *out;           // y or dx
    const float *mean;   // backward: saved statistics
    const float *rstd;
    const double *parts; // [nparts][C][3] (forward) or [nparts][C][2] (backward)
    int64_t nparts;
    int64_t count;       // backward: global batch * HW
    float *save_mean, *save_rstd, *running_mean, *running_var;  // forward outputs
    float *dgamma, *dbeta;                                       // backward outputs
    int64_t batch, C, HW;
    float eps, momentum;
};
// Folds of stage-1 partials into per-channel binary64 arrays: per_channel
// partials per channel; for per-unit partials (V > 0) partial j counts
// min(cpk, q - (j mod nch)*cpk)*V values, for per-plane partials (V = 0) HW.
cudaError_t launch_bn_fold_stats(const float2 *ws, const void *x, double *stats, int64_t per_channel,
                                 int64_t C, int64_t HW, int nch, int cpk, int q, int V, int dtype,
                                 cudaStream_t s);
cudaError_t launch_bn_fold_sums(const float2 *ws, const float *rstd, double *sums,
                                int64_t per_channel, int64_t C, cudaStream_t s);
cudaError_t launch_bn_apply_stats(const BnSyncArgs &a, int dtype, int num_sms, cudaStream_t s);
// The cluster plan in statistics-only mode (a.stats_out set): one launch
// writes every channel's (count, mean, M2); *launched false when the plan
// cannot take the shape.
cudaError_t launch_bn_cluster_stats(const BnArgs &a, int dtype, cudaStream_t s, bool *launched);
cudaError_t launch_bn_apply_sums(const BnSyncArgs &a, int dtype, int num_sms, cudaStream_t s);

}  // namespace nrm
