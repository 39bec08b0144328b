// row_kernels.cuh -- the row operators (LayerNorm, RMSNorm, residual add +
// RMSNorm) as three kernel families, templated on operator, I/O type and
// launch shape, plus the launch switch that maps a Plan onto them.
//
//   row_cta_kernel      one CTA per row; the row is loaded once into
//                       registers with 16-byte accesses, reduced (warp
//                       shuffles, then one shared-memory exchange), normalized
//                       from registers and stored.  x is read from HBM once.
//   row_warp_kernel     one warp per row (short rows, many rows); reduction
//                       by shuffles only.
//   row_pipe_kernel     persistent CTAs of several row groups; each group streams
//                       whole rows into its own ring of shared-memory stages
//                       with bulk asynchronous copies completed on mbarriers,
//                       so rows are always in flight while others are reduced
//                       (row_pipe.cuh).
//   row_persist_kernel  persistent CTAs; the next row's packs are loaded into
//                       registers while the current row is reduced (and
//                       later rows are prefetched into L2), and the
//                       parameters are widened to binary32 in shared memory
//                       once per CTA.
//   row_wraw_kernel     warp per row with the raw packs of the whole row in
//                       registers; shuffle-only reductions; long rows.
//   row_generic_kernel  any N and any alignment: scalar accesses, one CTA per
//                       row, the row read twice (statistics, then output).
//
// The mapping of a row onto a CTA with a shuffle reduction and a per-warp
// exchange through shared memory follows the CUDA fused RMSNorm kernel page
// (diycv.top, §3-§4) and the LayerNorm walkthrough (lpnh.cn/news/2756757, §4-§5);
// unlike both, the row stays in registers (no second read) and the LayerNorm
// statistics come from a shifted, corrected two-pass over the registers, not
// from sums of x and x^2.
#pragma once

#include "nrm_device.cuh"
#include "nrm_internal.h"

namespace nrm {

// LayerNorm statistics (register-resident rows): a corrected two-pass over
// the values held in registers,
//   m0 = sum(x) / N                                   (first group-wide sum)
//   e  = x - m0;  c = sum(e) / N;  M2 = sum(e^2) - N c^2   (second, fused sum)
//   mean = m0 + c,  var = M2 / N,  y = ((e - c) * rstd) * gamma + beta.
// m0 may carry the rounding error of a binary32 sum of N values; c, a sum of
// the small centred values e, removes it, so the mean is accurate to a few
// roundoffs of the spread.  For rows with a large mean and a small spread
// (mean 1000, std 1) e = x - m0 is exact (x and m0 within a factor 2), so
// nothing is lost to cancellation, and sum(e^2) is a sum of small positive
// terms.  Two float sums per row; no divisions per element or per combine.
//
// Arithmetic is done pairwise with the packed binary32 instructions of
// sm_100+ (two IEEE operations per instruction): the row operators are close
// to instruction-bound at GB300's bandwidth, so halving the arithmetic
// instruction count is what lets them stream at HBM speed.

// Row-group reducers: the row is spread over one warp or over one CTA.
struct WarpRed {
    __device__ __forceinline__ float sum(float v) { return warp_sum_all(v); }
    __device__ __forceinline__ float2 sum2(float2 v) { return warp_sum_all(v); }
};

template <int NW> struct CtaRed {
    float *s1;
    float2 *s2;
    __device__ __forceinline__ float sum(float v) { return cta_sum_all<NW>(v, s1); }
    __device__ __forceinline__ float2 sum2(float2 v) { return cta_sum_all<NW>(v, s2); }
};

// Where a row's 16-byte packs come from: global memory (register path) or a
// shared-memory stage filled by a bulk copy (x, then residual, back to back).
template <typename T> struct GlobalSrc {
    const T *x;    // row start in global memory
    const T *res;
    __device__ __forceinline__ uint4 x_pack(int idx) const { return ld_stream(x + (size_t)idx * IO<T>::V); }
    __device__ __forceinline__ uint4 r_pack(int idx) const { return ld_stream(res + (size_t)idx * IO<T>::V); }
};

template <typename T> struct SmemSrc {
    const unsigned char *stage;
    uint32_t row_bytes;
    __device__ __forceinline__ uint4 x_pack(int idx) const {
        return reinterpret_cast<const uint4 *>(stage)[idx];
    }
    __device__ __forceinline__ uint4 r_pack(int idx) const {
        return reinterpret_cast<const uint4 *>(stage + row_bytes)[idx];
    }
};

// Where the parameters (gamma, beta / w) come from: global memory in their
// storage type, or shared memory already widened to binary32 (gamma at
// [0, N), beta at [N, 2N)), filled once per persistent CTA.
template <typename T> struct GlobalParams {
    const T *p0, *p1;
    __device__ __forceinline__ void p0_pack(int idx, float2 *f) const {
        if (p0) IO2<T>::unpack(ld_param(p0 + (size_t)idx * IO<T>::V), f);
        else
#pragma unroll
            for (int h = 0; h < IO2<T>::H; ++h) f[h] = f2(1.f);
    }
    __device__ __forceinline__ void p1_pack(int idx, float2 *f) const {
        if (p1) IO2<T>::unpack(ld_param(p1 + (size_t)idx * IO<T>::V), f);
        else
#pragma unroll
            for (int h = 0; h < IO2<T>::H; ++h) f[h] = f2(0.f);
    }
};

// Shared-memory layout: float4 q[param][quarter][pack] with the 4 (binary32
// packs) or 8 (16-bit packs) values of pack i split into consecutive float4
// planes, so the threads of a warp read consecutive 16-byte words (no bank
// conflicts).  Filled by fill_smem_params.
template <typename T> struct SmemParams {
    const float4 *q;
    int P;  // packs per row
    static constexpr int Q = IO<T>::V / 4;  // float4 per pack
    __device__ __forceinline__ void load(int param, int idx, float2 *f) const {
#pragma unroll
        for (int h = 0; h < Q; ++h) {
            const float4 t = q[((size_t)param * Q + h) * P + idx];
            f[2 * h] = make_float2(t.x, t.y);
            f[2 * h + 1] = make_float2(t.z, t.w);
        }
    }
    __device__ __forceinline__ void p0_pack(int idx, float2 *f) const { load(0, idx, f); }
    __device__ __forceinline__ void p1_pack(int idx, float2 *f) const { load(1, idx, f); }
};

// Widen parameters into the SmemParams layout (absent gamma/w = 1, beta = 0),
// one 16-byte pack per thread and step (the plans that use it need 16-byte
// aligned parameters and N a multiple of the pack width).
template <typename T, int NPARAM, int THREADS>
__device__ __forceinline__ void fill_smem_params(const RowArgs &a, float *sp) {
    constexpr int V = IO<T>::V, Q = V / 4, H = IO2<T>::H;
    const int P = (int)(a.N / V);
    const T *src[2] = {static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
    const float dflt[2] = {1.f, 0.f};
    float4 *q = reinterpret_cast<float4 *>(sp);
    for (int idx = threadIdx.x; idx < P; idx += THREADS) {
#pragma unroll
        for (int p = 0; p < NPARAM; ++p) {
            float2 f[H];
            if (src[p]) IO2<T>::unpack(ld_param(src[p] + (size_t)idx * V), f);
            else
#pragma unroll
                for (int h = 0; h < H; ++h) f[h] = f2(dflt[p]);
#pragma unroll
            for (int h = 0; h < Q; ++h)
                q[((size_t)p * Q + h) * P + idx] =
                    make_float4(f[2 * h].x, f[2 * h].y, f[2 * h + 1].x, f[2 * h + 1].y);
        }
    }
}

// Parameters kept in shared memory in their storage type: the raw 16-byte
// packs of gamma (w) at [0, P) and beta at [P, 2P), copied once per CTA and
// unpacked per use (half the shared memory of SmemParams at 16-bit types).
// An absent parameter is never read: 1 (gamma, w) or 0 (beta).
template <typename T> struct SmemRawParams {
    const uint4 *q;
    int P;
    bool has0, has1;
    __device__ __forceinline__ void p0_pack(int idx, float2 *f) const {
        if (has0) IO2<T>::unpack(q[idx], f);
        else
#pragma unroll
            for (int h = 0; h < IO2<T>::H; ++h) f[h] = f2(1.f);
    }
    __device__ __forceinline__ void p1_pack(int idx, float2 *f) const {
        if (has1) IO2<T>::unpack(q[P + idx], f);
        else
#pragma unroll
            for (int h = 0; h < IO2<T>::H; ++h) f[h] = f2(0.f);
    }
};

// Copy the present parameters into the SmemRawParams layout.
template <typename T, int NPARAM, int THREADS>
__device__ __forceinline__ void fill_smem_raw_params(const RowArgs &a, uint4 *q) {
    constexpr int V = IO<T>::V;
    const int P = (int)(a.N / V);
    const T *src[2] = {static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
    for (int idx = threadIdx.x; idx < P; idx += THREADS)
#pragma unroll
        for (int p = 0; p < NPARAM; ++p)
            if (src[p]) q[(size_t)p * P + idx] = ld_param(src[p] + (size_t)idx * V);
}

// Where a plan keeps its parameters (Plan::smem_params).
enum ParamsIn { PARAMS_GLOBAL = 0, PARAMS_SMEM_F32 = 1, PARAMS_SMEM_RAW = 2 };

// Dynamic shared-memory bytes of the parameters for a ParamsIn mode.
template <int OP, typename T>
inline size_t params_smem_bytes(int mode, int64_t N) {
    const size_t n = (size_t)N * (OP == OP_LN ? 2 : 1);
    return mode == PARAMS_SMEM_F32 ? n * sizeof(float) : mode == PARAMS_SMEM_RAW ? n * sizeof(T) : 0;
}

struct NoHook {
    __device__ __forceinline__ void operator()() const {}
};

// Everything after the loads of one row: the row is spread over a group whose
// member `t` owns packs t, t + STRIDE, ...; rx (and rr, the residual packs of
// add+RMS) hold its raw 16-byte packs.  `after_sync` runs right after the
// first group-wide sum, when every member has its values in registers (the
// bulk-copy pipeline refills the stage there).
// FULL: the row is exactly STRIDE x PACKS packs, so no pack index needs a
// bounds test.
template <int OP, typename T, int PACKS, int STRIDE, class Red, class Prm, class Hook,
          bool FULL = false>
__device__ __forceinline__ void row_compute(const RowArgs &a, const int64_t row, const int t,
                                            Red &red, const uint4 (&rx)[PACKS],
                                            const uint4 (&rr)[PACKS], const Prm &prm,
                                            const Hook &after_sync, const bool lead = true) {
    using io2 = IO2<T>;
    constexpr int V = IO<T>::V;
    constexpr int H = io2::H;
    const int P = (int)(a.N / V);  // 16-byte packs per row (< 2^31 by construction)
    const float fN = a.fN;
    const float invN = a.invN;
    T *__restrict__ Y = static_cast<T *>(a.y) + row * a.ldy;
    T *__restrict__ RO = static_cast<T *>(a.res_out) + row * a.ldro;

    // v: the row's values (add+RMS: the rounded residual-stream value)
    float2 v[PACKS][H];
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int idx = t + k * STRIDE;
        if (FULL || idx < P) {
            io2::unpack(rx[k], v[k]);
            if (OP == OP_ADD_RMS) {
                float2 r[H];
                io2::unpack(rr[k], r);
#pragma unroll
                for (int h = 0; h < H; ++h) v[k][h] = __fadd2_rn(v[k][h], r[h]);
                const uint4 packed = io2::pack(v[k]);  // round once to T
                st_stream(RO + (size_t)idx * V, packed);
                io2::unpack(packed, v[k]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < H; ++h) v[k][h] = f2(0.f);  // contributes nothing
        }
    }

    // ---- S3-S6: statistics ----
    float rstd, c = 0.f;
    if (OP == OP_LN) {
        float2 acc = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
#pragma unroll
            for (int h = 0; h < H; ++h) acc = __fadd2_rn(acc, v[k][h]);
        const float tot = red.sum(acc.x + acc.y);
        after_sync();
        // m0 = tot / N, corrected once: a constant row (tot = N x exactly)
        // gives m0 == x, hence e == 0, c == 0 and y == beta bit for bit.
        float m0 = tot * invN;
        m0 = fmaf(fmaf(-m0, fN, tot), invN, m0);
        const float2 nm = f2(-m0);
        float2 e1 = f2(0.f), e2 = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (FULL || t + k * STRIDE < P) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 e = __fadd2_rn(v[k][h], nm);
                    v[k][h] = e;
                    e1 = __fadd2_rn(e1, e);
                    e2 = __ffma2_rn(e, e, e2);
                }
            }
        }
        const float2 E = red.sum2(make_float2(e1.x + e1.y, e2.x + e2.y));
        c = E.x * invN;
        const float var = fmaxf(fmaf(-c, c, E.y * invN), 0.f);
        rstd = rsqrtf(var + a.eps);
        if (t == 0 && lead) {
            if (a.mean) a.mean[row] = m0 + c;
            if (a.rstd) a.rstd[row] = rstd;
        }
    } else {
        float2 ss = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
#pragma unroll
            for (int h = 0; h < H; ++h) ss = __ffma2_rn(v[k][h], v[k][h], ss);
        rstd = rsqrtf(fmaf(red.sum(ss.x + ss.y), invN, a.eps));
        after_sync();
        if (t == 0 && lead && a.rstd) a.rstd[row] = rstd;
    }

    // ---- S7/S8: parameters, normalize, round once, store ----
    const float2 r2 = f2(rstd), nc = f2(-c);
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int idx = t + k * STRIDE;
        if (FULL || idx < P) {
            float2 out[H], g[H];
            prm.p0_pack(idx, g);
            if (OP == OP_LN) {
                float2 b[H];
                prm.p1_pack(idx, b);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    out[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(v[k][h], nc), r2), g[h], b[h]);
            } else {
#pragma unroll
                for (int h = 0; h < H; ++h) out[h] = __fmul2_rn(__fmul2_rn(v[k][h], r2), g[h]);
            }
            st_stream(Y + (size_t)idx * V, io2::pack(out));
        }
    }
}

// Issue every load of one row (S1/S2) before any arithmetic.
template <int OP, int PACKS, int STRIDE, class Src, bool FULL = false>
__device__ __forceinline__ void row_load(const Src &src, const int t, const int P,
                                         uint4 (&rx)[PACKS], uint4 (&rr)[PACKS]) {
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int idx = t + k * STRIDE;
        if (FULL || idx < P) {
            rx[k] = src.x_pack(idx);
            if (OP == OP_ADD_RMS) rr[k] = src.r_pack(idx);
        }
    }
}

// One row: load, then compute.
template <int OP, typename T, int PACKS, int STRIDE, class Red, class Src, class Prm, class Hook,
          bool FULL = false>
__device__ __forceinline__ void row_body(const RowArgs &a, const int64_t row, const int t,
                                         Red &red, const Src &src, const Prm &prm,
                                         const Hook &after_sync, const bool lead = true) {
    uint4 rx[PACKS], rr[PACKS];
    row_load<OP, PACKS, STRIDE, Src, FULL>(src, t, (int)(a.N / IO<T>::V), rx, rr);
    row_compute<OP, T, PACKS, STRIDE, Red, Prm, Hook, FULL>(a, row, t, red, rx, rr, prm, after_sync,
                                                           lead);
}

// Resident CTAs per SM the CTA and persistent kernels are compiled for
// (__launch_bounds__ minimum blocks, which caps registers at 65536 /
// (CTAs x THREADS)), measured on GB300 with cold L2:
//  * at most 2 packs per thread: 1280 threads per SM (five 256-thread CTAs,
//    at most 51 registers) kept the most row loads in flight; 1024 and 1536
//    were slower (add+RMSNorm 4096 x 4096 bf16: 19.17 us against 19.90 and
//    19.27); plain RMSNorm 1024 threads (2048 x 4096 fp16: 5.92 us against
//    6.18 at 1280 and 6.15 at 1536);
//  * LayerNorm with 4 packs per thread in CTAs of at most 256 threads: 896
//    threads (seven 128-thread CTAs, at most 73 registers): 12.3 us at
//    4096 x 4096 bf16 against 13.4 us uncapped (92 registers, five CTAs) and
//    12.9 / 12.7 us at six / eight; the exact-row instance (no bounds tests,
//    no spills at 64 registers) 1024 threads: eight CTAs, 10.17-10.19 us
//    against 10.39-10.40 us at seven (with the row requested before the
//    dependent-launch wait);
//  * anything else is left uncapped (caps made it spill or run slower; the
//    persistent 512 x 4 LayerNorm at 16384 bf16 runs 13.98 us uncapped at 96
//    registers, one CTA per SM, and 15.9 us capped to two CTAs).
// NRM_CTA_MIN_THREADS / NRM_RMS_MIN_THREADS / NRM_LN4_MIN_THREADS /
// NRM_LN4_FULL_MIN_THREADS override the caps for experiments.
#ifndef NRM_CTA_MIN_THREADS
#define NRM_CTA_MIN_THREADS 1280
#endif
#ifndef NRM_ROW_PDL
#define NRM_ROW_PDL 1
#endif
#ifndef NRM_LN4_MIN_THREADS
#define NRM_LN4_MIN_THREADS 896
#endif
#ifndef NRM_LN4_FULL_MIN_THREADS
#define NRM_LN4_FULL_MIN_THREADS 1024
#endif
#ifndef NRM_RMS_MIN_THREADS
#define NRM_RMS_MIN_THREADS 1024
#endif
// Launch with programmatic stream serialization when NRM_ROW_PDL (the
// kernels then order themselves with griddepcontrol.wait).
template <typename K, typename... Args>
inline cudaError_t launch_row(K kernel, unsigned grid, unsigned threads, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = NRM_ROW_PDL ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int OP, int THREADS, int PACKS, bool FULL = false>
constexpr int row_min_blocks() {
    return (OP == OP_RMS && PACKS <= 2 && NRM_RMS_MIN_THREADS / THREADS > 0) ? NRM_RMS_MIN_THREADS / THREADS
           : (PACKS <= 2 && NRM_CTA_MIN_THREADS / THREADS > 0) ? NRM_CTA_MIN_THREADS / THREADS
           : (OP != OP_ADD_RMS && PACKS == 4 && THREADS <= 512 && FULL &&
              NRM_LN4_FULL_MIN_THREADS / THREADS > 0)
               ? NRM_LN4_FULL_MIN_THREADS / THREADS
           : (OP == OP_LN && PACKS == 4 && THREADS <= 256 && NRM_LN4_MIN_THREADS / THREADS > 0)
               ? NRM_LN4_MIN_THREADS / THREADS
               : 1;
}

template <int OP, typename T, int THREADS, int PACKS, bool FULL = false>
__global__ void __launch_bounds__(THREADS, (row_min_blocks<OP, THREADS, PACKS, FULL>()))
    row_cta_kernel(const RowArgs a, const int64_t pf) {
    constexpr int NW = THREADS / 32;
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    const T *X = static_cast<const T *>(a.x);
    const T *R = static_cast<const T *>(a.res);
#if NRM_ROW_PDL
    // launched as a programmatic dependent: wait for the previous grid on the
    // stream (its outputs may be this call's inputs), then let the next one
    // get its CTAs resident while this grid runs.  A CTA that becomes
    // resident while the previous grid still runs first asks L2 for its own
    // row: L2 is where writes become coherent, so data the previous grid
    // writes afterwards still reaches the loads issued after the wait.
    if (pf > 0 && threadIdx.x == 0 && blockIdx.x < a.rows) {
        const uint32_t bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
        prefetch_l2_bulk(X + blockIdx.x * a.ldx, bytes);
        if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + blockIdx.x * a.ldr, bytes);
    }
    pdl_wait();
    pdl_launch_dependents();
#endif
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
        if (pf > 0 && threadIdx.x == 0 && row + pf < a.rows) {
            const uint32_t bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
            prefetch_l2_bulk(X + (row + pf) * a.ldx, bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + (row + pf) * a.ldr, bytes);
        }
        CtaRed<NW> red{&s1[parity][0], &s2[parity][0]};
        const GlobalSrc<T> src{X + row * a.ldx, R + row * a.ldr};
        const GlobalParams<T> prm{static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
        row_body<OP, T, PACKS, THREADS, CtaRed<NW>, GlobalSrc<T>, GlobalParams<T>, NoHook, FULL>(
            a, row, threadIdx.x, red, src, prm, NoHook{});
    }
}

// ---------------------------------------------------------------------------
// Cluster split: one row over the CS CTAs of a thread-block cluster (the
// LayerNorm walkthrough, lpnh.cn/news/2756757, §1.1 and §4.1, splits a row
// that outgrows one block across several; here the blocks are a cluster and
// their partial sums meet in distributed shared memory).  CTA rank r holds
// the contiguous slice [r S, (r+1) S) of the row's P = CS S packs in
// registers (x still read from HBM once); each row-wide sum is a CTA sum,
// published in the CTA's shared memory, a cluster barrier, and a read of the
// CS partials in rank order (lane k of every warp reads rank k's partial,
// then shuffles), so every thread of the cluster gets the same bits.  It
// serves rows too long for one CTA's registers and grids with too few rows
// to fill the SMs.
// ---------------------------------------------------------------------------
// Sum of the CS CTAs' published partials, rank order, same bits in every lane.
template <int CS>
__device__ __forceinline__ float cluster_gather_sum(const float *slot) {
    const int lane = threadIdx.x & 31;
    const float mine = lane < CS ? ld_dsmem(slot, (uint32_t)lane) : 0.f;
    float r = __shfl_sync(0xffffffffu, mine, 0);
#pragma unroll
    for (int k = 1; k < CS; ++k) r += __shfl_sync(0xffffffffu, mine, k);
    return r;
}

template <int NW, int CS> struct ClusterRed {
    float *s1;    // CTA-level exchange slots (CtaRed's)
    float2 *s2;
    float *c1;    // this CTA's published partials: c1[0]; c2[0], c2[1]
    float *c2;
    __device__ __forceinline__ float sum(float v) {
        const float t = cta_sum_all<NW>(v, s1);
        if (threadIdx.x == 0) c1[0] = t;
        cluster_arrive();
        cluster_wait();
        return cluster_gather_sum<CS>(c1);
    }
    __device__ __forceinline__ float2 sum2(float2 v) {
        const float2 t = cta_sum_all<NW>(v, s2);
        if (threadIdx.x == 0) {
            c2[0] = t.x;
            c2[1] = t.y;
        }
        cluster_arrive();
        cluster_wait();
        return make_float2(cluster_gather_sum<CS>(c2), cluster_gather_sum<CS>(c2 + 1));
    }
};

// Persistent clusters: cluster k handles rows k, k + G/CS, ... (G/CS = the
// clusters that fit at once), asking L2 for its next row while it reduces
// the current one.  A partial slot of one parity is rewritten two rows
// later, after at least one more cluster barrier, which every peer reaches
// only once its reads of that slot are done; a last cluster barrier keeps
// every CTA resident until its peers have read its partials.
template <int OP, typename T, int THREADS, int PACKS, int CS, bool FULL>
__global__ void __launch_bounds__(THREADS, (row_min_blocks<OP, THREADS, PACKS, FULL>()))
    row_cluster_kernel(const RowArgs a) {
    constexpr int NW = THREADS / 32;
    constexpr int V = IO<T>::V;
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    __shared__ float c1[2][1];
    __shared__ float c2[2][2];
    const int rank = (int)cluster_rank();
    const int64_t ncl = gridDim.x / CS;
    const int S = (int)(a.N / V) / CS;          // packs per CTA slice
    const int64_t off = (int64_t)rank * S * V;  // first element of this CTA's slice
    RowArgs b = a;
    b.N = (int64_t)S * V;  // the slice (a.fN, a.invN stay those of the row)
    b.y = static_cast<T *>(a.y) + off;
    if (OP == OP_ADD_RMS) b.res_out = static_cast<T *>(a.res_out) + off;
    const T *X = static_cast<const T *>(a.x) + off;
    const T *R = OP == OP_ADD_RMS ? static_cast<const T *>(a.res) + off : nullptr;
    const T *P0 = a.p0 ? static_cast<const T *>(a.p0) + off : nullptr;
    const T *P1 = a.p1 ? static_cast<const T *>(a.p1) + off : nullptr;
    const int64_t first = blockIdx.x / CS;
#if NRM_ROW_PDL
    // as row_cta_kernel: the CTA's slice of its first row is requested from
    // L2 before the wait for the previous grid
    if (threadIdx.x == 0 && first < a.rows) {
        const uint32_t bytes = (uint32_t)S * 16u;
        prefetch_l2_bulk(X + first * a.ldx, bytes);
        if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + first * a.ldr, bytes);
    }
    pdl_wait();
    pdl_launch_dependents();
#endif
    int parity = 0;
    for (int64_t row = first; row < a.rows; row += ncl, parity ^= 1) {
        // the cluster's next row is requested from L2 while this one is reduced
        if (threadIdx.x == 0 && row + ncl < a.rows) {
            const uint32_t bytes = (uint32_t)S * 16u;
            prefetch_l2_bulk(X + (row + ncl) * a.ldx, bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + (row + ncl) * a.ldr, bytes);
        }
        ClusterRed<NW, CS> red{&s1[parity][0], &s2[parity][0], &c1[parity][0], &c2[parity][0]};
        const GlobalSrc<T> src{X + row * a.ldx, OP == OP_ADD_RMS ? R + row * a.ldr : nullptr};
        const GlobalParams<T> prm{P0, P1};
        row_body<OP, T, PACKS, THREADS, ClusterRed<NW, CS>, GlobalSrc<T>, GlobalParams<T>, NoHook,
                 FULL>(b, row, threadIdx.x, red, src, prm, NoHook{}, rank == 0);
    }
    cluster_arrive();
    cluster_wait();
}

// Persistent register pipeline: CTA b handles rows b, b + G, ... (G =
// gridDim.x, as many CTAs as are resident).  Row r + G's packs are loaded
// into registers before row r is reduced, so every CTA always has a row in
// flight; parameters are widened to binary32 in shared memory once per CTA
// (SmemParams layout) when smem_params is set.  With pf_waves > 0, thread 0
// also asks L2 for the row pf_waves rows beyond the one in registers, so the
// register prefetch of later rows hits L2.
template <int OP, typename T, int THREADS, int PACKS>
__global__ void __launch_bounds__(THREADS, (row_min_blocks<OP, THREADS, PACKS>()))
    row_persist_kernel(const RowArgs a, const int smem_params, const int pf_waves) {
    constexpr int NW = THREADS / 32;
    extern __shared__ __align__(16) float4 sparams[];
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    const int P = (int)(a.N / IO<T>::V);
    const T *X = static_cast<const T *>(a.x);
    const T *R = static_cast<const T *>(a.res);
#if NRM_ROW_PDL
    // programmatic dependent launch, as row_cta_kernel: the CTA's first two
    // rows are requested from L2 before the wait for the previous grid
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
        for (int64_t r = blockIdx.x; r < a.rows && r < (int64_t)blockIdx.x + 2 * gridDim.x; r += gridDim.x) {
            prefetch_l2_bulk(X + r * a.ldx, bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + r * a.ldr, bytes);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
#endif
    if (smem_params)
        fill_smem_params<T, (OP == OP_LN ? 2 : 1), THREADS>(a, reinterpret_cast<float *>(sparams));
    __syncthreads();
    const SmemParams<T> sprm{sparams, P};
    const GlobalParams<T> gprm{static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
    const int64_t G = gridDim.x;
    const int64_t pf = (int64_t)(pf_waves + 1) * G;
    const uint32_t row_bytes = (uint32_t)(a.N * (int64_t)sizeof(T));

    uint4 rx[PACKS], rr[PACKS];
    int64_t row = blockIdx.x;
    if (row < a.rows) {
        const GlobalSrc<T> src{X + row * a.ldx, R + row * a.ldr};
        row_load<OP, PACKS, THREADS>(src, threadIdx.x, P, rx, rr);
    }
    int parity = 0;
    for (; row < a.rows; row += G, parity ^= 1) {
        if (pf_waves > 0 && threadIdx.x == 0 && row + pf < a.rows) {
            prefetch_l2_bulk(X + (row + pf) * a.ldx, row_bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + (row + pf) * a.ldr, row_bytes);
        }
        uint4 nx[PACKS], nr[PACKS];
        const int64_t next = row + G;
        if (next < a.rows) {
            const GlobalSrc<T> src{X + next * a.ldx, R + next * a.ldr};
            row_load<OP, PACKS, THREADS>(src, threadIdx.x, P, nx, nr);
        }
        CtaRed<NW> red{&s1[parity][0], &s2[parity][0]};
        if (smem_params)
            row_compute<OP, T, PACKS, THREADS>(a, row, threadIdx.x, red, rx, rr, sprm, NoHook{});
        else
            row_compute<OP, T, PACKS, THREADS>(a, row, threadIdx.x, red, rx, rr, gprm, NoHook{});
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            rx[k] = nx[k];
            if (OP == OP_ADD_RMS) rr[k] = nr[k];
        }
    }
}

// Warp per row, raw packs in registers: each warp owns whole rows (row r of
// the grid-stride loop), issues all PACKS 16-byte loads of its row at once
// (a whole 4096-wide bf16 row, 8 KB, in flight per warp), reduces with
// shuffles only -- no CTA barrier -- and unpacks the packs again for each
// pass instead of holding binary32 copies.  The CTA's warps share the
// parameters widened to binary32 in shared memory (when smem_params).
// Sized so that an SM keeps well over 100 KB of row loads in flight, which
// GB300's loaded memory latency needs to stream at HBM speed.
template <int OP, typename T, int PACKS, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) row_wraw_kernel(const RowArgs a, const int smem_params,
                                                              const int pf_waves) {
    using io2 = IO2<T>;
    constexpr int V = IO<T>::V;
    constexpr int H = io2::H;
    extern __shared__ __align__(16) float4 sparams[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int P = (int)(a.N / V);
    const float fN = a.fN, invN = a.invN;
#if NRM_ROW_PDL
    // programmatic dependent launch, as row_cta_kernel: each warp's first row
    // is requested from L2 before the wait for the previous grid
    {
        const int64_t r0 = (int64_t)blockIdx.x * WARPS + warp;
        if (lane == 0 && r0 < a.rows) {
            const uint32_t bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
            prefetch_l2_bulk(static_cast<const T *>(a.x) + r0 * a.ldx, bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(static_cast<const T *>(a.res) + r0 * a.ldr, bytes);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
#endif
    if (smem_params)
        fill_smem_params<T, (OP == OP_LN ? 2 : 1), WARPS * 32>(a, reinterpret_cast<float *>(sparams));
    __syncthreads();
    const SmemParams<T> sprm{sparams, P};
    const GlobalParams<T> gprm{static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
    const T *X = static_cast<const T *>(a.x);
    const T *R = static_cast<const T *>(a.res);

    const int64_t pf = (int64_t)pf_waves * gridDim.x * WARPS;
    for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < a.rows;
         row += (int64_t)gridDim.x * WARPS) {
        if (pf > 0 && lane == 0 && row + pf < a.rows) {
            const uint32_t bytes = (uint32_t)(a.N * (int64_t)sizeof(T));
            prefetch_l2_bulk(X + (row + pf) * a.ldx, bytes);
            if (OP == OP_ADD_RMS) prefetch_l2_bulk(R + (row + pf) * a.ldr, bytes);
        }
        const T *xr = X + row * a.ldx;
        uint4 raw[PACKS];
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
            if (lane + 32 * k < P) raw[k] = ld_stream(xr + (size_t)(lane + 32 * k) * V);
        if (OP == OP_ADD_RMS) {
            const T *rr = R + row * a.ldr;
            T *RO = static_cast<T *>(a.res_out) + row * a.ldro;
#pragma unroll
            for (int k = 0; k < PACKS; ++k) {
                const int idx = lane + 32 * k;
                if (idx < P) {
                    float2 fx[H], fr[H];
                    io2::unpack(raw[k], fx);
                    io2::unpack(ld_stream(rr + (size_t)idx * V), fr);
#pragma unroll
                    for (int h = 0; h < H; ++h) fx[h] = __fadd2_rn(fx[h], fr[h]);
                    raw[k] = io2::pack(fx);  // round once to T
                    st_stream(RO + (size_t)idx * V, raw[k]);
                }
            }
        }
        // pass 1
        float2 acc = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (lane + 32 * k < P) {
                float2 f[H];
                io2::unpack(raw[k], f);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    acc = (OP == OP_LN) ? __fadd2_rn(acc, f[h]) : __ffma2_rn(f[h], f[h], acc);
            }
        }
        const float tot = warp_sum_all(acc.x + acc.y);
        float rstd, m0 = 0.f, c = 0.f;
        if (OP == OP_LN) {
            m0 = tot * invN;
            m0 = fmaf(fmaf(-m0, fN, tot), invN, m0);  // exact for constant rows
            const float2 nm = f2(-m0);
            float2 e1 = f2(0.f), e2 = f2(0.f);
#pragma unroll
            for (int k = 0; k < PACKS; ++k) {
                if (lane + 32 * k < P) {
                    float2 f[H];
                    io2::unpack(raw[k], f);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 e = __fadd2_rn(f[h], nm);
                        e1 = __fadd2_rn(e1, e);
                        e2 = __ffma2_rn(e, e, e2);
                    }
                }
            }
            const float2 E = warp_sum_all(make_float2(e1.x + e1.y, e2.x + e2.y));
            c = E.x * invN;
            const float var = fmaxf(fmaf(-c, c, E.y * invN), 0.f);
            rstd = rsqrtf(var + a.eps);
            if (lane == 0) {
                if (a.mean) a.mean[row] = m0 + c;
                if (a.rstd) a.rstd[row] = rstd;
            }
        } else {
            rstd = rsqrtf(fmaf(tot, invN, a.eps));
            if (lane == 0 && a.rstd) a.rstd[row] = rstd;
        }
        // pass 3: normalize, scale (and shift), round once, store
        T *Y = static_cast<T *>(a.y) + row * a.ldy;
        const float2 r2 = f2(rstd), nm = f2(-m0), nc = f2(-c);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            const int idx = lane + 32 * k;
            if (idx < P) {
                float2 f[H], g2[H], out[H];
                io2::unpack(raw[k], f);
                if (smem_params) sprm.p0_pack(idx, g2);
                else gprm.p0_pack(idx, g2);
                if (OP == OP_LN) {
                    float2 b2[H];
                    if (smem_params) sprm.p1_pack(idx, b2);
                    else gprm.p1_pack(idx, b2);
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        out[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(__fadd2_rn(f[h], nm), nc), r2),
                                            g2[h], b2[h]);
                } else {
#pragma unroll
                    for (int h = 0; h < H; ++h) out[h] = __fmul2_rn(__fmul2_rn(f[h], r2), g2[h]);
                }
                st_stream(Y + (size_t)idx * V, io2::pack(out));
            }
        }
    }
}

#include "row_pipe.cuh"

template <int OP, typename T, int PACKS, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) row_warp_kernel(const RowArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    WarpRed red;
    const T *X = static_cast<const T *>(a.x);
    const T *R = static_cast<const T *>(a.res);
    for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < a.rows;
         row += (int64_t)gridDim.x * WARPS) {
        const GlobalSrc<T> src{X + row * a.ldx, R + row * a.ldr};
        const GlobalParams<T> prm{static_cast<const T *>(a.p0), static_cast<const T *>(a.p1)};
        row_body<OP, T, PACKS, 32>(a, row, lane, red, src, prm, NoHook{});
    }
}

// Scalar fallback for any N and any (element-aligned) pointers.  Pass 1 keeps
// a Welford recurrence per thread over d = x - K (LayerNorm) or a sum of
// squares (RMS ops), writing residual_out on the way; pass 2 re-reads the row
// (x, or the residual_out this same thread wrote) and writes y.
template <int OP, typename T, int THREADS>
__global__ void __launch_bounds__(THREADS) row_generic_kernel(const RowArgs a) {
    using io = IO<T>;
    constexpr int NW = THREADS / 32;
    __shared__ float s_red[2][NW][3];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const float fN = (float)a.N;
    const T *__restrict__ X = static_cast<const T *>(a.x);
    const T *R = static_cast<const T *>(a.res);
    const T *__restrict__ G = static_cast<const T *>(a.p0);
    const T *__restrict__ Bt = static_cast<const T *>(a.p1);
    T *__restrict__ Y = static_cast<T *>(a.y);
    T *RO = static_cast<T *>(a.res_out);  // may alias R

    int buf = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, buf ^= 1) {
        const int64_t bx = row * a.ldx, br = row * a.ldr, bro = row * a.ldro, by = row * a.ldy;
        const float K = (OP == OP_LN) ? io::to_f(X[bx]) : 0.f;
        float n = 0.f, mean = 0.f, m2 = 0.f, ss = 0.f;
        for (int64_t i = tid; i < a.N; i += THREADS) {
            float v;
            if (OP == OP_ADD_RMS) {
                const T r = io::from_f(__fadd_rn(io::to_f(X[bx + i]), io::to_f(R[br + i])));
                RO[bro + i] = r;
                v = io::to_f(r);
            } else {
                v = io::to_f(X[bx + i]);
            }
            if (OP == OP_LN) {
                const float d = v - K;
                n += 1.f;
                const float delta = d - mean;
                mean += delta / n;
                m2 = fmaf(delta, d - mean, m2);
            } else {
                ss = fmaf(v, v, ss);
            }
        }
        float r0, r1 = 0.f, r2 = 0.f;
        if (OP == OP_LN) {
            Stats st = warp_stats_down(Stats{n, mean, m2});
            r0 = st.n; r1 = st.mean; r2 = st.m2;
        } else {
            r0 = warp_sum_down(ss);
        }
        if (lane == 0) {
            s_red[buf][warp][0] = r0;
            s_red[buf][warp][1] = r1;
            s_red[buf][warp][2] = r2;
        }
        __syncthreads();
        float rstd, shift = 0.f;
        if (OP == OP_LN) {
            Stats st{s_red[buf][0][0], s_red[buf][0][1], s_red[buf][0][2]};
            for (int w = 1; w < NW; ++w)
                st = combine(st, Stats{s_red[buf][w][0], s_red[buf][w][1], s_red[buf][w][2]});
            rstd = 1.0f / sqrtf(st.m2 / fN + a.eps);
            shift = st.mean;
            if (tid == 0) {
                if (a.mean) a.mean[row] = K + st.mean;
                if (a.rstd) a.rstd[row] = rstd;
            }
        } else {
            float tot = s_red[buf][0][0];
            for (int w = 1; w < NW; ++w) tot += s_red[buf][w][0];
            rstd = 1.0f / sqrtf(tot / fN + a.eps);
            if (tid == 0 && a.rstd) a.rstd[row] = rstd;
        }
        for (int64_t i = tid; i < a.N; i += THREADS) {
            float out;
            if (OP == OP_LN) {
                const float g = G ? io::to_f(G[i]) : 1.f;
                const float b = Bt ? io::to_f(Bt[i]) : 0.f;
                const float t = (io::to_f(X[bx + i]) - K) - shift;
                out = fmaf(t * rstd, g, b);
            } else {
                const float v = (OP == OP_ADD_RMS) ? io::to_f(RO[bro + i]) : io::to_f(X[bx + i]);
                const float w = G ? io::to_f(G[i]) : 1.f;
                out = (v * rstd) * w;
            }
            Y[by + i] = io::from_f(out);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch switch: Plan -> template instance.
// ---------------------------------------------------------------------------

// Row-group pipeline launch: dynamic shared memory = parameters (binary32,
// when smem_params) + groups x stages x stage bytes; grid = min(rows, SMs x
// resident CTAs per SM).  The shared-memory opt-in and the occupancy are
// computed once per device and size (per kernel instance), under a lock.
template <int OP, typename T, int GT, int PACKS, int G>
cudaError_t launch_pipe(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = row_pipe_kernel<OP, T, GT, PACKS, G>;
    if (p.stages < 2 || p.stages > kMaxStages || !a.fault || p.sms < 1)
        return cudaErrorInvalidConfiguration;
    const size_t stage = (size_t)a.N * sizeof(T) * (OP == OP_ADD_RMS ? 2 : 1);
    const size_t params = params_smem_bytes<OP, T>(p.smem_params, a.N);
    const size_t smem = params + stage * (size_t)p.stages * G;
    if (smem > (size_t)kSmemMax) return cudaErrorInvalidConfiguration;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), GT * G, smem, &per_sm);
    if (oe != cudaSuccess) return oe;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)p.sms * per_sm;
    const int64_t grid = a.rows < slots ? a.rows : slots;
    return launch_row(kernel, (unsigned)grid, GT * G, smem, s, a, p.stages, p.smem_params);
}

// Persistent launch: dynamic shared memory = parameters in
// binary32 (when smem_params), grid = min(rows, SMs x resident CTAs per SM).
template <int OP, typename T, int THREADS, int PACKS>
cudaError_t launch_persist(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = row_persist_kernel<OP, T, THREADS, PACKS>;
    if (p.sms < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = p.smem_params ? (size_t)a.N * sizeof(float) * (OP == OP_LN ? 2 : 1) : 0;
    if (smem > (size_t)kSmemMax) return cudaErrorInvalidConfiguration;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), THREADS, smem, &per_sm);
    if (oe != cudaSuccess) return oe;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)p.sms * per_sm;
    const int64_t grid = a.rows < slots ? a.rows : slots;
    return launch_row(kernel, (unsigned)grid, THREADS, smem, s, a, p.smem_params, p.prefetch);
}

// Warp-per-row launch: dynamic shared memory = parameters in binary32 (when
// smem_params), grid = min(ceil(rows / WARPS), SMs x resident CTAs per SM).
template <int OP, typename T, int PACKS, int WARPS>
cudaError_t launch_wraw(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = row_wraw_kernel<OP, T, PACKS, WARPS>;
    if (p.sms < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = p.smem_params ? (size_t)a.N * sizeof(float) * (OP == OP_LN ? 2 : 1) : 0;
    if (smem > (size_t)kSmemMax) return cudaErrorInvalidConfiguration;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), WARPS * 32, smem, &per_sm);
    if (oe != cudaSuccess) return oe;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t need = (a.rows + WARPS - 1) / WARPS;
    const int64_t slots = (int64_t)p.sms * per_sm;
    const int64_t grid = need < slots ? need : slots;
    return launch_row(kernel, (unsigned)grid, WARPS * 32, smem, s, a, p.smem_params, p.prefetch);
}

// CTA-per-row launch: grid = rows (clamped); the L2 prefetch distance is
// p.prefetch waves of resident CTAs (occupancy computed once per device and
// kernel instance).
template <int OP, typename T, int THREADS, int PACKS, bool FULL = false>
cudaError_t launch_cta(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = row_cta_kernel<OP, T, THREADS, PACKS, FULL>;
    int64_t pf = 0;
    if (p.prefetch > 0) {
        int per_sm = 0;
        const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), THREADS, 0, &per_sm);
        if (oe != cudaSuccess) return oe;
        pf = (int64_t)p.prefetch * p.sms * per_sm;
    }
#if NRM_ROW_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, pf);
    return e == cudaSuccess ? cudaGetLastError() : e;
#else
    kernel<<<(unsigned)p.grid, THREADS, 0, s>>>(a, pf);
    return cudaGetLastError();
#endif
}

// Cluster-split launch: as many clusters of CS CTAs as are resident at once
// (at most one per row); needs P divisible by CS (checked by the plan choice).
template <int OP, typename T, int THREADS, int PACKS, int CS, bool FULL>
cudaError_t launch_cluster(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = row_cluster_kernel<OP, T, THREADS, PACKS, CS, FULL>;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), THREADS, 0, &per_sm);
    if (oe != cudaSuccess) return oe;
    const int64_t resident = (int64_t)p.sms * (per_sm > 0 ? per_sm : 1) / CS;
    cudaLaunchConfig_t cfg = {};
    int64_t clusters = a.rows < resident ? a.rows : resident;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3((unsigned)(clusters * CS));
    cfg.blockDim = dim3(THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = NRM_ROW_PDL ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int OP, typename T>
cudaError_t launch_row(const RowArgs &a, const Plan &p, cudaStream_t s) {
    const dim3 grid((unsigned)p.grid);
    if (p.kind == PLAN_GENERIC) {
        switch (p.threads) {
        case 128: row_generic_kernel<OP, T, 128><<<grid, 128, 0, s>>>(a); break;
        case 256: row_generic_kernel<OP, T, 256><<<grid, 256, 0, s>>>(a); break;
        case 512: row_generic_kernel<OP, T, 512><<<grid, 512, 0, s>>>(a); break;
        default: return cudaErrorInvalidConfiguration;
        }
    } else if (p.kind == PLAN_WARP) {
        if (p.threads != 128) return cudaErrorInvalidConfiguration;
        switch (p.packs) {
        case 1: row_warp_kernel<OP, T, 1, 4><<<grid, 128, 0, s>>>(a); break;
        case 2: row_warp_kernel<OP, T, 2, 4><<<grid, 128, 0, s>>>(a); break;
        case 4: row_warp_kernel<OP, T, 4, 4><<<grid, 128, 0, s>>>(a); break;
        case 8: row_warp_kernel<OP, T, 8, 4><<<grid, 128, 0, s>>>(a); break;
        default: return cudaErrorInvalidConfiguration;
        }
    } else if (p.kind == PLAN_CTA) {
#define NRM_CTA_CASE(TH, PK)                                                       \
    if (p.threads == TH && p.packs == PK) return launch_cta<OP, T, TH, PK>(a, p, s);
// the automatic shapes at power-of-two N also come without bounds tests
// (LayerNorm 4096x4096 bf16 12.2 -> 11.4 us; RMSNorm measured 2 % slower
// that way, so it keeps the tested form)
#define NRM_CTA_FULL_CASE(TH, PK)                                                  \
    if ((OP != OP_RMS || (PK == 4 && TH == 128)) && p.threads == TH && p.packs == PK && \
        a.N / IO<T>::V == TH * PK)                                                  \
        return launch_cta<OP, T, TH, PK, true>(a, p, s);
        NRM_CTA_FULL_CASE(128, 4) NRM_CTA_FULL_CASE(256, 2) NRM_CTA_FULL_CASE(256, 4)
        NRM_CTA_FULL_CASE(512, 4)
#undef NRM_CTA_FULL_CASE
        NRM_CTA_CASE(128, 1) NRM_CTA_CASE(256, 1) NRM_CTA_CASE(512, 1) NRM_CTA_CASE(1024, 1)
        NRM_CTA_CASE(128, 2) NRM_CTA_CASE(256, 2) NRM_CTA_CASE(512, 2) NRM_CTA_CASE(1024, 2)
        NRM_CTA_CASE(128, 4) NRM_CTA_CASE(256, 4) NRM_CTA_CASE(512, 4) NRM_CTA_CASE(1024, 4)
#undef NRM_CTA_CASE
        return cudaErrorInvalidConfiguration;
    } else if (p.kind == PLAN_CLUSTER) {
        // p.groups = CTAs per cluster; the slice is exactly THREADS x PACKS
        // packs (FULL, no bounds tests) or fits it
#define NRM_CLUSTER_CASE(TH, PK, CS)                                               \
    if (p.threads == TH && p.packs == PK && p.groups == CS) {                      \
        if (a.N / IO<T>::V == (int64_t)TH * PK * CS)                              \
            return launch_cluster<OP, T, TH, PK, CS, true>(a, p, s);              \
        return launch_cluster<OP, T, TH, PK, CS, false>(a, p, s);                 \
    }
        NRM_CLUSTER_CASE(128, 1, 2) NRM_CLUSTER_CASE(128, 1, 4) NRM_CLUSTER_CASE(128, 2, 2)
        NRM_CLUSTER_CASE(128, 2, 4) NRM_CLUSTER_CASE(128, 4, 2) NRM_CLUSTER_CASE(128, 4, 4)
        NRM_CLUSTER_CASE(128, 4, 8) NRM_CLUSTER_CASE(256, 4, 2)
#undef NRM_CLUSTER_CASE
        return cudaErrorInvalidConfiguration;
    } else if (p.kind == PLAN_WRAW) {
#define NRM_WRAW_CASE(PK, WP)                                                      \
    if (p.packs == PK && p.threads == WP * 32) return launch_wraw<OP, T, PK, WP>(a, p, s);
        NRM_WRAW_CASE(4, 8) NRM_WRAW_CASE(8, 8) NRM_WRAW_CASE(16, 8) NRM_WRAW_CASE(16, 16)
        NRM_WRAW_CASE(8, 16) NRM_WRAW_CASE(32, 8)
#undef NRM_WRAW_CASE
        return cudaErrorInvalidConfiguration;
    } else if (p.kind == PLAN_PERSIST) {
#define NRM_PERSIST_CASE(TH, PK)                                                   \
    if (p.threads == TH && p.packs == PK) return launch_persist<OP, T, TH, PK>(a, p, s);
        NRM_PERSIST_CASE(128, 4) NRM_PERSIST_CASE(256, 1) NRM_PERSIST_CASE(256, 2)
        NRM_PERSIST_CASE(256, 4) NRM_PERSIST_CASE(512, 1) NRM_PERSIST_CASE(512, 2)
        NRM_PERSIST_CASE(512, 4) NRM_PERSIST_CASE(1024, 2)
#undef NRM_PERSIST_CASE
        return cudaErrorInvalidConfiguration;
    } else if (p.kind == PLAN_TMA) {
#define NRM_PIPE_CASE(GT, PK, GR)                                                  \
    if (p.threads == GT && p.packs == PK && p.groups == GR)                        \
        return launch_pipe<OP, T, GT, PK, GR>(a, p, s);
        NRM_PIPE_CASE(128, 4, 1) NRM_PIPE_CASE(128, 4, 2) NRM_PIPE_CASE(128, 4, 4)
        NRM_PIPE_CASE(128, 4, 8) NRM_PIPE_CASE(128, 8, 1) NRM_PIPE_CASE(128, 8, 2)
        NRM_PIPE_CASE(128, 8, 4) NRM_PIPE_CASE(256, 2, 1) NRM_PIPE_CASE(256, 2, 2)
        NRM_PIPE_CASE(256, 2, 4) NRM_PIPE_CASE(256, 4, 1) NRM_PIPE_CASE(256, 4, 2)
        NRM_PIPE_CASE(256, 4, 4) NRM_PIPE_CASE(512, 4, 1) NRM_PIPE_CASE(512, 4, 2)
#undef NRM_PIPE_CASE
        return cudaErrorInvalidConfiguration;
    } else {
        return cudaErrorInvalidConfiguration;
    }
    return cudaGetLastError();
}

}  // namespace nrm
