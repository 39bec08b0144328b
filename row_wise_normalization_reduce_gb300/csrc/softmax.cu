// softmax.cu -- row softmax over [rows, N], the same reduce-then-normalize
// pattern as the norms (LLM-ops page, smarter.xin, section 1 "Softmax"):
//
//   m = max_j x_j,   d = sum_j exp(x_j - m),   y_i = exp(x_i - m) / d
//
// The page's online form keeps a running (max, sum) pair and merges two pairs
// by rescaling both sums to the larger max:
//   (ma, da) + (mb, db) = (M, da * exp(ma - M) + db * exp(mb - M)),  M = max(ma, mb).
//
// CTA plan: one CTA per row holds the row in registers.  Each thread takes
// the max of its own values, then e_i = exp(x_i - m_t) and their sum d_t (one
// exponential per element); the (m_t, d_t) pairs are merged with the rule
// above by a warp butterfly and one shared-memory exchange (so the row needs
// a single CTA-wide reduction, not a max and then a sum), and the output is
// y_i = e_i * (exp(m_t - m) / d), one multiply per element.  Rows of the next
// wave are prefetched into L2 as in the norm kernels.
//
// Cluster plan: the same with one row split over the CS CTAs of a
// thread-block cluster, CTA rank r holding the contiguous slice [r S, (r+1) S)
// of the row's packs; after its CTA-wide merge each CTA publishes its
// (max, sum) pair in shared memory, and after a cluster barrier every warp
// reads the CS pairs over distributed shared memory and merges them in rank
// order (same bits everywhere).  For rows too few to fill the SMs.
//
// Generic plan (any N, any alignment): one CTA per row streams the row once
// with the per-element online update to get (m, d), merges, then reads the
// row again to write y.
//
// Exponentials: expf for binary32 outputs (CUDA documents at most 2 ulp);
// for binary16/bfloat16 outputs the fast __expf, whose documented error
// (2 + floor(|1.173 x|) binary32 ulp, below 1e-5 relative wherever exp(x) is
// a normal binary32) is far inside the 1-ulp tolerance of those types.
// Statistics and outputs are binary32 until the single rounding to the
// output type.
#include <cmath>
#include <cstdint>

#include "nrm_device.cuh"
#include "nrm_internal.h"

namespace nrm {

namespace {

struct MaxSum {
    float m, d;
};

template <typename T> __device__ __forceinline__ float smx_exp(float x) { return __expf(x); }
template <> __device__ __forceinline__ float smx_exp<float>(float x) { return expf(x); }

// Maximum of three values in one instruction (sm_100+ three-input max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The CTA plan's exponentials of a pair, for d = x - m_t <= 0, scaled by
// kSmxScale<T>.  Binary32 outputs: expf(d), unscaled.  16-bit outputs:
// 2^16 exp(d) = 2^(d log2 e + 16), the exponent formed pairwise with one
// fused multiply-add and PTX's ex2.approx.ftz (an error of a few binary32
// ulp, like __expf; with the rounding of d log2 e, below 1e-5 relative for
// |d| < 100, far inside the 1-ulp tolerance of binary16 and bfloat16).  The
// 2^16 scale keeps every exponential whose output can be a nonzero
// bfloat16 (down to its smallest subnormal, 2^-133) a normal binary32, so
// the flush to zero of the fast instruction only drops values that round to
// zero anyway; the sums carry the same exact power-of-two scale, which the
// output's 1/d removes and the reported row sum divides out.
template <typename T> struct SmxScale { static constexpr float v = 65536.0f; };
template <> struct SmxScale<float> { static constexpr float v = 1.0f; };

template <typename T> __device__ __forceinline__ float2 smx_exp_pair(float2 d) {
    const float2 t = __ffma2_rn(d, f2(1.44269504088896341f), f2(16.0f));
    float2 r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(t.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(t.y));
    return r;
}
template <> __device__ __forceinline__ float2 smx_exp_pair<float>(float2 d) {
    return make_float2(expf(d.x), expf(d.y));
}

// Merge of two (max, sum) pairs (the rescaling rule above).  A side with no
// elements (m = -inf, d = 0) leaves the other unchanged; the merge is
// symmetric in its arguments bit for bit (max and + commute), so butterfly
// partners agree.
template <typename T>
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b) {
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    const float M = fmaxf(a.m, b.m);
    return MaxSum{M, a.d * smx_exp<T>(a.m - M) + b.d * smx_exp<T>(b.m - M)};
}

__device__ __forceinline__ MaxSum ms_shfl_xor(MaxSum v, int o) {
    return MaxSum{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.d, o)};
}

// CTA-wide merge returned to every thread (same bits everywhere): warp
// butterfly, one exchange through `slot` (two alternating slots per CTA, as
// cta_sum_all), then a butterfly over the NW warp results.
template <typename T, int NW>
__device__ __forceinline__ MaxSum cta_merge_all(MaxSum v, float2 *slot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ms_merge<T>(v, ms_shfl_xor(v, o));
    if (NW == 1) return v;
    if (lane == 0) slot[warp] = make_float2(v.m, v.d);
    __syncthreads();
    const float2 w = slot[lane & (NW - 1)];
    v = MaxSum{w.x, w.y};
#pragma unroll
    for (int o = NW / 2; o > 0; o >>= 1) v = ms_merge<T>(v, ms_shfl_xor(v, o));
    return v;
}

// ---------------------------------------------------------------------------
// CTA plan
// ---------------------------------------------------------------------------
// FULL: the row is exactly THREADS x PACKS packs (no bounds tests).
// Resident 128-thread CTAs per SM the exact-row CTA plan is compiled for
// (NRM_SMX128_MIN_BLOCKS, at most 48 registers at ten): bf16 4096 x 4096 on
// GB300 11.81 us at ten against 12.23 us uncapped (52 registers, nine CTAs)
// and 12.45 us at twelve (spills).  The bounds-tested and cluster instances
// take eight (64 registers; at ten the 16-bit ones spill).
#ifndef NRM_SMX128_MIN_BLOCKS
#define NRM_SMX128_MIN_BLOCKS 10
#endif
// CS > 1: the cluster plan (launched with clusters of CS CTAs; P divisible
// by CS).
template <typename T, int THREADS, int PACKS, int CS, bool FULL = false>
__global__ void __launch_bounds__(THREADS, (THREADS == 128 ? (CS == 1 && FULL ? NRM_SMX128_MIN_BLOCKS : 8) : 1))
    softmax_cta_kernel(const RowArgs a, const int64_t pf) {
    using io2 = IO2<T>;
    constexpr int V = IO<T>::V;
    constexpr int H = io2::H;
    constexpr int NW = THREADS / 32;
    __shared__ float2 slot[2][NW];
    __shared__ float2 pub[2];  // cluster plan: this CTA's (max, sum) of the row
    const int t = threadIdx.x;
    const int rank = CS > 1 ? (int)cluster_rank() : 0;
    const int P = (int)(a.N / V) / CS;  // packs of this CTA's slice of the row
    const int64_t off = (int64_t)rank * P * V;
    const T *X = static_cast<const T *>(a.x) + off;
    const int64_t first = blockIdx.x / CS, step = gridDim.x / CS;
    const uint32_t slice_bytes = (uint32_t)P * 16u;
    // launched as a programmatic dependent (as the norm kernels): the CTA's
    // own row is requested from L2 first, then the kernel waits for the
    // previous grid on the stream and lets the next one become resident
    if ((pf > 0 || CS > 1) && t == 0 && first < a.rows) prefetch_l2_bulk(X + first * a.ldx, slice_bytes);
    pdl_wait();
    pdl_launch_dependents();
    int parity = 0;
    for (int64_t row = first; row < a.rows; row += step, parity ^= 1) {
        if (pf > 0 && t == 0 && row + pf < a.rows) prefetch_l2_bulk(X + (row + pf) * a.ldx, slice_bytes);
        const T *xr = X + row * a.ldx;
        uint4 raw[PACKS];
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
            if (FULL || t + k * THREADS < P) raw[k] = ld_stream(xr + (size_t)(t + k * THREADS) * V);
        float2 v[PACKS][H];
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (FULL || t + k * THREADS < P) {
                io2::unpack(raw[k], v[k]);
#pragma unroll
                for (int h = 0; h < H; ++h) mt = fmax3(mt, v[k][h].x, v[k][h].y);
            }
        }
        // e = exp(x - m_t); a thread whose values are all -inf (masked) holds
        // e = 0 and m_t = -inf, which the merge treats as empty
        const float2 nsh = f2(mt == -INFINITY ? 0.f : -mt);
        float2 acc = f2(0.f);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (FULL || t + k * THREADS < P) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    v[k][h] = smx_exp_pair<T>(__fadd2_rn(v[k][h], nsh));
                    acc = __fadd2_rn(acc, v[k][h]);
                }
            }
        }
        const float dt = acc.x + acc.y;
        MaxSum r = cta_merge_all<T, NW>(MaxSum{mt, dt}, slot[parity]);
        if constexpr (CS > 1) {
            // a slot of one parity is rewritten two rows later, after another
            // cluster barrier that every peer reaches only once it has read it
            if (t == 0) pub[parity] = make_float2(r.m, r.d);
            cluster_arrive();
            cluster_wait();
            const int lane = t & 31;
            const float2 mine = lane < CS ? ld_dsmem(&pub[parity], (uint32_t)lane)
                                          : make_float2(-INFINITY, 0.f);
            r = MaxSum{__shfl_sync(0xffffffffu, mine.x, 0), __shfl_sync(0xffffffffu, mine.y, 0)};
#pragma unroll
            for (int k = 1; k < CS; ++k)
                r = ms_merge<T>(r, MaxSum{__shfl_sync(0xffffffffu, mine.x, k),
                                          __shfl_sync(0xffffffffu, mine.y, k)});
        }
        if (t == 0 && rank == 0) {
            if (a.mean) a.mean[row] = r.m;                      // row max
            if (a.rstd) a.rstd[row] = r.d / SmxScale<T>::v;     // row sum of exp(x - max)
        }
        const float s = (mt == -INFINITY ? 0.f : smx_exp<T>(mt - r.m)) / r.d;
        const float2 s2 = f2(s);
        T *Y = static_cast<T *>(a.y) + off + row * a.ldy;
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            const int idx = t + k * THREADS;
            if (FULL || idx < P) {
                float2 o[H];
#pragma unroll
                for (int h = 0; h < H; ++h) o[h] = __fmul2_rn(v[k][h], s2);
                st_stream(Y + (size_t)idx * V, io2::pack(o));
            }
        }
    }
    if constexpr (CS > 1) {
        // stay resident until every peer has read this CTA's pairs
        cluster_arrive();
        cluster_wait();
    }
}

// ---------------------------------------------------------------------------
// Generic plan: any N, element-aligned pointers; two reads of the row.
// ---------------------------------------------------------------------------
template <typename T, int THREADS>
__global__ void __launch_bounds__(THREADS) softmax_generic_kernel(const RowArgs a) {
    constexpr int NW = THREADS / 32;
    __shared__ float2 slot[2][NW];
    const T *X = static_cast<const T *>(a.x);
    T *Y = static_cast<T *>(a.y);
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
        const int64_t bx = row * a.ldx, by = row * a.ldy;
        // the online update of the LLM-ops page, one element at a time
        MaxSum st{-INFINITY, 0.f};
        for (int64_t i = threadIdx.x; i < a.N; i += THREADS) {
            const float x = IO<T>::to_f(X[bx + i]);
            if (x == -INFINITY) continue;
            const float M = fmaxf(st.m, x);
            st.d = (st.m == -INFINITY ? 0.f : st.d * smx_exp<T>(st.m - M)) + smx_exp<T>(x - M);
            st.m = M;
        }
        const MaxSum r = cta_merge_all<T, NW>(st, slot[parity]);
        if (threadIdx.x == 0) {
            if (a.mean) a.mean[row] = r.m;
            if (a.rstd) a.rstd[row] = r.d;
        }
        const float inv = 1.0f / r.d;
        for (int64_t i = threadIdx.x; i < a.N; i += THREADS)
            Y[by + i] = IO<T>::from_f(smx_exp<T>(IO<T>::to_f(X[bx + i]) - r.m) * inv);
    }
}

template <typename T, int THREADS, int PACKS, bool FULL = false, int CS = 1>
cudaError_t launch_softmax_cta(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = softmax_cta_kernel<T, THREADS, PACKS, CS, FULL>;
    int64_t pf = 0;
    if (CS == 1 && p.prefetch > 0) {
        int per_sm = 0;
        const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), THREADS, 0, &per_sm);
        if (oe != cudaSuccess) return oe;
        pf = (int64_t)p.prefetch * p.sms * per_sm;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);  // rows x CS (clamped)
    cfg.blockDim = dim3(THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CS > 1 ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, pf);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename T>
cudaError_t launch_softmax_t(const RowArgs &a, const Plan &p, cudaStream_t s) {
    const dim3 grid((unsigned)p.grid);
    if (p.kind == PLAN_GENERIC) {
        switch (p.threads) {
        case 128: softmax_generic_kernel<T, 128><<<grid, 128, 0, s>>>(a); break;
        case 256: softmax_generic_kernel<T, 256><<<grid, 256, 0, s>>>(a); break;
        case 512: softmax_generic_kernel<T, 512><<<grid, 512, 0, s>>>(a); break;
        default: return cudaErrorInvalidConfiguration;
        }
        return cudaGetLastError();
    }
    if (p.kind == PLAN_CLUSTER) {
#define NRM_SMXC_CASE(TH, PK, CS)                                                   \
    if (p.threads == TH && p.packs == PK && p.groups == CS) {                       \
        if (a.N / IO<T>::V == (int64_t)TH * PK * CS)                               \
            return launch_softmax_cta<T, TH, PK, true, CS>(a, p, s);               \
        return launch_softmax_cta<T, TH, PK, false, CS>(a, p, s);                  \
    }
        NRM_SMXC_CASE(128, 1, 4) NRM_SMXC_CASE(128, 1, 8) NRM_SMXC_CASE(128, 2, 2)
        NRM_SMXC_CASE(128, 2, 4) NRM_SMXC_CASE(128, 4, 2) NRM_SMXC_CASE(128, 4, 4)
#undef NRM_SMXC_CASE
        return cudaErrorInvalidConfiguration;
    }
    if (p.kind != PLAN_CTA) return cudaErrorInvalidConfiguration;
#define NRM_SMX_CASE(TH, PK) \
    if (p.threads == TH && p.packs == PK) return launch_softmax_cta<T, TH, PK>(a, p, s);
    if (p.threads == 128 && p.packs == 4 && a.N / IO<T>::V == 512)
        return launch_softmax_cta<T, 128, 4, true>(a, p, s);
    if (p.threads == 256 && p.packs == 4 && a.N / IO<T>::V == 1024)
        return launch_softmax_cta<T, 256, 4, true>(a, p, s);
    NRM_SMX_CASE(128, 1) NRM_SMX_CASE(256, 1) NRM_SMX_CASE(128, 4) NRM_SMX_CASE(256, 2)
    NRM_SMX_CASE(256, 4) NRM_SMX_CASE(512, 4) NRM_SMX_CASE(1024, 4)
#undef NRM_SMX_CASE
    return cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t launch_softmax(const RowArgs &a, const Plan &p, int dtype, cudaStream_t s) {
    switch (dtype) {
    case DT_F32: return launch_softmax_t<float>(a, p, s);
    case DT_F16: return launch_softmax_t<__half>(a, p, s);
    case DT_BF16: return launch_softmax_t<__nv_bfloat16>(a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
