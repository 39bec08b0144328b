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
// Resident 128-thread CTAs per SM the CTA plan is compiled for
// (NRM_SMX128_MIN_BLOCKS, at most 48 registers at ten): bf16 4096 x 4096 on
// GB300 11.81 us at ten against 12.23 us uncapped (52 registers, nine CTAs)
// and 12.45 us at twelve (spills).
#ifndef NRM_SMX128_MIN_BLOCKS
#define NRM_SMX128_MIN_BLOCKS 10
#endif
template <typename T, int THREADS, int PACKS, bool FULL = false>
__global__ void __launch_bounds__(THREADS, (THREADS == 128 ? NRM_SMX128_MIN_BLOCKS : 1))
    softmax_cta_kernel(const RowArgs a, const int64_t pf) {
    using io2 = IO2<T>;
    constexpr int V = IO<T>::V;
    constexpr int H = io2::H;
    constexpr int NW = THREADS / 32;
    __shared__ float2 slot[2][NW];
    const int t = threadIdx.x;
    const int P = (int)(a.N / V);
    const T *X = static_cast<const T *>(a.x);
    // launched as a programmatic dependent (as the norm kernels): the CTA's
    // own row is requested from L2 first, then the kernel waits for the
    // previous grid on the stream and lets the next one become resident
    if (pf > 0 && t == 0 && blockIdx.x < a.rows)
        prefetch_l2_bulk(X + blockIdx.x * a.ldx, (uint32_t)(a.N * (int64_t)sizeof(T)));
    pdl_wait();
    pdl_launch_dependents();
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
        if (pf > 0 && t == 0 && row + pf < a.rows)
            prefetch_l2_bulk(X + (row + pf) * a.ldx, (uint32_t)(a.N * (int64_t)sizeof(T)));
        const T *xr = X + row * a.ldx;
        uint4 raw[PACKS];
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
            if (FULL || t + k * THREADS < P) raw[k] = ld_stream(xr + (size_t)(t + k * THREADS) * V);
        float2 v[PACKS][H];
        float2 mx = f2(-INFINITY);
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (FULL || t + k * THREADS < P) {
                io2::unpack(raw[k], v[k]);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    mx = make_float2(fmaxf(mx.x, v[k][h].x), fmaxf(mx.y, v[k][h].y));
            }
        }
        // e = exp(x - m_t); a thread whose values are all -inf (masked) holds
        // e = 0 and m_t = -inf, which the merge treats as empty
        const float mt = fmaxf(mx.x, mx.y);
        const float sh = mt == -INFINITY ? 0.f : mt;
        float dt = 0.f;
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            if (FULL || t + k * THREADS < P) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    v[k][h] = make_float2(smx_exp<T>(v[k][h].x - sh), smx_exp<T>(v[k][h].y - sh));
                    dt += v[k][h].x + v[k][h].y;
                }
            }
        }
        const MaxSum r = cta_merge_all<T, NW>(MaxSum{mt, dt}, slot[parity]);
        if (t == 0) {
            if (a.mean) a.mean[row] = r.m;  // row max
            if (a.rstd) a.rstd[row] = r.d;  // row sum of exp(x - max)
        }
        const float s = (mt == -INFINITY ? 0.f : smx_exp<T>(mt - r.m)) / r.d;
        const float2 s2 = f2(s);
        T *Y = static_cast<T *>(a.y) + row * a.ldy;
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

template <typename T, int THREADS, int PACKS, bool FULL = false>
cudaError_t launch_softmax_cta(const RowArgs &a, const Plan &p, cudaStream_t s) {
    auto kernel = softmax_cta_kernel<T, THREADS, PACKS, FULL>;
    int64_t pf = 0;
    if (p.prefetch > 0) {
        int per_sm = 0;
        const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), THREADS, 0, &per_sm);
        if (oe != cudaSuccess) return oe;
        pf = (int64_t)p.prefetch * p.sms * per_sm;
    }
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
