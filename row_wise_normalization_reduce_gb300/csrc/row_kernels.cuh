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

// LayerNorm statistics (register-resident rows).  With K = x[row, 0], the
// row's first element, every value is first shifted, d = x - K: for 16-bit
// inputs d is exact in binary32 whenever x and K are within 2^16 of each other
// in magnitude, so rows with a large mean and a small spread (mean 1000,
// std 1) lose nothing to cancellation.  Then a corrected two-pass over the
// values held in registers:
//   m0 = sum(d) / N                      (first CTA-wide sum)
//   e  = d - m0;  c = sum(e) / N;  M2 = sum(e^2) - N c^2   (second, fused sum)
//   mean = K + m0 + c,  var = M2 / N,  y = ((e - c) * rstd) * gamma + beta.
// The correction c removes the rounding error of the first sum, so the mean
// is accurate to a few units in the last place of the spread, and e is
// centered exactly enough that sum(e^2) has no cancellation.  Two float
// sums per row replace per-thread (count, mean, M2) combines, which need a
// division at every step and would make a 4096-wide bf16 row issue-bound.

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

// One row, spread over a group whose member `t` owns packs t, t + STRIDE, ...
template <int OP, typename T, int PACKS, int STRIDE, class Red>
__device__ __forceinline__ void row_body(const RowArgs &a, const int64_t row, const int t,
                                         Red &red) {
    using io = IO<T>;
    constexpr int V = io::V;
    const int64_t P = a.N / V;  // 16-byte packs per row
    const float fN = (float)a.N;
    const int64_t base = row * a.N;
    const T *__restrict__ X = static_cast<const T *>(a.x);
    const T *__restrict__ R = static_cast<const T *>(a.res);
    const T *__restrict__ G = static_cast<const T *>(a.p0);
    const T *__restrict__ Bt = static_cast<const T *>(a.p1);
    T *__restrict__ Y = static_cast<T *>(a.y);
    T *__restrict__ RO = static_cast<T *>(a.res_out);

    // ---- S1/S2: issue every load of the row before any arithmetic ----
    uint4 rx[PACKS];
    uint4 rr[PACKS];
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int64_t idx = t + (int64_t)k * STRIDE;
        if (idx < P) {
            rx[k] = ld_stream(X + base + idx * V);
            if (OP == OP_ADD_RMS) rr[k] = ld_stream(R + base + idx * V);
        }
    }
    const float K = (OP == OP_LN) ? io::to_f(X[base]) : 0.f;

    // v: LayerNorm d = x - K; RMS x; add+RMS the rounded residual-stream value
    float v[PACKS][V];
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int64_t idx = t + (int64_t)k * STRIDE;
        if (idx < P) {
            if (OP == OP_ADD_RMS) {
                float fx[V], fr[V], s[V];
                io::unpack(rx[k], fx);
                io::unpack(rr[k], fr);
#pragma unroll
                for (int j = 0; j < V; ++j) s[j] = __fadd_rn(fx[j], fr[j]);
                const uint4 packed = io::pack(s);  // round once to T
                st_stream(RO + base + idx * V, packed);
                io::unpack(packed, v[k]);
            } else {
                io::unpack(rx[k], v[k]);
                if (OP == OP_LN)
#pragma unroll
                    for (int j = 0; j < V; ++j) v[k][j] -= K;
            }
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j) v[k][j] = 0.f;  // contributes nothing
        }
    }

    // ---- S3-S6: statistics ----
    float rstd, m0 = 0.f, c = 0.f;
    if (OP == OP_LN) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j) s += v[k][j];
        m0 = red.sum(s) / fN;
        float e1 = 0.f, e2 = 0.f;
#pragma unroll
        for (int k = 0; k < PACKS; ++k) {
            const int64_t idx = t + (int64_t)k * STRIDE;
            if (idx < P)
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const float e = v[k][j] - m0;
                    v[k][j] = e;
                    e1 += e;
                    e2 = fmaf(e, e, e2);
                }
        }
        const float2 E = red.sum2(make_float2(e1, e2));
        c = E.x / fN;
        const float var = fmaxf(fmaf(-c, c, E.y / fN), 0.f);
        rstd = 1.0f / sqrtf(var + a.eps);
        if (t == 0) {
            if (a.mean) a.mean[row] = K + (m0 + c);
            if (a.rstd) a.rstd[row] = rstd;
        }
    } else {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < PACKS; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j) ss = fmaf(v[k][j], v[k][j], ss);
        rstd = 1.0f / sqrtf(red.sum(ss) / fN + a.eps);
        if (t == 0 && a.rstd) a.rstd[row] = rstd;
    }

    // ---- S7/S8: parameters, normalize, round once, store ----
#pragma unroll
    for (int k = 0; k < PACKS; ++k) {
        const int64_t idx = t + (int64_t)k * STRIDE;
        if (idx < P) {
            float out[V];
            if (OP == OP_LN) {
                float g[V], b[V];
                if (G) io::unpack(ld_param(G + idx * V), g);
                else
#pragma unroll
                    for (int j = 0; j < V; ++j) g[j] = 1.f;
                if (Bt) io::unpack(ld_param(Bt + idx * V), b);
                else
#pragma unroll
                    for (int j = 0; j < V; ++j) b[j] = 0.f;
#pragma unroll
                for (int j = 0; j < V; ++j) out[j] = fmaf((v[k][j] - c) * rstd, g[j], b[j]);
            } else {
                float w[V];
                if (G) io::unpack(ld_param(G + idx * V), w);
                else
#pragma unroll
                    for (int j = 0; j < V; ++j) w[j] = 1.f;
#pragma unroll
                for (int j = 0; j < V; ++j) out[j] = (v[k][j] * rstd) * w[j];
            }
            st_stream(Y + base + idx * V, io::pack(out));
        }
    }
}

template <int OP, typename T, int THREADS, int PACKS>
__global__ void __launch_bounds__(THREADS) row_cta_kernel(const RowArgs a) {
    constexpr int NW = THREADS / 32;
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, parity ^= 1) {
        CtaRed<NW> red{&s1[parity][0], &s2[parity][0]};
        row_body<OP, T, PACKS, THREADS>(a, row, threadIdx.x, red);
    }
}

template <int OP, typename T, int PACKS, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) row_warp_kernel(const RowArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    WarpRed red;
    for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < a.rows;
         row += (int64_t)gridDim.x * WARPS)
        row_body<OP, T, PACKS, 32>(a, row, lane, red);
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
        const int64_t base = row * a.N;
        const float K = (OP == OP_LN) ? io::to_f(X[base]) : 0.f;
        float n = 0.f, mean = 0.f, m2 = 0.f, ss = 0.f;
        for (int64_t i = tid; i < a.N; i += THREADS) {
            float v;
            if (OP == OP_ADD_RMS) {
                const T r = io::from_f(__fadd_rn(io::to_f(X[base + i]), io::to_f(R[base + i])));
                RO[base + i] = r;
                v = io::to_f(r);
            } else {
                v = io::to_f(X[base + i]);
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
                const float t = (io::to_f(X[base + i]) - K) - shift;
                out = fmaf(t * rstd, g, b);
            } else {
                const float v = (OP == OP_ADD_RMS) ? io::to_f(RO[base + i]) : io::to_f(X[base + i]);
                const float w = G ? io::to_f(G[i]) : 1.f;
                out = (v * rstd) * w;
            }
            Y[base + i] = io::from_f(out);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch switch: Plan -> template instance.
// ---------------------------------------------------------------------------
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
    if (p.threads == TH && p.packs == PK) {                                        \
        row_cta_kernel<OP, T, TH, PK><<<grid, TH, 0, s>>>(a);                      \
        return cudaGetLastError();                                                 \
    }
        NRM_CTA_CASE(128, 1) NRM_CTA_CASE(256, 1) NRM_CTA_CASE(512, 1) NRM_CTA_CASE(1024, 1)
        NRM_CTA_CASE(128, 2) NRM_CTA_CASE(256, 2) NRM_CTA_CASE(512, 2) NRM_CTA_CASE(1024, 2)
        NRM_CTA_CASE(256, 4) NRM_CTA_CASE(512, 4) NRM_CTA_CASE(1024, 4)
#undef NRM_CTA_CASE
        return cudaErrorInvalidConfiguration;
    } else {
        return cudaErrorInvalidConfiguration;
    }
    return cudaGetLastError();
}

template <int OP>
cudaError_t launch_row_dtype(const RowArgs &a, const Plan &p, int dtype, cudaStream_t s) {
    switch (dtype) {
    case DT_F32: return launch_row<OP, float>(a, p, s);
    case DT_F16: return launch_row<OP, __half>(a, p, s);
    case DT_BF16: return launch_row<OP, __nv_bfloat16>(a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
