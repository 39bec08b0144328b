// bn_sync.cu -- the pieces of synchronized BatchNorm, for a batch split over
// processes (BatchNorm CUDA implementation walkthrough,
// jianying88.com/news/30214, §7.1: each device reduces its own part, the
// partial statistics are combined across devices, then every device
// normalizes -- and runs the backward -- with the global statistics).
//
// Forward:  partial stats  per-channel (count, mean, M2) of the local batch
//                          in binary64, for the exchange;
//           apply stats    fold the exchanged [nparts][C] triples in rank
//                          order (every process gets the same bits),
//                          normalize the local batch, write save_* and the
//                          running statistics (global count).
// Backward: partial sums   per-channel (sum dy, sum dy * xhat) in binary64;
//           apply sums     fold the exchanged pairs, write dx of the local
//                          batch and dgamma/dbeta (global sums).
//
// The exchange itself (an all-gather of the small binary64 arrays) is the
// caller's: the library has no communicator.  The local reductions reuse the
// stage-1 kernels of bn.cu and bn_bwd.cu (per unit of at most 1024 packs when
// the planes are 16-byte aligned packs, per plane otherwise); the folds below
// combine in binary64.  The apply kernels walk the tensor as one flat array
// of packs (as the inference kernel) with a per-channel table every CTA folds
// from the exchanged parts; per-plane kernels cover the other layouts.
#include <cmath>
#include <cstdint>

#include "bn_common.cuh"

namespace nrm {

namespace {

constexpr int BSY_THREADS = 256;

struct DStats {
    double n, mean, m2;
};

// Chan's pairwise combine (LLM-ops page, smarter.xin, "Welford combine"),
// in binary64.  An empty side leaves the other unchanged.
__device__ __forceinline__ DStats dcombine(const DStats &a, const DStats &b) {
    const double n = a.n + b.n;
    if (n == 0.0) return a;
    const double d = b.mean - a.mean;
    return DStats{n, a.mean + d * (b.n / n), a.m2 + b.m2 + d * d * (a.n * (b.n / n))};
}

// One warp per channel: fold the channel's `per_channel` partials (mean, M2)
// of d = x - K (K = x[0, c, 0]) in order; stats[c] = (count, mean, M2) of x.
// Partial j covers count(j) values: HW for per-plane partials; for per-unit
// partials (chunks of at most cpk packs of V values) min(cpk, q - k*cpk) * V,
// k = j mod nch.
template <typename T>
__global__ void bn_fold_stats_kernel(const float2 *ws, const void *x, double *stats,
                                     int64_t per_channel, int64_t C, int64_t HW, int nch, int cpk,
                                     int q, int V) {
    // a programmatic dependent of the statistics kernel
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (c >= C) return;
    DStats st{0.0, 0.0, 0.0};
    for (int64_t j = lane; j < per_channel; j += 32) {
        const float2 p = ws[c * per_channel + j];
        const int k = (int)(j % nch);
        const double n = V ? (double)(min(cpk, q - k * cpk) * V) : (double)HW;
        st = dcombine(st, DStats{n, (double)p.x, (double)p.y});
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const DStats t{__shfl_xor_sync(0xffffffffu, st.n, o), __shfl_xor_sync(0xffffffffu, st.mean, o),
                       __shfl_xor_sync(0xffffffffu, st.m2, o)};
        st = lane < (lane ^ o) ? dcombine(st, t) : dcombine(t, st);
    }
    if (lane == 0) {
        const double K = (double)bn_elem<T>(x, c * HW);
        stats[3 * c + 0] = st.n;
        stats[3 * c + 1] = K + st.mean;
        stats[3 * c + 2] = st.m2;
    }
}

// One warp per channel: sums[c] = (sum dy, rstd_c * sum dy * (x - mean_c))
// over the channel's `per_channel` partials.
__global__ void bn_fold_sums_kernel(const float2 *ws, const float *rstd, double *sums,
                                    int64_t per_channel, int64_t C) {
    pdl_wait();  // a programmatic dependent of the stream's previous kernel
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t c = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (c >= C) return;
    double s1 = 0.0, s2 = 0.0;
    for (int64_t j = lane; j < per_channel; j += 32) {
        const float2 q = ws[c * per_channel + j];
        s1 += (double)q.x;
        s2 += (double)q.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double t1 = __shfl_xor_sync(0xffffffffu, s1, o);
        const double t2 = __shfl_xor_sync(0xffffffffu, s2, o);
        s1 = lane < (lane ^ o) ? s1 + t1 : t1 + s1;
        s2 = lane < (lane ^ o) ? s2 + t2 : t2 + s2;
    }
    if (lane == 0) {
        sums[2 * c + 0] = s1;
        sums[2 * c + 1] = s2 * (double)rstd[c];
    }
}

// Per (n, c) plane: fold the nparts exchanged triples in rank order, then
// normalize with the shifted mean (K = x[0, c, 0] of this process's batch, so
// x - K is exact for channels with a large mean).
template <typename T>
__global__ void __launch_bounds__(BSY_THREADS) bn_apply_stats_kernel(const BnSyncArgs a) {
    constexpr int V = IO<T>::V;
    __shared__ float s_stat[2][3];
    const int tid = threadIdx.x;
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const T *X = static_cast<const T *>(a.x);
    T *Y = static_cast<T *>(a.out);
    const bool vec = (HW % V == 0) && bn_aligned16(a.x) && bn_aligned16(a.out);
    int buf = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, buf ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        const float K = bn_elem<T>(a.x, c * HW);
        if (tid == 0) {
            DStats st{0.0, 0.0, 0.0};
            for (int64_t r = 0; r < a.nparts; ++r) {
                const double *q = a.parts + 3 * (r * a.C + c);
                st = dcombine(st, DStats{q[0], q[1], q[2]});
            }
            const double var = st.m2 / st.n;
            const double rstd = 1.0 / sqrt(var + (double)a.eps);
            s_stat[buf][0] = (float)(st.mean - (double)K);  // shifted mean
            s_stat[buf][1] = (float)rstd;
            if (n == 0) {
                if (a.save_mean) a.save_mean[c] = (float)st.mean;
                if (a.save_rstd) a.save_rstd[c] = (float)rstd;
                const double m = (double)a.momentum;
                if (a.running_mean)
                    a.running_mean[c] = (float)((1.0 - m) * a.running_mean[c] + m * st.mean);
                if (a.running_var)
                    a.running_var[c] =
                        (float)((1.0 - m) * a.running_var[c] + m * var * st.n / (st.n - 1.0));
            }
        }
        __syncthreads();
        const float md = s_stat[buf][0], rs = s_stat[buf][1];
        const float g = bn_param<T>(a.gamma, c, 1.f);
        const float b = bn_param<T>(a.beta, c, 0.f);
        const T *xp = X + p * HW;
        T *yp = Y + p * HW;
        if (vec) {
            for (int64_t i = tid; i < HW / V; i += BSY_THREADS) {
                float f[V], o[V];
                IO<T>::unpack(ld_stream(xp + V * i), f);
#pragma unroll
                for (int j = 0; j < V; ++j) o[j] = fmaf(((f[j] - K) - md) * rs, g, b);
                st_stream(yp + V * i, IO<T>::pack(o));
            }
        } else {
            for (int64_t i = tid; i < HW; i += BSY_THREADS)
                yp[i] = IO<T>::from_f(fmaf(((IO<T>::to_f(xp[i]) - K) - md) * rs, g, b));
        }
    }
}

// Per (n, c) plane: fold the nparts exchanged sums in rank order, then
// dx = gamma * rstd * ((dy - s1/count) - xhat * s2/count).
template <typename T>
__global__ void __launch_bounds__(BSY_THREADS) bn_apply_sums_kernel(const BnSyncArgs a) {
    constexpr int V = IO<T>::V;
    __shared__ float s_sum[2][2];
    const int tid = threadIdx.x;
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const T *X = static_cast<const T *>(a.x);
    const T *G = static_cast<const T *>(a.dy);
    T *D = static_cast<T *>(a.out);
    const bool vec = (HW % V == 0) && bn_aligned16(a.x) && bn_aligned16(a.dy) &&
                     bn_aligned16(a.out);
    int buf = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, buf ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        if (tid == 0) {
            double s1 = 0.0, s2 = 0.0;
            for (int64_t r = 0; r < a.nparts; ++r) {
                s1 += a.parts[2 * (r * a.C + c) + 0];
                s2 += a.parts[2 * (r * a.C + c) + 1];
            }
            s_sum[buf][0] = (float)(s1 / (double)a.count);
            s_sum[buf][1] = (float)(s2 / (double)a.count);
            if (n == 0) {
                if (a.dbeta) a.dbeta[c] = (float)s1;
                if (a.dgamma) a.dgamma[c] = (float)s2;
            }
        }
        __syncthreads();
        const float ma = s_sum[buf][0], mb = s_sum[buf][1];
        const float mean = a.mean[c], rstd = a.rstd[c];
        const float gr = bn_param<T>(a.gamma, c, 1.f) * rstd;
        const T *xp = X + p * HW;
        const T *gp = G + p * HW;
        T *dp = D + p * HW;
        if (vec) {
            for (int64_t i = tid; i < HW / V; i += BSY_THREADS) {
                float fx[V], fg[V], o[V];
                IO<T>::unpack(ld_stream(xp + V * i), fx);
                IO<T>::unpack(ld_stream(gp + V * i), fg);
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const float xh = (fx[j] - mean) * rstd;
                    o[j] = gr * fmaf(-xh, mb, fg[j] - ma);
                }
                st_stream(dp + V * i, IO<T>::pack(o));
            }
        } else {
            for (int64_t i = tid; i < HW; i += BSY_THREADS) {
                const float xh = (IO<T>::to_f(xp[i]) - mean) * rstd;
                dp[i] = IO<T>::from_f(gr * fmaf(-xh, mb, IO<T>::to_f(gp[i]) - ma));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Flat apply kernels (16-byte packs, C <= kSyncTable): the tensor as one
// array of packs over a resident grid, as the inference kernel; every CTA
// first folds the exchanged parts of all channels into a shared-memory table
// (CTA 0 also writes the per-channel outputs).
// ---------------------------------------------------------------------------
constexpr int kSyncTable = 2048;
constexpr int BSY_PACKS = 4;  // packs in flight per thread

template <typename T>
__global__ void __launch_bounds__(BSY_THREADS) bn_apply_stats_flat_kernel(const BnSyncArgs a,
                                                                          const uint32_t total,
                                                                          const FastDiv per_plane,
                                                                          const FastDiv channels) {
    // a programmatic dependent of the stream's previous kernel (the fold, or
    // the exchange of the parts): wait before reading anything
    pdl_wait();
    pdl_launch_dependents();
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    extern __shared__ float4 tab[];  // [C] {mean_hi, mean_lo, rstd, gamma}, then [C] beta
    float *tb = reinterpret_cast<float *>(tab + a.C);
    // every CTA builds the table; GB300's binary64 rate is low, so the
    // binary64 work per channel is the fold of the parts alone, and the
    // variance and rstd are formed in binary32 from the binary64 M2 and count
    // (division, square root and reciprocal correctly rounded: rstd within a
    // few ulp of the binary64 value)
    for (int64_t c = threadIdx.x; c < a.C; c += BSY_THREADS) {
        const double *q0 = a.parts + 3 * c;
        DStats st{q0[0], q0[1], q0[2]};
        for (int64_t r = 1; r < a.nparts; ++r) {
            const double *q = a.parts + 3 * (r * a.C + c);
            st = dcombine(st, DStats{q[0], q[1], q[2]});
        }
        const float rstd = 1.0f / sqrtf((float)st.m2 / (float)st.n + a.eps);
        const float hi = (float)st.mean;
        // the mean as hi + lo: (x - hi) - lo keeps x - mean exact-ish for
        // channels with a large mean
        tab[c] = make_float4(hi, (float)(st.mean - (double)hi), rstd, bn_param<T>(a.gamma, c, 1.f));
        tb[c] = bn_param<T>(a.beta, c, 0.f);
        if (blockIdx.x == 0) {
            if (a.save_mean) a.save_mean[c] = hi;
            if (a.save_rstd) a.save_rstd[c] = rstd;
            const double m = (double)a.momentum;
            if (a.running_mean)
                a.running_mean[c] = (float)((1.0 - m) * a.running_mean[c] + m * st.mean);
            if (a.running_var)
                a.running_var[c] = (float)((1.0 - m) * a.running_var[c] + m * st.m2 / (st.n - 1.0));
        }
    }
    __syncthreads();
    const uint4 *X = static_cast<const uint4 *>(a.x);
    uint4 *Y = static_cast<uint4 *>(a.out);
    const uint32_t stride = gridDim.x * BSY_THREADS;
    for (uint32_t base = blockIdx.x * BSY_THREADS + threadIdx.x; base < total;
         base += stride * BSY_PACKS) {
        uint4 v[BSY_PACKS];
#pragma unroll
        for (int j = 0; j < BSY_PACKS; ++j)
            if (base + j * stride < total) v[j] = ld_stream(X + base + j * stride);
#pragma unroll
        for (int j = 0; j < BSY_PACKS; ++j) {
            const uint32_t i = base + j * stride;
            if (i < total) {
                const uint32_t plane = fast_div(i, per_plane);
                const uint32_t c = plane - fast_div(plane, channels) * channels.d;
                const float4 k = tab[c];
                const float2 nh = f2(-k.x), nl = f2(-k.y), r2 = f2(k.z), g2 = f2(k.w),
                             b2 = f2(tb[c]);
                float2 f[H], o[H];
                io2::unpack(v[j], f);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(__fadd2_rn(f[h], nh), nl), r2), g2, b2);
                st_stream(Y + i, io2::pack(o));
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(BSY_THREADS) bn_apply_sums_flat_kernel(const BnSyncArgs a,
                                                                         const uint32_t total,
                                                                         const FastDiv per_plane,
                                                                         const FastDiv channels) {
    // a programmatic dependent of the stream's previous kernel (the fold, or
    // the exchange of the parts): wait before reading anything
    pdl_wait();
    pdl_launch_dependents();
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    extern __shared__ float4 tab[];  // [C] {mean, rstd, gamma*rstd, s1/count}, then [C] s2/count
    float *tb = reinterpret_cast<float *>(tab + a.C);
    for (int64_t c = threadIdx.x; c < a.C; c += BSY_THREADS) {
        double s1 = 0.0, s2 = 0.0;
        for (int64_t r = 0; r < a.nparts; ++r) {
            s1 += a.parts[2 * (r * a.C + c) + 0];
            s2 += a.parts[2 * (r * a.C + c) + 1];
        }
        // binary32 divisions of the binary64 sums (GB300's binary64 rate is low)
        const float rstd = a.rstd[c];
        const float cnt = (float)a.count;
        tab[c] = make_float4(a.mean[c], rstd, bn_param<T>(a.gamma, c, 1.f) * rstd, (float)s1 / cnt);
        tb[c] = (float)s2 / cnt;
        if (blockIdx.x == 0) {
            if (a.dbeta) a.dbeta[c] = (float)s1;
            if (a.dgamma) a.dgamma[c] = (float)s2;
        }
    }
    __syncthreads();
    const uint4 *X = static_cast<const uint4 *>(a.x);
    const uint4 *G = static_cast<const uint4 *>(a.dy);
    uint4 *D = static_cast<uint4 *>(a.out);
    const uint32_t stride = gridDim.x * BSY_THREADS;
    for (uint32_t base = blockIdx.x * BSY_THREADS + threadIdx.x; base < total;
         base += stride * BSY_PACKS) {
        uint4 vx[BSY_PACKS], vg[BSY_PACKS];
#pragma unroll
        for (int j = 0; j < BSY_PACKS; ++j)
            if (base + j * stride < total) {
                vx[j] = ld_stream(X + base + j * stride);
                vg[j] = ld_stream(G + base + j * stride);
            }
#pragma unroll
        for (int j = 0; j < BSY_PACKS; ++j) {
            const uint32_t i = base + j * stride;
            if (i < total) {
                const uint32_t plane = fast_div(i, per_plane);
                const uint32_t c = plane - fast_div(plane, channels) * channels.d;
                const float4 k = tab[c];
                const float2 nm = f2(-k.x), r2 = f2(k.y), gr = f2(k.z), na = f2(-k.w),
                             nb = f2(-tb[c]);
                float2 fx[H], fg[H], o[H];
                io2::unpack(vx[j], fx);
                io2::unpack(vg[j], fg);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 xh = __fmul2_rn(__fadd2_rn(fx[h], nm), r2);
                    o[h] = __fmul2_rn(gr, __ffma2_rn(xh, nb, __fadd2_rn(fg[h], na)));
                }
                st_stream(D + i, io2::pack(o));
            }
        }
    }
}

// The flat plans' launch: HW a whole number of packs, 16-byte aligned
// tensors, a table that fits, pack indices within 32 bits.
template <typename T>
bool bn_flat_ok(const BnSyncArgs &a, bool bwd) {
    constexpr int V = IO<T>::V;
    const int64_t total = a.batch * a.C * (a.HW / V);
    // pack indices, and the loop's base + BSY_PACKS strides, stay below 2^32
    return a.HW % V == 0 && a.C <= kSyncTable && total < ((int64_t)1 << 31) &&
           bn_aligned16(a.x) && bn_aligned16(a.out) && (!bwd || bn_aligned16(a.dy));
}

template <typename T, typename K>
cudaError_t launch_bn_flat(K kernel, const BnSyncArgs &a, int num_sms, cudaStream_t s) {
    constexpr int V = IO<T>::V;
    const int64_t total = a.batch * a.C * (a.HW / V);
    const int64_t need = (total + BSY_THREADS * BSY_PACKS - 1) / (BSY_THREADS * BSY_PACKS);
    const int64_t slots = (int64_t)num_sms * 8;
    const unsigned grid = (unsigned)(need < slots ? need : slots);
    const size_t smem = (size_t)a.C * (sizeof(float4) + sizeof(float));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(BSY_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, (uint32_t)total,
                                             make_fastdiv((uint32_t)(a.HW / V)), make_fastdiv((uint32_t)a.C));
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename T>
cudaError_t launch_apply_stats_t(const BnSyncArgs &a, int num_sms, cudaStream_t s) {
    if (bn_flat_ok<T>(a, false)) return launch_bn_flat<T>(bn_apply_stats_flat_kernel<T>, a, num_sms, s);
    bn_apply_stats_kernel<T><<<bn_grid(a.batch * a.C, num_sms), BSY_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_apply_sums_t(const BnSyncArgs &a, int num_sms, cudaStream_t s) {
    if (bn_flat_ok<T>(a, true)) return launch_bn_flat<T>(bn_apply_sums_flat_kernel<T>, a, num_sms, s);
    bn_apply_sums_kernel<T><<<bn_grid(a.batch * a.C, num_sms), BSY_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bn_unit_stats_host(const BnArgs &a, int dtype, int num_sms, cudaStream_t s,
                                      int *nch, int *cpk, int *q) {
    BnChunks u;
    const cudaError_t e = launch_bn_unit_stats(a, dtype, num_sms, s, &u);
    *nch = u.nch;
    *cpk = u.cpk;
    *q = u.q;
    return e;
}

cudaError_t launch_bn_bwd_unit_sums_host(const BnBwdArgs &a, int dtype, int num_sms,
                                         cudaStream_t s, int *nch) {
    BnChunks u;
    const cudaError_t e = launch_bn_bwd_unit_sums(a, dtype, num_sms, s, &u);
    *nch = u.nch;
    return e;
}

cudaError_t launch_bn_fold_stats(const float2 *ws, const void *x, double *stats, int64_t per_channel,
                                 int64_t C, int64_t HW, int nch, int cpk, int q, int V, int dtype,
                                 cudaStream_t s) {
    // one channel (warp) per CTA, so the channels' binary64 folds run on
    // different SMs (GB300's binary64 rate per SM is low)
    if (C < 1 || C > 0x7fffffff) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)C;
    switch (dtype) {
    case DT_F32:
        return launch_pdl(bn_fold_stats_kernel<float>, grid, 32, s, true, ws, x, stats, per_channel, C, HW,
                          nch, cpk, q, V);
    case DT_F16:
        return launch_pdl(bn_fold_stats_kernel<__half>, grid, 32, s, true, ws, x, stats, per_channel, C, HW,
                          nch, cpk, q, V);
    case DT_BF16:
        return launch_pdl(bn_fold_stats_kernel<__nv_bfloat16>, grid, 32, s, true, ws, x, stats, per_channel,
                          C, HW, nch, cpk, q, V);
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_bn_fold_sums(const float2 *ws, const float *rstd, double *sums,
                                int64_t per_channel, int64_t C, cudaStream_t s) {
    if (C < 1 || C > 0x7fffffff) return cudaErrorInvalidValue;
    return launch_pdl(bn_fold_sums_kernel, (unsigned)C, 32, s, true, ws, rstd, sums, per_channel, C);
}

cudaError_t launch_bn_apply_stats(const BnSyncArgs &a, int dtype, int num_sms, cudaStream_t s) {
    switch (dtype) {
    case DT_F32: return launch_apply_stats_t<float>(a, num_sms, s);
    case DT_F16: return launch_apply_stats_t<__half>(a, num_sms, s);
    case DT_BF16: return launch_apply_stats_t<__nv_bfloat16>(a, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bn_apply_sums(const BnSyncArgs &a, int dtype, int num_sms, cudaStream_t s) {
    switch (dtype) {
    case DT_F32: return launch_apply_sums_t<float>(a, num_sms, s);
    case DT_F16: return launch_apply_sums_t<__half>(a, num_sms, s);
    case DT_BF16: return launch_apply_sums_t<__nv_bfloat16>(a, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
