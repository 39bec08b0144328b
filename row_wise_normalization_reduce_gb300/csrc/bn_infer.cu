// bn_infer.cu -- BatchNorm2d inference forward over NCHW data: every element
// is normalized with its channel's running statistics (BatchNorm CUDA
// implementation walkthrough, jianying88.com/news/30214, §2.4: inference
// replaces the batch's mean and variance by the running ones), so the pass
// is element-wise and bound by one read of x and one write of y.
//
//   y = ((x - running_mean_c) * rstd_c) * gamma_c + beta_c,
//   rstd_c = 1 / sqrt(running_var_c + eps)
//
// The unfolded form is kept (rather than y = x * s_c + t_c): it costs nothing
// at HBM speed and avoids the cancellation of x * s_c against t_c when the
// running mean is large compared with the spread.
//
// Main plan (16-byte packs, C <= 2048): the tensor is one flat array of
// 16-byte packs walked by a grid of resident CTAs (BNI_PACKS packs in flight
// per thread, consecutive threads on consecutive packs), so every SM streams
// until the end whatever the plane size.  A pack's channel is
// (pack / packs_per_plane) mod C, by multiply-high division; the channel
// constants (mean, rstd, gamma, beta) are computed once per CTA into a
// shared-memory table.
//
// Fallback plans: the CTA's threads are split into groups of TPP threads (a
// power of two, at most the CTA), one (n, c) plane per group; a group walks
// its plane with 16-byte packs, or elements when the layout does not allow
// packs.
#include <cmath>
#include <cstdint>

#include "bn_common.cuh"

namespace nrm {

namespace {

constexpr int BNI_THREADS = 256;
constexpr int BNI_PACKS = 4;

struct ChannelConst {
    float mean, rstd, g, b;
};

template <typename T>
__device__ __forceinline__ ChannelConst bn_infer_const(const BnInferArgs &a, int64_t c) {
    ChannelConst k;
    k.mean = a.running_mean[c];
    k.rstd = 1.0f / sqrtf(a.running_var[c] + a.eps);
    k.g = bn_param<T>(a.gamma, c, 1.f);
    k.b = bn_param<T>(a.beta, c, 0.f);
    return k;
}

constexpr int BNI_MAX_TABLE = 2048;  // channels of the shared-memory table (32 KB)

// Resident CTAs per SM the flat kernel is compiled for (registers): binary32
// fits 8 (32 registers), the 16-bit types 6 (their unpacking needs 40).
template <typename T> constexpr int bni_ctas_per_sm() { return sizeof(T) == 4 ? 8 : 6; }

template <typename T>
__global__ void __launch_bounds__(BNI_THREADS, bni_ctas_per_sm<T>()) bn_infer_flat_kernel(const BnInferArgs a,
                                                                    const uint32_t total,
                                                                    const FastDiv per_plane,
                                                                    const FastDiv channels) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    extern __shared__ float4 table[];  // C entries
    for (int c = threadIdx.x; c < (int)a.C; c += BNI_THREADS) {
        const ChannelConst k = bn_infer_const<T>(a, c);
        table[c] = make_float4(-k.mean, k.rstd, k.g, k.b);
    }
    __syncthreads();
    const uint4 *X = static_cast<const uint4 *>(a.x);
    uint4 *Y = static_cast<uint4 *>(a.y);
    const uint32_t stride = gridDim.x * BNI_THREADS;
    for (uint32_t base = blockIdx.x * BNI_THREADS + threadIdx.x; base < total;
         base += stride * BNI_PACKS) {
        uint4 v[BNI_PACKS];
#pragma unroll
        for (int j = 0; j < BNI_PACKS; ++j) {
            const uint32_t i = base + j * stride;
            if (i < total) v[j] = ld_stream(X + i);
        }
#pragma unroll
        for (int j = 0; j < BNI_PACKS; ++j) {
            const uint32_t i = base + j * stride;
            if (i < total) {
                const uint32_t plane = fast_div(i, per_plane);
                const uint32_t c = plane - fast_div(plane, channels) * channels.d;
                const float4 k = table[c];
                const float2 nm = f2(k.x), r2 = f2(k.y), g2 = f2(k.z), b2 = f2(k.w);
                float2 f[H], o[H];
                io2::unpack(v[j], f);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(f[h], nm), r2), g2, b2);
                st_stream(Y + i, io2::pack(o));
            }
        }
    }
}

// Vector plan: HW a multiple of the pack width, x and y 16-byte aligned.
template <typename T>
__global__ void __launch_bounds__(BNI_THREADS) bn_infer_vec_kernel(const BnInferArgs a,
                                                                   const int tpp_log2) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    const int tpp = 1 << tpp_log2;
    const int sub = threadIdx.x >> tpp_log2, li = threadIdx.x & (tpp - 1);
    const int ppi = BNI_THREADS >> tpp_log2;  // planes per CTA step
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const int q = (int)(HW / IO<T>::V);
    for (int64_t p = (int64_t)blockIdx.x * ppi + sub; p < planes; p += (int64_t)gridDim.x * ppi) {
        const ChannelConst k = bn_infer_const<T>(a, p % a.C);
        const float2 nm = f2(-k.mean), r2 = f2(k.rstd), g2 = f2(k.g), b2 = f2(k.b);
        const uint4 *xp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + p * HW);
        uint4 *yp = reinterpret_cast<uint4 *>(static_cast<T *>(a.y) + p * HW);
        for (int base = li; base < q; base += tpp * BNI_PACKS) {
            uint4 v[BNI_PACKS];
#pragma unroll
            for (int j = 0; j < BNI_PACKS; ++j)
                if (base + j * tpp < q) v[j] = ld_stream(xp + base + j * tpp);
#pragma unroll
            for (int j = 0; j < BNI_PACKS; ++j)
                if (base + j * tpp < q) {
                    float2 f[H], o[H];
                    io2::unpack(v[j], f);
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(f[h], nm), r2), g2, b2);
                    st_stream(yp + base + j * tpp, io2::pack(o));
                }
        }
    }
}

// Scalar plan: any HW, element-aligned pointers; the same plane grouping
// with one element per access.
template <typename T>
__global__ void __launch_bounds__(BNI_THREADS) bn_infer_scalar_kernel(const BnInferArgs a,
                                                                      const int tpp_log2) {
    const int tpp = 1 << tpp_log2;
    const int sub = threadIdx.x >> tpp_log2, li = threadIdx.x & (tpp - 1);
    const int ppi = BNI_THREADS >> tpp_log2;
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const T *X = static_cast<const T *>(a.x);
    T *Y = static_cast<T *>(a.y);
    for (int64_t p = (int64_t)blockIdx.x * ppi + sub; p < planes; p += (int64_t)gridDim.x * ppi) {
        const ChannelConst k = bn_infer_const<T>(a, p % a.C);
        for (int64_t i = li; i < HW; i += tpp) {
            const float v = IO<T>::to_f(X[p * HW + i]);
            Y[p * HW + i] = IO<T>::from_f(fmaf((v - k.mean) * k.rstd, k.g, k.b));
        }
    }
}

// Threads per plane: the plane's work items (packs or elements) rounded up to
// a power of two, between 32 and the CTA size.
int tpp_log2_for(int64_t items) {
    int l = 5;
    while (l < 8 && ((int64_t)1 << l) < items) ++l;
    return l;
}

template <typename T>
cudaError_t launch_bn_infer_t(const BnInferArgs &a, int num_sms, cudaStream_t s, int *used) {
    constexpr int V = IO<T>::V;
    const int64_t planes = a.batch * a.C;
    const bool vec = a.bn_plan != BN_PLAN_SCALAR && a.HW % V == 0 && a.HW / V < (1 << 30) &&
                     bn_aligned16(a.x) && bn_aligned16(a.y);
    *used = vec ? PLAN_CTA : PLAN_GENERIC;
    const int64_t total = planes * (a.HW / V);
    if (vec && a.C <= BNI_MAX_TABLE &&
        total < ((int64_t)1 << 32) - (int64_t)num_sms * 8 * BNI_THREADS * BNI_PACKS) {
        const int64_t need = (total + BNI_THREADS * BNI_PACKS - 1) / (BNI_THREADS * BNI_PACKS);
        const int64_t slots = (int64_t)num_sms * bni_ctas_per_sm<T>();
        const unsigned grid = (unsigned)(need < slots ? need : slots);
        bn_infer_flat_kernel<T><<<grid, BNI_THREADS, (size_t)a.C * sizeof(float4), s>>>(
            a, (uint32_t)total, make_fastdiv((uint32_t)(a.HW / V)), make_fastdiv((uint32_t)a.C));
        return cudaGetLastError();
    }
    const int l = tpp_log2_for(vec ? a.HW / V : a.HW);
    const int64_t ppi = BNI_THREADS >> l;
    const unsigned grid = bn_grid((planes + ppi - 1) / ppi, num_sms);
    if (vec) bn_infer_vec_kernel<T><<<grid, BNI_THREADS, 0, s>>>(a, l);
    else bn_infer_scalar_kernel<T><<<grid, BNI_THREADS, 0, s>>>(a, l);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bn_infer(const BnInferArgs &a, int dtype, int num_sms, cudaStream_t s,
                            int *used) {
    switch (dtype) {
    case DT_F32: return launch_bn_infer_t<float>(a, num_sms, s, used);
    case DT_F16: return launch_bn_infer_t<__half>(a, num_sms, s, used);
    case DT_BF16: return launch_bn_infer_t<__nv_bfloat16>(a, num_sms, s, used);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
