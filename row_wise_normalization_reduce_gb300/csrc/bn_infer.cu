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
// Mapping: the CTA's threads are split into groups of TPP threads (a power of
// two, at most the CTA), one (n, c) plane per group; a group walks its plane
// with 16-byte packs (PACKS in flight per thread).  Small planes thus share a
// CTA instead of leaving most of its threads idle, and a plane's constants
// are computed once per thread, not per element.
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
    const int l = tpp_log2_for(vec ? a.HW / V : a.HW);
    const int64_t ppi = BNI_THREADS >> l;
    const unsigned grid = bn_grid((planes + ppi - 1) / ppi, num_sms);
    *used = vec ? PLAN_CTA : PLAN_GENERIC;
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
