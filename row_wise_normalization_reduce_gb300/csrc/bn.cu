// bn.cu -- BatchNorm2d training forward over NCHW binary32 data, as a
// two-phase channel reduction (BatchNorm CUDA implementation walkthrough,
// jianying88.com/news/30214, §2.1-§2.4 and its Welford discussion in §4.3):
//
//   phase 1  one CTA per (n, c) plane (H*W contiguous values): partial
//            statistics (mean, M2) of the plane into the workspace;
//   phase 2  one CTA per plane: fold the batch's partials of its channel
//            (every CTA of a channel folds them in the same order, so all
//            agree bit for bit), normalize the plane and write y; the CTA of
//            plane n = 0 writes save_mean/save_rstd and the running statistics
//            (a single writer per channel).
//
// Phase 2 re-reads x; for tensors that fit in L2 (the 25.7 MB of a
// [32, 64, 56, 56] batch does) that second read is served from L2.
//
// All statistics of channel c are taken on d = x - K_c with K_c the channel's
// first element x[0, c, 0]: the shift keeps channels with a large mean and a
// small spread free of cancellation.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "nrm.h"
#include "nrm_device.cuh"
#include "nrm_internal.h"

namespace nrm {

namespace {

constexpr int BN_THREADS = 256;

__global__ void __launch_bounds__(BN_THREADS) bn_partial_kernel(const BnArgs a) {
    constexpr int NW = BN_THREADS / 32;
    __shared__ float s_red[2][NW][3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t planes = a.batch * a.C;
    const int64_t HW = a.HW;
    const bool vec = (HW % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0);
    float2 *ws = static_cast<float2 *>(a.ws);
    int buf = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, buf ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        const float *xp = a.x + p * HW;
        const float K = a.x[c * HW];  // x[0, c, 0]
        Stats st{0.f, 0.f, 0.f};
        if (vec) {
            const int64_t P = HW / 4;
            for (int64_t i = tid; i < P; i += BN_THREADS) {
                float f[4];
                IO<float>::unpack(ld_stream(xp + 4 * i), f);
                const float d0 = f[0] - K, d1 = f[1] - K, d2 = f[2] - K, d3 = f[3] - K;
                const float m = ((d0 + d1) + (d2 + d3)) * 0.25f;
                const float e0 = d0 - m, e1 = d1 - m, e2 = d2 - m, e3 = d3 - m;
                const float m2 = fmaf(e0, e0, fmaf(e1, e1, fmaf(e2, e2, e3 * e3)));
                st = combine(st, Stats{4.f, m, m2});
            }
        } else {
            for (int64_t i = tid; i < HW; i += BN_THREADS) {
                const float d = xp[i] - K;
                st.n += 1.f;
                const float delta = d - st.mean;
                st.mean += delta / st.n;
                st.m2 = fmaf(delta, d - st.mean, st.m2);
            }
        }
        st = warp_stats_down(st);
        if (lane == 0) {
            s_red[buf][warp][0] = st.n;
            s_red[buf][warp][1] = st.mean;
            s_red[buf][warp][2] = st.m2;
        }
        __syncthreads();
        if (tid == 0) {
            Stats t{s_red[buf][0][0], s_red[buf][0][1], s_red[buf][0][2]};
            for (int w = 1; w < NW; ++w)
                t = combine(t, Stats{s_red[buf][w][0], s_red[buf][w][1], s_red[buf][w][2]});
            ws[c * a.batch + n] = make_float2(t.mean, t.m2);
        }
    }
}

__global__ void __launch_bounds__(BN_THREADS) bn_apply_kernel(const BnArgs a) {
    __shared__ float s_stat[2][2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t planes = a.batch * a.C;
    const int64_t HW = a.HW;
    const float cnt = (float)(a.batch * HW);
    const bool vec = (HW % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(a.y) & 15) == 0);
    const float2 *ws = static_cast<const float2 *>(a.ws);
    int buf = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, buf ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        if (warp == 0) {
            Stats st{0.f, 0.f, 0.f};
            for (int64_t j = lane; j < a.batch; j += 32) {
                const float2 q = ws[c * a.batch + j];
                st = combine(st, Stats{(float)HW, q.x, q.y});
            }
            st = warp_stats_down(st);
            if (lane == 0) {
                s_stat[buf][0] = st.mean;
                s_stat[buf][1] = st.m2;
            }
        }
        __syncthreads();
        const float K = a.x[c * HW];
        const float md = s_stat[buf][0];
        const float var = s_stat[buf][1] / cnt;
        const float rstd = 1.0f / sqrtf(var + a.eps);
        if (n == 0 && tid == 0) {
            if (a.save_mean) a.save_mean[c] = K + md;
            if (a.save_rstd) a.save_rstd[c] = rstd;
            const float m = a.momentum;
            if (a.running_mean)
                a.running_mean[c] = fmaf(1.f - m, a.running_mean[c], m * (K + md));
            if (a.running_var) {
                const float unbiased = var * (cnt / (float)(a.batch * HW - 1));
                a.running_var[c] = fmaf(1.f - m, a.running_var[c], m * unbiased);
            }
        }
        const float g = a.gamma ? a.gamma[c] : 1.f;
        const float b = a.beta ? a.beta[c] : 0.f;
        const float *xp = a.x + p * HW;
        float *yp = a.y + p * HW;
        if (vec) {
            const int64_t P = HW / 4;
            for (int64_t i = tid; i < P; i += BN_THREADS) {
                float f[4], o[4];
                IO<float>::unpack(ld_stream(xp + 4 * i), f);
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = fmaf(((f[j] - K) - md) * rstd, g, b);
                st_stream(yp + 4 * i, IO<float>::pack(o));
            }
        } else {
            for (int64_t i = tid; i < HW; i += BN_THREADS)
                yp[i] = fmaf(((xp[i] - K) - md) * rstd, g, b);
        }
    }
}

}  // namespace

cudaError_t launch_bn_train_f32(const BnArgs &a, int num_sms, cudaStream_t s) {
    const int64_t planes = a.batch * a.C;
    const int64_t cap = (int64_t)num_sms * 64;
    const unsigned grid = (unsigned)(planes < cap ? planes : cap);
    bn_partial_kernel<<<grid, BN_THREADS, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bn_apply_kernel<<<grid, BN_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace nrm

// ---------------------------------------------------------------------------
// bn_fwd_train_noalloc: the same two kernels, with the per-plane partial
// statistics kept in a fixed array of this library instead of a workspace the
// caller allocates.  It is for callers that cannot allocate device memory
// when they call -- for example a runtime that reserves its whole device
// memory budget at start-up and forbids later allocations, or a component
// that is handed device pointers by another part of the program and has no
// allocator of its own.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it (kBnStaticPlanes float2 = 512 KB) until the process exits.
// Its name in host code is only a host-side stand-in, so the device address
// is taken with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on that device.  All calls on a device
// share the array: calls that overlap on the GPU (different streams without
// ordering) race on it.  Every partial a call reads it first writes in the
// same call, so nothing needs clearing between calls.
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kBnStaticPlanes = 65536;  // largest batch * C accepted
__device__ __align__(256) float2 g_bn_static_partials[kBnStaticPlanes];

constexpr int kMaxDevices = 64;
float2 *g_bn_static_ptr[kMaxDevices];
std::once_flag g_bn_static_once[kMaxDevices];

bool spans_overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

extern "C" int bn_fwd_train_noalloc(const void *x, const void *gamma, const void *beta, void *y,
                                    float *save_mean, float *save_rstd, float *running_mean,
                                    float *running_var, int64_t batch, int64_t C, int64_t HW,
                                    float eps, float momentum, int dtype, cudaStream_t stream) {
    using namespace nrm;
    if (dtype != NRM_F32 && dtype != NRM_F16 && dtype != NRM_BF16) return NRM_ERR_DTYPE;
    if (batch < 1 || C < 1 || HW < 1) return NRM_ERR_SHAPE;
    if ((uint64_t)batch > (uint64_t)INT64_MAX / (uint64_t)C / (uint64_t)HW / 4) return NRM_ERR_SHAPE;
    if (batch * HW < 2) return NRM_ERR_SHAPE;
    if (batch * C > kBnStaticPlanes) return NRM_ERR_TOO_LARGE;
    if (!std::isfinite(eps) || eps < 0.f || !(momentum >= 0.f && momentum <= 1.f))
        return NRM_ERR_VALUE;
    if (!x || !y) return NRM_ERR_NULL;
    if (dtype != NRM_F32) return NRM_ERR_UNSUPPORTED;
    const void *all[] = {x, gamma, beta, y, save_mean, save_rstd, running_mean, running_var};
    for (const void *p : all)
        if (p && (reinterpret_cast<uintptr_t>(p) & 3)) return NRM_ERR_VALUE;
    const size_t tb = (size_t)batch * (size_t)C * (size_t)HW * 4, cb = (size_t)C * 4;
    const void *ins[] = {x, gamma, beta};
    const size_t in_n[] = {tb, cb, cb};
    const void *outs[] = {y, save_mean, save_rstd, running_mean, running_var};
    const size_t out_n[] = {tb, cb, cb, cb, cb};
    for (int o = 0; o < 5; ++o) {
        for (int i = 0; i < 3; ++i)
            if (spans_overlap(outs[o], out_n[o], ins[i], in_n[i])) return NRM_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 5; ++o2)
            if (spans_overlap(outs[o], out_n[o], outs[o2], out_n[o2])) return NRM_ERR_ALIAS;
    }

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    std::call_once(g_bn_static_once[dev], [dev]() {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bn_static_partials) == cudaSuccess)
            g_bn_static_ptr[dev] = static_cast<float2 *>(p);
        else
            cudaGetLastError();
    });
    if (!g_bn_static_ptr[dev]) return NRM_ERR_DEVICE;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    BnArgs a{static_cast<const float *>(x), static_cast<const float *>(gamma),
             static_cast<const float *>(beta), static_cast<float *>(y), save_mean, save_rstd,
             running_mean, running_var, batch, C, HW, eps, momentum, g_bn_static_ptr[dev]};
    return launch_bn_train_f32(a, sms, stream) == cudaSuccess ? NRM_OK : NRM_ERR_LAUNCH;
}
