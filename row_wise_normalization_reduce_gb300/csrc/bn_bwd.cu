// bn_bwd.cu -- BatchNorm2d training backward over NCHW data, organised as the
// two stages of the BatchNorm CUDA implementation walkthrough
// (jianying88.com/news/30214, §3.1-§3.3): a channel reduction of the two
// sums, then an element-wise pass that broadcasts them.  With
// xhat = (x - mean_c) * rstd_c (mean_c, rstd_c saved by the training forward)
// and count = batch * H * W:
//
//   dbeta_c  = sum dy,   dgamma_c = sum dy * xhat,
//   dx = gamma_c * rstd_c * (dy - dbeta_c / count - xhat * dgamma_c / count).
//
// Unlike the page, which stores xhat in a temporary buffer during the
// forward pass, xhat is recomputed from x and the saved statistics: reading
// x costs the same bytes as reading a stored xhat, and the forward pass saves
// a full-tensor write.
//
// Stage 1 keeps per-plane partials (sum dy, sum dy * (x - mean_c)) in the
// workspace; stage 2 folds the batch's partials of its channel in a fixed
// order (every CTA of a channel gets the same bits) and writes dx; the CTA of
// plane n = 0 writes dgamma/dbeta.
//
// Streaming plan: one CTA per plane holds the plane's dy and x in registers;
// stage 2 is launched with programmatic stream serialization, loads its
// plane's dy and x first (for a batch that fits in L2 these reads hit L2),
// then waits for stage 1.  Scalar plan: any layout, plain loops.
#include <cmath>
#include <cstdint>

#include "bn_common.cuh"

namespace nrm {

namespace {

constexpr int BB_THREADS = 256;

// Fold the `count` partials of channel c (warp 0; lane j takes partials j,
// j + 32, ... in order, then a butterfly): the same bits in every CTA.
__device__ __forceinline__ float2 bn_bwd_fold(const float2 *ws, int64_t c, int64_t count) {
    float2 s = f2(0.f);
    const int lane = threadIdx.x & 31;
    for (int64_t j = lane; j < count; j += 32) {
        const float2 q = ws[c * count + j];
        s.x += q.x;
        s.y += q.y;
    }
    return warp_sum_all(s);
}

// ---------------------------------------------------------------------------
// Streaming plan: units are chunks of at most 1024 packs of one plane, and
// the channels are processed in groups whose dy and x fit comfortably in L2
// (bn_common.cuh), so stage 2 re-reads them from L2.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(BNS_THREADS) bn_bwd_sums_kernel(const BnBwdArgs a,
                                                                  const BnChunks u) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int NW = BNS_THREADS / 32;
    __shared__ float2 s2[2][NW];
    const int tid = threadIdx.x;
    const int64_t units = a.batch * u.G * u.nch, HW = a.HW;
    float2 *ws = static_cast<float2 *>(a.ws);
    // stage 2 may launch once every CTA of this grid has started (it waits
    // for this grid's completion before it reads the partials): started at
    // the top, it takes the SMs as this grid's last wave leaves them
    // ([32, 64, 56, 56] binary32: 19.58 -> 18.70 us against triggering at
    // the end)
    pdl_launch_dependents();
    int par = 0;
    for (int64_t idx = blockIdx.x; idx < units; idx += gridDim.x, par ^= 1) {
        const BnUnit w = bn_unit(u, idx);
        const int64_t base = (w.n * a.C + w.c) * HW;
        const uint4 *gp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.dy) + base) + w.off;
        const uint4 *xp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + base) + w.off;
        // default L2 policy: stage 2 reads the same chunks again
        uint4 vg[BNS_PACKS], vx[BNS_PACKS];
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) {
                vg[k] = __ldg(gp + tid + k * BNS_THREADS);
                vx[k] = __ldg(xp + tid + k * BNS_THREADS);
            }
        const float2 nm = f2(-a.mean[w.c]);
        float2 sg = f2(0.f), sgx = f2(0.f);
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) {
                float2 g[H], x[H];
                io2::unpack(vg[k], g);
                io2::unpack(vx[k], x);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    sg = __fadd2_rn(sg, g[h]);
                    sgx = __ffma2_rn(g[h], __fadd2_rn(x[h], nm), sgx);
                }
            }
        const float2 S = cta_sum_all<NW>(make_float2(hsum(sg), hsum(sgx)), s2[par]);
        if (tid == 0) ws[w.c * (a.batch * u.nch) + w.n * u.nch + w.k] = S;
    }
    pdl_wait();  // finish after the previous group's stage 2 (see bn.cu)
}

template <typename T>
__global__ void __launch_bounds__(BNS_THREADS) bn_bwd_dx_kernel(const BnBwdArgs a,
                                                                const BnChunks u) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    __shared__ float2 sums[2];
    const int tid = threadIdx.x;
    const int64_t units = a.batch * u.G * u.nch, HW = a.HW;
    const float cnt = (float)(a.batch * HW);
    const float2 *ws = static_cast<const float2 *>(a.ws);
    bool waited = false;
    int par = 0;
    for (int64_t idx = blockIdx.x; idx < units; idx += gridDim.x, par ^= 1) {
        const BnUnit w = bn_unit(u, idx);
        const int64_t base = (w.n * a.C + w.c) * HW;
        const uint4 *gp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.dy) + base) + w.off;
        const uint4 *xp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + base) + w.off;
        uint4 vg[BNS_PACKS], vx[BNS_PACKS];
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) {
                vg[k] = __ldcs(gp + tid + k * BNS_THREADS);
                vx[k] = __ldcs(xp + tid + k * BNS_THREADS);
            }
        if (!waited) {
            pdl_launch_dependents();  // the next group's stage 1 may start
            pdl_wait();  // stage 1 has finished and its partials are visible
            waited = true;
        }
        if (tid < 32) {
            const float2 S = bn_bwd_fold(ws, w.c, a.batch * u.nch);
            if (tid == 0) sums[par] = S;
        }
        __syncthreads();
        const float mean = a.mean[w.c], rstd = a.rstd[w.c];
        const float2 S = sums[par];
        const float dgamma = S.y * rstd;  // sum dy * xhat
        if (w.n == 0 && w.k == 0 && tid == 0) {
            if (a.dbeta) a.dbeta[w.c] = S.x;
            if (a.dgamma) a.dgamma[w.c] = dgamma;
        }
        const float gr = bn_param<T>(a.gamma, w.c, 1.f) * rstd;
        const float2 nm = f2(-mean), r2 = f2(rstd), na = f2(-(S.x / cnt)),
                     nb = f2(-(dgamma / cnt)), gr2 = f2(gr);
        uint4 *dp = reinterpret_cast<uint4 *>(static_cast<T *>(a.dx) + base) + w.off;
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) {
                float2 g[H], x[H], o[H];
                io2::unpack(vg[k], g);
                io2::unpack(vx[k], x);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 xh = __fmul2_rn(__fadd2_rn(x[h], nm), r2);
                    o[h] = __fmul2_rn(gr2, __ffma2_rn(xh, nb, __fadd2_rn(g[h], na)));
                }
                __stcs(dp + tid + k * BNS_THREADS, io2::pack(o));
            }
    }
    if (!waited) {
        pdl_launch_dependents();
        pdl_wait();
    }
}

// ---------------------------------------------------------------------------
// Scalar plan (any HW, element-aligned pointers)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(BB_THREADS) bn_bwd_partial_kernel(const BnBwdArgs a) {
    constexpr int NW = BB_THREADS / 32;
    __shared__ float2 s2[2][NW];
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const T *G = static_cast<const T *>(a.dy);
    const T *X = static_cast<const T *>(a.x);
    float2 *ws = static_cast<float2 *>(a.ws);
    int par = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, par ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        const float mean = a.mean[c];
        float sg = 0.f, sgx = 0.f;
        for (int64_t i = threadIdx.x; i < HW; i += BB_THREADS) {
            const float g = IO<T>::to_f(G[p * HW + i]);
            sg += g;
            sgx = fmaf(g, IO<T>::to_f(X[p * HW + i]) - mean, sgx);
        }
        const float2 S = cta_sum_all<NW>(make_float2(sg, sgx), s2[par]);
        if (threadIdx.x == 0) ws[c * a.batch + n] = S;
    }
}

template <typename T>
__global__ void __launch_bounds__(BB_THREADS) bn_bwd_apply_kernel(const BnBwdArgs a) {
    __shared__ float2 sums[2];
    const int64_t planes = a.batch * a.C, HW = a.HW;
    const float cnt = (float)(a.batch * HW);
    const T *G = static_cast<const T *>(a.dy);
    const T *X = static_cast<const T *>(a.x);
    T *D = static_cast<T *>(a.dx);
    const float2 *ws = static_cast<const float2 *>(a.ws);
    int par = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, par ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        if (threadIdx.x < 32) {
            const float2 S = bn_bwd_fold(ws, c, a.batch);
            if (threadIdx.x == 0) sums[par] = S;
        }
        __syncthreads();
        const float mean = a.mean[c], rstd = a.rstd[c];
        const float2 S = sums[par];
        const float dgamma = S.y * rstd;
        if (n == 0 && threadIdx.x == 0) {
            if (a.dbeta) a.dbeta[c] = S.x;
            if (a.dgamma) a.dgamma[c] = dgamma;
        }
        const float gr = bn_param<T>(a.gamma, c, 1.f) * rstd;
        const float ma = S.x / cnt, mb = dgamma / cnt;
        for (int64_t i = threadIdx.x; i < HW; i += BB_THREADS) {
            const float xh = (IO<T>::to_f(X[p * HW + i]) - mean) * rstd;
            const float t = fmaf(-xh, mb, IO<T>::to_f(G[p * HW + i]) - ma);
            D[p * HW + i] = IO<T>::from_f(gr * t);
        }
    }
}

template <typename T>
cudaError_t launch_bn_bwd_t(const BnBwdArgs &a, int num_sms, cudaStream_t s, int *used) {
    constexpr int V = IO<T>::V;
    const bool stream_ok = a.bn_plan != BN_PLAN_SCALAR && a.HW % V == 0 &&
                           a.HW / V < kBnMaxPlanePacks && bn_aligned16(a.dy) &&
                           bn_aligned16(a.x) && bn_aligned16(a.dx);
    // planes longer than one unit: the one-pass plan first (dy and x read
    // from HBM once; the streaming plan reads them twice once they exceed L2)
    const bool one_unit = a.HW / V <= kBnChunkPacks;
    if (stream_ok && ((a.bn_plan == BN_PLAN_AUTO && !one_unit) || a.bn_plan == BN_PLAN_FLOW)) {
        bool launched = false;
        const cudaError_t e = launch_bn_bwd_flow(a, bn_dtype<T>(), num_sms, s, &launched);
        if (launched || e != cudaSuccess) {
            *used = PLAN_PERSIST;
            return e;
        }
    }
    *used = stream_ok ? PLAN_CTA : PLAN_GENERIC;
    if (stream_ok) {
        BnChunks u = bn_chunks(a.HW / V);
        const int64_t G = bn_group_channels(a.C, 2 * a.batch * a.HW * (int64_t)sizeof(T),
                                            bn_group_budget());
        cudaError_t e = cudaSuccess;
        for (int64_t c0 = 0; c0 < a.C && e == cudaSuccess; c0 += G) {
            u.c0 = c0;
            u.G = (a.C - c0) < G ? (a.C - c0) : G;
            const unsigned grid = bn_grid(a.batch * u.G * u.nch, num_sms);
            e = launch_pdl(bn_bwd_sums_kernel<T>, grid, BNS_THREADS, s, c0 > 0, a, u);
            if (e == cudaSuccess) e = launch_pdl(bn_bwd_dx_kernel<T>, grid, BNS_THREADS, s, true, a, u);
        }
        return e;
    }
    const unsigned grid = bn_grid(a.batch * a.C, num_sms);
    bn_bwd_partial_kernel<T><<<grid, BB_THREADS, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bn_bwd_apply_kernel<T><<<grid, BB_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bn_bwd_unit_sums(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                                    BnChunks *u) {
    const int V = dtype == DT_F32 ? 4 : 8;
    *u = bn_chunks(a.HW / V);
    u->c0 = 0;
    u->G = a.C;
    const unsigned grid = bn_grid(a.batch * a.C * u->nch, num_sms);
    switch (dtype) {
    case DT_F32: bn_bwd_sums_kernel<float><<<grid, BNS_THREADS, 0, s>>>(a, *u); break;
    case DT_F16: bn_bwd_sums_kernel<__half><<<grid, BNS_THREADS, 0, s>>>(a, *u); break;
    case DT_BF16: bn_bwd_sums_kernel<__nv_bfloat16><<<grid, BNS_THREADS, 0, s>>>(a, *u); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_bn_bwd_plane_sums(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s) {
    const unsigned grid = bn_grid(a.batch * a.C, num_sms);
    switch (dtype) {
    case DT_F32: bn_bwd_partial_kernel<float><<<grid, BB_THREADS, 0, s>>>(a); break;
    case DT_F16: bn_bwd_partial_kernel<__half><<<grid, BB_THREADS, 0, s>>>(a); break;
    case DT_BF16: bn_bwd_partial_kernel<__nv_bfloat16><<<grid, BB_THREADS, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_bn_bwd(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                          int *used) {
    switch (dtype) {
    case DT_F32: return launch_bn_bwd_t<float>(a, num_sms, s, used);
    case DT_F16: return launch_bn_bwd_t<__half>(a, num_sms, s, used);
    case DT_BF16: return launch_bn_bwd_t<__nv_bfloat16>(a, num_sms, s, used);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
