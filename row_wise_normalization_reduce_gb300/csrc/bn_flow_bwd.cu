// bn_flow_bwd.cu -- BatchNorm2d training backward with dy and x read once
// from HBM, for planes longer than one streaming unit (BatchNorm CUDA
// implementation walkthrough, jianying88.com/news/30214, §3.1-§3.3), on the
// dataflow machinery of bn_flow.cuh:
//
//   dbeta_c  = sum dy,   dgamma_c = sum dy * xhat,   xhat = (x - mean_c) * rstd_c
//   dx = gamma_c * rstd_c * (dy - dbeta_c / cnt - xhat * dgamma_c / cnt)
//
// Statistics item: the chunks of dy and x in registers, their partial
// (sum dy, sum dy * (x - mean_c)) by one CTA-wide sum.
// Fold: the U partials summed in a fixed order (thread-strided, then warp
// butterflies, then the warps in order); the folding CTA writes dbeta and
// dgamma, and the result word holds dbeta / cnt (low half) and dgamma / cnt
// (high half).
// Apply item: dx from the re-read chunks (L2) and the result word.
#include <cmath>
#include <cstdint>

#include "bn_flow.cuh"

namespace nrm {

namespace {

constexpr int BNFB_PACKS = 4;  // per thread and tensor: 8 packs in registers

template <typename T>
__device__ __forceinline__ const uint4 *bwd_ptr(const void *t, const FlowIdx &w) {
    return reinterpret_cast<const uint4 *>(static_cast<const T *>(t) + w.base) + w.off;
}

// The chunks of dy and x of item w into registers: default L2 policy for
// statistics items (re-read by the apply items), evict-first for apply items.
template <typename T>
__device__ __forceinline__ void bwd_load(const BnBwdArgs &a, const FlowIdx &w, uint4 (&vg)[BNFB_PACKS],
                                         uint4 (&vx)[BNFB_PACKS]) {
    const uint4 *gp = bwd_ptr<T>(a.dy, w) + threadIdx.x;
    const uint4 *xp = bwd_ptr<T>(a.x, w) + threadIdx.x;
#pragma unroll
    for (int j = 0; j < BNFB_PACKS; ++j)
        if ((int)threadIdx.x + j * BNF_THREADS < w.len) {
            vg[j] = w.stats ? __ldg(gp + j * BNF_THREADS) : __ldcs(gp + j * BNF_THREADS);
            vx[j] = w.stats ? __ldg(xp + j * BNF_THREADS) : __ldcs(xp + j * BNF_THREADS);
        }
}

template <typename T>
__device__ __forceinline__ void bwd_prefetch(const BnBwdArgs &a, const FlowPlan &f, uint32_t i) {
    if (i >= f.items) return;
    const FlowIdx w = flow_item(f, (uint32_t)a.C, a.HW, i);
    if (w.stats) {
        prefetch_l2_bulk(bwd_ptr<T>(a.dy, w), (uint32_t)w.len * 16u);
        prefetch_l2_bulk(bwd_ptr<T>(a.x, w), (uint32_t)w.len * 16u);
    }
}

// Fold of channel c by the whole CTA; thread 0 publishes.
__device__ __forceinline__ void bwd_fold(const BnBwdArgs &a, const FlowPlan &f, uint32_t c, float2 *wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t *pc = f.part + (int64_t)c * f.U;
    float2 s = f2(0.f);
    for (uint32_t j = tid; j < f.U; j += BNF_THREADS) {
        const uint64_t word = poll_word(pc + j, a.wait_limit, a.fault);
        s.x += __uint_as_float((unsigned)word);
        s.y += __uint_as_float((unsigned)(word >> 32));
    }
    s = warp_sum_all(s);
    if (lane == 0) wsum[warp] = s;
    __syncthreads();
    if (tid == 0) {
        float2 t = wsum[0];
#pragma unroll
        for (int q = 1; q < BNF_NW; ++q) t = make_float2(t.x + wsum[q].x, t.y + wsum[q].y);
        const float dgamma = t.y * a.rstd[c];  // sum dy * xhat
        if (a.dbeta) a.dbeta[c] = t.x;
        if (a.dgamma) a.dgamma[c] = dgamma;
        const float cnt = (float)(a.batch * a.HW);
        st_relaxed_gpu(f.chst + c, pack_word(t.x / cnt, dgamma / cnt));
    }
}

template <typename T>
__global__ void __launch_bounds__(BNF_THREADS, 4) bn_flow_bwd_kernel(const BnBwdArgs a, const FlowPlan f) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int NW = BNF_NW;
    __shared__ float2 s2[2][NW];
    __shared__ float2 wsum[NW];
    __shared__ uint32_t s_tk[2], s_fold[2];
    __shared__ uint64_t s_stat[2];
    const int tid = threadIdx.x;
    const uint32_t C = (uint32_t)a.C, G = gridDim.x;
    const int64_t HW = a.HW;
    // thread 0's state: the ticket of the item after the current one, and the
    // channel whose completing increment is still to be checked
    uint32_t t_next = 0, pend_c = kNone;
    unsigned pend_old = 0;
    pdl_wait();  // the reset kernel has finished
    if (tid == 0) {
        s_tk[1] = atomicAdd(f.ticket, 1u);
        t_next = atomicAdd(f.ticket, 1u);
    }
    __syncthreads();
    uint32_t i = s_tk[1];
    if (i >= f.items) return;
    FlowIdx w = flow_item(f, C, HW, i);
    uint4 vg[BNFB_PACKS], vx[BNFB_PACKS];
    bwd_load<T>(a, w, vg, vx);
    if (tid == 0)
        for (uint32_t t = 1; t < f.pf; ++t) bwd_prefetch<T>(a, f, i + t * G);
    int par = 0;
    while (true) {
        if (tid == 0) {
            s_tk[par] = t_next;
            t_next = atomicAdd(f.ticket, 1u);  // the item after the next one
            s_fold[par] = pend_c != kNone && pend_old == f.U - 1 ? pend_c : kNone;
            pend_c = kNone;
            if (f.pf) bwd_prefetch<T>(a, f, i + f.pf * G);
        }
        const float mean = a.mean[w.c];
        uint32_t ni;
        if (w.stats) {
            const float2 nm = f2(-mean);
            float2 sg = f2(0.f), sgx = f2(0.f);
#pragma unroll
            for (int j = 0; j < BNFB_PACKS; ++j)
                if (tid + j * BNF_THREADS < w.len) {
                    float2 g[H], x[H];
                    io2::unpack(vg[j], g);
                    io2::unpack(vx[j], x);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        sg = __fadd2_rn(sg, g[h]);
                        sgx = __ffma2_rn(g[h], __fadd2_rn(x[h], nm), sgx);
                    }
                }
            // s_tk / s_fold become visible at this barrier
            const float2 S = cta_sum_all<NW>(make_float2(hsum(sg), hsum(sgx)), s2[par]);
            ni = s_tk[par];
            const uint32_t fc = s_fold[par];
            const uint32_t c = w.c, unit = w.unit;
            if (ni < f.items) {
                w = flow_item(f, C, HW, ni);
                bwd_load<T>(a, w, vg, vx);
            }
            if (tid == 0) {
                st_relaxed_gpu(f.part + (int64_t)c * f.U + unit, pack_word(S.x, S.y));
                pend_old = atomicAdd(f.cnt + c, 1u);
                pend_c = c;
            }
            if (fc != kNone) bwd_fold(a, f, fc, wsum);
        } else {
            __syncthreads();  // s_tk / s_fold visible
            ni = s_tk[par];
            const uint32_t fc = s_fold[par];
            // a pending fold first: this item may wait, the fold never waits
            // on anything but statistics items
            if (fc != kNone) bwd_fold(a, f, fc, wsum);
            if (tid == 0) s_stat[par] = poll_word(f.chst + w.c, a.wait_limit, a.fault);
            __syncthreads();
            const uint64_t word = s_stat[par];
            const float rstd = a.rstd[w.c];
            const float gr = bn_param<T>(a.gamma, w.c, 1.f) * rstd;
            const float2 nm = f2(-mean), r2 = f2(rstd), gr2 = f2(gr),
                         na = f2(-__uint_as_float((unsigned)word)),
                         nb = f2(-__uint_as_float((unsigned)(word >> 32)));
            uint4 *dp = reinterpret_cast<uint4 *>(static_cast<T *>(a.dx) + w.base) + w.off + tid;
#pragma unroll
            for (int j = 0; j < BNFB_PACKS; ++j)
                if (tid + j * BNF_THREADS < w.len) {
                    float2 g[H], x[H], o[H];
                    io2::unpack(vg[j], g);
                    io2::unpack(vx[j], x);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 xh = __fmul2_rn(__fadd2_rn(x[h], nm), r2);
                        o[h] = __fmul2_rn(gr2, __ffma2_rn(xh, nb, __fadd2_rn(g[h], na)));
                    }
                    __stcs(dp + j * BNF_THREADS, io2::pack(o));
                }
            if (ni < f.items) {
                w = flow_item(f, C, HW, ni);
                bwd_load<T>(a, w, vg, vx);
            }
        }
        if (ni >= f.items) break;
        i = ni;
        par ^= 1;
    }
    // the last item may have completed its channel
    if (tid == 0) s_fold[par ^ 1] = pend_c != kNone && pend_old == f.U - 1 ? pend_c : kNone;
    __syncthreads();
    if (s_fold[par ^ 1] != kNone) bwd_fold(a, f, s_fold[par ^ 1], wsum);
}

template <typename T>
cudaError_t launch_bn_bwd_flow_t(const BnBwdArgs &a, int num_sms, cudaStream_t s, bool *launched) {
    *launched = false;
    constexpr int V = IO<T>::V;
    if (a.HW % V != 0 || !bn_aligned16(a.dy) || !bn_aligned16(a.x) || !bn_aligned16(a.dx) ||
        !a.fault || !a.ws || !bn_aligned16(a.ws) || a.HW / V >= kBnMaxPlanePacks)
        return cudaSuccess;
    auto kernel = bn_flow_bwd_kernel<T>;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), BNF_THREADS, 0, &per_sm);
    if (oe != cudaSuccess) return oe;
    FlowPlan f;
    int64_t grid = 0;
    // chunks of at most BNF_THREADS * BNFB_PACKS = kBnChunkPacks packs, as
    // the workspace is sized; the lag counts the bytes of dy and x
    if (!flow_plan(a.batch, a.C, a.HW / V, BNF_THREADS * BNFB_PACKS, a.prefetch, per_sm, num_sms,
                   2 * a.batch * a.HW * (int64_t)sizeof(T), a.ws, a.ws_bytes, &f, &grid))
        return cudaSuccess;
    *launched = true;
    const cudaError_t e = flow_reset(f, a.C, num_sms, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, (unsigned)grid, BNF_THREADS, s, true, a, f);
}

}  // namespace

cudaError_t launch_bn_bwd_flow(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                               bool *launched) {
    switch (dtype) {
    case DT_F32: return launch_bn_bwd_flow_t<float>(a, num_sms, s, launched);
    case DT_F16: return launch_bn_bwd_flow_t<__half>(a, num_sms, s, launched);
    case DT_BF16: return launch_bn_bwd_flow_t<__nv_bfloat16>(a, num_sms, s, launched);
    default: *launched = false; return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
