// bn_flow.cu -- BatchNorm2d training forward with x read once from HBM, for
// planes longer than one streaming unit (BatchNorm CUDA implementation
// walkthrough, jianying88.com/news/30214, §2.1-§2.4: the same two phases,
// per-plane partial statistics then per-channel fold and normalization), on
// the dataflow machinery of bn_flow.cuh.
//
// Statistics item: the chunk in registers, its exact partial (mean, M2) on
// d = x - K (K = x[0, c, 0]) by the corrected two-pass of bn_unit_partial.
// Fold: the U partials combined in a fixed order (Chan's pairwise rule, so
// the bits do not depend on which CTA folds); the folding CTA writes
// save_mean/save_rstd and the running statistics, and the result word holds
// the channel's shifted mean (low half) and rstd (high half).
// Apply item: y = ((x - K) - mean_d) * rstd * gamma + beta.
//
// The loads of a CTA's next item are issued as soon as the registers of the
// current one are free (after its partial statistics, or after its stores),
// and thread 0 prefetches into L2 the chunk of the item pf * grid numbers
// ahead of its own.
#include <cmath>
#include <cstdint>

#include "bn_flow.cuh"

namespace nrm {

namespace {

// Resident CTAs per SM for PACKS 16-byte packs per thread (register caps
// without spills: 48 and 64 registers).
template <int PACKS> constexpr int bnf_min_blocks() { return PACKS <= 4 ? 5 : 4; }

template <typename T>
__device__ __forceinline__ const uint4 *flow_ptr(const BnArgs &a, const FlowIdx &w) {
    return reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + w.base) + w.off;
}

// The chunk of item w into registers: statistics items read with the
// default L2 policy (the apply items re-read the data from L2), apply items
// evict-first (last use).
template <typename T, int PACKS>
__device__ __forceinline__ void flow_load(const BnArgs &a, const FlowIdx &w, uint4 (&v)[PACKS]) {
    const uint4 *xp = flow_ptr<T>(a, w) + threadIdx.x;
#pragma unroll
    for (int j = 0; j < PACKS; ++j)
        if ((int)threadIdx.x + j * BNF_THREADS < w.len)
            v[j] = w.stats ? __ldg(xp + j * BNF_THREADS) : __ldcs(xp + j * BNF_THREADS);
}

// L2 prefetch of item i's chunk if it is a statistics item.
template <typename T>
__device__ __forceinline__ void flow_prefetch(const BnArgs &a, const FlowPlan &f, uint32_t i) {
    if (i >= f.items) return;
    const FlowIdx w = flow_item(f, (uint32_t)a.C, a.HW, i);
    if (w.stats) prefetch_l2_bulk(flow_ptr<T>(a, w), (uint32_t)w.len * 16u);
}

// Fold of channel c by the whole CTA; thread 0 publishes.
template <typename T>
__device__ __forceinline__ void flow_fold(const BnArgs &a, const FlowPlan &f, uint32_t c, Stats *wred) {
    constexpr int V = IO<T>::V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t *pc = f.part + (int64_t)c * f.U;
    Stats st{0.f, 0.f, 0.f};
    for (uint32_t j = tid; j < f.U; j += BNF_THREADS) {
        const uint64_t word = poll_word(pc + j, a.wait_limit, a.fault);
        const float cn = (float)(flow_chunk_len(f, j) * V);
        st = combine(st, Stats{cn, __uint_as_float((unsigned)word), __uint_as_float((unsigned)(word >> 32))});
    }
    st = warp_stats_down(st);
    if (lane == 0) wred[warp] = st;
    __syncthreads();
    if (tid == 0) {
        Stats t = wred[0];
#pragma unroll
        for (int q = 1; q < BNF_NW; ++q) t = combine(t, wred[q]);
        const float var = t.m2 / (float)(a.batch * a.HW);
        const float rstd = 1.0f / sqrtf(var + a.eps);
        bn_write_channel_stats(a, c, bn_elem<T>(a.x, (int64_t)c * a.HW), t.mean, var, rstd);
        st_relaxed_gpu(f.chst + c, pack_word(t.mean, rstd));
    }
}

template <typename T, int PACKS>
__global__ void __launch_bounds__(BNF_THREADS, bnf_min_blocks<PACKS>())
    bn_flow_kernel(const BnArgs a, const FlowPlan f) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int NW = BNF_NW;
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    __shared__ Stats wred[NW];
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
    uint4 v[PACKS];
    flow_load<T, PACKS>(a, w, v);
    if (tid == 0)
        for (uint32_t t = 1; t < f.pf; ++t) flow_prefetch<T>(a, f, i + t * G);
    int par = 0;
    while (true) {
        if (tid == 0) {
            s_tk[par] = t_next;
            t_next = atomicAdd(f.ticket, 1u);  // the item after the next one
            s_fold[par] = pend_c != kNone && pend_old == f.U - 1 ? pend_c : kNone;
            pend_c = kNone;
            if (f.pf) flow_prefetch<T>(a, f, i + f.pf * G);
        }
        const float K = bn_elem<T>(a.x, (int64_t)w.c * HW);
        uint32_t ni;
        if (w.stats) {
            // s_tk / s_fold become visible at the first barrier of the partial
            const float2 r = bn_unit_partial<T, PACKS>(v, w.len, K, s1[par], s2[par]);
            ni = s_tk[par];
            const uint32_t fc = s_fold[par];
            const uint32_t c = w.c, unit = w.unit;
            if (ni < f.items) {
                w = flow_item(f, C, HW, ni);
                flow_load<T, PACKS>(a, w, v);
            }
            if (tid == 0) {
                st_relaxed_gpu(f.part + (int64_t)c * f.U + unit, pack_word(r.x, r.y));
                pend_old = atomicAdd(f.cnt + c, 1u);
                pend_c = c;
            }
            if (fc != kNone) flow_fold<T>(a, f, fc, wred);
        } else {
            __syncthreads();  // s_tk / s_fold visible
            ni = s_tk[par];
            const uint32_t fc = s_fold[par];
            // a pending fold first: this item may wait, the fold never waits
            // on anything but statistics items
            if (fc != kNone) flow_fold<T>(a, f, fc, wred);
            if (tid == 0) s_stat[par] = poll_word(f.chst + w.c, a.wait_limit, a.fault);
            __syncthreads();
            const uint64_t word = s_stat[par];
            const float md = __uint_as_float((unsigned)word);
            const float rstd = __uint_as_float((unsigned)(word >> 32));
            const float g = bn_param<T>(a.gamma, w.c, 1.f);
            const float bb = bn_param<T>(a.beta, w.c, 0.f);
            const float2 nk = f2(-K), nmd = f2(-md), r2 = f2(rstd), g2 = f2(g), b2 = f2(bb);
            uint4 *yp = reinterpret_cast<uint4 *>(static_cast<T *>(a.y) + w.base) + w.off + tid;
#pragma unroll
            for (int j = 0; j < PACKS; ++j)
                if (tid + j * BNF_THREADS < w.len) {
                    float2 fv[H], o[H];
                    io2::unpack(v[j], fv);
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(__fadd2_rn(fv[h], nk), nmd), r2), g2, b2);
                    __stcs(yp + j * BNF_THREADS, io2::pack(o));
                }
            if (ni < f.items) {
                w = flow_item(f, C, HW, ni);
                flow_load<T, PACKS>(a, w, v);
            }
        }
        if (ni >= f.items) break;
        i = ni;
        par ^= 1;
    }
    // the last item may have completed its channel
    if (tid == 0) s_fold[par ^ 1] = pend_c != kNone && pend_old == f.U - 1 ? pend_c : kNone;
    __syncthreads();
    if (s_fold[par ^ 1] != kNone) flow_fold<T>(a, f, s_fold[par ^ 1], wred);
}

template <typename T, int PACKS>
cudaError_t launch_bn_flow_t(const BnArgs &a, int num_sms, cudaStream_t s, bool *launched) {
    *launched = false;
    constexpr int V = IO<T>::V;
    if (a.HW % V != 0 || !bn_aligned16(a.x) || !bn_aligned16(a.y) || !a.fault || !a.ws ||
        !bn_aligned16(a.ws) || a.HW / V >= kBnMaxPlanePacks)
        return cudaSuccess;
    auto kernel = bn_flow_kernel<T, PACKS>;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), BNF_THREADS, 0, &per_sm);
    if (oe != cudaSuccess) return oe;
    FlowPlan f;
    int64_t grid = 0;
    // chunks of at most BNF_THREADS * PACKS packs (never more chunks than the
    // kBnChunkPacks units the workspace is sized for)
    if (!flow_plan(a.batch, a.C, a.HW / V, BNF_THREADS * PACKS, a.prefetch, per_sm, num_sms,
                   a.batch * a.HW * (int64_t)sizeof(T), a.ws, a.ws_bytes, &f, &grid))
        return cudaSuccess;
    *launched = true;
    const cudaError_t e = flow_reset(f, a.C, num_sms, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, (unsigned)grid, BNF_THREADS, s, true, a, f);
}

template <typename T>
cudaError_t launch_bn_flow_p(const BnArgs &a, int num_sms, cudaStream_t s, bool *launched) {
    // four packs per thread while a plane fits one CTA that way, eight beyond
    // (fewer, larger items: each item costs a fixed chain of latencies)
    const int packs = a.packs ? a.packs : (a.HW / IO<T>::V <= BNF_THREADS * 4 ? 4 : 8);
    if (packs == 4) return launch_bn_flow_t<T, 4>(a, num_sms, s, launched);
    if (packs == 8) return launch_bn_flow_t<T, 8>(a, num_sms, s, launched);
    *launched = false;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bn_flow(const BnArgs &a, int dtype, int num_sms, cudaStream_t s, bool *launched) {
    switch (dtype) {
    case DT_F32: return launch_bn_flow_p<float>(a, num_sms, s, launched);
    case DT_F16: return launch_bn_flow_p<__half>(a, num_sms, s, launched);
    case DT_BF16: return launch_bn_flow_p<__nv_bfloat16>(a, num_sms, s, launched);
    default: *launched = false; return cudaErrorInvalidValue;
    }
}

}  // namespace nrm
