// bn_flow.cu -- BatchNorm2d training forward with x read once from HBM, for
// channels too large for the shared memory of one cluster (BatchNorm CUDA
// implementation walkthrough, jianying88.com/news/30214, §2.1-§2.4: the same
// two phases, per-plane partial statistics then per-channel fold and
// normalization).
//
// The two phases run in one persistent kernel as a dataflow over work items.
// An item is one unit (a chunk of at most kBnChunkPacks 16-byte packs of one
// (n, c) plane, bn_common.cuh), either a statistics item or a normalize item.
// The items are numbered in blocks of one channel's U = batch * nch units:
//
//   S(0) S(1) ... S(L-1)  S(L) A(0)  S(L+1) A(1) ...  S(C-1) A(C-1-L)  A(C-L) ... A(C-1)
//
// S(c) = statistics items of channel c, A(c) = its normalize items, so each
// channel is normalized L channels after its statistics were taken.  The
// host picks L so that the items in flight at one time (about one per
// resident CTA) rarely reach a channel whose statistics are still open, while
// the x of the last L channels stays far below L2's capacity: the normalize
// items re-read x from L2, and HBM sees x once and y once.
//
// Statistics item: the chunk in registers, its exact partial (mean, M2) on
// d = x - K (K = x[0, c, 0]) stored as one 64-bit word, then a relaxed
// increment of the channel's counter.  The CTA whose increment completes the
// channel folds it at the start of its next item: it reads the U partial
// words, each until it no longer holds the "open" pattern (64-bit
// single-copy-atomic accesses, so the partials need no fence), combines them
// in a fixed order (so the bits do not depend on who folds), writes
// save_mean/save_rstd and the running statistics, and stores the channel's
// (mean, rstd) as one 64-bit word.
// Normalize item: its chunk is already in flight; thread 0 polls the
// channel's 64-bit word until it is no longer open, and the CTA writes y.
//
// CTAs take items in number order from a ticket counter (relaxed atomics,
// fetched two items ahead).  A normalize item waits only for the fold of its
// channel; every statistics item of that channel has a smaller number and
// never waits, and the fold is done before the folding CTA's next item can
// wait on anything.  So the oldest unfinished item can always proceed,
// whatever number of CTAs is resident.  Every wait is bounded by the
// library's wait limit; a thread that gives up raises the fault bit and the
// kernel goes on (that call's outputs are then undefined), so it always ends.
//
// The partial words, counters, statistics words and ticket counter are reset
// by a small kernel launched before the flow kernel in stream order; the flow
// kernel is a programmatic dependent launch of it and waits for it
// (griddepcontrol.wait) before its first ticket.
//
// The loads of a CTA's next item are issued as soon as the registers of the
// current one are free (after its partial statistics, or after its stores),
// and thread 0 prefetches into L2 the chunk of the item pf * grid numbers
// ahead of its own.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "bn_common.cuh"

namespace nrm {

namespace {

constexpr int BNF_THREADS = BNS_THREADS;
constexpr int BNF_NW = BNF_THREADS / 32;
// Resident CTAs per SM for PACKS 16-byte packs per thread (register caps
// without spills: 48 and 64 registers).
template <int PACKS> constexpr int bnf_min_blocks() { return PACKS <= 4 ? 5 : 4; }
// High word of a partial or statistics word until it is stored (a NaN
// pattern no result takes: M2 is clamped at zero and a computed rstd that is
// NaN is stored as 0x7fffffff).
constexpr unsigned kOpen = 0xffffffffu;
constexpr uint32_t kNone = 0xffffffffu;

struct FlowPlan {
    BnChunks u;           // unit layout over all channels
    uint32_t U;           // units per channel (batch * nch)
    uint32_t L;           // channels between a channel's statistics and its normalization
    uint32_t items;       // 2 * C * U
    uint32_t pf;          // L2 prefetch distance in multiples of the grid (0: none)
    FastDiv divU, divN;   // by U and by nch
    uint64_t *part;       // per-unit partials (mean bits low, M2 bits high), [c * U + n * nch + k]
    uint64_t *chst;       // per channel: shifted mean bits low, rstd bits high
    unsigned *cnt;        // per channel: statistics units done
    unsigned *ticket;     // next item number
};

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t pack_word(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

// Bounded poll of a 64-bit word until its high half is no longer open; on
// giving up the fault bit is raised and the open word returned.
__device__ __forceinline__ uint64_t poll_word(const uint64_t *p, unsigned limit, unsigned *fault) {
    uint64_t word = (uint64_t)kOpen << 32;
    for (unsigned tries = 0; tries < limit; ++tries) {
        word = ld_relaxed_gpu(p);
        if ((unsigned)(word >> 32) != kOpen) return word;
        __nanosleep(32);
    }
    atomicOr(fault, FAULT_WAIT);
    return word;
}

struct FlowIdx {
    bool stats;
    uint32_t c, unit;
    int off, len;          // first pack of the chunk within its plane, packs in it
    int64_t base;          // first element of the plane
};

// Item i -> (statistics?, channel, unit within the channel) per the block
// layout above, and the unit's chunk.
__device__ __forceinline__ FlowIdx flow_item(const FlowPlan &f, uint32_t C, int64_t HW, uint32_t i) {
    FlowIdx w;
    const uint32_t b = fast_div(i, f.divU);
    w.unit = i - b * f.U;
    if (b < f.L) {
        w.stats = true;
        w.c = b;
    } else if (b < 2 * C - f.L) {
        const uint32_t r = b - f.L;
        w.stats = (r & 1) == 0;
        w.c = (r >> 1) + (w.stats ? f.L : 0);
    } else {
        w.stats = false;
        w.c = b - C;
    }
    const uint32_t n = fast_div(w.unit, f.divN);
    const int k = (int)(w.unit - n * (uint32_t)f.u.nch);
    w.off = k * f.u.cpk;
    w.len = min(f.u.cpk, f.u.q - w.off);
    w.base = ((int64_t)n * C + w.c) * HW;
    return w;
}

template <typename T>
__device__ __forceinline__ const uint4 *flow_ptr(const BnArgs &a, const FlowIdx &w) {
    return reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + w.base) + w.off;
}

// The chunk of item w into registers: statistics items read with the
// default L2 policy (the normalize items re-read the data from L2), normalize
// items evict-first (last use).
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

// Opens every partial and statistics word (16 bytes per thread and step: the
// two areas are padded to 16 bytes), zeroes the counters and the ticket.
__global__ void __launch_bounds__(256) bn_flow_reset_kernel(uint4 *words, int64_t quads, unsigned *cnt,
                                                            int64_t C, unsigned *ticket) {
    pdl_launch_dependents();
    const uint4 open = make_uint4(0u, kOpen, 0u, kOpen);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (int64_t i = t; i < quads; i += stride) words[i] = open;
    for (int64_t i = t; i < C; i += stride) cnt[i] = 0u;
    if (t == 0) *ticket = 0u;
}

// Fold of channel c by the whole CTA (see the header); thread 0 publishes.
template <typename T>
__device__ __forceinline__ void flow_fold(const BnArgs &a, const FlowPlan &f, uint32_t c, Stats *wred) {
    constexpr int V = IO<T>::V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t *pc = f.part + (int64_t)c * f.U;
    Stats st{0.f, 0.f, 0.f};
    for (uint32_t j = tid; j < f.U; j += BNF_THREADS) {
        const uint64_t word = poll_word(pc + j, a.wait_limit, a.fault);
        const int kk = (int)(j - fast_div(j, f.divN) * (uint32_t)f.u.nch);
        const float cn = (float)(min(f.u.cpk, f.u.q - kk * f.u.cpk) * V);
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
        const float rs = __float_as_uint(rstd) == kOpen ? __uint_as_float(0x7fffffffu) : rstd;
        st_relaxed_gpu(f.chst + c, pack_word(t.mean, rs));
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

// L2 bytes the lag may keep in flight (x of L channels, their y on its way
// out as well): a fraction of GB300's 126 MB L2.
constexpr int64_t kFlowL2Budget = (int64_t)40 << 20;

template <typename T, int PACKS>
cudaError_t launch_bn_flow_t(const BnArgs &a, int num_sms, cudaStream_t s, bool *launched) {
    *launched = false;
    constexpr int V = IO<T>::V;
    if (a.HW % V != 0 || !bn_aligned16(a.x) || !bn_aligned16(a.y) || !a.fault || !a.ws ||
        !bn_aligned16(a.ws) || a.HW / V >= kBnMaxPlanePacks)
        return cudaSuccess;
    // chunks of at most BNF_THREADS * PACKS packs (never more chunks than the
    // kBnChunkPacks units the workspace is sized for)
    BnChunks u;
    u.c0 = 0;
    u.G = a.C;
    u.q = (int)(a.HW / V);
    u.nch = std::max(1, (u.q + BNF_THREADS * PACKS - 1) / (BNF_THREADS * PACKS));
    u.cpk = (u.q + u.nch - 1) / u.nch;
    const int64_t U = a.batch * u.nch, items = 2 * a.C * U;
    // 32-bit item numbers, with room for i + pf * grid
    if (items > 0x3fffffff || a.ws_bytes < bn_flow_ws_bytes(a.C, a.C * U)) return cudaSuccess;
    FlowPlan f;
    f.u = u;
    f.U = (uint32_t)U;
    f.items = (uint32_t)items;
    f.pf = a.prefetch == 0 ? 2u : a.prefetch == 1 ? 0u : (uint32_t)std::min(a.prefetch - 1, 8);
    f.divU = make_fastdiv(f.U);
    f.divN = make_fastdiv((uint32_t)u.nch);
    auto kernel = bn_flow_kernel<T, PACKS>;
    int per_sm = 0;
    const cudaError_t oe = resident_ctas(reinterpret_cast<const void *>(kernel), BNF_THREADS, 0, &per_sm);
    if (oe != cudaSuccess) return oe;
    if (per_sm < 1) return cudaSuccess;
    const int64_t cap = (int64_t)per_sm * num_sms;
    const int64_t grid = items < cap ? items : cap;
    // lag: past the items in flight at once (about `grid`; before the first
    // normalize block the item numbers advance one block of U per channel),
    // within the L2 budget
    const int64_t chan_bytes = a.batch * a.HW * (int64_t)sizeof(T);
    int64_t L = (grid + U - 1) / U + 2;
    const int64_t Lmax = kFlowL2Budget / (chan_bytes > 0 ? chan_bytes : 1);
    if (L > Lmax) L = Lmax;
    if (L > a.C) L = a.C;
    if (L < 1) L = 1;
    f.L = (uint32_t)L;
    // workspace: partials (padded to 16 bytes), statistics words (padded to
    // 16 bytes), counters, ticket -- within bn_flow_ws_bytes
    char *ws = static_cast<char *>(a.ws);
    const size_t part_bytes = ((size_t)(a.C * U) * 8 + 15) & ~(size_t)15;
    const size_t chst_bytes = ((size_t)a.C * 8 + 15) & ~(size_t)15;
    f.part = reinterpret_cast<uint64_t *>(ws);
    f.chst = reinterpret_cast<uint64_t *>(ws + part_bytes);
    f.cnt = reinterpret_cast<unsigned *>(ws + part_bytes + chst_bytes);
    f.ticket = f.cnt + a.C;
    *launched = true;
    const int64_t quads = (int64_t)((part_bytes + chst_bytes) / 16);
    const int64_t rgrid = std::min<int64_t>(std::max<int64_t>((quads + 1023) / 1024, 1), num_sms);
    bn_flow_reset_kernel<<<(unsigned)rgrid, 256, 0, s>>>(reinterpret_cast<uint4 *>(ws), quads, f.cnt,
                                                         a.C, f.ticket);
    cudaError_t e = cudaGetLastError();
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
