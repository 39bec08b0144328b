// bn_flow.cuh -- the dataflow machinery shared by the one-pass BatchNorm
// kernels (bn_flow.cu: training forward; bn_flow_bwd.cu: training backward).
//
// Both run the two phases of a per-channel reduction (statistics, then an
// element-wise pass that needs them) in one persistent kernel over work
// items.  An item is a chunk of at most BNF_THREADS * PACKS 16-byte packs of
// one (n, c) plane, either a statistics item or an apply item.  The items are
// numbered in blocks of one channel's U = batch * nch chunks:
//
//   S(0) S(1) ... S(L-1)  S(L) A(0)  S(L+1) A(1) ...  S(C-1) A(C-1-L)  A(C-L) ... A(C-1)
//
// S(c) = statistics items of channel c, A(c) = its apply items, so each
// channel is applied L channels after its statistics were taken.  The host
// picks L so that the items in flight at one time (about one per resident
// CTA) rarely reach a channel whose statistics are still open, while the
// inputs of the last L channels stay far below L2's capacity: the apply items
// re-read them from L2, and HBM sees each input once.
//
// A statistics item stores its partial as one 64-bit word, then makes a
// relaxed increment of the channel's counter; the CTA whose increment
// completes the channel folds it at the start of its next item, reading the
// U partial words, each until it no longer holds the "open" pattern (64-bit
// single-copy-atomic accesses, so the partials need no fence), and stores the
// channel's result as one 64-bit word.  An apply item polls that word.
//
// CTAs take items in number order from a ticket counter (relaxed atomics,
// fetched two items ahead).  An apply item waits only for the fold of its
// channel; every statistics item of that channel has a smaller number and
// never waits, and a fold is done before the folding CTA's next item can
// wait on anything.  So the oldest unfinished item can always proceed,
// whatever number of CTAs is resident.  Every wait is bounded by the
// library's wait limit; a thread that gives up raises the fault bit and the
// kernel goes on (that call's outputs are then undefined), so it always ends.
//
// The partial words, counters, result words and ticket counter are reset by
// a small kernel launched before the flow kernel in stream order; the flow
// kernel is a programmatic dependent launch of it and waits for it
// (griddepcontrol.wait) before its first ticket.
#pragma once

#include <algorithm>
#include <cstdint>

#include "bn_common.cuh"

namespace nrm {

namespace {

constexpr int BNF_THREADS = BNS_THREADS;
constexpr int BNF_NW = BNF_THREADS / 32;
// High word of a partial or result word until it is stored (a NaN pattern
// that no stored value takes: the writers store a computed NaN as 0x7fffffff).
constexpr unsigned kOpen = 0xffffffffu;
constexpr uint32_t kNone = 0xffffffffu;
// L2 bytes the lag may keep in flight (the inputs of L channels, their
// outputs on the way out as well): a fraction of GB300's 126 MB L2.
// NRM_FLOW_L2_MB overrides it for experiments.
#ifndef NRM_FLOW_L2_MB
#define NRM_FLOW_L2_MB 40
#endif
constexpr int64_t kFlowL2Budget = (int64_t)NRM_FLOW_L2_MB << 20;

struct FlowPlan {
    BnChunks u;           // chunk layout over all channels
    uint32_t U;           // chunks per channel (batch * nch)
    uint32_t L;           // channels between a channel's statistics and its apply items
    uint32_t items;       // 2 * C * U
    uint32_t pf;          // L2 prefetch distance in multiples of the grid (0: none)
    FastDiv divU, divN;   // by U and by nch
    uint64_t *part;       // per-chunk partials, [c * U + n * nch + k]
    uint64_t *chst;       // per channel: the folded result word
    unsigned *cnt;        // per channel: statistics items done
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
// A word of two binary32 values; a high half that would read as open is
// stored as the canonical NaN.
__device__ __forceinline__ uint64_t pack_word(float lo, float hi) {
    unsigned h = __float_as_uint(hi);
    if (h == kOpen) h = 0x7fffffffu;
    return ((uint64_t)h << 32) | __float_as_uint(lo);
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

// Item i -> (statistics?, channel, chunk within the channel) per the block
// layout above, and the chunk's place.
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

// Packs of chunk k of a plane (the last chunk may be shorter).
__device__ __forceinline__ int flow_chunk_len(const FlowPlan &f, uint32_t j) {
    const int kk = (int)(j - fast_div(j, f.divN) * (uint32_t)f.u.nch);
    return min(f.u.cpk, f.u.q - kk * f.u.cpk);
}

// Opens every partial and result word (16 bytes per thread and step: the two
// areas are padded to 16 bytes), zeroes the counters and the ticket.
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

// Host side: the plan for planes of q packs split into chunks of at most
// chunk_cap packs, `per_sm` resident CTAs per SM, `chan_bytes` input bytes per
// channel (for the lag), the workspace carved as partials | result words |
// counters | ticket.  Returns false (nothing launched) when the item numbers
// or the workspace do not allow the plan; *grid is the CTA count.
inline bool flow_plan(int64_t batch, int64_t C, int64_t q, int chunk_cap, int prefetch, int per_sm,
                      int num_sms, int64_t chan_bytes, void *ws, size_t ws_bytes, FlowPlan *f,
                      int64_t *grid) {
    BnChunks u;
    u.c0 = 0;
    u.G = C;
    u.q = (int)q;
    u.nch = std::max(1, (u.q + chunk_cap - 1) / chunk_cap);
    u.cpk = (u.q + u.nch - 1) / u.nch;
    const int64_t U = batch * u.nch, items = 2 * C * U;
    // 32-bit item numbers, with room for i + pf * grid
    if (per_sm < 1 || items > 0x3fffffff || ws_bytes < bn_flow_ws_bytes(C, C * U)) return false;
    f->u = u;
    f->U = (uint32_t)U;
    f->items = (uint32_t)items;
    f->pf = prefetch == 0 ? 2u : prefetch == 1 ? 0u : (uint32_t)std::min(prefetch - 1, 8);
    f->divU = make_fastdiv(f->U);
    f->divN = make_fastdiv((uint32_t)u.nch);
    const int64_t cap = (int64_t)per_sm * num_sms;
    *grid = items < cap ? items : cap;
    // lag: past the items in flight at once (about `grid`; before the first
    // apply block the item numbers advance one block of U per channel),
    // within the L2 budget
    int64_t L = (*grid + U - 1) / U + 2;
    const int64_t Lmax = kFlowL2Budget / (chan_bytes > 0 ? chan_bytes : 1);
    if (L > Lmax) L = Lmax;
    if (L > C) L = C;
    if (L < 1) L = 1;
    f->L = (uint32_t)L;
    char *w = static_cast<char *>(ws);
    const size_t part_bytes = ((size_t)(C * U) * 8 + 15) & ~(size_t)15;
    f->part = reinterpret_cast<uint64_t *>(w);
    f->chst = reinterpret_cast<uint64_t *>(w + part_bytes);
    f->cnt = reinterpret_cast<unsigned *>(w + part_bytes + (((size_t)C * 8 + 15) & ~(size_t)15));
    f->ticket = f->cnt + C;
    return true;
}

// The reset kernel for plan f (in stream order, not a dependent launch).
inline cudaError_t flow_reset(const FlowPlan &f, int64_t C, int num_sms, cudaStream_t s) {
    const int64_t quads = (int64_t)((reinterpret_cast<char *>(f.cnt) - reinterpret_cast<char *>(f.part)) / 16);
    const int64_t rgrid = std::min<int64_t>(std::max<int64_t>((quads + 1023) / 1024, 1), num_sms);
    bn_flow_reset_kernel<<<(unsigned)rgrid, 256, 0, s>>>(reinterpret_cast<uint4 *>(f.part), quads, f.cnt, C,
                                                         f.ticket);
    return cudaGetLastError();
}

}  // namespace

}  // namespace nrm
