// bn.cu -- BatchNorm2d training forward over NCHW data (binary32, binary16 or
// bfloat16 storage; statistics in binary32), as a two-phase channel reduction
// (BatchNorm CUDA implementation walkthrough, jianying88.com/news/30214,
// §2.1-§2.4 and its Welford discussion in §4.3):
//
//   phase 1  partial statistics (mean, M2) of each (n, c) plane (H*W
//            contiguous values);
//   phase 2  fold the batch's partials of a channel (every CTA of a channel
//            folds them in the same order, so all agree bit for bit),
//            normalize and write y; one CTA per channel writes
//            save_mean/save_rstd and the running statistics.
//
// Three plans carry the two phases: one thread-block cluster per channel
// holding the channel in shared memory (a single read of x), two streaming
// kernels chained by programmatic dependent launch (the second read of x is
// served from L2 for batches that fit there), and a scalar two-kernel plan
// for any layout.
//
// All statistics of channel c are taken on d = x - K_c with K_c the channel's
// first element x[0, c, 0]: the shift keeps channels with a large mean and a
// small spread free of cancellation.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bn_common.cuh"
#include "nrm.h"

namespace nrm {

namespace {

// ---------------------------------------------------------------------------
// Scalar two-kernel plan (any HW, any element-aligned pointers).
// ---------------------------------------------------------------------------
constexpr int BN_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(BN_THREADS) bn_partial_kernel(const BnArgs a) {
    constexpr int NW = BN_THREADS / 32;
    constexpr int V = IO<T>::V;
    __shared__ float s_red[2][NW][3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t planes = a.batch * a.C;
    const int64_t HW = a.HW;
    const T *X = static_cast<const T *>(a.x);
    const bool vec = (HW % V == 0) && bn_aligned16(a.x);
    float2 *ws = static_cast<float2 *>(a.ws);
    int buf = 0;
    for (int64_t p = blockIdx.x; p < planes; p += gridDim.x, buf ^= 1) {
        const int64_t n = p / a.C, c = p - n * a.C;
        const T *xp = X + p * HW;
        const float K = bn_elem<T>(a.x, c * HW);  // x[0, c, 0]
        Stats st{0.f, 0.f, 0.f};
        if (vec) {
            const int64_t P = HW / V;
            for (int64_t i = tid; i < P; i += BN_THREADS) {
                float f[V];
                IO<T>::unpack(ld_stream(xp + V * i), f);
                // exact local two-pass over the pack's V values
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < V; ++j) s += f[j] - K;
                const float m = s * (1.f / V);
                float m2 = 0.f;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const float e = (f[j] - K) - m;
                    m2 = fmaf(e, e, m2);
                }
                st = combine(st, Stats{(float)V, m, m2});
            }
        } else {
            for (int64_t i = tid; i < HW; i += BN_THREADS) {
                const float d = IO<T>::to_f(xp[i]) - K;
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

template <typename T>
__global__ void __launch_bounds__(BN_THREADS) bn_apply_kernel(const BnArgs a) {
    constexpr int V = IO<T>::V;
    __shared__ float s_stat[2][2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t planes = a.batch * a.C;
    const int64_t HW = a.HW;
    const float cnt = (float)(a.batch * HW);
    const T *X = static_cast<const T *>(a.x);
    T *Y = static_cast<T *>(a.y);
    const bool vec = (HW % V == 0) && bn_aligned16(a.x) && bn_aligned16(a.y);
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
        const float K = bn_elem<T>(a.x, c * HW);
        const float md = s_stat[buf][0];
        const float var = s_stat[buf][1] / cnt;
        const float rstd = 1.0f / sqrtf(var + a.eps);
        if (n == 0 && tid == 0) bn_write_channel_stats(a, c, K, md, var, rstd);
        const float g = bn_param<T>(a.gamma, c, 1.f);
        const float b = bn_param<T>(a.beta, c, 0.f);
        const T *xp = X + p * HW;
        T *yp = Y + p * HW;
        if (vec) {
            const int64_t P = HW / V;
            for (int64_t i = tid; i < P; i += BN_THREADS) {
                float f[V], o[V];
                IO<T>::unpack(ld_stream(xp + V * i), f);
#pragma unroll
                for (int j = 0; j < V; ++j) o[j] = fmaf(((f[j] - K) - md) * rstd, g, b);
                st_stream(yp + V * i, IO<T>::pack(o));
            }
        } else {
            for (int64_t i = tid; i < HW; i += BN_THREADS)
                yp[i] = IO<T>::from_f(fmaf(((IO<T>::to_f(xp[i]) - K) - md) * rstd, g, b));
        }
    }
}

// ---------------------------------------------------------------------------
// Streaming two-kernel plan (16-byte aligned planes of any size).
//
// The work is cut into units, chunks of at most 1024 packs of one plane
// (bn_common.cuh), and the channels into groups whose x fits comfortably in
// L2.  Per group:
// bn_stats_kernel: one CTA per unit holds the chunk in registers and computes
// its exact partial statistics on d = x - K (K = x[0, c, 0]) with a corrected
// two-pass: (mean_d, M2) into the workspace.  It then allows the dependent
// launch to start.
// bn_norm_kernel (launched with programmatic stream serialization): each CTA
// loads its chunk of x into registers first -- x is an input, and the group
// was just read, so these reads hit L2 -- then waits for the statistics
// kernel (griddepcontrol.wait), folds the channel's partials in a fixed order
// (every CTA of a channel gets the same bits), normalizes and writes y.  The
// CTA of unit (n = 0, chunk 0) writes save_mean/save_rstd and the running
// statistics.  It lets the next group's statistics kernel start as soon as
// its own loads are issued, so that kernel fills the SMs this one frees; that
// kernel waits at its end for this one to finish (griddepcontrol.wait), so
// each call's last kernel completes after all of the call's kernels.  No
// kernel of the chain waits on a grid that is not fully resident: a
// dependent grid starts only once every CTA of its primary has started.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(BNS_THREADS) bn_stats_kernel(const BnArgs a, const BnChunks u) {
    constexpr int NW = BNS_THREADS / 32;
    __shared__ float s1[2][NW];
    __shared__ float2 s2[2][NW];
    const int tid = threadIdx.x;
    const int64_t units = a.batch * u.G * u.nch, HW = a.HW;
    float2 *ws = static_cast<float2 *>(a.ws);
    if (u.c0 == 0) {
        // first group, a programmatic dependent of the stream's previous
        // kernel: request the first unit's chunk from L2, then wait for that
        // kernel (its outputs may be x, and it may still read the workspace)
        if (tid == 0 && blockIdx.x < units) {
            const BnUnit w = bn_unit(u, blockIdx.x);
            prefetch_l2_bulk(reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) +
                                                             (w.n * a.C + w.c) * HW) + w.off,
                             (uint32_t)w.len * 16u);
        }
        pdl_wait();
    }
    // the normalize kernel may launch once every CTA of this grid has started
    // (it waits for this grid's completion before it reads the partials)
    pdl_launch_dependents();
    int par = 0;
    for (int64_t idx = blockIdx.x; idx < units; idx += gridDim.x, par ^= 1) {
        const BnUnit w = bn_unit(u, idx);
        const uint4 *xp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) +
                                                          (w.n * a.C + w.c) * HW) + w.off;
        // first read of x: default L2 policy, so the normalize kernel's second
        // read finds it in L2 (a streaming, evict-first read would lose it)
        uint4 v[BNS_PACKS];
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) v[k] = __ldg(xp + tid + k * BNS_THREADS);
        const float K = bn_elem<T>(a.x, w.c * HW);
        const float2 r = bn_unit_partial<T>(v, w.len, K, s1[par], s2[par]);
        if (tid == 0) ws[w.c * (a.batch * u.nch) + w.n * u.nch + w.k] = r;
    }
    // A later group's statistics kernel overlaps the previous group's
    // normalize kernel; it finishes only after that kernel has, so the end of
    // the last kernel of a call implies the end of all of them.
    pdl_wait();
}

template <typename T>
__global__ void __launch_bounds__(BNS_THREADS) bn_norm_kernel(const BnArgs a, const BnChunks u) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int V = IO<T>::V;
    __shared__ float stat[2][3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t units = a.batch * u.G * u.nch, HW = a.HW;
    const int64_t per_channel = a.batch * u.nch;  // partials per channel
    const float ctot = (float)(a.batch * HW);
    const float2 *ws = static_cast<const float2 *>(a.ws);
    bool waited = false;
    int par = 0;
    for (int64_t idx = blockIdx.x; idx < units; idx += gridDim.x, par ^= 1) {
        const BnUnit w = bn_unit(u, idx);
        const int64_t base = (w.n * a.C + w.c) * HW;
        const uint4 *xp = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.x) + base) + w.off;
        uint4 v[BNS_PACKS];
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) v[k] = __ldcs(xp + tid + k * BNS_THREADS);
        const float K = bn_elem<T>(a.x, w.c * HW);
        if (!waited) {
            pdl_launch_dependents();  // the next group's statistics may start
            pdl_wait();  // the statistics kernel has finished and its writes are visible
            waited = true;
        }
        if (warp == 0) {
            Stats st{0.f, 0.f, 0.f};
            for (int64_t j = lane; j < per_channel; j += 32) {
                const float2 qq = ws[w.c * per_channel + j];
                const int kk = (int)(j % u.nch);
                const float cn = (float)(min(u.cpk, u.q - kk * u.cpk) * V);
                st = combine(st, Stats{cn, qq.x, qq.y});
            }
            st = warp_stats_down(st);
            if (lane == 0) {
                const float var = st.m2 / ctot;
                stat[par][0] = st.mean;
                stat[par][1] = 1.0f / sqrtf(var + a.eps);
                stat[par][2] = var;
            }
        }
        __syncthreads();
        const float md = stat[par][0], rstd = stat[par][1];
        if (w.n == 0 && w.k == 0 && tid == 0) bn_write_channel_stats(a, w.c, K, md, stat[par][2], rstd);
        const float g = bn_param<T>(a.gamma, w.c, 1.f);
        const float bb = bn_param<T>(a.beta, w.c, 0.f);
        const float2 nk = f2(-K), nmd = f2(-md), r2 = f2(rstd), g2 = f2(g), b2 = f2(bb);
        uint4 *yp = reinterpret_cast<uint4 *>(static_cast<T *>(a.y) + base) + w.off;
#pragma unroll
        for (int k = 0; k < BNS_PACKS; ++k)
            if (tid + k * BNS_THREADS < w.len) {
                float2 f[H], o[H];
                io2::unpack(v[k], f);
#pragma unroll
                for (int h = 0; h < H; ++h)
                    o[h] = __ffma2_rn(__fmul2_rn(__fadd2_rn(__fadd2_rn(f[h], nk), nmd), r2), g2, b2);
                __stcs(yp + tid + k * BNS_THREADS, io2::pack(o));
            }
    }
    if (!waited) {
        pdl_launch_dependents();
        pdl_wait();
    }
}

// ---------------------------------------------------------------------------
// Thread-block clusters over channels (a single-launch plan).
//
// Cluster k (cs CTAs, 2 to 16) handles channels k, k + K, k + 2K, ... (K
// clusters).  The cs CTAs split the batch: CTA rank r owns planes n in
// [r*ppc, min((r+1)*ppc, batch)) of the channel.  When every channel has a
// resident cluster a CTA needs one shared-memory buffer; otherwise it holds
// two when they fit, and while channel i is reduced and written from one
// buffer the planes of channel i+1 stream into the other; else one, the
// cluster taking its channels one after another.  The planes arrive as one
// bulk asynchronous copy per plane, each completing on its own mbarrier, or
// (16-bit planes, BOX) as one tiled tensor copy of all of them on one
// mbarrier; x is read from HBM once.
//
// Statistics in one pass, plane by plane as the copies land: thread t keeps
// (count, sum e, sum e^2) of e = x - K_t over its packs, K_t its own first
// value (a per-thread shift: a far-off K_t only affects that thread's few
// values, whose sums stay small).  From these each thread forms its mean
// relative to the channel shift K = x[0, c, 0] and its M2; the CTA merges
// them exactly with two CTA-wide sums (the mean, then M2_t + n_t (m_t -
// m)^2, a sum of non-negative terms), publishes (count, mean, M2), and after
// a cluster barrier every CTA folds the cs partials over distributed shared
// memory in rank order (all agree bit for bit).  Then it normalizes its
// planes, y = ((x - K) - md) * (rstd * gamma) + beta, and writes y.  Rank 0
// writes save_mean/save_rstd and the running statistics.  In statistics-only
// mode (STATS, for synchronized BatchNorm) rank 0 instead writes the
// channel's binary64 (count, mean, M2) and nothing is normalized.  The barrier that
// protects the partials is split: each CTA arrives right after its fold and
// waits only before it writes the next channel's partial (or exits), so it
// overlaps the stores of y.  Every bulk-copy wait is bounded; on a give-up
// the thread raises a fault bit, the CTA stops issuing copies, keeps taking
// part in every barrier, and drains its copies in flight before exiting.
// ---------------------------------------------------------------------------
constexpr int BNC_THREADS = 512;
constexpr int kBnMaxPpc = 16;  // planes per CTA (one mbarrier each per buffer)

// How a CTA's planes of one channel arrive: BnBox<false>, one bulk copy per
// plane, each on its own barrier; BnBox<true>, one tiled tensor copy (TMA) of
// the box HW as k x HW / k, one channel, ppc planes, on one barrier.
template <bool BOX> struct BnBox {};
template <> struct BnBox<true> {
    CUtensorMap map;  // 64-byte aligned, first
    uint32_t bytes;   // the box's bytes (out-of-range planes included)
};

// The loads of channel c's planes n0 .. n0 + np - 1 into `buf`.
template <typename T, bool BOX>
__device__ __forceinline__ void bn_issue_planes(const BnArgs &a, uint4 *buf, uint64_t *bars,
                                                int64_t c, int64_t n0, int np, int q,
                                                uint32_t plane_bytes, const BnBox<BOX> &box) {
    if constexpr (BOX) {
        mbar_arrive_expect_tx(&bars[0], box.bytes);
        tma_load_4d(buf, &box.map, 0, 0, (int)c, (int)n0, &bars[0]);
        return;
    }
    for (int j = 0; j < np; ++j) {
        mbar_arrive_expect_tx(&bars[j], plane_bytes);
        bulk_g2s(buf + (size_t)j * q, static_cast<const T *>(a.x) + ((n0 + j) * a.C + c) * a.HW,
                 plane_bytes, &bars[j]);
    }
}

// binary32: four 512-thread CTAs per SM (at most 32 registers): with fewer,
// the 8-CTA clusters of a 64-channel batch no longer all fit at once.
// 16-bit and statistics only: two (the compiler takes about 42 registers;
// [32, 64, 56, 56] bfloat16 9.67 -> 9.33 us, [64, 64, 112, 112] 67.3 ->
// 65.5 us; the binary32 normalize measured 11.78 -> 11.88 us that way and
// keeps four).
template <typename T, bool BOX, bool STATS>
__global__ void __launch_bounds__(BNC_THREADS, (sizeof(T) == 2 || STATS) ? 2 : 4)
    bn_cluster_kernel(const BnArgs a, const int ppc, const int nbuf,
                      const __grid_constant__ BnBox<BOX> box) {
    namespace cg = cooperative_groups;
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int V = IO<T>::V;
    constexpr int NW = BNC_THREADS / 32;
    extern __shared__ __align__(128) uint4 sx[];  // nbuf (1 or 2) buffers of ppc planes
    __shared__ __align__(8) uint64_t bar[2][kBnMaxPpc];
    __shared__ float s1[2][NW];
    __shared__ float s2[2][NW];
    __shared__ float part[2][3];  // count, mean, M2 of this CTA's planes (shifted by K)
    __shared__ float stat[2][4];  // combined shifted mean, rstd, biased variance, M2
    __shared__ int s_fail;        // some wait of this CTA gave up

    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x;
    const int64_t C = a.C, HW = a.HW;
    const int64_t K_clusters = gridDim.x / cs;
    const int64_t first_c = blockIdx.x / cs;
    const int64_t n0 = (int64_t)rank * ppc;
    const int64_t left = a.batch - n0;
    const int np = (int)(left <= 0 ? 0 : left < ppc ? left : ppc);
    const int q = (int)(HW / V);  // 16-byte packs per plane
    const int tp = np * q;        // packs of this CTA's planes
    const uint32_t plane_bytes = (uint32_t)(HW * (int64_t)sizeof(T));
    // each buffer starts at a multiple of 128 bytes (a tensor copy's rule)
    const size_t buf_packs = ((size_t)ppc * q + 7) & ~(size_t)7;
    const float cnt = (float)np * (float)HW;
    const float ctot = (float)(a.batch * HW);

    // thread 0's bookkeeping: iteration whose planes were last issued into
    // each buffer (for the drain after a give-up)
    int last_issued0 = -1, last_issued1 = -1;
    // programmatic dependent launch: the CTA's planes of its first channel are
    // requested from L2 before the wait for the previous grid (L2 is where
    // that grid's writes become coherent; the bulk copies come after the wait)
    if (tid == 0 && np > 0 && first_c < C)
        for (int j = 0; j < np; ++j)
            prefetch_l2_bulk(static_cast<const T *>(a.x) + ((n0 + j) * C + first_c) * HW, plane_bytes);
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        s_fail = 0;
        for (int j = 0; j < (BOX ? 1 : np); ++j) {
            mbar_init(&bar[0][j], 1);
            mbar_init(&bar[1][j], 1);
        }
        fence_mbar_init();
        for (int b = 0; b < nbuf; ++b) {
            const int64_t c = first_c + b * K_clusters;
            if (np > 0 && c < C) {
                bn_issue_planes<T, BOX>(a, sx + b * buf_packs, bar[b], c, n0, np, q, plane_bytes, box);
                if (b == 0) last_issued0 = 0;
                else last_issued1 = 1;
            }
        }
    }
    __syncthreads();

    int i = 0;
    for (int64_t c = first_c; c < C; c += K_clusters, ++i) {
        // channel i sits in buffer i mod nbuf, that buffer's (i / nbuf)-th use
        const int b = nbuf == 2 ? (i & 1) : 0;
        const uint4 *buf = sx + b * buf_packs;
        const uint32_t par = (uint32_t)((nbuf == 2 ? i >> 1 : i) & 1);
        const float K = bn_elem<T>(a.x, c * HW);  // x[0, c, 0]
        // second half of the previous channel's barrier: every peer has folded
        // that channel's partials before any partial is written again
        if (i > 0) cluster_wait();

        // one pass, plane by plane as the copies land (flat pack index idx of
        // the buffer; thread t owns idx = t, t + THREADS, ...)
        float tn = 0.f, tK = 0.f;
        bool have = false;
        float2 a1 = f2(0.f), a2 = f2(0.f);
        int idx = tid;
        // with a box, its one barrier covers every plane
        if (BOX && idx < tp && !mbar_wait_bounded(&bar[b][0], par, a.wait_limit)) {
            s_fail = 1;  // read by thread 0 after the next __syncthreads
            atomicOr(a.fault, FAULT_WAIT);
        }
        for (int j = 0; j < np; ++j) {
            const int end = (j + 1) * q;
            if (idx >= end) continue;
            if (!BOX && !mbar_wait_bounded(&bar[b][j], par, a.wait_limit)) {
                s_fail = 1;  // read by thread 0 after the next __syncthreads
                atomicOr(a.fault, FAULT_WAIT);
            }
            for (; idx < end; idx += BNC_THREADS) {
                float2 f[H];
                io2::unpack(buf[idx], f);
                if (!have) {
                    tK = f[0].x;
                    have = true;
                }
                const float2 nk = f2(-tK);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 e = __fadd2_rn(f[h], nk);
                    a1 = __fadd2_rn(a1, e);
                    a2 = __ffma2_rn(e, e, a2);
                }
                tn += (float)V;
            }
        }
        // the thread's mean relative to K and its M2, merged over the CTA
        const float S1 = hsum(a1), S2 = hsum(a2);
        const float mt = tn > 0.f ? S1 / tn : 0.f;
        const float m2t = tn > 0.f ? fmaxf(fmaf(-S1, mt, S2), 0.f) : 0.f;
        const float mdt = tn > 0.f ? (tK - K) + mt : 0.f;
        const float md_r = np ? cta_sum_all<NW>(tn * mdt, s1[b]) / cnt : 0.f;
        const float dm = mdt - md_r;
        const float m2_r = cta_sum_all<NW>(fmaf(tn * dm, dm, m2t), s2[b]);
        if (tid == 0) {
            part[b][0] = cnt;
            part[b][1] = md_r;
            part[b][2] = m2_r;
        }
        cluster.sync();  // every partial of this channel is written

        // fold the cs partials in rank order: lanes 0..cs-1 of warp 0 read them
        // from the peers' shared memory in parallel, lane 0 combines
        if (tid < 32) {
            float pn = 0.f, pm = 0.f, p2 = 0.f;
            if (tid < cs) {
                const float *pr = cluster.map_shared_rank(&part[b][0], tid);
                pn = pr[0];
                pm = pr[1];
                p2 = pr[2];
            }
            Stats st{0.f, 0.f, 0.f};
            for (int r = 0; r < cs; ++r)
                st = combine(st, Stats{__shfl_sync(0xffffffffu, pn, r),
                                       __shfl_sync(0xffffffffu, pm, r),
                                       __shfl_sync(0xffffffffu, p2, r)});
            if (tid == 0) {
                const float var = st.m2 / ctot;
                stat[b][0] = st.mean;
                stat[b][1] = 1.0f / sqrtf(var + a.eps);
                stat[b][2] = var;
                stat[b][3] = st.m2;
            }
        }
        // nobody reads a peer's partial of this channel after this point:
        // arrive now, wait before the next channel (or exit), so the barrier
        // overlaps the stores of y instead of waiting for them
        cluster_arrive();
        __syncthreads();
        const float md = stat[b][0], rstd = stat[b][1];
        if constexpr (STATS) {
            // statistics only: the channel's binary64 (count, mean, M2)
            if (rank == 0 && tid == 0) {
                a.stats_out[3 * c + 0] = (double)ctot;
                a.stats_out[3 * c + 1] = (double)K + (double)md;
                a.stats_out[3 * c + 2] = (double)stat[b][3];
            }
        } else {
            if (rank == 0 && tid == 0) bn_write_channel_stats(a, c, K, md, stat[b][2], rstd);

            // normalize from shared memory: y = ((x - K) - md) * (rstd * gamma) + beta
            const float g = bn_param<T>(a.gamma, c, 1.f);
            const float bb = bn_param<T>(a.beta, c, 0.f);
            const float2 nk = f2(-K), nmd = f2(-md), A2 = f2(rstd * g), b2 = f2(bb);
            idx = tid;
            for (int j = 0; j < np && idx < tp; ++j) {
                const int end = (j + 1) * q;
                uint4 *yp = reinterpret_cast<uint4 *>(static_cast<T *>(a.y) + ((n0 + j) * C + c) * HW) -
                            (size_t)j * q;
                for (; idx < end; idx += BNC_THREADS) {
                    float2 f[H], o[H];
                    io2::unpack(buf[idx], f);
#pragma unroll
                    for (int h = 0; h < H; ++h)
                        o[h] = __ffma2_rn(__fadd2_rn(__fadd2_rn(f[h], nk), nmd), A2, b2);
                    __stcs(yp + idx, io2::pack(o));
                }
            }
        }
        __syncthreads();  // every thread is done with this buffer; s_fail is visible
        const int64_t next = c + nbuf * K_clusters;
        if (tid == 0 && np > 0 && next < C && !s_fail) {
            fence_proxy_async_smem();
            bn_issue_planes<T, BOX>(a, sx + b * buf_packs, bar[b], next, n0, np, q, plane_bytes, box);
            if (b == 0) last_issued0 = i + nbuf;
            else last_issued1 = i + nbuf;
        }
    }
    if (i > 0) cluster_wait();  // peers are done reading this CTA's last partials
    if (tid == 0 && s_fail) {
        // wait (bounded) for the copies of every plane's last issued phase; a
        // phase that already completed returns at once
        for (int b = 0; b < 2; ++b) {
            const int li = b == 0 ? last_issued0 : last_issued1;
            if (li < 0) continue;
            for (int j = 0; j < (BOX ? 1 : np); ++j)
                if (!mbar_wait_bounded(&bar[b][j], (uint32_t)((nbuf == 2 ? li >> 1 : li) & 1), 1u << 22))
                    atomicOr(a.fault, FAULT_DRAIN);
        }
    }
}

// Plan choice (measured on GB300 at [32, 64, 56, 56] binary32: cluster
// 11.8 us, streaming 17.3 us, one-pass 32.4 us, scalar 24.3 us).  One cluster of up to 8 CTAs
// per channel when the channel's planes fit the clusters' shared memory and
// every channel's cluster can be resident at once (one buffer); when there
// are more channels than resident clusters, each cluster pipelines its
// channels through two buffers.  Otherwise the streaming two kernels when
// the planes are 16-byte aligned and one unit long; else the scalar plan.
// one tiled tensor copy per CTA and channel for 16-bit planes (0: per-plane
// bulk copies; a measurement hook)
#ifndef NRM_BN_TMAP
#define NRM_BN_TMAP 1
#endif
// one-buffer cluster plan for channels too large for two buffers per CTA
#ifndef NRM_BN_ONE_BUFFER
#define NRM_BN_ONE_BUFFER 1
#endif

// cuTensorMapEncodeTiled through the runtime's driver entry point (nothing
// links against the driver library); null when unavailable.
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of the cluster kernel's loads: x seen as [batch][C][HW / k][k]
// (k innermost), box k x HW / k x 1 x ppc, so one tiled copy brings a CTA its
// ppc planes of one channel, laid out plane after plane as the per-plane
// copies would.  False (per-plane copies) when no view fits the tensor-copy
// rules: innermost box side a multiple of 16 bytes, every box side at most
// 256, strides multiples of 16 bytes (buffers sit at multiples of 128 bytes).
template <typename T>
bool bn_box_map(const BnArgs &a, int64_t ppc, size_t buf, CUtensorMap *m, uint32_t *box_bytes) {
    const int64_t es = (int64_t)sizeof(T), HW = a.HW;
    if (!NRM_BN_TMAP || !bn_aligned16(a.x) || (HW * es) % 16 || buf % 128 || ppc > 256 ||
        a.batch > 0x7fffffff || a.C > 0x7fffffff)
        return false;
    int64_t k = 0;
    for (int64_t d = 256; d >= 1 && !k; --d)
        if (HW % d == 0 && (d * es) % 16 == 0 && HW / d <= 256) k = d;
    const auto enc = tmap_encoder();
    if (!k || !enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)k, (cuuint64_t)(HW / k), (cuuint64_t)a.C,
                                (cuuint64_t)a.batch};
    const cuuint64_t strides[3] = {(cuuint64_t)(k * es), (cuuint64_t)(HW * es),
                                   (cuuint64_t)(a.C * HW * es)};
    const cuuint32_t box[4] = {(cuuint32_t)k, (cuuint32_t)(HW / k), 1u, (cuuint32_t)ppc};
    const cuuint32_t unit[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapDataType dt = sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : bn_dtype<T>() == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (enc(m, dt, 4, const_cast<void *>(a.x), dims, strides, box, unit,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    *box_bytes = (uint32_t)(ppc * HW * es);  // at most buf
    return true;
}

// Launch of one instance (per-plane copies, or one box) for cs CTAs per
// cluster of ppc planes each, buffers of buf bytes.  two_buf: the CTAs may
// hold two buffers (channels pipelined through them when not every channel
// has a resident cluster); else one, each cluster taking its channels one
// after another.
template <typename T, bool BOX, bool STATS>
cudaError_t launch_bn_cluster_k(const BnArgs &a, cudaStream_t s, bool *launched, int cs,
                                int64_t ppc, size_t buf, bool two_buf, const BnBox<BOX> &box) {
    auto kernel = bn_cluster_kernel<T, BOX, STATS>;
    static std::mutex mu;  // one per instance
    static int attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64 && !attr_done[dev]) {
            // 16-CTA clusters are a non-portable size
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemMax) == cudaSuccess &&
                cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                    cudaSuccess)
                attr_done[dev] = 1;
            else
                cudaGetLastError();
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(BNC_THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(a.C * cs));
    // one buffer if every channel gets its own resident cluster
    cfg.dynamicSmemBytes = buf;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return cudaSuccess;
    }
    int64_t k = a.C;
    int nbuf = 1;
    if (clusters < a.C || (a.max_clusters > 0 && a.max_clusters < a.C)) {
        if (two_buf) {
            cfg.dynamicSmemBytes = 2 * buf;
            nbuf = 2;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
                cudaGetLastError();
                return cudaSuccess;
            }
        }
        k = clusters;
        if (a.max_clusters > 0 && a.max_clusters < k) k = a.max_clusters;
    }
    if (k < 1) return cudaSuccess;
    cfg.gridDim = dim3((unsigned)(k * cs));
    *launched = true;
    cfg.numAttrs = 2;  // the occupancy queries above take the cluster shape alone
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, (int)ppc, nbuf, box);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename T>
cudaError_t launch_bn_cluster(const BnArgs &a, cudaStream_t s, bool *launched) {
    *launched = false;
    if (a.C > 0x7fffffff / 16) return cudaSuccess;
    // A CTA holds ppc = ceil(batch / cs) planes of a channel in a buffer of
    // buf bytes (rounded up to 128, as the kernel lays the buffers out).
    auto ppc_of = [&](int cs) { return (a.batch + cs - 1) / cs; };
    auto buf_of = [&](int cs) {
        return ((size_t)ppc_of(cs) * (size_t)a.HW * sizeof(T) + 127) & ~(size_t)127;
    };
    auto fits = [&](int cs, int nb) {
        return ppc_of(cs) <= kBnMaxPpc && nb * buf_of(cs) <= (size_t)(nb == 2 ? 200 : 220) * 1024;
    };
    // clusters of 4 CTAs when a CTA's two buffers fit (measured at
    // [32, 64, 56, 56]: binary32 11.8 us against 12.5 us with 8, bfloat16
    // 10.3 against 10.9), else 8; for 16-bit planes too large for that, one
    // buffer per CTA in clusters of 4, 8 or 16, each cluster taking its
    // channels one after another ([64, 64, 112, 112] bfloat16, 8 CTAs of
    // 196 KB: 66.3 us against 87.7 us for the one-pass plan; binary32, 16
    // CTAs of 196 KB: 110.4 us against 98.6, so binary32 leaves these shapes
    // to the one-pass plan).  A forced size wins.
    int cs = a.cluster_size;
    bool two_buf = true;
    if (cs == 2 || cs == 4 || cs == 8 || cs == 16) {
        while (cs > 1 && cs > a.batch) cs >>= 1;
        two_buf = fits(cs, 2);
        if (!two_buf && !(NRM_BN_ONE_BUFFER && fits(cs, 1))) return cudaSuccess;
    } else {
        cs = 0;
        for (int c : {4, 8})
            if (!cs && fits(c, 2)) cs = c;
        if (!cs && NRM_BN_ONE_BUFFER && sizeof(T) == 2) {
            two_buf = false;
            for (int c : {4, 8, 16})
                if (!cs && fits(c, 1)) cs = c;
        }
        if (!cs) return cudaSuccess;
        while (cs > 1 && cs > a.batch) cs >>= 1;
        two_buf = fits(cs, 2);
    }
    const int64_t ppc = ppc_of(cs);
    const size_t buf = buf_of(cs);
    // 16-bit planes arrive as one tiled tensor copy per CTA and channel where
    // the shape allows ([32, 64, 56, 56] bfloat16: 10.66 -> 9.58 us; the
    // per-plane copies' fixed cost dominates small planes); binary32 keeps
    // the per-plane copies, whose planes are reduced as each lands (12.5 us
    // with one box against 11.8)
    // statistics only (a.stats_out): an instance without the normalize
    if constexpr (sizeof(T) == 2) {
        BnBox<true> box;
        std::memset(&box, 0, sizeof(box));
        if (bn_box_map<T>(a, ppc, buf, &box.map, &box.bytes))
            return a.stats_out
                       ? launch_bn_cluster_k<T, true, true>(a, s, launched, cs, ppc, buf, two_buf, box)
                       : launch_bn_cluster_k<T, true, false>(a, s, launched, cs, ppc, buf, two_buf, box);
    }
    return a.stats_out ? launch_bn_cluster_k<T, false, true>(a, s, launched, cs, ppc, buf, two_buf,
                                                            BnBox<false>{})
                       : launch_bn_cluster_k<T, false, false>(a, s, launched, cs, ppc, buf, two_buf,
                                                             BnBox<false>{});
}

template <typename T>
cudaError_t launch_bn_stream(const BnArgs &a, int num_sms, cudaStream_t s) {
    BnChunks u = bn_chunks(a.HW / IO<T>::V);
    const int64_t G = bn_group_channels(a.C, a.batch * a.HW * (int64_t)sizeof(T),
                                        bn_group_budget());
    cudaError_t e = cudaSuccess;
    for (int64_t c0 = 0; c0 < a.C && e == cudaSuccess; c0 += G) {
        u.c0 = c0;
        u.G = (a.C - c0) < G ? (a.C - c0) : G;
        const unsigned grid = bn_grid(a.batch * u.G * u.nch, num_sms);
        // every statistics kernel is a programmatic dependent: the first
        // group's waits for the stream's earlier work before it touches
        // memory, later groups read other channels and only overlap the
        // previous group's normalize kernel
        e = launch_pdl(bn_stats_kernel<T>, grid, BNS_THREADS, s, true, a, u);
        if (e == cudaSuccess) e = launch_pdl(bn_norm_kernel<T>, grid, BNS_THREADS, s, true, a, u);
    }
    return e;
}

template <typename T>
cudaError_t launch_bn_train_t(const BnArgs &a, int num_sms, cudaStream_t s, int *used) {
    constexpr int V = IO<T>::V;
    const bool aligned = (a.HW % V == 0) && bn_aligned16(a.x) && bn_aligned16(a.y);
    const bool stream_ok = aligned && a.HW / V < kBnMaxPlanePacks;
    if (aligned && a.fault &&
        (a.bn_plan == BN_PLAN_AUTO || a.bn_plan == BN_PLAN_CLUSTER || a.bn_plan == BN_PLAN_NO_STREAM)) {
        bool launched = false;
        const cudaError_t e = launch_bn_cluster<T>(a, s, &launched);
        if (launched) {
            *used = PLAN_TMA;
            return e;
        }
    }
    // automatic choice beyond the cluster plan: planes of one unit take the
    // streaming plan; longer planes the one-pass plan (measured at
    // [64, 64, 112, 112] binary32: 104 us, against 108 us for the scalar
    // plan's two passes over x and 150 us for the streaming plan; at
    // [32, 64, 56, 56] the streaming plan's 18.6 us beats its 33 us)
    const bool one_unit = a.HW / V <= kBnChunkPacks;
    if (((a.bn_plan == BN_PLAN_AUTO || a.bn_plan == BN_PLAN_NO_STREAM) && !one_unit) ||
        a.bn_plan == BN_PLAN_FLOW) {
        bool launched = false;
        const cudaError_t e = launch_bn_flow(a, bn_dtype<T>(), num_sms, s, &launched);
        if (launched || e != cudaSuccess) {
            *used = PLAN_PERSIST;
            return e;
        }
    }
    if (stream_ok && ((a.bn_plan == BN_PLAN_AUTO && one_unit) || a.bn_plan == BN_PLAN_STREAM)) {
        *used = PLAN_CTA;
        return launch_bn_stream<T>(a, num_sms, s);
    }
    *used = PLAN_GENERIC;
    const unsigned grid = bn_grid(a.batch * a.C, num_sms);
    bn_partial_kernel<T><<<grid, BN_THREADS, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bn_apply_kernel<T><<<grid, BN_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bn_cluster_stats(const BnArgs &a, int dtype, cudaStream_t s, bool *launched) {
    *launched = false;
    if (!a.stats_out || !a.fault) return cudaSuccess;
    switch (dtype) {
    case DT_F32:
        if (a.HW % 4 || !bn_aligned16(a.x)) return cudaSuccess;
        return launch_bn_cluster<float>(a, s, launched);
    case DT_F16:
        if (a.HW % 8 || !bn_aligned16(a.x)) return cudaSuccess;
        return launch_bn_cluster<__half>(a, s, launched);
    case DT_BF16:
        if (a.HW % 8 || !bn_aligned16(a.x)) return cudaSuccess;
        return launch_bn_cluster<__nv_bfloat16>(a, s, launched);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bn_unit_stats(const BnArgs &a, int dtype, int num_sms, cudaStream_t s,
                                 BnChunks *u) {
    const int V = dtype == DT_F32 ? 4 : 8;
    *u = bn_chunks(a.HW / V);
    u->c0 = 0;
    u->G = a.C;
    const unsigned grid = bn_grid(a.batch * a.C * u->nch, num_sms);
    // a programmatic dependent: one group (c0 = 0), so the kernel waits for
    // the stream's previous kernel before it touches memory
    switch (dtype) {
    case DT_F32: return launch_pdl(bn_stats_kernel<float>, grid, BNS_THREADS, s, true, a, *u);
    case DT_F16: return launch_pdl(bn_stats_kernel<__half>, grid, BNS_THREADS, s, true, a, *u);
    case DT_BF16: return launch_pdl(bn_stats_kernel<__nv_bfloat16>, grid, BNS_THREADS, s, true, a, *u);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bn_plane_stats(const BnArgs &a, int dtype, int num_sms, cudaStream_t s) {
    const unsigned grid = bn_grid(a.batch * a.C, num_sms);
    switch (dtype) {
    case DT_F32: bn_partial_kernel<float><<<grid, BN_THREADS, 0, s>>>(a); break;
    case DT_F16: bn_partial_kernel<__half><<<grid, BN_THREADS, 0, s>>>(a); break;
    case DT_BF16: bn_partial_kernel<__nv_bfloat16><<<grid, BN_THREADS, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_bn_train(const BnArgs &a, int dtype, int num_sms, cudaStream_t s, int *used) {
    switch (dtype) {
    case DT_F32: return launch_bn_train_t<float>(a, num_sms, s, used);
    case DT_F16: return launch_bn_train_t<__half>(a, num_sms, s, used);
    case DT_BF16: return launch_bn_train_t<__nv_bfloat16>(a, num_sms, s, used);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nrm

// ---------------------------------------------------------------------------
// The fixed partials array of bn_fwd_train_noalloc (entry point in api.cpp):
// the same plans as bn_fwd_train; the plans that keep partial statistics in
// global memory (streaming, scalar and one-pass) keep them here instead of
// in a workspace the caller allocates.  It is for callers that cannot
// allocate device memory when they call -- for example a runtime that
// reserves its whole device memory budget at start-up and forbids later
// allocations, or a component that is handed device pointers by another part
// of the program and has no allocator of its own.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it (kBnFixedPlanes float2 = 512 KB) until the process exits.
// Its name in host code is only a host-side stand-in, so the device address
// is taken with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on that device.  All calls on a device
// share the array: calls that overlap on the GPU (different streams without
// ordering) race on it.  Every partial a call reads it first writes in the
// same call, and the one-pass plan's reset kernel clears its control words,
// so nothing needs clearing between calls.
// ---------------------------------------------------------------------------
namespace {

__device__ __align__(256) float2 g_bn_fixed_partials[nrm::kBnFixedPlanes];

constexpr int kMaxDevices = 64;
void *g_bn_fixed_ptr[kMaxDevices];
std::once_flag g_bn_fixed_once[kMaxDevices];

}  // namespace

int nrm::bn_fixed_workspace(void **ws, size_t *bytes) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    std::call_once(g_bn_fixed_once[dev], [dev]() {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bn_fixed_partials) == cudaSuccess)
            g_bn_fixed_ptr[dev] = p;
        else
            cudaGetLastError();
    });
    if (!g_bn_fixed_ptr[dev]) return NRM_ERR_DEVICE;
    *ws = g_bn_fixed_ptr[dev];
    *bytes = sizeof(g_bn_fixed_partials);
    return NRM_OK;
}
