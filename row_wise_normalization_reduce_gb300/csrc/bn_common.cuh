// bn_common.cuh -- pieces shared by the BatchNorm kernels (training forward,
// inference forward, training backward): element and parameter access in the
// storage type, programmatic dependent launch, and the per-channel fold of
// per-plane partials.
#pragma once

#include "nrm_device.cuh"
#include "nrm_internal.h"

namespace nrm {

// Element i of a tensor stored as T, widened to binary32.
template <typename T>
__device__ __forceinline__ float bn_elem(const void *p, int64_t i) {
    return IO<T>::to_f(static_cast<const T *>(p)[i]);
}

// Per-channel parameter in its storage type, or `dflt` when absent.
template <typename T>
__device__ __forceinline__ float bn_param(const void *p, int64_t c, float dflt) {
    return p ? IO<T>::to_f(static_cast<const T *>(p)[c]) : dflt;
}

// Sum of the pair of binary32 halves of a pack-sized accumulator.
__device__ __forceinline__ float hsum(float2 v) { return v.x + v.y; }

__host__ __device__ __forceinline__ bool bn_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Writes save_mean/save_rstd and the running statistics of channel c from
// its shifted mean md (d = x - K), biased variance and rstd.
__device__ __forceinline__ void bn_write_channel_stats(const BnArgs &a, int64_t c, float K,
                                                       float md, float var, float rstd) {
    if (a.save_mean) a.save_mean[c] = K + md;
    if (a.save_rstd) a.save_rstd[c] = rstd;
    const float m = a.momentum;
    if (a.running_mean) a.running_mean[c] = fmaf(1.f - m, a.running_mean[c], m * (K + md));
    if (a.running_var) {
        const float cnt = (float)(a.batch * a.HW);
        const float unbiased = var * (cnt / (float)(a.batch * a.HW - 1));
        a.running_var[c] = fmaf(1.f - m, a.running_var[c], m * unbiased);
    }
}

// One tiled copy of a 4-D box (TMA, cp.async.bulk.tensor) described by the
// tensor map `tmap` (a __grid_constant__ kernel parameter) at coordinates
// (c0, c1, c2, c3), innermost first, into this CTA's shared memory (128-byte
// aligned), counted on `bar` (the whole box's bytes, out-of-range elements
// included, which arrive as zeros).
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

// Division of 32-bit unsigned integers by a run-time constant d (1 <= d <
// 2^31) with a multiply-high, shift and add: the round-up method of
// Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication" (PLDI 1994), section 4.  With l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1, n / d = (mulhi(n, m) + n) >> l for
// every 32-bit n (the sum is formed in 64 bits).
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while (((uint64_t)1 << f.l) < d) ++f.l;
    f.m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << f.l) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f) {
    return (uint32_t)(((uint64_t)__umulhi(n, f.m) + n) >> f.l);
}

// ---------------------------------------------------------------------------
// Work units of the streaming BatchNorm plans.  A unit is a chunk of at most
// kBnChunkPacks 16-byte packs of one (n, c) plane (all chunks of a plane but
// the last have the same size), held in registers by one CTA of BNS_THREADS
// threads x BNS_PACKS packs.  A launch covers the units of one channel group
// [c0, c0 + G); the units of a group are ordered n-major, then channel, then
// chunk.  Per-unit partials sit at ws[c * (batch * nch) + n * nch + k].
// ---------------------------------------------------------------------------
constexpr int BNS_THREADS = 256;
constexpr int BNS_PACKS = 4;
static_assert(BNS_THREADS * BNS_PACKS == kBnChunkPacks, "a CTA holds one unit in registers");
constexpr int64_t kBnMaxPlanePacks = kBnUnitPlaneLimit;  // chunking exact below this

struct BnChunks {
    int64_t c0, G;  // channel group
    int q;          // packs per plane
    int nch;        // chunks per plane
    int cpk;        // packs per chunk (the last chunk may have fewer)
};

inline BnChunks bn_chunks(int64_t packs_per_plane) {
    BnChunks u;
    u.c0 = 0;
    u.G = 0;
    u.q = (int)packs_per_plane;
    u.nch = (int)((packs_per_plane + kBnChunkPacks - 1) / kBnChunkPacks);
    if (u.nch < 1) u.nch = 1;
    u.cpk = (int)((packs_per_plane + u.nch - 1) / u.nch);
    return u;
}

struct BnUnit {
    int64_t n, c;
    int k;    // chunk of the plane
    int off;  // first pack of the chunk within the plane
    int len;  // packs in the chunk
};

__device__ __forceinline__ BnUnit bn_unit(const BnChunks &u, int64_t idx) {
    BnUnit r;
    r.k = (int)(idx % u.nch);
    const int64_t t = idx / u.nch;
    r.c = u.c0 + t % u.G;
    r.n = t / u.G;
    r.off = r.k * u.cpk;
    r.len = min(u.cpk, u.q - r.off);
    return r;
}

// Exact partial statistics of one unit held in registers by a CTA of
// BNS_THREADS threads (pack tid + k * BNS_THREADS in v[k], k < PACKS, valid
// below len):
// a corrected two-pass on d = x - K, returned as (mean of d, M2) with the
// same bits in every thread.  Two CTA-wide sums through s1 and s2, which the
// caller alternates between consecutive units.
template <typename T, int PACKS = BNS_PACKS>
__device__ __forceinline__ float2 bn_unit_partial(const uint4 (&v)[PACKS], int len, float K,
                                                  float *s1, float2 *s2) {
    using io2 = IO2<T>;
    constexpr int H = io2::H;
    constexpr int NW = BNS_THREADS / 32;
    const int tid = threadIdx.x;
    const float cnt = (float)(len * IO<T>::V);
    const float2 nk = f2(-K);
    float2 acc = f2(0.f);
#pragma unroll
    for (int k = 0; k < PACKS; ++k)
        if (tid + k * BNS_THREADS < len) {
            float2 f[H];
            io2::unpack(v[k], f);
#pragma unroll
            for (int h = 0; h < H; ++h) acc = __fadd2_rn(acc, __fadd2_rn(f[h], nk));
        }
    const float tot = cta_sum_all<NW>(hsum(acc), s1);
    const float m0 = tot / cnt;
    const float2 nkm = f2(-m0);
    float2 e1 = f2(0.f), e2 = f2(0.f);
#pragma unroll
    for (int k = 0; k < PACKS; ++k)
        if (tid + k * BNS_THREADS < len) {
            float2 f[H];
            io2::unpack(v[k], f);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float2 e = __fadd2_rn(__fadd2_rn(f[h], nk), nkm);
                e1 = __fadd2_rn(e1, e);
                e2 = __ffma2_rn(e, e, e2);
            }
        }
    const float2 E = cta_sum_all<NW>(make_float2(hsum(e1), hsum(e2)), s2);
    const float cc = E.x / cnt;
    return make_float2(m0 + cc, fmaxf(fmaf(-cnt * cc, cc, E.y), 0.f));
}

// Channels per group so that a group's input bytes stay within `budget`
// (the second stage then re-reads them from L2).
inline int64_t bn_group_channels(int64_t C, int64_t bytes_per_channel, int64_t budget) {
    int64_t g = bytes_per_channel > 0 ? budget / bytes_per_channel : C;
    return g < 1 ? 1 : g > C ? C : g;
}

// Grid of a grid-stride kernel over `units` work items: at most 64 CTAs per SM.
inline unsigned bn_grid(int64_t units, int num_sms) {
    const int64_t cap = (int64_t)num_sms * 64;
    return (unsigned)(units < cap ? units : cap);
}

// Launch with programmatic stream serialization (the kernel may start before
// the previous one on the stream has finished; it orders itself with
// griddepcontrol.wait where it needs to).
template <typename K, typename... Args>
inline cudaError_t launch_pdl(K kernel, unsigned grid, unsigned threads, cudaStream_t s, bool pdl,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// Stage 1 of the streaming plans alone over all channels (synchronized
// BatchNorm): per-unit partials into a.ws, the unit layout in *u.  The
// planes must be 16-byte aligned and a whole number of packs.
cudaError_t launch_bn_unit_stats(const BnArgs &a, int dtype, int num_sms, cudaStream_t s,
                                 BnChunks *u);
cudaError_t launch_bn_bwd_unit_sums(const BnBwdArgs &a, int dtype, int num_sms, cudaStream_t s,
                                    BnChunks *u);

// The one-pass plan (bn_flow.cu) for 16-byte aligned planes of whole packs
// and a workspace of at least bn_flow_ws_bytes: *launched tells whether it
// ran (false: the layout or the workspace does not allow it).
cudaError_t launch_bn_flow(const BnArgs &a, int dtype, int num_sms, cudaStream_t s, bool *launched);

template <typename T> constexpr int bn_dtype();
template <> constexpr int bn_dtype<float>() { return DT_F32; }
template <> constexpr int bn_dtype<__half>() { return DT_F16; }
template <> constexpr int bn_dtype<__nv_bfloat16>() { return DT_BF16; }

// Input bytes per channel group of the streaming BatchNorm plans (api.cpp;
// nrm_set_bn_group_bytes), 0 for a single group.
size_t bn_group_bytes();
inline int64_t bn_group_budget() {
    const size_t b = bn_group_bytes();
    return b == 0 || b > (size_t)INT64_MAX ? INT64_MAX : (int64_t)b;
}

}  // namespace nrm
