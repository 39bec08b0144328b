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

// Input bytes per channel group of the streaming BatchNorm plans (api.cpp;
// nrm_set_bn_group_bytes), 0 for a single group.
size_t bn_group_bytes();
inline int64_t bn_group_budget() {
    const size_t b = bn_group_bytes();
    return b == 0 || b > (size_t)INT64_MAX ? INT64_MAX : (int64_t)b;
}

}  // namespace nrm
