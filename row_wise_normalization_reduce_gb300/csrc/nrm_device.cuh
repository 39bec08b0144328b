// nrm_device.cuh -- device building blocks of the normalization kernels:
// 16-byte vector I/O with binary32 conversion, and the reduction engine
// (warp shuffles, CTA combine through shared memory) for sums and for
// (count, mean, M2) statistics.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nrm {

// ---------------------------------------------------------------------------
// Vector I/O.  A "pack" is 16 bytes: 4 binary32 or 8 half-width values.  The
// fused RMSNorm page (diycv.top, §3.1) packs 4 elements per access; on GB300
// a full 16-byte access per thread is the widest single load/store.
// ---------------------------------------------------------------------------
template <typename T> struct IO;

template <> struct IO<float> {
    static constexpr int V = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float *f) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
};

template <> struct IO<__half> {
    static constexpr int V = 8;
    __device__ __forceinline__ static void unpack(const uint4 &r, float *f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float to_f(__half v) { return __half2float(v); }
    __device__ __forceinline__ static __half from_f(float v) { return __float2half_rn(v); }
};

template <> struct IO<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ __forceinline__ static void unpack(const uint4 &r, float *f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // a bfloat16 is the top half of a binary32: widening is a shift
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Pairwise views of a pack: H = V/2 float2 values, for the packed binary32
// arithmetic of sm_100+ (__fadd2_rn, __fmul2_rn, __ffma2_rn: two IEEE
// round-to-nearest operations per instruction, bit-identical to the scalar
// ones).
template <typename T> struct IO2;

template <> struct IO2<float> {
    static constexpr int H = 2;
    __device__ __forceinline__ static void unpack(const uint4 &r, float2 *f) {
        f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    __device__ __forceinline__ static uint4 pack(const float2 *f) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                          __float_as_uint(f[1].x), __float_as_uint(f[1].y));
    }
};

template <> struct IO2<__half> {
    static constexpr int H = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float2 *f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
    }
    __device__ __forceinline__ static uint4 pack(const float2 *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __float22half2_rn(f[i]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <> struct IO2<__nv_bfloat16> {
    static constexpr int H = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float2 *f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
    __device__ __forceinline__ static uint4 pack(const float2 *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __float22bfloat162_rn(f[i]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Streaming 16-byte load of data read once (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte load of data every CTA re-reads (parameters): keep it cached.
__device__ __forceinline__ uint4 ld_param(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Streaming 16-byte store (evict-first in the caches).
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

// Ask L2 to fetch [p, p + bytes) from HBM (bytes a multiple of 16, p 16-byte
// aligned).  A hint: no register holds the data and nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: the primary grid allows the secondary one to
// start (launch_dependents); the secondary waits until the primary grid has
// completed and its memory operations are visible (wait).  Both are no-ops in
// a kernel launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Reduction engine.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum_down(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    return v;  // complete in lane 0
}

// Partial statistics of a set of values: count, mean, and M2 = sum of squared
// deviations from that mean.
struct Stats {
    float n, mean, m2;
};

// Pairwise combine of two partial statistics (the parallel form of the
// Welford update; LLM-ops page, smarter.xin, "Welford combine" section):
//   n = na + nb, d = mb - ma, mean = ma + d*nb/n, M2 = M2a + M2b + d^2*na*nb/n.
// An empty side (n = 0) leaves the other unchanged.
__device__ __forceinline__ Stats combine(const Stats &a, const Stats &b) {
    const float n = a.n + b.n;
    if (n == 0.f) return a;
    const float fb = b.n / n;
    const float d = b.mean - a.mean;
    Stats r;
    r.n = n;
    r.mean = fmaf(d, fb, a.mean);
    r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
    return r;
}

__device__ __forceinline__ Stats warp_stats_down(Stats s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Stats t;
        t.n = __shfl_down_sync(0xffffffffu, s.n, o);
        t.mean = __shfl_down_sync(0xffffffffu, s.mean, o);
        t.m2 = __shfl_down_sync(0xffffffffu, s.m2, o);
        s = combine(s, t);
    }
    return s;  // complete in lane 0
}

// Broadcast lane 0's value to the whole warp.
__device__ __forceinline__ float warp_bcast0(float v) { return __shfl_sync(0xffffffffu, v, 0); }

// Butterfly sums: every lane ends with the same bits (a + b == b + a exactly in
// IEEE arithmetic, so partners at each level compute identical values).
__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float2 warp_sum_all(float2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

// Butterfly over groups of NW lanes (NW a power of two): every lane ends
// with the sum of its group.
template <int NW>
__device__ __forceinline__ float group_sum_all(float v) {
#pragma unroll
    for (int o = NW / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
template <int NW>
__device__ __forceinline__ float2 group_sum_all(float2 v) {
#pragma unroll
    for (int o = NW / 2; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

// CTA-wide sum returned to every thread, with one __syncthreads: warps reduce
// by butterfly, lane 0 of each warp publishes its partial, then every warp
// reads the NW partials (lane l takes partial l % NW) and finishes with a
// log2(NW)-level butterfly (same data, same order, so every thread gets the
// same bits).  `slot` must not be rewritten until every thread has passed the
// next __syncthreads of the CTA (callers alternate two slots).
template <int NW>
__device__ __forceinline__ float cta_sum_all(float v, float *slot) {
    static_assert(NW >= 1 && NW <= 32 && (NW & (NW - 1)) == 0, "1..32 warps, power of two");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_all(v);
    if (NW == 1) return v;
    if (lane == 0) slot[warp] = v;
    __syncthreads();
    return group_sum_all<NW>(slot[lane & (NW - 1)]);
}
template <int NW>
__device__ __forceinline__ float2 cta_sum_all(float2 v, float2 *slot) {
    static_assert(NW >= 1 && NW <= 32 && (NW & (NW - 1)) == 0, "1..32 warps, power of two");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_all(v);
    if (NW == 1) return v;
    if (lane == 0) slot[warp] = v;
    __syncthreads();
    return group_sum_all<NW>(slot[lane & (NW - 1)]);
}

// Named barrier over `count` threads (a multiple of 32), id 1..15 (id 0 is
// the barrier of __syncthreads).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Sum over a group of NW warps synchronised by named barrier `bar_id`, returned
// to every thread of the group (same bits everywhere, as cta_sum_all).
template <int NW>
__device__ __forceinline__ float group_cta_sum(float v, float *slot, int bar_id) {
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & (NW - 1);
    v = warp_sum_all(v);
    if (NW == 1) return v;
    if (lane == 0) slot[warp] = v;
    named_sync(bar_id, NW * 32);
    return group_sum_all<NW>(slot[lane & (NW - 1)]);
}
template <int NW>
__device__ __forceinline__ float2 group_cta_sum(float2 v, float2 *slot, int bar_id) {
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & (NW - 1);
    v = warp_sum_all(v);
    if (NW == 1) return v;
    if (lane == 0) slot[warp] = v;
    named_sync(bar_id, NW * 32);
    return group_sum_all<NW>(slot[lane & (NW - 1)]);
}

// As group_cta_sum, and also OR `flag` over the group in the same barrier
// (bar.red.or): every thread learns whether any thread of the group raised it.
template <int NW>
__device__ __forceinline__ float group_cta_sum_or(float v, float *slot, int bar_id, bool flag,
                                                  bool &any) {
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & (NW - 1);
    v = warp_sum_all(v);
    if (lane == 0) slot[warp] = v;
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag), "r"(bar_id), "r"(NW * 32)
        : "memory");
    any = r != 0;
    return group_sum_all<NW>(slot[lane & (NW - 1)]);
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (global -> shared) completed on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the asynchronous (copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier shared-memory accesses before later
// asynchronous-proxy writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One try of the phase with the given parity.  The hint lets the hardware
// suspend the thread for up to kWaitHintNs (it resumes as soon as the phase
// completes), so a waiting warp does not spin on the issue slots.
constexpr uint32_t kWaitHintNs = 1000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "n"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, trying at most
// `limit` times (each try suspends for at most kWaitHintNs); false means the
// wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Rank of this CTA in its thread-block cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Loads from CTA `rank`'s shared memory at the address of `p` in this CTA
// (distributed shared memory of the cluster).
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    return remote;
}
__device__ __forceinline__ float ld_dsmem(const float *p, uint32_t rank) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(dsmem_addr(p, rank)) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_dsmem(const float2 *p, uint32_t rank) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"(dsmem_addr(p, rank))
                 : "memory");
    return v;
}

// Cluster barrier in two halves: arrive (release: this thread's earlier
// memory accesses, including reads of peers' shared memory, are done) and
// wait (acquire).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace nrm
