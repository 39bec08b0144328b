// bn_common.cuh -- pieces shared by the BatchNorm kernels (training forward,
// inference forward, training backward): element and parameter access in the
// storage type, programmatic dependent launch, and the per-channel fold of
// per-plane partials.
#pragma once

#include "nrm_device.cuh"
#include "nrm_internal.h"

namespace nrm {

// Programmatic dependent launch: the primary grid allows the secondary one to
// start (launch_dependents); the secondary waits until the primary grid has
// completed and its memory operations are visible (wait).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Grid of a grid-stride kernel over `units` work items: at most 64 CTAs per SM.
inline unsigned bn_grid(int64_t units, int num_sms) {
    const int64_t cap = (int64_t)num_sms * 64;
    return (unsigned)(units < cap ? units : cap);
}

}  // namespace nrm
