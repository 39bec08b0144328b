// fault.cu -- the device fault word.  Kernels with bounded waits set bits of
// it when a wait gives up (they then drain their copies and return instead of
// hanging); the host reads and clears it with nrm_device_fault().
#include <cuda_runtime.h>

#include <mutex>

#include "nrm.h"
#include "nrm_internal.h"

namespace nrm {

namespace {
__device__ unsigned g_fault_word;

constexpr int kMaxDevices = 64;
unsigned *g_fault_ptr[kMaxDevices];
std::once_flag g_fault_once[kMaxDevices];
}  // namespace

// The symbol's host-side name is not a device address: take the device
// address once per device, with that device current.
unsigned *fault_word() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::call_once(g_fault_once[dev], [dev]() {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fault_word) == cudaSuccess)
            g_fault_ptr[dev] = static_cast<unsigned *>(p);
        else
            cudaGetLastError();
    });
    return g_fault_ptr[dev];
}

}  // namespace nrm

extern "C" int nrm_device_fault(unsigned *bits, int clear) {
    unsigned *p = nrm::fault_word();
    if (!p) return NRM_ERR_DEVICE;
    unsigned v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return NRM_ERR_DEVICE;
    }
    if (clear && v) {
        const unsigned zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return NRM_ERR_DEVICE;
        }
    }
    if (bits) *bits = v;
    return NRM_OK;
}
