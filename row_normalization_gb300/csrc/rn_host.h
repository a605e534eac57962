// rn_host.h -- host-side helpers shared by the entry points: argument checks
// and a per-device cache of the properties the schedules depend on.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/row_norm.h"

namespace rn {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory one CTA may opt into
    int cc_major = 0;
    int cc_minor = 0;
};

// Properties of the current device, queried once per device.  Returns
// nullptr when there is no usable device.
inline const DeviceInfo *current_device_info() {
    static DeviceInfo infos[kMaxDevices];
    static std::atomic<int> ready[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    if (ready[dev].load(std::memory_order_acquire)) return &infos[dev];
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    infos[dev] = d;
    ready[dev].store(1, std::memory_order_release);
    return &infos[dev];
}

inline int current_device_index() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

// Reads (and optionally clears) the status word of the QK translation unit.
int qk_status(unsigned int *out, int clear);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? RN_OK : RN_ERR_LAUNCH;
}

}  // namespace rn
