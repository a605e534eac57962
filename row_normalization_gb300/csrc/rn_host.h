// rn_host.h -- host-side helpers shared by the entry points: a per-device
// cache of the properties the schedules depend on, alignment checks, and the
// format-independent row-norm call that the C entry points hand to the
// translation unit of each element format.
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

// One row-normalization call, independent of the element format.
enum RowOp { ROW_RMS = 0, ROW_L2 = 1, ROW_ADD_RMS = 2, ROW_LN = 3 };

struct RowCall {
    int op;                // RowOp
    const uint16_t *x;     // [M, N]
    const uint16_t *r;     // residual [M, N] (ROW_ADD_RMS)
    const uint16_t *w;     // weight [N] (all but ROW_L2)
    const uint16_t *b;     // bias [N] or null (ROW_LN)
    float eps;
    int64_t M, N;
    uint16_t *h;           // x + r out [M, N] (ROW_ADD_RMS)
    uint16_t *y;           // [M, N]
    int schedule;
    uint64_t timeout_ns;
    int debug_flags;
    rn_stream_t stream;
    void *workspace;       // RN_WORKSPACE_BYTES of zeroed device memory, or null
};

// Row kernels instantiated per element format (rows_bf16.cu, rows_f16.cu).
int rows_run_bf16(const RowCall &c);
int rows_run_f16(const RowCall &c);
int rows_status_bf16(unsigned int *out, int clear);
int rows_status_f16(unsigned int *out, int clear);
int rows_select_schedule(int op, int64_t M, int64_t N, bool ws = false);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


}  // namespace rn
