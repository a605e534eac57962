// rows_bf16.cu -- the row-normalization kernels instantiated for bf16, and
// rmsnorm_fwd_noalloc, the RMSNorm entry point whose scratch is a fixed
// array of this library instead of a buffer the caller allocates.
#include <mutex>

#include "row_kernels.cuh"

namespace rn {

int rows_run_bf16(const RowCall &c) { return rows_run<Bf16>(c); }

int rows_status_bf16(unsigned int *out, int clear) { return rows_status_word(out, clear); }

int rows_select_schedule(int op, int64_t M, int64_t N, bool ws) { return rows_select(op, M, N, ws); }

// ---- scratch for rmsnorm_fwd_noalloc ----------------------------------------
// The dynamic unit order of the row ring keeps two counters in device memory
// (rmsnorm_fwd_ws takes them from the caller's workspace).  For callers that
// cannot allocate device memory, this array holds them instead: every device
// that loads the library carries its own copy of it until the process exits.
static_assert(RN_NOALLOC_SCRATCH_BYTES >= RN_WORKSPACE_BYTES, "scratch smaller than a workspace");
static __device__ __align__(256) unsigned char g_noalloc_scratch[RN_NOALLOC_SCRATCH_BYTES];

// The array's device address on the current device.  On the host the name
// g_noalloc_scratch stands for a host-side shadow, not the device memory, so
// the address is asked of the runtime once per device (with that device
// current) and kept.
static int noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    const int dev = current_device_index();
    if (dev < 0 || dev >= kMaxDevices) return RN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return RN_ERR_DEVICE;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return RN_OK;
}

}  // namespace rn

extern "C" int rmsnorm_fwd_noalloc(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M,
                                   int64_t N, rn_bf16 *y, rn_stream_t stream) {
    // The arguments are checked before anything is enqueued, with the limits
    // of rmsnorm_fwd.  The scratch needed is the same few bytes whatever M
    // and N are, so no size is refused for lack of scratch.
    const int rc = rn::check_rows(M, N);
    if (rc != RN_OK) return rc;
    if (M == 0) return RN_OK;
    if (!x || !w || !y) return RN_ERR_NULL;
    if (!rn::aligned16(x) || !rn::aligned16(w) || !rn::aligned16(y)) return RN_ERR_ALIGN;
    void *scratch = nullptr;
    const int src = rn::noalloc_scratch(&scratch);
    if (src != RN_OK) return src;
    // The counters must start at zero.  A completed launch leaves them so,
    // but calls that overlapped on the GPU (which race on the one array)
    // could leave them otherwise; clearing them here, in stream order,
    // confines such a race to the calls that overlapped.
    if (cudaMemsetAsync(scratch, 0, RN_WORKSPACE_BYTES, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return RN_ERR_LAUNCH;
    }
    const rn::RowCall c{rn::ROW_RMS, reinterpret_cast<const uint16_t *>(x), nullptr,
                        reinterpret_cast<const uint16_t *>(w), nullptr, eps, M, N, nullptr,
                        reinterpret_cast<uint16_t *>(y), RN_SCHED_AUTO, 0, 0, stream, scratch};
    return rn::rows_run_bf16(c);
}
