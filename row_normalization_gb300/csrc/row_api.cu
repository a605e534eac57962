// row_api.cu -- the C entry points of the row norms (include/row_norm.h), the
// library's status word and its error strings.  Argument checks and launches
// live with the kernels (row_kernels.cuh); this file only routes each call to
// the translation unit of its element format.
#include "rn_host.h"

namespace {

int run(int op, int dtype, const void *x, const void *r, const void *w, const void *b, float eps,
        int64_t M, int64_t N, void *h, void *y, int schedule, uint64_t timeout_ns,
        int debug_flags, rn_stream_t stream, void *workspace = nullptr) {
    const rn::RowCall c{op,
                        static_cast<const uint16_t *>(x),
                        op == rn::ROW_ADD_RMS ? static_cast<const uint16_t *>(r) : nullptr,
                        op == rn::ROW_L2 ? nullptr : static_cast<const uint16_t *>(w),
                        op == rn::ROW_LN ? static_cast<const uint16_t *>(b) : nullptr,
                        eps,
                        M,
                        N,
                        op == rn::ROW_ADD_RMS ? static_cast<uint16_t *>(h) : nullptr,
                        static_cast<uint16_t *>(y),
                        schedule,
                        timeout_ns,
                        debug_flags,
                        stream,
                        workspace};
    if (dtype == RN_DTYPE_BF16) return rn::rows_run_bf16(c);
    if (dtype == RN_DTYPE_F16) return rn::rows_run_f16(c);
    return RN_ERR_ARG;
}

}  // namespace

extern "C" {

int rmsnorm_fwd(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M, int64_t N, rn_bf16 *y,
                rn_stream_t stream) {
    return run(rn::ROW_RMS, RN_DTYPE_BF16, x, nullptr, w, nullptr, eps, M, N, nullptr, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int rmsnorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M, int64_t N,
                      rn_bf16 *y, int schedule, uint64_t wait_timeout_ns, int debug_flags,
                      rn_stream_t stream) {
    return run(rn::ROW_RMS, RN_DTYPE_BF16, x, nullptr, w, nullptr, eps, M, N, nullptr, y, schedule,
               wait_timeout_ns, debug_flags, stream);
}

int rmsnorm_select_schedule(int64_t M, int64_t N) {
    return rn::rows_select_schedule(rn::ROW_RMS, M, N);
}

int l2norm_fwd(const rn_bf16 *x, float eps, int64_t M, int64_t N, rn_bf16 *y,
               rn_stream_t stream) {
    return run(rn::ROW_L2, RN_DTYPE_BF16, x, nullptr, nullptr, nullptr, eps, M, N, nullptr, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int l2norm_fwd_sched(const rn_bf16 *x, float eps, int64_t M, int64_t N, rn_bf16 *y,
                     int schedule, uint64_t wait_timeout_ns, int debug_flags,
                     rn_stream_t stream) {
    return run(rn::ROW_L2, RN_DTYPE_BF16, x, nullptr, nullptr, nullptr, eps, M, N, nullptr, y,
               schedule, wait_timeout_ns, debug_flags, stream);
}

int layernorm_fwd(const rn_bf16 *x, const rn_bf16 *w, const rn_bf16 *b, float eps, int64_t M,
                  int64_t N, rn_bf16 *y, rn_stream_t stream) {
    return run(rn::ROW_LN, RN_DTYPE_BF16, x, nullptr, w, b, eps, M, N, nullptr, y, RN_SCHED_AUTO,
               0, 0, stream);
}

int layernorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *w, const rn_bf16 *b, float eps,
                        int64_t M, int64_t N, rn_bf16 *y, int schedule, uint64_t wait_timeout_ns,
                        int debug_flags, rn_stream_t stream) {
    return run(rn::ROW_LN, RN_DTYPE_BF16, x, nullptr, w, b, eps, M, N, nullptr, y, schedule,
               wait_timeout_ns, debug_flags, stream);
}

int layernorm_select_schedule(int64_t M, int64_t N) {
    return rn::rows_select_schedule(rn::ROW_LN, M, N);
}

int add_rmsnorm_fwd(const rn_bf16 *x, const rn_bf16 *residual, const rn_bf16 *w, float eps,
                    int64_t M, int64_t N, rn_bf16 *h_out, rn_bf16 *y, rn_stream_t stream) {
    return run(rn::ROW_ADD_RMS, RN_DTYPE_BF16, x, residual, w, nullptr, eps, M, N, h_out, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int add_rmsnorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *residual, const rn_bf16 *w,
                          float eps, int64_t M, int64_t N, rn_bf16 *h_out, rn_bf16 *y,
                          int schedule, uint64_t wait_timeout_ns, int debug_flags,
                          rn_stream_t stream) {
    return run(rn::ROW_ADD_RMS, RN_DTYPE_BF16, x, residual, w, nullptr, eps, M, N, h_out, y,
               schedule, wait_timeout_ns, debug_flags, stream);
}

int add_rmsnorm_select_schedule(int64_t M, int64_t N) {
    return rn::rows_select_schedule(rn::ROW_ADD_RMS, M, N);
}

int rmsnorm_fwd_f16(const rn_f16 *x, const rn_f16 *w, float eps, int64_t M, int64_t N, rn_f16 *y,
                    rn_stream_t stream) {
    return run(rn::ROW_RMS, RN_DTYPE_F16, x, nullptr, w, nullptr, eps, M, N, nullptr, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int l2norm_fwd_f16(const rn_f16 *x, float eps, int64_t M, int64_t N, rn_f16 *y,
                   rn_stream_t stream) {
    return run(rn::ROW_L2, RN_DTYPE_F16, x, nullptr, nullptr, nullptr, eps, M, N, nullptr, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int add_rmsnorm_fwd_f16(const rn_f16 *x, const rn_f16 *residual, const rn_f16 *w, float eps,
                        int64_t M, int64_t N, rn_f16 *h_out, rn_f16 *y, rn_stream_t stream) {
    return run(rn::ROW_ADD_RMS, RN_DTYPE_F16, x, residual, w, nullptr, eps, M, N, h_out, y,
               RN_SCHED_AUTO, 0, 0, stream);
}

int layernorm_fwd_f16(const rn_f16 *x, const rn_f16 *w, const rn_f16 *b, float eps, int64_t M,
                      int64_t N, rn_f16 *y, rn_stream_t stream) {
    return run(rn::ROW_LN, RN_DTYPE_F16, x, nullptr, w, b, eps, M, N, nullptr, y, RN_SCHED_AUTO, 0,
               0, stream);
}

int row_norm_fwd_ex(int op, int dtype, const void *x, const void *residual, const void *w,
                    const void *b, float eps, int64_t M, int64_t N, void *h_out, void *y,
                    int schedule, uint64_t wait_timeout_ns, int debug_flags, rn_stream_t stream) {
    if (op < RN_OP_RMSNORM || op > RN_OP_LAYERNORM) return RN_ERR_ARG;
    return run(op, dtype, x, residual, w, b, eps, M, N, h_out, y, schedule, wait_timeout_ns,
               debug_flags, stream);
}

int rmsnorm_fwd_ws(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M, int64_t N,
                   rn_bf16 *y, void *workspace, rn_stream_t stream) {
    return run(rn::ROW_RMS, RN_DTYPE_BF16, x, nullptr, w, nullptr, eps, M, N, nullptr, y,
               RN_SCHED_AUTO, 0, 0, stream, workspace);
}

int row_norm_fwd_ws(int op, int dtype, const void *x, const void *residual, const void *w,
                    const void *b, float eps, int64_t M, int64_t N, void *h_out, void *y,
                    void *workspace, int schedule, uint64_t wait_timeout_ns, int debug_flags,
                    rn_stream_t stream) {
    if (op < RN_OP_RMSNORM || op > RN_OP_LAYERNORM) return RN_ERR_ARG;
    return run(op, dtype, x, residual, w, b, eps, M, N, h_out, y, schedule, wait_timeout_ns,
               debug_flags, stream, workspace);
}

int row_norm_select_schedule(int op, int64_t M, int64_t N) {
    if (op < RN_OP_RMSNORM || op > RN_OP_LAYERNORM) return RN_ERR_ARG;
    return rn::rows_select_schedule(op, M, N);
}

int row_norm_select_schedule_ws(int op, int64_t M, int64_t N) {
    if (op < RN_OP_RMSNORM || op > RN_OP_LAYERNORM) return RN_ERR_ARG;
    return rn::rows_select_schedule(op, M, N, true);
}

int rn_device_status(unsigned int *out, int clear) {
    if (!out) return RN_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return RN_ERR_DEVICE;
    }
    unsigned int a = 0, b = 0, q = 0;
    int rc = rn::rows_status_bf16(&a, clear);
    if (rc == RN_OK) rc = rn::rows_status_f16(&b, clear);
    if (rc == RN_OK) rc = rn::qk_status(&q, clear);
    if (rc != RN_OK) return rc;
    *out = a | b | q;
    return RN_OK;
}

const char *rn_error_string(int code) {
    switch (code) {
        case RN_OK: return "ok";
        case RN_ERR_NULL: return "a required pointer is NULL";
        case RN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
        case RN_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case RN_ERR_LAUNCH: return "CUDA kernel launch failed";
        case RN_ERR_DEVICE: return "no usable CUDA device";
        case RN_ERR_ARG: return "invalid argument";
    }
    return "unknown status code";
}

int rn_version(void) { return 101; }

}  // extern "C"
