/*
 * row_norm.h -- C ABI of the GB300 (sm_103a) row-normalization library
 * (bf16, and IEEE fp16 for the row norms).
 *
 * Operations
 *   rmsnorm_fwd       y = x * 1/sqrt(mean(x^2) + eps) * w, row by row.
 *                     "[Inductor] Codegen Gluon", section 3.1 (MVP: RMSNorm
 *                     with TMA-cached reused input): x feeds both the x*x
 *                     reduction and the x * rstd * weight pass, and is read
 *                     from HBM once.
 *   qk_norm_rope_fwd  per-head RMSNorm of the query and key heads of a packed
 *                     QKV tensor, followed by neox rotary embedding, in place.
 *                     "[pretuned] Optimize fused_qk_norm_rope on B200",
 *                     section "Summary": load each head's rotary halves once,
 *                     reduce over the whole head in registers, apply the Q/K
 *                     weight and the rotation, store each half once; partial
 *                     rotary still normalises the non-rotary tail.
 *   rope_cos_sin_table  builds the cos/sin table the rotary step reads
 *                     (fp32 entries; rope_cos_sin_table_bf16 for bf16 ones,
 *                     which qk_norm_rope_fwd_ex_bf16_table reads).
 *   l2norm_fwd        y = x / max(||x||_2, eps), row by row: one reduction, a
 *                     scale by the inverse norm ("[Inductor] Codegen Gluon",
 *                     section 3.2).
 *   layernorm_fwd     y = (x - mean) / sqrt(var + eps) * w + b, row by row
 *                     (biased variance), the same single HBM pass:
 *                     "TorchInductor: from ATen IR to Triton kernel", section
 *                     14.12.2, and "[Inductor] Codegen Gluon", section 3.2.
 *   add_rmsnorm_fwd   h = x + residual (written out) and y = rmsnorm(h), one
 *                     kernel: the norm / residual-add chain fused ("TorchInductor:
 *                     from ATen IR to Triton kernel", sections 14.3 and 14.27).
 *
 * Conventions shared by every entry point
 *   - bf16 tensors are passed as pointers to their raw 16-bit patterns
 *     (rn_bf16); fp32 and int64 tensors as float* and int64_t*.
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc'd or managed) on
 *     the current CUDA device, 16-byte aligned, densely packed row-major.
 *   - The caller owns every buffer (the *_ws forms also take a small
 *     caller-owned workspace).  The library allocates no device memory,
 *     never synchronises, and enqueues its kernels on `stream` (NULL = the
 *     legacy default stream).  Results are ready when the stream reaches
 *     that point.  The calls can be captured into a CUDA graph.
 *   - Kernels launch with programmatic dependent launch: a kernel may be
 *     scheduled while the previous launch on the stream is finishing, but it
 *     waits for that launch to complete (and its writes to be visible)
 *     before it reads or writes any tensor, so stream order holds exactly
 *     as for ordinary launches.
 *   - Every function returns RN_OK (0) or a negative RN_ERR_* code.  Argument
 *     errors are detected on the host before anything is launched; nothing is
 *     written in that case.  RN_ERR_LAUNCH reports a failed launch.
 *   - Zero rows (M == 0 or T == 0) is a no-op that returns RN_OK.
 *   - Arithmetic: bf16 inputs are widened to fp32 at the point of use, all
 *     sums and products run in fp32, and each output is rounded once to
 *     bf16 (round to nearest even).
 *   - Row statistics are fp32 sums: a bf16 row whose sum of squares passes
 *     the fp32 range (about 3.4e38; values near 2^63 / sqrt(N) and above)
 *     gets a zero scale, and so zero outputs.
 *   - The row norms also take IEEE fp16 tensors (rn_f16; the *_f16 entry
 *     points and row_norm_fwd_ex): the same fp32 arithmetic, one rounding
 *     to fp16 at the store (overflow to infinity, subnormals kept).
 *     "[Inductor] Codegen Gluon", section 3.2, widens the eligible inputs
 *     of the fused norm to fp16.
 */
#ifndef ROW_NORM_H
#define ROW_NORM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raw bf16 bit pattern (sign, 8-bit exponent, 7-bit mantissa). */
typedef uint16_t rn_bf16;

/* Raw IEEE binary16 bit pattern (sign, 5-bit exponent, 10-bit mantissa). */
typedef uint16_t rn_f16;

/* ABI-identical to cudaStream_t / CUstream. */
typedef struct CUstream_st *rn_stream_t;

enum {
    RN_OK = 0,
    RN_ERR_NULL = -1,     /* a required pointer is NULL                        */
    RN_ERR_ALIGN = -2,    /* a tensor pointer is not 16-byte aligned           */
    RN_ERR_SHAPE = -3,    /* a size is negative, unsupported or inconsistent   */
    RN_ERR_LAUNCH = -4,   /* the CUDA launch failed (cudaGetLastError)         */
    RN_ERR_DEVICE = -5,   /* no usable CUDA device / device query failed       */
    RN_ERR_ARG = -6       /* another invalid argument (unknown option value)   */
};

/* Bits of the per-device status word that kernels raise instead of trapping. */
enum {
    RN_STATUS_WAIT_TIMEOUT = 1u,  /* a pipeline wait ran out; that launch's
                                     output is incomplete                     */
    RN_STATUS_BAD_POSITION = 2u   /* qk_norm_rope_fwd_checked met a position
                                     outside [0, max_pos)                     */
};

/* Static description of a code.  Never NULL. */
const char *rn_error_string(int code);

/* Library version as 10000*major + 100*minor + patch. */
int rn_version(void);

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                    */
/* ------------------------------------------------------------------------ */

/* y[r, :] = bf16( x[r, :] * 1/sqrt(sum_j x[r, j]^2 / N + eps) * w[:] )
 *
 *   x    [M, N] bf16, row-major, read once.
 *   w    [N] bf16.
 *   eps  added to the mean of squares inside the square root.
 *   y    [M, N] bf16, written once.  Must not overlap x or w.
 *   Requirements: M >= 0; 8 <= N <= 65536 and N % 8 == 0 (rows start on
 *   16-byte boundaries); x, w, y 16-byte aligned.
 * The schedule (warp per row, CTA per row, or a persistent CTA per SM that
 * streams rows through a shared-memory ring with bulk async copies) is
 * chosen from (M, N) and the SM count.  Errors: RN_ERR_NULL, RN_ERR_ALIGN,
 * RN_ERR_SHAPE, RN_ERR_DEVICE, RN_ERR_LAUNCH. */
int rmsnorm_fwd(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M,
                int64_t N, rn_bf16 *y, rn_stream_t stream);

/* Schedules that rmsnorm_fwd_sched can force (for tests and measurement). */
enum {
    RN_SCHED_AUTO = 0,
    RN_SCHED_WARP_ROW = 1,    /* one warp per row, row in registers (N <= 2048;
                                 RMSNorm and L2Norm up to 4096)                    */
    RN_SCHED_CTA_ROW = 2,     /* one CTA per row, row in registers               */
    RN_SCHED_PERSIST_BULK = 3 /* persistent CTAs, bulk-copy shared-memory ring
                                 (N a power of two, 1024 <= N <= 32768)          */
};

/* rmsnorm_fwd with an explicit schedule.  `schedule` is one of RN_SCHED_*;
 * a schedule that cannot serve (M, N) returns RN_ERR_SHAPE.
 * `wait_timeout_ns` bounds every pipeline wait of the persistent schedule
 * (0 = the default of 2 s); when one runs out, the kernel raises
 * RN_STATUS_WAIT_TIMEOUT in the status word, drains its own copies and
 * returns.  `debug_flags` is 0 in normal use.  Tests and tuning set:
 *   bit 0      the persistent schedule never issues its copies, so its
 *              waits run out (exercises the timeout path);
 *   bits 4-7   persistent schedule: CTAs per SM (0 = the tuned value),
 *              lowered to what the SM's shared memory (at two stages a
 *              CTA) and registers hold at once;
 *   bits 8-12  persistent schedule: ring stages, capped by shared memory
 *              (0 = the tuned value).
 * Setting bits 4-12 also keeps LayerNorm at generic widths on its one-CTA
 * layout (its multi-CTA layouts are chosen only when both are 0). */
int rmsnorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *w, float eps,
                      int64_t M, int64_t N, rn_bf16 *y, int schedule,
                      uint64_t wait_timeout_ns, int debug_flags,
                      rn_stream_t stream);

/* The schedule (RN_SCHED_*) that rmsnorm_fwd launches for (M, N) on the
 * current device; RN_ERR_SHAPE / RN_ERR_DEVICE as rmsnorm_fwd would return.
 * Host-only query: launches nothing. */
int rmsnorm_select_schedule(int64_t M, int64_t N);

/* L2Norm, one HBM pass: y[r, :] = bf16( x[r, :] / max(||x[r, :]||_2, eps) ).
 * No weight.  Requirements, errors and schedules as rmsnorm_fwd (the same
 * kernels run it with a unit weight and the L2 scale). */
int l2norm_fwd(const rn_bf16 *x, float eps, int64_t M, int64_t N, rn_bf16 *y,
               rn_stream_t stream);

/* l2norm_fwd with an explicit schedule, wait limit and test flags, as
 * rmsnorm_fwd_sched. */
int l2norm_fwd_sched(const rn_bf16 *x, float eps, int64_t M, int64_t N, rn_bf16 *y,
                     int schedule, uint64_t wait_timeout_ns, int debug_flags,
                     rn_stream_t stream);

/* LayerNorm, one HBM pass:
 *   mean_r = sum_j x[r, j] / N,  var_r = sum_j (x[r, j] - mean_r)^2 / N
 *   y[r, :] = bf16( (x[r, :] - mean_r) * 1/sqrt(var_r + eps) * w[:] + b[:] )
 * The row stays in registers for two exact passes (mean, then the centred
 * sum of squares), so the variance does not suffer from E[x^2] - mean^2
 * cancellation.  b may be NULL (no bias).  Requirements and errors as
 * rmsnorm_fwd (b, when given, 16-byte aligned).  The persistent schedule
 * serves power-of-two N from 1024 to 16384; wider rows use a row schedule. */
int layernorm_fwd(const rn_bf16 *x, const rn_bf16 *w, const rn_bf16 *b, float eps,
                  int64_t M, int64_t N, rn_bf16 *y, rn_stream_t stream);

/* layernorm_fwd with an explicit schedule, wait limit and test flags, as
 * rmsnorm_fwd_sched. */
int layernorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *w, const rn_bf16 *b,
                        float eps, int64_t M, int64_t N, rn_bf16 *y, int schedule,
                        uint64_t wait_timeout_ns, int debug_flags,
                        rn_stream_t stream);

/* The schedule (RN_SCHED_*) layernorm_fwd launches for (M, N) on the current
 * device.  Host-only query: launches nothing. */
int layernorm_select_schedule(int64_t M, int64_t N);

/* Fused residual add + RMSNorm, one pass:
 *   h[r, j] = bf16(x[r, j] + residual[r, j])   (the exact sum rounded once)
 *   y[r, :] = bf16( h[r, :] * 1/sqrt(sum_j h[r, j]^2 / N + eps) * w[:] )
 * y is computed from the rounded h, so the result is exactly that of the two
 * unfused operations; fusing saves the HBM round trip of h.
 *   x, residual  [M, N] bf16, each read once.
 *   h_out        [M, N] bf16 output; may be `residual` itself (in-place
 *                residual update) or `x`.
 *   y            [M, N] bf16 output; may be `x` itself.  Must differ from h_out.
 * Outputs may equal an input pointer exactly but must not partially overlap
 * one.  Requirements and errors as rmsnorm_fwd; h_out == y gives RN_ERR_ARG.
 * The persistent schedule streams x and residual rows through its ring
 * (N a power of two, 1024 <= N <= 16384); 32768-wide rows use a row schedule. */
int add_rmsnorm_fwd(const rn_bf16 *x, const rn_bf16 *residual, const rn_bf16 *w,
                    float eps, int64_t M, int64_t N, rn_bf16 *h_out, rn_bf16 *y,
                    rn_stream_t stream);

/* The schedule (RN_SCHED_*) add_rmsnorm_fwd launches for (M, N) on the
 * current device.  Host-only query: launches nothing. */
int add_rmsnorm_select_schedule(int64_t M, int64_t N);

/* add_rmsnorm_fwd with an explicit schedule, wait limit and test flags, as
 * rmsnorm_fwd_sched. */
int add_rmsnorm_fwd_sched(const rn_bf16 *x, const rn_bf16 *residual,
                          const rn_bf16 *w, float eps, int64_t M, int64_t N,
                          rn_bf16 *h_out, rn_bf16 *y, int schedule,
                          uint64_t wait_timeout_ns, int debug_flags,
                          rn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* fp16 row norms, and one entry point for every row norm and format          */
/* ------------------------------------------------------------------------ */

/* Element formats and operations of row_norm_fwd_ex. */
enum { RN_DTYPE_BF16 = 0, RN_DTYPE_F16 = 1 };
enum {
    RN_OP_RMSNORM = 0,      /* rmsnorm_fwd:     x, w            -> y      */
    RN_OP_L2NORM = 1,       /* l2norm_fwd:      x               -> y      */
    RN_OP_ADD_RMSNORM = 2,  /* add_rmsnorm_fwd: x, residual, w  -> h, y   */
    RN_OP_LAYERNORM = 3     /* layernorm_fwd:   x, w, b (or NULL) -> y    */
};

/* The four row norms on fp16 tensors: the same contracts, sizes, checks and
 * errors as their bf16 namesakes above, every tensor rn_f16. */
int rmsnorm_fwd_f16(const rn_f16 *x, const rn_f16 *w, float eps, int64_t M,
                    int64_t N, rn_f16 *y, rn_stream_t stream);
int l2norm_fwd_f16(const rn_f16 *x, float eps, int64_t M, int64_t N, rn_f16 *y,
                   rn_stream_t stream);
int add_rmsnorm_fwd_f16(const rn_f16 *x, const rn_f16 *residual, const rn_f16 *w,
                        float eps, int64_t M, int64_t N, rn_f16 *h_out, rn_f16 *y,
                        rn_stream_t stream);
int layernorm_fwd_f16(const rn_f16 *x, const rn_f16 *w, const rn_f16 *b,
                      float eps, int64_t M, int64_t N, rn_f16 *y,
                      rn_stream_t stream);

/* Any row norm (op = RN_OP_*) in either format (dtype = RN_DTYPE_*), with an
 * explicit schedule, wait limit and test flags as rmsnorm_fwd_sched.  Every
 * tensor is a DEVICE pointer to 16-bit patterns of `dtype`; the pointers an
 * op does not use (residual and h_out outside RN_OP_ADD_RMSNORM, w for
 * RN_OP_L2NORM, b outside RN_OP_LAYERNORM) are ignored and may be NULL.
 * Errors as the op's own entry point; an unknown op or dtype is RN_ERR_ARG. */
int row_norm_fwd_ex(int op, int dtype, const void *x, const void *residual,
                    const void *w, const void *b, float eps, int64_t M, int64_t N,
                    void *h_out, void *y, int schedule, uint64_t wait_timeout_ns,
                    int debug_flags, rn_stream_t stream);

/* The schedule (RN_SCHED_*) row_norm_fwd_ex picks under RN_SCHED_AUTO for op
 * and (M, N) on the current device; the same for both formats. */
int row_norm_select_schedule(int op, int64_t M, int64_t N);

/* The same for the workspace forms (rmsnorm_fwd_ws, row_norm_fwd_ws under
 * RN_SCHED_AUTO).  With a workspace the persistent ring can take its units in
 * the dynamic order, and RMSNorm 4096 wide then stays on the ring at every
 * row count, where the plain forms take one warp per row from 128 rows an SM.
 * Host-only query: launches nothing. */
int row_norm_select_schedule_ws(int op, int64_t M, int64_t N);

/* ------------------------------------------------------------------------ */
/* Fused Q/K RMSNorm + neox RoPE                                              */
/* ------------------------------------------------------------------------ */

/* In place on qkv [T, (Hq + 2*Hkv) * D] bf16: token t holds Hq query heads,
 * then Hkv key heads, then Hkv value heads, D contiguous elements each.
 * For every query head (weight wq) and key head (weight wk):
 *   n_j = x_j * 1/sqrt(sum_k x_k^2 / D + eps) * w_j      (all D elements)
 *   for i < r/2 (r = rotary_dim), c = cos_sin[pos, i], s = cos_sin[pos, r/2 + i]:
 *     o_i = n_i*c - n_{i+r/2}*s,   o_{i+r/2} = n_{i+r/2}*c + n_i*s
 *   o_j = n_j for r <= j < D
 * and o is stored back, rounded once to bf16.  Value heads are neither read
 * nor written.
 *
 *   wq, wk     [D] bf16.
 *   cos_sin    [max_pos, r] fp32, row p = [cos(p f_0..) | sin(p f_0..)]
 *              (see rope_cos_sin_table).
 *   positions  [T] int64; every entry must lie in [0, max_pos) of the table
 *              the caller passes: this entry point does not check them (a
 *              position outside the table reads outside cos_sin).  Use
 *              qk_norm_rope_fwd_checked for untrusted positions.
 *   Requirements: T >= 0, Hq >= 0, Hkv >= 0; D in {64, 128, 256};
 *   rotary_dim in {D, D/2, D/4}; T * (Hq + Hkv) < 2^31; qkv, wq, wk and
 *   cos_sin 16-byte aligned, positions 8-byte aligned.
 * The schedule (1, 2 or 4 heads per warp; persistent grid for large T) is
 * chosen from T.  Errors: RN_ERR_NULL, RN_ERR_ALIGN, RN_ERR_SHAPE,
 * RN_ERR_DEVICE, RN_ERR_LAUNCH. */
int qk_norm_rope_fwd(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                     const float *cos_sin, const int64_t *positions, int64_t T,
                     int Hq, int Hkv, int D, int rotary_dim, float eps,
                     rn_stream_t stream);

/* As qk_norm_rope_fwd, but every position is checked against max_pos: the
 * heads of a token whose position lies outside [0, max_pos) are left
 * untouched and RN_STATUS_BAD_POSITION is OR-ed into *d_err_flag (a device
 * int the caller owns and clears).  max_pos >= 1. */
int qk_norm_rope_fwd_checked(rn_bf16 *qkv, const rn_bf16 *wq,
                             const rn_bf16 *wk, const float *cos_sin,
                             const int64_t *positions, int64_t T, int Hq,
                             int Hkv, int D, int rotary_dim, float eps,
                             int64_t max_pos, int *d_err_flag,
                             rn_stream_t stream);

/* Schedules that qk_norm_rope_fwd_sched can force. */
enum {
    RN_QK_AUTO = 0,
    RN_QK_HEAD_PER_WARP = 1,   /* 32 lanes per head                      */
    RN_QK_TWO_HEADS = 2,       /* 16 lanes per head                      */
    RN_QK_FOUR_HEADS = 4,      /* 8 lanes per head                       */
    RN_QK_PERSISTENT = 8,      /* 8 lanes per head, persistent grid       */
    RN_QK_BULK = 16,           /* persistent CTAs stream whole tokens'
                                  query/key regions and cos/sin rows
                                  through a bulk-copy shared-memory ring */
    RN_QK_PAIRS = 32           /* two heads of a token per lane group
                                  sharing one cos/sin slice (4 lanes per
                                  head at D 64, 8 at D 128, 16 at D 256),
                                  grid of two whole waves.  At D 128 the
                                  results are bit-identical to RN_QK_BULK
                                  (neox, fp32 table) or RN_QK_FOUR_HEADS
                                  (GPT-J or a bf16 table)                 */
};

/* qk_norm_rope_fwd with an explicit schedule (one of RN_QK_*).
 * `wait_timeout_ns` and `debug_flags` act on RN_QK_BULK as on
 * rmsnorm_fwd_sched's persistent schedule (bit 0: never issue the copies;
 * bits 8-12: ring stages, 2 or more; bits 16-21: tokens per stage, 1-32;
 * a shared-memory overflow is RN_ERR_SHAPE); 0 and 0 in normal use. */
int qk_norm_rope_fwd_sched(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                           const float *cos_sin, const int64_t *positions,
                           int64_t T, int Hq, int Hkv, int D, int rotary_dim,
                           float eps, int schedule, uint64_t wait_timeout_ns,
                           int debug_flags, rn_stream_t stream);

/* Rotary pairing styles for qk_norm_rope_fwd_ex. */
enum {
    RN_ROPE_NEOX = 0,  /* pairs (i, i + r/2): the half-split layout (default)   */
    RN_ROPE_GPTJ = 1   /* pairs (2i, 2i + 1): interleaved neighbours; the same
                          table row, c = cos_sin[pos, i], s = cos_sin[pos, r/2+i],
                          rotates pair i: o_{2i} = n_{2i} c - n_{2i+1} s,
                          o_{2i+1} = n_{2i+1} c + n_{2i} s                      */
};

/* The general form of the fused Q/K norm + RoPE: every other qk_norm_rope_fwd*
 * entry point is this one with some arguments fixed.
 *   rope_style   RN_ROPE_NEOX or RN_ROPE_GPTJ (else RN_ERR_ARG).
 *   max_pos      0: positions trusted (as qk_norm_rope_fwd); > 0: checked as
 *                qk_norm_rope_fwd_checked, flagging into *d_err_flag.
 *   schedule, wait_timeout_ns, debug_flags: as qk_norm_rope_fwd_sched. */
int qk_norm_rope_fwd_ex(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                        const float *cos_sin, const int64_t *positions, int64_t T,
                        int Hq, int Hkv, int D, int rotary_dim, float eps,
                        int rope_style, int64_t max_pos, int *d_err_flag,
                        int schedule, uint64_t wait_timeout_ns, int debug_flags,
                        rn_stream_t stream);

/* qk_norm_rope_fwd_ex with a bf16 table: cos_sin [max_pos, r] holds bf16
 * entries (the same layout; see rope_cos_sin_table_bf16), which the rotation
 * uses widened exactly to fp32.  Every other argument, requirement and error
 * is that of qk_norm_rope_fwd_ex; cos_sin is 16-byte aligned.  The table's
 * bytes per token halve (r * 2 instead of r * 4). */
int qk_norm_rope_fwd_ex_bf16_table(rn_bf16 *qkv, const rn_bf16 *wq,
                                   const rn_bf16 *wk, const rn_bf16 *cos_sin,
                                   const int64_t *positions, int64_t T, int Hq,
                                   int Hkv, int D, int rotary_dim, float eps,
                                   int rope_style, int64_t max_pos,
                                   int *d_err_flag, int schedule,
                                   uint64_t wait_timeout_ns, int debug_flags,
                                   rn_stream_t stream);

/* The schedule (RN_QK_*) that qk_norm_rope_fwd picks for T tokens of heads
 * with D = 128 and rotary_dim = 128 (RN_ERR_SHAPE if T < 0).  Host-only
 * query: launches nothing. */
int qk_norm_rope_select_schedule(int64_t T);

/* The same for any layout: the pick depends on T, D and rotary_dim (measured
 * per layout).  RN_ERR_SHAPE if T < 0 or (D, rotary_dim) is not a layout
 * qk_norm_rope_fwd takes.  When it picks RN_QK_BULK for a token wider than the
 * ring's shared memory, qk_norm_rope_fwd runs RN_QK_PERSISTENT instead.
 * Host-only query: launches nothing. */
int qk_norm_rope_select_schedule_ex(int64_t T, int D, int rotary_dim);

/* cos_sin[p, i] = cos(p * f_i), cos_sin[p, r/2 + i] = sin(p * f_i),
 * f_i = theta^(-2i/r), for p < max_pos, i < r/2 (r = rotary_dim, even, > 0).
 * Computed on the device in fp64 and rounded once to fp32; written to the
 * caller's DEVICE buffer cos_sin [max_pos, r] fp32.  theta > 0. */
int rope_cos_sin_table(double theta, int64_t max_pos, int rotary_dim,
                       float *cos_sin, rn_stream_t stream);

/* rope_cos_sin_table written to a caller-owned HOST buffer: the same table
 * (cos half, then sin half, of p * theta^(-2i/r); angle, pow, cos and sin in
 * fp64, each entry rounded once to fp32), computed on the calling CPU thread
 * with the C library's pow, cos and sin.  Synchronous; launches nothing and
 * needs no GPU.  cos_sin_host [max_pos, r] fp32 in ordinary host memory
 * (pageable or pinned), 4-byte aligned.  The fp64 pow, cos and sin of the
 * host's C library and of the device may differ in the last bit.  An entry of
 * this table and of rope_cos_sin_table then differs by one fp32 step at most,
 * except where cos or sin is close to zero: there the angle's last-bit
 * difference (below 1e-10 for positions up to 2^17) can move a tiny entry by
 * more steps, while the absolute difference stays below 1e-10.  The table is
 * an input of the fused kernel, which uses whatever entries it is given.  Errors: RN_ERR_SHAPE (max_pos < 0,
 * rotary_dim odd or <= 0, theta not > 0), RN_ERR_NULL (cos_sin_host NULL
 * with max_pos > 0), RN_ERR_ALIGN (cos_sin_host not 4-byte aligned).
 * max_pos = 0 writes nothing and returns RN_OK.
 * ("[pretuned] Optimize fused_qk_norm_rope on B200", "Summary": the cos/sin
 * row of each token's position feeds the rotation.) */
int rope_cos_sin_table_host(double theta, int64_t max_pos, int rotary_dim,
                            float *cos_sin_host);

/* rope_cos_sin_table with bf16 entries: the same fp64 angles and trig, each
 * entry rounded once from double to bf16 (ties to even; not through fp32,
 * which would round twice); written to the caller's DEVICE buffer
 * cos_sin [max_pos, r] bf16, 16-byte aligned. */
int rope_cos_sin_table_bf16(double theta, int64_t max_pos, int rotary_dim,
                            rn_bf16 *cos_sin, rn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Workspace forms: dynamic unit order on the persistent rings                */
/* ------------------------------------------------------------------------ */

/* Bytes of device memory one workspace needs. */
#define RN_WORKSPACE_BYTES 256

/* The persistent row schedule (the ring RN_SCHED_PERSIST_BULK: a
 * warp-specialised persistent kernel, "[Inductor] Codegen Gluon", section
 * 3.3) gives each CTA a fixed round-robin share of the units (R rows each)
 * by default.  The SMs of one GPU do not all stream from HBM at the same
 * rate (on a GB300 some SMs finish such a share up to 15% later than the
 * rest), so a launch lasts as long as its slowest SMs.  With a workspace,
 * each CTA takes about 70% of its share in the fixed order and every later
 * unit from a counter in the workspace: CTAs on faster SMs take more units
 * and all finish within about a stage of each other.  Launches of fewer
 * than six units a CTA keep the fixed order, and so does LayerNorm, whose
 * heavier per-row work measured mixed with the dynamic one.  The outputs are bit-identical
 * either way (a row gets the same arithmetic whichever CTA takes it).  (The
 * fused Q/K token ring measured no gain from this order and takes no
 * workspace.)
 *
 * The workspace:
 *   - RN_WORKSPACE_BYTES of DEVICE memory on the current device, 16-byte
 *     aligned (else RN_ERR_ALIGN), owned by the caller;
 *   - zero-filled by the caller before its first use (cudaMemset); every
 *     launch leaves it zero again when it completes, also one whose waits
 *     ran out (RN_STATUS_WAIT_TIMEOUT);
 *   - serves any number of calls that run one after another (the same
 *     stream, or streams ordered by events); calls whose kernels may run at
 *     the same time need separate workspaces;
 *   - NULL selects the fixed order: the call is then exactly the form
 *     without a workspace.
 * Schedules other than the ring never touch it. */

/* rmsnorm_fwd with a workspace; otherwise the same contract and errors. */
int rmsnorm_fwd_ws(const rn_bf16 *x, const rn_bf16 *w, float eps, int64_t M,
                   int64_t N, rn_bf16 *y, void *workspace, rn_stream_t stream);

/* row_norm_fwd_ex (any row norm, either format, explicit schedule, wait
 * limit and test flags) with a workspace. */
int row_norm_fwd_ws(int op, int dtype, const void *x, const void *residual,
                    const void *w, const void *b, float eps, int64_t M, int64_t N,
                    void *h_out, void *y, void *workspace, int schedule,
                    uint64_t wait_timeout_ns, int debug_flags, rn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* RMSNorm without any caller allocation                                      */
/* ------------------------------------------------------------------------ */

/* Bytes of the library's own scratch array behind rmsnorm_fwd_noalloc (one
 * per device that loads the library, held until the process exits). */
#define RN_NOALLOC_SCRATCH_BYTES 256

/* rmsnorm_fwd_ws with the workspace taken from a fixed scratch array of
 * RN_NOALLOC_SCRATCH_BYTES declared inside the library, so that the caller
 * allocates nothing at all.  This is for callers that cannot hand the library
 * a buffer: a plug-in running inside a host framework that owns the device's
 * memory pool and gives the plug-in no way to draw from it, or a serving
 * process that forbids every device allocation after start-up so that its
 * memory use stays fixed and no allocator call (which may synchronise the
 * device) lands on its hot path.  The pages describe no such entry point;
 * it exists for these callers only.
 *   - Same arguments, limits, results and errors as rmsnorm_fwd; the scratch
 *     needed is the same few bytes for every M and N, so no size is refused
 *     for lack of scratch (sizes outside rmsnorm_fwd's limits give
 *     RN_ERR_SHAPE).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  RN_ERR_DEVICE if the lookup fails.
 *   - Each call clears the counters it needs (a cudaMemsetAsync of the
 *     scratch on `stream`) before its kernel.  Calls no allocation routine.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents: calls whose kernels may overlap on the GPU (different
 *     streams, not ordered) race on it and can compute wrong rows.  Order
 *     them, or give each stream rmsnorm_fwd_ws and a workspace of its own. */
int rmsnorm_fwd_noalloc(const rn_bf16 *x, const rn_bf16 *w, float eps,
                        int64_t M, int64_t N, rn_bf16 *y, rn_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status word                                                                */
/* ------------------------------------------------------------------------ */

/* Reads (and, if clear != 0, resets) the current device's status word: an
 * OR of RN_STATUS_* bits raised by kernels since the last reset.
 * Synchronous: waits for the device to finish its queued work. */
int rn_device_status(unsigned int *out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* ROW_NORM_H */
