// row_kernels.cuh -- the row-normalization kernels for sm_103a, written once
// over a 16-bit element format (bf16 or IEEE fp16; the fp32 arithmetic is the
// same for both) and instantiated by one translation unit per format.
//
//   RMSNorm    y[r, :] = round( x[r, :] * 1/sqrt(sum_j x[r, j]^2 / N + eps) * w[:] )
//   L2Norm     y[r, :] = round( x[r, :] / max(||x[r, :]||_2, eps) )
//   add+RMS    h = round(x + res), y = RMSNorm(h)
//   LayerNorm  y[r, :] = round( (x[r, :] - mean) / sqrt(var + eps) * w[:] + b[:] )
//
// "[Inductor] Codegen Gluon", section 3.1: x feeds both the x*x reduction and
// the x * rstd * weight pass.  Every schedule here reads each element of x
// from HBM exactly once, keeps it (16-bit) in registers or shared memory
// between the two passes, widens to fp32 at the point of use, and writes each
// output once with a single rounding.  Section 3.2 of the same page widens
// the eligible inputs to fp16 and to rows that are not a power of two wide.
//
// Schedules:
//   warp_rows        one warp per row, the row in registers (N <= 2048).
//   cta_rows         one CTA per row, the row in registers, one CTA-wide
//                    reduction through shared memory (any N up to 65536).
//   persistent_bulk  one CTA per SM.  A producer warp streams R-row units of
//                    x into an S-stage shared-memory ring with 1D bulk
//                    copies (cp.async.bulk, completion on a per-stage
//                    mbarrier); consumer warps pull each unit into registers
//                    once, release the stage, reduce, and store y.  The
//                    weight stays in registers for the CTA's whole life.
//
// Each including translation unit gets its own status word (g_status) and
// reads it back through rows_status_word().
#pragma once

#include "rn_common.cuh"
#include "rn_host.h"

namespace rn {

static __device__ unsigned int g_status = 0u;

__device__ __forceinline__ void raise_status(unsigned int bits) { atomicOr(&g_status, bits); }

// Sum of squares of the 8 elements in a 16-byte vector, in fp32 (pairwise):
// each square is exact, formed straight from the packed halves.
template <class E>
__device__ __forceinline__ float sumsq8(uint4 v) {
    const float a = E::sq_acc(0.f, v.x);
    const float b = E::sq_acc(0.f, v.y);
    const float c = E::sq_acc(0.f, v.z);
    const float d = E::sq_acc(0.f, v.w);
    return (a + b) + (c + d);
}

// y = round((x * rstd) * w) for 8 packed elements.
template <class E>
__device__ __forceinline__ uint4 scale8(uint4 xv, uint4 wv, float rstd) {
    uint4 o;
    o.x = E::pack(E::lo(xv.x) * rstd * E::lo(wv.x), E::hi(xv.x) * rstd * E::hi(wv.x));
    o.y = E::pack(E::lo(xv.y) * rstd * E::lo(wv.y), E::hi(xv.y) * rstd * E::hi(wv.y));
    o.z = E::pack(E::lo(xv.z) * rstd * E::lo(wv.z), E::hi(xv.z) * rstd * E::hi(wv.z));
    o.w = E::pack(E::lo(xv.w) * rstd * E::lo(wv.w), E::hi(xv.w) * rstd * E::hi(wv.w));
    return o;
}

// h = round(x + r) for 8 packed elements.  Each sum is formed in fp32 and
// rounded once, which gives the correctly rounded exact sum in both formats.
// bf16: the fp32 sum is exact when the exponents are within 16 of each other;
// otherwise the smaller addend is below 2^-16 of the larger, too small to
// reach a rounding midpoint.  fp16: both addends are multiples of 2^-24 below
// 2^16, so the fp32 sum is exact unless the exponents differ by 14 or more,
// and then the smaller addend stays under a quarter of the larger's half-step
// (the fp32 result stays on the larger addend's side of every midpoint).
template <class E>
__device__ __forceinline__ uint4 add8(uint4 a, uint4 b) {
    uint4 o;
    o.x = E::pack(E::lo(a.x) + E::lo(b.x), E::hi(a.x) + E::hi(b.x));
    o.y = E::pack(E::lo(a.y) + E::lo(b.y), E::hi(a.y) + E::hi(b.y));
    o.z = E::pack(E::lo(a.z) + E::lo(b.z), E::hi(a.z) + E::hi(b.z));
    o.w = E::pack(E::lo(a.w) + E::lo(b.w), E::hi(a.w) + E::hi(b.w));
    return o;
}

// LayerNorm pieces: sum of 8, the sum of deviations from `m` with the sum of
// their squares, and y = ((x - m) [+ nc]) * rstd * w (+ b) rounded once.  The
// widening of x is folded into mixed-precision adds and subtracts (pair_sum,
// sub2), which round exactly as widen-then-add does.
template <class E>
__device__ __forceinline__ float sum8(uint4 v) {
    return (E::pair_sum(v.x) + E::pair_sum(v.y)) + (E::pair_sum(v.z) + E::pair_sum(v.w));
}

// Adds the deviations x_k - m of 8 packed elements and their squares to two
// sets of fp32-pair accumulators (words x, y to a; z, w to b): each pair is
// consumed at once (few registers) and the two sets halve the dependent
// chains.  The row's sums are dev_sum(sd) and dev_sum(sq).
struct DevAcc {
    float2 sd_a, sq_a, sd_b, sq_b;
};

__device__ __forceinline__ DevAcc dev_zero() {
    const float2 z = make_float2(0.f, 0.f);
    return {z, z, z, z};
}

template <class E>
__device__ __forceinline__ void dev8(uint4 v, float m, DevAcc &acc) {
    float2 d = E::sub2(v.x, m);
    acc.sd_a = __fadd2_rn(acc.sd_a, d);
    acc.sq_a = __ffma2_rn(d, d, acc.sq_a);
    d = E::sub2(v.z, m);
    acc.sd_b = __fadd2_rn(acc.sd_b, d);
    acc.sq_b = __ffma2_rn(d, d, acc.sq_b);
    d = E::sub2(v.y, m);
    acc.sd_a = __fadd2_rn(acc.sd_a, d);
    acc.sq_a = __ffma2_rn(d, d, acc.sq_a);
    d = E::sub2(v.w, m);
    acc.sd_b = __fadd2_rn(acc.sd_b, d);
    acc.sq_b = __ffma2_rn(d, d, acc.sq_b);
}

// (sum of deviations, sum of squared deviations) held in `acc`.
__device__ __forceinline__ float2 dev_sums(const DevAcc &acc) {
    const float2 d = __fadd2_rn(acc.sd_a, acc.sd_b);
    const float2 q = __fadd2_rn(acc.sq_a, acc.sq_b);
    return make_float2(d.x + d.y, q.x + q.y);
}

// Centring of a row whose mean is large against its spread.  The first
// reduction's fp32 mean m is off by up to |mean| * 2^-24 plus its sum's
// rounding, and that error would move every x - m by the same amount.  A
// second reduction over the deviations d = x - m (exact, or within 2^-24 of
// |d|) gives the correction c = sum(d) / N, which is small against the
// spread, and the variance sum(d^2) / N - c^2 without cancellation.  The
// output then takes (x - m) * rstd - c * rstd as one fused multiply-add in
// place of the product (x - m) * rstd, leaving an error of order 2^-24 of
// |x - mean| * rstd instead of |mean| * rstd.  Rows centred on the first
// reduction's mean pass ncr = +0, which gives the plain product's bits.
struct Centring {
    float rstd;  // 1 / sqrt(var + eps)
    float ncr;   // -c * rstd
};

__device__ __forceinline__ Centring centre(float sum_d, float sum_d2, int N, float eps) {
    const float c = sum_d / static_cast<float>(N);
    const float var = fmaxf(sum_d2 / static_cast<float>(N) - c * c, 0.f);
    const float rstd = __frsqrt_rn(var + eps);
    return {rstd, -c * rstd};
}

// Same, on fp32 pairs (Blackwell FFMA2): per pair one subtract, one fused
// multiply-add by rstd (with the centring correction), one fused
// multiply-add with (w, b).
template <class E>
__device__ __forceinline__ uint32_t ln2w(uint32_t x, uint32_t w, uint32_t b, float m, float2 r,
                                         float2 ncr) {
    const float2 d = __ffma2_rn(E::sub2(x, m), r, ncr);
    const float2 y = __ffma2_rn(d, make_float2(E::lo(w), E::hi(w)), make_float2(E::lo(b), E::hi(b)));
    return E::pack(y.x, y.y);
}

template <class E>
__device__ __forceinline__ uint4 ln8(uint4 xv, uint4 wv, uint4 bv, float m, float rstd,
                                     float ncr) {
    const float2 r = make_float2(rstd, rstd);
    const float2 c = make_float2(ncr, ncr);
    uint4 o;
    o.x = ln2w<E>(xv.x, wv.x, bv.x, m, r, c);
    o.y = ln2w<E>(xv.y, wv.y, bv.y, m, r, c);
    o.z = ln2w<E>(xv.z, wv.z, bv.z, m, r, c);
    o.w = ln2w<E>(xv.w, wv.w, bv.w, m, r, c);
    return o;
}

// ln8 with the weights already widened to fp32 pairs (w[0..3]).
template <class E>
__device__ __forceinline__ uint32_t ln2f(uint32_t x, float2 w, uint32_t b, float m, float2 r,
                                         float2 ncr) {
    const float2 y = __ffma2_rn(__ffma2_rn(E::sub2(x, m), r, ncr), w, make_float2(E::lo(b), E::hi(b)));
    return E::pack(y.x, y.y);
}

template <class E>
__device__ __forceinline__ uint4 ln8w(uint4 xv, const float2 *w, uint4 bv, float m, float rstd,
                                      float ncr) {
    const float2 r = make_float2(rstd, rstd);
    const float2 c = make_float2(ncr, ncr);
    uint4 o;
    o.x = ln2f<E>(xv.x, w[0], bv.x, m, r, c);
    o.y = ln2f<E>(xv.y, w[1], bv.y, m, r, c);
    o.z = ln2f<E>(xv.z, w[2], bv.z, m, r, c);
    o.w = ln2f<E>(xv.w, w[3], bv.w, m, r, c);
    return o;
}

// Bias chunk, or zeros when there is no bias.
__device__ __forceinline__ uint4 bias16(const uint16_t *b, int c) {
    return b ? ld_ro16(b + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float row_rstd(float ss, int N, float eps) {
    return __frsqrt_rn(ss / static_cast<float>(N) + eps);
}

// Per-row scale: RMSNorm's 1/sqrt(ss/N + eps), or with `l2` the L2Norm's
// 1/max(sqrt(ss), eps) (a correctly rounded rsqrt when the norm exceeds eps).
__device__ __forceinline__ float row_scale(float ss, int N, float eps, int l2) {
    if (!l2) return row_rstd(ss, N, eps);
    return sqrtf(ss) > eps ? __frsqrt_rn(ss) : 1.0f / eps;
}

// Weight chunk, or eight ones in the element format when there is no weight.
template <class E>
__device__ __forceinline__ uint4 weight16(const uint16_t *w, int c) {
    return w ? ld_ro16(w + 8 * c) : make_uint4(E::kOne2, E::kOne2, E::kOne2, E::kOne2);
}

// ---------------------------------------------------------------------------
// warp_rows: one warp per row; lane l holds 16-byte chunks l, l+32, ...
// ---------------------------------------------------------------------------
// With ADD, the row is h = round(x + r) (stored to h_out) and y = rmsnorm(h).
// With LN, y = layernorm(x) = (x - mean) * rstd * w + b (b may be null).
template <class E, int VPT, bool ADD, bool LN>
__global__ void __launch_bounds__(256) rms_warp_rows_kernel(const uint16_t *x,
                                                            const uint16_t *__restrict__ w,
                                                            float eps, int64_t M, int N,
                                                            uint16_t *y, const uint16_t *r,
                                                            uint16_t *h_out, const uint16_t *b,
                                                            int l2) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int cpr = N >> 3;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); row < M;
         row += static_cast<int64_t>(gridDim.x) * wpb) {
        const uint16_t *xr = x + row * N;
        uint4 v[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = lane + 32 * i;
            v[i] = (c < cpr) ? ld_stream16(xr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        }
        if constexpr (ADD) {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = lane + 32 * i;
                if (c < cpr) {
                    v[i] = add8<E>(v[i], ld_stream16(r + row * N + 8 * c));
                    st16(h_out + row * N + 8 * c, v[i]);
                }
            }
        }
        uint16_t *yr = y + row * N;
        if constexpr (LN) {
            // the sum and the sum of squares in one pass; the centred second
            // pass only where the mean is large against the spread (the same
            // rule as the persistent schedule; a butterfly sum leaves the
            // same bits in every lane, so the branch is warp-uniform)
            float s1 = 0.f, q1 = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {  // absent chunks are zero
                s1 += sum8<E>(v[i]);
                q1 += sumsq8<E>(v[i]);
            }
            const float mean = warp_sum(s1) / static_cast<float>(N);
            const float var = warp_sum(q1) / static_cast<float>(N) - mean * mean;
            Centring ce{__frsqrt_rn(var + eps), 0.f};
            if (!(var > 0.f && mean * mean <= 4.f * var)) {
                DevAcc acc = dev_zero();
#pragma unroll
                for (int i = 0; i < VPT; ++i)
                    if (lane + 32 * i < cpr) dev8<E>(v[i], mean, acc);
                const float2 ds = dev_sums(acc);
                ce = centre(warp_sum(ds.x), warp_sum(ds.y), N, eps);
            }
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = lane + 32 * i;
                if (c < cpr)
                    st16(yr + 8 * c,
                         ln8<E>(v[i], ld_ro16(w + 8 * c), bias16(b, c), mean, ce.rstd, ce.ncr));
            }
        } else {
            // With up to 4 chunks a lane the weights' loads go out with the
            // row's, ahead of the reduction; with 8 the extra registers cost
            // more occupancy than the early loads gain (2048-wide rows).
            constexpr bool EARLY_W = VPT <= 4 && !ADD;
            uint4 wv[EARLY_W ? VPT : 1];
            if constexpr (EARLY_W) {
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    const int c = lane + 32 * i;
                    if (c < cpr) wv[i] = weight16<E>(w, c);
                }
            }
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) ss += sumsq8<E>(v[i]);
            ss = warp_sum(ss);
            const float rstd = row_scale(ss, N, eps, l2);
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = lane + 32 * i;
                if (c < cpr)
                    st16(yr + 8 * c, scale8<E>(v[i], EARLY_W ? wv[i] : weight16<E>(w, c), rstd));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// cta_rows: one CTA per row; thread t holds chunks t, t+nt, ...
// ---------------------------------------------------------------------------
template <class E, int VPT, int MAXT, bool ADD, bool LN>
__global__ void __launch_bounds__(MAXT) rms_cta_rows_kernel(const uint16_t *x,
                                                            const uint16_t *__restrict__ w,
                                                            float eps, int64_t M, int N,
                                                            uint16_t *y, const uint16_t *r,
                                                            uint16_t *h_out, const uint16_t *b,
                                                            int l2) {
    __shared__ float red[2][32];
    __shared__ float red2[2][32];  // LayerNorm's sums of squares
    __shared__ float red3[2][32];  // LayerNorm's centred squares (large-mean rows)
    __shared__ float red4[2][32];  // and their deviations
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int nw = nt >> 5;
    const int cpr = N >> 3;
    int par = 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, par ^= 1) {
        const uint16_t *xr = x + row * N;
        uint4 v[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int c = tid + nt * i;
            v[i] = (c < cpr) ? ld_stream16(xr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        }
        if constexpr (ADD) {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = tid + nt * i;
                if (c < cpr) {
                    v[i] = add8<E>(v[i], ld_stream16(r + row * N + 8 * c));
                    st16(h_out + row * N + 8 * c, v[i]);
                }
            }
        }
        uint16_t *yr = y + row * N;
        if constexpr (LN) {
            // one CTA reduction of the sum and the sum of squares; a second
            // over the centred squares only where the mean is large against
            // the spread (every thread reads the same partials in the same
            // order, so the branch is uniform)
            float s1 = 0.f, q1 = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {  // absent chunks are zero
                s1 += sum8<E>(v[i]);
                q1 += sumsq8<E>(v[i]);
            }
            s1 = warp_sum(s1);
            q1 = warp_sum(q1);
            if ((tid & 31) == 0) {
                red[par][tid >> 5] = s1;
                red2[par][tid >> 5] = q1;
            }
            __syncthreads();
            float t1 = 0.f, u1 = 0.f;
            for (int k = 0; k < nw; ++k) {
                t1 += red[par][k];
                u1 += red2[par][k];
            }
            const float mean = t1 / static_cast<float>(N);
            const float var = u1 / static_cast<float>(N) - mean * mean;
            Centring ce{__frsqrt_rn(var + eps), 0.f};
            if (!(var > 0.f && mean * mean <= 4.f * var)) {
                DevAcc acc = dev_zero();
#pragma unroll
                for (int i = 0; i < VPT; ++i)
                    if (tid + nt * i < cpr) dev8<E>(v[i], mean, acc);
                const float2 ds = dev_sums(acc);
                const float2 dv = make_float2(warp_sum(ds.x), warp_sum(ds.y));
                if ((tid & 31) == 0) {
                    red3[par][tid >> 5] = dv.y;
                    red4[par][tid >> 5] = dv.x;
                }
                __syncthreads();
                float t2 = 0.f, d2 = 0.f;
                for (int k = 0; k < nw; ++k) {
                    t2 += red3[par][k];
                    d2 += red4[par][k];
                }
                ce = centre(d2, t2, N, eps);
            }
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = tid + nt * i;
                if (c < cpr)
                    st16(yr + 8 * c,
                         ln8<E>(v[i], ld_ro16(w + 8 * c), bias16(b, c), mean, ce.rstd, ce.ncr));
            }
            continue;
        }
        // The weights' loads go out with the row's, ahead of the reduction
        // (at 1024 threads, 64 registers a thread, they are streamed at the
        // end instead).
        uint4 wv[MAXT < 1024 ? VPT : 1];
        if constexpr (MAXT < 1024) {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = tid + nt * i;
                if (c < cpr) wv[i] = weight16<E>(w, c);
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) ss += sumsq8<E>(v[i]);
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[par][tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int k = 0; k < nw; ++k) tot += red[par][k];
        const float rstd = row_scale(tot, N, eps, l2);
        if constexpr (MAXT < 1024) {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = tid + nt * i;
                if (c < cpr) st16(yr + 8 * c, scale8<E>(v[i], wv[i], rstd));
            }
        } else {
            // 64 registers a thread at 1024 threads: stream the weights
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int c = tid + nt * i;
                if (c < cpr) st16(yr + 8 * c, scale8<E>(v[i], weight16<E>(w, c), rstd));
            }
        }
        // red[par] is rewritten two rows later, after the next barrier: safe.
    }
}

// ---------------------------------------------------------------------------
// persistent_bulk
// ---------------------------------------------------------------------------
struct BulkArgs {
    const uint16_t *x;
    const uint16_t *w;
    uint16_t *y;
    const uint16_t *r;  // residual (fused add) or nullptr
    uint16_t *h;        // x + r output (fused add) or nullptr
    const uint16_t *b;  // LayerNorm bias or nullptr
    int l2;             // L2Norm scale instead of RMSNorm's (w may then be null)
    int64_t M;
    int N;
    float eps;
    int stages;
    int debug;
    uint64_t timeout_ns;
    unsigned long long *ws;  // dynamic unit order (two zeroed words), or nullptr: round-robin
};

// Per-warp partial sums of row rr sit at [rr * kRedStride + warp]: the lane
// that finishes row rr reads its row's partials along a run of consecutive
// words, and the R such lanes fall in different banks (stride 33, not 32).
constexpr int kRedStride = 33;

// Shared memory: [stages x (R rows of x [+ R rows of r])][full mbarriers]
//                [empty mbarriers][partial sums 6 x R x 33 floats][flags: 4 ints]
//                [unit of each stage: stages x int64 (dynamic unit order)]
// (three double-buffered sets of partial sums; LayerNorm reduces up to four
// quantities a row and has four sets, 8 x R x 33 floats)
// `nin` is the number of row inputs streamed through the ring (1, or 2 with
// the fused residual add).
constexpr int bulk_red_sets(bool ln) { return ln ? 8 : 6; }

__host__ __device__ constexpr size_t bulk_smem_bytes(int stages, int R, int N, int nin = 1,
                                                     bool ln = false) {
    return static_cast<size_t>(stages) * nin * R * N * 2 + static_cast<size_t>(stages) * 16 +
           static_cast<size_t>(bulk_red_sets(ln)) * R * kRedStride * 4 + 16 +
           static_cast<size_t>(stages) * 8;
}

// NT consumer threads (N / 8 / VPR of them) plus one producer warp.
// NT <= 0 is the generic form: the consumer count comes from the launch
// (blockDim.x - 32, a multiple of 32; at most 256 for NT == 0, 512 for
// NT == -1, 192 for NT == -2) and chunks past the end of a row (any
// N % 8 == 0) are masked.
template <int VPR, int R, int NT>
constexpr int bulk_max_threads() {
    return NT > 0 ? NT + 32 : (NT == 0 ? 288 : (NT == -2 ? 224 : 544));
}

// Generic LayerNorm with at most two chunks per thread is built for two CTAs
// per SM (96 registers, no spills): its per-row chain wants a second CTA's
// warps more than it wants registers.  The other forms keep one CTA's full
// register budget (the fused add spills at the two-CTA bound; RMSNorm and the
// fused add measured no gain from a second CTA; power-of-two LayerNorm with
// 1-CTA registers is faster over many rows).
// NT == -2 is a second build of generic LayerNorm at 8 chunks a thread, for
// two CTAs of at most 192 consumers (128 registers, no spills, against 165 in
// the one-CTA build): the launcher takes it only where the one-CTA build's
// registers leave one CTA an SM (12288-wide rows: 0.76 -> 0.83 of the copy).
template <int VPR, int NT, bool LN>
constexpr int bulk_min_ctas() { return ((LN && NT == 0 && VPR <= 2) || NT == -2) ? 2 : 1; }

template <class E, int VPR, int R, int NT, bool ADD, bool LN>
__global__ void __launch_bounds__(bulk_max_threads<VPR, R, NT>(), bulk_min_ctas<VPR, NT, LN>())
    rms_persistent_bulk_kernel(const BulkArgs a) {
    constexpr bool GENERIC = NT <= 0;
    static_assert(!(ADD && LN), "the fused add is an RMSNorm prologue");
    constexpr int NIN = ADD ? 2 : 1;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = a.stages;
    const int N = a.N;
    const uint32_t row_bytes = static_cast<uint32_t>(N) * 2u;
    const uint32_t stage_bytes = row_bytes * R * NIN;  // x rows, then r rows
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t *empty = full + S;
    float *red = reinterpret_cast<float *>(empty + S);
    // flags[0], flags[1]: "consumers give up" for even / odd units (decided
    // before a named barrier, read after it); flags[2]: "someone gave up",
    // polled inside waits so nobody waits out a full timeout needlessly.
    volatile int *flags = reinterpret_cast<volatile int *>(red + bulk_red_sets(LN) * R * kRedStride);
    // dynamic unit order: the unit each stage holds, -1 for "no more units"
    volatile int64_t *unit_of = reinterpret_cast<volatile int64_t *>(flags + 4);

    const int nt = GENERIC ? static_cast<int>(blockDim.x) - 32 : NT;
    const int NW = nt / 32;
    const int cpr = N >> 3;
    // chunk j of this thread lies inside the row (always, for exact covers)
    auto live = [&](int tid_, int j) { return !GENERIC || tid_ + j * nt < cpr; };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        fence_mbar_init();
    }
    pdl_trigger();
    pdl_wait();
    __syncthreads();

    // Unit order: round-robin (UnitSchedule), or with a workspace the dynamic
    // order of DynUnits over units of R consecutive rows, for launches of six
    // units a CTA and more (below that the CTAs would all reach the counter
    // at once, and the short launch measured slower for it).  LayerNorm is
    // built without the dynamic order: its heavier consumers measured mixed
    // with it (+4% at 8192 x 12288, -5% at 32768 x 4096), and its run-time
    // checks alone cost LayerNorm's instruction-bound consumers about 4%.
    const int64_t total_units = (a.M + R - 1) / R;
    const bool dyn = !LN && a.ws != nullptr && total_units >= 6 * static_cast<int64_t>(gridDim.x);
    const UnitSchedule sched(a.M, gridDim.x, R);
    const int64_t bid = blockIdx.x;
    const int64_t n_units = dyn ? INT64_MAX : sched.units(bid);
    const DynUnits du(a.ws, static_cast<int64_t>(gridDim.x), bid, total_units, S);

    if (warp == NW) {
        // ---- producer ----
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int64_t k = 0;
            bool marked = false;                   // the "no more units" stage was armed
            int64_t u_cur = dyn ? du.first(0) : 0;  // the unit of iteration k (dynamic order)
            for (; k < n_units; ++k) {
                const int s = static_cast<int>(k % S);
                // the unit of iteration k + 1: static, or fetched now and first
                // read an iteration later, after two empty waits and a copy
                // issue have hidden the round trip
                int64_t u_after = 0;
                if (dyn) u_after = k + 1 < du.lead ? du.first(k + 1) : du.fetch();
                const int64_t u = u_cur;
                if (k >= S) {
                    const uint32_t par = static_cast<uint32_t>((k / S - 1) & 1);
                    if (!mbar_wait_bounded(&empty[s], par, a.timeout_ns, &flags[2])) {
                        flags[2] = 1;
                        raise_status(RN_STATUS_WAIT_TIMEOUT);
                        break;
                    }
                }
                int64_t r0;
                int rows;
                if (dyn) {
                    if (u >= total_units) {
                        unit_of[s] = -1;  // a stage with no bytes: the consumers stop here
                        mbar_arrive(&full[s]);
                        marked = true;
                        break;
                    }
                    unit_of[s] = u;
                    r0 = u * R;
                    rows = static_cast<int>(a.M - r0 < R ? a.M - r0 : R);
                    u_cur = u_after;
                } else {
                    sched.unit(bid, k, &r0, &rows);
                }
                const uint32_t bytes = static_cast<uint32_t>(rows) * row_bytes;
                mbar_arrive_expect_tx(&full[s], bytes * NIN);
                if (!(a.debug & 1)) {
                    uint8_t *dst = ring + static_cast<size_t>(s) * stage_bytes;
                    bulk_copy_g2s(dst, a.x + r0 * N, bytes, &full[s], pol);
                    if constexpr (ADD)
                        bulk_copy_g2s(dst + row_bytes * R, a.r + r0 * N, bytes, &full[s], pol);
                }
            }
            if (dyn) du.finish();
            // Drain: every copy issued into this CTA's ring lands before the
            // CTA may exit.  The last use of each stage is among the last S
            // (the last S - 1 when the stop marker re-armed stage k % S, whose
            // previous unit the consumers had already released).
            const int64_t issued = k;
            const int64_t first_kk = issued - S + (marked ? 1 : 0);
            const uint64_t t0 = globaltimer_ns();
            for (int64_t kk = (first_kk > 0 ? first_kk : 0); kk < issued; ++kk) {
                const uint64_t spent = globaltimer_ns() - t0;
                const uint64_t budget = spent < a.timeout_ns ? a.timeout_ns - spent : 0;
                if (!mbar_wait_bounded(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), budget,
                                       nullptr)) {
                    raise_status(RN_STATUS_WAIT_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ---- consumers ----
    const int tid = threadIdx.x;
    uint4 wv[VPR];
#pragma unroll
    for (int j = 0; j < VPR; ++j)
        wv[j] = live(tid, j) ? weight16<E>(a.w, tid + j * nt) : make_uint4(0u, 0u, 0u, 0u);
    uint4 bv[LN ? VPR : 1];  // LayerNorm bias, held like the weights
    // With at most 256 consumers (3 warps a scheduler, up to 170 registers a
    // thread) and at most 4 chunks a thread, LayerNorm keeps its weights
    // widened to fp32 pairs: one fused multiply-add a pair and no widening of
    // w per row.  Other layouts keep them packed (512 consumers put 5 warps on
    // one scheduler: 96 registers; 8 chunks would spill).  The bias stays
    // packed.
    constexpr bool WIDE_W = LN && NT <= 256 && VPR <= 4;
    float2 wf[WIDE_W ? VPR * 4 : 1];
    if constexpr (LN) {
#pragma unroll
        for (int j = 0; j < VPR; ++j)
            bv[j] = live(tid, j) ? bias16(a.b, tid + j * nt) : make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (WIDE_W) {
#pragma unroll
        for (int j = 0; j < VPR; ++j) {
            wf[4 * j + 0] = make_float2(E::lo(wv[j].x), E::hi(wv[j].x));
            wf[4 * j + 1] = make_float2(E::lo(wv[j].y), E::hi(wv[j].y));
            wf[4 * j + 2] = make_float2(E::lo(wv[j].z), E::hi(wv[j].z));
            wf[4 * j + 3] = make_float2(E::lo(wv[j].w), E::hi(wv[j].w));
        }
    }

    for (int64_t k = 0; k < n_units; ++k) {
        int64_t r0 = 0;
        int rows = 0;
        if (!dyn) sched.unit(bid, k, &r0, &rows);
        // Keep the weights packed (16-bit) across rows: without this the
        // compiler hoists their fp32 widening out of the loop and doubles
        // the register footprint.
        if constexpr (!WIDE_W) {
#pragma unroll
            for (int j = 0; j < VPR; ++j)
                asm volatile("" : "+r"(wv[j].x), "+r"(wv[j].y), "+r"(wv[j].z), "+r"(wv[j].w));
        }
        if constexpr (LN) {
#pragma unroll
            for (int j = 0; j < VPR; ++j)
                asm volatile("" : "+r"(bv[j].x), "+r"(bv[j].y), "+r"(bv[j].z), "+r"(bv[j].w));
        }
        const int s = static_cast<int>(k % S);
        const uint32_t par = static_cast<uint32_t>((k / S) & 1);
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], par, a.timeout_ns, &flags[2]));
        // Dynamic order: the stage names its unit; the stop marker is a unit
        // with no rows, which still goes through the barrier below, so every
        // consumer warp leaves at the same unit.
        bool last = false;
        if (dyn && ok) {
            const int64_t u = unit_of[s];
            last = u < 0;
            r0 = last ? 0 : u * R;
            rows = last ? 0 : static_cast<int>(a.M - r0 < R ? a.M - r0 : R);
        }
        const uint8_t *st = ring + static_cast<size_t>(s) * stage_bytes;
        uint4 xv[R][VPR];
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
#pragma unroll
            for (int j = 0; j < VPR; ++j)
                xv[rr][j] = (ok && !last && live(tid, j))
                                ? ld_shared16(st + rr * row_bytes + 16u * (tid + j * nt))
                                : make_uint4(0u, 0u, 0u, 0u);
        if constexpr (ADD) {
            // h = x + r, stored at once; the rest of the row works on h
#pragma unroll
            for (int rr = 0; rr < R; ++rr)
#pragma unroll
                for (int j = 0; j < VPR; ++j)
                    xv[rr][j] = add8<E>(xv[rr][j],
                                     (ok && !last && live(tid, j))
                                         ? ld_shared16(st + (R + rr) * row_bytes + 16u * (tid + j * nt))
                                         : make_uint4(0u, 0u, 0u, 0u));
            if (ok) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr)
                    if (rr < rows)
#pragma unroll
                        for (int j = 0; j < VPR; ++j)
                            if (live(tid, j)) st16(a.h + (r0 + rr) * N + 8 * (tid + j * nt), xv[rr][j]);
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (ok) {
                mbar_arrive(&empty[s]);
            } else {
                flags[k & 1] = 1;
                flags[2] = 1;
                raise_status(RN_STATUS_WAIT_TIMEOUT);
            }
        }
        if constexpr (LN) {
            // LayerNorm: one CTA reduction of each row's sum and sum of
            // squares.  Where the mean is small against the spread (mean^2 <=
            // 4 var) the variance follows directly as E[x^2] - mean^2 (the
            // fp32 cancellation costs at most ~2 bits of a 2^-23 error).  A
            // unit with a row outside that bound (a large mean, a constant
            // row) takes a second reduction over the centred squares, the
            // exact two-pass form.  Every warp finishes the same partials in
            // the same order, so the choice is uniform over the CTA.
            float s1[R], q1[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                float acc = 0.f, acq = 0.f;
#pragma unroll
                for (int j = 0; j < VPR; ++j) {
                    acc += sum8<E>(xv[rr][j]);
                    acq += sumsq8<E>(xv[rr][j]);
                }
                s1[rr] = warp_sum(acc);
                q1[rr] = warp_sum(acq);
            }
            float *rbs = red + (k & 1) * R * kRedStride;        // sums
            float *rbq = red + (2 + (k & 1)) * R * kRedStride;  // sums of squares
            float *rbc = red + (4 + (k & 1)) * R * kRedStride;  // centred squares
            float *rbd = red + (6 + (k & 1)) * R * kRedStride;  // and deviations
            if (lane == 0) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr) {
                    rbs[rr * kRedStride + warp] = s1[rr];
                    rbq[rr * kRedStride + warp] = q1[rr];
                }
            }
            named_bar_sync(1, nt);
            if (flags[k & 1] || last) break;  // same decision in every consumer warp
            // lane rr finishes row rr's statistics once; shuffles hand them out
            float my_mean = 0.f, my_rstd = 0.f, my_ncr = 0.f;
            bool my_exact = false;
            if (lane < R) {
                float t = 0.f, u = 0.f;
                for (int q = 0; q < NW; ++q) {
                    t += rbs[lane * kRedStride + q];
                    u += rbq[lane * kRedStride + q];
                }
                my_mean = t / static_cast<float>(N);
                const float var = u / static_cast<float>(N) - my_mean * my_mean;
                my_exact = lane < rows && !(var > 0.f && my_mean * my_mean <= 4.f * var);
                my_rstd = __frsqrt_rn(var + a.eps);
            }
            float mean[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) mean[rr] = __shfl_sync(0xffffffffu, my_mean, rr);
            if (__any_sync(0xffffffffu, my_exact)) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr) {
                    DevAcc acc = dev_zero();
#pragma unroll
                    for (int j = 0; j < VPR; ++j)
                        if (live(tid, j)) dev8<E>(xv[rr][j], mean[rr], acc);
                    const float2 ds = dev_sums(acc);
                    const float dsum = warp_sum(ds.x);
                    const float qsum = warp_sum(ds.y);
                    if (lane == 0) {
                        rbd[rr * kRedStride + warp] = dsum;
                        rbc[rr * kRedStride + warp] = qsum;
                    }
                }
                named_bar_sync(1, nt);
                if (lane < R) {
                    float t = 0.f, u = 0.f;
                    for (int q = 0; q < NW; ++q) {
                        t += rbc[lane * kRedStride + q];
                        u += rbd[lane * kRedStride + q];
                    }
                    const Centring ce = centre(u, t, N, a.eps);
                    my_rstd = ce.rstd;
                    my_ncr = ce.ncr;
                }
            }
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const float rstd = __shfl_sync(0xffffffffu, my_rstd, rr);
                const float ncr = __shfl_sync(0xffffffffu, my_ncr, rr);
                if (rr < rows) {
                    uint16_t *yr = a.y + (r0 + rr) * N;
#pragma unroll
                    for (int j = 0; j < VPR; ++j)
                        if (live(tid, j))
                            st16(yr + 8 * (tid + j * nt),
                                 WIDE_W ? ln8w<E>(xv[rr][j], &wf[4 * j], bv[j], mean[rr], rstd, ncr)
                                        : ln8<E>(xv[rr][j], wv[j], bv[j], mean[rr], rstd, ncr));
                }
            }
        } else {
            float ss[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < VPR; ++j) acc += sumsq8<E>(xv[rr][j]);
                ss[rr] = warp_sum(acc);
            }
            // Same for x: hold it packed across the barrier, widen again after.
#pragma unroll
            for (int rr = 0; rr < R; ++rr)
#pragma unroll
                for (int j = 0; j < VPR; ++j)
                    asm volatile("" : "+r"(xv[rr][j].x), "+r"(xv[rr][j].y), "+r"(xv[rr][j].z),
                                 "+r"(xv[rr][j].w));
            float *rb = red + (k & 1) * R * kRedStride;
            if (lane == 0) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr) rb[rr * kRedStride + warp] = ss[rr];
            }
            named_bar_sync(1, nt);
            if (flags[k & 1] || last) break;  // same decision in every consumer warp
            // Lane rr finishes row rr's sum and scale once; a shuffle hands it
            // to the warp (instead of every thread redoing all R rows).
            float my_scale = 0.f;
            if (lane < R) {
                float tot = 0.f;
                for (int q = 0; q < NW; ++q) tot += rb[lane * kRedStride + q];
                my_scale = row_scale(tot, N, a.eps, a.l2);
            }
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const float rstd = __shfl_sync(0xffffffffu, my_scale, rr);
                if (rr < rows) {
                    uint16_t *yr = a.y + (r0 + rr) * N;
#pragma unroll
                    for (int j = 0; j < VPR; ++j)
                        if (live(tid, j))
                            st16(yr + 8 * (tid + j * nt), scale8<E>(xv[rr][j], wv[j], rstd));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Everything one launch needs; r and h are set only for the fused residual
// add, b only for LayerNorm.
struct RowJob {
    const uint16_t *x;
    const uint16_t *w;
    float eps;
    int64_t M;
    int N;
    uint16_t *y;
    const uint16_t *r;
    uint16_t *h;
    const uint16_t *b;  // LayerNorm bias (may be null)
    int l2;             // L2Norm instead of RMSNorm (w may be null: unit weights)
    unsigned long long *ws = nullptr;  // workspace: dynamic unit order on the ring
};

template <class E, bool ADD, bool LN>
static int launch_warp_rows(const RowJob &j, cudaStream_t st, const DeviceInfo &dev) {
    const int cpr = j.N >> 3;
    const int wpb = 8;
    const int64_t want = (j.M + wpb - 1) / wpb;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 64;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
#define RN_WARP(V)                                                                              \
    return launch_pdl(rms_warp_rows_kernel<E, V, ADD, LN>, dim3(grid), dim3(32 * wpb), 0, st, j.x, \
                      j.w, j.eps, j.M, j.N, j.y, j.r, j.h, j.b, j.l2)
    if (cpr <= 32) RN_WARP(1);
    if (cpr <= 64) RN_WARP(2);
    if (cpr <= 128) RN_WARP(4);
    if (cpr <= 256) RN_WARP(8);
    if constexpr (!ADD && !LN) {
        // RMSNorm and L2Norm rows up to 4096 wide: 12 or 16 chunks a lane
        // (120 registers, no spills; two CTAs of 8 warps an SM, 8 KiB of
        // loads in flight a warp).  The fused add and LayerNorm fit too but
        // measured well behind their rings, so they are not built this way.
        if (cpr <= 384) RN_WARP(12);
        if (cpr <= 512) RN_WARP(16);
    }
#undef RN_WARP
    return RN_ERR_SHAPE;
}

template <class E, bool ADD, bool LN>
static int launch_cta_rows(const RowJob &j, cudaStream_t st, const DeviceInfo &dev) {
    const int cpr = j.N >> 3;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 2048;
    const unsigned grid = static_cast<unsigned>(j.M < cap ? j.M : cap);
    // Threads: enough 16-byte chunks per thread to keep several loads in
    // flight, at most 1024 threads.
    auto nthreads = [&](int vpt) {
        int t = (cpr + vpt - 1) / vpt;
        return ((t + 31) / 32) * 32;
    };
#define RN_CTA(V, T)                                                                           \
    return launch_pdl(rms_cta_rows_kernel<E, V, T, ADD, LN>, dim3(grid), dim3(nthreads(V)), 0, st, \
                      j.x, j.w, j.eps, j.M, j.N, j.y, j.r, j.h, j.b, j.l2)
    if (cpr <= 512) RN_CTA(1, 512);
    if (cpr <= 1024) RN_CTA(2, 512);
    if (cpr <= 2048) RN_CTA(4, 512);
    if (cpr <= 4096) RN_CTA(8, 512);
    if (cpr <= 8192) RN_CTA(8, 1024);
#undef RN_CTA
    return RN_ERR_SHAPE;
}

// Geometry of the persistent schedule, measured on GB300 (back-to-back
// launches of one shape, two alternating buffer sets): NT consumer threads x
// VPR 16-byte chunks cover one row exactly, R rows make a stage, `stages`
// stages per CTA, `ctas` co-resident CTAs per SM.  About 64 KiB in flight per
// SM (two 32 KiB stages) streams best at every width from 4096 to 16384:
// deeper rings and 64 KiB stages measured slower (more concurrent DRAM
// streams, no more bandwidth).  Short launches are dominated by their ramp:
// 4096-wide rows run two CTAs per SM up to M = 4096 rows and a third stage up
// to 8192; launches of 4096 rows take a third stage at widths 8192 and 16384.  With the fused residual add a
// stage carries R rows of x and R rows of r, so R is halved where needed to
// keep a stage at 64 KiB or less; 32768-wide rows do not fit two such stages
// and take the CTA-per-row schedule.
struct BulkGeometry {
    int nt, vpr, R, stages, ctas;
    bool generic;        // masked instantiation with a run-time consumer count
    bool tight = false;  // LayerNorm's two-CTA build at 8 chunks a thread (NT == -2)
};

// Rows that are not a power-of-two width (any N % 8 == 0 from 512 to 32768)
// run the generic instantiation: the fewest chunks per thread (1, 2, 4 or 8)
// that keep the consumers at 256 threads or fewer (N <= 16384), else 8 chunks
// and up to 512 threads (plain RMSNorm only: the fused forms would spill);
// R = 8 / VPR rows a stage.
static bool bulk_geometry_generic(int N, bool add, bool ln, BulkGeometry *g) {
    if (N < 512 || N > 32768 || N % 8 != 0) return false;
    const int cpr = N >> 3;
    // Plain RMSNorm / L2Norm fit up to 512 consumers without spilling and want
    // the warps; the fused forms carry more per thread and stay at 256.
    const int cap = (add || ln) ? 256 : 512;
    int vpr = 1;
    while (vpr < 8 && (cpr + vpr - 1) / vpr > cap) vpr *= 2;
    const int per = (cpr + vpr - 1) / vpr;
    if (per > cap) return false;
    // LayerNorm runs every consumer the layout allows (chunks past the row
    // are masked): its heavier per-row work wants the warps (3-5% measured);
    // the other forms use just enough threads to cover the row.
    const int nt = ln ? cap : ((per + 31) / 32) * 32;
    const int R = 8 / vpr;
    const size_t stage = static_cast<size_t>(add ? 2 : 1) * R * N * 2;
    if (2 * stage > 200 * 1024) return false;  // two stages must fit with room to spare
    // About 64 KiB in flight per SM, as the tuned power-of-two layouts have:
    // small stages get a deeper ring (2 to 4 stages).
    int stages = static_cast<int>((65536 + stage - 1) / stage);
    if (stages < 2) stages = 2;
    if (stages > 4) stages = 4;
    // LayerNorm with at most two chunks a thread: two CTAs per SM, two stages
    // each (the second CTA lifted 16384 x 3072 from 0.68 to 0.79 of the copy;
    // deeper rings measured 1% behind).
    if (ln && vpr <= 2) {
        *g = {nt, vpr, R, 2, 2, true};
        return true;
    }
    *g = {nt, vpr, R, stages, 1, true};
    return true;
}

static bool bulk_geometry(int64_t M, int N, bool add, bool ln, bool dyn, BulkGeometry *g) {
    const bool few_rows = M <= 8192;
    if ((N & (N - 1)) != 0 || N < 1024) return bulk_geometry_generic(N, add, ln, g);
    if (ln) {
        // LayerNorm keeps its mean and the bias loads live too: 4-row stages at
        // 4096 and no ring at 32768 (both spill otherwise).
        switch (N) {
            case 1024: *g = {128, 1, 8, 2, 1, false}; break;
            case 2048: *g = {256, 1, 8, 2, 1, false}; break;
            case 4096:
                // Up to 8192 rows the generic layout (the same 4-row stages)
                // at two CTAs per SM (8192 rows: 0.73 -> 0.85); over more rows
                // one CTA with the full register budget and a third stage.
                if (few_rows) return bulk_geometry_generic(N, add, ln, g);
                *g = {256, 2, 4, 3, 1, false};  // 3 stages: 0.96 -> 0.98 at 65536 rows
                break;
            // A third stage pays for LayerNorm (slower consumers than RMSNorm,
            // whose two-stage rings measured 3-5% ahead of three) at 8192
            // (16384 rows: 0.94 -> 0.97); at 16384 it measured even.
            case 8192: *g = {256, 4, 2, 3, 1, false}; break;
            // 256 x 8 (measured ahead of 512 x 4), in the generic instantiation:
            // the same layout measured 3% ahead of the one built for 16384.
            case 16384: return bulk_geometry_generic(N, add, ln, g);
            default: return false;
        }
        return true;
    }
    if (add) {
        switch (N) {
            case 1024: *g = {128, 1, 8, 2, 1, false}; break;
            case 2048: *g = {256, 1, 8, 2, 1, false}; break;
            case 4096: *g = {256, 2, 4, 2, 1, false}; break;
            case 8192: *g = {256, 4, 2, 2, 1, false}; break;
            case 16384: *g = {512, 4, 1, 2, 1, false}; break;
            default: return false;
        }
        return true;
    }
    // A third stage pays only on the shortest launches (4096 rows), where the
    // ramp is a larger share of the time.
    const int short_stages = M <= 4096 ? 3 : 2;
    switch (N) {
        case 1024: *g = {128, 1, 8, 2, 1, false}; break;
        case 2048: *g = {256, 1, 8, 2, 1, false}; break;
        case 4096:
            // Two CTAs per SM through 4096 rows, then one CTA.  In the dynamic
            // unit order four stages (128 KiB in flight an SM): alone even with
            // two or three (8192 rows: 0.843 against 0.847 of the copy; 32768
            // rows: 0.979 against 0.983), and inside a sequence of differently
            // shaped launches, where the ring starts behind a wider one, 7 us
            // shorter at 8192 rows and 22 us for 16384 and 32768 rows together
            // (against two stages and one warp per row).  In the fixed order
            // four stages measured 3-10% slower alone (32768 rows: 0.969 ->
            // 0.876): three stages through 8192 rows, then two.
            if (M <= 4096)
                *g = BulkGeometry{256, 2, 4, 2, 2, false};
            else
                *g = BulkGeometry{256, 2, 4, dyn ? 4 : (few_rows ? 3 : 2), 1, false};
            break;
        case 8192: *g = {256, 4, 2, short_stages, 1, false}; break;
        // Three 32 KiB stages at every row count in the dynamic unit order,
        // 1% ahead of two from 8192 rows (32768 rows: 1.012 -> 1.024 of the
        // copy); in the fixed order two from 8192 rows (three: 0.992 -> 0.962).
        case 16384: *g = {512, 4, 1, dyn ? 3 : short_stages, 1, false}; break;
        case 32768: *g = {512, 8, 1, 2, 1, false}; break;
        default: return false;
    }
    return true;
}

// How many CTAs of one instantiation of the ring an SM holds at once with
// `nt` consumers and `smem` bytes of dynamic shared memory (registers, shared
// memory and threads all counted), or -1 when the runtime cannot say.  Opts
// the instantiation into `smem_cap` bytes of shared memory on first use.
template <class E, int VPR, int R, int NT, bool ADD, bool LN>
static int bulk_fit(int nt, size_t smem, int smem_cap) {
    static std::atomic<int> attr_done[kMaxDevices];
    // last answer per device: (consumers << 20 | smem) << 8 | CTAs, plus bit 63
    static std::atomic<uint64_t> cache[kMaxDevices];
    const auto kernel = rms_persistent_bulk_kernel<E, VPR, R, NT, ADD, LN>;
    const int dev = current_device_index();
    if (dev < 0 || dev >= kMaxDevices) return -1;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cap) !=
            cudaSuccess) {
            cudaGetLastError();
            return -1;
        }
        attr_done[dev].store(1, std::memory_order_release);
    }
    const uint64_t key = (static_cast<uint64_t>(nt) << 20 | static_cast<uint64_t>(smem)) << 8;
    const uint64_t hit = cache[dev].load(std::memory_order_acquire);
    if ((hit >> 63) && ((hit & ~(1ull << 63)) >> 8) == (key >> 8)) return static_cast<int>(hit & 0xFF);
    int fit = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kernel, nt + 32, smem) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (fit > 255) fit = 255;
    cache[dev].store((1ull << 63) | key | static_cast<uint64_t>(fit), std::memory_order_release);
    return fit;
}

// Launches one instantiation of the ring on min(M, SMs x ctas) CTAs.  A
// request for more than one CTA per SM is clamped to what the SM holds at
// once: CTAs beyond that would run as a second wave behind the first instead
// of beside it.
template <class E, int VPR, int R, int NT, bool ADD, bool LN>
static int launch_bulk_inst(const BulkArgs &a, int sm_count, int ctas, size_t smem, int smem_cap,
                            cudaStream_t st, int nt = NT) {
    const int fit = bulk_fit<E, VPR, R, NT, ADD, LN>(nt, smem, smem_cap);
    if (fit < 0) return RN_ERR_DEVICE;
    if (fit == 0) return RN_ERR_SHAPE;
    if (ctas > fit) ctas = fit;
    int64_t grid = static_cast<int64_t>(sm_count) * ctas;
    if (grid > a.M) grid = a.M;
    return launch_pdl(rms_persistent_bulk_kernel<E, VPR, R, NT, ADD, LN>,
                      dim3(static_cast<unsigned>(grid)), dim3(nt + 32), smem, st, a);
}

// LayerNorm at a generic width: the layout with the most chunks a thread
// (1, 2, 4 or 8) whose consumers, rounded up to whole warps, cover the row
// with at most `max_masked_tenths` tenths of their chunk slots masked, number
// at least three warps, and leave room for two or three such CTAs on an SM,
// each with a two-stage ring (at 8 chunks, in the two-CTA build when the
// one-CTA build's registers leave room for one).  Several independent CTAs a
// SM keep the per-row chain of LayerNorm (reduce, derive mean and scale,
// normalise) in flight in parallel; one CTA with more threads on the same row
// does not (16384 x 5120: 0.65 -> 0.93 of the copy; 6144: 0.75 -> 0.88;
// 3072: 0.79 -> 0.85).  Returns false, `geo` untouched, when none qualifies.
template <class E>
static bool ln_multi_cta_try(int N, int smem_cap, int max_masked_tenths, BulkGeometry *geo) {
    const int cpr = N >> 3;
    for (int v = 8; v >= 1; v >>= 1) {
        const int per = (cpr + v - 1) / v;
        if (per > 256) return false;  // fewer chunks a thread only need more consumers
        const int nt = ((per + 31) / 32) * 32;
        // at most max_masked_tenths tenths of the chunk slots masked
        if (nt < 96 || 10LL * cpr < (10LL - max_masked_tenths) * nt * v) continue;
        const int R = 8 / v;
        if (2ull * R * N * 2 > 200 * 1024) continue;
        const size_t smem = bulk_smem_bytes(2, R, N, 1, true);
        int fit = -1;
        switch (v) {
            case 8:
                fit = bulk_fit<E, 8, 1, 0, false, true>(nt, smem, smem_cap);
                if (fit < 2 && nt <= 192) {  // the two-CTA build, at fewer registers
                    const int f2 = bulk_fit<E, 8, 1, -2, false, true>(nt, smem, smem_cap);
                    if (f2 >= 2) {
                        *geo = {nt, v, R, 2, f2 < 3 ? f2 : 3, true, true};
                        return true;
                    }
                }
                break;
            case 4: fit = bulk_fit<E, 4, 2, 0, false, true>(nt, smem, smem_cap); break;
            case 2: fit = bulk_fit<E, 2, 4, 0, false, true>(nt, smem, smem_cap); break;
            case 1: fit = bulk_fit<E, 1, 8, 0, false, true>(nt, smem, smem_cap); break;
        }
        if (fit >= 2) {
            *geo = {nt, v, R, 2, fit < 3 ? fit : 3, true};
            return true;
        }
    }
    return false;
}

template <class E>
static void ln_multi_cta_layout(int N, int smem_cap, BulkGeometry *geo) {
    // A tenth of the slots masked at most; failing that, a fifth, which still
    // beats one CTA an SM (6656: 0.81 -> 0.82, 7168: 0.87 -> 0.88 of the copy).
    if (!ln_multi_cta_try<E>(N, smem_cap, 1, geo)) ln_multi_cta_try<E>(N, smem_cap, 2, geo);
}

template <class E, bool ADD, bool LN>
static int launch_persistent_bulk(const RowJob &j, cudaStream_t st, const DeviceInfo &dev,
                                  uint64_t timeout_ns, int debug_flags) {
    constexpr int NIN = ADD ? 2 : 1;
    BulkGeometry geo;
    const int N = j.N;
    // The geometry for the dynamic unit order when the kernel will take it: a
    // workspace, and six units a CTA or more (the kernel's own test).
    bool dyn = !LN && j.ws != nullptr;
    if (!bulk_geometry(j.M, N, ADD, LN, dyn, &geo)) return RN_ERR_SHAPE;
    if (dyn && (j.M + geo.R - 1) / geo.R < 6LL * dev.sm_count * geo.ctas) {
        dyn = false;
        bulk_geometry(j.M, N, ADD, LN, dyn, &geo);
    }
    const int smem_cap = dev.max_smem_optin < 232448 ? dev.max_smem_optin : 232448;
    if constexpr (LN) {
        if (geo.generic && (debug_flags & 0x1FF0) == 0) ln_multi_cta_layout<E>(N, smem_cap, &geo);
    }
    const size_t stage_cost = static_cast<size_t>(NIN) * geo.R * N * 2 + 16;
    int max_stages = static_cast<int>((smem_cap - bulk_smem_bytes(0, geo.R, N, NIN, LN)) / stage_cost);
    if (max_stages > 16) max_stages = 16;
    int stages = geo.stages;
    const int forced_stages = (debug_flags >> 8) & 0x1F;
    if (forced_stages > 0) stages = forced_stages;
    int ctas_per_sm = (debug_flags >> 4) & 0xF;
    if (ctas_per_sm <= 0) ctas_per_sm = geo.ctas;
    // The CTAs of an SM share its shared memory: give up stages first (down
    // to two a CTA), then CTAs.  Registers are checked at launch.
    while (ctas_per_sm > 1 && max_stages / ctas_per_sm < 2) --ctas_per_sm;
    if (stages * ctas_per_sm > max_stages) stages = max_stages / ctas_per_sm;
    if (stages < 2) return RN_ERR_SHAPE;
    const size_t smem = bulk_smem_bytes(stages, geo.R, N, NIN, LN);
    BulkArgs a{j.x, j.w, j.y, j.r, j.h, j.b, j.l2, j.M, N, j.eps, stages, debug_flags & 1,
               timeout_ns ? timeout_ns : 2000000000ull, j.ws};
    const int sm = dev.sm_count, c = ctas_per_sm;
    if (geo.generic) {
        if constexpr (ADD || LN) {  // at most 256 consumers
            switch (geo.vpr) {
                case 1: return launch_bulk_inst<E, 1, 8, 0, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 2: return launch_bulk_inst<E, 2, 4, 0, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 4: return launch_bulk_inst<E, 4, 2, 0, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 8:
                    if constexpr (LN) {
                        if (geo.tight)
                            return launch_bulk_inst<E, 8, 1, -2, ADD, LN>(a, sm, c, smem, smem_cap, st,
                                                                          geo.nt);
                    }
                    return launch_bulk_inst<E, 8, 1, 0, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
            }
        } else {  // up to 512 consumers
            switch (geo.vpr) {
                case 1: return launch_bulk_inst<E, 1, 8, -1, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 2: return launch_bulk_inst<E, 2, 4, -1, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 4: return launch_bulk_inst<E, 4, 2, -1, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
                case 8: return launch_bulk_inst<E, 8, 1, -1, ADD, LN>(a, sm, c, smem, smem_cap, st, geo.nt);
            }
        }
        return RN_ERR_SHAPE;
    }
    switch (N) {
        case 1024: return launch_bulk_inst<E, 1, 8, 128, ADD, LN>(a, sm, c, smem, smem_cap, st);
        case 2048: return launch_bulk_inst<E, 1, 8, 256, ADD, LN>(a, sm, c, smem, smem_cap, st);
        case 4096: return launch_bulk_inst<E, 2, 4, 256, ADD, LN>(a, sm, c, smem, smem_cap, st);
        case 8192: return launch_bulk_inst<E, 4, 2, 256, ADD, LN>(a, sm, c, smem, smem_cap, st);
        case 16384:
            if constexpr (!LN) return launch_bulk_inst<E, 4, 1, 512, ADD, LN>(a, sm, c, smem, smem_cap, st);
            break;
        case 32768:
            if constexpr (!ADD && !LN)
                return launch_bulk_inst<E, 8, 1, 512, ADD, LN>(a, sm, c, smem, smem_cap, st);
            break;
    }
    return RN_ERR_SHAPE;
}

static int auto_schedule(int64_t M, int N, bool add, bool ln, bool l2, bool ws,
                         const DeviceInfo &dev) {
    BulkGeometry geo;
    // Up to 2048-wide rows one warp per row is ahead of the ring; wider rows
    // take the ring wherever it applies (3072-wide RMSNorm rows measured 0.85
    // of the copy on the ring against 0.60 one CTA per row) from 6 rows per SM
    // up: with fewer, one CTA per row keeps every row in flight at once and
    // measured ahead (608 x 16384: 0.90 against 0.76).  The fused add below
    // 4096-wide generic rows also stays on one CTA per row, which keeps twice
    // the loads in flight and measured ahead (0.94-0.97 against 0.89-0.94).
    if (N <= 2048 && M >= 4LL * dev.sm_count) return RN_SCHED_WARP_ROW;
    // Rows up to 4096 wide over many rows: one warp per row, loads straight
    // into registers.
    //   L2Norm (no weights: more warps an SM) from 12 rows a SM, ahead of the
    //     ring at every count measured from 2048 rows, 3072 or 4096 wide
    //     (4096 x 4096: 0.80 -> 0.87, 12288 x 4096: 0.89 -> 0.94, 32768 x
    //     4096: 0.98 -> 1.01 of the copy; even at 1024 rows).
    //   RMSNorm from 128 rows a SM (32768 x 3584: 0.89 -> 0.97), except 4096
    //     wide with a workspace: there the ring's four stages in the dynamic
    //     unit order are even with one warp per row alone (65536 rows: 1.01)
    //     or ahead (24576 rows: 0.943 -> 0.958), and 11-12 us shorter a
    //     launch behind a wider one (32768 rows).
    if (!add && !ln && N <= 4096) {
        if (l2 && M >= 12LL * dev.sm_count) return RN_SCHED_WARP_ROW;
        if (!l2 && !(ws && N == 4096) && M >= 128LL * dev.sm_count) return RN_SCHED_WARP_ROW;
    }
    if (bulk_geometry(M, N, add, ln, ws, &geo) && M >= 6LL * dev.sm_count &&
        !(add && geo.generic && N < 4096))
        return RN_SCHED_PERSIST_BULK;
    if (N <= 2048 && M < 64) return RN_SCHED_WARP_ROW;
    return RN_SCHED_CTA_ROW;
}

static int check_rows(int64_t M, int64_t N) {
    if (M < 0 || N < 8 || N > 65536 || (N % 8) != 0) return RN_ERR_SHAPE;
    return RN_OK;
}

template <class E, bool ADD, bool LN>
static int rows_dispatch(const RowJob &j, int schedule, uint64_t timeout_ns, int debug_flags,
                         rn_stream_t stream) {
    if (schedule < RN_SCHED_AUTO || schedule > RN_SCHED_PERSIST_BULK) return RN_ERR_ARG;
    const DeviceInfo *dev = current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (schedule == RN_SCHED_AUTO)
        schedule = auto_schedule(j.M, j.N, ADD, LN, j.l2 != 0, j.ws != nullptr, *dev);
    switch (schedule) {
        case RN_SCHED_WARP_ROW: return launch_warp_rows<E, ADD, LN>(j, st, *dev);
        case RN_SCHED_CTA_ROW: return launch_cta_rows<E, ADD, LN>(j, st, *dev);
        case RN_SCHED_PERSIST_BULK:
            return launch_persistent_bulk<E, ADD, LN>(j, st, *dev, timeout_ns, debug_flags);
    }
    return RN_ERR_ARG;
}

// Validates one call and launches it in the element format E.
template <class E>
static int rows_run(const RowCall &c) {
    const int rc = check_rows(c.M, c.N);
    if (rc != RN_OK) return rc;
    if (c.op < ROW_RMS || c.op > ROW_LN) return RN_ERR_ARG;
    if (c.M == 0) return RN_OK;
    const bool need_w = c.op != ROW_L2;
    const bool add = c.op == ROW_ADD_RMS;
    if (!c.x || !c.y || (need_w && !c.w) || (add && (!c.r || !c.h))) return RN_ERR_NULL;
    if (!aligned16(c.x) || !aligned16(c.y) || (c.w && !aligned16(c.w)) ||
        (add && (!aligned16(c.r) || !aligned16(c.h))) ||
        (c.op == ROW_LN && c.b && !aligned16(c.b)) || (c.workspace && !aligned16(c.workspace)))
        return RN_ERR_ALIGN;
    if (add && c.h == c.y) return RN_ERR_ARG;  // two different outputs
    RowJob j{c.x, c.op == ROW_L2 ? nullptr : c.w, c.eps, c.M, static_cast<int>(c.N), c.y,
             nullptr, nullptr, nullptr, c.op == ROW_L2 ? 1 : 0,
             static_cast<unsigned long long *>(c.workspace)};
    if (add) {
        j.r = c.r;
        j.h = c.h;
        return rows_dispatch<E, true, false>(j, c.schedule, c.timeout_ns, c.debug_flags, c.stream);
    }
    if (c.op == ROW_LN) {
        j.b = c.b;
        return rows_dispatch<E, false, true>(j, c.schedule, c.timeout_ns, c.debug_flags, c.stream);
    }
    return rows_dispatch<E, false, false>(j, c.schedule, c.timeout_ns, c.debug_flags, c.stream);
}

// The schedule rows_run picks in RN_SCHED_AUTO (the same for both formats:
// only the element size enters the geometry).
static int rows_select(int op, int64_t M, int64_t N, bool ws) {
    if (check_rows(M, N) != RN_OK) return RN_ERR_SHAPE;
    const DeviceInfo *dev = current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    return auto_schedule(M, static_cast<int>(N), op == ROW_ADD_RMS, op == ROW_LN, op == ROW_L2, ws,
                         *dev);
}

// Reads (and optionally clears) this translation unit's status word; the
// caller has synchronised the device.
static int rows_status_word(unsigned int *out, int clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) {
        cudaGetLastError();
        return RN_ERR_DEVICE;
    }
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) {
            cudaGetLastError();
            return RN_ERR_DEVICE;
        }
    }
    *out = v;
    return RN_OK;
}

}  // namespace rn
