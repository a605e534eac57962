// qk_norm_rope.cu -- fused per-head Q/K RMSNorm + neox RoPE, in place on
// packed QKV, and the rotary cos/sin table builder (sm_103a).
//
// "[pretuned] Optimize fused_qk_norm_rope on B200", section "Summary": each
// query/key head is loaded once as its two rotary halves (plus the
// non-rotary tail when rotary_dim < head_dim), reduced over the whole head
// while register-resident, scaled by the Q or K weight, rotated, and stored
// once.  No shared memory, no block barrier, no store-then-reload.
//
// Lane layout: a head of D elements is owned by LPH lanes (LPH = 8, 16 or
// 32, i.e. 4, 2 or 1 heads per warp, the schedules that section lists for
// large, medium and tiny token counts).  Lane `sub` of the group holds
//   x[sub*A     .. sub*A + A)        first rotary half   (A = r/2 / LPH)
//   x[r/2+sub*A .. r/2+sub*A + A)    second rotary half  (its rotation partners)
//   x[r+sub*B   .. r+sub*B + B)      tail                (B = (D-r) / LPH)
// so every neox pair (i, i + r/2) sits in one lane and the rotation needs no
// shuffle; only the sum of squares crosses lanes (log2(LPH) xor-shuffles).
#include "rn_common.cuh"
#include "rn_host.h"

namespace rn {

// ---- vector helpers -----------------------------------------------------------

// CNT consecutive bf16 -> fp32.  The pointer is aligned to the widest of
// 16/8/4/2 bytes that divides 2*CNT (the host validates the layouts).
template <int CNT>
__device__ __forceinline__ void load_bf(const uint16_t *p, float (&o)[CNT]) {
    if constexpr ((CNT * 2) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 8; ++k) {
            const uint4 v = *reinterpret_cast<const uint4 *>(p + 8 * k);
            o[8 * k + 0] = bf_lo(v.x); o[8 * k + 1] = bf_hi(v.x);
            o[8 * k + 2] = bf_lo(v.y); o[8 * k + 3] = bf_hi(v.y);
            o[8 * k + 4] = bf_lo(v.z); o[8 * k + 5] = bf_hi(v.z);
            o[8 * k + 6] = bf_lo(v.w); o[8 * k + 7] = bf_hi(v.w);
        }
    } else if constexpr ((CNT * 2) % 8 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p + 4 * k);
            o[4 * k + 0] = bf_lo(v.x); o[4 * k + 1] = bf_hi(v.x);
            o[4 * k + 2] = bf_lo(v.y); o[4 * k + 3] = bf_hi(v.y);
        }
    } else if constexpr ((CNT * 2) % 4 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(p + 2 * k);
            o[2 * k + 0] = bf_lo(v); o[2 * k + 1] = bf_hi(v);
        }
    } else {
#pragma unroll
        for (int k = 0; k < CNT; ++k) o[k] = __uint_as_float(static_cast<uint32_t>(p[k]) << 16);
    }
}

template <int CNT>
__device__ __forceinline__ void store_bf(uint16_t *p, const float (&v)[CNT]) {
    if constexpr ((CNT * 2) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 8; ++k) {
            uint4 u;
            u.x = pack_bf2(v[8 * k + 0], v[8 * k + 1]);
            u.y = pack_bf2(v[8 * k + 2], v[8 * k + 3]);
            u.z = pack_bf2(v[8 * k + 4], v[8 * k + 5]);
            u.w = pack_bf2(v[8 * k + 6], v[8 * k + 7]);
            *reinterpret_cast<uint4 *>(p + 8 * k) = u;
        }
    } else if constexpr ((CNT * 2) % 8 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k) {
            uint2 u;
            u.x = pack_bf2(v[4 * k + 0], v[4 * k + 1]);
            u.y = pack_bf2(v[4 * k + 2], v[4 * k + 3]);
            *reinterpret_cast<uint2 *>(p + 4 * k) = u;
        }
    } else if constexpr ((CNT * 2) % 4 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k)
            *reinterpret_cast<uint32_t *>(p + 2 * k) = pack_bf2(v[2 * k + 0], v[2 * k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < CNT; ++k) {
            __nv_bfloat16 b = __float2bfloat16_rn(v[k]);
            p[k] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
}

template <int CNT>
__device__ __forceinline__ void load_f32(const float *p, float (&o)[CNT]) {
    if constexpr (CNT % 4 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p + 4 * k));
            o[4 * k + 0] = v.x; o[4 * k + 1] = v.y; o[4 * k + 2] = v.z; o[4 * k + 3] = v.w;
        }
    } else if constexpr (CNT % 2 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k) {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(p + 2 * k));
            o[2 * k + 0] = v.x; o[2 * k + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < CNT; ++k) o[k] = __ldg(p + k);
    }
}

// ---- the fused kernel -----------------------------------------------------------

struct QkArgs {
    uint16_t *qkv;
    const uint16_t *wq;
    const uint16_t *wk;
    const float *cos_sin;
    const int64_t *pos;
    int64_t T;
    int Hq;
    int Hkv;
    float eps;
    int64_t max_pos;  // > 0: check positions against it; 0: trust them
    int *err;         // checked mode: RN_STATUS_BAD_POSITION is OR-ed in here
};

template <int D, int R, int LPH>
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const QkArgs a) {
    constexpr int H2 = R / 2;
    constexpr int A = H2 / LPH;
    constexpr int B = (D - R) / LPH;
    constexpr int HPW = 32 / LPH;
    static_assert(A * LPH == H2 && B * LPH == D - R && A >= 1, "bad lane layout");

    const int lane = threadIdx.x & 31;
    const int sub = lane % LPH;
    const int grp = lane / LPH;
    const uint32_t hpt = static_cast<uint32_t>(a.Hq + a.Hkv);  // normed heads per token
    const uint32_t total = static_cast<uint32_t>(a.T) * hpt;   // host: < 2^31
    const int64_t W = static_cast<int64_t>(a.Hq + 2 * a.Hkv) * D;
    const uint64_t warp0 =
        (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;

    for (uint64_t base = warp0 * HPW; base < total; base += nwarps * HPW) {
        const uint32_t g = static_cast<uint32_t>(base) + grp;
        const bool active = g < total;
        const uint32_t t = active ? g / hpt : 0u;
        const uint32_t h = active ? g - t * hpt : 0u;
        uint16_t *head = a.qkv + static_cast<int64_t>(t) * W + static_cast<int64_t>(h) * D;

        int64_t p = active ? __ldg(a.pos + t) : 0;
        bool ok = active;
        if (a.max_pos > 0 && active && (p < 0 || p >= a.max_pos)) {
            ok = false;
            if (sub == 0) atomicOr(a.err, RN_STATUS_BAD_POSITION);
        }
        if (!ok) p = 0;  // keeps every address in range; nothing is stored

        float x1[A], x2[A], x3[B > 0 ? B : 1];
        if (ok) {
            load_bf<A>(head + sub * A, x1);
            load_bf<A>(head + H2 + sub * A, x2);
            if constexpr (B > 0) load_bf<B>(head + R + sub * B, x3);
        } else {
#pragma unroll
            for (int i = 0; i < A; ++i) x1[i] = x2[i] = 0.f;
#pragma unroll
            for (int i = 0; i < (B > 0 ? B : 1); ++i) x3[i] = 0.f;
        }
        float c[A], s[A];
        const float *cs = a.cos_sin + p * R;
        load_f32<A>(cs + sub * A, c);
        load_f32<A>(cs + H2 + sub * A, s);

        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < A; ++i) ss = fmaf(x2[i], x2[i], fmaf(x1[i], x1[i], ss));
        if constexpr (B > 0) {
#pragma unroll
            for (int i = 0; i < B; ++i) ss = fmaf(x3[i], x3[i], ss);
        }
        ss = group_sum<LPH>(ss);
        const float rstd = __frsqrt_rn(ss / static_cast<float>(D) + a.eps);

        const uint16_t *wp = (h < static_cast<uint32_t>(a.Hq)) ? a.wq : a.wk;
        float w1[A], w2[A];
        load_bf<A>(wp + sub * A, w1);
        load_bf<A>(wp + H2 + sub * A, w2);

        float o1[A], o2[A];
#pragma unroll
        for (int i = 0; i < A; ++i) {
            const float n1 = x1[i] * rstd * w1[i];
            const float n2 = x2[i] * rstd * w2[i];
            o1[i] = n1 * c[i] - n2 * s[i];
            o2[i] = n2 * c[i] + n1 * s[i];
        }
        if (ok) {
            store_bf<A>(head + sub * A, o1);
            store_bf<A>(head + H2 + sub * A, o2);
        }
        if constexpr (B > 0) {
            float w3[B];
            load_bf<B>(wp + R + sub * B, w3);
#pragma unroll
            for (int i = 0; i < B; ++i) x3[i] = x3[i] * rstd * w3[i];
            if (ok) store_bf<B>(head + R + sub * B, x3);
        }
    }
}

// ---- table builder ----------------------------------------------------------------

// fp64 angle and trig, rounded once to fp32.
__global__ void rope_table_kernel(double theta, int64_t max_pos, int r, float *out) {
    const int h = r / 2;
    const int64_t n = max_pos * h;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = idx / h;
        const int i = static_cast<int>(idx - p * h);
        const double f = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(r));
        const double ang = static_cast<double>(p) * f;
        double sv, cv;
        sincos(ang, &sv, &cv);
        out[p * r + i] = __double2float_rn(cv);
        out[p * r + h + i] = __double2float_rn(sv);
    }
}

// ---- host side ----------------------------------------------------------------------

template <int D, int R, int LPH>
static int launch_qk(const QkArgs &a, bool persistent, cudaStream_t st, const DeviceInfo &dev) {
    constexpr int HPW = 32 / LPH;
    constexpr int kThreads = 256;
    const uint64_t total = static_cast<uint64_t>(a.T) * static_cast<uint64_t>(a.Hq + a.Hkv);
    const uint64_t warps = (total + HPW - 1) / HPW;
    uint64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
    if (persistent) {
        const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * 8;  // 8 x 256 threads per SM
        if (blocks > cap) blocks = cap;
    }
    if (blocks > 0x7fffffffULL) blocks = 0x7fffffffULL;
    qk_norm_rope_kernel<D, R, LPH><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(a);
    return launch_status();
}

// Largest lanes-per-head <= the request that tiles both rotary halves and
// the tail of this (D, rotary_dim); 8 always does.
template <int D, int R>
static int launch_qk_lph(const QkArgs &a, int lph, bool persistent, cudaStream_t st,
                         const DeviceInfo &dev) {
    constexpr int H2 = R / 2;
    if constexpr (H2 % 32 == 0 && (D - R) % 32 == 0) {
        if (lph >= 32) return launch_qk<D, R, 32>(a, persistent, st, dev);
    }
    if constexpr (H2 % 16 == 0 && (D - R) % 16 == 0) {
        if (lph >= 16) return launch_qk<D, R, 16>(a, persistent, st, dev);
    }
    if constexpr (H2 % 8 == 0 && (D - R) % 8 == 0) {
        return launch_qk<D, R, 8>(a, persistent, st, dev);
    }
    return RN_ERR_SHAPE;
}

// Heads-per-warp schedule by token count: one head per warp for 1-2
// tokens, two through 256 tokens, four (persistent grid) beyond.
static int auto_qk_schedule(int64_t T) {
    if (T <= 2) return RN_QK_HEAD_PER_WARP;
    if (T <= 256) return RN_QK_TWO_HEADS;
    return RN_QK_PERSISTENT;
}

static int qk_dispatch(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                       const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                       int Hkv, int D, int rotary_dim, float eps, int64_t max_pos, int *err,
                       int schedule, rn_stream_t stream) {
    if (T < 0 || Hq < 0 || Hkv < 0) return RN_ERR_SHAPE;
    if (D != 64 && D != 128 && D != 256) return RN_ERR_SHAPE;
    if (rotary_dim != D && rotary_dim != D / 2 && rotary_dim != D / 4) return RN_ERR_SHAPE;
    if (static_cast<uint64_t>(T) * static_cast<uint64_t>(Hq + Hkv) >= (1ull << 31))
        return RN_ERR_SHAPE;
    if (T == 0 || Hq + Hkv == 0) return RN_OK;
    if (!qkv || !wq || !wk || !cos_sin || !positions) return RN_ERR_NULL;
    if (!aligned16(qkv) || !aligned16(wq) || !aligned16(wk) || !aligned16(cos_sin) ||
        !aligned16(positions))
        return RN_ERR_ALIGN;
    int lph;
    bool persistent = false;
    if (schedule == RN_QK_AUTO) schedule = auto_qk_schedule(T);
    switch (schedule) {
        case RN_QK_HEAD_PER_WARP: lph = 32; break;
        case RN_QK_TWO_HEADS: lph = 16; break;
        case RN_QK_FOUR_HEADS: lph = 8; break;
        case RN_QK_PERSISTENT: lph = 8; persistent = true; break;
        default: return RN_ERR_ARG;
    }
    const DeviceInfo *dev = current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    QkArgs a{reinterpret_cast<uint16_t *>(qkv), wq, wk, cos_sin, positions, T, Hq, Hkv,
             eps, max_pos, err};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int r = rotary_dim;
#define RN_QK_GO(D_, R_)                                                               \
    if (D == (D_) && r == (R_)) return launch_qk_lph<D_, R_>(a, lph, persistent, st, *dev);
    RN_QK_GO(64, 64) RN_QK_GO(64, 32) RN_QK_GO(64, 16)
    RN_QK_GO(128, 128) RN_QK_GO(128, 64) RN_QK_GO(128, 32)
    RN_QK_GO(256, 256) RN_QK_GO(256, 128) RN_QK_GO(256, 64)
#undef RN_QK_GO
    return RN_ERR_SHAPE;
}

}  // namespace rn

extern "C" {

int qk_norm_rope_fwd(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk, const float *cos_sin,
                     const int64_t *positions, int64_t T, int Hq, int Hkv, int D,
                     int rotary_dim, float eps, rn_stream_t stream) {
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps, 0,
                           nullptr, RN_QK_AUTO, stream);
}

int qk_norm_rope_fwd_sched(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                           const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                           int Hkv, int D, int rotary_dim, float eps, int schedule,
                           rn_stream_t stream) {
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps, 0,
                           nullptr, schedule, stream);
}

int qk_norm_rope_fwd_checked(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                             const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                             int Hkv, int D, int rotary_dim, float eps, int64_t max_pos,
                             int *d_err_flag, rn_stream_t stream) {
    if (max_pos < 1) return RN_ERR_SHAPE;
    if (!d_err_flag && T > 0 && Hq + Hkv > 0) return RN_ERR_NULL;
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                           max_pos, d_err_flag, RN_QK_AUTO, stream);
}

int qk_norm_rope_select_schedule(int64_t T) {
    if (T < 0) return RN_ERR_SHAPE;
    return rn::auto_qk_schedule(T);
}

int rope_cos_sin_table(double theta, int64_t max_pos, int rotary_dim, float *cos_sin,
                       rn_stream_t stream) {
    if (max_pos < 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0.0))
        return RN_ERR_SHAPE;
    if (max_pos == 0) return RN_OK;
    if (!cos_sin) return RN_ERR_NULL;
    if (!rn::aligned16(cos_sin)) return RN_ERR_ALIGN;
    const rn::DeviceInfo *dev = rn::current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    const int64_t n = max_pos * (rotary_dim / 2);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev->sm_count) * 16;
    if (blocks > cap) blocks = cap;
    rn::rope_table_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                            reinterpret_cast<cudaStream_t>(stream)>>>(theta, max_pos, rotary_dim,
                                                                       cos_sin);
    return rn::launch_status();
}

}  // extern "C"
