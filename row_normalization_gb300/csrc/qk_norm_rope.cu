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
#include <cmath>

#include "rn_common.cuh"
#include "rn_host.h"

namespace rn {

// This translation unit's status word (RN_STATUS_* bits); rn_device_status()
// ORs it with the other units' words.
static __device__ unsigned int g_qk_status = 0u;

__device__ __forceinline__ void raise_qk_status(unsigned int bits) { atomicOr(&g_qk_status, bits); }

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

// CNT consecutive fp32 from shared memory (plain loads; __ldg is global-only).
template <int CNT>
__device__ __forceinline__ void load_f32_smem(const float *p, float (&o)[CNT]) {
    if constexpr (CNT % 4 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k) {
            const float4 v = *reinterpret_cast<const float4 *>(p + 4 * k);
            o[4 * k + 0] = v.x; o[4 * k + 1] = v.y; o[4 * k + 2] = v.z; o[4 * k + 3] = v.w;
        }
    } else if constexpr (CNT % 2 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k) {
            const float2 v = *reinterpret_cast<const float2 *>(p + 2 * k);
            o[2 * k + 0] = v.x; o[2 * k + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < CNT; ++k) o[k] = p[k];
    }
}

// ---- the fused kernel -----------------------------------------------------------

struct QkArgs {
    uint16_t *qkv;
    const uint16_t *wq;
    const uint16_t *wk;
    const void *cos_sin;  // fp32 or bf16 [max_pos, R]: the kernels' TB parameter says which
    const int64_t *pos;
    int64_t T;
    int Hq;
    int Hkv;
    float eps;
    int64_t max_pos;  // > 0: check positions against it; 0: trust them
    int *err;         // checked mode: RN_STATUS_BAD_POSITION is OR-ed in here
};

// STYLE 0: neox pairs (i, i + r/2).  STYLE 1: GPT-J pairs (2i, 2i + 1): the
// lane's rotary slice is then 2A contiguous elements, de-interleaved into the
// same (first, second) arrays so the arithmetic is shared.  TB: the cos/sin
// table holds bf16 entries (widened exactly to fp32 on load) instead of fp32.
template <int D, int R, int LPH, int STYLE, bool TB>
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const QkArgs a) {
    constexpr int H2 = R / 2;
    constexpr int A = H2 / LPH;
    constexpr int B = (D - R) / LPH;
    constexpr int HPW = 32 / LPH;
    static_assert(A * LPH == H2 && B * LPH == D - R && A >= 1, "bad lane layout");
    pdl_trigger();
    pdl_wait();

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
        // The head's loads do not wait for the position: only the cos/sin
        // row and the store depend on it (a token rejected below is read but
        // never written).
        float x1[A], x2[A], x3[B > 0 ? B : 1];
        if (active) {
            if constexpr (STYLE == 0) {
                load_bf<A>(head + sub * A, x1);
                load_bf<A>(head + H2 + sub * A, x2);
            } else {
                float xr[2 * A];
                load_bf<2 * A>(head + sub * 2 * A, xr);
#pragma unroll
                for (int i = 0; i < A; ++i) {
                    x1[i] = xr[2 * i];
                    x2[i] = xr[2 * i + 1];
                }
            }
            if constexpr (B > 0) load_bf<B>(head + R + sub * B, x3);
        } else {
#pragma unroll
            for (int i = 0; i < A; ++i) x1[i] = x2[i] = 0.f;
#pragma unroll
            for (int i = 0; i < (B > 0 ? B : 1); ++i) x3[i] = 0.f;
        }
        // the weights do not wait for the reduction either
        const uint16_t *wp = (h < static_cast<uint32_t>(a.Hq)) ? a.wq : a.wk;
        float w1[A], w2[A];
        if constexpr (STYLE == 0) {
            load_bf<A>(wp + sub * A, w1);
            load_bf<A>(wp + H2 + sub * A, w2);
        } else {
            float wr[2 * A];
            load_bf<2 * A>(wp + sub * 2 * A, wr);
#pragma unroll
            for (int i = 0; i < A; ++i) {
                w1[i] = wr[2 * i];
                w2[i] = wr[2 * i + 1];
            }
        }
        bool ok = active;
        if (a.max_pos > 0 && active && (p < 0 || p >= a.max_pos)) {
            ok = false;
            if (sub == 0) atomicOr(a.err, RN_STATUS_BAD_POSITION);
        }
        if (!ok) p = 0;  // keeps every address in range; nothing is stored
        float c[A], s[A];
        if constexpr (TB) {  // bf16 entries, widened exactly
            const uint16_t *cs = static_cast<const uint16_t *>(a.cos_sin) + p * R;
            load_bf<A>(cs + sub * A, c);
            load_bf<A>(cs + H2 + sub * A, s);
        } else {
            const float *cs = static_cast<const float *>(a.cos_sin) + p * R;
            load_f32<A>(cs + sub * A, c);
            load_f32<A>(cs + H2 + sub * A, s);
        }

        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < A; ++i) ss = fmaf(x2[i], x2[i], fmaf(x1[i], x1[i], ss));
        if constexpr (B > 0) {
#pragma unroll
            for (int i = 0; i < B; ++i) ss = fmaf(x3[i], x3[i], ss);
        }
        ss = group_sum<LPH>(ss);
        const float rstd = __frsqrt_rn(ss / static_cast<float>(D) + a.eps);

        float o1[A], o2[A];
#pragma unroll
        for (int i = 0; i < A; ++i) {
            const float n1 = x1[i] * rstd * w1[i];
            const float n2 = x2[i] * rstd * w2[i];
            o1[i] = n1 * c[i] - n2 * s[i];
            o2[i] = n2 * c[i] + n1 * s[i];
        }
        if (ok) {
            if constexpr (STYLE == 0) {
                store_bf<A>(head + sub * A, o1);
                store_bf<A>(head + H2 + sub * A, o2);
            } else {
                float orr[2 * A];
#pragma unroll
                for (int i = 0; i < A; ++i) {
                    orr[2 * i] = o1[i];
                    orr[2 * i + 1] = o2[i];
                }
                store_bf<2 * A>(head + sub * 2 * A, orr);
            }
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

// ---- persistent schedule: tokens streamed through a bulk-copy ring -------------
//
// One CTA per SM: 16 consumer warps (8 for 256-wide heads) and 1 producer warp.  A unit is `tps`
// consecutive tokens; for each, the producer copies the token's contiguous
// query+key region (H heads x D bf16; the value heads are skipped) and the
// cos/sin row its position selects into a stage of a shared-memory ring with
// 1D bulk copies, all completing on the stage's mbarrier.  Producer lane i
// owns token i of the unit and loads its position one unit ahead.
//
// Consumer warps take four heads at a time from the stage (8 lanes per head:
// the lane layout of qk_norm_rope_kernel) and keep wq and wk in registers as
// packed bf16.  The arithmetic runs on fp32 pairs (Blackwell's packed
// FFMA2/FMUL2), the results are stored in place with 16-byte writes, and each
// warp releases the stage once it has read its heads.  Which warp takes which
// quad of heads rotates from stage to stage, so no warp is always the one with
// the extra quad.  No CTA-wide barrier after set-up.

struct QkBulkArgs {
    QkArgs q;
    int tps;          // tokens per stage (<= 32: one producer lane per token)
    int stages;
    int debug;        // bit 0: never issue the copies (exercises the timeout path)
    uint64_t inv_h;   // ceil(2^32 / H): token slot of stage head hh = (hh * inv_h) >> 32
                      // (exact for hh, H < 2^16; 2^32 itself when H == 1)
    uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t qk_bulk_smem_bytes(int stages, int tps, int tok_bytes,
                                                        int cs_bytes) {
    return static_cast<size_t>(stages) * tps * (tok_bytes + cs_bytes) +  // ring
           static_cast<size_t>(stages) * 16 +                            // full + empty
           static_cast<size_t>(stages) * tps * 4 +                       // token valid flags
           16;                                                           // abort flag
}

__device__ __forceinline__ void bulk_copy_g2s_plain(void *dst_smem, const void *src_gmem,
                                                    uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// load_f32_smem for the CNT consecutive floats that lane `sub` (of the 8 lanes
// serving one head) owns at p = base + sub * CNT.  A 16-byte-per-lane shared
// load is served 8 lanes at a time; with CNT = 8 lanes sub and sub + 4 sit
// 128 bytes apart, so reading both 16-byte halves in the same order puts two
// lanes on every bank group.  Lanes 4-7 read their halves in the other order,
// which gives the 8 lanes 8 distinct bank groups per load.
template <int CNT>
__device__ __forceinline__ void load_f32_smem_lanes(const float *p, float (&o)[CNT], int sub) {
    if constexpr (CNT == 8) {
        const bool sw = (sub & 4) != 0;
        const float4 a = *reinterpret_cast<const float4 *>(p + (sw ? 4 : 0));
        const float4 b = *reinterpret_cast<const float4 *>(p + (sw ? 0 : 4));
        o[0] = sw ? b.x : a.x; o[1] = sw ? b.y : a.y; o[2] = sw ? b.z : a.z; o[3] = sw ? b.w : a.w;
        o[4] = sw ? a.x : b.x; o[5] = sw ? a.y : b.y; o[6] = sw ? a.z : b.z; o[7] = sw ? a.w : b.w;
    } else {
        load_f32_smem<CNT>(p, o);
    }
}

__device__ __forceinline__ float2 bf2f(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }

// CNT (even) consecutive bf16 as CNT/2 packed words; same alignment rules as load_bf.
template <int CNT>
__device__ __forceinline__ void load_words(const uint16_t *p, uint32_t (&o)[CNT / 2]) {
    static_assert(CNT % 2 == 0, "even counts only");
    if constexpr ((CNT * 2) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 8; ++k) {
            const uint4 v = *reinterpret_cast<const uint4 *>(p + 8 * k);
            o[4 * k + 0] = v.x; o[4 * k + 1] = v.y; o[4 * k + 2] = v.z; o[4 * k + 3] = v.w;
        }
    } else if constexpr ((CNT * 2) % 8 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p + 4 * k);
            o[2 * k + 0] = v.x; o[2 * k + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k) o[k] = *reinterpret_cast<const uint32_t *>(p + 2 * k);
    }
}

template <int CNT>
__device__ __forceinline__ void store_words(uint16_t *p, const uint32_t (&v)[CNT / 2]) {
    if constexpr ((CNT * 2) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 8; ++k)
            *reinterpret_cast<uint4 *>(p + 8 * k) =
                make_uint4(v[4 * k + 0], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    } else if constexpr ((CNT * 2) % 8 == 0) {
#pragma unroll
        for (int k = 0; k < CNT / 4; ++k)
            *reinterpret_cast<uint2 *>(p + 4 * k) = make_uint2(v[2 * k + 0], v[2 * k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < CNT / 2; ++k) *reinterpret_cast<uint32_t *>(p + 2 * k) = v[k];
    }
}

__device__ __forceinline__ uint32_t pack_f2(float2 v) { return pack_bf2(v.x, v.y); }

// Consumer threads: 16 warps, or 8 for 256-wide heads (twice the per-lane state).
template <int D>
constexpr int qk_bulk_consumers() { return D >= 256 ? 256 : 512; }

// Normalise + rotate one head's lane slice with the given weights (packed
// bf16): o = rotate(x * rstd * w), tail = x * rstd * w.  fp32 pairs.
template <int A2, int B2, bool TAIL>
__device__ __forceinline__ void qk_rotate_slice(const uint32_t (&x1)[A2], const uint32_t (&x2)[A2],
                                                const uint32_t (&x3)[B2], const uint32_t (&w1)[A2],
                                                const uint32_t (&w2)[A2], const uint32_t (&w3)[B2],
                                                const float (&c)[2 * A2],
                                                const float (&sn)[2 * A2], float rstd,
                                                uint32_t (&o1)[A2], uint32_t (&o2)[A2],
                                                uint32_t (&o3)[B2]) {
    const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
    for (int i = 0; i < A2; ++i) {
        const float2 n1 = __fmul2_rn(__fmul2_rn(bf2f(x1[i]), r2), bf2f(w1[i]));
        const float2 n2 = __fmul2_rn(__fmul2_rn(bf2f(x2[i]), r2), bf2f(w2[i]));
        const float2 cc = make_float2(c[2 * i], c[2 * i + 1]);
        const float2 sv = make_float2(sn[2 * i], sn[2 * i + 1]);
        const float2 nsv = make_float2(-sn[2 * i], -sn[2 * i + 1]);
        o1[i] = pack_f2(__ffma2_rn(n1, cc, __fmul2_rn(n2, nsv)));
        o2[i] = pack_f2(__ffma2_rn(n2, cc, __fmul2_rn(n1, sv)));
    }
    if constexpr (TAIL) {
#pragma unroll
        for (int i = 0; i < B2; ++i) o3[i] = pack_f2(__fmul2_rn(__fmul2_rn(bf2f(x3[i]), r2), bf2f(w3[i])));
    }
}

// GPT-J slice: the lane's 2A contiguous rotary elements arrive as two arrays of
// A/2 words (x1 then x2); every word is one pair (2j, 2j + 1) and rotates by
// (c_j, s_j): (e, o) -> (e c - o s, o c + e s).  Same signature as
// qk_rotate_slice, so the caller picks by style.
__device__ __forceinline__ uint32_t gptj_pair(uint32_t x, uint32_t w, float2 r2, float c, float s) {
    const float2 n = __fmul2_rn(__fmul2_rn(bf2f(x), r2), bf2f(w));
    const float2 t = __fmul2_rn(n, make_float2(c, c));
    return pack_f2(__ffma2_rn(make_float2(n.y, n.x), make_float2(-s, s), t));
}

template <int A2, int B2, bool TAIL>
__device__ __forceinline__ void qk_rotate_slice_gptj(const uint32_t (&x1)[A2],
                                                     const uint32_t (&x2)[A2],
                                                     const uint32_t (&x3)[B2],
                                                     const uint32_t (&w1)[A2],
                                                     const uint32_t (&w2)[A2],
                                                     const uint32_t (&w3)[B2],
                                                     const float (&c)[2 * A2],
                                                     const float (&sn)[2 * A2], float rstd,
                                                     uint32_t (&o1)[A2], uint32_t (&o2)[A2],
                                                     uint32_t (&o3)[B2]) {
    const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
    for (int i = 0; i < A2; ++i) {
        o1[i] = gptj_pair(x1[i], w1[i], r2, c[i], sn[i]);
        o2[i] = gptj_pair(x2[i], w2[i], r2, c[A2 + i], sn[A2 + i]);
    }
    if constexpr (TAIL) {
#pragma unroll
        for (int i = 0; i < B2; ++i) o3[i] = pack_f2(__fmul2_rn(__fmul2_rn(bf2f(x3[i]), r2), bf2f(w3[i])));
    }
}

template <int STYLE, int A2, int B2, bool TAIL>
__device__ __forceinline__ void qk_rotate(const uint32_t (&x1)[A2], const uint32_t (&x2)[A2],
                                          const uint32_t (&x3)[B2], const uint32_t (&w1)[A2],
                                          const uint32_t (&w2)[A2], const uint32_t (&w3)[B2],
                                          const float (&c)[2 * A2], const float (&sn)[2 * A2],
                                          float rstd, uint32_t (&o1)[A2], uint32_t (&o2)[A2],
                                          uint32_t (&o3)[B2]) {
    if constexpr (STYLE == 0)
        qk_rotate_slice<A2, B2, TAIL>(x1, x2, x3, w1, w2, w3, c, sn, rstd, o1, o2, o3);
    else
        qk_rotate_slice_gptj<A2, B2, TAIL>(x1, x2, x3, w1, w2, w3, c, sn, rstd, o1, o2, o3);
}

// The same operation as qk_norm_rope_kernel, with two heads per group of LPH
// lanes and round: heads j and j + G of the warp's 2G (G = 32 / LPH groups).
// The launch is bound by the bytes in flight, and two thirds of a lane's
// in-flight registers in qk_norm_rope_kernel hold its cos/sin slice, which the
// heads of a warp load alike when they belong to one token.  Here both heads of
// a group belong to one token whenever 2G divides the normed heads per token
// (40 at D 128, LPH 8), so one cos/sin slice serves both (a second row is read
// only when the two tokens differ), and the heads stay packed bf16 until they
// are reduced: twice the heads in flight a warp for a quarter more registers.
//
// Lanes per head by layout (pair_lph): 4 lanes at D 64, 8 at D 128, 16 at
// D 256, so that at full rotary each lane's two rotary pieces are 8 elements
// (16-byte loads) at every D.  At 8 lanes for every D, a D 64 lane moved 8-byte
// pieces and a D 256 lane held 32 cos/sin floats (two CTAs an SM): 0.70 and
// 0.68 of the copy at 4096 tokens (D 64 rotary 64; D 256 rotary 256), against
// 0.84 and 0.95 with 4 and 16 lanes.
//
// Arithmetic: neox heads with an fp32 table take the token ring's (fp32
// pairs, two accumulators, qk_rotate); at D 128 (the ring's lane layout)
// their results are bit-identical to RN_QK_BULK, and the packed form measured
// 1% (rotary 128) to 8% (rotary 64) faster at 2048-4096 tokens than the
// scalar one.  GPT-J pairs and bf16 tables keep qk_norm_rope_kernel's scalar
// form (bit-identical to RN_QK_FOUR_HEADS at D 128), where the packed one
// measured 1-5% slower.
template <int D, int R, int LPH, int STYLE, bool TB>
__global__ void __launch_bounds__(256, 3) qk_pair_kernel(const QkArgs a) {
    constexpr int G = 32 / LPH;  // groups a warp
    constexpr int H2 = R / 2;
    constexpr int A = H2 / LPH;
    constexpr int B = (D - R) / LPH;
    constexpr int A2 = A / 2;
    constexpr int B2 = B > 0 ? B / 2 : 1;
    constexpr bool PACKED = STYLE == 0 && !TB;
    static_assert(A * LPH == H2 && B * LPH == D - R && A % 2 == 0 && B % 2 == 0, "bad layout");
    pdl_trigger();
    pdl_wait();

    const int lane = threadIdx.x & 31;
    const int sub = lane % LPH;
    const int grp = lane / LPH;
    // the lane's two rotary pieces: neox A elements of each half, GPT-J 2A
    // contiguous elements (two A-runs)
    const int off1 = STYLE == 0 ? sub * A : sub * 2 * A;
    const int off2 = STYLE == 0 ? H2 + sub * A : sub * 2 * A + A;
    const uint32_t hpt = static_cast<uint32_t>(a.Hq + a.Hkv);  // normed heads per token
    const uint32_t total = static_cast<uint32_t>(a.T) * hpt;   // host: < 2^31
    const int64_t W = static_cast<int64_t>(a.Hq + 2 * a.Hkv) * D;
    const uint64_t warp0 = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;

    for (uint64_t base = warp0 * 2 * G; base < total; base += nwarps * 2 * G) {
        uint32_t th[2], hh[2];
        bool act[2];
        uint16_t *head[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t g = static_cast<uint32_t>(base) + grp + G * j;
            act[j] = g < total;
            th[j] = act[j] ? g / hpt : 0u;
            hh[j] = act[j] ? g - th[j] * hpt : 0u;
            head[j] = a.qkv + static_cast<int64_t>(th[j]) * W + static_cast<int64_t>(hh[j]) * D;
        }
        int64_t p = act[0] ? __ldg(a.pos + th[0]) : 0;
        uint32_t x1[2][A2], x2[2][A2], x3[2][B2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (act[j]) {
                load_words<A>(head[j] + off1, x1[j]);
                load_words<A>(head[j] + off2, x2[j]);
                if constexpr (B > 0) load_words<B>(head[j] + R + sub * B, x3[j]);
            } else {
#pragma unroll
                for (int i = 0; i < A2; ++i) x1[j][i] = x2[j][i] = 0u;
#pragma unroll
                for (int i = 0; i < B2; ++i) x3[j][i] = 0u;
            }
        }
        // a rejected position: read but never written (as qk_norm_rope_kernel)
        auto accept = [&](int64_t &pp, bool active) {
            bool ok = active;
            if (a.max_pos > 0 && active && (pp < 0 || pp >= a.max_pos)) {
                ok = false;
                if (sub == 0) atomicOr(a.err, RN_STATUS_BAD_POSITION);
            }
            if (!ok) pp = 0;
            return ok;
        };
        float c[A], sn[A];
        auto load_cs = [&](int64_t pp) {
            if constexpr (TB) {
                const uint16_t *cs = static_cast<const uint16_t *>(a.cos_sin) + pp * R;
                load_bf<A>(cs + sub * A, c);
                load_bf<A>(cs + H2 + sub * A, sn);
            } else {
                const float *cs = static_cast<const float *>(a.cos_sin) + pp * R;
                load_f32<A>(cs + sub * A, c);
                load_f32<A>(cs + H2 + sub * A, sn);
            }
        };
        const bool ok0 = accept(p, act[0]);
        load_cs(p);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            bool ok = ok0;
            if (j == 1 && (th[1] != th[0] || !act[1])) {  // the second head is another token's
                int64_t p1 = act[1] ? __ldg(a.pos + th[1]) : 0;
                ok = accept(p1, act[1]);
                load_cs(p1);
            }
            const uint16_t *wp = (hh[j] < static_cast<uint32_t>(a.Hq)) ? a.wq : a.wk;
            if constexpr (PACKED) {
                float2 acc = make_float2(0.f, 0.f), acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < A2; ++i) {
                    const float2 u = bf2f(x1[j][i]);
                    const float2 v = bf2f(x2[j][i]);
                    acc = __ffma2_rn(u, u, acc);
                    acc2 = __ffma2_rn(v, v, acc2);
                }
                if constexpr (B > 0) {
#pragma unroll
                    for (int i = 0; i < B2; ++i) {
                        const float2 u = bf2f(x3[j][i]);
                        if (i & 1)
                            acc2 = __ffma2_rn(u, u, acc2);
                        else
                            acc = __ffma2_rn(u, u, acc);
                    }
                }
                const float ss = group_sum<LPH>((acc.x + acc.y) + (acc2.x + acc2.y));
                // D is a power of two: multiplying by 1/D is the exact division.
                const float rstd = __frsqrt_rn(ss * (1.0f / static_cast<float>(D)) + a.eps);
                uint32_t w1[A2], w2[A2], w3[B2];
                load_words<A>(wp + off1, w1);
                load_words<A>(wp + off2, w2);
                if constexpr (B > 0) load_words<B>(wp + R + sub * B, w3);
                uint32_t o1[A2], o2[A2], o3[B2];
                qk_rotate<STYLE, A2, B2, (B > 0)>(x1[j], x2[j], x3[j], w1, w2, w3, c, sn, rstd, o1,
                                                 o2, o3);
                if (ok) {
                    store_words<A>(head[j] + off1, o1);
                    store_words<A>(head[j] + off2, o2);
                    if constexpr (B > 0) store_words<B>(head[j] + R + sub * B, o3);
                }
            } else {
                // qk_norm_rope_kernel's arithmetic, element by element
                float e1[A], e2[A];
#pragma unroll
                for (int i = 0; i < A; ++i) {
                    if constexpr (STYLE == 0) {
                        e1[i] = (i & 1) ? bf_hi(x1[j][i / 2]) : bf_lo(x1[j][i / 2]);
                        e2[i] = (i & 1) ? bf_hi(x2[j][i / 2]) : bf_lo(x2[j][i / 2]);
                    } else {  // word i of the lane's 2A-run is the pair (x1, x2) of element i
                        const uint32_t w = i < A2 ? x1[j][i] : x2[j][i - A2];
                        e1[i] = bf_lo(w);
                        e2[i] = bf_hi(w);
                    }
                }
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < A; ++i) ss = fmaf(e2[i], e2[i], fmaf(e1[i], e1[i], ss));
                if constexpr (B > 0) {
#pragma unroll
                    for (int i = 0; i < B2; ++i) {
                        const float lo = bf_lo(x3[j][i]), hi = bf_hi(x3[j][i]);
                        ss = fmaf(hi, hi, fmaf(lo, lo, ss));
                    }
                }
                ss = group_sum<LPH>(ss);
                const float rstd = __frsqrt_rn(ss / static_cast<float>(D) + a.eps);
                float w1[A], w2[A];
                if constexpr (STYLE == 0) {
                    load_bf<A>(wp + sub * A, w1);
                    load_bf<A>(wp + H2 + sub * A, w2);
                } else {
                    float wr[2 * A];
                    load_bf<2 * A>(wp + sub * 2 * A, wr);
#pragma unroll
                    for (int i = 0; i < A; ++i) {
                        w1[i] = wr[2 * i];
                        w2[i] = wr[2 * i + 1];
                    }
                }
                float o1[A], o2[A];
#pragma unroll
                for (int i = 0; i < A; ++i) {
                    const float n1 = e1[i] * rstd * w1[i];
                    const float n2 = e2[i] * rstd * w2[i];
                    o1[i] = n1 * c[i] - n2 * sn[i];
                    o2[i] = n2 * c[i] + n1 * sn[i];
                }
                if (ok) {
                    if constexpr (STYLE == 0) {
                        store_bf<A>(head[j] + sub * A, o1);
                        store_bf<A>(head[j] + H2 + sub * A, o2);
                    } else {
                        float orr[2 * A];
#pragma unroll
                        for (int i = 0; i < A; ++i) {
                            orr[2 * i] = o1[i];
                            orr[2 * i + 1] = o2[i];
                        }
                        store_bf<2 * A>(head[j] + sub * 2 * A, orr);
                    }
                }
                if constexpr (B > 0) {
                    float w3[B], e3[B];
                    load_bf<B>(wp + R + sub * B, w3);
#pragma unroll
                    for (int i = 0; i < B2; ++i) {
                        e3[2 * i] = bf_lo(x3[j][i]) * rstd * w3[2 * i];
                        e3[2 * i + 1] = bf_hi(x3[j][i]) * rstd * w3[2 * i + 1];
                    }
                    if (ok) store_bf<B>(head[j] + R + sub * B, e3);
                }
            }
        }
    }
}

template <int D, int R, int STYLE, bool TB>
__global__ void __launch_bounds__(qk_bulk_consumers<D>() + 32, 1)
    qk_persistent_bulk_kernel(const QkBulkArgs args) {
    constexpr int LPH = 8;
    constexpr int HPW = 32 / LPH;
    constexpr int NT = qk_bulk_consumers<D>();
    constexpr int NW = NT / 32;
    constexpr int H2 = R / 2;
    constexpr int A = H2 / LPH;          // elements per lane per rotary half
    constexpr int B = (D - R) / LPH;     // tail elements per lane
    constexpr int A2 = A / 2;
    constexpr int B2 = B > 0 ? B / 2 : 1;
    static_assert(A * LPH == H2 && B * LPH == D - R && A % 2 == 0 && B % 2 == 0,
                  "bad lane layout");
    extern __shared__ __align__(128) uint8_t smem[];

    const QkArgs &a = args.q;
    const int S = args.stages;
    const int TPS = args.tps;
    const int Hq = a.Hq;
    const int H = a.Hq + a.Hkv;
    const uint32_t tok_bytes = static_cast<uint32_t>(H) * D * 2;
    const uint32_t cs_bytes = R * (TB ? 2 : 4);
    const uint32_t stage_bytes = static_cast<uint32_t>(TPS) * (tok_bytes + cs_bytes);
    const int64_t W = static_cast<int64_t>(a.Hq + 2 * a.Hkv) * D;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t *empty = full + S;
    volatile int *valid = reinterpret_cast<volatile int *>(empty + S);  // [S][TPS]
    volatile int *abort_flag = valid + S * TPS;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    pdl_trigger();
    pdl_wait();
    __syncthreads();

    const UnitSchedule sched(a.T, gridDim.x, TPS);
    const int64_t bid = blockIdx.x;
    const int64_t n_units = sched.units(bid);

    if (warp == NW) {
        // ---- producer warp ----
        const uint64_t pol = l2_policy_evict_first();
        int64_t p_next = 0;
        if (n_units > 0) {
            int64_t r0;
            int rows;
            sched.unit(bid, 0, &r0, &rows);
            if (lane < rows) p_next = __ldg(a.pos + r0 + lane);
        }
        int64_t k = 0;
        for (; k < n_units; ++k) {
            const int s = static_cast<int>(k % S);
            if (k >= S) {
                const uint32_t par = static_cast<uint32_t>((k / S - 1) & 1);
                const bool ok = __all_sync(
                    0xffffffffu, mbar_wait_bounded(&empty[s], par, args.timeout_ns, abort_flag));
                if (!ok) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        raise_qk_status(RN_STATUS_WAIT_TIMEOUT);
                    }
                    break;
                }
            }
            int64_t r0;
            int rows;
            sched.unit(bid, k, &r0, &rows);
            const int64_t p = p_next;
            if (k + 1 < n_units) {
                int64_t r1;
                int rows1;
                sched.unit(bid, k + 1, &r1, &rows1);
                if (lane < rows1) p_next = __ldg(a.pos + r1 + lane);
            }
            bool pos_ok = true;
            if (lane < rows) {
                if (a.max_pos > 0 && (p < 0 || p >= a.max_pos)) {
                    pos_ok = false;
                    atomicOr(a.err, RN_STATUS_BAD_POSITION);
                }
                valid[s * TPS + lane] = pos_ok ? 1 : 0;
            }
            __threadfence_block();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(rows) * (tok_bytes + cs_bytes));
            __syncwarp();
            if (lane < rows && !(args.debug & 1)) {
                uint8_t *st = ring + static_cast<size_t>(s) * stage_bytes;
                bulk_copy_g2s(st + lane * tok_bytes, a.qkv + (r0 + lane) * W, tok_bytes, &full[s],
                              pol);
                // A rejected position still completes the stage's byte count
                // (row 0 is copied); its token is flagged and never stored.
                bulk_copy_g2s_plain(st + static_cast<size_t>(TPS) * tok_bytes + lane * cs_bytes,
                                    static_cast<const uint8_t *>(a.cos_sin) +
                                        (pos_ok ? p : 0) * static_cast<int64_t>(cs_bytes),
                                    cs_bytes, &full[s]);
            }
        }
        if (lane == 0) {
            // Drain: every copy issued into this CTA's ring lands before exit.
            const int64_t issued = k;
            const uint64_t t0 = globaltimer_ns();
            for (int64_t kk = (issued > S ? issued - S : 0); kk < issued; ++kk) {
                const uint64_t spent = globaltimer_ns() - t0;
                const uint64_t budget = spent < args.timeout_ns ? args.timeout_ns - spent : 0;
                if (!mbar_wait_bounded(&full[kk % S], static_cast<uint32_t>((kk / S) & 1), budget,
                                       nullptr)) {
                    raise_qk_status(RN_STATUS_WAIT_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ---- consumer warps ----
    const int sub = lane % LPH;
    const int grp = lane / LPH;
    // Element offsets of the lane's two rotary pieces: neox takes A elements
    // from each half, GPT-J 2A contiguous elements (split in two A-runs).
    const int off1 = STYLE == 0 ? sub * A : sub * 2 * A;
    const int off2 = STYLE == 0 ? H2 + sub * A : sub * 2 * A + A;
    uint32_t wq1[A2], wq2[A2], wq3[B2], wk1[A2], wk2[A2], wk3[B2];
    load_words<A>(a.wq + off1, wq1);
    load_words<A>(a.wq + off2, wq2);
    load_words<A>(a.wk + off1, wk1);
    load_words<A>(a.wk + off2, wk2);
    if constexpr (B > 0) {
        load_words<B>(a.wq + R + sub * B, wq3);
        load_words<B>(a.wk + R + sub * B, wk3);
    }

    for (int64_t k = 0; k < n_units; ++k) {
        const int s = static_cast<int>(k % S);
        const uint32_t par = static_cast<uint32_t>((k / S) & 1);
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait_bounded(&full[s], par, args.timeout_ns, abort_flag));
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1;
                raise_qk_status(RN_STATUS_WAIT_TIMEOUT);
            }
            break;
        }
        int64_t r0;
        int rows;
        sched.unit(bid, k, &r0, &rows);
        const uint8_t *st = ring + static_cast<size_t>(s) * stage_bytes;
        const uint8_t *cs_base = st + static_cast<size_t>(TPS) * tok_bytes;
        const int heads = rows * H;
        const int quads = (heads + HPW - 1) / HPW;
        for (int q = static_cast<int>((warp + k) % NW); q < quads; q += NW) {
            const uint32_t hh = static_cast<uint32_t>(q * HPW + grp);
            const bool act = hh < static_cast<uint32_t>(heads);
            const uint32_t ts =
                act ? static_cast<uint32_t>((static_cast<uint64_t>(hh) * args.inv_h) >> 32) : 0u;
            const uint32_t h = act ? hh - ts * H : 0u;
            const bool good = act && valid[s * TPS + ts] != 0;
            const uint16_t *xs =
                reinterpret_cast<const uint16_t *>(st + ts * tok_bytes) + static_cast<size_t>(h) * D;
            uint32_t x1[A2], x2[A2], x3[B2];
            load_words<A>(xs + off1, x1);
            load_words<A>(xs + off2, x2);
            if constexpr (B > 0) load_words<B>(xs + R + sub * B, x3);
            float c[A], sn[A];
            if constexpr (TB) {
                // 8 lanes read one 2A-byte run each, one contiguous span: no
                // bank is shared within a phase, so no reordering is needed.
                const uint16_t *cs = reinterpret_cast<const uint16_t *>(cs_base) + ts * R;
                load_bf<A>(cs + sub * A, c);
                load_bf<A>(cs + H2 + sub * A, sn);
            } else {
                const float *cs = reinterpret_cast<const float *>(cs_base) + ts * R;
                load_f32_smem_lanes<A>(cs + sub * A, c, sub);
                load_f32_smem_lanes<A>(cs + H2 + sub * A, sn, sub);
            }

            // two independent accumulators: half the dependent FMA chain
            float2 acc = make_float2(0.f, 0.f), acc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < A2; ++i) {
                const float2 u = bf2f(x1[i]);
                const float2 v = bf2f(x2[i]);
                acc = __ffma2_rn(u, u, acc);
                acc2 = __ffma2_rn(v, v, acc2);
            }
            if constexpr (B > 0) {
#pragma unroll
                for (int i = 0; i < B2; ++i) {
                    const float2 u = bf2f(x3[i]);
                    if (i & 1)
                        acc2 = __ffma2_rn(u, u, acc2);
                    else
                        acc = __ffma2_rn(u, u, acc);
                }
            }
            const float ss = group_sum<LPH>((acc.x + acc.y) + (acc2.x + acc2.y));
            // D is a power of two: multiplying by 1/D is the exact division.
            const float rstd = __frsqrt_rn(ss * (1.0f / static_cast<float>(D)) + a.eps);
            const bool isq = h < static_cast<uint32_t>(Hq);
            uint32_t o1[A2], o2[A2], o3[B2];
            // The quad's heads are usually all query or all key heads: pick the
            // weights once for the warp instead of element by element.
            if (__all_sync(0xffffffffu, isq || !act)) {
                qk_rotate<STYLE, A2, B2, (B > 0)>(x1, x2, x3, wq1, wq2, wq3, c, sn, rstd, o1, o2, o3);
            } else if (__all_sync(0xffffffffu, !isq || !act)) {
                qk_rotate<STYLE, A2, B2, (B > 0)>(x1, x2, x3, wk1, wk2, wk3, c, sn, rstd, o1, o2, o3);
            } else {
                uint32_t w1[A2], w2[A2], w3[B2];
#pragma unroll
                for (int i = 0; i < A2; ++i) {
                    w1[i] = isq ? wq1[i] : wk1[i];
                    w2[i] = isq ? wq2[i] : wk2[i];
                }
#pragma unroll
                for (int i = 0; i < B2; ++i) w3[i] = isq ? wq3[i] : wk3[i];
                qk_rotate<STYLE, A2, B2, (B > 0)>(x1, x2, x3, w1, w2, w3, c, sn, rstd, o1, o2, o3);
            }
            if (good) {
                uint16_t *head = a.qkv + (r0 + ts) * W + static_cast<int64_t>(h) * D;
                store_words<A>(head + off1, o1);
                store_words<A>(head + off2, o2);
                if constexpr (B > 0) store_words<B>(head + R + sub * B, o3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// ---- table builder ----------------------------------------------------------------

// fp64 angle and trig, rounded once to the table's element type (fp32, or
// bf16 straight from the double: going through fp32 would round twice).
__device__ __forceinline__ void put_table(float *p, double v) { *p = __double2float_rn(v); }
__device__ __forceinline__ void put_table(uint16_t *p, double v) {
    const __nv_bfloat16 b = __double2bfloat16(v);
    *p = *reinterpret_cast<const uint16_t *>(&b);
}

template <class OUT>
__global__ void rope_table_kernel(double theta, int64_t max_pos, int r, OUT *out) {
    pdl_trigger();
    pdl_wait();
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
        put_table(out + p * r + i, cv);
        put_table(out + p * r + h + i, sv);
    }
}

// ---- host side ----------------------------------------------------------------------

template <int D, int R, int LPH, int STYLE, bool TB>
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
    return launch_pdl(qk_norm_rope_kernel<D, R, LPH, STYLE, TB>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kThreads), 0, st, a);
}

// Lanes per head of qk_pair_kernel: 16-byte rotary pieces a lane.
template <int D>
constexpr int pair_lph() { return D == 64 ? 4 : (D == 128 ? 8 : 16); }

// Two heads per lane group (qk_pair_kernel) on a grid of two whole waves:
// SMs x twice the CTAs an SM holds at once.  Grids that are not a whole
// number of waves measured 3-10% slower at 2048-4096 tokens, and one wave
// loses at 4096 tokens: with two, the second wave's CTAs take the place of
// whichever finish first, which evens out the SMs' unequal rates.
template <int D, int R, int STYLE, bool TB>
static int launch_qk_pairs(const QkArgs &a, cudaStream_t st, const DeviceInfo &dev) {
    constexpr int LPH = pair_lph<D>();
    static std::atomic<int> fit_cache[kMaxDevices];
    const int dev_idx = current_device_index();
    if (dev_idx < 0 || dev_idx >= kMaxDevices) return RN_ERR_DEVICE;
    int fit = fit_cache[dev_idx].load(std::memory_order_acquire);
    if (fit <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, qk_pair_kernel<D, R, LPH, STYLE, TB>,
                                                          256, 0) != cudaSuccess || fit <= 0) {
            cudaGetLastError();
            return RN_ERR_DEVICE;
        }
        fit_cache[dev_idx].store(fit, std::memory_order_release);
    }
    const uint64_t total = static_cast<uint64_t>(a.T) * static_cast<uint64_t>(a.Hq + a.Hkv);
    const uint64_t per_block = 8 * 2 * (32 / LPH);  // 8 warps x 2 heads a group a round
    uint64_t blocks = (total + per_block - 1) / per_block;
    const uint64_t cap = static_cast<uint64_t>(dev.sm_count) * 2 * static_cast<uint64_t>(fit);
    if (blocks > cap) blocks = cap;
    return launch_pdl(qk_pair_kernel<D, R, LPH, STYLE, TB>, dim3(static_cast<unsigned>(blocks)),
                      dim3(256), 0, st, a);
}

// Largest lanes-per-head <= the request that tiles both rotary halves and
// the tail of this (D, rotary_dim); 8 always does.
template <int D, int R, int STYLE, bool TB>
static int launch_qk_lph(const QkArgs &a, int lph, bool persistent, cudaStream_t st,
                         const DeviceInfo &dev) {
    constexpr int H2 = R / 2;
    if constexpr (H2 % 32 == 0 && (D - R) % 32 == 0) {
        if (lph >= 32) return launch_qk<D, R, 32, STYLE, TB>(a, persistent, st, dev);
    }
    if constexpr (H2 % 16 == 0 && (D - R) % 16 == 0) {
        if (lph >= 16) return launch_qk<D, R, 16, STYLE, TB>(a, persistent, st, dev);
    }
    if constexpr (H2 % 8 == 0 && (D - R) % 8 == 0) {
        return launch_qk<D, R, 8, STYLE, TB>(a, persistent, st, dev);
    }
    return RN_ERR_SHAPE;
}

template <int D, int R, int STYLE, bool TB>
static int launch_qk_bulk(const QkArgs &a, cudaStream_t st, const DeviceInfo &dev,
                          uint64_t timeout_ns, int debug_flags) {
    static std::atomic<int> attr_done[kMaxDevices];
    const int H = a.Hq + a.Hkv;
    const int tok_bytes = H * D * 2;
    const int cs_bytes = R * (TB ? 2 : 4);
    // About 32 KiB a stage; 44 KiB when the rotation spans the whole head,
    // whose consumers hold a stage longer (more arithmetic per token): 4
    // tokens a stage instead of 3 at D = 128, measured on GB300.
    int tps = (R == D ? 45056 : 32768) / (tok_bytes + cs_bytes);
    const int forced_tps = (debug_flags >> 16) & 0x3F;
    if (forced_tps > 0) tps = forced_tps;
    if (tps < 1) tps = 1;
    if (tps > 32) tps = 32;
    // Consumers hold a stage while they compute, so four stages keep about
    // three in flight.
    int stages = 4;
    const int forced = (debug_flags >> 8) & 0x1F;
    if (forced >= 2) stages = forced;
    const int smem_cap = dev.max_smem_optin < 232448 ? dev.max_smem_optin : 232448;
    // a forced stage count takes precedence over the stage size
    while (tps > 1 && qk_bulk_smem_bytes(stages, tps, tok_bytes, cs_bytes) > static_cast<size_t>(smem_cap))
        --tps;
    const size_t smem = qk_bulk_smem_bytes(stages, tps, tok_bytes, cs_bytes);
    if (smem > static_cast<size_t>(smem_cap)) return RN_ERR_SHAPE;
    const int dev_idx = current_device_index();
    if (dev_idx < 0 || dev_idx >= kMaxDevices) return RN_ERR_DEVICE;
    if (!attr_done[dev_idx].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(qk_persistent_bulk_kernel<D, R, STYLE, TB>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_cap) != cudaSuccess) {
            cudaGetLastError();
            return RN_ERR_DEVICE;
        }
        attr_done[dev_idx].store(1, std::memory_order_release);
    }
    int64_t grid = dev.sm_count;
    if (grid > a.T) grid = a.T;
    const uint64_t inv_h = ((1ull << 32) + H - 1) / H;
    QkBulkArgs b{a, tps, stages, debug_flags & 1, inv_h, timeout_ns ? timeout_ns : 2000000000ull};
    return launch_pdl(qk_persistent_bulk_kernel<D, R, STYLE, TB>, dim3(static_cast<unsigned>(grid)),
                      dim3(qk_bulk_consumers<D>() + 32), smem, st, b);
}

// Schedule by token count and layout (measured on GB300 in steady state,
// back-to-back launches, positions uniform over 131072 rows): one head per
// warp for 1-2 tokens, two heads per warp through 256 tokens; beyond that the
// bulk-copy token ring above `ring_above` tokens (its deeper prefetch pays
// for its longer start-up), else the pairs (qk_pair_kernel) from `pairs_from`
// through `pairs_upto` tokens, else four heads per warp on a persistent grid.
//   D 128: the pairs lead the four-heads grid by 3-15% from 1024 tokens at
//     rotary 128 and 64 (within 2% at 1536, rotary 64) and from 1792 at
//     rotary 32, and the ring by 4-10% through 5120 tokens (4608 at rotary
//     64); from 6144 they are even, and the ring leads from 8192-12288.
//   D 64: the pairs lead from 1024 tokens (3072 at rotary 16) at every count
//     up to 65536 (0.82-0.91 of the copy from 4096 on, rotary 64); the ring
//     stays behind them (tokens of 5 KB: 0.54-0.74).
//   D 256: the pairs lead from the first persistent counts at rotary 256 and
//     128 (rotary 256: 0.94 at 4096 tokens, 0.93 at 65536; the ring 0.57 and
//     0.71), the ring from 8192 at rotary 128; at rotary 64 the pairs lead
//     from 512 to 4096 and the four-heads grid beyond (0.86-0.97).
struct QkRule {
    int D, r;
    int64_t pairs_from;  // 0: never
    int64_t pairs_upto;  // 0: no limit
    int64_t ring_above;  // 0: never
};
static constexpr QkRule kQkRules[] = {
    {64, 64, 1024, 0, 0},       {64, 32, 1024, 0, 0},       {64, 16, 3072, 0, 0},
    {128, 128, 1024, 0, 5120},  {128, 64, 1024, 0, 4096},  {128, 32, 1792, 0, 5120},
    {256, 256, 1, 0, 0},        {256, 128, 1, 0, 6144},    {256, 64, 512, 4096, 0},
};

// RN_ERR_SHAPE for a layout no schedule serves.
static int auto_qk_schedule(int64_t T, int D, int r) {
    const QkRule *rule = nullptr;
    for (const QkRule &q : kQkRules)
        if (q.D == D && q.r == r) rule = &q;
    if (!rule) return RN_ERR_SHAPE;
    if (T <= 2) return RN_QK_HEAD_PER_WARP;
    if (T <= 256) return RN_QK_TWO_HEADS;
    if (rule->ring_above > 0 && T > rule->ring_above) return RN_QK_BULK;
    if (rule->pairs_from > 0 && T >= rule->pairs_from &&
        (rule->pairs_upto == 0 || T <= rule->pairs_upto))
        return RN_QK_PAIRS;
    return RN_QK_PERSISTENT;
}

template <int STYLE, bool TB>
static int qk_launch(const QkArgs &a, int D, int r, int schedule, bool automatic, int lph,
                     bool persistent, cudaStream_t st, const DeviceInfo &dev,
                     uint64_t timeout_ns, int debug_flags) {
    if (schedule == RN_QK_BULK) {
        int rc = RN_ERR_SHAPE;
#define RN_QK_BULK_GO(D_, R_)                                                           \
    if (D == (D_) && r == (R_))                                                         \
        rc = launch_qk_bulk<D_, R_, STYLE, TB>(a, st, dev, timeout_ns, debug_flags);
        // (64, 16) leaves one element per lane per half: the warp schedules serve it.
        RN_QK_BULK_GO(64, 64) RN_QK_BULK_GO(64, 32)
        RN_QK_BULK_GO(128, 128) RN_QK_BULK_GO(128, 64) RN_QK_BULK_GO(128, 32)
        RN_QK_BULK_GO(256, 256) RN_QK_BULK_GO(256, 128) RN_QK_BULK_GO(256, 64)
#undef RN_QK_BULK_GO
        if (rc != RN_ERR_SHAPE || !automatic) return rc;
        persistent = true;  // a token too wide for the ring: the warp grid serves it
    }
    if (schedule == RN_QK_PAIRS) {
#define RN_QK_PAIRS_GO(D_, R_) \
    if (D == (D_) && r == (R_)) return launch_qk_pairs<D_, R_, STYLE, TB>(a, st, dev);
        RN_QK_PAIRS_GO(64, 64) RN_QK_PAIRS_GO(64, 32) RN_QK_PAIRS_GO(64, 16)
        RN_QK_PAIRS_GO(128, 128) RN_QK_PAIRS_GO(128, 64) RN_QK_PAIRS_GO(128, 32)
        RN_QK_PAIRS_GO(256, 256) RN_QK_PAIRS_GO(256, 128) RN_QK_PAIRS_GO(256, 64)
#undef RN_QK_PAIRS_GO
        return RN_ERR_SHAPE;
    }
#define RN_QK_GO(D_, R_)                                                               \
    if (D == (D_) && r == (R_)) return launch_qk_lph<D_, R_, STYLE, TB>(a, lph, persistent, st, dev);
    RN_QK_GO(64, 64) RN_QK_GO(64, 32) RN_QK_GO(64, 16)
    RN_QK_GO(128, 128) RN_QK_GO(128, 64) RN_QK_GO(128, 32)
    RN_QK_GO(256, 256) RN_QK_GO(256, 128) RN_QK_GO(256, 64)
#undef RN_QK_GO
    return RN_ERR_SHAPE;
}

// `cos_sin` holds fp32 entries, or bf16 ones when table_bf16.
static int qk_dispatch(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                       const void *cos_sin, const int64_t *positions, int64_t T, int Hq,
                       int Hkv, int D, int rotary_dim, float eps, int64_t max_pos, int *err,
                       int schedule, uint64_t timeout_ns, int debug_flags, rn_stream_t stream,
                       int style = RN_ROPE_NEOX, bool table_bf16 = false) {
    if (style != RN_ROPE_NEOX && style != RN_ROPE_GPTJ) return RN_ERR_ARG;
    if (T < 0 || Hq < 0 || Hkv < 0) return RN_ERR_SHAPE;
    if (D != 64 && D != 128 && D != 256) return RN_ERR_SHAPE;
    if (rotary_dim != D && rotary_dim != D / 2 && rotary_dim != D / 4) return RN_ERR_SHAPE;
    if (static_cast<uint64_t>(T) * static_cast<uint64_t>(Hq + Hkv) >= (1ull << 31))
        return RN_ERR_SHAPE;
    if (T == 0 || Hq + Hkv == 0) return RN_OK;
    if (!qkv || !wq || !wk || !cos_sin || !positions) return RN_ERR_NULL;
    // positions are read one int64 at a time: 8-byte alignment suffices
    if (!aligned16(qkv) || !aligned16(wq) || !aligned16(wk) || !aligned16(cos_sin) ||
        (reinterpret_cast<uintptr_t>(positions) & 7u) != 0)
        return RN_ERR_ALIGN;
    int lph;
    bool persistent = false;
    const bool automatic = schedule == RN_QK_AUTO;
    if (automatic) {
        schedule = auto_qk_schedule(T, D, rotary_dim);
        if (schedule < 0) return schedule;
    }
    switch (schedule) {
        case RN_QK_HEAD_PER_WARP: lph = 32; break;
        case RN_QK_TWO_HEADS: lph = 16; break;
        case RN_QK_FOUR_HEADS: lph = 8; break;
        case RN_QK_PERSISTENT: lph = 8; persistent = true; break;
        case RN_QK_BULK: lph = 8; break;
        case RN_QK_PAIRS: lph = 8; persistent = true; break;
        default: return RN_ERR_ARG;
    }
    const DeviceInfo *dev = current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    QkArgs a{reinterpret_cast<uint16_t *>(qkv), wq, wk, cos_sin, positions, T, Hq, Hkv,
             eps, max_pos, err};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
#define RN_QK_STYLE(S_, TB_)                                                                \
    return qk_launch<S_, TB_>(a, D, rotary_dim, schedule, automatic, lph, persistent, st, *dev, \
                              timeout_ns, debug_flags)
    if (style == RN_ROPE_GPTJ) {
        if (table_bf16) RN_QK_STYLE(1, true);
        RN_QK_STYLE(1, false);
    }
    if (table_bf16) RN_QK_STYLE(0, true);
    RN_QK_STYLE(0, false);
#undef RN_QK_STYLE
}

int qk_status(unsigned int *out, int clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_qk_status, sizeof v) != cudaSuccess) {
        cudaGetLastError();
        return RN_ERR_DEVICE;
    }
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_qk_status, &zero, sizeof zero) != cudaSuccess) {
            cudaGetLastError();
            return RN_ERR_DEVICE;
        }
    }
    *out = v;
    return RN_OK;
}

}  // namespace rn

extern "C" {

int qk_norm_rope_fwd(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk, const float *cos_sin,
                     const int64_t *positions, int64_t T, int Hq, int Hkv, int D,
                     int rotary_dim, float eps, rn_stream_t stream) {
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps, 0,
                           nullptr, RN_QK_AUTO, 0, 0, stream);
}

int qk_norm_rope_fwd_sched(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                           const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                           int Hkv, int D, int rotary_dim, float eps, int schedule,
                           uint64_t wait_timeout_ns, int debug_flags, rn_stream_t stream) {
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps, 0,
                           nullptr, schedule, wait_timeout_ns, debug_flags, stream);
}

int qk_norm_rope_fwd_checked(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                             const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                             int Hkv, int D, int rotary_dim, float eps, int64_t max_pos,
                             int *d_err_flag, rn_stream_t stream) {
    if (max_pos < 1) return RN_ERR_SHAPE;
    if (!d_err_flag && T > 0 && Hq + Hkv > 0) return RN_ERR_NULL;
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                           max_pos, d_err_flag, RN_QK_AUTO, 0, 0, stream);
}

int qk_norm_rope_fwd_ex(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                        const float *cos_sin, const int64_t *positions, int64_t T, int Hq,
                        int Hkv, int D, int rotary_dim, float eps, int rope_style,
                        int64_t max_pos, int *d_err_flag, int schedule,
                        uint64_t wait_timeout_ns, int debug_flags, rn_stream_t stream) {
    if (max_pos < 0) return RN_ERR_SHAPE;
    if (max_pos > 0 && !d_err_flag && T > 0 && Hq + Hkv > 0) return RN_ERR_NULL;
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                           max_pos, d_err_flag, schedule, wait_timeout_ns, debug_flags, stream,
                           rope_style);
}

int qk_norm_rope_fwd_ex_bf16_table(rn_bf16 *qkv, const rn_bf16 *wq, const rn_bf16 *wk,
                                   const rn_bf16 *cos_sin, const int64_t *positions, int64_t T,
                                   int Hq, int Hkv, int D, int rotary_dim, float eps,
                                   int rope_style, int64_t max_pos, int *d_err_flag, int schedule,
                                   uint64_t wait_timeout_ns, int debug_flags, rn_stream_t stream) {
    if (max_pos < 0) return RN_ERR_SHAPE;
    if (max_pos > 0 && !d_err_flag && T > 0 && Hq + Hkv > 0) return RN_ERR_NULL;
    return rn::qk_dispatch(qkv, wq, wk, cos_sin, positions, T, Hq, Hkv, D, rotary_dim, eps,
                           max_pos, d_err_flag, schedule, wait_timeout_ns, debug_flags, stream,
                           rope_style, true);
}

int qk_norm_rope_select_schedule(int64_t T) {
    if (T < 0) return RN_ERR_SHAPE;
    return rn::auto_qk_schedule(T, 128, 128);
}

int qk_norm_rope_select_schedule_ex(int64_t T, int D, int rotary_dim) {
    if (T < 0) return RN_ERR_SHAPE;
    return rn::auto_qk_schedule(T, D, rotary_dim);
}

}  // extern "C"

namespace rn {

template <class OUT>
static int build_rope_table(double theta, int64_t max_pos, int rotary_dim, OUT *cos_sin,
                            rn_stream_t stream) {
    if (max_pos < 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0.0))
        return RN_ERR_SHAPE;
    if (max_pos == 0) return RN_OK;
    if (!cos_sin) return RN_ERR_NULL;
    if (!aligned16(cos_sin)) return RN_ERR_ALIGN;
    const DeviceInfo *dev = current_device_info();
    if (!dev) return RN_ERR_DEVICE;
    const int64_t n = max_pos * (rotary_dim / 2);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev->sm_count) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(rope_table_kernel<OUT>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                      reinterpret_cast<cudaStream_t>(stream), theta, max_pos, rotary_dim, cos_sin);
}

}  // namespace rn

extern "C" {

int rope_cos_sin_table(double theta, int64_t max_pos, int rotary_dim, float *cos_sin,
                       rn_stream_t stream) {
    return rn::build_rope_table(theta, max_pos, rotary_dim, cos_sin, stream);
}

// Host form: one column i at a time, so f_i = theta^(-2i/r) is evaluated once
// per column; every entry is the fp64 cos or sin of p * f_i rounded once to
// fp32 (a C++ double -> float conversion rounds to nearest, ties to even).
int rope_cos_sin_table_host(double theta, int64_t max_pos, int rotary_dim, float *cos_sin_host) {
    if (max_pos < 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0.0)) return RN_ERR_SHAPE;
    if (max_pos == 0) return RN_OK;
    if (!cos_sin_host) return RN_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(cos_sin_host) & 3u) return RN_ERR_ALIGN;
    const int h = rotary_dim / 2;
    for (int i = 0; i < h; ++i) {
        const double f = std::pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(rotary_dim));
        float *col = cos_sin_host + i;
        for (int64_t p = 0; p < max_pos; ++p) {
            const double ang = static_cast<double>(p) * f;
            col[p * rotary_dim] = static_cast<float>(std::cos(ang));
            col[p * rotary_dim + h] = static_cast<float>(std::sin(ang));
        }
    }
    return RN_OK;
}

int rope_cos_sin_table_bf16(double theta, int64_t max_pos, int rotary_dim, rn_bf16 *cos_sin,
                            rn_stream_t stream) {
    return rn::build_rope_table(theta, max_pos, rotary_dim, reinterpret_cast<uint16_t *>(cos_sin),
                                stream);
}

}  // extern "C"
