// rn_common.cuh -- device helpers shared by the row-normalization kernels.
//
// The 16-bit element formats (bf16, IEEE fp16) with their mixed-precision
// operations, 16-byte global accesses, programmatic-dependent-launch hooks
// and the launch helper, and thin inline-PTX wrappers for the
// Hopper/Blackwell asynchronous-copy machinery the persistent schedules use:
// mbarriers (arrive, expect-tx, parity wait) and 1D bulk copies
// (cp.async.bulk, global -> this CTA's shared memory, completion signalled on
// an mbarrier).  No tensor maps and no multicast.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/row_norm.h"

namespace rn {

// ---- bf16 <-> fp32 ----------------------------------------------------------

// Two bf16 packed in a 32-bit word -> two fp32 (exact: bf16 is the top half
// of a binary32).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two fp32 -> two bf16 rounded to nearest even, packed (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---- element formats -----------------------------------------------------------
// A 16-bit element format: widen the two halves of a packed word to fp32
// (exact) and narrow two fp32 back with one round-to-nearest-even.

// Besides widening and narrowing, each format offers three operations on the
// packed halves as mixed-precision instructions (16-bit operand, fp32 other
// operand and result; sm_100 and later), which fold the widening into the
// arithmetic and round exactly as widen-then-operate does:
//   sq_acc(acc, u)  acc + lo(u)^2 + hi(u)^2  (two fused multiply-adds; each
//                   square is exact in fp32);
//   pair_sum(u)     lo(u) + hi(u), rounded once;
//   sub2(u, m)      (lo(u) - m, hi(u) - m), each rounded once.

struct Bf16 {
    static constexpr uint32_t kOne2 = 0x3F803F80u;  // two 1.0
    __device__ static __forceinline__ float lo(uint32_t u) { return bf_lo(u); }
    __device__ static __forceinline__ float hi(uint32_t u) { return bf_hi(u); }
    __device__ static __forceinline__ uint32_t pack(float a, float b) { return pack_bf2(a, b); }
    __device__ static __forceinline__ float sq_acc(float acc, uint32_t u) {
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
            "fma.rn.f32.bf16 %0, l, l, %0;\n\tfma.rn.f32.bf16 %0, h, h, %0;\n\t}"
            : "+f"(acc) : "r"(u));
        return acc;
    }
    __device__ static __forceinline__ float pair_sum(uint32_t u) {
        float r;
        asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 t;\n\tmov.b32 {l, h}, %1;\n\t"
            "add.rn.f32.bf16 t, l, 0f80000000;\n\tadd.rn.f32.bf16 %0, h, t;\n\t}"
            : "=f"(r) : "r"(u));
        return r;
    }
    __device__ static __forceinline__ float2 sub2(uint32_t u, float m) {
        float2 r;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
            : "=f"(r.x), "=f"(r.y) : "r"(u), "f"(m));
        return r;
    }
};

// IEEE binary16: overflow rounds to infinity, subnormals are kept.
struct F16 {
    static constexpr uint32_t kOne2 = 0x3C003C00u;  // two 1.0
    // widening as a mixed-precision add of -0 (exact, signs and specials
    // kept), which measured faster than the conversion instruction
    __device__ static __forceinline__ float lo(uint32_t u) {
        float r;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, l, 0f80000000;\n\t}"
            : "=f"(r) : "r"(u));
        return r;
    }
    __device__ static __forceinline__ float hi(uint32_t u) {
        float r;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, h, 0f80000000;\n\t}"
            : "=f"(r) : "r"(u));
        return r;
    }
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __device__ static __forceinline__ float sq_acc(float acc, uint32_t u) {
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
            "fma.rn.f32.f16 %0, l, l, %0;\n\tfma.rn.f32.f16 %0, h, h, %0;\n\t}"
            : "+f"(acc) : "r"(u));
        return acc;
    }
    __device__ static __forceinline__ float pair_sum(uint32_t u) {
        float r;
        asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 t;\n\tmov.b32 {l, h}, %1;\n\t"
            "add.rn.f32.f16 t, l, 0f80000000;\n\tadd.rn.f32.f16 %0, h, t;\n\t}"
            : "=f"(r) : "r"(u));
        return r;
    }
    __device__ static __forceinline__ float2 sub2(uint32_t u, float m) {
        float2 r;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "sub.rn.f32.f16 %0, l, %3;\n\tsub.rn.f32.f16 %1, h, %3;\n\t}"
            : "=f"(r.x), "=f"(r.y) : "r"(u), "f"(m));
        return r;
    }
};

// ---- programmatic dependent launch ---------------------------------------------
// Every kernel here is launched with programmatic stream serialisation: its
// CTAs may be scheduled while the previous launch in the stream is still
// finishing, which hides the launch gap between back-to-back kernels.  Each
// kernel lets its own successor do the same (pdl_trigger) and then waits,
// before its first global memory access, until the previous launch has
// completed and its writes are visible (pdl_wait).  Both are no-ops when the
// neighbouring launch does not take part.

__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` with programmatic stream serialisation; RN_OK or
// RN_ERR_LAUNCH.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return RN_ERR_LAUNCH;
    }
    return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_LAUNCH;
}

// ---- global memory ----------------------------------------------------------

// Read-once 16-byte load (streaming: evict first from L1/L2).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
// Read-only 16-byte load that may be reused (weights): normal caching.
__device__ __forceinline__ uint4 ld_ro16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st16(void *p, uint4 v) {
    *reinterpret_cast<uint4 *>(p) = v;
}

// ---- reductions ---------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over aligned groups of G lanes (G a power of two <= 32).
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- shared memory / mbarrier / bulk copy -------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (the bulk-copy
// engine) before any copy is issued against it.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Parity wait with a wall-clock limit.  Returns false if the limit ran out or
// *abort became non-zero (another role gave up) before the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns,
                                                  const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// 1D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; completion is counted on
// `bar` as transaction bytes.  Evict-first L2 policy: each byte is read once.
__device__ __forceinline__ void bulk_copy_g2s(void *dst_smem, const void *src_gmem,
                                              uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Named barrier over `nthreads` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 ld_shared16(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Which rows (or tokens) the k-th unit of persistent CTA b covers.  Units go round-robin: round q
// gives CTA b rows [q*G*R + b*R, +R), so at any moment the grid streams one
// contiguous band of memory.  A last, partial round is re-split evenly (rows
// per CTA ceil(rem / G)) so no CTA is left with a whole extra unit.
struct UnitSchedule {
    int64_t full_rounds;  // rounds in which every CTA gets R rows
    int64_t rem;          // rows left for the final round
    int64_t last_r;       // rows per CTA in the final round
    int64_t G;
    int R;

    __device__ __forceinline__ UnitSchedule(int64_t M, int64_t G_, int R_) : G(G_), R(R_) {
        full_rounds = M / (G * R);
        rem = M - full_rounds * G * R;
        last_r = (rem + G - 1) / G;
    }
    __device__ __forceinline__ int64_t units(int64_t b) const {
        return full_rounds + ((rem > 0 && b * last_r < rem) ? 1 : 0);
    }
    __device__ __forceinline__ void unit(int64_t b, int64_t k, int64_t *r0, int *rows) const {
        if (k < full_rounds) {
            *r0 = k * G * R + b * R;
            *rows = R;
        } else {
            *r0 = full_rounds * G * R + b * last_r;
            const int64_t left = rem - b * last_r;
            *rows = static_cast<int>(left < last_r ? left : last_r);
        }
    }
};

// Dynamic unit order of a persistent grid (the row ring).  CTA b takes its first `lead`
// units statically (unit k * G + b for k < lead) and every later one from a
// counter in the caller's workspace: ws[0] counts the units handed out after
// the static ones, so a CTA whose SM streams faster takes more of them and
// all CTAs finish within about a stage of each other.  (Under a fixed
// round-robin some SMs of a GB300 finish up to 15% later than the rest.)
// The static lead is about 70% of a CTA's fair share (and at least the ring
// depth): the dynamic rest absorbs such a spread, and the CTAs reach the
// counter spread out in time rather than all at once.  ws[1] counts the
// producers that have finished; the last one sets both words back to zero,
// so the workspace is zero again when the grid completes, and the next
// launch that uses it touches it only after that completion (stream order,
// or griddepcontrol.wait under programmatic dependent launch).
struct DynUnits {
    unsigned long long *ws;
    int64_t G;
    int64_t b;
    int64_t lead;

    __device__ __forceinline__ DynUnits(unsigned long long *ws_, int64_t G_, int64_t b_,
                                        int64_t total_units, int stages)
        : ws(ws_), G(G_), b(b_) {
        const int64_t share = total_units * 7 / (10 * G_);
        lead = share > stages ? share : stages;
    }

    __device__ __forceinline__ int64_t first(int64_t k) const { return k * G + b; }
    // The next unit after the static ones (atomic: the caller should issue it
    // early and use the result late, to hide the round trip).
    __device__ __forceinline__ int64_t fetch() const {
        return lead * G + static_cast<int64_t>(atomicAdd(ws, 1ull));
    }
    // Called once by every CTA's producer after its last fetch.
    __device__ __forceinline__ void finish() const {
        if (atomicAdd(ws + 1, 1ull) == static_cast<unsigned long long>(G - 1)) {
            atomicExch(ws, 0ull);
            atomicExch(ws + 1, 0ull);
        }
    }
};

}  // namespace rn
