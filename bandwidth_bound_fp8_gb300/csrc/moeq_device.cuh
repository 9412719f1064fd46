// Device-side building blocks shared by the libmoeq kernels (sm_103a):
// inline-PTX wrappers for mbarriers, TMA bulk-tensor loads, the global timer,
// and the E4M3 conversions, plus the per-group live activation quantiser.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeq.h"

namespace moeq {

constexpr int kGroup = MOEQ_GROUP;
constexpr int kMaxTok = MOEQ_MAX_TOKENS;
// Bounded waits: a wait that has not finished after this long records
// MOEQ_ERR_TIMEOUT in the device status word and gives up.
constexpr unsigned long long kWaitLimitNs = 2000ull * 1000ull * 1000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete sleeps (up to
// kSleepHintNs, woken early when the phase completes) instead of returning at
// once: a waiting warp takes no issue slots from the warps that work.
constexpr uint32_t kSleepHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepHintNs)
        : "memory");
    return done != 0;
}

// Sleeping wait for the phase with the given parity; gives up (returns
// false) when *abort becomes non-zero or after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) when *abort becomes non-zero or after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// Start a global line on its way into L2 (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Starts `bytes` (multiple of 16, 16-byte aligned) of global memory on its
// way into L2 with a bulk copy that has no destination.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// fp32 store with an L2 eviction-priority hint.
__device__ __forceinline__ void st_global_hint(float* p, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16, 16-byte aligned ends) into
// shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation (warp-collective), 1-CTA MMAs of kind::f8f6f4 and
// loads of the fp32 accumulators, as inline PTX.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes, 8-row atoms of 1024 bytes (1024-aligned),
// 16-byte chunk c of row r at chunk c ^ (r % 8).  Advancing the start address
// by 32 bytes selects the next K = 32 slice of the atom.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    uint64_t d = static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;             // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride byte offset: one 8-row atom
    d |= static_cast<uint64_t>(1) << 46;             // descriptor version
    d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B E4M3, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// The mbarrier completes one arrival when every MMA issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// N consecutive fp32 columns (N = 4, 8 or 16) of this thread's TMEM lane
// (warp w reads lanes 32*(w%4) ..), without waiting: the registers are valid
// after tmem_wait_ld, so several loads can overlap.
template <int N>
__device__ __forceinline__ void tmem_ld_nowait(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else {
        static_assert(N == 16, "tmem_ld_nowait: 4, 8 or 16 columns");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// gpu-scope acquire load / release store of a flag in global memory.
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// gpu-scope atomic add with acquire-release semantics; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Orders generic-proxy memory accesses with async-proxy (bulk copy) ones.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
// The same, for global memory only: generic writes (or reads acquired) in
// global memory ordered against bulk copies that read it.  The unqualified
// fence also covers shared memory, where this CTA's own bulk copies may be
// landing, and costs more while they are in flight.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Named barrier over the consumer warps only (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- E4M3
// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448.
// Returns (code(hi) << 8) | code(lo).
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (low byte first) -> two exact fp16 values.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    __half2 v = *reinterpret_cast<__half2*>(&h);
    return __half22float2(v);
}

// Four E4M3 codes packed in a u32 (byte 0 = lowest k) -> four exact floats.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float2& a, float2& b) {
    a = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xFFFFu)));
    b = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16)));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Load 4 consecutive activation elements (k .. k+3) of row `row` as fp32,
// through L2 (coherent with writes by other CTAs of the same kernel).
template <bool kF32>
__device__ __forceinline__ float4 load_act4(const void* a, size_t ld, int row, int k) {
    if (kF32) {
        const float* p = static_cast<const float*>(a) + static_cast<size_t>(row) * ld + k;
        return __ldcg(reinterpret_cast<const float4*>(p));
    } else {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(a) + static_cast<size_t>(row) * ld + k;
        uint2 raw = __ldcg(reinterpret_cast<const uint2*>(p));
        float4 r;
        r.x = __uint_as_float(raw.x << 16);
        r.y = __uint_as_float(raw.x & 0xFFFF0000u);
        r.z = __uint_as_float(raw.y << 16);
        r.w = __uint_as_float(raw.y & 0xFFFF0000u);
        return r;
    }
}

// One warp quantises one 1 x 128 group (GLM-5.2 x10 §1, §8c: live FP8
// activation quantisation).  Lane l holds elements 4l .. 4l+3 in v.
//   s = fl32(amax / 448); code = RNE_satfinite(fl32(x / s)); s == 0 -> signed zero.
// Returns the 4 codes packed little-endian (element 4l in byte 0) and the
// scale through *s_out; also writes the 4 decoded (exact) values to dec.
__device__ __forceinline__ uint32_t quant_group_warp(float4 v, float* s_out, float4* dec) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 448.0f);
    uint32_t codes;
    if (s == 0.0f) {
        codes = (signbit(v.x) ? 0x80u : 0u) | (signbit(v.y) ? 0x8000u : 0u) |
                (signbit(v.z) ? 0x800000u : 0u) | (signbit(v.w) ? 0x80000000u : 0u);
    } else {
        const uint16_t c01 = e4m3x2_from_f32(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s));
        const uint16_t c23 = e4m3x2_from_f32(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s));
        codes = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
    }
    float2 d01, d23;
    e4m3x4_to_f32(codes, d01, d23);
    *dec = make_float4(d01.x, d01.y, d23.x, d23.y);
    *s_out = s;
    return codes;
}

}  // namespace moeq
