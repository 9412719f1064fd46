// The engine's tcgen05 instantiations: the MMA-issuing lane and the
// epilogue warps that promote the TMEM accumulators (the rest of the engine
// is in moeq_stream.cuh).
#include "moeq_stream.cuh"

namespace moeq {

// Swap-AB: the 128 weight rows of a tile are the MMA's M, the (up to 16)
// tokens of the segment its N, K = 128 per tile in four K = 32 steps.  Each
// stage's tiles accumulate into their own TMEM columns (a fresh sum per
// 128-wide K group), so the per-group scales are applied in fp32 by the
// epilogue warps, as the CUDA-core path does.  One lane issues the MMAs; its
// commits free the weight stage and hand the accumulators to the epilogue.
template <bool kMma>
__device__ __noinline__ void mma_issue_loop(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, int lane) {
    constexpr uint32_t kIdesc = umma_idesc_e4m3(128, kMmaN);
    const uint32_t tmem = sm.tmem_base, stage0 = smem_u32(stages);
    long long c = 0, it = 0, last = -1;
    bool ok = true;
    while (ok) {
        const int cs = static_cast<int>(c & 1);
        if (!mbar_wait_or_abort(&sm.prep_full[cs], static_cast<uint32_t>((c >> 1) & 1), sm, a.status)) break;
        const ChunkDesc d = sm.chunk[cs];
        if (d.kind < 0 || sm.abort_flag) break;
        const uint32_t bslot = smem_u32(sm.act[cs]);
        for (int ku = d.ku0; ku < d.ku1; ++ku, ++it) {
            const int s = static_cast<int>(it % kStages), b = static_cast<int>(it % kTmemBufs);
            ok = mbar_wait_or_abort(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status);
            if (ok && it >= kTmemBufs)
                ok = mbar_wait_or_abort(&sm.tmem_empty[b], static_cast<uint32_t>(((it / kTmemBufs) - 1) & 1), sm,
                                        a.status);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const int ntile = d.kind == kKindGU ? 2 : min(2, a.op[kKindDN].KB - 2 * ku);
                for (int tt = 0; tt < ntile; ++tt) {
                    const int gl = (d.kind == kKindGU ? ku : 2 * ku + tt) - d.g0;
                    const uint32_t aaddr = stage0 + static_cast<uint32_t>(s * kStageBytes + tt * kTile);
                    const uint32_t baddr = bslot + static_cast<uint32_t>(gl * kMmaGroupBytes);
                    const uint32_t dcol = tmem + static_cast<uint32_t>((b * 2 + tt) * kMmaN);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f8(dcol, umma_desc_sw128(aaddr + 32 * k), umma_desc_sw128(baddr + 32 * k), kIdesc, k);
                }
                umma_commit(&sm.mma_done[b]);
                umma_commit(&sm.empty[s]);
            }
            __syncwarp();
            last = it;
        }
        ++c;
    }
    // every MMA issued must have completed before TMEM is freed (bounded; a
    // wait that runs out is an error of the launch: its results are void)
    if (last >= 0) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&sm.mma_done[last % kTmemBufs], static_cast<uint32_t>((last / kTmemBufs) & 1))) {
            if (global_timer_ns() - t0 > 100ull * 1000ull * 1000ull) {
                if (lane == 0) record_error(a.status, MOEQ_ERR_TIMEOUT);
                break;
            }
        }
    }
}

// One stage for the epilogue: each tile's NT token columns of this thread's
// TMEM lane, scaled by s_a[t][g] * s_w and added to the running sums.  Both
// tiles' loads (and their scales) are issued before the one wait.
template <int NT, int NA>
__device__ __forceinline__ void epi_fma(float (&acc)[NA], const uint32_t (&r)[NT], const float4* sa, float sw) {
#pragma unroll
    for (int q = 0; q < NT / 4; ++q) {
        const float4 x = sa[q];
        acc[4 * q] = fmaf(__uint_as_float(r[4 * q]), x.x * sw, acc[4 * q]);
        acc[4 * q + 1] = fmaf(__uint_as_float(r[4 * q + 1]), x.y * sw, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(__uint_as_float(r[4 * q + 2]), x.z * sw, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(__uint_as_float(r[4 * q + 3]), x.w * sw, acc[4 * q + 3]);
    }
}

// One stage for the epilogue: each tile's NT token columns of this thread's
// TMEM lane, scaled by s_a[t][g] * s_w and added to the running sums (gate_up:
// the gate and up tiles to acc0 and acc1; down: both K groups to acc0).  Up
// to 8 columns both tiles' loads are issued before one wait; with 16 the two
// tiles' registers do not fit beside the sums, so they go one after the other.
template <int NT, int KIND, int NA>
__device__ __forceinline__ void mma_epi_stage(const SmemTail& sm, uint32_t tcol, int cs, const ChunkDesc& d, int ku,
                                              int kb_dn, float (&acc0)[kMmaN], float (&acc1)[NA]) {
    constexpr bool gu = KIND == kKindGU;
    const bool two = gu || 2 * ku + 1 < kb_dn;
    const int gl0 = (gu ? ku : 2 * ku) - d.g0, gl1 = gu ? gl0 : gl0 + 1;
    const float sw0 = sm.sw[cs][0][gl0], sw1 = sm.sw[cs][gu ? 1 : 0][gl1];
    const float4* a0 = reinterpret_cast<const float4*>(&sm.act_s[cs][gl0 * kMmaN]);
    const float4* a1 = reinterpret_cast<const float4*>(&sm.act_s[cs][gl1 * kMmaN]);
    if constexpr (NT <= 8) {
        uint32_t r0[NT], r1[NT];
        tmem_ld_nowait<NT>(tcol, r0);
        if (two) tmem_ld_nowait<NT>(tcol + static_cast<uint32_t>(kMmaN), r1);
        tmem_wait_ld();
        epi_fma<NT>(acc0, r0, a0, sw0);
        if (two) {
            if constexpr (gu)
                epi_fma<NT>(acc1, r1, a1, sw1);
            else
                epi_fma<NT>(acc0, r1, a1, sw1);
        }
    } else {
        uint32_t r[NT];
        tmem_ld_nowait<NT>(tcol, r);
        tmem_wait_ld();
        epi_fma<NT>(acc0, r, a0, sw0);
        if (two) {
            tmem_ld_nowait<NT>(tcol + static_cast<uint32_t>(kMmaN), r);
            tmem_wait_ld();
            if constexpr (gu)
                epi_fma<NT>(acc1, r, a1, sw1);
            else
                epi_fma<NT>(acc0, r, a1, sw1);
        }
    }
}

// The epilogue warps: set e (warps 4e .. 4e+3) takes the stages with
// it % 2 == e; warp w owns TMEM lanes 32*(w%4) .. +31 = rows of each tile.
// At a segment's end set 1 stores its sums in the result slot and set 0 adds
// its own (a fixed order) and publishes the slot like the CUDA-core consumers.
// One segment, with its running sums in registers (NT token columns).
template <int NT, int KIND>
__device__ __noinline__ void mma_epi_segment(const StreamArgs& a, SmemTail& sm, int set, uint32_t tlane, int r,
                                             int ntok, float* res, int ld, int rs, long long& c_io,
                                             long long& it_io) {
    constexpr int NA = KIND == kKindGU ? kMmaN : 1;   // up-tile sums: gate_up only
    const int kb_dn = a.op[kKindDN].KB;
    const int lane = threadIdx.x & 31;
    long long c = c_io, it = it_io;
    float acc0[kMmaN], acc1[NA];   // gate (or down) and up sums per token (NT used)
#pragma unroll
    for (int t = 0; t < kMmaN; ++t) acc0[t] = 0.0f;
#pragma unroll
    for (int t = 0; t < NA; ++t) acc1[t] = 0.0f;
    for (bool first = true;; first = false) {
        const int cs = static_cast<int>(c & 1);
        if (!first) mbar_wait_or_abort(&sm.prep_full[cs], static_cast<uint32_t>((c >> 1) & 1), sm, a.status);
        const ChunkDesc d = sm.chunk[cs];
        for (int ku = d.ku0; ku < d.ku1 && !sm.abort_flag; ++ku, ++it) {
            if ((it & 1) != set) continue;
            const int b = static_cast<int>(it % kTmemBufs);
            if (!mbar_wait_or_abort(&sm.mma_done[b], static_cast<uint32_t>((it / kTmemBufs) & 1), sm, a.status))
                break;
            tc_fence_after();
            mma_epi_stage<NT, KIND, NA>(sm, tlane + static_cast<uint32_t>(b * 2 * kMmaN), cs, d, ku, kb_dn, acc0, acc1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tmem_empty[b]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.act_empty[cs]);
        ++c;
        if (d.seg_end || sm.abort_flag) break;
    }
    c_io = c;
    it_io = it;
    if (set == 1) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < ntok) {
                res[r * ld + t] = acc0[t];
                if constexpr (KIND == kKindGU) res[(128 + r) * ld + t] = acc1[t];
            }
        }
    }
    named_sync(5, kEpiWarps * 32);
    if (set == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < ntok) {
                res[r * ld + t] += acc0[t];
                if constexpr (KIND == kKindGU) res[(128 + r) * ld + t] += acc1[t];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.res_full[rs]);
    }
}

template <bool kMma>
__device__ __noinline__ void mma_epilogue_loop(const StreamArgs& a, SmemTail& sm, int warp, int lane) {
    const ResRing ring(a);
    const int set = warp / 4, quad = warp % 4;
    const uint32_t tlane = sm.tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const int r = quad * 32 + lane;
    long long c = 0, it = 0, sidx = 0;
    for (;;) {
        const int rs = ring.slot(sidx);
        if (sidx >= ring.ns) mbar_wait_or_abort(&sm.res_empty[rs], ring.parity(sidx) ^ 1u, sm, a.status);
        const int cs0 = static_cast<int>(c & 1);
        mbar_wait_or_abort(&sm.prep_full[cs0], static_cast<uint32_t>((c >> 1) & 1), sm, a.status);
        const int kind = sm.chunk[cs0].kind;
        if (kind < 0 || sm.abort_flag) {
            if (set == 0) {
                // pass the end on to both finish warps (see the CUDA-core consumers)
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.res_full[rs]);
                const long long s2 = sidx + 1;
                if (s2 >= ring.ns)
                    mbar_wait_or_abort(&sm.res_empty[ring.slot(s2)], ring.parity(s2) ^ 1u, sm, a.status);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.res_full[ring.slot(s2)]);
            }
            break;
        }
        const int ntok = sm.chunk[cs0].ntok;
        float* res = ring.at(sm, sidx);
        if (kind == kKindGU) {
            if (ntok <= 4)
                mma_epi_segment<4, kKindGU>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
            else if (ntok <= 8)
                mma_epi_segment<8, kKindGU>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
            else
                mma_epi_segment<16, kKindGU>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
        } else {
            if (ntok <= 4)
                mma_epi_segment<4, kKindDN>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
            else if (ntok <= 8)
                mma_epi_segment<8, kKindDN>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
            else
                mma_epi_segment<16, kKindDN>(a, sm, set, tlane, r, ntok, res, ring.ld, rs, c, it);
        }
        ++sidx;
    }
}

cudaError_t launch_stream_mma(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    return launch_mode<true>(args, grid, cooperative, stream);
}

}  // namespace moeq
