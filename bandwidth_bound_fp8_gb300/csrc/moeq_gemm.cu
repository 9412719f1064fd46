// Expert GEMM with the live activation quantisation fused into its prologue
// (GLM-5.2 x10 §4, "PQ-GEMM": quantisation inside the GEMM, no activation
// round trip through HBM), split-K over every SM (§1) and a deterministic
// fp32 split-K reduction, for the M = 1..16 decode / draft-verification case.
//
// Work decomposition ("units").  A unit is one 128-row block (two for
// gate_up: the gate block and its matching up block) of one unique expert
// times one 128-wide K group: 16 KiB (32 KiB) of FP8 weights.  Units are
// ordered (unique expert, row block, K group) and the grid -- one persistent
// CTA per SM -- takes contiguous, equal shares of them, so every SM streams
// the same number of bytes whatever the number of experts.  A CTA's share
// splits into segments (runs of one row block); only a CTA's first and last
// segment can be partial in K, so each CTA leaves at most two fp32 partials.
// The last CTA to finish a row block (atomic ticket, no waiting) sums the
// partials in CTA order -- the same order every run -- and applies the
// epilogue (SwiGLU for gate_up).
//
// Inside a CTA: warp 8 is the producer; one lane issues TMA bulk-tensor
// loads of the units into a ring of shared-memory stages (mbarrier
// full/empty pairs).  Warps 0-7 consume: they quantise the segment's
// activation groups (per token, 1 x 128, s = amax/448) into shared memory,
// then for every stage each lane takes 16 bytes of one weight row, turns
// them into fp32 (exact) and accumulates products with the decoded
// activation codes using paired fp32 FMAs.  Lanes keep running sums across
// K groups (scaled per group by s_a * s_w) and reduce across the 8 lanes of
// a row with warp shuffles at the end of the segment.
#include "moeq_device.cuh"
#include "moeq_internal.h"

namespace moeq {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kActCap = 8192;                 // decoded activation floats in shared memory
constexpr int kActScaleCap = kActCap / kGroup;
constexpr int kMaxKG = MOEQ_MAX_K / kGroup;
constexpr int kAccLd = kMaxTok + 1;           // padded row stride of the accumulator tile

template <int NBOX>
struct Cfg {
    static constexpr int kRows = 128 * NBOX;                 // weight rows per unit
    static constexpr int kStageBytes = 16384 * NBOX;
    static constexpr int kStages = NBOX == 2 ? 5 : 10;       // 160 KiB ring either way
    static constexpr int kRowsPerWarp = kRows / kConsumerWarps;
    static constexpr int kPasses = kRowsPerWarp / 4;         // 4 rows per warp instruction
};

struct SmemTail {
    float act[kActCap];               // decoded activations, [tok][group][permuted k]
    float act_s[kActScaleCap];        // activation scales [tok][group]
    float sw[2][kMaxKG];              // weight scales of the segment, per box
    float acc[256 * kAccLd];          // per (row, token) sums, row stride kAccLd
    uint64_t full[10];
    uint64_t empty[10];
    int abort_flag;
    int last_flag;
};

template <int NBOX>
constexpr size_t smem_bytes() {
    return 1024 + static_cast<size_t>(Cfg<NBOX>::kStages) * Cfg<NBOX>::kStageBytes + sizeof(SmemTail);
}

// Position of element k (0..127) of a group in the shared activation layout:
// lane l8 = k/16 reads its four float4 (k = 16*l8 + 4i .. +3) at (8i + l8)*4,
// so the 8 lanes of a quarter-warp hit 8 consecutive 16-byte chunks.
__device__ __forceinline__ int act_pos(int k) { return (((k & 15) >> 2) * 8 + (k >> 4)) * 4 + (k & 3); }

__device__ __forceinline__ void consumer_sync() { named_sync(1, kConsumers); }

__device__ __forceinline__ long long unit_lo(long long c, long long T, long long G) { return c * T / G; }
// The CTA whose share [unit_lo(c), unit_lo(c+1)) holds unit u.
__device__ __forceinline__ long long cta_of_unit(long long u, long long T, long long G) {
    return ((u + 1) * G - 1) / T;
}

__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

// One stage, tokens t0 .. t0+MT-1 (clamped to ntok-1 for loads): per lane
// and pass, the dot product of its 16 weight bytes with the 16 matching
// decoded activations, one float per (pass, token).
template <int NBOX, int MT>
__device__ __forceinline__ void stage_dot(const uint8_t* st, const float* act_g, int tok_ld, int t0, int ntok,
                                          int cw, int lane, float (&part)[Cfg<NBOX>::kPasses][MT]) {
    using C = Cfg<NBOX>;
    const int l8 = lane & 7;
    const int rsub = lane >> 3;
    float2 a[MT][8];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int tt = min(t0 + t, ntok - 1);
        const float4* ap = reinterpret_cast<const float4*>(act_g + tt * tok_ld);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ap[i * 8 + l8];
            a[t][2 * i] = make_float2(v.x, v.y);
            a[t][2 * i + 1] = make_float2(v.z, v.w);
        }
    }
#pragma unroll
    for (int p = 0; p < C::kPasses; ++p) {
        const int row = cw * C::kRowsPerWarp + p * 4 + rsub;
        const uint4 w = *reinterpret_cast<const uint4*>(st + row * 128 + l8 * 16);
        float2 wf[8];
        e4m3x4_to_f32(w.x, wf[0], wf[1]);
        e4m3x4_to_f32(w.y, wf[2], wf[3]);
        e4m3x4_to_f32(w.z, wf[4], wf[5]);
        e4m3x4_to_f32(w.w, wf[6], wf[7]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float2 d = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 8; ++j) d = __ffma2_rn(wf[j], a[t][j], d);
            part[p][t] = d.x + d.y;
        }
    }
}

__device__ __forceinline__ float reduce8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

struct SegCtx {
    int ue, rb, g0, g1, expert, p0, ntok;
    bool valid;
};

template <int NBOX, bool kF32>
__device__ __forceinline__ void quantise_chunk(const GemmArgs& args, SmemTail& sm, const SegCtx& sc, int ga, int gb,
                                               int U, int cw, int lane) {
    const int ngc = gb - ga;
    const int KG = args.K / kGroup;
    const bool dump = sc.valid && args.qdump != nullptr && sc.rb == 0 && (args.a_row == nullptr || sc.ue == U - 1);
    for (int item = cw; item < sc.ntok * ngc; item += kConsumerWarps) {
        const int t = item / ngc, gl = item % ngc, gg = ga + gl;
        const int p = sc.p0 + t;
        int row = args.a_row ? __ldg(args.a_row + p) : p;
        if (row < 0 || row >= args.rows_a) {
            if (lane == 0) record_error(args.status, MOEQ_ERR_INVALID_ARG);
            row = 0;
        }
        const float4 v = load_act4<kF32>(args.a, static_cast<size_t>(args.K), row, gg * kGroup + lane * 4);
        float s;
        float4 dec;
        const uint32_t codes = quant_group_warp(v, &s, &dec);
        float* dst = sm.act + (t * ngc + gl) * kGroup;
        *reinterpret_cast<float4*>(dst + act_pos(lane * 4)) = dec;
        if (lane == 0) sm.act_s[t * ngc + gl] = s;
        if (dump) {
            *reinterpret_cast<uint32_t*>(args.qdump + static_cast<size_t>(row) * args.K + gg * kGroup + lane * 4) =
                codes;
            if (lane == 0) args.sdump[static_cast<size_t>(row) * KG + gg] = s;
        }
    }
}

// Epilogue from the accumulator tile: SwiGLU (gate rows 0..127, up rows
// 128..255) or a plain store of the 128 rows.
template <int NBOX>
__device__ __forceinline__ void epilogue(const GemmArgs& args, const SmemTail& sm, const SegCtx& sc, int ctid) {
    if (!sc.valid) return;
    for (int idx = ctid; idx < 128 * sc.ntok; idx += kConsumers) {
        const int i = idx & 127, t = idx >> 7;
        float* o = args.out + static_cast<size_t>(sc.p0 + t) * args.out_ld + sc.rb * 128 + i;
        if (NBOX == 2) {
            const float g = sm.acc[i * kAccLd + t];
            const float u = sm.acc[(128 + i) * kAccLd + t];
            *o = __fdiv_rn(g, 1.0f + expf(-g)) * u;
        } else {
            *o = sm.acc[i * kAccLd + t];
        }
    }
}

// Streams the K groups [g0, g1) of one segment and leaves one sum per
// (row, token) in sm.acc.  MODE = 1, 2, 4: up to that many tokens, running
// sums in registers; MODE = 0: any number of tokens, four at a time, with
// the cross-lane reduction done per group into sm.acc.
template <int NBOX, bool kF32, int MODE>
__device__ __forceinline__ void run_segment(const GemmArgs& args, SmemTail& sm, const uint8_t* stages,
                                            const SegCtx& sc, int U, int cw, int lane, int ctid, long long& it) {
    using C = Cfg<NBOX>;
    constexpr int MT = MODE == 0 ? 4 : MODE;
    const int box = (cw * C::kRowsPerWarp) / 128;
    if (MODE == 0)
        for (int i = ctid; i < C::kRows * kMaxTok; i += kConsumers) sm.acc[(i / kMaxTok) * kAccLd + i % kMaxTok] = 0.f;
    float acc[C::kPasses][MT];
#pragma unroll
    for (int p = 0; p < C::kPasses; ++p)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[p][t] = 0.0f;

    const int gpc = max(1, kActCap / (kGroup * sc.ntok));
    for (int ga = sc.g0; ga < sc.g1; ga += gpc) {
        const int gb = min(sc.g1, ga + gpc);
        const int ngc = gb - ga;
        consumer_sync();  // activation buffer free
        quantise_chunk<NBOX, kF32>(args, sm, sc, ga, gb, U, cw, lane);
        consumer_sync();  // activation buffer full
        for (int g = ga; g < gb; ++g, ++it) {
            const int s = static_cast<int>(it % C::kStages);
            if (!mbar_wait_bounded(&sm.full[s], static_cast<uint32_t>((it / C::kStages) & 1), &sm.abort_flag)) {
                // Give up on the data but keep the control flow (and so every
                // named barrier) identical across the consumer warps.
                record_error(args.status, MOEQ_ERR_TIMEOUT);
                sm.abort_flag = 1;
            }
            const uint8_t* st = stages + s * C::kStageBytes;
            const float* act_g = sm.act + (g - ga) * kGroup;
            const int tok_ld = ngc * kGroup;
            const float swg = sm.sw[box][g - sc.g0];
            if (MODE != 0) {
                float part[C::kPasses][MT];
                stage_dot<NBOX, MT>(st, act_g, tok_ld, 0, sc.ntok, cw, lane, part);
                float scl[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) scl[t] = sm.act_s[min(t, sc.ntok - 1) * ngc + (g - ga)] * swg;
#pragma unroll
                for (int p = 0; p < C::kPasses; ++p)
#pragma unroll
                    for (int t = 0; t < MT; ++t) acc[p][t] = fmaf(part[p][t], scl[t], acc[p][t]);
            } else {
                for (int t0 = 0; t0 < sc.ntok; t0 += 4) {
                    float part[C::kPasses][4];
                    stage_dot<NBOX, 4>(st, act_g, tok_ld, t0, sc.ntok, cw, lane, part);
#pragma unroll
                    for (int p = 0; p < C::kPasses; ++p) {
                        const int row = cw * C::kRowsPerWarp + p * 4 + (lane >> 3);
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float v = reduce8(part[p][t]);
                            if ((lane & 7) == 0 && t0 + t < sc.ntok)
                                sm.acc[row * kAccLd + t0 + t] += v * (sm.act_s[(t0 + t) * ngc + (g - ga)] * swg);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
    }
    if (MODE != 0) {
#pragma unroll
        for (int p = 0; p < C::kPasses; ++p) {
            const int row = cw * C::kRowsPerWarp + p * 4 + (lane >> 3);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v = reduce8(acc[p][t]);
                if ((lane & 7) == 0 && t < sc.ntok) sm.acc[row * kAccLd + t] = v;
            }
        }
    }
}

template <int NBOX, bool kF32>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const GemmArgs args) {
    using C = Cfg<NBOX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemTail& sm = *reinterpret_cast<SmemTail*>(stages + C::kStages * C::kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KG = args.K / kGroup;
    int U = __ldg(args.n_uniq);
    if (U > args.max_uniq || U < 0) {  // a plan the call cannot hold: report, and clamp
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(args.status, MOEQ_ERR_INVALID_ARG);
        U = U < 0 ? 0 : args.max_uniq;
    }
    const long long upe = static_cast<long long>(args.RB) * KG;  // units per expert
    const long long T = static_cast<long long>(U) * upe;
    const long long G = gridDim.x, c = blockIdx.x;
    const long long u_lo = unit_lo(c, T, G), u_hi = unit_lo(c + 1, T, G);

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (u_lo >= u_hi) return;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&wmap);
            const uint64_t pol = l2_evict_first_policy();
            long long issued = 0;
            int cur_ue = -1, expert = 0;
            for (long long u = u_lo; u < u_hi; ++u) {
                const int ue = static_cast<int>(u / upe);
                const int rem = static_cast<int>(u % upe);
                const int rb = rem / KG, g = rem % KG;
                if (ue != cur_ue) {
                    cur_ue = ue;
                    expert = __ldg(args.uniq + ue);
                    if (expert < 0 || expert >= args.n_experts) expert = 0;  // reported by the consumers
                }
                const int s = static_cast<int>(issued % C::kStages);
                if (issued >= C::kStages) {
                    const uint32_t par = static_cast<uint32_t>((issued / C::kStages - 1) & 1);
                    if (!mbar_wait_bounded(&sm.empty[s], par, &sm.abort_flag)) {
                        record_error(args.status, MOEQ_ERR_TIMEOUT);
                        sm.abort_flag = 1;
                    }
                }
                if (sm.abort_flag) break;
                uint8_t* dst = stages + s * C::kStageBytes;
                const int row0 = expert * args.rows_per_expert + rb * 128;
                mbar_arrive_expect_tx(&sm.full[s], C::kStageBytes);
                tma_load_2d(dst, &wmap, g * kGroup, row0, &sm.full[s], pol);
                if (NBOX == 2) tma_load_2d(dst + 16384, &wmap, g * kGroup, row0 + args.up_offset, &sm.full[s], pol);
                ++issued;
            }
            if (sm.abort_flag) {
                // Let the copies already issued land before the CTA may exit
                // (bounded, 100 ms per stage).
                for (long long j = max(0LL, issued - C::kStages); j < issued; ++j) {
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(&sm.full[j % C::kStages], static_cast<uint32_t>((j / C::kStages) & 1)) &&
                           global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp, ctid = tid;
    long long it = 0;
    long long u = u_lo;
    while (u < u_hi) {
        SegCtx sc;
        sc.ue = static_cast<int>(u / upe);
        const int rem = static_cast<int>(u % upe);
        sc.rb = rem / KG;
        sc.g0 = rem % KG;
        const long long seg_end = min(u_hi, u - sc.g0 + KG);
        sc.g1 = sc.g0 + static_cast<int>(seg_end - u);
        sc.expert = __ldg(args.uniq + sc.ue);
        sc.p0 = __ldg(args.offs + sc.ue);
        sc.ntok = __ldg(args.offs + sc.ue + 1) - sc.p0;
        // A plan entry this call cannot serve (bad expert id, pair range
        // outside `out`, more than kMaxTok tokens) is reported and streamed
        // without writing any output, so every index stays in bounds.
        sc.valid = sc.expert >= 0 && sc.expert < args.n_experts && sc.p0 >= 0 && sc.ntok >= 1 &&
                   sc.ntok <= kMaxTok && sc.p0 + sc.ntok <= args.max_pairs;
        if (!sc.valid) {
            if (ctid == 0) record_error(args.status, MOEQ_ERR_INVALID_ARG);
            sc.expert = 0;
            sc.p0 = 0;
            sc.ntok = 1;
        }
        const int nseg = sc.g1 - sc.g0;

        consumer_sync();  // previous segment's readers of sw / acc are done
        for (int i = ctid; i < nseg * NBOX; i += kConsumers) {
            const int b = i / nseg, gg = sc.g0 + i % nseg;
            const int rbox = sc.rb + (b ? args.up_offset / 128 : 0);
            sm.sw[b][gg - sc.g0] =
                __ldg(args.sw + (static_cast<size_t>(sc.expert) * (args.rows_per_expert / 128) + rbox) * KG + gg);
        }
        if (sc.ntok <= 1)
            run_segment<NBOX, kF32, 1>(args, sm, stages, sc, U, cw, lane, ctid, it);
        else if (sc.ntok <= 2)
            run_segment<NBOX, kF32, 2>(args, sm, stages, sc, U, cw, lane, ctid, it);
        else if (sc.ntok <= 4)
            run_segment<NBOX, kF32, 4>(args, sm, stages, sc, U, cw, lane, ctid, it);
        else
            run_segment<NBOX, kF32, 0>(args, sm, stages, sc, U, cw, lane, ctid, it);
        consumer_sync();

        // ------------------------------------------------------------ finalise
        if (sc.g0 == 0 && sc.g1 == KG) {
            epilogue<NBOX>(args, sm, sc, ctid);
        } else {
            const long long r = static_cast<long long>(sc.ue) * args.RB + sc.rb;  // row-block id
            const long long c_lo = cta_of_unit(r * KG, T, G);
            const long long c_hi = cta_of_unit(r * KG + KG - 1, T, G);
            const int my_slot = static_cast<int>(2 * c + ((u_lo / KG) == r ? 0 : 1));
            float* mine = args.partials + static_cast<size_t>(my_slot) * kMaxTok * C::kRows;
            for (int idx = ctid; idx < C::kRows * sc.ntok; idx += kConsumers) {
                const int row = idx % C::kRows, t = idx / C::kRows;
                mine[t * C::kRows + row] = sm.acc[row * kAccLd + t];
            }
            __threadfence();
            consumer_sync();
            if (ctid == 0) {
                int n = 0;
                for (long long cc = c_lo; cc <= c_hi; ++cc) n += unit_lo(cc, T, G) < unit_lo(cc + 1, T, G);
                const int old = atomicAdd(args.tickets + r, 1);
                sm.last_flag = (old == n - 1);
            }
            consumer_sync();
            if (sm.last_flag) {
                __threadfence();
                for (int idx = ctid; idx < C::kRows * sc.ntok; idx += kConsumers) {
                    const int row = idx % C::kRows, t = idx / C::kRows;
                    float v = 0.0f;
                    for (long long cc = c_lo; cc <= c_hi; ++cc) {
                        const long long lo = unit_lo(cc, T, G);
                        if (lo >= unit_lo(cc + 1, T, G)) continue;
                        const int slot = static_cast<int>(2 * cc + ((lo / KG) == r ? 0 : 1));
                        v += __ldcg(args.partials + (static_cast<size_t>(slot) * kMaxTok + t) * C::kRows + row);
                    }
                    sm.acc[row * kAccLd + t] = v;
                }
                consumer_sync();
                epilogue<NBOX>(args, sm, sc, ctid);
                if (ctid == 0) args.tickets[r] = 0;
            }
        }
        u = seg_end;
    }
}

template <int NBOX, bool kF32>
static cudaError_t launch_one(const CUtensorMap& map, const GemmArgs& args, int grid, cudaStream_t stream) {
    constexpr size_t bytes = smem_bytes<NBOX>();
    static_assert(bytes <= 232448, "shared memory budget");
    static bool configured = false;  // per instantiation; attribute is per device-function
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<NBOX, kF32>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    expert_gemm_kernel<NBOX, kF32><<<grid, kThreads, bytes, stream>>>(map, args);
    return cudaGetLastError();
}

cudaError_t launch_expert_gemm(const CUtensorMap& map, const GemmArgs& args, int nbox, int grid,
                               cudaStream_t stream) {
    if (nbox == 2) return args.a_f32 ? launch_one<2, true>(map, args, grid, stream)
                                     : launch_one<2, false>(map, args, grid, stream);
    return args.a_f32 ? launch_one<1, true>(map, args, grid, stream) : launch_one<1, false>(map, args, grid, stream);
}

size_t gemm_partials_floats(int nbox, int grid) {
    return static_cast<size_t>(2) * grid * kMaxTok * 128 * nbox;
}

}  // namespace moeq
