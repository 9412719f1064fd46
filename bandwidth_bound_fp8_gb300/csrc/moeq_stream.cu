// The weight-streaming expert GEMM engine: one persistent CTA per SM pulls
// FP8 weight tiles from HBM through a ring of shared-memory stages with 1-D
// bulk copies and reduces them against live-quantised activations.
//
// GLM-5.2 x10 is the source of the method: decode streams every active
// expert weight from HBM once with little arithmetic on top (bandwidth
// model); the activations are quantised to FP8 live, in front of the GEMM
// (§1, §8c), fused into it instead of round-tripping through HBM (§4,
// "PQ-GEMM"); K is split so that every SM streams (§1, split-K); tokens
// verified together share one read of each expert (§5-§6).
//
// Work.  A unit is one stage: for gate_up the gate tile and the up tile of
// one 128-row block at one 128-wide K group (32 KiB), for down two
// consecutive K tiles of one 128-row block (32 KiB).  Work comes in lists
// (for the layer: shared-expert gate_up, routed gate_up, shared down, routed
// down); every CTA takes a contiguous, equal share of every list.  A share
// splits into segments (runs of one row block); only its first and last can
// be partial in K, so each CTA leaves at most two fp32 partials per list; the
// last CTA to finish a row block (atomic ticket) sums them in CTA order and
// runs the epilogue, so results do not depend on timing.
//
// Inside a CTA warp 16 is the producer (one lane issues the bulk copies) and
// warps 0-15 consume: they quantise the segment's activation groups (per
// token, 1 x 128, s = amax/448, RNE to E4M3) into shared memory, then each
// lane takes 16 bytes of a weight row per pass, widens them exactly to fp32
// and accumulates products with the decoded activation codes in paired fp32
// FMAs, scaling per K group by s_a * s_w.
//
// Layer fusion (cooperative launch, all CTAs resident): CTA 0 computes the
// routing plan while the other CTAs stream the shared expert, which needs no
// routing; gate_up epilogues publish per-(expert, row block) readiness of h;
// down segments wait (bounded) for their expert's h while their weights are
// already in flight; the down epilogue that completes the last expert of a
// (token, row block) also writes the combined bf16 output.
#include "moeq_device.cuh"
#include "moeq_internal.h"
#include "moeq_route.cuh"

namespace moeq {

constexpr int kCW = 16;                // consumer warps
constexpr int kConsumers = kCW * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTile = 16384;
constexpr int kStageBytes = 2 * kTile;
constexpr int kStages = 5;
constexpr int kActCap = 6144;          // decoded activation floats in shared memory
constexpr int kActScaleCap = kActCap / kGroup;
constexpr int kMaxKG = MOEQ_MAX_K / kGroup;
constexpr int kAccLd = kMaxTok + 1;
constexpr int kUnitRows = 256;         // rows of a gate_up unit (gate + up); down units use 128

struct SmemTail {
    union {
        float act[kActCap];            // decoded activations [tok][group][permuted k]
        RouteScratch route;            // plan computation (CTA 0, before any activation)
    };
    float act_s[kActScaleCap];         // activation scales [tok][group]
    float sw[2][kMaxKG];               // weight scales of the segment
    float acc[kUnitRows * kAccLd];     // one sum per (row, token)
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort_flag;
    int last_flag;
    int n_comb;
    int comb_tok[kMaxTok];
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(SmemTail);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void consumer_sync() { named_sync(1, kConsumers); }
__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

// Position of element k (0..127) of a group in the shared activation layout:
// lane l8 reads its four float4 (k = 16*l8 + 4i .. +3) at (8i + l8)*4, so the
// eight lanes of a row hit eight consecutive 16-byte chunks.
__device__ __forceinline__ int act_pos(int k) { return (((k & 15) >> 2) * 8 + (k >> 4)) * 4 + (k & 3); }

// ------------------------------------------------------------------ work lists
struct ListInfo {
    int kind, src, n_exp, RB, KU;
    long long T, G, c;   // units, participating CTAs, this CTA's index among them
    long long lo, hi;    // this CTA's share [lo, hi)
};

__device__ __forceinline__ long long unit_lo(long long c, long long T, long long G) { return c * T / G; }
__device__ __forceinline__ long long cta_of_unit(long long u, long long T, long long G) {
    return ((u + 1) * G - 1) / T;
}

__device__ __forceinline__ bool list_needs_plan(const StreamArgs& a, int li) {
    return a.list_src[li] != kSrcShared;
}

__device__ __forceinline__ ListInfo list_info(const StreamArgs& a, int li, int U) {
    ListInfo L;
    L.kind = a.list_kind[li];
    L.src = a.list_src[li];
    L.n_exp = L.src == kSrcShared ? 1 : (L.src == kSrcPlanAll ? U : U - 1);
    if (L.n_exp < 0) L.n_exp = 0;
    const Operand& op = a.op[L.kind];
    L.RB = op.RB;
    L.KU = L.kind == kKindGU ? op.KB : (op.KB + 1) / 2;
    L.T = static_cast<long long>(L.n_exp) * L.RB * L.KU;
    // While CTA 0 routes, the shared expert's gate_up goes to the other CTAs.
    const bool skip0 = a.fused_route && L.src == kSrcShared && L.kind == kKindGU && gridDim.x > 1;
    L.G = gridDim.x - (skip0 ? 1 : 0);
    L.c = static_cast<long long>(blockIdx.x) - (skip0 ? 1 : 0);
    if (L.c < 0 || L.T == 0) {
        L.lo = L.hi = 0;
    } else {
        L.lo = unit_lo(L.c, L.T, L.G);
        L.hi = unit_lo(L.c + 1, L.T, L.G);
    }
    return L;
}

struct ExpertRef {
    int expert, p0, ntok, slot;
    bool shared_static, valid;
};

__device__ __forceinline__ ExpertRef expert_ref(const StreamArgs& a, int src, int e_local) {
    ExpertRef r;
    if (src == kSrcShared) {
        r.expert = a.shared_id;
        r.p0 = a.shared_p0;
        r.ntok = a.M;
        r.slot = a.max_uniq - 1;
        r.shared_static = true;
    } else {
        r.expert = __ldcg(a.uniq + e_local);
        r.p0 = __ldcg(a.offs + e_local);
        r.ntok = __ldcg(a.offs + e_local + 1) - r.p0;
        r.slot = e_local;
        r.shared_static = false;
    }
    r.valid = r.expert >= 0 && r.expert < a.n_experts && r.p0 >= 0 && r.ntok >= 1 && r.ntok <= kMaxTok &&
              r.p0 + r.ntok <= a.max_pairs;
    return r;
}

__device__ __forceinline__ const uint8_t* tile_ptr(const Operand& op, int e, int nb, int kb) {
    return op.w + ((static_cast<size_t>(e) * op.NB + nb) * op.KB + kb) * kTile;
}

// Bounded spin until *flag == want (acquire).  On timeout records the error,
// sets the CTA's abort flag and returns false.
__device__ __forceinline__ bool wait_flag(const int* flag, int want, int* status, volatile int* abort) {
    if (ld_acquire(flag) == want) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire(flag) == want) return true;
        if ((i & 31u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                record_error(status, MOEQ_ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void producer(const StreamArgs& a, SmemTail& sm, uint8_t* stages, int epoch) {
    const uint64_t pol = l2_evict_first_policy();
    long long issued = 0;
    int U = 0;
    bool have_plan = !a.fused_route;
    for (int li = 0; li < a.n_lists; ++li) {
        if (list_needs_plan(a, li)) {
            if (!have_plan) {
                wait_flag(a.route_flag, epoch, a.status, &sm.abort_flag);
                have_plan = true;
            }
            U = __ldcg(a.n_uniq);
            if (U < 0 || U > a.max_uniq) U = 0;  // reported by the consumers
        }
        const ListInfo L = list_info(a, li, U);
        const Operand& op = a.op[L.kind];
        int cur = -1, expert = 0;
        for (long long u = L.lo; u < L.hi; ++u) {
            const int e_local = static_cast<int>(u / (static_cast<long long>(L.RB) * L.KU));
            const int rem = static_cast<int>(u % (static_cast<long long>(L.RB) * L.KU));
            const int rb = rem / L.KU, ku = rem % L.KU;
            if (e_local != cur) {
                cur = e_local;
                expert = L.src == kSrcShared ? a.shared_id : __ldcg(a.uniq + e_local);
                if (expert < 0 || expert >= a.n_experts) expert = 0;
            }
            const int s = static_cast<int>(issued % kStages);
            if (issued >= kStages) {
                if (!mbar_wait_bounded(&sm.empty[s], static_cast<uint32_t>((issued / kStages - 1) & 1),
                                       &sm.abort_flag)) {
                    record_error(a.status, MOEQ_ERR_TIMEOUT);
                    sm.abort_flag = 1;
                }
            }
            if (sm.abort_flag) goto drain;
            {
                uint8_t* dst = stages + static_cast<size_t>(s) * kStageBytes;
                if (L.kind == kKindGU) {
                    mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
                    bulk_load(dst, tile_ptr(op, expert, rb, ku), kTile, &sm.full[s], pol);
                    bulk_load(dst + kTile, tile_ptr(op, expert, L.RB + rb, ku), kTile, &sm.full[s], pol);
                } else {
                    const int nt = min(2, op.KB - 2 * ku);
                    mbar_arrive_expect_tx(&sm.full[s], nt * kTile);
                    bulk_load(dst, tile_ptr(op, expert, rb, 2 * ku), nt * kTile, &sm.full[s], pol);
                }
            }
            ++issued;
        }
    }
    return;
drain:
    // Let the copies already issued land before the CTA may exit (bounded).
    for (long long j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&sm.full[j % kStages], static_cast<uint32_t>((j / kStages) & 1)) &&
               global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
        }
    }
}

// ------------------------------------------------------------------ consumers
// Quantise activation groups [g0, g1) of the segment's tokens into shared
// memory (decoded values and scales).  Loads are issued four items at a time.
// Out of line: it runs once per chunk and its division sequences would
// otherwise crowd the registers of the streaming loop.
template <bool kF32>
__device__ __noinline__ void quantise(const StreamArgs& a, const Operand& op, SmemTail& sm, const ExpertRef& r,
                                      int g0, int g1, bool dump, int cw, int lane) {
    const int ng = g1 - g0;
    const int items = r.ntok * ng;
    for (int base = cw; base < items; base += 4 * kCW) {
        float4 v[4];
        int row[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int item = base + b * kCW;
            row[b] = -1;
            if (item < items) {
                const int t = item / ng, gg = g0 + item % ng;
                const int p = r.p0 + t;
                // gate_up reads token rows (the shared expert's pairs are tokens
                // 0..M-1 before any plan exists); down reads pair rows.
                int rr = op.a_row ? (r.shared_static ? t : __ldcg(op.a_row + p)) : p;
                if (rr < 0 || rr >= op.rows_a) {
                    if (lane == 0) record_error(a.status, MOEQ_ERR_INVALID_ARG);
                    rr = 0;
                }
                row[b] = rr;
                v[b] = load_act4<kF32>(op.a, static_cast<size_t>(op.K), rr, gg * kGroup + lane * 4);
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int item = base + b * kCW;
            if (item >= items) break;
            const int t = item / ng, gl = item % ng, gg = g0 + gl;
            float s;
            float4 dec;
            const uint32_t codes = quant_group_warp(v[b], &s, &dec);
            *reinterpret_cast<float4*>(sm.act + (t * ng + gl) * kGroup + act_pos(lane * 4)) = dec;
            if (lane == 0) sm.act_s[t * ng + gl] = s;
            if (dump) {
                *reinterpret_cast<uint32_t*>(op.qdump + static_cast<size_t>(row[b]) * op.K + gg * kGroup +
                                             lane * 4) = codes;
                if (lane == 0) op.sdump[static_cast<size_t>(row[b]) * op.KB + gg] = s;
            }
        }
    }
}

// Per lane and pass: dot product of its 16 weight bytes (row `rows_base +
// 4p + lane/8`, logical chunk lane%8) with the matching decoded activations
// of tokens t0 .. t0+MT-1 (loads clamped to the last token).
template <int MT, int PASSES>
__device__ __forceinline__ void tile_dot(const uint8_t* tile, int rows_base, const float* act_g, int tok_ld, int t0,
                                         int ntok, int lane, float (&part)[PASSES][MT]) {
    const int l8 = lane & 7, rsub = lane >> 3;
    float2 av[MT][8];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const float4* ap = reinterpret_cast<const float4*>(act_g + min(t0 + t, ntok - 1) * tok_ld);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ap[i * 8 + l8];
            av[t][2 * i] = make_float2(v.x, v.y);
            av[t][2 * i + 1] = make_float2(v.z, v.w);
        }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int row = rows_base + p * 4 + rsub;
        const uint4 w = *reinterpret_cast<const uint4*>(tile + row * 128 + ((l8 ^ (row & 7)) << 4));
        float2 wf[8];
        e4m3x4_to_f32(w.x, wf[0], wf[1]);
        e4m3x4_to_f32(w.y, wf[2], wf[3]);
        e4m3x4_to_f32(w.z, wf[4], wf[5]);
        e4m3x4_to_f32(w.w, wf[6], wf[7]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float2 d = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 8; ++j) d = __ffma2_rn(wf[j], av[t][j], d);
            part[p][t] = d.x + d.y;
        }
    }
}

// As tile_dot for tokens T0 .. T0+MT-1, but folds each pass straight into
// running sums: acc[p][T0 + t] += dot * scl[T0 + t].
template <int MT, int PASSES, int T0, int MTOT>
__device__ __forceinline__ void tile_dot_acc(const uint8_t* tile, int rows_base, const float* act_g, int tok_ld,
                                             int ntok, int lane, const float (&scl)[MTOT],
                                             float (&acc)[PASSES][MTOT]) {
    const int l8 = lane & 7, rsub = lane >> 3;
    float2 av[MT][8];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const float4* ap = reinterpret_cast<const float4*>(act_g + min(T0 + t, ntok - 1) * tok_ld);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ap[i * 8 + l8];
            av[t][2 * i] = make_float2(v.x, v.y);
            av[t][2 * i + 1] = make_float2(v.z, v.w);
        }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int row = rows_base + p * 4 + rsub;
        const uint4 w = *reinterpret_cast<const uint4*>(tile + row * 128 + ((l8 ^ (row & 7)) << 4));
        float2 wf[8];
        e4m3x4_to_f32(w.x, wf[0], wf[1]);
        e4m3x4_to_f32(w.y, wf[2], wf[3]);
        e4m3x4_to_f32(w.z, wf[4], wf[5]);
        e4m3x4_to_f32(w.w, wf[6], wf[7]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float2 d = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 8; ++j) d = __ffma2_rn(wf[j], av[t][j], d);
            acc[p][T0 + t] = fmaf(d.x + d.y, scl[T0 + t], acc[p][T0 + t]);
        }
    }
}

__device__ __forceinline__ float reduce8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

// One segment: units [ku0, ku1) of row block rb of expert r.  Leaves one sum
// per (unit row, token) in sm.acc.  MODE 1/2/4: up to that many tokens with
// running sums in registers; MODE 0: any count, two tokens at a time, each
// K group reduced across lanes into sm.acc.
template <int KIND, bool kF32, int MODE>
__device__ __forceinline__ void run_segment(const StreamArgs& a, SmemTail& sm, const uint8_t* stages,
                                            const ExpertRef& r, int rb, int ku0, int ku1, bool dump, int cw,
                                            int lane, int ctid, long long& it) {
    const Operand& op = a.op[KIND];
    constexpr int MT = MODE == 0 ? 2 : MODE;
    constexpr int PASSES = KIND == kKindGU ? 4 : 2;   // 4-row passes per warp and tile
    constexpr int GPU = KIND == kKindGU ? 1 : 2;      // K groups per unit
    // gate_up: warp w covers rows (w%8)*16.. of tile w/8; down: rows w*8.. of both tiles
    const int tile_w = KIND == kKindGU ? (cw >> 3) : 0;
    const int rows_base = KIND == kKindGU ? (cw & 7) * 16 : cw * 8;
    const int acc_row0 = KIND == kKindGU ? tile_w * 128 + rows_base : rows_base;
    if (MODE == 0)
        for (int i = ctid; i < kUnitRows * kMaxTok; i += kConsumers) sm.acc[(i / kMaxTok) * kAccLd + i % kMaxTok] = 0.f;
    float acc[PASSES][MT];
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[p][t] = 0.0f;

    const int upc = max(1, (kActCap / (kGroup * r.ntok)) / GPU);  // units per activation chunk
    for (int ua = ku0; ua < ku1; ua += upc) {
        const int ub = min(ku1, ua + upc);
        const int g0 = ua * GPU, g1 = min(op.KB, ub * GPU);
        consumer_sync();   // activation buffer free
        quantise<kF32>(a, op, sm, r, g0, g1, dump, cw, lane);
        consumer_sync();   // activation buffer full
        const int ng = g1 - g0;
        const int tok_ld = ng * kGroup;
        for (int ku = ua; ku < ub; ++ku, ++it) {
            const int s = static_cast<int>(it % kStages);
            if (!mbar_wait_bounded(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), &sm.abort_flag)) {
                // Keep the control flow (and so every named barrier) identical
                // across the consumer warps; the results are void.
                record_error(a.status, MOEQ_ERR_TIMEOUT);
                sm.abort_flag = 1;
            }
            const uint8_t* st = stages + static_cast<size_t>(s) * kStageBytes;
            const int ntile = KIND == kKindGU ? 1 : min(2, op.KB - 2 * ku);
            for (int tt = 0; tt < ntile; ++tt) {
                const int g = KIND == kKindGU ? ku : 2 * ku + tt;
                const uint8_t* tile = st + (KIND == kKindGU ? tile_w : tt) * kTile;
                const float* act_g = sm.act + (g - g0) * kGroup;
                const float swg = sm.sw[tile_w][g - ku0 * GPU];
                if (MODE != 0) {
                    float scl[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) scl[t] = sm.act_s[min(t, r.ntok - 1) * ng + (g - g0)] * swg;
                    if (MT <= 2) {
                        tile_dot_acc<MT, PASSES, 0, MT>(tile, rows_base, act_g, tok_ld, r.ntok, lane, scl, acc);
                    } else {  // four tokens as two pairs: fewer live registers
                        tile_dot_acc<2, PASSES, 0, MT>(tile, rows_base, act_g, tok_ld, r.ntok, lane, scl, acc);
                        tile_dot_acc<2, PASSES, 2, MT>(tile, rows_base, act_g, tok_ld, r.ntok, lane, scl, acc);
                    }
                } else {
                    for (int t0 = 0; t0 < r.ntok; t0 += 2) {
                        float part[PASSES][2];
                        tile_dot<2, PASSES>(tile, rows_base, act_g, tok_ld, t0, r.ntok, lane, part);
#pragma unroll
                        for (int p = 0; p < PASSES; ++p) {
                            const int row = acc_row0 + p * 4 + (lane >> 3);
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const float v = reduce8(part[p][t]);
                                if ((lane & 7) == 0 && t0 + t < r.ntok)
                                    sm.acc[row * kAccLd + t0 + t] += v * (sm.act_s[(t0 + t) * ng + (g - g0)] * swg);
                            }
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
        for (int p = 0; p < PASSES; ++p) {
            const int row = acc_row0 + p * 4 + (lane >> 3);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v = reduce8(acc[p][t]);
                if ((lane & 7) == 0 && t < r.ntok) sm.acc[row * kAccLd + t] = v;
            }
        }
    }
}

// The wide-token modes run out of line so that their register needs do not
// constrain the one- and two-token loops (the common case at M <= 16).
template <int KIND, bool kF32, int MODE>
__device__ __noinline__ void run_segment_cold(const StreamArgs& a, SmemTail& sm, const uint8_t* stages,
                                              const ExpertRef& r, int rb, int ku0, int ku1, bool dump, int cw,
                                              int lane, int ctid, long long& it) {
    run_segment<KIND, kF32, MODE>(a, sm, stages, r, rb, ku0, ku1, dump, cw, lane, ctid, it);
}

// Epilogue of a finished row block: gate_up -> h = silu(gate) * up and, in
// the layer, the readiness flag of (expert, row block); down -> y and, in the
// layer, the combine of every token whose last expert this was.
template <int KIND>
__device__ __forceinline__ void epilogue(const StreamArgs& a, SmemTail& sm, const ExpertRef& r, int rb, int ctid,
                                         int epoch) {
    const Operand& op = a.op[KIND];
    if (r.valid) {
        for (int idx = ctid; idx < 128 * r.ntok; idx += kConsumers) {
            const int i = idx & 127, t = idx >> 7;
            float* o = op.out + static_cast<size_t>(r.p0 + t) * op.out_ld + rb * 128 + i;
            if (KIND == kKindGU) {
                const float g = sm.acc[i * kAccLd + t];
                const float u = sm.acc[(128 + i) * kAccLd + t];
                *o = __fdiv_rn(g, 1.0f + expf(-g)) * u;
            } else {
                *o = sm.acc[i * kAccLd + t];
            }
        }
    }
    if (KIND == kKindGU && a.fused_route) {
        __threadfence();
        consumer_sync();
        if (ctid == 0) st_release(a.h_ready + static_cast<size_t>(r.slot) * op.RB + rb, epoch);
    }
    if (KIND == kKindDN && a.fused_combine) {
        __threadfence();
        if (ctid == 0) sm.n_comb = 0;
        consumer_sync();
        if (ctid < r.ntok && r.valid) {
            const int tok = r.shared_static ? ctid : __ldcg(a.pair_tok + r.p0 + ctid);
            if (tok >= 0 && tok < a.M) {
                const int old = atomicAdd(a.comb + tok * op.RB + rb, 1);
                if (old == a.top_k) sm.comb_tok[atomicAdd(&sm.n_comb, 1)] = tok;
            }
        }
        consumer_sync();
        const int nc = sm.n_comb;
        if (nc) __threadfence();
        for (int j = 0; j < nc; ++j) {
            const int tok = sm.comb_tok[j];
            if (ctid < 128) {
                const int n = rb * 128 + ctid;
                const int* po = a.pair_of + tok * (a.top_k + 1);
                float accv = __ldcg(op.out + static_cast<size_t>(__ldcg(po + a.top_k)) * op.out_ld + n);
                for (int jj = 0; jj < a.top_k; ++jj)
                    accv = fmaf(__ldcg(a.topk_w + tok * a.top_k + jj),
                                __ldcg(op.out + static_cast<size_t>(__ldcg(po + jj)) * op.out_ld + n), accv);
                a.out_bf16[static_cast<size_t>(tok) * op.out_ld + n] = __float2bfloat16_rn(accv);
            }
            if (ctid == 0) a.comb[tok * op.RB + rb] = 0;
        }
    }
}

template <int KIND, bool kF32>
__device__ __forceinline__ void run_list(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, int li, int U, int cw, int lane,
                         int ctid, long long& it, int epoch) {
    const ListInfo L = list_info(a, li, U);
    const Operand& op = a.op[KIND];
    constexpr int kRows = KIND == kKindGU ? 256 : 128;
    const long long upe = static_cast<long long>(L.RB) * L.KU;
    long long u = L.lo;
    while (u < L.hi) {
        const int e_local = static_cast<int>(u / upe);
        const int rem = static_cast<int>(u % upe);
        const int rb = rem / L.KU, ku0 = rem % L.KU;
        const long long seg_end = min(L.hi, u - ku0 + L.KU);
        const int ku1 = ku0 + static_cast<int>(seg_end - u);
        ExpertRef r = expert_ref(a, L.src, e_local);
        if (!r.valid) {
            if (ctid == 0) record_error(a.status, MOEQ_ERR_INVALID_ARG);
            r.expert = 0;
            r.p0 = 0;
            r.ntok = 1;
        }
        // down in the layer: this expert's h must be complete (bounded wait)
        if (KIND == kKindDN && a.fused_route && ctid == 0) {
            const int nrb = a.op[kKindGU].RB;
            for (int j = 0; j < nrb; ++j)
                if (!wait_flag(a.h_ready + static_cast<size_t>(r.slot) * nrb + j, epoch, a.status, &sm.abort_flag))
                    break;
        }
        consumer_sync();   // previous segment's readers of sw / acc are done; h is ready
        const int nsw = KIND == kKindGU ? (ku1 - ku0) : (min(op.KB, 2 * ku1) - 2 * ku0);
        for (int i = ctid; i < nsw * (KIND == kKindGU ? 2 : 1); i += kConsumers) {
            const int b = i / nsw, gl = i % nsw;
            const int g = (KIND == kKindGU ? ku0 : 2 * ku0) + gl;
            const int nb = rb + (b ? L.RB : 0);
            sm.sw[b][gl] = __ldg(op.sw + (static_cast<size_t>(r.expert) * op.NB + nb) * op.KB + g);
        }
        const bool dump = r.valid && op.qdump != nullptr && rb == 0 &&
                          (KIND == kKindDN || r.shared_static || e_local == L.n_exp - 1);
        if (r.ntok <= 1)
            run_segment<KIND, kF32, 1>(a, sm, stages, r, rb, ku0, ku1, dump, cw, lane, ctid, it);
        else if (r.ntok <= 2)
            run_segment<KIND, kF32, 2>(a, sm, stages, r, rb, ku0, ku1, dump, cw, lane, ctid, it);
        else if (r.ntok <= 4)
            run_segment_cold<KIND, kF32, 4>(a, sm, stages, r, rb, ku0, ku1, dump, cw, lane, ctid, it);
        else
            run_segment_cold<KIND, kF32, 0>(a, sm, stages, r, rb, ku0, ku1, dump, cw, lane, ctid, it);
        consumer_sync();

        if (ku0 == 0 && ku1 == L.KU) {
            epilogue<KIND>(a, sm, r, rb, ctid, epoch);
        } else {
            const long long rblk = static_cast<long long>(e_local) * L.RB + rb;
            const long long c_lo = cta_of_unit(rblk * L.KU, L.T, L.G);
            const long long c_hi = cta_of_unit(rblk * L.KU + L.KU - 1, L.T, L.G);
            float* part_base = a.partials + static_cast<size_t>(li) * a.partial_list_floats;
            const int my_slot = static_cast<int>(2 * L.c + ((L.lo / L.KU) == rblk ? 0 : 1));
            float* mine = part_base + static_cast<size_t>(my_slot) * kMaxTok * kRows;
            for (int idx = ctid; idx < kRows * r.ntok; idx += kConsumers) {
                const int row = idx % kRows, t = idx / kRows;
                mine[t * kRows + row] = sm.acc[row * kAccLd + t];
            }
            __threadfence();
            consumer_sync();
            if (ctid == 0) {
                int n = 0;
                for (long long cc = c_lo; cc <= c_hi; ++cc) n += unit_lo(cc, L.T, L.G) < unit_lo(cc + 1, L.T, L.G);
                const int old = atomicAdd(a.tickets[li] + rblk, 1);
                sm.last_flag = (old == n - 1);
            }
            consumer_sync();
            if (sm.last_flag) {
                __threadfence();
                for (int idx = ctid; idx < kRows * r.ntok; idx += kConsumers) {
                    const int row = idx % kRows, t = idx / kRows;
                    float v = 0.0f;
                    for (long long cc = c_lo; cc <= c_hi; ++cc) {
                        const long long lo = unit_lo(cc, L.T, L.G);
                        if (lo >= unit_lo(cc + 1, L.T, L.G)) continue;
                        const int slot = static_cast<int>(2 * cc + ((lo / L.KU) == rblk ? 0 : 1));
                        v += __ldcg(part_base + (static_cast<size_t>(slot) * kMaxTok + t) * kRows + row);
                    }
                    sm.acc[row * kAccLd + t] = v;
                }
                consumer_sync();
                if (ctid == 0) a.tickets[li][rblk] = 0;
                epilogue<KIND>(a, sm, r, rb, ctid, epoch);
            }
        }
        u = seg_end;
    }
}

struct ConsumerSync {
    __device__ __forceinline__ void operator()() const { consumer_sync(); }
};

template <bool kGuF32, bool kDnF32>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemTail& sm = *reinterpret_cast<SmemTail*>(stages + static_cast<size_t>(kStages) * kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCW);
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    const int epoch = a.fused_route ? ld_relaxed(a.epoch) + 1 : 0;
    __syncthreads();

    if (warp == kCW) {
        if (lane == 0) producer(a, sm, stages, epoch);
        return;
    }

    const int cw = warp, ctid = tid;
    if (a.fused_route && blockIdx.x == 0) {
        route_compute<kConsumers>(a.logits, a.M, a.E_routed, a.top_k, a.plan, sm.route, ctid, ConsumerSync{});
        __threadfence();
        consumer_sync();
        if (ctid == 0) st_release(a.route_flag, epoch);
    }
    long long it = 0;
    int U = 0;
    bool have_plan = !a.fused_route;
    for (int li = 0; li < a.n_lists; ++li) {
        if (list_needs_plan(a, li)) {
            if (!have_plan) {
                if (ctid == 0) wait_flag(a.route_flag, epoch, a.status, &sm.abort_flag);
                consumer_sync();
                have_plan = true;
            }
            U = __ldcg(a.n_uniq);
            if (U < 0 || U > a.max_uniq) {
                if (ctid == 0) record_error(a.status, MOEQ_ERR_INVALID_ARG);
                U = 0;
            }
        }
        if (a.list_kind[li] == kKindGU)
            run_list<kKindGU, kGuF32>(a, sm, stages, li, U, cw, lane, ctid, it, epoch);
        else
            run_list<kKindDN, kDnF32>(a, sm, stages, li, U, cw, lane, ctid, it, epoch);
    }

    if (a.fused_route) {
        // The last CTA to finish publishes the epoch for the next launch.
        consumer_sync();
        if (ctid == 0) {
            __threadfence();
            const int old = atomicAdd(a.done, 1);
            if (old == static_cast<int>(gridDim.x) - 1) {
                *a.done = 0;
                __threadfence();
                st_release(a.epoch, epoch);
            }
        }
    }
}

size_t stream_partials_floats(int grid) { return static_cast<size_t>(2) * grid * kMaxTok * kUnitRows; }

template <bool G32, bool D32>
static cudaError_t launch_t(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(stream_kernel<G32, D32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = cooperative ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_kernel<G32, D32>, args);
}

cudaError_t launch_stream(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    const bool g = args.op[kKindGU].a_f32 != 0, d = args.op[kKindDN].a_f32 != 0;
    if (g) return d ? launch_t<true, true>(args, grid, cooperative, stream) : launch_t<true, false>(args, grid, cooperative, stream);
    return d ? launch_t<false, true>(args, grid, cooperative, stream) : launch_t<false, false>(args, grid, cooperative, stream);
}

}  // namespace moeq
