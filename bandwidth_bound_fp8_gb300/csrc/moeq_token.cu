// The one-token MoE layer kernel: route, live quantisation of x, gate_up +
// SwiGLU, live quantisation of h, down and the combine for a single token,
// in one launch with no CTA ever waiting for another.
//
// GLM-5.2 x10 is the source of the method: decode streams every active
// expert's FP8 weights from HBM once with little arithmetic on top
// (bandwidth model: at batch 1 a layer is a read of its top-8 experts plus
// the shared one); the activations are quantised to FP8 live in front of each
// GEMM (§1, §8c), fused into the GEMM rather than round-tripping through HBM
// (§4, "PQ-GEMM"); K is split so that every SM streams (§1, split-K).
//
// Work.  A column is one (expert slot, kb): the gate rows kb*128.. and the up
// rows I+kb*128.. of gate_up over all of H (2 x H/128 tiles), then down's K
// group kb -- the 128 h values this column produces -- against all of down's
// H rows (H/128 tiles).  At the layer's shapes that is 9 slots x 16 = 144
// columns of 2.25 MB on 152 SMs, one per CTA.  gate_up never leaves the CTA:
// the h group a column needs for its down is the one it just computed.  Down
// leaves, per 256-row unit of the output, one fp32 partial per column and
// counts itself in (a release add on the unit's counter in the workspace).
// A unit's 16 parts (16 rows each) are summed, and the bf16 output formed, by
// warps that have nothing else to do: those of the CTAs without a column
// (or, with none to spare, every CTA once its stream is done), each waiting
// for its unit's count to reach ncols.  The streams themselves never wait for another CTA, and a CTA that
// finds no part left exits.  Every CTA takes the down units in the same order
// (the measured faster DRAM pattern), so the units complete one after another
// as the slowest stream passes them, and their sums overlap the rest of it.
//
// Warp roles (576 threads, one CTA per SM):
//   warps 0-15  consumers: per 32 KiB stage, each lane widens 16 weight bytes
//               of a row exactly to fp32 and accumulates paired fp32 FMAs with
//               the decoded activation codes (x for gate_up, h for down);
//   warp 16     producer: routes (all lanes), then one lane issues the bulk
//               copies of every stage into a ring of kStages;
//   warp 17     ticket warp: as the consumers store down partials it counts
//               them in (one gpu-scope fence per batch of arrivals).
// Launched with programmatic dependent launch: the next kernel's CTAs may
// start as this one's exit; everything before griddepcontrol.wait only reads
// weights (which nothing writes) and this CTA's own shared memory.
#include "moeq_device.cuh"
#include "moeq_internal.h"
#include "moeq_route.cuh"

namespace moeq {
namespace {

constexpr int kCW = 16;                        // consumer warps
constexpr int kConsumers = kCW * 32;
constexpr int kProducerWarp = kCW;
constexpr int kTicketWarp = kCW + 1;
constexpr int kThreads = (kCW + 2) * 32;
constexpr int kTile = 16384;
constexpr int kStageBytes = 2 * kTile;
constexpr int kStages = 4;
constexpr int kMaxKB = kTokenMaxH / 128;       // K groups of x
constexpr int kMaxUnits = kTokenMaxH / 256;    // 256-row output units of down
constexpr int kParts = kCW;                    // a unit's rows split by consumer warp (16 rows each)
constexpr int kTailUnits = 4;                  // the last down units, summed by the column CTAs

struct Smem {
    alignas(16) float xdec[kTokenMaxH];   // decoded x codes, each group in the consumer layout
    float xs[kMaxKB];                  // x scales
    float swg[2][kMaxKB];              // the column's gate and up weight-scale rows
    float swd[2 * kMaxUnits];          // the column's down weight scales, one per row block
    float gsum[256];                   // the column's gate (0..127) and up (128..255) sums
    alignas(16) float hdec[128];       // decoded h codes (consumer layout) ...
    float hs;                          // ... and their scale
    int topk_id[kTokenMaxTopK];
    float topk_w[kTokenMaxTopK];
    int uniq[kTokenMaxTopK];           // routed experts, ascending
    int pick_rank[kTokenMaxTopK];      // position of pick j in uniq
    int slot_pick[kTokenMaxTopK];      // the pick at position s of uniq
    float rvals[kTokenMaxTopK];        // picked logits (routing scratch)
    int wdone[kCW];                    // down partials stored, per consumer warp (monotonic)
    int abort_flag;
    uint64_t full[kStages], empty[kStages];
    uint64_t plan_bar;
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(offsetof(Smem, xdec) % 16 == 0 && offsetof(Smem, hdec) % 16 == 0, "float4 accesses");
static_assert((static_cast<size_t>(kStages) * kStageBytes) % 1024 == 0, "the tail starts 1024-aligned");

__device__ __forceinline__ void consumer_sync() { named_sync(1, kConsumers); }
__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Smem& sm, int* status) {
    if (mbar_wait_sleep_bounded(bar, parity, &sm.abort_flag)) return true;
    record_error(status, MOEQ_ERR_TIMEOUT);
    sm.abort_flag = 1;
    return false;
}

// Position of element k (0..127) of a group in the consumer layout: lane l8
// reads its four float4 (k = 16*l8 + 4i .. +3) at (8i + l8)*4, so the eight
// lanes of a row read eight consecutive 16-byte chunks.
__device__ __forceinline__ int act_pos(int k) { return (((k & 15) >> 2) * 8 + (k >> 4)) * 4 + (k & 3); }

// Column j of the launch: slot group g = j / RB (0: the shared expert,
// g >= 1: the routed expert uniq[g - 1]) and K group kb of down.
struct Column {
    int g, kb, expert, pair;
};

__device__ __forceinline__ Column column(const TokenArgs& a, const Smem& sm, int j) {
    Column c;
    c.g = j / a.RB;
    c.kb = j - c.g * a.RB;
    c.expert = c.g == 0 ? a.E_routed : sm.uniq[c.g - 1];
    c.pair = c.g == 0 ? a.top_k : c.g - 1;   // pairs of the plan: routed in uniq order, then shared
    return c;
}

__device__ __forceinline__ const uint8_t* gu_tile(const TokenArgs& a, int e, int nb, int kb) {
    return a.w_gu + ((static_cast<size_t>(e) * (2 * a.RB) + nb) * a.KB + kb) * kTile;
}
__device__ __forceinline__ const uint8_t* dn_tile(const TokenArgs& a, int e, int nb, int kb) {
    return a.w_d + ((static_cast<size_t>(e) * a.KB + nb) * a.RB + kb) * kTile;
}

// The down units in stream order (the same for every CTA).
__device__ __forceinline__ int unit_of(const TokenArgs&, int i) { return i; }

// ------------------------------------------------------------------ producer
// Issues stage t (0 .. KB-1 gate_up, then KB/2 down units) of column col.
__device__ __forceinline__ void issue_stage(const TokenArgs& a, Smem& sm, uint8_t* stages, const Column& col, int t,
                                            long long n, uint64_t pol) {
    const int s = static_cast<int>(n % kStages);
    uint8_t* dst = stages + static_cast<size_t>(s) * kStageBytes;
    mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
    if (t < a.KB) {
        bulk_load(dst, gu_tile(a, col.expert, col.kb, t), kTile, &sm.full[s], pol);
        bulk_load(dst + kTile, gu_tile(a, col.expert, a.RB + col.kb, t), kTile, &sm.full[s], pol);
    } else {
        const int u = unit_of(a, t - a.KB);
        bulk_load(dst, dn_tile(a, col.expert, 2 * u, col.kb), kTile, &sm.full[s], pol);
        bulk_load(dst + kTile, dn_tile(a, col.expert, 2 * u + 1, col.kb), kTile, &sm.full[s], pol);
    }
}

// The shared expert's weights need no plan and no input: every CTA starts
// its share of them (one 16 KiB tile per lane) towards L2 before it waits for
// the previous kernel, so that HBM streams through that kernel's tail and
// this one's routing; the shared expert's CTAs then find them in L2.
__device__ __forceinline__ void prefetch_shared_expert(const TokenArgs& a, int lane) {
    const long long G = gridDim.x, c = blockIdx.x;
    const long long gu_tiles = 2LL * a.RB * a.KB, tiles = gu_tiles + static_cast<long long>(a.KB) * a.RB;
    const long long lo = tiles * c / G, hi = tiles * (c + 1) / G;
    for (long long t = lo + lane; t < hi; t += 32) {
        const uint8_t* src = t < gu_tiles ? gu_tile(a, a.E_routed, 0, 0) + t * kTile
                                          : dn_tile(a, a.E_routed, 0, 0) + (t - gu_tiles) * kTile;
        bulk_prefetch_l2(src, kTile);
    }
}

// Routing of the one token (GLM-5.2 x10 bandwidth model: its top-8 experts).
template <int NPER>
__device__ __forceinline__ void route_one_token(const TokenArgs& a, Smem& sm, int lane) {
    uint32_t key[NPER];
    route_load_keys<NPER>(a.logits, a.E_routed, lane, key);
    route_topk_keys<NPER>(key, a.E_routed, a.top_k, lane, sm.topk_id, sm.rvals);
}

// Routing of the token by the producer warp: top-k with ties to the lower
// id, softmax over the picks, picks sorted by id into the slots; CTA 0 also
// writes the plan out.
__device__ void producer_route(const TokenArgs& a, Smem& sm, int lane) {
    const int k = a.top_k;
    if (a.E_routed <= 256)
        route_one_token<8>(a, sm, lane);
    else
        route_one_token<kRouteMaxE / 32>(a, sm, lane);
    __syncwarp();
    float ex = 0.0f;
    int id = 0x7fffffff;
    if (lane < k) {
        ex = expf(sm.rvals[lane] - sm.rvals[0]);
        id = sm.topk_id[lane];
    }
    float den = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += __shfl_sync(0xffffffffu, id, i) < id;
    const float w = lane < k ? __fdiv_rn(ex, den) : 0.0f;
    if (lane < k) {
        sm.topk_w[lane] = w;
        sm.uniq[rank] = id;
        sm.pick_rank[lane] = rank;
        sm.slot_pick[rank] = lane;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.plan_bar);
    if (blockIdx.x == 0) {
        // CTA 0 hands the plan to the caller (one token: every routed expert
        // has one pair, in uniq order; the shared expert's pair is last)
        const moeq_route_plan& p = a.plan;
        if (lane < k) {
            p.topk_id[lane] = id;
            p.topk_w[lane] = w;
            p.uniq[rank] = id;
            p.offs[lane] = lane;
            p.pair_tok[lane] = 0;
            p.pair_of[lane] = rank;
        }
        if (lane == 0) {
            p.uniq[k] = a.E_routed;
            p.offs[k] = k;
            p.offs[k + 1] = k + 1;
            p.pair_tok[k] = 0;
            p.pair_of[k] = k;
            *p.n_uniq = k + 1;
        }
    }
}

__device__ void producer_warp(const TokenArgs& a, Smem& sm, uint8_t* stages, int lane) {
    const int G = gridDim.x, c = blockIdx.x, k = a.top_k;
    const int stages_per_col = a.KB + a.KB / 2;
    const uint64_t pol = l2_evict_first_policy();
    long long issued = 0;
    // The logits and x are the previous kernel's to write until
    // griddepcontrol.wait; their lines can still be brought into L2 now (L2
    // is where every SM's writes meet), so the reads after the wait are hits.
    {
        const int lg_lines = (a.E_routed * 4 + 127) / 128, x_lines = (a.H * 2 + 127) / 128;
        for (int i = lane; i < lg_lines + x_lines; i += 32)
            prefetch_l2(i < lg_lines ? reinterpret_cast<const char*>(a.logits) + 128 * i
                                     : reinterpret_cast<const char*>(a.x) + 128 * (i - lg_lines));
    }
    prefetch_shared_expert(a, lane);
    // The shared expert's columns (the first RB) need no plan: start them now.
    // When the logits are known not to come from the kernel ahead, the token
    // is routed now too, and a routed first column starts as well.
    const bool routed_now = a.route_early && k > 0;
    if (routed_now) producer_route(a, sm, lane);
    int pre = 0;
    if (c < a.ncols && (c < a.RB || routed_now)) {
        const Column col = column(a, sm, c);
        pre = min(kStages, stages_per_col);
        if (lane == 0)
            for (int t = 0; t < pre; ++t) issue_stage(a, sm, stages, col, t, issued++, pol);
    }
    issued = pre;
    pdl_wait();
    if (k == 0) {   // a dense FFN: the one expert, no routing
        if (lane == 0) mbar_arrive(&sm.plan_bar);
    } else if (!routed_now) {
        producer_route(a, sm, lane);
    }
    if (lane != 0) return;
    for (int j = c; j < a.ncols && !sm.abort_flag; j += G) {
        const Column col = column(a, sm, j);
        for (int t = (j == c ? pre : 0); t < stages_per_col; ++t) {
            const int s = static_cast<int>(issued % kStages);
            if (issued >= kStages &&
                !wait_or_abort(&sm.empty[s], static_cast<uint32_t>((issued / kStages - 1) & 1), sm, a.status))
                break;
            issue_stage(a, sm, stages, col, t, issued++, pol);
        }
    }
    if (sm.abort_flag) {
        // let the copies in flight land before the CTA may exit (bounded)
        for (long long i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&sm.full[i % kStages], static_cast<uint32_t>((i / kStages) & 1)) &&
                   global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
            }
        }
    }
}

// ------------------------------------------------------------------ consumers
// Sum of four per-lane partials (rows 4p + rsub, p = 0..3) over the eight
// lanes of each row, transposed: returns, in every lane, the full sum of row
// 4 * (l8 >> 1) + rsub (lanes l8 and l8 ^ 1 hold the same value).
__device__ __forceinline__ float reduce_rows4(float d0, float d1, float d2, float d3, int l8) {
    const bool b2 = (l8 & 4) != 0, b1 = (l8 & 2) != 0;
    float k0 = b2 ? d2 : d0, k1 = b2 ? d3 : d1;
    const float s0 = b2 ? d0 : d2, s1 = b2 ? d1 : d3;
    k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
    float kk = b1 ? k1 : k0;
    const float ss = b1 ? k0 : k1;
    kk += __shfl_xor_sync(0xffffffffu, ss, 2);
    kk += __shfl_xor_sync(0xffffffffu, kk, 1);
    return kk;
}

// Lane's 16 weight bytes of a row (logical chunk l8) dotted with its 16
// activation values: paired fp32 FMAs on exactly widened E4M3 codes.
__device__ __forceinline__ float row_dot(const uint8_t* tile, int row, int l8, const float2 (&av)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(tile + row * 128 + ((l8 ^ (row & 7)) << 4));
    float2 wf[8];
    e4m3x4_to_f32(w.x, wf[0], wf[1]);
    e4m3x4_to_f32(w.y, wf[2], wf[3]);
    e4m3x4_to_f32(w.z, wf[4], wf[5]);
    e4m3x4_to_f32(w.w, wf[6], wf[7]);
    float2 d = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) d = __ffma2_rn(wf[j], av[j], d);
    return d.x + d.y;
}

__device__ __forceinline__ void load_act(const float* grp, int l8, float2 (&av)[8]) {
    const float4* ap = reinterpret_cast<const float4*>(grp);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v = ap[i * 8 + l8];
        av[2 * i] = make_float2(v.x, v.y);
        av[2 * i + 1] = make_float2(v.z, v.w);
    }
}

// Live quantisation of x (GLM-5.2 x10 §1, §8c: 1 x 128 groups, s = amax/448,
// RNE to E4M3): every CTA quantises all of x into its shared memory; the
// warp's groups are all loaded before any is quantised.
__device__ void quantise_x(const TokenArgs& a, Smem& sm, int cw, int lane) {
    constexpr int kPer = kMaxKB / kCW;
    float4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int g = cw + i * kCW;
        v[i] = g < a.KB ? load_act4<false>(a.x, static_cast<size_t>(a.H), 0, g * 128 + lane * 4)
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int g = cw + i * kCW;
        if (g < a.KB) {   // warp-uniform
            float sc;
            float4 dec;
            const uint32_t codes = quant_group_warp(v[i], &sc, &dec);
            *reinterpret_cast<float4*>(sm.xdec + g * 128 + act_pos(lane * 4)) = dec;
            if (lane == 0) sm.xs[g] = sc;
            if (a.q_x && blockIdx.x == 0) {
                *reinterpret_cast<uint32_t*>(a.q_x + g * 128 + lane * 4) = codes;
                if (lane == 0) a.s_x[g] = sc;
            }
        }
    }
}

__device__ void load_column_scales(const TokenArgs& a, Smem& sm, const Column& col, int tid) {
    const int NBg = 2 * a.RB;
    if (tid < a.KB) {
        sm.swg[0][tid] = __ldg(a.s_gu + (static_cast<size_t>(col.expert) * NBg + col.kb) * a.KB + tid);
    } else if (tid >= 128 && tid < 128 + a.KB) {
        const int q = tid - 128;
        sm.swg[1][q] = __ldg(a.s_gu + (static_cast<size_t>(col.expert) * NBg + a.RB + col.kb) * a.KB + q);
    } else if (tid >= 256 && tid < 256 + a.KB) {
        const int nb = tid - 256;
        sm.swd[nb] = __ldg(a.s_d + (static_cast<size_t>(col.expert) * a.KB + nb) * a.RB + col.kb);
    }
}

// One column for one consumer warp: gate_up over every K group of x, SwiGLU
// and the live quantisation of h (warp 0), then down's K group kb against
// every output row, one 256-row unit per stage.
__device__ bool consume_column(const TokenArgs& a, Smem& sm, const uint8_t* stages, const Column& col, int j, int cw,
                               int lane, long long& it, int& stored) {
    const int l8 = lane & 7, rsub = lane >> 3;
    const int half = cw >> 3;                     // gate_up: 0 gate, 1 up; down: tile 2u + half
    const int rows_base = (cw & 7) * 16;
    float acc0 = 0.0f, acc1 = 0.0f, acc2 = 0.0f, acc3 = 0.0f;
    for (int t = 0; t < a.KB; ++t, ++it) {
        const int s = static_cast<int>(it % kStages);
        if (!__all_sync(0xffffffffu, wait_or_abort(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status)))
            return false;
        const uint8_t* tile = stages + static_cast<size_t>(s) * kStageBytes + half * kTile;
        float2 av[8];
        load_act(sm.xdec + t * 128, l8, av);
        const float scl = sm.xs[t] * sm.swg[half][t];
        const float d0 = row_dot(tile, rows_base + rsub, l8, av);
        const float d1 = row_dot(tile, rows_base + 4 + rsub, l8, av);
        const float d2 = row_dot(tile, rows_base + 8 + rsub, l8, av);
        const float d3 = row_dot(tile, rows_base + 12 + rsub, l8, av);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
        acc0 = fmaf(d0, scl, acc0);
        acc1 = fmaf(d1, scl, acc1);
        acc2 = fmaf(d2, scl, acc2);
        acc3 = fmaf(d3, scl, acc3);
    }
    const float r = reduce_rows4(acc0, acc1, acc2, acc3, l8);
    if ((l8 & 1) == 0) sm.gsum[half * 128 + rows_base + 4 * (l8 >> 1) + rsub] = r;
    consumer_sync();
    if (cw == 0) {
        // SwiGLU (gate rows first, then up rows) and the live quantisation of
        // the h group this column owns -- down's K group kb
        float hv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float g = sm.gsum[4 * lane + q], u = sm.gsum[128 + 4 * lane + q];
            hv[q] = __fdiv_rn(g, 1.0f + expf(-g)) * u;
        }
        const float4 h4 = make_float4(hv[0], hv[1], hv[2], hv[3]);
        const size_t hoff = static_cast<size_t>(col.pair) * a.I + col.kb * 128 + 4 * lane;
        *reinterpret_cast<float4*>(a.h + hoff) = h4;
        float sc;
        float4 dec;
        const uint32_t codes = quant_group_warp(h4, &sc, &dec);
        *reinterpret_cast<float4*>(sm.hdec + act_pos(4 * lane)) = dec;
        if (lane == 0) sm.hs = sc;
        if (a.q_h) {
            *reinterpret_cast<uint32_t*>(a.q_h + hoff) = codes;
            if (lane == 0) a.s_h[col.pair * a.RB + col.kb] = sc;
        }
    }
    consumer_sync();
    float2 hv[8];
    load_act(sm.hdec, l8, hv);
    // the routing weight of this column's expert (1 for the shared one) goes
    // into its partials, so that a unit's output is the plain sum of them
    const float sa = sm.hs * (col.g == 0 ? 1.0f : sm.topk_w[sm.slot_pick[col.g - 1]]);
    const uint64_t keep = l2_evict_last_policy();
    const int nu = a.KB / 2;
    for (int i = 0; i < nu; ++i, ++it) {
        const int s = static_cast<int>(it % kStages);
        if (!__all_sync(0xffffffffu, wait_or_abort(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status)))
            return false;
        const uint8_t* tile = stages + static_cast<size_t>(s) * kStageBytes + half * kTile;
        const float d0 = row_dot(tile, rows_base + rsub, l8, hv);
        const float d1 = row_dot(tile, rows_base + 4 + rsub, l8, hv);
        const float d2 = row_dot(tile, rows_base + 8 + rsub, l8, hv);
        const float d3 = row_dot(tile, rows_base + 12 + rsub, l8, hv);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
        const int u = unit_of(a, i);
        const float v = reduce_rows4(d0, d1, d2, d3, l8) * (sa * sm.swd[2 * u + half]);
        // the partials stay in L2 (evict last) until a summing warp reads them,
        // while the weight stream passes through it
        if ((l8 & 1) == 0)
            st_global_hint(a.part + ((static_cast<size_t>(u) * kParts + cw) * a.ncols + j) * 16 + 4 * (l8 >> 1) + rsub,
                           v, keep);
        __syncwarp();
        // the ticket warp learns of the stored partials four units at a time,
        // and of each of the last kTailUnits at once
        ++stored;
        if (lane == 0 && ((i & 3) == 3 || i >= nu - kTailUnits)) {
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&sm.wdone[cw]) = stored;
        }
    }
    return true;
}

// ------------------------------------------------------------------ combine
// One part of a completed unit: rows (2u + w/8)*128 + (w%8)*16 .. +15 of the
// output.  Every column's partial already carries its expert's routing
// weight, so the output is their plain sum: lane (row quad q = lane % 4,
// column class c8 = lane / 4) adds the columns c8, c8 + 8, ... in order (all
// its loads in flight at once, from L2), a fixed butterfly over the eight
// column classes adds those, and lanes 0..3 round their four rows to bf16.
__device__ void combine_part(const TokenArgs& a, int u, int w, int lane) {
    const float4* src = reinterpret_cast<const float4*>(a.part + (static_cast<size_t>(u) * kParts + w) * a.ncols * 16);
    const int n4 = a.ncols * 4;
    constexpr int kBatch = 19;   // up to 152 columns in one batch
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int f0 = lane; f0 < n4; f0 += 32 * kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int f = f0 + 32 * b;
            v[b] = f < n4 ? __ldcg(src + f) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            acc.x += v[b].x;
            acc.y += v[b].y;
            acc.z += v[b].z;
            acc.w += v[b].w;
        }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (lane < 4) {
        const int n = (2 * u + (w >> 3)) * 128 + (w & 7) * 16 + 4 * lane;
        if (a.out_f32) {
            *reinterpret_cast<float4*>(a.out_f32 + n) = acc;
        } else {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 packed;
            packed.x = *reinterpret_cast<const uint32_t*>(&lo);
            packed.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(a.out + n) = packed;
        }
    }
}

// The parts this warp sums, in unit order.  The units complete one after
// another as the slowest stream passes them.  All but the last kTailUnits
// are summed while the streams go on, by the CTAs without a column when there
// are some (part p = 16u + w to spare CTA p % n_spare, warp (p / n_spare) %
// 16, so a unit's 16 parts land on 16 different warps), else by every CTA
// once its stream is done (part p to CTA p % G).  The last units complete at
// the very end, when every column CTA is free: their parts are spread one per
// CTA over the column CTAs.  A part waits (bounded) for its unit's count to
// reach ncols.
__device__ void sum_part_when_complete(const TokenArgs& a, Smem& sm, int p, int lane, bool& ok_out) {
    const int u = p / kParts;
    int ok = 0;
    if (lane == 0) {
        const int* cnt = a.tickets + u;
        const unsigned long long t0 = global_timer_ns();
        for (uint32_t i = 0;; ++i) {
            if (ld_relaxed(cnt) >= a.ncols) {
                ok = ld_acquire(cnt) >= a.ncols;   // acquires the unit's partials
                break;
            }
            if ((i & 7u) == 7u) {
                if (sm.abort_flag) break;
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    record_error(a.status, MOEQ_ERR_TIMEOUT);
                    sm.abort_flag = 1;
                    break;
                }
            }
            __nanosleep(64);
        }
    }
    ok_out = __shfl_sync(0xffffffffu, ok, 0) != 0;
    if (ok_out) combine_part(a, u, p % kParts, lane);
}

__device__ void combine_worker(const TokenArgs& a, Smem& sm, int cw, int lane) {
    const int G = gridDim.x, c = blockIdx.x, nu = a.KB / 2, n_spare = G - a.ncols;
    const int tail = min(kTailUnits, nu), early = (nu - tail) * kParts;
    bool ok = true;
    if (n_spare > 0) {
        if (c >= a.ncols)
            for (int p = (c - a.ncols) + n_spare * cw; p < early && ok; p += n_spare * kCW)
                sum_part_when_complete(a, sm, p, lane, ok);
    } else {
        for (int p = c + G * cw; p < early && ok; p += G * kCW) sum_part_when_complete(a, sm, p, lane, ok);
    }
    const int nc = min(a.ncols, G);
    if (c < nc)
        for (int q = c + nc * cw; q < tail * kParts && ok; q += nc * kCW) sum_part_when_complete(a, sm, early + q, lane, ok);
}

// The ticket warp: as the consumer warps store down partials, count each
// (column, unit) in -- one gpu-scope fence releases every partial stored so
// far (observed through the warps' progress counters), then one
// fire-and-forget add per arrival.  A unit is complete once its count reaches
// ncols; the summing warps watch the counts.
__device__ void ticket_warp(const TokenArgs& a, Smem& sm, int lane) {
    const int G = gridDim.x, c = blockIdx.x, nu = a.KB / 2;
    const int my_cols = c < a.ncols ? (a.ncols - 1 - c) / G + 1 : 0;
    const int total = my_cols * nu;
    int done = 0;
    unsigned long long t0 = global_timer_ns();
    while (done < total && !sm.abort_flag) {
        const int mine = lane < kCW ? reinterpret_cast<volatile int*>(sm.wdone)[lane] : 0x7fffffff;
        const int avail = __reduce_min_sync(0xffffffffu, mine);
        if (avail <= done) {
            __nanosleep(32);
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (lane == 0) record_error(a.status, MOEQ_ERR_TIMEOUT);
                sm.abort_flag = 1;
            }
            continue;
        }
        t0 = global_timer_ns();
        __threadfence();   // releases the partials stored by every consumer warp so far
        for (int q = done + lane; q < avail; q += 32) atomicAdd(a.tickets + unit_of(a, q % nu), 1);
        done = avail;
    }
}

__device__ void consumer_warp(const TokenArgs& a, Smem& sm, const uint8_t* stages, int cw, int lane) {
    const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
    if (c < a.ncols) {
        // the first column is known before griddepcontrol.wait when it is the
        // shared expert's, or when the token is routed ahead of the wait
        const bool first_early = c < a.RB || (a.route_early && a.top_k > 0);
        if (first_early) {
            if (c >= a.RB) {
                if (lane == 0) wait_or_abort(&sm.plan_bar, 0, sm, a.status);
                __syncwarp();
            }
            load_column_scales(a, sm, column(a, sm, c), tid);
        }
        pdl_wait();
        quantise_x(a, sm, cw, lane);
        long long it = 0;
        int stored = 0;
        for (int j = c; j < a.ncols; j += G) {
            if (j != c || !first_early) {
                if (lane == 0) wait_or_abort(&sm.plan_bar, 0, sm, a.status);
                __syncwarp();
                consumer_sync();   // the previous column's scales are no longer read
                load_column_scales(a, sm, column(a, sm, j), tid);
            }
            consumer_sync();       // x quantised, the column's scales loaded
            if (__any_sync(0xffffffffu, sm.abort_flag)) return;
            const Column col = column(a, sm, j);
            if (!consume_column(a, sm, stages, col, j, cw, lane, it, stored)) return;
        }
    } else {
        pdl_wait();
    }
    combine_worker(a, sm, cw, lane);
}

__global__ void __launch_bounds__(kThreads, 1) token_kernel(const __grid_constant__ TokenArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem& sm = *reinterpret_cast<Smem*>(stages + static_cast<size_t>(kStages) * kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        pdl_launch_dependents();
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCW);
        }
        mbar_init(&sm.plan_bar, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (tid < kCW) sm.wdone[tid] = 0;
    __syncthreads();
    if (warp == kProducerWarp) {
        producer_warp(a, sm, stages, lane);
    } else if (warp == kTicketWarp) {
        pdl_wait();
        ticket_warp(a, sm, lane);
    } else {
        consumer_warp(a, sm, stages, warp, lane);
    }
    __syncwarp();
    // The last CTA to get here clears the units' counts for the next launch:
    // every other CTA has stopped reading them.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(a.gq + kGqCtas, 1) == static_cast<int>(gridDim.x) - 1) {
            __threadfence();
            const int nu = a.KB / 2;
            for (int i = 0; i < nu; ++i) a.tickets[i] = 0;
            a.gq[kGqCtas] = 0;
        }
    }
}

}  // namespace

cudaError_t launch_token(const TokenArgs& args, int grid, bool pdl, cudaStream_t stream) {
    static int configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 64 && !configured[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, token_kernel, args);
}

}  // namespace moeq
