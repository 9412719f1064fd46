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
// consecutive K tiles of one 128-row block (32 KiB), for down by K group
// (one token) two row blocks' tiles of one K group (32 KiB).  Work comes in
// lists (for the layer: gate_up, then down, each over the shared expert
// first and then the routed experts of the plan).  When the row blocks of a
// list nearly fill the grid in whole numbers per CTA (one token: 144 gate_up
// blocks on 152 SMs), each CTA takes whole row blocks and nothing is split.
// One token goes on with down by K group: the CTA that finished gate_up
// block kb of a pair streams down's tiles (nb, kb) for every nb (its own h
// group against all of down's rows) and stores fp32 sums per (pair, kb,
// row); a combine over K groups ends the launch.  Otherwise every CTA takes a contiguous, equal share
// of the list's units (stream-K); a share splits into segments (runs of one
// row block) of which only the first and last can be partial in K, so each
// CTA leaves at most two fp32 partials per list; the last CTA to finish a
// row block (atomic ticket) sums them in CTA order and runs the epilogue, so
// results do not depend on timing.  A segment splits into chunks whose
// quantised activations fit one shared-memory slot.
//
// Warp roles (640 threads):
//   warps 0-15  consumers: per stage, each lane widens 16 weight bytes of a
//               row exactly to fp32 and accumulates paired fp32 FMAs with the
//               decoded activation codes, scaling per K group by s_a * s_w;
//               at a segment's end they leave one sum per (row, token);
//   warp 16     producer: one lane issues the bulk copies of every unit;
//   warp 17     prep: prepares the next chunk (plan lookup, weight scales,
//               bulk copies of its quantised activation groups) while the
//               consumers stream the current one;
//   warps 18-19 finish: finish segments (split-K partials and the ticketed
//               reduction, SwiGLU or plain store, readiness flags, the
//               combine) off the streaming path, even and odd segments.
// Live quantisation (per token, 1 x 128, s = amax/448, RNE to E4M3) happens
// once per (row, group) inside the kernel: the given inputs in a first phase
// spread over all CTAs, h in the gate_up finish that produces it.  The
// decoded codes stay in an L2-resident workspace buffer in the consumers'
// layout, so preparing a chunk is a few bulk copies.
// The roles meet only through mbarriers: the stage ring (full/empty), two
// activation slots (prep_full/act_empty) and two result slots
// (res_full/res_empty); no role waits on another CTA while the others owe
// it progress, so the cross-CTA dependencies (plan, h) cannot deadlock.
//
// Layer fusion (cooperative launch, all CTAs resident): every CTA computes
// the routing plan itself into shared memory (a few microseconds, no
// cross-CTA wait; CTA 0 also writes it out), while CTAs whose first blocks
// belong to the shared expert already stream them; gate_up finishes publish
// per-(expert, row block) readiness of h (already quantised); the prep warp
// waits (bounded) for an expert's h before loading it for down, while the
// producer already streams down weights;
// the down finish that completes the last expert of a (token, row block)
// also writes the combined bf16 output.
#pragma once

#include "moeq_device.cuh"
#include "moeq_internal.h"
#include "moeq_route.cuh"

namespace moeq {

constexpr int kCW = 16;                  // consumer warps
constexpr int kConsumers = kCW * 32;
constexpr int kProducerWarp = kCW;
constexpr int kPrepWarp = kCW + 1;
constexpr int kFinishWarp0 = kCW + 2;    // finishes even segments
constexpr int kFinishWarp1 = kCW + 3;    // finishes odd segments
constexpr int kThreads = (kCW + 4) * 32;
constexpr int kTile = 16384;
constexpr int kStageBytes = 2 * kTile;
constexpr int kStages = 4;
constexpr int kActSlot = 6144;           // decoded activation floats per slot
constexpr int kChunkGroups = kActSlot / kGroup;
// tcgen05 path: a slot holds the chunk's activation codes as the MMA's B
// operand, 2 KiB per K group (16 token rows x 128 bytes, 128-byte swizzle).
constexpr int kMmaN = 16;                              // tokens per MMA (rows of B)
constexpr int kMmaGroupBytes = kMmaN * 128;
constexpr int kMmaChunkGroups = kActSlot * 4 / kMmaGroupBytes;   // 12
constexpr int kActScales = kMaxTok * kMmaChunkGroups;           // >= kChunkGroups
constexpr int kTmemBufs = 4;                           // accumulator sets (one per stage in flight)
constexpr int kTmemCols = kTmemBufs * 2 * kMmaN;       // 128 columns: 2 tiles x 16 tokens per set
constexpr int kEpiSets = 2;                            // epilogue warp sets, alternating stages
constexpr int kEpiWarps = 4 * kEpiSets;                // warps 0-7: warp w reads TMEM lanes 32*(w%4) ..
constexpr int kMmaWarp = kEpiWarps;
constexpr int kUnitRows = 256;           // rows of a gate_up unit (gate + up); down units use 128
constexpr int kResPool = 2 * kUnitRows * (kMaxTok + 1);   // result slot floats (two at 16 tokens)
constexpr int kMaxRes = 8;               // result slots at most
constexpr int kSegRing = 16;             // segment metadata entries (>= kMaxRes + 8, see prep_warp)

struct ChunkDesc {
    int kind;          // kKindGU / kKindDN / kKindDC; -1: no more work
    int ku0, ku1;      // units [ku0, ku1) of the segment's row block
    int g0, ng;        // K groups of this chunk's activations
    int ntok;
    int seg_end;       // the segment's last chunk
    int p0;            // down by K group: the pair whose sums the chunk leaves
};

struct SegMeta {       // what the helper needs to finish a segment
    int kind, li, e_local, rb, j, ku0, ku1;   // j: the row block's position in the list
    int expert, p0, ntok, slot, shared_static, valid;
    long long T, G, c, lo;
    int KU, RB;
};

// The layer's routing plan, computed by every CTA into shared memory (same
// members as moeq_route_plan; M <= kMaxTok, top_k <= kRouteMaxK).
constexpr int kLocalUniq = kMaxTok * kRouteMaxK + 1;
constexpr int kLocalPairs = kMaxTok * (kRouteMaxK + 1);
struct LocalPlan {
    int topk_id[kMaxTok * kRouteMaxK];
    float topk_w[kMaxTok * kRouteMaxK];
    int n_uniq;
    int uniq[kLocalUniq];
    int offs[kLocalUniq + 1];
    int pair_tok[kLocalPairs];
    int pair_of[kLocalPairs];
};

// Where the roles read the plan: the CTA's LocalPlan (layer) or the caller's
// plan in global memory (standalone calls).  Generic pointers.
struct PlanView {
    const int* n_uniq;
    const int* uniq;
    const int* offs;
    const int* pair_tok;
    const int* pair_of;
    const float* topk_w;
};

struct SmemTail {
    float act[2][kActSlot];              // decoded activations [tok][group][permuted k]
    float act_s[2][kActScales];          // activation scales: [tok][group]; tcgen05 path [group][16 tok]
    float sw[2][2][kChunkGroups];        // weight scales per slot, per tile
    union {
        float res[kResPool];             // result slots: one sum per (row, token), see ResRing
        RouteScratch route;              // plan computation: done before any chunk, so before any result
    };
    float hloc[kGroup];                  // one token: the h group this CTA finished (decoded codes) ...
    float hloc_s;                        // ... and its scale
    ChunkDesc chunk[2];
    SegMeta seg[kSegRing];               // by segment index % kSegRing (see prep_warp)
    LocalPlan plan;
    PlanView pv;
    int n_segments;                      // total, written by the prep warp before its end marker
    int finish_done;                     // finish warps that have ended
    uint64_t full[kStages], empty[kStages];
    uint64_t prep_full[2], act_empty[2], res_full[kMaxRes], res_empty[kMaxRes];
    uint64_t plan_bar;                   // the LocalPlan is complete (layer)
    uint64_t xq_bar;                     // x is quantised into act[0] / act_s[0] (xloc)
    uint64_t hloc_bar;                   // hloc is written (hloc)
    uint64_t mma_done[kTmemBufs], tmem_empty[kTmemBufs];   // tcgen05 path
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(SmemTail);
static_assert(kActSlot >= kDcCombineFloats, "the down-by-K-group combine works in one activation slot");
static_assert(kActSlot >= kXLocalMaxK, "one token's x fits one activation slot");
static_assert(offsetof(SmemTail, sw) % 16 == 0 && (kChunkGroups * 4) % 16 == 0,
              "weight-scale rows are bulk-copy destinations");
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void consumer_sync() { named_sync(1, kConsumers); }

// Result slots: segment s publishes its sums in slot s % ns, element (row, t)
// at row * ld + t.  ld is the odd number >= the launch's largest token count
// per expert, so short launches get more slots (8 at one token, 2 at 16) and
// the consumers run further ahead of the finish warps.
struct ResRing {
    int ns, ld;
    __device__ __forceinline__ explicit ResRing(const StreamArgs& a)
        : ns(min(kMaxRes, kResPool / (kUnitRows * (a.max_ntok | 1)))), ld(a.max_ntok | 1) {}
    __device__ __forceinline__ int slot(long long sidx) const { return static_cast<int>(sidx % ns); }
    __device__ __forceinline__ uint32_t parity(long long sidx) const { return static_cast<uint32_t>((sidx / ns) & 1); }
    __device__ __forceinline__ float* at(SmemTail& sm, long long sidx) const {
        return sm.res + static_cast<size_t>(slot(sidx)) * kUnitRows * ld;
    }
};
__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

// The operand a list kind streams: down by K group streams down's tiles.
__device__ __forceinline__ const Operand& kind_op(const StreamArgs& a, int kind) {
    return a.op[kind == kKindDC ? kKindDN : kind];
}

// Row blocks per expert of a list kind: its output row blocks, or for down
// by K group its K groups (each the h of one gate_up row block).
__device__ __forceinline__ int kind_rbs(const StreamArgs& a, int kind) {
    return kind == kKindDC ? a.op[kKindDN].KB : a.op[kind].RB;
}

// Position of element k (0..127) of a group in the shared activation layout:
// lane l8 reads its four float4 (k = 16*l8 + 4i .. +3) at (8i + l8)*4, so the
// eight lanes of a row hit eight consecutive 16-byte chunks.
__device__ __forceinline__ int act_pos(int k) { return (((k & 15) >> 2) * 8 + (k >> 4)) * 4 + (k & 3); }

// tcgen05 path: lane l's four codes (bytes 4l .. 4l+3 of a 128-byte group)
// into all 8 swizzle phases of that group: phase p at chunk (l/4) ^ p.
__device__ __forceinline__ void store_code_phases(uint8_t* group0, size_t phase_stride, int lane, uint32_t codes) {
    const int c = lane >> 2, off = (lane & 3) * 4;
#pragma unroll
    for (int p = 0; p < 8; ++p)
        *reinterpret_cast<uint32_t*>(group0 + p * phase_stride + ((c ^ p) << 4) + off) = codes;
}

// ------------------------------------------------------------------ work lists
struct ListInfo {
    int kind, src, n_exp, e0, RB, KU;  // experts e0 .. e0+n_exp-1 of the list's source (see list_expert)
    bool dp;             // whole row blocks: `per` consecutive blocks per CTA
    int per;
    long long T, G, c;   // units, CTAs, this CTA's index
    long long lo, hi;    // this CTA's share [lo, hi)
};

__device__ __forceinline__ long long unit_lo(long long c, long long T, long long G) { return c * T / G; }
__device__ __forceinline__ long long cta_of_unit(long long u, long long T, long long G) {
    return ((u + 1) * G - 1) / T;
}

// Row blocks per CTA when whole blocks are dealt out: used when the CTAs
// that get `per` blocks are at least 90% of the grid (the rest idle in this
// list; the streaming rate is the memory's, not the SM count's).
__device__ __forceinline__ int dp_blocks_per_cta(long long n_rb, long long G) {
    if (n_rb <= 0) return 0;
    const long long per = (n_rb + G - 1) / G, used = (n_rb + per - 1) / per;
    return used * 10 >= G * 9 ? static_cast<int>(per) : 0;
}

// Whether this CTA needs the plan to know its share of list li.  The layer's
// lists start with the shared expert, which needs none: for one token (where
// the plan's expert count is known in advance) with whole blocks per CTA, the
// CTAs whose blocks all belong to it start before the plan.
__device__ __forceinline__ bool list_needs_plan(const StreamArgs& a, int li) {
    if (a.list_src[li] == kSrcShared || a.list_src[li] == kSrcPlanAll) return false;
    if (a.list_src[li] != kSrcLayer || a.M > 1) return true;
    const int rbs = kind_rbs(a, a.list_kind[li]);
    const int per = dp_blocks_per_cta(static_cast<long long>(a.max_uniq) * rbs, gridDim.x);
    return !(per > 0 && (static_cast<long long>(blockIdx.x) + 1) * per <= rbs);
}

// U: unique experts of the plan (shared included), or -1 while unknown
// (only where list_needs_plan is false).
__device__ __forceinline__ ListInfo list_info(const StreamArgs& a, int li, int U) {
    ListInfo L;
    L.kind = a.list_kind[li];
    L.src = a.list_src[li];
    const Operand& op = kind_op(a, L.kind);
    L.RB = kind_rbs(a, L.kind);
    // units per row block: K groups (gate_up), K tile pairs (down), row
    // block pairs (down by K group)
    L.KU = L.kind == kKindGU ? op.KB : L.kind == kKindDC ? op.NB / 2 : (op.KB + 1) / 2;
    const int routed = U > 1 ? U - 1 : 0, half = (routed + 1) / 2;
    L.e0 = L.src == kSrcPlanRoutedB ? half : 0;
    L.n_exp = L.src == kSrcShared ? 1
            : (L.src == kSrcLayer || L.src == kSrcPlanAll) ? (U < 0 ? 1 : U)
            : L.src == kSrcPlanRoutedA ? half : routed - half;
    L.G = gridDim.x;
    L.c = blockIdx.x;
    L.T = static_cast<long long>(L.n_exp) * L.RB * L.KU;
    // one-token layers decide on the plan's bound (their expert count, known
    // before the plan), everything else on the plan's actual expert count
    const long long n_dec = (L.src == kSrcLayer && a.M == 1) ? a.max_uniq : L.n_exp;
    L.per = dp_blocks_per_cta(n_dec * L.RB, L.G);
    L.dp = L.per > 0;
    if (L.dp) {
        const long long n_rb = static_cast<long long>(L.n_exp) * L.RB;
        L.lo = min(L.c * L.per, n_rb) * L.KU;
        L.hi = min((L.c + 1) * L.per, n_rb) * L.KU;
    } else if (L.T == 0) {
        L.lo = L.hi = 0;
    } else {
        L.lo = unit_lo(L.c, L.T, L.G);
        L.hi = unit_lo(L.c + 1, L.T, L.G);
    }
    return L;
}

// Expert e_local of a list.  The layer's shared expert (tokens 0..M-1, its
// pairs after the routed ones, known before the plan) is a list of its own
// or the first expert of a kSrcLayer list, followed there by the plan's
// routed experts; the halves are runs of the plan's routed experts; a
// standalone call's list is its plan.
struct ExpertRef {
    int expert, p0, ntok, slot, shared_static;
};

__device__ __forceinline__ ExpertRef list_expert(const StreamArgs& a, const PlanView& pv, const ListInfo& L,
                                                 int e_local) {
    const int src = L.src;
    ExpertRef r;
    if (src == kSrcShared || (src == kSrcLayer && e_local == 0)) {
        r.expert = a.shared_id;
        r.p0 = a.shared_p0;
        r.ntok = a.M;
        r.slot = a.max_uniq - 1;
        r.shared_static = 1;
    } else {
        const int ue = L.e0 + e_local - (src == kSrcLayer ? 1 : 0);
        r.expert = pv.uniq[ue];
        r.p0 = pv.offs[ue];
        r.ntok = pv.offs[ue + 1] - r.p0;
        r.slot = ue;
        r.shared_static = 0;
    }
    return r;
}

// The (expert, row block) at row-block position j of a list.  Lists of a
// multi-token layer spread the shared expert's row blocks evenly among the
// routed ones (block k at position floor(k * n / RB) of n): its blocks carry
// every token, so no CTA gets more than its share of them.  Otherwise
// positions run expert by expert.
__device__ __forceinline__ void list_rb(const StreamArgs& a, const ListInfo& L, int j, int& e_local, int& rb) {
    if (L.src == kSrcLayer && a.M > 1 && L.n_exp > 1) {
        const long long n = static_cast<long long>(L.n_exp) * L.RB, R = L.RB;
        const int before = static_cast<int>((j * R + n - 1) / n);          // shared blocks at positions < j
        const int upto = static_cast<int>(((j + 1) * R + n - 1) / n);      // ... at positions <= j
        if (upto > before) {
            e_local = 0;
            rb = before;
        } else {
            const int q = j - before;
            e_local = 1 + q / L.RB;
            rb = q % L.RB;
        }
    } else {
        e_local = j / L.RB;
        rb = j % L.RB;
    }
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

__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, SmemTail& sm, int* status) {
    if (mbar_wait_bounded(bar, parity, &sm.abort_flag)) return true;
    record_error(status, MOEQ_ERR_TIMEOUT);
    sm.abort_flag = 1;
    return false;
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void producer(const StreamArgs& a, SmemTail& sm, uint8_t* stages, int epoch) {
    const uint64_t pol = l2_evict_first_policy();
    long long issued = 0;
    int U = -1;
    for (int li = 0; li < a.n_lists && !sm.abort_flag; ++li) {
        if (U < 0 && (list_needs_plan(a, li) || a.list_src[li] == kSrcPlanAll)) {
            if (a.fused_route) mbar_wait_or_abort(&sm.plan_bar, 0, sm, a.status);
            U = *sm.pv.n_uniq;
            if (U < 0 || U > a.max_uniq) U = 0;  // reported by the prep warp
        }
        const ListInfo L = list_info(a, li, U);
        const Operand& op = kind_op(a, L.kind);
        int cur = -1, expert = 0;
        for (int u = static_cast<int>(L.lo); u < static_cast<int>(L.hi); ++u) {
            const int jb = u / L.KU, ku = u - jb * L.KU;
            int e_local, rb;
            list_rb(a, L, jb, e_local, rb);
            if (e_local != cur) {
                cur = e_local;
                expert = list_expert(a, sm.pv, L, e_local).expert;
                if (expert < 0 || expert >= a.n_experts) expert = 0;
            }
            const int s = static_cast<int>(issued % kStages);
            if (issued >= kStages)
                mbar_wait_or_abort(&sm.empty[s], static_cast<uint32_t>((issued / kStages - 1) & 1), sm, a.status);
            if (sm.abort_flag) break;
            uint8_t* dst = stages + static_cast<size_t>(s) * kStageBytes;
            if (L.kind == kKindGU) {
                // one token, one block per CTA: the first stage also brings
                // the gate and up weight-scale rows of the block (the first
                // chunk's, all K groups) into the first chunk's scale slots,
                // so they land with the first tiles rather than behind them
                const bool swb = a.swb && issued == 0;
                const uint32_t sw_bytes = static_cast<uint32_t>(op.KB) * 4u;
                mbar_arrive_expect_tx(&sm.full[s], 2 * kTile + (swb ? 2u * sw_bytes : 0u));
                bulk_load(dst, tile_ptr(op, expert, rb, ku), kTile, &sm.full[s], pol);
                bulk_load(dst + kTile, tile_ptr(op, expert, L.RB + rb, ku), kTile, &sm.full[s], pol);
                if (swb) {
                    bulk_load(sm.sw[0][0], op.sw + (static_cast<size_t>(expert) * op.NB + rb) * op.KB, sw_bytes,
                              &sm.full[s], pol);
                    bulk_load(sm.sw[0][1], op.sw + (static_cast<size_t>(expert) * op.NB + L.RB + rb) * op.KB,
                              sw_bytes, &sm.full[s], pol);
                }
            } else if (L.kind == kKindDC) {
                // row blocks 2ku and 2ku+1 of down at K group rb
                mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
                bulk_load(dst, tile_ptr(op, expert, 2 * ku, rb), kTile, &sm.full[s], pol);
                bulk_load(dst + kTile, tile_ptr(op, expert, 2 * ku + 1, rb), kTile, &sm.full[s], pol);
            } else {
                const int nt = min(2, op.KB - 2 * ku);
                mbar_arrive_expect_tx(&sm.full[s], nt * kTile);
                bulk_load(dst, tile_ptr(op, expert, rb, 2 * ku), nt * kTile, &sm.full[s], pol);
            }
            ++issued;
        }
    }
    if (sm.abort_flag) {
        // Let the copies already issued land before the CTA may exit (bounded).
        for (long long j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&sm.full[j % kStages], static_cast<uint32_t>((j / kStages) & 1)) &&
                   global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
            }
        }
    }
}

// ------------------------------------------------------------------ helper
// Bounded spin until *cnt >= want (acquire).
__device__ __forceinline__ bool wait_count(const int* cnt, int want, int* status, volatile int* abort) {
    if (ld_acquire(cnt) - want >= 0) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire(cnt) - want >= 0) return true;
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

// Stage a chunk into slot cs: bulk copies of the already quantised
// (decoded, consumer-layout) activation rows of groups [g0, g0+ng), their
// scales, the weight scales and the descriptor.  Every load is issued before
// any is waited for; prep_full[cs] completes when the copied bytes land.
template <bool kMma>
__device__ __forceinline__ void prep_chunk(const StreamArgs& a, const Operand& op, SmemTail& sm, long long c,
                                           long long sidx, const SegMeta& m, const ListInfo& L, const ChunkDesc& d,
                                           int lane) {
    const int cs = static_cast<int>(c & 1);
    const int g0 = d.g0, ng = d.ng;
    int row = 0;
    if (lane < m.ntok) {
        const int p = m.p0 + lane;
        // gate_up reads token rows (the shared expert's pairs are tokens
        // 0..M-1); down reads pair rows.
        row = m.kind == kKindGU ? (m.shared_static ? lane : sm.pv.pair_tok[p]) : p;
        if (row < 0 || row >= op.rows_a) {
            record_error(a.status, MOEQ_ERR_INVALID_ARG);
            row = 0;
        }
    }
    // one token's x quantised by this CTA itself: codes and scales are
    // already in slot 0 (the first chunk's), only the weight scales remain
    const bool xl = !kMma && a.xloc && m.kind == kKindGU && c == 0;
    // scales: activation (ntok x ng) then weight (1 or 2 tiles x ng), all
    // loads first; only as many 32-wide passes as there are values
    const int n_as = xl ? 0 : m.ntok * ng, n_all = n_as + (xl && a.swb ? 0 : ng * (m.kind == kKindGU ? 2 : 1));
    const float* sw0 = op.sw + (static_cast<size_t>(m.expert) * op.NB + m.rb) * op.KB + g0;
    const size_t sw_up = static_cast<size_t>(L.RB) * op.KB;   // the up tile's row block
    constexpr int kPer = (kActScales + 2 * kChunkGroups + 31) / 32;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (32 * j >= n_all) break;                  // uniform
        const int i = lane + 32 * j;
        int rt = 0;
        if (32 * j < n_as) rt = __shfl_sync(0xffffffffu, row, min(i / ng, m.ntok - 1));   // uniform
        float x = 0.0f;
        if (i < n_as) {
            x = __ldcg(op.as + static_cast<size_t>(rt) * op.KB + g0 + i % ng);
        } else if (i < n_all) {
            const int q = i - n_as, b = q >= ng;
            x = __ldg(sw0 + (b ? sw_up : 0) + (q - b * ng));
        }
        v[j] = x;
    }
    // The slot is free once the consumers are done with chunk c - 2: the
    // scale loads above are already in flight while this waits.
    if (c >= 2) mbar_wait_or_abort(&sm.act_empty[cs], static_cast<uint32_t>(((c >> 1) - 1) & 1), sm, a.status);
    if (d.ku0 == m.ku0 && lane == 0) sm.seg[sidx % kSegRing] = m;
    const uint32_t bytes = static_cast<uint32_t>(ng) * kGroup * 4u;
    // after an abort no copy is issued (the consumers stop reading)
    const bool live = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort_flag) == 0, 0);
    fence_proxy_async();
    if (!live) {
    } else if constexpr (kMma) {
        // B operand: token t's codes of group gl become row t of that group's
        // 16 x 128-byte block, whose 128-byte swizzle puts chunk c at c ^ (t % 8):
        // one bulk copy per (token, group) from the code phase t % 8
        const uint8_t* codes = reinterpret_cast<const uint8_t*>(op.aq);
        const size_t phase_stride = static_cast<size_t>(op.rows_a) * op.K;
        uint8_t* slot = reinterpret_cast<uint8_t*>(sm.act[cs]);
        const int total = ng * m.ntok;
        for (int base = 0; base < total; base += 32) {
            const int i = base + lane;
            const int t = i % m.ntok, gl = i / m.ntok;
            const int rt = __shfl_sync(0xffffffffu, row, t);
            if (i < total)
                bulk_load(slot + gl * kMmaGroupBytes + (t >> 3) * 1024 + (t & 7) * 128,
                          codes + (t & 7) * phase_stride + static_cast<size_t>(rt) * op.K + (g0 + gl) * kGroup, 128,
                          &sm.prep_full[cs], l2_evict_first_policy());
        }
    } else {
        if (!xl && lane < m.ntok)
            bulk_load(sm.act[cs] + lane * ng * kGroup, op.aq + (static_cast<size_t>(row) * op.KB + g0) * kGroup,
                      bytes, &sm.prep_full[cs], l2_evict_first_policy());
    }
    if constexpr (kMma) {
        // token-minor, padded with zeros to kMmaN tokens
        for (int i = lane; i < ng * kMmaN; i += 32) sm.act_s[cs][i] = 0.0f;
        __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (32 * j >= n_all) break;
        const int i = lane + 32 * j;
        if (i < n_as) {
            sm.act_s[cs][kMma ? (i % ng) * kMmaN + i / ng : i] = v[j];
        } else if (i < n_all) {
            const int q = i - n_as, b = q >= ng;
            sm.sw[cs][b][q - b * ng] = v[j];
        }
    }
    if (lane == 0) sm.chunk[cs] = d;
    __syncwarp();
    if (lane == 0) {
        if (live && !xl)
            mbar_arrive_expect_tx(&sm.prep_full[cs], kMma ? static_cast<uint32_t>(ng * m.ntok) * 128u
                                                           : bytes * static_cast<uint32_t>(m.ntok));
        else
            mbar_arrive(&sm.prep_full[cs]);
    }
}

// Stage a chunk of down by K group into slot cs: the pair's quantised h
// group m.rb, its scale, and the weight scales of both tiles of each unit.
// The weight scales are loaded first; then, for the segment's first chunk,
// the wait for the h group: from this CTA's own finish warp in shared
// memory (hloc), else the group's readiness flag and one 512-byte bulk copy
// of its decoded codes.  One token: the pair has one row.
__device__ __forceinline__ void prep_chunk_dc(const StreamArgs& a, SmemTail& sm, long long c, long long sidx,
                                              const SegMeta& m, const ChunkDesc& d, int lane, int epoch) {
    const Operand& op = a.op[kKindDN];
    const int cs = static_cast<int>(c & 1);
    const int n_sw = 2 * (d.ku1 - d.ku0);   // <= 2 * kChunkGroups
    constexpr int kPer = (2 * kChunkGroups + 31) / 32;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int q = lane + 32 * j, nb = 2 * (d.ku0 + (q >> 1)) + (q & 1);
        v[j] = q < n_sw ? __ldg(op.sw + (static_cast<size_t>(m.expert) * op.NB + nb) * op.KB + m.rb) : 0.0f;
    }
    if (d.ku0 == m.ku0) {
        if (a.hloc) {
            if (lane == 0) mbar_wait_or_abort(&sm.hloc_bar, 0, sm, a.status);
        } else if (lane == 0) {
            wait_flag(a.h_ready + static_cast<size_t>(m.slot) * a.op[kKindGU].RB + m.rb, epoch, a.status,
                      &sm.abort_flag);
        }
        __syncwarp();
    }
    if (c >= 2) mbar_wait_or_abort(&sm.act_empty[cs], static_cast<uint32_t>(((c >> 1) - 1) & 1), sm, a.status);
    if (d.ku0 == m.ku0 && lane == 0) sm.seg[sidx % kSegRing] = m;
    const bool live = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort_flag) == 0, 0);
    if (a.hloc) {
        *reinterpret_cast<float4*>(sm.act[cs] + 4 * lane) = *reinterpret_cast<const float4*>(sm.hloc + 4 * lane);
        if (lane == 0) sm.act_s[cs][0] = sm.hloc_s;
    } else {
        fence_proxy_async();
        if (live && lane == 0)
            bulk_load(sm.act[cs], op.aq + (static_cast<size_t>(m.p0) * op.KB + m.rb) * kGroup, kGroup * 4u,
                      &sm.prep_full[cs], l2_evict_first_policy());
        if (lane == 0) sm.act_s[cs][0] = __ldcg(op.as + static_cast<size_t>(m.p0) * op.KB + m.rb);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int q = lane + 32 * j;
        if (q < n_sw) sm.sw[cs][q & 1][q >> 1] = v[j];
    }
    if (lane == 0) sm.chunk[cs] = d;
    __syncwarp();
    if (lane == 0) {
        if (live && !a.hloc)
            mbar_arrive_expect_tx(&sm.prep_full[cs], kGroup * 4u);
        else
            mbar_arrive(&sm.prep_full[cs]);
    }
}

// Finish one segment from its result slot: gate_up -> h = silu(gate) * up
// and (layer) the readiness flag of (expert, row block); down -> y and
// (layer) the combine of every token whose last expert this was.
static __device__ __noinline__ void helper_epilogue(const StreamArgs& a, SmemTail& sm, const SegMeta& m,
                                             const float* res, int ld, int lane, int epoch) {
    const PlanView& pv = sm.pv;
    const Operand& op = a.op[m.kind];
    if (m.valid && m.kind == kKindGU) {
        // lane owns h columns 4*lane .. 4*lane+3 of this row block; in the
        // layer the 128 columns are one K group of down: quantise it here,
        // once, for every down CTA that will read it.
        const Operand& dn = a.op[kKindDN];
        for (int t = 0; t < m.ntok; ++t) {
            float hv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = 4 * lane + j;
                const float g = res[i * ld + t];
                const float u = res[(128 + i) * ld + t];
                hv[j] = __fdiv_rn(g, 1.0f + expf(-g)) * u;
            }
            const float4 h4 = make_float4(hv[0], hv[1], hv[2], hv[3]);
            const size_t p = static_cast<size_t>(m.p0 + t);
            if (a.hloc) {
                // this CTA's own down by K group takes the group from shared
                // memory, before any of the global writes below
                float sc;
                float4 dec;
                quant_group_warp(h4, &sc, &dec);
                *reinterpret_cast<float4*>(sm.hloc + act_pos(4 * lane)) = dec;
                if (lane == 0) sm.hloc_s = sc;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.hloc_bar);
            }
            *reinterpret_cast<float4*>(op.out + p * op.out_ld + m.rb * 128 + 4 * lane) = h4;
            if (a.h_to_dn) {
                float sc;
                float4 dec;
                const uint32_t hc = quant_group_warp(h4, &sc, &dec);
                if (a.mma)
                    store_code_phases(reinterpret_cast<uint8_t*>(dn.aq) + p * dn.K + m.rb * kGroup,
                                      static_cast<size_t>(dn.rows_a) * dn.K, lane, hc);
                else
                    *reinterpret_cast<float4*>(dn.aq + (p * dn.KB + m.rb) * kGroup + act_pos(4 * lane)) = dec;
                if (lane == 0) dn.as[p * dn.KB + m.rb] = sc;
                if (a.qh_dump) {
                    *reinterpret_cast<uint32_t*>(a.qh_dump + p * dn.K + m.rb * kGroup + 4 * lane) = hc;
                    if (lane == 0) a.sh_dump[p * dn.KB + m.rb] = sc;
                }
            }
        }
    } else if (m.valid) {
        for (int idx = lane; idx < 128 * m.ntok; idx += 32) {
            const int i = idx & 127, t = idx >> 7;
            op.out[static_cast<size_t>(m.p0 + t) * op.out_ld + m.rb * 128 + i] = res[i * ld + t];
        }
    }
    if (m.kind == kKindGU && a.fused_route) {
        fence_proxy_async();   // h codes are read back by bulk copies
        __syncwarp();
        if (lane == 0) st_release(a.h_ready + static_cast<size_t>(m.slot) * op.RB + m.rb, epoch);
    }
    if (m.kind == kKindDN && a.fused_combine) {
        __syncwarp();   // y rows of every lane before the (acq_rel) combine tickets
        int tok = -1, last = 0;
        if (lane < m.ntok && m.valid) {
            tok = m.shared_static ? lane : pv.pair_tok[m.p0 + lane];
            if (tok >= 0 && tok < a.M) last = atom_add_acq_rel(a.comb + tok * op.RB + m.rb, 1) == a.top_k;
        }
        uint32_t todo = __ballot_sync(0xffffffffu, last);
        __syncwarp();   // the ticket lanes' acquires before every lane's loads
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int tk = __shfl_sync(0xffffffffu, tok, src);
            const int* po = pv.pair_of + tk * (a.top_k + 1);
            // lane owns columns 4*lane .. 4*lane+3; all slots' rows in flight
            const int n = m.rb * 128 + 4 * lane;
            const int ps = po[a.top_k];
            float4 accv = __ldcg(reinterpret_cast<const float4*>(op.out + static_cast<size_t>(ps) * op.out_ld + n));
            for (int j0 = 0; j0 < a.top_k; j0 += 4) {
                float4 yv[4];
                float wv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j0 + j < a.top_k) {
                        const int pj = po[j0 + j];
                        wv[j] = pv.topk_w[tk * a.top_k + j0 + j];
                        yv[j] = __ldcg(reinterpret_cast<const float4*>(op.out + static_cast<size_t>(pj) * op.out_ld + n));
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j0 + j < a.top_k) {
                        accv.x = fmaf(wv[j], yv[j].x, accv.x);
                        accv.y = fmaf(wv[j], yv[j].y, accv.y);
                        accv.z = fmaf(wv[j], yv[j].z, accv.z);
                        accv.w = fmaf(wv[j], yv[j].w, accv.w);
                    }
                }
            }
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(accv.x, accv.y), hi2 = __floats2bfloat162_rn(accv.z, accv.w);
            uint2 packed;
            packed.x = *reinterpret_cast<uint32_t*>(&lo2);
            packed.y = *reinterpret_cast<uint32_t*>(&hi2);
            *reinterpret_cast<uint2*>(a.out_bf16 + static_cast<size_t>(tk) * op.out_ld + n) = packed;
            if (lane == 0) a.comb[tk * op.RB + m.rb] = 0;
        }
    }
}

// Finish segment number `sidx`, whose result the consumers have published.
static __device__ __noinline__ void finish_segment(const StreamArgs& a, SmemTail& sm, long long sidx, int lane, int epoch) {
    const ResRing ring(a);
    const int ld = ring.ld;
    const SegMeta m = sm.seg[sidx % kSegRing];
    if (m.kind == kKindDC) return;   // its sums went out from the consumers
    float* res = ring.at(sm, sidx);
    const int rows = m.kind == kKindGU ? 256 : 128;
    if (!(m.ku0 == 0 && m.ku1 == m.KU)) {
        // split K: publish this CTA's partial, take a ticket, and if this is
        // the last contribution sum all of them in CTA order.
        const long long rblk = m.j;   // the row block's position: its units are rblk*KU ..
        const long long c_lo = cta_of_unit(rblk * m.KU, m.T, m.G);
        const long long c_hi = cta_of_unit(rblk * m.KU + m.KU - 1, m.T, m.G);
        const int n_c = static_cast<int>(c_hi - c_lo + 1);   // CTAs the row block spans
        const int lg = m.kind == kKindGU ? 8 : 7;             // log2(rows)
        float* part_base = a.partials + static_cast<size_t>(m.li) * a.partial_list_floats;
        const int my_slot = static_cast<int>(2 * m.c + ((m.lo / m.KU) == rblk ? 0 : 1));
        float* mine = part_base + static_cast<size_t>(my_slot) * kMaxTok * rows;
        const int nitems = rows * m.ntok;
        for (int idx = lane; idx < nitems; idx += 32) mine[idx] = res[(idx & (rows - 1)) * ld + (idx >> lg)];
        // Lane j resolves CTA c_lo + b + j: the slot of its partial of this
        // row block, null when that CTA holds no unit (all lanes in parallel).
        auto resolve = [&](int b) -> const float* {
            const long long cc = c_lo + b + lane;
            if (cc > c_hi) return nullptr;
            const long long lo = unit_lo(cc, m.T, m.G);
            if (lo >= unit_lo(cc + 1, m.T, m.G)) return nullptr;
            return part_base + static_cast<size_t>(2 * cc + ((lo / m.KU) == rblk ? 0 : 1)) * kMaxTok * rows;
        };
        const float* src0 = resolve(0);
        int n = __popc(__ballot_sync(0xffffffffu, src0 != nullptr));
        for (int b = 32; b < n_c; b += 32) n += __popc(__ballot_sync(0xffffffffu, resolve(b) != nullptr));
        // The warp barrier orders every lane's partial before lane 0's ticket;
        // the acq_rel ticket publishes them and, for the last contribution,
        // acquires everyone else's.
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel(a.tickets[m.li] + rblk, 1) == n - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();   // lane 0's acquire before every lane's loads
        if (last) {
            // kWin contributors' partials are loaded together, then added in
            // CTA order (absent CTAs add +0).
            constexpr int kWin = 8, kPer = 4;
            for (int base = 0; base < nitems; base += kPer * 32) {
                float v[kPer];
#pragma unroll
                for (int j = 0; j < kPer; ++j) v[j] = 0.0f;
                for (int b = 0; b < n_c; b += 32) {
                    const float* sb = b == 0 ? src0 : resolve(b);
                    const int nw = min(32, n_c - b);
                    for (int w0 = 0; w0 < nw; w0 += kWin) {
                        float w[kWin][kPer];
#pragma unroll
                        for (int q = 0; q < kWin; ++q) {
                            const float* sq = reinterpret_cast<const float*>(
                                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(sb), w0 + q));
#pragma unroll
                            for (int j = 0; j < kPer; ++j) {
                                const int idx = base + j * 32 + lane;
                                w[q][j] = (sq != nullptr && idx < nitems) ? __ldcg(sq + idx) : 0.0f;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < kWin; ++q)
#pragma unroll
                            for (int j = 0; j < kPer; ++j) v[j] += w[q][j];
                    }
                }
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int idx = base + j * 32 + lane;
                    if (idx < nitems) res[(idx & (rows - 1)) * ld + (idx >> lg)] = v[j];
                }
            }
            __syncwarp();
            if (lane == 0) a.tickets[m.li][rblk] = 0;
            helper_epilogue(a, sm, m, res, ld, lane, epoch);
        }
    } else {
        helper_epilogue(a, sm, m, res, ld, lane, epoch);
    }
}

// The prep warp walks the same lists / segments as the producer, cut into
// chunks, and prepares each chunk (scales, activation rows, descriptor) at
// most two chunks ahead of the consumers.  Segment metadata goes to
// seg[segment % kSegRing]: when segment S+R is written the consumers have
// started S+R-2, so they found the slots of S+R-2-ns and S+R-3-ns finished;
// one of the two has the parity of S, and each finish warp finishes its
// segments in order, so S is finished once R >= ns + 3.
template <bool kMma>
__device__ __forceinline__ void prep_warp(const StreamArgs& a, SmemTail& sm, int lane, int epoch) {
    long long c = 0;         // chunks prepared
    long long sidx = 0;      // segments started
    bool have_input = false;
    // The lists need the plan, and its scratch shares memory with the result
    // slots: the layer's prep warp starts once the CTA's plan is complete (so
    // every result is written after it).
    if (a.fused_route) {
        if (lane == 0) mbar_wait_or_abort(&sm.plan_bar, 0, sm, a.status);
        __syncwarp();
    }
    // one token: this CTA's consumers quantise all of x into act[0] (the
    // first chunk's slot); otherwise every CTA's share goes to the workspace
    if (a.xloc) {
        if (lane == 0) mbar_wait_or_abort(&sm.xq_bar, 0, sm, a.status);
        __syncwarp();
    }
    int U = *sm.pv.n_uniq;
    if (U < 0 || U > a.max_uniq) {
        if (lane == 0) record_error(a.status, MOEQ_ERR_INVALID_ARG);
        U = 0;
    }
    for (int li = 0; li < a.n_lists && !sm.abort_flag; ++li) {
        const ListInfo L = list_info(a, li, U);
        const Operand& op = kind_op(a, L.kind);
        const int GPU = L.kind == kKindDN ? 2 : 1;   // K groups per unit
        for (int u = static_cast<int>(L.lo); u < static_cast<int>(L.hi) && !sm.abort_flag;) {
            SegMeta m;
            m.kind = L.kind;
            m.li = li;
            m.j = u / L.KU;
            m.ku0 = u - m.j * L.KU;
            list_rb(a, L, m.j, m.e_local, m.rb);
            const int seg_end_u = min(static_cast<int>(L.hi), u - m.ku0 + L.KU);
            m.ku1 = m.ku0 + (seg_end_u - u);
            const ExpertRef er = list_expert(a, sm.pv, L, m.e_local);
            m.expert = er.expert;
            m.p0 = er.p0;
            m.ntok = er.ntok;
            m.slot = er.slot;
            m.shared_static = er.shared_static;
            m.valid = m.expert >= 0 && m.expert < a.n_experts && m.p0 >= 0 && m.ntok >= 1 && m.ntok <= a.max_ntok &&
                      m.p0 + m.ntok <= a.max_pairs;
            if (!m.valid) {
                if (lane == 0) record_error(a.status, MOEQ_ERR_INVALID_ARG);
                m.expert = 0;
                m.p0 = 0;
                m.ntok = 1;
            }
            m.T = L.T;
            m.G = L.G;
            m.c = L.c;
            m.lo = L.lo;
            m.KU = L.KU;
            m.RB = L.RB;
            // activations quantised by the kernel's first phase: all CTAs' shares
            if (op.quant_input && !have_input && !a.xloc) {
                if (lane == 0) wait_count(a.a_cnt, epoch * static_cast<int>(gridDim.x), a.status, &sm.abort_flag);
                __syncwarp();
                have_input = true;
            }
            // down in the layer needs this expert's complete h (lanes check the
            // row-block flags in parallel); the finish warp keeps finishing
            if (m.kind == kKindDN && a.fused_route) {
                const int nrb = a.op[kKindGU].RB;
                for (int j = lane; j < nrb; j += 32)
                    wait_flag(a.h_ready + static_cast<size_t>(m.slot) * nrb + j, epoch, a.status, &sm.abort_flag);
                __syncwarp();
                fence_proxy_async();
            }
            // units per chunk: as many as a slot holds (down by K group: as
            // many as the weight-scale slots hold), evened out over the row
            // block's chunks (so no chunk is a short remainder)
            const int cu_max = m.kind == kKindDC ? kChunkGroups
                             : kMma ? kMmaChunkGroups / GPU : max(1, (kActSlot / (kGroup * m.ntok)) / GPU);
            const int n_chunks = (L.KU + cu_max - 1) / cu_max;
            const int cu = (L.KU + n_chunks - 1) / n_chunks;
            for (int ua = m.ku0; ua < m.ku1; ua += cu) {
                const int ub = min(m.ku1, ua + cu);
                ChunkDesc d;
                d.kind = m.kind;
                d.ku0 = ua;
                d.ku1 = ub;
                d.g0 = m.kind == kKindDC ? m.rb : ua * GPU;
                d.ng = m.kind == kKindDC ? 1 : min(op.KB, ub * GPU) - d.g0;
                d.ntok = m.ntok;
                d.seg_end = ub == m.ku1;
                d.p0 = m.p0;
                // each ends with the prep_full arrival
                if (m.kind == kKindDC)
                    prep_chunk_dc(a, sm, c, sidx, m, d, lane, epoch);
                else
                    prep_chunk<kMma>(a, op, sm, c, sidx, m, L, d, lane);
                ++c;
            }
            ++sidx;
            u = seg_end_u;
        }
    }
    if (sm.abort_flag) {
        // Copies of the last two chunks may still be landing in their slots:
        // wait for them (bounded) before the CTA may exit.
        for (long long j = c > 2 ? c - 2 : 0; j < c; ++j) {
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&sm.prep_full[j & 1], static_cast<uint32_t>((j >> 1) & 1)) &&
                   global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
            }
        }
    }
    // end marker (the consumers pass it on to the finish warp)
    const int cs = static_cast<int>(c & 1);
    if (c >= 2) mbar_wait_or_abort(&sm.act_empty[cs], static_cast<uint32_t>(((c >> 1) - 1) & 1), sm, a.status);
    if (lane == 0) {
        sm.n_segments = static_cast<int>(sidx);
        sm.chunk[cs].kind = -1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.prep_full[cs]);
}

// Finish warp w finishes segments w, w+2, w+4, ... in order as the
// consumers publish them, until the consumers pass on the end marker.
__device__ __forceinline__ void finish_warp(const StreamArgs& a, SmemTail& sm, int w, int lane, int epoch) {
    const ResRing ring(a);
    for (long long sidx = w;; sidx += 2) {
        const int rs = ring.slot(sidx);
        mbar_wait_or_abort(&sm.res_full[rs], ring.parity(sidx), sm, a.status);
        if (sm.abort_flag || sidx >= static_cast<volatile int&>(sm.n_segments)) break;
        finish_segment(a, sm, sidx, lane, epoch);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.res_empty[rs]);
    }
}

// ------------------------------------------------------------------ consumers
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

// As tile_dot for tokens T0 .. T0+MT-1, folding each pass straight into
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

// One segment, chunk after chunk, for one consumer warp.  Leaves one sum per
// (row of this warp, token) in the result slot res (row stride ld).  MODE 1/2: up to that many
// tokens with running sums in registers; MODE 0: any count, two tokens at a
// time, each K group reduced across lanes into the result slot.
template <int KIND, int MODE>
__device__ __forceinline__ void consume_segment(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, float* res,
                                                int ld, int cw, int lane, long long& c, long long& it) {
    constexpr int MT = MODE == 0 ? 2 : MODE;
    constexpr int PASSES = KIND == kKindGU ? 4 : 2;   // 4-row passes per warp and tile
    // gate_up: warp w covers rows (w%8)*16.. of tile w/8; down: rows w*8.. of both tiles
    const int tile_w = KIND == kKindGU ? (cw >> 3) : 0;
    const int rows_base = KIND == kKindGU ? (cw & 7) * 16 : cw * 8;
    const int acc_row0 = KIND == kKindGU ? tile_w * 128 + rows_base : rows_base;
    const int ntok = sm.chunk[c & 1].ntok;
    if (MODE == 0)
        for (int i = lane; i < PASSES * 4 * ntok; i += 32) res[(acc_row0 + i / ntok) * ld + i % ntok] = 0.f;
    float acc[PASSES][MT];
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[p][t] = 0.0f;

    for (bool first = true;; first = false) {
        const int cs = static_cast<int>(c & 1);
        if (!first) mbar_wait_or_abort(&sm.prep_full[cs], static_cast<uint32_t>((c >> 1) & 1), sm, a.status);
        const ChunkDesc d = sm.chunk[cs];
        const float* act = sm.act[cs];
        const float* act_s = sm.act_s[cs];
        const int tok_ld = d.ng * kGroup;
        for (int ku = d.ku0; ku < d.ku1; ++ku, ++it) {
            const int s = static_cast<int>(it % kStages);
            mbar_wait_or_abort(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status);
            const uint8_t* st = stages + static_cast<size_t>(s) * kStageBytes;
            const int ntile = KIND == kKindGU ? 1 : min(2, a.op[KIND].KB - 2 * ku);
            for (int tt = 0; tt < ntile; ++tt) {
                const int gl = (KIND == kKindGU ? ku : 2 * ku + tt) - d.g0;
                const uint8_t* tile = st + (KIND == kKindGU ? tile_w : tt) * kTile;
                const float* act_g = act + gl * kGroup;
                const float swg = sm.sw[cs][tile_w][gl];
                if (MODE != 0) {
                    float scl[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) scl[t] = act_s[min(t, ntok - 1) * d.ng + gl] * swg;
                    tile_dot_acc<MT, PASSES, 0, MT>(tile, rows_base, act_g, tok_ld, ntok, lane, scl, acc);
                } else {
                    for (int t0 = 0; t0 < ntok; t0 += 2) {
                        float part[PASSES][2];
                        tile_dot<2, PASSES>(tile, rows_base, act_g, tok_ld, t0, ntok, lane, part);
#pragma unroll
                        for (int p = 0; p < PASSES; ++p) {
                            const int row = acc_row0 + p * 4 + (lane >> 3);
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const float v = reduce8(part[p][t]);
                                if ((lane & 7) == 0 && t0 + t < ntok)
                                    res[row * ld + t0 + t] += v * (act_s[(t0 + t) * d.ng + gl] * swg);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.act_empty[cs]);
        ++c;
        if (d.seg_end || sm.abort_flag) break;
    }
    if (MODE != 0) {
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int row = acc_row0 + p * 4 + (lane >> 3);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v = reduce8(acc[p][t]);
                if ((lane & 7) == 0 && t < ntok) res[row * ld + t] = v;
            }
        }
    }
}

// Every mode runs out of line: each gets the whole register budget for its
// streaming loop, and the consumer's outer state is saved once per segment.
template <int KIND, int MODE>
__device__ __noinline__ void consume_segment_cold(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, float* res,
                                                  int ld, int cw, int lane, long long& c_io, long long& it_io) {
    long long c = c_io, it = it_io;   // in registers for the streaming loop
    consume_segment<KIND, MODE>(a, sm, stages, res, ld, cw, lane, c, it);
    c_io = c;
    it_io = it;
}

template <int KIND>
__device__ __forceinline__ void consume_dispatch(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, float* res,
                                                 int ld, int ntok, int cw, int lane, long long& c, long long& it) {
    if (ntok <= 1)
        consume_segment_cold<KIND, 1>(a, sm, stages, res, ld, cw, lane, c, it);
    else if (ntok <= 2)
        consume_segment_cold<KIND, 2>(a, sm, stages, res, ld, cw, lane, c, it);
    else
        consume_segment_cold<KIND, 0>(a, sm, stages, res, ld, cw, lane, c, it);
}

// Down by K group, one token: a unit holds tiles (2u, kb) and (2u+1, kb),
// 256 output rows over the one K group kb of h; warp w takes rows
// (w%8)*16 .. +15 of tile w/8, as gate_up does.  Each unit's sums are
// complete for that group: scaled by s_h * s_w and stored as the pair's
// (kb, row) sums, 16 consecutive floats per warp.
static __device__ __noinline__ void consume_dc(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, int cw, int lane,
                                        long long& c_io, long long& it_io) {
    long long c = c_io, it = it_io;
    const Operand& op = a.op[kKindDN];
    const size_t H = static_cast<size_t>(op.NB) * 128;
    const int tile_w = cw >> 3, rows_base = (cw & 7) * 16;
    const int l8 = lane & 7, rsub = lane >> 3;
    for (bool first = true;; first = false) {
        const int cs = static_cast<int>(c & 1);
        if (!first) mbar_wait_or_abort(&sm.prep_full[cs], static_cast<uint32_t>((c >> 1) & 1), sm, a.status);
        const ChunkDesc d = sm.chunk[cs];
        // the group's decoded codes, the same for every unit of the chunk
        float2 av[8];
        const float4* ap = reinterpret_cast<const float4*>(sm.act[cs]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ap[i * 8 + l8];
            av[2 * i] = make_float2(v.x, v.y);
            av[2 * i + 1] = make_float2(v.z, v.w);
        }
        const float sa = sm.act_s[cs][0];
        float* dst = a.dc_part + (static_cast<size_t>(d.p0) * op.KB + d.g0) * H + rows_base + lane;
        for (int ku = d.ku0; ku < d.ku1; ++ku, ++it) {
            const int s = static_cast<int>(it % kStages);
            mbar_wait_or_abort(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status);
            const uint8_t* tile = stages + static_cast<size_t>(s) * kStageBytes + tile_w * kTile;
            float r = 0.0f;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int row = rows_base + p * 4 + rsub;
                const uint4 w = *reinterpret_cast<const uint4*>(tile + row * 128 + ((l8 ^ (row & 7)) << 4));
                float2 wf[8];
                e4m3x4_to_f32(w.x, wf[0], wf[1]);
                e4m3x4_to_f32(w.y, wf[2], wf[3]);
                e4m3x4_to_f32(w.z, wf[4], wf[5]);
                e4m3x4_to_f32(w.w, wf[6], wf[7]);
                float2 dd = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < 8; ++j) dd = __ffma2_rn(wf[j], av[j], dd);
                // row rows_base + 4p + q ends in lane 8q; lane 4p + q takes it
                const float v = __shfl_sync(0xffffffffu, reduce8(dd.x + dd.y), (lane & 3) * 8);
                if ((lane >> 2) == p) r = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            if (lane < 16) dst[static_cast<size_t>(2 * ku + tile_w) * 128] = r * (sa * sm.sw[cs][tile_w][ku - d.ku0]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.act_empty[cs]);
        ++c;
        if (d.seg_end || sm.abort_flag) break;
    }
    c_io = c;
    it_io = it;
}

// ------------------------------------------------------------------ tcgen05 path
// (defined in the translation unit that instantiates the tcgen05 kernels)
template <bool kMma>
__device__ __noinline__ void mma_issue_loop(const StreamArgs& a, SmemTail& sm, const uint8_t* stages, int lane);
template <bool kMma>
__device__ __noinline__ void mma_epilogue_loop(const StreamArgs& a, SmemTail& sm, int warp, int lane);

// the routing half of the consumers (warps 0 .. kCW/2-1)
struct RouteSync {
    __device__ __forceinline__ void operator()() const { named_sync(2, kConsumers / 2); }
};

// The kernel's first phase: the inputs given as activations (x for gate_up;
// for a standalone down call, its input) are live-quantised once, each
// (row, 128-group) by one consumer warp of one CTA, into the decoded
// consumer layout that chunk loads copy from.
template <bool kGuF32, bool kDnF32, bool kMma>
__device__ __noinline__ void quantise_inputs(const StreamArgs& a, int warp, int nwarps, int lane) {
    const long long G = gridDim.x, c = blockIdx.x;
    const long long n0 = a.op[0].quant_input ? static_cast<long long>(a.op[0].rows_a) * a.op[0].KB : 0;
    const long long n1 = a.op[1].quant_input ? static_cast<long long>(a.op[1].rows_a) * a.op[1].KB : 0;
    const long long n = n0 + n1;
    const long long lo = c * n / G, hi = (c + 1) * n / G;
    for (long long i = lo + warp; i < hi; i += nwarps) {
        const int k = i < n0 ? 0 : 1;
        const Operand& op = a.op[k];
        const long long j = i < n0 ? i : i - n0;
        const int row = static_cast<int>(j / op.KB), g = static_cast<int>(j % op.KB);
        const float4 v = (k == 0 ? kGuF32 : kDnF32)
                             ? load_act4<true>(op.a, static_cast<size_t>(op.K), row, g * kGroup + lane * 4)
                             : load_act4<false>(op.a, static_cast<size_t>(op.K), row, g * kGroup + lane * 4);
        float sc;
        float4 dec;
        const uint32_t codes = quant_group_warp(v, &sc, &dec);
        if constexpr (kMma)
            store_code_phases(reinterpret_cast<uint8_t*>(op.aq) + static_cast<size_t>(row) * op.K + g * kGroup,
                              static_cast<size_t>(op.rows_a) * op.K, lane, codes);
        else
            *reinterpret_cast<float4*>(op.aq + (static_cast<size_t>(row) * op.KB + g) * kGroup + act_pos(lane * 4)) = dec;
        if (lane == 0) op.as[static_cast<size_t>(row) * op.KB + g] = sc;
        if (op.qdump) {
            *reinterpret_cast<uint32_t*>(op.qdump + static_cast<size_t>(row) * op.K + g * kGroup + lane * 4) = codes;
            if (lane == 0) op.sdump[static_cast<size_t>(row) * op.KB + g] = sc;
        }
    }
}

// The combine after down by K group (consumer threads, after their last
// segment).  Every CTA counts itself in dc_cnt once its sums are out; then
// CTA c combines output columns [c*H/G, (c+1)*H/G): per pair, the sum over
// K groups in group order, then out = y_shared + sum_j w_j y_j in the
// plan's order of picks, rounded once to bf16.  One token.
static __device__ __noinline__ void dc_combine(const StreamArgs& a, SmemTail& sm, int tid, int epoch) {
    consumer_sync();   // every consumer's sums are stored ...
    if (tid == 0) {
        __threadfence();   // ... and thread 0's fence releases them with the count
        atom_add_acq_rel(a.dc_cnt, 1);
        wait_count(a.dc_cnt, epoch * static_cast<int>(gridDim.x), a.status, &sm.abort_flag);
    }
    consumer_sync();   // thread 0's acquire before every thread's loads
    if (sm.abort_flag) return;
    const Operand& op = a.op[kKindDN];
    const int H = op.NB * 128, KB = op.KB, k = a.top_k, P = k + 1;
    const long long G = gridDim.x, cta = blockIdx.x;
    const int n0 = static_cast<int>(cta * H / G), W = static_cast<int>((cta + 1) * H / G) - n0;
    float* ys = sm.act[0];   // [P][W]: the activation slots are idle now
    for (int i = tid; i < P * W; i += kConsumers) {
        const int p = i / W, n = n0 + i % W;
        const float* src = a.dc_part + static_cast<size_t>(p) * KB * H + n;
        float v = 0.0f;
#pragma unroll 16
        for (int kb = 0; kb < KB; ++kb) v += __ldcg(src + static_cast<size_t>(kb) * H);
        ys[i] = v;
    }
    consumer_sync();
    const int* po = sm.pv.pair_of;   // token 0
    for (int i = tid; i < W; i += kConsumers) {
        float acc = ys[po[k] * W + i];
        for (int j = 0; j < k; ++j) acc = fmaf(sm.pv.topk_w[j], ys[po[j] * W + i], acc);
        a.out_bf16[n0 + i] = __float2bfloat16_rn(acc);
    }
}

// One token, x quantised by each CTA for itself: every 128-group of row 0
// by one warp, decoded codes straight into act[0] (group g at g*128, the
// consumer layout) and the scales into act_s[0]: the first chunk's slot.
// The warp's groups are all loaded before any is quantised (one round trip).
constexpr int kXLocalPer = kXLocalMaxK / kGroup / (kCW / 2);   // groups per warp of the quantising half
static_assert(kXLocalPer * kGroup * (kCW / 2) == kXLocalMaxK, "x groups split evenly over the warps");
template <bool kF32>
__device__ __noinline__ void quantise_x_local(const StreamArgs& a, SmemTail& sm, int warp, int lane) {
    const Operand& op = a.op[kKindGU];
    constexpr int nwarps = kCW / 2;
    float4 v[kXLocalPer];
#pragma unroll
    for (int i = 0; i < kXLocalPer; ++i) {
        const int g = warp + i * nwarps;
        v[i] = g < op.KB ? load_act4<kF32>(op.a, static_cast<size_t>(op.K), 0, g * kGroup + lane * 4)
                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < kXLocalPer; ++i) {
        const int g = warp + i * nwarps;
        if (g < op.KB) {   // warp-uniform
            float sc;
            float4 dec;
            quant_group_warp(v[i], &sc, &dec);
            *reinterpret_cast<float4*>(sm.act[0] + g * kGroup + act_pos(lane * 4)) = dec;
            if (lane == 0) sm.act_s[0][g] = sc;
        }
    }
}

// CTA 0 hands its copy of the plan to the caller (the kernel never reads it).
static __device__ __noinline__ void copy_plan_out(const StreamArgs& a, const LocalPlan& lp, int tid) {
    const int M = a.M, k = a.top_k, U = lp.n_uniq, P = M * (k + 1);
    constexpr int kN = kConsumers / 2;
    for (int i = tid; i < M * k; i += kN) {
        a.plan.topk_id[i] = lp.topk_id[i];
        a.plan.topk_w[i] = lp.topk_w[i];
    }
    for (int i = tid; i <= U; i += kN) {
        if (i < U) a.plan.uniq[i] = lp.uniq[i];
        a.plan.offs[i] = lp.offs[i];
    }
    for (int i = tid; i < P; i += kN) {
        a.plan.pair_tok[i] = lp.pair_tok[i];
        a.plan.pair_of[i] = lp.pair_of[i];
    }
    if (tid == 0) *a.plan.n_uniq = U;
}

template <bool kGuF32, bool kDnF32, bool kMma>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ StreamArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemTail& sm = *reinterpret_cast<SmemTail*>(stages + static_cast<size_t>(kStages) * kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        // the tcgen05 path frees a stage by one MMA commit and has four
        // epilogue warps in place of the sixteen consumer warps
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kMma ? 1 : kCW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.prep_full[s], 1);
            mbar_init(&sm.act_empty[s], kMma ? kEpiWarps : kCW);
        }
        for (int s = 0; s < kMaxRes; ++s) {
            mbar_init(&sm.res_full[s], kMma ? 4 : kCW);   // tcgen05 path: epilogue set 0 publishes
            mbar_init(&sm.res_empty[s], 1);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(&sm.mma_done[b], 1);
            mbar_init(&sm.tmem_empty[b], 4);   // the four warps of the set that owns the buffer
        }
        mbar_init(&sm.plan_bar, 1);
        mbar_init(&sm.xq_bar, 1);
        mbar_init(&sm.hloc_bar, 1);
        if (a.fused_route) {
            sm.pv.n_uniq = &sm.plan.n_uniq;
            sm.pv.uniq = sm.plan.uniq;
            sm.pv.offs = sm.plan.offs;
            sm.pv.pair_tok = sm.plan.pair_tok;
            sm.pv.pair_of = sm.plan.pair_of;
            sm.pv.topk_w = sm.plan.topk_w;
        } else {
            sm.pv.n_uniq = a.n_uniq;
            sm.pv.uniq = a.uniq;
            sm.pv.offs = a.offs;
            sm.pv.pair_tok = a.pair_tok;
            sm.pv.pair_of = a.pair_of;
            sm.pv.topk_w = a.topk_w;
        }
        sm.abort_flag = 0;
        sm.n_segments = 0x7fffffff;
        sm.finish_done = 0;
        fence_mbar_init();
    }
    if (kMma && warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tc_fence_before();
    }
    if (a.fused_route && warp < kCW) {
        // the logits (and one token's x) are read right after the barrier
        // below: start their lines towards L2 now
        const int lg_lines = (a.M * a.E_routed * 4 + 127) / 128;
        if (tid < lg_lines) prefetch_l2(reinterpret_cast<const char*>(a.logits) + 128 * tid);
        const int x_lines = a.xloc ? (a.op[kKindGU].K * (a.op[kKindGU].a_f32 ? 4 : 2) + 127) / 128 : 0;
        if (tid < x_lines) prefetch_l2(static_cast<const char*>(a.op[kKindGU].a) + 128 * tid);
    }
    const int epoch = ld_relaxed(a.epoch) + 1;
    // every launch adds one per CTA to dc_cnt (keeping it at epoch * grid);
    // down by K group counts in its combine
    if (tid == 0 && !a.dc) atomicAdd(a.dc_cnt, 1);
    __syncthreads();

    if (warp == kProducerWarp) {
        if (lane == 0) producer(a, sm, stages, epoch);
        return;
    }
    if (warp == kPrepWarp) {
        prep_warp<kMma>(a, sm, lane, epoch);
        return;
    }
    if (warp == kFinishWarp0 || warp == kFinishWarp1) {
        finish_warp(a, sm, warp - kFinishWarp0, lane, epoch);
        // the second finish warp to end closes the CTA's work
        if (lane == 0 && atomicAdd(&sm.finish_done, 1) == 1) {
            // The last CTA to finish publishes the epoch for the next launch.
            __threadfence();
            if (atomicAdd(a.done, 1) == static_cast<int>(gridDim.x) - 1) {
                *a.done = 0;
                __threadfence();
                st_release(a.epoch, epoch);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp;
    if (!a.fused_route) {
        quantise_inputs<kGuF32, kDnF32, kMma>(a, cw, kCW, lane);
        fence_proxy_async();
        __threadfence();
        consumer_sync();
        if (tid == 0) atomicAdd(a.a_cnt, 1);
    } else if (cw >= kCW / 2 && a.xloc) {
        // half the consumers quantise all of one token's x into this CTA's
        // first activation slot (the count keeps a_cnt at epoch * grid) ...
        quantise_x_local<kGuF32>(a, sm, cw - kCW / 2, lane);
        named_sync(3, kConsumers / 2);
        if (cw == kCW / 2 && lane == 0) {
            mbar_arrive(&sm.xq_bar);
            atomicAdd(a.a_cnt, 1);
        }
    } else if (cw >= kCW / 2) {
        // half the consumers quantise this CTA's share of the inputs ...
        quantise_inputs<kGuF32, kDnF32, kMma>(a, cw - kCW / 2, kCW / 2, lane);
        fence_proxy_async();
        __threadfence();
        named_sync(3, kConsumers / 2);
        if (cw == kCW / 2 && lane == 0) atomicAdd(a.a_cnt, 1);
    } else {
        // ... while the other half routes: every CTA for itself (identical,
        // deterministic plans)
        moeq_route_plan lp;
        lp.topk_id = sm.plan.topk_id;
        lp.topk_w = sm.plan.topk_w;
        lp.n_uniq = &sm.plan.n_uniq;
        lp.uniq = sm.plan.uniq;
        lp.offs = sm.plan.offs;
        lp.pair_tok = sm.plan.pair_tok;
        lp.pair_of = sm.plan.pair_of;
        route_compute<kConsumers / 2>(a.logits, a.M, a.E_routed, a.top_k, lp, sm.route, tid, RouteSync{});
        RouteSync{}();
        if (blockIdx.x == 0) copy_plan_out(a, sm.plan, tid);
        if (tid == 0) mbar_arrive(&sm.plan_bar);
    }
    if constexpr (kMma) {
        // tcgen05 path: warps 0-7 read the accumulators, warp 8 issues the
        // MMAs and owns the TMEM allocation; the other consumer warps are done
        if (cw < kEpiWarps) {
            tc_fence_after();
            mma_epilogue_loop<kMma>(a, sm, cw, lane);
            tc_fence_before();
        } else if (cw == kMmaWarp) {
            tc_fence_after();
            mma_issue_loop<kMma>(a, sm, stages, lane);
        }
        if (cw <= kMmaWarp) {
            named_sync(4, (kEpiWarps + 1) * 32);
            if (cw == kMmaWarp) {
                tc_fence_after();
                tmem_dealloc(sm.tmem_base, kTmemCols);
            }
        }
        return;
    }
    const ResRing ring(a);
    long long c = 0, it = 0, sidx = 0;
    for (;;) {
        const int rs = ring.slot(sidx);
        // the slot's previous segment (sidx - ns) must be finished
        if (sidx >= ring.ns) mbar_wait_or_abort(&sm.res_empty[rs], ring.parity(sidx) ^ 1u, sm, a.status);
        const int cs = static_cast<int>(c & 1);
        mbar_wait_or_abort(&sm.prep_full[cs], static_cast<uint32_t>((c >> 1) & 1), sm, a.status);
        const int kind = sm.chunk[cs].kind;
        if (kind < 0 || sm.abort_flag) {
            // pass the end on to both finish warps: as segment sidx (the
            // warp of its parity waits for it) and as segment sidx + 1 (the
            // other warp), each in its slot once that slot is free
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.res_full[rs]);
            const long long s2 = sidx + 1;
            if (s2 >= ring.ns) mbar_wait_or_abort(&sm.res_empty[ring.slot(s2)], ring.parity(s2) ^ 1u, sm, a.status);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.res_full[ring.slot(s2)]);
            break;
        }
        const int ntok = sm.chunk[cs].ntok;
        float* res = ring.at(sm, sidx);
        if (kind == kKindGU)
            consume_dispatch<kKindGU>(a, sm, stages, res, ring.ld, ntok, cw, lane, c, it);
        else if (kind == kKindDC)
            consume_dc(a, sm, stages, cw, lane, c, it);
        else
            consume_dispatch<kKindDN>(a, sm, stages, res, ring.ld, ntok, cw, lane, c, it);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.res_full[rs]);
        ++sidx;
    }
    if (a.dc) dc_combine(a, sm, tid, epoch);
}

// Launch one instantiation (persistent, one CTA per SM, all shared memory).
// Internal linkage: each library instance (and translation unit) keeps its
// own per-device "attribute set" flags and kernel handles.
template <bool G32, bool D32, bool kMma>
static cudaError_t launch_t(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    static int configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(stream_kernel<G32, D32, kMma>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
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
    return cudaLaunchKernelEx(&cfg, stream_kernel<G32, D32, kMma>, args);
}

template <bool kMma>
static cudaError_t launch_mode(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream) {
    const bool g = args.op[kKindGU].a_f32 != 0, d = args.op[kKindDN].a_f32 != 0;
    if (g)
        return d ? launch_t<true, true, kMma>(args, grid, cooperative, stream)
                 : launch_t<true, false, kMma>(args, grid, cooperative, stream);
    return d ? launch_t<false, true, kMma>(args, grid, cooperative, stream)
             : launch_t<false, false, kMma>(args, grid, cooperative, stream);
}

}  // namespace moeq
