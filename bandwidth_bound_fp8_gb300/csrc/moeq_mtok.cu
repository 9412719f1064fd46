// The multi-token MoE layer kernel (1..16 tokens: decode and draft
// verification): route, live quantisation of x, gate_up + SwiGLU, live
// quantisation of h, down and the combine in one launch, the GEMMs on the
// tcgen05 tensor cores.
//
// GLM-5.2 x10 is the source of the method: tokens verified together read
// each expert once (§5-§6); a decode layer is a read of its active experts'
// FP8 weights (bandwidth model); the activations are quantised live in front
// of each GEMM (§1, §8c), fused into it (§4); the per-block scales stay out
// of the tensor-core accumulator -- a fresh TMEM sum per 128-wide K group,
// promoted in fp32 -- so that loads and MMAs pipeline (§2-§3).
//
// Work.  As in the one-token kernel, a column is (unique expert, kb): the
// gate rows kb*128.. and the up rows I+kb*128.. over all of H (KB stages of
// two tiles), then down's K group kb -- the 128 h values the column forms
// itself -- against every output row (KB/2 stages of two tiles).  The
// column's tokens are its expert's; its MMAs take every token (N = 16
// accumulator columns, token n in column n) and the epilogue keeps the
// column's own.  The shared expert's columns -- every token's, the costliest
// to finish -- are spaced evenly among the routed ones, so that they fall on
// different CTAs.  Every column streams the same bytes
// whatever its token count, so the launch's stages (ncols x 3KB/2) are dealt
// out evenly
// (stream-K): a CTA's range may begin inside one column and end inside
// another.  The CTA streams the head of the column its range ends in FIRST
// and publishes what the rest of that column needs (the gate and up sums so
// far, or h's codes once gate_up is complete), then its whole columns, and
// LAST the tail of the column its range begins in -- whose head the previous
// CTA published at its very start, so that wait is over long before it
// comes.  Down leaves one fp32 partial per (token, column, output row),
// already scaled by its expert's routing weight; once every CTA has stored
// its partials, each token's 16-row parts are summed in a fixed order and
// rounded to bf16.
//
// Warp roles (384 threads, one CTA per SM):
//   warps 0-5   at the start, the routing of every token (each CTA for itself);
//   warps 6-11  at the start, the live quantisation of x: each 1 x 128 group
//               once in the whole grid (one warp each), into one copy in
//               L2 laid out as gate_up's B operand, counted in per K group;
//               then warp 6 waits for each K group's count and releases the
//               group (its scales in shared memory) to the producer;
//   warp 0      producer: one lane issues the bulk copies of each stage; a
//               gate_up stage also carries the x codes of its K group for
//               every token;
//   warp 1      MMA: one lane issues the tcgen05 MMAs (2 tiles x 4 K steps
//               per stage) into one of four TMEM accumulator sets;
//   warps 2-5   epilogue: each thread owns one TMEM lane (a row of the
//               tiles) and promotes each stage's sums with the block scales;
//               SwiGLU and h's quantisation; down's partials;
//   warp 7      tickets: as the epilogue stores down partials it counts each
//               (column, output unit) in (one gpu-scope fence per batch);
//   warps 8-11  the sums: each (token, 16 output rows) once its unit's count
//               shows every column in -- the units complete one after another
//               as the last columns' down stages pass them, so the sums
//               overlap the end of the streams.
// Launched with programmatic dependent launch: before griddepcontrol.wait a
// CTA only starts its share of the shared expert's weights towards L2.
//
// One instantiation per mode (the template parameter):
//   kMtokLayer    the MoE layer, as above;
//   kMtokDense    a dense FFN (top_k = 0, no routing: the one expert is the
//                 "shared" one, serving every token); with fewer columns
//                 than CTAs the CTAs left over stream the columns' first
//                 gate_up stages (share_of);
//   kMtokGateUp   gate_up + SwiGLU alone over a caller's plan, h to global;
//   kMtokDown     down alone over a caller's plan: each piece's epilogue
//                 quantises its rows of a into a shared-memory B operand,
//                 and the stages, independent of one another, are dealt
//                 over every CTA.
#include "moeq_device.cuh"
#include "moeq_internal.h"
#include "moeq_route.cuh"

// The gate_up-alone instantiation leaves the epilogue's h step once h is
// written, so the rest of that step is unreachable there by design.
#pragma nv_diag_suppress 128

namespace moeq {
namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4, kQuantWarp0 = 6, kQuantWarps = 6;
constexpr int kTicketWarp = 7, kSumWarp0 = 8, kSumWarps = 4;
constexpr int kRouteThreads = kQuantWarp0 * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kTile = 16384;
constexpr int kN = 16;                                 // MMA N: token columns of the accumulators
constexpr int kXGroupBytes = kMtokXGroupBytes;         // one K group of x codes: B operand of gate_up
constexpr int kStageBytes = 2 * kTile + kXGroupBytes;  // 34 KiB: two weight tiles + the x group
constexpr int kStages = 4;
constexpr int kTmemBufs = 4;
constexpr int kTmemCols = kTmemBufs * 2 * kN;          // 128
constexpr int kMaxKB = kTokenMaxH / 128;
constexpr int kMaxPicks = kMaxTok * kRouteMaxK;
constexpr int kParts = 16;                             // 16-row parts of a 256-row output unit
constexpr uint32_t kIdesc = umma_idesc_e4m3(128, kN);
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-aligned");
static_assert(kXGroupBytes == kN * 128, "x group: 16 token rows of 128 bytes");
static_assert(kMtokSlotBytes >= 2 * kN * 128 * 4 + kXGroupBytes + kN * 4, "split slot size");

// The route plan of the launch, in shared memory.
struct PlanSmem {
    int topk_id[kMaxPicks];
    float topk_w[kMaxPicks];
    int n_uniq;
    int uniq[kMaxPicks + 1];
    int offs[kMaxPicks + 2];
    int pair_tok[kMaxTok * (kRouteMaxK + 1)];
    int pair_of[kMaxTok * (kRouteMaxK + 1)];
};

// One piece of a column: stages [t0, t1) of column j (0 .. GS-1 gate_up,
// GS .. GS+NU-1 down's output units; down alone: GS = 0 and the column is
// an expert's K group), with what the epilogue needs of it.
struct ColInfo {
    float sw[3][kMaxKB];   // gate and up weight scales per K group of x; down's per row block
    float rw[kN];          // routing weight of the token's pick of this expert (1: the shared one)
    float xsc[kN];         // down mode: the activation scale of each row at the column's K group
    int pbase[kN];         // the token's partials of this column: offset in `part` of unit 0, row 0
    int pair[kN];          // the (token, expert) pair: row of h and of its dumps
    uint32_t tmask;        // tokens of the column
    int j, t0, t1, expert, kb;
};

struct Smem {
    alignas(1024) uint8_t hbuf[kXGroupBytes];   // h codes: down's B operand (token n in row n, 128B swizzle)
    alignas(1024) uint8_t abuf[2][kXGroupBytes];   // down alone: a's codes of a piece's K group (B operand),
                                                   // by piece parity
    float sx[kMaxKB][kN];                       // x scales per (K group, token)
    float hs[kN], hw[kN];                       // h scales; h scale x routing weight
    float amax[kEpiWarps][kN];
    ColInfo col[2];
    PlanSmem plan;
    RouteScratch rs;
    uint64_t full[kStages], empty[kStages], mma_done[kTmemBufs], tmem_empty[kTmemBufs], h_ready, a_ready[2];
    uint64_t xq_bar[kMaxKB];
    uint32_t tmem_base;
    int wdone[kEpiWarps];                       // down stages whose partials each epilogue warp has stored
    int abort_flag;
    int last_cta;                               // this CTA is the last one out
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void epi_sync() { named_sync(1, kEpiThreads); }
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Sleeping bounded wait (producer, epilogue); on expiry the launch is
// aborted with MOEQ_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_sleep(uint64_t* bar, uint32_t parity, Smem& sm, int* status) {
    if (mbar_wait_sleep_bounded(bar, parity, &sm.abort_flag)) return true;
    record_error(status, MOEQ_ERR_TIMEOUT);
    sm.abort_flag = 1;
    return false;
}
// Spinning bounded wait (the MMA lane: issue latency matters there).
__device__ __forceinline__ bool wait_spin(uint64_t* bar, uint32_t parity, Smem& sm, int* status) {
    if (mbar_wait_bounded(bar, parity, &sm.abort_flag)) return true;
    record_error(status, MOEQ_ERR_TIMEOUT);
    sm.abort_flag = 1;
    return false;
}

// Bounded wait for a global flag to become non-zero (acquire); one thread.
__device__ bool wait_flag(const int* flag, Smem& sm, int* status) {
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire(flag) != 0) return true;
        if ((i & 7u) == 7u) {
            if (sm.abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                record_error(status, MOEQ_ERR_TIMEOUT);
                sm.abort_flag = 1;
                return false;
            }
        }
        __nanosleep(128);
    }
}

__device__ __forceinline__ const uint8_t* gu_tile(const MtokArgs& a, int e, int nb, int kb) {
    return a.w_gu + ((static_cast<size_t>(e) * (2 * a.RB) + nb) * a.KB + kb) * kTile;
}
__device__ __forceinline__ const uint8_t* dn_tile(const MtokArgs& a, int e, int nb, int kb) {
    return a.w_d + ((static_cast<size_t>(e) * a.KB + nb) * a.RB + kb) * kTile;
}
__device__ __forceinline__ uint8_t* xq_group(const MtokArgs& a, int t) {
    return a.xq + static_cast<size_t>(t) * kXGroupBytes;
}
__device__ __forceinline__ uint8_t* slot_at(const MtokArgs& a, int b) {
    return a.slots + static_cast<size_t>(b) * kMtokSlotBytes;
}

// ------------------------------------------------------------------ share
// This CTA's share of the launch's stages: the head of column head_j (stages
// [0, head_t1)), whole columns [j0, j1), the tail of column tail_j (stages
// [tail_t0, tail_t1)).  With more columns than CTAs the stages are dealt
// evenly (a range then holds at most one head and one tail).  With no more
// columns than CTAs it depends on the launch:
//   kShareColumns (the MoE layer): one column per CTA;
//   kShareHelp (the dense layer): one column per CTA, and the CTAs left over
//     (helpers) stream the first g0 gate_up stages of every column, each
//     helper a few columns' heads in turn, handing their sums on through
//     the column's own slot; g0 is as large as lets every head be done
//     before its column's owner has streamed the rest of gate_up: the
//     busiest helper's h heads take h g0 <= GS - g0 stages, so
//     g0 = GS / (h + 1) with h = ceil(columns / helpers).  Only while a
//     helper has at most two heads of at least 8 stages: each piece costs
//     its CTA a column set-up and a hand-over of about a microsecond or
//     two, which many small heads would put on the owners' path;
//   kShareChain (gate_up alone): the stages dealt evenly over min(G, 2 ncols)
//     CTAs, so that a range is at least half a column and a column spans at
//     most three CTAs -- a range may lie inside one column (a "tail" that
//     ends before the column does: a middle piece, which takes the sums of
//     the CTA before and hands them on to the CTA after);
//   kShareFree (down alone, every stage its own partial): dealt evenly over
//     the whole grid.
constexpr int kShareColumns = 0, kShareChain = 1, kShareFree = 2, kShareHelp = 3;
struct Share {
    int head_j, head_t1, j0, j1, tail_j, tail_t0, tail_t1, np;
    int help;            // kShareHelp with helpers: splits hand on through the column's slot
    int hj0, hstep, g0;  // a helper's heads: columns hj0, hj0 + hstep, ..., stages [0, g0)
};

__device__ Share share_of(int ncols, int spc, int gs, int kind) {
    const int G = gridDim.x, c = blockIdx.x;
    Share s;
    s.head_j = s.tail_j = -1;
    s.head_t1 = s.tail_t0 = 0;
    s.tail_t1 = spc;
    s.help = s.hj0 = s.hstep = s.g0 = 0;
    const int nh = G - ncols, hmax = nh > 0 ? (ncols + nh - 1) / nh : 0;
    const int g0 = kind == kShareHelp && ncols > 0 && nh > 0 ? min(gs / (hmax + 1), gs - 1) : 0;
    if (g0 >= 8 && hmax <= 2) {
        s.help = 1;
        s.g0 = g0;
        s.j0 = s.j1 = 0;
        if (c < ncols) {
            // the owner: the rest of column c
            s.tail_j = c;
            s.tail_t0 = g0;
        } else {
            s.hj0 = c - ncols;
            s.hstep = nh;
        }
        s.np = c < ncols ? 1 : (ncols - (c - ncols) + nh - 1) / nh;
        return s;
    }
    if ((kind == kShareChain || kind == kShareFree) && ncols <= G) {
        const int Gs = kind == kShareChain ? min(G, 2 * ncols) : G;
        const long long S = static_cast<long long>(ncols) * spc;
        const long long lo = S * min(c, Gs) / Gs, hi = S * min(c + 1, Gs) / Gs;
        const int jx = static_cast<int>(lo / spc), bx = static_cast<int>(lo - static_cast<long long>(jx) * spc);
        const int jy = static_cast<int>(hi / spc), ey = static_cast<int>(hi - static_cast<long long>(jy) * spc);
        s.j0 = s.j1 = 0;
        if (jy == jx) {
            // inside one column (or empty)
            if (ey > bx) {
                s.tail_j = jx;
                s.tail_t0 = bx;
                s.tail_t1 = ey;
            }
        } else {
            // the range is no longer than a column here, so it spans at
            // most two: the end of column jx, then the start of column jy
            s.tail_j = jx;
            s.tail_t0 = bx;
            if (ey > 0) {
                s.head_j = jy;
                s.head_t1 = ey;
            }
        }
    } else if (ncols <= G) {
        s.j0 = c < ncols ? c : 0;
        s.j1 = c < ncols ? c + 1 : 0;
    } else {
        // the range is longer than a column (ncols > G), so it holds at most
        // one head and one tail, of different columns
        const long long S = static_cast<long long>(ncols) * spc;
        const long long lo = S * c / G, hi = S * (c + 1) / G;
        const int jx = static_cast<int>(lo / spc), bx = static_cast<int>(lo - static_cast<long long>(jx) * spc);
        const int jy = static_cast<int>(hi / spc), ey = static_cast<int>(hi - static_cast<long long>(jy) * spc);
        if (bx > 0) {
            s.tail_j = jx;
            s.tail_t0 = bx;
        }
        if (ey > 0) {
            s.head_j = jy;
            s.head_t1 = ey;
        }
        s.j0 = bx > 0 ? jx + 1 : jx;
        s.j1 = jy;
    }
    s.np = (s.head_j >= 0) + (s.j1 - s.j0) + (s.tail_j >= 0);
    return s;
}

// Piece i of the share, in processing order: head, whole columns, tail (or
// a helper's heads).
__device__ __forceinline__ void piece_at(const Share& s, int i, int spc, int& j, int& t0, int& t1) {
    if (s.hstep > 0) {
        j = s.hj0 + i * s.hstep;
        t0 = 0;
        t1 = s.g0;
        return;
    }
    if (s.head_j >= 0) {
        if (i == 0) {
            j = s.head_j;
            t0 = 0;
            t1 = s.head_t1;
            return;
        }
        --i;
    }
    if (i < s.j1 - s.j0) {
        j = s.j0 + i;
        t0 = 0;
        t1 = spc;
        return;
    }
    j = s.tail_j;
    t0 = s.tail_t0;
    t1 = s.tail_t1;
}

// ------------------------------------------------------------------ routing
// Every CTA routes all tokens into its shared memory (the plan definition of
// moeq_route), with warps 0-5; CTA 0 also writes the plan out.
struct RouteSync {
    __device__ void operator()() const { named_sync(2, kRouteThreads); }
};
template <int MODE>
__device__ void route_all(const MtokArgs& a, Smem& sm, int tid) {
    moeq_route_plan p;
    p.topk_id = sm.plan.topk_id;
    p.topk_w = sm.plan.topk_w;
    p.n_uniq = &sm.plan.n_uniq;
    p.uniq = sm.plan.uniq;
    p.offs = sm.plan.offs;
    p.pair_tok = sm.plan.pair_tok;
    p.pair_of = sm.plan.pair_of;
    if (MODE == kMtokGateUp || MODE == kMtokDown) {
        // the caller's plan (unique experts, their pair ranges, gate_up: each
        // pair's token), checked as the persistent engine checks it: an
        // expert out of range, a pair range that is empty, out of range or
        // wider than one MMA's 16 rows, or (gate_up) a token out of range or
        // twice on one expert leaves MOEQ_ERR_INVALID_ARG and no work
        const int U0 = __ldcg(a.plan.n_uniq);
        const int U = U0 >= 0 && U0 <= a.max_uniq ? U0 : 0;
        const int cap = MODE == kMtokGateUp ? a.M : min(a.max_pairs, kN);
        if (tid == 0) sm.rs.total[0] = U0 != U;
        for (int i = tid; i < U; i += kRouteThreads) sm.plan.uniq[i] = __ldcg(a.plan.uniq + i);
        for (int i = tid; i <= U; i += kRouteThreads) sm.plan.offs[i] = __ldcg(a.plan.offs + i);
        named_sync(2, kRouteThreads);
        for (int g = tid; g < U; g += kRouteThreads) {
            const int e = sm.plan.uniq[g], r0 = sm.plan.offs[g], r1 = sm.plan.offs[g + 1];
            bool ok = e >= 0 && e < a.n_experts && r0 >= 0 && r1 > r0 && r1 - r0 <= cap && r1 <= a.max_pairs;
            if (MODE == kMtokGateUp && ok) {
                uint32_t seen = 0;
                for (int q = r0; q < r1; ++q) {
                    const int n = __ldcg(a.plan.pair_tok + q);
                    ok = ok && n >= 0 && n < a.M && !((seen >> n) & 1u);
                    if (!ok) break;
                    seen |= 1u << n;
                    sm.plan.pair_tok[q] = n;
                }
            }
            if (!ok) atomicOr(&sm.rs.total[0], 1);
        }
        named_sync(2, kRouteThreads);
        if (tid == 0) {
            const bool bad = sm.rs.total[0] != 0;
            if (bad) record_error(a.status, MOEQ_ERR_INVALID_ARG);
            sm.plan.n_uniq = bad ? 0 : U;
            if (bad) sm.plan.offs[0] = 0;
        }
        named_sync(2, kRouteThreads);
        return;
    }
    if (a.top_k == 0) {
        // a dense FFN: no routing -- one expert (index E_routed) serving
        // every token, one pair per token
        if (tid == 0) {
            sm.plan.n_uniq = 1;
            sm.plan.uniq[0] = a.E_routed;
            sm.plan.offs[0] = 0;
            sm.plan.offs[1] = a.M;
        }
        if (tid < a.M) {
            sm.plan.pair_tok[tid] = tid;
            sm.plan.pair_of[tid] = tid;
        }
        named_sync(2, kRouteThreads);
        return;
    }
    if (a.M == 1) {
        // one token: one warp, no block barrier
        if (tid < 32) {
            if (a.E_routed <= 256)
                route_one_token_warp<8>(a.logits, a.E_routed, a.top_k, tid, p, sm.rs.id[0], sm.rs.lv[0]);
            else
                route_one_token_warp<kRouteMaxE / 32>(a.logits, a.E_routed, a.top_k, tid, p, sm.rs.id[0], sm.rs.lv[0]);
        }
    } else {
        route_compute<kRouteThreads>(a.logits, a.M, a.E_routed, a.top_k, p, sm.rs, tid, RouteSync{});
    }
    named_sync(2, kRouteThreads);
    if (blockIdx.x == 0) {
        const int M = a.M, k = a.top_k, U = sm.plan.n_uniq, P = sm.plan.offs[U];
        for (int i = tid; i < M * k; i += kRouteThreads) {
            a.plan.topk_id[i] = sm.plan.topk_id[i];
            a.plan.topk_w[i] = sm.plan.topk_w[i];
        }
        for (int i = tid; i < U; i += kRouteThreads) a.plan.uniq[i] = sm.plan.uniq[i];
        for (int i = tid; i <= U; i += kRouteThreads) a.plan.offs[i] = sm.plan.offs[i];
        for (int i = tid; i < P; i += kRouteThreads) a.plan.pair_tok[i] = sm.plan.pair_tok[i];
        for (int i = tid; i < M * (k + 1); i += kRouteThreads) a.plan.pair_of[i] = sm.plan.pair_of[i];
        if (tid == 0) *a.plan.n_uniq = U;
    }
}

// ------------------------------------------------------------------ x
// Live quantisation of x (GLM-5.2 x10 §1, §8c: 1 x 128 groups, s = amax/448,
// RNE to E4M3), once in the whole grid: group (t, n) -- K group t of token
// n, t-major -- goes to warp q of the quantising warps (6-11 of every CTA),
// which writes its codes into row n of K group t of the one copy in L2 (the
// gate_up stages' B operand: token n in row n of an 8-row, 128-byte-swizzled
// atom pair) and its scale beside it, then counts itself in K group t.
// (layer, dense and gate_up: down alone quantises its rows of a per piece)
__device__ void quantise_x(const MtokArgs& a, int wq, int lane) {
    const int M = a.M, ngroups = M * a.KX;
    for (int q = blockIdx.x * kQuantWarps + wq; q < ngroups; q += gridDim.x * kQuantWarps) {
        const int t = q / M, n = q - t * M;
        const float4 v = a.x_f32 ? load_act4<true>(a.x, static_cast<size_t>(a.x_ld), n, t * 128 + 4 * lane)
                                 : load_act4<false>(a.x, static_cast<size_t>(a.x_ld), n, t * 128 + 4 * lane);
        float sc;
        float4 dec;
        const uint32_t codes = quant_group_warp(v, &sc, &dec);
        // token n in row n of K group t's 16 rows (128-byte swizzle)
        *reinterpret_cast<uint32_t*>(xq_group(a, t) + n * 128 + (((lane >> 2) ^ (n & 7)) << 4) + (lane & 3) * 4) =
            codes;
        if (lane == 0) a.xs[t * kN + n] = sc;
        if (a.q_x) {
            *reinterpret_cast<uint32_t*>(a.q_x + static_cast<size_t>(n) * a.x_ld + t * 128 + 4 * lane) = codes;
            if (lane == 0) a.s_x[n * a.KX + t] = sc;
        }
        fence_proxy_async_global();   // the codes are read by bulk copies (async proxy)
        __threadfence();       // ... and by other CTAs: released by the count below
        __syncwarp();
        if (lane == 0) atomicAdd(a.cnt + kMtokX + kMtokPad * t, 1);
    }
}


// Warp 6, once the plan is known: lane l watches K groups l and l + 32,
// each on its own (bounded) -- once a group's count shows all M tokens in,
// the lane takes its scales into shared memory and releases it to the
// producer and the epilogue.
__device__ void x_ready(const MtokArgs& a, Smem& sm, int lane) {
    constexpr int kPer = (kMaxKB + 31) / 32;
    bool done[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) done[i] = lane + 32 * i >= a.KX;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        bool all = true;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (done[i]) continue;
            const int t = lane + 32 * i;
            if (ld_relaxed(a.cnt + kMtokX + kMtokPad * t) >= a.M && ld_acquire(a.cnt + kMtokX + kMtokPad * t) >= a.M) {
                fence_proxy_async_global();
                for (int n = 0; n < kN; ++n) sm.sx[t][n] = n < a.M ? __ldcg(a.xs + t * kN + n) : 0.0f;
                mbar_arrive(&sm.xq_bar[t]);
                done[i] = true;
            } else {
                all = false;
            }
        }
        if (all) break;
        if (sm.abort_flag) break;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_error(a.status, MOEQ_ERR_TIMEOUT);
            sm.abort_flag = 1;
            break;
        }
        __nanosleep(64);
    }
}

// ------------------------------------------------------------------ producer
// Column j's (unique expert slot g, K group kb): the routed experts' columns
// in expert-major order (each expert's gate rows, then up rows, one run of
// tiles after another), with the shared expert's columns -- every token's,
// the costliest to finish -- spaced evenly among them (one after every U - 1
// routed columns), so that they fall on different CTAs.
__device__ __forceinline__ void col_of(int j, int U, int RB, int& g, int& kb) {
    const int b = j / U, o = j - b * U;
    if (o == U - 1) {
        g = U - 1;
        kb = b;
    } else {
        const int r = b * (U - 1) + o;
        g = r / RB;
        kb = r - g * RB;
    }
}

// Returns the number of stages issued (all of the share's, unless aborted).
// A gate_up stage's weight tiles go out at once; its x group follows as soon
// as that K group is released (at the start of the launch x may still be on
// its way), so that x's quantisation overlaps the first tiles' latency.
// Before the producer blocks on a free stage, every deferred x copy is out.
template <int MODE>
__device__ long long producer(const MtokArgs& a, Smem& sm, uint8_t* stages, const Share& sh, int spc) {
    const uint64_t pol = l2_evict_first_policy();
    constexpr bool down = MODE == kMtokDown;
    const uint32_t gu_xbytes = static_cast<uint32_t>(a.M) * 128;
    // a gate_up stage's x copy waits for its K group's release: (stage, K group)
    int pend_s[kStages], pend_t[kStages];
    int npend = 0;
    auto flush = [&]() -> bool {
        for (int q = 0; q < npend; ++q) {
            if (!wait_sleep(&sm.xq_bar[pend_t[q]], 0, sm, a.status)) return false;
            bulk_load(stages + static_cast<size_t>(pend_s[q]) * kStageBytes + 2 * kTile, xq_group(a, pend_t[q]),
                      gu_xbytes, &sm.full[pend_s[q]], pol);
        }
        npend = 0;
        return true;
    };
    auto x_copy = [&](int s, int t) {
        if (npend == 0 && mbar_try_wait(&sm.xq_bar[t], 0)) {
            bulk_load(stages + static_cast<size_t>(s) * kStageBytes + 2 * kTile, xq_group(a, t), gu_xbytes,
                      &sm.full[s], pol);
        } else {
            pend_s[npend] = s;
            pend_t[npend] = t;
            ++npend;
        }
    };
    long long it = 0;
    for (int i = 0; i < sh.np && !sm.abort_flag; ++i) {
        int j, t0, t1, g, kb;
        piece_at(sh, i, spc, j, t0, t1);
        col_of(j, sm.plan.n_uniq, a.RB, g, kb);
        const int e = sm.plan.uniq[g];
        for (int t = t0; t < t1; ++t, ++it) {
            const int s = static_cast<int>(it % kStages);
            if (it >= kStages) {
                if (!flush()) return it;
                if (!wait_sleep(&sm.empty[s], static_cast<uint32_t>((it / kStages - 1) & 1), sm, a.status))
                    return it;
            }
            uint8_t* dst = stages + static_cast<size_t>(s) * kStageBytes;
            if (!down && t < a.GS) {
                mbar_arrive_expect_tx(&sm.full[s], 2 * kTile + gu_xbytes);
                bulk_load(dst, gu_tile(a, e, kb, t), kTile, &sm.full[s], pol);
                bulk_load(dst + kTile, gu_tile(a, e, a.RB + kb, t), kTile, &sm.full[s], pol);
                x_copy(s, t);
            } else {
                const int u = t - a.GS;
                mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
                bulk_load(dst, dn_tile(a, e, 2 * u, kb), kTile, &sm.full[s], pol);
                bulk_load(dst + kTile, dn_tile(a, e, 2 * u + 1, kb), kTile, &sm.full[s], pol);
            }
        }
    }
    flush();
    return it;
}

// After an abort: let the copies in flight land before the CTA may exit (bounded).
__device__ void producer_drain(Smem& sm, long long issued) {
    for (long long i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&sm.full[i % kStages], static_cast<uint32_t>((i / kStages) & 1)) &&
               global_timer_ns() - t0 < 100ull * 1000ull * 1000ull) {
        }
    }
}

// ------------------------------------------------------------------ MMA
// One lane: per stage, 2 tiles x 4 K steps into accumulator set it % 4
// (tile 0 at columns 32b .. 32b+15, tile 1 at 32b+16 ..).  gate_up's B is
// the stage's x group; down's is h's codes, ready once h_ready completes.
template <int MODE>
__device__ long long mma_issuer(const MtokArgs& a, Smem& sm, const uint8_t* stages, const Share& sh, int spc,
                                int lane) {
    const uint32_t stage0 = smem_u32(stages), hb = smem_u32(sm.hbuf);
    const uint32_t ab[2] = {smem_u32(sm.abuf[0]), smem_u32(sm.abuf[1])};
    long long it = 0, last = -1;
    int hcount = 0;
    for (int i = 0; i < sh.np; ++i) {
        int j, t0, t1;
        piece_at(sh, i, spc, j, t0, t1);
        for (int t = t0; t < t1; ++t, ++it) {
            const int s = static_cast<int>(it % kStages), b = static_cast<int>(it % kTmemBufs);
            if (!wait_spin(&sm.full[s], static_cast<uint32_t>((it / kStages) & 1), sm, a.status)) return last;
            if (it >= kTmemBufs &&
                !wait_spin(&sm.tmem_empty[b], static_cast<uint32_t>(((it / kTmemBufs) - 1) & 1), sm, a.status))
                return last;
            if ((MODE == kMtokLayer || MODE == kMtokDense) && t == max(t0, a.GS)) {   // the piece's first down stage: its h codes
                if (!wait_spin(&sm.h_ready, static_cast<uint32_t>(hcount & 1), sm, a.status)) return last;
                ++hcount;
            }
            if (MODE == kMtokDown && t == t0) {   // down alone: the piece's rows of a, quantised by the epilogue
                if (!wait_spin(&sm.a_ready[i & 1], static_cast<uint32_t>((i >> 1) & 1), sm, a.status)) return last;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sa = stage0 + static_cast<uint32_t>(s * kStageBytes);
                const uint32_t bb = MODE == kMtokDown ? ab[i & 1] : (t < a.GS ? sa + 2 * kTile : hb);
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const uint32_t d = sm.tmem_base + static_cast<uint32_t>((b * 2 + tt) * kN);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f8(d, umma_desc_sw128(sa + tt * kTile + 32 * k), umma_desc_sw128(bb + 32 * k), kIdesc, k);
                }
                umma_commit(&sm.mma_done[b]);
                umma_commit(&sm.empty[s]);
            }
            __syncwarp();
            last = it;
        }
    }
    return last;
}

// ------------------------------------------------------------------ epilogue
// Column info of piece i (scales, and per token: membership, pick, pair).
template <int MODE>
__device__ void load_col(const MtokArgs& a, Smem& sm, const Share& sh, int spc, int i, int etid) {
    ColInfo& ci = sm.col[i & 1];
    int j, t0, t1;
    piece_at(sh, i, spc, j, t0, t1);
    int g, kb;
    col_of(j, sm.plan.n_uniq, a.RB, g, kb);
    const int e = sm.plan.uniq[g];
    const int KB = a.KB, NBg = 2 * a.RB;
    for (int q = etid; q < 3 * KB; q += kEpiThreads) {
        const int which = q / KB, t = q - which * KB;
        if (which < 2 && MODE == kMtokDown) continue;     // no gate_up
        if (which == 2 && MODE == kMtokGateUp) continue;  // no down
        float v;
        if (which < 2)
            v = __ldg(a.s_gu + (static_cast<size_t>(e) * NBg + which * a.RB + kb) * KB + t);
        else
            v = __ldg(a.s_d + (static_cast<size_t>(e) * KB + t) * a.RB + kb);
        ci.sw[which][t] = v;
    }
    if (MODE == kMtokDown) {
        // down alone: the piece's rows of a at K group kb (the expert's pair
        // rows offs[g] ..), quantised here into the piece's B operand and
        // their scales into the column info.  Buffer i & 1 was piece i - 2's,
        // whose MMAs are complete: this runs before the epilogue takes piece
        // i - 1's stages, after it took all of piece i - 2's.  The piece
        // that holds the column's first stage writes the optional dump.
        const int r0 = sm.plan.offs[g], nr = min(sm.plan.offs[g + 1] - r0, kN);
        const int w = etid >> 5, lane = etid & 31;
        uint8_t* b = sm.abuf[i & 1];
        constexpr int kRows = kN / kEpiWarps;   // a warp's rows: w, w + 4, ...
        float4 v[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int n = w + q * kEpiWarps;
            if (n < nr)
                v[q] = a.x_f32 ? load_act4<true>(a.x, static_cast<size_t>(a.x_ld), r0 + n, kb * 128 + 4 * lane)
                               : load_act4<false>(a.x, static_cast<size_t>(a.x_ld), r0 + n, kb * 128 + 4 * lane);
        }
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int n = w + q * kEpiWarps;
            if (n < nr) {
                float sc;
                float4 dec;
                const uint32_t codes = quant_group_warp(v[q], &sc, &dec);
                *reinterpret_cast<uint32_t*>(b + n * 128 + (((lane >> 2) ^ (n & 7)) << 4) + (lane & 3) * 4) = codes;
                if (lane == 0) ci.xsc[n] = sc;
                if (a.q_x && t0 == 0) {
                    *reinterpret_cast<uint32_t*>(a.q_x + static_cast<size_t>(r0 + n) * a.x_ld + kb * 128 + 4 * lane) =
                        codes;
                    if (lane == 0) a.s_x[(r0 + n) * a.KX + kb] = sc;
                }
            }
        }
        fence_proxy_async_smem();   // the codes are read by the MMAs (async proxy)
        epi_sync();
        if (etid == 0) mbar_arrive(&sm.a_ready[i & 1]);
    }
    if (etid < 32) {
        const int n = etid, k = a.top_k, U = sm.plan.n_uniq, nu = a.NU;
        int pair = -1, slot = 0;
        float w = 0.0f, xsc = 0.0f;
        if (MODE == kMtokDown) {
            // row n of the column: the expert's pair row offs[g] + n
            if (n < min(sm.plan.offs[g + 1] - sm.plan.offs[g], kN)) {
                pair = sm.plan.offs[g] + n;
                w = 1.0f;
                xsc = ci.xsc[n];
            }
        } else if (n < a.M) {
            for (int p = sm.plan.offs[g]; p < sm.plan.offs[g + 1]; ++p)
                if (sm.plan.pair_tok[p] == n) pair = p;
            if (pair >= 0) {
                if (MODE == kMtokGateUp || g == U - 1) {
                    slot = k;
                    w = 1.0f;
                } else {
                    for (int q = 0; q < k; ++q)
                        if (sm.plan.topk_id[n * k + q] == e) {
                            slot = q;
                            w = sm.plan.topk_w[n * k + q];
                        }
                }
            }
        }
        const uint32_t m = __ballot_sync(0xffffffffu, pair >= 0);
        if (n < kN) {
            // partials: [row][unit][slot][kb][256 rows] (row: token, or down's pair row)
            const int row = MODE == kMtokDown ? (pair >= 0 ? pair : 0) : n;
            ci.rw[n] = w;
            ci.xsc[n] = xsc;
            ci.pbase[n] = ((row * nu * (k + 1) + slot) * a.RB + kb) * 256;
            ci.pair[n] = pair;
        }
        if (n == 0) {
            ci.tmask = m;
            ci.j = j;
            ci.t0 = t0;
            ci.t1 = t1;
            ci.expert = e;
            ci.kb = kb;
        }
    }
}

template <int NT>
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t (&r0)[NT], uint32_t (&r1)[NT]) {
    tmem_ld_nowait<NT>(taddr, r0);
    tmem_ld_nowait<NT>(taddr + kN, r1);
    tmem_wait_ld();
}

// The epilogue's view of one stage's accumulators: wait for its MMAs, load
// both tiles' NT token columns of this thread's lane, free the set.
template <int NT>
__device__ __forceinline__ bool epi_take(const MtokArgs& a, Smem& sm, long long it, uint32_t tlane,
                                         uint32_t (&r0)[NT], uint32_t (&r1)[NT], int lane) {
    const int b = static_cast<int>(it % kTmemBufs);
    const bool ok = wait_sleep(&sm.mma_done[b], static_cast<uint32_t>((it / kTmemBufs) & 1), sm, a.status);
    tc_fence_after();
    tmem_ld2<NT>(tlane + static_cast<uint32_t>(b * 2 * kN), r0, r1);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.tmem_empty[b]);
    return ok;
}

template <int NT, int MODE>
__device__ void epilogue(const MtokArgs& a, Smem& sm, const Share& sh, int spc, int warp, int lane) {
    const int etid = (warp - kEpiWarp0) * 32 + lane, quad = warp & 3;
    const int r = quad * 32 + lane;                       // the TMEM lane: row of the tiles
    const uint32_t tlane = sm.tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const int GS = a.GS, k = a.top_k, c = blockIdx.x;
    constexpr bool layer = MODE == kMtokLayer || MODE == kMtokDense, down_only = MODE == kMtokDown;
    const int ustride = (k + 1) * a.RB * 256;   // partials of one output unit, per token
    long long it = 0;
    int stored = 0;
    if (sh.np > 0) load_col<MODE>(a, sm, sh, spc, 0, etid);
    for (int i = 0; i < sh.np; ++i) {
        epi_sync();   // piece i's column info is loaded; the previous piece's is no longer read
        if (i + 1 < sh.np) load_col<MODE>(a, sm, sh, spc, i + 1, etid);
        const ColInfo& ci = sm.col[i & 1];
        const int t0 = ci.t0, t1 = ci.t1, kb = ci.kb;
        const uint32_t tmask = ci.tmask;
        float accg[NT], accu[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) accg[n] = accu[n] = 0.0f;

        // gate_up: stages [t0, min(t1, GS))
        for (int t = t0; t < min(t1, GS); ++t, ++it) {
            uint32_t rg[NT], ru[NT];
            epi_take<NT>(a, sm, it, tlane, rg, ru, lane);
            wait_sleep(&sm.xq_bar[t], 0, sm, a.status);   // x's scales of group t (returns at once after the first)
            const float sg = ci.sw[0][t], su = ci.sw[1][t];
            const float4* sx4 = reinterpret_cast<const float4*>(sm.sx[t]);
#pragma unroll
            for (int q = 0; q < NT / 4; ++q) {
                const float4 x = sx4[q];
                const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    accg[4 * q + z] = fmaf(__uint_as_float(rg[4 * q + z]), sg * xs[z], accg[4 * q + z]);
                    accu[4 * q + z] = fmaf(__uint_as_float(ru[4 * q + z]), su * xs[z], accu[4 * q + z]);
                }
            }
        }

        // a split inside gate_up hands on through the slot and flag of the
        // CTA boundary (b before, b + 1 after this CTA), or with helpers
        // through the column's own
        const int slot_in = sh.help ? ci.j : c, slot_out = sh.help ? ci.j : c + 1;
        if (!down_only && t0 > 0 && t0 <= GS) {
            // the tail (or a middle piece) of a column split inside gate_up:
            // the sums of the CTA before + this CTA's
            if (etid == 0) wait_flag(a.cnt + kMtokFlags + slot_in, sm, a.status);
            epi_sync();
            const float* gu = reinterpret_cast<const float*>(slot_at(a, slot_in));
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                accg[n] = __ldcg(gu + n * 128 + r) + accg[n];
                accu[n] = __ldcg(gu + (kN + n) * 128 + r) + accu[n];
            }
        }
        if (!down_only && t1 <= GS && t1 < spc) {
            // the head (or a middle piece) of a column split inside gate_up:
            // hand the sums so far on to the CTA after
            float* gu = reinterpret_cast<float*>(slot_at(a, slot_out));
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                gu[n * 128 + r] = accg[n];
                gu[(kN + n) * 128 + r] = accu[n];
            }
            __threadfence();
            epi_sync();
            if (etid == 0) st_release(a.cnt + kMtokFlags + slot_out, 1);
            continue;
        }
        if (down_only) {
            // down alone: the rows' codes come with every stage
        } else if (t0 <= GS) {
            // SwiGLU and the live quantisation of h (GLM-5.2 x10 §8c): per
            // token of the column, its 128 h values form one group (the
            // rows of the other tokens keep finite codes from before: their
            // accumulator columns are never used)
            float h[NT], m[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                h[n] = 0.0f;
                if ((tmask >> n) & 1u) {
                    const float gv = accg[n];
                    h[n] = __fdiv_rn(gv, 1.0f + expf(-gv)) * accu[n];
                    if (a.h) a.h[static_cast<size_t>(ci.pair[n]) * a.I + kb * 128 + r] = h[n];
                }
                m[n] = fabsf(h[n]);
            }
            if (!layer) continue;   // gate_up alone: h is the result
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    if ((tmask >> n) & 1u) m[n] = fmaxf(m[n], __shfl_xor_sync(0xffffffffu, m[n], o));
            }
            if (lane == 0) {
#pragma unroll
                for (int n = 0; n < NT; ++n) sm.amax[quad][n] = m[n];
            }
            epi_sync();
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if ((tmask >> n) & 1u) {
                    const float amax =
                        fmaxf(fmaxf(sm.amax[0][n], sm.amax[1][n]), fmaxf(sm.amax[2][n], sm.amax[3][n]));
                    const float s = __fdiv_rn(amax, 448.0f);
                    const uint8_t code =
                        s == 0.0f ? (signbit(h[n]) ? 0x80u : 0u)
                                  : static_cast<uint8_t>(e4m3x2_from_f32(__fdiv_rn(h[n], s), 0.0f) & 0xFFu);
                    sm.hbuf[n * 128 + ((((r >> 4) ^ (n & 7))) << 4) + (r & 15)] = code;
                    if (a.q_h) {
                        a.q_h[static_cast<size_t>(ci.pair[n]) * a.I + kb * 128 + r] = code;
                        if (r == 0) a.s_h[ci.pair[n] * a.RB + kb] = s;
                    }
                    if (etid == n) {
                        sm.hs[n] = s;
                        sm.hw[n] = s * ci.rw[n];
                    }
                }
            }
            fence_proxy_async_smem();   // h's codes are read by the MMAs (async proxy)
            epi_sync();
            if (t1 < spc) {
                // the head of a column split inside down: publish h's codes and scales
                uint8_t* sl = slot_at(a, c + 1);
                reinterpret_cast<uint4*>(sl + 2 * kN * 128 * 4)[etid] = reinterpret_cast<const uint4*>(sm.hbuf)[etid];
                if (etid < kN) reinterpret_cast<float*>(sl + 2 * kN * 128 * 4 + kXGroupBytes)[etid] = sm.hs[etid];
                __threadfence();
                epi_sync();
                if (etid == 0) st_release(a.cnt + kMtokFlags + c + 1, 1);
            }
        } else {
            // the tail of a column split inside down: h's codes from the head
            if (etid == 0) wait_flag(a.cnt + kMtokFlags + c, sm, a.status);
            epi_sync();
            const uint8_t* sl = slot_at(a, c);
            reinterpret_cast<uint4*>(sm.hbuf)[etid] = __ldcg(reinterpret_cast<const uint4*>(sl + 2 * kN * 128 * 4) + etid);
            if (etid < kN) {
                const float s = __ldcg(reinterpret_cast<const float*>(sl + 2 * kN * 128 * 4 + kXGroupBytes) + etid);
                sm.hs[etid] = s;
                sm.hw[etid] = s * ci.rw[etid];
            }
            fence_proxy_async_smem();
            epi_sync();
        }
        if (layer && etid == 0) mbar_arrive(&sm.h_ready);

        // down: stages [max(t0, GS), t1), unit u = t - GS; partials scaled by
        // the row's activation scale (h's, or down alone: a's), its routing
        // weight and the block's weight scale
        for (int t = max(t0, GS); t < t1; ++t, ++it) {
            uint32_t d0[NT], d1[NT];
            epi_take<NT>(a, sm, it, tlane, d0, d1, lane);
            const int u = t - GS;
            const float s0 = ci.sw[2][2 * u], s1 = ci.sw[2][2 * u + 1];
            float* pu = a.part + static_cast<size_t>(u) * ustride + r;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if ((tmask >> n) & 1u) {
                    const float hwn = down_only ? ci.xsc[n] : sm.hw[n];
                    float* p = pu + ci.pbase[n];
                    p[0] = __uint_as_float(d0[n]) * (hwn * s0);
                    p[128] = __uint_as_float(d1[n]) * (hwn * s1);
                }
            }
            // the ticket warp learns of the stored partials
            ++stored;
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                *reinterpret_cast<volatile int*>(&sm.wdone[warp - kEpiWarp0]) = stored;
            }
        }
    }
}

// ------------------------------------------------------------------ combine
// Token n's rows 256u + 16w .. +15: the fixed-order sum of its (k+1) x RB
// partials (slot-major, each already carrying its routing weight), as in
// the one-token kernel: lane (row quad lane % 4, column class lane / 4) adds
// its columns in order, a fixed butterfly adds the classes, lanes 0..3 round
// to bf16.
__device__ void combine_part(const MtokArgs& a, int n, int u, int w, int lane) {
    const int nu = a.NU, ncol = (a.top_k + 1) * a.RB;
    const float* base = a.part + (static_cast<size_t>(n) * nu + u) * ncol * 256 + 16 * w;
    const int n4 = ncol * 4;
    constexpr int kBatch = 12;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int f0 = lane; f0 < n4; f0 += 32 * kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int f = f0 + 32 * b;
            v[b] = f < n4 ? __ldcg(reinterpret_cast<const float4*>(base + (f >> 2) * 256) + (f & 3))
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
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
        const size_t o = static_cast<size_t>(n) * a.H + 256 * u + 16 * w + 4 * lane;
        if (a.out_f32) {
            *reinterpret_cast<float4*>(a.out_f32 + o) = acc;
        } else {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 packed;
            packed.x = *reinterpret_cast<const uint32_t*>(&lo);
            packed.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(a.out + o) = packed;
        }
    }
}

// ------------------------------------------------------------------ counts
// The unit of this CTA's q-th down stage (its pieces' down stages in order).
__device__ int unit_of_down_stage(const Share& sh, int spc, int KB, int q) {
    for (int i = 0; i < sh.np; ++i) {
        int j, t0, t1;
        piece_at(sh, i, spc, j, t0, t1);
        const int d0 = max(t0, KB), nd = max(0, t1 - d0);
        if (q < nd) return d0 - KB + q;   // KB: gate_up stages per column
        q -= nd;
    }
    return 0;
}

// Warp 7: as the epilogue warps store down partials (their progress
// counters in shared memory), one gpu-scope fence releases every partial
// stored so far, then one fire-and-forget add per (column, unit) arrival.
// A unit is complete once its count reaches ncols.
__device__ void ticket_warp(const MtokArgs& a, Smem& sm, const Share& sh, int spc, int lane) {
    const int GS = a.GS;
    int total = 0;
    for (int i = 0; i < sh.np; ++i) {
        int j, t0, t1;
        piece_at(sh, i, spc, j, t0, t1);
        total += max(0, t1 - max(t0, GS));
    }
    int done = 0;
    unsigned long long t0 = global_timer_ns();
    while (done < total && !sm.abort_flag) {
        const int mine = lane < kEpiWarps ? reinterpret_cast<volatile int*>(sm.wdone)[lane] : 0x7fffffff;
        const int avail = __reduce_min_sync(0xffffffffu, mine);
        if (avail <= done) {
            __nanosleep(64);
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (lane == 0) record_error(a.status, MOEQ_ERR_TIMEOUT);
                sm.abort_flag = 1;
            }
            continue;
        }
        t0 = global_timer_ns();
        __threadfence();   // releases the partials stored by every epilogue warp so far
        for (int q = done + lane; q < avail; q += 32) atomicAdd(a.cnt + kMtokU + kMtokPad * unit_of_down_stage(sh, spc, GS, q), 1);
        done = avail;
    }
}

// Warps 8-11: the sums, in unit order (task p: unit p / (16M), then token,
// then 16-row part), each once its unit's count shows all ncols columns in
// (bounded wait).
template <int MODE>
__device__ void sum_worker(const MtokArgs& a, Smem& sm, int ncols, int wi, int lane) {
    // the rows summed: the tokens, or (down alone) the plan's pair rows
    const int row0 = MODE == kMtokDown ? sm.plan.offs[0] : 0;
    const int rows = MODE == kMtokDown ? sm.plan.offs[sm.plan.n_uniq] - row0 : a.M;
    const int nu = a.NU, per_unit = rows * kParts, ntask = nu * per_unit;
    for (int p = blockIdx.x * kSumWarps + wi; p < ntask; p += gridDim.x * kSumWarps) {
        const int u = p / per_unit, rem = p - u * per_unit;
        int ok = 0;
        if (lane == 0) {
            const int* cnt = a.cnt + kMtokU + kMtokPad * u;
            const unsigned long long t0 = global_timer_ns();
            for (uint32_t i = 0;; ++i) {
                if (ld_relaxed(cnt) >= ncols) {
                    ok = ld_acquire(cnt) >= ncols;   // acquires the unit's partials
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
                // few polls while the unit is far from complete
                __nanosleep(ld_relaxed(cnt) * 4 < ncols * 3 ? 1024 : 64);
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        combine_part(a, row0 + rem / kParts, u, rem % kParts, lane);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) mtok_kernel(const __grid_constant__ MtokArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem& sm = *reinterpret_cast<Smem*>(stages + static_cast<size_t>(kStages) * kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, G = gridDim.x;
    if (tid == 0) pdl_launch_dependents();
    if (tid < kStages) {
        mbar_init(&sm.full[tid], 1);
        mbar_init(&sm.empty[tid], 1);
    } else if (tid >= 32 && tid < 32 + kTmemBufs) {
        mbar_init(&sm.mma_done[tid - 32], 1);
        mbar_init(&sm.tmem_empty[tid - 32], kEpiWarps);
    } else if (tid == 64) {
        mbar_init(&sm.h_ready, 1);
        mbar_init(&sm.a_ready[0], 1);
        mbar_init(&sm.a_ready[1], 1);
        sm.abort_flag = 0;
    } else if (tid >= 96 && tid < 96 + kMaxKB) {
        mbar_init(&sm.xq_bar[tid - 96], 1);
    }
    fence_mbar_init();
    if (tid < kEpiWarps) sm.wdone[tid] = 0;
    // rows M .. 15 of every stage's x group and all of h's codes stay zero:
    // their accumulator columns are never used, but stay finite
    for (int q = tid; q < kStages * kXGroupBytes / 16; q += kThreads) {
        const int s = q / (kXGroupBytes / 16), o = (q % (kXGroupBytes / 16)) * 16;
        *reinterpret_cast<uint4*>(stages + static_cast<size_t>(s) * kStageBytes + 2 * kTile + o) = make_uint4(0, 0, 0, 0);
    }
    for (int q = tid; q < kXGroupBytes / 16; q += kThreads) reinterpret_cast<uint4*>(sm.hbuf)[q] = make_uint4(0, 0, 0, 0);
    for (int q = tid; q < 2 * kXGroupBytes / 16; q += kThreads)
        reinterpret_cast<uint4*>(&sm.abuf[0][0])[q] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == kMmaWarp) tmem_alloc(&sm.tmem_base, kTmemCols);
    // before the previous kernel is done: this CTA's share of the shared
    // expert's weights towards L2 (nothing writes weights)
    if (warp == kMmaWarp + 2) {
        // the logits and x are the previous kernel's to write until
        // griddepcontrol.wait; their lines can still be brought into L2 now
        // (L2 is where every SM's writes meet), so the reads after the wait hit
        const int lg_lines = (a.M * a.E_routed * 4 + 127) / 128, x_lines = (a.M * a.x_ld * (a.x_f32 ? 4 : 2) + 127) / 128;
        for (int i = lane; i < lg_lines + x_lines; i += 32)
            prefetch_l2(i < lg_lines ? reinterpret_cast<const char*>(a.logits) + 128 * i
                                     : reinterpret_cast<const char*>(a.x) + 128 * (i - lg_lines));
    }
    if (warp == kProducerWarp && a.top_k > 0) {
        const long long gu_tiles = 2LL * a.RB * a.KB, tiles = gu_tiles + static_cast<long long>(a.KB) * a.RB;
        const long long lo = tiles * blockIdx.x / G, hi = tiles * (blockIdx.x + 1) / G;
        for (long long t = lo + lane; t < hi; t += 32) {
            const uint8_t* src = t < gu_tiles ? gu_tile(a, a.E_routed, 0, 0) + t * kTile
                                              : dn_tile(a, a.E_routed, 0, 0) + (t - gu_tiles) * kTile;
            bulk_prefetch_l2(src, kTile);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Routing reads only the logits.  When they are the caller's inputs (no
    // kernel ahead writes them, as in a stack of layers), warps 0-5 route
    // before griddepcontrol.wait, and the producer issues its first weight
    // tiles before it too (x's codes follow once quantised, after the wait).
    // Everything that writes global memory or reads the previous kernel's
    // output waits first.
    const bool early = a.route_early != 0;
    if (warp < kQuantWarp0) {
        if (!early) pdl_wait();
        route_all<MODE>(a, sm, tid);           // the plan in every CTA's shared memory (warps 0-5)
        named_arrive(3, kThreads - 32);        // ... and for warps 7-11
    } else {
        pdl_wait();
        // (down alone: each piece's epilogue quantises its rows of a itself)
        if (MODE != kMtokDown) quantise_x(a, warp - kQuantWarp0, lane);
        if (warp != kQuantWarp0) named_sync(3, kThreads - 32);
    }
    if (warp == kQuantWarp0) {
        // warp 6 goes on at once to release x's K groups as the grid's
        // quantisation completes (it needs no plan)
        if (MODE != kMtokDown) x_ready(a, sm, lane);
    } else {
        const int U = sm.plan.n_uniq, ncols = U * a.RB, spc = a.GS + a.NU;
        const Share sh =
            share_of(ncols, spc, a.GS,
                     MODE == kMtokDown     ? kShareFree
                     : MODE == kMtokGateUp ? kShareChain
                     : MODE == kMtokDense  ? kShareHelp
                                           : kShareColumns);
        if (warp == kProducerWarp) {
            if (lane == 0) {
                const long long issued = producer<MODE>(a, sm, stages, sh, spc);
                if (sm.abort_flag) producer_drain(sm, issued);
            }
        } else if (warp == kMmaWarp) {
            const long long last = mma_issuer<MODE>(a, sm, stages, sh, spc, lane);
            if (last >= 0) {
                // every MMA issued has completed before TMEM is freed (bounded)
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(&sm.mma_done[last % kTmemBufs], static_cast<uint32_t>((last / kTmemBufs) & 1))) {
                    if (global_timer_ns() - t0 > 100ull * 1000ull * 1000ull) {
                        if (lane == 0) record_error(a.status, MOEQ_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        } else if (warp < kEpiWarp0 + kEpiWarps) {
            if (early) pdl_wait();
            if (a.ntmax <= 4)
                epilogue<4, MODE>(a, sm, sh, spc, warp, lane);
            else if (a.ntmax <= 8)
                epilogue<8, MODE>(a, sm, sh, spc, warp, lane);
            else
                epilogue<16, MODE>(a, sm, sh, spc, warp, lane);
        } else if (warp == kTicketWarp) {
            ticket_warp(a, sm, sh, spc, lane);
        } else {
            sum_worker<MODE>(a, sm, ncols, warp - kSumWarp0, lane);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(sm.tmem_base, kTmemCols);
    // the last CTA out (every other CTA's counting and summing done) clears
    // the counts and flags for the next launch, with all its threads (the
    // next kernel's griddepcontrol.wait waits for this)
    if (tid == 0) {
        __threadfence();
        sm.last_cta = atomicAdd(a.cnt + kMtokFin, 1) == G - 1;
    }
    __syncthreads();
    if (sm.last_cta) {
        __threadfence();
        // (down alone counts no K group of its input)
        const int n_x = MODE == kMtokDown ? 0 : a.KX, n_u = a.NU, n = n_x + n_u + G + 1;
        for (int i = tid; i < n; i += kThreads) {
            const int o = i < n_x ? kMtokX + kMtokPad * i
                                  : (i < n_x + n_u ? kMtokU + kMtokPad * (i - n_x) : kMtokFlags + (i - n_x - n_u));
            a.cnt[o] = 0;
        }
        if (tid == 0) a.cnt[kMtokFin] = 0;
    }
}

}  // namespace

size_t mtok_smem_bytes() { return kSmemBytes; }

// One instantiation per mode: the layer path carries none of the
// standalone modes' branches.
cudaError_t launch_mtok(const MtokArgs& args, int grid, bool pdl, cudaStream_t stream) {
    if (args.mode < kMtokLayer || args.mode > kMtokDense) return cudaErrorInvalidValue;
    void (*const kernels[4])(MtokArgs) = {mtok_kernel<kMtokLayer>, mtok_kernel<kMtokGateUp>, mtok_kernel<kMtokDown>,
                                          mtok_kernel<kMtokDense>};
    static int configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 64 && !configured[dev]) {
        for (auto k : kernels) {
            const cudaError_t e =
                cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
            if (e != cudaSuccess) return e;
        }
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
    return cudaLaunchKernelEx(&cfg, kernels[args.mode], args);
}

}  // namespace moeq
