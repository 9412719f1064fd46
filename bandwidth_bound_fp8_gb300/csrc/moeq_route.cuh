// Routing plan computation shared by the standalone route kernel and the
// fused layer kernel (where one CTA computes it while the others already
// stream the shared expert).  GLM-5.2 x10, bandwidth model: every token
// activates its top-8 experts; §5-§6: tokens verified in one pass share one
// read of each expert, so the plan lists each expert once with its tokens.
//
// Definition (the page fixes none of it; this library's reading):
//   topk_id[m, j]: the j-th largest logit of token m, ties to the lower id;
//   topk_w[m, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k picks;
//   uniq: routed experts in ascending id, then the shared expert (id E);
//   offs/pair_tok: the pairs of each unique expert, tokens ascending;
//   pair_of[m, j]: the pair of (token m, slot j), slot k = shared.
#pragma once

#include <float.h>

#include "moeq_device.cuh"

namespace moeq {

constexpr int kRouteMaxE = MOEQ_MAX_EXPERTS;
constexpr int kRouteMaxK = MOEQ_MAX_TOPK;

struct RouteScratch {
    int id[MOEQ_MAX_TOKENS][kRouteMaxK];
    float lv[MOEQ_MAX_TOKENS][kRouteMaxK];
    int cnt[kRouteMaxE];
    int poff[kRouteMaxE];
    int total[2];
};

// Order-preserving map of a float to an unsigned key (-0 folded onto +0, so
// that equal values tie exactly as they compare).
__device__ __forceinline__ uint32_t route_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float route_key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of one token's logits by one warp: lane l holds experts l, l+32, ...;
// each round takes the warp maximum of the key, then the smallest expert id
// holding it (ties to the lower id), with two warp reductions.
template <int NPER>
__device__ __forceinline__ void route_load_keys(const float* __restrict__ l, int E, int lane, uint32_t (&key)[NPER]) {
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? route_key(__ldcg(l + e)) : 0u;
    }
}

// The selection itself, on keys already loaded by route_load_keys.
template <int NPER>
__device__ __forceinline__ void route_topk_keys(const uint32_t (&key)[NPER], int E, int k, int lane, int* ids,
                                                float* vals) {
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const bool ok = (lane + 32 * i < E) && !((taken >> i) & 1u);
            if (ok && (bi < 0 || key[i] > bk)) {
                bk = key[i];
                bi = i;
            }
        }
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const int cand = (bi >= 0 && bk == wk) ? lane + 32 * bi : 0x7fffffff;
        const int we = __reduce_min_sync(0xffffffffu, cand);
        if ((we & 31) == lane) taken |= 1u << (we >> 5);
        if (lane == 0) {
            ids[j] = we;
            vals[j] = route_key_value(wk);
        }
    }
    __syncwarp();
}

template <int NPER>
__device__ __forceinline__ void route_topk_warp(const float* __restrict__ l, int E, int k, int lane, int* ids,
                                                float* vals) {
    uint32_t key[NPER];
    route_load_keys<NPER>(l, E, lane, key);
    route_topk_keys<NPER>(key, E, k, lane, ids, vals);
}

// The plan of ONE token by one warp, with no block barrier: top-k as
// above, the softmax over the picks (the same butterfly and division as
// route_compute, so the same bits), the picks ascending as the unique list
// (one pair each, in that order) and the shared expert last.  `ids`/`vals`
// are k-entry scratch (the warp's own).
template <int NPER>
__device__ __forceinline__ void route_one_token_warp(const float* __restrict__ l, int E, int k, int lane,
                                                     const moeq_route_plan& plan, int* ids, float* vals) {
    route_topk_warp<NPER>(l, E, k, lane, ids, vals);
    float ex = 0.0f;
    int id = 0x7fffffff;
    if (lane < k) {
        ex = expf(vals[lane] - vals[0]);
        id = ids[lane];
    }
    float den = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += __shfl_sync(0xffffffffu, id, i) < id;
    if (lane < k) {
        plan.topk_id[lane] = id;
        plan.topk_w[lane] = __fdiv_rn(ex, den);
        plan.uniq[rank] = id;
        plan.offs[lane] = lane;
        plan.pair_tok[lane] = 0;
        plan.pair_of[lane] = rank;
    }
    if (lane == 0) {
        plan.uniq[k] = E;
        plan.offs[k] = k;
        plan.offs[k + 1] = k + 1;
        plan.pair_tok[k] = 0;
        plan.pair_of[k] = k;
        *plan.n_uniq = k + 1;
    }
    __syncwarp();
}

// Computes the plan with NT threads (tid in [0, NT)); `sync` is a barrier
// over exactly those threads.  Writes every plan member to global memory;
// the caller makes the writes visible (fence + flag) as it needs.
template <int NT, typename Sync>
__device__ __forceinline__ void route_compute(const float* __restrict__ logits, int M, int E, int k,
                                              const moeq_route_plan& plan, RouteScratch& s, int tid, Sync sync) {
    constexpr int kWarps = NT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += NT) s.cnt[e] = 0;

    for (int m = warp; m < M; m += kWarps) {
        const float* l = logits + static_cast<size_t>(m) * E;
        if (E <= 256)
            route_topk_warp<8>(l, E, k, lane, s.id[m], s.lv[m]);
        else
            route_topk_warp<kRouteMaxE / 32>(l, E, k, lane, s.id[m], s.lv[m]);
        float ex = 0.0f;
        if (lane < k) ex = expf(s.lv[m][lane] - s.lv[m][0]);
        float den = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane < k) {
            plan.topk_id[m * k + lane] = s.id[m][lane];
            plan.topk_w[m * k + lane] = __fdiv_rn(ex, den);
        }
    }
    sync();
    for (int i = tid; i < M * k; i += NT) atomicAdd(&s.cnt[s.id[i / k][i % k]], 1);
    sync();
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int used = 0, pairs = 0;
        for (int e = e0; e < min(E, e0 + per); ++e) {
            used += s.cnt[e] > 0;
            pairs += s.cnt[e];
        }
        int used_x = used, pairs_x = pairs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, used_x, o);
            const int b = __shfl_up_sync(0xffffffffu, pairs_x, o);
            if (lane >= o) {
                used_x += a;
                pairs_x += b;
            }
        }
        int u = used_x - used, p = pairs_x - pairs;
        for (int e = e0; e < min(E, e0 + per); ++e) {
            s.poff[e] = p;
            if (s.cnt[e] > 0) {
                plan.uniq[u] = e;
                plan.offs[u] = p;
                ++u;
            }
            p += s.cnt[e];
        }
        if (lane == 31) {
            s.total[0] = used_x;
            s.total[1] = pairs_x;
        }
    }
    sync();
    for (int i = tid; i < M * k; i += NT) {
        const int m = i / k, j = i % k, e = s.id[m][j];
        int rank = 0;
        for (int m2 = 0; m2 < m; ++m2)
            for (int j2 = 0; j2 < k; ++j2) rank += s.id[m2][j2] == e;
        const int p = s.poff[e] + rank;
        plan.pair_tok[p] = m;
        plan.pair_of[m * (k + 1) + j] = p;
    }
    const int U = s.total[0], P = s.total[1];
    for (int m = tid; m < M; m += NT) {
        plan.pair_tok[P + m] = m;
        plan.pair_of[m * (k + 1) + k] = P + m;
    }
    if (tid == 0) {
        plan.uniq[U] = E;
        plan.offs[U] = P;
        plan.offs[U + 1] = P + M;
        *plan.n_uniq = U + 1;
    }
}

}  // namespace moeq
