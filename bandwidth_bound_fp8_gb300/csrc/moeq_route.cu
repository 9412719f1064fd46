// Routing (top-k + softmax over the picks + expert deduplication) and the
// routing-weighted combine.  GLM-5.2 x10, bandwidth model: each token
// activates its top-8 experts; §5-§6: tokens verified in one pass share one
// read of each expert's weights, so the plan lists every expert once with
// all the tokens that use it.
#include <float.h>

#include "moeq_device.cuh"
#include "moeq_internal.h"

namespace moeq {

constexpr int kRouteThreads = 512;  // one warp per token, MOEQ_MAX_TOKENS warps
constexpr int kMaxE = MOEQ_MAX_EXPERTS;
constexpr int kMaxK = MOEQ_MAX_TOPK;

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ logits, int M, int E,
                                                              int k, moeq_route_plan plan) {
    __shared__ int s_id[kMaxTokens][kMaxK];
    __shared__ float s_lv[kMaxTokens][kMaxK];
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_poff[kMaxE];
    __shared__ int s_total[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;

    // ---- top-k per token: k rounds of a warp arg-max, ties to the lower id.
    if (warp < M) {
        const float* l = logits + static_cast<size_t>(warp) * E;
        constexpr int kPer = kMaxE / 32;
        float v[kPer];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? l[e] : -FLT_MAX;
        }
        for (int j = 0; j < k; ++j) {
            float bv = -FLT_MAX;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == 0) {
                s_id[warp][j] = be;
                s_lv[warp][j] = bv;
            }
            __syncwarp();
        }
        // softmax over the k picks, relative to the largest (the first pick)
        float ex = 0.0f;
        if (lane < k) ex = expf(s_lv[warp][lane] - s_lv[warp][0]);
        float den = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (lane < k) {
            plan.topk_id[warp * k + lane] = s_id[warp][lane];
            plan.topk_w[warp * k + lane] = __fdiv_rn(ex, den);
        }
    }
    __syncthreads();

    // ---- per-expert token counts
    for (int i = tid; i < M * k; i += blockDim.x) atomicAdd(&s_cnt[s_id[i / k][i % k]], 1);
    __syncthreads();

    // ---- exclusive scans over experts (one warp; each lane owns a run of experts)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int used = 0, pairs = 0;
        for (int e = e0; e < min(E, e0 + per); ++e) {
            used += s_cnt[e] > 0;
            pairs += s_cnt[e];
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
        int u = used_x - used, p = pairs_x - pairs;  // exclusive
        for (int e = e0; e < min(E, e0 + per); ++e) {
            s_poff[e] = p;
            if (s_cnt[e] > 0) {
                plan.uniq[u] = e;
                plan.offs[u] = p;
                ++u;
            }
            p += s_cnt[e];
        }
        if (lane == 31) {
            s_total[0] = used_x;   // unique routed experts
            s_total[1] = pairs_x;  // routed pairs = M * k
        }
    }
    __syncthreads();

    // ---- pairs: tokens ascending within each expert
    for (int i = tid; i < M * k; i += blockDim.x) {
        const int m = i / k, j = i % k, e = s_id[m][j];
        int rank = 0;
        for (int m2 = 0; m2 < m; ++m2)
            for (int j2 = 0; j2 < k; ++j2) rank += s_id[m2][j2] == e;
        const int p = s_poff[e] + rank;
        plan.pair_tok[p] = m;
        plan.pair_of[m * (k + 1) + j] = p;
    }
    // ---- the shared expert, id E, serves every token and comes last
    const int U = s_total[0], P = s_total[1];
    for (int m = tid; m < M; m += blockDim.x) {
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

cudaError_t launch_route(const float* logits, int M, int E, int k, const moeq_route_plan& plan,
                         cudaStream_t stream) {
    route_kernel<<<1, kRouteThreads, 0, stream>>>(logits, M, E, k, plan);
    return cudaGetLastError();
}

// out[m, n] = bf16(y[shared] + sum_j w_j * y[pair_j]) in slot order.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, int N, moeq_route_plan plan,
                                                      int k, __nv_bfloat16* __restrict__ out) {
    const int m = blockIdx.y;
    const int n = blockIdx.x * 256 + threadIdx.x;
    if (n >= N) return;
    const int* po = plan.pair_of + m * (k + 1);
    float acc = y[static_cast<size_t>(po[k]) * N + n];
    for (int j = 0; j < k; ++j) acc = fmaf(plan.topk_w[m * k + j], y[static_cast<size_t>(po[j]) * N + n], acc);
    out[static_cast<size_t>(m) * N + n] = __float2bfloat16_rn(acc);
}

cudaError_t launch_combine(const float* y, int N, const moeq_route_plan& plan, int M, int k, void* out,
                           cudaStream_t stream) {
    dim3 grid((N + 255) / 256, M);
    combine_kernel<<<grid, 256, 0, stream>>>(y, N, plan, k, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
}

}  // namespace moeq
