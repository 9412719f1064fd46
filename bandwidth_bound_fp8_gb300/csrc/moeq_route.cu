// Routing (top-k + softmax over the picks + expert deduplication) and the
// routing-weighted combine.  GLM-5.2 x10, bandwidth model: each token
// activates its top-8 experts; §5-§6: tokens verified in one pass share one
// read of each expert's weights, so the plan lists every expert once with
// all the tokens that use it.
#include "moeq_device.cuh"
#include "moeq_internal.h"
#include "moeq_route.cuh"

namespace moeq {

constexpr int kRouteThreads = 512;  // 16 warps: one per token at M = 16

struct BlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ logits, int M, int E,
                                                              int k, moeq_route_plan plan) {
    __shared__ RouteScratch scratch;
    route_compute<kRouteThreads>(logits, M, E, k, plan, scratch, threadIdx.x, BlockSync{});
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
