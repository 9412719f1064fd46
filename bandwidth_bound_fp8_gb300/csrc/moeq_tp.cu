// Tensor-parallel combine: the rank-order sum of R shards' fp32 partial
// outputs, rounded to bf16 (GLM-5.2 x10, bandwidth model: TP8 splits every
// expert over 8 cards, so each card streams 1/8 of the layer's bytes; the
// layer's output is then the sum of the cards' partial outputs).
#include "moeq_device.cuh"
#include "moeq_internal.h"

namespace moeq {
namespace {

// One thread per 4 consecutive outputs: partial r = 0, 1, .. R-1 added in
// that order in fp32, then rounded to bf16.
__global__ void tp_reduce_kernel(const float* __restrict__ part, int R, size_t n, __nv_bfloat16* __restrict__ out) {
    const size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    float4 acc = __ldcg(reinterpret_cast<const float4*>(part + i));
    for (int r = 1; r < R; ++r) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(part + static_cast<size_t>(r) * n + i));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&lo);
    packed.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + i) = packed;
}

}  // namespace

cudaError_t launch_tp_reduce(const float* part, int R, int M, int H, void* out, cudaStream_t stream) {
    const size_t n = static_cast<size_t>(M) * H;   // a multiple of 4 (H % 128 == 0)
    const int threads = 256;
    const unsigned blocks = static_cast<unsigned>((n / 4 + threads - 1) / threads);
    tp_reduce_kernel<<<blocks, threads, 0, stream>>>(part, R, n, static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
}

}  // namespace moeq
