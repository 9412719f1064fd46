// Standalone quantisation kernels: live activation quantisation (the same
// per-group routine the GEMM prologues fuse) and offline 128 x 128 block
// quantisation of expert weights.
#include "moeq_device.cuh"
#include "moeq_internal.h"

namespace moeq {

// One warp per (row, group): 8 warps per block, grid.x covers rows*groups.
template <bool kF32>
__global__ void __launch_bounds__(256) quant_act_kernel(const void* __restrict__ x, int M, int K,
                                                        uint8_t* __restrict__ q, float* __restrict__ s) {
    const int G = K / kGroup;
    const long long item = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (item >= static_cast<long long>(M) * G) return;
    const int lane = threadIdx.x & 31;
    const int row = static_cast<int>(item / G);
    const int g = static_cast<int>(item % G);
    const int k = g * kGroup + lane * 4;
    float4 v = load_act4<kF32>(x, static_cast<size_t>(K), row, k);
    float sc;
    float4 dec;
    const uint32_t codes = quant_group_warp(v, &sc, &dec);
    *reinterpret_cast<uint32_t*>(q + static_cast<size_t>(row) * K + k) = codes;
    if (lane == 0) s[static_cast<size_t>(row) * G + g] = sc;
}

cudaError_t launch_quant_act(const void* x, int x_f32, int M, int K, uint8_t* q, float* s,
                             cudaStream_t stream) {
    const long long items = static_cast<long long>(M) * (K / kGroup);
    const unsigned blocks = static_cast<unsigned>((items + 7) / 8);
    if (x_f32)
        quant_act_kernel<true><<<blocks, 256, 0, stream>>>(x, M, K, q, s);
    else
        quant_act_kernel<false><<<blocks, 256, 0, stream>>>(x, M, K, q, s);
    return cudaGetLastError();
}

// Byte offset of element (r, k) of a tile: rows of 128 bytes, the 16-byte
// chunk k/16 of row r stored at chunk (k/16) ^ (r % 8).
__device__ __forceinline__ int tile_chunk(int r, int chunk) { return r * 128 + ((chunk ^ (r & 7)) << 4); }

// One block of 256 threads per 128 x 128 weight block.  Each thread owns
// half a row (64 consecutive elements): thread t -> row t/2, columns
// (t%2)*64 .. +63.  amax over the block, s = fl32(amax/448), then codes,
// written tile-major (see the layout in moeq_internal.h).
__global__ void __launch_bounds__(256) quant_weight_kernel(const float* __restrict__ w, int N, int K,
                                                           uint8_t* __restrict__ q, float* __restrict__ s) {
    __shared__ float red[8];
    const int kb = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
    const int KB = K / kGroup, NB = N / kGroup;
    const int t = threadIdx.x;
    const int r = t >> 1;
    const int c0 = (t & 1) * 64;
    const size_t base = (static_cast<size_t>(e) * N + static_cast<size_t>(nb) * kGroup + r) * K +
                        static_cast<size_t>(kb) * kGroup + c0;
    const float4* src = reinterpret_cast<const float4*>(w + base);
    float4 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = __ldg(src + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
    amax = warp_max(amax);
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    if (t < 32) {
        float m = t < 8 ? red[t] : 0.0f;
        m = warp_max(m);
        if (t == 0) red[0] = m;
    }
    __syncthreads();
    const float sc = __fdiv_rn(red[0], 448.0f);
    const size_t tile = (static_cast<size_t>(e) * NB + nb) * KB + kb;
    if (t == 0) s[tile] = sc;
    uint32_t out[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (sc == 0.0f) {
            out[i] = (signbit(v[i].x) ? 0x80u : 0u) | (signbit(v[i].y) ? 0x8000u : 0u) |
                     (signbit(v[i].z) ? 0x800000u : 0u) | (signbit(v[i].w) ? 0x80000000u : 0u);
        } else {
            const uint16_t c01 = e4m3x2_from_f32(__fdiv_rn(v[i].x, sc), __fdiv_rn(v[i].y, sc));
            const uint16_t c23 = e4m3x2_from_f32(__fdiv_rn(v[i].z, sc), __fdiv_rn(v[i].w, sc));
            out[i] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
        }
    }
    uint8_t* dst = q + tile * (kGroup * kGroup);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(dst + tile_chunk(r, (c0 >> 4) + i)) =
            make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
}

cudaError_t launch_quant_weight(const float* w, int E, int N, int K, uint8_t* q, float* s,
                                cudaStream_t stream) {
    dim3 grid(K / kGroup, N / kGroup, E);
    quant_weight_kernel<<<grid, 256, 0, stream>>>(w, N, K, q, s);
    return cudaGetLastError();
}

// Row-major codes [E, N, K] -> the tile-major layout (a pure permutation).
__global__ void __launch_bounds__(256) pack_weight_kernel(const uint8_t* __restrict__ src, int N, int K,
                                                          uint8_t* __restrict__ dst) {
    const int kb = blockIdx.x, nb = blockIdx.y, e = blockIdx.z;
    const int KB = K / kGroup, NB = N / kGroup;
    const int t = threadIdx.x, r = t >> 1, c0 = (t & 1) * 64;
    const uint4* in = reinterpret_cast<const uint4*>(
        src + (static_cast<size_t>(e) * N + static_cast<size_t>(nb) * kGroup + r) * K + static_cast<size_t>(kb) * kGroup + c0);
    uint8_t* out = dst + ((static_cast<size_t>(e) * NB + nb) * KB + kb) * (kGroup * kGroup);
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(out + tile_chunk(r, (c0 >> 4) + i)) = __ldg(in + i);
}

cudaError_t launch_pack_weight(const uint8_t* q_rows, int E, int N, int K, uint8_t* q_tiles, cudaStream_t stream) {
    dim3 grid(K / kGroup, N / kGroup, E);
    pack_weight_kernel<<<grid, 256, 0, stream>>>(q_rows, N, K, q_tiles);
    return cudaGetLastError();
}

}  // namespace moeq
