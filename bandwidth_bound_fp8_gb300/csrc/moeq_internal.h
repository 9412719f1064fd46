// Host-side declarations shared by the libmoeq translation units.  The C ABI
// (include/moeq.h) validates arguments and then calls these launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moeq.h"

namespace moeq {

// Geometry of one expert-GEMM launch (gate_up or down).
struct GemmArgs {
    const void* a;              // activations [rows_a, K] bf16 or fp32
    int a_f32;                  // 1: fp32, 0: bf16
    const int32_t* a_row;       // row of `a` used by pair p; nullptr = p itself
    int K;                      // reduction length (multiple of 128)
    int rows_per_expert;        // rows of one expert's weight matrix (2I or N)
    int up_offset;              // gate_up: row offset of the up half (I); down: 0
    int RB;                     // 128-row output blocks per expert (I/128 or N/128)
    const float* sw;            // weight scales [E, rows_per_expert/128, K/128]
    const int32_t* uniq;        // plan
    const int32_t* offs;
    const int32_t* n_uniq;
    float* out;                 // [max_pairs, out_ld]
    int out_ld;
    uint8_t* qdump;             // optional [rows_a, K]
    float* sdump;               // optional [rows_a, K/128]
    int* tickets;               // [max_uniq * RB], zero between launches
    float* partials;            // [2 * grid, kMaxTok, rows per unit]
    int* status;                // device status word
    int n_experts;              // experts in the weight tensor (plan ids must be below)
    int max_uniq;               // plan capacity: U read on the device is clamped to it
    int max_pairs;              // rows of `out`
    int rows_a;                 // rows of `a`
};

constexpr int kMaxTokens = MOEQ_MAX_TOKENS;

// Expert GEMM with fused activation quantisation.  nbox = 2: gate_up with
// SwiGLU epilogue; nbox = 1: plain output.
cudaError_t launch_expert_gemm(const CUtensorMap& map, const GemmArgs& args, int nbox, int grid,
                               cudaStream_t stream);
size_t gemm_partials_floats(int nbox, int grid);

cudaError_t launch_quant_act(const void* x, int x_f32, int M, int K, uint8_t* q, float* s,
                             cudaStream_t stream);
cudaError_t launch_quant_weight(const float* w, int E, int N, int K, uint8_t* q, float* s,
                                cudaStream_t stream);
cudaError_t launch_route(const float* logits, int M, int E, int k, const moeq_route_plan& plan,
                         cudaStream_t stream);
cudaError_t launch_combine(const float* y, int N, const moeq_route_plan& plan, int M, int k,
                           void* out, cudaStream_t stream);

}  // namespace moeq
