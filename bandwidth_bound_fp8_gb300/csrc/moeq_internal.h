// Host-side declarations shared by the libmoeq translation units.  The C ABI
// (include/moeq.h) validates arguments and then calls these launchers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moeq.h"

namespace moeq {

constexpr int kMaxTokens = MOEQ_MAX_TOKENS;
constexpr int kMmaMinTokens = 8;  // launches with this many tokens per expert (or more) run the tcgen05 path
constexpr int kMaxLists = 6;
constexpr int kKindGU = 0;  // gate_up: a stage holds the gate tile and the up tile of one K group
constexpr int kKindDN = 1;  // down: a stage holds two consecutive K tiles of one row block
constexpr int kKindDC = 2;  // down by K group (one token): a stage holds two row blocks' tiles of one K group
// Down by K group needs the combine's per-pair sums of one CTA's output
// columns in one activation slot: max_pairs * ceil(H / grid) floats at most.
constexpr int kDcCombineFloats = 6144;
constexpr int kSrcShared = 0;      // the layer's shared expert alone, known before routing
constexpr int kSrcPlanAll = 1;     // every unique expert of the caller's plan (standalone calls)
constexpr int kSrcLayer = 2;       // the layer: its shared expert first, then the plan's routed experts
constexpr int kSrcPlanRoutedA = 3; // the first half of the plan's routed experts
constexpr int kSrcPlanRoutedB = 4; // the second half (down of half A hides the finish of half B's h)

// One GEMM operand set.  Weights are tile-major: tile (e, nb, kb) -- the
// 128 x 128 block of rows nb*128.. and columns kb*128.. of expert e -- is 16
// KiB at w + ((e * NB + nb) * KB + kb) * 16384, rows of 128 bytes, the 16-byte
// chunk c of row r stored at chunk c ^ (r % 8).
struct Operand {
    const uint8_t* w;
    const float* sw;      // [E, NB, KB]
    int K, KB, NB, RB;    // RB = output row blocks per expert (I/128 for gate_up, N/128 for down)
    const void* a;        // activations [rows_a, K], bf16 or fp32 (gate_up: token rows; down: pair rows)
    int a_f32;
    int rows_a;
    float* out;           // [max_pairs, out_ld]
    int out_ld;
    uint8_t* qdump;       // optional [rows_a, K]
    float* sdump;         // optional [rows_a, K/128]
    float* aq;            // workspace: decoded activation codes [rows_a, K] in the consumer layout, or
                          // (tcgen05 path) E4M3 codes [8][rows_a, K]: phase p holds each 128-byte
                          // group with its 16-byte chunk c at chunk c ^ p
    float* as;            // workspace: activation scales [rows_a, K/128]
    int quant_input;      // 1: the kernel's first phase quantises `a` into aq/as
};

struct StreamArgs {
    Operand op[2];
    int n_lists;
    int list_kind[kMaxLists];
    int list_src[kMaxLists];
    // plan (device)
    const int32_t* n_uniq;
    const int32_t* uniq;
    const int32_t* offs;
    const int32_t* pair_tok;
    const int32_t* pair_of;
    const float* topk_w;
    int n_experts, max_uniq, max_pairs;
    // the layer's shared expert (id, first pair, token count)
    int shared_id, shared_p0, M;
    int max_ntok;             // largest token (pair) count of one expert: 1 .. kMaxTokens
    // layer fusion
    int fused_route;          // every CTA computes the plan into shared memory; CTA 0 writes `plan`
    const float* logits;
    int E_routed, top_k;
    moeq_route_plan plan;     // writable plan (fused route)
    int fused_combine;        // the down epilogue also writes out_bf16
    __nv_bfloat16* out_bf16;
    // workspace
    int* status;
    int* epoch;
    int* done;
    int* a_cnt;               // CTAs done with the input quantisation phase (epoch * grid when all are)
    int h_to_dn;              // layer: the gate_up finish also quantises h into op[down].aq/as
    uint8_t* qh_dump;         // layer, optional: h's codes [max_pairs, I] ...
    float* sh_dump;           // ... and scales [max_pairs, I/128]
    int mma;                  // 1: tcgen05 path (activation codes kept as E4M3 bytes in aq)
    int* tickets[kMaxLists];
    float* partials;          // per list: 2 * grid slots of kMaxTokens * 256 floats
    size_t partial_list_floats;
    int* h_ready;             // [max_uniq, RB of gate_up]: epoch of the last write of h
    int* comb;                // [M, RB of down]
    // down by K group (layer, one token, CUDA cores): the CTA that finished
    // h's row block kb of a pair streams down's tiles (nb, kb) for every nb
    // and leaves fp32 sums per (pair, kb, output column); after every CTA
    // has counted itself in dc_cnt, each CTA combines a slice of columns.
    int dc;
    float* dc_part;           // [max_pairs, K groups of down, H]
    int* dc_cnt;              // every launch adds one per CTA (epoch * grid once all have)
    // one token, whole blocks, one gate_up block per CTA: each CTA quantises
    // all of x itself into its first activation slot (xloc), and hands the
    // h group it finishes to its own down by K group in shared memory (hloc)
    int xloc, hloc;
    // with xloc: the CTA's first stage also brings its gate_up chunk's two
    // rows of weight scales (bulk copies, 16-byte aligned rows)
    int swb;
};

// Whole row blocks per CTA for n_rb blocks on G CTAs, or 0 for stream-K: the
// engine's rule (whole blocks when the CTAs that get some are >= 90 % of G).
inline int dp_blocks_per_cta_host(long long n_rb, long long G) {
    if (n_rb <= 0) return 0;
    const long long per = (n_rb + G - 1) / G, used = (n_rb + per - 1) / per;
    return used * 10 >= G * 9 ? static_cast<int>(per) : 0;
}
// x fits one activation slot (decoded fp32 codes of one token)
constexpr int kXLocalMaxK = 6144;

// The one-token layer kernel (moeq_token.cu): x fits its shared memory, the
// routed picks plus the shared expert fit its per-slot sums.
constexpr int kTokenMaxH = 6144;
constexpr int kTokenMaxTopK = 8;

struct TokenArgs {
    const __nv_bfloat16* x;      // [H]
    const float* logits;         // [E_routed]
    int H, I, KB, RB;            // KB = H/128 (gate_up K groups, down row blocks), RB = I/128
    int E_routed, top_k;
    int ncols;                   // (top_k + 1) * RB columns (expert slot, down K group)
    const uint8_t* w_gu;         // tile-major [E_routed + 1, 2I, H]
    const float* s_gu;           // [E_routed + 1, 2I/128, H/128]
    const uint8_t* w_d;          // tile-major [E_routed + 1, H, I]
    const float* s_d;            // [E_routed + 1, H/128, I/128]
    __nv_bfloat16* out;          // [H]
    float* out_f32;              // or, when set, [H] fp32: the unrounded sum (a tensor-parallel shard's partial)
    moeq_route_plan plan;        // written by CTA 0
    float* h;                    // [top_k + 1, I]
    uint8_t* q_x;                // optional [H] and [H/128]: x's codes and scales
    float* s_x;
    uint8_t* q_h;                // optional [top_k + 1, I] and [top_k + 1, I/128]: h's codes and scales
    float* s_h;
    int* status;
    int* tickets;                // [H/256] arrivals per output unit, zero between launches
    int* gq;                     // kGqUnits ints, zero between launches
    float* part;                 // [H/256][16][ncols][16] down partials
    int route_early;             // 1: the logits are not written by the kernel ahead on the stream,
                                 // so the token is routed (and its first column started) before
                                 // griddepcontrol.wait
};
// Completion state of the one-token kernel (ints): CTAs finished.
constexpr int kGqCtas = 0, kGqUnits = 4;

cudaError_t launch_token(const TokenArgs& args, int grid, bool pdl, cudaStream_t stream);

// The multi-token layer kernel (moeq_mtok.cu): 1..16 tokens on the tcgen05
// tensor cores, H a multiple of 256 up to kTokenMaxH, top_k up to 16.  Its
// modes: the layer (routing; top_k = 0: a dense FFN), gate_up + SwiGLU
// alone, and down alone, the last two over a caller's plan.
constexpr int kMtokLayer = 0, kMtokGateUp = 1, kMtokDown = 2, kMtokDense = 3;   // kMtokDense: the layer with
                                                                             // no routing (top_k = 0)
struct MtokArgs {
    const void* x;               // [M, x_ld] bf16 (or fp32 with x_f32): the layer's x, gate_up's x, down's a
    const float* logits;         // [M, E_routed]
    int M, H, I, KB, RB;         // layer and gate_up: KB = H/128, RB = I/128; down: M pair rows, H = N,
                                 // KB = N/128 row blocks, RB = K/128 K groups, I = K
    int mode;                    // kMtokLayer, kMtokGateUp, kMtokDown or kMtokDense
    int GS, NU;                  // per column: gate_up stages (KB or 0) and down units of 256 rows (KB/2 or 0)
    int KX, x_ld, x_f32;         // the quantised input's K groups, row length and type
    int ntmax;                   // most rows (tokens or pairs) one column serves: 1..16
    int n_experts, max_uniq, max_pairs;   // gate_up or down alone: the bounds the caller's plan is checked against
    int E_routed, top_k;
    const uint8_t* w_gu;         // tile-major [E_routed + 1, 2I, H]
    const float* s_gu;           // [E_routed + 1, 2I/128, H/128]
    const uint8_t* w_d;          // tile-major [E_routed + 1, H, I]
    const float* s_d;            // [E_routed + 1, H/128, I/128]
    __nv_bfloat16* out;          // [M, H]
    float* out_f32;              // or, when set, [M, H] fp32: the unrounded sums (a tensor-parallel shard's partial)
    moeq_route_plan plan;        // the layer: written by CTA 0; gate_up or down alone: the caller's, read
    float* h;                    // [max_pairs, I], or null: not written (the layer's h dump)
    uint8_t* q_x;                // optional [M, H] and [M, H/128]: x's codes and scales
    float* s_x;
    uint8_t* q_h;                // optional [max_pairs, I] and [max_pairs, I/128]: h's codes and scales
    float* s_h;
    int* status;
    int* cnt;                    // kMtokFlags + grid + 1 ints, zero between launches
    uint8_t* slots;              // [grid + 1][kMtokSlotBytes]: what a split column's head publishes
    uint8_t* xq;                 // [KX][16 * 128]: x's codes, token n in row n (gate_up's B operand;
    float* xs;                   // [KX][16]: x's scales                          unused by down alone)
    float* part;                 // [M][H/256][top_k + 1][RB][256] down partials (down alone: M pair rows,
                                 // H = N, top_k = 0, RB = K/128)
    int route_early;             // 1: the logits are not written by the kernel ahead on the stream, so
                                 // the tokens are routed (and the first weight tiles issued) before
                                 // griddepcontrol.wait
};
// counts (ints): CTAs done, quantised groups per K group of x, down partials
// stored per 256-row output unit, and the split columns' flags (one per CTA
// boundary).  The counts that every CTA polls sit one per 128-byte line
// (stride kMtokPad ints), so that the polls spread over L2.
constexpr int kMtokPad = 32;
constexpr int kMtokFin = 0, kMtokX = kMtokPad, kMtokU = kMtokX + kMtokPad * (kTokenMaxH / 128),
              kMtokFlags = kMtokU + kMtokPad * (kTokenMaxH / 256);
constexpr int kMtokSlotBytes = 18688;
constexpr int kMtokXGroupBytes = 16 * 128;   // one K group of x's codes for up to 16 tokens
constexpr int kMtokMaxTopK = 16;

cudaError_t launch_mtok(const MtokArgs& args, int grid, bool pdl, cudaStream_t stream);

// Tensor-parallel combine (moeq_tp.cu): out = bf16(sum over r in order of part[r]).
cudaError_t launch_tp_reduce(const float* part, int R, int M, int H, void* out, cudaStream_t stream);

size_t stream_partials_floats(int grid);
cudaError_t launch_stream(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream);
cudaError_t launch_stream_mma(const StreamArgs& args, int grid, bool cooperative, cudaStream_t stream);

cudaError_t launch_quant_act(const void* x, int x_f32, int M, int K, uint8_t* q, float* s,
                             cudaStream_t stream);
cudaError_t launch_quant_weight(const float* w, int E, int N, int K, uint8_t* q, float* s,
                                cudaStream_t stream);
cudaError_t launch_pack_weight(const uint8_t* q_rows, int E, int N, int K, uint8_t* q_tiles,
                               cudaStream_t stream);
cudaError_t launch_route(const float* logits, int M, int E, int k, const moeq_route_plan& plan,
                         cudaStream_t stream);
cudaError_t launch_combine(const float* y, int N, const moeq_route_plan& plan, int M, int k,
                           void* out, cudaStream_t stream);

}  // namespace moeq
