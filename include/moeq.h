/*
 * libmoeq -- FP8 live-quantised MoE expert projection for small decode
 * batches (M = 1..16 tokens: plain decode and multi-token draft
 * verification), written for NVIDIA GB300 (sm_103a).
 *
 * Citations.  "GLM-5.2 x10" is the blog.sionic.ai page titled
 * "GPU 커널부터 새로 짜서 GLM-5.2 속도 10배 올리기"; "§n" is its numbered
 * section.  The page states the problem this library solves -- decode is a
 * stream of FP8 expert weights from HBM with very little arithmetic on top
 * (bandwidth model), the activations are quantised to FP8 live in front of
 * each GEMM (§1, §8c), that quantisation is fused into the GEMM instead of
 * round-tripping through HBM (§4, "PQ-GEMM"), K is split across the SMs so
 * that enough of them stream weights (§1, split-K), and several tokens
 * verified together share one read of each expert (§5-§6) -- but it prints no
 * interface.  The calls below are this library's own statement of it.
 *
 * Numeric contract (the page fixes none of it; these are this library's
 * choices, applied identically by every call):
 *   - FP8 is OCP E4M3FN (bias 7, max 448, no infinities);
 *   - activations are quantised per token in groups of 1 x 128 along K:
 *     s = fl32(amax / 448), q = RNE_satfinite(fl32(x / s)); a group whose
 *     s is 0 gets signed-zero codes;
 *   - weights carry one fp32 scale per 128 x 128 block;
 *   - weight codes are stored TILE-MAJOR (the HBM layout every GEMM call
 *     streams): the 128 x 128 block (nb, kb) of expert e -- rows nb*128..,
 *     columns kb*128.. of its [N, K] matrix -- is one contiguous 16 KiB tile
 *     at byte offset ((e * N/128 + nb) * K/128 + kb) * 16384; inside a tile
 *     row r occupies bytes r*128 .. r*128+127 and its 16-byte chunk c (columns
 *     16c .. 16c+15) sits at chunk position c ^ (r % 8).  Each tile is then
 *     one sequential 16 KiB read, and the chunk rotation keeps shared-memory
 *     reads conflict-free.  moeq_quant_weight writes this layout and
 *     moeq_pack_weight converts row-major codes to it; scales stay row-major
 *     [E, N/128, K/128];
 *   - GEMMs accumulate in fp32: y = sum_g s_a * s_w * sum_{k in g} q_a * q_w.
 *
 * Conventions for every call:
 *   - tensor pointers are DEVICE pointers owned by the caller, row-major,
 *     16-byte aligned (fp32 scale arrays and routing arrays: 4-byte);
 *     `stream` is a cudaStream_t passed as void*;
 *   - calls are asynchronous on `stream` and never synchronise the host
 *     (except moeq_read_device_status, which says so);
 *   - the library makes no device allocation at run time: the caller
 *     passes a workspace sized by moeq_workspace_size /
 *     moeq_gemm_workspace_size, zeroed once with moeq_workspace_init; kernels
 *     leave it reusable; one workspace must not be used by two calls that may
 *     run concurrently.  The one exception, moeq_expert_gemm_down_noalloc,
 *     uses a fixed 8 MiB static device array that the library holds on every
 *     device it is loaded on;
 *   - arguments are validated on the host first; on any error nothing is
 *     launched and the status says why;
 *   - inputs must be finite (NaN/Inf inputs give unspecified results).
 */
#ifndef MOEQ_H
#define MOEQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moeq_status {
    MOEQ_OK = 0,
    MOEQ_ERR_INVALID_ARG = 1,       /* null pointer, misaligned pointer, bad enum, M out of range */
    MOEQ_ERR_UNSUPPORTED_SHAPE = 2, /* K, N, H or I not a multiple of 128, or above the limits */
    MOEQ_ERR_WORKSPACE = 3,         /* workspace null or smaller than required */
    MOEQ_ERR_CUDA = 4,              /* a CUDA runtime call failed (launch, attribute, memset) */
    MOEQ_ERR_TIMEOUT = 5,           /* a bounded device-side wait gave up (device status word) */
    MOEQ_ERR_DEVICE = 6             /* no CUDA device, or not a compute capability 10.3 part */
} moeq_status;

typedef enum moeq_dtype { MOEQ_BF16 = 0, MOEQ_F32 = 1 } moeq_dtype;

#define MOEQ_GROUP 128          /* quantisation group along K, and weight block edge */
#define MOEQ_MAX_TOKENS 16      /* M limit: decode plus draft verification */
#define MOEQ_MAX_EXPERTS 1024   /* routed experts limit of moeq_route */
#define MOEQ_MAX_TOPK 16
#define MOEQ_MAX_K 32768        /* K (H or I) limit of the GEMM calls */
#define MOEQ_MAX_LAYERS 256     /* L limit of moeq_moe_stack */
#define MOEQ_STACK_EAGER 1      /* moeq_moe_stack flag: launch the layers directly, no graph */

/* Human-readable text of a status (static storage, never NULL). */
const char* moeq_status_string(moeq_status s);

/* ABI version, bumped whenever a signature or struct below changes. */
int moeq_abi_version(void);

/* ------------------------------------------------------------------------ */
/* Routing plan (GLM-5.2 x10, bandwidth model: top-8 experts per token;     */
/* §5-§6: tokens verified together share one weight read, so experts are    */
/* deduplicated).  All members point to caller-owned device memory.         */
/*   topk_id [M, top_k]   j-th largest logit of token m, ties -> lower id   */
/*   topk_w  [M, top_k]   softmax over the top_k picked logits              */
/*   n_uniq  [1]          U = unique routed experts + 1 (the shared one)    */
/*   uniq    [max_uniq]   routed expert ids ascending, then E_routed        */
/*                        (the shared expert's id) last                     */
/*   offs    [max_uniq+1] pairs of unique expert u are offs[u]..offs[u+1]-1 */
/*   pair_tok[max_pairs]  token of each (token, expert) pair, ascending     */
/*                        within an expert                                  */
/*   pair_of [M, top_k+1] pair of (token m, slot j); slot top_k = shared    */
/* ------------------------------------------------------------------------ */
typedef struct moeq_route_plan {
    int32_t* topk_id;
    float* topk_w;
    int32_t* n_uniq;
    int32_t* uniq;
    int32_t* offs;
    int32_t* pair_tok;
    int32_t* pair_of;
} moeq_route_plan;

/* min(E_routed, M * top_k) + 1: the most unique experts a plan can hold. */
int moeq_max_uniq(int M, int E_routed, int top_k);
/* M * top_k + M: (token, expert) pairs including the shared expert. */
int moeq_max_pairs(int M, int top_k);
/* Bytes of one device buffer that moeq_route_plan_carve splits into a plan. */
size_t moeq_route_plan_bytes(int M, int E_routed, int top_k);
/* Point the members of *plan into `base` (device memory of at least
 * moeq_route_plan_bytes bytes, 16-byte aligned).  Host-only, no launch. */
moeq_status moeq_route_plan_carve(void* base, size_t bytes, int M, int E_routed, int top_k,
                                  moeq_route_plan* plan);

/* ------------------------------------------------------------------------ */
/* Workspace.                                                               */
/* ------------------------------------------------------------------------ */
/* Bytes needed by moeq_moe_layer for M tokens, hidden H, expert
 * intermediate I, n_experts_incl_shared = E_routed + 1, top_k.  Depends on
 * the current device's SM count; returns 0 on invalid arguments or when no
 * device is present.  At M == 1 it includes the fp32 sums of down by K group
 * (max_pairs * I/128 * H floats: 3.5 MB for H 6144, I 2048, top-8). */
size_t moeq_workspace_size(int M, int H, int I, int n_experts_incl_shared, int top_k);
/* Bytes needed by one standalone GEMM call.  gate_up (is_gate_up = 1):
 * rows_out = I, K = H, rows_in = M; down (is_gate_up = 0): rows_out = N,
 * K = K, rows_in = max_pairs.  max_uniq as for the plan the call is given.
 * Depends on the current device's SM count; 0 on invalid arguments. */
size_t moeq_gemm_workspace_size(int rows_out, int K, int rows_in, int max_uniq, int is_gate_up);
/* Diagnostics for failure-injection tests: the byte offset, inside a       */
/* moeq_moe_layer workspace, of one int count that the multi-token kernel   */
/* waits on (which = 0: the quantised groups of x's K group 0; 1: the down  */
/* partials stored for output unit 0), or 0 when the call's shape does not  */
/* run that kernel.  A count set out of reach makes the kernel's bounded    */
/* wait run out (MOEQ_ERR_TIMEOUT); re-initialise the workspace after.      */
size_t moeq_layer_ws_count_offset(int M, int H, int I, int n_experts_incl_shared, int top_k, int which);
/* The same for a standalone GEMM call's workspace (the arguments of        */
/* moeq_gemm_workspace_size): the offset of the count of x's K group 0      */
/* (which = 0, gate_up only) or of output unit 0 (which = 1, down only),    */
/* or 0 when the call's shape does not run the multi-token kernel.          */
size_t moeq_gemm_ws_count_offset(int rows_out, int K, int rows_in, int max_uniq, int is_gate_up, int which);
/* Zero the workspace (split-K tickets and the device status word) on
 * `stream`.  Needed once after allocation; kernels leave it zeroed.  After a
 * launch that recorded an error (e.g. a bounded wait that gave up, which
 * ends the kernel early) the workspace state is undefined: zero it again. */
moeq_status moeq_workspace_init(void* ws, size_t ws_bytes, void* stream);
/* SYNCHRONOUS: copy the device status word (0 or a moeq_status that a
 * kernel recorded, e.g. MOEQ_ERR_TIMEOUT) to *device_status.  Waits for the
 * work already queued on the current device. */
moeq_status moeq_read_device_status(const void* ws, size_t ws_bytes, int* device_status);

/* ------------------------------------------------------------------------ */
/* moeq_quant_act -- live activation quantisation (GLM-5.2 x10 §1, §8c).   */
/* x [M, K] (bf16 or fp32) -> q [M, K] E4M3 codes, s [M, K/128] fp32.       */
/* Standalone form of the prologue that the GEMM calls fuse.                */
/* M in [1, 4096], K a multiple of 128 up to MOEQ_MAX_K.                    */
/* ------------------------------------------------------------------------ */
moeq_status moeq_quant_act(const void* x, moeq_dtype x_dtype, int M, int K,
                           uint8_t* q, float* s, void* stream);

/* moeq_quant_weight -- offline block quantisation of E expert matrices.    */
/* w [E, N, K] fp32 row-major -> q: E*N*K codes in the tile-major layout,   */
/* s [E, N/128, K/128] fp32, one scale per 128 x 128 block with the same    */
/* codec as the activations (s = fl32(amax/448), RNE, saturating).          */
moeq_status moeq_quant_weight(const float* w, int E, int N, int K,
                              uint8_t* q, float* s, void* stream);

/* moeq_pack_weight -- row-major E4M3 codes [E, N, K] -> the tile-major      */
/* layout (a permutation of bytes; q_rows and q_tiles must not overlap).    */
moeq_status moeq_pack_weight(const uint8_t* q_rows, int E, int N, int K,
                             uint8_t* q_tiles, void* stream);

/* moeq_route -- top-k routing plus expert deduplication for M tokens.     */
/* logits [M, E_routed] fp32 -> *plan (see moeq_route_plan).                */
/* M in [1, MOEQ_MAX_TOKENS], E_routed <= MOEQ_MAX_EXPERTS,                 */
/* top_k in [1, min(E_routed, MOEQ_MAX_TOPK)].                              */
moeq_status moeq_route(const float* logits, int M, int E_routed, int top_k,
                       const moeq_route_plan* plan, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_expert_gemm_gateup_swiglu -- quant(x) fused into the gate_up FP8    */
/* GEMM of every unique expert of a plan, split-K over all SMs with a       */
/* deterministic fp32 reduction, and the SwiGLU epilogue                    */
/* (GLM-5.2 x10 §1: split-K; §4: quantisation fused into the GEMM).         */
/* For M <= 16 and H <= 6144 it runs the multi-token kernel's gate_up mode  */
/* (tcgen05; columns of 128 h rows dealt over the SMs, a split column's     */
/* sums handed on); otherwise the persistent engine (tcgen05 at every row   */
/* count unless MOEQ_MMA_MIN_TOKENS sets a crossover).                      */
/*   x       [M, H] bf16 or fp32, M <= MOEQ_MAX_TOKENS                      */
/*   w_gu    n_experts x [2I, H] E4M3 tile-major: gate rows [0, I), up rows */
/*           [I, 2I)                                                        */
/*   s_gu    [n_experts, 2I/128, H/128] fp32                                */
/*   uniq/offs/pair_tok/n_uniq_dev: the plan (device), U read on the device */
/*   h       [max_pairs, I] fp32: h[p] = silu(gate . x[tok(p)]) * (up . x)  */
/*   q_x_opt [M, H], s_x_opt [M, H/128]: optional dump of the codes and     */
/*           scales the fused prologue used, for the tokens of the plan's   */
/*           last unique expert (the shared expert, which serves them all)  */
/* H and I multiples of 128, H <= MOEQ_MAX_K.  An expert holds at most M    */
/* pairs (its tokens are distinct); a plan that breaks this, or names an    */
/* expert or pair out of range, leaves MOEQ_ERR_INVALID_ARG in the          */
/* workspace status (moeq_read_device_status).                              */
/* ------------------------------------------------------------------------ */
moeq_status moeq_expert_gemm_gateup_swiglu(
    const void* x, moeq_dtype x_dtype, int M, int H, int I,
    const uint8_t* w_gu, const float* s_gu, int n_experts,
    const int32_t* uniq, const int32_t* offs, const int32_t* pair_tok,
    const int32_t* n_uniq_dev, int max_uniq, int max_pairs,
    float* h, uint8_t* q_x_opt, float* s_x_opt,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_expert_gemm_down -- quant(a) fused into the down FP8 GEMM of every  */
/* unique expert, split-K, deterministic fp32 reduction.  For N a multiple  */
/* of 256 up to 6144 (and its partials, max_pairs x N x K/128 floats,       */
/* within 256 MiB) it runs the multi-token kernel's down mode (tcgen05; its */
/* stages dealt over every SM); otherwise the engine (tcgen05 at every row */
/* count unless MOEQ_MMA_MIN_TOKENS sets a crossover).                      */
/*   a       [max_pairs, K] bf16 or fp32; row p is the input of pair p      */
/*           (h from the gate_up call, or x for a dense projection)         */
/*   w_d     n_experts x [N, K] E4M3 tile-major; s_d [n_experts, N/128,     */
/*           K/128] fp32                                                    */
/*   y       [max_pairs, N] fp32, row p = W_d[expert(p)] applied to a[p]    */
/*   q_a_opt [max_pairs, K], s_a_opt [max_pairs, K/128]: optional dump of   */
/*           the fused prologue's codes and scales                          */
/* A plan for a dense layer is uniq = {0}, offs = {0, M}, n_uniq = 1.       */
/* An expert holds at most min(max_pairs, MOEQ_MAX_TOKENS) pairs; a plan    */
/* that breaks this, or names an expert or pair out of range, leaves        */
/* MOEQ_ERR_INVALID_ARG in the workspace status.                            */
/* ------------------------------------------------------------------------ */
moeq_status moeq_expert_gemm_down(
    const void* a, moeq_dtype a_dtype, int K, int N,
    const uint8_t* w_d, const float* s_d, int n_experts,
    const int32_t* uniq, const int32_t* offs, const int32_t* n_uniq_dev,
    int max_uniq, int max_pairs,
    float* y, uint8_t* q_a_opt, float* s_a_opt,
    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_expert_gemm_down_noalloc -- moeq_expert_gemm_down with no caller     */
/* workspace.  The pages have no counterpart: it exists for callers that     */
/* cannot lend a workspace and cannot allocate on their path (a plain C      */
/* host issuing one projection with no device buffer to spare, or an engine  */
/* whose device memory is committed to its own pools and whose decode step   */
/* may not call cudaMalloc, which can synchronise the device).               */
/*   Arguments, layouts and results are those of moeq_expert_gemm_down,      */
/*   without ws / ws_bytes: it runs the kernel that call runs, bit for bit  */
/*   the same, except where the multi-token kernel's areas would not fit    */
/*   the scratch below, when it runs the persistent engine instead.         */
/*   device_status_opt: NULL, or a caller-owned device int32 that receives   */
/*   the launch's device status word (0 = MOEQ_OK, else a moeq_status) on    */
/*   the stream after the launch.                                            */
/* Scratch: the library's own static device array of 8 MiB per device       */
/*   (counts and partials; on the engine also decoded activations and       */
/*   scales, and split-K tickets).  A problem that fits neither kernel's    */
/*   areas in it returns MOEQ_ERR_WORKSPACE and launches nothing; the dense */
/*   projection (K 2048, N 4096, one token) needs ~0.3 MiB on the multi-token */
/*   kernel, and K = 32768 with 16 rows ~7 MiB on the engine.  Its counters must be  */
/*   zero when a launch starts: every call zeroes them on `stream` itself    */
/*   (cudaMemsetAsync), so nothing has to be zero beforehand.                */
/* Set-up: the first call on each device looks up that device's scratch      */
/*   address (cudaGetSymbolAddress, with the device current) and caches it;  */
/*   make that first call before any stream capture.                         */
/* Concurrency: every call on a device uses the same scratch, so calls that  */
/*   may overlap in time (other streams, other host threads) race: issue     */
/*   them on one stream.                                                     */
/* Allocates no device or host memory.                                       */
/* ------------------------------------------------------------------------ */
moeq_status moeq_expert_gemm_down_noalloc(
    const void* a, moeq_dtype a_dtype, int K, int N,
    const uint8_t* w_d, const float* s_d, int n_experts,
    const int32_t* uniq, const int32_t* offs, const int32_t* n_uniq_dev,
    int max_uniq, int max_pairs,
    float* y, uint8_t* q_a_opt, float* s_a_opt,
    int32_t* device_status_opt, void* stream);

/* moeq_combine -- out[m] = bf16_RNE(y[pair_of[m][top_k]] +                 */
/*   sum_{j < top_k} topk_w[m][j] * y[pair_of[m][j]]), fp32, in slot order. */
/* y [max_pairs, N] fp32, out [M, N] bf16.  top_k may be 0 (dense layer:    */
/* pair_of[m][0] is then the only term, weight 1).                          */
moeq_status moeq_combine(const float* y, int N, const moeq_route_plan* plan, int M, int top_k,
                         void* out_bf16, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_dense_ffn -- one dense FFN for M tokens, in ONE kernel:             */
/*   out = bf16( down( quant( silu(gate) * up ) ) ), gate/up = gate_up(quant(x)) */
/*   (GLM-5.2 x10 §4: the live quantisation fused into the GEMMs -- the      */
/*   "PQ-GEMM" FFN; §1: K split so that every SM streams.)  The multi-token  */
/*   kernel of moeq_moe_layer with no routing (top_k = 0): one column per    */
/*   128-wide K group of down streams that group's gate and up rows for     */
/*   every token, forms and quantises the group, and streams down's K group */
/*   against every output row; the fp32 partials of each (token, 16 output  */
/*   rows) are summed in a fixed order by idle warps.  With fewer columns   */
/*   (I/128) than SMs, the SMs left over stream the first part of the       */
/*   columns' gate_up and hand the sums on.  With MOEQ_MTOK_MIN_TOKENS       */
/*   above 1, one token runs the one-token kernel (CUDA cores) instead.     */
/*   Launched with programmatic dependent launch (see                       */
/*   moeq_moe_layer): the weights must not be written by the kernel right   */
/*   ahead of this call on the same stream, except by moeq_quant_weight /    */
/*   moeq_pack_weight, which this library tracks.                          */
/*   M      1 .. MOEQ_MAX_TOKENS                                            */
/*   x      [M, H] bf16; H a multiple of 256, at most 6144; I a multiple    */
/*           of 128                                                         */
/*   w_gu/s_gu [1, 2I, H] tile-major + [1, 2I/128, H/128]: gate rows [0, I), */
/*           up rows [I, 2I); w_d/s_d [1, H, I] + [1, H/128, I/128]          */
/*   out    [M, H] bf16                                                     */
/*   h_opt [M, I] f32, q_x_opt/s_x_opt [M, H] u8 + [M, H/128] f32,          */
/*   q_h_opt/s_h_opt [M, I] u8 + [M, I/128] f32: optional dumps (each pair  */
/*           both or neither) of h and of both live quantisations           */
/*   ws     moeq_dense_ffn_workspace_size(M, H, I) bytes (0 for shapes out  */
/*           of range or with no device), zeroed once                       */
/* ------------------------------------------------------------------------ */
size_t moeq_dense_ffn_workspace_size(int M, int H, int I);
moeq_status moeq_dense_ffn(const void* x, int M, int H, int I,
                           const uint8_t* w_gu, const float* s_gu,
                           const uint8_t* w_d, const float* s_d,
                           void* out, float* h_opt,
                           uint8_t* q_x_opt, float* s_x_opt,
                           uint8_t* q_h_opt, float* s_h_opt,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_moe_layer -- one MoE FFN layer for M tokens, in ONE kernel:         */
/*   route -> [quant x + gate_up + SwiGLU] -> [quant h + down] -> combine   */
/*   (GLM-5.2 x10: bandwidth model -- a decode layer reads its top-8        */
/*   experts plus the shared one; §1 and §8c -- live FP8 quantisation of    */
/*   the activations in front of each GEMM; §4 -- fused into it; §1 --      */
/*   split-K so that every SM streams; §5-§6 -- tokens verified together     */
/*   read each expert once.)                                                */
/*   y not asked for, top_k <= 16, H <= 6144 and H % 256 == 0: the          */
/*   multi-token kernel, on the tcgen05 tensor cores.  A column is (unique  */
/*   expert, 128-wide K group of down): the h group's gate and up rows over */
/*   all of H, then down's K group against every output row; the column's   */
/*   MMAs take every token and keep its expert's.  The columns' stages are  */
/*   dealt out evenly over the SMs (a column may be split between two CTAs, */
/*   whose second part comes last in its CTA's order), x is quantised once  */
/*   in the grid, and each token's 16 output rows are summed in a fixed     */
/*   order (and rounded to bf16) by idle warps as soon as their output unit */
/*   is complete.  It is launched with programmatic dependent launch: the   */
/*   next kernel on the stream may start as its CTAs finish, and waits      */
/*   (griddepcontrol.wait) before it reads anything this one writes.  With  */
/*   MOEQ_MTOK_MIN_TOKENS=2 one token runs the one-token kernel instead     */
/*   (CUDA cores, top_k <= 8; the kernel of moeq_dense_ffn).                */
/*   Otherwise: one persistent CTA per SM (cooperative launch).  Every CTA  */
/*   routes for itself while CTAs whose first blocks are the shared         */
/*   expert's already stream them; down waits per expert for its h, and the */
/*   combine runs in the down epilogue (M == 1 without y on the persistent  */
/*   engine streams down by K group instead).                               */
/*   All paths give out within the same bound; their fp32 rounding orders   */
/*   differ.                                                                */
/*   x      [M, H] bf16; logits [M, E_routed] fp32                          */
/*   w_gu/s_gu, w_d/s_d: E_routed + 1 experts (tile-major codes), the       */
/*           shared expert last                                             */
/*   out    [M, H] bf16                                                     */
/*   plan_opt, h_opt [max_pairs, I], y_opt [max_pairs, H]: optional         */
/*           caller buffers that receive the plan and the intermediates     */
/*           (NULL: kept in the workspace; a non-NULL y_opt selects the     */
/*           row-block down path, which is the one that forms y)            */
/*   q_x_opt [M, H] u8 + s_x_opt [M, H/128] f32: optional, both or neither: */
/*           the codes and scales of x's live quantisation (a2)             */
/*   q_h_opt [max_pairs, I] u8 + s_h_opt [max_pairs, I/128] f32: optional,  */
/*           both or neither: the codes and scales of h's live quantisation */
/*           (a5), the ones the down GEMM multiplies, h being the layer's   */
/*           own fp32 h (h_opt)                                             */
/*   events_opt: NULL, or 2 cudaEvent_t recorded on `stream` right before   */
/*           and right after the layer's kernel, for the caller's timing    */
/* A workspace serves one layer call at a time: consecutive calls on one    */
/* stream may share it, concurrent calls may not.                           */
/* ------------------------------------------------------------------------ */
moeq_status moeq_moe_layer(const void* x, const float* logits,
                           int M, int H, int I, int E_routed, int top_k,
                           const uint8_t* w_gu, const float* s_gu,
                           const uint8_t* w_d, const float* s_d,
                           void* out, const moeq_route_plan* plan_opt,
                           float* h_opt, float* y_opt,
                           uint8_t* q_x_opt, float* s_x_opt,
                           uint8_t* q_h_opt, float* s_h_opt,
                           void* const* events_opt,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Tensor parallelism (GLM-5.2 x10, bandwidth model: TP8 splits every       */
/* expert over 8 cards, each card streaming 1/8 of the layer's bytes).      */
/* Rank r of R holds, for every expert, the I-slice [r*I/R, (r+1)*I/R) of   */
/* the gate rows and of the up rows of gate_up, and the same K-slice of     */
/* down (I/R a multiple of 128): a layer with intermediate I/R.  Its fp32   */
/* partial out is the sum over its slice; the layer's output is            */
/* bf16(sum over r = 0 .. R-1, in that order, of the partials).  h groups   */
/* never straddle slices, so each rank's live quantisation of h is the      */
/* unsharded one's.                                                         */
/*                                                                          */
/* moeq_tp_shard_weights -- rank `rank`'s shard of full tile-major weights  */
/*   (E experts, the shared one included): w_gu_shard [E, 2I/R, H] (gate    */
/*   slice then up slice) + s_gu_shard [E, 2I/(128R), H/128], w_d_shard     */
/*   [E, H, I/R] + s_d_shard [E, H/128, I/(128R)].  Whole 128 x 128 tiles   */
/*   and their scales are copied (strided device-to-device copies on        */
/*   `stream`; no arithmetic).                                              */
/* moeq_moe_layer_shard -- moeq_moe_layer on one rank's shard (I_shard =    */
/*   I/R), writing the fp32 partial out_partial [M, H] instead of bf16;     */
/*   routing, x's quantisation and the plan are the full layer's.  Served   */
/*   by the one-token and multi-token kernels only (H a multiple of 256 up  */
/*   to 6144, top_k <= 8 at one token): other calls return                  */
/*   MOEQ_ERR_UNSUPPORTED_SHAPE.  Workspace: moeq_workspace_size(M, H,      */
/*   I_shard, E_routed + 1, top_k).                                         */
/* moeq_tp_reduce -- out_bf16 [M, H] = bf16(sum_r partials[r]) over         */
/*   partials [R, M, H] fp32 (all ranks' partials, gathered in rank order), */
/*   added in rank order.                                                   */
/* The exchange of the partials between GPUs (an all-gather) is the        */
/* caller's (bandwidth_bound_fp8_gb300/tp.py uses torch.distributed).       */
/* ------------------------------------------------------------------------ */
moeq_status moeq_tp_shard_weights(int E, int H, int I, int R, int rank,
                                  const uint8_t* w_gu, const float* s_gu,
                                  const uint8_t* w_d, const float* s_d,
                                  uint8_t* w_gu_shard, float* s_gu_shard,
                                  uint8_t* w_d_shard, float* s_d_shard, void* stream);
moeq_status moeq_moe_layer_shard(const void* x, const float* logits,
                                 int M, int H, int I_shard, int E_routed, int top_k,
                                 const uint8_t* w_gu, const float* s_gu,
                                 const uint8_t* w_d, const float* s_d,
                                 float* out_partial, const moeq_route_plan* plan_opt,
                                 float* h_opt, uint8_t* q_x_opt, float* s_x_opt,
                                 uint8_t* q_h_opt, float* s_h_opt,
                                 void* ws, size_t ws_bytes, void* stream);
moeq_status moeq_tp_reduce(const float* partials, int R, int M, int H, void* out_bf16, void* stream);

/* ------------------------------------------------------------------------ */
/* moeq_moe_stack -- one decode step through L MoE layers in sequence, as   */
/*   ONE CUDA graph (GLM-5.2 x10 §8b: graph replay takes the host's         */
/*   per-kernel launch cost out of a decode step).  Layer l runs            */
/*   moeq_moe_layer on x_l (x_0 = x, x_l = layer l-1's bf16 output) with     */
/*   its own logits and weights.  The first call with a given set of        */
/*   arguments captures the L launches and instantiates the graph; every    */
/*   later call with the same arguments (pointers included) launches it on  */
/*   `stream`, so new data in the same buffers needs no host work.  Up to   */
/*   16 graphs are kept per process (least recently used dropped); a call   */
/*   made while `stream` is being captured by the caller, or with           */
/*   MOEQ_STACK_EAGER, launches the layers directly instead.                */
/*   Layers after the first route before they wait for the layer ahead     */
/*   (their logits are inputs, which no layer writes).                      */
/*   L      1 .. MOEQ_MAX_LAYERS                                            */
/*   x      [M, H] bf16                                                     */
/*   logits [L, M, E_routed] fp32, contiguous                               */
/*   w_gu, s_gu, w_d, s_d: HOST arrays of L device pointers, layer l's      */
/*           weights as moeq_moe_layer takes them (read during the call;    */
/*           the arrays may be freed after it)                              */
/*   out    [L, M, H] bf16: every layer's output (layer L-1's is the        */
/*           stack's); must not overlap x, logits or the weights            */
/*   flags  0 or MOEQ_STACK_EAGER                                           */
/*   ws     moeq_stack_workspace_size(L, M, H, I, E_routed + 1, top_k)      */
/*           bytes, zeroed once with moeq_workspace_init; it holds one      */
/*           layer workspace and every layer's route plan (moeq_stack_plan  */
/*           gives layer l's).  A graph records the workspace's address: do */
/*           not free a workspace while a call that used it may still run.  */
/* Errors: every layer's arguments are checked before anything is launched  */
/* or captured (the statuses of moeq_moe_layer); a failed capture or        */
/* instantiation returns MOEQ_ERR_CUDA and keeps nothing.                   */
/* ------------------------------------------------------------------------ */
size_t moeq_stack_workspace_size(int L, int M, int H, int I, int n_experts_incl_shared, int top_k);
moeq_status moeq_moe_stack(int L, const void* x, const float* logits,
                           int M, int H, int I, int E_routed, int top_k,
                           const uint8_t* const* w_gu, const float* const* s_gu,
                           const uint8_t* const* w_d, const float* const* s_d,
                           void* out, int flags, void* ws, size_t ws_bytes, void* stream);
/* Layer `layer`'s route plan inside a stack workspace (pointers only; the  */
/* plan is written by the stack's calls).                                   */
moeq_status moeq_stack_plan(void* ws, size_t ws_bytes, int L, int M, int H, int I, int E_routed, int top_k,
                            int layer, moeq_route_plan* plan);
/* Destroy every graph moeq_moe_stack keeps (a graph still running is freed */
/* when it completes).  The next stack call captures again.                 */
moeq_status moeq_stack_release_graphs(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ_H */
