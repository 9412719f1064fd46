// The C ABI of libmoeq (include/moeq.h): argument validation, workspace
// layout, TMA tensor-map construction and the launch sequence.  Every check
// runs on the host before anything is launched.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "moeq_internal.h"

using namespace moeq;

namespace {

constexpr int kAbiVersion = 1;

struct DeviceInfo {
    int ok = 0;
    int sms = 0;
};

DeviceInfo current_device() {
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DeviceInfo{};
    }
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1);
    if (!cache[dev].sms) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return DeviceInfo{};
        }
        cache[dev].sms = sms;
        cache[dev].ok = (major == 10 && minor == 3);
    }
    return cache[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

moeq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOEQ_OK : MOEQ_ERR_CUDA; }

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D map over the FP8 weights seen as [rows, K] bytes, 128 x 128 boxes,
// no swizzle (each box lands as 128 rows of 128 contiguous bytes).
bool weight_map(CUtensorMap* map, const uint8_t* w, uint64_t rows, uint64_t K) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ workspace
// Standalone GEMM workspace: [status int (256 B)] [tickets] [partials].
struct GemmWs {
    size_t tickets, partials, end;
};

GemmWs gemm_ws_layout(size_t base, int RB, int max_uniq, int nbox, int grid) {
    GemmWs l;
    l.tickets = align_up(base, 256);
    l.partials = align_up(l.tickets + sizeof(int) * static_cast<size_t>(RB) * max_uniq, 256);
    l.end = l.partials + sizeof(float) * gemm_partials_floats(nbox, grid);
    return l;
}

struct LayerWs {
    size_t plan, h, y, end;
    GemmWs gu, dn;
};

LayerWs layer_ws_layout(int M, int H, int I, int E, int k, int grid) {
    LayerWs l;
    const int mu = moeq_max_uniq(M, E, k), mp = moeq_max_pairs(M, k);
    l.plan = 256;
    l.h = align_up(l.plan + moeq_route_plan_bytes(M, E, k), 256);
    l.y = align_up(l.h + sizeof(float) * static_cast<size_t>(mp) * I, 256);
    const size_t after = l.y + sizeof(float) * static_cast<size_t>(mp) * H;
    l.gu = gemm_ws_layout(after, I / 128, mu, 2, grid);
    l.dn = gemm_ws_layout(l.gu.end, H / 128, mu, 1, grid);
    l.end = l.dn.end;
    return l;
}

struct PlanLayout {
    size_t topk_id, topk_w, n_uniq, uniq, offs, pair_tok, pair_of, end;
};

PlanLayout plan_layout(int M, int E, int k) {
    PlanLayout p;
    const int mu = moeq_max_uniq(M, E, k), mp = moeq_max_pairs(M, k);
    p.topk_id = 0;
    p.topk_w = align_up(p.topk_id + 4 * static_cast<size_t>(M) * k, 16);
    p.n_uniq = align_up(p.topk_w + 4 * static_cast<size_t>(M) * k, 16);
    p.uniq = align_up(p.n_uniq + 4, 16);
    p.offs = align_up(p.uniq + 4 * static_cast<size_t>(mu), 16);
    p.pair_tok = align_up(p.offs + 4 * static_cast<size_t>(mu + 1), 16);
    p.pair_of = align_up(p.pair_tok + 4 * static_cast<size_t>(mp), 16);
    p.end = align_up(p.pair_of + 4 * static_cast<size_t>(M) * (k + 1), 16);
    return p;
}

bool route_args_ok(int M, int E, int k) {
    return M >= 1 && M <= MOEQ_MAX_TOKENS && E >= 1 && E <= MOEQ_MAX_EXPERTS && k >= 1 && k <= MOEQ_MAX_TOPK &&
           k <= E;
}

bool plan_ok(const moeq_route_plan* p) {
    return p && p->topk_id && p->topk_w && p->n_uniq && p->uniq && p->offs && p->pair_tok && p->pair_of;
}

// Shared body of the two GEMM calls, after their own argument checks.
moeq_status run_gemm(const void* a, int a_f32, const int32_t* a_row, int K, int rows_per_expert, int up_offset,
                     int RB, int nbox, const uint8_t* w, const float* sw, int n_experts, const int32_t* uniq,
                     const int32_t* offs, const int32_t* n_uniq, int max_uniq, int max_pairs, int rows_a,
                     float* out, int out_ld,
                     uint8_t* qdump, float* sdump, void* ws, const GemmWs& wl, const DeviceInfo& dev,
                     cudaStream_t stream) {
    CUtensorMap map;
    if (!weight_map(&map, w, static_cast<uint64_t>(n_experts) * rows_per_expert, static_cast<uint64_t>(K)))
        return MOEQ_ERR_CUDA;
    GemmArgs g;
    g.a = a;
    g.a_f32 = a_f32;
    g.a_row = a_row;
    g.K = K;
    g.rows_per_expert = rows_per_expert;
    g.up_offset = up_offset;
    g.RB = RB;
    g.sw = sw;
    g.uniq = uniq;
    g.offs = offs;
    g.n_uniq = n_uniq;
    g.out = out;
    g.out_ld = out_ld;
    g.qdump = qdump;
    g.sdump = sdump;
    char* base = static_cast<char*>(ws);
    g.tickets = reinterpret_cast<int*>(base + wl.tickets);
    g.partials = reinterpret_cast<float*>(base + wl.partials);
    g.status = reinterpret_cast<int*>(base);
    g.n_experts = n_experts;
    g.max_uniq = max_uniq;
    g.max_pairs = max_pairs;
    g.rows_a = rows_a;
    return cuda_status(launch_expert_gemm(map, g, nbox, dev.sms, stream));
}

}  // namespace

// ====================================================================== ABI
extern "C" {

const char* moeq_status_string(moeq_status s) {
    switch (s) {
        case MOEQ_OK: return "ok";
        case MOEQ_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad dtype or M)";
        case MOEQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (dimensions must be multiples of 128 within limits)";
        case MOEQ_ERR_WORKSPACE: return "workspace missing or too small";
        case MOEQ_ERR_CUDA: return "a CUDA runtime call failed";
        case MOEQ_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        case MOEQ_ERR_DEVICE: return "no CUDA device of compute capability 10.3";
    }
    return "unknown status";
}

int moeq_abi_version(void) { return kAbiVersion; }

int moeq_max_uniq(int M, int E_routed, int top_k) {
    if (M < 1 || E_routed < 1 || top_k < 0) return 0;
    return std::min(E_routed, M * top_k) + 1;
}

int moeq_max_pairs(int M, int top_k) {
    if (M < 1 || top_k < 0) return 0;
    return M * top_k + M;
}

size_t moeq_route_plan_bytes(int M, int E_routed, int top_k) {
    if (!route_args_ok(M, E_routed, top_k)) return 0;
    return plan_layout(M, E_routed, top_k).end;
}

moeq_status moeq_route_plan_carve(void* base, size_t bytes, int M, int E_routed, int top_k, moeq_route_plan* plan) {
    if (!base || !plan || !aligned16(base)) return MOEQ_ERR_INVALID_ARG;
    if (!route_args_ok(M, E_routed, top_k)) return MOEQ_ERR_INVALID_ARG;
    const PlanLayout l = plan_layout(M, E_routed, top_k);
    if (bytes < l.end) return MOEQ_ERR_WORKSPACE;
    char* b = static_cast<char*>(base);
    plan->topk_id = reinterpret_cast<int32_t*>(b + l.topk_id);
    plan->topk_w = reinterpret_cast<float*>(b + l.topk_w);
    plan->n_uniq = reinterpret_cast<int32_t*>(b + l.n_uniq);
    plan->uniq = reinterpret_cast<int32_t*>(b + l.uniq);
    plan->offs = reinterpret_cast<int32_t*>(b + l.offs);
    plan->pair_tok = reinterpret_cast<int32_t*>(b + l.pair_tok);
    plan->pair_of = reinterpret_cast<int32_t*>(b + l.pair_of);
    return MOEQ_OK;
}

size_t moeq_workspace_size(int M, int H, int I, int n_experts_incl_shared, int top_k) {
    const int E = n_experts_incl_shared - 1;
    if (!route_args_ok(M, E, top_k) || H <= 0 || I <= 0 || H % 128 || I % 128 || H > MOEQ_MAX_K || I > MOEQ_MAX_K)
        return 0;
    const DeviceInfo dev = current_device();
    if (!dev.sms) return 0;
    return layer_ws_layout(M, H, I, E, top_k, dev.sms).end;
}

size_t moeq_gemm_workspace_size(int rows_out, int max_uniq, int is_gate_up) {
    if (rows_out <= 0 || rows_out % 128 || max_uniq < 1) return 0;
    const DeviceInfo dev = current_device();
    if (!dev.sms) return 0;
    return gemm_ws_layout(256, rows_out / 128, max_uniq, is_gate_up ? 2 : 1, dev.sms).end;
}

moeq_status moeq_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < 256 || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream)));
}

moeq_status moeq_read_device_status(const void* ws, size_t ws_bytes, int* device_status) {
    if (!ws || ws_bytes < 256 || !device_status) return MOEQ_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOEQ_ERR_CUDA;
    return cuda_status(cudaMemcpy(device_status, ws, sizeof(int), cudaMemcpyDeviceToHost));
}

moeq_status moeq_quant_act(const void* x, moeq_dtype x_dtype, int M, int K, uint8_t* q, float* s, void* stream) {
    if (!x || !q || !s || !aligned16(x) || !aligned16(q) || !aligned4(s)) return MOEQ_ERR_INVALID_ARG;
    if (x_dtype != MOEQ_BF16 && x_dtype != MOEQ_F32) return MOEQ_ERR_INVALID_ARG;
    if (M < 1 || M > 4096) return MOEQ_ERR_INVALID_ARG;
    if (K <= 0 || K % 128 || K > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    return cuda_status(launch_quant_act(x, x_dtype == MOEQ_F32, M, K, q, s, as_stream(stream)));
}

moeq_status moeq_quant_weight(const float* w, int E, int N, int K, uint8_t* q, float* s, void* stream) {
    if (!w || !q || !s || !aligned16(w) || !aligned16(q) || !aligned4(s)) return MOEQ_ERR_INVALID_ARG;
    if (E < 1 || E > 65535) return MOEQ_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || N % 128 || K % 128 || N / 128 > 65535 || K / 128 > 65535)
        return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    return cuda_status(launch_quant_weight(w, E, N, K, q, s, as_stream(stream)));
}

moeq_status moeq_route(const float* logits, int M, int E_routed, int top_k, const moeq_route_plan* plan,
                       void* stream) {
    if (!logits || !plan_ok(plan)) return MOEQ_ERR_INVALID_ARG;
    if (!route_args_ok(M, E_routed, top_k)) return MOEQ_ERR_INVALID_ARG;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    return cuda_status(launch_route(logits, M, E_routed, top_k, *plan, as_stream(stream)));
}

moeq_status moeq_expert_gemm_gateup_swiglu(const void* x, moeq_dtype x_dtype, int M, int H, int I,
                                           const uint8_t* w_gu, const float* s_gu, int n_experts,
                                           const int32_t* uniq, const int32_t* offs, const int32_t* pair_tok,
                                           const int32_t* n_uniq_dev, int max_uniq, int max_pairs, float* h,
                                           uint8_t* q_x_opt, float* s_x_opt, void* ws, size_t ws_bytes,
                                           void* stream) {
    if (!x || !w_gu || !s_gu || !uniq || !offs || !pair_tok || !n_uniq_dev || !h) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gu) || !aligned16(h) || !aligned4(s_gu)) return MOEQ_ERR_INVALID_ARG;
    if ((q_x_opt == nullptr) != (s_x_opt == nullptr)) return MOEQ_ERR_INVALID_ARG;
    if (q_x_opt && !aligned16(q_x_opt)) return MOEQ_ERR_INVALID_ARG;
    if (x_dtype != MOEQ_BF16 && x_dtype != MOEQ_F32) return MOEQ_ERR_INVALID_ARG;
    if (M < 1 || M > MOEQ_MAX_TOKENS || n_experts < 1 || max_uniq < 1 || max_pairs < 1) return MOEQ_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 128 || I % 128 || H > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(n_experts) * 2 * I >= (1LL << 31)) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const GemmWs wl = gemm_ws_layout(256, I / 128, max_uniq, 2, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < wl.end) return MOEQ_ERR_WORKSPACE;
    return run_gemm(x, x_dtype == MOEQ_F32, pair_tok, H, 2 * I, I, I / 128, 2, w_gu, s_gu, n_experts, uniq, offs,
                    n_uniq_dev, max_uniq, max_pairs, M, h, I, q_x_opt, s_x_opt, ws, wl, dev, as_stream(stream));
}

moeq_status moeq_expert_gemm_down(const void* a, moeq_dtype a_dtype, int K, int N, const uint8_t* w_d,
                                  const float* s_d, int n_experts, const int32_t* uniq, const int32_t* offs,
                                  const int32_t* n_uniq_dev, int max_uniq, int max_pairs, float* y, uint8_t* q_a_opt,
                                  float* s_a_opt, void* ws, size_t ws_bytes, void* stream) {
    if (!a || !w_d || !s_d || !uniq || !offs || !n_uniq_dev || !y) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w_d) || !aligned16(y) || !aligned4(s_d)) return MOEQ_ERR_INVALID_ARG;
    if ((q_a_opt == nullptr) != (s_a_opt == nullptr)) return MOEQ_ERR_INVALID_ARG;
    if (q_a_opt && !aligned16(q_a_opt)) return MOEQ_ERR_INVALID_ARG;
    if (a_dtype != MOEQ_BF16 && a_dtype != MOEQ_F32) return MOEQ_ERR_INVALID_ARG;
    if (n_experts < 1 || max_uniq < 1 || max_pairs < 1) return MOEQ_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || K % 128 || N % 128 || K > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(n_experts) * N >= (1LL << 31)) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const GemmWs wl = gemm_ws_layout(256, N / 128, max_uniq, 1, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < wl.end) return MOEQ_ERR_WORKSPACE;
    return run_gemm(a, a_dtype == MOEQ_F32, nullptr, K, N, 0, N / 128, 1, w_d, s_d, n_experts, uniq, offs,
                    n_uniq_dev, max_uniq, max_pairs, max_pairs, y, N, q_a_opt, s_a_opt, ws, wl, dev,
                    as_stream(stream));
}

moeq_status moeq_combine(const float* y, int N, const moeq_route_plan* plan, int M, int top_k, void* out_bf16,
                         void* stream) {
    if (!y || !plan || !plan->pair_of || !out_bf16 || (top_k > 0 && !plan->topk_w)) return MOEQ_ERR_INVALID_ARG;
    if (M < 1 || M > MOEQ_MAX_TOKENS || top_k < 0 || top_k > MOEQ_MAX_TOPK) return MOEQ_ERR_INVALID_ARG;
    if (N <= 0 || N % 128) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    return cuda_status(launch_combine(y, N, *plan, M, top_k, out_bf16, as_stream(stream)));
}

moeq_status moeq_moe_layer(const void* x, const float* logits, int M, int H, int I, int E_routed, int top_k,
                           const uint8_t* w_gu, const float* s_gu, const uint8_t* w_d, const float* s_d, void* out,
                           const moeq_route_plan* plan_opt, float* h_opt, float* y_opt, void* const* events_opt,
                           void* ws, size_t ws_bytes, void* stream) {
    if (!x || !logits || !w_gu || !s_gu || !w_d || !s_d || !out) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gu) || !aligned16(w_d) || !aligned16(out) || !aligned4(s_gu) || !aligned4(s_d))
        return MOEQ_ERR_INVALID_ARG;
    if ((h_opt && !aligned16(h_opt)) || (y_opt && !aligned16(y_opt))) return MOEQ_ERR_INVALID_ARG;
    if (plan_opt && !plan_ok(plan_opt)) return MOEQ_ERR_INVALID_ARG;
    if (!route_args_ok(M, E_routed, top_k)) return MOEQ_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 128 || I % 128 || H > MOEQ_MAX_K || I > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const long long n_exp = static_cast<long long>(E_routed) + 1;
    if (n_exp * 2 * I >= (1LL << 31) || n_exp * H >= (1LL << 31)) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const LayerWs l = layer_ws_layout(M, H, I, E_routed, top_k, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < l.end) return MOEQ_ERR_WORKSPACE;

    char* base = static_cast<char*>(ws);
    moeq_route_plan plan;
    if (plan_opt) {
        plan = *plan_opt;
    } else {
        moeq_route_plan_carve(base + l.plan, l.h - l.plan, M, E_routed, top_k, &plan);
    }
    float* h = h_opt ? h_opt : reinterpret_cast<float*>(base + l.h);
    float* y = y_opt ? y_opt : reinterpret_cast<float*>(base + l.y);
    const int mu = moeq_max_uniq(M, E_routed, top_k);
    cudaStream_t st = as_stream(stream);
    auto mark = [&](int i) -> cudaError_t {
        return events_opt ? cudaEventRecord(static_cast<cudaEvent_t>(events_opt[i]), st) : cudaSuccess;
    };

    if (mark(0) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (launch_route(logits, M, E_routed, top_k, plan, st) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (mark(1) != cudaSuccess) return MOEQ_ERR_CUDA;
    const int mp = moeq_max_pairs(M, top_k);
    moeq_status s = run_gemm(x, 0, plan.pair_tok, H, 2 * I, I, I / 128, 2, w_gu, s_gu, E_routed + 1, plan.uniq,
                             plan.offs, plan.n_uniq, mu, mp, M, h, I, nullptr, nullptr, ws, l.gu, dev, st);
    if (s != MOEQ_OK) return s;
    if (mark(2) != cudaSuccess) return MOEQ_ERR_CUDA;
    s = run_gemm(h, 1, nullptr, I, H, 0, H / 128, 1, w_d, s_d, E_routed + 1, plan.uniq, plan.offs, plan.n_uniq, mu,
                 mp, mp, y, H, nullptr, nullptr, ws, l.dn, dev, st);
    if (s != MOEQ_OK) return s;
    if (mark(3) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (launch_combine(y, H, plan, M, top_k, out, st) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (mark(4) != cudaSuccess) return MOEQ_ERR_CUDA;
    return MOEQ_OK;
}

}  // extern "C"
