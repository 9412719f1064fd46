// The C ABI of libmoeq (include/moeq.h): argument validation, workspace
// layout and the launches.  Every check
// runs on the host before anything is launched.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "moeq_internal.h"

using namespace moeq;

namespace {

constexpr int kAbiVersion = 2;

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

// Token count (per expert) from which the engine's layer launches take the
// tcgen05 path: 8, where it measured faster than the CUDA cores.  The
// environment variable MOEQ_MMA_MIN_TOKENS overrides it, for the GEMM calls
// too (read once; 17 or more keeps every launch on the CUDA cores, 1 sends
// every launch to the tensor cores).
int mma_min_tokens() {
    static const int v = [] {
        const char* e = std::getenv("MOEQ_MMA_MIN_TOKENS");
        const int x = e ? std::atoi(e) : 0;
        return x >= 1 ? x : kMmaMinTokens;
    }();
    return v;
}
// The standalone GEMM calls that fall to the engine are those beyond the
// multi-token kernel's shapes, chiefly large-N projections (the LM head:
// 163 us on tcgen05 against 175 us on the CUDA cores at one token, 170
// against 594 at four), so they take tcgen05 at every row count unless
// MOEQ_MMA_MIN_TOKENS says otherwise.
int gemm_mma_min_tokens() {
    static const bool set = [] {
        const char* e = std::getenv("MOEQ_MMA_MIN_TOKENS");
        return e && std::atoi(e) >= 1;
    }();
    return set ? mma_min_tokens() : 1;
}

// The one-token layer kernel serves M = 1 layers on the CUDA cores unless
// MOEQ_TOKEN_KERNEL=0 (then the persistent engine does, as it does for every
// other M); MOEQ_PDL=0 launches it without programmatic dependent launch.
// Both read once.
bool env_flag(const char* name, bool dflt) {
    const char* e = std::getenv(name);
    if (!e || !*e) return dflt;
    return std::atoi(e) != 0;
}
bool token_kernel_enabled() {
    static const bool v = env_flag("MOEQ_TOKEN_KERNEL", true);
    return v;
}
bool pdl_enabled() {
    static const bool v = env_flag("MOEQ_PDL", true);
    return v;
}
// Layers of 1..16 tokens run the multi-token kernel unless
// MOEQ_MTOK_KERNEL=0 (then the persistent engine does); MOEQ_MTOK_MIN_TOKENS
// (default 1) moves its lower end, 2 handing one-token layers to the
// one-token kernel.  Both read once.
bool mtok_kernel_enabled() {
    static const bool v = env_flag("MOEQ_MTOK_KERNEL", true);
    return v;
}
int mtok_min_tokens() {
    static const int v = [] {
        const char* e = std::getenv("MOEQ_MTOK_MIN_TOKENS");
        const int x = e ? std::atoi(e) : 0;
        return x >= 1 ? x : 1;
    }();
    return v;
}
// The standalone GEMM calls spread over every SM; MOEQ_GRID_LIMIT=n (read
// once) caps them at n CTAs, for experiments that compare split widths.
int gemm_grid(int sms) {
    static const int lim = [] {
        const char* e = std::getenv("MOEQ_GRID_LIMIT");
        const int x = e ? std::atoi(e) : 0;
        return x >= 1 ? x : 0;
    }();
    return lim ? std::min(lim, sms) : sms;
}

// The one-token kernel reads weights before it waits for the kernel ahead of
// it on the stream (programmatic dependent launch).  This library's own
// weight writers (moeq_quant_weight, moeq_pack_weight) note their stream
// here; a layer call that directly follows one on the same stream launches
// without programmatic dependence, so it reads the weights only after the
// writer has finished.
std::atomic<uintptr_t> g_weight_write_stream{0};
inline uintptr_t stream_key(void* s) { return s ? reinterpret_cast<uintptr_t>(s) : uintptr_t(1); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

moeq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOEQ_OK : MOEQ_ERR_CUDA; }

// ------------------------------------------------------------------ workspace
// Header (256 B): status word, epoch, done ticket, input-quantisation count,
// down-by-K-group count.
constexpr size_t kOffStatus = 0, kOffEpoch = 4, kOffDone = 8, kOffACnt = 16, kOffDcCnt = 20, kHeader = 256;

struct StreamWs {
    size_t aq[2], as[2];
    size_t tickets[kMaxLists];
    size_t partials;
    size_t h_ready, comb, end;
};

// Quantised-activation buffers (rows x K floats + rows x K/128 scales per
// operand), ticket and partial areas for the given lists, from `base`.
StreamWs stream_ws_layout(size_t base, const int* aq_rows, const int* aq_k, int n_lists, const int* tickets_per_list,
                          int grid, int h_ready_n, int comb_n) {
    StreamWs l;
    size_t off = align_up(base, 256);
    for (int k = 0; k < 2; ++k) {
        // decoded fp32 codes (CUDA-core path) or 8 swizzle phases of the
        // E4M3 codes (tcgen05 path): 8 bytes per element covers both
        l.aq[k] = off;
        off = align_up(off + 8 * static_cast<size_t>(aq_rows[k]) * aq_k[k], 256);
        l.as[k] = off;
        off = align_up(off + sizeof(float) * static_cast<size_t>(aq_rows[k]) * (aq_k[k] / 128), 256);
    }
    for (int i = 0; i < kMaxLists; ++i) {
        l.tickets[i] = off;
        if (i < n_lists) off = align_up(off + sizeof(int) * static_cast<size_t>(tickets_per_list[i]), 256);
    }
    l.partials = off;
    off = align_up(off + sizeof(float) * stream_partials_floats(grid) * n_lists, 256);
    l.h_ready = off;
    off = align_up(off + sizeof(int) * static_cast<size_t>(h_ready_n), 256);
    l.comb = off;
    l.end = align_up(off + sizeof(int) * static_cast<size_t>(comb_n), 256);
    return l;
}

struct LayerWs {
    size_t plan, h, y, dc, tok_tickets;
    size_t mt_cnt, mt_slots, mt_xq, mt_xs, mt_part;   // multi-token kernel (M >= 2)
    StreamWs s;
};

LayerWs layer_ws_layout(int M, int H, int I, int E, int k, int grid) {
    LayerWs l;
    const int mu = moeq_max_uniq(M, E, k), mp = moeq_max_pairs(M, k);
    l.plan = kHeader;
    l.h = align_up(l.plan + moeq_route_plan_bytes(M, E, k), 256);
    l.y = align_up(l.h + sizeof(float) * static_cast<size_t>(mp) * I, 256);
    // one token: down by K group's sums per (pair, K group of down, column)
    l.dc = align_up(l.y + sizeof(float) * static_cast<size_t>(mp) * H, 256);
    // one token: the token kernel's partials share that area; its arrival
    // counts (one per 256 output rows) and completion count follow
    l.tok_tickets = align_up(l.dc + (M == 1 ? sizeof(float) * static_cast<size_t>(mp) * (I / 128) * H : 0), 256);
    const size_t tok_end =
        l.tok_tickets + (M == 1 ? sizeof(int) * (static_cast<size_t>((H + 255) / 256) + kGqUnits) : 0);
    // the multi-token kernel's counts and flags, split-column slots, x's
    // codes and scales, and the down partials (for the token counts it serves)
    const bool mt = M >= mtok_min_tokens();
    l.mt_cnt = align_up(tok_end, 256);
    l.mt_slots = align_up(l.mt_cnt + (mt ? sizeof(int) * (kMtokFlags + grid + 1) : 0), 256);
    l.mt_xq = align_up(l.mt_slots + (mt ? static_cast<size_t>(grid + 1) * kMtokSlotBytes : 0), 256);
    l.mt_xs = align_up(l.mt_xq + (mt ? static_cast<size_t>(H / 128) * kMtokXGroupBytes : 0), 256);
    l.mt_part = align_up(l.mt_xs + (mt ? sizeof(float) * static_cast<size_t>(H / 128) * 16 : 0), 256);
    const size_t after =
        l.mt_part + (mt ? sizeof(float) * static_cast<size_t>(M) * H * (k + 1) * (I / 128) : 0);
    // tickets of the layer's lists: M == 1 uses the first two (whole lists),
    // M > 1 all six (shared, half A, half B of each kind)
    const int rbmax = mu * ((H > I ? H : I) / 128);
    const int tk[6] = {rbmax, rbmax, rbmax, rbmax, rbmax, rbmax};
    const int rows[2] = {M, mp}, ks[2] = {H, I};
    l.s = stream_ws_layout(after, rows, ks, 6, tk, grid, mu * (I / 128), M * (H / 128));
    return l;
}

// kind 0: gate_up (input rows = tokens), kind 1: down (input rows = pairs)
StreamWs gemm_ws_layout(int kind, int RB, int K, int rows_a, int max_uniq, int grid) {
    const int tk[1] = {RB * max_uniq};
    int rows[2] = {0, 0}, ks[2] = {128, 128};
    rows[kind] = rows_a;
    ks[kind] = K;
    return stream_ws_layout(kHeader, rows, ks, 1, tk, grid, 0, 0);
}

// The multi-token kernel's areas for a standalone GEMM call (gate_up alone or
// down alone), from `base` on: counts and flags, and for gate_up the
// split-column slots and x's codes and scales (16 token rows per K group),
// for down the partials [pair][N/256][K/128][256] (down quantises its rows
// of a in shared memory).
struct MtokGemmWs {
    size_t cnt, slots, xq, xs, part, end;
};

MtokGemmWs mtok_gemm_ws(bool gate_up, int rows_out, int K, int rows_in, int grid, size_t base) {
    MtokGemmWs l;
    const size_t KX = static_cast<size_t>(K / 128);
    l.cnt = align_up(base, 256);
    l.slots = align_up(l.cnt + sizeof(int) * (kMtokFlags + grid + 1), 256);
    l.xq = align_up(l.slots + (gate_up ? static_cast<size_t>(grid + 1) * kMtokSlotBytes : 0), 256);
    l.xs = align_up(l.xq + (gate_up ? KX * kMtokXGroupBytes : 0), 256);
    l.part = align_up(l.xs + (gate_up ? sizeof(float) * KX * 16 : 0), 256);
    l.end = align_up(l.part + (gate_up ? 0 : sizeof(float) * rows_in * static_cast<size_t>(rows_out) * KX), 256);
    return l;
}

// The standalone calls run the multi-token kernel where it takes them: at
// most 16 tokens (gate_up; down: at most 16 rows per expert, as the call
// requires of every plan), gate_up's K up to 6144, down's N up to 6144 and a
// multiple of 256 (down's K is free: it counts no K group of a, but its
// partials, rows x N x K/128 floats, stay within 256 MiB), and a plan that
// fits the kernel's shared copy of it.  The kernel checks the plan as the
// persistent engine does.
constexpr int kMtokMaxPairs = MOEQ_MAX_TOKENS * (MOEQ_MAX_TOPK + 1);
constexpr int kMtokMaxSlots = MOEQ_MAX_TOKENS * MOEQ_MAX_TOPK;
bool gateup_mtok_ok(int M, int H, int max_uniq, int max_pairs) {
    return mtok_kernel_enabled() && M <= MOEQ_MAX_TOKENS && H <= kTokenMaxH && max_pairs <= kMtokMaxPairs &&
           max_uniq <= kMtokMaxSlots;
}
bool down_mtok_ok(int K, int N, int max_uniq, int max_pairs) {
    const size_t part_bytes = sizeof(float) * static_cast<size_t>(max_pairs) * N * (K / 128);
    return mtok_kernel_enabled() && N % 256 == 0 && N <= kTokenMaxH && K <= MOEQ_MAX_K &&
           max_pairs <= kMtokMaxPairs && max_uniq <= kMtokMaxSlots && part_bytes <= (size_t{256} << 20);
}

// The arguments of the multi-token kernel's standalone modes.
MtokArgs mtok_gemm_args(bool gate_up, const void* x, int x_f32, int rows, int K, int rows_out, const uint8_t* w,
                        const float* sw, const int32_t* uniq, const int32_t* offs, const int32_t* pair_tok,
                        const int32_t* n_uniq, int n_experts, int max_uniq, int max_pairs, float* out,
                        uint8_t* q_opt, float* s_opt, void* ws, const MtokGemmWs& l) {
    char* base = static_cast<char*>(ws);
    MtokArgs t = {};
    t.x = x;
    t.x_f32 = x_f32;
    t.x_ld = K;
    t.M = rows;
    t.KX = K / 128;
    t.top_k = 0;
    t.E_routed = 0;
    t.n_experts = n_experts;
    t.max_uniq = max_uniq;
    t.max_pairs = max_pairs;
    t.plan.n_uniq = const_cast<int32_t*>(n_uniq);
    t.plan.uniq = const_cast<int32_t*>(uniq);
    t.plan.offs = const_cast<int32_t*>(offs);
    t.plan.pair_tok = const_cast<int32_t*>(pair_tok);
    if (gate_up) {
        // x [M, H]; h [pairs, I]: H = K, I = rows_out / 2
        t.mode = kMtokGateUp;
        t.H = K;
        t.I = rows_out / 2;
        t.KB = K / 128;
        t.RB = rows_out / 256;
        t.GS = t.KB;
        t.NU = 0;
        t.ntmax = rows;
        t.w_gu = w;
        t.s_gu = sw;
        t.h = out;
    } else {
        // a [pairs, K]; y [pairs, N]: N = rows_out
        t.mode = kMtokDown;
        t.H = rows_out;
        t.I = K;
        t.KB = rows_out / 128;
        t.RB = K / 128;
        t.GS = 0;
        t.NU = rows_out / 256;
        t.ntmax = rows < MOEQ_MAX_TOKENS ? rows : MOEQ_MAX_TOKENS;
        t.w_d = w;
        t.s_d = sw;
        t.out_f32 = out;
    }
    t.q_x = q_opt;
    t.s_x = s_opt;
    t.status = reinterpret_cast<int*>(base + kOffStatus);
    t.cnt = reinterpret_cast<int*>(base + l.cnt);
    t.slots = gate_up ? reinterpret_cast<uint8_t*>(base + l.slots) : nullptr;
    t.xq = reinterpret_cast<uint8_t*>(base + l.xq);
    t.xs = reinterpret_cast<float*>(base + l.xs);
    t.part = gate_up ? nullptr : reinterpret_cast<float*>(base + l.part);
    return t;
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

void fill_ws(StreamArgs& a, void* ws, const StreamWs& l, int grid) {
    char* base = static_cast<char*>(ws);
    a.partial_list_floats = stream_partials_floats(grid);
    a.status = reinterpret_cast<int*>(base + kOffStatus);
    a.epoch = reinterpret_cast<int*>(base + kOffEpoch);
    a.done = reinterpret_cast<int*>(base + kOffDone);
    a.a_cnt = reinterpret_cast<int*>(base + kOffACnt);
    a.dc_cnt = reinterpret_cast<int*>(base + kOffDcCnt);
    for (int k = 0; k < 2; ++k) {
        a.op[k].aq = reinterpret_cast<float*>(base + l.aq[k]);
        a.op[k].as = reinterpret_cast<float*>(base + l.as[k]);
    }
    for (int i = 0; i < kMaxLists; ++i) a.tickets[i] = reinterpret_cast<int*>(base + l.tickets[i]);
    a.partials = reinterpret_cast<float*>(base + l.partials);
    a.h_ready = reinterpret_cast<int*>(base + l.h_ready);
    a.comb = reinterpret_cast<int*>(base + l.comb);
}

// ------------------------------------------------------------------ layer
// One moeq_moe_layer call's arguments.
struct LayerCall {
    const void* x;
    const float* logits;
    int M, H, I, E_routed, top_k;
    const uint8_t* w_gu;
    const float* s_gu;
    const uint8_t* w_d;
    const float* s_d;
    void* out;
    float* out_f32;   // a tensor-parallel shard's fp32 partial instead of out
    const moeq_route_plan* plan_opt;
    float* h_opt;
    float* y_opt;
    uint8_t* q_x_opt;
    float* s_x_opt;
    uint8_t* q_h_opt;
    float* s_h_opt;
    void* const* events_opt;
    void* ws;
    size_t ws_bytes;
};

// The fused one-token and multi-token kernels serve a call (the persistent
// engine serves the rest).
bool mtok_path(const LayerCall& c) {
    return c.M >= mtok_min_tokens() && !c.y_opt && mtok_kernel_enabled() && c.top_k <= kMtokMaxTopK &&
           c.H <= kTokenMaxH && c.H % 256 == 0;
}
bool token_path(const LayerCall& c) {
    return c.M == 1 && !mtok_path(c) && (c.out_f32 || c.M < mma_min_tokens()) && !c.y_opt &&
           token_kernel_enabled() && c.top_k <= kTokenMaxTopK && c.H <= kTokenMaxH && c.H % 256 == 0;
}

// Host-side checks of one layer call (nothing is launched).
moeq_status layer_check(const LayerCall& c, const DeviceInfo& dev) {
    void* const dst = c.out_f32 ? static_cast<void*>(c.out_f32) : c.out;
    if (!c.x || !c.logits || !c.w_gu || !c.s_gu || !c.w_d || !c.s_d || !dst) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(c.x) || !aligned16(c.w_gu) || !aligned16(c.w_d) || !aligned16(dst) || !aligned4(c.s_gu) ||
        !aligned4(c.s_d))
        return MOEQ_ERR_INVALID_ARG;
    if ((c.h_opt && !aligned16(c.h_opt)) || (c.y_opt && !aligned16(c.y_opt))) return MOEQ_ERR_INVALID_ARG;
    if ((c.q_x_opt == nullptr) != (c.s_x_opt == nullptr) || (c.q_h_opt == nullptr) != (c.s_h_opt == nullptr))
        return MOEQ_ERR_INVALID_ARG;
    if ((c.q_x_opt && (!aligned16(c.q_x_opt) || !aligned4(c.s_x_opt))) ||
        (c.q_h_opt && (!aligned16(c.q_h_opt) || !aligned4(c.s_h_opt))))
        return MOEQ_ERR_INVALID_ARG;
    if (c.plan_opt && !plan_ok(c.plan_opt)) return MOEQ_ERR_INVALID_ARG;
    if (!route_args_ok(c.M, c.E_routed, c.top_k)) return MOEQ_ERR_INVALID_ARG;
    const int H = c.H, I = c.I;
    if (H <= 0 || I <= 0 || H % 128 || I % 128 || H > MOEQ_MAX_K || I > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    // an fp32 partial comes from the fused kernels only
    if (c.out_f32 && !token_path(c) && !mtok_path(c)) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const LayerWs l = layer_ws_layout(c.M, H, I, c.E_routed, c.top_k, dev.sms);
    if (!c.ws || !aligned16(c.ws) || c.ws_bytes < l.s.end) return MOEQ_ERR_WORKSPACE;
    return MOEQ_OK;
}

// The launch of one checked layer call.  route_early: the logits are not
// written by the kernel ahead on the stream (the one-token kernel may then
// route before it waits for that kernel); allow_pdl: the weights are not
// either.
moeq_status layer_launch(const LayerCall& c, const DeviceInfo& dev, bool route_early, bool allow_pdl,
                         cudaStream_t st) {
    const void* x = c.x;
    const float* logits = c.logits;
    const int M = c.M, H = c.H, I = c.I, E_routed = c.E_routed, top_k = c.top_k;
    const uint8_t *w_gu = c.w_gu, *w_d = c.w_d;
    const float *s_gu = c.s_gu, *s_d = c.s_d;
    void* out = c.out;
    const moeq_route_plan* plan_opt = c.plan_opt;
    float *h_opt = c.h_opt, *y_opt = c.y_opt, *s_x_opt = c.s_x_opt, *s_h_opt = c.s_h_opt;
    uint8_t *q_x_opt = c.q_x_opt, *q_h_opt = c.q_h_opt;
    void* const* events_opt = c.events_opt;
    void* ws = c.ws;
    const LayerWs l = layer_ws_layout(M, H, I, E_routed, top_k, dev.sms);
    char* base = static_cast<char*>(ws);
    moeq_route_plan plan;
    if (plan_opt)
        plan = *plan_opt;
    else
        moeq_route_plan_carve(base + l.plan, l.h - l.plan, M, E_routed, top_k, &plan);
    float* h = h_opt ? h_opt : reinterpret_cast<float*>(base + l.h);
    float* y = y_opt ? y_opt : reinterpret_cast<float*>(base + l.y);
    const int mu = moeq_max_uniq(M, E_routed, top_k), mp = moeq_max_pairs(M, top_k);

    // One token on the CUDA cores (no per-pair y asked for): the one-token
    // kernel, which needs no co-resident grid and no cross-CTA wait.
    if (token_path(c)) {
        TokenArgs t = {};
        t.x = static_cast<const __nv_bfloat16*>(x);
        t.logits = logits;
        t.H = H;
        t.I = I;
        t.KB = H / 128;
        t.RB = I / 128;
        t.E_routed = E_routed;
        t.top_k = top_k;
        t.ncols = (top_k + 1) * (I / 128);
        t.w_gu = w_gu;
        t.s_gu = s_gu;
        t.w_d = w_d;
        t.s_d = s_d;
        t.out = static_cast<__nv_bfloat16*>(out);
        t.out_f32 = c.out_f32;
        t.plan = plan;
        t.h = h;
        t.q_x = q_x_opt;
        t.s_x = s_x_opt;
        t.q_h = q_h_opt;
        t.s_h = s_h_opt;
        t.status = reinterpret_cast<int*>(base + kOffStatus);
        t.tickets = reinterpret_cast<int*>(base + l.tok_tickets);
        t.gq = t.tickets + H / 256;
        t.part = reinterpret_cast<float*>(base + l.dc);
        t.route_early = route_early ? 1 : 0;
        if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[0]), st) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        if (launch_token(t, dev.sms, pdl_enabled() && allow_pdl, st) != cudaSuccess) return MOEQ_ERR_CUDA;
        if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[1]), st) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        return MOEQ_OK;
    }

    // 2..16 tokens (no per-pair y asked for): the multi-token kernel, on the
    // tensor cores, with no cross-CTA wait inside its streams.
    if (mtok_path(c)) {
        MtokArgs t = {};
        t.x = static_cast<const __nv_bfloat16*>(x);
        t.logits = logits;
        t.M = M;
        t.H = H;
        t.I = I;
        t.KB = H / 128;
        t.RB = I / 128;
        t.E_routed = E_routed;
        t.top_k = top_k;
        t.w_gu = w_gu;
        t.s_gu = s_gu;
        t.w_d = w_d;
        t.s_d = s_d;
        t.out = static_cast<__nv_bfloat16*>(out);
        t.out_f32 = c.out_f32;
        t.plan = plan;
        t.h = h_opt;   // h only when asked for (the kernel needs none of its own)
        t.q_x = q_x_opt;
        t.s_x = s_x_opt;
        t.q_h = q_h_opt;
        t.s_h = s_h_opt;
        t.status = reinterpret_cast<int*>(base + kOffStatus);
        t.cnt = reinterpret_cast<int*>(base + l.mt_cnt);
        t.slots = reinterpret_cast<uint8_t*>(base + l.mt_slots);
        t.xq = reinterpret_cast<uint8_t*>(base + l.mt_xq);
        t.xs = reinterpret_cast<float*>(base + l.mt_xs);
        t.part = reinterpret_cast<float*>(base + l.mt_part);
        t.route_early = route_early ? 1 : 0;
        t.mode = kMtokLayer;
        t.GS = t.KB;
        t.NU = t.KB / 2;
        t.KX = t.KB;
        t.x_ld = H;
        t.x_f32 = 0;
        t.ntmax = M;
        if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[0]), st) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        if (launch_mtok(t, dev.sms, pdl_enabled() && allow_pdl, st) != cudaSuccess) return MOEQ_ERR_CUDA;
        if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[1]), st) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        return MOEQ_OK;
    }

    StreamArgs a = {};
    Operand& g = a.op[kKindGU];
    g.w = w_gu;
    g.sw = s_gu;
    g.K = H;
    g.KB = H / 128;
    g.NB = 2 * I / 128;
    g.RB = I / 128;
    g.a = x;
    g.a_f32 = 0;
    g.rows_a = M;
    g.out = h;
    g.out_ld = I;
    g.quant_input = 1;
    g.qdump = q_x_opt;
    g.sdump = s_x_opt;
    Operand& d = a.op[kKindDN];
    d.w = w_d;
    d.sw = s_d;
    d.K = I;
    d.KB = I / 128;
    d.NB = H / 128;
    d.RB = H / 128;
    d.a = h;
    d.a_f32 = 1;
    d.rows_a = mp;
    d.out = y;
    d.out_ld = H;
    a.mma = M >= mma_min_tokens();
    // One token on the CUDA cores (unless y is asked for): down by K group.
    // The CTA that finished gate_up row block kb of a pair goes on with
    // down's tiles (nb, kb) for every nb, so no CTA waits for another's h;
    // a combine over the K groups' sums ends the launch.
    const int dc_cols = (H + dev.sms - 1) / dev.sms;
    a.dc = M == 1 && !a.mma && !y_opt && (H / 128) % 2 == 0 && mp * dc_cols <= kDcCombineFloats;
    // One gate_up block per CTA (whole blocks, as the engine deals them):
    // each CTA quantises all of x for itself, and down by K group takes the
    // h group the CTA finished itself from shared memory.
    const bool one_block = dp_blocks_per_cta_host(static_cast<long long>(mu) * (I / 128), dev.sms) == 1;
    a.xloc = M == 1 && !a.mma && H <= kXLocalMaxK && one_block && !q_x_opt;
    a.hloc = a.dc && one_block;
    a.swb = a.xloc && aligned16(s_gu) && (H / 128) % 4 == 0;
    if (M == 1 || M >= mma_min_tokens()) {
        // one token, or the tcgen05 path (where a stage costs the same for 1
        // or 16 tokens): the routed experts' blocks and the shared expert's
        // cost the same, so each kind is one list, dealt out in whole row
        // blocks where they nearly fill the grid
        a.n_lists = 2;
        a.list_kind[0] = kKindGU;
        a.list_src[0] = kSrcLayer;
        a.list_kind[1] = a.dc ? kKindDC : kKindDN;
        a.list_src[1] = kSrcLayer;
    } else {
        // the shared expert serves all M tokens (M times a routed block's
        // arithmetic): its own lists spread it over every CTA; the routed
        // experts come in two halves so that down of the first hides the
        // finish of the second's h
        a.n_lists = 6;
        const int kinds[6] = {kKindGU, kKindGU, kKindGU, kKindDN, kKindDN, kKindDN};
        const int srcs[6] = {kSrcShared, kSrcPlanRoutedA, kSrcPlanRoutedB, kSrcShared, kSrcPlanRoutedA, kSrcPlanRoutedB};
        for (int i = 0; i < 6; ++i) {
            a.list_kind[i] = kinds[i];
            a.list_src[i] = srcs[i];
        }
    }
    a.n_uniq = plan.n_uniq;
    a.uniq = plan.uniq;
    a.offs = plan.offs;
    a.pair_tok = plan.pair_tok;
    a.pair_of = plan.pair_of;
    a.topk_w = plan.topk_w;
    a.n_experts = E_routed + 1;
    a.max_uniq = mu;
    a.max_pairs = mp;
    a.max_ntok = M;
    a.shared_id = E_routed;
    a.shared_p0 = M * top_k;
    a.M = M;
    a.fused_route = 1;
    a.logits = logits;
    a.E_routed = E_routed;
    a.top_k = top_k;
    a.plan = plan;
    a.fused_combine = 1;
    a.out_bf16 = static_cast<__nv_bfloat16*>(out);
    a.h_to_dn = 1;
    a.qh_dump = q_h_opt;
    a.sh_dump = s_h_opt;
    fill_ws(a, ws, l.s, dev.sms);
    a.dc_part = reinterpret_cast<float*>(base + l.dc);

    if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[0]), st) != cudaSuccess)
        return MOEQ_ERR_CUDA;
    if (launch_stream(a, dev.sms, true, st) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (events_opt && cudaEventRecord(static_cast<cudaEvent_t>(events_opt[1]), st) != cudaSuccess)
        return MOEQ_ERR_CUDA;
    return MOEQ_OK;
}

// ------------------------------------------------------------------ stack
// A stack's workspace: one layer workspace at offset 0 (its header holds the
// status word, so moeq_read_device_status reads a stack's workspace as it
// reads a layer's), then one route plan per layer.
struct StackWs {
    size_t layer_bytes, plan0, plan_stride, end;
};

StackWs stack_ws_layout(int L, size_t layer_bytes, int M, int E_routed, int top_k) {
    StackWs w;
    w.layer_bytes = layer_bytes;
    w.plan0 = align_up(layer_bytes, 256);
    w.plan_stride = align_up(moeq_route_plan_bytes(M, E_routed, top_k), 256);
    w.end = w.plan0 + static_cast<size_t>(L) * w.plan_stride;
    return w;
}

// Instantiated stack graphs, keyed by the device and every argument of the
// call that captured them; the least recently used is dropped beyond
// kStackGraphs (a graph that is still running is freed when it completes).
struct StackGraph {
    std::vector<uintptr_t> key;
    cudaGraphExec_t exec;
    unsigned long long used;
};
constexpr size_t kStackGraphs = 16;
std::mutex g_stack_mu;
std::vector<StackGraph> g_stack_graphs;
unsigned long long g_stack_clock = 0;

// A non-blocking stream per device on which the library captures (capture
// issues no work, so the caller's stream, which may be the legacy default
// stream, never needs to be put into capture mode).
cudaStream_t capture_stream(int dev) {
    static std::vector<cudaStream_t> streams;
    if (static_cast<int>(streams.size()) <= dev) streams.resize(dev + 1, nullptr);
    if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        streams[dev] = nullptr;
    }
    return streams[dev];
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
    return layer_ws_layout(M, H, I, E, top_k, dev.sms).s.end;
}

size_t moeq_layer_ws_count_offset(int M, int H, int I, int n_experts_incl_shared, int top_k, int which) {
    const int E = n_experts_incl_shared - 1;
    if (!moeq_workspace_size(M, H, I, n_experts_incl_shared, top_k) || M < mtok_min_tokens()) return 0;
    const size_t base = layer_ws_layout(M, H, I, E, top_k, current_device().sms).mt_cnt;
    switch (which) {
    case 0: return base + sizeof(int) * kMtokX;   // K group 0 of x: quantised groups in
    case 1: return base + sizeof(int) * kMtokU;   // output unit 0: down partials stored
    default: return 0;
    }
}

size_t moeq_gemm_ws_count_offset(int rows_out, int K, int rows_in, int max_uniq, int is_gate_up, int which) {
    if (!moeq_gemm_workspace_size(rows_out, K, rows_in, max_uniq, is_gate_up)) return 0;
    const bool mt = is_gate_up ? gateup_mtok_ok(rows_in, K, max_uniq, rows_in * (MOEQ_MAX_TOPK + 1))
                               : down_mtok_ok(K, rows_out, max_uniq, rows_in);
    if (!mt || (which == 1 && is_gate_up)) return 0;
    if (which == 0 && !is_gate_up) return 0;   // down alone quantises a per piece: no count
    const DeviceInfo dev = current_device();
    const size_t end = gemm_ws_layout(is_gate_up ? 0 : 1, rows_out / 128, K, rows_in, max_uniq, dev.sms).end;
    const size_t base = mtok_gemm_ws(is_gate_up != 0, is_gate_up ? 2 * rows_out : rows_out, K, rows_in, dev.sms, end).cnt;
    switch (which) {
    case 0: return base + sizeof(int) * kMtokX;
    case 1: return base + sizeof(int) * kMtokU;
    default: return 0;
    }
}

size_t moeq_gemm_workspace_size(int rows_out, int K, int rows_in, int max_uniq, int is_gate_up) {
    if (rows_out <= 0 || rows_out % 128 || max_uniq < 1 || K <= 0 || K % 128 || K > MOEQ_MAX_K || rows_in < 1)
        return 0;
    const DeviceInfo dev = current_device();
    if (!dev.sms) return 0;
    const size_t end = gemm_ws_layout(is_gate_up ? 0 : 1, rows_out / 128, K, rows_in, max_uniq, dev.sms).end;
    // room for the multi-token kernel where it may serve the call
    if (is_gate_up ? gateup_mtok_ok(rows_in, K, max_uniq, rows_in * (MOEQ_MAX_TOPK + 1))
                   : down_mtok_ok(K, rows_out, max_uniq, rows_in))
        return mtok_gemm_ws(is_gate_up != 0, is_gate_up ? 2 * rows_out : rows_out, K, rows_in, dev.sms, end).end;
    return end;
}

moeq_status moeq_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < kHeader || !aligned16(ws)) return MOEQ_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream)));
}

moeq_status moeq_read_device_status(const void* ws, size_t ws_bytes, int* device_status) {
    if (!ws || ws_bytes < kHeader || !device_status) return MOEQ_ERR_INVALID_ARG;
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
    g_weight_write_stream.store(stream_key(stream));
    return cuda_status(launch_quant_weight(w, E, N, K, q, s, as_stream(stream)));
}

moeq_status moeq_pack_weight(const uint8_t* q_rows, int E, int N, int K, uint8_t* q_tiles, void* stream) {
    if (!q_rows || !q_tiles || !aligned16(q_rows) || !aligned16(q_tiles)) return MOEQ_ERR_INVALID_ARG;
    if (E < 1 || E > 65535) return MOEQ_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || N % 128 || K % 128 || N / 128 > 65535 || K / 128 > 65535)
        return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    g_weight_write_stream.store(stream_key(stream));
    return cuda_status(launch_pack_weight(q_rows, E, N, K, q_tiles, as_stream(stream)));
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
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const StreamWs wl = gemm_ws_layout(0, I / 128, H, M, max_uniq, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < wl.end) return MOEQ_ERR_WORKSPACE;
    if (gateup_mtok_ok(M, H, max_uniq, max_pairs)) {
        const MtokGemmWs ml = mtok_gemm_ws(true, 2 * I, H, M, dev.sms, wl.end);
        if (ws_bytes < ml.end) return MOEQ_ERR_WORKSPACE;
        const MtokArgs t = mtok_gemm_args(true, x, x_dtype == MOEQ_F32, M, H, 2 * I, w_gu, s_gu, uniq, offs, pair_tok,
                                          n_uniq_dev, n_experts, max_uniq, max_pairs, h, q_x_opt, s_x_opt, ws, ml);
        uintptr_t key = stream_key(stream);
        const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(key, 0);
        return cuda_status(launch_mtok(t, gemm_grid(dev.sms), pdl_enabled() && !after_weight_write, as_stream(stream)));
    }
    StreamArgs a = {};
    Operand& o = a.op[kKindGU];
    o.quant_input = 1;
    o.w = w_gu;
    o.sw = s_gu;
    o.K = H;
    o.KB = H / 128;
    o.NB = 2 * I / 128;
    o.RB = I / 128;
    o.a = x;
    o.a_f32 = x_dtype == MOEQ_F32;
    o.rows_a = M;
    o.out = h;
    o.out_ld = I;
    o.qdump = q_x_opt;
    o.sdump = s_x_opt;
    a.n_lists = 1;
    a.list_kind[0] = kKindGU;
    a.list_src[0] = kSrcPlanAll;
    a.n_uniq = n_uniq_dev;
    a.uniq = uniq;
    a.offs = offs;
    a.pair_tok = pair_tok;
    a.n_experts = n_experts;
    a.max_uniq = max_uniq;
    a.max_pairs = max_pairs;
    a.max_ntok = M;   // the pairs of one expert are distinct tokens
    a.mma = a.max_ntok >= gemm_mma_min_tokens();
    a.M = M;
    fill_ws(a, ws, wl, dev.sms);
    return cuda_status(launch_stream(a, gemm_grid(dev.sms), true, as_stream(stream)));
}

moeq_status moeq_expert_gemm_down(const void* a_in, moeq_dtype a_dtype, int K, int N, const uint8_t* w_d,
                                  const float* s_d, int n_experts, const int32_t* uniq, const int32_t* offs,
                                  const int32_t* n_uniq_dev, int max_uniq, int max_pairs, float* y, uint8_t* q_a_opt,
                                  float* s_a_opt, void* ws, size_t ws_bytes, void* stream) {
    if (!a_in || !w_d || !s_d || !uniq || !offs || !n_uniq_dev || !y) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(a_in) || !aligned16(w_d) || !aligned16(y) || !aligned4(s_d)) return MOEQ_ERR_INVALID_ARG;
    if ((q_a_opt == nullptr) != (s_a_opt == nullptr)) return MOEQ_ERR_INVALID_ARG;
    if (q_a_opt && !aligned16(q_a_opt)) return MOEQ_ERR_INVALID_ARG;
    if (a_dtype != MOEQ_BF16 && a_dtype != MOEQ_F32) return MOEQ_ERR_INVALID_ARG;
    if (n_experts < 1 || max_uniq < 1 || max_pairs < 1) return MOEQ_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || K % 128 || N % 128 || K > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const StreamWs wl = gemm_ws_layout(1, N / 128, K, max_pairs, max_uniq, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < wl.end) return MOEQ_ERR_WORKSPACE;
    if (down_mtok_ok(K, N, max_uniq, max_pairs)) {
        const MtokGemmWs ml = mtok_gemm_ws(false, N, K, max_pairs, dev.sms, wl.end);
        if (ws_bytes < ml.end) return MOEQ_ERR_WORKSPACE;
        const MtokArgs t = mtok_gemm_args(false, a_in, a_dtype == MOEQ_F32, max_pairs, K, N, w_d, s_d, uniq, offs,
                                          nullptr, n_uniq_dev, n_experts, max_uniq, max_pairs, y, q_a_opt, s_a_opt, ws,
                                          ml);
        uintptr_t key = stream_key(stream);
        const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(key, 0);
        return cuda_status(launch_mtok(t, gemm_grid(dev.sms), pdl_enabled() && !after_weight_write, as_stream(stream)));
    }
    StreamArgs a = {};
    Operand& o = a.op[kKindDN];
    o.quant_input = 1;
    o.w = w_d;
    o.sw = s_d;
    o.K = K;
    o.KB = K / 128;
    o.NB = N / 128;
    o.RB = N / 128;
    o.a = a_in;
    o.a_f32 = a_dtype == MOEQ_F32;
    o.rows_a = max_pairs;
    o.out = y;
    o.out_ld = N;
    o.qdump = q_a_opt;
    o.sdump = s_a_opt;
    a.n_lists = 1;
    a.list_kind[0] = kKindDN;
    a.list_src[0] = kSrcPlanAll;
    a.n_uniq = n_uniq_dev;
    a.uniq = uniq;
    a.offs = offs;
    a.n_experts = n_experts;
    a.max_uniq = max_uniq;
    a.max_pairs = max_pairs;
    a.max_ntok = max_pairs < MOEQ_MAX_TOKENS ? max_pairs : MOEQ_MAX_TOKENS;
    a.mma = a.max_ntok >= gemm_mma_min_tokens();
    fill_ws(a, ws, wl, dev.sms);
    return cuda_status(launch_stream(a, gemm_grid(dev.sms), true, as_stream(stream)));
}

// ------------------------------------------------------------------ no-alloc down
// moeq_expert_gemm_down without a caller workspace, for callers that cannot
// lend one and cannot allocate on their path: a plain C host issuing one
// projection with no device buffer of its own to spare, or an engine whose
// device memory is wholly committed to its own pools, where cudaMalloc (which
// may synchronise the device) is not allowed in the decode step.  Its scratch
// is this file's static device array; a launch needs at most
// kNoAllocScratchBytes of it (header, decoded activations and scales,
// tickets, split-K partials), larger problems are refused.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of this device's copy of the scratch, looked up once per
// device (with that device current) and cached.
static moeq_status noalloc_scratch(void** out) {
    static std::mutex mu;
    static std::vector<void*> addr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOEQ_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(addr.size()) <= dev) addr.resize(dev + 1, nullptr);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MOEQ_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return MOEQ_OK;
}

moeq_status moeq_expert_gemm_down_noalloc(const void* a_in, moeq_dtype a_dtype, int K, int N, const uint8_t* w_d,
                                          const float* s_d, int n_experts, const int32_t* uniq, const int32_t* offs,
                                          const int32_t* n_uniq_dev, int max_uniq, int max_pairs, float* y,
                                          uint8_t* q_a_opt, float* s_a_opt, int32_t* device_status_opt,
                                          void* stream) {
    if (!a_in || !w_d || !s_d || !uniq || !offs || !n_uniq_dev || !y) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(a_in) || !aligned16(w_d) || !aligned16(y) || !aligned4(s_d)) return MOEQ_ERR_INVALID_ARG;
    if ((q_a_opt == nullptr) != (s_a_opt == nullptr)) return MOEQ_ERR_INVALID_ARG;
    if (q_a_opt && !aligned16(q_a_opt)) return MOEQ_ERR_INVALID_ARG;
    if (device_status_opt && !aligned4(device_status_opt)) return MOEQ_ERR_INVALID_ARG;
    if (a_dtype != MOEQ_BF16 && a_dtype != MOEQ_F32) return MOEQ_ERR_INVALID_ARG;
    if (n_experts < 1 || max_uniq < 1 || max_pairs < 1) return MOEQ_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || K % 128 || N % 128 || K > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    void* ws = nullptr;
    cudaStream_t cs = as_stream(stream);
    const MtokGemmWs ml = mtok_gemm_ws(false, N, K, max_pairs, dev.sms, kHeader);
    if (down_mtok_ok(K, N, max_uniq, max_pairs) && ml.end <= kNoAllocScratchBytes) {
        // the path moeq_expert_gemm_down takes: the multi-token kernel, its
        // areas right after the header, its counts zeroed on the stream
        // first (when they do not fit the scratch, the engine below)
        const moeq_status st = noalloc_scratch(&ws);
        if (st != MOEQ_OK) return st;
        if (cudaMemsetAsync(ws, 0, kHeader, cs) != cudaSuccess ||
            cudaMemsetAsync(static_cast<char*>(ws) + ml.cnt, 0, ml.slots - ml.cnt, cs) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        const MtokArgs t = mtok_gemm_args(false, a_in, a_dtype == MOEQ_F32, max_pairs, K, N, w_d, s_d, uniq, offs,
                                          nullptr, n_uniq_dev, n_experts, max_uniq, max_pairs, y, q_a_opt, s_a_opt, ws,
                                          ml);
        if (launch_mtok(t, gemm_grid(dev.sms), false, cs) != cudaSuccess) return MOEQ_ERR_CUDA;
        if (device_status_opt &&
            cudaMemcpyAsync(device_status_opt, static_cast<char*>(ws) + kOffStatus, sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
            return MOEQ_ERR_CUDA;
        return MOEQ_OK;
    }
    const StreamWs wl = gemm_ws_layout(1, N / 128, K, max_pairs, max_uniq, dev.sms);
    if (wl.end > kNoAllocScratchBytes) return MOEQ_ERR_WORKSPACE;   // beyond the static maximum
    const moeq_status st = noalloc_scratch(&ws);
    if (st != MOEQ_OK) return st;
    // The counters (header: status word, epoch, input-quantisation count;
    // the split-K tickets) must be zero when a launch starts: zero them on
    // the stream first.  The activation buffers between them need no zeroing.
    if (cudaMemsetAsync(ws, 0, kHeader, cs) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (cudaMemsetAsync(static_cast<char*>(ws) + wl.tickets[0], 0, wl.partials - wl.tickets[0], cs) != cudaSuccess)
        return MOEQ_ERR_CUDA;
    StreamArgs a = {};
    Operand& o = a.op[kKindDN];
    o.quant_input = 1;
    o.w = w_d;
    o.sw = s_d;
    o.K = K;
    o.KB = K / 128;
    o.NB = N / 128;
    o.RB = N / 128;
    o.a = a_in;
    o.a_f32 = a_dtype == MOEQ_F32;
    o.rows_a = max_pairs;
    o.out = y;
    o.out_ld = N;
    o.qdump = q_a_opt;
    o.sdump = s_a_opt;
    a.n_lists = 1;
    a.list_kind[0] = kKindDN;
    a.list_src[0] = kSrcPlanAll;
    a.n_uniq = n_uniq_dev;
    a.uniq = uniq;
    a.offs = offs;
    a.n_experts = n_experts;
    a.max_uniq = max_uniq;
    a.max_pairs = max_pairs;
    a.max_ntok = max_pairs < MOEQ_MAX_TOKENS ? max_pairs : MOEQ_MAX_TOKENS;
    a.mma = a.max_ntok >= gemm_mma_min_tokens();   // the path moeq_expert_gemm_down takes
    fill_ws(a, ws, wl, dev.sms);
    if (launch_stream(a, dev.sms, true, cs) != cudaSuccess) return MOEQ_ERR_CUDA;
    if (device_status_opt &&
        cudaMemcpyAsync(device_status_opt, static_cast<char*>(ws) + kOffStatus, sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return MOEQ_ERR_CUDA;
    return MOEQ_OK;
}

// ------------------------------------------------------------------ dense FFN
// M tokens through one dense FFN: the multi-token kernel with no routing
// (top_k = 0: the one expert serves every token), or, for one token with
// MOEQ_MTOK_MIN_TOKENS above 1, the one-token kernel with no routing.
// Workspace: header, h [M, I], then the multi-token kernel's areas (counts,
// split-column slots, x's codes and scales, partials [M][H/256][1][I/128]
// [256]) and the one-token kernel's (partials [I/128, H], arrival counts).
struct DenseWs {
    size_t h, mt_cnt, mt_slots, mt_xq, mt_xs, mt_part, part, tickets, end;
};

DenseWs dense_ws_layout(int M, int H, int I, int grid) {
    DenseWs l;
    l.h = kHeader;
    l.mt_cnt = align_up(l.h + sizeof(float) * static_cast<size_t>(M) * I, 256);
    l.mt_slots = align_up(l.mt_cnt + sizeof(int) * (kMtokFlags + grid + 1), 256);
    l.mt_xq = align_up(l.mt_slots + static_cast<size_t>(grid + 1) * kMtokSlotBytes, 256);
    l.mt_xs = align_up(l.mt_xq + static_cast<size_t>(H / 128) * kMtokXGroupBytes, 256);
    l.mt_part = align_up(l.mt_xs + sizeof(float) * static_cast<size_t>(H / 128) * 16, 256);
    l.part = align_up(l.mt_part + sizeof(float) * static_cast<size_t>(M) * H * (I / 128), 256);
    l.tickets = align_up(l.part + (M == 1 ? sizeof(float) * static_cast<size_t>(I / 128) * H : 0), 256);
    l.end = align_up(l.tickets + sizeof(int) * (static_cast<size_t>(H / 256) + kGqUnits), 256);
    return l;
}

bool dense_shape_ok(int M, int H, int I) {
    return M >= 1 && M <= MOEQ_MAX_TOKENS && H > 0 && I > 0 && H % 256 == 0 && I % 128 == 0 && H <= kTokenMaxH &&
           I <= MOEQ_MAX_K && (M == 1 || (mtok_kernel_enabled() && M >= mtok_min_tokens()));
}

size_t moeq_dense_ffn_workspace_size(int M, int H, int I) {
    if (!dense_shape_ok(M, H, I)) return 0;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return 0;
    return dense_ws_layout(M, H, I, dev.sms).end;
}

moeq_status moeq_dense_ffn(const void* x, int M, int H, int I, const uint8_t* w_gu, const float* s_gu,
                           const uint8_t* w_d, const float* s_d, void* out, float* h_opt, uint8_t* q_x_opt,
                           float* s_x_opt, uint8_t* q_h_opt, float* s_h_opt, void* ws, size_t ws_bytes,
                           void* stream) {
    if (!x || !w_gu || !s_gu || !w_d || !s_d || !out) return MOEQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gu) || !aligned16(w_d) || !aligned16(out) || !aligned4(s_gu) || !aligned4(s_d))
        return MOEQ_ERR_INVALID_ARG;
    if (h_opt && !aligned16(h_opt)) return MOEQ_ERR_INVALID_ARG;
    if ((q_x_opt == nullptr) != (s_x_opt == nullptr) || (q_h_opt == nullptr) != (s_h_opt == nullptr))
        return MOEQ_ERR_INVALID_ARG;
    if ((q_x_opt && (!aligned16(q_x_opt) || !aligned4(s_x_opt))) || (q_h_opt && (!aligned16(q_h_opt) || !aligned4(s_h_opt))))
        return MOEQ_ERR_INVALID_ARG;
    if (M < 1 || M > MOEQ_MAX_TOKENS) return MOEQ_ERR_INVALID_ARG;
    if (!dense_shape_ok(M, H, I)) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const DenseWs l = dense_ws_layout(M, H, I, dev.sms);
    if (!ws || !aligned16(ws) || ws_bytes < l.end) return MOEQ_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    float* h = h_opt ? h_opt : reinterpret_cast<float*>(base + l.h);
    uintptr_t key = stream_key(stream);
    const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(key, 0);
    const bool pdl = pdl_enabled() && !after_weight_write;
    if (mtok_kernel_enabled() && M >= mtok_min_tokens()) {
        MtokArgs t = {};
        t.x = static_cast<const __nv_bfloat16*>(x);
        t.logits = nullptr;
        t.M = M;
        t.H = H;
        t.I = I;
        t.KB = H / 128;
        t.RB = I / 128;
        t.E_routed = 0;   // expert 0 is the one expert
        t.top_k = 0;
        t.w_gu = w_gu;
        t.s_gu = s_gu;
        t.w_d = w_d;
        t.s_d = s_d;
        t.out = static_cast<__nv_bfloat16*>(out);
        t.h = h_opt;   // h only when asked for (the kernel needs none of its own)
        t.q_x = q_x_opt;
        t.s_x = s_x_opt;
        t.q_h = q_h_opt;
        t.s_h = s_h_opt;
        t.status = reinterpret_cast<int*>(base + kOffStatus);
        t.cnt = reinterpret_cast<int*>(base + l.mt_cnt);
        t.slots = reinterpret_cast<uint8_t*>(base + l.mt_slots);
        t.xq = reinterpret_cast<uint8_t*>(base + l.mt_xq);
        t.xs = reinterpret_cast<float*>(base + l.mt_xs);
        t.part = reinterpret_cast<float*>(base + l.mt_part);
        t.mode = kMtokDense;
        t.GS = t.KB;
        t.NU = t.KB / 2;
        t.KX = t.KB;
        t.x_ld = H;
        t.x_f32 = 0;
        t.ntmax = M;
        return cuda_status(launch_mtok(t, dev.sms, pdl, as_stream(stream)));
    }
    TokenArgs t = {};
    t.x = static_cast<const __nv_bfloat16*>(x);
    t.logits = nullptr;
    t.H = H;
    t.I = I;
    t.KB = H / 128;
    t.RB = I / 128;
    t.E_routed = 0;   // expert 0 is the one expert
    t.top_k = 0;
    t.ncols = I / 128;
    t.w_gu = w_gu;
    t.s_gu = s_gu;
    t.w_d = w_d;
    t.s_d = s_d;
    t.out = static_cast<__nv_bfloat16*>(out);
    t.h = h;
    t.q_x = q_x_opt;
    t.s_x = s_x_opt;
    t.q_h = q_h_opt;
    t.s_h = s_h_opt;
    t.status = reinterpret_cast<int*>(base + kOffStatus);
    t.tickets = reinterpret_cast<int*>(base + l.tickets);
    t.gq = t.tickets + H / 256;
    t.part = reinterpret_cast<float*>(base + l.part);
    return cuda_status(launch_token(t, dev.sms, pdl, as_stream(stream)));
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
                           const moeq_route_plan* plan_opt, float* h_opt, float* y_opt, uint8_t* q_x_opt,
                           float* s_x_opt, uint8_t* q_h_opt, float* s_h_opt, void* const* events_opt, void* ws,
                           size_t ws_bytes, void* stream) {
    const LayerCall c{x,     logits,  M,        H,     I,       E_routed, top_k,   w_gu,    s_gu,      w_d, s_d,
                      out,   nullptr, plan_opt, h_opt, y_opt,   q_x_opt,  s_x_opt, q_h_opt, s_h_opt,   events_opt,
                      ws,    ws_bytes};
    const DeviceInfo dev = current_device();
    const moeq_status st = layer_check(c, dev);
    if (st != MOEQ_OK) return st;
    uintptr_t key = stream_key(stream);
    const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(key, 0);
    return layer_launch(c, dev, false, !after_weight_write, as_stream(stream));
}

moeq_status moeq_moe_layer_shard(const void* x, const float* logits, int M, int H, int I_shard, int E_routed,
                                 int top_k, const uint8_t* w_gu, const float* s_gu, const uint8_t* w_d,
                                 const float* s_d, float* out_partial, const moeq_route_plan* plan_opt, float* h_opt,
                                 uint8_t* q_x_opt, float* s_x_opt, uint8_t* q_h_opt, float* s_h_opt, void* ws,
                                 size_t ws_bytes, void* stream) {
    LayerCall c = {};
    c.x = x;
    c.logits = logits;
    c.M = M;
    c.H = H;
    c.I = I_shard;
    c.E_routed = E_routed;
    c.top_k = top_k;
    c.w_gu = w_gu;
    c.s_gu = s_gu;
    c.w_d = w_d;
    c.s_d = s_d;
    c.out_f32 = out_partial;
    c.plan_opt = plan_opt;
    c.h_opt = h_opt;
    c.q_x_opt = q_x_opt;
    c.s_x_opt = s_x_opt;
    c.q_h_opt = q_h_opt;
    c.s_h_opt = s_h_opt;
    c.ws = ws;
    c.ws_bytes = ws_bytes;
    const DeviceInfo dev = current_device();
    const moeq_status st = layer_check(c, dev);
    if (st != MOEQ_OK) return st;
    uintptr_t key = stream_key(stream);
    const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(key, 0);
    return layer_launch(c, dev, false, !after_weight_write, as_stream(stream));
}

moeq_status moeq_tp_shard_weights(int E, int H, int I, int R, int rank, const uint8_t* w_gu, const float* s_gu,
                                  const uint8_t* w_d, const float* s_d, uint8_t* w_gu_shard, float* s_gu_shard,
                                  uint8_t* w_d_shard, float* s_d_shard, void* stream) {
    if (!w_gu || !s_gu || !w_d || !s_d || !w_gu_shard || !s_gu_shard || !w_d_shard || !s_d_shard)
        return MOEQ_ERR_INVALID_ARG;
    if (E < 1 || R < 1 || rank < 0 || rank >= R) return MOEQ_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 128 || I % (128 * R) || H > MOEQ_MAX_K || I > MOEQ_MAX_K)
        return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    const size_t tile = 16384, KB = H / 128, RB = I / 128, RBs = RB / R;
    cudaStream_t st = as_stream(stream);
    // gate_up, per expert: row blocks [r*RBs, (r+1)*RBs) (gate) and RB + that
    // (up), each a contiguous run of RBs * KB tiles; its scales likewise
    const size_t gu_run = RBs * KB * tile, gu_pitch = 2 * RB * KB * tile, gus_pitch = 2 * RBs * KB * tile;
    const size_t sg_run = RBs * KB * 4, sg_pitch = 2 * RB * KB * 4, sgs_pitch = 2 * RBs * KB * 4;
    const size_t E_ = static_cast<size_t>(E);
    for (int half = 0; half < 2; ++half) {
        const size_t rb0 = half * RB + rank * RBs;
        if (cudaMemcpy2DAsync(w_gu_shard + half * gu_run, gus_pitch, w_gu + rb0 * KB * tile, gu_pitch, gu_run, E_,
                              cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpy2DAsync(reinterpret_cast<char*>(s_gu_shard) + half * sg_run, sgs_pitch,
                              reinterpret_cast<const char*>(s_gu) + rb0 * KB * 4, sg_pitch, sg_run, E_,
                              cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return MOEQ_ERR_CUDA;
    }
    // down, per (expert, row block): K groups [r*RBs, (r+1)*RBs), a
    // contiguous run of RBs tiles; its scales likewise
    if (cudaMemcpy2DAsync(w_d_shard, RBs * tile, w_d + rank * RBs * tile, RB * tile, RBs * tile, E_ * KB,
                          cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
        cudaMemcpy2DAsync(s_d_shard, RBs * 4, s_d + rank * RBs, RB * 4, RBs * 4, E_ * KB, cudaMemcpyDeviceToDevice,
                          st) != cudaSuccess)
        return MOEQ_ERR_CUDA;
    // the shards are weights the layer kernels read before they wait for the
    // kernel ahead of them: note the writing stream (see moeq_quant_weight)
    g_weight_write_stream.store(stream_key(stream));
    return MOEQ_OK;
}

moeq_status moeq_tp_reduce(const float* partials, int R, int M, int H, void* out_bf16, void* stream) {
    if (!partials || !out_bf16 || !aligned16(partials) || !aligned16(out_bf16)) return MOEQ_ERR_INVALID_ARG;
    if (R < 1 || M < 1 || M > MOEQ_MAX_TOKENS) return MOEQ_ERR_INVALID_ARG;
    if (H <= 0 || H % 128) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    if (!current_device().ok) return MOEQ_ERR_DEVICE;
    return cuda_status(launch_tp_reduce(partials, R, M, H, out_bf16, as_stream(stream)));
}

size_t moeq_stack_workspace_size(int L, int M, int H, int I, int n_experts_incl_shared, int top_k) {
    if (L < 1 || L > MOEQ_MAX_LAYERS) return 0;
    const size_t lb = moeq_workspace_size(M, H, I, n_experts_incl_shared, top_k);
    if (!lb) return 0;
    return stack_ws_layout(L, lb, M, n_experts_incl_shared - 1, top_k).end;
}

moeq_status moeq_stack_plan(void* ws, size_t ws_bytes, int L, int M, int H, int I, int E_routed, int top_k, int layer,
                            moeq_route_plan* plan) {
    if (!ws || !plan || layer < 0 || layer >= L) return MOEQ_ERR_INVALID_ARG;
    const size_t need = moeq_stack_workspace_size(L, M, H, I, E_routed + 1, top_k);
    if (!need) return MOEQ_ERR_INVALID_ARG;
    if (ws_bytes < need) return MOEQ_ERR_WORKSPACE;
    const StackWs w = stack_ws_layout(L, moeq_workspace_size(M, H, I, E_routed + 1, top_k), M, E_routed, top_k);
    return moeq_route_plan_carve(static_cast<char*>(ws) + w.plan0 + static_cast<size_t>(layer) * w.plan_stride,
                                 w.plan_stride, M, E_routed, top_k, plan);
}

moeq_status moeq_moe_stack(int L, const void* x, const float* logits, int M, int H, int I, int E_routed, int top_k,
                           const uint8_t* const* w_gu, const float* const* s_gu, const uint8_t* const* w_d,
                           const float* const* s_d, void* out, int flags, void* ws, size_t ws_bytes, void* stream) {
    if (L < 1 || L > MOEQ_MAX_LAYERS || !w_gu || !s_gu || !w_d || !s_d || !x || !logits || !out)
        return MOEQ_ERR_INVALID_ARG;
    if (flags & ~MOEQ_STACK_EAGER) return MOEQ_ERR_INVALID_ARG;
    if (!route_args_ok(M, E_routed, top_k)) return MOEQ_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 128 || I % 128 || H > MOEQ_MAX_K || I > MOEQ_MAX_K) return MOEQ_ERR_UNSUPPORTED_SHAPE;
    const DeviceInfo dev = current_device();
    if (!dev.ok) return MOEQ_ERR_DEVICE;
    const size_t need = moeq_stack_workspace_size(L, M, H, I, E_routed + 1, top_k);
    if (!ws || !aligned16(ws) || ws_bytes < need) return MOEQ_ERR_WORKSPACE;
    const StackWs w = stack_ws_layout(L, moeq_workspace_size(M, H, I, E_routed + 1, top_k), M, E_routed, top_k);

    // every layer's call, checked before anything is launched or captured
    std::vector<LayerCall> calls(L);
    std::vector<moeq_route_plan> plans(L);
    const size_t x_bytes = static_cast<size_t>(M) * H * 2;
    for (int l = 0; l < L; ++l) {
        moeq_stack_plan(ws, ws_bytes, L, M, H, I, E_routed, top_k, l, &plans[l]);
        LayerCall& c = calls[l];
        c = LayerCall{};
        c.x = l == 0 ? x : static_cast<const char*>(out) + (l - 1) * x_bytes;
        c.logits = logits + static_cast<size_t>(l) * M * E_routed;
        c.M = M;
        c.H = H;
        c.I = I;
        c.E_routed = E_routed;
        c.top_k = top_k;
        c.w_gu = w_gu[l];
        c.s_gu = s_gu[l];
        c.w_d = w_d[l];
        c.s_d = s_d[l];
        c.out = static_cast<char*>(out) + l * x_bytes;
        c.plan_opt = &plans[l];
        c.ws = ws;
        c.ws_bytes = w.layer_bytes;
        const moeq_status st = layer_check(c, dev);
        if (st != MOEQ_OK) return st;
    }
    cudaStream_t st = as_stream(stream);
    uintptr_t skey = stream_key(stream);
    const bool after_weight_write = g_weight_write_stream.compare_exchange_strong(skey, 0);

    // Layer l > 0 reads logits that no layer of the stack writes, so it may
    // route before it waits for layer l - 1; layer 0 follows whatever came
    // before it on the stream.
    auto launch_all = [&](cudaStream_t s, bool first_pdl) -> moeq_status {
        for (int l = 0; l < L; ++l) {
            const moeq_status r = layer_launch(calls[l], dev, l > 0, l > 0 || first_pdl, s);
            if (r != MOEQ_OK) return r;
        }
        return MOEQ_OK;
    };
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        cudaGetLastError();
        return MOEQ_ERR_CUDA;
    }
    // Eager on request, and inside the caller's own capture (the launches
    // become part of the caller's graph).
    if ((flags & MOEQ_STACK_EAGER) || cap != cudaStreamCaptureStatusNone) return launch_all(st, !after_weight_write);

    int devid = 0;
    if (cudaGetDevice(&devid) != cudaSuccess) return MOEQ_ERR_CUDA;
    std::vector<uintptr_t> key = {static_cast<uintptr_t>(devid), static_cast<uintptr_t>(L), static_cast<uintptr_t>(M),
                                  static_cast<uintptr_t>(H), static_cast<uintptr_t>(I),
                                  static_cast<uintptr_t>(E_routed), static_cast<uintptr_t>(top_k),
                                  reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(logits),
                                  reinterpret_cast<uintptr_t>(out), reinterpret_cast<uintptr_t>(ws), ws_bytes};
    for (int l = 0; l < L; ++l) {
        key.push_back(reinterpret_cast<uintptr_t>(w_gu[l]));
        key.push_back(reinterpret_cast<uintptr_t>(s_gu[l]));
        key.push_back(reinterpret_cast<uintptr_t>(w_d[l]));
        key.push_back(reinterpret_cast<uintptr_t>(s_d[l]));
    }
    std::lock_guard<std::mutex> lock(g_stack_mu);
    StackGraph* hit = nullptr;
    for (StackGraph& g : g_stack_graphs)
        if (g.key == key) hit = &g;
    if (!hit) {
        // capture on first use
        cudaStream_t cs = capture_stream(devid);
        if (!cs) return MOEQ_ERR_CUDA;
        if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            cudaGetLastError();
            return MOEQ_ERR_CUDA;
        }
        const moeq_status r = launch_all(cs, false);
        cudaGraph_t graph = nullptr;
        const cudaError_t e = cudaStreamEndCapture(cs, &graph);
        cudaGraphExec_t exec = nullptr;
        const bool ok = r == MOEQ_OK && e == cudaSuccess && graph &&
                        cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
        if (graph) cudaGraphDestroy(graph);
        if (!ok) {
            cudaGetLastError();
            return r != MOEQ_OK ? r : MOEQ_ERR_CUDA;
        }
        if (g_stack_graphs.size() >= kStackGraphs) {
            auto lru = std::min_element(g_stack_graphs.begin(), g_stack_graphs.end(),
                                        [](const StackGraph& a, const StackGraph& b) { return a.used < b.used; });
            cudaGraphExecDestroy(lru->exec);
            g_stack_graphs.erase(lru);
        }
        g_stack_graphs.push_back(StackGraph{std::move(key), exec, 0});
        hit = &g_stack_graphs.back();
    }
    hit->used = ++g_stack_clock;
    return cuda_status(cudaGraphLaunch(hit->exec, st));
}

moeq_status moeq_stack_release_graphs(void) {
    std::lock_guard<std::mutex> lock(g_stack_mu);
    for (StackGraph& g : g_stack_graphs) cudaGraphExecDestroy(g.exec);
    g_stack_graphs.clear();
    return MOEQ_OK;
}

}  // extern "C"
