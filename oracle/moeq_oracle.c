/*
 * moeq oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the libmoeq hot path
 * computes: live per-token FP8 (OCP E4M3FN) activation quantisation, block-
 * scaled FP8 weight GEMMs, top-k MoE routing with expert deduplication, the
 * SwiGLU between gate_up and down, and the routing-weighted combine.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
 * this library.  It shares no source, header, table or helper with the CUDA
 * path in bandwidth_bound_fp8_gb300/csrc, and the CUDA path never calls it.
 *
 * Citations.  "GLM-5.2 x10" is the blog.sionic.ai page titled
 * "GPU 커널부터 새로 짜서 GLM-5.2 속도 10배 올리기"; "§n" is its numbered
 * section.  That page describes the method (live FP8 activation quantisation
 * in front of an FP8 weight GEMM, §1 and §8c; quantisation fused into the GEMM,
 * §4; top-8 MoE routing, bandwidth model) but prints no formula for the scale,
 * the group shape, the rounding or the routing weights.  This file fixes them
 * as follows (every reading is listed with its reason in the design notes):
 *   - activation groups are 1 x 128 per token, weight blocks 128 x 128;
 *   - scale s = fl32(amax / 448), code = RNE_satfinite_e4m3(fl32(x / s));
 *     a group with s == 0 gets signed-zero codes;
 *   - routing = top-k of the logits (ties to the lower expert id), weights =
 *     softmax over the k picked logits; one shared expert with weight 1;
 *   - gate rows [0, I) and up rows [I, 2I) of the gate_up weight,
 *     h = silu(gate) * up, kept in fp32 between the two GEMMs.
 *
 * Parity status of every function is pinned by tests/test_oracle_*.py.
 * Floating point: compile WITHOUT -ffast-math and with -ffp-contract=off, so
 * that every float expression below is one IEEE-754 operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Planted-mistake switch, used only by the mutation test that shows the     */
/* pins catch plausible slips.  0 = correct oracle.                          */
/* ------------------------------------------------------------------------ */
static int g_fault = 0;
void orc_set_fault(int f) { g_fault = f; }
int orc_get_fault(void) { return g_fault; }

/* ------------------------------------------------------------------------ */
/* E4M3FN codec (OCP 8-bit floating point, E4M3 variant).                     */
/* Fields: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no          */
/* infinities; S.1111.111 is NaN; largest finite magnitude 448; smallest      */
/* subnormal 2^-9.                                                            */
/* ------------------------------------------------------------------------ */
double orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);             /* 0.mmm * 2^(1-7) */
    else
        mag = ldexp((double)(8 + m), e - 10);   /* 1.mmm * 2^(e-7) */
    if (g_fault == 1 && e == 0) mag *= 2.0;     /* planted: subnormal scale */
    return sign ? -mag : mag;
}

/* Midpoint between the magnitudes of codes c and c+1 (exact in fp64). */
static double mid_above(int c)
{
    return 0.5 * (orc_e4m3_decode((uint8_t)c) + orc_e4m3_decode((uint8_t)(c + 1)));
}

/* Round-to-nearest-even with saturation to +-448, by a linear scan over the
 * finite grid (the definition).  The sign of v is copied, so -0 and negative
 * values that round to zero give 0x80. */
uint8_t orc_e4m3_encode_scan(double v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    int c;
    for (c = 0; c < 0x7E; ++c) {
        double mid = mid_above(c);
        if (a < mid) return (uint8_t)((neg << 7) | c);
        if (a == mid) {                          /* tie: even mantissa LSB */
            int pick = (c & 1) ? c + 1 : c;
            return (uint8_t)((neg << 7) | pick);
        }
    }
    return (uint8_t)((neg << 7) | 0x7E);         /* >= 448: saturate */
}

/* Same result as orc_e4m3_encode_scan, found by bisection over the 126
 * midpoints instead of a scan (used for the large weight tensors).  The
 * midpoints are tabulated from mid_above on every call's entry check, so
 * the table always reflects the decode definition in force. */
uint8_t orc_e4m3_encode(double v)
{
    static double mids[0x7E];
    static int mids_fault = -1;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    int lo = 0, hi = 0x7D;  /* answer in [lo, hi]: smallest c with a <= mid(c) */
    int c;
    if (mids_fault != g_fault) {
        for (c = 0; c < 0x7E; ++c) mids[c] = mid_above(c);
        mids_fault = g_fault;
    }
    if (a > mids[0x7D]) return (uint8_t)((neg << 7) | 0x7E);
    while (lo < hi) {
        int mc = (lo + hi) / 2;
        if (a <= mids[mc]) hi = mc; else lo = mc + 1;
    }
    c = lo;
    if (c < 0x7E && a == mids[c] && (c & 1)) c = c + 1;
    if (g_fault == 2 && c < 0x7E && a == mids[c] && !(c & 1)) c = c + 1; /* planted: ties away */
    return (uint8_t)((neg << 7) | c);
}

/* bf16 bit pattern -> float (exact: bf16 is the top half of a binary32). */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* double -> bf16 bit pattern, round to nearest even, directly from fp64. */
uint16_t orc_f64_to_bf16(double v)
{
    double a = fabs(v), r;
    float f;
    uint32_t u;
    int e;
    if (v != v) return 0x7FC0;
    if (a == 0.0) {
        r = 0.0;
    } else if (a < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(a, 133)), -133);       /* subnormal grid */
    } else {
        frexp(a, &e);                                    /* a in [2^(e-1), 2^e) */
        r = ldexp(nearbyint(ldexp(a, 8 - e)), e - 8);    /* 8 significant bits */
    }
    f = (float)(signbit(v) ? -r : r);                    /* exact */
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* Live activation quantisation (GLM-5.2 x10 §1, §8c): per row m and per     */
/* 128-wide group g, s = fl32(amax/448), q = RNE_sat(fl32(x/s)).             */
/* ------------------------------------------------------------------------ */
static void quant_group(const float* x, int n, uint8_t* q, float* s_out)
{
    float amax = 0.0f, s;
    int k;
    for (k = 0; k < n; ++k) {
        float a = fabsf(x[k]);
        if (a > amax) amax = a;
    }
    s = amax / 448.0f;
    if (g_fault == 3) s = amax / 447.0f;                 /* planted: wrong constant */
    *s_out = s;
    for (k = 0; k < n; ++k) {
        if (s == 0.0f) {
            q[k] = signbit(x[k]) ? 0x80 : 0x00;
        } else {
            float v = x[k] / s;                           /* one IEEE division */
            q[k] = orc_e4m3_encode((double)v);
        }
    }
}

/* x: [M, K] fp32 row-major; q: [M, K]; s: [M, K/128]. Returns 0, or -1 if K % 128. */
int orc_quant_act_f32(const float* x, int M, int K, uint8_t* q, float* s)
{
    int m, g, G = K / 128;
    if (K % 128) return -1;
    for (m = 0; m < M; ++m)
        for (g = 0; g < G; ++g)
            quant_group(x + (size_t)m * K + (size_t)g * 128, 128,
                        q + (size_t)m * K + (size_t)g * 128, s + (size_t)m * G + g);
    return 0;
}

/* Same for bf16 input (bit patterns); the bf16 -> fp32 widening is exact. */
int orc_quant_act_bf16(const uint16_t* x, int M, int K, uint8_t* q, float* s)
{
    size_t i, n = (size_t)M * K;
    float* xf = (float*)malloc(n * sizeof(float) + 1);
    int rc;
    if (!xf) return -2;
    for (i = 0; i < n; ++i) xf[i] = orc_bf16_to_f32(x[i]);
    rc = orc_quant_act_f32(xf, M, K, q, s);
    free(xf);
    return rc;
}

/* Weight quantisation: one scale per 128 x 128 block, same codec.
 * w: [N, K] fp32; q: [N, K]; s: [N/128, K/128]. */
int orc_quant_weight(const float* w, int N, int K, uint8_t* q, float* s)
{
    int nb, kb, r, k, NB = N / 128, KB = K / 128;
    if (N % 128 || K % 128) return -1;
    for (nb = 0; nb < NB; ++nb)
        for (kb = 0; kb < KB; ++kb) {
            float amax = 0.0f, sc;
            for (r = 0; r < 128; ++r)
                for (k = 0; k < 128; ++k) {
                    float a = fabsf(w[(size_t)(nb * 128 + r) * K + kb * 128 + k]);
                    if (a > amax) amax = a;
                }
            sc = amax / 448.0f;
            s[(size_t)nb * KB + kb] = sc;
            for (r = 0; r < 128; ++r)
                for (k = 0; k < 128; ++k) {
                    size_t i = (size_t)(nb * 128 + r) * K + kb * 128 + k;
                    if (sc == 0.0f) q[i] = signbit(w[i]) ? 0x80 : 0x00;
                    else q[i] = orc_e4m3_encode((double)(w[i] / sc));
                }
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block-scaled FP8 GEMM, y = A W^T with A = diag-scaled codes per 1x128      */
/* group and W = codes per 128x128 block:                                     */
/*   y[m,n] = sum_g sa[m,g] * sw[n/128,g] * sum_{k in g} qa[m,k] * qw[n,k]    */
/* The inner sum is exact in fp64: each product of two E4M3 values is an      */
/* integer multiple of 2^-18 below 2^18, and 128 of them need fewer than 53   */
/* bits.  T[m,n] = the same sum over absolute values of every scaled term,    */
/* the scale the parity tolerance is stated against.                          */
/* qa: [M,K], sa: [M,K/128], qw: [N,K], sw: [N/128,K/128]; y, T: [M,N].        */
/* ------------------------------------------------------------------------ */
int orc_gemm(const uint8_t* qa, const float* sa, int M,
             const uint8_t* qw, const float* sw, int N, int K,
             double* y, double* T)
{
    double dec[256];
    int m, n, g, k, G = K / 128;
    if (K % 128 || N % 128) return -1;
    for (k = 0; k < 256; ++k) dec[k] = orc_e4m3_decode((uint8_t)k);
    for (m = 0; m < M; ++m)
        for (n = 0; n < N; ++n) {
            double acc = 0.0, tacc = 0.0;
            for (g = 0; g < G; ++g) {
                const uint8_t* a = qa + (size_t)m * K + (size_t)g * 128;
                const uint8_t* w = qw + (size_t)n * K + (size_t)g * 128;
                double inner = 0.0, inner_abs = 0.0, scale;
                int kend = (g_fault == 4) ? 127 : 128;   /* planted: dropped term */
                for (k = 0; k < kend; ++k) {
                    double p = dec[a[k]] * dec[w[k]];
                    if (g_fault == 8)                        /* planted: transposed operand */
                        p = dec[a[k]] * dec[qw[((size_t)(g * 128 + k) * N + n) % ((size_t)N * K)]];
                    inner += p;
                    inner_abs += fabs(p);
                }
                scale = (double)sa[(size_t)m * G + g] * (double)sw[(size_t)(n / 128) * G + g];
                if (g_fault == 5) scale = (double)sa[(size_t)m * G + g] *
                                          (double)sw[(size_t)g * (N / 128) + n / 128]; /* planted: transposed scales */
                acc += scale * inner;
                tacc += fabs(scale) * inner_abs;
            }
            y[(size_t)m * N + n] = acc;
            if (T) T[(size_t)m * N + n] = tacc;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k routing with deduplication (GLM-5.2 x10: top-8 experts per token;    */
/* several tokens verified in one pass share one weight read, §5-§6).         */
/*   topk_id[m,j]: j-th largest logit of row m, ties to the lower id;         */
/*   topk_w[m,j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k picks;    */
/*   uniq[0..U-1]: routed experts used by any token, ascending, then the      */
/*   shared expert (id E) last, so n_uniq = U_routed + 1;                     */
/*   offs[u]..offs[u+1]: the pairs of unique expert u, tokens ascending;      */
/*   pair_tok[p]: token of pair p;  pair_of[m, j]: pair of (token m, slot j), */
/*   slot k being the shared expert.  Returns the number of pairs.            */
/* ------------------------------------------------------------------------ */
int orc_route(const float* logits, int M, int E, int k,
              int32_t* topk_id, double* topk_w, int32_t* n_uniq, int32_t* uniq,
              int32_t* offs, int32_t* pair_tok, int32_t* pair_of)
{
    int m, j, e, u, p;
    int* cnt;
    int* uid;
    if (k < 1 || k > E || M < 1) return -1;
    cnt = (int*)calloc((size_t)E + 1, sizeof(int));
    uid = (int*)calloc((size_t)E + 1, sizeof(int));
    if (!cnt || !uid) { free(cnt); free(uid); return -2; }

    for (m = 0; m < M; ++m) {
        const float* l = logits + (size_t)m * E;
        double den = 0.0, lmax;
        for (j = 0; j < k; ++j) {                        /* selection, one pick at a time */
            int best = -1;
            for (e = 0; e < E; ++e) {
                int taken = 0, t;
                for (t = 0; t < j; ++t) if (topk_id[(size_t)m * k + t] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: ties keep lower id */
                else if (g_fault == 6 && l[e] == l[best]) best = e; /* planted: ties to higher id */
            }
            topk_id[(size_t)m * k + j] = best;
        }
        lmax = (double)l[topk_id[(size_t)m * k]];
        for (j = 0; j < k; ++j) den += exp((double)l[topk_id[(size_t)m * k + j]] - lmax);
        for (j = 0; j < k; ++j)
            topk_w[(size_t)m * k + j] = exp((double)l[topk_id[(size_t)m * k + j]] - lmax) / den;
    }

    for (m = 0; m < M; ++m)
        for (j = 0; j < k; ++j) cnt[topk_id[(size_t)m * k + j]]++;
    u = 0; p = 0;
    for (e = 0; e < E; ++e) {
        if (!cnt[e]) continue;
        uid[e] = u;
        uniq[u] = e;
        offs[u] = p;
        for (m = 0; m < M; ++m)                          /* tokens ascending */
            for (j = 0; j < k; ++j)
                if (topk_id[(size_t)m * k + j] == e) {
                    pair_tok[p] = m;
                    pair_of[(size_t)m * (k + 1) + j] = p;
                    ++p;
                }
        ++u;
    }
    uniq[u] = E;                                         /* shared expert last */
    offs[u] = p;
    for (m = 0; m < M; ++m) {
        pair_tok[p] = m;
        pair_of[(size_t)m * (k + 1) + k] = p;
        ++p;
    }
    ++u;
    offs[u] = p;
    *n_uniq = u;
    free(cnt);
    free(uid);
    return p;
}

/* SwiGLU between the two GEMMs: h = silu(gate) * up = gate/(1+e^-gate) * up,
 * evaluated in fp64 and rounded once to fp32 (the dtype of h). */
float orc_swiglu(double gate, double up)
{
    double silu = gate / (1.0 + exp(-gate));
    if (g_fault == 7) silu = gate / (1.0 + exp(gate));   /* planted: wrong sign */
    return (float)(silu * up);
}

/* Elementwise SwiGLU over arrays: h[i] = orc_swiglu(gate[i], up[i]). */
void orc_swiglu_vec(const double* gate, const double* up, int n, float* h)
{
    int i;
    for (i = 0; i < n; ++i) h[i] = orc_swiglu(gate[i], up[i]);
}

/* ------------------------------------------------------------------------ */
/* One MoE layer:                                                             */
/*   route -> quant(x) -> per pair: gate_up GEMM -> SwiGLU -> h (fp32)        */
/*   -> quant(h) -> down GEMM -> y -> out[m] = y[shared(m)] + sum_j w_j y[j]  */
/* Weights are passed per expert id (0..E, E = shared); only the experts the  */
/* routing touches are read, so the others may be NULL.                       */
/*   qgu[e]: [2I, H] codes, sgu[e]: [2I/128, H/128];                          */
/*   qd[e]:  [H, I] codes,  sd[e]:  [H/128, I/128].                           */
/* Outputs (caller-allocated, P_max = M*k + M pairs):                         */
/*   out_bf16 [M,H], out64 [M,H], Tout [M,H], h [P_max,I], y64 [P_max,H],     */
/*   Ty [P_max,H], qx [M,H], sx [M,H/128], qh [P_max,I], sh [P_max,I/128],    */
/*   routing outputs as orc_route.  Returns the pair count, < 0 on error.     */
/* ------------------------------------------------------------------------ */
int orc_moe_layer(const uint16_t* x_bf16, const float* logits,
                  int M, int H, int I, int E, int k,
                  const uint8_t* const* qgu, const float* const* sgu,
                  const uint8_t* const* qd, const float* const* sd,
                  uint16_t* out_bf16, double* out64, double* Tout,
                  float* h, double* y64, double* Ty,
                  uint8_t* qx, float* sx, uint8_t* qh, float* sh,
                  int32_t* topk_id, double* topk_w, int32_t* n_uniq, int32_t* uniq,
                  int32_t* offs, int32_t* pair_tok, int32_t* pair_of)
{
    int P, u, p, i, m, j, n;
    double* gu;
    if (H % 128 || I % 128) return -1;
    P = orc_route(logits, M, E, k, topk_id, topk_w, n_uniq, uniq, offs, pair_tok, pair_of);
    if (P < 0) return P;
    if (orc_quant_act_bf16(x_bf16, M, H, qx, sx)) return -3;
    gu = (double*)malloc(sizeof(double) * 2 * (size_t)I);
    if (!gu) return -2;

    for (u = 0; u < *n_uniq; ++u) {                      /* gate_up + SwiGLU */
        int e = uniq[u];
        if (!qgu[e] || !sgu[e]) { free(gu); return -4; }
        for (p = offs[u]; p < offs[u + 1]; ++p) {
            int t = pair_tok[p];
            orc_gemm(qx + (size_t)t * H, sx + (size_t)t * (H / 128), 1,
                     qgu[e], sgu[e], 2 * I, H, gu, NULL);
            for (i = 0; i < I; ++i) h[(size_t)p * I + i] = orc_swiglu(gu[i], gu[I + i]);
        }
    }
    free(gu);

    if (orc_quant_act_f32(h, P, I, qh, sh)) return -3;   /* live quant of h */

    for (u = 0; u < *n_uniq; ++u) {                      /* down */
        int e = uniq[u];
        if (!qd[e] || !sd[e]) return -4;
        for (p = offs[u]; p < offs[u + 1]; ++p)
            orc_gemm(qh + (size_t)p * I, sh + (size_t)p * (I / 128), 1,
                     qd[e], sd[e], H, I, y64 + (size_t)p * H, Ty + (size_t)p * H);
    }

    for (m = 0; m < M; ++m)                              /* combine */
        for (n = 0; n < H; ++n) {
            int ps = pair_of[(size_t)m * (k + 1) + k];
            double acc = (g_fault == 9) ? 0.0 : y64[(size_t)ps * H + n]; /* planted: shared dropped */
            double tacc = Ty[(size_t)ps * H + n];
            for (j = 0; j < k; ++j) {
                int pj = pair_of[(size_t)m * (k + 1) + j];
                double w = topk_w[(size_t)m * k + j];
                acc += w * y64[(size_t)pj * H + n];
                tacc += w * Ty[(size_t)pj * H + n];
            }
            out64[(size_t)m * H + n] = acc;
            Tout[(size_t)m * H + n] = tacc;
            out_bf16[(size_t)m * H + n] = orc_f64_to_bf16(acc);
        }
    return P;
}
