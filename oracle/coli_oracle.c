/*
 * coli_oracle.c -- plain, slow, step-by-step CPU oracle for the quantized MoE
 * feed-forward layer (int4 routed experts, Q8_0 activations, F32 router).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library.
 *
 * Sources (the colibri pages; cited by page title and section):
 *   [P1] "colibri: a pure-C inference engine that runs a 744B MoE model on a
 *        25GB-RAM consumer PC" (discuss.pytorch.kr), section "Key features"
 *        (Q8_0-style int8 activations, integer dot kernels, int8/int4/int2
 *        packing bit-identical to the int8 container).
 *   [P2] "Open-source engine that ran 744B GLM-5.2 on a 25GB-RAM laptop"
 *        (jeff.news), section "Attention and kernels" (DeepSeek-V3-style sigmoid
 *        router, shared expert; Q8_0 int8 activations with an integer matmul).
 *   [P3] "Colibri: an AI engine running a 744B model in 25GB of RAM"
 *        (alphamatch.ai), sections "Optimised integer kernels" and "Technical
 *        excellence" (batch-union MoE for prefill).
 *   [P5] "GLM-5.2-colibri-int4" model card (aitrends.kr), sections "TL;DR",
 *        "Good to know" and "Technical features" (packed int4 nibbles in U8 with
 *        per-row F32 scales; np.rint matching the engine's lrintf; router in F32).
 *
 * Where the pages leave a step open, the layer's specification fixes it (shapes,
 * the weight quantiser q = clamp(lrintf(w/s), -7, 7) with s = max|row|/7,
 * low-nibble-first packing with a +8 offset, Q8_0 blocks of 32 with an F32
 * scale, top-k with lowest-index ties, renormalised selected weights times the
 * routed scale, SwiGLU experts).  The remaining open points are fixed by the
 * plainest reading, each one named at the function that takes it.
 *
 * Precision: the pages fix F32 for the router and for every scale, and int32
 * for the block dot products, so the oracle computes in F32 exactly where the
 * method does and in exact integers elsewhere.  It must be compiled with
 * -ffp-contract=off: every fused multiply-add it performs is an explicit fmaf.
 * Threading (OpenMP) is only over independent outputs, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))
/* status of orc_moe_forward_w for a weight container other than 4 or 8 bits */
#define ORC_E_WBITS (-1000000)

/* ------------------------------------------------------------------------- */
/* Bit helpers                                                               */
/* ------------------------------------------------------------------------- */
static float orc_bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ------------------------------------------------------------------------- */
/* O1  int4 weight container: per-row F32 scale, packed nibbles  [P5 TL;DR,   */
/*     Technical features; P1 Key features]                                  */
/* ------------------------------------------------------------------------- */
/* One row of K weights (one output neuron's input vector) becomes K/2 bytes:
 * s = max_k |w_k| / 7 (an IEEE F32 divide), q_k = clamp(lrintf(w_k / s), -7, 7)
 * (the division is taken literally, not as a multiply by 1/s), nibble = q + 8,
 * byte j = nibble(2j) | nibble(2j+1) << 4.  An all-zero row has s = 0 and
 * every q = 0 (reading: the pages are silent about empty rows). */
ORC_API void orc_pack_int4_rows(const float *w, int rows, int K, uint8_t *packed, float *scale)
{
    for (int r = 0; r < rows; ++r) {
        const float *wr = w + (size_t)r * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float a = fabsf(wr[k]);
            if (a > amax) amax = a;
        }
        float s = amax / 7.0f;
        scale[r] = s;
        uint8_t *pr = packed + (size_t)r * (K / 2);
        for (int j = 0; j < K / 2; ++j) {
            int nib[2];
            for (int h = 0; h < 2; ++h) {
                long q = 0;
                if (s > 0.0f) {
                    q = lrintf(wr[2 * j + h] / s);
                    if (q < -7) q = -7;
                    if (q > 7) q = 7;
                }
                nib[h] = (int)q + 8;
            }
            pr[j] = (uint8_t)(nib[0] | (nib[1] << 4));
        }
    }
}

/* Inverse of the packing: signed codes q in [-8, 7] from the nibbles. */
ORC_API void orc_unpack_int4_rows(const uint8_t *packed, int rows, int K, int8_t *q)
{
    for (int r = 0; r < rows; ++r) {
        const uint8_t *pr = packed + (size_t)r * (K / 2);
        int8_t *qr = q + (size_t)r * K;
        for (int j = 0; j < K / 2; ++j) {
            qr[2 * j] = (int8_t)((pr[j] & 0x0F) - 8);
            qr[2 * j + 1] = (int8_t)((pr[j] >> 4) - 8);
        }
    }
}

/* int8 weight container (the pages' int8 head and their int8 container, to
 * which the int4 packing decodes bit-identically) [P1 Key features]: one
 * two's-complement byte per weight, s = max_k |w_k| / 127 (an IEEE F32
 * divide), q_k = clamp(lrintf(w_k / s), -127, 127); an all-zero row has s = 0
 * and every q = 0 (the same reading as the int4 container). */
ORC_API void orc_pack_int8_rows(const float *w, int rows, int K, int8_t *q, float *scale)
{
    for (int r = 0; r < rows; ++r) {
        const float *wr = w + (size_t)r * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float a = fabsf(wr[k]);
            if (a > amax) amax = a;
        }
        float sr = amax / 127.0f;
        scale[r] = sr;
        int8_t *qr = q + (size_t)r * K;
        for (int k = 0; k < K; ++k) {
            long v = 0;
            if (sr > 0.0f) {
                v = lrintf(wr[k] / sr);
                if (v < -127) v = -127;
                if (v > 127) v = 127;
            }
            qr[k] = (int8_t)v;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* O2  Q8_0-style activation quantiser  [P1 Key features; P2 Attention and    */
/*     kernels; P3 Optimised integer kernels; rounding per P5 TL;DR]         */
/* ------------------------------------------------------------------------- */
/* Per block of 32: amax = max|x|, d = amax / 127 (F32), id = d ? 1/d : 0,
 * q = clamp(lrintf(x * id), -127, 127), stored scale d in F32.  "Q8_0 style"
 * follows the ggml heritage, so the code is x * (1/d), not x / d (reading).
 * lrintf rounds half to even under the default rounding mode, as np.rint does. */
ORC_API void orc_q8_0(const float *x, int n, int8_t *q, float *d)
{
    for (int b = 0; b < n / 32; ++b) {
        const float *xb = x + 32 * b;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float db = amax / 127.0f;
        float id = (db != 0.0f) ? 1.0f / db : 0.0f;
        d[b] = db;
        for (int i = 0; i < 32; ++i) {
            long v = lrintf(xb[i] * id);
            if (v < -127) v = -127;
            if (v > 127) v = 127;
            q[32 * b + i] = (int8_t)v;
        }
    }
}

/* lrintf itself, exposed so the tests can check the rounding rule. */
ORC_API long orc_lrintf(float v) { return lrintf(v); }

/* ------------------------------------------------------------------------- */
/* Own exponential and sigmoid (same IEEE operation sequence on every side)  */
/* ------------------------------------------------------------------------- */
/* Cody and Waite range reduction (W. J. Cody, W. Waite, "Software Manual for
 * the Elementary Functions", 1980): z = n ln2 + r with n = rint(z log2 e) and
 * r computed with a two-part ln2, then e^r by its Taylor series to degree 7
 * (|r| <= ln2/2 makes the truncation error ~5e-9 relative), then scaling by 2^n
 * through the exponent bits.  Constants are the F32 roundings of log2(e), of ln2
 * (high part) and of ln2 - high (low part), and of 1/k!. */
static const float ORC_LOG2E = 0x1.715476p+0f;
static const float ORC_LN2_HI = 0x1.62e430p-1f;
static const float ORC_LN2_LO = -0x1.05c610p-29f;
static const float ORC_INV_FACT[8] = {
    0x1.000000p+0f, 0x1.000000p+0f, 0x1.000000p-1f, 0x1.555556p-3f,
    0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f,
};

ORC_API float orc_exp(float z)
{
    if (z > 88.0f) return INFINITY;
    if (z < -87.0f) return 0.0f;
    float t = z * ORC_LOG2E;
    float n = rintf(t);
    float r = fmaf(-n, ORC_LN2_HI, z);
    r = fmaf(-n, ORC_LN2_LO, r);
    float p = ORC_INV_FACT[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, r, ORC_INV_FACT[k]);
    int ni = (int)n;
    float two_n = orc_bits_to_float((uint32_t)(ni + 127) << 23);
    return p * two_n;
}

/* sigma(z) = 1 / (1 + e^-z) */
ORC_API float orc_sigmoid(float z)
{
    return 1.0f / (1.0f + orc_exp(-z));
}

/* ------------------------------------------------------------------------- */
/* O3  DeepSeek-V3-style sigmoid router, F32  [P2 Attention and kernels;      */
/*     P5 Good to know: router kept in F32]                                  */
/* ------------------------------------------------------------------------- */
/* Canonical F32 reduction order of one router logit (a build choice: the pages
 * say only "F32 router"; bit-exact expert indices need one fixed order).
 * The H inputs are cut into chunks of 4 consecutive elements; chunk c feeds
 * partial sum p[c mod 256], chunks taken in ascending order, the 4 elements of
 * a chunk in ascending order, each step p = fmaf(x_k, W_ek, p) from p = +0.
 * The 256 partials are then folded as 8 groups of 32: within a group, for
 * o = 16, 8, 4, 2, 1, every member j becomes p[j] + p[j ^ o] (all members
 * updated from the previous values); member 0 of group g is S_g.  The 8 S_g
 * are folded the same way with o = 4, 2, 1, and member 0 is the logit. */
static float orc_fold(float *v, int n)
{
    float tmp[32];
    for (int o = n / 2; o >= 1; o /= 2) {
        for (int j = 0; j < n; ++j) tmp[j] = v[j] + v[j ^ o];
        for (int j = 0; j < n; ++j) v[j] = tmp[j];
    }
    return v[0];
}

ORC_API float orc_router_logit(const float *x, const float *w, int H)
{
    float p[256];
    for (int j = 0; j < 256; ++j) p[j] = 0.0f;
    for (int c = 0; c < H / 4; ++c)
        for (int i = 0; i < 4; ++i)
            p[c % 256] = fmaf(x[4 * c + i], w[4 * c + i], p[c % 256]);
    float s[8];
    for (int g = 0; g < 8; ++g) s[g] = orc_fold(p + 32 * g, 32);
    return orc_fold(s, 8);
}

/* Route T tokens.  sigma_e = sigmoid(logit_e); selection key sel_e = sigma_e +
 * bias_e; the k experts with the largest key are chosen, ties going to the lower
 * expert index, listed in rank order (largest key first).  The bias steers the
 * selection only (DeepSeek-V3's auxiliary-loss-free balancing: the gate weight
 * uses sigma, not sigma + bias).  No group-limited routing (nothing on the pages
 * asks for it).  Weights: S = sum of the selected sigma in rank order starting
 * from 0, w_r = (sigma_r / S) * routed_scale.  Optional outputs (NULL to skip):
 * logits [T][E] and sigma [T][E]. */
ORC_API void orc_route(const float *x, int T, int H, const float *W, const float *bias, int E,
                       int k, float routed_scale, int32_t *idx, float *wout,
                       float *logits_out, float *sigma_out)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        float *sig = (float *)malloc(sizeof(float) * E);
        float *sel = (float *)malloc(sizeof(float) * E);
        char *taken = (char *)calloc(E, 1);
        for (int e = 0; e < E; ++e) {
            float z = orc_router_logit(x + (size_t)t * H, W + (size_t)e * H, H);
            if (logits_out) logits_out[(size_t)t * E + e] = z;
            sig[e] = orc_sigmoid(z);
            if (sigma_out) sigma_out[(size_t)t * E + e] = sig[e];
            sel[e] = sig[e] + bias[e];
        }
        float S = 0.0f;
        for (int r = 0; r < k; ++r) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || sel[e] > sel[best]) best = e; /* strict: lower index wins ties */
            }
            taken[best] = 1;
            idx[(size_t)t * k + r] = best;
            S = S + sig[best];
        }
        for (int r = 0; r < k; ++r) {
            float sr = sig[idx[(size_t)t * k + r]];
            wout[(size_t)t * k + r] = (sr / S) * routed_scale;
        }
        free(sig); free(sel); free(taken);
    }
}

/* Pre-norm of one layer of a stacked decoder (a reading: the multi-layer
 * sweep of the benchmark configurations chains layers with a residual add;
 * without a norm the SwiGLU output grows as the square of its input and the
 * stream overflows within a few layers, so each layer reads RMSNorm(x) as in
 * GLM-class decoders, with no learned gain).  Per token: ss = sum of x_k^2 in
 * the router's canonical order (the router dot of x with itself), ms = ss / H,
 * r = 1 / sqrtf(ms + eps), xn_k = x_k * r; every step one IEEE operation. */
ORC_API void orc_rmsnorm(const float *x, int T, int H, float eps, float *xn)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *xt = x + (size_t)t * H;
        const float ss = orc_router_logit(xt, xt, H);
        const float ms = ss / (float)H;
        const float r = 1.0f / sqrtf(ms + eps);
        for (int k = 0; k < H; ++k) xn[(size_t)t * H + k] = xt[k] * r;
    }
}

/* ------------------------------------------------------------------------- */
/* O4  Batch-union dispatch: histogram and stable permutation  [P3 Technical  */
/*     excellence: batch-union MoE in prefill]                               */
/* ------------------------------------------------------------------------- */
/* The T*k (token, rank) pairs, pair p = t*k + r, are sorted by expert with a
 * stable counting sort (reading: token-major stability is the plainest order):
 * counts[e]; offsets = exclusive scan over ascending e (offsets[E] = T*k);
 * pos(p) = offsets[e_p] + #{p' < p : e_p' = e_p}; perm[pos] = p; inv[p] = pos. */
ORC_API void orc_dispatch(const int32_t *idx, int T, int k, int E, int32_t *counts,
                          int32_t *offsets, int32_t *perm, int32_t *inv)
{
    int P = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int p = 0; p < P; ++p) counts[idx[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int p = 0; p < P; ++p) {
        int e = idx[p];
        int pos = offsets[e] + fill[e];
        fill[e] += 1;
        perm[pos] = p;
        inv[p] = pos;
    }
    free(fill);
}

/* ------------------------------------------------------------------------- */
/* O5  Integer dot products and the expert FFN  [P1 Key features; P2         */
/*     Attention and kernels; P3 Optimised integer kernels]                  */
/* ------------------------------------------------------------------------- */
/* I[r][b] = sum over the 32 elements of block b of (nibble - 8) * qx, in int32. */
ORC_API void orc_block_dots(const uint8_t *w4, int rows, int K, const int8_t *q, int32_t *I)
{
    int nb = K / 32;
    for (int r = 0; r < rows; ++r) {
        const uint8_t *pr = w4 + (size_t)r * (K / 2);
        for (int b = 0; b < nb; ++b) {
            int32_t acc = 0;
            for (int i = 0; i < 32; ++i) {
                int k = 32 * b + i;
                uint8_t byte = pr[k / 2];
                int nib = (k & 1) ? (byte >> 4) : (byte & 0x0F);
                acc += (nib - 8) * (int32_t)q[k];
            }
            I[(size_t)r * nb + b] = acc;
        }
    }
}

/* Weight code k of a row in a container of `wbits` bits per weight: 4 is the
 * packed int4 container (nibble - 8), 8 the int8 container (the byte). */
static int orc_wcode(const uint8_t *row, int wbits, int k)
{
    if (wbits == 8) return (int)(int8_t)row[k];
    uint8_t byte = row[k / 2];
    int nib = (k & 1) ? (byte >> 4) : (byte & 0x0F);
    return nib - 8;
}

/* One output row: y = s_row * acc, where acc = 0 and, for blocks b ascending,
 * acc = fmaf(d_b, (float)I_b, acc) with I_b the int32 sum over block b of
 * code * q (reading: the per-row scale is applied once, after the block sum). */
static float orc_row_dot_w(const uint8_t *row, int wbits, float s_row, int K, const int8_t *q, const float *d)
{
    float acc = 0.0f;
    for (int b = 0; b < K / 32; ++b) {
        int32_t I = 0;
        for (int i = 0; i < 32; ++i) {
            int k = 32 * b + i;
            I += orc_wcode(row, wbits, k) * (int32_t)q[k];
        }
        acc = fmaf(d[b], (float)I, acc);
    }
    return s_row * acc;
}

static float orc_row_dot(const uint8_t *row4, float s_row, int K, const int8_t *q, const float *d)
{
    return orc_row_dot_w(row4, 4, s_row, K, q, d);
}

/* Block dots of the int8 container: I[r][b] = sum over block b of w8 * q. */
ORC_API void orc_block_dots_w8(const int8_t *w8, int rows, int K, const int8_t *q, int32_t *I)
{
    int nb = K / 32;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            int32_t acc = 0;
            for (int i = 0; i < 32; ++i)
                acc += (int32_t)w8[(size_t)r * K + 32 * b + i] * (int32_t)q[32 * b + i];
            I[(size_t)r * nb + b] = acc;
        }
}

ORC_API void orc_rows_dot(const uint8_t *w4, const float *s, int rows, int K, const int8_t *q,
                          const float *d, float *out)
{
    for (int r = 0; r < rows; ++r)
        out[r] = orc_row_dot(w4 + (size_t)r * (K / 2), s[r], K, q, d);
}

/* One SwiGLU expert on one token.  Expert layout: gate [F][H], up [F][H],
 * down [H][F] (int4, rows of K/2 bytes, back to back); row scales
 * [gate F | up F | down H].  g_i, u_i by orc_row_dot over qx; h_i = (g_i *
 * sigma(g_i)) * u_i; h is Q8_0-quantised (F/32 blocks) into qh, dh; then
 * y_j = orc_row_dot(down_j) over qh.  Optional outputs g, u, h may be NULL. */
ORC_API int orc_expert_ffn_w(const uint8_t *ew, int wbits, const float *ers, int H, int F,
                             const int8_t *qx, const float *dx, int8_t *qh, float *dh, float *y,
                             float *g_out, float *u_out, float *h_out)
{
    /* the two containers: 4 (packed nibbles) or 8 (one int8 code per byte) */
    if (wbits != 4 && wbits != 8) return -1;
    /* a row of K weights takes K * wbits / 8 bytes */
    const size_t rh = (size_t)H * wbits / 8, rf = (size_t)F * wbits / 8;
    const uint8_t *gate = ew;
    const uint8_t *up = ew + (size_t)F * rh;
    const uint8_t *down = ew + (size_t)2 * F * rh;
    float *h = (float *)malloc(sizeof(float) * F);
    for (int i = 0; i < F; ++i) {
        float g = orc_row_dot_w(gate + (size_t)i * rh, wbits, ers[i], H, qx, dx);
        float u = orc_row_dot_w(up + (size_t)i * rh, wbits, ers[F + i], H, qx, dx);
        h[i] = (g * orc_sigmoid(g)) * u;
        if (g_out) g_out[i] = g;
        if (u_out) u_out[i] = u;
        if (h_out) h_out[i] = h[i];
    }
    orc_q8_0(h, F, qh, dh);
    for (int j = 0; j < H; ++j)
        y[j] = orc_row_dot_w(down + (size_t)j * rf, wbits, ers[2 * F + j], F, qh, dh);
    free(h);
    return 0;
}

ORC_API void orc_expert_ffn(const uint8_t *ew4, const float *ers, int H, int F,
                            const int8_t *qx, const float *dx, int8_t *qh, float *dh, float *y,
                            float *g_out, float *u_out, float *h_out)
{
    (void)orc_expert_ffn_w(ew4, 4, ers, H, F, qx, dx, qh, dh, y, g_out, u_out, h_out);
}

/* ------------------------------------------------------------------------- */
/* O6  The whole layer: quantise, route, dispatch, experts, combine          */
/* ------------------------------------------------------------------------- */
/* out_t = y_shared,t + sum over r = 0..k-1 of w_{t,r} * y_{e_{t,r},t}, as
 * acc = y_shared; acc = fmaf(w_r, y_r, acc) in rank order.  The shared expert
 * has weight 1 (DeepSeek-V3 heritage; the pages are silent).  Expert weights
 * are given per expert (ew4[e], ers[e]); a NULL entry is allowed for an expert
 * no token selects, so callers may supply only the experts a sample touches.
 * Returns 0, -(1 + e) if a selected expert e was not supplied, or
 * ORC_E_WBITS for a container other than 4 or 8 bits.
 * Optional intermediates (NULL to skip): qx [T][H], dx [T][H/32], idx [T][k],
 * w [T][k], y_routed [T][k][H] (pair order), y_shared [T][H]. */
ORC_API int orc_moe_forward_w(const float *x, int T, int H, int F, int E, int k, float routed_scale,
                              const float *router_w, const float *router_b, int wbits,
                              const uint8_t *const *ew4, const float *const *ers,
                              const uint8_t *sw4, const float *srs, float *out,
                              int8_t *qx_out, float *dx_out, int32_t *idx_out, float *w_out,
                              float *yr_out, float *ys_out)
{
    if (wbits != 4 && wbits != 8) return ORC_E_WBITS;
    int8_t *qx = (int8_t *)malloc((size_t)T * H);
    float *dx = (float *)malloc(sizeof(float) * (size_t)T * (H / 32));
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    float *w = (float *)malloc(sizeof(float) * (size_t)T * k);
    float *yr = (float *)malloc(sizeof(float) * (size_t)T * k * H);
    float *ys = (float *)malloc(sizeof(float) * (size_t)T * H);
    int status = 0;

    for (int t = 0; t < T; ++t)
        orc_q8_0(x + (size_t)t * H, H, qx + (size_t)t * H, dx + (size_t)t * (H / 32));
    orc_route(x, T, H, router_w, router_b, E, k, routed_scale, idx, w, NULL, NULL);
    for (int p = 0; p < T * k; ++p)
        if (!ew4[idx[p]] || !ers[idx[p]]) { status = -(1 + idx[p]); goto done; }

    #pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < T * k + T; ++p) {
        int8_t *qh = (int8_t *)malloc((size_t)F);
        float *dh = (float *)malloc(sizeof(float) * (F / 32));
        if (p < T * k) {
            int t = p / k, e = idx[p];
            (void)orc_expert_ffn_w(ew4[e], wbits, ers[e], H, F, qx + (size_t)t * H, dx + (size_t)t * (H / 32),
                                   qh, dh, yr + (size_t)p * H, NULL, NULL, NULL);
        } else {
            int t = p - T * k;
            (void)orc_expert_ffn_w(sw4, wbits, srs, H, F, qx + (size_t)t * H, dx + (size_t)t * (H / 32),
                                   qh, dh, ys + (size_t)t * H, NULL, NULL, NULL);
        }
        free(qh); free(dh);
    }

    for (int t = 0; t < T; ++t)
        for (int j = 0; j < H; ++j) {
            float acc = ys[(size_t)t * H + j];
            for (int r = 0; r < k; ++r)
                acc = fmaf(w[(size_t)t * k + r], yr[((size_t)t * k + r) * H + j], acc);
            out[(size_t)t * H + j] = acc;
        }

    if (qx_out) memcpy(qx_out, qx, (size_t)T * H);
    if (dx_out) memcpy(dx_out, dx, sizeof(float) * (size_t)T * (H / 32));
    if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * k);
    if (w_out) memcpy(w_out, w, sizeof(float) * (size_t)T * k);
    if (yr_out) memcpy(yr_out, yr, sizeof(float) * (size_t)T * k * H);
    if (ys_out) memcpy(ys_out, ys, sizeof(float) * (size_t)T * H);
done:
    free(qx); free(dx); free(idx); free(w); free(yr); free(ys);
    return status;
}

ORC_API int orc_moe_forward(const float *x, int T, int H, int F, int E, int k, float routed_scale,
                            const float *router_w, const float *router_b,
                            const uint8_t *const *ew4, const float *const *ers,
                            const uint8_t *sw4, const float *srs, float *out,
                            int8_t *qx_out, float *dx_out, int32_t *idx_out, float *w_out,
                            float *yr_out, float *ys_out)
{
    return orc_moe_forward_w(x, T, H, F, E, k, routed_scale, router_w, router_b, 4, ew4, ers, sw4, srs, out,
                             qx_out, dx_out, idx_out, w_out, yr_out, ys_out);
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP), and a
 * setter (n <= 0 restores the default); results do not depend on it. */
#ifdef _OPENMP
#include <omp.h>
static int orc_default_threads = 0;
ORC_API int orc_num_threads(void) { return omp_get_max_threads(); }
ORC_API void orc_set_threads(int n)
{
    if (orc_default_threads == 0) orc_default_threads = omp_get_max_threads();
    omp_set_num_threads(n > 0 ? n : orc_default_threads);
}
#else
ORC_API int orc_num_threads(void) { return 1; }
ORC_API void orc_set_threads(int n) { (void)n; }
#endif
