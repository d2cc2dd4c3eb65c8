/*
 * CPU oracle of the routed-expert W4A8 MoE layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * and reference legs may load this library.  The product path never calls
 * it, and it shares no code with the CUDA kernels: everything below is a
 * plain, slow restatement of what the layer computes, one (token, expert)
 * pair at a time, in fp64 except where an integer is decided.
 *
 * Source: "Two 96 GB Ascend cards run Qwen3.8 Flash-Next" (ai-pulse-lab.com,
 * 2026-10-03), section 3 "Keep low-bit weights packed and do the work on the
 * NPU": tokens are routed to experts on the device, the grouped expert
 * projections run on the packed W4 bank with fused gate/up handling, blocked
 * (per-group) reduction and W4A8 execution, instead of expanding the bank;
 * the same section's eager reference dequantises the packed weights and
 * calls a plain matmul.  The page gives no formulas; the numeric details
 * below are the workloads' stated recipe, and where that is silent the
 * plainest reading (each one is named at the function that takes it).
 *
 * Steps (notation: T tokens, H hidden, I expert intermediate, E routed
 * experts, S shared experts, k = top_k, g = int4 group along K):
 *   route     top-k of the logits (descending, ties to the lower index),
 *             softmax over the selected k (= softmax, top-k, renormalise);
 *   permute   stable counting sort of the flattened pairs i = t*k + j by
 *             expert id: counts, exclusive offsets, perm, inverse;
 *   gemm1     per pair p = (t, e), row n < 2I, group q:
 *             P1[n][q] = sum_{k in q} x_q[t][k] * W13[e][n][k]   (int32),
 *             G[n] = x_scale[t] * sum_q s13[e][n][q] * P1[n][q];
 *   act       h[i] = SiLU(G[i]) * G[I + i], SiLU(z) = z / (1 + e^-z);
 *   requant   s_h = max_i |h[i]| / 127, h_q = clamp(RNE(h / s_h), -127, 127);
 *   gemm2     P2[n][q] = sum_{k in q} h_q[k] * W2[e][n][k],
 *             Y[n] = s_h * sum_q s2[e][n][q] * P2[n][q];
 *   combine   out[t] = sum_j w[t][j] * Y(t, ids[t][j]) + sum_s Y(t, E + s).
 *
 * Compiled with -std=c11 -ffp-contract=off (no fused multiply-add), so the
 * results do not depend on the host architecture or the thread count.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* Packed int4 storage: element 2j in the low nibble of byte j, element
 * 2j+1 in the high nibble, two's complement (sign-extended on unpack). */
int orc_unpack(uint8_t byte, int high) {
    int v = high ? (byte >> 4) & 0xF : byte & 0xF;
    return v >= 8 ? v - 16 : v;
}

/*
 * Packed 2-bit storage (mixed 2/4-bit banks): element 4j + p sits in bits
 * 2p, 2p+1 of byte j of the row, a two's-complement 2-bit number in [-2, 1]
 * (the same low-bits-first order as the 4-bit packing).  A 2-bit row keeps
 * the 4-bit row's length, K/2 bytes, of which the first K/4 hold the codes
 * (reading: the storage of a slot does not depend on its width, so one bank
 * array serves both; only the bytes read halve).
 */
int orc_unpack2(uint8_t byte, int pos) {
    int v = (byte >> (2 * pos)) & 0x3;
    return v >= 2 ? v - 4 : v;
}

/* Code k of a packed row of `bits` (4 or 2) bits per code. */
static int code_at(const uint8_t* row, int64_t k, int bits) {
    return bits == 2 ? orc_unpack2(row[k >> 2], (int)(k & 3)) : orc_unpack(row[k >> 1], (int)(k & 1));
}

/*
 * route: for each token choose k experts by repeated scans for the largest
 * remaining logit (a strictly larger value replaces the candidate, so equal
 * values keep the lower index; -0.0 and +0.0 compare equal).  A NaN logit
 * ranks below every number and NaNs among themselves by index (reading: the
 * page is silent on invalid logits; this keeps k distinct experts per token).  Selecting on
 * the logits picks the same set as selecting on the softmax probabilities,
 * because exp is increasing.  Weights: exp(l_j - m) / sum over the selected
 * of exp(l - m), m the largest selected logit -- the renormalised top-k of
 * the full softmax, since the full denominator cancels.
 */
int orc_route(int64_t T, int64_t E, int64_t k, const float* logits, int32_t* ids, double* w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return 1;
    char* taken = (char*)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best] || (isnan(l[best]) && !isnan(l[e]))) best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
        }
        double m = (double)l[ids[t * k]];
        double den = 0.0;
        for (int64_t j = 0; j < k; ++j) den += exp((double)l[ids[t * k + j]] - m);
        for (int64_t j = 0; j < k; ++j) w[t * k + j] = exp((double)l[ids[t * k + j]] - m) / den;
    }
    free(taken);
    return 0;
}

/*
 * permute: counting sort of the T*k flattened pairs by expert id, stable in
 * the flattened index.  counts[e] pairs go to expert e; offsets is the
 * exclusive prefix sum (E+1 entries, offsets[E] = T*k); perm[pos] is the
 * flattened pair index at sorted position pos; inv[i] is the position of i.
 */
int orc_permute(int64_t T, int64_t E, int64_t k, const int32_t* ids,
                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv) {
    int64_t n = T * k;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return 1;
        counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = ids[i];
        int32_t pos = offsets[e] + cursor[e];
        cursor[e] += 1;
        perm[pos] = (int32_t)i;
        inv[i] = pos;
    }
    free(cursor);
    return 0;
}

/*
 * Per-group integer partial sums of one int8 activation row `a` (length K)
 * against `rows` packed weight rows of length K: P[n * (K/g) + q] =
 * sum over k in [q*g, (q+1)*g) of a[k] * code(W[n], k).  |P| <= g*127*8.
 */
void orc_partials_bits(const int8_t* a, int64_t K, const uint8_t* W, int64_t rows, int64_t g, int bits,
                       int32_t* P) {
    int64_t ng = K / g;
    for (int64_t n = 0; n < rows; ++n) {
        const uint8_t* row = W + n * (K / 2);
        for (int64_t q = 0; q < ng; ++q) {
            int32_t acc = 0;
            for (int64_t kk = q * g; kk < (q + 1) * g; ++kk) acc += (int32_t)a[kk] * code_at(row, kk, bits);
            P[n * ng + q] = acc;
        }
    }
}

void orc_partials(const int8_t* a, int64_t K, const uint8_t* W, int64_t rows, int64_t g, int32_t* P) {
    orc_partials_bits(a, K, W, rows, g, 4, P);
}

/* Dequantised row sums: out[n] = a_scale * sum_q s[n][q] * P[n][q] (fp64). */
static void combine_groups(const int32_t* P, const float* s, int64_t rows, int64_t ng, double a_scale, double* out) {
    for (int64_t n = 0; n < rows; ++n) {
        double acc = 0.0;
        for (int64_t q = 0; q < ng; ++q) acc += (double)s[n * ng + q] * (double)P[n * ng + q];
        out[n] = a_scale * acc;
    }
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * gemm1 + act for one pair: G (optional, 2I values) and h (I values).
 * w13e/s13e point at the expert's slot: rows [0, I) are the gate
 * projection, rows [I, 2I) the up projection (reading: the fused bank is
 * the plain concatenation gate-then-up).  P1 (optional) receives the int32
 * partials [2I][H/g].
 */
static void hidden_bits(const int8_t* x, float x_scale, const uint8_t* w13e, const float* s13e,
                        int64_t H, int64_t I, int64_t g, int bits, int32_t* P1, double* G, double* h) {
    int64_t ng = H / g;
    int32_t* P = P1 ? P1 : (int32_t*)malloc((size_t)(2 * I * ng) * sizeof(int32_t));
    double* Gv = G ? G : (double*)malloc((size_t)(2 * I) * sizeof(double));
    orc_partials_bits(x, H, w13e, 2 * I, g, bits, P);
    combine_groups(P, s13e, 2 * I, ng, (double)x_scale, Gv);
    for (int64_t i = 0; i < I; ++i) h[i] = orc_silu(Gv[i]) * Gv[I + i];
    if (!P1) free(P);
    if (!G) free(Gv);
}

void orc_hidden(const int8_t* x, float x_scale, const uint8_t* w13e, const float* s13e,
                int64_t H, int64_t I, int64_t g, int32_t* P1, double* G, double* h) {
    hidden_bits(x, x_scale, w13e, s13e, H, I, g, 4, P1, G, h);
}

/*
 * requant: symmetric int8 code per pair row (reading: one scale per
 * (token, expert) row, since each expert's intermediate is its own
 * vector).  The integer decision is taken in fp32, the precision of the
 * device kernels: h32 = fp32(h), s_h = max |h32| / 127 (fp32 division),
 * h_q = RNE(h32 / s_h) (fp32 division), clamped to [-127, 127]; an all-zero
 * row gets s_h = 0 and h_q = 0.
 */
void orc_requant(const double* h, int64_t I, int8_t* hq, float* sh) {
    float amax = 0.0f;
    for (int64_t i = 0; i < I; ++i) {
        float a = fabsf((float)h[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *sh = s;
    for (int64_t i = 0; i < I; ++i) {
        float q = (s > 0.0f) ? rintf((float)h[i] / s) : 0.0f;
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        hq[i] = (int8_t)q;
    }
}

/*
 * S0, the activations' quantisation, for callers that hand the layer bf16
 * activations: per token, s = max_h |x[t][h]| / 127 and
 * q = clamp(RNE(x / s), -127, 127), an all-zero row giving s = 0 and q = 0
 * (the same per-token symmetric int8 recipe as the workloads' inputs).
 * x holds bf16 bit patterns; each is widened exactly to fp32 (the 16 bits
 * become the high half of the fp32 word).  The integer decision is taken in
 * fp32, the precision of the device kernels: fp32 maximum, fp32 division
 * by 127, fp32 division x / s, round half to even.
 */
void orc_quantize_bf16(const uint16_t* x, int64_t T, int64_t H, int8_t* x_q, float* x_scale) {
    for (int64_t t = 0; t < T; ++t) {
        float amax = 0.0f;
        for (int64_t h = 0; h < H; ++h) {
            uint32_t bits = (uint32_t)x[t * H + h] << 16;
            float v;
            memcpy(&v, &bits, sizeof v);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float s = amax / 127.0f;
        x_scale[t] = s;
        for (int64_t h = 0; h < H; ++h) {
            uint32_t bits = (uint32_t)x[t * H + h] << 16;
            float v;
            memcpy(&v, &bits, sizeof v);
            float q = (s > 0.0f) ? rintf(v / s) : 0.0f;
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            x_q[t * H + h] = (int8_t)q;
        }
    }
}

/* gemm2 for one pair: Y[n] = s_h * sum_q s2[n][q] * P2[n][q]; P2 optional [H][I/g]. */
static void down_bits(const int8_t* hq, float sh, const uint8_t* w2e, const float* s2e,
                      int64_t H, int64_t I, int64_t g, int bits, int32_t* P2, double* y) {
    int64_t ng = I / g;
    int32_t* P = P2 ? P2 : (int32_t*)malloc((size_t)(H * ng) * sizeof(int32_t));
    orc_partials_bits(hq, I, w2e, H, g, bits, P);
    combine_groups(P, s2e, H, ng, (double)sh, y);
    if (!P2) free(P);
}

void orc_down(const int8_t* hq, float sh, const uint8_t* w2e, const float* s2e,
              int64_t H, int64_t I, int64_t g, int32_t* P2, double* y) {
    down_bits(hq, sh, w2e, s2e, H, I, g, 4, P2, y);
}

/* Y of one (token, slot) pair; hq/sh (optional) receive the requantised intermediate;
 * slot_bits (optional, [E+S], 2 or 4) gives each slot's code width (default 4). */
static void pair_output_bits(const orc_dims_t* d, const int8_t* x_q, const float* x_scale,
                             const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                             const uint8_t* slot_bits, int64_t t, int64_t slot, int8_t* hq_out, float* sh_out,
                             double* y) {
    int64_t H = d->H, I = d->I, g = d->group;
    int bits = slot_bits ? slot_bits[slot] : 4;
    double* h = (double*)malloc((size_t)I * sizeof(double));
    int8_t* hq = (int8_t*)malloc((size_t)I);
    float sh;
    hidden_bits(x_q + t * H, x_scale[t], w13 + slot * (2 * I) * (H / 2), s13 + slot * (2 * I) * (H / g),
                H, I, g, bits, NULL, NULL, h);
    orc_requant(h, I, hq, &sh);
    down_bits(hq, sh, w2 + slot * H * (I / 2), s2 + slot * H * (I / g), H, I, g, bits, NULL, y);
    if (hq_out) memcpy(hq_out, hq, (size_t)I);
    if (sh_out) *sh_out = sh;
    free(h);
    free(hq);
}

void orc_pair_output(const orc_dims_t* d, const int8_t* x_q, const float* x_scale,
                     const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                     int64_t t, int64_t slot, int8_t* hq_out, float* sh_out, double* y) {
    pair_output_bits(d, x_q, x_scale, w13, s13, w2, s2, NULL, t, slot, hq_out, sh_out, y);
}

/*
 * The whole layer for the listed tokens: out[r][:] for token tokens[r].
 * combine (reading: the shared expert is always on, with weight 1 and no
 * gate, added after the routed sum): out[t] = sum_j w[t][j] * Y(t, ids[t][j])
 * + sum_s Y(t, E + s), summed in that fixed order in fp64.  Each token only
 * needs its own routing, so a sample of tokens costs only its own pairs.
 */
int orc_forward_tokens_mixed(const orc_dims_t* d, const int8_t* x_q, const float* x_scale, const float* logits,
                             const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                             const uint8_t* slot_bits, int64_t n_sel, const int64_t* tokens, double* out) {
    int64_t H = d->H, E = d->E, k = d->top_k;
    if (d->T < 0 || d->H < 1 || d->I < 1 || E < 1 || k < 1 || k > E || d->n_shared < 0 || d->group < 1 ||
        d->H % d->group || d->I % d->group || d->group % 2)
        return 1;
    for (int64_t r = 0; r < n_sel; ++r)
        if (tokens[r] < 0 || tokens[r] >= d->T) return 1;
    int bad = 0;
    #pragma omp parallel for schedule(dynamic, 1) reduction(|:bad)
    for (int64_t r = 0; r < n_sel; ++r) {
        int64_t t = tokens[r];
        int32_t* ids = (int32_t*)malloc((size_t)k * sizeof(int32_t));
        double* w = (double*)malloc((size_t)k * sizeof(double));
        double* y = (double*)malloc((size_t)H * sizeof(double));
        double* o = out + r * H;
        if (orc_route(1, E, k, logits + t * E, ids, w)) bad = 1;
        for (int64_t n = 0; n < H; ++n) o[n] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            pair_output_bits(d, x_q, x_scale, w13, s13, w2, s2, slot_bits, t, ids[j], NULL, NULL, y);
            for (int64_t n = 0; n < H; ++n) o[n] += w[j] * y[n];
        }
        for (int64_t s = 0; s < d->n_shared; ++s) {
            pair_output_bits(d, x_q, x_scale, w13, s13, w2, s2, slot_bits, t, E + s, NULL, NULL, y);
            for (int64_t n = 0; n < H; ++n) o[n] += y[n];
        }
        free(ids);
        free(w);
        free(y);
    }
    return bad;
}

int orc_forward_tokens(const orc_dims_t* d, const int8_t* x_q, const float* x_scale, const float* logits,
                       const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                       int64_t n_sel, const int64_t* tokens, double* out) {
    return orc_forward_tokens_mixed(d, x_q, x_scale, logits, w13, s13, w2, s2, NULL, n_sel, tokens, out);
}
