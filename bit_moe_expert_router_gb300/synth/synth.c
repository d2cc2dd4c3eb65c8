/*
 * Seeded synthetic inputs for the routed-expert W4A8 MoE layer.
 *
 * This module only produces the data the layer consumes: random deviates,
 * the bf16-rounded activations and their per-token int8 code, router logits
 * with the workloads' popularity biases, and the packed int4 expert bank.
 * It holds none of the layer's own arithmetic (routing, grouping, the
 * projections, the activation, the requantisation or the combine); both the
 * CPU oracle and the CUDA path consume what it writes.
 *
 * Random numbers: SplitMix64 (S. Vigna, public-domain reference, 2015) used
 * as a counter-based generator, value(stream, i) = mix(base(stream) +
 * (i + 1) * gamma), so every element depends only on (seed, stream, index)
 * and any thread count gives the same bytes.  Normal deviates come from the
 * Box-Muller transform (Box & Muller, 1958) on consecutive pairs.
 *
 * Packed int4 format (the bank's storage format): two signed 4-bit codes
 * per byte, element 2j in the low nibble and element 2j+1 in the high
 * nibble, two's complement.  Scales are fp32, one per (row, K-group).
 *
 * Compiled with -std=c11 -ffp-contract=off so that no multiply-add is fused
 * on either host architecture.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Base of stream `stream` under `seed`. */
uint64_t synth_stream_base(uint64_t seed, uint64_t stream) {
    return sm_mix(sm_mix(seed + SM_GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

uint64_t synth_u64(uint64_t base, uint64_t i) { return sm_mix(base + (i + 1) * SM_GAMMA); }

/* Uniform in the open interval (0, 1): 53 random bits, centred in their cell. */
static inline double u01(uint64_t base, uint64_t i) {
    return ((double)(synth_u64(base, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal deviate number i of the stream (Box-Muller, pair i/2). */
static inline double normal_at(uint64_t base, uint64_t i) {
    uint64_t j = i & ~1ULL;
    double u1 = u01(base, j), u2 = u01(base, j + 1);
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (i & 1ULL) ? r * sin(a) : r * cos(a);
}

/* out[i] = sigma * deviate (first + i), i < n: both members of each Box-Muller pair at once. */
static void fill_normals(uint64_t base, uint64_t first, int64_t n, double sigma, float* out) {
    int64_t i = 0;
    if ((first & 1ULL) && n > 0) { out[0] = (float)(sigma * normal_at(base, first)); i = 1; }
    for (; i + 1 < n; i += 2) {
        uint64_t j = first + (uint64_t)i;
        double r = sqrt(-2.0 * log(u01(base, j)));
        double a = 6.283185307179586476925286766559 * u01(base, j + 1);
        out[i] = (float)(sigma * (r * cos(a)));
        out[i + 1] = (float)(sigma * (r * sin(a)));
    }
    if (i < n) out[i] = (float)(sigma * normal_at(base, first + (uint64_t)i));
}

/* n normal deviates of the stream, starting at index first, times sigma, as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, int64_t n, double sigma, float* out) {
    uint64_t base = synth_stream_base(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(sigma * normal_at(base, first + (uint64_t)i));
}

/* n uniform deviates in (0,1) (fp64), used for seeded choices and permutations. */
void synth_uniform_f64(uint64_t seed, uint64_t stream, int64_t n, double* out) {
    uint64_t base = synth_stream_base(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = u01(base, (uint64_t)i);
}

/* fp32 -> bf16 with round-to-nearest-even, returned as fp32 (NaN not expected). */
static inline float round_bf16(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;
    float r;
    memcpy(&r, &b, 4);
    return r;
}

/*
 * Activations: x[t, :] ~ N(0,1) (stream 1) -> fp32 -> bf16 (RNE), then the
 * per-token symmetric int8 code: s = absmax / 127 (fp32), q = RNE(x / s) in
 * fp32, clamped to [-127, 127]; an all-zero row gets s = 0 and q = 0.
 * x_bf16 (optional, may be NULL) receives the bf16-rounded values as fp32.
 */
void synth_activations(uint64_t seed, int64_t T, int64_t H, int8_t* x_q, float* x_scale, float* x_bf16) {
    uint64_t base = synth_stream_base(seed, 1);
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        float* row = (float*)malloc((size_t)H * sizeof(float));
        float amax = 0.0f;
        fill_normals(base, (uint64_t)(t * H), H, 1.0, row);
        for (int64_t h = 0; h < H; ++h) {
            float v = round_bf16(row[h]);
            row[h] = v;
            float a = fabsf(v);
            if (a > amax) amax = a;
            if (x_bf16) x_bf16[t * H + h] = v;
        }
        float s = amax / 127.0f;
        x_scale[t] = s;
        for (int64_t h = 0; h < H; ++h) {
            float q = (s > 0.0f) ? rintf(row[h] / s) : 0.0f;
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            x_q[t * H + h] = (int8_t)q;
        }
        free(row);
    }
}

/*
 * One packed weight matrix of an expert slot: rows x K values ~ N(0, sigma)
 * drawn from `stream` at element offset (slot * rows + r) * K + k, quantised
 * per (row, K-group of g): s = absmax / qmax (fp32), q = clamp(RNE(w / s),
 * qlo, qhi); packed two per byte, low nibble first.  An all-zero group gets
 * s = 0 and q = 0.  codes (optional, may be NULL) receives the int8 codes.
 */
void synth_weight_matrix(uint64_t seed, uint64_t stream, int64_t slot, int64_t rows, int64_t K, int64_t g,
                         double sigma, int qmax, int qlo, int qhi,
                         uint8_t* packed, float* scales, int8_t* codes) {
    uint64_t base = synth_stream_base(seed, stream);
    int64_t ng = K / g;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float* w = (float*)malloc((size_t)K * sizeof(float));
        int8_t* q = (int8_t*)malloc((size_t)K);
        uint64_t off = (uint64_t)((slot * rows + r) * K);
        fill_normals(base, off, K, sigma, w);
        for (int64_t gi = 0; gi < ng; ++gi) {
            float amax = 0.0f;
            for (int64_t k = gi * g; k < (gi + 1) * g; ++k) {
                float a = fabsf(w[k]);
                if (a > amax) amax = a;
            }
            float s = amax / (float)qmax;
            scales[r * ng + gi] = s;
            for (int64_t k = gi * g; k < (gi + 1) * g; ++k) {
                float v = (s > 0.0f) ? rintf(w[k] / s) : 0.0f;
                if (v > (float)qhi) v = (float)qhi;
                if (v < (float)qlo) v = (float)qlo;
                q[k] = (int8_t)v;
            }
        }
        for (int64_t j = 0; j < K / 2; ++j)
            packed[r * (K / 2) + j] = (uint8_t)(((uint8_t)q[2 * j] & 0x0Fu) | (((uint8_t)q[2 * j + 1] & 0x0Fu) << 4));
        if (codes) memcpy(codes + r * K, q, (size_t)K);
        free(w);
        free(q);
    }
}
