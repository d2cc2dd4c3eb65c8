/*
 * CPU oracle of the routed-expert W4A8 MoE layer -- TEST INFRASTRUCTURE ONLY.
 * See oracle.c for the definitions and their sources.  Nothing in the
 * product path includes this header.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

typedef struct {
    int64_t T, H, I, E, n_shared, top_k, group;
} orc_dims_t;

int orc_unpack(uint8_t byte, int high);
int orc_unpack2(uint8_t byte, int pos);
int orc_route(int64_t T, int64_t E, int64_t k, const float* logits, int32_t* ids, double* w);
int orc_permute(int64_t T, int64_t E, int64_t k, const int32_t* ids,
                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv);
void orc_partials(const int8_t* a, int64_t K, const uint8_t* W, int64_t rows, int64_t g, int32_t* P);
void orc_partials_bits(const int8_t* a, int64_t K, const uint8_t* W, int64_t rows, int64_t g, int bits,
                       int32_t* P);
double orc_silu(double z);
void orc_hidden(const int8_t* x, float x_scale, const uint8_t* w13e, const float* s13e,
                int64_t H, int64_t I, int64_t g, int32_t* P1, double* G, double* h);
void orc_requant(const double* h, int64_t I, int8_t* hq, float* sh);
void orc_quantize_bf16(const uint16_t* x, int64_t T, int64_t H, int8_t* x_q, float* x_scale);
void orc_down(const int8_t* hq, float sh, const uint8_t* w2e, const float* s2e,
              int64_t H, int64_t I, int64_t g, int32_t* P2, double* y);
void orc_pair_output(const orc_dims_t* d, const int8_t* x_q, const float* x_scale,
                     const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                     int64_t t, int64_t slot, int8_t* hq_out, float* sh_out, double* y);
int orc_forward_tokens(const orc_dims_t* d, const int8_t* x_q, const float* x_scale, const float* logits,
                       const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                       int64_t n_sel, const int64_t* tokens, double* out);
int orc_forward_tokens_mixed(const orc_dims_t* d, const int8_t* x_q, const float* x_scale, const float* logits,
                             const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                             const uint8_t* slot_bits, int64_t n_sel, const int64_t* tokens, double* out);
#endif
