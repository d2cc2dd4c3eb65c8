// tcgen05 grouped-GEMM engine (prefill_tc.cu): launcher interface.
#pragma once

#include <cuda_fp16.h>

#include "kernels.h"

namespace moe {

constexpr int kTcMaxSlots = 1039;  // bank slots (E + S) one launch can group

enum class TcMode { kGateUp, kDown, kGateUpPartials, kDownPartials };

struct TcArgs {
    // A operand: packed int4 weight rows of every bank slot with their group scales
    const uint8_t* w;         // [slots][rows_per_slot][K/2]
    const float* ws;          // [slots][rows_per_slot][K/g]
    int64_t rows_per_slot;    // 2I (gate/up) or H (down)
    int64_t K;                // H (gate/up) or I (down)
    int g;
    int64_t I, H;
    // B operand: fp16 rows (K order permuted inside 8-value groups), by pair row
    const __half* b;          // [rows][K]
    const int32_t* b_row;     // pair row -> row of b_scale (null: identity)
    int64_t b_rows;           // rows of b; a B row outside [0, b_rows) reads zeros
    const float* b_scale;     // gate/up: per B row (x_scale); down: per pair row (s_h)
    // grouping of the pair rows by bank slot
    const int32_t* seg_off;
    const int32_t* seg_cnt;
    int n_slots;
    // outputs
    float* h;                 // [P][I]        gate/up
    float* y;                 // [P][H]        down
    int32_t* partials;        // [P][rows_per_slot][K/g]  partials modes
    Header* hdr;              // status word for the bounded waits
};

bool tc_supported(int64_t H, int64_t I, int64_t g);
cudaError_t launch_tc_gemm(TcMode mode, const TcArgs& a, cudaStream_t st);

// x_q int8 [T][H] -> fp16 [rows][H] in the engine's K order, row r taken from
// token row_token[r] (null: r); a token outside [0, T) gives a zero row.
cudaError_t launch_prep_x16(const int8_t* x_q, int64_t T, int64_t H, const int32_t* row_token, int64_t rows, __half* x16,
                            cudaStream_t st);
// h fp32 [P][I] -> row maxima of |h| (amax bits [P]), s_h [P] and the requantised codes as fp16
// [P][I] in the engine's K order; with h null, the int8 codes `hq_in` [P][I] are converted as given.
cudaError_t launch_prep_h16(const float* h, uint32_t* amax, const int8_t* hq_in, int64_t P, int64_t I, __half* h16,
                            float* s_h, cudaStream_t st);

}  // namespace moe
