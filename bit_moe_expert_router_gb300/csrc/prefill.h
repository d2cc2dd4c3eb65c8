// tcgen05 grouped-GEMM engine (prefill_tc.cu): launcher interface.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace moe {

constexpr int kTcMaxSlots = 1039;  // bank slots (E + S) one launch can group

// kGateUp      gate/up projection, h = SiLU(gate) * up written by pair row
// kDown        down projection, Y[pair row] = s_h * sum_q s2 P2 written in bf16 for the combine
// kDownY       the same Y in fp32 (checking copies)
// k*Partials   the int32 partial of every group, per pair row
enum class TcMode { kGateUp, kDown, kDownY, kGateUpPartials, kDownPartials };

struct TcArgs {
    // A operand: packed int4 weight rows of every bank slot with their group scales
    const uint8_t* w;         // [slots][rows_per_slot][K/2]
    const float* ws;          // [slots][rows_per_slot][K/g]
    const uint8_t* slot_bits; // code width of each slot (2 or 4), or null (all 4): a 2-bit row holds its
                              // K codes in its first K/4 bytes, element 4j + p in bits 2p, 2p+1 of byte j
    const int64_t* w_off;     // with slot_bits: compact storage, slot e's rows at w + w_off[e], each K/4
                              // (2-bit) or K/2 (4-bit) bytes after the one before; or null (K/2 stride)
    int64_t rows_per_slot;    // 2I (gate/up) or H (down)
    int64_t K;                // H (gate/up) or I (down)
    int g;
    int64_t I, H;
    // B operand, fp16 rows by pair row in the engine's K order (pairs (0,4) (1,5) (2,6) (3,7) of
    // every 8 values): the activations gathered per pair (gate/up) or the requantised h (down)
    const __half* b;          // [b_rows][K]
    int64_t b_rows;           // rows of b; a B row past the end reads zeros
    const float* b_scale;     // gate/up: x_scale by token (through row_token); down: s_h by pair row
    // grouping of the pair rows by bank slot
    const int32_t* seg_off;
    const int32_t* seg_cnt;
    const int32_t* row_token;  // pair row -> token
    int n_slots;
    // outputs
    float* h;                 // [P][I]        kGateUp
    __nv_bfloat16* yb;        // [P][H]        kDown
    float* y;                 // [P][H]        kDownY
    int32_t* partials;        // [P][rows_per_slot][K/g]  partials modes
    Header* hdr;              // status word for the bounded waits
};

bool tc_supported(int64_t H, int64_t I, int64_t g);
cudaError_t launch_tc_gemm(TcMode mode, const TcArgs& a, cudaStream_t st);

// x_q int8 [T][H] -> fp16 [rows][H] in the engine's K order, row r taken from token row_token[r]; a
// token outside [0, T) gives a zero row.
cudaError_t launch_prep_x16(const int8_t* x_q, int64_t T, int64_t H, const int32_t* row_token, int64_t rows, __half* x16,
                            cudaStream_t st);
// out[t] = sum_j wts[t][j] * Y[inv[t*k + j]] + sum_s Y[Tk + s*T + t] from bf16 Y [P][H], in that fixed
// order in fp32 (overwrites out).
cudaError_t launch_combine_bf16(const __nv_bfloat16* y, const float* wts, const int32_t* inv, int64_t T, int64_t H,
                                int64_t k, int64_t S, float* out, cudaStream_t st);
// h fp32 [P][I] -> row maxima of |h| (amax bits [P]), s_h [P] and the requantised codes as fp16
// [P][I] in the engine's K order; with h null, the int8 codes `hq_in` [P][I] are converted as given.
cudaError_t launch_prep_h16(const float* h, uint32_t* amax, const int8_t* hq_in, int64_t P, int64_t I, __half* h16,
                            float* s_h, cudaStream_t st);

}  // namespace moe
