// Fused decode engine (decode.cu): launcher interface.
#pragma once

#include "kernels.h"

namespace moe {

constexpr int kDecodeMaxT = 32;        // tokens per launch
constexpr int kDecodeMaxPairs = 512;   // routed (or listed) pair rows per launch (< kFlagWords slots)
constexpr int kMaxI = 2048;            // expert intermediate size (I / 512 in {1, 3})

enum class DecodeMode { kForward, kGemm1Partials, kGemm2Partials };

struct DecodeArgs {
    const int8_t* x_q;
    const float* x_scale;
    const uint16_t* x_bf16;  // forward: bf16 activations [T][H] quantised in the kernel (x_q / x_scale unused), or null
    const float* logits;
    const int32_t* ids_in;   // forward: routing supplied by the caller ([T][k] ids, clamped to [0, E)), or null
    const float* wts_in;     //          its weights [T][k] (logits unused)
    const uint8_t* slot_bits;  // forward: code width of each bank slot [E+S] (2 or 4), or null (all 4)
    const int64_t* w13_off;    // forward with slot_bits: compact storage, slot e's gate/up rows at w13 + w13_off[e]
    const int64_t* w2_off;     //   and its down rows at w2 + w2_off[e], each row at its slot's width; or null
    const uint8_t* w13;
    const float* s13;
    const uint8_t* w2;
    const float* s2;
    int T, H, I, E, S, k, g;
    // pair-list modes (pairs sorted by slot)
    const int32_t* pair_token;
    const int32_t* pair_slot;
    int n_pairs;
    const int8_t* h_q_in;    // [n_pairs][I] (gemm2 partials)
    // outputs
    float* out;              // [T][H]
    int32_t* p1;             // [n_pairs][2I][H/g]
    int32_t* p2;             // [n_pairs][H][I/g]
    // workspace
    Header* hdr;
    uint32_t* row_max;       // [P] running max |h| per pair row (float bits), cleared before the launch
    int8_t* hq_g;            // [P][I] requantised rows, each 8-byte group split even|odd
    float* sh_g;             // [P] their scales
    float* h;                // [P][I]
    uint32_t* amax;          // [P] row maxima (debug copies; may be null)
    float* y;                // [P][H] (debug copies; may be null)
    // the routing of the launch (debug copies, written by CTA 0; may be null): ids and weights
    // [T][k], perm [T*k] (pair row -> pair) and inv [T*k] (pair -> pair row)
    int32_t* ids_out;
    float* wts_out;
    int32_t* perm_out;
    int32_t* inv_out;
};

// Byte offsets of the shared-memory arrays of one launch.
struct DecodePlan {
    int rows_pc;      // down-projection output rows per CTA
    int smem_slots;   // slots whose down-projection slice is staged in shared memory
    int smem_bytes;
    int off_ids, off_wts, off_pos, off_pair_of, off_row_tok, off_slot_e, off_slot_row0, off_slot_cnt, off_slot_bw, off_slot_cum,
        off_n_slots, off_xs, off_sh, off_x, off_xm, off_hq, off_y, off_first, off_eqc, off_wmax, off_w2bar, off_row_slot, off_w2s;
};

// mixed: the forward kernel for mixed 2/4-bit banks (a second activation staging area).
bool decode_plan(int64_t T, int64_t H, int64_t I, int64_t E, int64_t S, int64_t k, int64_t g, int64_t n_pairs,
                 DecodeMode mode, int grid, int max_smem, DecodePlan* out, bool mixed = false);
bool decode_shape_supported(int64_t H, int64_t I);
int decode_grid();
int decode_max_smem();
cudaError_t launch_decode(DecodeMode mode, const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st);
cudaError_t launch_barrier_timeout_probe(Header* hdr, cudaStream_t st);

}  // namespace moe
