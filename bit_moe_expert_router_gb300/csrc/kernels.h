// Internal launchers of the W4A8 MoE kernels (host side; no argument checks --
// the C ABI in api.cu validates everything before calling these).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Router: ids/wts [T][k] from logits [T][E].
// ids [T][k] <- ids_in clamped into [0, E), wts <- wts_in (a routing supplied by the caller).
cudaError_t launch_route_supplied(const int32_t* ids_in, const float* wts_in, int64_t T, int64_t E, int64_t k,
                                  int32_t* ids, float* wts, cudaStream_t st);
cudaError_t launch_route_topk(const float* logits, int64_t T, int64_t E, int64_t k, int32_t* ids, float* wts,
                              cudaStream_t st);

// Counting sort of n = T*k pair ids (values < E) plus the grouped-GEMM tile
// schedule over E + S slots (shared slot s covers rows Tk + s*T .. + T).
// tok_map (optional): token of flattened pair i; default i / k.
struct SortArgs {
    const int32_t* ids;
    int64_t T, k, E, S;
    const int32_t* tok_map;
    // outputs in the workspace
    int32_t* chunk_counts;
    int32_t* seg_cnt;
    int32_t* seg_off;
    int32_t* perm;
    int32_t* inv;
    int32_t* row_token;
    int32_t* tile_slot;
    int32_t* tile_row0;
    Header* hdr;
    uint32_t* amax;      // cleared for all P rows (may be null)
    int64_t P;
    // optional copies for the API (may be null)
    int32_t* counts_out;
    int32_t* offsets_out;
};
cudaError_t launch_sort(const SortArgs& a, cudaStream_t st);

// Copy of up to kStageBufs buffers (byte counts multiples of 4, addresses
// 16-byte aligned) by one kernel; sources may be host memory mapped into
// the device address space, read once over the host link.
constexpr int kStageBufs = 3;
struct StageArgs {
    const void* src[kStageBufs];
    void* dst[kStageBufs];
    int64_t bytes[kStageBufs];
};
cudaError_t launch_stage_copy(const StageArgs& a, cudaStream_t st);

// S0 of bf16 activations [T][H] (bit patterns): per token s = max|x| / 127,
// q = clamp(RNE(x / s), -127, 127) in IEEE fp32; an all-zero row gives s = 0.
cudaError_t launch_quantize_bf16(const uint16_t* x, int64_t T, int64_t H, int8_t* x_q, float* x_scale,
                                 cudaStream_t st);

enum class Gemm1Mode { kHidden, kPartials };
enum class Gemm2Mode { kOutput, kPartials };

struct Gemm1Args {
    const int8_t* x_q;
    const float* x_scale;    // kHidden only
    const uint8_t* w13;
    const float* s13;        // kHidden only
    int64_t T, H, I, g;      // rows naming a token >= T read zeros
    const int32_t* seg_off;
    const int32_t* seg_cnt;
    const int32_t* row_token;
    const int32_t* tile_slot;
    const int32_t* tile_row0;
    const Header* hdr;
    float* h;                // [P][I]      kHidden
    uint32_t* amax;          // [P]         kHidden
    int32_t* p1;             // [P][2I][H/g] kPartials
};
cudaError_t launch_gemm1(Gemm1Mode mode, const Gemm1Args& a, int max_tiles, cudaStream_t st);

struct Gemm2Args {
    const float* h;          // [P][I] fp32 (kOutput) ...
    const uint32_t* amax;    // ... with its row maxima
    const int8_t* h_q;       // [P][I] int8 (kPartials)
    const uint8_t* w2;
    const float* s2;         // kOutput only
    int64_t H, I, g;
    const int32_t* seg_off;
    const int32_t* seg_cnt;
    const int32_t* tile_slot;
    const int32_t* tile_row0;
    const Header* hdr;
    float* y;                // [P][H]      kOutput
    int32_t* p2;             // [P][H][I/g] kPartials
};
cudaError_t launch_gemm2(Gemm2Mode mode, const Gemm2Args& a, int max_tiles, cudaStream_t st);

struct CombineArgs {
    const float* y;          // [P][H]
    const float* wts;        // [T][k]
    const int32_t* inv;      // [T*k]
    int64_t T, H, k, S;
    float* out;              // [T][H]
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

// Debug copies of the requantised intermediate: h_q [P][I], s_h [P].
cudaError_t launch_requant_copy(const float* h, const uint32_t* amax, int64_t P, int64_t I, int8_t* h_q, float* s_h,
                                cudaStream_t st);

int num_sms();

}  // namespace moe
