// Shared device helpers and the workspace layout of the W4A8 MoE layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_w4a8.h"

namespace moe {

constexpr int kWarp = 32;
constexpr int kChunk = 256;    // pairs per chunk of the counting sort (one scatter warp each)
constexpr int kTileM = 64;     // pair rows per grouped-GEMM tile
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxShared = 8;
constexpr int kMaxGroup = 256;
constexpr int kMaxDim = 65536;  // largest H and I: keeps every workspace size far from overflow

// Status word values written by device code into the workspace header.
constexpr uint32_t kDevOk = 0;
constexpr uint32_t kDevTimeout = 1;

// ---------------------------------------------------------------- workspace
// Every array starts on a 256-byte boundary.  Sizes follow the layer dims;
// P = T*k + T*S pair rows.  The header holds device-side counters.
struct Header {
    uint32_t status;        // kDevOk / kDevTimeout
    uint32_t n_tiles;       // grouped-GEMM m-tiles of this call
    uint32_t bar_arrive;    // grid barriers: arrivals so far (fused decode kernel)
    uint32_t pad[61];
};

constexpr int kFlagWords = 1024;  // per-call words after the header, cleared with it (decode: row maxima)

struct WsLayout {
    int64_t Tk = 0, P = 0, n_chunks = 0, max_tiles = 0, slots = 0;
    size_t hdr = 0, flags = 0, ids = 0, wts = 0, seg_cnt = 0, seg_off = 0, perm = 0, inv = 0, row_token = 0,
           chunk_counts = 0, tile_slot = 0, tile_row0 = 0, amax = 0, h = 0, hq = 0, sh = 0, y = 0, x16 = 0, h16 = 0,
           total = 0;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t S, int64_t k) {
    WsLayout L;
    L.Tk = T * k;
    L.P = T * k + T * S;
    L.slots = E + S;
    L.n_chunks = (L.Tk + kChunk - 1) / kChunk;
    L.max_tiles = (L.P + kTileM - 1) / kTileM + L.slots;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.hdr = take(sizeof(Header));
    L.flags = take(sizeof(uint32_t) * kFlagWords);
    L.ids = take(sizeof(int32_t) * L.Tk);
    L.wts = take(sizeof(float) * L.Tk);
    L.seg_cnt = take(sizeof(int32_t) * L.slots);
    L.seg_off = take(sizeof(int32_t) * (L.slots + 1));
    L.perm = take(sizeof(int32_t) * L.Tk);
    L.inv = take(sizeof(int32_t) * L.Tk);
    L.row_token = take(sizeof(int32_t) * L.P);
    L.chunk_counts = take(sizeof(int32_t) * L.n_chunks * E);
    L.tile_slot = take(sizeof(int32_t) * L.max_tiles);
    L.tile_row0 = take(sizeof(int32_t) * L.max_tiles);
    L.amax = take(sizeof(uint32_t) * L.P);
    L.h = take(sizeof(float) * L.P * I);
    L.hq = take(static_cast<size_t>(L.P) * I);
    L.sh = take(sizeof(float) * L.P);
    L.y = take(sizeof(float) * L.P * H);
    // tcgen05 engine operands (fp16), by pair row: the gathered activations and the requantised h
    L.x16 = take(2 * static_cast<size_t>(L.P) * H);
    L.h16 = take(2 * static_cast<size_t>(L.P) * I);
    L.total = o;
    return L;
}

template <typename T>
inline T* ws_at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes = 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Packed int4 word (8 codes, element 2j in the low nibble of byte j) ->
// two words of four int8 lanes holding 16 * code: `even` has elements
// 0,2,4,6 and `odd` elements 1,3,5,7.  Moving each nibble into the high
// half of its byte makes the byte's two's-complement value 16 * code, so no
// sign extension is needed; dot products come out 16x and are shifted back.
__device__ __forceinline__ void unpack_int4x8_x16(uint32_t w, uint32_t& even, uint32_t& odd) {
    even = (w << 4) & 0xF0F0F0F0u;
    odd = w & 0xF0F0F0F0u;
}

// Eight consecutive int8 values (two words) -> their even and odd elements.
__device__ __forceinline__ void deinterleave_int8x8(uint32_t w0, uint32_t w1, uint32_t& even, uint32_t& odd) {
    even = __byte_perm(w0, w1, 0x6420);
    odd = __byte_perm(w0, w1, 0x7531);
}

// D = A(16x32 s8, row) * B(32x8 s8, col) + C, int32 accumulate.
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Requantisation scale and code, decided in fp32 with IEEE division.
__device__ __forceinline__ float requant_scale(uint32_t amax_bits) {
    return __fdiv_rn(__uint_as_float(amax_bits), 127.0f);
}
__device__ __forceinline__ int requant_code(float h, float s) {
    if (!(s > 0.0f)) return 0;
    float q = rintf(__fdiv_rn(h, s));
    q = fminf(fmaxf(q, -127.0f), 127.0f);
    return static_cast<int>(q);
}

// The same code from s and its reciprocal rs = 1 / s (correctly rounded): h * rs
// is within 2^-23 relative of h / s (|h / s| <= 127), so it rounds to the same
// integer unless it lies within 1e-4 of a half-integer; only then is the exact
// division computed.  The rare exact path is kept out of line (the run-once
// code of a launch is fetched cold, so it is kept small).
static __device__ __noinline__ float rint_div_exact(float h, float s) { return rintf(__fdiv_rn(h, s)); }

__device__ __forceinline__ int requant_code_fast(float h, float s, float rs) {
    if (!(s > 0.0f)) return 0;
    const float f = h * rs;
    const float d = fabsf(f - floorf(f) - 0.5f);
    float q = rintf(f);
    if (d < 1e-4f) q = rint_div_exact(h, s);
    q = fminf(fmaxf(q, -127.0f), 127.0f);
    return static_cast<int>(q);
}

}  // namespace moe
