// Fused decode engine of the W4A8 MoE layer: one cooperative persistent launch.
//
// For small batches the layer is bound by the bytes of the touched experts'
// packed weights ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next", section 3:
// keep the W4 bank packed and do the work on the device; section 5: no host
// round trips inside the token loop, fused operators for decode steps made of
// many small launches).  One launch does everything and streams each touched
// expert's bytes from HBM once:
//
//   phase 0  every CTA routes all T tokens itself (the same deterministic
//            result in every CTA, so nothing is exchanged; one warp per token,
//            k rounds of a warp arg-max) while its other warps stage the
//            activations in shared memory (int8 input split even|odd; bf16
//            input quantised here first: S0, s = max|x| / 127, RNE codes);
//            then it groups the pairs stably by expert into pair rows and builds
//            the slot table (touched experts ascending, then the shared
//            experts; with each slot's code width for a mixed 2/4-bit bank)
//            from per-expert token masks and expert presence bits (a pair's
//            slot is a popcount of the presence bits below its expert, its row
//            in the slot a popcount of its expert's mask below its token), and
//            a per-slot cost prefix.
//   phase 1  gate/up projection with dp4a on the CUDA cores: units of two
//            intermediate indices (2 gate rows + the 2 matching up rows) of
//            one slot; each warp takes a contiguous unit range of equal cost
//            (streaming + per-token work, so the always-on shared expert's
//            multi-token units weigh more).  A warp loads one unit at a
//            time into registers (16-byte loads; lane l loads pieces l,
//            l + 32, ... of each row, so each warp load reads 512 contiguous
//            bytes) -- the other 15 warps of the SM cover its latency; each
//            lane folds the exact int32 sum of each piece with its group
//            scale, and a 4-row reduce-scatter across the warp (6 shuffles)
//            gives the row sums; h = SiLU(G_gate) * G_up goes to the workspace
//            and |h| into the warp's running row maximum in shared memory
//            (merged into the global row maxima with one atomic max per CTA
//            and row at the end of the phase).  2-bit slots (the MIXED
//            instantiation) load half-length rows and multiply them with a
//            second, mod-4 ordered copy of the activations.  Meanwhile each CTA
//            has the bulk-copy engine copy its slice of the down-projection
//            bank (its output rows of every touched slot) into shared memory,
//            or warms it in L2 where shared memory runs out.
//   barrier  grid barrier 1 (each CTA adds its arrival and polls the count;
//            bounded: on timeout the status word records it and the CTAs
//            leave).
//   phase 2  requantisation spread over the grid (row p on CTA p mod grid,
//            one warp: s_h = max/127 from the row maximum, RNE codes) into the
//            workspace; grid barrier 2; every CTA copies the P requantised
//            rows into shared memory, runs the down projection for its output
//            rows of every touched slot (one thread per (pair row, output
//            row), whole-K dot product) and combines
//            out[t][n] = sum_j w[t][j] Y[(t,j)][n] + shared in a fixed order:
//            no atomics on the output, deterministic.
//
// The same kernel serves the partials entry points (phase 1 or phase 2
// alone, pairs given as a list instead of routed); there each K group's
// int32 partial is summed in integers over the lanes of the group, so the
// bit-exact checks run through this engine's integer core.
//
// Unpack: a nibble moved into the high half of its byte is an int8 lane
// holding 16 * code (unpack_int4x8_x16), so dp4a sums are 16x and exact;
// the unpack yields even and odd elements, and the activations are stored
// with every 8-byte group split into its even and odd elements to match.
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "decode.h"

namespace moe {
namespace {

constexpr int kThreadsD = 512;
static_assert(kDecodeMaxPairs + kDecodeMaxT * kMaxShared <= kFlagWords, "row maxima live in the cleared words");
constexpr int kWarpsD = kThreadsD / 32;

// Bounded waits: give up after about one second of wall-clock time (the
// global timer), with an iteration cap as a second bound.
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kSpinCap = 1u << 26;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global to shared memory, its completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number `k` (1-based) of this launch; the arrival counter
// starts at zero (cleared before the launch).  Each CTA adds its arrival and
// polls the counter itself until all k * grid arrivals are in (one L2 round
// trip less than a separate release word written by the last arriver).
// Bounded: false on timeout.
__device__ bool grid_barrier(Header* hdr, uint32_t k) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(&hdr->bar_arrive, 1u);
        const uint32_t target = k * gridDim.x;
        const uint64_t t0 = global_ns();
        uint32_t it = 0;
        while (ld_acquire(&hdr->bar_arrive) < target) {
            if (++it > kSpinCap || global_ns() - t0 > kWaitNs) {
                atomicOr(&hdr->status, kDevTimeout);
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// Byte offset of row r of slot e in a packed bank of `rows` rows per slot and
// rb4 bytes per 4-bit row: the uniform layout (every row rb4 bytes), or the
// compact one (slot e at off[e], low four bits cleared so every 16-byte load
// stays aligned; rows at the slot's own width, rb4 / 2 for a 2-bit slot).
__device__ __forceinline__ int64_t bank_row(const int64_t* off, int64_t e, int64_t rows, int64_t r, int64_t rb4,
                                            bool two) {
    return off ? (__ldg(off + e) & ~int64_t(15)) + r * (two ? rb4 / 2 : rb4) : (e * rows + r) * rb4;
}

// Order-preserving 32-bit key of a float: larger float -> larger key; -0.0
// and +0.0 map to the same key (the sum with +0.0 turns -0.0 into +0.0).  A
// NaN gets key 1: below every number (-inf is 0x007FFFFF), above the 0 of a
// taken or absent expert, so NaNs are picked last, by index.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 1u;
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Bounded wait for the first phase of the slice-copy barrier; false (and the
// status word set) if it runs out.
__device__ bool w2_wait(uint64_t* bar, Header* hdr) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, 0)) return true;
        if ((it & 15) == 15) {
            const uint64_t t = global_ns();
            if (t0 == 0) t0 = t;
            if (t - t0 > kWaitNs || it > kSpinCap) {
                atomicOr(&hdr->status, kDevTimeout);
                return false;
            }
        }
    }
}

// Routing of all T tokens, one warp per token (tokens dealt over the
// CTA's warps).  Lane l holds the order keys of experts l, l + 32, ...
// (NJ * 32 >= E).  Exact top-k in (key desc, id asc) order by k rounds of a
// warp arg-max: each lane keeps its best untaken (key, id) -- strict > over
// its keys keeps the lowest id on ties -- the round's winner is the largest
// key, lowest id among the lanes holding it, and only the winning lane
// rescans its keys.  The code is short on purpose: it runs once per launch
// and is fetched cold.  Then the weights: softmax over the k selected
// logits, relative to the largest.  ids/wts: [T][k]; warps 0 .. nw-1 take part.
template <int NJ>
__device__ void route_tokens(const float* __restrict__ logits, int T, int E, int k, int* ids, float* wts, int nw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = warp; t < T; t += nw) {
        uint32_t key[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            // 0 is below every finite key, and k <= E real experts are always left
            key[j] = e < E ? order_key(__ldg(logits + static_cast<int64_t>(t) * E + e)) : 0u;
        }
        uint32_t bk = 0;
        int bj = 0;
        auto lane_best = [&]() {
            bk = key[0];
            bj = 0;
#pragma unroll
            for (int j = 1; j < NJ; ++j)
                if (key[j] > bk) {
                    bk = key[j];
                    bj = j;
                }
        };
        lane_best();
        for (int r = 0; r < k; ++r) {
            const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t mine = static_cast<uint32_t>(lane + 32 * bj);
            const uint32_t mi = __reduce_min_sync(0xffffffffu, bk == mk ? mine : 0xFFFFFFFFu);
            if (lane == 0) {
                ids[t * k + r] = static_cast<int>(mi);
                wts[t * k + r] = key_value(mk);
            }
            if (mine == mi) {  // the winner drops the taken key and rescans
#pragma unroll
                for (int j = 0; j < NJ; ++j)
                    if (j == bj) key[j] = 0u;
                lane_best();
            }
        }
        __syncwarp();
        // softmax over the selected logits, relative to the largest (position 0)
        const float my_v = lane < k ? wts[t * k + lane] : 0.0f;
        const float m = __shfl_sync(0xffffffffu, my_v, 0);
        const float ex = lane < k ? expf(my_v - m) : 0.0f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane < k) wts[t * k + lane] = ex / sum;
        __syncwarp();
    }
}

// 16 int8 -> the same 16 bytes with each 8-byte group split into its even
// elements (first word) and odd elements (second word).
__device__ __forceinline__ uint4 split16(uint4 v) {
    uint4 r;
    r.x = __byte_perm(v.x, v.y, 0x6420);
    r.y = __byte_perm(v.x, v.y, 0x7531);
    r.z = __byte_perm(v.z, v.w, 0x6420);
    r.w = __byte_perm(v.z, v.w, 0x7531);
    return r;
}

// 16 int8 -> the same 16 bytes in mod-4 order: word p holds elements p, p + 4,
// p + 8, p + 12 (the lanes a 2-bit word unpacks into with one shift and mask).
__device__ __forceinline__ uint4 mod4_16(uint4 v) {
    uint4 r;
    r.x = __byte_perm(__byte_perm(v.x, v.y, 0x0040), __byte_perm(v.z, v.w, 0x0040), 0x5410);
    r.y = __byte_perm(__byte_perm(v.x, v.y, 0x0051), __byte_perm(v.z, v.w, 0x0051), 0x5410);
    r.z = __byte_perm(__byte_perm(v.x, v.y, 0x0062), __byte_perm(v.z, v.w, 0x0062), 0x5410);
    r.w = __byte_perm(__byte_perm(v.x, v.y, 0x0073), __byte_perm(v.z, v.w, 0x0073), 0x5410);
    return r;
}

// 16 * (dot of 8 packed codes `w` with the 8 split activation bytes xe|xo) + acc.
__device__ __forceinline__ int dot8(uint32_t w, uint32_t xe, uint32_t xo, int acc) {
    uint32_t e, o;
    unpack_int4x8_x16(w, e, o);
    acc = __dp4a(static_cast<int>(xe), static_cast<int>(e), acc);
    return __dp4a(static_cast<int>(xo), static_cast<int>(o), acc);
}

// 16 * dot of 32 packed codes (uint4) with 32 split activation bytes (two uint4).
__device__ __forceinline__ int dot32(const uint4& w, const uint4& xa, const uint4& xb) {
    int acc = dot8(w.x, xa.x, xa.y, 0);
    acc = dot8(w.y, xa.z, xa.w, acc);
    acc = dot8(w.z, xb.x, xb.y, acc);
    return dot8(w.w, xb.z, xb.w, acc);
}

// Sixteen packed 2-bit codes (element 4j + p in bits 2p, 2p+1 of byte j) ->
// four int8 lane words holding 64 * code, in the split activation order:
// e0 = elements 0,2,4,6; o0 = 1,3,5,7; e1 = 8,10,12,14; o1 = 9,11,13,15.
// Each code is moved to bits 6-7 of its byte (byte_perm duplicates the
// source byte into the two lanes it feeds).
__device__ __forceinline__ void unpack_int2x16_x64(uint32_t w, uint32_t& e0, uint32_t& o0, uint32_t& e1, uint32_t& o1) {
    const uint32_t t0 = __byte_perm(w, 0u, 0x1100), t1 = __byte_perm(w, 0u, 0x3322);
    e0 = ((t0 << 6) & 0x00C000C0u) | ((t0 << 2) & 0xC000C000u);
    o0 = ((t0 << 4) & 0x00C000C0u) | (t0 & 0xC000C000u);
    e1 = ((t1 << 6) & 0x00C000C0u) | ((t1 << 2) & 0xC000C000u);
    o1 = ((t1 << 4) & 0x00C000C0u) | (t1 & 0xC000C000u);
}

// 64 * dot of 64 packed 2-bit codes (uint4) with 64 split activation bytes (four uint4).
__device__ __forceinline__ int dot64_2bit(const uint4& w, const uint4& xa, const uint4& xb, const uint4& xc,
                                          const uint4& xd) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    const uint4 xv[4] = {xa, xb, xc, xd};
    int acc = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t e0, o0, e1, o1;
        unpack_int2x16_x64(wv[i], e0, o0, e1, o1);
        acc = __dp4a(static_cast<int>(xv[i].x), static_cast<int>(e0), acc);
        acc = __dp4a(static_cast<int>(xv[i].y), static_cast<int>(o0), acc);
        acc = __dp4a(static_cast<int>(xv[i].z), static_cast<int>(e1), acc);
        acc = __dp4a(static_cast<int>(xv[i].w), static_cast<int>(o1), acc);
    }
    return acc;
}

struct Smem {
    int* ids;         // [rows]
    float* wts;       // [rows]
    int* pos;         // [rows] pair -> row
    int* pair_of;     // [rows] row -> pair
    int* row_tok;     // [P]
    int* slot_e;      // [MS]
    int* slot_row0;   // [MS]
    int* slot_cnt;    // [MS]
    int* slot_bw;     // [MS] code width of the slot (4, or 2 in a mixed bank)
    int* slot_cum;    // [MS + 1] phase-1 cost prefix
    int* n_slots;     // [1]
    float* xs;        // [T]
    float* sh;        // [P]
    uint8_t* x;       // [T][H + 16] split layout
    uint8_t* xm;      // [T][H + 16] mod-4 layout (mixed banks only)
    uint8_t* hq;      // [P][I + 16] split layout
    float* y;         // [P][rows_pc]
    int* first;       // [rows] pair is the first of its expert (by pair index)
    int* eqc;         // [rows] pairs with the same expert
    float* wmax;      // [warps][P] each warp's running max |h| per pair row
    int* row_slot;    // [P] slot of each pair row
    uint64_t* w2bar;  // completion of the down-projection slice copies
    uint8_t* w2s;     // [smem_slots][slot_stride] staged down-projection slices
};

__device__ Smem carve(uint8_t* base, const DecodePlan& pl) {
    Smem s;
    s.ids = reinterpret_cast<int*>(base + pl.off_ids);
    s.wts = reinterpret_cast<float*>(base + pl.off_wts);
    s.pos = reinterpret_cast<int*>(base + pl.off_pos);
    s.pair_of = reinterpret_cast<int*>(base + pl.off_pair_of);
    s.row_tok = reinterpret_cast<int*>(base + pl.off_row_tok);
    s.slot_e = reinterpret_cast<int*>(base + pl.off_slot_e);
    s.slot_row0 = reinterpret_cast<int*>(base + pl.off_slot_row0);
    s.slot_cnt = reinterpret_cast<int*>(base + pl.off_slot_cnt);
    s.slot_bw = reinterpret_cast<int*>(base + pl.off_slot_bw);
    s.slot_cum = reinterpret_cast<int*>(base + pl.off_slot_cum);
    s.n_slots = reinterpret_cast<int*>(base + pl.off_n_slots);
    s.xs = reinterpret_cast<float*>(base + pl.off_xs);
    s.sh = reinterpret_cast<float*>(base + pl.off_sh);
    s.x = base + pl.off_x;
    s.xm = base + pl.off_xm;
    s.hq = base + pl.off_hq;
    s.y = reinterpret_cast<float*>(base + pl.off_y);
    s.first = reinterpret_cast<int*>(base + pl.off_first);
    s.eqc = reinterpret_cast<int*>(base + pl.off_eqc);
    s.wmax = reinterpret_cast<float*>(base + pl.off_wmax);
    s.row_slot = reinterpret_cast<int*>(base + pl.off_row_slot);
    s.w2bar = reinterpret_cast<uint64_t*>(base + pl.off_w2bar);
    s.w2s = base + pl.off_w2s;
    return s;
}

// Phase-1 cost of one unit of a slot with `cnt` tokens (streaming + per-token work), in units fitted to
// measured per-CTA phase times: a 4-token unit of a 4-bit slot takes ~2.1x a 1-token unit.
__device__ __forceinline__ int unit_cost(int cnt, int bits) { return (bits == 2 ? 5 : 9) + 8 * cnt; }

// PC1 = H / 2048 (64-value pieces per lane per row), PC2 = I / 512 (16-value pieces per lane per row).
// MIXED (forward only): the bank mixes 2-bit and 4-bit slots (a.slot_bits); the plain
// instantiation carries none of the 2-bit code.
template <DecodeMode MODE, int PC1, int PC2, bool MIXED = false>
__global__ void __launch_bounds__(kThreadsD, 1) decode_kernel(DecodeArgs a, DecodePlan pl) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const Smem s = carve(smem_raw, pl);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the shape is a template parameter (the host checks a.H and a.I against it),
    // so the index arithmetic below divides by constants
    constexpr int H = 2048 * PC1, I = 512 * PC2;
    const int T = a.T, k = a.k, g = a.g;
    const int ng1 = H / g, ng2 = I / g;
    constexpr int XS = H + 16, HQS = I + 16;
    constexpr int RS = I / 2 + 16;  // staged down-projection row stride
    const bool routed = MODE == DecodeMode::kForward;

    if (tid == 0) {
        mbar_init(s.w2bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }

    // ---------------------------------------------------------------- phase 0
    // Warps 0 .. nrw-1 route (one token each at a time); the others stage the
    // activations meanwhile ([t][H + 16], each 8-byte group split even|odd).
    // When every warp routes, every thread stages afterwards.
    constexpr int per_tok = H / 16;
    const int n_xp = MODE == DecodeMode::kGemm2Partials ? 0 : T * per_tok;
    const int nrw = routed && !a.ids_in ? min(T, kWarpsD) : 0;
    int n_rows;  // routed/listed pair rows before the shared rows
    if (routed) {
        if (a.ids_in) {  // routing supplied by the caller
            for (int i = tid; i < T * k; i += kThreadsD) {
                s.ids[i] = min(max(a.ids_in[i], 0), a.E - 1);
                s.wts[i] = a.wts_in[i];
            }
        } else if (warp < nrw) {
            if (a.E <= 512) route_tokens<16>(a.logits, T, a.E, k, s.ids, s.wts, nrw);
            else route_tokens<kMaxExperts / 32>(a.logits, T, a.E, k, s.ids, s.wts, nrw);
        }
        n_rows = T * k;
    } else {
        n_rows = a.n_pairs;  // listed pairs; out-of-range slots and tokens are clamped (never read out of bounds)
        for (int r = tid; r < n_rows; r += kThreadsD) s.ids[r] = min(max(a.pair_slot[r], 0), a.E - 1);
    }
    if (MODE == DecodeMode::kForward && !MIXED && a.x_bf16) {
        // S0 on the device: the warps that do not route quantise the bf16
        // activations (s = max|x| / 127, q = RNE(x / s) decided in fp32, clamped
        // to +-127; zero row: s = 0, q = 0) into the split staging layout.  wpt
        // warps share a token: each finds the row maximum itself (no sync) and
        // codes the 8-value groups i = part, part + wpt, ... of every lane
        // (group lane + 32 i).  Codes come from x * (1/s) with the exact
        // division only near a half-step, as in the requantisation.
        constexpr int NV = H / 256;  // 8-value groups per lane
        const int w0 = nrw < kWarpsD ? nrw : 0, nws = kWarpsD - w0;
        const int wpt = max(1, min(NV, nws / max(T, 1))), ntw = nws / wpt, rel = warp - w0;
        if (warp >= w0 && rel < ntw * wpt)
            for (int t = rel / wpt; t < T; t += ntw) {
                const int part = rel % wpt;
                const uint4* xr = reinterpret_cast<const uint4*>(a.x_bf16 + static_cast<int64_t>(t) * H);
                float amax = 0.f;
#pragma unroll 4
                for (int i = 0; i < NV; ++i) {
                    const uint4 v = xr[lane + 32 * i];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[j] << 16)), fabsf(__uint_as_float(wv[j] & 0xFFFF0000u))));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                const float sc = __fdiv_rn(amax, 127.0f);
                const float rs = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
                if (lane == 0 && part == 0) s.xs[t] = sc;
                for (int i = part; i < NV; i += wpt) {
                    const uint4 v = xr[lane + 32 * i];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    uint32_t packed[2] = {0u, 0u};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t b = (j & 1) ? (wv[j >> 1] & 0xFFFF0000u) : (wv[j >> 1] << 16);
                        packed[j >> 2] |= (static_cast<uint32_t>(requant_code_fast(__uint_as_float(b), sc, rs)) & 0xFFu)
                                          << (8 * (j & 3));
                    }
                    *reinterpret_cast<uint2*>(s.x + t * XS + 8 * (lane + 32 * i)) =
                        make_uint2(__byte_perm(packed[0], packed[1], 0x6420), __byte_perm(packed[0], packed[1], 0x7531));
                }
            }
    } else if (MODE != DecodeMode::kGemm2Partials) {
        const int st0 = nrw < kWarpsD ? 32 * nrw : 0, nst = kThreadsD - st0;
        if (tid >= st0) {
#pragma unroll 4
            for (int o = tid - st0; o < n_xp; o += nst) {
                const int t = o / per_tok, c = o % per_tok;
                const uint4 v = *reinterpret_cast<const uint4*>(a.x_q + static_cast<int64_t>(t) * H + 16 * c);
                *reinterpret_cast<uint4*>(s.x + t * XS + 16 * c) = split16(v);
                if (MIXED) *reinterpret_cast<uint4*>(s.xm + t * XS + 16 * c) = mod4_16(v);
            }
            for (int t = tid - st0; t < T; t += nst) s.xs[t] = routed ? a.x_scale[t] : 1.0f;
        }
    }
    // routed: per-expert token masks and expert presence bits for the grouping below, in the
    // requantised-row area (first written in phase 2)
    uint32_t* emask = reinterpret_cast<uint32_t*>(s.hq);  // [E] bit t: token t picked the expert
    uint32_t* pres = emask + a.E;                          // [EW] bit e: expert e was picked
    int* pbase = reinterpret_cast<int*>(pres + (a.E + 31) / 32);  // [EW] experts picked in earlier words
    const int EW = (a.E + 31) / 32;
    // (supplied routing may repeat an expert within a token: it takes the scans below)
    const bool bitmaps = routed && !a.ids_in;
    if (bitmaps)
        for (int i = tid; i < a.E + EW; i += kThreadsD) emask[i] = 0u;
    __syncthreads();
    const int S = routed ? a.S : 0;
    if (bitmaps) {
        // Grouping from bitmaps (T <= 32, and top-k picks an expert at most once per token): a pair's
        // slot is the number of picked experts below its expert, its row within the slot the number
        // of earlier tokens that picked the same expert -- the stable order by (expert, pair index).
        for (int i = tid; i < n_rows; i += kThreadsD) {
            const int e = s.ids[i];
            atomicOr(emask + e, 1u << (i / k));
            atomicOr(pres + (e >> 5), 1u << (e & 31));
        }
        __syncthreads();
        if (warp == 0) {  // exclusive prefix of the presence popcounts; the shared slots after the routed ones
            int run = 0;
            for (int b0 = 0; b0 < EW; b0 += 32) {
                const int wi = b0 + lane;
                const int c = wi < EW ? __popc(pres[wi]) : 0;
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                if (wi < EW) pbase[wi] = run + incl - c;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            for (int sh = lane; sh < S; sh += 32) {
                s.slot_e[run + sh] = a.E + sh;
                s.slot_row0[run + sh] = n_rows + sh * T;
                s.slot_cnt[run + sh] = T;
                s.slot_bw[run + sh] = (MIXED && a.slot_bits) ? (a.slot_bits[a.E + sh] == 2 ? 2 : 4) : 4;
            }
            if (lane == 0) s.n_slots[0] = run + S;
        }
        __syncthreads();
        for (int i = tid; i < n_rows; i += kThreadsD) {
            const int e = s.ids[i], t = i / k;
            const uint32_t m = emask[e];
            const int u = pbase[e >> 5] + __popc(pres[e >> 5] & ((1u << (e & 31)) - 1u));
            const int within = __popc(m & ((1u << t) - 1u));
            if (within == 0) {
                s.slot_e[u] = e;
                s.slot_cnt[u] = __popc(m);
                s.slot_bw[u] = (MIXED && a.slot_bits) ? (a.slot_bits[e] == 2 ? 2 : 4) : 4;
            }
            s.first[i] = u;  // (scratch here: the pair's slot and its rank within the slot)
            s.eqc[i] = within;
        }
        __syncthreads();
        if (warp == 0) {  // first pair row of each routed slot: exclusive prefix of the counts
            const int nr = s.n_slots[0] - S;
            int run = 0;
            for (int b0 = 0; b0 < nr; b0 += 32) {
                const int u = b0 + lane;
                const int c = u < nr ? s.slot_cnt[u] : 0;
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                if (u < nr) s.slot_row0[u] = run + incl - c;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        __syncthreads();
        for (int i = tid; i < n_rows; i += kThreadsD) {
            const int p = s.slot_row0[s.first[i]] + s.eqc[i];
            s.pos[i] = p;
            s.pair_of[p] = i;
            s.row_tok[p] = i / k;
        }
    } else {
        // stable rank of each pair by expert id (n_rows <= kDecodeMaxPairs), whether
        // it is its expert's first pair, and how many pairs share its expert
        for (int i = tid; i < n_rows; i += kThreadsD) {
            const int e = s.ids[i];
            int p = 0, eq = 0;
            bool first = true;
#pragma unroll 4
            for (int j = 0; j < n_rows; ++j) {
                const int f = s.ids[j];
                p += (f < e) || (f == e && j < i);
                eq += f == e;
                first = first && !(f == e && j < i);
            }
            s.pos[i] = p;
            s.pair_of[p] = i;
            s.row_tok[p] = routed ? i / k : (MODE == DecodeMode::kGemm1Partials ? min(max(a.pair_token[i], 0), T - 1) : p);
            s.first[i] = first;
            s.eqc[i] = eq;
        }
        __syncthreads();
        // slot table: touched experts ascending (slot = number of smaller touched
        // experts), then the shared experts
        for (int i = tid; i < n_rows; i += kThreadsD) {
            if (!s.first[i]) continue;
            const int e = s.ids[i];
            int u = 0;
#pragma unroll 4
            for (int j = 0; j < n_rows; ++j) u += s.first[j] && s.ids[j] < e;
            s.slot_e[u] = e;
            s.slot_row0[u] = s.pos[i];
            s.slot_cnt[u] = s.eqc[i];
            s.slot_bw[u] = (MIXED && a.slot_bits) ? (a.slot_bits[e] == 2 ? 2 : 4) : 4;
        }
        if (warp == 0) {
            int nr = 0;
            for (int b0 = 0; b0 < n_rows; b0 += 32)
                nr += __popc(__ballot_sync(0xffffffffu, b0 + lane < n_rows && s.first[b0 + lane]));
            for (int sh = lane; sh < S; sh += 32) {
                s.slot_e[nr + sh] = a.E + sh;
                s.slot_row0[nr + sh] = n_rows + sh * T;
                s.slot_cnt[nr + sh] = T;
                s.slot_bw[nr + sh] = (MIXED && a.slot_bits) ? (a.slot_bits[a.E + sh] == 2 ? 2 : 4) : 4;
            }
            if (lane == 0) s.n_slots[0] = nr + S;
        }
    }
    for (int r = tid; r < T * S; r += kThreadsD) s.row_tok[n_rows + r] = r % T;
    if (routed && blockIdx.x == 0 && a.ids_out) {  // debug copies of the routing (every CTA holds the same)
        for (int i = tid; i < n_rows; i += kThreadsD) {
            a.ids_out[i] = s.ids[i];
            a.wts_out[i] = s.wts[i];
            a.inv_out[i] = s.pos[i];
            a.perm_out[s.pos[i]] = i;
        }
    }
    const int P_all = n_rows + T * S;
    if (MODE == DecodeMode::kForward)
        for (int i = tid; i < kWarpsD * P_all; i += kThreadsD) s.wmax[i] = 0.f;
    __syncthreads();
    const int n_slots = s.n_slots[0];
    for (int u = warp; u < n_slots; u += kWarpsD)  // pair row -> its slot
        for (int m = lane; m < s.slot_cnt[u]; m += 32) s.row_slot[s.slot_row0[u] + m] = u;
    if (warp == 0) {  // phase-1 cost prefix over slots (streaming + per-token work), warp scan
        int run = 0;
        for (int b0 = 0; b0 < n_slots; b0 += 32) {
            const int u = b0 + lane;
            const int c = u < n_slots ? (I / 2) * unit_cost(s.slot_cnt[u], s.slot_bw[u]) : 0;
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (u < n_slots) s.slot_cum[u] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s.slot_cum[n_slots] = run;
    }
    __syncthreads();

    // This CTA's down-projection slice (rows [n0, n0 + nrows) of every slot):
    // the first n_smem slots are copied into shared memory by the bulk-copy
    // engine (one copy per row, so the rows keep their padded stride, and one
    // for the scales; completion on one mbarrier), the rest warmed in L2.
    // Warp w stages slots w, w + 8, ..., a few per phase-1 unit (lane r issues
    // row r's copy).
    const int n0 = blockIdx.x * pl.rows_pc;
    const int nrows = max(0, min(pl.rows_pc, H - n0));
    const int n_smem = MODE == DecodeMode::kForward && nrows > 0 ? min(n_slots, pl.smem_slots) : 0;
    const int slot_stride = pl.rows_pc * RS + pl.rows_pc * ng2 * 4;
    const int lines_s = (nrows * ng2 * 4 + 127) / 128;
    if (tid == 0 && n_smem > 0) {  // every staged byte counted before any copy can land
        uint32_t bytes = 0;  // a 2-bit slot's rows are copied at half length
        for (int u = 0; u < n_smem; ++u) bytes += nrows * ((MIXED && s.slot_bw[u] == 2 ? I / 4 : I / 2) + ng2 * 4);
        mbar_expect_tx(s.w2bar, bytes);
    }
    __syncthreads();
    int next_slot = warp;  // next slot this warp stages (copies or warms)
    auto stage_some = [&](int budget) {
        for (int b = 0; b < budget && next_slot < n_slots; ++b, next_slot += kWarpsD) {
            const int u = next_slot;
            const int64_t e = s.slot_e[u];
            const bool two = MIXED && s.slot_bw[u] == 2;
            const int64_t* off = MIXED ? a.w2_off : nullptr;
            const uint8_t* wsrc = a.w2 + bank_row(off, e, H, n0, I / 2, two);
            const uint8_t* ssrc = reinterpret_cast<const uint8_t*>(a.s2 + (e * H + n0) * ng2);
            const int rb = two ? I / 4 : I / 2;       // bytes of a row that hold codes
            const int rstr = off && two ? I / 4 : I / 2;  // bytes from one row to the next
            if (u < n_smem) {
                uint8_t* base = s.w2s + u * slot_stride;
                for (int r = lane; r <= nrows; r += 32) {  // lane r: row r; lane nrows: the scales
                    if (r < nrows) bulk_g2s(base + r * RS, wsrc + r * rstr, rb, s.w2bar);
                    else bulk_g2s(base + pl.rows_pc * RS, ssrc, nrows * ng2 * 4, s.w2bar);
                }
            } else {
                const int lpr = rb / 128, lines_w = nrows * lpr;  // 128-byte lines of the code bytes of each row
                for (int c = lane; c < lines_w + lines_s; c += 32)
                    prefetch_l2(c < lines_w ? wsrc + (c / lpr) * rstr + 128 * (c % lpr) : ssrc + 128 * (c - lines_w));
            }
        }
    };

    // ---------------------------------------------------------------- phase 1
    if (MODE != DecodeMode::kGemm2Partials) {
        constexpr int DEPTH = 1;  // units loaded per warp at a time (the SM's other warps hide the latency)
        const int upe = I / 2;                    // units per slot
        // each warp takes a contiguous unit range of equal cost: a CTA's warps
        // stream neighbouring rows, and few slots (pages) per SM
        const int64_t Ctot = s.slot_cum[n_slots];
        const int64_t W = static_cast<int64_t>(gridDim.x) * kWarpsD;
        const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsD + warp;
        auto unit_at = [&](int64_t cpos) -> int64_t {
            int lo = 0, hi = n_slots;  // last slot with cum <= cpos
            while (hi - lo > 1) {
                const int mid = (lo + hi) / 2;
                if (s.slot_cum[mid] <= cpos) lo = mid;
                else hi = mid;
            }
            const int c = unit_cost(s.slot_cnt[lo], s.slot_bw[lo]);
            int64_t within = (cpos - s.slot_cum[lo] + c - 1) / c;
            if (within > upe) within = upe;
            return static_cast<int64_t>(lo) * upe + within;
        };
        const int64_t Ua = unit_at(gw * Ctot / W), Ub = unit_at((gw + 1) * Ctot / W);
        const int nun = static_cast<int>(Ub - Ua);
        const int stage_budget = MODE == DecodeMode::kForward ? (n_slots + kWarpsD - 1) / kWarpsD / max(nun, 1) + 1 : 0;

        // lane l owns the 16-byte pieces l + 32 p of each row (32 codes each, p <
        // NP): every load instruction of a warp reads 512 contiguous bytes
        constexpr int NP = 2 * PC1;
        uint4 wr[DEPTH][4][NP];
        float sr[DEPTH][4][NP];
        // K group of piece p of this lane, (32 lane + 1024 p) / g, by a multiply and
        // a shift: with m = ceil(2^24 / g), floor(n m / 2^24) = floor(n / g) for n g < 2^24
        const uint32_t gmag = ((1u << 24) + static_cast<uint32_t>(g) - 1) / static_cast<uint32_t>(g);
        auto gq = [&](int p) { return static_cast<int>((static_cast<uint32_t>(32 * lane + 1024 * p) * gmag) >> 24); };
        // a 2-bit row: lane l owns the 16-byte pieces l + 32 p (64 codes each, p < PC1)
        auto gq2 = [&](int p) { return static_cast<int>((static_cast<uint32_t>(64 * lane + 2048 * p) * gmag) >> 24); };
        auto issue = [&](int un, int d) {
            const int64_t U = Ua + un;
            const int u = static_cast<int>(U / upe), ip = static_cast<int>(U % upe);
            const int64_t e = s.slot_e[u];
            const bool two = MIXED && s.slot_bw[u] == 2;  // half the bytes per row
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int64_t rr = (r >= 2 ? I : 0) + 2 * ip + (r & 1), row = e * 2 * I + rr;
                const uint8_t* wp = a.w13 + bank_row(MIXED ? a.w13_off : nullptr, e, 2 * I, rr, H / 2, two);
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    if (two && p >= PC1) break;
                    wr[d][r][p] = ld_stream16(wp + 16 * lane + 512 * p);
                    if (MODE == DecodeMode::kForward) sr[d][r][p] = __ldg(a.s13 + row * ng1 + (two ? gq2(p) : gq(p)));
                }
            }
        };
#pragma unroll
        for (int d = 0; d < DEPTH; ++d)
            if (d < nun) issue(d, d);
        const int lpg = g / 32;  // lanes per K group (per piece index)
        for (int base = 0; base < nun; base += DEPTH) {
#pragma unroll
            for (int d = 0; d < DEPTH; ++d) {
                const int un = base + d;
                if (un >= nun) break;
                const uint4(&w)[4][NP] = wr[d];
                const float(&sc)[4][NP] = sr[d];
                const int64_t U = Ua + un;
                const int u = static_cast<int>(U / upe), ip = static_cast<int>(U % upe);
                const int row0 = s.slot_row0[u], cnt = s.slot_cnt[u];
                const bool two = MIXED && s.slot_bw[u] == 2;
                for (int m = 0; m < cnt; ++m) {
                    const int prow = row0 + m;
                    const int t = s.row_tok[prow];
                    float v[4];
                    if (two) {  // 2-bit slot: 64 codes per piece, sums are 64 x the int32 partials
#pragma unroll
                        for (int r = 0; r < 4; ++r) v[r] = 0.f;
#pragma unroll
                        for (int p = 0; p < PC1; ++p) {
                            // activations in mod-4 order: lane word q of a 2-bit word is one shift and one mask
                            const uint4* xp = reinterpret_cast<const uint4*>(s.xm + t * XS + 64 * lane + 2048 * p);
                            int acc[4] = {0, 0, 0, 0};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {  // word i: 16 codes against 16 activation bytes
                                const uint4 xv = xp[i];
#pragma unroll
                                for (int r = 0; r < 4; ++r) {
                                    const uint32_t wd = i == 0 ? w[r][p].x : i == 1 ? w[r][p].y : i == 2 ? w[r][p].z : w[r][p].w;
                                    acc[r] = __dp4a(static_cast<int>(xv.x), static_cast<int>((wd << 6) & 0xC0C0C0C0u), acc[r]);
                                    acc[r] = __dp4a(static_cast<int>(xv.y), static_cast<int>((wd << 4) & 0xC0C0C0C0u), acc[r]);
                                    acc[r] = __dp4a(static_cast<int>(xv.z), static_cast<int>((wd << 2) & 0xC0C0C0C0u), acc[r]);
                                    acc[r] = __dp4a(static_cast<int>(xv.w), static_cast<int>(wd & 0xC0C0C0C0u), acc[r]);
                                }
                            }
#pragma unroll
                            for (int r = 0; r < 4; ++r) v[r] = fmaf(static_cast<float>(acc[r] >> 6), sc[r][p], v[r]);
                        }
                    } else {
                    int P[4][NP];
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        const uint8_t* xp = s.x + t * XS + 32 * lane + 1024 * p;
                        const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
                        const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
#pragma unroll
                        for (int r = 0; r < 4; ++r) P[r][p] = dot32(w[r][p], x0, x1);
                    }
                    if (MODE == DecodeMode::kGemm1Partials) {
#pragma unroll
                        for (int r = 0; r < 4; ++r)
#pragma unroll
                            for (int p = 0; p < NP; ++p) {
                                int v = P[r][p];
                                for (int off = 1; off < lpg; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                                if ((lane % lpg) == 0) {
                                    const int64_t wrow = (r >= 2 ? I : 0) + 2 * ip + (r & 1);
                                    a.p1[(static_cast<int64_t>(prow) * 2 * I + wrow) * ng1 + gq(p)] = v >> 4;
                                }
                            }
                        continue;
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        v[r] = 0.f;
#pragma unroll
                        for (int p = 0; p < NP; ++p) v[r] = fmaf(static_cast<float>(P[r][p] >> 4), sc[r][p], v[r]);
                    }
                    }  // 4-bit slot
                    // reduce-scatter of the 4 row sums: lane keeps row 2*bit4 + bit3
                    const bool b4 = lane & 16, b3 = lane & 8;
                    float k0 = b4 ? v[2] : v[0], k1 = b4 ? v[3] : v[1];
                    const float s0 = b4 ? v[0] : v[2], s1 = b4 ? v[1] : v[3];
                    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
                    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
                    float kk = b3 ? k1 : k0;
                    kk += __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
                    kk += __shfl_xor_sync(0xffffffffu, kk, 4);
                    kk += __shfl_xor_sync(0xffffffffu, kk, 2);
                    kk += __shfl_xor_sync(0xffffffffu, kk, 1);
                    const float upv = __shfl_xor_sync(0xffffffffu, kk, 16);  // up row of the same index
                    float hm = 0.f;
                    if (!b4 && (lane & 7) == 0) {
                        const float xs = s.xs[t];
                        const float hv = silu_f32(kk * xs) * (upv * xs);
                        a.h[static_cast<int64_t>(prow) * I + 2 * ip + (b3 ? 1 : 0)] = hv;
                        hm = fabsf(hv);
                    }
                    if (MODE == DecodeMode::kForward) {
                        // this warp's running maximum of the row (lane 0 owns the warp's entry)
                        hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 8));
                        if (lane == 0) s.wmax[warp * P_all + prow] = fmaxf(s.wmax[warp * P_all + prow], hm);
                    }
                }
                if (un + DEPTH < nun) issue(un + DEPTH, d);  // refill this ring slot
                if (MODE == DecodeMode::kForward) stage_some(stage_budget);
            }
        }
    }
    if (MODE == DecodeMode::kGemm1Partials) return;
    if (MODE == DecodeMode::kForward) {
        stage_some(1 << 30);  // whatever phase 1 did not cover
        __syncthreads();
        for (int p = tid; p < P_all; p += kThreadsD) {
            float m = 0.f;
            for (int w = 0; w < kWarpsD; ++w) m = fmaxf(m, s.wmax[w * P_all + p]);
            if (m > 0.f) atomicMax(a.row_max + p, __float_as_uint(m));
        }
    }

    // ---------------------------------------------------------------- barrier
    if (MODE == DecodeMode::kForward && !grid_barrier(a.hdr, 1)) {
        if (n_smem > 0) w2_wait(s.w2bar, a.hdr);  // the CTA's bulk copies land before it leaves
        __syncthreads();
        return;
    }

    // ---------------------------------------------------------------- phase 2
    const int P = n_rows + T * S;
    const int per_row = I / 16;
    if (MODE == DecodeMode::kForward) {
        // (a) requantisation, spread over the grid: row p goes to CTA p % grid,
        // one warp per row -- s_h from the row maximum, RNE codes -- stored
        // split even|odd to the workspace; a second grid barrier publishes them
        for (int p = static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * warp; p < P;
             p += static_cast<int>(gridDim.x) * kWarpsD) {
            // the row's h values and its maximum in one round trip (PC2 = 1: 16 values
            // per lane; larger I: the rest per chunk below)
            const float4* src0 = reinterpret_cast<const float4*>(a.h + static_cast<int64_t>(p) * I + 16 * lane);
            float4 f[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) f[q] = __ldcg(src0 + q);
            const uint32_t mb = __ldcg(a.row_max + p);
            const float sc = requant_scale(mb);
            const float rs = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
            if (lane == 0) {
                a.sh_g[p] = sc;
                if (a.amax) a.amax[p] = mb;
            }
#pragma unroll
            for (int c2 = 0; c2 < PC2; ++c2) {  // 16 values per lane per 512-value chunk
                if (c2 > 0) {
                    const float4* src = reinterpret_cast<const float4*>(a.h + static_cast<int64_t>(p) * I + 512 * c2 + 16 * lane);
#pragma unroll
                    for (int q = 0; q < 4; ++q) f[q] = __ldcg(src + q);
                }
                uint2* dst = reinterpret_cast<uint2*>(a.hq_g + static_cast<int64_t>(p) * I + 512 * c2 + 16 * lane);
#pragma unroll
                for (int q = 0; q < 2; ++q) {  // 8 values -> one 8-byte group, split even|odd
                    const float4 f0 = f[2 * q], f1 = f[2 * q + 1];
                    const uint32_t w0 = (requant_code_fast(f0.x, sc, rs) & 0xFF) | ((requant_code_fast(f0.y, sc, rs) & 0xFF) << 8) |
                                        ((requant_code_fast(f0.z, sc, rs) & 0xFF) << 16) |
                                        ((static_cast<uint32_t>(requant_code_fast(f0.w, sc, rs)) & 0xFF) << 24);
                    const uint32_t w1 = (requant_code_fast(f1.x, sc, rs) & 0xFF) | ((requant_code_fast(f1.y, sc, rs) & 0xFF) << 8) |
                                        ((requant_code_fast(f1.z, sc, rs) & 0xFF) << 16) |
                                        ((static_cast<uint32_t>(requant_code_fast(f1.w, sc, rs)) & 0xFF) << 24);
                    dst[q] = make_uint2(__byte_perm(w0, w1, 0x6420), __byte_perm(w0, w1, 0x7531));
                }
            }
        }
        if (!grid_barrier(a.hdr, 2)) {
            if (n_smem > 0) w2_wait(s.w2bar, a.hdr);
            __syncthreads();
            return;
        }
        // (b) every CTA copies all P requantised rows (already split) and their scales
        for (int o = tid; o < P * per_row; o += kThreadsD) {
            const int p = o / per_row, c = o % per_row;
            cp_async16(s.hq + p * HQS + 16 * c, a.hq_g + static_cast<int64_t>(p) * I + 16 * c);
        }
        for (int p = tid; p < P; p += kThreadsD) s.sh[p] = __ldcg(a.sh_g + p);
        cp_async_commit();
    } else {
        for (int o = tid; o < P * per_row; o += kThreadsD) {
            const int p = o / per_row, c = o % per_row;
            const uint4 v = *reinterpret_cast<const uint4*>(a.h_q_in + static_cast<int64_t>(p) * I + 16 * c);
            *reinterpret_cast<uint4*>(s.hq + p * HQS + 16 * c) = split16(v);
        }
    }
    cp_async_wait<0>();
    if (MODE == DecodeMode::kForward && n_smem > 0 && !w2_wait(s.w2bar, a.hdr)) {
        __syncthreads();
        return;
    }
    __syncthreads();
    if (nrows == 0) return;

    // (b) down projection: one thread per (pair row, output row), running the
    // whole K = I dot product of the row's slot (no cross-lane sums); the
    // threads of one pair row share its activation row (broadcast reads)
    {
        const int n_items = P * nrows;
        for (int L = tid; L < n_items; L += kThreadsD) {
            const int p = L / nrows, r = L % nrows;
            const int u = s.row_slot[p];
            const int64_t e = s.slot_e[u];
            const bool in_smem = u < n_smem;
            const uint8_t* wrow = in_smem ? s.w2s + u * slot_stride + r * RS
                                          : a.w2 + bank_row(MIXED ? a.w2_off : nullptr, e, H, n0 + r, I / 2,
                                                            MIXED && s.slot_bw[u] == 2);
            const float* srow = in_smem ? reinterpret_cast<const float*>(s.w2s + u * slot_stride + pl.rows_pc * RS) + r * ng2
                                        : a.s2 + (e * H + n0 + r) * ng2;
            const uint8_t* xrow = s.hq + p * HQS;
            const bool two = MIXED && s.slot_bw[u] == 2;
            float acc = 0.f;
            for (int q = 0; q < ng2; ++q) {
                int Pq = 0;
                if (two) {
                    for (int c = 0; c < g / 64; ++c) {  // 64 codes (16 packed bytes) per step
                        const int kb = q * (g / 4) + 16 * c;
                        const uint4 wv = in_smem ? *reinterpret_cast<const uint4*>(wrow + kb) : ld_stream16(wrow + kb);
                        const uint4* xp = reinterpret_cast<const uint4*>(xrow + 4 * kb);
                        Pq += dot64_2bit(wv, xp[0], xp[1], xp[2], xp[3]) >> 2;  // 16 x the partial, as below
                    }
                } else {
                    for (int c = 0; c < g / 32; ++c) {  // 32 codes (16 packed bytes) per step
                        const int kb = q * (g / 2) + 16 * c;
                        const uint4 wv = in_smem ? *reinterpret_cast<const uint4*>(wrow + kb) : ld_stream16(wrow + kb);
                        const uint4 xa = *reinterpret_cast<const uint4*>(xrow + 2 * kb);
                        const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 2 * kb + 16);
                        Pq += dot32(wv, xa, xb);
                    }
                }
                if (MODE == DecodeMode::kGemm2Partials) {
                    a.p2[(static_cast<int64_t>(p) * H + n0 + r) * ng2 + q] = Pq >> 4;
                } else {
                    const float sc = in_smem ? srow[q] : __ldg(srow + q);
                    acc = fmaf(static_cast<float>(Pq >> 4), sc, acc);
                }
            }
            if (MODE == DecodeMode::kForward) {
                const float yv = acc * s.sh[p];
                s.y[p * pl.rows_pc + r] = yv;
                if (a.y) a.y[static_cast<int64_t>(p) * H + n0 + r] = yv;
            }
        }
    }
    if (MODE == DecodeMode::kGemm2Partials) return;
    __syncthreads();

    // (c) combine, fixed order: routed pairs j = 0..k-1, then the shared experts
    for (int o = tid; o < T * nrows; o += kThreadsD) {
        const int t = o / nrows, r = o % nrows;
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = fmaf(s.wts[t * k + j], s.y[s.pos[t * k + j] * pl.rows_pc + r], acc);
        for (int sh = 0; sh < S; ++sh) acc += s.y[(n_rows + sh * T + t) * pl.rows_pc + r];
        a.out[static_cast<int64_t>(t) * H + n0 + r] = acc;
    }
}

// Two CTAs: CTA 0 waits at the grid barrier, CTA 1 never arrives, so the
// bounded wait runs out and records the timeout in the status word.
__global__ void barrier_timeout_probe_kernel(Header* hdr) {
    if (blockIdx.x != 0) return;
    grid_barrier(hdr, 1);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <DecodeMode MODE, int PC1, int PC2, bool MIXED = false>
cudaError_t launch_mode(const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    auto kern = decode_kernel<MODE, PC1, PC2, MIXED>;
    // The dynamic shared memory limit is one value per kernel: set it once per
    // device to the largest size any plan may ask for.
    static std::mutex mu;
    static std::map<int, bool> attr_set;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set.count(dev)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, decode_max_smem());
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    if (pl.smem_bytes > decode_max_smem()) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsD);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = MODE == DecodeMode::kForward ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a, pl);
}

template <int PC1, int PC2>
cudaError_t launch_shape(DecodeMode mode, const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    if (mode == DecodeMode::kForward)
        return a.slot_bits ? launch_mode<DecodeMode::kForward, PC1, PC2, true>(a, pl, grid, st)
                           : launch_mode<DecodeMode::kForward, PC1, PC2, false>(a, pl, grid, st);
    if (mode == DecodeMode::kGemm1Partials) return launch_mode<DecodeMode::kGemm1Partials, PC1, PC2>(a, pl, grid, st);
    return launch_mode<DecodeMode::kGemm2Partials, PC1, PC2>(a, pl, grid, st);
}

}  // namespace

// (H / 2048, I / 512) shapes the engine is compiled for.
bool decode_shape_supported(int64_t H, int64_t I) {
    if (H % 2048 != 0 || I % 512 != 0) return false;
    const int64_t p1 = H / 2048, p2 = I / 512;
    return (p1 == 1 || p1 == 2) && (p2 >= 1 && p2 <= 4);
}

// Shared-memory plan of one launch (host side; the kernel reads the offsets).
bool decode_plan(int64_t T, int64_t H, int64_t I, int64_t E, int64_t S, int64_t k, int64_t g, int64_t n_pairs,
                 DecodeMode mode, int grid, int max_smem, DecodePlan* out, bool mixed) {
    if (!decode_shape_supported(H, I) || g % 64 != 0 || g > 512 || (I / g) % 4 != 0 || E > kMaxExperts) return false;
    const int64_t rows = mode == DecodeMode::kForward ? T * k : n_pairs;
    const int64_t Sx = mode == DecodeMode::kForward ? S : 0;
    const int64_t P = rows + T * Sx;
    if (T > kDecodeMaxT || rows > kDecodeMaxPairs || P > kDecodeMaxPairs + kDecodeMaxT * kMaxShared) return false;
    if (mode != DecodeMode::kForward && rows < 1) return false;
    const int64_t MS = rows + Sx;
    DecodePlan pl{};
    pl.rows_pc = static_cast<int>((H + grid - 1) / grid);
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) {
        o = align_up(o, al);
        size_t at = o;
        o += bytes;
        return static_cast<int>(at);
    };
    pl.off_ids = take(4 * rows, 16);
    pl.off_wts = take(4 * rows, 16);
    pl.off_pos = take(4 * rows, 16);
    pl.off_pair_of = take(4 * rows, 16);
    pl.off_row_tok = take(4 * P, 16);
    pl.off_slot_e = take(4 * MS, 16);
    pl.off_slot_row0 = take(4 * MS, 16);
    pl.off_slot_cnt = take(4 * MS, 16);
    pl.off_slot_bw = take(4 * MS, 16);
    pl.off_slot_cum = take(4 * (MS + 1), 16);
    pl.off_n_slots = take(16, 16);
    pl.off_xs = take(4 * T, 16);
    pl.off_sh = take(4 * P, 16);
    pl.off_x = take(mode == DecodeMode::kGemm2Partials ? 0 : T * (H + 16), 128);
    pl.off_xm = take(mode == DecodeMode::kForward && mixed ? T * (H + 16) : 0, 128);
    // (the forward kernel's grouping uses this area as scratch before phase 2 writes it: E + 2 (E + 31) / 32 words)
    pl.off_hq = take(mode == DecodeMode::kGemm1Partials ? 0
                     : std::max<int64_t>(P * (I + 16), mode == DecodeMode::kForward ? 4 * (E + 2 * ((E + 31) / 32)) : 0),
                     128);
    pl.off_y = take(mode == DecodeMode::kForward ? 4 * P * pl.rows_pc : 0, 16);
    pl.off_first = take(4 * rows, 16);
    pl.off_eqc = take(4 * rows, 16);
    pl.off_wmax = take(mode == DecodeMode::kForward ? 4 * kWarpsD * P : 0, 16);
    pl.off_w2bar = take(8, 16);
    pl.off_row_slot = take(4 * P, 16);
    pl.off_w2s = static_cast<int>(align_up(o, 128));
    const size_t slot_bytes =
        static_cast<size_t>(pl.rows_pc) * (I / 2 + 16) + static_cast<size_t>(pl.rows_pc) * (I / g) * 4;
    const size_t fixed = pl.off_w2s;
    if (fixed > static_cast<size_t>(max_smem)) return false;
    const int64_t fit = mode == DecodeMode::kForward ? static_cast<int64_t>((max_smem - fixed) / slot_bytes) : 0;
    pl.smem_slots = static_cast<int>(std::min<int64_t>(fit, MS));
    pl.smem_bytes = static_cast<int>(fixed + pl.smem_slots * slot_bytes);
    *out = pl;
    return true;
}

int decode_grid() { return num_sms(); }

int decode_max_smem() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cached[dev] = v > 1024 ? v - 1024 : 0;  // leave room for static shared memory
    }
    return cached[dev];
}

cudaError_t launch_decode(DecodeMode mode, const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    if (mode == DecodeMode::kForward) {
        // status, barrier counters and the per-slot counters that follow the header
        cudaError_t e = cudaMemsetAsync(a.hdr, 0, sizeof(Header) + sizeof(uint32_t) * kFlagWords, st);
        if (e != cudaSuccess) return e;
    }
    const int p1 = a.H / 2048, p2 = a.I / 512;
    if (a.H != 2048 * p1 || a.I != 512 * p2) return cudaErrorInvalidValue;  // the kernel's shape is compiled in
    if (p1 == 1 && p2 == 1) return launch_shape<1, 1>(mode, a, pl, grid, st);
    if (p1 == 2 && p2 == 1) return launch_shape<2, 1>(mode, a, pl, grid, st);
    if (p1 == 1 && p2 == 2) return launch_shape<1, 2>(mode, a, pl, grid, st);
    if (p1 == 2 && p2 == 2) return launch_shape<2, 2>(mode, a, pl, grid, st);
    if (p1 == 1 && p2 == 3) return launch_shape<1, 3>(mode, a, pl, grid, st);
    if (p1 == 2 && p2 == 3) return launch_shape<2, 3>(mode, a, pl, grid, st);
    if (p1 == 1 && p2 == 4) return launch_shape<1, 4>(mode, a, pl, grid, st);
    if (p1 == 2 && p2 == 4) return launch_shape<2, 4>(mode, a, pl, grid, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_barrier_timeout_probe(Header* hdr, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(hdr, 0, 16, st);
    if (e != cudaSuccess) return e;
    barrier_timeout_probe_kernel<<<2, 32, 0, st>>>(hdr);
    return cudaGetLastError();
}

}  // namespace moe
