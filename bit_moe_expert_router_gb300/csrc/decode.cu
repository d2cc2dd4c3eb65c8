// Fused decode engine of the W4A8 MoE layer: one cooperative persistent launch.
//
// For small batches the layer is bound by the bytes of the touched experts'
// packed weights ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next", section 3:
// keep the W4 bank packed and do the work on the device; section 5: no host
// round trips inside the token loop, fused operators for decode steps made of
// many small launches).  One launch does everything, streaming each touched
// expert's bytes from HBM exactly once:
//
//   phase 0  every CTA routes all T tokens itself (same deterministic result
//            in every CTA, so no exchange is needed), sorts the pairs stably
//            by expert into pair rows, builds the slot table (touched experts
//            in ascending order, then the shared experts), stages the
//            activations in shared memory, and starts TMA bulk copies of its
//            own slice of the down-projection bank (its output rows, every
//            touched slot) into shared memory (L2 prefetch for what does not
//            fit).
//   phase 1  gate/up projection: the (slot, intermediate index) units are split
//            evenly over all warps of the grid; a warp streams the unit's gate
//            row and up row (16-byte loads, round-robin over lanes), unpacks the
//            nibbles in registers and accumulates with dp4a; each K group's
//            exact int32 partial is folded into fp32 with its scale, then
//            h = SiLU(G_gate) * G_up goes to the workspace.
//   barrier  one grid-wide barrier (bounded wait; on timeout the status word
//            records it and the CTAs leave after their copies have landed).
//   phase 2  every CTA requantises all pair rows (row max -> s_h, RNE codes)
//            into shared memory, runs the down projection for its output rows
//            of every touched slot from the staged slice (half-warp per weight
//            row), and combines out[t][n] = sum_j w[t][j] Y[(t,j)][n] + shared
//            in a fixed order -- no atomics, deterministic.
//
// The same kernel also serves the partials entry points (phase 1 or phase 2
// alone, pairs given as a list instead of routed) so the bit-exact int32
// checks run through this engine's integer core.
//
// Nibble unpack as in the grouped engine: a nibble moved into the high half
// of its byte is an int8 lane holding 16 * code; dp4a gives 16 * P exactly.
// Activations are stored in shared memory with each 8-byte group split into
// its even and odd elements, matching the unpack's even/odd output words.
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "decode.h"

namespace moe {
namespace {

constexpr int kThreadsD = 512;
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

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// Bounded wait for the TMA transactions of phase `parity`; false on timeout.
__device__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < kSpinCap; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) break;
        __nanosleep(128);
    }
    return false;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number `k` (1-based) of this launch; the counters start
// at zero (cleared before the launch).  Bounded: false on timeout.
__device__ bool grid_barrier(Header* hdr, uint32_t k) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        const uint32_t old = atomicAdd(&hdr->bar_arrive, 1u);
        if (old == k * gridDim.x - 1) {
            __threadfence();
            atomicExch(&hdr->bar_gen, k);
        } else {
            const uint64_t t0 = global_ns();
            uint32_t it = 0;
            while (ld_acquire(&hdr->bar_gen) < k) {
                if (++it > kSpinCap || global_ns() - t0 > kWaitNs) {
                    atomicOr(&hdr->status, kDevTimeout);
                    ok = 0;
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// (v, e) beats (bv, be): larger value, or equal value and lower index.
__device__ __forceinline__ bool beats(float v, int e, float bv, int be) { return v > bv || (v == bv && e < be); }

// One warp routes token t: ids/w of its k selected experts into shared memory.
__device__ void route_token_warp(const float* __restrict__ l, int E, int k, int* ids, float* wts) {
    const int lane = threadIdx.x & 31;
    float v[kMaxExperts / 32];
    uint32_t taken = 0;
    const int nj = (E + 31) / 32;
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        v[j] = (j < nj && e < E) ? __ldg(l + e) : -INFINITY;
        if (!(j < nj && e < E)) taken |= 1u << j;
    }
    float my_v = 0.f;
    int my_e = 0;
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int be = INT32_MAX;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {
            const int e = lane + 32 * j;
            if (!(taken >> j & 1u) && beats(v[j], e, bv, be)) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (beats(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == s) {
            my_v = bv;
            my_e = be;
        }
    }
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - m) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        ids[lane] = my_e;
        wts[lane] = ex / sum;
    }
}

// Eight int8 values -> (even elements word, odd elements word).
__device__ __forceinline__ uint2 split_even_odd(uint32_t w0, uint32_t w1) {
    uint2 r;
    r.x = __byte_perm(w0, w1, 0x6420);
    r.y = __byte_perm(w0, w1, 0x7531);
    return r;
}

// 16 int8 (uint4) -> same 16 bytes with each 8-byte group split even|odd.
__device__ __forceinline__ uint4 split16(uint4 v) {
    const uint2 a = split_even_odd(v.x, v.y), b = split_even_odd(v.z, v.w);
    return make_uint4(a.x, a.y, b.x, b.y);
}

// dp4a over one packed 16-byte weight chunk (32 codes) against 32 activation
// bytes stored split (xa: codes 0..15, xb: codes 16..31).
__device__ __forceinline__ int dot_chunk(const uint4 w, const uint4 xa, const uint4 xb, int acc) {
    uint32_t e, o;
    unpack_int4x8_x16(w.x, e, o);
    acc = __dp4a(static_cast<int>(xa.x), static_cast<int>(e), acc);
    acc = __dp4a(static_cast<int>(xa.y), static_cast<int>(o), acc);
    unpack_int4x8_x16(w.y, e, o);
    acc = __dp4a(static_cast<int>(xa.z), static_cast<int>(e), acc);
    acc = __dp4a(static_cast<int>(xa.w), static_cast<int>(o), acc);
    unpack_int4x8_x16(w.z, e, o);
    acc = __dp4a(static_cast<int>(xb.x), static_cast<int>(e), acc);
    acc = __dp4a(static_cast<int>(xb.y), static_cast<int>(o), acc);
    unpack_int4x8_x16(w.w, e, o);
    acc = __dp4a(static_cast<int>(xb.z), static_cast<int>(e), acc);
    acc = __dp4a(static_cast<int>(xb.w), static_cast<int>(o), acc);
    return acc;
}

struct Smem {
    uint64_t* bar;
    int* flags;       // [0] abort
    int* ids;         // [T*k]
    float* wts;       // [T*k]
    int* pos;         // [T*k] pair -> row
    int* pair_of;     // [T*k] row -> pair
    int* row_tok;     // [P]
    int* slot_e;      // [MS]
    int* slot_row0;   // [MS]
    int* slot_cnt;    // [MS]
    int* n_slots;     // [1]
    float* xs;        // [T]
    float* sh;        // [P]
    uint8_t* x;       // [T*H] phase-1 layout
    uint8_t* hq;      // [P*I] phase-2 layout
    float* y;         // [P*rows_pc]
    uint8_t* w2s;     // [smem_slots][slot_bytes]
};

__device__ Smem carve(uint8_t* base, const DecodePlan& pl) {
    Smem s;
    s.bar = reinterpret_cast<uint64_t*>(base + pl.off_bar);
    s.flags = reinterpret_cast<int*>(base + pl.off_flags);
    s.ids = reinterpret_cast<int*>(base + pl.off_ids);
    s.wts = reinterpret_cast<float*>(base + pl.off_wts);
    s.pos = reinterpret_cast<int*>(base + pl.off_pos);
    s.pair_of = reinterpret_cast<int*>(base + pl.off_pair_of);
    s.row_tok = reinterpret_cast<int*>(base + pl.off_row_tok);
    s.slot_e = reinterpret_cast<int*>(base + pl.off_slot_e);
    s.slot_row0 = reinterpret_cast<int*>(base + pl.off_slot_row0);
    s.slot_cnt = reinterpret_cast<int*>(base + pl.off_slot_cnt);
    s.n_slots = reinterpret_cast<int*>(base + pl.off_n_slots);
    s.xs = reinterpret_cast<float*>(base + pl.off_xs);
    s.sh = reinterpret_cast<float*>(base + pl.off_sh);
    s.x = base + pl.off_x;
    s.hq = base + pl.off_hq;
    s.y = reinterpret_cast<float*>(base + pl.off_y);
    s.w2s = base + pl.off_w2s;
    return s;
}

template <DecodeMode MODE, int C1, int C2>
__global__ void __launch_bounds__(kThreadsD, 1) decode_kernel(DecodeArgs a, DecodePlan pl) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const Smem s = carve(smem_raw, pl);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, H = a.H, I = a.I, k = a.k, g = a.g;
    const int lpg1 = g / 32;                 // lanes per K group (one 16-byte chunk = 32 codes per lane)
    // C1 = H / 1024: phase-1 chunks per lane per row; C2 = I / 512: phase-2 chunks per lane per row
    const int ng1 = H / g, ng2 = I / g;
    const bool routed = MODE == DecodeMode::kForward;

    // ---------------------------------------------------------------- phase 0
    if (tid == 0) {
        s.flags[0] = 0;
        if (MODE == DecodeMode::kForward) mbar_init(s.bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    int n_rows;  // routed/listed pair rows before the shared rows
    if (routed) {
        for (int t = warp; t < T; t += kWarpsD)
            route_token_warp(a.logits + static_cast<int64_t>(t) * a.E, a.E, k, s.ids + t * k, s.wts + t * k);
        n_rows = T * k;
    } else {
        n_rows = a.n_pairs;  // listed pairs; out-of-range slots and tokens are clamped (never read out of bounds)
        for (int r = tid; r < n_rows; r += kThreadsD) s.ids[r] = min(max(a.pair_slot[r], 0), a.E - 1);
    }
    __syncthreads();
    // stable rank of each pair by expert id (n_rows <= kDecodeMaxPairs)
    for (int i = tid; i < n_rows; i += kThreadsD) {
        const int e = s.ids[i];
        int p = 0;
        for (int j = 0; j < n_rows; ++j) {
            const int f = s.ids[j];
            p += (f < e) || (f == e && j < i);
        }
        s.pos[i] = p;
        s.pair_of[p] = i;
        s.row_tok[p] = routed ? i / k : (MODE == DecodeMode::kGemm1Partials ? min(max(a.pair_token[i], 0), T - 1) : 0);
    }
    const int S = routed ? a.S : 0;
    for (int r = tid; r < T * S; r += kThreadsD) s.row_tok[n_rows + r] = r % T;
    __syncthreads();
    for (int r = tid; r < n_rows; r += kThreadsD) {
        const int e = s.ids[s.pair_of[r]];
        if (r == 0 || s.ids[s.pair_of[r - 1]] != e) {
            int u = 0;
            for (int q = 1; q <= r; ++q) u += s.ids[s.pair_of[q]] != s.ids[s.pair_of[q - 1]];
            s.slot_e[u] = e;
            s.slot_row0[u] = r;
        }
    }
    if (tid == 0) {
        int nr = 0;
        for (int q = 0; q < n_rows; ++q) nr += (q == 0 || s.ids[s.pair_of[q]] != s.ids[s.pair_of[q - 1]]);
        for (int sh = 0; sh < S; ++sh) {
            s.slot_e[nr + sh] = a.E + sh;
            s.slot_row0[nr + sh] = n_rows + sh * T;
        }
        s.n_slots[0] = nr + S;
    }
    __syncthreads();
    const int n_slots = s.n_slots[0];
    const int n_routed_slots = n_slots - S;
    for (int u = tid; u < n_slots; u += kThreadsD) {
        const int end = u + 1 < n_routed_slots ? s.slot_row0[u + 1] : (u < n_routed_slots ? n_rows : T);
        s.slot_cnt[u] = u < n_routed_slots ? end - s.slot_row0[u] : T;
    }
    // activations in the phase-1 layout: [t][chunk j][half][lane][16 B], each 8-byte group split even|odd
    if (MODE != DecodeMode::kGemm2Partials) {
        const int per_tok = H / 16;
        for (int o = tid; o < T * per_tok; o += kThreadsD) {
            const int t = o / per_tok, c = o % per_tok;
            const int j = c / 64, half = (c / 32) % 2, l = c % 32;
            const int k0 = 32 * (32 * j + l) + 16 * half;
            const uint4 v = *reinterpret_cast<const uint4*>(a.x_q + static_cast<int64_t>(t) * H + k0);
            *reinterpret_cast<uint4*>(s.x + static_cast<int64_t>(t) * H + c * 16) = split16(v);
        }
        for (int t = tid; t < T; t += kThreadsD) s.xs[t] = routed ? a.x_scale[t] : 1.0f;
    }
    __syncthreads();

    // phase-2 slice of this CTA and its staging
    const int n0 = blockIdx.x * pl.rows_pc;
    const int nrows = max(0, min(pl.rows_pc, H - n0));
    const int slot_w_bytes = pl.rows_pc * (I / 2), slot_s_bytes = pl.rows_pc * ng2 * 4;
    const int n_smem = MODE == DecodeMode::kForward ? min(n_slots, pl.smem_slots) : 0;
    if (MODE == DecodeMode::kForward && tid == 0) {
        if (nrows > 0 && n_smem > 0) {
            const uint32_t wb = nrows * (I / 2), sb = nrows * ng2 * 4;
            mbar_arrive_expect_tx(s.bar, static_cast<uint32_t>(n_smem) * (wb + sb));
            for (int u = 0; u < n_smem; ++u) {
                const int64_t e = s.slot_e[u];
                uint8_t* dst = s.w2s + static_cast<int64_t>(u) * (slot_w_bytes + slot_s_bytes);
                bulk_g2s(dst, a.w2 + (e * H + n0) * (I / 2), wb, s.bar);
                bulk_g2s(dst + slot_w_bytes, a.s2 + (e * H + n0) * ng2, sb, s.bar);
            }
        } else {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(s.bar)) : "memory");
        }
        for (int u = n_smem; u < n_slots && nrows > 0; ++u) {
            const int64_t e = s.slot_e[u];
            bulk_prefetch_l2(a.w2 + (e * H + n0) * (I / 2), nrows * (I / 2));
            bulk_prefetch_l2(a.s2 + (e * H + n0) * ng2, nrows * ng2 * 4);
        }
    }

    // ---------------------------------------------------------------- phase 1
    if (MODE != DecodeMode::kGemm2Partials) {
        const int64_t N1 = static_cast<int64_t>(n_slots) * I;
        const int64_t W = static_cast<int64_t>(gridDim.x) * kWarpsD;
        const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsD + warp;
        const int64_t U0 = gw * N1 / W, U1 = (gw + 1) * N1 / W;
        constexpr int kMaxC1 = C1;
        uint4 wg[kMaxC1], wu[kMaxC1];
        float sg[kMaxC1], su[kMaxC1];
        auto load_unit = [&](int64_t U, uint4* g_, uint4* u_, float* sg_, float* su_) {
            const int u = static_cast<int>(U / I), i = static_cast<int>(U % I);
            const int64_t e = s.slot_e[u];
            const uint8_t* rg = a.w13 + (e * 2 * I + i) * static_cast<int64_t>(H / 2);
            const uint8_t* ru = rg + static_cast<int64_t>(I) * (H / 2);
#pragma unroll
            for (int j = 0; j < kMaxC1; ++j)
                if (j < C1) {
                    g_[j] = ld_stream16(rg + 16 * (32 * j + lane));
                    u_[j] = ld_stream16(ru + 16 * (32 * j + lane));
                    if (MODE == DecodeMode::kForward) {
                        const int q = (32 * (32 * j + lane)) / g;
                        sg_[j] = __ldg(a.s13 + (e * 2 * I + i) * ng1 + q);
                        su_[j] = __ldg(a.s13 + (e * 2 * I + I + i) * ng1 + q);
                    }
                }
        };
        if (U0 < U1) load_unit(U0, wg, wu, sg, su);
        for (int64_t U = U0; U < U1; ++U) {
            uint4 cg[kMaxC1], cu[kMaxC1];
            float csg[kMaxC1], csu[kMaxC1];
#pragma unroll
            for (int j = 0; j < kMaxC1; ++j) {
                cg[j] = wg[j];
                cu[j] = wu[j];
                csg[j] = sg[j];
                csu[j] = su[j];
            }
            if (U + 1 < U1) load_unit(U + 1, wg, wu, sg, su);
            const int u = static_cast<int>(U / I), i = static_cast<int>(U % I);
            const int row0 = s.slot_row0[u], cnt = s.slot_cnt[u];
            for (int m = 0; m < cnt; ++m) {
                const int r = row0 + m;
                const int t = s.row_tok[r];
                int ag[kMaxC1], au[kMaxC1];
#pragma unroll
                for (int j = 0; j < kMaxC1; ++j)
                    if (j < C1) {
                        const uint8_t* xp = s.x + static_cast<int64_t>(t) * H + j * 1024 + lane * 16;
                        const uint4 xa = *reinterpret_cast<const uint4*>(xp);
                        const uint4 xb = *reinterpret_cast<const uint4*>(xp + 512);
                        ag[j] = dot_chunk(cg[j], xa, xb, 0);
                        au[j] = dot_chunk(cu[j], xa, xb, 0);
                    }
                // sum the lanes of each K group (consecutive lanes)
                for (int off = 1; off < lpg1; off <<= 1)
#pragma unroll
                    for (int j = 0; j < kMaxC1; ++j)
                        if (j < C1) {
                            ag[j] += __shfl_xor_sync(0xffffffffu, ag[j], off);
                            au[j] += __shfl_xor_sync(0xffffffffu, au[j], off);
                        }
                const bool leader = (lane % lpg1) == 0;
                if (MODE == DecodeMode::kGemm1Partials) {
                    if (leader) {
                        int32_t* dst = a.p1 + static_cast<int64_t>(r) * (2 * I) * ng1;
#pragma unroll
                        for (int j = 0; j < kMaxC1; ++j)
                            if (j < C1) {
                                const int q = (32 * (32 * j + lane)) / g;
                                dst[static_cast<int64_t>(i) * ng1 + q] = ag[j] >> 4;
                                dst[static_cast<int64_t>(I + i) * ng1 + q] = au[j] >> 4;
                            }
                    }
                    continue;
                }
                float vg = 0.f, vu = 0.f;
                if (leader) {
#pragma unroll
                    for (int j = 0; j < kMaxC1; ++j)
                        if (j < C1) {
                            vg = fmaf(static_cast<float>(ag[j] >> 4), csg[j], vg);
                            vu = fmaf(static_cast<float>(au[j] >> 4), csu[j], vu);
                        }
                }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    vg += __shfl_xor_sync(0xffffffffu, vg, off);
                    vu += __shfl_xor_sync(0xffffffffu, vu, off);
                }
                if (lane == 0) {
                    const float xs = s.xs[t];
                    a.h[static_cast<int64_t>(r) * I + i] = silu_f32(vg * xs) * (vu * xs);
                }
            }
        }
    }
    if (MODE == DecodeMode::kGemm1Partials) return;

    // ---------------------------------------------------------------- barrier
    bool ok = true;
    if (MODE == DecodeMode::kForward) ok = grid_barrier(a.hdr, 1);
    if (!ok) {
        // leave only once this CTA's own bulk copies have landed
        if (tid == 0 && n_smem > 0 && nrows > 0) mbar_wait_bounded(s.bar, 0);
        __syncthreads();
        return;
    }

    // ---------------------------------------------------------------- phase 2
    const int P = n_rows + T * S;
    // (a) int8 rows in the phase-2 layout: [p][chunk j][half][lane 0..15][16 B]
    if (MODE == DecodeMode::kForward) {
        for (int p = warp; p < P; p += kWarpsD) {
            const float* hrow = a.h + static_cast<int64_t>(p) * I;
            float v[C2][16];
            float m = 0.f;
            const int nout = I / 16 / 32;  // 16-byte outputs per lane
#pragma unroll
            for (int c = 0; c < C2; ++c)
                if (c < nout) {
                    const int o = lane + 32 * c;
                    const int j = o / 32, half = (o / 16) % 2, l = o % 16;
                    const int k0 = 32 * (16 * j + l) + 16 * half;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(hrow + k0 + 4 * q));
                        v[c][4 * q] = f.x;
                        v[c][4 * q + 1] = f.y;
                        v[c][4 * q + 2] = f.z;
                        v[c][4 * q + 3] = f.w;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) m = fmaxf(m, fabsf(v[c][q]));
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            const float sc = requant_scale(__float_as_uint(m));
#pragma unroll
            for (int c = 0; c < C2; ++c)
                if (c < nout) {
                    const int o = lane + 32 * c;
                    uint32_t wds[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        wds[q] = (requant_code(v[c][4 * q], sc) & 0xFF) |
                                 ((requant_code(v[c][4 * q + 1], sc) & 0xFF) << 8) |
                                 ((requant_code(v[c][4 * q + 2], sc) & 0xFF) << 16) |
                                 ((static_cast<uint32_t>(requant_code(v[c][4 * q + 3], sc)) & 0xFF) << 24);
                    *reinterpret_cast<uint4*>(s.hq + static_cast<int64_t>(p) * I + o * 16) =
                        split16(make_uint4(wds[0], wds[1], wds[2], wds[3]));
                }
            if (lane == 0) {
                s.sh[p] = sc;
                if (a.amax && blockIdx.x == 0) a.amax[p] = __float_as_uint(m);
            }
        }
    } else {  // kGemm2Partials: rows given as int8
        const int per_row = I / 16;
        for (int o = tid; o < P * per_row; o += kThreadsD) {
            const int p = o / per_row, c = o % per_row;
            const int j = c / 32, half = (c / 16) % 2, l = c % 16;
            const int k0 = 32 * (16 * j + l) + 16 * half;
            const uint4 v = *reinterpret_cast<const uint4*>(a.h_q_in + static_cast<int64_t>(p) * I + k0);
            *reinterpret_cast<uint4*>(s.hq + static_cast<int64_t>(p) * I + c * 16) = split16(v);
        }
    }
    __syncthreads();
    if (MODE == DecodeMode::kForward && n_smem > 0 && nrows > 0) {
        if (tid == 0 && !mbar_wait_bounded(s.bar, 0)) {
            atomicOr(&a.hdr->status, kDevTimeout);
            s.flags[0] = 1;
        }
        __syncthreads();
        if (s.flags[0]) {
            if (tid == 0) mbar_wait_bounded(s.bar, 0);
            __syncthreads();
            return;
        }
    }
    if (nrows == 0) return;

    // (b) down projection: half-warp teams over (slot, row) units
    {
        const int team = warp * 2 + (lane >> 4), n_teams = kWarpsD * 2, l = lane & 15;
        const unsigned hmask = 0xFFFFu << (lane & 16);
        const int lpg2 = g / 32;
        const int n_units = n_slots * nrows;
        constexpr int kMaxC2 = C2;
        for (int U = team; U < n_units; U += n_teams) {
            const int u = U / nrows, r = U % nrows;
            const int64_t e = s.slot_e[u];
            uint4 w[kMaxC2];
            float sc[kMaxC2];
#pragma unroll
            for (int j = 0; j < kMaxC2; ++j)
                if (j < C2) {
                    const int q = (32 * (16 * j + l)) / g;
                    if (u < n_smem) {
                        const uint8_t* base = s.w2s + static_cast<int64_t>(u) * (slot_w_bytes + slot_s_bytes);
                        w[j] = *reinterpret_cast<const uint4*>(base + r * (I / 2) + 16 * (16 * j + l));
                        sc[j] = reinterpret_cast<const float*>(base + slot_w_bytes)[r * ng2 + q];
                    } else {
                        const uint8_t* row = a.w2 + (e * H + n0 + r) * static_cast<int64_t>(I / 2);
                        w[j] = *reinterpret_cast<const uint4*>(row + 16 * (16 * j + l));
                        sc[j] = MODE == DecodeMode::kForward ? __ldg(a.s2 + (e * H + n0 + r) * ng2 + q) : 0.f;
                    }
                }
            const int row0 = s.slot_row0[u], cnt = s.slot_cnt[u];
            for (int m = 0; m < cnt; ++m) {
                const int p = row0 + m;
                int acc[kMaxC2];
#pragma unroll
                for (int j = 0; j < kMaxC2; ++j)
                    if (j < C2) {
                        const uint8_t* xp = s.hq + static_cast<int64_t>(p) * I + j * 512 + l * 16;
                        acc[j] = dot_chunk(w[j], *reinterpret_cast<const uint4*>(xp),
                                           *reinterpret_cast<const uint4*>(xp + 256), 0);
                    }
                for (int off = 1; off < lpg2; off <<= 1)
#pragma unroll
                    for (int j = 0; j < kMaxC2; ++j)
                        if (j < C2) acc[j] += __shfl_xor_sync(hmask, acc[j], off);
                const bool leader = (l % lpg2) == 0;
                if (MODE == DecodeMode::kGemm2Partials) {
                    if (leader) {
                        int32_t* dst = a.p2 + (static_cast<int64_t>(p) * H + n0 + r) * ng2;
#pragma unroll
                        for (int j = 0; j < kMaxC2; ++j)
                            if (j < C2) dst[(32 * (16 * j + l)) / g] = acc[j] >> 4;
                    }
                    continue;
                }
                float v = 0.f;
                if (leader) {
#pragma unroll
                    for (int j = 0; j < kMaxC2; ++j)
                        if (j < C2) v = fmaf(static_cast<float>(acc[j] >> 4), sc[j], v);
                }
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) v += __shfl_xor_sync(hmask, v, off);
                if (l == 0) {
                    const float yv = v * s.sh[p];
                    s.y[p * pl.rows_pc + r] = yv;
                    if (a.y) a.y[static_cast<int64_t>(p) * H + n0 + r] = yv;
                }
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

}  // namespace

// Shared-memory plan of one launch (host side; the kernel reads the offsets).
bool decode_plan(int64_t T, int64_t H, int64_t I, int64_t E, int64_t S, int64_t k, int64_t g, int64_t n_pairs,
                 DecodeMode mode, int grid, int max_smem, DecodePlan* out) {
    if (!decode_shape_supported(H, I) || I > kMaxI || (I / g) % 4 != 0 || g % 32 != 0 || g > 1024) return false;
    if (E > kMaxExperts) return false;
    const int64_t rows = mode == DecodeMode::kForward ? T * k : n_pairs;
    const int64_t Sx = mode == DecodeMode::kForward ? S : 0;
    const int64_t P = rows + T * Sx;
    if (T > kDecodeMaxT || rows > kDecodeMaxPairs || P > kDecodeMaxPairs + kDecodeMaxT * kMaxShared) return false;
    const int64_t MS = rows + Sx;
    DecodePlan pl{};
    pl.rows_pc = static_cast<int>((H + grid - 1) / grid);
    pl.rows_pc = (pl.rows_pc + 1) / 2 * 2;
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) {
        o = align_up(o, al);
        size_t at = o;
        o += bytes;
        return static_cast<int>(at);
    };
    pl.off_bar = take(8, 8);
    pl.off_flags = take(16, 16);
    pl.off_ids = take(4 * rows, 16);
    pl.off_wts = take(4 * rows, 16);
    pl.off_pos = take(4 * rows, 16);
    pl.off_pair_of = take(4 * rows, 16);
    pl.off_row_tok = take(4 * P, 16);
    pl.off_slot_e = take(4 * MS, 16);
    pl.off_slot_row0 = take(4 * MS, 16);
    pl.off_slot_cnt = take(4 * MS, 16);
    pl.off_n_slots = take(16, 16);
    pl.off_xs = take(4 * T, 16);
    pl.off_sh = take(4 * P, 16);
    pl.off_x = take(mode == DecodeMode::kGemm2Partials ? 0 : T * H, 128);
    pl.off_hq = take(mode == DecodeMode::kGemm1Partials ? 0 : P * I, 128);
    pl.off_y = take(mode == DecodeMode::kForward ? 4 * P * pl.rows_pc : 0, 16);
    pl.off_w2s = static_cast<int>(align_up(o, 128));
    const size_t slot_bytes = static_cast<size_t>(pl.rows_pc) * (I / 2) + static_cast<size_t>(pl.rows_pc) * (I / g) * 4;
    const size_t fixed = pl.off_w2s;
    if (fixed > static_cast<size_t>(max_smem)) return false;
    int64_t fit = mode == DecodeMode::kForward ? static_cast<int64_t>((max_smem - fixed) / slot_bytes) : 0;
    pl.smem_slots = static_cast<int>(std::min<int64_t>(fit, MS));
    pl.smem_bytes = static_cast<int>(fixed + pl.smem_slots * slot_bytes);
    *out = pl;
    return true;
}

namespace {
template <DecodeMode MODE, int C1, int C2>
cudaError_t launch_mode(const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    auto kern = decode_kernel<MODE, C1, C2>;
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

template <int C1, int C2>
cudaError_t launch_shape(DecodeMode mode, const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    if (mode == DecodeMode::kForward) return launch_mode<DecodeMode::kForward, C1, C2>(a, pl, grid, st);
    if (mode == DecodeMode::kGemm1Partials) return launch_mode<DecodeMode::kGemm1Partials, C1, C2>(a, pl, grid, st);
    return launch_mode<DecodeMode::kGemm2Partials, C1, C2>(a, pl, grid, st);
}
}  // namespace

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

// (H / 1024, I / 512) shapes the engine is compiled for.
bool decode_shape_supported(int64_t H, int64_t I) {
    if (H % 1024 != 0 || I % 512 != 0) return false;
    const int64_t c1 = H / 1024, c2 = I / 512;
    return (c2 == 1 && (c1 == 1 || c1 == 2 || c1 == 4)) || (c2 == 3 && (c1 == 2 || c1 == 4));
}

cudaError_t launch_decode(DecodeMode mode, const DecodeArgs& a, const DecodePlan& pl, int grid, cudaStream_t st) {
    if (mode == DecodeMode::kForward) {
        cudaError_t e = cudaMemsetAsync(a.hdr, 0, 16, st);  // status and barrier counters
        if (e != cudaSuccess) return e;
    }
    const int c1 = a.H / 1024, c2 = a.I / 512;
    if (c2 == 1 && c1 == 1) return launch_shape<1, 1>(mode, a, pl, grid, st);
    if (c2 == 1 && c1 == 2) return launch_shape<2, 1>(mode, a, pl, grid, st);
    if (c2 == 1 && c1 == 4) return launch_shape<4, 1>(mode, a, pl, grid, st);
    if (c2 == 3 && c1 == 2) return launch_shape<2, 3>(mode, a, pl, grid, st);
    if (c2 == 3 && c1 == 4) return launch_shape<4, 3>(mode, a, pl, grid, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_barrier_timeout_probe(Header* hdr, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(hdr, 0, 16, st);
    if (e != cudaSuccess) return e;
    barrier_timeout_probe_kernel<<<2, 32, 0, st>>>(hdr);
    return cudaGetLastError();
}

}  // namespace moe
