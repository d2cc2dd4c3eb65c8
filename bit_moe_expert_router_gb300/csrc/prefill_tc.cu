// Tensor-core (tcgen05) engine of the W4A8 MoE layer for large batches.
//
// The grouped expert projections are dense contractions once the tokens are
// grouped per expert ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next",
// section 3: grouped expert projections on the matrix unit, blocked
// reduction, W4A8, weights kept packed).  GB300 has no int8 tcgen05 MMA, so
// the operands go to the fp16 MMA (kind::f16): int4 codes and int8 values
// are exact in fp16, each product is exact in the fp32 accumulator and a
// 128-value K group sums to |P| <= 128 * 127 * 8 < 2^24, so every group's
// accumulator holds the exact int32 partial.  One group is accumulated per
// TMEM buffer and folded into fp32 registers with its weight scale by the
// epilogue warps while the tensor core fills the next buffer.
//
// Tile: M = 128 weight rows x N <= 128 tokens of one bank slot, one K
// group (128 values) per pipeline stage, 2 stages.  The A operand (the
// unpacked weights, fp16) goes to tensor memory -- each producer thread
// writes its row's 64 columns into its own lane with tcgen05.st -- and the
// B operand (token rows, fp16) to shared memory in the 128-byte-swizzled
// K-major layout the MMA reads; A thus never passes through shared memory,
// whose bandwidth the MMA's B reads and the B copies then share alone.
// Gate/up tiles interleave the rows (tile row 2j = gate row i, 2j + 1 = up
// row i, i = 64 m + j), so the SiLU(gate) * up product pairs neighbouring
// lanes.  The MMA width N is the token count of the tile rounded up to 16.
// Persistent CTAs (one per SM) walk the (slot, token tile, weight tile)
// items with the weight tile fastest, so the CTAs working at one time share
// the token tile in L2.  Tensor memory: 3 accumulators x 128 columns + 2 A
// stages x 64 columns = all 512 columns.  Three accumulators let the MMAs run
// two groups into the next item while the epilogue finishes an item (SiLU or
// scaling and the stores); that buys more than deeper A/B staging, since the
// producers keep ahead of the MMAs with two stages.
//
// Thirteen warps (four of them share one SM sub-partition, whose 16K-register
// file then caps a thread at 128 registers).  Warp roles: warps 0-7
// epilogue (warp w: TMEM lanes 32 (w % 4) .. +31 = tile rows, columns
// 64 (w / 4) .. +63), warps 8-11 producers (thread = tile row: unpack 64
// packed bytes of its weight row into fp16 and store them to its TMEM lane;
// warp 8 also issues the stage's two TMA tiles of token rows), warp 12 issues
// the MMAs (one thread)
// and owns the TMEM allocation.  Every wait is bounded; a timeout sets the
// status word and every role leaves cleanly.
//
// K order: the weight unpack turns a packed word (codes 0..7) into fp16
// pairs (0,4) (1,5) (2,6) (3,7); the token rows are converted to fp16 in
// the same order by the prep kernels, so both operands agree on K.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "prefill.h"

namespace moe {
namespace {

constexpr int kEpiWarps = 8;                 // two per TMEM lane quarter, 64 columns each
constexpr int kProdWarps = 4;
constexpr int kMmaWarp = kEpiWarps + kProdWarps;
constexpr int kTcThreads = 32 * (kMmaWarp + 1);
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kHalfN = 64;                   // columns per epilogue warp
constexpr int kNS = 2;                       // pipeline stages: A in tensor memory, B in shared memory
constexpr int kTileN = 128;
constexpr int kAtom = 16384;                 // 128 rows x 128 bytes
constexpr int kStage = 2 * kAtom;             // B: 128 token rows x 128 fp16 (two swizzled atoms)
constexpr int kACols = 64;                   // A: 128 rows x 128 fp16 = 64 tensor-memory columns per stage
constexpr int kMaxSlotsTc = kTcMaxSlots + 1;
constexpr int kAcc = 3;                      // accumulator buffers in tensor memory (128 columns each)
constexpr int kTmemCols = 512;               // kAcc * 128 accumulator columns + kNS * kACols A columns
constexpr int kRaw = 3;                      // packed weight rows in flight ahead of the unpack
constexpr int kRawStage = 128 * 64;          // 128 rows x 64 packed bytes (128 codes)
constexpr int kSmemTc =
    kNS * kStage + kRaw * kRawStage + 128 * 4 + 128 * 4 + (kMaxSlotsTc + 16) * 4 + 256 + 1024;
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(kAcc * 128 + kNS * kACols <= kTmemCols, "tensor-memory columns");

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
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

struct Ctl {
    volatile int* abort;
    Header* hdr;
};

// Bounded wait for phase `parity` of `bar`; false if the CTA aborted or the
// wait ran out (then the abort flag and the status word are set).
__device__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 31) {
            if (*c.abort) return false;
            const uint64_t t = global_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > kWaitNs) {
                *c.abort = 1;
                atomicOr(&c.hdr->status, kDevTimeout);
                return false;
            }
        }
    }
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both
// K-major, M = 128, N = n (a multiple of 16, at most 128).
__device__ __forceinline__ uint32_t idesc_f16(int n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | ((128u >> 4) << 24);
}

// MMA with the A operand read from tensor memory (lane = row, K along the columns)
// and B from shared memory (descriptor).
__device__ __forceinline__ void mma_f16_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// TMA: one box (64 fp16 x 128 rows from column x, row y) -> 16 KB of shared memory.
__device__ __forceinline__ void tma_tile2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// SiLU in fast fp32 (hardware exp2 approximation and fast reciprocal divide,
// a few ulp from z / (1 + exp(-z))).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ float ld_nc_f32(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
    return v;
}

// 64 consecutive 32-bit tensor-memory columns of this thread's lane <- v; waits for the store.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,"
        "%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]),
        "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]),
        "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]),
        "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}


// Eight packed int4 codes (element e at bits 4e) -> fp16 pairs (0,4) (1,5) (2,6) (3,7).
// A nibble n of a two's-complement code c satisfies n ^ 8 = c + 8.  Placed in
// the low 4 mantissa bits of fp16 0x6400 (1024) it gives 1024 + c + 8, so
// subtracting 1032 leaves c; placed 4 bits higher it gives 1024 + 16 (c + 8),
// and x / 16 - 72 = c (one exact fma).  Each (w & mask) ^ (0x6400.. | 8-bit)
// is a single three-input logic op.
__device__ __forceinline__ uint4 unpack_int4_f16(uint32_t w) {
    const __half2 sub = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
    const __half2 b72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));   // -72
    const uint32_t w8 = w >> 8;
    uint32_t p[4];
    p[0] = (w & 0x000F000Fu) ^ 0x64086408u;
    p[1] = (w & 0x00F000F0u) ^ 0x64806480u;
    p[2] = (w8 & 0x000F000Fu) ^ 0x64086408u;
    p[3] = (w8 & 0x00F000F0u) ^ 0x64806480u;
    uint32_t r[4];
    const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p[0]), sub);
    const __half2 h1 = __hfma2(*reinterpret_cast<const __half2*>(&p[1]), s16, b72);
    const __half2 h2 = __hsub2(*reinterpret_cast<const __half2*>(&p[2]), sub);
    const __half2 h3 = __hfma2(*reinterpret_cast<const __half2*>(&p[3]), s16, b72);
    r[0] = *reinterpret_cast<const uint32_t*>(&h0);
    r[1] = *reinterpret_cast<const uint32_t*>(&h1);
    r[2] = *reinterpret_cast<const uint32_t*>(&h2);
    r[3] = *reinterpret_cast<const uint32_t*>(&h3);
    return make_uint4(r[0], r[1], r[2], r[3]);
}


__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n)); }

// Named barrier that also ORs a predicate over its threads: every thread gets the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n bar.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(id), "r"(n), "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

struct Item {
    int slot, tt, mt, row0, ntok;
};

template <TcMode MODE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(TcArgs a, int n_mt, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* raw = smem + kNS * kStage;                           // [kRaw][128][64] packed weight rows
    float* colf = reinterpret_cast<float*>(raw + kRaw * kRawStage);  // [128] B-row scales of the item
    int* colp = reinterpret_cast<int*>(colf + 128);               // [128] pair rows of the item
    int* prefix = colp + 128;                                     // [kMaxSlotsTc + 1] items before each slot
    uint64_t* bars = reinterpret_cast<uint64_t*>(prefix + kMaxSlotsTc + 16);
    uint64_t* full = bars;
    uint64_t* empty = bars + kNS;
    uint64_t* accf = bars + 2 * kNS;
    uint64_t* acce = accf + kAcc;
    uint64_t* done = acce + kAcc;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int* warp_sums = abort_flag + 1;  // [kTcThreads / 32 + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool gateup = MODE == TcMode::kGateUp || MODE == TcMode::kGateUpPartials;
    constexpr bool partials = MODE == TcMode::kGateUpPartials || MODE == TcMode::kDownPartials;
    const int64_t K = a.K, rows_per_slot = a.rows_per_slot;
    const int ksteps = static_cast<int>(K / 128), spg = a.g / 128, ngrp = static_cast<int>(K / a.g);
    const Ctl ctl{abort_flag, a.hdr};

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            // 128 producer arrivals (A in tensor memory) + the TMA tiles' expect-tx arrival (B)
            mbar_init(full + s, 129);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < kAcc; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, kEpiThreads);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    // items of each slot -> exclusive prefix (every CTA computes it)
    {
        const int per = (a.n_slots + kTcThreads - 1) / kTcThreads;
        const int u0 = min(a.n_slots, tid * per), u1 = min(a.n_slots, (tid + 1) * per);
        int local = 0;
        for (int u = u0; u < u1; ++u) local += ((a.seg_cnt[u] + kTileN - 1) / kTileN) * n_mt;
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int w2 = 0; w2 < kTcThreads / 32; ++w2) {
                const int v = warp_sums[w2];
                warp_sums[w2] = run;
                run += v;
            }
            warp_sums[kTcThreads / 32] = run;
        }
        __syncthreads();
        int run = warp_sums[warp] + incl - local;
        for (int u = u0; u < u1; ++u) {
            prefix[u] = run;
            run += ((a.seg_cnt[u] + kTileN - 1) / kTileN) * n_mt;
        }
        if (tid == 0) prefix[a.n_slots] = warp_sums[kTcThreads / 32];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = prefix[a.n_slots];

    auto decode_item = [&](int item) {
        int lo = 0, hi = a.n_slots;  // last slot whose first item is <= item
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= item) lo = mid;
            else hi = mid;
        }
        Item it;
        it.slot = lo;
        const int local = item - prefix[lo];
        it.tt = local / n_mt;
        it.mt = local % n_mt;
        it.row0 = a.seg_off[lo] + kTileN * it.tt;
        it.ntok = min(kTileN, a.seg_off[lo] + a.seg_cnt[lo] - it.row0);
        return it;
    };
    // bank row of tile row r (gate/up: gate and up rows interleaved)
    auto weight_row = [&](int mt, int r) -> int64_t {
        if (gateup) return ((r & 1) ? a.I : 0) + 64 * mt + (r >> 1);
        return static_cast<int64_t>(128) * mt + r;
    };

    if (warp >= kEpiWarps && warp < kMmaWarp) {
        // ------------------------------------------------------------ producers
        // Each thread owns tile row pt.  The packed weight bytes for use
        // u + kRaw are copied (cp.async) into the raw ring while use u is
        // unpacked, so the unpack never waits for HBM.  The copies are
        // coalesced within the warp (4 lanes per row, 8 rows of 64 contiguous
        // bytes per instruction), so a lane waits for its own copies and then
        // syncs the warp before reading its row.
        const int pt = tid - kEpiThreads;
        const int pw = warp - kEpiWarps;
        // 16-byte chunk q of row pt sits at chunk q ^ rsw: eight consecutive rows
        // (64 bytes apart) then hit eight different bank groups
        const int rsw = (pt >> 1) & 3;
        int l_item = blockIdx.x, l_ks = 0;  // next use whose raw bytes are fetched
        const uint8_t* l_slot = nullptr;    // its slot's packed rows
        int l_mt = 0;
        if (l_item < total) {
            const Item it = decode_item(l_item);
            l_slot = a.w + static_cast<int64_t>(it.slot) * rows_per_slot * (K / 2);
            l_mt = it.mt;
        }
        int l_use = 0;
        const int piece = lane & 3;
        auto fetch_next = [&]() {
            if (l_item < total) {
                uint8_t* dst = raw + (l_use % kRaw) * kRawStage;
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // rows 32 pw + 8 q .. + 7, 4 lanes per row
                    const int row = 32 * pw + 8 * q + (lane >> 2);
                    const int rs = (row >> 1) & 3;
                    cp_async16(dst + row * 64 + 16 * (piece ^ rs),
                               l_slot + weight_row(l_mt, row) * (K / 2) + 64 * l_ks + 16 * piece);
                }
                ++l_use;
                if (++l_ks == ksteps) {
                    l_ks = 0;
                    l_item += gridDim.x;
                    if (l_item < total) {
                        const Item it = decode_item(l_item);
                        l_slot = a.w + static_cast<int64_t>(it.slot) * rows_per_slot * (K / 2);
                        l_mt = it.mt;
                    }
                }
            }
            cp_async_commit();  // one group per call, empty or not, so the group count stays aligned
        };
#pragma unroll
        for (int d = 0; d < kRaw; ++d) fetch_next();
        int use = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            const Item it = decode_item(item);
            if (named_bar_or(2, 128, !ok)) break;  // the four producer warps give up together
            for (int ks = 0; ks < ksteps; ++ks, ++use) {
                const int s = use % kNS;
                if (!wait_bar(empty + s, ((use / kNS) & 1) ^ 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the stage's previous MMAs (which read its A columns) are complete
                uint8_t* Bs = stages + s * kStage;
                // B, the 128 token rows of the stage (contiguous fp16 rows): two 2-D
                // TMA tiles, one per 128-byte-swizzled atom, issued by producer warp 0
                if (warp == kEpiWarps && lane == 0) {
                    mbar_expect_tx(full + s, kStage);
#pragma unroll
                    for (int at = 0; at < 2; ++at) tma_tile2d(Bs + at * kAtom, &bmap, 128 * ks + 64 * at, it.row0, full + s);
                }
                cp_async_wait<kRaw - 1>();  // this lane's copies for this use (issued kRaw calls ago) have landed
                __syncwarp();               // ... and the other lanes' copies of this warp's rows
                const uint4* rp = reinterpret_cast<const uint4*>(raw + (use % kRaw) * kRawStage + pt * 64);
                uint4 rw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) rw[q] = rp[q ^ rsw];
                // unpacked row -> this thread's tensor-memory lane, 64 columns of
                // fp16 pairs (column c holds K positions 2c, 2c + 1 of the stage)
                uint32_t av[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t words[4] = {rw[q].x, rw[q].y, rw[q].z, rw[q].w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const uint4 u4 = unpack_int4_f16(words[wi]);
                        const int c = 4 * (4 * q + wi);
                        av[c] = u4.x;
                        av[c + 1] = u4.y;
                        av[c + 2] = u4.z;
                        av[c + 3] = u4.w;
                    }
                }
                tmem_st64(tmem + (static_cast<uint32_t>(32 * (warp - kEpiWarps)) << 16) + kAcc * 128 + kACols * s, av);
                // the raw slot just consumed is refilled kRaw uses ahead, after every
                // lane of the warp has read its row from it
                __syncwarp();
                fetch_next();
                tc_fence_before();
                mbar_arrive(full + s);
            }
        }
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int use = 0, grp = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = decode_item(item);
                const uint32_t idesc = idesc_f16((it.ntok + 15) & ~15);
                for (int ks = 0; ks < ksteps; ++ks, ++use) {
                    const int s = use % kNS;
                    const int sub = ks % spg;
                    const int b = grp % kAcc;
                    if (!wait_bar(full + s, (use / kNS) & 1, ctl) ||
                        (sub == 0 && !wait_bar(acce + b, ((grp / kAcc) & 1) ^ 1, ctl))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b0 = smem_u32(stages + s * kStage);
                    const uint32_t ta = tmem + kAcc * 128 + kACols * s;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {  // K = 16 per MMA: 8 A columns, 32 B of a B row
                        const uint32_t off = (kk >> 2) * kAtom + 32 * (kk & 3);
                        mma_f16_ta(tmem + b * 128, ta + 8 * kk, sdesc(b0 + off), idesc, (sub > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(empty + s);
                    if (sub == spg - 1) {
                        mma_commit(accf + b);
                        ++grp;
                    }
                }
            }
            mma_commit(done);  // arrives once every MMA issued above has completed
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(done, 0)) {
                if (global_ns() - t0 > kWaitNs) {
                    atomicOr(&a.hdr->status, kDevTimeout);
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // warp w: TMEM lanes 32 (w % 4) .. +31 (tile rows), columns 64 (w / 4) .. +63
        const int quarter = warp & 3, c_base = kHalfN * (warp >> 2);
        const int r = 32 * quarter + lane;  // tile row
        int grp = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            const Item it = decode_item(item);
            if (tid < it.ntok) {
                const int p = it.row0 + tid;
                colp[tid] = p;
                if (!partials) colf[tid] = gateup ? a.b_scale[a.b_row ? a.b_row[p] : p] : a.b_scale[p];
            }
            named_bar(1, kEpiThreads);
            const int nloc = min(kHalfN, it.ntok - c_base);  // this warp's live columns (may be <= 0)
            const int64_t wrow = weight_row(it.mt, r);
            const float* srow = a.ws + (static_cast<int64_t>(it.slot) * rows_per_slot + wrow) * ngrp;
            float acc[kHalfN];
#pragma unroll
            for (int c = 0; c < kHalfN; ++c) acc[c] = 0.f;
            bool ok = true;
            // group scales two groups ahead (volatile loads: issued before the waits)
            float sc1 = partials ? 0.f : ld_nc_f32(srow), sc2 = (partials || ngrp < 2) ? 0.f : ld_nc_f32(srow + 1);
            for (int gq = 0; gq < ngrp; ++gq, ++grp) {
                const int b = grp % kAcc;
                const float sc = sc1;
                sc1 = sc2;
                if (!partials && gq + 2 < ngrp) sc2 = ld_nc_f32(srow + gq + 2);
                if (!wait_bar(accf + b, (grp / kAcc) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < kHalfN / 32; ++i) {
                    if (32 * i >= nloc) break;
                    uint32_t v[32];
                    tmem_ld32(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + b * 128 + c_base + 32 * i, v);
                    if (partials) {
                        int32_t* dst = a.partials + wrow * ngrp + gq;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (32 * i + c < nloc)
                                dst[static_cast<int64_t>(colp[c_base + 32 * i + c]) * rows_per_slot * ngrp] =
                                    __float2int_rn(__uint_as_float(v[c]));
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) acc[32 * i + c] = fmaf(__uint_as_float(v[c]), sc, acc[32 * i + c]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acce + b);
            }
            if (ok && MODE == TcMode::kGateUp) {
                // lanes 2j (gate) and 2j+1 (up) hold index i for every column: for a
                // column pair (c0, c1) the even lane finishes c0 and the odd lane c1
                const int64_t i = 64 * it.mt + (r >> 1);
                const bool odd = r & 1;
#pragma unroll
                for (int c0 = 0; c0 < kHalfN; c0 += 2) {
                    const int c = c0 + (odd ? 1 : 0);
                    const float other = __shfl_xor_sync(0xffffffffu, odd ? acc[c0] : acc[c0 + 1], 1);
                    const float gate = odd ? other : acc[c0], up = odd ? acc[c0 + 1] : other;
                    if (c < nloc) {
                        const float xs = colf[c_base + c];
                        a.h[static_cast<int64_t>(colp[c_base + c]) * a.I + i] = silu_fast(gate * xs) * (up * xs);
                    }
                }
            } else if (ok && MODE == TcMode::kDown) {
                const int64_t n = 128 * it.mt + r;
#pragma unroll
                for (int c = 0; c < kHalfN; ++c)
                    if (c < nloc) a.y[static_cast<int64_t>(colp[c_base + c]) * a.H + n] = acc[c] * colf[c_base + c];
            }
            // colf / colp are reused by the next item; leave together if any thread gave up
            if (named_bar_or(1, kEpiThreads, !ok)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
    }
}

// x_q int8 -> fp16 rows in the engine's K order (pairs (0,4)(1,5)(2,6)(3,7) per
// 8 values); out row r is token row_token[r] (null: r), zeros for a token
// outside [0, T).  Idx: the type of the element index 8 i (32-bit when
// rows * H fits, which keeps the row/column split a 32-bit division).
template <typename Idx>
__global__ void prep_x16_kernel(const int8_t* __restrict__ x, int64_t T, int64_t H, const int32_t* __restrict__ row_token,
                                int64_t n8, __half* __restrict__ out) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const Idx i8 = static_cast<Idx>(8 * i), Hx = static_cast<Idx>(H);
        const int64_t r = static_cast<int64_t>(i8 / Hx), c = static_cast<int64_t>(i8 % Hx);
        const int64_t t = row_token ? row_token[r] : r;
        uint2 v = make_uint2(0u, 0u);
        if (t >= 0 && t < T) v = *reinterpret_cast<const uint2*>(x + t * H + c);
        const int8_t* b = reinterpret_cast<const int8_t*>(&v);
        __half2 o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = __halves2half2(__int2half_rn(b[e]), __int2half_rn(b[e + 4]));
        *reinterpret_cast<uint4*>(out + 8 * i) = *reinterpret_cast<const uint4*>(o);
    }
}

// h fp32 -> requantised codes as fp16 in the engine's K order, one warp per
// pair row: the row maximum of |h| (-> amax bits and s_h = max / 127), then
// the codes (fp32 decision, IEEE division).  With hq_in (no h) the int8
// codes are converted as given.
__global__ void prep_h16_kernel(const float* __restrict__ h, uint32_t* __restrict__ amax,
                                const int8_t* __restrict__ hq_in, int64_t P, int64_t I, __half* __restrict__ out,
                                float* __restrict__ s_h) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < P; row += nw) {
        const float* hr = h ? h + row * I : nullptr;
        float s = 0.f;
        if (hr) {
            float m = 0.f;
            for (int64_t k = 8 * lane; k < I; k += 256) {
                const float4 f0 = *reinterpret_cast<const float4*>(hr + k);
                const float4 f1 = *reinterpret_cast<const float4*>(hr + k + 4);
                m = fmaxf(m, fmaxf(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f0.z), fabsf(f0.w))),
                                   fmaxf(fmaxf(fabsf(f1.x), fabsf(f1.y)), fmaxf(fabsf(f1.z), fabsf(f1.w)))));
            }
            m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
            s = requant_scale(__float_as_uint(m));
            if (lane == 0) {
                if (amax) amax[row] = __float_as_uint(m);
                if (s_h) s_h[row] = s;
            }
        }
        for (int64_t k = 8 * lane; k < I; k += 256) {
            int code[8];
            if (hr) {
                const float4 f0 = *reinterpret_cast<const float4*>(hr + k);
                const float4 f1 = *reinterpret_cast<const float4*>(hr + k + 4);
                const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) code[e] = requant_code(f[e], s);
            } else {
                const uint2 v = *reinterpret_cast<const uint2*>(hq_in + row * I + k);
                const int8_t* b = reinterpret_cast<const int8_t*>(&v);
#pragma unroll
                for (int e = 0; e < 8; ++e) code[e] = b[e];
            }
            __half2 o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = __halves2half2(__int2half_rn(code[e]), __int2half_rn(code[e + 4]));
            *reinterpret_cast<uint4*>(out + row * I + k) = *reinterpret_cast<const uint4*>(o);
        }
    }
}

// Tensor map of contiguous B rows (fp16 [b_rows][K]) for the TMA unit:
// boxes of 64 columns (128 bytes, the swizzle span) by 128 rows; rows past
// the end read zeros.
cudaError_t make_bmap(const TcArgs& a, CUtensorMap* map) {
    using Encode = PFN_cuTensorMapEncodeTiled_v12000;
    static Encode encode = nullptr;
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess) return e;
            if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
            encode = reinterpret_cast<Encode>(fn);
        }
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.b_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a.b), dims, strides, box, elem,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <TcMode MODE>
cudaError_t launch_mode_tc(const TcArgs& a, int n_mt, cudaStream_t st) {
    auto kern = tc_gemm_kernel<MODE>;
    static std::mutex mu;
    static std::map<int, bool> attr_set;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set.count(dev)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    alignas(64) CUtensorMap bmap{};
    if (cudaError_t e = make_bmap(a, &bmap); e != cudaSuccess) return e;
    kern<<<num_sms(), kTcThreads, kSmemTc, st>>>(a, n_mt, bmap);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int64_t H, int64_t I, int64_t g) {
    return g % 128 == 0 && H % 128 == 0 && I % 128 == 0 && H >= 128 && I >= 128;
}

cudaError_t launch_tc_gemm(TcMode mode, const TcArgs& a, cudaStream_t st) {
    if (a.n_slots < 1 || a.n_slots > kTcMaxSlots) return cudaErrorInvalidValue;
    const bool gateup = mode == TcMode::kGateUp || mode == TcMode::kGateUpPartials;
    const int n_mt = static_cast<int>(gateup ? a.I / 64 : a.H / 128);
    switch (mode) {
        case TcMode::kGateUp: return launch_mode_tc<TcMode::kGateUp>(a, n_mt, st);
        case TcMode::kDown: return launch_mode_tc<TcMode::kDown>(a, n_mt, st);
        case TcMode::kGateUpPartials: return launch_mode_tc<TcMode::kGateUpPartials>(a, n_mt, st);
        default: return launch_mode_tc<TcMode::kDownPartials>(a, n_mt, st);
    }
}

cudaError_t launch_prep_x16(const int8_t* x_q, int64_t T, int64_t H, const int32_t* row_token, int64_t rows, __half* x16,
                            cudaStream_t st) {
    const int64_t n8 = rows * H / 8;
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(blocks, 1));
    if (rows * H < (int64_t(1) << 32))
        prep_x16_kernel<uint32_t><<<grid, 256, 0, st>>>(x_q, T, H, row_token, n8, x16);
    else
        prep_x16_kernel<uint64_t><<<grid, 256, 0, st>>>(x_q, T, H, row_token, n8, x16);
    return cudaGetLastError();
}

cudaError_t launch_prep_h16(const float* h, uint32_t* amax, const int8_t* hq_in, int64_t P, int64_t I, __half* h16,
                            float* s_h, cudaStream_t st) {
    const int64_t blocks = std::min<int64_t>((P + 7) / 8, static_cast<int64_t>(num_sms()) * 8);
    prep_h16_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(h, amax, hq_in, P, I, h16,
                                                                                          s_h);
    return cudaGetLastError();
}

}  // namespace moe
