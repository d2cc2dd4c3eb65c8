// Tensor-core (tcgen05) engine of the W4A8 MoE layer for large batches.
//
// The grouped expert projections are dense contractions once the tokens are
// grouped per expert ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next",
// section 3: grouped expert projections on the matrix unit, blocked
// reduction, W4A8, weights kept packed).  GB300 has no fast int8 tcgen05
// MMA, so the operands go to the fp16 MMA (kind::f16).
//
// Two accumulation schedules:
//   Exact (gate/up, and both partials modes): int4 codes and int8 values are
//     exact in fp16, each product is exact in the fp32 accumulator and a
//     128-value K group sums to |P| <= 128 * 127 * 8 < 2^24, so every group's
//     accumulator holds the exact int32 partial.  Each group gets its own
//     tensor-memory buffer; the epilogue folds it into fp32 registers with
//     its weight scale (or writes the partial) while the tensor core fills
//     the other buffer.  The requantised intermediate depends on h at the
//     rounding level, so gate/up stays exact.
//   Scaled (down): the producers multiply each code by its group's scale
//     over the row's largest scale (a fraction of magnitude <= 1, rounded to
//     fp16, then the product rounded to fp16: within 2^-10 relative of the
//     dequantised weight) and one accumulator sums the item's whole K range;
//     the epilogue multiplies the row's largest scale back once.  One drain
//     per item instead of one per K group: the epilogue's work and its
//     hand-offs with the MMA thread drop by the group count, and the output
//     stores overlap the next item's MMAs.  The error enters the layer
//     output directly (no requantisation after it), far inside the output
//     tolerance.
//
// Tile: M = 128 weight rows x N <= 192 tokens of one bank slot, one K group
// (128 values) per B stage.  An M = 128, K = 16 MMA takes N / 2 cycles for
// N >= 64 on this GPU (64 at N = 128, 96 at N = 192, 128 at N = 256, A in
// tensor or shared memory alike) and ~45 cycles below that; wide token
// tiles spread each A stage (the unpack and its tensor-memory stores) and
// each accumulator drain over more tokens.  192 columns is the widest that
// leaves two accumulators and two A stages in the 512 columns of tensor
// memory (2 x 192 + 2 x 64).
//   A (the unpacked weights, fp16): the packed rows of a stage (128 rows x
//     128 codes) land in a 3-deep shared-memory ring as two 2-D TMA tiles of
//     64 rows, issued by a loader warp of their own (64-byte rows, 64-byte
//     swizzle; a 2-bit slot's 32-byte rows, 32-byte swizzle, through a map of
//     their own).  (The TMA tiles measured 5-7% faster per step than the
//     producers' own cp.async copies; an earlier TMA version, whose tiles
//     shared an issuing thread with the B tiles, measured slower.)  Each
//     producer thread unpacks its row's 128 codes and writes them to its own
//     tensor-memory lane with tcgen05.st, so the unpacked A never passes
//     through shared memory.  Gate/up tiles interleave the rows (tile row
//     2j = gate row i, 2j + 1 = up row i, i = 64 m + j): the SiLU(gate) * up
//     product pairs neighbouring lanes.
//   B (token rows, fp16, 128-byte-swizzled K-major atoms): contiguous rows
//     by pair row -- the activations gathered per pair (gate/up) or the
//     requantised h (down) -- loaded as two 2-D TMA tiles per stage by a
//     warp of its own, four stages deep.  (Gathering the activation rows
//     inside the kernel from a per-token table, by TMA tile::gather4 or by
//     16-byte cp.async copies, measured several times slower here: the row
//     requests cost far more than the bytes.)
// Persistent CTAs (one per SM) walk the (slot, token tile, weight tile)
// items with the weight tile fastest, so the CTAs working at one time share
// the token rows in L2.  An item's A stages and accumulator drains, which
// set its pace, do not depend on its width (a narrow tile only shortens its
// MMAs), so a static round-robin deal balances the grid.
//
// Epilogue.  Gate/up: h = SiLU(x_scale G_gate) * (x_scale G_up) by pair row.
// Down: Y = s_h * sum_q s2 P2 by pair row, stored in bf16 for the combine
// kernel, which sums each token's pairs in a fixed order in fp32 (adding the
// pairs into the output with device reductions instead measured several
// times slower: the reductions of one tile outlast its MMAs many times over).
// Both are stored straight from the registers: for one token column a
// warp's lanes hold consecutive output features, and a tile's pair rows are
// consecutive.
//
// Nineteen warps: 0 MMA issue (one thread; the tensor-memory allocation is
// the warp's), 1 the B tiles (one thread), 2-5 producers (thread = tile row
// of A, rows 32 (w % 4) .. +31; 2-9 for the down projection, two K halves
// per row) and then the epilogue (warp w: TMEM lanes 32 (w % 4) .. +31 =
// tile rows, a column range per group of four warps), 18 the A tiles (one
// thread).  The MMA thread does nothing but wait, issue and commit, and it
// has the lowest warp id: with busy warps beside it on its scheduler each of
// its instructions otherwise waited tens of cycles, and its loop has to stay
// inside the MMA time of a use.  Every wait is bounded (the waiting thread
// sleeps in the barrier test); a timeout sets the status word and every role
// leaves cleanly.
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

// Roles by warp.  The single-thread roles come first: a warp scheduler that has several ready
// warps favours the lower warp ids, and these threads' loops set the pace of everything else.
// A warp reaches only the tensor-memory lane quarter warp % 4, so the four producer warps and
// each group of four epilogue warps cover the four quarters in some order.
constexpr int kMmaWarp = 0;                  // MMA issue and the tensor-memory allocation
constexpr int kBWarp = 1;                    // B tiles
constexpr int kProdWarp0 = 2;                // producers, then the epilogue (split per mode below)
constexpr int kNumWarps = 19;
constexpr int kAWarp = kNumWarps - 1;        // packed A tiles by TMA
constexpr int kTcThreads = 32 * kNumWarps;
constexpr int kTileN = 192;                  // tokens per tile (MMA width <= 192)
constexpr int kAcc = 2;                      // accumulators in tensor memory
constexpr int kAStages = 2;                  // A stages in tensor memory: one K group (64 columns) each
constexpr int kACols = 64;
constexpr int kACol0 = kAcc * kTileN;        // first A column
constexpr int kTmemCols = 512;
constexpr int kBStages = 4;
constexpr int kBAtom = kTileN * 128;         // 192 rows x 128 bytes (64 fp16 of K)
constexpr int kBStage = 2 * kBAtom;          // 128 values of K
constexpr int kRaw = 3;                      // packed weight stages in flight
constexpr int kRawStage = 128 * 64;          // 128 rows x 64 packed bytes (128 codes)
constexpr int kMaxSlotsTc = kTcMaxSlots + 1;
// Shared-memory layout (byte offsets from the 1024-aligned base), one region after another.
constexpr int kOffB = 0;                                        // [kBStages][2 atoms][192 rows][128 B]
constexpr int kOffRaw = kOffB + kBStages * kBStage;             // [kRaw][128 rows][64 B], 64-byte swizzle
constexpr int kOffColp = kOffRaw + kRaw * kRawStage;            // int [2][192]: pair rows of the item (two items)
constexpr int kOffColf = kOffColp + 2 * kTileN * 4;             // float [2][192]: their scales
constexpr int kOffPrefix = kOffColf + 2 * kTileN * 4;           // int [kMaxSlotsTc + 1]: items before each slot
constexpr int kItab = 256;                                      // this CTA's first items, decoded once
constexpr int kOffItab = kOffPrefix + ((kMaxSlotsTc + 1) * 4 + 7) / 8 * 8;  // ItemRec [kItab]
constexpr int kOffBars = kOffItab + kItab * 8;                  // mbarriers, then small words
constexpr int kBarWords = kAStages + 2 * kBStages + 2 * kAcc + 1 + 2 * kRaw;
constexpr int kOffMisc = kOffBars + 8 * kBarWords;              // tmem holder, abort flag, warp sums
constexpr int kSmemUsed = kOffMisc + 4 * (2 + kNumWarps + 1);
constexpr int kSmemTc = kSmemUsed + 1024;                      // + room to align the base to 1024 bytes
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSleepNs = 20000;  // longest sleep inside one barrier test
static_assert(kAcc * kTileN + kAStages * kACols <= kTmemCols, "tensor-memory columns");

static_assert(kSmemTc <= 227 * 1024, "shared memory");
static_assert(kOffRaw % 1024 == 0 && kOffColp % 16 == 0 && kOffBars % 8 == 0, "region alignment");
static_assert(kRawStage == 128 * 64, "raw stage: 128 rows of 64 packed bytes");
static_assert((kOffB + kBStages * kBStage) >> 4 < (1 << 14), "B stages addressable by a matrix descriptor");

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
// The same test, but the thread may sleep in the instruction for up to `ns` nanoseconds (it is
// woken when the phase completes): a waiting warp then takes no issue slots from the warps
// doing the work.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
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
        if (mbar_wait_sleep(bar, parity, kSleepNs)) return true;
        if ((it & 7) == 7) {
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
// K-major, M = 128, N = n (a multiple of 16).
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

// TMA: 2-D box at (x, y) of `map` -> shared memory, completion counted on `bar`.
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

// 16 consecutive 32-bit tensor-memory columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
// 8 consecutive 32-bit tensor-memory columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* v) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }


// 32 consecutive 32-bit tensor-memory columns of this thread's lane <- v (no wait).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Eight packed int4 codes (element e at bits 4e) -> fp16 pairs (0,4) (1,5) (2,6) (3,7).
// A nibble n of a two's-complement code c satisfies n ^ 8 = c + 8.  Placed in
// the low 4 mantissa bits of fp16 0x6400 (1024) it gives 1024 + c + 8, so
// subtracting 1032 leaves c; placed 4 bits higher it gives 1024 + 16 (c + 8),
// and x / 16 - 72 = c (one exact fma).  Each (w & mask) ^ (0x6400.. | 8-bit)
// is a single three-input logic op.
__device__ __forceinline__ void unpack_int4_f16(uint32_t w, uint32_t* r) {
    const __half2 sub = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
    const __half2 b72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));   // -72
    const uint32_t w8 = w >> 8;
    uint32_t p[4];
    p[0] = (w & 0x000F000Fu) ^ 0x64086408u;
    p[1] = (w & 0x00F000F0u) ^ 0x64806480u;
    p[2] = (w8 & 0x000F000Fu) ^ 0x64086408u;
    p[3] = (w8 & 0x00F000F0u) ^ 0x64806480u;
    const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p[0]), sub);
    const __half2 h1 = __hfma2(*reinterpret_cast<const __half2*>(&p[1]), s16, b72);
    const __half2 h2 = __hsub2(*reinterpret_cast<const __half2*>(&p[2]), sub);
    const __half2 h3 = __hfma2(*reinterpret_cast<const __half2*>(&p[3]), s16, b72);
    r[0] = *reinterpret_cast<const uint32_t*>(&h0);
    r[1] = *reinterpret_cast<const uint32_t*>(&h1);
    r[2] = *reinterpret_cast<const uint32_t*>(&h2);
    r[3] = *reinterpret_cast<const uint32_t*>(&h3);
}

// Sixteen packed 2-bit codes (element 4j + p in bits 2p, 2p+1 of byte j, two's complement in
// [-2, 1]) -> fp16 pairs (0,4) (1,5) (2,6) (3,7) of each 8, the same K order as the int4 unpack.  A
// field f satisfies f ^ 2 = c + 2: in the low mantissa bits of fp16 0x6400 (1024) it gives
// 1024 + c + 2, and subtracting 1026 leaves c.  Bytes 0 and 1 hold codes 0-3 and 4-7, so spreading
// them to the two halves of a word lines each pair's codes up in one shift and one mask.
__device__ __forceinline__ void unpack_int2_f16(uint32_t w, uint32_t* r) {
    const __half2 sub = __halves2half2(__ushort_as_half(0x6402), __ushort_as_half(0x6402));  // 1026
    const uint32_t y0 = __byte_perm(w, 0u, 0x4140), y1 = __byte_perm(w, 0u, 0x4342);  // bytes (0,1), (2,3) -> halves
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t q0 = ((y0 >> (2 * p)) & 0x00030003u) ^ 0x64026402u;
        const uint32_t q1 = ((y1 >> (2 * p)) & 0x00030003u) ^ 0x64026402u;
        const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&q0), sub);
        const __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&q1), sub);
        r[p] = *reinterpret_cast<const uint32_t*>(&h0);
        r[4 + p] = *reinterpret_cast<const uint32_t*>(&h1);
    }
}

// Largest |scale| of a weight row's n groups (0 for an all-zero row).  The producers put each
// group's scale into A as a fraction of it and the epilogue multiplies it back: both read the same
// values, and a maximum does not depend on the order it is taken in.
__device__ __forceinline__ float row_scale_max(const float* s, int n) {
    float m = 0.f;
    for (int g = 0; g < n; ++g) m = fmaxf(m, fabsf(__ldg(s + g)));
    return m;
}

// Named barriers of n threads.  The non-aligned forms (barrier.sync / barrier.red, not bar.*):
// they are reached right after per-thread bounded spin waits, so a warp may arrive diverged, and
// the compiler does not reconverge a warp before an inline-asm barrier.

// Named barrier that also ORs a predicate over its threads: every thread gets the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n barrier.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(id), "r"(n), "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}



// Producer / epilogue split of the warps after the two single-thread roles.  The exact modes
// drain the accumulator every K group, so their epilogue gets 12 warps (64 columns each); the
// scaled (down) mode drains once per item and its producers carry the scaling, so it gets 8
// producers (each quarter's rows split in two K halves) and 8 epilogue warps (96 columns each).
template <TcMode M>
struct Roles {
    static constexpr bool scaled = M == TcMode::kDown || M == TcMode::kDownY;
    static constexpr int prod = scaled ? 8 : 4;
    static constexpr int epi0 = kProdWarp0 + prod;
    static constexpr int epi = kAWarp - epi0;
    static constexpr int cols = 4 * kTileN / epi;  // accumulator columns per epilogue warp
    static constexpr int parts = prod / 4;         // K parts of a stage, one per producer warp of a quarter
    static_assert(prod % 4 == 0 && epi % 4 == 0 && cols % 16 == 0 && 4 * kTileN % epi == 0, "warp split");
};

struct Item {
    int slot, mt, row0, ntok;
};
// A decoded item as kept in shared memory.
struct ItemRec {
    int row0;
    int16_t slot;
    uint8_t mt, ntok_m1;
};
static_assert(sizeof(ItemRec) == 8, "item record");

// COMPACT: the bank is in compact storage (a.w_off), a variant of its own (its A loader reads the
// slots' offsets; the uniform layout's needs none).
template <TcMode MODE, bool COMPACT = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(TcArgs a, int n_mt, const __grid_constant__ CUtensorMap bmap,
                   const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap amap2) {
    extern __shared__ uint8_t smem_raw[];
    // (offset from the __shared__ array itself, not an integer cast: the compiler then keeps every
    // access below in the shared state space and knows it cannot alias the global stores)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* bstages = smem + kOffB;
    uint8_t* raw = smem + kOffRaw;
    int* colp_buf = reinterpret_cast<int*>(smem + kOffColp);
    float* colf_buf = reinterpret_cast<float*>(smem + kOffColf);
    int* prefix = reinterpret_cast<int*>(smem + kOffPrefix);
    ItemRec* itab = reinterpret_cast<ItemRec*>(smem + kOffItab);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    // Use u: its A stage is u % kAStages, its B stage and its empty barrier u % kBStages.
    uint64_t* a_full = bars;                     // [kAStages] 128 producer arrivals (the last after B landed)
    uint64_t* b_full = a_full + kAStages;        // [kBStages] expect-tx arrival + TMA bytes
    uint64_t* empty = b_full + kBStages;         // [kBStages] MMA commit: use u's A and B stages are read
    uint64_t* accf = empty + kBStages;           // [kAcc] MMA commit at a group's end
    uint64_t* acce = accf + kAcc;                // [kAcc] epilogue arrivals
    uint64_t* done = acce + kAcc;
    uint64_t* raw_full = done + 1;               // [kRaw] expect-tx arrival + the A tile bytes
    uint64_t* raw_empty = raw_full + kRaw;       // [kRaw] the producers have unpacked the stage
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int* warp_sums = abort_flag + 1;  // [kNumWarps + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool gateup = MODE == TcMode::kGateUp || MODE == TcMode::kGateUpPartials;
    constexpr bool partials = MODE == TcMode::kGateUpPartials || MODE == TcMode::kDownPartials;
    // Down projection outputs: the group scales ride in A and one accumulator sums the item's
    // whole K range.  Every other mode keeps one exact int32 partial per K group.
    using R = Roles<MODE>;
    constexpr bool scaled = R::scaled;
    constexpr int kColsW = R::cols;
    constexpr int kEpiThreads = 32 * R::epi;
    const int64_t K = a.K, rows_per_slot = a.rows_per_slot;
    const int ksteps = static_cast<int>(K / 128), spg = a.g / 128, ngrp = static_cast<int>(K / a.g);
    const Ctl ctl{abort_flag, a.hdr};

    if (tid == 0) {
        for (int s = 0; s < kAStages; ++s) mbar_init(a_full + s, 32 * R::prod);
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(b_full + s, 1);  // expect-tx arrival + the TMA bytes
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < kAcc; ++b) {
            mbar_init(accf + b, 1);
            mbar_init(acce + b, kEpiThreads);
        }
        mbar_init(done, 1);
        for (int r = 0; r < kRaw; ++r) {
            mbar_init(raw_full + r, 1);
            mbar_init(raw_empty + r, 32 * R::prod);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == kMmaWarp) {  // (a converged warp; warp-aligned alloc)
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
        it.mt = local % n_mt;
        it.row0 = a.seg_off[lo] + kTileN * (local / n_mt);
        it.ntok = min(kTileN, a.seg_off[lo] + a.seg_cnt[lo] - it.row0);
        return it;
    };
    // This CTA's j-th item (item = blockIdx.x + j gridDim.x): its first kItab items are decoded
    // once here, so the single-thread loops read one record instead of searching the prefix.
    for (int j = tid; j < kItab; j += kTcThreads) {
        const int item = static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x);
        if (item < total) {
            const Item it = decode_item(item);
            itab[j] = ItemRec{it.row0, static_cast<int16_t>(it.slot), static_cast<uint8_t>(it.mt),
                              static_cast<uint8_t>(it.ntok - 1)};
        }
    }
    __syncthreads();
    auto item_at = [&](int j, int item) -> Item {
        if (j >= kItab) return decode_item(item);
        const ItemRec rec = itab[j];
        Item it;
        it.slot = rec.slot;
        it.mt = rec.mt;
        it.row0 = rec.row0;
        it.ntok = rec.ntok_m1 + 1;
        return it;
    };
    // bank row of tile row r (gate/up: gate and up rows interleaved)
    auto weight_row = [&](int mt, int r) -> int64_t {
        if (gateup) return ((r & 1) ? a.I : 0) + 64 * mt + (r >> 1);
        return static_cast<int64_t>(128) * mt + r;
    };

    if (warp >= kProdWarp0 && warp < R::epi0) {
        // ------------------------------------------------------------ producers
        // Thread pt owns tile row pt (TMEM lane pt), and this warp K part kh of
        // each stage (all of it, or one half).  The packed rows of a use arrive
        // in raw stage use % kRaw by TMA (the A loader warp); each thread reads
        // its row's part into registers, unpacks it into its tensor-memory lane
        // and only then releases the stage.
        constexpr int kPieces = 4 / R::parts;  // 16-byte pieces (32 codes) of a packed row per warp
        const int pw = warp & 3;  // this warp's tensor-memory lane quarter = its 32 tile rows
        const int kh = (warp - kProdWarp0) >> 2;
        const int pt = 32 * pw + lane;
        // Row of the raw stage holding tile row pt: its place in the stage's two 64-row boxes (gate/up:
        // the tile's gate rows, then its up rows; down: rows 0-63, then 64-127).
        const int arow = gateup ? ((pt & 1) ? 64 : 0) + (pt >> 1) : pt;
        const int rsw = (arow >> 1) & 3;  // 64-byte swizzle: 16-byte chunk q of box row r at q ^ ((r >> 1) & 3)
        bool ok = true;
        int use = 0;
        for (int item = blockIdx.x, j = 0; item < total && ok; item += gridDim.x, ++j) {
            // Scaled (down) modes: A carries each code times its group's scale over the row's
            // largest scale (|fraction| <= 1, so the fp16 product keeps 11 significant bits).
            // Other modes: A is the bare code.
            const float* srow = nullptr;
            float inv = 0.f;
            const bool two = a.slot_bits && a.slot_bits[item_at(j, item).slot] == 2;
            if (scaled) {
                const Item it = item_at(j, item);
                srow = a.ws + (static_cast<int64_t>(it.slot) * rows_per_slot + weight_row(it.mt, pt)) * ngrp;
                const float m = row_scale_max(srow, ngrp);
                inv = m > 0.f ? 1.0f / m : 0.f;
            }
            for (int ks = 0; ks < ksteps; ++ks, ++use) {
                const float sg = scaled ? __ldg(srow + ks / spg) : 0.f;  // (loaded ahead of the waits)
                // the stage's tiles have landed
                if (!__all_sync(0xffffffffu, wait_bar(raw_full + use % kRaw, (use / kRaw) & 1, ctl))) {
                    ok = false;
                    break;
                }
                uint4 rw[kPieces];
                if (two) {  // a 2-bit tile: 32-byte rows, 32-byte swizzle (chunk q at q ^ ((r >> 2) & 1))
                    const uint4* rp = reinterpret_cast<const uint4*>(raw + (use % kRaw) * kRawStage + arow * 32);
#pragma unroll
                    for (int q = 0; q < kPieces / 2; ++q) rw[q] = rp[(kh * (kPieces / 2) + q) ^ ((arow >> 2) & 1)];
                } else {
                    const uint4* rp = reinterpret_cast<const uint4*>(raw + (use % kRaw) * kRawStage + arow * 64);
#pragma unroll
                    for (int q = 0; q < kPieces; ++q) rw[q] = rp[(kh * kPieces + q) ^ rsw];
                }
                const int s = use % kAStages;
                // The A stage is free once the MMAs of use - kAStages have completed (warp-uniform
                // outcome: the tensor-memory stores below are warp-aligned).
                if (use >= kAStages) {
                    const int v = use - kAStages;
                    if (!__all_sync(0xffffffffu, wait_bar(empty + v % kBStages, (v / kBStages) & 1, ctl))) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();  // the stage's previous MMAs (which read its A columns) are complete
                // unpacked row part -> this thread's tensor-memory lane, 32 columns of fp16 pairs
                // per 64 codes (column c of the stage holds K positions 2c, 2c + 1)
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * pw) << 16) + kACol0 + kACols * s + 32 * kh * (kPieces / 2);
#pragma unroll
                for (int h2 = 0; h2 < kPieces / 2; ++h2) {
                    uint32_t av[32];
                    if (!two) {
                        const uint32_t words[8] = {rw[2 * h2].x, rw[2 * h2].y, rw[2 * h2].z, rw[2 * h2].w,
                                                   rw[2 * h2 + 1].x, rw[2 * h2 + 1].y, rw[2 * h2 + 1].z, rw[2 * h2 + 1].w};
#pragma unroll
                        for (int wi = 0; wi < 8; ++wi) unpack_int4_f16(words[wi], av + 4 * wi);
                    } else {  // 64 2-bit codes of piece h2
                        const uint32_t words[4] = {rw[h2].x, rw[h2].y, rw[h2].z, rw[h2].w};
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) unpack_int2_f16(words[wi], av + 8 * wi);
                    }
                    if (scaled) {
                        const __half2 f2 = __float2half2_rn(sg * inv);
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&av[e]), f2);
                            av[e] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                    }
                    tmem_st32(ta + 32 * h2, av);
                }
                tmem_st_wait();
                // The raw stage goes back to the loader only now that the unpack above has consumed the
                // loaded words (an arrival right after the loads let the next tile's TMA write overtake
                // loads still in flight: the async proxy is not ordered behind them).
                mbar_arrive(raw_empty + use % kRaw);
                // Thread 0 holds its arrival back until the use's B tiles have landed, so the MMA
                // thread waits on one barrier per use.
                if (!__all_sync(0xffffffffu, pt != 0 || kh != 0 || wait_bar(b_full + use % kBStages, (use / kBStages) & 1, ctl))) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(a_full + s);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue (lane 0)
        // Use u: wait for its B stage, a drained accumulator (at a group's
        // start) and its A stage; issue its 8 MMAs; release both stages to
        // the copies (and the accumulator to the epilogue at a group's end).
        // Nothing else runs on this thread: its loop has to stay well inside
        // the MMA time of a use.
        if (lane == 0) {
            bool ok = true;
            int use = 0, grp = 0;
            const int span = scaled ? ksteps : spg;  // uses summed in one accumulator
            const uint64_t bdesc0 = sdesc(smem_u32(bstages));
            for (int item = blockIdx.x, j = 0; item < total && ok; item += gridDim.x, ++j) {
                const uint32_t idesc = idesc_f16((item_at(j, item).ntok + 15) & ~15);
                for (int ks = 0; ks < ksteps; ++ks, ++use) {
                    const int sa = use % kAStages, sb = use % kBStages, sub = ks % span, b = grp % kAcc;
                    if (!wait_bar(a_full + sa, (use / kAStages) & 1, ctl) ||
                        (sub == 0 && !wait_bar(acce + b, ((grp / kAcc) & 1) ^ 1, ctl))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptor address field = byte address / 16: stage and K offsets add to it
                    const uint64_t bd = bdesc0 + static_cast<uint64_t>((sb * kBStage) >> 4);
                    const uint32_t ta = tmem + kACol0 + kACols * sa, td = tmem + b * kTileN;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // K = 16 per MMA: 8 A columns, 32 bytes of a B row
                        mma_f16_ta(td, ta + 8 * kk, bd + static_cast<uint64_t>(((kk >> 2) * kBAtom + 32 * (kk & 3)) >> 4),
                                   idesc, (sub > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(empty + sb);
                    if (sub == span - 1) {
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
    } else if (warp == kAWarp) {
        // ------------------------------------------------------------ A tiles (lane 0)
        // The packed rows of use u go into raw stage u % kRaw once the producers
        // have read use u - kRaw from it: two 2-D TMA tiles of 64 rows x 64 bytes
        // (128 codes), 64-byte swizzle (gate/up: the 64 gate rows, then the 64 up
        // rows of the weight tile; down: rows 0-63 and 64-127); a 2-bit slot's
        // tiles are 64 rows x 32 bytes, 32-byte swizzle.  A thread of its own: a
        // thread's copies to one barrier measured as waiting for its copies to
        // the barrier before.
        if (lane == 0) {
            int use = 0;
            bool ok = true;
            for (int item = blockIdx.x, j = 0; item < total && ok; item += gridDim.x, ++j) {
                const Item it = item_at(j, item);
                // a 2-bit slot: 32 bytes of a row per use, through its own map
                const bool two = a.slot_bits && a.slot_bits[it.slot] == 2;
                const CUtensorMap* map = two ? &amap2 : &amap;
                const int rb = two ? 32 : 64;
                // the slot's first row in the map's rows: uniform, or compact (its offset over its row
                // length; the offsets are multiples of it)
                const int ybase = COMPACT ? static_cast<int>((__ldg(a.w_off + it.slot) & ~int64_t(15)) / (two ? K / 4 : K / 2))
                                          : static_cast<int>(it.slot * rows_per_slot);
                const int y0 = ybase + (gateup ? 64 : 128) * it.mt;
                const int y1 = gateup ? static_cast<int>(ybase + a.I + 64 * it.mt) : y0 + 64;
                for (int ks = 0; ks < ksteps; ++ks, ++use) {
                    const int r = use % kRaw;
                    if (use >= kRaw && !wait_bar(raw_empty + r, ((use / kRaw) & 1) ^ 1, ctl)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = raw + r * kRawStage;
                    mbar_expect_tx(raw_full + r, 128 * rb);
                    tma_tile2d(dst, map, rb * ks, y0, raw_full + r);
                    tma_tile2d(dst + 64 * rb, map, rb * ks, y1, raw_full + r);
                }
            }
            // every tile issued above lands before the CTA leaves
            for (int u = max(0, use - kRaw); u < use; ++u) {
                const uint64_t t1 = global_ns();
                while (!mbar_try_wait(raw_full + u % kRaw, (u / kRaw) & 1) && global_ns() - t1 < kWaitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == kBWarp) {
        // ------------------------------------------------------------ B tiles (lane 0)
        // The token rows of use u go into stage u % kBStages once the MMAs of
        // use u - kBStages have released it: two 2-D TMA tiles of 64 K values.
        if (lane == 0) {
            int use = 0;
            bool ok = true;
            for (int item = blockIdx.x, j = 0; item < total && ok; item += gridDim.x, ++j) {
                const int row0 = item_at(j, item).row0;
                for (int ks = 0; ks < ksteps; ++ks, ++use) {
                    const int s = use % kBStages;
                    if (!wait_bar(empty + s, ((use / kBStages) & 1) ^ 1, ctl)) {
                        ok = false;
                        break;
                    }
                    uint8_t* Bs = bstages + s * kBStage;
                    mbar_expect_tx(b_full + s, kBStage);
                    tma_tile2d(Bs, &bmap, 128 * ks, row0, b_full + s);
                    tma_tile2d(Bs + kBAtom, &bmap, 128 * ks + 64, row0, b_full + s);
                }
            }
            // every tile issued above lands before the CTA leaves (after an abort the MMA thread
            // no longer waits for them): the last kBStages uses cover every stage still in flight
            for (int u = max(0, use - kBStages); u < use; ++u) {
                const uint64_t t1 = global_ns();
                while (!mbar_try_wait(b_full + u % kBStages, (u / kBStages) & 1) && global_ns() - t1 < kWaitNs) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // warp w: TMEM lanes 32 (w % 4) .. +31 (tile rows), columns kColsW ((w - epi0) / 4) .. +kColsW - 1
        const int quarter = warp & 3, c_base = kColsW * ((warp - R::epi0) >> 2);
        const int r = 32 * quarter + lane;  // tile row
        const int et = tid - 32 * R::epi0;  // epilogue thread index
        int grp = 0;
        // the pair rows and column scales of an item are loaded one item ahead (their global
        // loads then overlap the previous item's groups) into the other half of colp / colf
        auto load_cols = [&](int jj, int item, int& p_out, float& f_out) {
            p_out = -1;
            if (item < total && et < kTileN) {
                const Item nx = item_at(jj, item);
                if (et < nx.ntok) {
                    const int p = nx.row0 + et;
                    p_out = p;
                    f_out = MODE == TcMode::kGateUp ? __ldg(a.b_scale + __ldg(a.row_token + p))
                                                    : (partials ? 0.f : __ldg(a.b_scale + p));
                }
            }
        };
        {
            int p0 = -1;
            float f0 = 0.f;
            load_cols(0, blockIdx.x, p0, f0);
            if (p0 >= 0) {
                colp_buf[et] = p0;
                colf_buf[et] = f0;
            }
        }
        int j = 0;  // this CTA's item count
        bool ok = true;
        for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
            // Every epilogue thread learns whether any gave up; and every thread is done with
            // item j - 1, so its column tables (the other half) may be refilled during item j.
            if (named_bar_or(1, kEpiThreads, !ok)) break;
            const Item it = item_at(j, item);
            const int* colp = colp_buf + (j & 1) * kTileN;
            const float* colf = colf_buf + (j & 1) * kTileN;
            int np = -1;
            float nf = 0.f;
            load_cols(j + 1, item + gridDim.x, np, nf);  // the next item's (consumed after this one)
            const int nloc = min(kColsW, it.ntok - c_base);  // this warp's live columns (may be <= 0)
            const int64_t wrow = weight_row(it.mt, r);
            const float* srow = a.ws + (static_cast<int64_t>(it.slot) * rows_per_slot + wrow) * ngrp;
            if (partials) {
                // one accumulator per K group: its exact int32 partial, by pair row
                for (int gq = 0; gq < ngrp; ++gq, ++grp) {
                    const int b = grp % kAcc;
                    if (!__all_sync(0xffffffffu, wait_bar(accf + b, (grp / kAcc) & 1, ctl))) {  // loads are warp-aligned
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tb = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + b * kTileN + c_base;
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < kColsW / 16; ++i) {
                        if (16 * i >= nloc) break;
                        tmem_ld16(tb + 16 * i, v);
                        tmem_ld_wait();
                        int32_t* dst = a.partials + wrow * ngrp + gq;
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            if (16 * i + c < nloc)
                                dst[static_cast<int64_t>(colp[c_base + 16 * i + c]) * rows_per_slot * ngrp] =
                                    __float2int_rn(__uint_as_float(v[c]));
                    }
                    tc_fence_before();
                    mbar_arrive(acce + b);
                }
            } else if (!scaled) {
                // Gate/up: each K group's exact partial is folded into fp32 registers with its
                // scale (scales two groups ahead: issued before the waits)
                float acc[kColsW];
#pragma unroll
                for (int c = 0; c < kColsW; ++c) acc[c] = 0.f;
                float sc1 = __ldg(srow), sc2 = ngrp < 2 ? 0.f : __ldg(srow + 1);
                for (int gq = 0; gq < ngrp; ++gq, ++grp) {
                    const int b = grp % kAcc;
                    const float sc = sc1;
                    sc1 = sc2;
                    if (gq + 2 < ngrp) sc2 = __ldg(srow + gq + 2);
                    if (!__all_sync(0xffffffffu, wait_bar(accf + b, (grp / kAcc) & 1, ctl))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tb = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + b * kTileN + c_base;
#pragma unroll
                    for (int i = 0; i < kColsW / 16; ++i) {  // 16 columns at a time (64 running sums + 16 loaded)
                        if (16 * i < nloc) {
                            uint32_t v[16];
                            tmem_ld8(tb + 16 * i, v);
                            tmem_ld8(tb + 16 * i + 8, v + 8);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 16; ++c) acc[16 * i + c] = fmaf(__uint_as_float(v[c]), sc, acc[16 * i + c]);
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(acce + b);
                }
                if (!ok) continue;
                // h straight from the registers: lanes 2j (gate) and 2j+1 (up) hold index
                // i = 64 mt + j for every column; for a column pair (c0, c0 + 1) the even lane
                // finishes c0 and the odd lane c0 + 1, so each store instruction writes two
                // 64-byte row pieces.  The tile's pair rows are consecutive (row0 + column).
                const bool odd = r & 1;
                float* hp = a.h + static_cast<int64_t>(it.row0 + c_base + (odd ? 1 : 0)) * a.I + 64 * it.mt + (r >> 1);
#pragma unroll
                for (int q = 0; q < kColsW / 16; ++q) {
                    if (16 * q < nloc) {  // warp-uniform: the shuffles below are warp-wide
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int c0 = 16 * q + 2 * e;
                            const float xs = colf[c_base + c0 + (odd ? 1 : 0)];
                            const float other = __shfl_xor_sync(0xffffffffu, odd ? acc[c0] : acc[c0 + 1], 1);
                            const float gate = odd ? other : acc[c0], up = odd ? acc[c0 + 1] : other;
                            if (c0 + (odd ? 1 : 0) < nloc) *hp = silu_fast(gate * xs) * (up * xs);
                            hp += 2 * a.I;
                        }
                    }
                }
            } else {
                // Down: one accumulator holds the item's whole K range in units of the row's
                // largest scale.  It is read 16 columns at a time and handed back to the MMAs as
                // soon as its last columns are in registers; Y goes straight from the registers:
                // for one token column the lanes of a warp hold consecutive output features, so
                // each store instruction writes a 64-byte row piece, and the tile's pair rows are
                // consecutive (row0 + column).
                const float smax = row_scale_max(srow, ngrp);
                const int b = grp % kAcc;
                ++grp;
                if (!__all_sync(0xffffffffu, wait_bar(accf + b, ((grp - 1) / kAcc) & 1, ctl))) {
                    ok = false;
                    continue;
                }
                tc_fence_after();
                const uint32_t tb = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + b * kTileN + c_base;
                const int nq = nloc <= 0 ? 0 : min(kColsW / 16, (nloc + 15) / 16);  // chunks with live columns
                if (nq == 0) {
                    tc_fence_before();
                    mbar_arrive(acce + b);
                }
                const int64_t o0 = static_cast<int64_t>(it.row0 + c_base) * a.H + 128 * static_cast<int64_t>(it.mt) + r;
#pragma unroll
                for (int q = 0; q < kColsW / 16; ++q) {
                    if (q < nq) {  // warp-uniform: the loads below are warp-wide
                        uint32_t v[16];
                        tmem_ld16(tb + 16 * q, v);
                        tmem_ld_wait();
                        if (q == nq - 1) {
                            tc_fence_before();
                            mbar_arrive(acce + b);
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = 16 * q + e;
                            const float yv = __uint_as_float(v[e]) * smax * colf[c_base + c];
                            const int64_t o = o0 + static_cast<int64_t>(c) * a.H;
                            if (c < nloc) {
                                if (MODE == TcMode::kDown) a.yb[o] = __float2bfloat16_rn(yv);
                                else a.y[o] = yv;
                            }
                        }
                    }
                }
            }
            if (np >= 0) {
                colp_buf[((j + 1) & 1) * kTileN + et] = np;
                colf_buf[((j + 1) & 1) * kTileN + et] = nf;
            }
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
// 8 values); out row r is token row_token[r], zeros for a token outside
// [0, T).  Idx: the type of the element index 8 i (32-bit when rows * H fits,
// which keeps the row/column split a 32-bit division).
template <typename Idx>
__global__ void prep_x16_kernel(const int8_t* __restrict__ x, int64_t T, int64_t H, const int32_t* __restrict__ row_token,
                                int64_t n8, __half* __restrict__ out) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const Idx i8 = static_cast<Idx>(8 * i), Hx = static_cast<Idx>(H);
        const int64_t r = static_cast<int64_t>(i8 / Hx), c = static_cast<int64_t>(i8 % Hx);
        const int64_t t = row_token[r];
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
// the codes (RNE(h / s) decided in fp32: by the reciprocal, and by the IEEE
// division within 1e-4 of a half-step).  With hq_in (no h) the int8 codes are
// converted as given.
// NV > 0: I = 256 NV, each lane keeps its 8 NV values of the row in registers (one read of h);
// NV = 0: any I, the row read twice.
template <int NV>
__global__ void prep_h16_kernel(const float* __restrict__ h, uint32_t* __restrict__ amax,
                                const int8_t* __restrict__ hq_in, int64_t P, int64_t I, __half* __restrict__ out,
                                float* __restrict__ s_h) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    auto store8 = [&](int64_t row, int64_t k, const int (&code)[8]) {
        __half2 o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = __halves2half2(__int2half_rn(code[e]), __int2half_rn(code[e + 4]));
        *reinterpret_cast<uint4*>(out + row * I + k) = *reinterpret_cast<const uint4*>(o);
    };
    auto finish_max = [&](int64_t row, float m, float& s, float& rs) {
        m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
        s = requant_scale(__float_as_uint(m));
        rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
        if (lane == 0) {
            if (amax) amax[row] = __float_as_uint(m);
            if (s_h) s_h[row] = s;
        }
    };
    auto absmax8 = [](const float4& f0, const float4& f1) {
        return fmaxf(fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f0.z), fabsf(f0.w))),
                     fmaxf(fmaxf(fabsf(f1.x), fabsf(f1.y)), fmaxf(fabsf(f1.z), fabsf(f1.w))));
    };
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < P; row += nw) {
        const float* hr = h ? h + row * I : nullptr;
        if (!hr) {  // the codes as given
            for (int64_t k = 8 * lane; k < I; k += 256) {
                const uint2 v = *reinterpret_cast<const uint2*>(hq_in + row * I + k);
                const int8_t* b = reinterpret_cast<const int8_t*>(&v);
                int code[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) code[e] = b[e];
                store8(row, k, code);
            }
            continue;
        }
        float s, rs, m = 0.f;
        if (NV > 0) {
            float4 f[NV > 0 ? NV : 1][2];
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                f[v][0] = __ldcs(reinterpret_cast<const float4*>(hr + 8 * lane + 256 * v));
                f[v][1] = __ldcs(reinterpret_cast<const float4*>(hr + 8 * lane + 256 * v + 4));
                m = fmaxf(m, absmax8(f[v][0], f[v][1]));
            }
            finish_max(row, m, s, rs);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const float g[8] = {f[v][0].x, f[v][0].y, f[v][0].z, f[v][0].w, f[v][1].x, f[v][1].y, f[v][1].z, f[v][1].w};
                int code[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) code[e] = requant_code_fast(g[e], s, rs);
                store8(row, 8 * lane + 256 * v, code);
            }
        } else {
            for (int64_t k = 8 * lane; k < I; k += 256)
                m = fmaxf(m, absmax8(*reinterpret_cast<const float4*>(hr + k), *reinterpret_cast<const float4*>(hr + k + 4)));
            finish_max(row, m, s, rs);
            for (int64_t k = 8 * lane; k < I; k += 256) {
                const float4 f0 = *reinterpret_cast<const float4*>(hr + k);
                const float4 f1 = *reinterpret_cast<const float4*>(hr + k + 4);
                const float g[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                int code[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) code[e] = requant_code_fast(g[e], s, rs);
                store8(row, k, code);
            }
        }
    }
}

using Encode = PFN_cuTensorMapEncodeTiled_v12000;

cudaError_t get_encode(Encode* out) {
    static Encode encode = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
        encode = reinterpret_cast<Encode>(fn);
    }
    *out = encode;
    return cudaSuccess;
}

// Tensor map of the B rows of one launch: fp16 [b_rows][K], boxes of 64 values by 192 rows,
// 128-byte swizzle; rows past the end read zeros.
cudaError_t make_bmap(const TcArgs& a, CUtensorMap* bmap) {
    Encode encode = nullptr;
    if (cudaError_t e = get_encode(&encode); e != cudaSuccess) return e;
    const cuuint32_t elem[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.b_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTileN)};
    const CUresult r = encode(bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a.b), dims, strides, box, elem,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed weight rows of every slot as one 2-D uint8 tensor (K/2 bytes per row): 64-byte x 64-row
// boxes, 64-byte swizzle (16-byte chunk q of box row r at q ^ ((r >> 1) & 3)).
// two: the map of the 2-bit slots (32 code bytes of a row per 128 codes: 32-byte x 64-row boxes,
// 32-byte swizzle), whose rows are K/2 bytes apart in the uniform layout and K/4 in the compact one.
// Compact storage has no single row count: the map spans as many rows as a map may, and the slots'
// offsets (inside the caller's buffer) keep every box in it.
cudaError_t make_amap(const TcArgs& a, bool two, CUtensorMap* amap) {
    Encode encode = nullptr;
    if (cudaError_t e = get_encode(&encode); e != cudaSuccess) return e;
    const cuuint32_t elem[2] = {1, 1};
    const cuuint64_t pitch = static_cast<cuuint64_t>(a.w_off && two ? a.K / 4 : a.K / 2);
    const cuuint64_t rows = a.w_off ? std::min<cuuint64_t>((cuuint64_t(1) << 31) - 1, ((cuuint64_t(1) << 40) - 1) / pitch)
                                    : static_cast<cuuint64_t>(a.n_slots) * static_cast<cuuint64_t>(a.rows_per_slot);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(two ? a.K / 4 : a.K / 2), rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {two ? 32u : 64u, 64};
    const CUresult r = encode(amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.w), dims, strides, box, elem,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, two ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Fixed-order combine from bf16 Y: one thread per (token, 8 output columns).
__global__ void __launch_bounds__(256) combine_bf16_kernel(const __nv_bfloat16* __restrict__ y,
                                                           const float* __restrict__ wts, const int32_t* __restrict__ inv,
                                                           int64_t T, int64_t H, int64_t k, int64_t S,
                                                           float* __restrict__ out) {
    const int64_t H8 = H / 8, Tk = T * k, total = T * H8;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / H8, n = (idx % H8) * 8;
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        auto add_row = [&](int64_t row, float wj) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + row * H + n));
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[2 * e] = fmaf(wj, __uint_as_float(u[e] << 16), o[2 * e]);
                o[2 * e + 1] = fmaf(wj, __uint_as_float(u[e] & 0xFFFF0000u), o[2 * e + 1]);
            }
        };
        for (int64_t j = 0; j < k; ++j) add_row(inv[t * k + j], wts[t * k + j]);
        for (int64_t sh = 0; sh < S; ++sh) add_row(Tk + sh * T + t, 1.0f);
        float4* dst = reinterpret_cast<float4*>(out + t * H + n);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

template <TcMode MODE, bool COMPACT = false>
cudaError_t launch_mode_tc(const TcArgs& a, int n_mt, cudaStream_t st) {
    auto kern = tc_gemm_kernel<MODE, COMPACT>;
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
    alignas(64) CUtensorMap amap{}, amap2{};
    if (cudaError_t e = make_amap(a, false, &amap); e != cudaSuccess) return e;
    if (a.slot_bits)
        if (cudaError_t e = make_amap(a, true, &amap2); e != cudaSuccess) return e;
    kern<<<num_sms(), kTcThreads, kSmemTc, st>>>(a, n_mt, bmap, amap, amap2);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int64_t H, int64_t I, int64_t g) {
    // (weight tiles per slot: I / 64 for gate/up, H / 128 for down, each indexed in 8 bits)
    return g % 128 == 0 && H % 128 == 0 && I % 128 == 0 && H >= 128 && I >= 128 && I / 64 <= 256 && H / 128 <= 256;
}

cudaError_t launch_tc_gemm(TcMode mode, const TcArgs& a, cudaStream_t st) {
    if (a.n_slots < 1 || a.n_slots > kTcMaxSlots) return cudaErrorInvalidValue;
    // the weight rows are addressed as one 2-D tensor of int32 row coordinates
    if (static_cast<int64_t>(a.n_slots) * a.rows_per_slot >= (int64_t(1) << 31) || a.b_rows < 1 ||
        a.b_rows >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const bool gateup = mode == TcMode::kGateUp || mode == TcMode::kGateUpPartials;
    const int n_mt = static_cast<int>(gateup ? a.I / 64 : a.H / 128);
    if (n_mt < 1 || n_mt > 256) return cudaErrorInvalidValue;  // weight tile index kept in 8 bits
    switch (mode) {
        // (compact storage: a variant of its own)
        case TcMode::kGateUp:
            return a.w_off ? launch_mode_tc<TcMode::kGateUp, true>(a, n_mt, st)
                           : launch_mode_tc<TcMode::kGateUp>(a, n_mt, st);
        case TcMode::kDown:
            return a.w_off ? launch_mode_tc<TcMode::kDown, true>(a, n_mt, st)
                           : launch_mode_tc<TcMode::kDown>(a, n_mt, st);
        case TcMode::kDownY:
            return a.w_off ? launch_mode_tc<TcMode::kDownY, true>(a, n_mt, st)
                           : launch_mode_tc<TcMode::kDownY>(a, n_mt, st);
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

cudaError_t launch_combine_bf16(const __nv_bfloat16* y, const float* wts, const int32_t* inv, int64_t T, int64_t H,
                                int64_t k, int64_t S, float* out, cudaStream_t st) {
    const int64_t total = T * H / 8;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms()) * 16);
    combine_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(y, wts, inv, T, H, k, S, out);
    return cudaGetLastError();
}

cudaError_t launch_prep_h16(const float* h, uint32_t* amax, const int8_t* hq_in, int64_t P, int64_t I, __half* h16,
                            float* s_h, cudaStream_t st) {
    const int64_t blocks = std::min<int64_t>((P + 7) / 8, static_cast<int64_t>(num_sms()) * 8);
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(blocks, 1));
    switch (I) {  // rows of up to 1024 values stay in registers
        case 256: prep_h16_kernel<1><<<grid, 256, 0, st>>>(h, amax, hq_in, P, I, h16, s_h); break;
        case 512: prep_h16_kernel<2><<<grid, 256, 0, st>>>(h, amax, hq_in, P, I, h16, s_h); break;
        case 768: prep_h16_kernel<3><<<grid, 256, 0, st>>>(h, amax, hq_in, P, I, h16, s_h); break;
        case 1024: prep_h16_kernel<4><<<grid, 256, 0, st>>>(h, amax, hq_in, P, I, h16, s_h); break;
        default: prep_h16_kernel<0><<<grid, 256, 0, st>>>(h, amax, hq_in, P, I, h16, s_h); break;
    }
    return cudaGetLastError();
}

}  // namespace moe
