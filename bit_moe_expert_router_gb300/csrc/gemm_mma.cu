// Grouped W4A8 expert projections on the int8 tensor-core path (mma.sync s8).
//
// The projections run directly on the packed int4 bank with per-group
// (blocked) reduction and the gate and up halves handled in one tile
// ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next", section 3: keep the
// weights packed; fused gate/up, blocked reduction, dedicated W4A8
// execution).  Each CTA tile is 64 pair rows of one bank slot; the K loop
// runs one quantisation group (g values of K) per stage, double-buffered
// with cp.async.  Per group the warp accumulates exact int32 partial sums
// on the tensor cores and then folds them into fp32 with the group's weight
// scale, so the int32 partials of every group are available (partials mode)
// and the dequantised result never goes through a widened copy of the bank.
//
// Nibbles are unpacked in registers: a packed word moved into the high half
// of each byte is an int8 lane holding 16 * code (unpack_int4x8_x16), so the
// MMA yields 16 * P exactly (|16 P| <= 16 * g * 127 * 8 < 2^31) and P is an
// arithmetic shift away.  The unpack yields even and odd K elements in
// separate registers; the activation fragments are deinterleaved the same
// way, which only permutes the K order inside each 32-wide MMA step.
//
//   gemm1_kernel  A = gathered x_q rows, B = 64 gate rows + the matching 64
//                 up rows of w13; epilogue G = x_scale * sum_q s13 * P1,
//                 h = SiLU(G_gate) * G_up, h -> workspace and the per-row
//                 |h| maximum -> atomicMax (order-independent).
//   gemm2_kernel  A = h_q, requantised from h on the fly (fp32 decision);
//                 B = 128 rows of w2; epilogue Y = s_h * sum_q s2 * P2.
//   combine_kernel out[t] = sum_j w[t][j] Y[inv[t*k+j]] + sum_s Y[shared row].
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 128;  // 4 warps, 2 (M) x 2 (N)

__host__ __device__ constexpr int lda_bytes(int g) { return g + 32; }
__host__ __device__ constexpr int ldb_bytes(int g) { return g / 2 + 16; }
__host__ __device__ constexpr int stage_bytes(int g) {
    return kTileM * lda_bytes(g) + 128 * ldb_bytes(g) + 128 * 4;
}

struct Frag {
    int d[2][8][4];
};

// One group of K (g values) for a warp tile of 32 rows x 8 n-tiles.
// As/Bs point at the stage; brow_of(j) gives the B row of n-tile j.
template <typename BRow>
__device__ __forceinline__ void mma_group(const int8_t* As, const uint8_t* Bs, int g, int wm, BRow brow_of,
                                          int (&d)[2][8][4]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tq = lane & 3;
    const int lda = lda_bytes(g), ldb = ldb_bytes(g);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[mt][j][e] = 0;
    for (int ks = 0; ks < g / 32; ++ks) {
        uint32_t a[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int r = 32 * wm + 16 * mt + gid;
            const uint2 v0 = *reinterpret_cast<const uint2*>(As + r * lda + ks * 32 + 8 * tq);
            const uint2 v1 = *reinterpret_cast<const uint2*>(As + (r + 8) * lda + ks * 32 + 8 * tq);
            deinterleave_int8x8(v0.x, v0.y, a[mt][0], a[mt][2]);
            deinterleave_int8x8(v1.x, v1.y, a[mt][1], a[mt][3]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(Bs + (brow_of(j) + gid) * ldb + ks * 16 + 4 * tq);
            uint32_t b0, b1;
            unpack_int4x8_x16(w, b0, b1);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) mma_s8_16832(d[mt][j], a[mt], b0, b1);
        }
    }
}

struct TileInfo {
    int slot, row0, nrows;
};

__device__ __forceinline__ TileInfo tile_info(const int32_t* tile_slot, const int32_t* tile_row0, const int32_t* seg_off,
                                              const int32_t* seg_cnt, int tile) {
    TileInfo t;
    t.slot = tile_slot[tile];
    t.row0 = tile_row0[tile];
    t.nrows = min(kTileM, seg_off[t.slot] + seg_cnt[t.slot] - t.row0);
    return t;
}

// ------------------------------------------------------------------ gemm1
template <Gemm1Mode MODE>
__global__ void __launch_bounds__(kThreads) gemm1_kernel(Gemm1Args a, int n_ntiles) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int g = static_cast<int>(a.g);
    const int64_t H = a.H, I = a.I;
    const int ng = static_cast<int>(H / g);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tq = lane & 3;
    const int wm = warp >> 1, wn = warp & 1;
    const int lda = lda_bytes(g), ldb = ldb_bytes(g), sb = stage_bytes(g);
    const int a_chunks = g / 16, b_chunks = g / 32;  // 16-byte chunks per row per group
    const int64_t total = static_cast<int64_t>(a.hdr->n_tiles) * n_ntiles;

    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int tile = static_cast<int>(w / n_ntiles), nt = static_cast<int>(w % n_ntiles);
        const TileInfo ti = tile_info(a.tile_slot, a.tile_row0, a.seg_off, a.seg_cnt, tile);
        const int64_t i0 = static_cast<int64_t>(nt) * 64;
        const uint8_t* wbase = a.w13 + static_cast<int64_t>(ti.slot) * 2 * I * (H / 2);

        auto issue = [&](int q, int stage) {
            int8_t* As = reinterpret_cast<int8_t*>(smem + stage * sb);
            uint8_t* Bs = smem + stage * sb + kTileM * lda;
            float* Ss = reinterpret_cast<float*>(smem + stage * sb + kTileM * lda + 128 * ldb);
            for (int it = tid; it < kTileM * a_chunks; it += kThreads) {
                const int r = it / a_chunks, c = it % a_chunks;
                int64_t tok = r < ti.nrows ? a.row_token[ti.row0 + r] : -1;
                const bool ok = tok >= 0 && tok < a.T;
                if (!ok) tok = 0;
                cp_async16(As + r * lda + c * 16, a.x_q + tok * H + static_cast<int64_t>(q) * g + c * 16, ok ? 16 : 0);
            }
            for (int it = tid; it < 128 * b_chunks; it += kThreads) {
                const int rr = it / b_chunks, c = it % b_chunks;
                const int64_t wrow = rr < 64 ? i0 + rr : I + i0 + (rr - 64);
                cp_async16(Bs + rr * ldb + c * 16, wbase + wrow * (H / 2) + static_cast<int64_t>(q) * (g / 2) + c * 16);
            }
            if (MODE == Gemm1Mode::kHidden) {
                const int rr = tid;  // 128 threads, 128 rows
                const int64_t wrow = rr < 64 ? i0 + rr : I + i0 + (rr - 64);
                cp_async4(Ss + rr, a.s13 + (static_cast<int64_t>(ti.slot) * 2 * I + wrow) * ng + q);
            }
            cp_async_commit();
        };

        float acc[2][8][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;

        // B row of n-tile j: gate tiles 0..3, then the matching up tiles 4..7
        auto brow_of = [&](int j) { return j < 4 ? 32 * wn + 8 * j : 64 + 32 * wn + 8 * (j - 4); };

        issue(0, 0);
        for (int q = 0; q < ng; ++q) {
            if (q + 1 < ng) {
                issue(q + 1, (q + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const int stage = q & 1;
            const int8_t* As = reinterpret_cast<const int8_t*>(smem + stage * sb);
            const uint8_t* Bs = smem + stage * sb + kTileM * lda;
            const float* Ss = reinterpret_cast<const float*>(smem + stage * sb + kTileM * lda + 128 * ldb);
            int d[2][8][4];
            mma_group(As, Bs, g, wm, brow_of, d);
            if (MODE == Gemm1Mode::kHidden) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float s0 = Ss[brow_of(j) + 2 * tq], s1 = Ss[brow_of(j) + 2 * tq + 1];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        acc[mt][j][0] = fmaf(static_cast<float>(d[mt][j][0] >> 4), s0, acc[mt][j][0]);
                        acc[mt][j][1] = fmaf(static_cast<float>(d[mt][j][1] >> 4), s1, acc[mt][j][1]);
                        acc[mt][j][2] = fmaf(static_cast<float>(d[mt][j][2] >> 4), s0, acc[mt][j][2]);
                        acc[mt][j][3] = fmaf(static_cast<float>(d[mt][j][3] >> 4), s1, acc[mt][j][3]);
                    }
                }
            } else {
                const int64_t row_stride = 2 * I * ng;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int r = 32 * wm + 16 * mt + gid + 8 * half;
                        if (r >= ti.nrows) continue;
                        int32_t* dst = a.p1 + static_cast<int64_t>(ti.row0 + r) * row_stride;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int64_t wrow =
                                (j < 4 ? i0 + 32 * wn + 8 * j : I + i0 + 32 * wn + 8 * (j - 4)) + 2 * tq;
                            dst[wrow * ng + q] = d[mt][j][2 * half] >> 4;
                            dst[(wrow + 1) * ng + q] = d[mt][j][2 * half + 1] >> 4;
                        }
                    }
            }
            __syncthreads();
        }

        if (MODE == Gemm1Mode::kHidden) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = 32 * wm + 16 * mt + gid + 8 * half;
                    const bool ok = r < ti.nrows;
                    const int64_t pos = ti.row0 + r;
                    const float xs = ok ? a.x_scale[a.row_token[pos]] : 0.0f;
                    float m = 0.0f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float hv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float G = acc[mt][j][2 * half + e] * xs;
                            const float U = acc[mt][j + 4][2 * half + e] * xs;
                            hv[e] = silu_f32(G) * U;
                            m = fmaxf(m, fabsf(hv[e]));
                        }
                        if (ok) {
                            const int64_t col = i0 + 32 * wn + 8 * j + 2 * tq;
                            *reinterpret_cast<float2*>(a.h + pos * I + col) = make_float2(hv[0], hv[1]);
                        }
                    }
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    if (ok && tq == 0) atomicMax(a.amax + pos, __float_as_uint(m));
                }
        }
    }
}

// ------------------------------------------------------------------ gemm2
template <Gemm2Mode MODE>
__global__ void __launch_bounds__(kThreads) gemm2_kernel(Gemm2Args a, int n_ntiles) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float sh_s[kTileM];
    const int g = static_cast<int>(a.g);
    const int64_t H = a.H, I = a.I;
    const int ng = static_cast<int>(I / g);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tq = lane & 3;
    const int wm = warp >> 1, wn = warp & 1;
    const int lda = lda_bytes(g), ldb = ldb_bytes(g), sb = stage_bytes(g);
    const int a_chunks = g / 16, b_chunks = g / 32;
    const int64_t total = static_cast<int64_t>(a.hdr->n_tiles) * n_ntiles;

    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int tile = static_cast<int>(w / n_ntiles), nt = static_cast<int>(w % n_ntiles);
        const TileInfo ti = tile_info(a.tile_slot, a.tile_row0, a.seg_off, a.seg_cnt, tile);
        const int64_t n0 = static_cast<int64_t>(nt) * 128;
        const uint8_t* wbase = a.w2 + static_cast<int64_t>(ti.slot) * H * (I / 2);
        if (MODE == Gemm2Mode::kOutput) {
            for (int r = tid; r < kTileM; r += kThreads)
                sh_s[r] = r < ti.nrows ? requant_scale(a.amax[ti.row0 + r]) : 0.0f;
            __syncthreads();
        }

        // A: requantise h rows of group q into the stage (plain loads, fp32 decision).
        auto load_a_requant = [&](int q, int stage) {
            int8_t* As = reinterpret_cast<int8_t*>(smem + stage * sb);
            const int f4 = g / 4;  // float4 per row per group
            for (int it = tid; it < kTileM * f4; it += kThreads) {
                const int r = it / f4, c = it % f4;
                uint32_t packed = 0;
                if (r < ti.nrows) {
                    const float4 v = *reinterpret_cast<const float4*>(a.h + static_cast<int64_t>(ti.row0 + r) * I +
                                                                      static_cast<int64_t>(q) * g + 4 * c);
                    const float s = sh_s[r];
                    packed = (requant_code(v.x, s) & 0xFF) | ((requant_code(v.y, s) & 0xFF) << 8) |
                             ((requant_code(v.z, s) & 0xFF) << 16) | ((static_cast<uint32_t>(requant_code(v.w, s)) & 0xFF) << 24);
                }
                *reinterpret_cast<uint32_t*>(As + r * lda + 4 * c) = packed;
            }
        };
        auto issue = [&](int q, int stage) {
            int8_t* As = reinterpret_cast<int8_t*>(smem + stage * sb);
            uint8_t* Bs = smem + stage * sb + kTileM * lda;
            float* Ss = reinterpret_cast<float*>(smem + stage * sb + kTileM * lda + 128 * ldb);
            if (MODE == Gemm2Mode::kPartials) {
                for (int it = tid; it < kTileM * a_chunks; it += kThreads) {
                    const int r = it / a_chunks, c = it % a_chunks;
                    const bool ok = r < ti.nrows;
                    const int64_t row = ok ? ti.row0 + r : 0;
                    cp_async16(As + r * lda + c * 16, a.h_q + row * I + static_cast<int64_t>(q) * g + c * 16, ok ? 16 : 0);
                }
            }
            for (int it = tid; it < 128 * b_chunks; it += kThreads) {
                const int rr = it / b_chunks, c = it % b_chunks;
                cp_async16(Bs + rr * ldb + c * 16,
                           wbase + (n0 + rr) * (I / 2) + static_cast<int64_t>(q) * (g / 2) + c * 16);
            }
            if (MODE == Gemm2Mode::kOutput)
                cp_async4(Ss + tid, a.s2 + (static_cast<int64_t>(ti.slot) * H + n0 + tid) * ng + q);
            cp_async_commit();
        };

        float acc[2][8][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.0f;
        auto brow_of = [&](int j) { return 64 * wn + 8 * j; };

        issue(0, 0);
        if (MODE == Gemm2Mode::kOutput) load_a_requant(0, 0);
        for (int q = 0; q < ng; ++q) {
            if (q + 1 < ng) {
                issue(q + 1, (q + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const int stage = q & 1;
            const int8_t* As = reinterpret_cast<const int8_t*>(smem + stage * sb);
            const uint8_t* Bs = smem + stage * sb + kTileM * lda;
            const float* Ss = reinterpret_cast<const float*>(smem + stage * sb + kTileM * lda + 128 * ldb);
            int d[2][8][4];
            mma_group(As, Bs, g, wm, brow_of, d);
            if (MODE == Gemm2Mode::kOutput) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float s0 = Ss[brow_of(j) + 2 * tq], s1 = Ss[brow_of(j) + 2 * tq + 1];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        acc[mt][j][0] = fmaf(static_cast<float>(d[mt][j][0] >> 4), s0, acc[mt][j][0]);
                        acc[mt][j][1] = fmaf(static_cast<float>(d[mt][j][1] >> 4), s1, acc[mt][j][1]);
                        acc[mt][j][2] = fmaf(static_cast<float>(d[mt][j][2] >> 4), s0, acc[mt][j][2]);
                        acc[mt][j][3] = fmaf(static_cast<float>(d[mt][j][3] >> 4), s1, acc[mt][j][3]);
                    }
                }
                // the next group's activations go into the other stage (read two groups ago)
                if (q + 1 < ng) load_a_requant(q + 1, (q + 1) & 1);
            } else {
                const int64_t row_stride = H * ng;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int r = 32 * wm + 16 * mt + gid + 8 * half;
                        if (r >= ti.nrows) continue;
                        int32_t* dst = a.p2 + static_cast<int64_t>(ti.row0 + r) * row_stride;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int64_t n = n0 + brow_of(j) + 2 * tq;
                            dst[n * ng + q] = d[mt][j][2 * half] >> 4;
                            dst[(n + 1) * ng + q] = d[mt][j][2 * half + 1] >> 4;
                        }
                    }
            }
            __syncthreads();
        }

        if (MODE == Gemm2Mode::kOutput) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = 32 * wm + 16 * mt + gid + 8 * half;
                    if (r >= ti.nrows) continue;
                    const float s = sh_s[r];
                    float* dst = a.y + static_cast<int64_t>(ti.row0 + r) * H + n0;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float2*>(dst + brow_of(j) + 2 * tq) =
                            make_float2(acc[mt][j][2 * half] * s, acc[mt][j][2 * half + 1] * s);
                }
        }
        __syncthreads();  // sh_s is rewritten by the next tile
    }
}

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
    const int64_t H4 = a.H / 4, Tk = a.T * a.k;
    const int64_t total = a.T * H4;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / H4, n = (idx % H4) * 4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t j = 0; j < a.k; ++j) {
            const float wj = a.wts[t * a.k + j];
            const float4 y = *reinterpret_cast<const float4*>(a.y + static_cast<int64_t>(a.inv[t * a.k + j]) * a.H + n);
            o.x = fmaf(wj, y.x, o.x);
            o.y = fmaf(wj, y.y, o.y);
            o.z = fmaf(wj, y.z, o.z);
            o.w = fmaf(wj, y.w, o.w);
        }
        for (int64_t s = 0; s < a.S; ++s) {
            const float4 y = *reinterpret_cast<const float4*>(a.y + (Tk + s * a.T + t) * a.H + n);
            o.x += y.x;
            o.y += y.y;
            o.z += y.z;
            o.w += y.w;
        }
        *reinterpret_cast<float4*>(a.out + t * a.H + n) = o;
    }
}

__global__ void requant_copy_kernel(const float* h, const uint32_t* amax, int64_t P, int64_t I, int8_t* h_q, float* s_h) {
    const int64_t total = P * I;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = idx / I;
        const float s = requant_scale(amax[r]);
        if (h_q) h_q[idx] = static_cast<int8_t>(requant_code(h[idx], s));
        if (s_h && idx % I == 0) s_h[r] = s;
    }
}

// Resident CTAs per SM of a kernel at a dynamic shared memory size; the
// attribute and the occupancy query run once per (kernel, size, device).
template <typename K>
int grid_for(K kernel, int smem_bytes, int64_t max_work) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), smem_bytes, dev);
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            per_sm = it->second;
        } else {
            // one limit per kernel: the largest stage size any group width needs
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * stage_bytes(kMaxGroup));
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem_bytes);
            per_sm = std::max(per_sm, 1);
            cache[key] = per_sm;
        }
    }
    const int64_t grid = static_cast<int64_t>(num_sms()) * per_sm;
    return static_cast<int>(std::max<int64_t>(1, std::min(grid, max_work)));
}

}  // namespace

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

cudaError_t launch_gemm1(Gemm1Mode mode, const Gemm1Args& a, int max_tiles, cudaStream_t st) {
    const int n_ntiles = static_cast<int>(a.I / 64);
    const int smem = 2 * stage_bytes(static_cast<int>(a.g));
    const int64_t work = static_cast<int64_t>(max_tiles) * n_ntiles;
    if (mode == Gemm1Mode::kHidden) {
        auto k = gemm1_kernel<Gemm1Mode::kHidden>;
        k<<<grid_for(k, smem, work), kThreads, smem, st>>>(a, n_ntiles);
    } else {
        auto k = gemm1_kernel<Gemm1Mode::kPartials>;
        k<<<grid_for(k, smem, work), kThreads, smem, st>>>(a, n_ntiles);
    }
    return cudaGetLastError();
}

cudaError_t launch_gemm2(Gemm2Mode mode, const Gemm2Args& a, int max_tiles, cudaStream_t st) {
    const int n_ntiles = static_cast<int>(a.H / 128);
    const int smem = 2 * stage_bytes(static_cast<int>(a.g));
    const int64_t work = static_cast<int64_t>(max_tiles) * n_ntiles;
    if (mode == Gemm2Mode::kOutput) {
        auto k = gemm2_kernel<Gemm2Mode::kOutput>;
        k<<<grid_for(k, smem, work), kThreads, smem, st>>>(a, n_ntiles);
    } else {
        auto k = gemm2_kernel<Gemm2Mode::kPartials>;
        k<<<grid_for(k, smem, work), kThreads, smem, st>>>(a, n_ntiles);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    const int64_t total = a.T * (a.H / 4);
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
    combine_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_requant_copy(const float* h, const uint32_t* amax, int64_t P, int64_t I, int8_t* h_q, float* s_h,
                                cudaStream_t st) {
    const int64_t total = P * I;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms()) * 8);
    requant_copy_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(h, amax, P, I, h_q, s_h);
    return cudaGetLastError();
}

}  // namespace moe
