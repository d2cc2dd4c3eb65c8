// Routing and grouping of the W4A8 MoE layer.
//
// Tokens are routed to experts on the device, and the (token, expert) pairs
// are grouped per expert so the projections can run as grouped GEMMs
// ("Two 96 GB Ascend cards run Qwen3.8 Flash-Next", section 3: route tokens
// to experts on the device; routing and tile reuse).
//
//   route_topk_kernel  one warp per token: the k largest logits (ties to
//                      the lower index), softmax over the selected k.
//   count_kernel       per-chunk expert histogram (chunks of kChunk pairs).
//   scan_kernel        one block: expert offsets, per-chunk bases, segment
//                      table of all E + S bank slots and the m-tile schedule.
//   scatter_kernel     one warp per chunk: stable placement of each pair at
//                      base + its rank among equal ids (warp match + popc).
#include <float.h>
#include <math.h>

#include <algorithm>

#include "kernels.h"

namespace moe {
namespace {

// Order-preserving 32-bit key of a logit: a larger float gives a larger key, -0.0 and +0.0 the same
// key, and a NaN key 1 -- below every number (-inf is 0x007FFFFF) and above the 0 of an absent
// expert -- so NaNs rank last, among themselves by index.  key_value inverts it for numbers.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v != v) return 1u;
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kRouteWarps = 8;  // tokens per block, one warp each
constexpr int kRouteCand = 64;  // candidate keys a warp ranks directly

// Top-k of each token by (key desc, id asc), one warp per token; lane l holds the keys of experts
// l, l + 32, ...  Threshold: the k-th largest of the 32 lane maxima (k <= 32).  At least k keys reach
// it, so every pick does, and so does every key better than a pick: the picks are the k best of the
// keys >= the threshold, whose ranks among themselves are counted directly (a few more than k keys
// qualify as a rule).  When more than kRouteCand qualify, k rounds of a warp-wide arg-max instead.
// Weights: softmax over the k picked logits, relative to the largest.
template <int MAXJ>
__global__ void __launch_bounds__(32 * kRouteWarps) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                     int k, int32_t* __restrict__ ids,
                                                                     float* __restrict__ wts) {
    __shared__ uint32_t cand_k[kRouteWarps][kRouteCand];
    __shared__ int cand_i[kRouteWarps][kRouteCand];
    __shared__ uint32_t picked[kRouteWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kRouteWarps + warp;
    if (t >= T) return;
    const float* l = logits + static_cast<int64_t>(t) * E;
    uint32_t key[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
        const int e = lane + 32 * j;
        key[j] = e < E ? order_key(__ldg(l + e)) : 0u;
    }
    uint32_t lm = key[0];
#pragma unroll
    for (int j = 1; j < MAXJ; ++j) lm = max(lm, key[j]);
    int rk = 0;  // rank of this lane's maximum among the lanes' (ties by lane)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t o = __shfl_sync(0xffffffffu, lm, j);
        rk += o > lm || (o == lm && j < lane);
    }
    const uint32_t th = __shfl_sync(0xffffffffu, lm, __ffs(__ballot_sync(0xffffffffu, rk == k - 1)) - 1);
    int c = 0;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) c += key[j] >= th;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const int C = __shfl_sync(0xffffffffu, incl, 31);
    int my_e = 0;
    uint32_t my_k = 0;
    if (C <= kRouteCand) {
        int w = incl - c;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
            if (key[j] >= th) {
                cand_k[warp][w] = key[j];
                cand_i[warp][w] = lane + 32 * j;
                ++w;
            }
        __syncwarp();
        for (int i = lane; i < C; i += 32) {
            const uint32_t kk = cand_k[warp][i];
            const int ii = cand_i[warp][i];
            int r = 0;
            for (int j = 0; j < C; ++j) r += cand_k[warp][j] > kk || (cand_k[warp][j] == kk && cand_i[warp][j] < ii);
            if (r < k) {
                picked[warp][r] = kk;
                ids[static_cast<int64_t>(t) * k + r] = ii;
            }
        }
        __syncwarp();
        if (lane < k) my_k = picked[warp][lane];
    } else {
        uint32_t bk = 0;
        int bj = 0;
        auto lane_best = [&]() {
            bk = key[0];
            bj = 0;
#pragma unroll
            for (int j = 1; j < MAXJ; ++j)
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
            if (lane == r) {
                my_k = mk;
                my_e = static_cast<int>(mi);
            }
            if (mine == mi) {  // the winner drops the taken key and rescans
#pragma unroll
                for (int j = 0; j < MAXJ; ++j)
                    if (j == bj) key[j] = 0u;
                lane_best();
            }
        }
        if (lane < k) ids[static_cast<int64_t>(t) * k + lane] = my_e;
    }
    // softmax over the selected logits, relative to the largest (position 0)
    const float my_v = lane < k ? key_value(my_k) : 0.0f;
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - m) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) wts[static_cast<int64_t>(t) * k + lane] = ex / sum;
}

// Chunk c's expert histogram -> chunk_counts[e * n_chunks + c] (expert-major: one expert's counts over
// the chunks are contiguous for the scan).
__global__ void __launch_bounds__(256) count_kernel(SortArgs a, int64_t n, int64_t n_chunks) {
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t c = blockIdx.x;
    const int64_t i_end = min(n, (c + 1) * kChunk);
    for (int64_t i = c * kChunk + threadIdx.x; i < i_end; i += blockDim.x) {
        const int e = a.ids[i];
        if (static_cast<unsigned>(e) < static_cast<unsigned>(a.E)) atomicAdd(&hist[e], 1);  // out-of-range ids are dropped
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.chunk_counts[e * n_chunks + c] = hist[e];
    // side jobs spread over the grid: clear the row maxima, name the shared rows' tokens
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (a.amax)
        for (int64_t r = gid; r < a.P; r += stride) a.amax[r] = 0u;
    for (int64_t r = gid; r < a.T * a.S; r += stride) a.row_token[n + r] = static_cast<int32_t>(r % a.T);
}

// In-place exclusive scan of data[0..n) (n <= 4 * blockDim.x); returns the total.
__device__ int block_exclusive_scan(int* data, int n, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    int loc[4];
    int s = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int idx = tid * 4 + j;
        loc[j] = idx < n ? data[idx] : 0;
        s += loc[j];
    }
    int incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) warp_sums[lane] = wi - ws;  // exclusive
        if (lane == 31) warp_sums[32] = wi;        // total
    }
    __syncthreads();
    int run = warp_sums[wid] + incl - s;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int idx = tid * 4 + j;
        if (idx < n) data[idx] = run;
        run += loc[j];
    }
    int total = warp_sums[32];
    __syncthreads();
    return total;
}

// Per expert, one warp: the exclusive prefix of its chunk counts (contiguous, expert-major) in place,
// 256 chunks a step with each lane's 8 counts loaded together; the expert's total -> seg_cnt[e].
__global__ void __launch_bounds__(256) chunk_scan_kernel(SortArgs a, int64_t n_chunks) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (e >= a.E) return;
    int32_t* cc = a.chunk_counts + static_cast<int64_t>(e) * n_chunks;
    int run = 0;
    for (int64_t base = 0; base < n_chunks; base += 256) {
        int v[8], loc = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = base + 8 * lane + j;
            v[j] = c < n_chunks ? cc[c] : 0;
            loc += v[j];
        }
        int incl = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int r = run + incl - loc;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = base + 8 * lane + j;
            if (c < n_chunks) cc[c] = r;
            r += v[j];
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) a.seg_cnt[e] = run;
}

__global__ void __launch_bounds__(1024) scan_kernel(SortArgs a, int64_t n_chunks) {
    __shared__ int tot[kMaxExperts + kMaxShared + 1];
    __shared__ int tiles[kMaxExperts + kMaxShared + 1];
    __shared__ int warp_sums[33];
    const int E = static_cast<int>(a.E), slots = static_cast<int>(a.E + a.S);
    // the experts' totals from chunk_scan_kernel (no chunks: none)
    for (int e = threadIdx.x; e < E; e += blockDim.x) tot[e] = n_chunks > 0 ? a.seg_cnt[e] : 0;
    for (int s = threadIdx.x; s < a.S; s += blockDim.x) tot[E + s] = static_cast<int>(a.T);
    __syncthreads();
    for (int s = threadIdx.x; s < slots; s += blockDim.x) {
        a.seg_cnt[s] = tot[s];
        if (a.counts_out && s < E) a.counts_out[s] = tot[s];
        tiles[s] = (tot[s] + kTileM - 1) / kTileM;
    }
    __syncthreads();
    int total_rows = block_exclusive_scan(tot, slots, warp_sums);  // tot -> segment offsets
    int n_tiles = block_exclusive_scan(tiles, slots, warp_sums);   // tiles -> tile offsets
    for (int s = threadIdx.x; s <= slots; s += blockDim.x) {
        int off = s < slots ? tot[s] : total_rows;
        a.seg_off[s] = off;
        if (a.offsets_out && s <= E) a.offsets_out[s] = off;
    }
    for (int s = threadIdx.x; s < slots; s += blockDim.x) {
        int cnt = a.seg_cnt[s];
        int nt = (cnt + kTileM - 1) / kTileM;
        for (int j = 0; j < nt; ++j) {
            a.tile_slot[tiles[s] + j] = s;
            a.tile_row0[tiles[s] + j] = tot[s] + j * kTileM;
        }
    }
    if (threadIdx.x == 0) {
        a.hdr->n_tiles = static_cast<uint32_t>(n_tiles);
        a.hdr->status = kDevOk;
    }
}

__global__ void __launch_bounds__(32) scatter_kernel(SortArgs a, int64_t n, int64_t n_chunks) {
    extern __shared__ int cursor[];
    const int lane = threadIdx.x;
    const int64_t c = blockIdx.x;
    // the chunk's first row of each expert: the expert's segment offset + the earlier chunks' count
    for (int e = lane; e < a.E; e += 32) cursor[e] = a.seg_off[e] + a.chunk_counts[e * n_chunks + c];
    __syncwarp();
    const int64_t i0 = c * kChunk, i_end = min(n, i0 + kChunk);
    int id_next = i0 + lane < i_end ? a.ids[i0 + lane] : -1;  // the next batch's ids are loaded one batch ahead
    for (int64_t base = i0; base < i_end; base += 32) {
        const int64_t i = base + lane;
        const int id = id_next;
        id_next = base + 32 + lane < i_end ? a.ids[base + 32 + lane] : -1;
        const bool valid = static_cast<unsigned>(id) < static_cast<unsigned>(a.E);
        const int e = valid ? id : -1 - lane;  // absent or out-of-range lanes match nobody
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        if (valid) {
            const int pos = cursor[e] + rank;
            a.perm[pos] = static_cast<int32_t>(i);
            a.inv[i] = pos;
            a.row_token[pos] = a.tok_map ? a.tok_map[i] : static_cast<int32_t>(i / a.k);
        }
        __syncwarp();
        if (valid && rank == 0) cursor[e] += __popc(same);
        __syncwarp();
    }
}

}  // namespace

namespace {
// Routing supplied by the caller: ids clamped into [0, E) (no expert id can address memory outside the
// bank), weights as given.
__global__ void route_supplied_kernel(const int32_t* __restrict__ ids_in, const float* __restrict__ wts_in, int64_t n,
                                      int E, int32_t* __restrict__ ids, float* __restrict__ wts) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        ids[i] = min(max(ids_in[i], 0), E - 1);
        wts[i] = wts_in[i];
    }
}
}  // namespace

cudaError_t launch_route_supplied(const int32_t* ids_in, const float* wts_in, int64_t T, int64_t E, int64_t k,
                                  int32_t* ids, float* wts, cudaStream_t st) {
    const int64_t n = T * k;
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 1024));
    route_supplied_kernel<<<std::max(blocks, 1u), 256, 0, st>>>(ids_in, wts_in, n, static_cast<int>(E), ids, wts);
    return cudaGetLastError();
}

cudaError_t launch_route_topk(const float* logits, int64_t T, int64_t E, int64_t k, int32_t* ids, float* wts,
                              cudaStream_t st) {
    const int warps = kRouteWarps;
    dim3 grid(static_cast<unsigned>((T + warps - 1) / warps)), block(32 * warps);
    const int Ti = static_cast<int>(T), Ei = static_cast<int>(E), ki = static_cast<int>(k);
    if (E <= 32) route_topk_kernel<1><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    else if (E <= 64) route_topk_kernel<2><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    else if (E <= 128) route_topk_kernel<4><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    else if (E <= 256) route_topk_kernel<8><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    else if (E <= 512) route_topk_kernel<16><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    else route_topk_kernel<32><<<grid, block, 0, st>>>(logits, Ti, Ei, ki, ids, wts);
    return cudaGetLastError();
}

cudaError_t launch_sort(const SortArgs& a, cudaStream_t st) {
    const int64_t n = a.T * a.k;
    const int64_t n_chunks = (n + kChunk - 1) / kChunk;
    const size_t hist_bytes = sizeof(int) * a.E;
    if (n_chunks > 0) {
        count_kernel<<<static_cast<unsigned>(n_chunks), 256, hist_bytes, st>>>(a, n, n_chunks);
    } else if (a.amax) {
        cudaMemsetAsync(a.amax, 0, sizeof(uint32_t) * a.P, st);
    }
    if (n_chunks > 0) chunk_scan_kernel<<<static_cast<unsigned>((a.E + 7) / 8), 256, 0, st>>>(a, n_chunks);
    scan_kernel<<<1, 1024, 0, st>>>(a, n_chunks);
    if (n_chunks > 0) scatter_kernel<<<static_cast<unsigned>(n_chunks), 32, hist_bytes, st>>>(a, n, n_chunks);
    return cudaGetLastError();
}

// Grid-stride copy of the staged buffers: 16-byte words, then the 4-byte tail.
__global__ void stage_copy_kernel(StageArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
    for (int b = 0; b < kStageBufs; ++b) {
        const int64_t n16 = a.bytes[b] / 16, n4 = a.bytes[b] / 4;
        const uint4* s16 = static_cast<const uint4*>(a.src[b]);
        uint4* d16 = static_cast<uint4*>(a.dst[b]);
        for (int64_t i = i0; i < n16; i += stride) d16[i] = s16[i];
        const uint32_t* s4 = static_cast<const uint32_t*>(a.src[b]);
        uint32_t* d4 = static_cast<uint32_t*>(a.dst[b]);
        for (int64_t i = 4 * n16 + i0; i < n4; i += stride) d4[i] = s4[i];
    }
}

cudaError_t launch_stage_copy(const StageArgs& a, cudaStream_t st) {
    int64_t total = 0;
    for (int b = 0; b < kStageBufs; ++b) total += a.bytes[b];
    if (total == 0) return cudaSuccess;
    // about 32 KB per block, at most a wave of 152 blocks
    const int64_t blocks = std::min<int64_t>(std::max<int64_t>(total / 32768, 1), 152);
    stage_copy_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
    return cudaGetLastError();
}

// One warp per token: the row maximum, then the codes (8 values per step).
__global__ void quantize_bf16_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H, int8_t* __restrict__ x_q,
                                     float* __restrict__ x_scale) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + t * H);
    const int64_t n8 = H / 8;  // H is a multiple of 128
    float amax = 0.f;
    for (int64_t i = lane; i < n8; i += 32) {
        const uint4 v = xr[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[j] << 16)), fabsf(__uint_as_float(wv[j] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = __fdiv_rn(amax, 127.0f);
    if (lane == 0) x_scale[t] = sc;
    uint2* qr = reinterpret_cast<uint2*>(x_q + t * H);
    for (int64_t i = lane; i < n8; i += 32) {
        const uint4 v = xr[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t b = (j & 1) ? (wv[j >> 1] & 0xFFFF0000u) : (wv[j >> 1] << 16);
            float q = sc > 0.0f ? rintf(__fdiv_rn(__uint_as_float(b), sc)) : 0.0f;
            q = fminf(fmaxf(q, -127.0f), 127.0f);
            packed[j >> 2] |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xFFu) << (8 * (j & 3));
        }
        qr[i] = make_uint2(packed[0], packed[1]);
    }
}

cudaError_t launch_quantize_bf16(const uint16_t* x, int64_t T, int64_t H, int8_t* x_q, float* x_scale,
                                 cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int warps = 8;
    quantize_bf16_kernel<<<static_cast<unsigned>((T + warps - 1) / warps), 32 * warps, 0, st>>>(x, T, H, x_q, x_scale);
    return cudaGetLastError();
}

}  // namespace moe
