// C ABI of the routed-expert W4A8 MoE layer: argument checks, workspace
// carving, engine choice and the launch sequences.  Host code only; every
// step of the layer runs in the kernels of route.cu, gemm_mma.cu, decode.cu
// and prefill_tc.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include "decode.h"
#include "kernels.h"
#include "moe_w4a8.h"
#include "prefill.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace {

using moe::WsLayout;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const moe_dims_t* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->H < 1 || d->I < 1 || d->E < 1 || d->n_shared < 0 || d->top_k < 1 || d->top_k > d->E ||
        d->group < 32 || d->group % 32 != 0 || d->H % d->group != 0 || d->I % d->group != 0)
        return MOE_ERR_INVALID_ARG;
    if (d->E > moe::kMaxExperts || d->n_shared > moe::kMaxShared || d->top_k > moe::kMaxTopK ||
        d->group > moe::kMaxGroup || d->I % 64 != 0 || d->H % 128 != 0 || d->H > moe::kMaxDim ||
        d->I > moe::kMaxDim)
        return MOE_ERR_UNSUPPORTED;
    const int64_t P = d->T * (d->top_k + d->n_shared);
    if (d->T > (int64_t(1) << 24) || P >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_ptrs(std::initializer_list<const void*> ptrs) {
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

WsLayout layout_of(const moe_dims_t* d) { return moe::ws_layout(d->T, d->H, d->I, d->E, d->n_shared, d->top_k); }

// Workspace of the partials entry points: the grouping of n_pairs pairs
// over E + S slots, plus the fp16 activation rows of the pairs.
WsLayout partials_layout(const moe_dims_t* d, int64_t n_pairs) {
    return moe::ws_layout(std::max<int64_t>(n_pairs, 1), d->H, d->I, d->E + d->n_shared, 0, 1);
}


int check_ws(const WsLayout& L, const void* ws, size_t bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

thread_local char g_last_error[256] = "";

int cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return MOE_OK;
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                          \
    do {                                       \
        int _rc = (expr);                      \
        if (_rc != MOE_OK) return _rc;         \
    } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status((expr), #expr))

struct Views {
    moe::Header* hdr;
    uint32_t* flags;
    int8_t* hq;
    float* sh;
    int32_t *ids, *seg_cnt, *seg_off, *perm, *inv, *row_token, *chunk_counts, *tile_slot, *tile_row0;
    float *wts, *h, *y;
    uint32_t* amax;
    __half *x16, *h16;
};

Views views(void* ws, const WsLayout& L) {
    Views v;
    v.hdr = moe::ws_at<moe::Header>(ws, L.hdr);
    v.flags = moe::ws_at<uint32_t>(ws, L.flags);
    v.hq = moe::ws_at<int8_t>(ws, L.hq);
    v.sh = moe::ws_at<float>(ws, L.sh);
    v.ids = moe::ws_at<int32_t>(ws, L.ids);
    v.wts = moe::ws_at<float>(ws, L.wts);
    v.seg_cnt = moe::ws_at<int32_t>(ws, L.seg_cnt);
    v.seg_off = moe::ws_at<int32_t>(ws, L.seg_off);
    v.perm = moe::ws_at<int32_t>(ws, L.perm);
    v.inv = moe::ws_at<int32_t>(ws, L.inv);
    v.row_token = moe::ws_at<int32_t>(ws, L.row_token);
    v.chunk_counts = moe::ws_at<int32_t>(ws, L.chunk_counts);
    v.tile_slot = moe::ws_at<int32_t>(ws, L.tile_slot);
    v.tile_row0 = moe::ws_at<int32_t>(ws, L.tile_row0);
    v.amax = moe::ws_at<uint32_t>(ws, L.amax);
    v.h = moe::ws_at<float>(ws, L.h);
    v.y = moe::ws_at<float>(ws, L.y);
    v.x16 = moe::ws_at<__half>(ws, L.x16);
    v.h16 = moe::ws_at<__half>(ws, L.h16);
    return v;
}

moe::SortArgs sort_args(const Views& v, const int32_t* ids, int64_t T, int64_t k, int64_t E, int64_t S, int64_t P) {
    moe::SortArgs a{};
    a.ids = ids;
    a.T = T;
    a.k = k;
    a.E = E;
    a.S = S;
    a.tok_map = nullptr;
    a.chunk_counts = v.chunk_counts;
    a.seg_cnt = v.seg_cnt;
    a.seg_off = v.seg_off;
    a.perm = v.perm;
    a.inv = v.inv;
    a.row_token = v.row_token;
    a.tile_slot = v.tile_slot;
    a.tile_row0 = v.tile_row0;
    a.hdr = v.hdr;
    a.amax = v.amax;
    a.P = P;
    a.counts_out = nullptr;
    a.offsets_out = nullptr;
    return a;
}

// The fused decode engine's plan for a forward call, if the sizes fit it.
bool decode_forward_plan(const moe_dims_t* d, moe::DecodePlan* pl, bool mixed = false) {
    return moe::decode_plan(d->T, d->H, d->I, d->E, d->n_shared, d->top_k, d->group, 0, moe::DecodeMode::kForward,
                            moe::decode_grid(), moe::decode_max_smem(), pl, mixed);
}

int run_decode(const int8_t* x_q, const float* x_scale, const float* logits, const uint8_t* w13, const float* s13,
               const uint8_t* w2, const float* s2, const moe_dims_t* d, float* out, const Views& v,
               const moe::DecodePlan& pl, float* y_debug, cudaStream_t st, const uint16_t* x_bf16 = nullptr,
               const uint8_t* slot_bits = nullptr, bool route_debug = false, const int32_t* ids_in = nullptr,
               const float* wts_in = nullptr, const int64_t* w13_off = nullptr, const int64_t* w2_off = nullptr) {
    moe::DecodeArgs a{};
    a.x_q = x_q;
    a.x_scale = x_scale;
    a.x_bf16 = x_bf16;
    a.slot_bits = slot_bits;
    a.w13_off = w13_off;
    a.w2_off = w2_off;
    a.logits = logits;
    a.ids_in = ids_in;
    a.wts_in = wts_in;
    a.w13 = w13;
    a.s13 = s13;
    a.w2 = w2;
    a.s2 = s2;
    a.T = static_cast<int>(d->T);
    a.H = static_cast<int>(d->H);
    a.I = static_cast<int>(d->I);
    a.E = static_cast<int>(d->E);
    a.S = static_cast<int>(d->n_shared);
    a.k = static_cast<int>(d->top_k);
    a.g = static_cast<int>(d->group);
    a.out = out;
    a.hdr = v.hdr;
    a.row_max = v.flags;
    a.hq_g = v.hq;
    a.sh_g = v.sh;
    a.h = v.h;
    a.amax = v.amax;
    a.y = y_debug;
    if (route_debug) {  // leave the routing in the workspace arrays the other engines fill
        a.ids_out = v.ids;
        a.wts_out = v.wts;
        a.perm_out = v.perm;
        a.inv_out = v.inv;
    }
    MOE_CUDA(moe::launch_decode(moe::DecodeMode::kForward, a, pl, moe::decode_grid(), st));
    return MOE_OK;
}

int combine_out(const moe_dims_t* d, float* out, const WsLayout& L, const Views& v, float* y_debug, cudaStream_t st);

bool tc_fits(const moe_dims_t* d) {
    return moe::tc_supported(d->H, d->I, d->group) && d->E + d->n_shared <= moe::kTcMaxSlots;
}

moe::TcArgs tc_args(const uint8_t* w, const float* ws, int64_t rows_per_slot, int64_t K, const moe_dims_t* d,
                    const __half* b, int64_t b_rows, const float* b_scale, const Views& v, int n_slots) {
    moe::TcArgs a{};
    a.w = w;
    a.ws = ws;
    a.rows_per_slot = rows_per_slot;
    a.K = K;
    a.g = static_cast<int>(d->group);
    a.I = d->I;
    a.H = d->H;
    a.b = b;
    a.b_rows = b_rows;
    a.b_scale = b_scale;
    a.seg_off = v.seg_off;
    a.seg_cnt = v.seg_cnt;
    a.row_token = v.row_token;
    a.n_slots = n_slots;
    a.hdr = v.hdr;
    return a;
}

// gemm1 + act, requant, gemm2 and the combine on the tcgen05 engine (routing and grouping done).
// y_debug: also the per-pair outputs Y in fp32.
// slot_bits: each slot's code width (2 or 4) of a mixed bank, or null.
int run_tc_gemms(const int8_t* x_q, const float* x_scale, const uint8_t* w13, const float* s13, const uint8_t* w2,
                 const float* s2, const moe_dims_t* d, float* out, const WsLayout& L, const Views& v, float* y_debug,
                 cudaStream_t st, const uint8_t* slot_bits = nullptr, const int64_t* w13_off = nullptr,
                 const int64_t* w2_off = nullptr) {
    const int n_slots = static_cast<int>(d->E + d->n_shared);
    // the activations gathered by pair row (fp16, the engine's K order): contiguous B tiles for gate/up
    MOE_CUDA(moe::launch_prep_x16(x_q, d->T, d->H, v.row_token, L.P, v.x16, st));
    moe::TcArgs g1 = tc_args(w13, s13, 2 * d->I, d->H, d, v.x16, L.P, x_scale, v, n_slots);
    g1.slot_bits = slot_bits;
    g1.w_off = w13_off;
    g1.h = v.h;
    MOE_CUDA(moe::launch_tc_gemm(moe::TcMode::kGateUp, g1, st));
    MOE_CUDA(moe::launch_prep_h16(v.h, v.amax, nullptr, L.P, d->I, v.h16, v.sh, st));
    moe::TcArgs g2 = tc_args(w2, s2, d->H, d->I, d, v.h16, L.P, v.sh, v, n_slots);
    g2.slot_bits = slot_bits;
    g2.w_off = w2_off;
    __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(v.y);  // the Y area holds bf16 Y here
    g2.yb = yb;
    MOE_CUDA(moe::launch_tc_gemm(moe::TcMode::kDown, g2, st));
    MOE_CUDA(moe::launch_combine_bf16(yb, v.wts, v.inv, d->T, d->H, d->top_k, d->n_shared, out, st));
    if (y_debug) {
        g2.y = y_debug;
        MOE_CUDA(moe::launch_tc_gemm(moe::TcMode::kDownY, g2, st));
    }
    return MOE_OK;
}

// route + permute + gemm1 + gemm2 + combine on the workspace views.
int run_layer(const int8_t* x_q, const float* x_scale, const float* logits, const uint8_t* w13, const float* s13,
              const uint8_t* w2, const float* s2, const moe_dims_t* d, float* out, const WsLayout& L, const Views& v,
              cudaStream_t st, int engine = MOE_ENGINE_AUTO, float* y_debug = nullptr, bool route_debug = false,
              const int32_t* ids_in = nullptr, const float* wts_in = nullptr) {
    if (engine == MOE_ENGINE_AUTO || engine == MOE_ENGINE_DECODE) {
        moe::DecodePlan pl;
        if (decode_forward_plan(d, &pl))
            return run_decode(x_q, x_scale, logits, w13, s13, w2, s2, d, out, v, pl, y_debug, st, nullptr, nullptr,
                              route_debug, ids_in, wts_in);
        if (engine == MOE_ENGINE_DECODE) return MOE_ERR_UNSUPPORTED;
    }
    const bool tc = engine == MOE_ENGINE_TCGEN05 || (engine == MOE_ENGINE_AUTO && tc_fits(d));
    if (tc && !tc_fits(d)) return MOE_ERR_UNSUPPORTED;
    if (ids_in) MOE_CUDA(moe::launch_route_supplied(ids_in, wts_in, d->T, d->E, d->top_k, v.ids, v.wts, st));
    else MOE_CUDA(moe::launch_route_topk(logits, d->T, d->E, d->top_k, v.ids, v.wts, st));
    MOE_CUDA(moe::launch_sort(sort_args(v, v.ids, d->T, d->top_k, d->E, d->n_shared, L.P), st));
    if (tc) return run_tc_gemms(x_q, x_scale, w13, s13, w2, s2, d, out, L, v, y_debug, st);

    moe::Gemm1Args g1{};
    g1.x_q = x_q;
    g1.x_scale = x_scale;
    g1.w13 = w13;
    g1.s13 = s13;
    g1.T = d->T;
    g1.H = d->H;
    g1.I = d->I;
    g1.g = d->group;
    g1.seg_off = v.seg_off;
    g1.seg_cnt = v.seg_cnt;
    g1.row_token = v.row_token;
    g1.tile_slot = v.tile_slot;
    g1.tile_row0 = v.tile_row0;
    g1.hdr = v.hdr;
    g1.h = v.h;
    g1.amax = v.amax;
    MOE_CUDA(moe::launch_gemm1(moe::Gemm1Mode::kHidden, g1, static_cast<int>(L.max_tiles), st));

    moe::Gemm2Args g2{};
    g2.h = v.h;
    g2.amax = v.amax;
    g2.w2 = w2;
    g2.s2 = s2;
    g2.H = d->H;
    g2.I = d->I;
    g2.g = d->group;
    g2.seg_off = v.seg_off;
    g2.seg_cnt = v.seg_cnt;
    g2.tile_slot = v.tile_slot;
    g2.tile_row0 = v.tile_row0;
    g2.hdr = v.hdr;
    g2.y = v.y;
    MOE_CUDA(moe::launch_gemm2(moe::Gemm2Mode::kOutput, g2, static_cast<int>(L.max_tiles), st));
    return combine_out(d, out, L, v, y_debug, st);
}

int combine_out(const moe_dims_t* d, float* out, const WsLayout& L, const Views& v, float* y_debug, cudaStream_t st) {
    moe::CombineArgs c{};
    c.y = v.y;
    c.wts = v.wts;
    c.inv = v.inv;
    c.T = d->T;
    c.H = d->H;
    c.k = d->top_k;
    c.S = d->n_shared;
    c.out = out;
    MOE_CUDA(moe::launch_combine(c, st));
    if (y_debug) MOE_CUDA(cudaMemcpyAsync(y_debug, v.y, sizeof(float) * L.P * d->H, cudaMemcpyDeviceToDevice, st));
    return MOE_OK;
}

}  // namespace

MOE_API int moe_w4a8_version(void) { return MOE_W4A8_ABI_VERSION; }

MOE_API const char* moe_w4a8_last_error(void) { return g_last_error; }

MOE_API const char* moe_w4a8_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or inconsistent sizes)";
        case MOE_ERR_UNSUPPORTED: return "sizes beyond the kernels' limits";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA launch error";
        case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
        default: return "unknown status";
    }
}

MOE_API size_t moe_w4a8_workspace_size(const moe_dims_t* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return layout_of(d).total;
}

MOE_API size_t moe_w4a8_partials_workspace_size(const moe_dims_t* d, int64_t n_pairs) {
    if (check_dims(d) != MOE_OK || n_pairs < 0 || n_pairs >= (int64_t(1) << 24)) return 0;
    return partials_layout(d, n_pairs).total;
}

MOE_API int moe_w4a8_engine_for(const moe_dims_t* d) {
    if (check_dims(d) != MOE_OK) return -1;
    moe::DecodePlan pl;
    if (decode_forward_plan(d, &pl)) return MOE_ENGINE_DECODE;
    return tc_fits(d) ? MOE_ENGINE_TCGEN05 : MOE_ENGINE_GROUPED;
}

MOE_API int moe_w4a8_forward(const int8_t* x_q, const float* x_scale, const float* router_logits,
                             const uint8_t* w13_packed, const float* w13_scale, const uint8_t* w2_packed,
                             const float* w2_scale, const moe_dims_t* d, float* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    return run_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L,
                     views(workspace, L), static_cast<cudaStream_t>(stream));
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Staging area after the layer's workspace: x_q, x_scale, logits, out.
struct HostStage {
    size_t x_q, x_scale, logits, out, total;
};
HostStage host_stage_of(const moe_dims_t* d, const WsLayout& L) {
    HostStage h;
    h.x_q = align256(L.total);
    h.x_scale = h.x_q + align256(static_cast<size_t>(d->T) * d->H);
    h.logits = h.x_scale + align256(sizeof(float) * d->T);
    h.out = h.logits + align256(sizeof(float) * d->T * d->E);
    h.total = h.out + align256(sizeof(float) * d->T * d->H);
    return h;
}

// Where a caller's host-side buffer lives: 1 = page-locked host memory
// mapped into the device address space (*dev = its device address),
// 2 = device or managed memory (*dev = p), 0 = pageable host memory,
// -1 = the runtime could not classify it.
int host_buffer_kind(const void* p, void** dev) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (a.type == cudaMemoryTypeHost) {
        if (!a.devicePointer) return 0;
        *dev = a.devicePointer;
        return 1;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dev = const_cast<void*>(p);
        return 2;
    }
    return 0;
}

}  // namespace

MOE_API size_t moe_w4a8_forward_host_workspace_size(const moe_dims_t* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return host_stage_of(d, layout_of(d)).total;
}

MOE_API int moe_w4a8_forward_host(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                  const uint8_t* w13_packed, const float* w13_scale, const uint8_t* w2_packed,
                                  const float* w2_scale, const moe_dims_t* d, float* out, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    const WsLayout L = layout_of(d);
    const HostStage hs = host_stage_of(d, L);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < hs.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    // classify every buffer before anything is enqueued
    const void* src[3] = {x_q, x_scale, router_logits};
    const size_t bytes[3] = {static_cast<size_t>(d->T) * d->H, sizeof(float) * d->T, sizeof(float) * d->T * d->E};
    const size_t off[3] = {hs.x_q, hs.x_scale, hs.logits};
    int kind[3];
    void* dev[3] = {nullptr, nullptr, nullptr};
    for (int b = 0; b < 3; ++b)
        if ((kind[b] = host_buffer_kind(src[b], &dev[b])) < 0) return MOE_ERR_INVALID_ARG;
    void* out_dev = nullptr;
    const int out_kind = host_buffer_kind(out, &out_dev);
    if (out_kind < 0) return MOE_ERR_INVALID_ARG;

    const void* in_dev[3];
    moe::StageArgs sa{};
    for (int b = 0; b < 3; ++b) {
        if (kind[b] == 2) {  // device-accessible memory: used in place
            in_dev[b] = dev[b];
        } else if (kind[b] == 1) {  // mapped page-locked memory: one kernel reads it over the host link
            sa.src[b] = dev[b];
            sa.dst[b] = ws + off[b];
            sa.bytes[b] = static_cast<int64_t>(bytes[b]);
            in_dev[b] = ws + off[b];
        } else {  // pageable: the driver stages the copy
            MOE_CUDA(cudaMemcpyAsync(ws + off[b], src[b], bytes[b], cudaMemcpyHostToDevice, st));
            in_dev[b] = ws + off[b];
        }
    }
    MOE_CUDA(moe::launch_stage_copy(sa, st));
    float* layer_out = out_kind == 0 ? reinterpret_cast<float*>(ws + hs.out) : static_cast<float*>(out_dev);
    MOE_TRY(run_layer(static_cast<const int8_t*>(in_dev[0]), static_cast<const float*>(in_dev[1]),
                      static_cast<const float*>(in_dev[2]), w13_packed, w13_scale, w2_packed, w2_scale, d, layer_out, L,
                      views(workspace, L), st));
    if (out_kind == 0)
        MOE_CUDA(cudaMemcpyAsync(out, layer_out, sizeof(float) * d->T * d->H, cudaMemcpyDeviceToHost, st));
    return MOE_OK;
}

namespace {
// Staging area of moe_w4a8_forward_bf16 after the layer's workspace: x_q [T][H], x_scale [T].
size_t bf16_stage_xq(const WsLayout& L) { return align256(L.total); }
size_t bf16_stage_xs(const moe_dims_t* d, const WsLayout& L) {
    return bf16_stage_xq(L) + align256(static_cast<size_t>(d->T) * d->H);
}
size_t bf16_stage_total(const moe_dims_t* d, const WsLayout& L) {
    return bf16_stage_xs(d, L) + align256(sizeof(float) * d->T);
}
}  // namespace

MOE_API size_t moe_w4a8_forward_bf16_workspace_size(const moe_dims_t* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return bf16_stage_total(d, layout_of(d));
}

MOE_API int moe_w4a8_forward_bf16(const uint16_t* x_bf16, const float* router_logits, const uint8_t* w13_packed,
                                  const float* w13_scale, const uint8_t* w2_packed, const float* w2_scale,
                                  const moe_dims_t* d, float* out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_bf16, router_logits, out}));
    const WsLayout L = layout_of(d);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < bf16_stage_total(d, L)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Views v = views(workspace, L);
    moe::DecodePlan pl;
    if (decode_forward_plan(d, &pl))  // the fused kernel quantises the activations itself
        return run_decode(nullptr, nullptr, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, v, pl,
                          nullptr, st, x_bf16);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int8_t* x_q = reinterpret_cast<int8_t*>(ws + bf16_stage_xq(L));
    float* x_scale = reinterpret_cast<float*>(ws + bf16_stage_xs(d, L));
    MOE_CUDA(moe::launch_quantize_bf16(x_bf16, d->T, d->H, x_q, x_scale, st));
    return run_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L, v, st);
}

MOE_API int moe_w4a8_forward_w2w4(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                  const uint8_t* w13_packed, const float* w13_scale, const uint8_t* w2_packed,
                                  const float* w2_scale, const uint8_t* slot_bits, const moe_dims_t* d, float* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (!slot_bits) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    const Views v = views(workspace, L);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    moe::DecodePlan pl;
    if (decode_forward_plan(d, &pl, true))  // small batches: the decode engine
        return run_decode(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, v, pl,
                          nullptr, st, nullptr, slot_bits);
    if (!tc_fits(d)) return MOE_ERR_UNSUPPORTED;  // large batches: the tcgen05 engine's sizes
    MOE_CUDA(moe::launch_route_topk(router_logits, d->T, d->E, d->top_k, v.ids, v.wts, st));
    MOE_CUDA(moe::launch_sort(sort_args(v, v.ids, d->T, d->top_k, d->E, d->n_shared, L.P), st));
    return run_tc_gemms(x_q, x_scale, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L, v, nullptr, st,
                        slot_bits);
}

MOE_API int moe_w4a8_mixed_bank_layout(const uint8_t* slot_bits, const moe_dims_t* d, int64_t* w13_off,
                                       int64_t* w2_off, int64_t* w13_bytes, int64_t* w2_bytes) {
    MOE_TRY(check_dims(d));
    if (!slot_bits || !w13_off || !w2_off || !w13_bytes || !w2_bytes) return MOE_ERR_INVALID_ARG;
    // (the dims checks keep H and I multiples of 64: every 2-bit row, and so every offset, is a multiple
    // of 16 bytes)
    int64_t o13 = 0, o2 = 0;
    for (int64_t e = 0; e < d->E + d->n_shared; ++e) {
        const bool two = slot_bits[e] == 2;
        w13_off[e] = o13;
        w2_off[e] = o2;
        o13 += 2 * d->I * (two ? d->H / 4 : d->H / 2);
        o2 += d->H * (two ? d->I / 4 : d->I / 2);
    }
    *w13_bytes = o13;
    *w2_bytes = o2;
    return MOE_OK;
}

MOE_API int moe_w4a8_forward_w2w4_compact(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                          const uint8_t* w13_packed, const int64_t* w13_off, const float* w13_scale,
                                          const uint8_t* w2_packed, const int64_t* w2_off, const float* w2_scale,
                                          const uint8_t* slot_bits, const moe_dims_t* d, float* out,
                                          void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (!slot_bits || !w13_off || !w2_off) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    const Views v = views(workspace, L);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    moe::DecodePlan pl;
    if (decode_forward_plan(d, &pl, true))  // small batches: the decode engine
        return run_decode(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, v, pl,
                          nullptr, st, nullptr, slot_bits, false, nullptr, nullptr, w13_off, w2_off);
    if (!tc_fits(d)) return MOE_ERR_UNSUPPORTED;  // large batches: the tcgen05 engine's sizes
    MOE_CUDA(moe::launch_route_topk(router_logits, d->T, d->E, d->top_k, v.ids, v.wts, st));
    MOE_CUDA(moe::launch_sort(sort_args(v, v.ids, d->T, d->top_k, d->E, d->n_shared, L.P), st));
    return run_tc_gemms(x_q, x_scale, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L, v, nullptr, st,
                        slot_bits, w13_off, w2_off);
}

MOE_API int moe_w4a8_forward_debug(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                   const uint8_t* w13_packed, const float* w13_scale, const uint8_t* w2_packed,
                                   const float* w2_scale, const moe_dims_t* d, float* out, int8_t* h_q, float* s_h,
                                   float* y, int engine, void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    for (const void* p : {static_cast<const void*>(h_q), static_cast<const void*>(s_h), static_cast<const void*>(y)})
        if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    const Views v = views(workspace, L);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (engine < MOE_ENGINE_AUTO || engine > MOE_ENGINE_TCGEN05) return MOE_ERR_INVALID_ARG;
    MOE_TRY(run_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L, v, st,
                      engine, y, true));
    if (h_q || s_h) MOE_CUDA(moe::launch_requant_copy(v.h, v.amax, L.P, d->I, h_q, s_h, st));
    return MOE_OK;
}

MOE_API int moe_w4a8_forward_routed(const int8_t* x_q, const float* x_scale, const int32_t* topk_ids,
                                   const float* topk_w, const uint8_t* w13_packed, const float* w13_scale,
                                   const uint8_t* w2_packed, const float* w2_scale, const moe_dims_t* d, float* out,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, topk_ids, topk_w, out}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    return run_layer(x_q, x_scale, nullptr, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L,
                     views(workspace, L), static_cast<cudaStream_t>(stream), MOE_ENGINE_AUTO, nullptr, false, topk_ids,
                     topk_w);
}

MOE_API int moe_w4a8_debug_routing(const moe_dims_t* d, const void* workspace, size_t workspace_bytes,
                                   int32_t* topk_ids, float* topk_w, int32_t* perm, int32_t* inv, void* stream) {
    MOE_TRY(check_dims(d));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({topk_ids, topk_w, perm, inv}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, const_cast<void*>(workspace), workspace_bytes));
    const Views v = views(const_cast<void*>(workspace), L);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n = static_cast<size_t>(d->T * d->top_k);
    MOE_CUDA(cudaMemcpyAsync(topk_ids, v.ids, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    MOE_CUDA(cudaMemcpyAsync(topk_w, v.wts, n * sizeof(float), cudaMemcpyDeviceToDevice, st));
    MOE_CUDA(cudaMemcpyAsync(perm, v.perm, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    MOE_CUDA(cudaMemcpyAsync(inv, v.inv, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    return MOE_OK;
}

MOE_API int moe_w4a8_route(const float* router_logits, const moe_dims_t* d, int32_t* topk_ids, float* topk_w,
                           int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace,
                           size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({router_logits, topk_ids, topk_w, counts, offsets, perm, inv}));
    const WsLayout L = layout_of(d);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    Views v = views(workspace, L);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    MOE_CUDA(moe::launch_route_topk(router_logits, d->T, d->E, d->top_k, topk_ids, topk_w, st));
    moe::SortArgs a = sort_args(v, topk_ids, d->T, d->top_k, d->E, d->n_shared, L.P);
    a.perm = perm;
    a.inv = inv;
    a.counts_out = counts;
    a.offsets_out = offsets;
    MOE_CUDA(moe::launch_sort(a, st));
    return MOE_OK;
}

namespace {
// Grouping of an explicit pair list by bank slot (sorted ascending): the
// counting sort over E + S slots with one "expert" per pair.
int group_pairs(const moe_dims_t* d, const int32_t* pair_token, const int32_t* pair_slot, int64_t n_pairs,
                void* workspace, size_t workspace_bytes, cudaStream_t st, WsLayout* L_out, Views* v_out) {
    const WsLayout L = partials_layout(d, n_pairs);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    Views v = views(workspace, L);
    moe::SortArgs a = sort_args(v, pair_slot, n_pairs, 1, d->E + d->n_shared, 0, L.P);
    a.tok_map = pair_token;
    a.amax = nullptr;
    MOE_CUDA(moe::launch_sort(a, st));
    *L_out = L;
    *v_out = v;
    return MOE_OK;
}
}  // namespace

// The decode engine's integer core on an explicit pair list (phase 1 or phase 2 alone).
int decode_partials(moe::DecodeMode mode, const moe_dims_t* d, const int8_t* x_or_hq, const uint8_t* w,
                    const int32_t* pair_token, const int32_t* pair_slot, int64_t n_pairs, int32_t* p, void* workspace,
                    size_t workspace_bytes, cudaStream_t st) {
    const int64_t T = mode == moe::DecodeMode::kGemm1Partials ? d->T : 0;
    moe::DecodePlan pl;
    if (!moe::decode_plan(T, d->H, d->I, d->E, 0, 1, d->group, n_pairs, mode, moe::decode_grid(),
                          moe::decode_max_smem(), &pl))
        return MOE_ERR_UNSUPPORTED;
    const WsLayout L = partials_layout(d, n_pairs);
    MOE_TRY(check_ws(L, workspace, workspace_bytes));
    Views v = views(workspace, L);
    moe::DecodeArgs a{};
    a.x_q = mode == moe::DecodeMode::kGemm1Partials ? x_or_hq : nullptr;
    a.h_q_in = mode == moe::DecodeMode::kGemm2Partials ? x_or_hq : nullptr;
    a.w13 = w;
    a.w2 = w;
    a.T = static_cast<int>(T);
    a.H = static_cast<int>(d->H);
    a.I = static_cast<int>(d->I);
    a.E = static_cast<int>(d->E + d->n_shared);
    a.S = 0;
    a.k = 1;
    a.g = static_cast<int>(d->group);
    a.pair_token = pair_token;
    a.pair_slot = pair_slot;
    a.n_pairs = static_cast<int>(n_pairs);
    a.p1 = p;
    a.p2 = p;
    a.hdr = v.hdr;
    MOE_CUDA(moe::launch_decode(mode, a, pl, moe::decode_grid(), st));
    return MOE_OK;
}

MOE_API int moe_w4a8_gemm1_partials(const int8_t* x_q, const uint8_t* w13_packed, const moe_dims_t* d,
                                    const int32_t* pair_token, const int32_t* pair_slot, int64_t n_pairs, int32_t* p1,
                                    int engine, void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    if (n_pairs < 0 || n_pairs >= (int64_t(1) << 24)) return MOE_ERR_INVALID_ARG;
    if (engine < MOE_ENGINE_AUTO || engine > MOE_ENGINE_TCGEN05) return MOE_ERR_INVALID_ARG;
    if (n_pairs == 0) return MOE_OK;
    if (d->E + d->n_shared > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_ptrs({x_q, w13_packed, pair_token, pair_slot, p1}));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (engine == MOE_ENGINE_DECODE)
        return decode_partials(moe::DecodeMode::kGemm1Partials, d, x_q, w13_packed, pair_token, pair_slot, n_pairs,
                               p1, workspace, workspace_bytes, st);
    WsLayout L;
    Views v;
    MOE_TRY(group_pairs(d, pair_token, pair_slot, n_pairs, workspace, workspace_bytes, st, &L, &v));
    const int n_slots = static_cast<int>(d->E + d->n_shared);
    if (engine == MOE_ENGINE_TCGEN05) {
        if (!tc_fits(d)) return MOE_ERR_UNSUPPORTED;
        MOE_CUDA(moe::launch_prep_x16(x_q, d->T, d->H, v.row_token, L.P, v.x16, st));
        moe::TcArgs a = tc_args(w13_packed, nullptr, 2 * d->I, d->H, d, v.x16, L.P, nullptr, v, n_slots);
        a.partials = p1;
        MOE_CUDA(moe::launch_tc_gemm(moe::TcMode::kGateUpPartials, a, st));
        return MOE_OK;
    }
    moe::Gemm1Args g1{};
    g1.x_q = x_q;
    g1.w13 = w13_packed;
    g1.T = d->T;
    g1.H = d->H;
    g1.I = d->I;
    g1.g = d->group;
    g1.seg_off = v.seg_off;
    g1.seg_cnt = v.seg_cnt;
    g1.row_token = v.row_token;
    g1.tile_slot = v.tile_slot;
    g1.tile_row0 = v.tile_row0;
    g1.hdr = v.hdr;
    g1.p1 = p1;
    MOE_CUDA(moe::launch_gemm1(moe::Gemm1Mode::kPartials, g1, static_cast<int>(L.max_tiles), st));
    return MOE_OK;
}

MOE_API int moe_w4a8_gemm2_partials(const int8_t* h_q, const uint8_t* w2_packed, const moe_dims_t* d,
                                    const int32_t* pair_slot, int64_t n_pairs, int32_t* p2, int engine,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    MOE_TRY(check_dims(d));
    if (n_pairs < 0 || n_pairs >= (int64_t(1) << 24)) return MOE_ERR_INVALID_ARG;
    if (engine < MOE_ENGINE_AUTO || engine > MOE_ENGINE_TCGEN05) return MOE_ERR_INVALID_ARG;
    if (n_pairs == 0) return MOE_OK;
    if (d->E + d->n_shared > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_ptrs({h_q, w2_packed, pair_slot, p2}));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (engine == MOE_ENGINE_DECODE)
        return decode_partials(moe::DecodeMode::kGemm2Partials, d, h_q, w2_packed, pair_slot, pair_slot, n_pairs, p2,
                               workspace, workspace_bytes, st);
    WsLayout L;
    Views v;
    MOE_TRY(group_pairs(d, pair_slot, pair_slot, n_pairs, workspace, workspace_bytes, st, &L, &v));
    const int n_slots = static_cast<int>(d->E + d->n_shared);
    if (engine == MOE_ENGINE_TCGEN05) {
        if (!tc_fits(d)) return MOE_ERR_UNSUPPORTED;
        MOE_CUDA(moe::launch_prep_h16(nullptr, nullptr, h_q, n_pairs, d->I, v.h16, nullptr, st));
        moe::TcArgs a = tc_args(w2_packed, nullptr, d->H, d->I, d, v.h16, n_pairs, nullptr, v, n_slots);
        a.partials = p2;
        MOE_CUDA(moe::launch_tc_gemm(moe::TcMode::kDownPartials, a, st));
        return MOE_OK;
    }
    moe::Gemm2Args g2{};
    g2.h_q = h_q;
    g2.w2 = w2_packed;
    g2.H = d->H;
    g2.I = d->I;
    g2.g = d->group;
    g2.seg_off = v.seg_off;
    g2.seg_cnt = v.seg_cnt;
    g2.tile_slot = v.tile_slot;
    g2.tile_row0 = v.tile_row0;
    g2.hdr = v.hdr;
    g2.p2 = p2;
    MOE_CUDA(moe::launch_gemm2(moe::Gemm2Mode::kPartials, g2, static_cast<int>(L.max_tiles), st));
    return MOE_OK;
}

namespace {
int noalloc_scratch(void** out);
}  // namespace

MOE_API int moe_w4a8_device_status(const void* workspace, size_t workspace_bytes, void* stream) {
    void* scratch = nullptr;
    if (!workspace) {  // the built-in array of moe_w4a8_forward_noalloc on the current device
        MOE_TRY(noalloc_scratch(&scratch));
        workspace = scratch;
        workspace_bytes = MOE_W4A8_NOALLOC_SCRATCH_BYTES;
    }
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < sizeof(moe::Header))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t status = 0;
    MOE_CUDA(cudaMemcpyAsync(&status, workspace, sizeof(status), cudaMemcpyDeviceToHost, st));
    MOE_CUDA(cudaStreamSynchronize(st));
    return (status & moe::kDevTimeout) ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

MOE_API int moe_w4a8_selftest_barrier_timeout(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < sizeof(moe::Header))
        return MOE_ERR_INVALID_ARG;
    MOE_CUDA(moe::launch_barrier_timeout_probe(static_cast<moe::Header*>(workspace), static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

// ------------------------------------------------------------------ no-alloc variant
// The scratch array of moe_w4a8_forward_noalloc.  Host code must not pass
// `g_noalloc_scratch` itself to a kernel (on the host it names a stand-in,
// not device memory); its device address is looked up on every call, with
// the calling device current, so a context that was reset and re-created
// (the module reloaded, the array possibly moved) gets its new address.
namespace {
constexpr size_t kNoAllocBytes = MOE_W4A8_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of the scratch array on the current device.  The first
// lookup in a context loads the library's device code there.
int noalloc_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress");
    *out = p;
    return MOE_OK;
}
}  // namespace

MOE_API int moe_w4a8_forward_noalloc(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                     const uint8_t* w13_packed, const float* w13_scale, const uint8_t* w2_packed,
                                     const float* w2_scale, const moe_dims_t* d, float* out, void* stream) {
    MOE_TRY(check_dims(d));
    MOE_TRY(check_ptrs({w13_packed, w13_scale, w2_packed, w2_scale}));
    if (d->T == 0) return MOE_OK;
    MOE_TRY(check_ptrs({x_q, x_scale, router_logits, out}));
    const WsLayout L = layout_of(d);
    if (L.total > kNoAllocBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    MOE_TRY(noalloc_scratch(&ws));
    return run_layer(x_q, x_scale, router_logits, w13_packed, w13_scale, w2_packed, w2_scale, d, out, L,
                     views(ws, L), static_cast<cudaStream_t>(stream));
}
