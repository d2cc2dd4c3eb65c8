/*
 * moe_w4a8.h -- C ABI of the routed-expert W4A8 MoE layer (CUDA, sm_103a).
 *
 * What it computes.  Source: "Two 96 GB Ascend cards run Qwen3.8 Flash-Next:
 * hardware notes, vLLM work, benchmarks and next steps" (ai-pulse-lab.com,
 * 2026-10-03), section 3, "Keep low-bit weights packed and do the work on
 * the NPU": tokens are routed to experts on the device and the grouped
 * expert projections run directly on the packed W4 bank -- fused gate/up,
 * blocked (per-group) reduction, W4A8 execution -- instead of expanding the
 * bank into a larger temporary; the same section's eager reference
 * dequantises the packed weights and calls a plain matmul (same result,
 * slower, far more memory).  The page prints no formulas; the numeric
 * recipe below is the layer's stated W4A8 format.
 *
 * Notation: T tokens, H hidden, I expert intermediate, E routed experts,
 * S shared experts, k = top_k, g = int4 quantisation group along K.
 *
 *   route    per token: the k largest logits (descending; equal logits go
 *            to the lower expert index), weights w[t][j] = softmax over the
 *            selected k logits (= softmax, top-k, renormalise).
 *   permute  stable counting sort of the flattened pairs i = t*k + j by
 *            expert: counts[E], offsets[E+1] (exclusive), perm[pos] = i,
 *            inv[i] = pos.
 *   gemm1    per pair p = (t, e), row n < 2I, group q:
 *            P1[p][n][q] = sum_{kk in q} x_q[t][kk] * W13[e][n][kk]  (int32)
 *            G[p][n] = x_scale[t] * sum_q s13[e][n][q] * P1[p][n][q]
 *   act      h[p][i] = SiLU(G[p][i]) * G[p][I + i],  SiLU(z) = z/(1+e^-z)
 *   requant  s_h[p] = max_i |h[p][i]| / 127 (fp32),
 *            h_q[p][i] = clamp(RNE(h[p][i] / s_h[p]), -127, 127); s_h = 0
 *            gives h_q = 0
 *   gemm2    P2[p][n][q] = sum_{kk in q} h_q[p][kk] * W2[e][n][kk]  (int32)
 *            Y[p][n] = s_h[p] * sum_q s2[e][n][q] * P2[p][n][q]
 *   combine  out[t][n] = sum_j w[t][j] * Y[(t, ids[t][j])][n]
 *                        + sum_s Y[(t, E + s)][n]   (fixed order; overwrite)
 *
 * Data layout (all row-major, contiguous, no padding):
 *   x_q      int8    [T][H]        per-token symmetric int8 activations
 *   x_scale  float   [T]           their scales
 *   logits   float   [T][E]        router logits
 *   w13      uint8   [E+S][2I][H/2] packed int4: element 2j in the low
 *                                   nibble of byte j, 2j+1 in the high
 *                                   nibble, two's complement; rows [0, I)
 *                                   are the gate projection, [I, 2I) up
 *   s13      float   [E+S][2I][H/g]
 *   w2       uint8   [E+S][H][I/2] same packing
 *   s2       float   [E+S][H][I/g]
 *   out      float   [T][H]        fully overwritten
 * Bank slots E .. E+S-1 are the always-on shared experts (weight 1).
 * "Pair rows" are ordered by sorted position: routed pair i sits at row
 * inv[i] (0 .. T*k-1), the shared pair (t, E+s) at row T*k + s*T + t.
 *
 * Ownership and streams.  Every pointer is a device pointer owned by the
 * caller, except where an argument says host.  The library allocates
 * nothing, keeps no state between calls and never synchronises: each call
 * only enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  The workspace carries all intermediates; calls that may run at
 * the same time need distinct workspaces.
 *
 * Errors.  Host-detected errors are returned before anything is enqueued:
 * MOE_ERR_INVALID_ARG for a null or misaligned pointer (16-byte alignment
 * is required for every array), non-positive sizes, top_k outside [1, E],
 * g not a multiple of 32, or H or I not a multiple of g;
 * MOE_ERR_UNSUPPORTED for sizes beyond the kernels' limits (E > 1024,
 * S > 8, top_k > 32, g > 256, I not a multiple of 64, H not a multiple of
 * 128, H or I > 65536, T > 2^24); MOE_ERR_WORKSPACE_TOO_SMALL; MOE_ERR_CUDA if a launch is
 * rejected.  Errors that occur while the kernels run surface at
 * the caller's next synchronisation, as for any CUDA work.  T = 0 is valid
 * and enqueues nothing.
 */
#ifndef MOE_W4A8_H
#define MOE_W4A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_W4A8_ABI_VERSION 4

/* Engines (the `engine` argument of the checking entry points).  AUTO picks
 * what moe_w4a8_forward picks: the fused decode engine when the batch fits
 * it (T <= 32, T*k <= 512 pairs, H = 2048 or 4096, I = 512, 1024, 1536 or 2048, g a
 * multiple of 64 with I/g a multiple of 4), else the tcgen05 engine when g
 * is a multiple of 128, else the grouped mma.sync engine.
 *   GROUPED  grouped GEMMs on the legacy int8 mma.sync path (any valid dims)
 *   DECODE   one cooperative kernel per call, dp4a on the CUDA cores
 *   TCGEN05  grouped GEMMs on the fifth-generation tensor cores (tcgen05.mma,
 *            fp16 operands holding the exact int4 / int8 values, accumulator
 *            in tensor memory; g a multiple of 128) */
#define MOE_ENGINE_AUTO (-1)
#define MOE_ENGINE_GROUPED 0
#define MOE_ENGINE_DECODE 1
#define MOE_ENGINE_TCGEN05 2

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_DEVICE_TIMEOUT = 5
} moe_status_t;

/* Layer sizes.  n_shared = S; group = g. */
typedef struct {
    int64_t T, H, I, E, n_shared, top_k, group;
} moe_dims_t;

/* ABI version of the loaded library (MOE_W4A8_ABI_VERSION of its build).
 * The Python binding refuses a library whose version differs. */
int moe_w4a8_version(void);

/* Static text for a status code (never NULL). */
const char* moe_w4a8_status_string(int status);

/* The CUDA error behind this thread's most recent MOE_ERR_CUDA (the failing
 * call and CUDA's message), or "" if there was none.  Never NULL. */
const char* moe_w4a8_last_error(void);

/* Bytes of workspace moe_w4a8_forward and moe_w4a8_route need for `d`
 * (0 if `d` is invalid).  Host call, no device work. */
size_t moe_w4a8_workspace_size(const moe_dims_t* d);

/* Bytes of workspace moe_w4a8_gemm1_partials and moe_w4a8_gemm2_partials
 * need for `d` and n_pairs pairs (0 if `d` is invalid or n_pairs is
 * outside [0, 2^24)). */
size_t moe_w4a8_partials_workspace_size(const moe_dims_t* d, int64_t n_pairs);

/* The engine moe_w4a8_forward uses for `d` on the current device
 * (MOE_ENGINE_DECODE, MOE_ENGINE_TCGEN05 or MOE_ENGINE_GROUPED), or -1 if
 * `d` is invalid.  The decode engine is one kernel launch per call (after
 * a memset of its barrier counters); the grouped mma.sync engine is seven
 * launches, the tcgen05 engine nine. */
int moe_w4a8_engine_for(const moe_dims_t* d);

/*
 * The whole layer: route, permute, gemm1 + act + requant, gemm2, combine.
 * out [T][H] is overwritten.  workspace: device memory of at least
 * moe_w4a8_workspace_size(d) bytes, 256-byte aligned, contents arbitrary
 * on entry (the call initialises what it uses).
 */
int moe_w4a8_forward(const int8_t* x_q, const float* x_scale, const float* router_logits,
                     const uint8_t* w13_packed, const float* w13_scale,
                     const uint8_t* w2_packed, const float* w2_scale,
                     const moe_dims_t* d, float* out,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Routing and grouping alone (the first two steps of moe_w4a8_forward, same
 * kernels): topk_ids int32 [T][k], topk_w float [T][k], counts int32 [E],
 * offsets int32 [E+1], perm int32 [T*k], inv int32 [T*k].
 */
int moe_w4a8_route(const float* router_logits, const moe_dims_t* d,
                   int32_t* topk_ids, float* topk_w, int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The layer with its intermediates exposed, for checking: with engine =
 * MOE_ENGINE_AUTO it runs exactly the kernels of moe_w4a8_forward (another
 * engine value forces that engine; MOE_ERR_UNSUPPORTED if the sizes do not
 * fit it) and additionally copies out h_q int8 [P][I] and s_h float [P]
 * (P = T*k + T*S pair rows, in pair-row order), and Y float [P][H] (the
 * per-pair down-projection outputs).  Any of the three may be NULL.
 */
int moe_w4a8_forward_debug(const int8_t* x_q, const float* x_scale, const float* router_logits,
                           const uint8_t* w13_packed, const float* w13_scale,
                           const uint8_t* w2_packed, const float* w2_scale,
                           const moe_dims_t* d, float* out, int8_t* h_q, float* s_h, float* y,
                           int engine, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The layer with the routing supplied by the caller -- an expert-routing
 * cache (the page's serving notes name one among the optimisations measured
 * at the API boundary, section 6): the ids and weights an earlier call
 * computed for the same tokens (moe_w4a8_route, moe_w4a8_debug_routing) or
 * any routing the caller keeps, so the call skips the top-k.  topk_ids
 * int32 [T][k] (the expert of pair t*k + j; each row should hold k distinct
 * experts -- an id outside [0, E) is clamped into it, and a repeated expert
 * is grouped and weighted like any other pair, never read out of bounds) and
 * topk_w float [T][k] (the pair weights, used as given), both 16-byte-aligned
 * device arrays; router_logits are not needed.  Everything else (engines,
 * workspace, errors) as for moe_w4a8_forward.  Given the routing
 * moe_w4a8_forward computes for these inputs, the result equals its output
 * bit for bit.
 */
int moe_w4a8_forward_routed(const int8_t* x_q, const float* x_scale, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13_packed, const float* w13_scale,
                            const uint8_t* w2_packed, const float* w2_scale,
                            const moe_dims_t* d, float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The routing used by the last moe_w4a8_forward_debug call on `workspace`
 * (any engine; the decode engine copies its own in-kernel routing there):
 * topk_ids int32 [T][k] and topk_w float [T][k] in rank order (largest
 * logit first, ties by lower expert id), perm int32 [T*k] (pair row ->
 * pair index t*k + j) and inv int32 [T*k] (pair index -> pair row), as
 * moe_w4a8_route returns them.  All four are device pointers; the copies
 * are enqueued on `stream`.  The values are unspecified if no forward_debug
 * call with the same dims has run on this workspace.
 */
int moe_w4a8_debug_routing(const moe_dims_t* d, const void* workspace, size_t workspace_bytes,
                           int32_t* topk_ids, float* topk_w, int32_t* perm, int32_t* inv, void* stream);

/*
 * Int32 partial sums of the gate/up projection for an explicit list of
 * pairs, through the main loop of the chosen engine (MOE_ENGINE_GROUPED,
 * MOE_ENGINE_DECODE or MOE_ENGINE_TCGEN05; AUTO means GROUPED): for pair r
 * (token pair_token[r], bank slot pair_slot[r], both int32 device arrays
 * of n_pairs entries), p1[r][n][q] = P1 for n < 2I, q < H/g.  pair_slot
 * must be sorted ascending; a pair_token outside [0, T) reads a zero row.
 * Workspace: moe_w4a8_partials_workspace_size(d, n_pairs) bytes.
 */
int moe_w4a8_gemm1_partials(const int8_t* x_q, const uint8_t* w13_packed, const moe_dims_t* d,
                            const int32_t* pair_token, const int32_t* pair_slot, int64_t n_pairs,
                            int32_t* p1, int engine, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Int32 partial sums of the down projection for given int8 rows: for pair
 * r with activation row h_q[r][:] (int8 [n_pairs][I]) and bank slot
 * pair_slot[r] (sorted ascending), p2[r][n][q] = P2 for n < H, q < I/g,
 * through the chosen engine's main loop (as for moe_w4a8_gemm1_partials).
 */
int moe_w4a8_gemm2_partials(const int8_t* h_q, const uint8_t* w2_packed, const moe_dims_t* d,
                            const int32_t* pair_slot, int64_t n_pairs,
                            int32_t* p2, int engine, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Device-side status of the last call that used `workspace`: synchronises
 * `stream`, then reads the status word the kernels keep at the start of the
 * workspace.  MOE_OK, or MOE_ERR_DEVICE_TIMEOUT if one of the engine's
 * bounded waits (the decode engine's grid barrier or its bulk-copy wait,
 * about one second each) ran out -- the kernels then skip the rest of the
 * work and the output is not valid.  A diagnostic call (it blocks the host);
 * not for the hot loop.  With workspace NULL (workspace_bytes ignored) it
 * reads the status word of the built-in array of moe_w4a8_forward_noalloc on
 * the current device, i.e. of the last no-alloc call there.
 */
int moe_w4a8_device_status(const void* workspace, size_t workspace_bytes, void* stream);

/*
 * Self-test of the bounded device waits: enqueues a two-CTA kernel in
 * which one CTA waits at the decode engine's grid barrier for a CTA that
 * never arrives.  The wait gives up after its limit (about a second) and
 * records the timeout in the workspace status word, so a following
 * moe_w4a8_device_status returns MOE_ERR_DEVICE_TIMEOUT; nothing faults and
 * the context stays usable.  workspace: at least 256 bytes, 256-aligned.
 */
int moe_w4a8_selftest_barrier_timeout(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of the library's built-in scratch array used by
 * moe_w4a8_forward_noalloc (16 MiB).
 */
#define MOE_W4A8_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * moe_w4a8_forward without a caller-supplied workspace.  (The pages have no
 * counterpart; this is a library convenience.)
 *
 * For callers that cannot allocate device memory when they run the layer:
 * plugin hosts and inference runtimes that own all device memory and hand
 * out only the tensors they manage, code that must not call cudaMalloc on
 * its hot path (it synchronises the device and can fail under memory
 * pressure), or embedded runtimes that allocate everything once at start-up.
 * The intermediates live in one fixed array inside the library, of
 * MOE_W4A8_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the
 * library holds until the process exits.  This call allocates nothing and
 * calls no allocating routine.
 *
 * Arguments, layouts, errors and the result are those of moe_w4a8_forward;
 * the caller still passes the inputs and `out`.  Layers whose
 * moe_w4a8_workspace_size(d) exceeds the array return
 * MOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued (for the 512-expert
 * decode layer, H=2048, I=512, top-10, one shared expert, that is T > ~128).
 *
 * Every call looks up the array's device address on the current device (so
 * a context that was reset and re-created is served at the array's new
 * address); the first lookup in a context loads the library's device code,
 * so make the first call on a device before capturing any stream into a
 * CUDA graph.  A bounded device wait that ran out inside a no-alloc call is
 * reported by moe_w4a8_device_status(NULL, 0, stream).  All calls on a device share the one array: two calls whose
 * kernels may overlap on the GPU (different streams without ordering
 * between them) race and produce wrong results; serialise them.  Nothing
 * from a previous call is reused -- each call initialises what it reads.
 */
int moe_w4a8_forward_noalloc(const int8_t* x_q, const float* x_scale, const float* router_logits,
                             const uint8_t* w13_packed, const float* w13_scale,
                             const uint8_t* w2_packed, const float* w2_scale,
                             const moe_dims_t* d, float* out, void* stream);

/*
 * Bytes of device workspace moe_w4a8_forward_host needs for `d`: the
 * moe_w4a8_forward workspace plus room for the staged inputs and output
 * (0 if `d` is invalid).  Host call, no device work.
 */
size_t moe_w4a8_forward_host_workspace_size(const moe_dims_t* d);

/*
 * moe_w4a8_forward with the activations, scales, logits and output in HOST
 * memory (the weights and the workspace stay device memory).  (The pages
 * have no counterpart; this is the step a host-side caller makes each
 * decode step, with the transfers done by the library.)
 *
 * x_q, x_scale, router_logits, out: host pointers, layouts as for
 * moe_w4a8_forward, 16-byte aligned.  Page-locked memory mapped into the
 * device address space (cudaHostAlloc / cudaMallocHost / pinned tensors;
 * with unified addressing every such allocation is mapped) is used in place: one
 * small kernel reads the inputs over the host link into the workspace, and
 * the layer writes `out` directly into host memory -- no copy engine
 * transfers.  Pageable memory is accepted too: it goes through
 * cudaMemcpyAsync (staged by the driver, which may block the calling
 * thread).  Device or managed memory is used as is.
 *
 * As with any asynchronous transfer, the inputs must stay unchanged and
 * `out` must not be read until `stream` has passed this call (synchronise
 * the stream or an event recorded after it).  workspace: device memory of
 * at least moe_w4a8_forward_host_workspace_size(d) bytes, 256-byte aligned.
 * Errors as for moe_w4a8_forward; a pointer the runtime cannot classify
 * (cudaPointerGetAttributes fails) is MOE_ERR_INVALID_ARG.
 */
int moe_w4a8_forward_host(const int8_t* x_q, const float* x_scale, const float* router_logits,
                          const uint8_t* w13_packed, const float* w13_scale,
                          const uint8_t* w2_packed, const float* w2_scale,
                          const moe_dims_t* d, float* out,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace moe_w4a8_forward_bf16 needs for `d` (the
 * moe_w4a8_forward workspace plus T*H + 4T bytes, each area 256-aligned;
 * 0 if `d` is invalid).  Host call, no device work. */
size_t moe_w4a8_forward_bf16_workspace_size(const moe_dims_t* d);

/*
 * The layer from bf16 activations: S0, the per-token quantisation, runs on
 * the device as part of the call (section 5 of the page: keep the decode
 * step's work on the device, no host round trips).  x_bf16: device array
 * [T][H] of bf16 bit patterns (16-byte aligned).  Per token t:
 * x_scale[t] = max_h |x[t][h]| / 127 and x_q[t][h] = clamp(RNE(x[t][h] /
 * x_scale[t]), -127, 127), decided in IEEE fp32 (an all-zero row gives
 * x_scale = 0 and x_q = 0) -- the per-token symmetric int8 activations that
 * moe_w4a8_forward takes -- then the layer as moe_w4a8_forward.  The decode
 * engine quantises inside its single kernel (the warps that do not route
 * do it while the others route); the other engines run one quantisation
 * kernel first.  Same codes as the recipe, so the result equals
 * moe_w4a8_forward on the quantised activations bit for bit.
 * workspace: at least moe_w4a8_forward_bf16_workspace_size(d) bytes,
 * 256-byte aligned.  Other arguments and errors as for moe_w4a8_forward.
 */
int moe_w4a8_forward_bf16(const uint16_t* x_bf16, const float* router_logits,
                          const uint8_t* w13_packed, const float* w13_scale,
                          const uint8_t* w2_packed, const float* w2_scale,
                          const moe_dims_t* d, float* out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * The layer on a mixed 2/4-bit bank (the page's mixed W2/W4 expert
 * checkpoint, section "GLM is my next, harder model", and the grouped mixed
 * W2/W4 expert path of "Known issues and work in progress"): slot_bits, a
 * device array of E+S bytes,
 * gives each bank slot's code width, 4 or 2.  A 4-bit slot is stored as in
 * moe_w4a8_forward.  A 2-bit slot keeps the same row length (K/2 bytes per
 * row of K codes, both projections) but holds its codes in the first K/4
 * bytes, four per byte: element 4j + p in bits 2p and 2p+1 of byte j, a
 * two's-complement number in [-2, 1]; the rest of the row is never read.
 * Scales are unchanged (one per row and group).  A 2-bit slot's code bytes
 * -- what a decode step streams -- are half those of a 4-bit slot.
 * Small batches run on the decode engine (T <= 32, T*k <= 512, H in
 * {2048, 4096}, I in {512, 1024, 1536, 2048}, g a multiple of 64 with I/g a multiple
 * of 4), larger ones on the tcgen05 engine (H and I multiples of 128, g a
 * multiple of 128, E+S <= 1039); other sizes return MOE_ERR_UNSUPPORTED.  A null slot_bits is
 * MOE_ERR_INVALID_ARG (it needs no particular alignment; a value other than
 * 2 is read as 4).  Other arguments, workspace (moe_w4a8_workspace_size)
 * and errors as for moe_w4a8_forward; with every slot 4-bit the result
 * equals moe_w4a8_forward's bit for bit.
 */
int moe_w4a8_forward_w2w4(const int8_t* x_q, const float* x_scale, const float* router_logits,
                          const uint8_t* w13_packed, const float* w13_scale,
                          const uint8_t* w2_packed, const float* w2_scale, const uint8_t* slot_bits,
                          const moe_dims_t* d, float* out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Compact storage of a mixed 2/4-bit bank.  moe_w4a8_forward_w2w4 keeps a
 * 2-bit slot at the int4 row length, so the bank takes the same HBM either
 * way.  The compact layout puts each slot's rows back to back at the slot's
 * own code width -- K/4 bytes per row for a 2-bit slot, K/2 for a 4-bit
 * slot (same codes, same packing within a row) -- and the slots one after
 * another in slot order, so a 2-bit expert takes half the bank bytes of a
 * 4-bit one.  Host function, no device work: from slot_bits (HOST, E+S
 * bytes, 2 or 4; any other value is read as 4) it writes each slot's byte
 * offset in the gate/up bank and in the down bank (HOST int64 arrays of E+S
 * entries) and each bank's size in bytes.  Every offset is a multiple of 16
 * (H and I are multiples of 64).  Errors: MOE_ERR_INVALID_ARG for a null
 * pointer; dims are checked as for moe_w4a8_forward (MOE_ERR_INVALID_ARG,
 * MOE_ERR_UNSUPPORTED).
 */
int moe_w4a8_mixed_bank_layout(const uint8_t* slot_bits, const moe_dims_t* d, int64_t* w13_off, int64_t* w2_off,
                               int64_t* w13_bytes, int64_t* w2_bytes);

/*
 * moe_w4a8_forward_w2w4 on a bank in compact storage: slot e's rows begin
 * at w13_packed + w13_off[e] (2I rows of H codes) and w2_packed + w2_off[e]
 * (H rows of I codes), DEVICE int64 arrays of E+S entries (for example the
 * layout above), each row K/4 bytes (2-bit slot) or K/2 bytes (4-bit slot)
 * after the one before.  Each offset must be a multiple of its slot's row
 * length (K/2 bytes, or K/4 for a 2-bit slot), as the layout above gives:
 * the tcgen05 engine addresses slot e's rows from w_off[e] / row length,
 * and the kernels clear the offsets' low four bits, so a wrong offset reads
 * wrong bytes, never a misaligned address.  Like the bank pointers
 * themselves, the offsets must lie inside the caller's buffers: they are
 * not checked.  Scales, slot_bits, engines,
 * size limits and errors as for moe_w4a8_forward_w2w4 (null offsets:
 * MOE_ERR_INVALID_ARG); the output equals moe_w4a8_forward_w2w4's on the
 * same codes bit for bit.
 */
int moe_w4a8_forward_w2w4_compact(const int8_t* x_q, const float* x_scale, const float* router_logits,
                                  const uint8_t* w13_packed, const int64_t* w13_off, const float* w13_scale,
                                  const uint8_t* w2_packed, const int64_t* w2_off, const float* w2_scale,
                                  const uint8_t* slot_bits, const moe_dims_t* d, float* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4A8_H */
