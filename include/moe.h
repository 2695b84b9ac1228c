/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts FFN hot path.
 *
 * One GPU, one stream per call, no host synchronisation on the hot path:
 *
 *   moe_route_topk        router logits -> top-k expert ids and weights
 *                         (moe_route_topk_sigmoid: sigmoid scores + routing
 *                         bias; moe_route_topk_bwd: the logits gradient)
 *   moe_permute           tokens -> expert-contiguous rows, group sizes and
 *                         offsets written on the device
 *   moe_grouped_ffn_fwd   grouped gate/up GEMM + SwiGLU, grouped down GEMM
 *   moe_unpermute_combine weighted top-k combine back to token order
 *   moe_grouped_ffn_bwd   dSwiGLU + grouped dgrad / wgrad GEMMs
 *   moe_grouped_quantize_mxfp8 / moe_grouped_ffn_fwd_mxfp8  MXFP8 path
 *   moe_dequantize_rows_mxfp8 / moe_dequantize_weights_mxfp8  operands of
 *                         the MXFP8 path's straight-through backward
 *
 * Conventions for every call:
 *   - Pointers named in a call's doc as "device" are device pointers owned by
 *     the caller; the library never frees or keeps them past the call, and
 *     allocates no device memory on these paths.
 *   - bf16 tensors are passed as moe_bf16_t (the raw 16-bit pattern).
 *   - Matrices are dense row-major with the innermost dimension contiguous
 *     and no padding between rows, unless stated otherwise.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting.  Problem sizes that
 *     depend on routing are read on the device, so every call can be
 *     captured in a CUDA graph.
 *   - Host-side argument errors return a status before anything is
 *     enqueued.  Errors found in device data (an expert id outside [-1, E),
 *     a wait that timed out) set bits in the device error word at offset 0
 *     of the workspace; read it with moe_read_device_error (the one call
 *     that synchronises).  Kernels never trap.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef uint16_t moe_bf16_t;          /* bf16 bit pattern */
typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a null pointer, a negative or inconsistent size */
    MOE_ERR_UNSUPPORTED = 2,   /* a size outside what the kernels handle (alignment, limits) */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch, encode, copy) */
    MOE_ERR_DEVICE_DATA = 4,   /* returned by moe_read_device_error when the word is non-zero */
    MOE_ERR_WORKSPACE = 5,     /* workspace null or smaller than moe_workspace_bytes */
} moe_status_t;

/* Bits of the device error word (uint32 at workspace offset 0). */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1u  /* a topk id outside [-1, E): route treated as dropped */
#define MOE_DEVERR_TIMEOUT       0x2u  /* a bounded device wait gave up; outputs are invalid */
#define MOE_DEVERR_CAPACITY      0x4u  /* routed rows exceed rows_cap; extra rows not written */
#define MOE_DEVERR_BOUNDS        0x8u  /* bounds-check builds only (-DMOE_BOUNDS_CHECK): group
                                          offsets that a GEMM read were not non-decreasing within
                                          [0, rows_cap]; the GEMM computed nothing */

/* Alignment: the kernels move 16-byte vectors.  The row tensors of moe_permute (x, x_perm),
 * moe_permute_static_scratch, moe_unpermute_combine (y_perm, out), moe_combine_bwd
 * (dY, y_perm, dy_perm), moe_unpermute_sum (dx_perm, dx), moe_grouped_quantize_mxfp8 (in,
 * data) and moe_quantize_weights_mxfp8 (data) must start on a 16-byte boundary; the
 * GEMMs' operands and outputs must too (their TMA descriptors).  A misaligned pointer gives
 * MOE_ERR_UNSUPPORTED before anything is launched. */

/* Human-readable name of a status (static storage). */
MOE_API const char *moe_status_string(moe_status_t status);

/* ABI version of this header (incremented on incompatible changes). */
MOE_API int moe_abi_version(void);

/* ------------------------------------------------------------------ */
/* Workspace                                                           */
/* ------------------------------------------------------------------ */

/* Bytes of device workspace that moe_permute, moe_grouped_ffn_fwd(_mxfp8)
 * and moe_grouped_ffn_bwd need for a problem with T tokens, E experts and
 * top-k: the error word (offset 0) plus the permutation's per-chunk expert
 * counts.  Returns 0 for invalid sizes. */
MOE_API size_t moe_workspace_bytes(int64_t T, int E, int k);

/* Zero the error word (and any state) of a workspace, on `stream`. */
MOE_API moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* Limit, in ns, of the device spin waits of the grouped GEMMs that use this
 * workspace (every pipeline mbarrier wait of moe_grouped_* and the calls built on
 * them), written into the workspace header on `stream`; 0 restores the default of
 * 2 s (as does moe_workspace_init).  A wait that runs past the limit sets
 * MOE_DEVERR_TIMEOUT in the error word; the kernel then lets the copies and MMAs
 * it has issued finish, frees its tensor memory and exits, leaving the call's
 * outputs invalid and the context usable.  Failure detection ("[JAX] Expert
 * Parallelism: JAX primitives + VJPs", commit log: kernel contracts are trusted and
 * errors surface instead of being sanitised) and a short limit to exercise that
 * path.  Errors: MOE_ERR_WORKSPACE (null or too small), MOE_ERR_CUDA. */
MOE_API moe_status_t moe_workspace_set_wait_limit(void *ws, size_t ws_bytes, uint32_t limit_ns,
                                                  moe_stream_t stream);

/* Copy the device error word to *out (synchronises `stream`).  Returns
 * MOE_OK if the word is 0, MOE_ERR_DEVICE_DATA if any bit is set,
 * MOE_ERR_CUDA if the copy failed. */
MOE_API moe_status_t moe_read_device_error(const void *ws, moe_stream_t stream, uint32_t *out);

/* ------------------------------------------------------------------ */
/* A1  Top-k routing                                                    */
/* ------------------------------------------------------------------ */

/* Top-k routing over fp32 router logits ("[JAX] Expert Parallelism: JAX
 * primitives + VJPs", commit log: fused top-k router with fp32 logits; the
 * score function, a softmax over the k selected logits, is the workload's).
 *
 *   logits   device fp32 [T, E]
 *   topk_idx device int32 [T, k] out: for each token the k experts ranked
 *            first by (logit descending, expert id ascending); +0 and -0
 *            are equal; NaN ranks below -inf.  Slot j is the j-th ranked.
 *   topk_w   device fp32 [T, k] out: w_j = exp(l_j - l_0) / sum_i exp(l_i
 *            - l_0) over the selected logits; all 0 when l_0 = -inf.
 *
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0 (T = 0 is a no-op).
 * Logits must be finite or -inf for the weights to be defined.
 * Errors: MOE_ERR_INVALID_ARG (null pointer with T > 0, negative T),
 * MOE_ERR_UNSUPPORTED (E or k out of range), MOE_ERR_CUDA. */
MOE_API moe_status_t moe_route_topk(const float *logits, int64_t T, int E, int k,
                            int32_t *topk_idx, float *topk_w, moe_stream_t stream);

/* Sigmoid variant of the top-k router ("[JAX] Expert Parallelism: JAX
 * primitives + VJPs", commit log: sigmoid scores, the expert routing bias of
 * the sigmoid-bias configurations, and the kernel's weights / (sum + 1e-20)
 * normalisation).
 *
 *   logits      device fp32 [T, E]; score s_e = sigmoid(l_e) in fp32
 *   expert_bias device fp32 [E] or NULL (all zero): added to the scores for
 *               the selection only
 *   normalize   0: w_j = s_j;  else w_j = s_j / (sum of the k selected s + 1e-20)
 *   topk_idx    device int32 [T, k] out: the k experts ranked first by
 *               (s_e + b_e descending, expert id ascending); a NaN logit ranks
 *               last (its weight is 0)
 *   topk_w      device fp32 [T, k] out: the weights above (never NaN for
 *               finite or -inf logits: all-zero scores give zero weights)
 *
 * Limits and errors as moe_route_topk. */
MOE_API moe_status_t moe_route_topk_sigmoid(const float *logits, const float *expert_bias, int64_t T, int E,
                                            int k, int normalize, int32_t *topk_idx, float *topk_w,
                                            moe_stream_t stream);

#define MOE_SCORE_SOFTMAX 0   /* moe_route_topk */
#define MOE_SCORE_SIGMOID 1   /* moe_route_topk_sigmoid */

/* Router backward: the fp32 logits cotangent from the weights' cotangent
 * ("[JAX] Expert Parallelism: JAX primitives + VJPs", commit log: the
 * router's backward gives an fp32 cotangent of the fp32-promoted logits).
 * The selection is taken as given (piecewise constant: unselected experts and
 * the routing bias get no gradient); the weights are recomputed in fp32 from
 * the logits over the valid selected ids.
 *
 *   logits    device fp32 [T, E] (the forward's input)
 *   topk_idx  device int32 [T, k] (the forward's selection); ids outside
 *             [0, E) are skipped (no logit receives their gradient)
 *   d_topk_w  device fp32 [T, k] (e.g. from moe_combine_bwd)
 *   score_fn  MOE_SCORE_SOFTMAX: dl_j = w_j (g_j - sum_i w_i g_i)
 *             MOE_SCORE_SIGMOID: ds_j = normalize ? (g_j - sum_i w_i g_i) /
 *             (S + 1e-20) : g_j, dl_j = ds_j s_j (1 - s_j), S = sum of the
 *             selected scores
 *   d_logits  device fp32 [T, E] out, dense: 0 where not selected; an expert
 *             selected twice receives the sum
 *
 * Limits as moe_route_topk.  Errors: MOE_ERR_INVALID_ARG (null pointer with
 * T > 0, negative T, unknown score_fn), MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API moe_status_t moe_route_topk_bwd(const float *logits, const int32_t *topk_idx, const float *d_topk_w,
                                        int64_t T, int E, int k, int score_fn, int normalize, float *d_logits,
                                        moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A2  Permutation into expert-contiguous order                         */
/* ------------------------------------------------------------------ */

/* One-GPU counterpart of the expert-parallel dispatch ("[JAX] Expert
 * Parallelism", commit log: receive buffer laid out expert-major, per-expert
 * token counts fed to the grouped GEMM from device memory; "Add MoE +
 * expert-parallel Python API surface, PyTorch reference, and tests":
 * "-1 = dropped route", other ids out of range are an error).
 *
 * Routes are flattened r = t*k + j.  Route r with id e in [0, E) gets row
 * group_offsets[e] + #{r' < r : id(r') == e} (stable order); each group
 * occupies round_up(group_sizes[e], align) rows.
 *
 *   x             device bf16 [T, H] tokens
 *   topk_idx      device int32 [T, k]; -1 = dropped route; an id outside
 *                 [-1, E) sets MOE_DEVERR_BAD_EXPERT_ID and is dropped
 *   x_perm        device bf16 [rows_cap, H] out: row dst_of_route[r] holds
 *                 x[r / k]; padding rows (align > 1) are zero; rows past
 *                 group_offsets[E] are not written
 *   rows_cap      capacity of x_perm / src_of_row; must be >= T*k +
 *                 E*(align-1) so that every route fits
 *   dst_of_route  device int32 [T, k] out: row of each route, -1 if dropped
 *   src_of_row    device int32 [rows_cap] out: route r of each row, -1 for
 *                 padding rows; rows past group_offsets[E] are not written
 *   group_sizes   device int32 [E] out: routes per expert
 *   group_offsets device int32 [E+1] out: first row of each group;
 *                 group_offsets[E] = rows used
 *   ws, ws_bytes  device workspace of at least moe_workspace_bytes(T,E,k)
 *                 bytes, initialised once with moe_workspace_init
 *
 * Limits: H % 8 == 0, 1 <= E <= 1024, 1 <= k <= 32, 1 <= align <= 1024.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA; device: MOE_DEVERR_BAD_EXPERT_ID. */
MOE_API moe_status_t moe_permute(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T, int H,
                         int E, int k, int align, moe_bf16_t *x_perm, int64_t rows_cap,
                         int32_t *dst_of_route, int32_t *src_of_row, int32_t *group_sizes,
                         int32_t *group_offsets, void *ws, size_t ws_bytes,
                         moe_stream_t stream);

/* moe_permute for callers that cannot allocate device memory.  The pages
 * have no counterpart of this call; it exists for hosts whose device memory
 * is owned by someone else -- a framework's caching allocator or a fixed
 * arena sized up front, where a stray cudaMalloc breaks the memory budget --
 * and for plain C or plugin callers with no way to manage a workspace buffer.
 *
 * Same arguments, results and limits as moe_permute, except:
 *   - no workspace: the scratch (error word and per-chunk expert counts)
 *     lives in a fixed 256 KiB array inside this library's device image,
 *     resident on every GPU that loads the library until the process exits;
 *   - problems whose scratch exceeds it are rejected with
 *     MOE_ERR_UNSUPPORTED: ceil(T*k / 2048) * E must be <= 65472;
 *   - error_word: device uint32 out (nullable) that receives this call's
 *     device error bits (MOE_DEVERR_*), stream-ordered after the call.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current, and the lookup is
 * repeated when the device's current context is no longer the one the address
 * was taken in (after cudaDeviceReset, or under another context); make the
 * first call in each context before any stream capture.  Every call shares
 * the one array, so calls that overlap on the GPU (for example on two
 * streams at once) race and give undefined results; serialise them. */
MOE_API moe_status_t moe_permute_static_scratch(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T,
                                                int H, int E, int k, int align, moe_bf16_t *x_perm,
                                                int64_t rows_cap, int32_t *dst_of_route,
                                                int32_t *src_of_row, int32_t *group_sizes,
                                                int32_t *group_offsets, uint32_t *error_word,
                                                moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A3 + A4  Grouped expert FFN, forward                                 */
/* ------------------------------------------------------------------ */

/* For every expert e and every row i in [group_offsets[e], group_offsets[e+1]):
 *   g = x_perm[i] W_gate[e],  u = x_perm[i] W_up[e]     (fp32 accumulation)
 *   h[i] = bf16(silu(g) * u)                            (SwiGLU, fp32)
 *   y_perm[i] = bf16(h[i] W_down[e])                    (fp32 accumulation)
 * ("Add MoE + expert-parallel Python API surface, PyTorch reference, and
 * tests", Summary: local SwiGLU experts silu(gate) * up, the fc1_c stash;
 * "[Draft][JAX] MoE block optimization", diagram: fused grouped GEMM and
 * SwiGLU, then the down projection.)
 *
 *   x_perm        device bf16 [rows_cap, H] (from moe_permute)
 *   W_gate, W_up  device bf16 [E, H, F]
 *   W_down        device bf16 [E, F, H]
 *   group_offsets device int32 [E+1] (from moe_permute); read on the device
 *   rows_cap      rows of x_perm / h / y_perm; group_offsets[E] <= rows_cap
 *   h             device bf16 [rows_cap, F] out (rows of groups only)
 *   y_perm        device bf16 [rows_cap, H] out (rows of groups only): the
 *                 expert outputs in 2-byte slots, as the pages' combine carries
 *                 them ("[JAX] Expert Parallelism: JAX primitives + VJPs",
 *                 commit log)
 *   fc1_c         device bf16 [rows_cap, 2F] out, or NULL: the pre-SwiGLU
 *                 accumulators rounded to bf16, gate in columns [0, F) and
 *                 up in [F, 2F); needed by moe_grouped_ffn_bwd
 *   ws, ws_bytes  workspace (error word)
 *
 * Limits: H % 128 == 0, F % 128 == 0, 1 <= E <= 1024, rows_cap < 2^31.
 * Rows outside every group are neither read into results nor written.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA; device: MOE_DEVERR_TIMEOUT. */
MOE_API moe_status_t moe_grouped_ffn_fwd(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                 const moe_bf16_t *W_up, const moe_bf16_t *W_down,
                                 const int32_t *group_offsets, int E, int H, int F,
                                 int64_t rows_cap, moe_bf16_t *h, moe_bf16_t *y_perm,
                                 moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                 moe_stream_t stream);

/* The two halves of moe_grouped_ffn_fwd, callable on their own (same
 * arguments, same limits and errors):
 *   moe_grouped_fc1_swiglu  x_perm -> h (and the optional fc1_c stash)
 *   moe_grouped_fc2         h -> y_perm */
MOE_API moe_status_t moe_grouped_fc1_swiglu(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                            const moe_bf16_t *W_up, const int32_t *group_offsets,
                                            int E, int H, int F, int64_t rows_cap, moe_bf16_t *h,
                                            moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                            moe_stream_t stream);
MOE_API moe_status_t moe_grouped_fc2(const moe_bf16_t *h, const moe_bf16_t *W_down,
                                     const int32_t *group_offsets, int E, int H, int F,
                                     int64_t rows_cap, moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* The same two steps with the router weight applied early ("Add MoE +
 * expert-parallel Python API surface, PyTorch reference, and tests", Summary:
 * the router weight in the FC1 or FC2 epilogue; "[JAX] Expert Parallelism",
 * commit log: apply_topk_weights_early).  Row `row` of the permuted tensors
 * belongs to route src_of_row[row] (from moe_permute; -1 = padding row, weight
 * 0) and is scaled by topk_w[src_of_row[row]] (topk_w fp32 [T, k] read flat):
 *   moe_grouped_fc1_swiglu_weighted   h = bf16(w * silu(g) * u); fc1_c (if
 *                                      not NULL) keeps the unweighted g | u
 *   moe_grouped_fc2_weighted          y_perm = bf16(w * (h W_down)), the product in fp32
 * Combine such outputs with moe_unpermute_combine(..., topk_w = NULL, ...).
 * The three placements are one function in exact arithmetic; the FC1 one
 * rounds the weighted h to bf16, the FC2 one the weighted y.  Forward only: moe_grouped_ffn_bwd assumes
 * the weight is applied in the combine.  Other arguments, limits and errors as
 * above; src_of_row / topk_w NULL with rows_cap > 0 is MOE_ERR_INVALID_ARG. */
MOE_API moe_status_t moe_grouped_fc1_swiglu_weighted(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                                     const moe_bf16_t *W_up, const int32_t *group_offsets,
                                                     const int32_t *src_of_row, const float *topk_w, int E,
                                                     int H, int F, int64_t rows_cap, moe_bf16_t *h,
                                                     moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                                     moe_stream_t stream);
MOE_API moe_status_t moe_grouped_fc2_weighted(const moe_bf16_t *h, const moe_bf16_t *W_down,
                                              const int32_t *group_offsets, const int32_t *src_of_row,
                                              const float *topk_w, int E, int H, int F, int64_t rows_cap,
                                              moe_bf16_t *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Optional clamp of the SwiGLU inputs ("Add MoE + expert-parallel Python API surface,
 * PyTorch reference, and tests", Summary: local SwiGLU experts with an optional
 * DeepSeek-style clamp, inclusive clamp bounds; the pages give no values, so the
 * bounds are the caller's): the fp32 accumulators are clamped before SwiGLU,
 *   h = bf16(silu(clamp(g, gate_lo, gate_hi)) * clamp(u, up_lo, up_hi))   (times the
 *   route weight when src_of_row / topk_w are given, as moe_grouped_fc1_swiglu_weighted)
 * fc1_c (nullable) stashes the unclamped g | u.  The backward of a clamped forward uses
 * moe_grouped_dgrad_fc2_dswiglu_clamped with the same bounds: the dSwiGLU is taken at
 * the clamped values, and an input outside its interval gets derivative 0 (a value equal
 * to a bound is inside).  Infinite ends disable a side.  Errors: MOE_ERR_INVALID_ARG for
 * an empty interval or a NaN bound, else as the unclamped calls. */
MOE_API moe_status_t moe_grouped_fc1_swiglu_clamped(const moe_bf16_t *x_perm, const moe_bf16_t *W_gate,
                                                    const moe_bf16_t *W_up, const int32_t *group_offsets,
                                                    const int32_t *src_of_row, const float *topk_w, int E, int H,
                                                    int F, int64_t rows_cap, float gate_lo, float gate_hi,
                                                    float up_lo, float up_hi, moe_bf16_t *h, moe_bf16_t *fc1_c,
                                                    void *ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A5  Weighted unpermute / combine                                     */
/* ------------------------------------------------------------------ */

/* out[t] = bf16( sum_{j<k} topk_w[t,j] * y_perm[dst_of_route[t,j]] ), the
 * sum taken in fp32 in slot order; routes with dst -1 contribute nothing
 * ("Add MoE + expert-parallel Python API surface, PyTorch reference, and
 * tests", Summary: per-top-k combine; "[JAX] Expert Parallelism", sequence
 * diagram: the combine that returns expert outputs to token order).
 *
 *   y_perm       device bf16 [rows, H] (each value widened exactly to fp32)
 *   dst_of_route device int32 [T, k] (from moe_permute)
 *   topk_w       device fp32 [T, k], or NULL for weights 1 (the plain sum, when
 *                the router weight was already applied in FC1 or FC2)
 *   out          device bf16 [T, H] out
 *
 * Limits: H % 8 == 0, 1 <= k <= 32.  Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API moe_status_t moe_unpermute_combine(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                   const float *topk_w, int64_t T, int H, int k,
                                   moe_bf16_t *out, moe_stream_t stream);

/* The combine with the output encoded as MXFP8 along H ("Add MoE + expert-parallel
 * Python API surface, PyTorch reference, and tests", Summary: mxfp8 public outputs
 * as block-scaled tensors, logical unswizzled layout): the fp32 slot-order sum of
 * moe_unpermute_combine, then per 32 consecutive elements of a token row the MX
 * rule of the MXFP8 section below.  out_q: device uint8 [T, H] (E4M3 codes);
 * out_sf: device uint8 [T, H/32] (UE8M0 scale bytes, row-major).  topk_w may be
 * NULL (plain sum).  Limits: H % 32 == 0, 1 <= k <= 32; y_perm 16-byte and out_q
 * 8-byte aligned. */
MOE_API moe_status_t moe_unpermute_combine_mxfp8(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                                 const float *topk_w, int64_t T, int H, int k, uint8_t *out_q,
                                                 uint8_t *out_sf, moe_stream_t stream);

/* The combine with the output encoded as NVFP4 along H ("Add MoE + expert-parallel
 * Python API surface, PyTorch reference, and tests", Summary: nvfp4 public outputs as
 * block-scaled tensors, logical unswizzled layout; BlockScaledTensor: data plus one
 * scale per block, block_size 16 for nvfp4, no tensor-level scale).  The pages fix no
 * more of the format; the reading taken: the fp32 slot-order sum of
 * moe_unpermute_combine, then per 16 consecutive elements of a token row one FP8 E4M3
 * scale s = the smallest positive finite E4M3 value with 6 s >= the block's max |v|
 * (448 beyond 6 * 448, where elements saturate; byte 0 for an all-zero block) and
 * FP4 E2M1 elements = the magnitude in {0, 0.5, 1, 1.5, 2, 3, 4, 6} nearest |v| / s,
 * ties to the even code, sign bit (bit 3) set for v < 0.  Decoded value:
 * +-magnitude * s.
 *   out_q   device uint8 [T, H/2]: two codes per byte, element 2i in the low nibble
 *   out_sf  device uint8 [T, H/16]: the E4M3 scale bytes, row-major
 * topk_w may be NULL (plain sum).  Limits: H % 16 == 0, 1 <= k <= 32; y_perm 16-byte
 * and out_q 4-byte aligned (else MOE_ERR_UNSUPPORTED).  Errors as
 * moe_unpermute_combine. */
MOE_API moe_status_t moe_unpermute_combine_nvfp4(const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                                 const float *topk_w, int64_t T, int H, int k, uint8_t *out_q,
                                                 uint8_t *out_sf, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A6 + A7  MXFP8 path                                                  */
/* ------------------------------------------------------------------ */

/* MXFP8 = E4M3 elements with one UE8M0 scale per 32 consecutive elements along
 * the contraction dimension K ("Add MoE + expert-parallel Python API surface,
 * PyTorch reference, and tests", BlockScaledTensor: block size 32 for mxfp8;
 * "MoE training optimization": grouped MXFP8 quantize and grouped GEMM).
 * Scale of a block with maximum magnitude amax: the smallest 2^X with
 * amax / 2^X <= 448 (X = floor(log2 amax) - 8, +1 when amax's significand
 * exceeds 1.75), clamped to [-127, 127], stored as X + 127 (amax = 0 -> 0).
 * Elements: v / 2^X rounded to nearest even onto E4M3, saturated to +-448.
 *
 * Scale layouts:
 *   row-major    uint8 [rows][K/32]
 *   tile layout  the block-scaled MMA's operand layout.  Rows are cut into
 *                128-row tiles per group (tile ids run over the groups in
 *                order, ceil(rows_g / 128) tiles per group); each tile has one
 *                512-byte atom per 128 K elements, atoms ordered [tile][K/128],
 *                byte (m % 32) * 16 + (m / 32) * 4 + (kb % 4) for tile row m
 *                and 32-block kb.  Size: moe_mx_tile_scale_bytes(rows_cap, E, K).
 *   weights      [E][K/128][N/128] atoms of the same form, m = n % 128. */
MOE_API size_t moe_mx_tile_scale_bytes(int64_t rows_cap, int E, int K);

/* A6: quantise rows of a bf16 [rows, K] matrix along K.  data: uint8
 * [rows, K] out.  scale_rowmajor (nullable): [rows][K/32] out.  scale_tiles
 * (nullable): tile-layout scales of the groups given by group_offsets [G+1]
 * (required with scale_tiles; ws must then hold 256 + 4*(G+1) bytes).  At
 * least one scale output.  Limits: K % 128 == 0, G <= 1024. */
MOE_API moe_status_t moe_grouped_quantize_mxfp8(const moe_bf16_t *in, int64_t rows, int K,
                                                const int32_t *group_offsets, int G, uint8_t *data,
                                                uint8_t *scale_rowmajor, uint8_t *scale_tiles, void *ws,
                                                size_t ws_bytes, moe_stream_t stream);

/* Quantise expert weights W bf16 [E, K, N] (N contiguous) along K.  data:
 * E*K*N bytes of E4M3 codes as the MMA's K-major operand, tiled: one
 * contiguous 16 KB block per (expert, 128 K elements, 128 rows n), blocks
 * ordered [E][K/128][N/128]; inside a block row r = n % 128 takes 128 bytes
 * (the codes of k % 128 = 0..127) with its 16-byte chunk j stored at chunk
 * j ^ (r % 8) (the 128-byte swizzle), so each block is one bulk copy.
 * scales: the weights' tile layout ([E][K/128][N/128] 512-byte atoms,
 * E*K*N/32 bytes).  For W_gate / W_up pass K = H, N = F; for W_down K = F,
 * N = H.  Limits: K % 128 == 0, N % 128 == 0. */
MOE_API moe_status_t moe_quantize_weights_mxfp8(const moe_bf16_t *W, int E, int K, int N, uint8_t *data,
                                                uint8_t *scales, moe_stream_t stream);

/* moe_permute with the rows quantised to MXFP8 on the way (each token row is
 * read once): x_q uint8 [rows_cap, H] out (row dst_of_route[r] holds the
 * E4M3 codes of x[r / k]), x_sf tile-layout scales out
 * (moe_mx_tile_scale_bytes(rows_cap, E, H) bytes).  Other arguments and
 * outputs as moe_permute with align = 1.  Limits: H % 128 == 0; x 16-byte,
 * x_q 8-byte and x_sf 4-byte aligned (else MOE_ERR_UNSUPPORTED). */
MOE_API moe_status_t moe_permute_mxfp8(const moe_bf16_t *x, const int32_t *topk_idx, int64_t T, int H, int E,
                                       int k, uint8_t *x_q, uint8_t *x_sf, int64_t rows_cap,
                                       int32_t *dst_of_route, int32_t *src_of_row, int32_t *group_sizes,
                                       int32_t *group_offsets, void *ws, size_t ws_bytes, moe_stream_t stream);

/* A7: the grouped FFN on MXFP8 operands with block-scaled tcgen05 MMAs, fp32
 * accumulation:
 *   h = silu(x W_gate) * (x W_up) (fp32), quantised to MXFP8 along F:
 *       h_q uint8 [rows_cap, F], h_sf tile layout (moe_mx_tile_scale_bytes(rows_cap, E, F))
 *   y_perm = bf16(h W_down) [rows_cap, H]
 * x_q / x_sf from moe_permute_mxfp8; Wg_q, Wu_q (K = H, N = F) and Wd_q
 * (K = F, N = H) with their scales from moe_quantize_weights_mxfp8.  All code
 * and scale pointers 16-byte aligned.  Limits: H % 128 == 0, F % 128 == 0, E <= 1024.
 * moe_grouped_fc1_swiglu_mxfp8 and moe_grouped_fc2_mxfp8 are the two halves. */
MOE_API moe_status_t moe_grouped_ffn_fwd_mxfp8(const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q,
                                               const uint8_t *Wg_sf, const uint8_t *Wu_q, const uint8_t *Wu_sf,
                                               const uint8_t *Wd_q, const uint8_t *Wd_sf,
                                               const int32_t *group_offsets, int E, int H, int F,
                                               int64_t rows_cap, uint8_t *h_q, uint8_t *h_sf, moe_bf16_t *y_perm,
                                               void *ws, size_t ws_bytes, moe_stream_t stream);
/* moe_grouped_fc1_swiglu_mxfp8 also writes, when fc1_c is non-NULL, the bf16
 * stash of the fp32 accumulators g | u, bf16 [rows_cap, 2F], for the
 * straight-through backward (moe_dequantize_rows_mxfp8 below). */
MOE_API moe_status_t moe_grouped_fc1_swiglu_mxfp8(const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q,
                                                  const uint8_t *Wg_sf, const uint8_t *Wu_q, const uint8_t *Wu_sf,
                                                  const int32_t *group_offsets, int E, int H, int F,
                                                  int64_t rows_cap, uint8_t *h_q, uint8_t *h_sf,
                                                  moe_bf16_t *fc1_c, void *ws, size_t ws_bytes,
                                                  moe_stream_t stream);
/* moe_grouped_fc1_swiglu_mxfp8 with the SwiGLU inputs clamped (bounds and errors as
 * moe_grouped_fc1_swiglu_clamped); the straight-through backward then uses
 * moe_grouped_dgrad_fc2_dswiglu_clamped with the same bounds. */
MOE_API moe_status_t moe_grouped_fc1_swiglu_mxfp8_clamped(
    const uint8_t *x_q, const uint8_t *x_sf, const uint8_t *Wg_q, const uint8_t *Wg_sf, const uint8_t *Wu_q,
    const uint8_t *Wu_sf, const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap, float gate_lo,
    float gate_hi, float up_lo, float up_hi, uint8_t *h_q, uint8_t *h_sf, moe_bf16_t *fc1_c, void *ws,
    size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_fc2_mxfp8(const uint8_t *h_q, const uint8_t *h_sf, const uint8_t *Wd_q,
                                           const uint8_t *Wd_sf, const int32_t *group_offsets, int E, int H, int F,
                                           int64_t rows_cap, moe_bf16_t *y_perm, void *ws, size_t ws_bytes,
                                           moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A8  Backward                                                         */
/* ------------------------------------------------------------------ */

/* Backward of the expert FFN and the combine ("Add MoE + expert-parallel
 * Python API surface, PyTorch reference, and tests", Summary: the backward
 * re-dispatches gradient rows along the forward routes, recomputes SwiGLU
 * from the bf16 fc1_c stash, returns FP32 weight gradients and the route
 * (top-k weight) gradients; "[Draft][JAX] MoE block optimization": fused
 * grouped_gemm_dswiglu; "[JAX] Expert Parallelism", commit log: the wgrad of
 * an expert with no tokens is zero, never uninitialised).  For route
 * r = (t, j) -> expert e at permuted row i = dst_of_route[t, j]:
 *   dy_perm[i] = bf16(w[t,j] dY[t]);          d_topk_w[t,j] = <dY[t], y_perm[i]>
 *   dh = dy_perm[i] W_down[e]^T (fp32);       g, u = fc1_c[i] (bf16 stash)
 *   dgu[i] = bf16([dh u s (1 + g (1 - s)) | dh g s]),  s = sigmoid(g)
 *   dx_perm[i] = dgu[i] [W_gate[e]; W_up[e]]^T (fp32)
 *   dx[t] = bf16(sum_j dx_perm[row(t,j)])
 *   dW_down[e] = sum_i h[i]^T dy_perm[i];  [dW_gate|dW_up][e] = sum_i x_perm[i]^T dgu[i]
 *     (fp32, over the rows of group e; experts with no rows get exact zeros)
 * Shapes: dY, dx bf16 [T, H]; x_perm, dy_perm bf16 [rows_cap, H]; h bf16
 * [rows_cap, F]; fc1_c, dgu bf16 [rows_cap, 2F]; y_perm bf16 and dx_perm fp32
 * [rows_cap, H]; dW_gate, dW_up fp32 [E, H, F]; dW_down fp32 [E, F, H];
 * d_topk_w fp32 [T, k] (nullable; y_perm may then be NULL).  dy_perm, dgu
 * and dx_perm are caller-owned scratch.  group_sizes/group_offsets/
 * dst_of_route are the forward's (moe_permute); padding rows (align > 1)
 * get zero gradient rows.  Limits: H % 128 == 0, F % 128 == 0, E <= 1024,
 * 1 <= k <= 32.  Errors as for the forward calls. */
MOE_API moe_status_t moe_grouped_ffn_bwd(
    const moe_bf16_t *dY, const moe_bf16_t *x_perm, const moe_bf16_t *W_gate, const moe_bf16_t *W_up,
    const moe_bf16_t *W_down, const moe_bf16_t *fc1_c, const moe_bf16_t *h, const moe_bf16_t *y_perm,
    const int32_t *dst_of_route, const int32_t *group_sizes, const int32_t *group_offsets,
    const float *topk_w, int64_t T, int H, int F, int E, int k, int64_t rows_cap, moe_bf16_t *dy_perm,
    moe_bf16_t *dgu, float *dx_perm, moe_bf16_t *dx, float *dW_gate, float *dW_up, float *dW_down,
    float *d_topk_w, void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_grouped_ffn_bwd with the weight gradients stored as bf16 (the fp32 accumulators rounded
 * to nearest even once, the values moe_grouped_ffn_bwd stores rounded): dW_gate, dW_up bf16
 * [E, H, F], dW_down bf16 [E, F, H] ("[JAX] Expert Parallelism", commit log: outputs in the
 * input dtype).  Everything else as moe_grouped_ffn_bwd. */
MOE_API moe_status_t moe_grouped_ffn_bwd_bf16(
    const moe_bf16_t *dY, const moe_bf16_t *x_perm, const moe_bf16_t *W_gate, const moe_bf16_t *W_up,
    const moe_bf16_t *W_down, const moe_bf16_t *fc1_c, const moe_bf16_t *h, const moe_bf16_t *y_perm,
    const int32_t *dst_of_route, const int32_t *group_sizes, const int32_t *group_offsets,
    const float *topk_w, int64_t T, int H, int F, int E, int k, int64_t rows_cap, moe_bf16_t *dy_perm,
    moe_bf16_t *dgu, float *dx_perm, moe_bf16_t *dx, moe_bf16_t *dW_gate, moe_bf16_t *dW_up,
    moe_bf16_t *dW_down, float *d_topk_w, void *ws, size_t ws_bytes, moe_stream_t stream);

/* The steps of moe_grouped_ffn_bwd, callable on their own (same arguments,
 * limits and errors; each reads what the previous steps wrote):
 *   moe_combine_bwd               dY -> dy_perm (+ zero padding rows), d_topk_w
 *   moe_grouped_dgrad_fc2_dswiglu dy_perm, fc1_c -> dgu
 *   moe_grouped_dgrad_fc1         dgu -> dx_perm
 *   moe_grouped_wgrad             x_perm, h, dy_perm, dgu -> dW_gate, dW_up, dW_down
 *                                 (moe_grouped_wgrad_bf16: the same gradients stored as bf16)
 *   moe_unpermute_sum             dx_perm -> dx */
MOE_API moe_status_t moe_combine_bwd(const moe_bf16_t *dY, const moe_bf16_t *y_perm, const int32_t *dst_of_route,
                                     const float *topk_w, const int32_t *group_sizes,
                                     const int32_t *group_offsets, int64_t T, int H, int E, int k,
                                     int64_t rows_cap, moe_bf16_t *dy_perm, float *d_topk_w,
                                     moe_stream_t stream);
MOE_API moe_status_t moe_grouped_dgrad_fc2_dswiglu(const moe_bf16_t *dy_perm, const moe_bf16_t *W_down,
                                                   const moe_bf16_t *fc1_c, const int32_t *group_offsets,
                                                   int E, int H, int F, int64_t rows_cap, moe_bf16_t *dgu,
                                                   void *ws, size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_dgrad_fc2_dswiglu_clamped(const moe_bf16_t *dy_perm, const moe_bf16_t *W_down,
                                                           const moe_bf16_t *fc1_c, const int32_t *group_offsets,
                                                           int E, int H, int F, int64_t rows_cap, float gate_lo,
                                                           float gate_hi, float up_lo, float up_hi, moe_bf16_t *dgu,
                                                           void *ws, size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_dgrad_fc1(const moe_bf16_t *dgu, const moe_bf16_t *W_gate,
                                           const moe_bf16_t *W_up, const int32_t *group_offsets, int E,
                                           int H, int F, int64_t rows_cap, float *dx_perm, void *ws,
                                           size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_wgrad(const moe_bf16_t *x_perm, const moe_bf16_t *h,
                                       const moe_bf16_t *dy_perm, const moe_bf16_t *dgu,
                                       const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap,
                                       float *dW_gate, float *dW_up, float *dW_down, void *ws,
                                       size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_wgrad_bf16(const moe_bf16_t *x_perm, const moe_bf16_t *h,
                                            const moe_bf16_t *dy_perm, const moe_bf16_t *dgu,
                                            const int32_t *group_offsets, int E, int H, int F, int64_t rows_cap,
                                            moe_bf16_t *dW_gate, moe_bf16_t *dW_up, moe_bf16_t *dW_down, void *ws,
                                            size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_unpermute_sum(const float *dx_perm, const int32_t *dst_of_route, int64_t T, int H,
                                       int k, moe_bf16_t *dx, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* A8 on the MXFP8 path: straight-through backward                      */
/* ------------------------------------------------------------------ */

/* The backward of the MXFP8 forward treats every quantisation round trip as
 * the identity ("Add MoE + expert-parallel Python API surface, PyTorch
 * reference, and tests", Summary: quantization round-trips are
 * straight-through).  It is moe_grouped_ffn_bwd run on the values the forward's
 * block-scaled MMAs consumed: x_perm and h replaced by the dequantised x_q and
 * h_q rows, the weights by their dequantised codes, fc1_c from
 * moe_grouped_fc1_swiglu_mxfp8.  Gradients are with respect to the
 * unquantised x and weights.  Dequantised values (code * 2^(scale - 127)) are
 * exact in bf16 except below 2^-133, which flushes to zero.
 *
 * moe_dequantize_rows_mxfp8: codes uint8 [rows, K] with tile-layout scales of
 * the groups given by group_offsets [G+1] (as written by moe_permute_mxfp8 or
 * moe_grouped_fc1_swiglu_mxfp8) -> out bf16 [rows, K]; rows at or past
 * group_offsets[G] are written as zeros.  ws must hold 256 + 4*(G+1) bytes.
 * Limits: K % 128 == 0, G <= 1024; codes and out 16-byte aligned.
 *
 * moe_dequantize_weights_mxfp8: the inverse of moe_quantize_weights_mxfp8's
 * layout: tiled codes and weight scales -> W bf16 [E, K, N] (N contiguous).
 * Limits: K % 128 == 0, N % 128 == 0; data 16-byte aligned. */
MOE_API moe_status_t moe_dequantize_rows_mxfp8(const uint8_t *codes, const uint8_t *tile_scales,
                                               const int32_t *group_offsets, int G, int64_t rows, int K,
                                               moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_dequantize_weights_mxfp8(const uint8_t *data, const uint8_t *scales, int E, int K, int N,
                                                  moe_bf16_t *W, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
