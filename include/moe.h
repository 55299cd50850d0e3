/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts layer library
 * (libmoe.so): forward and backward of one MoE expert layer on one GPU.
 *
 * The layer (per dispatch chunk of T tokens, model width d, expert FFN width
 * f, E experts, k experts per token):
 *
 *   A1  L      = x Wg^T + beta                     router logits      [T,E]
 *   A2  idx, w = softmax top-k gate of L                             [T,k]
 *   A3  counts, offsets, pos, perm                 stable dispatch by expert
 *   A4  X_perm[pos[t,j]] = x[t]                    permute            [T*k,d]
 *   A5  per expert e over its segment of X_perm:
 *         h = X W1[e]^T + b1[e],  A = GELU(h),  Y_perm = A W2[e]^T + b2[e]
 *   A6  y[t] = sum_j w[t,j] Y_perm[pos[t,j]]       combine            [T,d]
 *   and the backward of each step (A7 combine, A8 expert FFN, A9 permute,
 *   A10 router).
 *
 * Sources for the method: the gating network's output decides each token's
 * experts, tokens are permuted and then assigned to their target experts in
 * order, and the experts run one after another over only their own tokens,
 * with no dispatch mask and no zero padding ("ES-MoE: Scaling Beyond the GPU
 * Memory Limit for Large Mixture-of-Experts Model Training", review, section
 * 3 "expert-wise offloading and processing" and "dynamic expert placement",
 * section 4 table row "sequential processing"); a dedicated FFN with a
 * per-expert linear over a scatter/gather layout that batches inputs by expert
 * ("FastMoE: A Fast Mixture-of-Expert Training System", review, "proposed
 * method"); dispatch in chunks with a cap on tokens per chunk ("Flattening
 * Every Memory Peak in Long-Context Mixture-of-Experts Training", abstract,
 * PipelinedLLEP).  The pages give no gate formula, GELU variant, tie rule or
 * precision; this library takes: softmax over all E logits, the k largest
 * logits (equal logits -> lower expert index; slot j = 0 is the largest),
 * w = softmax probability (k = 1 or renorm = 0) or the k probabilities divided
 * by their sum (renorm = 1); GELU(x) = x * Phi(x) (erf form).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Every pointer is a DEVICE pointer (cudaMalloc / torch CUDA memory) on the
 *    current device, 16-byte aligned, row-major and densely packed, unless
 *    stated otherwise.  Shapes come from `moe_shape`.
 *  - Ownership: the caller allocates and frees every buffer, including the
 *    workspace (size from moe_workspace_size).  The library never allocates,
 *    frees or synchronises, and keeps no state between calls other than
 *    cached device attributes.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Calls on one stream run in order; the same
 *    workspace must not be used by calls that may overlap.
 *  - Return value: MOE_OK, or MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED for bad
 *    arguments (nothing is launched), or MOE_ERR_CUDA when a launch fails.
 *    Errors that happen on the device after launch (a bounded wait that ran
 *    out, non-finite logits) are written to `*dev_status` (an int32 in device
 *    memory that the caller zeroes and reads after synchronising); the first
 *    error wins.  Kernels never trap and every device-side wait is bounded
 *    (default 1 s, environment variable MOE_WAIT_TIMEOUT_NS overrides).
 *  - dtype MOE_BF16: x, weights, biases and activations are bf16, arithmetic
 *    accumulates in fp32; the expert GEMMs run on the tcgen05 tensor cores and
 *    need d % 64 == 0 and f % 64 == 0.  dtype MOE_F32: everything fp32 with
 *    fp32 arithmetic on CUDA cores (no TF32).  Logits, gate weights, dw and
 *    every weight / bias gradient are fp32 in both.  The router (logits and
 *    its backward) runs on CUDA cores in fp32: the tensor cores are used only
 *    for the expert GEMMs unless MOE_ROUTER_TENSOR_CORES=1 (below).
 *  - Limits: T * k < 2^31, 1 <= k <= min(E, 16), 1 <= E <= 256.
 *
 * Environment variables (all optional)
 * ------------------------------------
 *  MOE_WAIT_TIMEOUT_NS      bound on every device-side wait, ns (default 1e9;
 *                           read once per process).
 *  The rest are read at every call:
 *  MOE_ROUTER_TENSOR_CORES  "1": bf16 router logits (d % 64 == 0) as one more
 *                           segment of the tcgen05 grouped GEMM with an fp32
 *                           epilogue instead of the CUDA-core kernel.
 *  MOE_GEMM_PAIR            "0": the expert GEMMs use single CTAs (128 x 256
 *                           tiles) instead of CTA pairs (256 x 256).
 *  MOE_GEMM_MAX_UNITS       n > 0: at most n CTAs (or CTA pairs) per expert
 *                           GEMM launch; each then walks more tiles.  For
 *                           tests; results are the same for every n.
 *  MOE_DEBUG_GEMM_WITHHOLD  "u:kb", for tests of the timeout path only: in
 *                           every expert GEMM launch, the producer of the CTA
 *                           (pair) holding work unit u stops before K block kb
 *                           and issues nothing more; that CTA's bounded wait
 *                           runs out, it writes MOE_ERR_TIMEOUT to *dev_status,
 *                           drains what it issued, frees its tensor memory and
 *                           exits.  The call's outputs are then incomplete.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = 1,     /* bad argument: null / misaligned pointer, bad size */
    MOE_ERR_UNSUPPORTED = 2, /* valid but unsupported shape or dtype */
    MOE_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
    MOE_ERR_TIMEOUT = 4,     /* device: a bounded wait ran out */
    MOE_ERR_NONFINITE = 5    /* device: a router logit was NaN or infinite */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef struct {
    int64_t T;      /* tokens in this call (one dispatch chunk), >= 0 */
    int32_t d;      /* model width */
    int32_t f;      /* expert FFN hidden width */
    int32_t E;      /* number of experts */
    int32_t k;      /* experts per token */
    int32_t dtype;  /* moe_dtype of x, weights, biases and activations */
    int32_t renorm; /* 1: divide the k gate probabilities by their sum */
} moe_shape;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_string(moe_status s);

/* Bytes of device workspace that every entry point below may use for a call
 * with this shape (the maximum over all of them; 0 on invalid shape).  The
 * workspace holds transient data only (per-block histograms, dH of the expert
 * backward, router-gradient partial sums); its contents need no
 * initialisation and are garbage after the call. */
MOE_API size_t moe_workspace_size(const moe_shape* s);

/* A1 + A2 + A3: router logits, softmax top-k gate and stable dispatch.
 * Source: the gating network decides each token's experts, and tokens are
 * assigned to their target experts in order with no dispatch mask ("ES-MoE",
 * review, section 3 "dynamic expert placement" and "expert-wise offloading
 * and processing"); the gate formula and tie rule are this library's reading
 * (header above).
 *   x       [T,d] dtype            tokens
 *   Wg      [E,d] dtype            router weight
 *   logit_bias [E] fp32 or NULL    fixed per-expert additive logit shift
 *   logits  [T,E] fp32             written when compute_logits != 0 (then
 *                                  x and Wg are read); READ as the given
 *                                  logits when compute_logits == 0 (then x,
 *                                  Wg and logit_bias are ignored and may be
 *                                  NULL)
 *   idx     [T,k] int32  out       selected experts, slot 0 = largest logit,
 *                                  equal logits -> lower expert index
 *   w       [T,k] fp32   out       gate weights
 *   counts  [E]   int32  out       tokens routed to each expert
 *   offsets [E+1] int32  out       exclusive prefix sum of counts; offsets[E] = T*k
 *   pos     [T,k] int32  out       row of slot (t,j) in the expert-sorted order:
 *                                  offsets[e] + number of tokens t' < t routed to e
 *   perm    [T*k] int32  out       inverse of pos: perm[pos[t*k+j]] = t*k+j
 *   ws      workspace, dev_status  see above (MOE_ERR_NONFINITE on NaN/Inf
 *                                  logits; the outputs then stay in range but
 *                                  are otherwise unspecified)
 * Deterministic: identical logits give bit-identical idx, counts, offsets,
 * pos and perm. */
MOE_API moe_status moe_route(const moe_shape* s, const void* x, const void* Wg,
                     const float* logit_bias, float* logits, int compute_logits,
                     int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                     int32_t* pos, int32_t* perm, void* ws, int32_t* dev_status,
                     moe_stream_t stream);

/* A4: X_perm[pos[t*k+j]] = x[t].   x [T,d], X_perm [T*k,d], dtype.
 * Source: the scatter half of the scatter/gather layout that batches the
 * inputs by expert ("FastMoE", review, "proposed method"); the token
 * permutation stage of "ES-MoE", review, section 3. */
MOE_API moe_status moe_permute(const moe_shape* s, const void* x, const int32_t* pos,
                       void* x_perm, moe_stream_t stream);

/* A5: expert FFN forward over the contiguous expert segments
 * [offsets[e], offsets[e+1]) of X_perm (offsets as produced by moe_route).
 * Source: each expert runs over only its own tokens, with no zero padding
 * ("ES-MoE", review, section 3 and section 4 table row "sequential
 * processing"); the per-expert Linear-GELU-Linear of FMoETransformerMLP /
 * FMoELinear ("FastMoE", review, "proposed method").
 *   W1 [E,f,d], b1 [E,f] (or NULL = 0), W2 [E,d,f], b2 [E,d] (or NULL), dtype
 *   with h = X W1[e]^T + b1[e], the pre-activation (not stored):
 *   G  [T*k,f] out  GELU'(h), kept for the backward (the only use of h there)
 *   A  [T*k,f] out  GELU(h)
 *   y_perm [T*k,d] out
 * Experts with no tokens read no weights. */
MOE_API moe_status moe_expert_ffn_fwd(const moe_shape* s, const void* x_perm,
                              const int32_t* offsets, const void* W1, const void* b1,
                              const void* W2, const void* b2, void* G, void* A,
                              void* y_perm, void* ws, int32_t* dev_status,
                              moe_stream_t stream);

/* NEXT-2, permute half: A4 fused into A5.  The same results as moe_permute
 * followed by moe_expert_ffn_fwd (bit for bit), without X_perm: the first
 * GEMM's operand loads read row r of the expert-sorted activations straight
 * from x, as x[perm[r] / k] (four rows per TMA tile::gather4 load on the
 * tensor-core path).  Source: the scatter half of the scatter/gather layout
 * ("FastMoE", review, "proposed method") and the token permutation that
 * "ES-MoE" (review, section 3) overlaps with the experts' compute, here folded
 * into the compute itself.
 *   x    [T,d] dtype        tokens of this chunk
 *   perm [T*k] int32        from moe_route of this chunk
 *   others as moe_expert_ffn_fwd. */
MOE_API moe_status moe_expert_ffn_fwd_gather(const moe_shape* s, const void* x,
                                             const int32_t* perm, const int32_t* offsets,
                                             const void* W1, const void* b1, const void* W2,
                                             const void* b2, void* G, void* A, void* y_perm,
                                             void* ws, int32_t* dev_status, moe_stream_t stream);

/* A6 (w != NULL): y[t] = sum_j w[t,j] * y_perm[pos[t,j]], j ascending, fp32
 * accumulation.  Source: the gather half of the scatter/gather layout
 * ("FastMoE", review, "proposed method"), weighted by the gate.  A9 (w == NULL): the permute backward, y[t] = sum_j
 * y_perm[pos[t,j]].   y_perm [T*k,d], y [T,d], dtype. */
MOE_API moe_status moe_combine_fwd(const moe_shape* s, const void* y_perm, const int32_t* pos,
                           const float* w, void* y, moe_stream_t stream);

/* A7: combine backward (the chain rule through A6; the pages describe the
 * backward only as each expert's backward pass, "ES-MoE", review, section 3).
 *   dy_perm[pos[t,j]] = w[t,j] * dy[t]            [T*k,d] dtype out
 *   dw[t,j]           = <dy[t], y_perm[pos[t,j]]> [T,k]   fp32  out */
MOE_API moe_status moe_combine_bwd(const moe_shape* s, const void* dy, const void* y_perm,
                           const int32_t* pos, const float* w, void* dy_perm, float* dw,
                           moe_stream_t stream);

/* A8: expert FFN backward over the same segments (each expert's backward
 * pass over its own tokens, "ES-MoE", review, section 3).
 *   dA = dY W2[e];  dH = dA * G (G = GELU'(h) from moe_expert_ffn_fwd);
 *   dx_perm = dH W1[e]
 *   dW2[e] (+)= dY^T A,  db2[e] (+)= sum_rows dY
 *   dW1[e] (+)= dH^T X,  db1[e] (+)= sum_rows dH
 * dy_perm, x_perm [T*k,d], G, A [T*k,f] dtype; dx_perm [T*k,d] dtype out;
 * dW1 [E,f,d], db1 [E,f], dW2 [E,d,f], db2 [E,d] fp32.  accumulate == 0
 * overwrites the weight/bias gradients (experts with no tokens get zeros);
 * accumulate != 0 adds to them (used across dispatch chunks).  The row sums
 * are taken in a fixed order: results are deterministic. */
MOE_API moe_status moe_expert_ffn_bwd(const moe_shape* s, const void* dy_perm, const void* x_perm,
                              const void* G, const void* A, const int32_t* offsets,
                              const void* W1, const void* W2, void* dx_perm, float* dW1,
                              float* db1, float* dW2, float* db2, int accumulate, void* ws,
                              int32_t* dev_status, moe_stream_t stream);

/* A8, data half, for one dispatch chunk: the activation gradients and db1.
 *   dA = dY W2[e];  dH = dA * G (G = GELU'(h) from moe_expert_ffn_fwd);
 *   dx_perm = dH W1[e];  db1[e] (+)= sum_rows dH
 * dy_perm [T*k,d], G [T*k,f] dtype in; dH [T*k,f] and dx_perm [T*k,d] dtype
 * out (dH is the caller's, for moe_expert_ffn_bwd_weights); db1 [E,f] fp32,
 * overwritten (accumulate == 0; experts with no tokens get zeros) or added to.
 * ws: workspace as for moe_expert_ffn_bwd.  Source: each expert's backward
 * pass over its own tokens ("ES-MoE", review, section 3). */
MOE_API moe_status moe_expert_ffn_bwd_data(const moe_shape* s, const void* dy_perm,
                                           const void* G, const int32_t* offsets,
                                           const void* W1, const void* W2, void* dH,
                                           void* dx_perm, float* db1, int accumulate, void* ws,
                                           int32_t* dev_status, moe_stream_t stream);

/* A8, weight half, over one or more dispatch chunks in one call.
 *   dW2[e] (+)= dY^T A,  db2[e] (+)= sum_rows dY,  dW1[e] (+)= dH^T X
 * summed over expert e's rows in every chunk.  For a pass split into dispatch
 * chunks ("Flattening Every Memory Peak in Long-Context Mixture-of-Experts
 * Training", abstract: a cap on the tokens of a dispatch chunk) whose rows the
 * caller keeps, this writes each gradient tile once per pass instead of once
 * per chunk, and each expert's reduction runs over its rows of all chunks in
 * chunk order (fp32 accumulation).
 *   s              d, f, E, k, dtype of the layer (s->T is not used)
 *   nchunks >= 1, chunk_T  HOST array [nchunks]: tokens of each chunk (>= 0)
 *   offsets        device int32 [nchunks][offsets_stride]: chunk c's expert
 *                  offsets (from its moe_route) at c * offsets_stride;
 *                  offsets_stride >= E+1 and a multiple of 4
 *   dy_perm, x_perm [R,d], dH, A [R,f] dtype, R = k * sum(chunk_T): chunk c's
 *                  rows follow chunk c-1's (chunk c holds chunk_T[c] * k rows,
 *                  in the expert-sorted order of its dispatch)
 *   dW1 [E,f,d], dW2 [E,d,f], db2 [E,d] fp32: overwritten (accumulate == 0;
 *                  experts with no rows get zeros) or added to
 *   ws, ws_bytes   device workspace and its size.  bf16: scratch for the
 *                  partial tiles of long reductions, which are cut into parts
 *                  so that a few long (expert, tile) reductions do not leave
 *                  most SMs idle; the parts are added in a fixed order, so the
 *                  result is deterministic for a given ws_bytes (any size works,
 *                  NULL / 0 included; less scratch means coarser parts; the
 *                  finest split needs moe_expert_ffn_bwd_weights_workspace_size
 *                  bytes).  fp32: at least moe_expert_ffn_bwd_weights_workspace_size.
 * R < 2^31. */
MOE_API moe_status moe_expert_ffn_bwd_weights(const moe_shape* s, int nchunks,
                                              const int64_t* chunk_T, const int32_t* offsets,
                                              int offsets_stride, const void* dy_perm,
                                              const void* x_perm, const void* dH, const void* A,
                                              float* dW1, float* dW2, float* db2, int accumulate,
                                              void* ws, size_t ws_bytes, int32_t* dev_status,
                                              moe_stream_t stream);

/* NEXT-2, permute half, in the weight gradient: moe_expert_ffn_bwd_weights
 * with dW1 = dH^T X reading X's rows through each chunk's perm instead of
 * X_perm (bit for bit the same results).
 *   x     [sum(chunk_T), d] dtype: the chunks' tokens, chunk c's after those
 *         of chunks < c
 *   perm  device int32: chunk c's perm (from its moe_route, chunk_T[c] * k
 *         entries) at c * perm_stride; perm_stride >= k * max(chunk_T)
 *   others as moe_expert_ffn_bwd_weights (the same workspace size). */
MOE_API moe_status moe_expert_ffn_bwd_weights_gather(const moe_shape* s, int nchunks,
                                                     const int64_t* chunk_T,
                                                     const int32_t* offsets, int offsets_stride,
                                                     const void* dy_perm, const void* x,
                                                     const int32_t* perm, int64_t perm_stride,
                                                     const void* dH, const void* A, float* dW1,
                                                     float* dW2, float* db2, int accumulate,
                                                     void* ws, size_t ws_bytes,
                                                     int32_t* dev_status, moe_stream_t stream);

/* Workspace bytes for moe_expert_ffn_bwd_weights (and its _gather form) with
 * these chunks (0 on bad arguments): the finest split of its reductions
 * (bf16), the column-sum partials (fp32). */
MOE_API size_t moe_expert_ffn_bwd_weights_workspace_size(const moe_shape* s, int nchunks,
                                                         const int64_t* chunk_T);

/* A10: router backward (the gating network is trained with the model,
 * "ES-MoE", review, section 3; the formulas are the chain rule through this
 * library's gate).  dL = d(gate weights)/d(logits)^T dw:
 *   renorm: dL[idx_j] = w_j (dw_j - sum_i w_i dw_i), zero elsewhere;
 *   else:   dL[e] = sum_j dw_j p[idx_j] (delta(e, idx_j) - p[e]), p = softmax(L).
 *   dx[t]   = [sum_j dx_perm[pos[t,j]]]  +  sum_e dL[t,e] Wg[e]
 *             (dx [T,d] dtype).  With dx_perm and pos given, the bracketed
 *             permute backward (A9) is fused in and dx is overwritten; with
 *             dx_perm == NULL, dx is read and the router term added to it.
 *   dWg    (+)= dL^T x                (dWg [E,d] fp32; accumulate as above)
 * perm / offsets are the dispatch of this chunk (used to sum each expert's
 * tokens in a fixed order).  The logit shift has no gradient. */
MOE_API moe_status moe_route_bwd(const moe_shape* s, const float* dw, const float* logits,
                         const int32_t* idx, const float* w, const int32_t* perm,
                         const int32_t* offsets, const void* x, const void* Wg,
                         const void* dx_perm, const int32_t* pos, void* dx,
                         float* dWg, int accumulate, void* ws, int32_t* dev_status,
                         moe_stream_t stream);

/* Routing (A1 + A2 + A3) without a caller-provided workspace.
 *
 * For callers that cannot allocate device memory: a plug-in whose host
 * framework owns every allocation and hands it only the tensors it reads and
 * writes, with no room for a workspace.  This entry point needs nothing beyond
 * those.  It is an interface convenience of this library; the MoE method
 * itself has no counterpart for it.
 *
 * Same arguments and results as moe_route, minus `ws`.  The per-block expert
 * histogram lives in a fixed scratch array inside libmoe.so (a static device
 * array of MOE_ROUTE_NOALLOC_MAX_SCRATCH int32, 1 MiB; every GPU that loads
 * the library keeps it until the process exits).
 *   - Size limit: E * ceil(T / 64) must not exceed MOE_ROUTE_NOALLOC_MAX_SCRATCH;
 *     larger shapes return MOE_ERR_UNSUPPORTED without launching anything.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  A failure there returns MOE_ERR_CUDA.  The
 *     address is looked up again when the device's context has changed since
 *     (after cudaDeviceReset), so that a new context never gets a stale one.
 *   - The library allocates and frees nothing on this path.
 *   - All calls share the one array and leave their contents in it; every
 *     entry a call reads is written earlier by the same call, so nothing needs
 *     clearing.  Calls whose work may overlap on the GPU (different streams,
 *     no ordering between them) race on the array and give wrong results:
 *     serialise them. */
#define MOE_ROUTE_NOALLOC_MAX_SCRATCH (1 << 18)
MOE_API moe_status moe_route_noalloc(const moe_shape* s, const void* x, const void* Wg,
                                     const float* logit_bias, float* logits,
                                     int compute_logits, int32_t* idx, float* w,
                                     int32_t* counts, int32_t* offsets, int32_t* pos,
                                     int32_t* perm, int32_t* dev_status, moe_stream_t stream);

/* Diagnostics: launch one kernel that waits on a device flag that nothing
 * sets, with the library's bounded wait (limit_ns nanoseconds), then writes
 * MOE_ERR_TIMEOUT to *dev_status and returns.  It exercises the timeout path
 * every pipelined kernel uses, without hanging the GPU. */
MOE_API moe_status moe_debug_bounded_wait(uint64_t limit_ns, int32_t* dev_status,
                                  moe_stream_t stream);

/* Launch option: the tensor-core expert GEMMs (moe_expert_ffn_* calls, bf16)
 * that the calling host thread launches from now on use at most `units` CTA
 * pairs (single CTAs with MOE_GEMM_PAIR=0); 0 restores the default, every
 * pair the GPU holds at once.  Capturing a CUDA graph records the launch as
 * made.  For overlapping other kernels with the GEMMs: a persistent GEMM grid
 * holds every SM, so kernels on another stream otherwise run only in its
 * gaps (the chunk pipeline of "MPipeMoE", "research method", and the
 * overlap of "ES-MoE", review, section 3, leave SMs to the side stream this
 * way).  The data-path GEMMs' results do not depend on it; the weight
 * gradients' split reductions do (their parts follow the grid), so callers
 * that want run-to-run identical weight gradients keep one setting for them.
 * MOE_GEMM_MAX_UNITS in the environment, when set, takes precedence.  Returns
 * MOE_ERR_INVALID for units < 0. */
MOE_API moe_status moe_set_gemm_max_units(int units);

/* Diagnostics: GELU(x) = x Phi(x) and GELU'(x) = Phi(x) + x phi(x) of n fp32
 * values, as the kernels evaluate them: fast != 0 selects the approximation
 * the bf16 expert-GEMM epilogues use (erf by Abramowitz & Stegun, "Handbook
 * of Mathematical Functions", formula 7.1.26, |error| <= 1.5e-7), fast == 0
 * the CUDA erff / expf form the fp32 path uses.  x, gelu, gelu_grad: [n]
 * fp32 device arrays. */
MOE_API moe_status moe_debug_gelu(int64_t n, const float* x, float* gelu, float* gelu_grad,
                                  int fast, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
