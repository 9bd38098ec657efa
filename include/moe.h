/*
 * moe.h -- C ABI of libmoe, the GB300 (sm_103a) forward pass of one sparse
 * Mixture-of-Experts FFN layer:
 *
 *     y = SharedExpert(x) + sum_{i in TopK(x . W_g^T + b)} w_i * Expert_i(x),
 *     w = softmax over only the K selected scores,
 *     Expert(x) = W_down (SiLU(W_gate x) * (W_up x))          (SwiGLU).
 *
 * Sources, by page title and section:
 *   [R] adg.csdn.net sparse-MoE explainer ("1.8T parameters, 2% active"),
 *       section 2.2: score every expert with a small linear router, keep the
 *       K best scores, softmax over those K, weighted sum of the K experts.
 *   [S] "Sparse MoE inference kernels: expert parallelism, dynamic routing
 *       gates and all-to-all overlap" (blog.llmgo.top): section 1.1 shared
 *       expert plus routed experts; section 1.2 W_gate/W_up/W_down experts
 *       and the decode (GEMV-like) vs prefill (GEMM) regimes; section 4.2
 *       grouped GEMM over an offsets array; section 4.3 token permutation
 *       (flatten, order by expert, gather, counts, offsets); FAQ Q1 experts
 *       with zero tokens are skipped.
 *   [C] "Computation and Data Movement for Inference", sections 4 and 15:
 *       routing records sorted by expert id so one weight load serves the
 *       whole bucket; outputs returned to token order, weighted and merged.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers except `shape` and `code_out` are DEVICE pointers on the
 *    current CUDA device, 16-byte aligned.  Storage is row-major; weights are
 *    [out][in] (nn.Linear layout):
 *        x [T][d], w_g [E][d], w_gate, w_up [E][I][d], w_down [E][d][I],
 *        ws_gate, ws_up [Is][d], ws_down [d][Is], bias [E] (fp32).
 *  - dtype: MOE_F32 (every activation and weight fp32; fp32 FMA arithmetic,
 *    no TF32) or MOE_BF16 (bf16 storage, fp32 accumulation).  Router scores
 *    and routing weights are always fp32; indices are int32.
 *  - Ownership: the caller allocates every buffer, including `workspace`
 *    (size from moe_workspace_bytes).  The library never allocates device
 *    memory, frees or synchronises; all work is ordered on `stream`.  When
 *    one call's tensor-core stage has both 256-row (CTA-pair) and 128-row
 *    tiles, the 128-row grids run on a second stream of the library's own,
 *    forked from `stream` with an event and joined back before the call's
 *    next kernel (so the call stays ordered on `stream` and graph capturable).
 *    MOE_CONCURRENT=0 keeps everything on `stream`; the 8-bit entry points
 *    use the second stream only with MOE_CONCURRENT=1.
 *  - Errors: argument errors return a non-zero moe_status immediately and
 *    enqueue nothing.  A failed launch returns MOE_ERR_CUDA.  Errors found
 *    on the device (index out of range, a bounded wait that ran out) are
 *    recorded in the workspace's error word and read with
 *    moe_get_device_error after the stream has been synchronised; each entry
 *    point that takes a workspace clears that word first.
 *  - Limits: 0 <= T, T*K < 2^31; 1 <= K <= min(E, 32); E <= 1024;
 *    d and I (and Is when > 0) multiples of 64; d, I, Is <= 16384.
 *    T == 0 is a no-op returning MOE_OK (pointers to T-sized arrays may
 *    then be NULL; moe_permute still zeroes counts and offsets).
 *  - Routing rule: top-K picks the largest scores, ties to the LOWER expert
 *    index (scores compared as floats, so -0.0 == +0.0); slot j of a token
 *    holds its j-th pick (descending score).  Flat slot f = t*K + j.
 *  - Threading: entry points are reentrant and keep no mutable global state
 *    beyond per-device attributes cached on first use and, per host thread
 *    and device, that second stream and its two events (made on first use
 *    outside stream capture, kept for the thread's lifetime).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, K > E, ...          */
    MOE_ERR_UNSUPPORTED = 2, /* legal but outside the limits above          */
    MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required  */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed        */
    MOE_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out              */
    MOE_ERR_BOUNDS = 6       /* device: an index was out of range           */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/*
 * Router rule (s = x . w_g^T, the raw score; b = bias or 0):
 *   MOE_ROUTER_SOFTMAX  key = s + b; the K largest keys; w = softmax over the
 *                       K selected keys [R section 2.2].
 *   MOE_ROUTER_SIGMOID  a = sigmoid(s); key = a + b (the bias steers the
 *                       selection only); the K largest keys;
 *                       w = a / (sum of the K selected a + 1e-6) -- the
 *                       DeepSeek-V3 auxiliary-loss-free routing [S section
 *                       2.2 and the dispatcher code of section 4.3].
 */
typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1 } moe_router;

typedef struct {
    int32_t T;            /* tokens                                         */
    int32_t d;            /* hidden size                                    */
    int32_t E;            /* routed experts                                 */
    int32_t K;            /* experts per token                              */
    int32_t inter;        /* routed expert intermediate size I              */
    int32_t inter_shared; /* shared expert intermediate size Is; 0 = none   */
    int32_t dtype;        /* moe_dtype                                      */
    int32_t router;       /* moe_router (0 = softmax over the K selected)   */
} moe_shape;

/* Text for a status code (static storage, never NULL). */
const char *moe_status_string(int32_t status);

/*
 * Bytes of workspace that every entry point below accepts for `shape`
 * (one size serves all of them).  Returns 0 for an invalid shape.
 */
size_t moe_workspace_bytes(const moe_shape *shape);

/*
 * Stage 1, routing [R section 2.2; S sections 2.1-2.2].
 *   s[t][e] = sum_k x[t][k] * w_g[e][k]   (fp32 accumulate)
 *   keys and weights by shape->router (see moe_router above);
 *   topk_idx[t][j], topk_w[t][j]: the K largest keys with ties to the lower
 *   index, slot j = j-th pick, and their weights.
 * bias [E] (fp32) may be NULL (no bias).  If logits_in [T][E] (fp32) is
 * non-NULL it replaces s (x and w_g are then ignored and may be NULL); the
 * bias still applies.  logits_out [T][E] (fp32) receives the keys if non-NULL.
 * Outputs: topk_idx [T][K] int32, topk_w [T][K] fp32.
 */
moe_status moe_route(const moe_shape *shape, const void *x, const void *w_g,
                     const float *bias, const float *logits_in,
                     float *logits_out, int32_t *topk_idx, float *topk_w,
                     void *workspace, size_t ws_bytes, void *stream);

/*
 * Stage 2, dispatch [S section 4.3; C section 15].
 *   counts[e]  = number of flat slots f with topk_idx[f] == e      [E]
 *   offsets    = exclusive scan of counts, offsets[E] = T*K         [E+1]
 *   perm[p]    = flat slot at sorted position p; slots ordered by expert
 *                id, and by increasing f within an expert (stable)   [T*K]
 *   inv_perm[f]= p with perm[p] == f                                 [T*K]
 *   x_perm[p]  = x[perm[p] / K]   (row gather; skipped if x or x_perm is
 *                NULL)                                        [T*K][d]
 * perm and inv_perm may be NULL if not wanted.  An expert id outside
 * [0, E) is recorded as MOE_ERR_BOUNDS on the device and its slot dropped.
 */
moe_status moe_permute(const moe_shape *shape, const int32_t *topk_idx,
                       const void *x, int32_t *counts, int32_t *offsets,
                       int32_t *perm, int32_t *inv_perm, void *x_perm,
                       void *workspace, size_t ws_bytes, void *stream);

/*
 * moe_permute without a workspace, for callers that cannot allocate device
 * memory (a runtime that reserves all of HBM for its own pool at start-up and
 * allows no cudaMalloc afterwards, or a plug-in handed only the tensors it
 * works on).  The pages have no counterpart: this is an interface variant,
 * not part of the layer.  Arguments and results are those of moe_permute.
 * Its scratch (error word, per-chunk histogram, token of each row, and the
 * inverse permutation when inv_perm is NULL) lives in a fixed 4 MiB device
 * array inside the library, which every GPU that loads the library holds
 * until the process exits.  Shapes whose scratch would exceed it -- about
 * (T*K + T*K/1024*E) * 4 bytes, doubled for T*K when inv_perm is NULL -- are
 * refused with MOE_ERR_UNSUPPORTED; other shapes are checked exactly as
 * moe_permute checks them.  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library call.  The first call on a device looks up the array's
 * device address (with that device current) and later calls in the same CUDA
 * context reuse it; make that first call before any stream capture.  A
 * context torn down and made again (cudaDeviceReset) counts as a new one: its
 * first call looks the address up again.  All calls share the array, and
 * calls whose work overlaps on the GPU race on it.  Device-side errors are
 * not reported: a dropped slot (expert id outside [0, E)) shows as
 * offsets[E] < T*K and inv_perm[f] == -1.
 */
moe_status moe_permute_noalloc(const moe_shape *shape, const int32_t *topk_idx,
                               const void *x, int32_t *counts, int32_t *offsets,
                               int32_t *perm, int32_t *inv_perm, void *x_perm,
                               void *stream);

/*
 * Stage 3, grouped expert FFN [S sections 1.2, 4.2; C section 15].
 * For each expert e and each row p in [offsets[e], offsets[e+1]):
 *   h = SiLU(w_gate[e] . x_perm[p]) * (w_up[e] . x_perm[p]),
 *   y_perm[p] = w_down[e] . h.
 * offsets [E+1] is a device array (as written by moe_permute); nothing on
 * the host reads it.  Experts with no rows read no weights.  Rows with few
 * tokens per expert stream each selected expert's weights once (GEMV path);
 * experts with many rows run on the tcgen05 tensor-core grouped GEMM.
 * Shape fields used: d, E, inter, dtype, T and K (rows = T*K).
 * inter_shared is ignored here: the shared expert is the same operation
 * with E = 1, K = 1, offsets = {0, T} and x in place of x_perm.
 * Output: y_perm [T*K][d] in the layer dtype.
 */
moe_status moe_expert_ffn(const moe_shape *shape, const void *x_perm,
                          const int32_t *offsets, const void *w_gate,
                          const void *w_up, const void *w_down, void *y_perm,
                          void *workspace, size_t ws_bytes, void *stream);

/*
 * Stage 4, combine [R section 2.2 step 4; S section 1.1; C section 4].
 *   y[t] = y_shared[t] + sum_{j=0..K-1} topk_w[t][j] * y_perm[inv_perm[t*K+j]]
 * accumulated in fp32 (shared term first, then j ascending) and rounded
 * once to the layer dtype.  y_shared [T][d] may be NULL (no shared expert).
 * Deterministic: a gather per token, no atomics.
 */
moe_status moe_combine(const moe_shape *shape, const void *y_perm,
                       const int32_t *inv_perm, const float *topk_w,
                       const void *y_shared, void *y, void *stream);

/*
 * The whole layer: route, dispatch, routed and shared expert FFN, combine,
 * enqueued on `stream` with no host synchronisation and no host read of
 * device data (usable inside CUDA graph capture).  ws_gate/ws_up/ws_down
 * must be non-NULL iff shape->inter_shared > 0.  bias may be NULL.
 * Output: y [T][d] in the layer dtype.
 */
moe_status moe_forward(const moe_shape *shape, const void *x, const void *w_g,
                       const float *bias, const void *w_gate, const void *w_up,
                       const void *w_down, const void *ws_gate,
                       const void *ws_up, const void *ws_down, void *y,
                       void *workspace, size_t ws_bytes, void *stream);

/*
 * ---- 8-bit expert weights ------------------------------------------------
 * [Q] "LLM from scratch, ch. 6" (foundations of inference optimisation),
 * section "second route: make every byte cheaper": weight quantisation
 * x_q = round(x / s) + z, x_hat = (x_q - z) s,
 * with the scale per tensor, per channel or per group; for memory-bound
 * decode one byte per weight instead of two halves the streamed bytes.
 *
 * Format: OCP E4M3 codes (1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; largest finite magnitude 448; S.1111.111 is NaN), zero
 * point 0, one fp32 scale per weight ROW (output channel):
 *     w_hat[r][c] = e4m3_value(code[r][c]) * scale[r].
 * The layer is the bf16 layer above with every expert matrix (routed and
 * shared) replaced by w_hat; x, w_g, y and the intermediates stay bf16.
 * Groups of at most 8 rows in calls whose groups are all small (at most 64
 * rows: decode) stream their codes through a GEMV that widens them to f16
 * (exact) for mma.sync, on exact bf16 activations.  The other groups run on
 * the tcgen05 tensor cores as E4M3 x E4M3 products (kind::f8f6f4), each bf16
 * activation row carried as two E4M3 planes, x ~ s * (value(hi) + value(lo))
 * with s = amax / 448 and lo the code of the fp32 remainder (within 2^-8 of
 * |x| relative plus 2^-10 s): a documented approximation of the exact layer
 * at about bf16's own resolution (MOE_W8_PLANES=0 widens the codes to bf16
 * instead, exactly, at about half the speed).  All accumulate in fp32 and
 * apply the row scale to the fp32 sums.
 */
typedef struct moe_fp8_experts {
    const uint8_t *w_gate;  /* [E][I][d] codes                       */
    const uint8_t *w_up;    /* [E][I][d] codes                       */
    const uint8_t *w_down;  /* [E][d][I] codes                       */
    const float *s_gate;    /* [E][I] row scales                     */
    const float *s_up;      /* [E][I]                                */
    const float *s_down;    /* [E][d]                                */
    const uint8_t *ws_gate; /* [Is][d] shared-expert codes, or NULL  */
    const uint8_t *ws_up;   /* [Is][d]                               */
    const uint8_t *ws_down; /* [d][Is]                               */
    const float *ss_gate;   /* [Is]                                  */
    const float *ss_up;     /* [Is]                                  */
    const float *ss_down;   /* [d]                                   */
} moe_fp8_experts;

/*
 * Per-row quantisation [Q]: for each row r of the row-major [rows][cols]
 * matrix w (dtype MOE_F32 or MOE_BF16), scale[r] = max_c |w[r][c]| / 448
 * (fp32 division; 1 for a row of zeros) and code[r][c] = the E4M3 value
 * nearest to w[r][c] / scale[r] (fp32 division; ties to an even mantissa;
 * magnitudes past 448 saturate).  w must be finite.  codes [rows][cols]
 * (uint8) and scales [rows] (fp32) are device buffers.  Limits: rows < 2^31,
 * cols a multiple of 16.  rows == 0 is a no-op.  An offline step (a user
 * converting bf16 checkpoints); enqueued on `stream`, no workspace.
 */
moe_status moe_quantize_fp8_rows(int64_t rows, int64_t cols, int32_t dtype,
                                 const void *w, uint8_t *codes, float *scales,
                                 void *stream);

/*
 * moe_expert_ffn with 8-bit expert weights: *w is a HOST struct of device
 * pointers (the ws_* / ss_* members are ignored here).  shape->dtype must be
 * MOE_BF16 and d, inter multiples of 128 (else MOE_ERR_UNSUPPORTED); scale
 * arrays 16-byte aligned.  Groups of at most 8 rows take the 8-bit GEMV when
 * T*K <= 64 (the bound this call has on a group), the rest the tensor cores.
 * Same workspace size as moe_expert_ffn.
 */
moe_status moe_expert_ffn_fp8(const moe_shape *shape, const void *x_perm,
                              const int32_t *offsets, const moe_fp8_experts *w,
                              void *y_perm, void *workspace, size_t ws_bytes,
                              void *stream);

/*
 * moe_forward with 8-bit expert weights (routed and shared): *w is a HOST
 * struct of device pointers; the ws_* / ss_* members must be non-NULL iff
 * shape->inter_shared > 0.  w_g stays bf16.  shape->dtype must be MOE_BF16
 * and d, inter, inter_shared multiples of 128 (else MOE_ERR_UNSUPPORTED).
 * Same workspace size as moe_forward; graph-capturable like moe_forward.
 */
moe_status moe_forward_fp8(const moe_shape *shape, const void *x, const void *w_g,
                           const float *bias, const moe_fp8_experts *w, void *y,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * ---- block-scaled 8-bit weights --------------------------------------------
 * [Q] lets a quantisation scale cover a tensor, a channel or a group.  Here a
 * group is a square block of 128 x 128 weights, the layout of DeepSeek-V3's
 * 8-bit checkpoints (DeepSeek-V3 served in FP8: "Model architecture feeding
 * back into inference systems: from MHA/GQA to DeepSeek MLA", blog.llmgo.top,
 * FAQ Q3): one fp32 scale per block of the STACKED matrix,
 *     w_hat[r][c] = e4m3_value(code[r][c]) * scale[r / 128][c / 128],
 * each block quantised by the per-row rule above applied to its elements
 * (scale = block amax / 448, fp32 divisions, ties to an even mantissa,
 * saturation at 448).
 *
 * moe_quantize_fp8_blocks: w [rows][cols] (MOE_F32 or MOE_BF16, finite) ->
 * codes [rows][cols] and scales [ceil(rows/128)][ceil(cols/128)] (row-major),
 * device buffers.  Limits: cols a multiple of 16 and < 2^31, ceil(rows/128) <=
 * 65535.  rows == 0 is a no-op.  Enqueued on `stream`, no workspace.  Pass a
 * stacked weight tensor as one matrix: w_gate [E][I][d] as rows = E*I.
 */
moe_status moe_quantize_fp8_blocks(int64_t rows, int64_t cols, int32_t dtype,
                                   const void *w, uint8_t *codes, float *scales,
                                   void *stream);

/*
 * moe_expert_ffn_fp8 / moe_forward_fp8 with block scales: the codes of
 * moe_fp8_experts as before, its scale members the block grids of
 * moe_quantize_fp8_blocks: s_gate, s_up [E*I/128][d/128]; s_down
 * [E*d/128][I/128]; ss_gate, ss_up [Is/128][d/128]; ss_down [d/128][Is/128].
 * Same limits (d, inter, inter_shared multiples of 128, so no block spans two
 * experts), workspace and errors as the row-scaled calls.  Groups of at most
 * 8 rows take the 8-bit GEMV (each 128-code K block's partial sums scaled and
 * added); larger groups take the tensor cores with the activations as two
 * E4M3 planes, each 128-deep K block multiplied into its own tensor-memory
 * accumulator and added, times its block scale, to fp32 sums in registers.
 */
moe_status moe_expert_ffn_fp8_blocks(const moe_shape *shape, const void *x_perm,
                                     const int32_t *offsets, const moe_fp8_experts *w,
                                     void *y_perm, void *workspace, size_t ws_bytes,
                                     void *stream);
moe_status moe_forward_fp8_blocks(const moe_shape *shape, const void *x, const void *w_g,
                                  const float *bias, const moe_fp8_experts *w, void *y,
                                  void *workspace, size_t ws_bytes, void *stream);

/*
 * ---- 8-bit weights AND 8-bit activations (W8A8) ----------------------------
 * [Q] names weights, activations and the KV cache as things a quantisation
 * method may act on.  Here the same per-row rule quantises the two
 * activations that enter an expert's matrix products:
 *     x_hat = e4m3_value(code(x row)) * s_x,      s_x = amax(x row) / 448
 *     h     = SiLU(W_gate_hat x_hat) * (W_up_hat x_hat)  (fp32, stored bf16)
 *     h_hat = e4m3_value(code(h row)) * s_h,      s_h = amax(h row) / 448
 *     y     = W_down_hat h_hat
 * (scales and codes decided exactly as in moe_quantize_fp8_rows: fp32
 * divisions, round to nearest even, saturation at 448), with the 8-bit
 * weights of moe_fp8_experts.  Both operands of every expert GEMM are E4M3,
 * multiplied on tcgen05 kind::f8f6f4 with fp32 accumulation; both row scales
 * are applied to the fp32 sums.  Every group runs on the tensor cores, so
 * this is the prefill path; for decode moe_forward_fp8 streams the same
 * weights with bf16 activations.  The router reads the unquantised x.
 * Limits and workspace as moe_forward_fp8 / moe_expert_ffn_fp8.
 */

/* moe_expert_ffn_fp8 with 8-bit activations: each x_perm row is quantised
 * (per row) before the gate/up GEMM, each h row after it. */
moe_status moe_expert_ffn_w8a8(const moe_shape *shape, const void *x_perm,
                               const int32_t *offsets, const moe_fp8_experts *w,
                               void *y_perm, void *workspace, size_t ws_bytes,
                               void *stream);

/* moe_forward_fp8 with every expert (routed and shared) run W8A8; each token's
 * row of x is quantised once and its codes gathered into expert order. */
moe_status moe_forward_w8a8(const moe_shape *shape, const void *x, const void *w_g,
                            const float *bias, const moe_fp8_experts *w, void *y,
                            void *workspace, size_t ws_bytes, void *stream);

/* The W8A8 calls on block-scaled weights: x and h quantised per row as above,
 * the weights' scales the 128 x 128 block grids of moe_quantize_fp8_blocks
 * (layout as for moe_forward_fp8_blocks).  One E4M3 x E4M3 MMA per 32-deep
 * slice; each 128-deep K block is multiplied into its own tensor-memory
 * accumulator and added, times its block scale, to fp32 sums in registers,
 * the activation row's scale applied at the end.  Limits, workspace and
 * errors as moe_forward_w8a8 / moe_expert_ffn_w8a8. */
moe_status moe_expert_ffn_w8a8_blocks(const moe_shape *shape, const void *x_perm,
                                      const int32_t *offsets, const moe_fp8_experts *w,
                                      void *y_perm, void *workspace, size_t ws_bytes,
                                      void *stream);
moe_status moe_forward_w8a8_blocks(const moe_shape *shape, const void *x, const void *w_g,
                                   const float *bias, const moe_fp8_experts *w, void *y,
                                   void *workspace, size_t ws_bytes, void *stream);

/*
 * Reads the device error word of `workspace` (a device pointer passed to a
 * previous call) into *code_out (a HOST pointer): MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_BOUNDS.  Synchronous (one 16-byte device-to-host copy of the error
 * record: code, where, padding); call it after the stream that ran the work
 * has been synchronised.
 */
moe_status moe_get_device_error(const void *workspace, int32_t *code_out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
