// internal.h -- host-side interfaces between the C-ABI layer (moe_api.cu) and
// the kernel files.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

struct DevError;

// Side of the square weight-scale blocks of block-scaled 8-bit weights.
constexpr int kWBlock = 128;

// Device-built work plan for the grouped expert FFN.  Group g < E is routed
// expert g with rows [offsets[g], offsets[g+1]) of the permuted row space;
// group E (when present) is the shared expert, whose rows are the T tokens.
struct FfnPlanHeader {
    int32_t n_gemv;    // groups handled by the streaming GEMV kernels (first list)
    int32_t n_mtiles;  // 128-row tiles of the single-SM tensor-core GEMM
    int32_t n_ptiles;  // 256-row tiles of the CTA-pair tensor-core GEMM
    int32_t n_gemv2;   // second GEMV list (groups above the small-row split), or 0
    // SM split when the pair-tile and single-tile GEMMs run side by side on two
    // streams: CTA pairs of the pair-tile grid and CTAs of the single-tile grid
    // that take tiles (the rest of each grid exits at once)
    int32_t units_pair;
    int32_t units_single;
    int32_t pad_[2];
};

// One routed/shared expert group as the FFN kernels see it.
struct FfnGroups {
    int E;             // routed experts (group E = shared, if has_shared)
    int has_shared;
    int d;             // hidden size
    int I, Is;         // intermediate sizes (routed, shared)
    int n_routed_rows; // T*K (rows of x_perm / h / y_perm)
    int max_group_rows; // bound on any group's rows (0: unknown); <= 32 selects the small-row ring
    int g8_prefetch;    // 8-bit GEMV: prefetch each warp's next weight blocks into L2
    int wblock;         // 8-bit weights: 0, s_* below are row scales; kWBlock, one
                        // scale per 128 x 128 block of the stacked matrices
    int T;             // tokens (rows of the shared group)
    const int32_t* offsets;  // [E+1] device
    const int32_t* row_src;  // [n_routed_rows] token of each routed row, or
                             // null: routed row p reads A row p directly
    const void* a_routed;    // rows of x_perm (or x when row_src is set)
    const void* a_perm;      // contiguous permuted rows for the tensor-core path's
                             // large row blocks when row_src is set (or null when
                             // no group can exceed tc_gather_max_rows(T))
    const void* a_shared;    // x [T][d] (shared group input)
    const void* w_gate;      // [E][I][d]
    const void* w_up;
    const void* w_down;      // [E][d][I]
    const void* ws_gate;     // [Is][d]
    const void* ws_up;
    const void* ws_down;     // [d][Is]
    // 8-bit weights: the w_* / ws_* pointers above hold E4M3 codes and these
    // the fp32 scale of each weight row (wblock = 0) or of each 128 x 128 block
    // (wblock = kWBlock: s_gate/s_up [E*I/128][d/128], s_down [E*d/128][I/128],
    // ss_gate/ss_up [Is/128][d/128], ss_down [d/128][Is/128])
    const float* s_gate;     // [E][I]
    const float* s_up;       // [E][I]
    const float* s_down;     // [E][d]
    const float* ss_gate;    // [Is]
    const float* ss_up;      // [Is]
    const float* ss_down;    // [d]
    // 8-bit activations (launch_ffn_tc_a8_*): a_perm / a_shared hold E4M3 codes
    // and these the fp32 scale of each row; h / h_s hold codes in place after
    // the gate/up GEMM (rows 2 * I / 2 * Is bytes apart)
    const float* sa_routed;  // [n_routed_rows]
    const float* sa_shared;  // [T]
    const float* sa_h;       // [n_routed_rows]: zero before the gate/up GEMM, which
    const float* sa_hs;      // [T]              raises it to max |h| (fp32 bits); the
                             // h quantiser turns it into the row scale
    void* h;                 // [n_routed_rows][I]
    void* h_s;               // [T][Is]
    void* y;                 // [n_routed_rows][d]
    void* y_s;               // [T][d]
};

// Workspace carving (all offsets 256-byte aligned).
struct WsLayout {
    size_t err, router_part, logits, topk_idx, topk_w, counts, offsets, perm, inv_perm,
        tok_of, blk_hist, plan, gemv_list, mtile_list, x_perm, h, h_s, y_perm, y_s, ascale, total;
    int router_splits, dispatch_blocks, max_mtiles;
};
WsLayout ws_layout(const moe_shape& s);

// ---- moe_api.cu ----
// The shape rules every entry point applies (MOE_ERR_INVALID_ARG or
// MOE_ERR_UNSUPPORTED before anything is enqueued).
moe_status check_shape(const moe_shape* s);

// ---- router.cu ----
int router_splits_for(const moe_shape& s);
cudaError_t launch_router_gemv(const moe_shape& s, const void* x, const void* w_g, float* part,
                               int splits, cudaStream_t st);
// a few tokens: GEMV and top-K in one launch (ticket: a zeroed counter)
bool fused_router_enabled();
bool router_fused_possible(const moe_shape& s);
cudaError_t launch_router_fused(const moe_shape& s, const void* x, const void* w_g, float* part,
                                int splits, const float* bias, float* logits_out,
                                int32_t* topk_idx, float* topk_w, unsigned int* ticket,
                                cudaStream_t st);
cudaError_t launch_topk_softmax(const moe_shape& s, const float* part, int splits,
                                const float* bias, float* logits_out, int32_t* topk_idx,
                                float* topk_w, cudaStream_t st);

// ---- dispatch.cu ----
int dispatch_blocks_for(int64_t n_slots);
cudaError_t launch_dispatch(const moe_shape& s, const int32_t* topk_idx, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* tok_of,
                            int32_t* blk_hist, DevError* err, cudaStream_t st);
cudaError_t launch_gather_rows(const moe_shape& s, const void* x, const int32_t* inv_perm,
                               void* x_perm, cudaStream_t st);
// E4M3 rows xq [T][d] and their scales sx [T] into expert order (d bytes per row)
cudaError_t launch_gather_codes(const moe_shape& s, const uint8_t* xq, const float* sx,
                                const int32_t* inv_perm, uint8_t* xq_perm, float* s_perm,
                                cudaStream_t st);

// ---- ffn_plan + ffn_gemv.cu ----
int gemv_max_rows();  // groups with at most this many rows take the GEMV path
// gemv_list holds 2 * (E + 1) entries: groups of 1..small_rows rows (all GEMV
// groups when small_rows is 0), then from entry E + 1 on the groups of
// small_rows + 1 .. gemv_limit rows.  mtile_list holds 2 * max_mtiles
// entries: single-SM tiles, then pair tiles (none when allow_pair is false).
cudaError_t launch_ffn_plan(const FfnGroups& g, int dtype, FfnPlanHeader* hdr,
                            int32_t* gemv_list, int4* mtile_list, int max_mtiles,
                            int gemv_limit, bool allow_pair, int small_rows, cudaStream_t st);
cudaError_t launch_ffn_gemv(const FfnGroups& g, int dtype, const FfnPlanHeader* hdr,
                            const int32_t* gemv_list, cudaStream_t st);
// Small batches (T*K <= 1024 slots, E <= 1024): the three dispatch kernels
// and the plan as one single-block launch with identical results
// (MOE_FUSED_DISPATCH=0, read per call, keeps the separate launches).
bool dispatch_plan_fusable(const moe_shape& s);
cudaError_t launch_dispatch_plan_small(const moe_shape& s, const int32_t* topk_idx, int32_t* counts,
                                       int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                       int32_t* tok_of, DevError* err, const FfnGroups& g,
                                       FfnPlanHeader* hdr, int32_t* gemv_list, int4* mtile_list,
                                       int max_mtiles, int gemv_limit, bool allow_pair,
                                       int small_rows, cudaStream_t st);

// ---- ffn_tc.cu (tcgen05 grouped GEMM) ----
bool tc_available();
int tc_tile_rows(bool pair);  // rows per tensor-core m-tile (single-SM or CTA pair)
int tc_pair_min_rows();       // fixed pair threshold (0: the plan picks the cheaper shape)
int tc_split_rho();          // > 0: the two tile shapes run side by side (plan's SM split cost)
bool tc_pair_possible(int64_t max_rows);  // a group of at most max_rows rows may take pair tiles
// per-CTA routed row blocks up to this size are gathered from x (batch of T tokens)
int tc_gather_max_rows(int64_t T);
// The combine fused into the shared expert's down projection (launch_ffn_tc
// with a shared group): each token's routed rows and weights, and the output.
struct CombineArgs {
    const int32_t* inv_perm;  // [T*K] routed row of each slot (< 0: dropped)
    const float* topk_w;      // [T*K]
    int K;
    void* y;                  // [T][d] layer output (bf16)
};
bool fused_combine_enabled();  // MOE_FUSED_COMBINE (read per call)
// may_pair: some group can reach tc_pair_min_rows() rows (else the pair
// launches are skipped).  cmb (with a shared group): the routed down launches
// skip the shared group, whose down projection then runs as one dense launch
// that also sums the routed rows into y -- no separate combine.
// shared_apart: the shared expert ran in launch_shared_apart's launches, and
// the grouped launches skip its group.
cudaError_t launch_ffn_tc(const FfnGroups& g, const FfnPlanHeader* hdr, const int4* mtile_list,
                          int max_mtiles, bool may_pair, DevError* err, cudaStream_t st,
                          const CombineArgs* cmb = nullptr, bool shared_apart = false);
// The shared expert of a batch of at most shared_apart_max_tokens() tokens in
// its own two launches on a side stream forked off st (true: enqueued, *status
// tells whether it worked; false: nothing enqueued); join_shared_apart makes
// st wait for it.
int shared_apart_max_tokens();
bool launch_shared_apart(const FfnGroups& g, DevError* err, cudaStream_t st, cudaError_t* status);
cudaError_t join_shared_apart(cudaStream_t st);
cudaError_t launch_router_tc(const moe_shape& s, const void* x, const void* w_g, float* scores,
                             DevError* err, cudaStream_t st);
// E4M3 expert weights with row scales (g.s_* set); bf16 activations; the
// plan's pair tiles (launched only when may_pair) and single-SM tiles
cudaError_t launch_ffn_tc_fp8(const FfnGroups& g, const FfnPlanHeader* hdr, const int4* mtile_list,
                              int max_mtiles, bool may_pair, DevError* err, cudaStream_t st);

// E4M3 weights and activations (kind::f8f6f4), the two GEMMs launched
// separately so the caller can quantise h in between
cudaError_t launch_ffn_tc_a8_gate_up(const FfnGroups& g, const FfnPlanHeader* hdr,
                                     const int4* mtile_list, int max_mtiles, bool may_pair,
                                     DevError* err, cudaStream_t st, int planes = 1);
cudaError_t launch_ffn_tc_a8_down(const FfnGroups& g, const FfnPlanHeader* hdr,
                                  const int4* mtile_list, int max_mtiles, bool may_pair,
                                  DevError* err, cudaStream_t st, int planes = 1);

// ---- ffn_gemv_fp8.cu (E4M3 weights, small groups) ----
int gemv8_max_rows();  // groups with at most this many rows take the 8-bit GEMV
bool gemv8_fits(int widest);  // its staged activation rows of this width fit in shared memory
int gemv8_small_rows();       // groups up to this size go to the first GEMV list
constexpr size_t kGemv8SmemLimit = 232448;
// both GEMV lists of the plan (limit: the plan's GEMV row limit)
cudaError_t launch_ffn_gemv_fp8(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list,
                                int limit, cudaStream_t st);

// ---- quant.cu ----
cudaError_t launch_quantize_fp8_rows(int64_t rows, int64_t cols, int dtype, const void* w,
                                     uint8_t* codes, float* scales, cudaStream_t st);
// one scale per 128 x 128 block: scales [ceil(rows/128)][ceil(cols/128)]
cudaError_t launch_quantize_fp8_blocks(int64_t rows, int64_t cols, int dtype, const void* w,
                                       uint8_t* codes, float* scales, cudaStream_t st);
// bf16 activation rows (cols <= 16384): row r read at w + r * ld_in elements,
// its codes written at codes + r * ld_out bytes (may be the row's own storage)
cudaError_t launch_quantize_act_rows(int64_t rows, int cols, const void* w, int64_t ld_in,
                                     uint8_t* codes, int64_t ld_out, float* scales,
                                     cudaStream_t st);
// The same quantisation with each row's max |value| already known: amax_scale[r]
// holds it as fp32 bits on entry and the row's scale on return.  One warp per
// row, walking it from low to high addresses, so codes may overwrite the row.
// Two E4M3 planes per value (a code and the code of its fp32 remainder),
// interleaved per 128-value block: [128 hi | 128 lo] bytes; cols a multiple
// of 128.  x rows to a separate buffer (ld_out bytes apart, 2 * cols used), or
// rows whose max |value| is known split in place (amax_scale: the max as fp32
// bits in, the row scale out).
cudaError_t launch_split_act_rows(int64_t rows, int cols, const void* w, int64_t ld_in,
                                  uint8_t* codes, int64_t ld_out, float* scales, cudaStream_t st);
cudaError_t launch_split_rows_known_amax(int64_t rows, int cols, void* w, int64_t ld,
                                         float* amax_scale, cudaStream_t st);
cudaError_t launch_quantize_rows_known_amax(int64_t rows, int cols, const void* w, int64_t ld_in,
                                            uint8_t* codes, int64_t ld_out, float* amax_scale,
                                            cudaStream_t st);

// ---- combine.cu ----
cudaError_t launch_combine(const moe_shape& s, const void* y_perm, const int32_t* inv_perm,
                           const float* topk_w, const void* y_shared, void* y, cudaStream_t st);

int device_sm_count();

// Launches with programmatic stream serialisation (MOE_PDL=0 turns it off, read
// per call): the kernel may start while the previous kernel of the stream
// finishes, and orders itself with pdl_wait().
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
