// moe_api.cu -- the C ABI declared in include/moe.h: argument checks,
// workspace carving and the launch sequence of each stage.  Host code only;
// the kernels live in router.cu, dispatch.cu, ffn_gemv.cu, ffn_tc.cu and
// combine.cu.  No entry point allocates, frees or synchronises (except
// moe_get_device_error, which is documented as synchronous).
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {

// The shape rules every entry point applies before it enqueues anything.
moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->d <= 0 || s->E <= 0 || s->K <= 0 || s->inter <= 0 || s->inter_shared < 0)
        return MOE_ERR_INVALID_ARG;
    if (s->K > s->E) return MOE_ERR_INVALID_ARG;
    if (s->dtype != MOE_F32 && s->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (s->router != MOE_ROUTER_SOFTMAX && s->router != MOE_ROUTER_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (s->K > 32 || s->E > 1024) return MOE_ERR_UNSUPPORTED;
    if (s->d % 64 || s->inter % 64 || s->inter_shared % 64) return MOE_ERR_UNSUPPORTED;
    if (s->d > 16384 || s->inter > 16384 || s->inter_shared > 16384) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s->T * s->K >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t esize(const moe_shape& s) { return s.dtype == MOE_BF16 ? 2 : 4; }

moe_status check_ws(const moe_shape& s, const void* ws, size_t bytes) {
    if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    if (bytes < ws_layout(s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

// Groups whose row count exceeds this take the tensor-core path.
int gemv_limit() { return gemv_max_rows(); }

// The GEMV kernels can get work only for fp32 layers or with a non-zero row limit.
bool gemv_possible(const moe_shape& s) { return s.dtype == MOE_F32 || gemv_limit() > 0; }

bool use_tc_router(const moe_shape& s) {
    return s.dtype == MOE_BF16 && s.T >= 128 && s.E >= 64;
}

// The workspace's error block: the device error record at its start, the fused
// router's ticket counter at kRouteTicket; every entry point clears the whole
// block before it enqueues work.
constexpr size_t kErrBlockBytes = 256;
constexpr size_t kRouteTicket = 128;
static_assert(sizeof(DevError) <= kRouteTicket, "error record and ticket overlap");

unsigned int* route_ticket(void* workspace, const WsLayout& L) {
    return reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + L.err + kRouteTicket);
}

// Stage 1 from x into topk_idx / topk_w (and the selection keys into
// logits_out when given): the tensor-core GEMM for large bf16 batches, one
// fused GEMV + top-K launch for a few tokens, else the split-K GEMV and then
// the top-K.  The error block must have been cleared on the stream.
cudaError_t launch_route(const moe_shape& s, const WsLayout& L, void* workspace, const void* x,
                         const void* w_g, const float* bias, float* logits_out, int32_t* topk_idx,
                         float* topk_w, DevError* err, cudaStream_t cs) {
    float* part = at<float>(workspace, L.router_part);
    int splits = L.router_splits;
    cudaError_t e;
    if (use_tc_router(s) && tc_available()) {
        e = launch_router_tc(s, x, w_g, part, err, cs);
        splits = 1;
    } else if (router_fused_possible(s)) {
        return launch_router_fused(s, x, w_g, part, splits, bias, logits_out, topk_idx, topk_w,
                                   route_ticket(workspace, L), cs);
    } else {
        e = launch_router_gemv(s, x, w_g, part, splits, cs);
    }
    if (e != cudaSuccess) return e;
    return launch_topk_softmax(s, part, splits, bias, logits_out, topk_idx, topk_w, cs);
}

// 8-bit weights: bf16 activations, K extents that whole 128-code boxes tile
moe_status check_fp8_shape(const moe_shape& s) {
    if (s.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (s.d % 128 || s.inter % 128 || s.inter_shared % 128) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Groups with at most this many rows take the 8-bit GEMV (0 when its staged
// activation rows would not fit in shared memory).  With row scales the GEMV
// serves only calls whose groups are all small (max_rows, the bound on any
// group, at most kGemv8MaxGroupBound): once some group can be large the
// tensor-core tiles run anyway, the small groups among them run swapped there,
// and the GEMV's own launches cost more than they save (measured on GB300,
// E4M3-weight DeepSeek-V3 T=512: 2063 us with the GEMV for groups of <= 8 rows,
// 1998 us without; T=64, every group small: 1614 us with it, 1646 without).
// MOE_GEMV8_MAX_ROWS, when set, applies to every call.
constexpr int64_t kGemv8MaxGroupBound = 64;
int gemv8_limit(const moe_shape& s, int64_t max_rows = 0, int wblock = 0) {
    const int widest = std::max(s.d, std::max(s.inter, s.inter_shared));
    if (!gemv8_fits(widest)) return 0;
    if (wblock == 0 && max_rows > kGemv8MaxGroupBound && getenv("MOE_GEMV8_MAX_ROWS") == nullptr)
        return 0;
    return gemv8_max_rows();
}

// 8-bit weights on CTA-pair tiles (MOE_W8_PAIR=1, read per call; default off).
// Measured on GB300: the pair variant (each CTA widens half of the n-block's
// weight rows) is slower than single-SM tiles on prefill shapes (Mixtral:
// 5.3 ms vs 3.65 ms), its handoffs crossing the cluster; it stays selectable
// and parity-tested.
bool w8_pair() {
    const char* e = getenv("MOE_W8_PAIR");
    return e && e[0] == '1';
}

// Whether the plan may give 8-bit-weight groups CTA-pair tiles: with 8-bit
// activations (two planes, or W8A8) and row scales, yes; with the codes widened
// in the GEMM, or with block scales, only when MOE_W8_PAIR=1.  Measured on GB300 (block scales,
// Mixtral-shaped stage on a 4-expert pool): 1.72 ms on pair tiles, 1.13 ms on
// single-SM tiles (row scales: 0.95 ms) -- per 128-deep K block the pair's MMA
// issuer waited ~1600 cycles for the peer CTA to release the accumulator,
// against ~400 on single tiles.
bool w8_pair_tiles(bool planes, int wblock) {
    if (wblock) return w8_pair();
    return planes || w8_pair();
}

// Tensor-core groups of the 8-bit-weight entry points carry their bf16
// activations as two E4M3 planes on the 8-bit-by-8-bit MMA (MOE_W8_PLANES,
// read per call; 0 widens the codes to bf16 inside the GEMM instead).
bool w8_planes() {
    const char* e = getenv("MOE_W8_PLANES");
    return !(e && e[0] == '0');
}

// routed code and scale pointers present and aligned; shared ones iff wanted
moe_status check_fp8_weights(const moe_fp8_experts* w, bool shared) {
    if (!w) return MOE_ERR_INVALID_ARG;
    const void* routed[] = {w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down};
    for (const void* p : routed)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!shared) return MOE_OK;
    const void* sh[] = {w->ws_gate, w->ws_up, w->ws_down, w->ss_gate, w->ss_up, w->ss_down};
    for (const void* p : sh)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

bool pdl_enabled() {
    const char* e = getenv("MOE_PDL");
    return !(e && e[0] == '0');
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev >= kMaxDevices) {
        int n = 1;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

WsLayout ws_layout(const moe_shape& s) {
    WsLayout L{};
    const int64_t T = s.T, E = s.E, K = s.K, d = s.d, I = s.inter, Is = s.inter_shared;
    const int64_t n = T * K;
    const size_t es = esize(s);
    L.router_splits = router_splits_for(s);
    L.dispatch_blocks = dispatch_blocks_for(n);
    L.max_mtiles = (int)(n / 128 + E + T / 128 + 2);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at_ = o;
        o = align_up(o + (bytes ? bytes : 1));
        return at_;
    };
    L.err = take(kErrBlockBytes);
    L.router_part = take(sizeof(float) * (size_t)(L.router_splits > 1 ? L.router_splits : 1) * T * E);
    L.logits = 0;
    L.topk_idx = take(sizeof(int32_t) * n);
    L.topk_w = take(sizeof(float) * n);
    L.counts = take(sizeof(int32_t) * (E + 1));
    L.offsets = take(sizeof(int32_t) * (E + 2));
    L.perm = take(sizeof(int32_t) * n);
    L.inv_perm = take(sizeof(int32_t) * n);
    L.tok_of = take(sizeof(int32_t) * n);
    L.blk_hist = take(sizeof(int32_t) * (size_t)L.dispatch_blocks * E);
    L.plan = take(sizeof(FfnPlanHeader));
    L.gemv_list = take(sizeof(int32_t) * 2 * (E + 1));  // two GEMV lists
    L.mtile_list = take(sizeof(int4) * 2 * (size_t)L.max_mtiles);  // single, then pair tiles
    L.x_perm = take(es * n * d);
    L.h = take(es * n * I);
    L.h_s = take(es * T * Is);
    L.y_perm = take(es * n * d);
    L.y_s = take(es * T * d);
    // 8-bit activations: row scales of x [T], x_perm [T*K], h [T*K], h_s [T]
    L.ascale = take(sizeof(float) * (size_t)(2 * T + 2 * n));
    L.total = o;
    return L;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int32_t status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_BOUNDS: return "index out of range on the device";
        default: return "unknown status";
    }
}

size_t moe_workspace_bytes(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    return ws_layout(*shape).total;
}

moe_status moe_route(const moe_shape* shape, const void* x, const void* w_g, const float* bias,
                     const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w,
                     void* workspace, size_t ws_bytes, void* stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (s.T == 0) return MOE_OK;
    if (!topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!logits_in && (!x || !w_g)) return MOE_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (w_g && !aligned16(w_g))) return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (logits_in)
        return cuda_status(launch_topk_softmax(s, logits_in, 1, bias, logits_out, topk_idx, topk_w, cs));
    return cuda_status(launch_route(s, L, workspace, x, w_g, bias, logits_out, topk_idx, topk_w,
                                    err, cs));
}

moe_status moe_permute(const moe_shape* shape, const int32_t* topk_idx, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                       void* x_perm, void* workspace, size_t ws_bytes, void* stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!counts || !offsets || (s.T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (s.T == 0) {
        // no slots: every count is zero and every offset is zero
        e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (s.E + 1), cs);
        return cuda_status(e);
    }
    int32_t* inv = inv_perm ? inv_perm : at<int32_t>(workspace, L.inv_perm);
    int32_t* tok = at<int32_t>(workspace, L.tok_of);
    e = launch_dispatch(s, topk_idx, counts, offsets, perm, inv, tok, at<int32_t>(workspace, L.blk_hist),
                        err, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (x && x_perm) e = launch_gather_rows(s, x, inv, x_perm, cs);
    return cuda_status(e);
}

moe_status moe_expert_ffn(const moe_shape* shape, const void* x_perm, const int32_t* offsets,
                          const void* w_gate, const void* w_up, const void* w_down, void* y_perm,
                          void* workspace, size_t ws_bytes, void* stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (s.T == 0) return MOE_OK;
    if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    const int64_t rows = (int64_t)s.T * s.K;
    const bool need_tc = s.dtype == MOE_BF16 && rows > gemv_limit();
    if (need_tc && !tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = 0;
    g.n_routed_rows = (int)rows;
    g.T = s.T;
    g.max_group_rows = (int)rows;
    g.offsets = offsets;
    g.row_src = nullptr;
    g.a_routed = x_perm;
    g.a_perm = x_perm;
    g.a_shared = x_perm;
    g.w_gate = w_gate;
    g.w_up = w_up;
    g.w_down = w_down;
    g.h = at<void>(workspace, L.h);
    g.h_s = nullptr;
    g.y = y_perm;
    g.y_s = nullptr;
    FfnPlanHeader* hdr = at<FfnPlanHeader>(workspace, L.plan);
    int32_t* glist = at<int32_t>(workspace, L.gemv_list);
    int4* mtiles = at<int4>(workspace, L.mtile_list);
    e = launch_ffn_plan(g, s.dtype, hdr, glist, mtiles, L.max_mtiles, gemv_limit(), true, 0, cs);
    if (e == cudaSuccess && gemv_possible(s)) e = launch_ffn_gemv(g, s.dtype, hdr, glist, cs);
    if (e == cudaSuccess && need_tc)
        e = launch_ffn_tc(g, hdr, mtiles, L.max_mtiles, tc_pair_possible(rows), err, cs);
    return cuda_status(e);
}

moe_status moe_combine(const moe_shape* shape, const void* y_perm, const int32_t* inv_perm,
                       const float* topk_w, const void* y_shared, void* y, void* stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (s.T == 0) return MOE_OK;
    if (!y_perm || !inv_perm || !topk_w || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm) || !aligned16(y) || (y_shared && !aligned16(y_shared)))
        return MOE_ERR_INVALID_ARG;
    if (s.T == 0) return MOE_OK;
    return cuda_status(launch_combine(s, y_perm, inv_perm, topk_w, y_shared, y, (cudaStream_t)stream));
}

moe_status moe_forward(const moe_shape* shape, const void* x, const void* w_g, const float* bias,
                       const void* w_gate, const void* w_up, const void* w_down,
                       const void* ws_gate, const void* ws_up, const void* ws_down, void* y,
                       void* workspace, size_t ws_bytes, void* stream) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const bool shared = s.inter_shared > 0;
    if (s.T == 0) return MOE_OK;
    if (!x || !w_g || !w_gate || !w_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (shared != (ws_gate && ws_up && ws_down)) return MOE_ERR_INVALID_ARG;
    if (shared && (ws_gate == nullptr || ws_up == nullptr || ws_down == nullptr)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w_g, w_gate, w_up, w_down, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (shared && (!aligned16(ws_gate) || !aligned16(ws_up) || !aligned16(ws_down)))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    const bool need_tc = s.dtype == MOE_BF16 && s.T > gemv_limit();
    if (need_tc && !tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 0. small batches: the shared expert (it reads only x) starts on a side
    //    stream, beside the routing and dispatch below
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = shared ? 1 : 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = s.inter_shared;
    g.T = s.T;
    g.a_shared = x;
    g.ws_gate = ws_gate;
    g.ws_up = ws_up;
    g.ws_down = ws_down;
    g.h_s = at<void>(workspace, L.h_s);
    g.y_s = at<void>(workspace, L.y_s);
    bool apart = false;
    if (need_tc && shared && !gemv_possible(s) && s.T <= shared_apart_max_tokens() &&
        !tc_pair_possible(s.T)) {
        apart = launch_shared_apart(g, err, cs, &e);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }

    // 1. router scores, top-K, softmax over the K
    int32_t* topk_idx = at<int32_t>(workspace, L.topk_idx);
    float* topk_w = at<float>(workspace, L.topk_w);
    e = launch_route(s, L, workspace, x, w_g, bias, nullptr, topk_idx, topk_w, err, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 2. dispatch (and, for small batches, the expert plan in the same launch)
    int32_t* counts = at<int32_t>(workspace, L.counts);
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv_perm);
    int32_t* tok = at<int32_t>(workspace, L.tok_of);
    // Both expert paths read routed rows from x through the row -> token map
    // (the tensor-core path with TMA gather4 for row blocks of at most
    // tc_gather_max_rows(T) rows).  Larger blocks need the contiguous permuted
    // copy, which is only built when a group can be that large (a group has at
    // most T rows: a token picks an expert once).
    void* x_perm = (need_tc && s.T > tc_gather_max_rows(s.T)) ? at<void>(workspace, L.x_perm) : nullptr;
    g.n_routed_rows = s.T * s.K;
    g.max_group_rows = s.T;  // a token picks an expert once; the shared group has T rows
    g.offsets = offsets;
    g.row_src = tok;
    g.a_routed = x;
    g.a_perm = x_perm;
    g.w_gate = w_gate;
    g.w_up = w_up;
    g.w_down = w_down;
    g.h = at<void>(workspace, L.h);
    g.y = at<void>(workspace, L.y_perm);
    FfnPlanHeader* hdr = at<FfnPlanHeader>(workspace, L.plan);
    int32_t* glist = at<int32_t>(workspace, L.gemv_list);
    int4* mtiles = at<int4>(workspace, L.mtile_list);
    int32_t* perm = at<int32_t>(workspace, L.perm);
    const bool fused = dispatch_plan_fusable(s);
    if (fused)
        e = launch_dispatch_plan_small(s, topk_idx, counts, offsets, perm, inv, tok, err, g, hdr,
                                       glist, mtiles, L.max_mtiles, gemv_limit(), true, 0, cs);
    else
        e = launch_dispatch(s, topk_idx, counts, offsets, perm, inv, tok,
                            at<int32_t>(workspace, L.blk_hist), err, cs);
    if (e == cudaSuccess && x_perm) e = launch_gather_rows(s, x, inv, x_perm, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 3. routed experts and the shared expert
    if (!fused)
        e = launch_ffn_plan(g, s.dtype, hdr, glist, mtiles, L.max_mtiles, gemv_limit(), true, 0, cs);
    if (e == cudaSuccess && gemv_possible(s)) e = launch_ffn_gemv(g, s.dtype, hdr, glist, cs);
    // 4. combine: with a shared expert on the tensor-core path, fused into the
    //    shared expert's down projection (its epilogue sums the routed rows)
    const bool fuse = need_tc && shared && !gemv_possible(s) && fused_combine_enabled();
    const CombineArgs cmb{inv, topk_w, s.K, y};
    // a group has at most T rows (a token picks an expert once)
    if (e == cudaSuccess && need_tc)
        e = launch_ffn_tc(g, hdr, mtiles, L.max_mtiles, tc_pair_possible(s.T), err, cs,
                          fuse && !apart ? &cmb : nullptr, apart);
    if (e == cudaSuccess && apart) e = join_shared_apart(cs);  // y_s is ready
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (fuse && !apart) return MOE_OK;
    return cuda_status(launch_combine(s, g.y, inv, topk_w, shared ? g.y_s : nullptr, y, cs));
}

moe_status moe_quantize_fp8_rows(int64_t rows, int64_t cols, int32_t dtype, const void* w,
                                 uint8_t* codes, float* scales, void* stream) {
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (rows >= ((int64_t)1 << 31) || cols % 16) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!w || !codes || !scales || !aligned16(w) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_fp8_rows(rows, cols, dtype, w, codes, scales,
                                                (cudaStream_t)stream));
}

moe_status moe_quantize_fp8_blocks(int64_t rows, int64_t cols, int32_t dtype, const void* w,
                                   uint8_t* codes, float* scales, void* stream) {
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    // the block grid: ceil(cols / 128) x ceil(rows / 128) thread blocks
    if ((rows + kWBlock - 1) / kWBlock > 65535 || cols % 16 || cols >= ((int64_t)1 << 31))
        return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!w || !codes || !scales || !aligned16(w) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_fp8_blocks(rows, cols, dtype, w, codes, scales,
                                                  (cudaStream_t)stream));
}

// The tensor-core groups of an 8-bit-weight call with two-plane activations:
// g.a_perm / g.a_shared hold the planes of the routed / shared rows and
// g.sa_routed / g.sa_shared their scales; the plan is built.  Gate/up GEMM
// (bf16 h, each row's max |h| raised from zero), h split into two planes in
// place, down GEMM.  Groups on the 8-bit GEMV have run before (their bf16 h
// rows, already consumed, are split along with the rest and never read).
static cudaError_t run_tc_planes(const moe_shape& s, FfnGroups& g, const WsLayout& L, void* ws,
                                 int64_t max_rows, bool pair, DevError* err, cudaStream_t cs) {
    FfnPlanHeader* hdr = at<FfnPlanHeader>(ws, L.plan);
    int4* mtiles = at<int4>(ws, L.mtile_list);
    const int64_t R = (int64_t)s.T * s.K;
    const bool may_pair = pair && tc_pair_possible(max_rows);
    cudaError_t e = cudaMemsetAsync(const_cast<float*>(g.sa_h), 0, sizeof(float) * R, cs);
    if (e == cudaSuccess && g.has_shared)
        e = cudaMemsetAsync(const_cast<float*>(g.sa_hs), 0, sizeof(float) * s.T, cs);
    if (e == cudaSuccess)
        e = launch_ffn_tc_a8_gate_up(g, hdr, mtiles, L.max_mtiles, may_pair, err, cs, 2);
    if (e == cudaSuccess)
        e = launch_split_rows_known_amax(R, s.inter, g.h, s.inter, const_cast<float*>(g.sa_h), cs);
    if (e == cudaSuccess && g.has_shared)
        e = launch_split_rows_known_amax(s.T, s.inter_shared, g.h_s, s.inter_shared,
                                         const_cast<float*>(g.sa_hs), cs);
    if (e == cudaSuccess)
        e = launch_ffn_tc_a8_down(g, hdr, mtiles, L.max_mtiles, may_pair, err, cs, 2);
    return e;
}

// moe_expert_ffn_fp8 (wblock = 0: row scales) and moe_expert_ffn_fp8_blocks
// (wblock = kWBlock: 128 x 128 block scales, whose tensor-core groups always
// take the two-plane path).
static moe_status expert_ffn_fp8_call(const moe_shape* shape, const void* x_perm,
                                      const int32_t* offsets, const moe_fp8_experts* w,
                                      void* y_perm, void* workspace, size_t ws_bytes, void* stream,
                                      int wblock) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_fp8_shape(s)) != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    if (!x_perm || !offsets || !y_perm || !aligned16(x_perm) || !aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_fp8_weights(w, false)) != MOE_OK) return st;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (!tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = 0;
    g.n_routed_rows = s.T * s.K;
    g.T = s.T;
    g.offsets = offsets;
    g.row_src = nullptr;
    g.a_routed = x_perm;
    g.a_perm = x_perm;
    g.a_shared = x_perm;
    g.w_gate = w->w_gate;
    g.w_up = w->w_up;
    g.w_down = w->w_down;
    g.s_gate = w->s_gate;
    g.s_up = w->s_up;
    g.s_down = w->s_down;
    g.wblock = wblock;
    g.max_group_rows = s.T * s.K;  // the offsets are the caller's
    g.h = at<void>(workspace, L.h);
    g.y = y_perm;
    FfnPlanHeader* hdr = at<FfnPlanHeader>(workspace, L.plan);
    int32_t* glist = at<int32_t>(workspace, L.gemv_list);
    int4* mtiles = at<int4>(workspace, L.mtile_list);
    const int64_t R = (int64_t)s.T * s.K;
    // a group has at most T*K rows here (the offsets are the caller's)
    const int lim = gemv8_limit(s, R, wblock);
    const bool planes = R > lim && (w8_planes() || wblock != 0);
    const bool pair = w8_pair_tiles(planes, wblock);
    if (planes) {
        // the rows' two planes (2d codes per row) and their scales
        float* sc = at<float>(workspace, L.ascale);
        g.a_perm = at<uint8_t>(workspace, L.x_perm);
        g.sa_routed = sc + s.T;
        g.sa_h = sc + s.T + R;
        e = launch_split_act_rows(R, s.d, x_perm, s.d, at<uint8_t>(workspace, L.x_perm),
                                  2 * (int64_t)s.d, sc + s.T, cs);
    }
    if (e == cudaSuccess)
        e = launch_ffn_plan(g, s.dtype, hdr, glist, mtiles, L.max_mtiles, lim, pair,
                            gemv8_small_rows(), cs);
    if (e == cudaSuccess && lim > 0) e = launch_ffn_gemv_fp8(g, hdr, glist, lim, cs);
    if (e == cudaSuccess && R > lim) {
        if (planes) e = run_tc_planes(s, g, L, workspace, R, pair, err, cs);
        else e = launch_ffn_tc_fp8(g, hdr, mtiles, L.max_mtiles, pair && tc_pair_possible(R), err, cs);
    }
    return cuda_status(e);
}

moe_status moe_expert_ffn_fp8(const moe_shape* shape, const void* x_perm, const int32_t* offsets,
                              const moe_fp8_experts* w, void* y_perm, void* workspace,
                              size_t ws_bytes, void* stream) {
    return expert_ffn_fp8_call(shape, x_perm, offsets, w, y_perm, workspace, ws_bytes, stream, 0);
}

moe_status moe_expert_ffn_fp8_blocks(const moe_shape* shape, const void* x_perm,
                                     const int32_t* offsets, const moe_fp8_experts* w,
                                     void* y_perm, void* workspace, size_t ws_bytes,
                                     void* stream) {
    return expert_ffn_fp8_call(shape, x_perm, offsets, w, y_perm, workspace, ws_bytes, stream,
                               kWBlock);
}

// moe_forward_fp8 (wblock = 0) and moe_forward_fp8_blocks (wblock = kWBlock).
static moe_status forward_fp8_call(const moe_shape* shape, const void* x, const void* w_g,
                                   const float* bias, const moe_fp8_experts* w, void* y,
                                   void* workspace, size_t ws_bytes, void* stream, int wblock) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_fp8_shape(s)) != MOE_OK) return st;
    const bool shared = s.inter_shared > 0;
    if (s.T == 0) return MOE_OK;
    if (!x || !w_g || !y || !aligned16(x) || !aligned16(w_g) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_fp8_weights(w, shared)) != MOE_OK) return st;
    if (!shared && w->ws_gate) return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (!tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 1. router (bf16 weights), top-K and weights
    int32_t* topk_idx = at<int32_t>(workspace, L.topk_idx);
    float* topk_w = at<float>(workspace, L.topk_w);
    e = launch_route(s, L, workspace, x, w_g, bias, nullptr, topk_idx, topk_w, err, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 2. dispatch (for small batches with the expert plan) and the permuted
    //    copy of the routed rows
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv_perm);
    int32_t* tok = at<int32_t>(workspace, L.tok_of);
    void* x_perm = at<void>(workspace, L.x_perm);
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = shared ? 1 : 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = s.inter_shared;
    g.n_routed_rows = s.T * s.K;
    g.T = s.T;
    g.offsets = offsets;
    g.row_src = nullptr;
    g.a_routed = x_perm;
    g.a_perm = x_perm;
    g.a_shared = x;
    g.w_gate = w->w_gate;
    g.w_up = w->w_up;
    g.w_down = w->w_down;
    g.s_gate = w->s_gate;
    g.s_up = w->s_up;
    g.s_down = w->s_down;
    g.ws_gate = w->ws_gate;
    g.ws_up = w->ws_up;
    g.ws_down = w->ws_down;
    g.ss_gate = w->ss_gate;
    g.ss_up = w->ss_up;
    g.ss_down = w->ss_down;
    g.wblock = wblock;
    g.max_group_rows = s.T;  // a token picks an expert once; the shared group has T rows
    g.h = at<void>(workspace, L.h);
    g.h_s = at<void>(workspace, L.h_s);
    g.y = at<void>(workspace, L.y_perm);
    g.y_s = at<void>(workspace, L.y_s);
    FfnPlanHeader* hdr = at<FfnPlanHeader>(workspace, L.plan);
    int32_t* glist = at<int32_t>(workspace, L.gemv_list);
    int4* mtiles = at<int4>(workspace, L.mtile_list);
    // a group has at most T rows (a token picks an expert once; the shared group has T)
    const int lim = gemv8_limit(s, s.T, wblock);
    const bool planes = s.T > lim && (w8_planes() || wblock != 0);
    const bool pair = w8_pair_tiles(planes, wblock);
    const int64_t R = (int64_t)s.T * s.K;
    float* sc = at<float>(workspace, L.ascale);
    uint8_t* xq = at<uint8_t>(workspace, L.y_s);  // x planes [T][2d], read before y_s is written
    if (planes) {
        // tensor-core groups read two-plane rows (routed: gathered into expert
        // order; shared: the x planes); GEMV groups read x through the row map
        g.row_src = tok;
        g.a_routed = x;
        g.a_perm = x_perm;
        g.a_shared = xq;
        g.sa_routed = sc + s.T;
        g.sa_shared = sc;
        g.sa_h = sc + s.T + R;
        g.sa_hs = sc + s.T + 2 * R;
    }
    int32_t* counts = at<int32_t>(workspace, L.counts);
    int32_t* perm = at<int32_t>(workspace, L.perm);
    const bool fused = dispatch_plan_fusable(s);
    if (fused)
        e = launch_dispatch_plan_small(s, topk_idx, counts, offsets, perm, inv, tok, err, g, hdr,
                                       glist, mtiles, L.max_mtiles, lim, pair, gemv8_small_rows(),
                                       cs);
    else
        e = launch_dispatch(s, topk_idx, counts, offsets, perm, inv, tok,
                            at<int32_t>(workspace, L.blk_hist), err, cs);
    if (e == cudaSuccess && !planes) e = launch_gather_rows(s, x, inv, x_perm, cs);
    if (e == cudaSuccess && planes) {
        moe_shape s2 = s;  // rows of 2d bytes: the two planes
        s2.d = 2 * s.d;
        e = launch_split_act_rows(s.T, s.d, x, s.d, xq, 2 * (int64_t)s.d, sc, cs);
        if (e == cudaSuccess)
            e = launch_gather_codes(s2, xq, sc, inv, (uint8_t*)x_perm, sc + s.T, cs);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 3. routed and shared experts, 8-bit weights: the 8-bit GEMV for small
    //    groups, tensor-core tiles for the rest
    if (!fused)
        e = launch_ffn_plan(g, s.dtype, hdr, glist, mtiles, L.max_mtiles, lim, pair,
                            gemv8_small_rows(), cs);
    if (e == cudaSuccess && lim > 0) e = launch_ffn_gemv_fp8(g, hdr, glist, lim, cs);
    if (e == cudaSuccess && s.T > lim) {
        if (planes) e = run_tc_planes(s, g, L, workspace, s.T, pair, err, cs);
        else e = launch_ffn_tc_fp8(g, hdr, mtiles, L.max_mtiles, pair && tc_pair_possible(s.T), err, cs);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 4. combine
    return cuda_status(launch_combine(s, g.y, inv, topk_w, shared ? g.y_s : nullptr, y, cs));
}

moe_status moe_forward_fp8(const moe_shape* shape, const void* x, const void* w_g, const float* bias,
                           const moe_fp8_experts* w, void* y, void* workspace, size_t ws_bytes,
                           void* stream) {
    return forward_fp8_call(shape, x, w_g, bias, w, y, workspace, ws_bytes, stream, 0);
}

moe_status moe_forward_fp8_blocks(const moe_shape* shape, const void* x, const void* w_g,
                                  const float* bias, const moe_fp8_experts* w, void* y,
                                  void* workspace, size_t ws_bytes, void* stream) {
    return forward_fp8_call(shape, x, w_g, bias, w, y, workspace, ws_bytes, stream, kWBlock);
}

// W8A8 expert stage on groups g whose a_perm / a_shared already hold E4M3 rows
// and sa_routed / sa_shared their scales: gate/up GEMM (bf16 h), h quantised in
// place, down GEMM.  Every group runs on the tensor cores (no GEMV list);
// max_rows bounds the rows of any group (pair launches are skipped when no
// group can take pair tiles).
static cudaError_t run_ffn_w8a8(const moe_shape& s, FfnGroups& g, const WsLayout& L, void* ws,
                                int64_t max_rows, bool planned, bool pair, DevError* err,
                                cudaStream_t cs) {
    FfnPlanHeader* hdr = at<FfnPlanHeader>(ws, L.plan);
    int32_t* glist = at<int32_t>(ws, L.gemv_list);
    int4* mtiles = at<int4>(ws, L.mtile_list);
    const int64_t R = (int64_t)s.T * s.K;
    const bool may_pair = pair && tc_pair_possible(max_rows);
    // the gate/up epilogue raises each h row's max |h| from zero
    cudaError_t e = cudaMemsetAsync(const_cast<float*>(g.sa_h), 0, sizeof(float) * R, cs);
    if (e == cudaSuccess && g.has_shared)
        e = cudaMemsetAsync(const_cast<float*>(g.sa_hs), 0, sizeof(float) * s.T, cs);
    if (e == cudaSuccess && !planned)
        e = launch_ffn_plan(g, s.dtype, hdr, glist, mtiles, L.max_mtiles, 0, pair, 0, cs);
    if (e == cudaSuccess)
        e = launch_ffn_tc_a8_gate_up(g, hdr, mtiles, L.max_mtiles, may_pair, err, cs);
    if (e == cudaSuccess)
        e = launch_quantize_rows_known_amax(R, s.inter, g.h, s.inter, (uint8_t*)g.h,
                                            2 * (int64_t)s.inter, const_cast<float*>(g.sa_h), cs);
    if (e == cudaSuccess && g.has_shared)
        e = launch_quantize_rows_known_amax(s.T, s.inter_shared, g.h_s, s.inter_shared,
                                            (uint8_t*)g.h_s, 2 * (int64_t)s.inter_shared,
                                            const_cast<float*>(g.sa_hs), cs);
    if (e == cudaSuccess) e = launch_ffn_tc_a8_down(g, hdr, mtiles, L.max_mtiles, may_pair, err, cs);
    return e;
}

// moe_expert_ffn_w8a8 (wblock = 0: row scales) and moe_expert_ffn_w8a8_blocks
// (wblock = kWBlock: 128 x 128 block scales, single-SM tiles unless MOE_W8_PAIR=1).
static moe_status expert_ffn_w8a8_call(const moe_shape* shape, const void* x_perm,
                                       const int32_t* offsets, const moe_fp8_experts* w,
                                       void* y_perm, void* workspace, size_t ws_bytes,
                                       void* stream, int wblock) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_fp8_shape(s)) != MOE_OK) return st;
    if (s.T == 0) return MOE_OK;
    if (!x_perm || !offsets || !y_perm || !aligned16(x_perm) || !aligned16(y_perm))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_fp8_weights(w, false)) != MOE_OK) return st;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (!tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t R = (int64_t)s.T * s.K;
    float* sc = at<float>(workspace, L.ascale);
    uint8_t* xq = at<uint8_t>(workspace, L.x_perm);
    e = launch_quantize_act_rows(R, s.d, x_perm, s.d, xq, s.d, sc + s.T, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = 0;
    g.n_routed_rows = (int)R;
    g.T = s.T;
    g.max_group_rows = (int)R;
    g.offsets = offsets;
    g.row_src = nullptr;
    g.a_routed = xq;
    g.a_perm = xq;
    g.a_shared = xq;
    g.w_gate = w->w_gate;
    g.w_up = w->w_up;
    g.w_down = w->w_down;
    g.s_gate = w->s_gate;
    g.s_up = w->s_up;
    g.s_down = w->s_down;
    g.wblock = wblock;
    g.sa_routed = sc + s.T;
    g.sa_shared = sc + s.T;
    g.sa_h = sc + s.T + R;
    g.sa_hs = sc + s.T + R;
    g.h = at<void>(workspace, L.h);
    g.y = y_perm;
    // a group has at most T*K rows here (the offsets are the caller's)
    return cuda_status(run_ffn_w8a8(s, g, L, workspace, R, false, w8_pair_tiles(true, wblock), err,
                                    cs));
}

moe_status moe_expert_ffn_w8a8(const moe_shape* shape, const void* x_perm, const int32_t* offsets,
                               const moe_fp8_experts* w, void* y_perm, void* workspace,
                               size_t ws_bytes, void* stream) {
    return expert_ffn_w8a8_call(shape, x_perm, offsets, w, y_perm, workspace, ws_bytes, stream, 0);
}

moe_status moe_expert_ffn_w8a8_blocks(const moe_shape* shape, const void* x_perm,
                                      const int32_t* offsets, const moe_fp8_experts* w,
                                      void* y_perm, void* workspace, size_t ws_bytes,
                                      void* stream) {
    return expert_ffn_w8a8_call(shape, x_perm, offsets, w, y_perm, workspace, ws_bytes, stream,
                                kWBlock);
}

// moe_forward_w8a8 (wblock = 0) and moe_forward_w8a8_blocks (wblock = kWBlock).
static moe_status forward_w8a8_call(const moe_shape* shape, const void* x, const void* w_g,
                                    const float* bias, const moe_fp8_experts* w, void* y,
                                    void* workspace, size_t ws_bytes, void* stream, int wblock) {
    moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if ((st = check_fp8_shape(s)) != MOE_OK) return st;
    const bool shared = s.inter_shared > 0;
    if (s.T == 0) return MOE_OK;
    if (!x || !w_g || !y || !aligned16(x) || !aligned16(w_g) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if ((st = check_fp8_weights(w, shared)) != MOE_OK) return st;
    if (!shared && w->ws_gate) return MOE_ERR_INVALID_ARG;
    if ((st = check_ws(s, workspace, ws_bytes)) != MOE_OK) return st;
    if (!tc_available()) return MOE_ERR_UNSUPPORTED;
    cudaStream_t cs = (cudaStream_t)stream;
    const WsLayout L = ws_layout(s);
    DevError* err = at<DevError>(workspace, L.err);
    cudaError_t e = cudaMemsetAsync(err, 0, kErrBlockBytes, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 1. router (bf16 x and weights), top-K and weights
    int32_t* topk_idx = at<int32_t>(workspace, L.topk_idx);
    float* topk_w = at<float>(workspace, L.topk_w);
    e = launch_route(s, L, workspace, x, w_g, bias, nullptr, topk_idx, topk_w, err, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 2. dispatch (for small batches with the expert plan); x quantised per
    //    token row, codes and scales gathered into expert order (x_perm region:
    //    permuted codes [T*K][d], then x codes [T][d])
    int32_t* offsets = at<int32_t>(workspace, L.offsets);
    int32_t* inv = at<int32_t>(workspace, L.inv_perm);
    int32_t* tok = at<int32_t>(workspace, L.tok_of);
    const int64_t R = (int64_t)s.T * s.K;
    float* sc = at<float>(workspace, L.ascale);
    uint8_t* xq_perm = at<uint8_t>(workspace, L.x_perm);
    uint8_t* xq = xq_perm + R * s.d;
    FfnGroups g{};
    g.E = s.E;
    g.has_shared = shared ? 1 : 0;
    g.d = s.d;
    g.I = s.inter;
    g.Is = s.inter_shared;
    g.n_routed_rows = (int)R;
    g.T = s.T;
    g.max_group_rows = s.T;  // a token picks an expert once; the shared group has T rows
    g.offsets = offsets;
    g.row_src = nullptr;
    g.a_routed = xq_perm;
    g.a_perm = xq_perm;
    g.a_shared = xq;
    g.w_gate = w->w_gate;
    g.w_up = w->w_up;
    g.w_down = w->w_down;
    g.s_gate = w->s_gate;
    g.s_up = w->s_up;
    g.s_down = w->s_down;
    g.ws_gate = w->ws_gate;
    g.ws_up = w->ws_up;
    g.ws_down = w->ws_down;
    g.ss_gate = w->ss_gate;
    g.ss_up = w->ss_up;
    g.ss_down = w->ss_down;
    g.wblock = wblock;
    g.sa_routed = sc + s.T;
    g.sa_shared = sc;
    g.sa_h = sc + s.T + R;
    g.sa_hs = sc + s.T + 2 * R;
    g.h = at<void>(workspace, L.h);
    g.h_s = at<void>(workspace, L.h_s);
    g.y = at<void>(workspace, L.y_perm);
    g.y_s = at<void>(workspace, L.y_s);
    int32_t* counts = at<int32_t>(workspace, L.counts);
    int32_t* perm = at<int32_t>(workspace, L.perm);
    const bool fused = dispatch_plan_fusable(s);
    const bool pair = w8_pair_tiles(true, wblock);
    if (fused)
        e = launch_dispatch_plan_small(s, topk_idx, counts, offsets, perm, inv, tok, err, g,
                                       at<FfnPlanHeader>(workspace, L.plan),
                                       at<int32_t>(workspace, L.gemv_list),
                                       at<int4>(workspace, L.mtile_list), L.max_mtiles, 0, pair, 0,
                                       cs);
    else
        e = launch_dispatch(s, topk_idx, counts, offsets, perm, inv, tok,
                            at<int32_t>(workspace, L.blk_hist), err, cs);
    if (e == cudaSuccess) e = launch_quantize_act_rows(s.T, s.d, x, s.d, xq, s.d, sc, cs);
    if (e == cudaSuccess) e = launch_gather_codes(s, xq, sc, inv, xq_perm, sc + s.T, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 3. routed and shared experts, W8A8 on the tensor cores
    // a group has at most T rows (a token picks an expert once; the shared group has T)
    e = run_ffn_w8a8(s, g, L, workspace, s.T, fused, pair, err, cs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 4. combine
    return cuda_status(launch_combine(s, g.y, inv, topk_w, shared ? g.y_s : nullptr, y, cs));
}

moe_status moe_forward_w8a8(const moe_shape* shape, const void* x, const void* w_g,
                            const float* bias, const moe_fp8_experts* w, void* y, void* workspace,
                            size_t ws_bytes, void* stream) {
    return forward_w8a8_call(shape, x, w_g, bias, w, y, workspace, ws_bytes, stream, 0);
}

moe_status moe_forward_w8a8_blocks(const moe_shape* shape, const void* x, const void* w_g,
                                   const float* bias, const moe_fp8_experts* w, void* y,
                                   void* workspace, size_t ws_bytes, void* stream) {
    return forward_w8a8_call(shape, x, w_g, bias, w, y, workspace, ws_bytes, stream, kWBlock);
}

moe_status moe_get_device_error(const void* workspace, int32_t* code_out) {
    if (!workspace || !code_out) return MOE_ERR_INVALID_ARG;
    DevError h{};
    if (cudaMemcpy(&h, workspace, sizeof(DevError), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    *code_out = h.code;
    return MOE_OK;
}

}  // extern "C"
