// router.cu -- stage 1: router scores, top-K with lower-index ties, softmax
// over the K selected scores.
//
// adg.csdn.net sparse-MoE explainer, section 2.2 (steps 1-3: a linear router
// scores every expert, the K best are kept, softmax over those K);
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 2.1 (linear
// gate projection followed by top-k).
//
// Scores are fp32 partial dot products written by a split-K streaming GEMV
// (W_g is read once per 8-token chunk; x through L1), summed in a fixed order
// by the top-K kernel so the result is deterministic.  For large bf16 batches
// the tensor-core GEMM in ffn_tc.cu produces the scores instead (split = 1).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterTok = 8;  // tokens per pass
constexpr int kMaxSplits = 8;  // split-K partials per score

// part[s][t][e] = sum_{k in split s} x[t][k] * w_g[e][k], for the units
// (token chunk, expert, split) this block's warps take
template <typename T>
__device__ __forceinline__ void router_gemv_units(const T* __restrict__ x, const T* __restrict__ w_g,
                                                  float* __restrict__ part, int Tn, int d, int E,
                                                  int splits) {
    constexpr int V = Elem<T>::kPerVec;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nvec = d / V;                       // 16-byte vectors per row
    const int vps = (nvec + splits - 1) / splits; // vectors per split
    const int64_t n_chunks = (Tn + kRouterTok - 1) / kRouterTok;
    const int64_t units = n_chunks * E * splits;
    for (int64_t u = (int64_t)blockIdx.x * kRouterWarps + warp; u < units;
         u += (int64_t)gridDim.x * kRouterWarps) {
        const int s = (int)(u % splits);
        const int e = (int)((u / splits) % E);
        const int c = (int)(u / ((int64_t)splits * E));
        const int v0 = s * vps;
        const int v1 = min(nvec, v0 + vps);
        const int t0 = c * kRouterTok;
        const int nt = min(kRouterTok, Tn - t0);
        float acc[kRouterTok];
#pragma unroll
        for (int m = 0; m < kRouterTok; ++m) acc[m] = 0.f;
        const T* wrow = w_g + (int64_t)e * d;
#pragma unroll 4
        for (int v = v0 + lane; v < v1; v += 32) {
            float wf[V];
            unpack(ld_stream(wrow + (int64_t)v * V), wf, (const T*)nullptr);
#pragma unroll
            for (int m = 0; m < kRouterTok; ++m) {
                if (m < nt) {
                    float xf[V];
                    unpack(ld_ro(x + (int64_t)(t0 + m) * d + (int64_t)v * V), xf, (const T*)nullptr);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[m] = fmaf(wf[q], xf[q], acc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < kRouterTok; ++m) {
            float r = warp_sum(acc[m]);
            if (lane == 0 && m < nt) part[((int64_t)s * Tn + t0 + m) * E + e] = r;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_gemv_kernel(const T* __restrict__ x, const T* __restrict__ w_g, float* __restrict__ part,
                   int Tn, int d, int E, int splits) {
    pdl_wait();
    pdl_trigger();
    router_gemv_units<T>(x, w_g, part, Tn, d, E, splits);
}

// Few experts, many tokens: part[t][e] = sum_k x[t][k] * w_g[e][k] with one
// warp per TT tokens and all E <= EM experts, so x is streamed from HBM once
// and the small W_g (E rows) is served from L1.  (The split-K kernel above
// reads x once per expert, which for E = 8 and thousands of tokens costs
// ~8x the x traffic.)
constexpr int kRouterTokWarps = 4;
template <typename T, int EM, int TT>
__global__ void __launch_bounds__(kRouterTokWarps * 32)
router_tokens_kernel(const T* __restrict__ x, const T* __restrict__ w_g, float* __restrict__ part,
                     int Tn, int d, int E) {
    pdl_wait();
    pdl_trigger();
    constexpr int V = Elem<T>::kPerVec;
    constexpr int kUnroll = EM <= 8 ? 2 : 1;  // steps whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nvec = d / V;
    const int64_t units = (Tn + TT - 1) / TT;
    for (int64_t u = (int64_t)blockIdx.x * kRouterTokWarps + warp; u < units;
         u += (int64_t)gridDim.x * kRouterTokWarps) {
        const int t0 = (int)(u * TT);
        const int nt = min(TT, Tn - t0);
        float acc[TT][EM];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < EM; ++e) acc[t][e] = 0.f;
#pragma unroll kUnroll
        for (int v = lane; v < nvec; v += 32) {
            // every load of the step first (x from HBM, W_g from L1), then the FMAs
            uint4 xv[TT], wv[EM];
#pragma unroll
            for (int t = 0; t < TT; ++t)
                xv[t] = t < nt ? ld_stream(x + (int64_t)(t0 + t) * d + (int64_t)v * V)
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int e = 0; e < EM; ++e)
                wv[e] = e < E ? ld_ro(w_g + (int64_t)e * d + (int64_t)v * V) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float xf[V];
                unpack(xv[t], xf, (const T*)nullptr);
#pragma unroll
                for (int e = 0; e < EM; ++e) {
                    float wf[V];
                    unpack(wv[e], wf, (const T*)nullptr);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[t][e] = fmaf(wf[q], xf[q], acc[t][e]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < EM; ++e) {
                if (e < E) {
                    const float r = warp_sum(acc[t][e]);
                    if (lane == 0 && t < nt) part[(int64_t)(t0 + t) * E + e] = r;
                }
            }
    }
}

// the token-major kernel serves E <= 32 from this many tokens on
constexpr int kRouterTokMinT = 256;
// the fused GEMV + top-K launch serves batches of at most this many tokens
// (its last block routes them all, two per warp at most)
constexpr int kFusedRouteMaxT = 16;

struct Cand {
    float key;  // what the selection compares
    float val;  // what the weights are formed from
    int e;
};
// a beats b: larger key, or equal key and lower index
__device__ __forceinline__ bool beats(const Cand& a, const Cand& b) {
    return a.e >= 0 && (b.e < 0 || a.key > b.key || (a.key == b.key && a.e < b.e));
}

// One warp per token.  Lane l holds experts e = l + 32*m.
//   MODE 0 (softmax router; explainer section 2.2): key = score + bias, and
//          w = softmax over the K selected keys.
//   MODE 1 (sigmoid router; llmgo page section 2.2 and the dispatcher code of
//          section 4.3): a = sigmoid(score), key = a + bias (the bias only
//          steers the selection), w = a / (sum of the selected a + 1e-6).
// logits_out receives the keys.
// The whole warp routes token t.  CG: read the partials through L2 only (they
// were written by other blocks of the same launch).
template <int MAXM, int MODE, bool CG>
__device__ __forceinline__ void topk_token(const float* __restrict__ part, int splits,
                                           const float* __restrict__ bias,
                                           float* __restrict__ logits_out,
                                           int32_t* __restrict__ topk_idx,
                                           float* __restrict__ topk_w, int Tn, int E, int K, int t,
                                           int lane) {
    float key[MAXM], val[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        const int e = lane + 32 * m;
        float k = 0.f, v = 0.f;
        if (e < E) {
            // fixed summation order over the split-K partials (deterministic)
            float pq[kMaxSplits];
#pragma unroll
            for (int q = 0; q < kMaxSplits; ++q) {
                const float* src = part + ((int64_t)q * Tn + t) * E + e;
                pq[q] = q < splits ? (CG ? __ldcg(src) : *src) : 0.f;
            }
            float s = pq[0];
#pragma unroll
            for (int q = 1; q < kMaxSplits; ++q)
                if (q < splits) s += pq[q];
            const float b = bias ? bias[e] : 0.f;
            if (MODE == 1) {
                v = 1.f / (1.f + expf(-s));
                k = v + b;
            } else {
                k = s + b;
                v = k;
            }
            if (logits_out) logits_out[(int64_t)t * E + e] = k;
        }
        key[m] = k;
        val[m] = v;
    }
    uint32_t taken = 0;
    float my_v = 0.f;  // lane j keeps the value of the j-th pick
    float k0 = 0.f;    // key of the first pick
    for (int j = 0; j < K; ++j) {
        Cand best{0.f, 0.f, -1};
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            const int e = lane + 32 * m;
            if (e < E && !(taken & (1u << m)) && (best.e < 0 || key[m] > best.key))
                best = Cand{key[m], val[m], e};
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            Cand other{__shfl_xor_sync(0xffffffffu, best.key, o),
                       __shfl_xor_sync(0xffffffffu, best.val, o),
                       __shfl_xor_sync(0xffffffffu, best.e, o)};
            if (beats(other, best)) best = other;
        }
        if ((best.e & 31) == lane) taken |= 1u << (best.e >> 5);
        if (lane == j) my_v = best.val;
        if (j == 0) k0 = best.key;
        if (lane == 0) topk_idx[(int64_t)t * K + j] = best.e;
    }
    if (MODE == 1) {
        const float a = lane < K ? my_v : 0.f;
        const float denom = warp_sum(a) + 1e-6f;
        if (lane < K) topk_w[(int64_t)t * K + lane] = a / denom;
    } else {
        const float ex = lane < K ? expf(my_v - k0) : 0.f;
        const float denom = warp_sum(ex);
        if (lane < K) topk_w[(int64_t)t * K + lane] = ex / denom;
    }
}

template <int MAXM, int MODE>
__global__ void __launch_bounds__(256)
topk_route_kernel(const float* __restrict__ part, int splits, const float* __restrict__ bias,
                  float* __restrict__ logits_out, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w, int Tn, int E, int K) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= Tn) return;
    topk_token<MAXM, MODE, false>(part, splits, bias, logits_out, topk_idx, topk_w, Tn, E, K, t,
                                  lane);
}

// A few tokens (T <= kFusedRouteMaxT): the split-K GEMV and the top-K in one
// launch.  Every block computes its (chunk, expert, split) partials as
// router_gemv_kernel does, makes them visible device-wide and takes a ticket;
// the block that takes the last ticket finds every partial written and routes
// the tokens, one warp per token (the same fixed-order sum of the partials and
// the same warp top-K as the two-launch path, so the same bits).  No block
// waits for another.  The ticket counter lives in the workspace's error block,
// which the entry point clears before the launch; the last block also puts it
// back to zero.
template <typename T, int MAXM, int MODE>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_fused_kernel(const T* __restrict__ x, const T* __restrict__ w_g, float* __restrict__ part,
                    int Tn, int d, int E, int splits, const float* __restrict__ bias,
                    float* __restrict__ logits_out, int32_t* __restrict__ topk_idx,
                    float* __restrict__ topk_w, int K, unsigned int* __restrict__ ticket) {
    pdl_wait();
    pdl_trigger();
    __shared__ int last;
    router_gemv_units<T>(x, w_g, part, Tn, d, E, splits);
    // the lanes that wrote partials make them visible device-wide before the ticket
    if ((threadIdx.x & 31) == 0) __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = warp; t < Tn; t += kRouterWarps)
        topk_token<MAXM, MODE, true>(part, splits, bias, logits_out, topk_idx, topk_w, Tn, E, K, t,
                                     lane);
    if (threadIdx.x == 0) *ticket = 0u;
}

}  // namespace

// about 224 16-byte vectors (7 per lane) of a W_g row per split; one split
// (full sums) on the token-major path
int router_splits_for(const moe_shape& s) {
    if (s.E <= 32 && s.T >= kRouterTokMinT) return 1;
    const int V = s.dtype == MOE_BF16 ? 8 : 4;
    int splits = (s.d / V) / 224;
    return splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
}

template <typename T>
cudaError_t launch_router_tokens(const moe_shape& s, const void* x, const void* w_g, float* part,
                                 cudaStream_t st) {
    const int tt = 2;
    int64_t blocks = ceil_div(ceil_div(s.T, tt), kRouterTokWarps);
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    const dim3 grid((unsigned)blocks), block(kRouterTokWarps * 32);
    if (s.E <= 8)
        return launch_pdl(router_tokens_kernel<T, 8, 2>, grid, block, 0, st, (const T*)x,
                          (const T*)w_g, part, s.T, s.d, s.E);
    if (s.E <= 16)
        return launch_pdl(router_tokens_kernel<T, 16, 2>, grid, block, 0, st, (const T*)x,
                          (const T*)w_g, part, s.T, s.d, s.E);
    return launch_pdl(router_tokens_kernel<T, 32, 2>, grid, block, 0, st, (const T*)x,
                      (const T*)w_g, part, s.T, s.d, s.E);
}

cudaError_t launch_router_gemv(const moe_shape& s, const void* x, const void* w_g, float* part,
                               int splits, cudaStream_t st) {
    if (splits == 1 && s.E <= 32 && s.T >= kRouterTokMinT)
        return s.dtype == MOE_BF16 ? launch_router_tokens<bf16>(s, x, w_g, part, st)
                                   : launch_router_tokens<float>(s, x, w_g, part, st);
    const int64_t units = ceil_div(s.T, kRouterTok) * (int64_t)s.E * splits;
    int64_t blocks = ceil_div(units, kRouterWarps);
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid((unsigned)blocks), block(kRouterWarps * 32);
    if (s.dtype == MOE_BF16)
        return launch_pdl(router_gemv_kernel<bf16>, grid, block, 0, st, (const bf16*)x,
                          (const bf16*)w_g, part, s.T, s.d, s.E, splits);
    return launch_pdl(router_gemv_kernel<float>, grid, block, 0, st, (const float*)x,
                      (const float*)w_g, part, s.T, s.d, s.E, splits);
}

bool router_fused_possible(const moe_shape& s) {
    return s.T > 0 && s.T <= kFusedRouteMaxT && fused_router_enabled();
}

// MOE_FUSED_ROUTER=1 (read per call) routes batches of at most 16 tokens in
// one launch.  Off by default: measured on GB300 (interleaved, 4 x 300 calls
// each) the fused launch was slower than the two launches -- DeepSeek-V3 decode
// 827.6 vs 818.3 us, T = 1 164.3 vs 163.2 us -- the last block's top-K starting
// only after every block's fence and ticket, where the separate top-K kernel
// is already resident and waiting.
bool fused_router_enabled() {
    const char* e = getenv("MOE_FUSED_ROUTER");
    return e && e[0] == '1';
}

cudaError_t launch_router_fused(const moe_shape& s, const void* x, const void* w_g, float* part,
                                int splits, const float* bias, float* logits_out,
                                int32_t* topk_idx, float* topk_w, unsigned int* ticket,
                                cudaStream_t st) {
    const int64_t units = ceil_div(s.T, kRouterTok) * (int64_t)s.E * splits;
    int64_t blocks = ceil_div(units, kRouterWarps);
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid((unsigned)blocks), block(kRouterWarps * 32);
    const int m = (int)ceil_div(s.E, 32);
    cudaError_t e;
#define MOE_FUSED(TT, M, MODE)                                                                    \
    e = launch_pdl(router_fused_kernel<TT, M, MODE>, grid, block, 0, st, (const TT*)x,            \
                   (const TT*)w_g, part, s.T, s.d, s.E, splits, bias, logits_out, topk_idx,       \
                   topk_w, s.K, ticket)
#define MOE_FUSED_M(TT, MODE)                    \
    if (m <= 1) MOE_FUSED(TT, 1, MODE);          \
    else if (m <= 2) MOE_FUSED(TT, 2, MODE);     \
    else if (m <= 4) MOE_FUSED(TT, 4, MODE);     \
    else if (m <= 8) MOE_FUSED(TT, 8, MODE);     \
    else if (m <= 16) MOE_FUSED(TT, 16, MODE);   \
    else MOE_FUSED(TT, 32, MODE)
    if (s.dtype == MOE_BF16) {
        if (s.router == MOE_ROUTER_SIGMOID) { MOE_FUSED_M(bf16, 1); } else { MOE_FUSED_M(bf16, 0); }
    } else {
        if (s.router == MOE_ROUTER_SIGMOID) { MOE_FUSED_M(float, 1); } else { MOE_FUSED_M(float, 0); }
    }
#undef MOE_FUSED_M
#undef MOE_FUSED
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_topk_softmax(const moe_shape& s, const float* part, int splits,
                                const float* bias, float* logits_out, int32_t* topk_idx,
                                float* topk_w, cudaStream_t st) {
    const unsigned blocks = (unsigned)ceil_div(s.T, 8);
    const int m = (int)ceil_div(s.E, 32);
#define MOE_TOPK(M, MODE)                                                                     \
    e = launch_pdl(topk_route_kernel<M, MODE>, dim3(blocks), dim3(256), 0, st, part, splits, bias, \
                   logits_out, topk_idx, topk_w, s.T, s.E, s.K)
#define MOE_TOPK_M(MODE)                    \
    if (m <= 1) MOE_TOPK(1, MODE);          \
    else if (m <= 2) MOE_TOPK(2, MODE);     \
    else if (m <= 4) MOE_TOPK(4, MODE);     \
    else if (m <= 8) MOE_TOPK(8, MODE);     \
    else if (m <= 16) MOE_TOPK(16, MODE);   \
    else MOE_TOPK(32, MODE)
    cudaError_t e;
    if (s.router == MOE_ROUTER_SIGMOID) {
        MOE_TOPK_M(1);
    } else {
        MOE_TOPK_M(0);
    }
#undef MOE_TOPK_M
#undef MOE_TOPK
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
