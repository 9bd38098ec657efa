// dispatch.cu -- stage 2: per-expert histogram, exclusive scan, stable
// permutation and row gather.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 4.3: flatten
// the [T, K] expert ids, order the slots by expert id, gather the token rows
// into one contiguous buffer, count tokens per expert and build the offsets a
// grouped GEMM consumes.  "Computation and Data Movement for Inference",
// section 15: sorting the routing records by expert lets one weight load serve
// the whole bucket.  The page's code sorts with an unstable argsort and an
// inclusive cumsum; here the order is stable by flat slot f = t*K + j and the
// offsets are exclusive with E+1 entries.
//
// Three kernels over chunks of 1024 slots:
//   hist    -- per-chunk expert histogram (shared-memory atomics; counts only,
//              so the order of the atomics does not matter)
//   scan    -- one block: counts, exclusive offsets, and each chunk's base
//              position per expert (chunk-major running sums)
//   scatter -- per chunk, the stable rank of every slot among the earlier
//              slots of its expert: rank inside the warp from __match_any_sync,
//              plus the exclusive sum over earlier warps of the chunk, plus the
//              chunk base.  Writes perm, inv_perm and the token of every row.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kChunk = 1024;  // slots per block (one per thread)

__device__ __forceinline__ bool valid_expert(int e, int E) { return e >= 0 && e < E; }

__global__ void __launch_bounds__(kChunk)
dispatch_hist_kernel(const int32_t* __restrict__ idx, int64_t n, int E,
                     int32_t* __restrict__ blk_hist, DevError* err) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t f = (int64_t)blockIdx.x * kChunk + threadIdx.x;
    if (f < n) {
        const int e = idx[f];
        if (valid_expert(e, E)) atomicAdd(&hist[e], 1);
        else record_error(err, MOE_ERR_BOUNDS, 200);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        blk_hist[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_tot, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        int32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

// one block of 1024 threads; E <= 1024
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int32_t* __restrict__ blk_hist, int nb, int E, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t total;
    const int e = threadIdx.x;
    int32_t c = 0;
    if (e < E)
        for (int b = 0; b < nb; ++b) c += blk_hist[(int64_t)b * E + e];
    const int32_t off = block_exclusive_scan(e < E ? c : 0, warp_tot, &total);
    if (e < E) {
        counts[e] = c;
        offsets[e] = off;
        int32_t run = off;
        for (int b = 0; b < nb; ++b) {
            const int32_t t = blk_hist[(int64_t)b * E + e];
            blk_hist[(int64_t)b * E + e] = run;  // base position of chunk b for expert e
            run += t;
        }
    }
    if (threadIdx.x == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(kChunk)
dispatch_scatter_kernel(const int32_t* __restrict__ idx, int64_t n, int E, int K,
                        const int32_t* __restrict__ blk_base, int32_t* __restrict__ perm,
                        int32_t* __restrict__ inv_perm, int32_t* __restrict__ tok_of) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t wcnt[];  // [32 warps][E]: counts, then exclusive prefix over warps
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int64_t f = (int64_t)blockIdx.x * kChunk + threadIdx.x;
    int e = f < n ? idx[f] : -1;
    if (!valid_expert(e, E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int32_t run = 0;
        for (int w = 0; w < 32; ++w) {
            const int32_t t = wcnt[w * E + x];
            wcnt[w * E + x] = run;
            run += t;
        }
    }
    __syncthreads();
    if (f < n) {
        if (e >= 0) {
            const int32_t p = blk_base[(int64_t)blockIdx.x * E + e] + wcnt[warp * E + e] + rank;
            if (perm) perm[p] = (int32_t)f;
            inv_perm[f] = p;
            tok_of[p] = (int32_t)(f / K);
        } else {
            inv_perm[f] = -1;  // dropped slot (out-of-range expert id)
        }
    }
}

// One warp per (token, 128 16-byte vectors of its row): the slice of x is read
// once (four loads in flight per lane) and written to the token's K permuted
// positions inv_perm[t*K + j], so x crosses HBM once even when it does not fit
// in L2, and a few tokens still spread over many warps.  Rows are opaque
// bytes (bf16, fp32 or E4M3 codes); with s_src set, the warp that copies the
// first slice of a row also copies the row's scale s_src[t] to s_dst[p].
constexpr int kGatherVecs = 32 * 4;  // vectors per warp item

__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_perm,
                   uint4* __restrict__ x_perm, int Tn, int K, int vec_per_row, int64_t n_rows,
                   const float* __restrict__ s_src, float* __restrict__ s_dst) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nchunks = (vec_per_row + kGatherVecs - 1) / kGatherVecs;
    const int64_t items = (int64_t)Tn * nchunks;
    for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < items;
         w += (int64_t)gridDim.x * 8) {
        const int64_t t = w / nchunks;
        const int v0 = (int)(w - t * nchunks) * kGatherVecs + lane;
        const int32_t my_p = lane < K ? inv_perm[t * K + lane] : -1;
        if (s_src != nullptr && v0 < 32 && my_p >= 0 && my_p < n_rows) s_dst[my_p] = s_src[t];
        const uint4* src = x + t * vec_per_row;
        uint4 tmp[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (v0 + 32 * q < vec_per_row) tmp[q] = __ldg(src + v0 + 32 * q);
        // warp-uniform trip count: every lane reaches the shuffles
        for (int j = 0; j < K; ++j) {
            const int32_t p = __shfl_sync(0xffffffffu, my_p, j);
            if (p < 0 || p >= n_rows) continue;  // dropped slot
            uint4* dst = x_perm + (int64_t)p * vec_per_row;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (v0 + 32 * q < vec_per_row) dst[v0 + 32 * q] = tmp[q];
        }
    }
}

}  // namespace

int dispatch_blocks_for(int64_t n_slots) { return (int)ceil_div(n_slots > 0 ? n_slots : 1, kChunk); }

cudaError_t launch_dispatch(const moe_shape& s, const int32_t* topk_idx, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* tok_of,
                            int32_t* blk_hist, DevError* err, cudaStream_t st) {
    const int64_t n = (int64_t)s.T * s.K;
    const int nb = dispatch_blocks_for(n);
    const size_t hist_smem = (size_t)s.E * sizeof(int32_t);
    const size_t scat_smem = (size_t)32 * s.E * sizeof(int32_t);
    // the scatter kernel's per-warp table needs up to 128 KB of shared memory
    cudaError_t e = cudaFuncSetAttribute(dispatch_scatter_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(32 * 1024 * sizeof(int32_t)));
    if (e == cudaSuccess)
        e = launch_pdl(dispatch_hist_kernel, dim3(nb), dim3(kChunk), hist_smem, st, topk_idx, n,
                       s.E, blk_hist, err);
    if (e == cudaSuccess)
        e = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(1024), 0, st, blk_hist, nb, s.E, counts,
                       offsets);
    if (e == cudaSuccess)
        e = launch_pdl(dispatch_scatter_kernel, dim3(nb), dim3(kChunk), scat_smem, st, topk_idx, n,
                       s.E, s.K, blk_hist, perm, inv_perm, tok_of);
    return e;
}

cudaError_t launch_gather_rows(const moe_shape& s, const void* x, const int32_t* inv_perm,
                               void* x_perm, cudaStream_t st) {
    const int64_t rows = (int64_t)s.T * s.K;
    const int esz = s.dtype == MOE_BF16 ? 2 : 4;
    const int vpr = s.d * esz / 16;
    int64_t blocks = ceil_div((int64_t)s.T * ceil_div(vpr, kGatherVecs), 8);
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, (const uint4*)x,
                      inv_perm, (uint4*)x_perm, s.T, s.K, vpr, rows, (const float*)nullptr,
                      (float*)nullptr);
}

cudaError_t launch_gather_codes(const moe_shape& s, const uint8_t* xq, const float* sx,
                                const int32_t* inv_perm, uint8_t* xq_perm, float* s_perm,
                                cudaStream_t st) {
    const int64_t rows = (int64_t)s.T * s.K;
    const int vpr = s.d / 16;
    int64_t blocks = ceil_div((int64_t)s.T * ceil_div(vpr, kGatherVecs), 8);
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                      (const uint4*)xq, inv_perm, (uint4*)xq_perm, s.T, s.K, vpr, rows, sx, s_perm);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_permute_noalloc: the dispatch stage for callers that cannot allocate.
//
// Some callers have no way to allocate device memory: a serving runtime that
// reserves all of HBM for its own pool at start-up and allows no cudaMalloc
// afterwards (cudaMalloc can also stall every stream of the device), or a
// plug-in that is handed only the tensors it works on and no allocator.  For
// them this entry point keeps the dispatch kernels' scratch -- the device error
// word, the per-chunk expert histogram, the token of every permuted row and,
// when the caller passes no inv_perm, the inverse permutation -- in the
// file-scope array below instead of a caller-provided workspace.
//
// The array (kNoAllocScratchBytes, 4 MiB) is held by every GPU that loads the
// library until the process exits.  In host code its name is a host-side
// stand-in, not a device address: the address the kernels get comes from
// cudaGetSymbolAddress, called with the device current.  The first call made
// on a device (in a given CUDA context) does that lookup and keeps the result
// for later calls in the same context, so make that first call before any
// stream capture.  The result is keyed on the context's unique id: after a
// cudaDeviceReset, or any other teardown and re-creation of the context, the
// module is loaded again, the array may sit elsewhere, and the next call
// looks it up again instead of handing the kernels a stale address.  Every
// call shares the array and it keeps the last call's contents, so the error
// word is cleared at the start of every call; calls whose work overlaps on the
// GPU (other streams, other threads) race on it.
// ---------------------------------------------------------------------------
static constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

#include <cuda.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocEntry {
    unsigned long long ctx_id = 0;  // unique id of the context the address belongs to (0: none)
    void* addr = nullptr;
};
std::mutex g_noalloc_mu;
NoAllocEntry g_noalloc[kNoAllocMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// the driver's cuCtxGetCurrent / cuCtxGetId, found through the runtime (no -lcuda)
template <typename F>
F driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(f);
}

// Unique id of the calling thread's current context (0 when none is current or
// the driver cannot say).
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
        get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch in the current device's current context.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocEntry& c = g_noalloc[dev];
    unsigned long long id = current_ctx_id();
    if (id != 0 && id == c.ctx_id && c.addr != nullptr) {
        *out = c.addr;
        return cudaSuccess;
    }
    // first call in this context (the lookup also makes the runtime's context
    // current when no runtime call on this thread has done so yet)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (id == 0) id = current_ctx_id();
    c.ctx_id = id;  // 0 (unknown context) is never matched: the next call looks up again
    c.addr = p;
    *out = p;
    return cudaSuccess;
}

size_t noalloc_align(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const moe_shape* shape, const int32_t* topk_idx,
                                          const void* x, int32_t* counts, int32_t* offsets,
                                          int32_t* perm, int32_t* inv_perm, void* x_perm,
                                          void* stream) {
    using namespace moe;
    // the shapes moe_permute accepts, no more
    const moe_status st = check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (!counts || !offsets || (s.T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)x & 15u) || ((uintptr_t)x_perm & 15u)) return MOE_ERR_INVALID_ARG;
    // scratch carving: error word | per-chunk histogram | token of each row | inverse permutation
    const int64_t n = (int64_t)s.T * s.K;
    const int nb = dispatch_blocks_for(n);
    const size_t off_hist = 256;
    const size_t off_tok = off_hist + noalloc_align(sizeof(int32_t) * (size_t)nb * s.E);
    const size_t off_inv = off_tok + noalloc_align(sizeof(int32_t) * (size_t)n);
    const size_t need = off_inv + (inv_perm ? 0 : noalloc_align(sizeof(int32_t) * (size_t)n));
    if (need > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
    void* base = nullptr;
    if (noalloc_scratch(&base) != cudaSuccess) return MOE_ERR_CUDA;
    uint8_t* b = static_cast<uint8_t*>(base);
    cudaStream_t cs = (cudaStream_t)stream;
    DevError* err = reinterpret_cast<DevError*>(b);
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(DevError), cs);  // last call's contents linger
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (s.T == 0) {
        e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (s.E + 1), cs);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    int32_t* hist = reinterpret_cast<int32_t*>(b + off_hist);
    int32_t* tok = reinterpret_cast<int32_t*>(b + off_tok);
    int32_t* inv = inv_perm ? inv_perm : reinterpret_cast<int32_t*>(b + off_inv);
    e = launch_dispatch(s, topk_idx, counts, offsets, perm, inv, tok, hist, err, cs);
    if (e == cudaSuccess && x && x_perm) e = launch_gather_rows(s, x, inv, x_perm, cs);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
