// combine.cu -- stage 4: back to token order, weighted sum of the K expert
// outputs, plus the shared expert.
//
// adg.csdn.net sparse-MoE explainer, section 2.2 step 4 (output is the
// weighted sum of the selected experts); "Sparse MoE inference kernels ..."
// (blog.llmgo.top), section 1.1 (shared expert output added to the routed
// sum); "Computation and Data Movement for Inference", section 4 (expert
// outputs return to token order, are weighted and merged).
//
// A gather per token (no atomics, deterministic): each thread owns one
// 16-byte vector of an output row, accumulates in fp32 -- shared term first,
// then j = 0..K-1 -- and rounds once.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ y_perm, const int32_t* __restrict__ inv_perm,
               const float* __restrict__ topk_w, const T* __restrict__ y_shared, T* __restrict__ y,
               int d, int K, int64_t n_rows) {
    pdl_wait();
    pdl_trigger();
    constexpr int V = Elem<T>::kPerVec;
    const int nvec = d / V;
    const int t = blockIdx.x;
    const int v = blockIdx.y * blockDim.x + threadIdx.x;
    if (v >= nvec) return;
    float acc[V];
    if (y_shared) {
        unpack(ld_ro(y_shared + (int64_t)t * d + (int64_t)v * V), acc, (const T*)nullptr);
    } else {
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] = 0.f;
    }
    for (int j = 0; j < K; ++j) {
        const int32_t p = inv_perm[(int64_t)t * K + j];
        if (p < 0 || p >= n_rows) continue;  // dropped slot
        const float w = topk_w[(int64_t)t * K + j];
        float f[V];
        unpack(ld_ro(y_perm + (int64_t)p * d + (int64_t)v * V), f, (const T*)nullptr);
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] = fmaf(w, f[k], acc[k]);
    }
    uint4 out;
    if constexpr (V == 4) {
        out = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                         __float_as_uint(acc[3]));
    } else {
        uint32_t w32[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
            w32[k] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        out = make_uint4(w32[0], w32[1], w32[2], w32[3]);
    }
    *reinterpret_cast<uint4*>(y + (int64_t)t * d + (int64_t)v * V) = out;
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, const void* y_perm, const int32_t* inv_perm,
                           const float* topk_w, const void* y_shared, void* y, cudaStream_t st) {
    const int V = s.dtype == MOE_BF16 ? 8 : 4;
    const int nvec = s.d / V;
    const dim3 grid((unsigned)s.T, (unsigned)ceil_div(nvec, 256));
    const int64_t rows = (int64_t)s.T * s.K;
    if (s.dtype == MOE_BF16)
        return launch_pdl(combine_kernel<bf16>, grid, dim3(256), 0, st, (const bf16*)y_perm,
                          inv_perm, topk_w, (const bf16*)y_shared, (bf16*)y, s.d, s.K, rows);
    return launch_pdl(combine_kernel<float>, grid, dim3(256), 0, st, (const float*)y_perm, inv_perm,
                      topk_w, (const float*)y_shared, (float*)y, s.d, s.K, rows);
}

}  // namespace moe
