// quant.cu -- per-row E4M3 quantisation of expert weights (moe_quantize_fp8_rows).
//
// "LLM from scratch, ch. 6", section "second route: make every byte
// cheaper": x_q = round(x / s) + z with a per-channel scale.  Here z = 0, the
// scale of row r is amax_r / 448 (448 = the largest finite E4M3 magnitude)
// and round is the hardware's round-to-nearest-even with saturation to
// +-448.  Both divisions are IEEE fp32 divisions, so a code is the same
// integer whatever machine computes it from the same fp32 quotient.
//
// One 256-thread block per row, two passes over the row (the second reads it
// from L1/L2): a max-reduction of |w|, then 16 codes per thread and step
// (one 16-byte store).  An offline conversion step, HBM bound.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ void load16(const float* src, float (&f)[16]) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 v = s4[k];
        f[4 * k] = v.x; f[4 * k + 1] = v.y; f[4 * k + 2] = v.z; f[4 * k + 3] = v.w;
    }
}

__device__ __forceinline__ void load16(const bf16* src, float (&f)[16]) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint4 v = s4[k];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[8 * k + 2 * j] = __uint_as_float(w[j] << 16);
            f[8 * k + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rows_kernel(const T* __restrict__ w, uint8_t* __restrict__ codes,
                     float* __restrict__ scales, int64_t cols) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kQuantThreads / 32];
    const int64_t r = blockIdx.x;
    const T* row = w + r * cols;
    const int64_t nvec = cols / 16;
    float amax = 0.0f;
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        float f[16];
        load16(row + v * 16, f);
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(f[k]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < kQuantThreads / 32 ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) red[0] = m;
    }
    __syncthreads();
    const float a = red[0];
    const float s = a > 0.0f ? a / 448.0f : 1.0f;
    if (threadIdx.x == 0) scales[r] = s;
    uint8_t* out = codes + r * cols;
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        float f[16];
        load16(row + v * 16, f);
        uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(f[k] / s, __NV_SATFINITE, __NV_E4M3);
            packed[k >> 2] |= (uint32_t)c << (8 * (k & 3));  // byte k of the 16-byte store
        }
        *reinterpret_cast<uint4*>(out + v * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

}  // namespace

cudaError_t launch_quantize_fp8_rows(int64_t rows, int64_t cols, int dtype, const void* w,
                                     uint8_t* codes, float* scales, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (dtype == MOE_BF16)
        return launch_pdl(quantize_rows_kernel<bf16>, dim3((unsigned)rows), dim3(kQuantThreads), 0,
                          st, (const bf16*)w, codes, scales, cols);
    return launch_pdl(quantize_rows_kernel<float>, dim3((unsigned)rows), dim3(kQuantThreads), 0, st,
                      (const float*)w, codes, scales, cols);
}

}  // namespace moe
