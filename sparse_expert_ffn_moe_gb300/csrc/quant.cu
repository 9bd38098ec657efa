// quant.cu -- per-row and per-block E4M3 quantisation of expert weights
// (moe_quantize_fp8_rows, moe_quantize_fp8_blocks) and of the activation rows
// of 8-bit-activation experts.
//
// "LLM from scratch, ch. 6", section "second route: make every byte
// cheaper": x_q = round(x / s) + z with a per-channel scale.  Here z = 0, the
// scale of row r is amax_r / 448 (448 = the largest finite E4M3 magnitude)
// and round is the hardware's round-to-nearest-even with saturation to
// +-448.  Both divisions are IEEE fp32 divisions, so a code is the same
// integer whatever machine computes it from the same fp32 quotient.
//
// Weights: one 256-thread block per row, two passes over the row (the second
// reads it from L1/L2): a max-reduction of |w|, then 16 codes per thread and
// step (one 16-byte store).  An offline conversion step, HBM bound.
// Activations (8-bit-activation experts): quantize_act_rows_kernel below; and
// bf16 activations as two E4M3 planes (a code and the code of its remainder)
// for the 8-bit-weight tensor-core path: split_*_kernel below.
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

// 128 x 128 block scales (moe_quantize_fp8_blocks): one 256-thread block per
// weight block (grid: column blocks x row blocks).  Each thread keeps its four
// 16-value vectors of the block in registers across the max-reduction, so the
// block is read once; the scale and code decisions are quantize_rows_kernel's,
// over the block's elements.  Edge blocks are ragged: rows past the matrix and
// columns past cols (cols a multiple of 16) are skipped.
constexpr int kQBlk = 128;
constexpr int kQBlkVecs = kQBlk * kQBlk / 16 / kQuantThreads;  // 4 vectors per thread

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
quantize_blocks_kernel(const T* __restrict__ w, uint8_t* __restrict__ codes,
                       float* __restrict__ scales, int64_t rows, int64_t cols) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kQuantThreads / 32];
    const int64_t r0 = (int64_t)blockIdx.y * kQBlk, c0 = (int64_t)blockIdx.x * kQBlk;
    const int64_t nr = min((int64_t)kQBlk, rows - r0), nc = min((int64_t)kQBlk, cols - c0);
    float f[kQBlkVecs][16];
    bool in[kQBlkVecs];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kQBlkVecs; ++j) {
        const int v = (int)threadIdx.x + j * kQuantThreads;  // 8 vectors per block row
        const int i = v >> 3, c = (v & 7) * 16;
        in[j] = i < nr && c < nc;
        if (in[j]) {
            load16(w + (r0 + i) * cols + c0 + c, f[j]);
#pragma unroll
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(f[j][k]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < kQuantThreads / 32; ++k) m = fmaxf(m, red[k]);
    const float s = m > 0.0f ? m / 448.0f : 1.0f;
    if (threadIdx.x == 0) scales[blockIdx.y * gridDim.x + blockIdx.x] = s;
#pragma unroll
    for (int j = 0; j < kQBlkVecs; ++j) {
        if (!in[j]) continue;
        const int v = (int)threadIdx.x + j * kQuantThreads;
        const int i = v >> 3, c = (v & 7) * 16;
        uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(f[j][k] / s, __NV_SATFINITE, __NV_E4M3);
            packed[k >> 2] |= (uint32_t)q << (8 * (k & 3));
        }
        *reinterpret_cast<uint4*>(codes + (r0 + i) * cols + c0 + c) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

// Activation rows (bf16, cols a multiple of 16 and at most 16384): one
// 256-thread block per row loads the whole row into registers (at most four
// 16-value vectors per thread) before any code is written, so the codes may
// overwrite the row's own storage.  Row r is read at w + r * ld_in (elements)
// and its codes written at codes + r * ld_out (bytes).  The same decisions as
// quantize_rows_kernel: scale = amax / 448, code = E4M3 nearest to v / scale.
constexpr int kActVecs = 4;

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&f)[16]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_act_rows_kernel(const bf16* w, int64_t ld_in, uint8_t* codes, int64_t ld_out,
                         float* __restrict__ scales, int cols) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kQuantThreads / 32];
    const int64_t r = blockIdx.x;
    const uint4* row = reinterpret_cast<const uint4*>(w + r * ld_in);
    const int nvec = cols / 16;
    uint4 v[kActVecs][2];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kActVecs; ++j) {
        const int vi = (int)threadIdx.x + j * kQuantThreads;
        if (vi < nvec) {
            v[j][0] = row[2 * vi];
            v[j][1] = row[2 * vi + 1];
            float f[16];
            unpack16(v[j][0], v[j][1], f);
#pragma unroll
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(f[k]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();  // every load of the row has completed past this point
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kQuantThreads / 32; ++i) m = fmaxf(m, red[i]);
    const float s = m > 0.0f ? m / 448.0f : 1.0f;
    if (threadIdx.x == 0) scales[r] = s;
    uint8_t* out = codes + r * ld_out;
#pragma unroll
    for (int j = 0; j < kActVecs; ++j) {
        const int vi = (int)threadIdx.x + j * kQuantThreads;
        if (vi < nvec) {
            float f[16];
            unpack16(v[j][0], v[j][1], f);
            uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(f[k] / s, __NV_SATFINITE, __NV_E4M3);
                packed[k >> 2] |= (uint32_t)c << (8 * (k & 3));
            }
            *reinterpret_cast<uint4*>(out + (int64_t)vi * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
}

// Rows whose max |value| is known (raised by the producing GEMM): no block
// reduction, one warp per row.  The warp walks its row from low to high
// addresses, 1024 values per step (16 per lane, two 512-value halves), and
// orders each step's loads before its stores with __syncwarp.  Codes of
// values [a, a + 1024) land on bytes [a, a + 1024), which hold bf16 values
// [a / 2, a / 2 + 512) -- all loaded at this step or an earlier one -- and
// every later load reads bytes past every earlier store, so the codes may
// overwrite the row in place.
constexpr int kRowsPerBlock = kQuantThreads / 32;

__global__ void __launch_bounds__(kQuantThreads)
quantize_rows_known_amax_kernel(const bf16* w, int64_t ld_in, uint8_t* codes, int64_t ld_out,
                                float* amax_scale, int cols, int64_t rows) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (r >= rows) return;
    const float m = __uint_as_float(reinterpret_cast<const uint32_t*>(amax_scale)[r]);
    const float s = m > 0.0f ? m / 448.0f : 1.0f;
    const uint4* row = reinterpret_cast<const uint4*>(w + r * ld_in);
    uint8_t* out = codes + r * ld_out;
    for (int c0 = 0; c0 < cols; c0 += 1024) {
        uint4 v[2][2];
        bool ok[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = c0 + j * 512 + lane * 16;
            ok[j] = e < cols;
            if (ok[j]) {
                v[j][0] = row[e / 8];
                v[j][1] = row[e / 8 + 1];
            }
        }
        __syncwarp();  // every lane's loads of this step precede any store of it
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (!ok[j]) continue;
            float f[16];
            unpack16(v[j][0], v[j][1], f);
            uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(f[k] / s, __NV_SATFINITE, __NV_E4M3);
                packed[k >> 2] |= (uint32_t)c << (8 * (k & 3));
            }
            *reinterpret_cast<uint4*>(out + c0 + j * 512 + lane * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
    __syncwarp();  // every lane has read the max before it is replaced by the scale
    if (lane == 0) amax_scale[r] = s;
}

// Two E4M3 planes per value (bf16 rows carried to the 8-bit-by-8-bit tensor
// cores): q = v / s, hi = E4M3(q), lo = E4M3(q - value(hi)); the fp32
// subtraction is exact.  The planes are interleaved per 128-value block --
// [128 hi codes | 128 lo codes] -- so a block's codes take exactly the 256
// bytes its bf16 values took, and one TMA box of 128 codes loads either plane.
__device__ __forceinline__ void split16(const float (&f)[16], float s, uint4& hi, uint4& lo) {
    uint32_t ph[4] = {0u, 0u, 0u, 0u}, pl[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float q = f[k] / s;
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
        const float vc = __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
        const __nv_fp8_storage_t c2 = __nv_cvt_float_to_fp8(q - vc, __NV_SATFINITE, __NV_E4M3);
        ph[k >> 2] |= (uint32_t)c << (8 * (k & 3));
        pl[k >> 2] |= (uint32_t)c2 << (8 * (k & 3));
    }
    hi = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    lo = make_uint4(pl[0], pl[1], pl[2], pl[3]);
}

// Activation rows (bf16, cols a multiple of 128 and at most 16384) to two
// planes: quantize_act_rows_kernel's block per row with its whole row in
// registers, the scale amax / 448, and values [16 v, 16 v + 16) of block
// b = v / 8 written at bytes 256 b + 16 (v % 8) (hi) and 256 b + 128 + 16 (v % 8)
// (lo) of the row's 2 * cols bytes at codes + r * ld_out.
__global__ void __launch_bounds__(kQuantThreads)
split_act_rows_kernel(const bf16* w, int64_t ld_in, uint8_t* codes, int64_t ld_out,
                      float* __restrict__ scales, int cols) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kQuantThreads / 32];
    const int64_t r = blockIdx.x;
    const uint4* row = reinterpret_cast<const uint4*>(w + r * ld_in);
    const int nvec = cols / 16;
    uint4 v[kActVecs][2];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kActVecs; ++j) {
        const int vi = (int)threadIdx.x + j * kQuantThreads;
        if (vi < nvec) {
            v[j][0] = row[2 * vi];
            v[j][1] = row[2 * vi + 1];
            float f[16];
            unpack16(v[j][0], v[j][1], f);
#pragma unroll
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(f[k]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();  // every load of the row has completed past this point
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kQuantThreads / 32; ++i) m = fmaxf(m, red[i]);
    const float s = m > 0.0f ? m / 448.0f : 1.0f;
    if (threadIdx.x == 0) scales[r] = s;
    uint8_t* out = codes + r * ld_out;
#pragma unroll
    for (int j = 0; j < kActVecs; ++j) {
        const int vi = (int)threadIdx.x + j * kQuantThreads;
        if (vi < nvec) {
            float f[16];
            unpack16(v[j][0], v[j][1], f);
            uint4 hi, lo;
            split16(f, s, hi, lo);
            uint8_t* blk = out + (int64_t)(vi >> 3) * 256 + (vi & 7) * 16;
            *reinterpret_cast<uint4*>(blk) = hi;
            *reinterpret_cast<uint4*>(blk + 128) = lo;
        }
    }
}

// Rows whose max |value| is known (raised by the producing GEMM), split into
// two planes in place: one warp per row, four 128-value blocks per step (lane
// l takes values 16 (l % 8) .. of block l / 8), every load of a step before
// any store of it (__syncwarp).  A block's planes land on exactly the 256
// bytes of its bf16 values, all loaded at this step, and later steps read
// only later blocks, so the codes may overwrite the row.
__global__ void __launch_bounds__(kQuantThreads)
split_rows_known_amax_kernel(bf16* w, int64_t ld, float* amax_scale, int cols, int64_t rows) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (r >= rows) return;
    const float m = __uint_as_float(reinterpret_cast<const uint32_t*>(amax_scale)[r]);
    const float s = m > 0.0f ? m / 448.0f : 1.0f;
    bf16* row = w + r * ld;
    for (int c0 = 0; c0 < cols; c0 += 512) {
        const int blk = c0 + (lane >> 3) * 128;    // first value of this lane's block
        const int e = blk + (lane & 7) * 16;       // first of its 16 values
        const bool ok = e < cols;
        uint4 a, b;
        if (ok) {
            a = reinterpret_cast<const uint4*>(row + e)[0];
            b = reinterpret_cast<const uint4*>(row + e)[1];
        }
        __syncwarp();  // every lane's loads of this step precede any store of it
        if (ok) {
            float f[16];
            unpack16(a, b, f);
            uint4 hi, lo;
            split16(f, s, hi, lo);
            uint8_t* dst = reinterpret_cast<uint8_t*>(row + blk) + (lane & 7) * 16;
            *reinterpret_cast<uint4*>(dst) = hi;
            *reinterpret_cast<uint4*>(dst + 128) = lo;
        }
    }
    __syncwarp();  // every lane has read the max before it is replaced by the scale
    if (lane == 0) amax_scale[r] = s;
}

}  // namespace

cudaError_t launch_split_act_rows(int64_t rows, int cols, const void* w, int64_t ld_in,
                                  uint8_t* codes, int64_t ld_out, float* scales, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 128 || cols > kActVecs * kQuantThreads * 16) return cudaErrorInvalidValue;
    return launch_pdl(split_act_rows_kernel, dim3((unsigned)rows), dim3(kQuantThreads), 0, st,
                      (const bf16*)w, ld_in, codes, ld_out, scales, cols);
}

cudaError_t launch_split_rows_known_amax(int64_t rows, int cols, void* w, int64_t ld,
                                         float* amax_scale, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 128) return cudaErrorInvalidValue;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    return launch_pdl(split_rows_known_amax_kernel, dim3((unsigned)blocks), dim3(kQuantThreads), 0,
                      st, (bf16*)w, ld, amax_scale, cols, rows);
}

cudaError_t launch_quantize_rows_known_amax(int64_t rows, int cols, const void* w, int64_t ld_in,
                                            uint8_t* codes, int64_t ld_out, float* amax_scale,
                                            cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 16) return cudaErrorInvalidValue;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    return launch_pdl(quantize_rows_known_amax_kernel, dim3((unsigned)blocks), dim3(kQuantThreads),
                      0, st, (const bf16*)w, ld_in, codes, ld_out, amax_scale, cols, rows);
}

cudaError_t launch_quantize_act_rows(int64_t rows, int cols, const void* w, int64_t ld_in,
                                     uint8_t* codes, int64_t ld_out, float* scales,
                                     cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (cols % 16 || cols > kActVecs * kQuantThreads * 16) return cudaErrorInvalidValue;
    return launch_pdl(quantize_act_rows_kernel, dim3((unsigned)rows), dim3(kQuantThreads), 0, st,
                      (const bf16*)w, ld_in, codes, ld_out, scales, cols);
}

cudaError_t launch_quantize_fp8_blocks(int64_t rows, int64_t cols, int dtype, const void* w,
                                       uint8_t* codes, float* scales, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((cols + kQBlk - 1) / kQBlk), (unsigned)((rows + kQBlk - 1) / kQBlk));
    if (dtype == MOE_BF16)
        return launch_pdl(quantize_blocks_kernel<bf16>, grid, dim3(kQuantThreads), 0, st,
                          (const bf16*)w, codes, scales, rows, cols);
    return launch_pdl(quantize_blocks_kernel<float>, grid, dim3(kQuantThreads), 0, st,
                      (const float*)w, codes, scales, rows, cols);
}

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
