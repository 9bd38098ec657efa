// common.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// device error word (first 16 bytes of every workspace)
// ---------------------------------------------------------------------------
struct DevError {
    int32_t code;    // moe_status (0 = none); first error wins
    int32_t where;   // kernel-specific detail (which wait / which index)
    int32_t pad[2];
};

__device__ __forceinline__ void record_error(DevError* err, int32_t code, int32_t where) {
    if (err != nullptr && atomicCAS(&err->code, 0, code) == 0) err->where = where;
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
using bf16 = __nv_bfloat16;

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static float to_f32(float v) { return v; }
    __device__ __forceinline__ static float from_f32(float v) { return v; }
};
template <> struct Elem<bf16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static float to_f32(bf16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static bf16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// unpack one 16-byte vector into fp32 values
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4], const float*) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], const bf16*) {
    // bf16 -> fp32 is a 16-bit shift of the bit pattern
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
}

// streaming 16-byte load that bypasses L1 allocation (weights are read once)
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// read-only 16-byte load through L1 (activations reused across warps)
__device__ __forceinline__ uint4 ld_ro(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// SiLU(g) * u in fp32: g / (1 + e^-g) * u, with the CUDA fast exponential and
// fast division (a few ulp; for g < -87 the denominator overflows and the
// result is 0).  Measured on the tcgen05 gate/up epilogue: the IEEE division
// cost 6 % of an 8-bit prefill layer call.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel calls pdl_wait() before it
// touches global memory that an earlier kernel of the stream writes or reads
// (the wait returns once the preceding grid has completed and its writes are
// visible; without a programmatic dependency it returns at once), and
// pdl_trigger() to let the next kernel of the stream be scheduled onto SMs as
// they free up, so its launch and prologue overlap this kernel's tail.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

}  // namespace moe
