// ffn_gemv_fp8.cu -- stage 3 for small groups with 8-bit (E4M3) expert weights:
// a weight-streaming GEMV.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 1.2: a decode
// expert multiplies one or two token vectors, so the work is a GEMV bound by
// the bytes of its weights; "LLM from scratch, ch. 6", section "second route:
// make every byte cheaper": one byte per weight instead of two halves them.
//
// Design.  tcgen05 would need the codes widened to bf16 in shared memory
// (~7 bytes of shared-memory traffic per byte read from HBM for a one-row
// group), and a CUDA-core dot product spends ~5 instructions per code on
// widening and FMAs; both stay far below the HBM rate.  Here each code goes
// HBM -> register once and is widened with one cvt per two codes (E4M3 ->
// f16, exact); the products run on the warp-level tensor-core instruction
// mma.m16n8k16 (f16 x f16 -> f32), whose N = 8 columns hold up to 8 token
// rows of the group.
//
// A warp owns 16 weight rows (gate/up: 8 gate rows and the 8 up rows of the
// same intermediate indices, so SiLU(g) * u is formed in the accumulator
// registers; down: 16 output rows).  Lane (g, t) = (lane / 4, lane % 4)
// loads 16 consecutive codes of rows g and g + 8 at K offset 16 t of each
// 64-code block, eight blocks in flight (256 bytes per lane, 128 KB per SM).
// The MMA's K order is a permutation of the true K order, the same for both
// operands (a dot product does not depend on the order of its terms): in the
// block's MMA number kk, lane t's fragment slots {2t, 2t+1} hold codes
// 16t+4kk+{0,1} and slots {2t+8, 2t+9} hold codes 16t+4kk+{2,3}; so A is one
// cvt of each 16-bit half of the lane's loaded words, and B is one 8-byte
// shared-memory load of the same four activation values.
//
// Activations: bf16 rows are staged in shared memory as f16, each token row
// scaled by an exact power of two 2^-e so that its largest magnitude lies in
// [2^14, 2^15): every bf16 value within 2^29 of the row maximum is exact in
// f16 and nothing overflows.  The fp32 sums are multiplied by 2^e and by the
// weight row's scale.
//
// Work: warp tasks (group, 16 weight rows); each block takes a contiguous
// range of tasks and walks it group by group, staging each group's activation
// rows once.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kG8Warps = 16;
constexpr int kG8Threads = kG8Warps * 32;
constexpr int kG8Tok = kGemv8Rows;  // activation rows per pass = MMA N (8)
constexpr int kG8U = 8;             // 64-code K blocks in flight per lane
constexpr int kG8Pad = 4;           // f16 padding per staged row (conflict-free B loads)
static_assert(kG8Tok == 8, "the MMA has 8 columns");

struct Group8 {
    int rows;
    int64_t row0;  // first routed row (0 for the shared group)
    bool shared;
    int inter;
    const uint8_t *wg, *wu, *wd;
    const float *sg, *su, *sd;
};

__device__ __forceinline__ Group8 group8(const FfnGroups& g, int grp) {
    Group8 v;
    if (grp < g.E) {
        const int32_t o0 = g.offsets[grp];
        v.rows = g.offsets[grp + 1] - o0;
        v.row0 = o0;
        v.shared = false;
        v.inter = g.I;
        const int64_t w = (int64_t)grp * g.I * g.d;
        v.wg = (const uint8_t*)g.w_gate + w;
        v.wu = (const uint8_t*)g.w_up + w;
        v.wd = (const uint8_t*)g.w_down + w;  // [E][d][I]: the same stride d*I
        v.sg = g.s_gate + (int64_t)grp * g.I;
        v.su = g.s_up + (int64_t)grp * g.I;
        v.sd = g.s_down + (int64_t)grp * g.d;
    } else {
        v.rows = g.T;
        v.row0 = 0;
        v.shared = true;
        v.inter = g.Is;
        v.wg = (const uint8_t*)g.ws_gate;
        v.wu = (const uint8_t*)g.ws_up;
        v.wd = (const uint8_t*)g.ws_down;
        v.sg = g.ss_gate;
        v.su = g.ss_up;
        v.sd = g.ss_down;
    }
    return v;
}

// two E4M3 codes (low byte first) -> f16x2 (low half first), exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return (uint32_t)hr.x | ((uint32_t)hr.y << 16);
}

// D += A(16x16, f16) * B(16x8, f16), fp32 accumulators
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Stage token rows c0 .. c0+nt-1 of group v (n values each) into act as f16
// scaled by 2^-e_m (rows nt..7 zero), with rs[m] = 2^e_m.  Routed rows come
// from the permuted copy (row0 + c0 + m), shared rows from the token rows.
// One warp per row.
__device__ __forceinline__ void stage_f16(__half* act, float* rs, const bf16* routed,
                                          const bf16* shared, const Group8& v, int c0, int nt,
                                          int n, int warp, int lane) {
    const int ld = n + kG8Pad;
    for (int m = warp; m < kG8Tok; m += kG8Warps) {
        uint2* dst = reinterpret_cast<uint2*>(act + (int64_t)m * ld);
        if (m >= nt) {
            for (int c = lane; c < n / 4; c += 32) dst[c] = make_uint2(0u, 0u);
            if (lane == 0) rs[m] = 0.0f;
            continue;
        }
        const int64_t row = v.shared ? (int64_t)(c0 + m) : v.row0 + c0 + m;
        const uint4* src = reinterpret_cast<const uint4*>((v.shared ? shared : routed) + row * n);
        float amax = 0.0f;
#pragma unroll 4
        for (int c = lane; c < n / 8; c += 32) {
            float f[8];
            unpack(ld_ro(src + c), f, (const bf16*)nullptr);
#pragma unroll
            for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int ex = 0;
        frexpf(amax, &ex);                  // amax = f 2^ex, 0.5 <= f < 1
        int e = amax > 0.0f ? ex - 15 : 0;  // amax 2^-e in [2^14, 2^15)
        e = max(-100, min(100, e));
        const float down = __int_as_float((127 - e) << 23);  // 2^-e, exact
        if (lane == 0) rs[m] = __int_as_float((127 + e) << 23);
#pragma unroll 4
        for (int c = lane; c < n / 8; c += 32) {
            float f[8];
            unpack(ld_ro(src + c), f, (const bf16*)nullptr);
            uint32_t hw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __half2 h2 = __floats2half2_rn(f[2 * k] * down, f[2 * k + 1] * down);
                hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[2 * c] = make_uint2(hw[0], hw[1]);
            dst[2 * c + 1] = make_uint2(hw[2], hw[3]);
        }
    }
}

// c += weight rows (p0: M rows 0-7 via lane group g, p1: M rows 8-15) of n
// codes times the staged activations (8 token columns)
__device__ __forceinline__ void mma_rows(const uint8_t* p0, const uint8_t* p1, int n,
                                         const __half* act, int lane, float (&c)[4]) {
    const int g = lane >> 2, t = lane & 3;
    const int nkb = n / 64;
    const __half* brow = act + (int64_t)g * (n + kG8Pad) + 16 * t;
    p0 += 16 * t;
    p1 += 16 * t;
    for (int kb0 = 0; kb0 < nkb; kb0 += kG8U) {
        uint4 w0[kG8U], w1[kG8U];
#pragma unroll
        for (int u = 0; u < kG8U; ++u) {
            const bool ok = kb0 + u < nkb;
            w0[u] = ok ? ld_stream(p0 + (int64_t)(kb0 + u) * 64) : make_uint4(0, 0, 0, 0);
            w1[u] = ok ? ld_stream(p1 + (int64_t)(kb0 + u) * 64) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kG8U; ++u) {
            if (kb0 + u >= nkb) break;
            const uint32_t r0[4] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w};
            const uint32_t r1[4] = {w1[u].x, w1[u].y, w1[u].z, w1[u].w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint2 b = *reinterpret_cast<const uint2*>(brow + (kb0 + u) * 64 + 4 * kk);
                mma16816(c, e4m3x2_to_f16x2(r0[kk]), e4m3x2_to_f16x2(r1[kk]),
                         e4m3x2_to_f16x2(r0[kk] >> 16), e4m3x2_to_f16x2(r1[kk] >> 16), b.x, b.y);
            }
        }
    }
}

// contiguous task range of this block
__device__ __forceinline__ void task_range(int64_t tasks, int64_t& u0, int64_t& u1) {
    u0 = tasks * blockIdx.x / gridDim.x;
    u1 = tasks * (blockIdx.x + 1) / gridDim.x;
}

// h = SiLU(s_g * (Q_gate x)) * (s_u * (Q_up x)) for the GEMV groups.
// Warp task: intermediate rows i0 .. i0+7 (MMA rows 0-7 gate, 8-15 up).
__global__ void __launch_bounds__(kG8Threads, 1)
gemv8_gate_up_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                     const int32_t* __restrict__ gemv_list) {
    extern __shared__ __align__(16) unsigned char smem8[];
    float* rs = reinterpret_cast<float*>(smem8);               // [8] 2^e of each token row
    __half* act = reinterpret_cast<__half*>(smem8 + 64);       // [8][d + pad]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, t = lane & 3;
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const int tpg = max_inter / 8;  // tasks per group
    int64_t u, u1;
    task_range((int64_t)hdr->n_gemv * tpg, u, u1);
    while (u < u1) {
        const int a = (int)(u / tpg);
        const Group8 v = group8(g, gemv_list[a]);
        const int64_t seg_end = min(u1, (int64_t)(a + 1) * tpg);
        for (int c0 = 0; c0 < v.rows; c0 += kG8Tok) {
            const int nt = min(kG8Tok, v.rows - c0);
            __syncthreads();  // earlier readers of act are done
            stage_f16(act, rs, (const bf16*)g.a_routed, (const bf16*)g.a_shared, v, c0, nt, g.d,
                      warp, lane);
            __syncthreads();
            for (int64_t k = u + warp; k < seg_end; k += kG8Warps) {
                const int i0 = (int)(k - (int64_t)a * tpg) * 8;
                if (i0 >= v.inter) continue;  // warp-uniform
                const int i = i0 + gq;
                float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_rows(v.wg + (int64_t)i * g.d, v.wu + (int64_t)i * g.d, g.d, act, lane, c);
                const float sg = v.sg[i], su = v.su[i];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int tok = 2 * t + q;
                    if (tok < nt) {
                        const float gv = c[q] * rs[tok] * sg, uv = c[2 + q] * rs[tok] * su;
                        bf16* h = v.shared ? (bf16*)g.h_s + (int64_t)(c0 + tok) * v.inter
                                           : (bf16*)g.h + (v.row0 + c0 + tok) * v.inter;
                        h[i] = __float2bfloat16_rn(silu_mul(gv, uv));
                    }
                }
            }
        }
        u = seg_end;
    }
}

// y = s_d * (Q_down h) for the GEMV groups.  Warp task: output rows j0 .. j0+15.
__global__ void __launch_bounds__(kG8Threads, 1)
gemv8_down_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                  const int32_t* __restrict__ gemv_list) {
    extern __shared__ __align__(16) unsigned char smem8[];
    float* rs = reinterpret_cast<float*>(smem8);
    __half* act = reinterpret_cast<__half*>(smem8 + 64);       // [8][inter + pad]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, t = lane & 3;
    const int tpg = g.d / 16;
    int64_t u, u1;
    task_range((int64_t)hdr->n_gemv * tpg, u, u1);
    while (u < u1) {
        const int a = (int)(u / tpg);
        const Group8 v = group8(g, gemv_list[a]);
        const int64_t seg_end = min(u1, (int64_t)(a + 1) * tpg);
        for (int c0 = 0; c0 < v.rows; c0 += kG8Tok) {
            const int nt = min(kG8Tok, v.rows - c0);
            __syncthreads();
            stage_f16(act, rs, (const bf16*)g.h, (const bf16*)g.h_s, v, c0, nt, v.inter, warp, lane);
            __syncthreads();
            for (int64_t k = u + warp; k < seg_end; k += kG8Warps) {
                const int j0 = (int)(k - (int64_t)a * tpg) * 16;
                const int j = j0 + gq;
                float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_rows(v.wd + (int64_t)j * v.inter, v.wd + (int64_t)(j + 8) * v.inter, v.inter,
                         act, lane, c);
                const float s0 = v.sd[j], s1 = v.sd[j + 8];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int tok = 2 * t + q;
                    if (tok < nt) {
                        bf16* y = v.shared ? (bf16*)g.y_s + (int64_t)(c0 + tok) * g.d
                                           : (bf16*)g.y + (v.row0 + c0 + tok) * g.d;
                        y[j] = __float2bfloat16_rn(c[q] * rs[tok] * s0);
                        y[j + 8] = __float2bfloat16_rn(c[2 + q] * rs[tok] * s1);
                    }
                }
            }
        }
        u = seg_end;
    }
}

size_t gemv8_smem(int n) { return 64 + (size_t)kG8Tok * (n + kG8Pad) * sizeof(__half); }

}  // namespace

// Groups of at most this many rows take the 8-bit GEMV path (MOE_GEMV8_MAX_ROWS,
// read on every call; default 8 -- one MMA column per row; 0 sends every group
// to the tcgen05 path; larger values take several passes of 8 rows).
int gemv8_max_rows() {
    const char* s = getenv("MOE_GEMV8_MAX_ROWS");
    const int x = s ? atoi(s) : kG8Tok;
    return x < 0 ? 0 : x;
}

bool gemv8_fits(int widest) { return gemv8_smem(widest) <= kGemv8SmemLimit; }

cudaError_t launch_ffn_gemv_fp8(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list,
                                cudaStream_t st) {
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const size_t smem_gu = gemv8_smem(g.d), smem_dn = gemv8_smem(max_inter);
    cudaError_t e = cudaFuncSetAttribute(gemv8_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_gu);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv8_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    gemv8_gate_up_kernel<<<sms, kG8Threads, smem_gu, st>>>(g, hdr, list);
    gemv8_down_kernel<<<sms, kG8Threads, smem_dn, st>>>(g, hdr, list);
    return cudaGetLastError();
}

}  // namespace moe
