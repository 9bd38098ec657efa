// ffn_gemv_fp8.cu -- stage 3 for small groups with 8-bit (E4M3) expert weights:
// a weight-streaming GEMV.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 1.2: a decode
// expert multiplies one or two token vectors, so the work is a GEMV bound by
// the bytes of its weights; "LLM from scratch, ch. 6", section "second route:
// make every byte cheaper": one byte per weight instead of two halves them.
//
// Design.  On tcgen05 the exact layer needs the codes widened to bf16 in
// shared memory (~7 bytes of shared-memory traffic per byte read from HBM for
// a one-row group), and the 8-bit MMA needs the bf16 activations as two E4M3
// planes and 128 rows (or 16, swapped) per MMA -- measured at DeepSeek-V3
// decode 488 us on that path against this GEMV's 482 us; a CUDA-core dot
// product spends ~5 instructions per code on widening and FMAs.  Here each code goes
// HBM -> register once and is widened with one cvt per two codes (E4M3 ->
// f16, exact); the products run on the warp-level tensor-core instruction
// mma.m16n8k16 (f16 x f16 -> f32); one or two MMAs per A fragment (8 or 16
// token rows of the group per pass, by what fits in shared memory).
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
// weight row's scale.  Row m stores its 8-byte slot s (4 values) at slot
// s ^ (m % 16) of the same 128-byte segment, so the B loads of a half-warp
// (4 token rows x 4 lanes) hit 16 distinct bank pairs.
//
// Work: warp tasks (group, 16 weight rows); each block takes a contiguous
// range of tasks and walks it group by group, staging each group's activation
// rows once.
//
// Block-scaled weights (BLK, one scale per 128 x 128 block): a warp's 16 rows
// lie in one block row, so each 128-code K block has one scale per MMA row
// half; its two 64-code blocks accumulate into fresh registers, which are
// then scaled and added to the running sums (the scale varies along K, so it
// cannot wait for the end of the dot product).
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kG8Warps = 16;
constexpr int kG8Threads = kG8Warps * 32;
constexpr int kG8Tok = 8;           // token rows per MMA (its N)
constexpr int kG8U = 8;             // 64-code K blocks in flight per lane

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
        // block scales: expert grp's block rows follow the previous experts' (I
        // and d are multiples of the block side)
        const int64_t bs = g.wblock ? (int64_t)(g.d / g.wblock) * (g.I / g.wblock) : 0;
        v.sg = g.s_gate + (g.wblock ? grp * bs : (int64_t)grp * g.I);
        v.su = g.s_up + (g.wblock ? grp * bs : (int64_t)grp * g.I);
        v.sd = g.s_down + (g.wblock ? grp * bs : (int64_t)grp * g.d);
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

// 8-byte slot s of staged row m (swizzled within its 128-byte segment)
__device__ __forceinline__ int sw_slot(int s, int m) { return (s & ~15) | ((s & 15) ^ (m & 15)); }

// Stage token rows c0 .. c0+nt-1 of group v (n values each) into act as f16
// scaled by 2^-e_m (rows nt .. rows-1 zero), with rs[m] = 2^e_m.  Routed rows
// come from the permuted copy (row0 + c0 + m), shared rows from the token
// rows.  One warp per row.
__device__ __forceinline__ void stage_f16(__half* act, float* rs, const bf16* routed,
                                          const bf16* shared, const Group8& v, int c0, int nt,
                                          int rows, int n, int warp, int lane,
                                          const int32_t* row_src = nullptr) {
    for (int m = warp; m < rows; m += kG8Warps) {
        uint2* dst = reinterpret_cast<uint2*>(act + (int64_t)m * n);
        if (m >= nt) {
            for (int c = lane; c < n / 4; c += 32) dst[c] = make_uint2(0u, 0u);
            if (lane == 0) rs[m] = 0.0f;
            continue;
        }
        // a routed row: its permuted copy, or (row_src) the token's row of x
        const int64_t prow = v.row0 + c0 + m;
        const int64_t row = v.shared ? (int64_t)(c0 + m) : (row_src ? (int64_t)row_src[prow] : prow);
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
            dst[sw_slot(2 * c, m)] = make_uint2(hw[0], hw[1]);
            dst[sw_slot(2 * c + 1, m)] = make_uint2(hw[2], hw[3]);
        }
    }
}

__device__ __forceinline__ void prefetch_l2(const void* a) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// c[nt] += weight rows (p0: MMA rows 0-7 via the lane's group g, p1: rows
// 8-15) of n codes times staged token rows 8 nt .. 8 nt + 7.  pf: while a
// step's kG8U blocks are in flight, the four lanes of each row ask L2 for the
// row's next kG8U blocks (512 bytes, one 128-byte line per lane), so the next
// step's loads find them in L2 -- twice the weight bytes in flight per SM
// without holding more registers.
// BLK: sc0 / sc1 are the block scales of rows p0 / p1 along K (one per 128
// codes); each 128-code block's products are scaled before they are summed.
template <int NTILE, int R, bool BLK = false>
__device__ __forceinline__ void mma_rows(const uint8_t* p0, const uint8_t* p1, int n,
                                         const __half* act, int lane, float (&c)[NTILE][4],
                                         int pf, const float* sc0 = nullptr,
                                         const float* sc1 = nullptr) {
    const int g = lane >> 2, t = lane & 3;
    const int nkb = n / 64;
    const uint8_t* const row0 = p0;
    const uint8_t* const row1 = p1;
    const uint2* arow[NTILE];
#pragma unroll
    for (int j = 0; j < NTILE; ++j)  // (rows past R are never read)
        arow[j] = reinterpret_cast<const uint2*>(act + (int64_t)min(8 * j + g, R - 1) * n);
    p0 += 16 * t;
    p1 += 16 * t;
    // BLK: the scales of a step are loaded one step ahead (measured on GB300,
    // DeepSeek-V3 decode: 515 -> 502 us per layer; loading them in the step that
    // uses them left the products waiting on the loads)
    constexpr int kSB = kG8U / 2;  // 128-code scale blocks per step
    float n0[kSB], n1[kSB];
    if constexpr (BLK) {
#pragma unroll
        for (int b = 0; b < kSB; ++b) {
            const bool ok = 2 * b < nkb;
            n0[b] = ok ? __ldg(sc0 + b) : 0.0f;
            n1[b] = ok ? __ldg(sc1 + b) : 0.0f;
        }
    }
    for (int kb0 = 0; kb0 < nkb; kb0 += kG8U) {
        if (pf) {
            const int off = (kb0 + pf * kG8U) * 64 + 128 * t;  // inside the row: off < n
            if (off < n) {
                prefetch_l2(row0 + off);
                prefetch_l2(row1 + off);
            }
        }
        float s0[kSB], s1[kSB];
        if constexpr (BLK) {  // this step's scales; the next step's requested
#pragma unroll
            for (int b = 0; b < kSB; ++b) {
                s0[b] = n0[b];
                s1[b] = n1[b];
                const bool ok = kb0 + kG8U + 2 * b < nkb;
                n0[b] = ok ? __ldg(sc0 + ((kb0 + kG8U) / 2 + b)) : 0.0f;
                n1[b] = ok ? __ldg(sc1 + ((kb0 + kG8U) / 2 + b)) : 0.0f;
            }
        }
        if (BLK && kb0 + kG8U <= nkb) {
            // BLK, a whole step: loads without bounds tests, and the B slots
            // as a base per (tile, kk) plus 16 slots per block.  Measured on
            // GB300 (DeepSeek-V3 shapes, interleaved runs, identical bits):
            // this step leaves the block-scaled kernels without register
            // spills -- decode T=8 478 vs 502 us per layer, T=1 141 vs 148,
            // T=64 1615 vs 1662.  Row scales keep the general step below
            // (with this one: T=8 474 vs 479 us but T=64 1604 vs 1593).
            uint4 w0[kG8U], w1[kG8U];
            const uint8_t* q0 = p0 + (int64_t)kb0 * 64;
            const uint8_t* q1 = p1 + (int64_t)kb0 * 64;
#pragma unroll
            for (int u = 0; u < kG8U; ++u) {
                w0[u] = ld_stream(q0 + u * 64);
                w1[u] = ld_stream(q1 + u * 64);
            }
            const uint2* bb[NTILE][4];
#pragma unroll
            for (int j = 0; j < NTILE; ++j)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    bb[j][kk] = arow[j] + 16 * kb0 + ((4 * t + kk) ^ ((8 * j + g) & 15));
            float cp[NTILE][4];
#pragma unroll
            for (int u = 0; u < kG8U; ++u) {
                if (BLK && (u & 1) == 0) {
#pragma unroll
                    for (int j = 0; j < NTILE; ++j) cp[j][0] = cp[j][1] = cp[j][2] = cp[j][3] = 0.0f;
                }
                const uint32_t r0[4] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w};
                const uint32_t r1[4] = {w1[u].x, w1[u].y, w1[u].z, w1[u].w};
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t a0 = e4m3x2_to_f16x2(r0[kk]), a1 = e4m3x2_to_f16x2(r1[kk]);
                    const uint32_t a2 = e4m3x2_to_f16x2(r0[kk] >> 16), a3 = e4m3x2_to_f16x2(r1[kk] >> 16);
#pragma unroll
                    for (int j = 0; j < NTILE; ++j) {
                        const uint2 b = (R >= 8 * (j + 1) || 8 * j + g < R) ? bb[j][kk][16 * u]
                                                                           : make_uint2(0u, 0u);
                        if constexpr (BLK) mma16816(cp[j], a0, a1, a2, a3, b.x, b.y);
                        else mma16816(c[j], a0, a1, a2, a3, b.x, b.y);
                    }
                }
                if (BLK && (u & 1) == 1) {
#pragma unroll
                    for (int j = 0; j < NTILE; ++j) {
                        c[j][0] = fmaf(s0[u >> 1], cp[j][0], c[j][0]);
                        c[j][1] = fmaf(s0[u >> 1], cp[j][1], c[j][1]);
                        c[j][2] = fmaf(s1[u >> 1], cp[j][2], c[j][2]);
                        c[j][3] = fmaf(s1[u >> 1], cp[j][3], c[j][3]);
                    }
                }
            }
            continue;
        }
        uint4 w0[kG8U], w1[kG8U];
#pragma unroll
        for (int u = 0; u < kG8U; ++u) {
            const bool ok = kb0 + u < nkb;
            w0[u] = ok ? ld_stream(p0 + (int64_t)(kb0 + u) * 64) : make_uint4(0, 0, 0, 0);
            w1[u] = ok ? ld_stream(p1 + (int64_t)(kb0 + u) * 64) : make_uint4(0, 0, 0, 0);
        }
        float cp[NTILE][4];  // BLK: the current 128-code block's products
#pragma unroll
        for (int u = 0; u < kG8U; ++u) {
            if (kb0 + u >= nkb) break;
            if (BLK && (u & 1) == 0) {
#pragma unroll
                for (int j = 0; j < NTILE; ++j) cp[j][0] = cp[j][1] = cp[j][2] = cp[j][3] = 0.0f;
            }
            const uint32_t r0[4] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w};
            const uint32_t r1[4] = {w1[u].x, w1[u].y, w1[u].z, w1[u].w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t a0 = e4m3x2_to_f16x2(r0[kk]), a1 = e4m3x2_to_f16x2(r1[kk]);
                const uint32_t a2 = e4m3x2_to_f16x2(r0[kk] >> 16), a3 = e4m3x2_to_f16x2(r1[kk] >> 16);
                const int slot = 16 * (kb0 + u) + 4 * t + kk;
#pragma unroll
                for (int j = 0; j < NTILE; ++j) {
                    // token rows past the R staged ones are zero columns
                    const uint2 b = (R >= 8 * (j + 1) || 8 * j + g < R) ? arow[j][sw_slot(slot, 8 * j + g)]
                                                                       : make_uint2(0u, 0u);
                    if constexpr (BLK) mma16816(cp[j], a0, a1, a2, a3, b.x, b.y);
                    else mma16816(c[j], a0, a1, a2, a3, b.x, b.y);
                }
            }
            if (BLK && (u & 1) == 1) {  // n is a multiple of 128: u = 1, 3, ... closes a block
#pragma unroll
                for (int j = 0; j < NTILE; ++j) {
                    c[j][0] = fmaf(s0[u >> 1], cp[j][0], c[j][0]);
                    c[j][1] = fmaf(s0[u >> 1], cp[j][1], c[j][1]);
                    c[j][2] = fmaf(s1[u >> 1], cp[j][2], c[j][2]);
                    c[j][3] = fmaf(s1[u >> 1], cp[j][3], c[j][3]);
                }
            }
        }
    }
}

// contiguous task range of this block
__device__ __forceinline__ void task_range(int64_t tasks, int64_t& u0, int64_t& u1) {
    u0 = tasks * blockIdx.x / gridDim.x;
    u1 = tasks * (blockIdx.x + 1) / gridDim.x;
}

// One warp, gate/up: intermediate rows i0 .. i0+7 (MMA rows 0-7 gate, 8-15 up)
// for staged token rows 0 .. nt-1 (nt <= 8 NTILE).
template <int NTILE, int R, bool BLK>
__device__ __forceinline__ void gate_up_task(const FfnGroups& g, const Group8& v, int i0, int c0,
                                             int nt, const __half* act, const float* rs, int lane) {
    const int t = lane & 3;
    const int i = i0 + (lane >> 2);
    float c[NTILE][4];
#pragma unroll
    for (int j = 0; j < NTILE; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
    // BLK: the scales of the block row holding rows i0 .. i0 + 7
    const int64_t brow = BLK ? (int64_t)(i0 / kWBlock) * (g.d / kWBlock) : 0;
    mma_rows<NTILE, R, BLK>(v.wg + (int64_t)i * g.d, v.wu + (int64_t)i * g.d, g.d, act, lane, c,
                            g.g8_prefetch, v.sg + brow, v.su + brow);
    const float sg = BLK ? 1.0f : v.sg[i], su = BLK ? 1.0f : v.su[i];
#pragma unroll
    for (int j = 0; j < NTILE; ++j)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int tok = 8 * j + 2 * t + q;
            if (tok < nt) {
                const float gv = c[j][q] * rs[tok] * sg, uv = c[j][2 + q] * rs[tok] * su;
                bf16* h = v.shared ? (bf16*)g.h_s + (int64_t)(c0 + tok) * v.inter
                                   : (bf16*)g.h + (v.row0 + c0 + tok) * v.inter;
                h[i] = __float2bfloat16_rn(silu_mul(gv, uv));
            }
        }
}

// One warp, down: output rows j0 .. j0+15 for staged token rows 0 .. nt-1.
template <int NTILE, int R, bool BLK>
__device__ __forceinline__ void down_task(const FfnGroups& g, const Group8& v, int j0, int c0,
                                          int nt, const __half* act, const float* rs, int lane) {
    const int t = lane & 3;
    const int jr = j0 + (lane >> 2);
    float c[NTILE][4];
#pragma unroll
    for (int j = 0; j < NTILE; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
    // BLK: rows j0 .. j0 + 15 share one block row
    const float* bs = v.sd + (BLK ? (int64_t)(j0 / kWBlock) * (v.inter / kWBlock) : 0);
    mma_rows<NTILE, R, BLK>(v.wd + (int64_t)jr * v.inter, v.wd + (int64_t)(jr + 8) * v.inter,
                            v.inter, act, lane, c, g.g8_prefetch, bs, bs);
    const float s0 = BLK ? 1.0f : v.sd[jr], s1 = BLK ? 1.0f : v.sd[jr + 8];
#pragma unroll
    for (int j = 0; j < NTILE; ++j)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int tok = 8 * j + 2 * t + q;
            if (tok < nt) {
                bf16* y = v.shared ? (bf16*)g.y_s + (int64_t)(c0 + tok) * g.d
                                   : (bf16*)g.y + (v.row0 + c0 + tok) * g.d;
                y[jr] = __float2bfloat16_rn(c[j][q] * rs[tok] * s0);
                y[jr + 8] = __float2bfloat16_rn(c[j][2 + q] * rs[tok] * s1);
            }
        }
}

// h = SiLU(s_g * (Q_gate x)) * (s_u * (Q_up x)) for the groups of one GEMV
// list (which = 0: first list, 1: second), up to R token rows per pass; a pass
// of at most 8 rows runs one MMA per A fragment.
template <int R, bool BLK>
__global__ void __launch_bounds__(kG8Threads, 1)
gemv8_gate_up_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                     const int32_t* __restrict__ list, int which) {
    pdl_wait();
    pdl_trigger();
    constexpr int NT = (R + kG8Tok - 1) / kG8Tok;
    extern __shared__ __align__(16) unsigned char smem8[];
    float* rs = reinterpret_cast<float*>(smem8);          // [R] 2^e of each token row
    __half* act = reinterpret_cast<__half*>(smem8 + 64);  // [R][d], swizzled slots
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const int tpg = max_inter / 8;  // tasks per group
    int64_t u, u1;
    task_range((int64_t)(which ? hdr->n_gemv2 : hdr->n_gemv) * tpg, u, u1);
    while (u < u1) {
        const int a = (int)(u / tpg);
        const Group8 v = group8(g, list[a]);
        const int64_t seg_end = min(u1, (int64_t)(a + 1) * tpg);
        for (int c0 = 0; c0 < v.rows; c0 += R) {
            const int nt = min(R, v.rows - c0);
            const int rows = (NT == 1 || nt <= kG8Tok) ? min(R, kG8Tok) : R;
            __syncthreads();  // earlier readers of act are done
            stage_f16(act, rs, (const bf16*)g.a_routed, (const bf16*)g.a_shared, v, c0, nt, rows,
                      g.d, warp, lane, g.row_src);
            __syncthreads();
            for (int64_t k = u + warp; k < seg_end; k += kG8Warps) {
                const int i0 = (int)(k - (int64_t)a * tpg) * 8;
                if (i0 >= v.inter) continue;  // warp-uniform
                if (NT == 1 || nt <= kG8Tok) gate_up_task<1, (R < kG8Tok ? R : kG8Tok), BLK>(g, v, i0, c0, nt, act, rs, lane);
                else gate_up_task<NT, R, BLK>(g, v, i0, c0, nt, act, rs, lane);
            }
        }
        u = seg_end;
    }
}

// y = s_d * (Q_down h) for the groups of one GEMV list, up to R token rows per pass.
template <int R, bool BLK>
__global__ void __launch_bounds__(kG8Threads, 1)
gemv8_down_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                  const int32_t* __restrict__ list, int which) {
    pdl_wait();
    pdl_trigger();
    constexpr int NT = (R + kG8Tok - 1) / kG8Tok;
    extern __shared__ __align__(16) unsigned char smem8[];
    float* rs = reinterpret_cast<float*>(smem8);
    __half* act = reinterpret_cast<__half*>(smem8 + 64);  // [R][inter], swizzled slots
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tpg = g.d / 16;
    int64_t u, u1;
    task_range((int64_t)(which ? hdr->n_gemv2 : hdr->n_gemv) * tpg, u, u1);
    while (u < u1) {
        const int a = (int)(u / tpg);
        const Group8 v = group8(g, list[a]);
        const int64_t seg_end = min(u1, (int64_t)(a + 1) * tpg);
        for (int c0 = 0; c0 < v.rows; c0 += R) {
            const int nt = min(R, v.rows - c0);
            const int rows = (NT == 1 || nt <= kG8Tok) ? min(R, kG8Tok) : R;
            __syncthreads();
            stage_f16(act, rs, (const bf16*)g.h, (const bf16*)g.h_s, v, c0, nt, rows, v.inter, warp,
                      lane);
            __syncthreads();
            for (int64_t k = u + warp; k < seg_end; k += kG8Warps) {
                const int j0 = (int)(k - (int64_t)a * tpg) * 16;
                if (NT == 1 || nt <= kG8Tok) down_task<1, (R < kG8Tok ? R : kG8Tok), BLK>(g, v, j0, c0, nt, act, rs, lane);
                else down_task<NT, R, BLK>(g, v, j0, c0, nt, act, rs, lane);
            }
        }
        u = seg_end;
    }
}

size_t gemv8_smem(int n, int rows) { return 64 + (size_t)rows * n * sizeof(__half); }

constexpr int kG8Small = 8;  // rows of the first GEMV list's groups (one MMA column tile)

// Shared memory a launch may use and still leave L1 room for the weight loads
// in flight (measured: the same kernel streams at ~50% of HBM with a 229 KB
// carve-out and ~85% with 115 KB).
constexpr size_t kG8FastSmem = 120 * 1024;

template <int R, bool BLK>
cudaError_t launch_gu_as(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list, int which,
                         cudaStream_t st) {
    const size_t sm = gemv8_smem(g.d, R);
    cudaError_t e = cudaFuncSetAttribute(gemv8_gate_up_kernel<R, BLK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv8_gate_up_kernel<R, BLK>, dim3(device_sm_count()), dim3(kG8Threads), sm, st, g,
                      hdr, list, which);
}

template <int R>
cudaError_t launch_gu(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list, int which,
                      cudaStream_t st) {
    return g.wblock ? launch_gu_as<R, true>(g, hdr, list, which, st)
                    : launch_gu_as<R, false>(g, hdr, list, which, st);
}

template <int R, bool BLK>
cudaError_t launch_dn_as(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list, int which,
                         int max_inter, cudaStream_t st) {
    const size_t sm = gemv8_smem(max_inter, R);
    cudaError_t e = cudaFuncSetAttribute(gemv8_down_kernel<R, BLK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv8_down_kernel<R, BLK>, dim3(device_sm_count()), dim3(kG8Threads), sm, st, g,
                      hdr, list, which);
}

template <int R>
cudaError_t launch_dn(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list, int which,
                      int max_inter, cudaStream_t st) {
    return g.wblock ? launch_dn_as<R, true>(g, hdr, list, which, max_inter, st)
                    : launch_dn_as<R, false>(g, hdr, list, which, max_inter, st);
}

}  // namespace

// Groups of at most this many rows take the 8-bit GEMV path (MOE_GEMV8_MAX_ROWS,
// read on every call; default 8 -- one MMA column tile; 0 sends every group to
// the tcgen05 path; larger values use the second list, 16 rows per pass).
// Measured on GB300 (DeepSeek-V3 shapes): 8 and 16 tie at T = 8, 8 is 3% faster
// at T = 64 and 16 is 0.8% faster at T = 512.
int gemv8_max_rows() {
    const char* s = getenv("MOE_GEMV8_MAX_ROWS");
    const int x = s ? atoi(s) : kG8Tok;
    return x < 0 ? 0 : x;
}

bool gemv8_fits(int widest) { return gemv8_smem(widest, kG8Tok) <= kGemv8SmemLimit; }

int gemv8_small_rows() { return kG8Small; }

// First list (groups of 1..8 rows): 8 staged rows, one MMA per A fragment.
// Second list (9..limit rows): 16 rows per pass where they fit in
// kG8FastSmem, else passes of 8.  Both lists' gate/up kernels run before the
// down kernels that read their h.
cudaError_t launch_ffn_gemv_fp8(const FfnGroups& g0, const FfnPlanHeader* hdr, const int32_t* list,
                                int limit, cudaStream_t st) {
    FfnGroups g = g0;
    // read per call: how many steps ahead the L2 prefetch runs (0: off)
    const char* pfe = getenv("MOE_G8_PREFETCH");
    g.g8_prefetch = pfe ? atoi(pfe) : 1;
    if (g.g8_prefetch < 0 || g.g8_prefetch > 4) g.g8_prefetch = 1;
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const int32_t* list2 = list + (g.E + 1);
    const bool second = limit > kG8Small;
    const bool gu16 = gemv8_smem(g.d, 2 * kG8Tok) <= kG8FastSmem;
    const bool dn16 = gemv8_smem(max_inter, 2 * kG8Tok) <= kG8FastSmem;
    cudaError_t e = launch_gu<kG8Small>(g, hdr, list, 0, st);
    if (e == cudaSuccess && second)
        e = gu16 ? launch_gu<2 * kG8Tok>(g, hdr, list2, 1, st) : launch_gu<kG8Tok>(g, hdr, list2, 1, st);
    if (e == cudaSuccess) e = launch_dn<kG8Small>(g, hdr, list, 0, max_inter, st);
    if (e == cudaSuccess && second)
        e = dn16 ? launch_dn<2 * kG8Tok>(g, hdr, list2, 1, max_inter, st)
                 : launch_dn<kG8Tok>(g, hdr, list2, 1, max_inter, st);
    return e;
}

}  // namespace moe
