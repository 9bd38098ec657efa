// ffn_gemv.cu -- stage 3 for groups with few rows: the SwiGLU expert FFN as a
// weight-streaming GEMV, plus the device-side work plan for stage 3.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 1.2: in decode
// an expert gets ~0.25 tokens on average, so its W_gate, W_up and W_down are
// loaded from HBM to multiply one or two vectors -- the work is a GEMV bound
// by memory bandwidth; FAQ Q1: experts with zero tokens are skipped.
// "Computation and Data Movement for Inference", section 16: decode experts
// share little, so what matters is streaming each selected expert once.
//
// Plan kernel (one block): from offsets[], split the groups (routed experts
// and the shared expert) into those with 1..limit rows (GEMV list) and those
// with more (list of 128-row tiles for the tensor-core GEMM).  Nothing on the
// host reads the counts.
//
// GEMV kernels: a work unit is (group, block of output rows).  The unit's
// activation rows (up to MT of them at a time) are staged in shared memory;
// each warp streams whole weight rows with 16-byte non-allocating loads,
// several in flight per lane, and reduces with shuffles.  Gate and up rows of
// the same index are streamed together so SiLU(g) * u is formed in registers.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsGU = 16;   // gate/up output rows per unit (2 per warp)
constexpr int kRowsDown = 16; // down output rows per unit

__device__ int32_t scan_1024(int32_t v, int32_t* sh, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
        int32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        sh[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t r = sh[warp] + incl - v;
    __syncthreads();
    return r;
}

// groups: E routed (+1 shared), up to 1024 per pass of one 1024-thread block.
// A group goes to a GEMV list (1..limit rows: the first list up to `small`
// rows when small > 0, the second list above), to the pair-tile list (at
// least pair_min rows, tiles of pair_m rows) or to the single-tile list
// (tiles of single_m rows).  Tile entries are (group, first row of the group,
// rows of the group, index of the m-tile within the group).
//
// SM split (split_rho > 0): the pair-tile and single-tile GEMMs then run side
// by side, and the plan divides the sms between them in proportion to their
// estimated work, in units of one MMA K step of one tile on one SM: a pair
// tile costs 2 (two SMs), a single-tile group max(tiles, split_rho / 100) --
// its few rows leave it bound by streaming the expert's weights, which costs
// about split_rho / 100 MMA steps per weight K step on one SM.
struct PlanArgs {
    int E, has_shared, T, limit, small, single_m, pair_min, pair_m, max_mtiles;
    int sms, split_rho;
    FfnPlanHeader* hdr;
    int32_t* gemv_list;
    int4* mtile_list;
};

// The plan, run by one 1024-thread block; offsets may point to global or
// shared memory.
__device__ void plan_groups(const int32_t* offsets, const PlanArgs& a) {
    const int E = a.E, has_shared = a.has_shared, T = a.T, limit = a.limit, small = a.small;
    const int single_m = a.single_m, pair_min = a.pair_min, pair_m = a.pair_m;
    const int max_mtiles = a.max_mtiles;
    FfnPlanHeader* hdr = a.hdr;
    int32_t* gemv_list = a.gemv_list;
    int4* mtile_list = a.mtile_list;
    __shared__ int32_t sh[32];
    __shared__ int32_t tot_g, tot_g2, tot_s, tot_p, tot_c, base_g, base_g2, base_s, base_p, base_c;
    if (threadIdx.x == 0) { base_g = 0; base_g2 = 0; base_s = 0; base_p = 0; base_c = 0; }
    __syncthreads();
    int32_t* gemv_list2 = gemv_list + (E + 1);
    int4* pair_list = mtile_list + max_mtiles;
    const int G = E + (has_shared ? 1 : 0);
    for (int g0 = 0; g0 < G; g0 += blockDim.x) {
        const int g = g0 + threadIdx.x;
        int32_t rows = 0, row0 = 0;
        if (g < E) { row0 = offsets[g]; rows = offsets[g + 1] - row0; }
        else if (g < G) { row0 = 0; rows = T; }
        const bool gemv_any = rows > 0 && rows <= limit;
        const bool to_gemv = gemv_any && (small <= 0 || rows <= small);
        const bool to_gemv2 = gemv_any && !to_gemv;
        // pair_min > 0: fixed threshold.  0: the cheaper shape by padded rows
        // over the measured tensor-pipe activity of each shape (pair ~85%,
        // single ~70% on GB300): pair if ceil(r/256)*256/85 < ceil(r/128)*128/70.
        const int64_t pad_p = (int64_t)(rows + pair_m - 1) / pair_m * pair_m;
        const int64_t pad_s = (int64_t)(rows + single_m - 1) / single_m * single_m;
        const bool to_pair = rows > limit && (pair_min > 0 ? rows >= pair_min : pad_p * 70 < pad_s * 85);
        const int32_t st = (rows > limit && !to_pair) ? (rows + single_m - 1) / single_m : 0;
        const int32_t pt = to_pair ? (rows + pair_m - 1) / pair_m : 0;
        const int32_t pg = scan_1024(to_gemv ? 1 : 0, sh, &tot_g);
        const int32_t pg2 = scan_1024(to_gemv2 ? 1 : 0, sh, &tot_g2);
        const int32_t ps = scan_1024(st, sh, &tot_s);
        const int32_t pp = scan_1024(pt, sh, &tot_p);
        (void)scan_1024(st > 0 ? max(st * 100, a.split_rho) : 0, sh, &tot_c);
        if (to_gemv) gemv_list[base_g + pg] = g;
        if (to_gemv2) gemv_list2[base_g2 + pg2] = g;
        for (int32_t i = 0; i < st; ++i) {
            const int32_t slot = base_s + ps + i;
            if (slot < max_mtiles) mtile_list[slot] = make_int4(g, row0, rows, i);
        }
        for (int32_t i = 0; i < pt; ++i) {
            const int32_t slot = base_p + pp + i;
            if (slot < max_mtiles) pair_list[slot] = make_int4(g, row0, rows, i);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            base_g += tot_g; base_g2 += tot_g2; base_s += tot_s; base_p += tot_p; base_c += tot_c;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        hdr->n_gemv = base_g;
        hdr->n_gemv2 = base_g2;
        hdr->n_mtiles = min(base_s, max_mtiles);
        hdr->n_ptiles = min(base_p, max_mtiles);
        const int sms = a.sms;
        int up = sms / 2, us = sms;
        if (a.split_rho > 0) {
            const int64_t cp = 200ll * base_p, cs = base_c;
            if (cp == 0) {
                up = 0;
            } else if (cs == 0) {
                us = 0;
            } else {
                int ss = (int)(((int64_t)sms * cs + (cp + cs) / 2) / (cp + cs));
                ss = max(2, min(sms - 2, ss));
                up = (sms - ss) / 2;
                us = sms - 2 * up;
            }
        }
        hdr->units_pair = up;
        hdr->units_single = us;
    }
}

__global__ void __launch_bounds__(1024)
ffn_plan_kernel(const int32_t* __restrict__ offsets, PlanArgs a) {
    pdl_wait();
    pdl_trigger();
    plan_groups(offsets, a);
}

// Dispatch and plan for a small batch (n = T*K <= 1024 slots, E <= 1024) in
// one block of 1024 threads: thread f holds slot f.  The same results as the
// three dispatch kernels and the plan kernel -- counts, exclusive offsets,
// the permutation stable by flat slot (rank inside the warp from
// __match_any_sync plus the exclusive sum over earlier warps), the token of
// every row, and the plan -- in one launch instead of four.
__global__ void __launch_bounds__(1024)
dispatch_plan_small_kernel(const int32_t* __restrict__ idx, int n, int K, int32_t* __restrict__ counts,
                           int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                           int32_t* __restrict__ inv_perm, int32_t* __restrict__ tok_of,
                           DevError* err, PlanArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t dyn[];
    const int E = a.E;
    int32_t* wcnt = dyn;                // [32 warps][E]: counts, then exclusive prefix over warps
    int32_t* off_sh = dyn + 32 * E;     // [E + 1]
    __shared__ int32_t sh[32];
    __shared__ int32_t total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int f = threadIdx.x;
    int e = f < n ? idx[f] : -1;
    if (f < n && !(e >= 0 && e < E)) {
        record_error(err, MOE_ERR_BOUNDS, 200);
        e = -1;
    }
    if (!(e >= 0 && e < E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    int32_t c = 0;  // thread x < E: the count of expert x
    if (threadIdx.x < E) {
        for (int w = 0; w < 32; ++w) {
            const int32_t t = wcnt[w * E + threadIdx.x];
            wcnt[w * E + threadIdx.x] = c;
            c += t;
        }
    }
    const int32_t off = scan_1024(threadIdx.x < E ? c : 0, sh, &total);
    if (threadIdx.x < E) {
        counts[threadIdx.x] = c;
        offsets[threadIdx.x] = off;
        off_sh[threadIdx.x] = off;
    }
    if (threadIdx.x == 0) {
        offsets[E] = total;
        off_sh[E] = total;
    }
    __syncthreads();
    if (f < n) {
        if (e >= 0) {
            const int32_t p = off_sh[e] + wcnt[warp * E + e] + rank;
            if (perm) perm[p] = f;
            inv_perm[f] = p;
            tok_of[p] = f / K;
        } else {
            inv_perm[f] = -1;  // dropped slot (out-of-range expert id)
        }
    }
    plan_groups(off_sh, a);
}

PlanArgs plan_args(const FfnGroups& g, int dtype, FfnPlanHeader* hdr, int32_t* gemv_list,
                   int4* mtile_list, int max_mtiles, int gemv_limit, bool allow_pair,
                   int small_rows) {
    PlanArgs a;
    a.E = g.E;
    a.has_shared = g.has_shared;
    a.T = g.T;
    // fp32 layers never use the tensor cores (no TF32): every group streams
    a.limit = dtype == MOE_F32 ? 0x7fffffff : gemv_limit;
    a.small = small_rows;
    a.single_m = tc_tile_rows(false);
    // a pair threshold no group can reach keeps every group on single tiles
    a.pair_min = allow_pair ? tc_pair_min_rows() : 0x7fffffff;
    a.pair_m = tc_tile_rows(true);
    a.max_mtiles = max_mtiles;
    a.sms = device_sm_count();
    a.split_rho = allow_pair ? tc_split_rho() : 0;
    a.hdr = hdr;
    a.gemv_list = gemv_list;
    a.mtile_list = mtile_list;
    return a;
}

struct GroupView {
    int rows;          // rows of this group
    int inter;         // intermediate size
    int64_t row0;      // first row in the routed row space (or 0 for shared)
    bool shared;
    const void *wg, *wu, *wd;
};

template <typename T>
__device__ __forceinline__ GroupView group_view(const FfnGroups& g, int grp) {
    GroupView v;
    if (grp < g.E) {
        const int32_t o0 = g.offsets[grp];
        v.rows = g.offsets[grp + 1] - o0;
        v.row0 = o0;
        v.inter = g.I;
        v.shared = false;
        const int64_t wgu = (int64_t)grp * g.I * g.d;
        v.wg = (const T*)g.w_gate + wgu;
        v.wu = (const T*)g.w_up + wgu;
        v.wd = (const T*)g.w_down + wgu;  // [E][d][I]: same stride d*I
    } else {
        v.rows = g.T;
        v.row0 = 0;
        v.inter = g.Is;
        v.shared = true;
        v.wg = g.ws_gate;
        v.wu = g.ws_up;
        v.wd = g.ws_down;
    }
    return v;
}

// h = SiLU(Wg x) * (Wu x) for a block of kRowsGU intermediate rows.
template <typename T, int MT, int U>
__global__ void __launch_bounds__(kThreads)
gemv_gate_up_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                    const int32_t* __restrict__ gemv_list) {
    pdl_wait();
    pdl_trigger();
    constexpr int V = Elem<T>::kPerVec;
    extern __shared__ uint4 xs[];  // [MT][d / V]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvec = g.d / V;
    const int n_groups = hdr->n_gemv;
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const int nrb = (max_inter + kRowsGU - 1) / kRowsGU;
    const int64_t units = (int64_t)n_groups * nrb;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int a = (int)(u / nrb), rb = (int)(u % nrb);
        const GroupView gv = group_view<T>(g, gemv_list[a]);
        if (rb * kRowsGU >= gv.inter) continue;  // uniform across the block
        for (int c0 = 0; c0 < gv.rows; c0 += MT) {
            const int nt = min(MT, gv.rows - c0);
            __syncthreads();  // previous readers of xs are done
            for (int i = threadIdx.x; i < nt * nvec; i += kThreads) {
                const int m = i / nvec, v = i - m * nvec;
                int64_t src_row;
                const T* base;
                if (gv.shared) { src_row = c0 + m; base = (const T*)g.a_shared; }
                else {
                    const int64_t p = gv.row0 + c0 + m;
                    src_row = g.row_src ? g.row_src[p] : p;
                    base = (const T*)g.a_routed;
                }
                xs[m * nvec + v] = ld_ro(base + src_row * g.d + (int64_t)v * V);
            }
            __syncthreads();
            for (int r = warp; r < kRowsGU; r += kWarps) {
                const int i = rb * kRowsGU + r;
                if (i >= gv.inter) break;
                const T* wg = (const T*)gv.wg + (int64_t)i * g.d;
                const T* wu = (const T*)gv.wu + (int64_t)i * g.d;
                float ag[MT], au[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) { ag[m] = 0.f; au[m] = 0.f; }
                for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
                    uint4 rg[U], ru[U];
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = v0 + 32 * q;
                        if (v < nvec) {
                            rg[q] = ld_stream(wg + (int64_t)v * V);
                            ru[q] = ld_stream(wu + (int64_t)v * V);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = v0 + 32 * q;
                        if (v < nvec) {
                            float fg[V], fu[V];
                            unpack(rg[q], fg, (const T*)nullptr);
                            unpack(ru[q], fu, (const T*)nullptr);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (m < nt) {
                                    float fx[V];
                                    unpack(xs[m * nvec + v], fx, (const T*)nullptr);
#pragma unroll
                                    for (int k = 0; k < V; ++k) {
                                        ag[m] = fmaf(fg[k], fx[k], ag[m]);
                                        au[m] = fmaf(fu[k], fx[k], au[m]);
                                    }
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float sg = warp_sum(ag[m]);
                    const float su = warp_sum(au[m]);
                    if (lane == m && m < nt) {
                        const T hv = Elem<T>::from_f32(silu_mul(sg, su));
                        if (gv.shared) ((T*)g.h_s)[(int64_t)(c0 + m) * gv.inter + i] = hv;
                        else ((T*)g.h)[(gv.row0 + c0 + m) * gv.inter + i] = hv;
                    }
                }
            }
        }
    }
}

// y = Wd h for a block of kRowsDown output rows.
template <typename T, int MT, int U>
__global__ void __launch_bounds__(kThreads)
gemv_down_kernel(FfnGroups g, const FfnPlanHeader* __restrict__ hdr,
                 const int32_t* __restrict__ gemv_list) {
    pdl_wait();
    pdl_trigger();
    constexpr int V = Elem<T>::kPerVec;
    extern __shared__ uint4 hs[];  // [MT][inter / V]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_groups = hdr->n_gemv;
    const int nrb = (g.d + kRowsDown - 1) / kRowsDown;
    const int64_t units = (int64_t)n_groups * nrb;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int a = (int)(u / nrb), rb = (int)(u % nrb);
        const GroupView gv = group_view<T>(g, gemv_list[a]);
        const int nvec = gv.inter / V;
        for (int c0 = 0; c0 < gv.rows; c0 += MT) {
            const int nt = min(MT, gv.rows - c0);
            __syncthreads();
            for (int i = threadIdx.x; i < nt * nvec; i += kThreads) {
                const int m = i / nvec, v = i - m * nvec;
                const T* src = gv.shared ? (const T*)g.h_s + (int64_t)(c0 + m) * gv.inter
                                         : (const T*)g.h + (gv.row0 + c0 + m) * gv.inter;
                hs[m * nvec + v] = ld_ro(src + (int64_t)v * V);
            }
            __syncthreads();
            for (int r = warp; r < kRowsDown; r += kWarps) {
                const int j = rb * kRowsDown + r;
                if (j >= g.d) break;
                const T* wd = (const T*)gv.wd + (int64_t)j * gv.inter;
                float acc[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = 0.f;
                for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
                    uint4 rw[U];
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = v0 + 32 * q;
                        if (v < nvec) rw[q] = ld_stream(wd + (int64_t)v * V);
                    }
#pragma unroll
                    for (int q = 0; q < U; ++q) {
                        const int v = v0 + 32 * q;
                        if (v < nvec) {
                            float fw[V];
                            unpack(rw[q], fw, (const T*)nullptr);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (m < nt) {
                                    float fh[V];
                                    unpack(hs[m * nvec + v], fh, (const T*)nullptr);
#pragma unroll
                                    for (int k = 0; k < V; ++k) acc[m] = fmaf(fw[k], fh[k], acc[m]);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float s = warp_sum(acc[m]);
                    if (lane == m && m < nt) {
                        const T yv = Elem<T>::from_f32(s);
                        if (gv.shared) ((T*)g.y_s)[(int64_t)(c0 + m) * g.d + j] = yv;
                        else ((T*)g.y)[(gv.row0 + c0 + m) * g.d + j] = yv;
                    }
                }
            }
        }
    }
}

template <typename T, int MT, int U>
cudaError_t launch_gemv_t(const FfnGroups& g, const FfnPlanHeader* hdr, const int32_t* list,
                          cudaStream_t st) {
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    const size_t smem_gu = (size_t)MT * g.d * sizeof(T);
    const size_t smem_dn = (size_t)MT * max_inter * sizeof(T);
    cudaError_t e;
    e = cudaFuncSetAttribute(gemv_gate_up_kernel<T, MT, U>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv_down_kernel<T, MT, U>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dn);
    if (e != cudaSuccess) return e;
    int occ_gu = 1, occ_dn = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_gu, gemv_gate_up_kernel<T, MT, U>, kThreads,
                                                  smem_gu);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_dn, gemv_down_kernel<T, MT, U>, kThreads,
                                                  smem_dn);
    const int sms = device_sm_count();
    e = launch_pdl(gemv_gate_up_kernel<T, MT, U>, dim3(sms * (occ_gu > 0 ? occ_gu : 1)),
                   dim3(kThreads), smem_gu, st, g, hdr, list);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv_down_kernel<T, MT, U>, dim3(sms * (occ_dn > 0 ? occ_dn : 1)),
                      dim3(kThreads), smem_dn, st, g, hdr, list);
}

}  // namespace

// bf16 groups with more rows than this take the tcgen05 GEMM.  Measured on
// GB300: the tensor-core path streams expert weights at 88-100% of HBM
// bandwidth even for one-row groups (its MMAs are idle most of the time), so
// the default sends every bf16 group there; the GEMV kernels serve fp32.
// Read on every call so a process can compare both paths on the same inputs.
int gemv_max_rows() {
    const char* s = getenv("MOE_GEMV_MAX_ROWS");
    const int x = s ? atoi(s) : 0;
    return x < 0 ? 0 : x;
}

cudaError_t launch_ffn_plan(const FfnGroups& g, int dtype, FfnPlanHeader* hdr, int32_t* gemv_list,
                            int4* mtile_list, int max_mtiles, int gemv_limit, bool allow_pair,
                            int small_rows, cudaStream_t st) {
    return launch_pdl(ffn_plan_kernel, dim3(1), dim3(1024), 0, st, g.offsets,
                      plan_args(g, dtype, hdr, gemv_list, mtile_list, max_mtiles, gemv_limit,
                                allow_pair, small_rows));
}

// Read on every call: MOE_FUSED_DISPATCH=0 keeps the four-launch path.
bool dispatch_plan_fusable(const moe_shape& s) {
    const char* v = getenv("MOE_FUSED_DISPATCH");
    if (v && v[0] == '0') return false;
    return (int64_t)s.T * s.K <= 1024 && s.E <= 1024;
}

cudaError_t launch_dispatch_plan_small(const moe_shape& s, const int32_t* topk_idx, int32_t* counts,
                                       int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                       int32_t* tok_of, DevError* err, const FfnGroups& g,
                                       FfnPlanHeader* hdr, int32_t* gemv_list, int4* mtile_list,
                                       int max_mtiles, int gemv_limit, bool allow_pair,
                                       int small_rows, cudaStream_t st) {
    const size_t smem = sizeof(int32_t) * (32 * (size_t)s.E + s.E + 1);
    cudaError_t e = cudaFuncSetAttribute(dispatch_plan_small_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(dispatch_plan_small_kernel, dim3(1), dim3(1024), smem, st, topk_idx,
                      s.T * s.K, s.K, counts, offsets, perm, inv_perm, tok_of, err,
                      plan_args(g, s.dtype, hdr, gemv_list, mtile_list, max_mtiles, gemv_limit,
                                allow_pair, small_rows));
}

cudaError_t launch_ffn_gemv(const FfnGroups& g, int dtype, const FfnPlanHeader* hdr,
                            const int32_t* gemv_list, cudaStream_t st) {
    if (dtype == MOE_BF16) return launch_gemv_t<bf16, 4, 4>(g, hdr, gemv_list, st);
    return launch_gemv_t<float, 2, 4>(g, hdr, gemv_list, st);
}

}  // namespace moe
