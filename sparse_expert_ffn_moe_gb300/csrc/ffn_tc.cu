// ffn_tc.cu -- stage 3 for groups with many rows (and the router GEMM of
// large batches): a persistent grouped GEMM on the 5th-generation tensor
// cores.  TMA streams 128-row activation tiles and 256-row weight tiles into a
// 4-stage shared-memory ring; one thread issues tcgen05.mma into a TMEM
// accumulator (two 128x256 fp32 accumulators, double-buffered so the epilogue
// of one tile overlaps the main loop of the next); four epilogue warps read
// TMEM with tcgen05.ld and write the result.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 4.2: one
// launch computes many GEMMs whose M differs per expert while K and N are
// shared, thread blocks take tiles from the per-expert offsets, and experts
// with no tokens are skipped (FAQ Q1).  "Computation and Data Movement for
// Inference", section 15: one weight load serves every token of the bucket.
//
// Tiles are (group, 128-row m-tile, n-block).  Within a group the m-tiles of
// a band of 8 vary fastest, so the CTAs working at the same moment share the
// same weight tiles through L2 and every weight tile is read from HBM about
// once per band.  Rows of an m-tile past its group's end belong to the next
// group (or lie past the tensor and read as zero): they are computed and
// never stored.
//
// Epilogues:
//   SWIGLU     B = [W_gate rows n..n+127 ; W_up rows n..n+127], so columns
//              0..127 of the accumulator hold gate and 128..255 up for the
//              same 128 intermediate indices: h = SiLU(g) * u -> bf16.
//   STORE_BF16 plain product -> bf16 (down projection).
//   STORE_F32  plain product -> fp32 (router scores).
//
// Every wait on an mbarrier is bounded (MOE_TC_TIMEOUT_MS, default 1000 ms
// of wall time); when one runs out the CTA records MOE_ERR_TIMEOUT in the
// workspace error word, all roles leave their loops, outstanding copies and
// MMAs are drained with bounded waits, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kBand = 8;
constexpr uint32_t kABytes = BM * BK * 2;     // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;     // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kThreadsTc = 192;               // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kTmemCols = 512;

enum Epi { EPI_SWIGLU = 0, EPI_STORE_BF16 = 1, EPI_STORE_F32 = 2 };

// Activation maps come in four box heights; a tile loads the smallest box that
// covers its valid rows, so a one-token expert does not pull 128 rows of
// other experts' activations through L2 for every k-block.  The MMA still
// reads all 128 rows of the stage: rows past the box hold stale data that
// only reach accumulator rows which are never stored.
constexpr int kABoxes = 4;  // 16, 32, 64, 128 rows
__host__ __device__ constexpr int abox_rows(int i) { return 16 << i; }

struct TcParams {
    CUtensorMap a[2][kABoxes];  // activations: [0] routed rows, [1] shared / dense rows
    CUtensorMap b0[2];  // weights (gate / down / router)
    CUtensorMap b1[2];  // up weights (SWIGLU only)
    const FfnPlanHeader* hdr;
    const int4* mtiles;
    const int32_t* offsets;
    int E;
    int max_mtiles;
    int dense_rows;     // > 0: one dense group of this many rows on the [1] maps
    int NB;             // n-blocks per m-tile
    int n_out[2];       // valid output columns (routed, shared)
    int kdim[2];        // reduction length (routed, shared)
    int wrows[2];       // rows per group in the stacked weight matrix
    void* out[2];       // output base (routed, shared)
    int64_t ld_out[2];  // output row stride (elements)
    DevError* err;
    unsigned long long timeout_ns;
};

struct Tile {
    int kind;       // 0 routed, 1 shared/dense
    int row0;       // first activation row (in the map of `kind`)
    int rows;       // valid rows (<= BM)
    int wrow0;      // first weight row of this n-block in the stacked matrix
    int n0;         // first output column
    int kblocks;
    bool valid;
};

template <int EPI>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, int t) {
    constexpr int kNCols = EPI == EPI_SWIGLU ? BN / 2 : BN;  // output columns per n-block
    Tile tl;
    const int NB = p.NB;
    int g, gr0, Mg, i;
    if (p.dense_rows > 0) {
        g = -1; gr0 = 0; Mg = p.dense_rows; i = t / NB;
    } else {
        const int4 e = p.mtiles[t / NB];
        g = e.x; gr0 = e.y; Mg = e.z; i = e.w;
    }
    const int q = t / NB;
    const int cnt = (Mg + BM - 1) / BM;
    const int tt = t - (q - i) * NB;               // index inside this group's tiles
    const int band = tt / (kBand * NB);
    const int bstart = band * kBand;
    const int bcnt = min(kBand, cnt - bstart);
    const int r = tt - band * kBand * NB;
    const int nb = r / bcnt;
    const int mi = bstart + r % bcnt;
    tl.kind = (p.dense_rows > 0 || g >= p.E) ? 1 : 0;
    tl.row0 = gr0 + mi * BM;
    tl.rows = min(BM, Mg - mi * BM);
    tl.n0 = nb * kNCols;
    tl.wrow0 = (tl.kind == 0 ? g * p.wrows[0] : 0) + tl.n0;
    tl.kblocks = (p.kdim[tl.kind] + BK - 1) / BK;
    tl.valid = tl.n0 < p.n_out[tl.kind] && tl.rows > 0;
    return tl;
}

struct SmemCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};

// Bounded wait: false (and the CTA-wide abort flag set) when the budget runs out
// or another role already gave up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, SmemCtl* ctl,
                                             const TcParams& p, int where) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (ctl->abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
                record_error(p.err, MOE_ERR_TIMEOUT, where);
                ctl->abort_flag = 1;
                return false;
            }
        }
    }
}

template <int EPI>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzle atoms
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kABytes;
    SmemCtl* ctl = (SmemCtl*)(smem + kStages * kStageBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.dense_rows > 0 ? (p.dense_rows + BM - 1) / BM
                                          : min(p.hdr->n_mtiles, p.max_mtiles)) * p.NB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&ctl->full[s], 1);
            ptx::mbar_init(&ctl->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&ctl->tfull[a], 1);
            ptx::mbar_init(&ctl->tempty[a], 4);
        }
        ptx::mbar_init(&ctl->drain, 1);
        ctl->abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        for (int k = 0; k < 2; ++k) {
            for (int b = 0; b < kABoxes; ++b) ptx::prefetch_tmap(&p.a[k][b]);
            ptx::prefetch_tmap(&p.b0[k]);
            if (EPI == EPI_SWIGLU) ptx::prefetch_tmap(&p.b1[k]);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<EPI>(p, t);
                if (!tl.valid) continue;
                const int ab = tl.rows <= 16 ? 0 : tl.rows <= 32 ? 1 : tl.rows <= 64 ? 2 : 3;
                const uint32_t a_bytes = (uint32_t)abox_rows(ab) * BK * 2;
                const CUtensorMap* ma = &p.a[tl.kind][ab];
                const CUtensorMap* mb0 = &p.b0[tl.kind];
                const CUtensorMap* mb1 = &p.b1[tl.kind];
                for (int kb = 0; kb < tl.kblocks; ++kb) {
                    if (!wait_bounded(&ctl->empty[stage], phase ^ 1u, ctl, p, 100)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&ctl->full[stage], kBBytes + a_bytes);
                    const int k0 = kb * BK;
                    ptx::tma_load_2d(sA + stage * kABytes, ma, &ctl->full[stage], k0, tl.row0);
                    if (EPI == EPI_SWIGLU) {
                        ptx::tma_load_2d(sB + stage * kBBytes, mb0, &ctl->full[stage], k0, tl.wrow0);
                        ptx::tma_load_2d(sB + stage * kBBytes + kBBytes / 2, mb1, &ctl->full[stage], k0,
                                         tl.wrow0);
                    } else {
                        ptx::tma_load_2d(sB + stage * kBBytes, mb0, &ctl->full[stage], k0, tl.wrow0);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // drain: every copy issued lands before the CTA exits
                for (int s = 0; s < kStages; ++s) {
                    if (!issued[s]) continue;
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (!ptx::mbar_try_wait(&ctl->full[s], issued_phase[s]) &&
                           ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<EPI>(p, t);
                if (!tl.valid) continue;
                if (!wait_bounded(&ctl->tempty[acc], acc_phase ^ 1u, ctl, p, 200)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                for (int kb = 0; kb < tl.kblocks; ++kb) {
                    if (!wait_bounded(&ctl->full[stage], phase, ctl, p, 201)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a_base = ptx::smem_u32(sA + stage * kABytes);
                    const uint32_t b_base = ptx::smem_u32(sB + stage * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = ptx::sw128_kmajor_desc(a_base + kk * 32);
                        const uint64_t bd = ptx::sw128_kmajor_desc(b_base + kk * 32);
                        ptx::tc_mma_f16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    any = true;
                    ptx::tc_commit(&ctl->empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::tc_commit(&ctl->tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok && any) {
                // drain: every MMA issued completes before TMEM is freed
                ptx::tc_commit(&ctl->drain);
                const uint64_t t0 = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(&ctl->drain, 0) &&
                       ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quad = warp & 3;               // TMEM lanes 32*quad .. 32*quad+31
        const int r = quad * 32 + lane;          // tile row owned by this thread
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const Tile tl = decode_tile<EPI>(p, t);
            if (!tl.valid) continue;
            // one lane waits, the warp follows its verdict (tcgen05.ld needs the whole warp)
            const int ok = lane == 0 ? (int)wait_bounded(&ctl->tfull[acc], acc_phase, ctl, p, 300) : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
            const bool row_ok = r < tl.rows;
            const int64_t orow = (int64_t)tl.row0 + r;
            const int nvalid = p.n_out[tl.kind];
            if (EPI == EPI_SWIGLU) {
                bf16* out = (bf16*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0;
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 16) {
                    uint32_t g[16], u[16];
                    ptx::tmem_ld16(tbase + c, g);
                    ptx::tmem_ld16(tbase + BN / 2 + c, u);
                    ptx::tmem_ld_wait();
                    if (row_ok && tl.n0 + c < nvalid) {
                        uint32_t w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float h0 = silu_mul(__uint_as_float(g[2 * k]), __uint_as_float(u[2 * k]));
                            const float h1 = silu_mul(__uint_as_float(g[2 * k + 1]), __uint_as_float(u[2 * k + 1]));
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                            w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else if (EPI == EPI_STORE_BF16) {
                bf16* out = (bf16*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(tbase + c, v);
                    ptx::tmem_ld_wait();
                    if (row_ok && tl.n0 + c < nvalid) {
                        uint32_t w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                            w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else {
                float* out = (float*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(tbase + c, v);
                    ptx::tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (tl.n0 + c + k < nvalid) out[c + k] = __uint_as_float(v[k]);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ctl->tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
    });
    return fn;
}

// 2-D bf16 map over a row-major [rows][cols] matrix, box = 64 columns x box_rows
// rows, 128-byte swizzle.  A matrix with no rows gets a 1-row placeholder that
// is never read.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (rows <= 0) rows = 1;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// the four activation maps of one matrix (box heights 16, 32, 64, 128 rows)
bool make_amaps(CUtensorMap (&m)[kABoxes], const void* base, int64_t rows, int64_t cols) {
    bool ok = true;
    for (int b = 0; b < kABoxes; ++b) ok &= make_map(&m[b], base, rows, cols, abox_rows(b));
    return ok;
}

unsigned long long timeout_ns() {
    static const unsigned long long v = [] {
        const char* s = getenv("MOE_TC_TIMEOUT_MS");
        const long long ms = s ? atoll(s) : 1000;
        return (unsigned long long)(ms > 0 ? ms : 1000) * 1000000ull;
    }();
    return v;
}

constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + sizeof(SmemCtl) + 64;

template <int EPI>
cudaError_t launch_tc(const TcParams& p, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    int grid = device_sm_count();
    if (p.dense_rows > 0) {
        const int tiles = (p.dense_rows + BM - 1) / BM * p.NB;
        if (tiles < grid) grid = tiles;
    }
    if (grid < 1) grid = 1;
    tc_gemm_kernel<EPI><<<grid, kThreadsTc, kSmemBytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool tc_available() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3 && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const FfnGroups& g, const FfnPlanHeader* hdr, const int4* mtile_list,
                          int max_mtiles, DevError* err, cudaStream_t st) {
    const int64_t R = g.n_routed_rows;
    // ---- gate/up: h = SiLU(x W_gate^T) * (x W_up^T)
    TcParams p{};
    bool ok = true;
    ok &= make_amaps(p.a[0], g.a_routed, R, g.d);
    ok &= make_map(&p.b0[0], g.w_gate, (int64_t)g.E * g.I, g.d, BN / 2);
    ok &= make_map(&p.b1[0], g.w_up, (int64_t)g.E * g.I, g.d, BN / 2);
    if (g.has_shared) {
        ok &= make_amaps(p.a[1], g.a_shared, g.T, g.d);
        ok &= make_map(&p.b0[1], g.ws_gate, g.Is, g.d, BN / 2);
        ok &= make_map(&p.b1[1], g.ws_up, g.Is, g.d, BN / 2);
    } else {
        for (int b = 0; b < kABoxes; ++b) p.a[1][b] = p.a[0][b];
        p.b0[1] = p.b0[0]; p.b1[1] = p.b1[0];
    }
    if (!ok) return cudaErrorInvalidValue;
    p.hdr = hdr;
    p.mtiles = mtile_list;
    p.offsets = g.offsets;
    p.E = g.E;
    p.max_mtiles = max_mtiles;
    p.dense_rows = 0;
    const int max_inter = g.has_shared && g.Is > g.I ? g.Is : g.I;
    p.NB = (max_inter + BN / 2 - 1) / (BN / 2);
    p.n_out[0] = g.I; p.n_out[1] = g.has_shared ? g.Is : 0;
    p.kdim[0] = g.d; p.kdim[1] = g.d;
    p.wrows[0] = g.I; p.wrows[1] = 0;
    p.out[0] = g.h; p.out[1] = g.h_s;
    p.ld_out[0] = g.I; p.ld_out[1] = g.Is;
    p.err = err;
    p.timeout_ns = timeout_ns();
    cudaError_t e = launch_tc<EPI_SWIGLU>(p, st);
    if (e != cudaSuccess) return e;

    // ---- down: y = h W_down^T
    TcParams q{};
    ok = true;
    ok &= make_amaps(q.a[0], g.h, R, g.I);
    ok &= make_map(&q.b0[0], g.w_down, (int64_t)g.E * g.d, g.I, BN);
    if (g.has_shared) {
        ok &= make_amaps(q.a[1], g.h_s, g.T, g.Is);
        ok &= make_map(&q.b0[1], g.ws_down, g.d, g.Is, BN);
    } else {
        for (int b = 0; b < kABoxes; ++b) q.a[1][b] = q.a[0][b];
        q.b0[1] = q.b0[0];
    }
    q.b1[0] = q.b0[0]; q.b1[1] = q.b0[1];
    if (!ok) return cudaErrorInvalidValue;
    q.hdr = hdr;
    q.mtiles = mtile_list;
    q.offsets = g.offsets;
    q.E = g.E;
    q.max_mtiles = max_mtiles;
    q.dense_rows = 0;
    q.NB = (g.d + BN - 1) / BN;
    q.n_out[0] = g.d; q.n_out[1] = g.has_shared ? g.d : 0;
    q.kdim[0] = g.I; q.kdim[1] = g.has_shared ? g.Is : g.I;
    q.wrows[0] = g.d; q.wrows[1] = 0;
    q.out[0] = g.y; q.out[1] = g.y_s;
    q.ld_out[0] = g.d; q.ld_out[1] = g.d;
    q.err = err;
    q.timeout_ns = timeout_ns();
    return launch_tc<EPI_STORE_BF16>(q, st);
}

// scores[T][E] (fp32) = x w_g^T on the tensor cores
cudaError_t launch_router_tc(const moe_shape& s, const void* x, const void* w_g, float* scores,
                             DevError* err, cudaStream_t st) {
    TcParams p{};
    bool ok = true;
    ok &= make_amaps(p.a[1], x, s.T, s.d);
    ok &= make_map(&p.b0[1], w_g, s.E, s.d, BN);
    if (!ok) return cudaErrorInvalidValue;
    for (int b = 0; b < kABoxes; ++b) p.a[0][b] = p.a[1][b];
    p.b0[0] = p.b0[1]; p.b1[0] = p.b0[1]; p.b1[1] = p.b0[1];
    p.hdr = nullptr;
    p.mtiles = nullptr;
    p.dense_rows = s.T;
    p.NB = (s.E + BN - 1) / BN;
    p.n_out[0] = p.n_out[1] = s.E;
    p.kdim[0] = p.kdim[1] = s.d;
    p.wrows[0] = p.wrows[1] = 0;
    p.out[0] = p.out[1] = scores;
    p.ld_out[0] = p.ld_out[1] = s.E;
    p.err = err;
    p.timeout_ns = timeout_ns();
    return launch_tc<EPI_STORE_F32>(p, st);
}

}  // namespace moe
