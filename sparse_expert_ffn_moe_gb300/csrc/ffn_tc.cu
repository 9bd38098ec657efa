// ffn_tc.cu -- stage 3 for bf16 expert groups (and the router GEMM of large
// batches): a persistent grouped GEMM on the 5th-generation tensor cores.
//
// "Sparse MoE inference kernels ..." (blog.llmgo.top), section 4.2: one
// launch computes many GEMMs whose M differs per expert while K and N are
// shared, thread blocks take tiles from the per-expert offsets, and experts
// with no tokens are skipped (FAQ Q1).  "Computation and Data Movement for
// Inference", section 15: one weight load serves every token of the bucket.
//
// Two tile shapes, one kernel template (every tcgen05 instruction of one
// kernel uses the same CTA-group size):
//   single (PAIR = false)  128 rows x 256 columns per CTA; a 4-stage ring of
//                          48 KB stages (128 activation rows + 256 weight
//                          rows of a 64-deep K step); tcgen05.mma.cta_group::1.
//   pair   (PAIR = true)   256 rows x 256 columns per cluster of 2 CTAs; each
//                          CTA holds 128 activation rows and 128 of the 256
//                          weight rows of a K step in a 7-stage ring of 32 KB
//                          stages; the even CTA issues tcgen05.mma.cta_group::2,
//                          which reads both CTAs' operands and leaves each
//                          CTA's 128 accumulator rows in its own tensor memory.
// A pair tile needs 32 KB per SM per K step instead of 48 KB, so the ring
// hides ~1.5x more memory latency and large groups run faster; but it pads
// ragged groups to 256 rows.  The plan kernel picks the shape per group by
// its padded rows over each shape's measured tensor-pipe activity (or, with
// MOE_PAIR_MIN_ROWS > 0, by a fixed row threshold) and writes one tile list
// per shape; each GEMM is one launch per list, and when a call has both, the
// pair-tile launch runs on the caller's stream and the single-tile launch on
// a second stream beside it, each on the share of the SMs the plan gives it.
//
// Both shapes keep two 128x256 fp32 accumulators per CTA in tensor memory
// (all 512 columns), double-buffered so the epilogue of one tile overlaps the
// main loop of the next (with block-scaled 8-bit weights, A8 = 3, they
// alternate per 128-deep K block instead).  Roles (192 threads per CTA): warp 0
// TMA producer; warp 1 MMA issuer and tensor-memory owner; warps 2-5 epilogue
// (the 8-bit-weight variant W8 adds converter warps 6-13; A8 = 3 runs eight
// epilogue warps, 2-9).
//
// Tiles are (group, m-tile, n-block).  Within a group the m-tiles of a band
// (1024 rows) vary fastest, so the CTAs working at the same moment share the
// same weight tiles through L2.  Rows of an m-tile past its group's end belong
// to the next group (or lie past the tensor and read as zero): they are
// computed and never stored.  The activation box is 16/32/64/128 rows, the
// smallest covering a CTA's valid rows (no load when a CTA has none).
//
// Epilogues:
//   SWIGLU     the 256 weight rows of an n-block are W_gate rows n..n+127
//              followed by W_up rows n..n+127 (in a pair: even CTA gate, odd
//              CTA up), so accumulator columns 0..127 are gate and 128..255
//              up for the same intermediate indices: h = SiLU(g) * u -> bf16.
//   STORE_BF16 plain product -> bf16 (down projection).
//   STORE_F32  plain product -> fp32 (router scores).
//   COMBINE    the shared expert's down projection fused with the combine:
//              a dense launch over the T tokens whose epilogue adds, to each
//              fp32 product y_s[t][c], w[t][j] * y_perm[inv_perm[t*K+j]][c]
//              for j = 0..K-1 (shared term first, then j ascending, one fp32
//              fma each -- the combine kernel's order), rounds once and
//              stores the layer output y.  The routed down launches skip the
//              shared group and have finished (stream order) before it starts.
//
// Every wait on an mbarrier is bounded (MOE_TC_TIMEOUT_MS, default 1000 ms
// of wall time); when one runs out the CTA records MOE_ERR_TIMEOUT in the
// workspace error word, its roles leave their loops, outstanding copies and
// MMAs are drained with bounded waits, tensor memory is freed (a pair always
// reaches the collective free) and the kernel returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BMC = 128;  // accumulator rows per CTA
constexpr int BN = 256;   // MMA N
constexpr int BK = 64;
constexpr int kMaxStages = 7;
constexpr uint32_t kABytes = BMC * BK * 2;  // 16 KB
// warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue.  Eight
// epilogue warps (two per tensor-memory lane quarter, half the columns each)
// measured 3 % faster on 8-bit DeepSeek-V3 prefill but 1 % slower on the bf16
// Mixtral and Zipf prefill layers, so each quarter keeps one warp.
constexpr int kThreadsTc = 192;
constexpr uint32_t kTmemCols = 512;

// Block-scaled 8-bit weights (A8 == 3: two activation planes as A8 == 2; A8 ==
// 4: one plane of per-row-quantised activations as A8 == 1; either with one
// weight scale per 128 x 128 block).  A block scale changes every 128 values
// of K, so it cannot be applied to an accumulator that sums all of K: each
// 128-deep K block (one ring stage) is multiplied into a fresh accumulator,
// and the epilogue warps add it, times the block's scale, to fp32 sums held in
// registers -- the two accumulators alternate per K block instead of per tile.
// Eight epilogue warps (two per tensor-memory lane quarter, half of the tile's
// 256 columns each) hold 128 sums per thread.  An accumulator is released once
// per CTA: the eight warps meet at a named barrier after their last read of it
// and one thread arrives.  The hand-off costs little on single-SM tiles (the
// MMA issuer waits ~90 cycles per K block, measured on GB300); across a CTA
// pair it waited ~1600 cycles for the peer's release, so block-scaled groups
// take single-SM tiles unless MOE_W8_PAIR=1.
constexpr int kThreadsBlk = 320;
constexpr uint32_t kBlkEpiBar = 1;  // named barrier of the eight epilogue warps
template <bool W8, int A8> constexpr int threads_of() {
    return W8 ? (6 + 8) * 32 : (A8 >= 3 ? kThreadsBlk : kThreadsTc);
}

// Small-row ring (SMA, single-SM bf16 or W8A8 tiles whose groups all have at most kSmaRows
// rows, e.g. every group of a decode batch of <= 32 tokens): an activation
// stage holds 32 rows (4 KB) instead of 128, so the ring carries 6 weight
// stages instead of 4 -- 50 % more weight bytes in flight per SM for the
// weight-streaming GEMMs of small batches.  The MMA still reads 128 activation
// rows; rows past the 32 loaded ones are whatever lies beyond the stage (never
// stored, like the unloaded rows of a short box in the full-size ring).
constexpr int kSmaRows = 32;

template <bool PAIR, bool SMA = false> struct Shape {
    static constexpr int kTileRows = PAIR ? 256 : 128;  // rows per tile
    static constexpr int kBRows = PAIR ? 128 : 256;     // weight rows per CTA per K step
    static constexpr int kStages = SMA ? 6 : (PAIR ? 7 : 4);
    static constexpr int kBand = PAIR ? 4 : 8;          // m-tiles per band (1024 rows)
    static constexpr uint32_t kAStride = SMA ? kSmaRows * BK * 2 : kABytes;  // bytes per A stage
    static constexpr uint32_t kBBytes = kBRows * BK * 2;
    static constexpr uint32_t kStageBytes = kAStride + kBBytes;
    // 4 x 48 KB (single), 7 x 32 KB (pair) or 6 x 36 KB (single, small rows)
    static constexpr uint32_t kRingBytes = kStages * kStageBytes;
    static_assert(kStages <= kMaxStages, "stage barriers");
    static_assert(kAStride % 1024 == 0, "128-byte-swizzle atoms need 1 KB aligned stages");
};

// 8-bit activations carried as two E4M3 planes (A8 == 2): each 128-code K
// block of an activation row is [128 hi codes | 128 lo codes] (the row's value
// is scale * (hi + lo)), so a stage holds two activation tiles, one per plane,
// and every K slice issues two kind::f8f6f4 MMAs into the same accumulator --
// the tensor time of one bf16 MMA, on 1-byte weights with no widening.  The
// ring: 4 stages of 48 KB (pair) or 3 of 64 KB (single); with the small-row
// ring (SMA: every group of at most kSmaRows rows) each plane holds 32 rows,
// 5 stages of 40 KB.
template <bool PAIR, bool SMA = false> struct A2Shape {
    static constexpr int kTileRows = Shape<PAIR>::kTileRows;
    static constexpr int kBRows = Shape<PAIR>::kBRows;
    static constexpr int kStages = SMA ? 5 : (PAIR ? 4 : 3);
    static constexpr int kBand = Shape<PAIR>::kBand;
    static constexpr uint32_t kAPlaneBytes = SMA ? kSmaRows * BK * 2 : kABytes;
    static constexpr uint32_t kAStride = 2 * kAPlaneBytes;  // hi and lo planes
    static constexpr uint32_t kBBytes = Shape<PAIR>::kBBytes;
    static constexpr uint32_t kStageBytes = kAStride + kBBytes;
    static constexpr uint32_t kRingBytes = kStages * kStageBytes;
    static_assert(kStages <= kMaxStages, "stage barriers");
    static_assert(kAPlaneBytes % 1024 == 0, "128-byte-swizzle atoms need 1 KB aligned planes");
};
template <bool PAIR, bool SMA, int A8> struct RingOf { using type = Shape<PAIR, SMA>; };
template <bool PAIR, bool SMA> struct RingOf<PAIR, SMA, 2> { using type = A2Shape<PAIR, SMA>; };
template <bool PAIR, bool SMA> struct RingOf<PAIR, SMA, 3> { using type = A2Shape<PAIR, SMA>; };

enum Epi { EPI_SWIGLU = 0, EPI_STORE_BF16 = 1, EPI_STORE_F32 = 2, EPI_COMBINE = 3 };

// 8-bit weights (W8).  TMA streams a CTA's E4M3 weight rows (256 for a
// single-SM tile, 128 per CTA of a pair) x 128 codes (two 64-deep K steps)
// into a raw ring; eight converter warps widen each K step to bf16 (exact:
// every E4M3 value is a bf16 value) into a ring of bf16 weight stages; the
// producer requests the activation tiles into their own ring.  The per-row
// weight scale factors out of the K sum and is applied in the epilogue.  In a
// pair each CTA widens only its own 128 weight rows.  Measured on GB300
// (Mixtral-shaped prefill): moving the activation loads from the converters
// to the producer and doubling the converter warps took the single-SM
// variant from 4.85 to 3.65 ms; the pair variant stays slower (5.3 ms), its
// stage handoffs crossing the cluster, so 8-bit groups use single-SM tiles
// unless MOE_W8_PAIR=1.
// Three rings: activation tiles (TMA, requested by the producer several K
// steps ahead), raw code tiles (TMA), and widened bf16 weight tiles (written
// by the converter warps); the MMA waits for one stage of each A and B ring.
constexpr int kW8ConvWarps = 8;  // converter warps per CTA (warps 6..13)
template <bool PAIR> struct W8Shape {
    static constexpr int kA = PAIR ? 4 : 3;                          // activation stages
    static constexpr int kConv = PAIR ? 5 : 3;                       // bf16 weight stages
    static constexpr int kRaw = PAIR ? 4 : 2;                        // raw code tiles
    static constexpr uint32_t kRawBytes = Shape<PAIR>::kBRows * 128;  // 16 / 32 KB
    static constexpr uint32_t kRingBytes =
        kA * kABytes + kConv * Shape<PAIR>::kBBytes + kRaw * kRawBytes;  // 208 KB
    // converter warps that fill a stage (of both CTAs in a pair)
    static constexpr int kConvArrivals = PAIR ? 2 * kW8ConvWarps : kW8ConvWarps;
};
static_assert(W8Shape<false>::kRingBytes == W8Shape<true>::kRingBytes, "one W8 ring size");
constexpr int kW8MaxA = 4;
constexpr int kW8MaxRaw = 4;
constexpr uint32_t kW8RingBytes = W8Shape<false>::kRingBytes;
constexpr int kThreadsW8 = (6 + kW8ConvWarps) * 32;  // + the converter warps
static_assert(threads_of<true, 0>() == kThreadsW8, "W8 threads");

// Activation maps come in four box heights; a CTA loads the smallest box that
// covers its valid rows.  The MMA still reads all 128 rows of the stage: rows
// past the box hold stale data that only reach accumulator rows which are
// never stored.
constexpr int kABoxes = 4;  // 16, 32, 64, 128 rows
__host__ __device__ constexpr int abox_rows(int i) { return 16 << i; }
__device__ __forceinline__ int abox_for(int rows) {
    return rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : 3;
}
__device__ __forceinline__ uint32_t abytes_for(int rows) {
    return rows <= 0 ? 0u : (uint32_t)abox_rows(abox_for(rows)) * BK * 2;
}

// Swapped single tiles.  A single-SM tile of few rows (at most
// MOE_SWAP_MAX_ROWS, default 64: the tail experts of a skewed routing, every
// group of a decode batch) would spend an M = 128 MMA on each K step although
// most of its rows are padding.  Such a tile runs with the operands swapped:
// the stage's 256 weight rows are the A operand, as two M = 128 halves (gate
// and up rows, or the n-block's first and second 128 output columns), and the
// activation box (16, 32 or 64 rows) is the B operand, N = the box height, so
// each K step costs 2 x 128 x N instead of 128 x 256 multiply-adds -- a
// quarter or less of the tensor work and energy for groups of <= 32 rows.
// The products land transposed in tensor memory (lane = weight row, column =
// activation row): the first half at columns 0..N-1, the second at
// 128..128+N-1 of the tile's accumulator.  The ring and the copies are
// unchanged; only the MMA issue and the epilogue differ (bf16 operands, no
// 8-bit rings or scales).
constexpr int kSwapMaxRows = 64;

// Routed rows of at most MOE_GATHER_MAX_ROWS per CTA can be gathered from x
// with tile::gather4 inside the GEMM instead of being copied into expert order
// first; larger row blocks load the contiguous permuted copy.  Measured on
// GB300 (interleaved A/B): on prefill shapes gathering is 4-7% slower, even at
// <= 32 rows per CTA (128 rows per CTA took ~2.5x the MMA time per stage), and
// 1% slower at T=64; for batches of a few tokens, where it also spares the
// separate copy launch, it is faster (T=1 161.0 -> 157.6 us, DeepSeek-V3
// decode 801.3 -> 795.3 us).  Default: every routed row of a batch of at most
// kGatherSmallT tokens is gathered in the GEMM (no permuted copy is made);
// larger batches use the copy.
constexpr int kGatherMaxRows = 0;
constexpr int kGatherSmallT = 16;
// Weight-streaming cost of a single-tile group, in hundredths of an MMA step
// per weight K step (the plan's SM split between the two tile shapes).
constexpr int kSplitRho = 150;

struct TcParams {
    CUtensorMap a[2][kABoxes];  // activations: [0] routed rows, [1] shared / dense rows
    CUtensorMap b0[2];          // weights (gate / down / router), box 128 rows
    CUtensorMap b1[2];          // up weights (SWIGLU only), box 128 rows
    CUtensorMap bw[2];          // weights, box 256 rows (single tiles, non-SWIGLU)
    CUtensorMap ag;             // x with a one-row box, for tile::gather4 of routed rows
    CUtensorMap q0[2];          // W8: E4M3 gate / down codes, box 128 rows x 128 codes
    CUtensorMap q1[2];          // W8: E4M3 up codes (SWIGLU only)
    CUtensorMap qw[2];          // W8: E4M3 codes, box 256 rows x 128 codes (non-SWIGLU)
    const float* sc0[2];        // W8, A8: scale of each gate / down weight row (A8 == 3:
                                // of each 128 x 128 block, [rows / 128][K / 128])
    const float* sc1[2];        // W8, A8: scale of each up weight row (A8 == 3: block)
    const float* sa[2];         // A8: scale of each activation row (routed, shared)
    unsigned int* hmax[2];      // A8 gate/up: per-row max |h| as fp32 bits, raised atomically
    CUtensorMap g64[2];         // half pair tiles, gate/up: gate rows, box 64 rows
    CUtensorMap u64[2];         // half pair tiles, gate/up: up rows, box 64 rows
    int half_tiles;             // pair tiles of <= 128 rows run as M = 128 (64 rows per CTA)
    int swap_max_rows;          // single tiles of at most this many rows (<= 64) run swapped
    int band;                   // m-tiles per band (0: the shape's default, Shape::kBand)
    int skip_shared;            // tiles of the shared group (kind 1) take no work here
    // COMBINE epilogue: the routed outputs and how to sum them into each token's row
    const bf16* cmb_yperm;      // y_perm [T*K][d]
    const int32_t* cmb_inv;     // inv_perm [T*K]: routed row of slot t*K + j (< 0: dropped)
    const float* cmb_w;         // topk_w [T*K]
    int cmb_K;
    int64_t cmb_rows;           // T*K (slots outside [0, cmb_rows) are dropped)
    int split;                  // take only the first hdr->units_pair / units_single units
    const int32_t* row_src;     // token of each routed row (gather from x), or null
    int gather_max;             // gather a CTA's routed rows when it has at most this many
    const FfnPlanHeader* hdr;
    const int4* mtiles;
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
    int test_stall;  // test hook: the producer issues no copy, so the bounded waits run out
};

struct Tile {
    int kind;   // 0 routed, 1 shared/dense
    int row0;   // first activation row of the tile (in the map of `kind`)
    int rows;   // valid rows of the tile
    int wrow0;  // first weight row of this n-block in the stacked matrix
    int n0;     // first output column
    int kblocks;
    bool valid;
    bool half;  // a pair tile of at most 128 rows, run with M = 128: 64 rows per CTA
    bool swap;  // a single tile of few rows, run with the operands swapped (see kSwap below)
    int nsw;    // swap: MMA N = the activation box height (16, 32 or 64 rows)
};

// KSTEP: elements of the reduction per K block (64 bf16 or 128 8-bit values,
// 128 bytes either way)
// The plan entry of tile t (group, first row, rows, m-tile index); a load
// whose result decode_tile_entry uses, so a role can issue it one tile ahead.
__device__ __forceinline__ int4 fetch_tile_entry(const TcParams& p, int t) {
    return p.dense_rows > 0 ? make_int4(-1, 0, p.dense_rows, t / p.NB) : p.mtiles[t / p.NB];
}

template <int EPI, bool PAIR, int KSTEP>
__device__ __forceinline__ Tile decode_tile_entry(const TcParams& p, int4 e, int t) {
    using S = Shape<PAIR>;
    constexpr int kNCols = EPI == EPI_SWIGLU ? BN / 2 : BN;  // output columns per n-block
    Tile tl;
    const int NB = p.NB;
    const int g = e.x, gr0 = e.y, Mg = e.z, i = e.w;
    const int q = t / NB;
    const int cnt = (Mg + S::kTileRows - 1) / S::kTileRows;
    const int tt = t - (q - i) * NB;  // index inside this group's tiles
    const int kb = p.band > 0 ? p.band : S::kBand;
    const int band = tt / (kb * NB);
    const int bstart = band * kb;
    const int bcnt = min(kb, cnt - bstart);
    const int r = tt - band * kb * NB;
    const int nb = r / bcnt;
    const int mi = bstart + r % bcnt;
    tl.kind = (p.dense_rows > 0 || g >= p.E) ? 1 : 0;
    tl.row0 = gr0 + mi * S::kTileRows;
    tl.rows = min(S::kTileRows, Mg - mi * S::kTileRows);
    tl.n0 = nb * kNCols;
    tl.wrow0 = (tl.kind == 0 ? g * p.wrows[0] : 0) + tl.n0;
    tl.kblocks = (p.kdim[tl.kind] + KSTEP - 1) / KSTEP;
    tl.valid = tl.n0 < p.n_out[tl.kind] && tl.rows > 0 && !(p.skip_shared && tl.kind == 1);
    tl.half = PAIR && p.half_tiles != 0 && tl.rows <= BMC;
    tl.swap = !PAIR && (EPI == EPI_SWIGLU || EPI == EPI_STORE_BF16) && tl.rows <= p.swap_max_rows;
    tl.nsw = abox_rows(abox_for(tl.rows));
    return tl;
}

template <int EPI, bool PAIR, int KSTEP>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, int n_tiles_in_list, int t) {
    (void)n_tiles_in_list;
    return decode_tile_entry<EPI, PAIR, KSTEP>(p, fetch_tile_entry(p, t), t);
}

struct SmemCtl {
    uint64_t full[kMaxStages];   // stage s landed (a pair: both CTAs' copies, on the even CTA)
    uint64_t empty[kMaxStages];  // the MMAs reading stage s completed (each CTA)
    uint64_t tfull[2];           // accumulator a is ready (each CTA)
    uint64_t tempty[2];          // the epilogue warps drained accumulator a (a pair: even CTA, 8 warps)
    uint64_t drain;
    uint64_t afull[kW8MaxA];      // W8: activation stage a landed (a pair: both CTAs' tiles, even CTA)
    uint64_t aempty[kW8MaxA];     // W8: the MMAs reading activation stage a completed (each CTA)
    uint64_t rfull[kW8MaxRaw];    // W8: this CTA's raw code tile r landed
    uint64_t rempty[kW8MaxRaw];   // W8: this CTA's 4 converter warps are done with raw tile r
    uint32_t tmem_base;
    volatile int abort_flag;
};

// Bounded wait: false (and the CTA-wide abort flag set) when the budget runs out
// or another role of this CTA already gave up.
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

template <bool PAIR>
__device__ __forceinline__ void cta_sync_all() {
    if constexpr (PAIR) {
        __syncwarp();  // the cluster barrier needs every warp converged
        ptx::cluster_sync();
    } else {
        __syncthreads();
    }
}

// two E4M3 codes (low byte first) -> two bf16 (low half first); exact
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(__half2(hr));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// W8 converter warp cw (0..3): rows RPW*cw .. RPW*cw+RPW-1 of K half h (codes
// 64h .. 64h+63 of each 128-code row) of a raw tile -> the bf16 weight tile of
// an MMA stage.  Both tiles use the 128-byte swizzle (16-byte chunk c of row r
// at chunk c ^ (r & 7)).  Lane 8j + 4s + q takes row 8*it + j + 4s: it reads
// code chunk 4h+q and writes bf16 chunks 2q and 2q+1, the odd one first when
// s = 1.  Each quarter-warp (8 lanes, one shared-memory wavefront of 16-byte
// accesses) then touches 8 distinct chunk positions on every load and store.
template <int RPW>  // weight rows per converter warp (64 single-SM, 32 in a pair)
__device__ __forceinline__ void convert_rows_w8(const uint8_t* raw, uint8_t* dst, int h, int cw,
                                                int lane) {
    const int q = lane & 3, s = (lane >> 2) & 1, j = lane >> 3;
#pragma unroll
    for (int it = 0; it < RPW / 8; ++it) {
        const int r = cw * RPW + it * 8 + j + 4 * s;
        const int x = r & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(raw + r * 128 + (((h * 4 + q) ^ x) << 4));
        uint4 lo, hi;
        lo.x = e4m3x2_to_bf16x2(v.x);
        lo.y = e4m3x2_to_bf16x2(v.x >> 16);
        lo.z = e4m3x2_to_bf16x2(v.y);
        lo.w = e4m3x2_to_bf16x2(v.y >> 16);
        hi.x = e4m3x2_to_bf16x2(v.z);
        hi.y = e4m3x2_to_bf16x2(v.z >> 16);
        hi.z = e4m3x2_to_bf16x2(v.w);
        hi.w = e4m3x2_to_bf16x2(v.w >> 16);
        const uint4 first = s ? hi : lo, second = s ? lo : hi;
        const int c_first = 2 * q + s, c_second = 2 * q + 1 - s;
        *reinterpret_cast<uint4*>(dst + r * 128 + ((c_first ^ x) << 4)) = first;
        *reinterpret_cast<uint4*>(dst + r * 128 + ((c_second ^ x) << 4)) = second;
    }
}

// 8-bit weights: the weight-row scales one epilogue warp needs for a tile,
// 8 per lane, requested before the warp waits for the tile's accumulator so the
// loads overlap the K loop (a short K loop -- 16 steps for a 2048-long 8-bit
// reduction -- would otherwise wait on one global load per 16 columns).  Each
// lane holds 8 consecutive scales: SWIGLU, lanes 0..n-1 the gate scales and
// lanes n..2n-1 the up scales (n = 16 for a full tile's 128 h columns, 8 for a
// half tile's 64); STORE, lanes 0..31 (or 0..15) the tile's 256 (or 128)
// output columns.  Columns past n_out read as 0 (never stored).
template <int EPI>
__device__ __forceinline__ void load_tile_scales(const TcParams& p, const Tile& tl, int hi, int lane,
                                                 int nvalid, float (&s)[8]) {
    const float* src = nullptr;
    int col = 0;  // first output (h or y) column of this lane's scales, relative to n0
    bool active;
    if (EPI == EPI_SWIGLU) {
        const int nl = (tl.half ? 64 : BN / 2) / 8;  // lanes per vector
        const bool up = lane >= nl;
        const int l = up ? lane - nl : lane;
        active = lane < 2 * nl;
        col = (tl.half ? 64 * hi : 0) + 8 * l;
        src = (up ? p.sc1[tl.kind] : p.sc0[tl.kind]) + tl.wrow0 + col;
    } else {
        active = 8 * lane < (tl.half ? BN / 2 : BN);
        col = (tl.half ? (BN / 2) * hi : 0) + 8 * lane;
        src = p.sc0[tl.kind] + tl.wrow0 + col;
    }
    if (active && tl.n0 + col < nvalid) {  // n_out is a multiple of 8: all 8 valid or none
        const float4 a = __ldg(reinterpret_cast<const float4*>(src));
        const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
        s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
        s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) s[k] = 0.0f;
    }
}

// 16 consecutive scales of load_tile_scales' layout, starting at vector lane
// `lane0` (the first of the 16 columns is a multiple of 8): every lane of the
// warp must call it.
__device__ __forceinline__ void tile_scales16(const float (&s)[8], int lane0, float (&out)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) out[k] = __shfl_sync(0xffffffffu, s[k & 7], lane0 + (k >> 3));
}

template <int EPI, bool PAIR, bool W8 = false, int A8 = 0, bool SMA = false>
__global__ void __launch_bounds__(threads_of<W8, A8>(), 1)
tc_gemm_kernel(const __grid_constant__ TcParams p) {
    static_assert(!(W8 && EPI == EPI_STORE_F32), "8-bit weights feed the expert GEMMs only");
    static_assert(!(SMA && (PAIR || W8)), "small-row ring: single-SM tiles without the W8 rings");
    static_assert(!(SMA && EPI == EPI_COMBINE), "small-row ring: expert GEMMs");
    static_assert(!(A8 && (W8 || EPI == EPI_STORE_F32)), "A8: 8-bit operands, expert GEMMs only");
    // activation tiles per stage: two E4M3 planes (A8 = 2, 3) or one
    constexpr uint32_t kAPlanes = (A8 == 2 || A8 == 3) ? 2u : 1u;
    constexpr bool kBlk = A8 >= 3;  // block-scaled weights: one accumulator hand-off per K block
    static_assert(!(kBlk && EPI != EPI_SWIGLU && EPI != EPI_STORE_BF16), "block scales: expert GEMMs");
    using S = typename RingOf<PAIR, SMA, A8>::type;
    using W = W8Shape<PAIR>;
    constexpr uint32_t kAStride = S::kAStride;  // bytes per activation stage (W8: kABytes)
    constexpr uint32_t kAPlane = kAStride / kAPlanes;  // bytes of one activation plane of a stage
    // A8: both operands E4M3 (kind::f8f6f4); a 128-byte K block holds 128 values
    constexpr int kKStep = A8 ? 2 * BK : BK;
    constexpr int kEpiWarps = kBlk ? 8 : 4;  // warps 2..5 (2..9)
    constexpr int kStages = W8 ? W::kConv : S::kStages;  // B stages (and A stages without W8)
    constexpr int kAStages = W8 ? W::kA : S::kStages;
    // swapped tiles (few rows): single-SM expert GEMMs on bf16 or 8-bit activations
    // (one or two planes) with row-scaled weights
    constexpr bool kSwap = !PAIR && !W8 && !kBlk && (EPI == EPI_SWIGLU || EPI == EPI_STORE_BF16);
    static_assert(!(EPI == EPI_COMBINE && (W8 || A8 || SMA)), "COMBINE: the bf16 shared down GEMM");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzle atoms (the same offset in both CTAs of a pair)
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kAStages * kAStride;
    uint8_t* sRaw = sB + kStages * S::kBBytes;  // W8 only
    SmemCtl* ctl = (SmemCtl*)(smem + (W8 ? kW8RingBytes : S::kRingBytes));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;  // 0 issues the MMAs
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int n_units_grid = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // W8: full = the converter warps (of both CTAs of a pair) wrote the bf16 weight tile
            ptx::mbar_init(&ctl->full[s], W8 ? W::kConvArrivals : 1);
            ptx::mbar_init(&ctl->empty[s], 1);
        }
        if constexpr (W8) {
            for (int a = 0; a < W::kA; ++a) {
                ptx::mbar_init(&ctl->afull[a], 1);
                ptx::mbar_init(&ctl->aempty[a], 1);
            }
            for (int r = 0; r < W::kRaw; ++r) {
                ptx::mbar_init(&ctl->rfull[r], 1);
                ptx::mbar_init(&ctl->rempty[r], kW8ConvWarps);
            }
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&ctl->tfull[a], 1);
            // block scales: one arrival per CTA per K block (after the epilogue
            // warps' named barrier); otherwise one per epilogue warp per tile
            ptx::mbar_init(&ctl->tempty[a], (PAIR ? 2 : 1) * (kBlk ? 1 : kEpiWarps));
        }
        ptx::mbar_init(&ctl->drain, 1);
        ctl->abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        if (p.row_src) ptx::prefetch_tmap(&p.ag);
        for (int k = 0; k < 2; ++k) {
            for (int b = 0; b < kABoxes; ++b) ptx::prefetch_tmap(&p.a[k][b]);
            if (W8) {
                if (EPI == EPI_SWIGLU) {
                    ptx::prefetch_tmap(&p.q0[k]);
                    ptx::prefetch_tmap(&p.q1[k]);
                } else {
                    ptx::prefetch_tmap(&p.qw[k]);
                }
            } else if (PAIR || EPI == EPI_SWIGLU) {
                ptx::prefetch_tmap(&p.b0[k]);
                if (EPI == EPI_SWIGLU) ptx::prefetch_tmap(&p.b1[k]);
            } else {
                ptx::prefetch_tmap(&p.bw[k]);
            }
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    cta_sync_all<PAIR>();  // barriers initialised (in both CTAs of a pair), tensor memory allocated
    ptx::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    // the prologue above overlaps the previous kernel; its outputs (plan, operands) are read below
    pdl_wait();
    const int list_len = p.dense_rows > 0
        ? (p.dense_rows + S::kTileRows - 1) / S::kTileRows
        : min(PAIR ? p.hdr->n_ptiles : p.hdr->n_mtiles, p.max_mtiles);
    // Side by side with the other tile shape, this grid keeps the plan's share
    // of the SMs; its other units take no tile and leave through the teardown.
    const int n_units = p.split ? min(n_units_grid, PAIR ? p.hdr->units_pair : p.hdr->units_single)
                                : n_units_grid;
    const int n_tiles = unit < n_units ? list_len * p.NB : 0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (warp 0)
        // Lane 0 runs the barrier handshake and the weight loads.  Routed
        // activation rows of moe_forward are gathered straight from x with
        // tile::gather4 (the row -> token map of the dispatch gives the rows):
        // lane l loads rows 4l..4l+3 of this CTA's block, so one stage takes up
        // to 32 gather instructions issued in parallel.
        if constexpr (W8) {
            // W8: lane 0 streams this CTA's raw code tiles (two K steps each; a
            // pair: the even CTA the gate rows or weight rows 0-127 of the
            // n-block, the odd CTA the up rows or rows 128-255) and its
            // activation tiles, each ring as far ahead as it has free stages.
            if (lane == 0) {
                int rs = 0, as = 0;
                uint32_t rph = 0, aph = 0;
                bool r_issued[W::kRaw], a_issued[W::kA];
                uint32_t r_phase[W::kRaw], a_phase[W::kA];
                for (int r = 0; r < W::kRaw; ++r) { r_issued[r] = false; r_phase[r] = 0; }
                for (int a = 0; a < W::kA; ++a) { a_issued[a] = false; a_phase[a] = 0; }
                const uint32_t afull0 = PAIR ? ptx::map_to_rank(&ctl->afull[0], 0) : 0u;
                bool ok = p.test_stall == 0;
                for (int t = unit; t < n_tiles && ok; t += n_units) {
                    const Tile tl = decode_tile<EPI, PAIR, kKStep>(p, list_len, t);
                    if (!tl.valid) continue;
                    const int rows_me = max(0, min(BMC, tl.rows - (int)rank * BMC));
                    const CUtensorMap* ma = &p.a[tl.kind][abox_for(rows_me)];
                    const int arow = tl.row0 + (int)rank * BMC;
                    // bytes of one activation stage (both CTAs' tiles in a pair)
                    const uint32_t abytes = PAIR ? abytes_for(min(BMC, tl.rows)) + abytes_for(tl.rows - BMC)
                                                 : abytes_for(rows_me);
                    for (int kb = 0; kb < tl.kblocks; ++kb) {
                        if ((kb & 1) == 0) {
                            if (!wait_bounded(&ctl->rempty[rs], rph ^ 1u, ctl, p, 110)) { ok = false; break; }
                            uint8_t* dst = sRaw + rs * W::kRawBytes;
                            // a box past the end of K or of the weight rows is zero-filled
                            // and still counts its full size
                            ptx::mbar_arrive_expect_tx(&ctl->rfull[rs], W::kRawBytes);
                            const int kr = kb >> 1;
                            if constexpr (PAIR) {
                                const CUtensorMap* mq = (EPI == EPI_SWIGLU && rank == 1) ? &p.q1[tl.kind]
                                                                                         : &p.q0[tl.kind];
                                const int qrow = tl.wrow0 + (EPI == EPI_SWIGLU ? 0 : (int)rank * S::kBRows);
                                ptx::tma_load_2d(dst, mq, &ctl->rfull[rs], kr * 128, qrow);
                            } else if (EPI == EPI_SWIGLU) {
                                ptx::tma_load_2d(dst, &p.q0[tl.kind], &ctl->rfull[rs], kr * 128, tl.wrow0);
                                ptx::tma_load_2d(dst + W::kRawBytes / 2, &p.q1[tl.kind], &ctl->rfull[rs],
                                                 kr * 128, tl.wrow0);
                            } else {
                                ptx::tma_load_2d(dst, &p.qw[tl.kind], &ctl->rfull[rs], kr * 128, tl.wrow0);
                            }
                            r_issued[rs] = true;
                            r_phase[rs] = rph;
                            if (++rs == W::kRaw) { rs = 0; rph ^= 1u; }
                        }
                        if (!wait_bounded(&ctl->aempty[as], aph ^ 1u, ctl, p, 111)) { ok = false; break; }
                        if constexpr (PAIR) {
                            const uint32_t ab = afull0 + (uint32_t)(as * sizeof(uint64_t));
                            if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl->afull[as], abytes);
                            if (rows_me > 0) ptx::tma_load_2d_pair(sA + as * kABytes, ma, ab, kb * BK, arow);
                        } else {
                            ptx::mbar_arrive_expect_tx(&ctl->afull[as], abytes);
                            ptx::tma_load_2d(sA + as * kABytes, ma, &ctl->afull[as], kb * BK, arow);
                        }
                        a_issued[as] = true;
                        a_phase[as] = aph;
                        if (++as == W::kA) { as = 0; aph ^= 1u; }
                    }
                }
                if (!ok || ctl->abort_flag) {
                    // every copy issued lands before teardown: raw tiles on this CTA's
                    // barriers; activation tiles on the even CTA's (the odd CTA cannot
                    // observe those, so it gives its copies a bounded time)
                    for (int r = 0; r < W::kRaw; ++r) {
                        if (!r_issued[r]) continue;
                        const uint64_t t0 = ptx::globaltimer_ns();
                        while (!ptx::mbar_try_wait(&ctl->rfull[r], r_phase[r]) &&
                               ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                    }
                    if (rank == 0) {
                        for (int a = 0; a < W::kA; ++a) {
                            if (!a_issued[a]) continue;
                            const uint64_t t0 = ptx::globaltimer_ns();
                            while (!ptx::mbar_try_wait(&ctl->afull[a], a_phase[a]) &&
                                   ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                            }
                        }
                    } else {
                        const uint64_t t0 = ptx::globaltimer_ns();
                        while (ptx::globaltimer_ns() - t0 < 2000000ull) {
                        }
                    }
                }
            }
        } else {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kMaxStages];
            bool issued[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            const uint32_t full0 = PAIR ? ptx::map_to_rank(&ctl->full[0], 0) : 0u;
            bool ok = p.test_stall == 0;
            for (int t = unit; t < n_tiles && ok; t += n_units) {
                const Tile tl = decode_tile<EPI, PAIR, kKStep>(p, list_len, t);
                if (!tl.valid) continue;
                const int crows = tl.half ? BMC / 2 : BMC;  // activation rows per CTA
                int rows_me = max(0, min(crows, tl.rows - (int)rank * crows));
                if constexpr (SMA) {
                    // the host sends only groups of <= kSmaRows rows here; anything
                    // longer is reported, and no copy spills past its 4 KB stage
                    if (rows_me > kSmaRows) {
                        if (lane == 0) record_error(p.err, MOE_ERR_BOUNDS, 60);
                        rows_me = kSmaRows;
                    }
                }
                const CUtensorMap* ma = &p.a[tl.kind][abox_for(rows_me)];
                const int arow = tl.row0 + (int)rank * crows;
                const bool gather = tl.kind == 0 && p.row_src != nullptr && rows_me <= p.gather_max;
                const int n4 = gather ? (rows_me + 3) / 4 : 0;
                int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
                if (lane < n4) {  // padding rows repeat the last valid row
                    const int b = 4 * lane, last = rows_me - 1;
                    r0 = p.row_src[arow + min(b, last)];
                    r1 = p.row_src[arow + min(b + 1, last)];
                    r2 = p.row_src[arow + min(b + 2, last)];
                    r3 = p.row_src[arow + min(b + 3, last)];
                }
                // bytes of one CTA's activation rows (each CTA of a pair decides by its own rows)
                const bool can_gather = tl.kind == 0 && p.row_src != nullptr;
                const int gmax = p.gather_max;
                const auto a_bytes = [can_gather, gmax](int rows) -> uint32_t {
                    return (can_gather && rows <= gmax) ? (uint32_t)((rows + 3) / 4) * 512u
                                                        : abytes_for(rows);
                };
                uint32_t tx;
                const CUtensorMap* mb;
                int brow;
                // Half gate/up pair tiles: each CTA loads the gate rows (smem rows 0-63)
                // and the up rows (64-127) of its 64 intermediate indices, so that with
                // M = 128 the gate and up sums of one index land in the same thread's
                // tensor-memory columns (c and 64 + c).
                const bool split64 = EPI == EPI_SWIGLU && tl.half;
                const int j64 = tl.wrow0 + (int)rank * (BMC / 2);
                const auto load_b_pair = [&](uint8_t* b_dst, uint32_t fb, int k0, const CUtensorMap* mbp,
                                             int browp) {
                    if (split64) {
                        ptx::tma_load_2d_pair(b_dst, &p.g64[tl.kind], fb, k0, j64);
                        ptx::tma_load_2d_pair(b_dst + 64 * 128, &p.u64[tl.kind], fb, k0, j64);
                    } else {
                        ptx::tma_load_2d_pair(b_dst, mbp, fb, k0, browp);
                    }
                };
                if constexpr (PAIR) {
                    tx = kAPlanes * (a_bytes(min(crows, tl.rows)) + a_bytes(max(0, tl.rows - crows))) +
                         2 * S::kBBytes;
                    mb = (EPI == EPI_SWIGLU && rank == 1) ? &p.b1[tl.kind] : &p.b0[tl.kind];
                    brow = tl.wrow0 + ((EPI == EPI_SWIGLU) ? 0 : (int)rank * S::kBRows);
                } else {
                    tx = kAPlanes * a_bytes(rows_me) + S::kBBytes;
                    mb = EPI == EPI_SWIGLU ? &p.b0[tl.kind] : &p.bw[tl.kind];
                    brow = tl.wrow0;
                }
                if (!gather) {
                    // lane 0 alone; the other lanes only keep the ring position
                    if (lane == 0) {
                        for (int kb = 0; kb < tl.kblocks; ++kb) {
                            if (!wait_bounded(&ctl->empty[stage], phase ^ 1u, ctl, p, 100)) { ok = false; break; }
                            const int k0 = kb * kKStep;
                            uint8_t* a_dst = sA + stage * kAStride;
                            uint8_t* b_dst = sB + stage * S::kBBytes;
                            if constexpr (PAIR) {
                                const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
                                if (rank == 0) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
                                if (rows_me > 0) {
                                    if constexpr (kAPlanes == 2) {  // hi and lo codes of K block kb
                                        ptx::tma_load_2d_pair(a_dst, ma, fb, 2 * k0, arow);
                                        ptx::tma_load_2d_pair(a_dst + kAPlane, ma, fb, 2 * k0 + 128, arow);
                                    } else {
                                        ptx::tma_load_2d_pair(a_dst, ma, fb, k0, arow);
                                    }
                                }
                                load_b_pair(b_dst, fb, k0, mb, brow);
                            } else {
                                ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
                                if constexpr (kAPlanes == 2) {
                                    ptx::tma_load_2d(a_dst, ma, &ctl->full[stage], 2 * k0, arow);
                                    ptx::tma_load_2d(a_dst + kAPlane, ma, &ctl->full[stage], 2 * k0 + 128, arow);
                                } else {
                                    ptx::tma_load_2d(a_dst, ma, &ctl->full[stage], k0, arow);
                                }
                                ptx::tma_load_2d(b_dst, mb, &ctl->full[stage], k0, brow);
                                if (EPI == EPI_SWIGLU)
                                    ptx::tma_load_2d(b_dst + S::kBBytes / 2, &p.b1[tl.kind], &ctl->full[stage], k0, brow);
                            }
                            issued[stage] = true;
                            issued_phase[stage] = phase;
                            if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
                        }
                    } else {
                        const int adv = stage + tl.kblocks;
                        phase ^= (uint32_t)((adv / S::kStages) & 1);
                        stage = adv % S::kStages;
                    }
                } else {
                    for (int kb = 0; kb < tl.kblocks; ++kb) {
                        const int okw = lane == 0 ? (int)wait_bounded(&ctl->empty[stage], phase ^ 1u, ctl, p, 100) : 0;
                        if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
                        const int k0 = kb * kKStep;
                        uint8_t* a_dst = sA + stage * kAStride;
                        uint8_t* b_dst = sB + stage * S::kBBytes;
                        if constexpr (PAIR) {
                            const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
                            if (lane == 0 && rank == 0) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
                            __syncwarp();
                            if (lane < n4) ptx::tma_gather4_pair(a_dst + lane * 512, &p.ag, fb, k0, r0, r1, r2, r3);
                            if (lane == 0) load_b_pair(b_dst, fb, k0, mb, brow);
                        } else {
                            if (lane == 0) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
                            __syncwarp();  // the byte count is posted before any gathered row lands
                            if (lane < n4)
                                ptx::tma_gather4(a_dst + lane * 512, &p.ag, &ctl->full[stage], k0, r0, r1, r2, r3);
                            if (lane == 0) {
                                ptx::tma_load_2d(b_dst, mb, &ctl->full[stage], k0, brow);
                                if (EPI == EPI_SWIGLU)
                                    ptx::tma_load_2d(b_dst + S::kBBytes / 2, &p.b1[tl.kind], &ctl->full[stage], k0, brow);
                            }
                        }
                        issued[stage] = true;
                        issued_phase[stage] = phase;
                        if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
                ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;  // every lane agrees to stop
            }
            if (!ok && lane == 0) {
                if (rank == 0) {
                    // drain: every copy issued (for a pair, both CTAs' copies land on
                    // this CTA's full barriers) lands before teardown
                    for (int s = 0; s < S::kStages; ++s) {
                        if (!issued[s]) continue;
                        const uint64_t t0 = ptx::globaltimer_ns();
                        while (!ptx::mbar_try_wait(&ctl->full[s], issued_phase[s]) &&
                               ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                    }
                } else {
                    // the odd CTA of a pair cannot observe the even CTA's barriers: give
                    // its copies in flight a bounded time to land before teardown
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (ptx::globaltimer_ns() - t0 < 2000000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (rank 0)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = A8 ? ptx::idesc_e4m3_f32(S::kTileRows, BN)
                                          : ptx::idesc_bf16_f32(S::kTileRows, BN);
            // half pair tiles: M = 128, 64 rows of A from each CTA
            constexpr uint32_t idesc_half = A8 ? ptx::idesc_e4m3_f32(BMC, BN)
                                               : ptx::idesc_bf16_f32(BMC, BN);
            int stage = 0;       // B stage (and A stage without W8)
            uint32_t phase = 0;
            int ast = 0;         // W8: A stage
            uint32_t aphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            // the next tile's plan entry is loaded while this tile's MMAs run (its load
            // took ~700 cycles per tile of this warp's time; measured 0.5 % faster on
            // the bf16 prefill layers, neutral elsewhere)
            int4 entry_next = unit < n_tiles ? fetch_tile_entry(p, unit) : make_int4(0, 0, 0, 0);
            for (int t = unit; t < n_tiles && ok; t += n_units) {
                const int4 entry = entry_next;
                if (t + n_units < n_tiles) entry_next = fetch_tile_entry(p, t + n_units);
                const Tile tl = decode_tile_entry<EPI, PAIR, kKStep>(p, entry, t);
                if (!tl.valid) continue;
                if (!kBlk && !wait_bounded(&ctl->tempty[acc], acc_phase ^ 1u, ctl, p, 200)) { ok = false; break; }
                ptx::tc_fence_after();
                uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                const uint32_t id_t = tl.half ? idesc_half : idesc;
                const bool swp = kSwap && tl.swap;
                // swapped: M = 128, N = the box rows (within the small-row ring's 32-row stage)
                const int n_sw = SMA ? min(tl.nsw, kSmaRows) : tl.nsw;
                const uint32_t id_sw = A8 ? ptx::idesc_e4m3_f32(BMC, n_sw) : ptx::idesc_bf16_f32(BMC, n_sw);
                for (int kb = 0; kb < tl.kblocks; ++kb) {
                    if constexpr (kBlk) {  // each K block into a drained accumulator
                        if (!wait_bounded(&ctl->tempty[acc], acc_phase ^ 1u, ctl, p, 203)) { ok = false; break; }
                        ptx::tc_fence_after();
                        d_tmem = tmem + (uint32_t)(acc * BN);
                    }
                    if (!wait_bounded(&ctl->full[stage], phase, ctl, p, 201)) { ok = false; break; }
                    if (W8 && !wait_bounded(&ctl->afull[ast], aphase, ctl, p, 202)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a_base = ptx::smem_u32(sA + (W8 ? ast : stage) * kAStride);
                    const uint32_t b_base = ptx::smem_u32(sB + stage * S::kBBytes);
                    if (kSwap && swp) {
                        // weight halves (rows 0-127 and 128-255 of the stage) times the
                        // activation rows: two M = 128, N = nsw products per 16-deep
                        // (bf16) or 32-deep (8-bit) slice, twice with two planes
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t xd = ptx::sw128_kmajor_desc(a_base + kk * 32);
                            const uint64_t w0 = ptx::sw128_kmajor_desc(b_base + kk * 32);
                            const uint64_t w1 = ptx::sw128_kmajor_desc(b_base + S::kBBytes / 2 + kk * 32);
                            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
                            if constexpr (A8) {
                                ptx::tc_mma_f8(d_tmem, w0, xd, id_sw, accum);
                                ptx::tc_mma_f8(d_tmem + BN / 2, w1, xd, id_sw, accum);
                                if constexpr (kAPlanes == 2) {  // the lo plane
                                    const uint64_t xd2 = ptx::sw128_kmajor_desc(a_base + kAPlane + kk * 32);
                                    ptx::tc_mma_f8(d_tmem, w0, xd2, id_sw, 1u);
                                    ptx::tc_mma_f8(d_tmem + BN / 2, w1, xd2, id_sw, 1u);
                                }
                            } else {
                                ptx::tc_mma_f16(d_tmem, w0, xd, id_sw, accum);
                                ptx::tc_mma_f16(d_tmem + BN / 2, w1, xd, id_sw, accum);
                            }
                        }
                        any = true;
                        ptx::tc_commit(&ctl->empty[stage]);
                        if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        continue;
                    }
#pragma unroll
                    // four MMAs per 128-byte K block: K = 16 bf16 or 32 E4M3 values each
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = ptx::sw128_kmajor_desc(a_base + kk * 32);
                        const uint64_t bd = ptx::sw128_kmajor_desc(b_base + kk * 32);
                        const uint32_t accum = ((kBlk ? 0 : kb) | kk) != 0 ? 1u : 0u;
                        if constexpr (A8) {
                            if constexpr (PAIR) ptx::tc_mma_f8_pair(d_tmem, ad, bd, id_t, accum);
                            else ptx::tc_mma_f8(d_tmem, ad, bd, idesc, accum);
                            if constexpr (kAPlanes == 2) {  // the lo plane times the same weights
                                const uint64_t ad2 = ptx::sw128_kmajor_desc(a_base + kAPlane + kk * 32);
                                if constexpr (PAIR) ptx::tc_mma_f8_pair(d_tmem, ad2, bd, id_t, 1u);
                                else ptx::tc_mma_f8(d_tmem, ad2, bd, idesc, 1u);
                            }
                        } else {
                            if constexpr (PAIR) ptx::tc_mma_f16_pair(d_tmem, ad, bd, id_t, accum);
                            else ptx::tc_mma_f16(d_tmem, ad, bd, idesc, accum);
                        }
                    }
                    any = true;
                    if constexpr (PAIR) ptx::tc_commit_pair(&ctl->empty[stage], 0x3);
                    else ptx::tc_commit(&ctl->empty[stage]);
                    if constexpr (W8) {
                        if constexpr (PAIR) ptx::tc_commit_pair(&ctl->aempty[ast], 0x3);
                        else ptx::tc_commit(&ctl->aempty[ast]);
                        if (++ast == W::kA) { ast = 0; aphase ^= 1u; }
                    }
                    if constexpr (kBlk) {
                        if constexpr (PAIR) ptx::tc_commit_pair(&ctl->tfull[acc], 0x3);
                        else ptx::tc_commit(&ctl->tfull[acc]);
                        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if constexpr (!kBlk) {
                    if constexpr (PAIR) ptx::tc_commit_pair(&ctl->tfull[acc], 0x3);
                    else ptx::tc_commit(&ctl->tfull[acc]);
                    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                }
            }
            if (!ok && any) {
                // drain: every MMA issued completes before tensor memory is freed
                if constexpr (PAIR) ptx::tc_commit_pair(&ctl->drain, 0x3);
                else ptx::tc_commit(&ctl->drain);
                const uint64_t t0 = ptx::globaltimer_ns();
                while (!ptx::mbar_try_wait(&ctl->drain, 0) &&
                       ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                }
            }
        }
    } else if (kBlk) {
        // ------------------------------------------------ epilogue, block-scaled weights (warps 2..9)
        // Warp pair (w, w + 4) shares tensor-memory lane quarter w & 3; `half`
        // picks its columns: SWIGLU, gate columns 64 half .. +63 and the up
        // columns 128 + 64 half .. +63 (the same intermediate indices, one
        // weight block row); STORE, output columns 128 half .. +127 (weight
        // block row wrow0 / 128 + half).  Per K block: wait for its accumulator,
        // add scale * products to the 128 register sums, free the accumulator.
        // After the tile's last K block: times the activation row's scale, store.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quad * 32 + lane;  // accumulator row owned by this thread
        const uint32_t tempty0 = PAIR ? ptx::map_to_rank(&ctl->tempty[0], 0) : 0u;
        constexpr int kPart = 64;  // columns of each of the two parts a thread sums
        const int c_a = EPI == EPI_SWIGLU ? kPart * half : 2 * kPart * half;
        const int c_b = EPI == EPI_SWIGLU ? BN / 2 + kPart * half : 2 * kPart * half + kPart;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int t = unit; t < n_tiles && ok; t += n_units) {
            const Tile tl = decode_tile<EPI, PAIR, kKStep>(p, list_len, t);
            if (!tl.valid) continue;
            const int rows_me = max(0, min(BMC, tl.rows - (int)rank * BMC));
            const bool row_ok = r < rows_me;
            const int arow_me = tl.row0 + (int)rank * BMC + r;
            const int nvalid = p.n_out[tl.kind];
            const int nkb = tl.kblocks;
            // the scales of this warp's weight block row(s) along K
            const int out0 = EPI == EPI_SWIGLU ? tl.n0 + kPart * half : tl.n0 + 2 * kPart * half;
            const bool cols_ok = out0 < nvalid;  // n_out is a multiple of 128
            const int64_t brow = (int64_t)(tl.wrow0 / kWBlock + (EPI == EPI_SWIGLU ? 0 : half)) * nkb;
            const float* s_a = p.sc0[tl.kind] + brow;
            const float* s_b = (EPI == EPI_SWIGLU ? p.sc1[tl.kind] : p.sc0[tl.kind]) + brow;
            const float sa = row_ok ? __ldg(p.sa[tl.kind] + arow_me) : 0.0f;
            float sum[2 * kPart];
#pragma unroll
            for (int k = 0; k < 2 * kPart; ++k) sum[k] = 0.0f;
            float ws_a = cols_ok ? __ldg(s_a) : 0.0f, ws_b = cols_ok ? __ldg(s_b) : 0.0f;
            for (int kb = 0; kb < nkb; ++kb) {
                // the next K block's scales are requested before this block's wait
                const bool nx = cols_ok && kb + 1 < nkb;
                const float nx_a = nx ? __ldg(s_a + kb + 1) : 0.0f;
                const float nx_b = nx ? __ldg(s_b + kb + 1) : 0.0f;
                const int okw = lane == 0 ? (int)wait_bounded(&ctl->tfull[acc], acc_phase, ctl, p, 310) : 0;
                const bool ready = __shfl_sync(0xffffffffu, okw, 0) != 0;
                if (ready) {
                    ptx::tc_fence_after();
                    const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll
                    for (int c = 0; c < kPart; c += 16) {
                        uint32_t va[16], vb[16];
                        ptx::tmem_ld16(tbase + c_a + c, va);
                        ptx::tmem_ld16(tbase + c_b + c, vb);
                        ptx::tmem_ld_wait();
                        // packed FMAs (measured on GB300: block-scaled stage 1.11 -> 1.07 ms)
#pragma unroll
                        for (int k = 0; k < 16; k += 2) {
                            ptx::fma2_f32(sum[c + k], sum[c + k + 1], ws_a, __uint_as_float(va[k]),
                                          __uint_as_float(va[k + 1]));
                            ptx::fma2_f32(sum[kPart + c + k], sum[kPart + c + k + 1], ws_b,
                                          __uint_as_float(vb[k]), __uint_as_float(vb[k + 1]));
                        }
                    }
                    ptx::tc_fence_before();
                }
                // Every epilogue warp reaches this barrier whatever its wait gave (its
                // only blocking step is that bounded wait), so it cannot hang; past it,
                // all eight have read the accumulator, or all leave together.
                if (!ptx::named_bar_and(kBlkEpiBar, 8 * 32, ready)) { ok = false; break; }
                if (warp == 2 && lane == 0) {
                    if constexpr (PAIR) ptx::mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
                    else ptx::mbar_arrive(&ctl->tempty[acc]);
                }
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                ws_a = nx_a;
                ws_b = nx_b;
            }
            if (!ok || !row_ok || !cols_ok) continue;
            bf16* out = (bf16*)p.out[tl.kind] + (int64_t)arow_me * p.ld_out[tl.kind] + out0;
            if constexpr (EPI == EPI_SWIGLU) {
                uint32_t hmax_bits = 0;
#pragma unroll
                for (int c = 0; c < kPart; c += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float h0 = silu_mul(sum[c + 2 * k] * sa, sum[kPart + c + 2 * k] * sa);
                        const float h1 = silu_mul(sum[c + 2 * k + 1] * sa, sum[kPart + c + 2 * k + 1] * sa);
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                        hmax_bits = max(hmax_bits, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
                    }
                    *reinterpret_cast<uint4*>(out + c) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                // the row's max |h| over every tile of the row, for its two-plane split
                if (hmax_bits != 0) atomicMax(p.hmax[tl.kind] + arow_me, hmax_bits << 16);
            } else {
#pragma unroll
                for (int c = 0; c < 2 * kPart; c += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(sum[c + 2 * k] * sa, sum[c + 2 * k + 1] * sa);
                        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    *reinterpret_cast<uint4*>(out + c) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    } else if (!W8 || warp < 6) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quad = warp & 3;       // TMEM lanes 32*quad .. 32*quad+31
        const int r = quad * 32 + lane;  // accumulator row owned by this thread
        const uint32_t tempty0 = PAIR ? ptx::map_to_rank(&ctl->tempty[0], 0) : 0u;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = unit; t < n_tiles; t += n_units) {
            const Tile tl = decode_tile<EPI, PAIR, kKStep>(p, list_len, t);
            if (!tl.valid) continue;
            // Half pair tiles (M = 128) leave each CTA 64 rows: tensor-memory lane L
            // holds row L & 63; lanes 0-63 hold output columns 0-127 of the n-block
            // and lanes 64-127 columns 128-255, in tensor-memory columns 0-127.
            const int crows = tl.half ? BMC / 2 : BMC;
            const int hi = tl.half ? (r >> 6) : 0;  // the same for the whole warp
            const int rr = tl.half ? (r & 63) : r;
            const int rows_me = max(0, min(crows, tl.rows - (int)rank * crows));
            const bool row_ok = rr < rows_me;
            const int arow_me = tl.row0 + (int)rank * crows + rr;  // activation row of this thread
            const int64_t orow = arow_me;
            const int nvalid = p.n_out[tl.kind];
            // scales are requested before the accumulator wait, so they arrive during
            // the K loop: A8, the activation row's scale (it factors out of every
            // output of the row); 8-bit weights, the tile's weight-row scales
            const float sa = (A8 && row_ok) ? __ldg(p.sa[tl.kind] + arow_me) : 1.0f;
            float sreg[8];
            if constexpr (W8 || A8) load_tile_scales<EPI>(p, tl, hi, lane, nvalid, sreg);
            // one lane waits, the warp follows its verdict (tcgen05.ld needs the whole warp)
            const int ok = lane == 0 ? (int)wait_bounded(&ctl->tfull[acc], acc_phase, ctl, p, 300) : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
            if (kSwap && tl.swap) {
                // Swapped tile: tensor-memory lane r is weight row r of the n-block --
                // h column n0 + r (gate sums in columns t, up sums in 128 + t), or y
                // columns n0 + r and n0 + 128 + r -- and column t is the tile's
                // activation row t.  A warp's 32 lanes store 32 adjacent columns of a row.
                const int col = tl.n0 + r;
                const int64_t ld = p.ld_out[tl.kind];
                bf16* base = (bf16*)p.out[tl.kind] + (int64_t)tl.row0 * ld;
                const int nsw = SMA ? min(tl.nsw, kSmaRows) : tl.nsw;
                // 8-bit operands: this lane's weight-row scales (gate and up, or the
                // two output columns' rows); each activation row's scale per batch
                float w_a = 1.0f, w_b = 1.0f;
                if constexpr (A8) {
                    if (EPI == EPI_SWIGLU) {
                        if (col < nvalid) {
                            w_a = __ldg(p.sc0[tl.kind] + tl.wrow0 + r);
                            w_b = __ldg(p.sc1[tl.kind] + tl.wrow0 + r);
                        }
                    } else {
                        if (col < nvalid) w_a = __ldg(p.sc0[tl.kind] + tl.wrow0 + r);
                        if (col + BN / 2 < nvalid) w_b = __ldg(p.sc0[tl.kind] + tl.wrow0 + BN / 2 + r);
                    }
                }
#pragma unroll 1
                for (int t0 = 0; t0 < nsw; t0 += 16) {
                    uint32_t a[16], b[16];
                    ptx::tmem_ld16(tbase + t0, a);
                    ptx::tmem_ld16(tbase + BN / 2 + t0, b);
                    const int nt = min(16, tl.rows - t0);  // valid activation rows in this batch
                    float sat[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        sat[k] = (A8 && k < nt) ? __ldg(p.sa[tl.kind] + tl.row0 + t0 + k) : 1.0f;
                    ptx::tmem_ld_wait();
                    if (EPI == EPI_SWIGLU) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            if (k < nt) {  // (uniform across the warp)
                                const __nv_bfloat16 hv = __float2bfloat16_rn(
                                    silu_mul(__uint_as_float(a[k]) * (w_a * sat[k]),
                                             __uint_as_float(b[k]) * (w_b * sat[k])));
                                if (col < nvalid) base[(int64_t)(t0 + k) * ld + col] = hv;
                                if constexpr (A8) {
                                    // the activation row's max |h| over this warp's 32 columns
                                    const uint32_t bits =
                                        col < nvalid ? (uint32_t)(__bfloat16_as_ushort(hv) & 0x7FFFu) : 0u;
                                    const uint32_t m = __reduce_max_sync(0xffffffffu, bits);
                                    if (lane == 0 && m != 0)
                                        atomicMax(p.hmax[tl.kind] + tl.row0 + t0 + k, m << 16);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            if (k < nt) {
                                bf16* dst = base + (int64_t)(t0 + k) * ld + col;
                                if (col < nvalid)
                                    dst[0] = __float2bfloat16_rn(__uint_as_float(a[k]) * (w_a * sat[k]));
                                if (col + BN / 2 < nvalid)
                                    dst[BN / 2] = __float2bfloat16_rn(__uint_as_float(b[k]) * (w_b * sat[k]));
                            }
                        }
                    }
                }
            } else if (EPI == EPI_SWIGLU && tl.half) {
                // tensor-memory columns 0-63: gate sums, 64-127: up sums of the same 64
                // intermediate indices (n0 + 64 hi ..) of this thread's row
                bf16* out = (bf16*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0 + 64 * hi;
                uint32_t hmax_bits = 0;
#pragma unroll 1
                for (int c = 0; c < 64; c += 16) {
                    uint32_t g[16], u[16];
                    ptx::tmem_ld16(tbase + c, g);
                    ptx::tmem_ld16(tbase + 64 + c, u);
                    const int hc = 64 * hi + c;  // first h column, relative to n0
                    const bool col_ok = tl.n0 + hc < nvalid;
                    float gs[16], us[16];
                    if constexpr (W8 || A8) {  // gate scales in lanes 0-7, up in 8-15
                        tile_scales16(sreg, c >> 3, gs);
                        tile_scales16(sreg, 8 + (c >> 3), us);
                    }
                    ptx::tmem_ld_wait();
                    if (row_ok && col_ok) {
                        if constexpr (W8 || A8) {
                            if constexpr (A8) {
#pragma unroll
                                for (int k = 0; k < 16; ++k) { gs[k] *= sa; us[k] *= sa; }
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) { gs[k] = 1.0f; us[k] = 1.0f; }
                        }
                        uint32_t w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float h0 = silu_mul(__uint_as_float(g[2 * k]) * gs[2 * k],
                                                      __uint_as_float(u[2 * k]) * us[2 * k]);
                            const float h1 = silu_mul(__uint_as_float(g[2 * k + 1]) * gs[2 * k + 1],
                                                      __uint_as_float(u[2 * k + 1]) * us[2 * k + 1]);
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                            w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        if constexpr (A8) {
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                hmax_bits = max(hmax_bits, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
                        }
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                if (A8 && row_ok && hmax_bits != 0) atomicMax(p.hmax[tl.kind] + arow_me, hmax_bits << 16);
            } else if (EPI == EPI_SWIGLU) {
                bf16* out = (bf16*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0;
                uint32_t hmax_bits = 0;  // A8: largest |h| this thread stored (bf16 bits)
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 16) {
                    uint32_t g[16], u[16];
                    ptx::tmem_ld16(tbase + c, g);
                    ptx::tmem_ld16(tbase + BN / 2 + c, u);
                    const bool col_ok = tl.n0 + c < nvalid;
                    float gs[16], us[16];
                    if constexpr (W8 || A8) {  // gate scales in lanes 0-15, up in 16-31
                        tile_scales16(sreg, c >> 3, gs);
                        tile_scales16(sreg, 16 + (c >> 3), us);
                    }
                    ptx::tmem_ld_wait();
                    if (row_ok && col_ok) {
                        if constexpr (W8 || A8) {
                            if constexpr (A8) {
#pragma unroll
                                for (int k = 0; k < 16; ++k) { gs[k] *= sa; us[k] *= sa; }
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) { gs[k] = 1.0f; us[k] = 1.0f; }
                        }
                        uint32_t w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float h0 = silu_mul(__uint_as_float(g[2 * k]) * gs[2 * k],
                                                      __uint_as_float(u[2 * k]) * us[2 * k]);
                            const float h1 = silu_mul(__uint_as_float(g[2 * k + 1]) * gs[2 * k + 1],
                                                      __uint_as_float(u[2 * k + 1]) * us[2 * k + 1]);
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                            w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        if constexpr (A8) {
                            // magnitudes of finite bf16 values order like their bit patterns
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                hmax_bits = max(hmax_bits, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
                        }
                        uint4* dst = reinterpret_cast<uint4*>(out + c);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                // A8: the row's max |h| over every tile of the row, for its quantiser
                if (A8 && row_ok && hmax_bits != 0) atomicMax(p.hmax[tl.kind] + arow_me, hmax_bits << 16);
            } else if (EPI == EPI_STORE_BF16 || EPI == EPI_COMBINE) {
                bf16* out = (bf16*)p.out[tl.kind] + orow * p.ld_out[tl.kind] + tl.n0;
                const int ncol = tl.half ? BN / 2 : BN;  // tensor-memory columns of this thread's row
                // COMBINE: the routed rows and weights of this row's token (the first 8
                // slots kept in registers for every column chunk)
                constexpr int kCmbSlots = 8;
                int32_t crow[kCmbSlots];
                float cw[kCmbSlots];
                if constexpr (EPI == EPI_COMBINE) {
#pragma unroll
                    for (int q = 0; q < kCmbSlots; ++q) {
                        crow[q] = -1;
                        cw[q] = 0.0f;
                        if (row_ok && q < p.cmb_K) {
                            const int64_t f = (int64_t)arow_me * p.cmb_K + q;
                            const int32_t r = __ldg(p.cmb_inv + f);
                            crow[q] = (r >= 0 && r < p.cmb_rows) ? r : -1;
                            cw[q] = __ldg(p.cmb_w + f);
                        }
                    }
                }
#pragma unroll 1
                for (int tc = 0; tc < ncol; tc += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(tbase + tc, v);
                    const int c = tc + (BN / 2) * hi;  // output column, relative to n0
                    const bool col_ok = tl.n0 + c < nvalid;
                    float ds[16];
                    if constexpr (W8 || A8) tile_scales16(sreg, tc >> 3, ds);
                    ptx::tmem_ld_wait();
                    if (row_ok && col_ok) {
                        if constexpr (W8 || A8) {
                            if constexpr (A8) {
#pragma unroll
                                for (int k = 0; k < 16; ++k) ds[k] *= sa;
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) ds[k] = 1.0f;
                        }
                        uint32_t w[8];
                        if constexpr (EPI == EPI_COMBINE) {
                            // y = y_s + sum_j w_j * y_perm[row_j], in fp32, j ascending
                            float acc[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) acc[k] = __uint_as_float(v[k]);
                            const int64_t ldy = p.ld_out[tl.kind];
                            const int64_t col = tl.n0 + c;
                            for (int j0 = 0; j0 < p.cmb_K; j0 += kCmbSlots) {
                                int32_t rr[kCmbSlots];
                                float ww[kCmbSlots];
#pragma unroll
                                for (int q = 0; q < kCmbSlots; ++q) {
                                    if (j0 == 0) {
                                        rr[q] = crow[q];
                                        ww[q] = cw[q];
                                    } else {
                                        rr[q] = -1;
                                        ww[q] = 0.0f;
                                        if (j0 + q < p.cmb_K) {
                                            const int64_t f = (int64_t)arow_me * p.cmb_K + j0 + q;
                                            const int32_t r = __ldg(p.cmb_inv + f);
                                            rr[q] = (r >= 0 && r < p.cmb_rows) ? r : -1;
                                            ww[q] = __ldg(p.cmb_w + f);
                                        }
                                    }
                                }
                                // every slot's 16 columns requested before any is summed
                                uint4 yv[kCmbSlots][2];
#pragma unroll
                                for (int q = 0; q < kCmbSlots; ++q) {
                                    if (rr[q] >= 0) {
                                        const uint4* src = reinterpret_cast<const uint4*>(
                                            p.cmb_yperm + (int64_t)rr[q] * ldy + col);
                                        yv[q][0] = __ldg(src);
                                        yv[q][1] = __ldg(src + 1);
                                    }
                                }
#pragma unroll
                                for (int q = 0; q < kCmbSlots; ++q) {
                                    if (rr[q] < 0) continue;
                                    const uint32_t u[8] = {yv[q][0].x, yv[q][0].y, yv[q][0].z, yv[q][0].w,
                                                           yv[q][1].x, yv[q][1].y, yv[q][1].z, yv[q][1].w};
#pragma unroll
                                    for (int k = 0; k < 8; ++k) {
                                        const float lo = __uint_as_float(u[k] << 16);
                                        const float hi2 = __uint_as_float(u[k] & 0xFFFF0000u);
                                        acc[2 * k] = fmaf(ww[q], lo, acc[2 * k]);
                                        acc[2 * k + 1] = fmaf(ww[q], hi2, acc[2 * k + 1]);
                                    }
                                }
                            }
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
                                w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                    __uint_as_float(v[2 * k]) * ds[2 * k], __uint_as_float(v[2 * k + 1]) * ds[2 * k + 1]);
                                w[k] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
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
            if (lane == 0) {
                if constexpr (PAIR) ptx::mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
                else ptx::mbar_arrive(&ctl->tempty[acc]);
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    } else {
        if constexpr (W8) {
            // -------------------------------------------- W8 converters (warps 6..9)
            // Per K step: wait for the raw tile (first half) and a free bf16
            // stage; every warp widens its weight rows to bf16, makes the writes
            // visible to the tensor core (async proxy) and arrives on full (a
            // pair: on the even CTA, whose MMA reads both CTAs' stages); after
            // the second half the raw tile is released.
            const int cw = warp - 6;
            const uint32_t full0 = PAIR ? ptx::map_to_rank(&ctl->full[0], 0) : 0u;
            int rs = 0, cs = 0;
            uint32_t rph = 0, cph = 0;
            bool ok = true;
            for (int t = unit; t < n_tiles && ok; t += n_units) {
                const Tile tl = decode_tile<EPI, PAIR, kKStep>(p, list_len, t);
                if (!tl.valid) continue;
                for (int kb = 0; kb < tl.kblocks; ++kb) {
                    const int h = kb & 1;
                    if (h == 0) {
                        const int okr = lane == 0 ? (int)wait_bounded(&ctl->rfull[rs], rph, ctl, p, 400) : 0;
                        if (!__shfl_sync(0xffffffffu, okr, 0)) { ok = false; break; }
                    }
                    const int oke = lane == 0 ? (int)wait_bounded(&ctl->empty[cs], cph ^ 1u, ctl, p, 401) : 0;
                    if (!__shfl_sync(0xffffffffu, oke, 0)) { ok = false; break; }
                    convert_rows_w8<S::kBRows / kW8ConvWarps>(sRaw + rs * W::kRawBytes,
                                                              sB + cs * S::kBBytes, h, cw, lane);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) ptx::mbar_arrive_cluster(full0 + (uint32_t)(cs * sizeof(uint64_t)));
                        else ptx::mbar_arrive(&ctl->full[cs]);
                    }
                    if (++cs == W::kConv) { cs = 0; cph ^= 1u; }
                    if (h == 1 || kb == tl.kblocks - 1) {
                        if (lane == 0) ptx::mbar_arrive(&ctl->rempty[rs]);
                        if (++rs == W::kRaw) { rs = 0; rph ^= 1u; }
                    }
                }
            }
        }
    }

    ptx::tc_fence_before();
    cta_sync_all<PAIR>();  // no role touches the other CTA's memory after this
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, kTmemCols);
        else ptx::tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (PAIR) cta_sync_all<PAIR>();
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

// 2-D map over a row-major [rows][cols] matrix of E4M3 codes with rows ld
// bytes apart (0: cols), box = 128 codes x box_rows rows, 128-byte swizzle
// (cols a multiple of 128, ld a multiple of 16).
bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows,
                 int64_t ld = 0) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (rows <= 0) rows = 1;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld > 0 ? ld : cols)};
    const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
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

// the four activation maps of a matrix of E4M3 codes (rows ld bytes apart)
bool make_amaps_u8(CUtensorMap (&m)[kABoxes], const void* base, int64_t rows, int64_t cols,
                   int64_t ld) {
    bool ok = true;
    for (int b = 0; b < kABoxes; ++b) ok &= make_map_u8(&m[b], base, rows, cols, abox_rows(b), ld);
    return ok;
}

// weight maps: box 128 rows (pair tiles and SWIGLU halves) and box 256 rows
bool make_wmaps(TcParams& p, int k, const void* base, int64_t rows, int64_t cols) {
    return make_map(&p.b0[k], base, rows, cols, 128) && make_map(&p.bw[k], base, rows, cols, 256);
}

// Read on every call (a test shortens it to see a wait run out quickly).
unsigned long long timeout_ns() {
    const char* s = getenv("MOE_TC_TIMEOUT_MS");
    const long long ms = s ? atoll(s) : 1000;
    return (unsigned long long)(ms > 0 ? ms : 1000) * 1000000ull;
}

// Test hook (off unless MOE_TC_TEST_STALL is set to a non-zero value): the
// producer issues no copy, so the MMA's bounded wait runs out and the kernel
// must report MOE_ERR_TIMEOUT and return with the context intact.
int test_stall() {
    const char* s = getenv("MOE_TC_TEST_STALL");
    return (s && atoi(s) != 0) ? 1 : 0;
}

template <bool PAIR, bool SMA = false, int A8 = 0>
constexpr size_t kSmemBytes = 1024 + RingOf<PAIR, SMA, A8>::type::kRingBytes + sizeof(SmemCtl) + 64;
constexpr size_t kSmemBytesW8 = 1024 + kW8RingBytes + sizeof(SmemCtl) + 64;
static_assert(kSmemBytes<true> <= 232448 && kSmemBytes<false> <= 232448 && kSmemBytes<false, true> <= 232448,
              "shared memory exceeds the per-CTA limit");
static_assert(kSmemBytes<true, false, 2> <= 232448 && kSmemBytes<false, false, 2> <= 232448 &&
                  kSmemBytes<false, true, 2> <= 232448,
              "two-plane shared memory exceeds the per-CTA limit");
static_assert(kSmemBytesW8 <= 232448, "W8 shared memory exceeds the per-CTA limit");

// allow_pdl = false: the grid starts only when the previous kernel of the
// stream has finished (so units that take no tile do not hold SMs meanwhile).
template <int EPI, bool PAIR, bool W8 = false, int A8 = 0, bool SMA = false>
cudaError_t launch_tc(const TcParams& p, cudaStream_t st, bool allow_pdl = true) {
    constexpr size_t smem = W8 ? kSmemBytesW8 : kSmemBytes<PAIR, SMA, A8>;
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<EPI, PAIR, W8, A8, SMA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    int units = PAIR ? sms / 2 : sms;
    if (p.dense_rows > 0) {
        const int tiles = (p.dense_rows + Shape<PAIR>::kTileRows - 1) / Shape<PAIR>::kTileRows * p.NB;
        if (tiles < units) units = tiles;
    }
    if (units < 1) units = 1;
    if constexpr (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * units);
        cfg.blockDim = dim3(threads_of<W8, A8>());
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = allow_pdl && pdl_enabled() ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<EPI, PAIR, W8, A8, SMA>, p);
        if (e != cudaSuccess) return e;
    } else if (allow_pdl) {
        e = launch_pdl(tc_gemm_kernel<EPI, PAIR, W8, A8, SMA>, dim3(units),
                       dim3(threads_of<W8, A8>()), smem, st, p);
        if (e != cudaSuccess) return e;
    } else {
        tc_gemm_kernel<EPI, PAIR, W8, A8, SMA><<<units, threads_of<W8, A8>(), smem, st>>>(p);
    }
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

int tc_tile_rows(bool pair) { return pair ? Shape<true>::kTileRows : Shape<false>::kTileRows; }

// Read on every call: MOE_GATHER_MAX_ROWS (0 disables the in-GEMM gather;
// capped at 128, the rows of one CTA's block); unset, kGatherSmallT for a
// batch of at most that many tokens T (a group has at most T rows) and 0 above.
int tc_gather_max_rows(int64_t T) {
    const char* s = getenv("MOE_GATHER_MAX_ROWS");
    const int x = s ? atoi(s) : (T <= kGatherSmallT ? kGatherSmallT : kGatherMaxRows);
    return x < 0 ? 0 : (x > BMC ? BMC : x);
}

// Pair tiles of at most 128 rows (a group's last m-tile) run as M = 128 MMAs
// (MOE_HALF_TILES=0, read per call, keeps them at M = 256).
int half_tiles() {
    const char* s = getenv("MOE_HALF_TILES");
    return (s && s[0] == '0') ? 0 : 1;
}

// m-tiles per band of the CTA-pair tiles (MOE_BAND_PAIR, read per call; 0:
// Shape<true>::kBand = 4).  A band's weight n-blocks are swept once per band,
// so wider bands re-read a large group's weights fewer times (the Zipf
// prefill's hottest expert, 14016 rows, sweeps its weights 14 times at 4 pair
// m-tiles per band); its activation rows (8 x 256 rows x d) stay in L2 across
// the band's n-blocks.  Measured (ABBA, Zipf prefill): expert stage 9.63 ms at
// 4, 9.44 ms at 8, 9.45 ms at 16; Mixtral (one band per expert either way)
// unchanged.
constexpr int kBandPair = 8;
int band_pair() {
    const char* s = getenv("MOE_BAND_PAIR");
    const int x = s ? atoi(s) : kBandPair;
    return x < 0 ? 0 : (x > 64 ? 64 : x);
}

// Single tiles of at most this many rows run swapped (MOE_SWAP_MAX_ROWS, read
// per call; 0 turns it off; capped at 64, the largest swapped N) -- in calls
// where some group can have more rows (max_group_rows > 64, or unknown).  When
// every group is small the GEMMs stream weights, HBM bound, and two narrow
// MMAs per 16-deep slice cost more issue latency than one wide one: measured
// on DeepSeek-V3 decode, expert stage 0.771 ms swapped vs 0.758 ms not, T=64
// 2.810 vs 2.792 ms layer (8-bit activations: W8A8 decode 461 vs 447 us).
// With large groups beside them (skewed prefill) the tail's saved tensor
// energy buys clock under the power cap instead, and for 8-bit tiles, which
// spend two (W8A8) to four (two planes) times the tensor work of a bf16 tile
// on a small group's padding rows, it shortens the tensor work itself: W8A8
// Zipf prefill 6498 -> 6396 us, E4M3-weight T=512 2133 -> 2063 us.
int swap_max_rows(int max_group_rows = 0) {
    if (max_group_rows > 0 && max_group_rows <= kSwapMaxRows) return 0;
    const char* s = getenv("MOE_SWAP_MAX_ROWS");
    const int x = s ? atoi(s) : kSwapMaxRows;
    return x < 0 ? 0 : (x > kSwapMaxRows ? kSwapMaxRows : x);
}

// Groups of at most 32 rows take the small-row ring (MOE_SMALL_RING=0, read
// per call, keeps the full-size one).
bool small_ring() {
    const char* s = getenv("MOE_SMALL_RING");
    return !(s && s[0] == '0');
}

// A second stream and its fork/join events, one set per host thread and
// device, made on first use (not while the caller's stream is being captured:
// that call runs the two tile shapes one after the other instead).  Kept for
// the thread's lifetime, like a library handle.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream(cudaStream_t st) {
    constexpr int kMaxDevices = 64;
    static thread_local SideStream cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream& c = cache[dev];
    if (c.s && c.fork && c.join) return &c;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    if (!c.s && cudaStreamCreateWithFlags(&c.s, cudaStreamNonBlocking) != cudaSuccess) c.s = nullptr;
    if (!c.fork && cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess) c.fork = nullptr;
    if (!c.join && cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess) c.join = nullptr;
    if (c.s && c.fork && c.join) return &c;
    cudaGetLastError();
    return nullptr;
}

// Fork the side stream off st (it waits for everything enqueued on st so far);
// join() makes st wait for everything enqueued on the side stream.
cudaError_t fork_side(SideStream* side, cudaStream_t st) {
    cudaError_t e = cudaEventRecord(side->fork, st);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(side->s, side->fork, 0);
}

cudaError_t join_side(SideStream* side, cudaStream_t st) {
    cudaError_t e = cudaEventRecord(side->join, side->s);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(st, side->join, 0);
}

// Side by side for the 8-bit paths only when MOE_CONCURRENT=1 (read per
// call): measured neutral to 2 % slower there, against neutral to 3 % faster
// for bf16, where it is on unless MOE_CONCURRENT=0.
bool side_by_side(bool eight_bit) {
    if (!eight_bit) return tc_split_rho() > 0;
    const char* c = getenv("MOE_CONCURRENT");
    return c && c[0] == '1';
}

// The streams of the two tile shapes for the GEMMs enqueued while it lives:
// pair tiles on st, single tiles on the side stream (forked off st here and
// joined back by finish() or the destructor) when both shapes may occur and
// side-by-side running is on; otherwise both on st.
struct TwoShapes {
    SideStream* side = nullptr;
    cudaStream_t st, st2;
    TwoShapes(bool may_pair, cudaStream_t s, bool eight_bit) : st(s), st2(s) {
        side = may_pair && side_by_side(eight_bit) ? side_stream(s) : nullptr;
        if (side && fork_side(side, s) != cudaSuccess) {
            cudaGetLastError();
            side = nullptr;
        }
        if (side) st2 = side->s;
    }
    int split() const { return side ? 1 : 0; }
    cudaError_t finish(cudaError_t e) {
        if (side) {
            const cudaError_t j = join_side(side, st);
            side = nullptr;
            if (e == cudaSuccess) e = j;
        }
        return e;
    }
    ~TwoShapes() { finish(cudaSuccess); }
};

// One GEMM over both tile lists; pdl as launch_tc's allow_pdl; small_rows:
// every group has at most kSmaRows rows (single tiles then take the small-row
// ring; not with W8's rings).
template <int EPI, bool W8 = false, int A8 = 0>
cudaError_t launch_shapes(TcParams& p, const int4* pair_list, const int4* single_list, bool may_pair,
                          const TwoShapes& sh, bool pdl, bool small_rows = false) {
    p.split = sh.split();
    cudaError_t e = cudaSuccess;
    if (may_pair) {
        p.mtiles = pair_list;
        p.band = band_pair();
        e = launch_tc<EPI, true, W8, A8>(p, sh.st, pdl);
    }
    if (e == cudaSuccess) {
        p.mtiles = single_list;
        p.band = 0;
        if constexpr (!W8) {
            if (small_rows && small_ring()) return launch_tc<EPI, false, false, A8, true>(p, sh.st2, pdl);
        }
        e = launch_tc<EPI, false, W8, A8>(p, sh.st2, pdl);
    }
    return e;
}

// Groups with at least this many rows take 256-row pair tiles.
// MOE_PAIR_MIN_ROWS > 0 sets a fixed threshold; unset or 0 lets the plan pick
// the cheaper tile shape per group (padding over measured efficiency).
int tc_pair_min_rows() {
    const char* s = getenv("MOE_PAIR_MIN_ROWS");
    const int x = s ? atoi(s) : 0;
    return x < 0 ? 0 : x;
}

// Pair-tile and single-tile GEMMs of one call run side by side on two streams,
// with the SMs split by the plan; the value is the plan's weight-streaming cost
// of a single-tile group in hundredths of an MMA step (MOE_SPLIT_RHO, read per
// call).  MOE_CONCURRENT=0 runs them one after the other on the caller's stream.
int tc_split_rho() {
    const char* c = getenv("MOE_CONCURRENT");
    if (c && c[0] == '0') return 0;
    const char* s = getenv("MOE_SPLIT_RHO");
    const int r = s ? atoi(s) : kSplitRho;
    return r < 1 ? 1 : r;
}

// Some group with at most max_rows rows could take pair tiles.
bool tc_pair_possible(int64_t max_rows) {
    const int pm = tc_pair_min_rows();
    return pm > 0 ? max_rows >= pm : max_rows > Shape<false>::kTileRows;
}

// Batches of at most this many tokens run the shared expert apart
// (MOE_SHARED_APART, read per call).  Off (0) by default: measured on GB300
// (interleaved, 4 x 100 calls each) it is slower -- T=1 197 vs 160 us,
// DeepSeek-V3 decode 806 vs 800 us, T=64 unchanged: the shared expert's SMs
// hold back some units of the persistent routed grid, whose tiles are
// assigned by unit, so the routed GEMM ends later than the routing it hid.
constexpr int kSharedApartMaxT = 0;
int shared_apart_max_tokens() {
    const char* s = getenv("MOE_SHARED_APART");
    const int x = s ? atoi(s) : kSharedApartMaxT;
    return x < 0 ? 0 : (x > Shape<false>::kTileRows ? Shape<false>::kTileRows : x);
}

// The shared expert of a small batch in two dense launches (single-SM tiles,
// swapped for <= 64 rows) on the side stream, forked off st: it reads only x
// and its own weights, so it runs while the router, the dispatch and the
// gather of the routed rows run on st -- on a handful of SMs, streaming its
// weights while HBM would otherwise sit idle behind those latency-bound
// kernels.  The grouped launches then skip the shared group (shared_apart),
// and join_shared_apart() makes st wait for y_s before the combine.  Returns
// false (nothing enqueued) when no side stream can be had (first use inside a
// stream capture): the caller keeps the shared group in the grouped launches.
bool launch_shared_apart(const FfnGroups& g, DevError* err, cudaStream_t st, cudaError_t* status) {
    *status = cudaSuccess;
    if (!g.has_shared || g.T > Shape<false>::kTileRows) return false;
    SideStream* side = side_stream(st);
    if (!side) return false;
    cudaError_t e = fork_side(side, st);
    if (e != cudaSuccess) { *status = e; return true; }
    TcParams p{};
    bool ok = make_amaps(p.a[1], g.a_shared, g.T, g.d);
    ok &= make_map(&p.b0[1], g.ws_gate, g.Is, g.d, 128);
    ok &= make_map(&p.b1[1], g.ws_up, g.Is, g.d, 128);
    TcParams q{};
    ok &= make_amaps(q.a[1], g.h_s, g.T, g.Is);
    ok &= make_wmaps(q, 1, g.ws_down, g.d, g.Is);
    if (!ok) { *status = cudaErrorInvalidValue; return true; }
    for (TcParams* t : {&p, &q}) {
        for (int b = 0; b < kABoxes; ++b) t->a[0][b] = t->a[1][b];
        t->ag = t->a[1][0];
        t->half_tiles = half_tiles();
        t->swap_max_rows = swap_max_rows(g.T);
        t->hdr = nullptr;
        t->mtiles = nullptr;
        t->dense_rows = g.T;
        t->err = err;
        t->timeout_ns = timeout_ns();
        t->test_stall = test_stall();
    }
    // gate/up: h_s = SiLU(x Ws_gate^T) * (x Ws_up^T)
    p.b0[0] = p.b0[1]; p.b1[0] = p.b1[1]; p.bw[0] = p.bw[1] = p.b0[1];
    p.g64[0] = p.g64[1] = p.b0[1]; p.u64[0] = p.u64[1] = p.b1[1];
    p.NB = (g.Is + BN / 2 - 1) / (BN / 2);
    p.n_out[0] = p.n_out[1] = g.Is;
    p.kdim[0] = p.kdim[1] = g.d;
    p.out[0] = p.out[1] = g.h_s;
    p.ld_out[0] = p.ld_out[1] = g.Is;
    // down: y_s = h_s Ws_down^T
    q.b0[0] = q.b0[1]; q.bw[0] = q.bw[1]; q.b1[0] = q.b1[1] = q.b0[1];
    q.NB = (g.d + BN - 1) / BN;
    q.n_out[0] = q.n_out[1] = g.d;
    q.kdim[0] = q.kdim[1] = g.Is;
    q.out[0] = q.out[1] = g.y_s;
    q.ld_out[0] = q.ld_out[1] = g.d;
    e = launch_tc<EPI_SWIGLU, false>(p, side->s);
    if (e == cudaSuccess) e = launch_tc<EPI_STORE_BF16, false>(q, side->s);
    *status = e;
    return true;
}

cudaError_t join_shared_apart(cudaStream_t st) {
    SideStream* side = side_stream(st);
    return side ? join_side(side, st) : cudaErrorInvalidResourceHandle;
}

// The combine fused into the shared expert's down projection (MOE_FUSED_COMBINE=1,
// read per call).  Off by default: measured on GB300 (interleaved A/B, the same
// box) it is slower on every workload -- Zipf prefill 10.97 vs 10.44 ms,
// DeepSeek-V3 T=4096 4.08 vs 3.87 ms, decode 823 vs 800 us, T=1 185 vs 161 us:
// the shared expert's down tiles no longer fill the SMs the routed down tiles
// leave idle, and its launch waits for every routed row, while the combine it
// replaces is a short bandwidth-bound pass.
bool fused_combine_enabled() {
    const char* e = getenv("MOE_FUSED_COMBINE");
    return e && e[0] == '1';
}

cudaError_t launch_ffn_tc(const FfnGroups& g, const FfnPlanHeader* hdr, const int4* mtile_list,
                          int max_mtiles, bool may_pair, DevError* err, cudaStream_t st,
                          const CombineArgs* cmb, bool shared_apart) {
    const int64_t R = g.n_routed_rows;
    const int4* single_list = mtile_list;
    const int4* pair_list = mtile_list + max_mtiles;
    // ---- gate/up: h = SiLU(x W_gate^T) * (x W_up^T)
    TcParams p{};
    bool ok = true;
    if (g.row_src) {
        // small routed row blocks are gathered from x [T][d] by token index,
        // large ones loaded from the permuted copy (present whenever a group
        // can exceed the gather limit)
        ok &= make_map(&p.ag, g.a_routed, g.T, g.d, 1);
        if (g.a_perm) ok &= make_amaps(p.a[0], g.a_perm, R, g.d);
        else ok &= make_amaps(p.a[0], g.a_routed, g.T, g.d);
        p.row_src = g.row_src;
        p.gather_max = tc_gather_max_rows(g.T);
    } else {
        ok &= make_amaps(p.a[0], g.a_routed, R, g.d);
        p.ag = p.a[0][0];
        p.row_src = nullptr;
    }
    ok &= make_map(&p.b0[0], g.w_gate, (int64_t)g.E * g.I, g.d, 128);
    ok &= make_map(&p.b1[0], g.w_up, (int64_t)g.E * g.I, g.d, 128);
    ok &= make_map(&p.g64[0], g.w_gate, (int64_t)g.E * g.I, g.d, 64);
    ok &= make_map(&p.u64[0], g.w_up, (int64_t)g.E * g.I, g.d, 64);
    if (g.has_shared) {
        ok &= make_amaps(p.a[1], g.a_shared, g.T, g.d);
        ok &= make_map(&p.b0[1], g.ws_gate, g.Is, g.d, 128);
        ok &= make_map(&p.b1[1], g.ws_up, g.Is, g.d, 128);
        ok &= make_map(&p.g64[1], g.ws_gate, g.Is, g.d, 64);
        ok &= make_map(&p.u64[1], g.ws_up, g.Is, g.d, 64);
    } else {
        for (int b = 0; b < kABoxes; ++b) p.a[1][b] = p.a[0][b];
        p.b0[1] = p.b0[0]; p.b1[1] = p.b1[0];
        p.g64[1] = p.g64[0]; p.u64[1] = p.u64[0];
    }
    p.half_tiles = half_tiles();
    p.swap_max_rows = swap_max_rows(g.max_group_rows);
    p.skip_shared = shared_apart ? 1 : 0;  // the shared expert runs in its own launches
    p.bw[0] = p.b0[0]; p.bw[1] = p.b0[1];  // unused by the SWIGLU epilogue
    if (!ok) return cudaErrorInvalidValue;
    p.hdr = hdr;
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
    p.test_stall = test_stall();
    // pair tiles on st, single tiles on the side stream, each on its share of
    // the SMs; the down GEMMs follow on the same streams, joined at the end
    TwoShapes sh(may_pair, st, false);
    const bool small = g.max_group_rows > 0 && g.max_group_rows <= kSmaRows;
    cudaError_t e = launch_shapes<EPI_SWIGLU>(p, pair_list, single_list, may_pair, sh, true, small);
    if (e != cudaSuccess) return sh.finish(e);

    // ---- down: y = h W_down^T
    TcParams q{};
    ok = true;
    ok &= make_amaps(q.a[0], g.h, R, g.I);
    ok &= make_wmaps(q, 0, g.w_down, (int64_t)g.E * g.d, g.I);
    if (g.has_shared) {
        ok &= make_amaps(q.a[1], g.h_s, g.T, g.Is);
        ok &= make_wmaps(q, 1, g.ws_down, g.d, g.Is);
    } else {
        for (int b = 0; b < kABoxes; ++b) q.a[1][b] = q.a[0][b];
        q.b0[1] = q.b0[0]; q.bw[1] = q.bw[0];
    }
    q.b1[0] = q.b0[0]; q.b1[1] = q.b0[1];
    if (!ok) return sh.finish(cudaErrorInvalidValue);
    q.half_tiles = half_tiles();
    q.swap_max_rows = swap_max_rows(g.max_group_rows);
    q.hdr = hdr;
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
    q.test_stall = test_stall();
    const bool fuse = cmb != nullptr && g.has_shared && !shared_apart;
    q.skip_shared = (fuse || shared_apart) ? 1 : 0;
    // side by side, the down grids start only when their stream's gate/up grid ended
    e = launch_shapes<EPI_STORE_BF16>(q, pair_list, single_list, may_pair, sh, sh.side == nullptr, small);
    e = sh.finish(e);
    if (!fuse || e != cudaSuccess) return e;

    // ---- shared down + combine: y[t] = h_s[t] Ws_down^T + sum_j w[t][j] y_perm[inv[t*K+j]]
    // (a dense launch over the T token rows, after every routed row is written)
    TcParams r{};
    ok = make_amaps(r.a[1], g.h_s, g.T, g.Is);
    ok &= make_wmaps(r, 1, g.ws_down, g.d, g.Is);
    if (!ok) return cudaErrorInvalidValue;
    for (int b = 0; b < kABoxes; ++b) r.a[0][b] = r.a[1][b];
    r.b0[0] = r.b0[1]; r.bw[0] = r.bw[1]; r.b1[0] = r.b0[1]; r.b1[1] = r.b0[1];
    r.ag = r.a[1][0];
    r.half_tiles = half_tiles();
    r.hdr = nullptr;
    r.mtiles = nullptr;
    r.dense_rows = g.T;
    r.NB = (g.d + BN - 1) / BN;
    r.n_out[0] = r.n_out[1] = g.d;
    r.kdim[0] = r.kdim[1] = g.Is;
    r.wrows[0] = r.wrows[1] = 0;
    r.out[0] = r.out[1] = cmb->y;
    r.ld_out[0] = r.ld_out[1] = g.d;
    r.err = err;
    r.timeout_ns = timeout_ns();
    r.test_stall = test_stall();
    r.cmb_yperm = (const bf16*)g.y;
    r.cmb_inv = cmb->inv_perm;
    r.cmb_w = cmb->topk_w;
    r.cmb_K = cmb->K;
    r.cmb_rows = g.n_routed_rows;
    return g.T > Shape<false>::kTileRows ? launch_tc<EPI_COMBINE, true>(r, st)
                                         : launch_tc<EPI_COMBINE, false>(r, st);
}

// The expert FFN with E4M3 weights: the same two GEMMs on single-SM tiles
// (every plan entry in the single list), routed rows from the permuted copy.
cudaError_t launch_ffn_tc_fp8(const FfnGroups& g, const FfnPlanHeader* hdr, const int4* mtile_list,
                              int max_mtiles, bool may_pair, DevError* err, cudaStream_t st) {
    const int4* single_list = mtile_list;
    const int4* pair_list = mtile_list + max_mtiles;
    const int64_t R = g.n_routed_rows;
    // ---- gate/up: h = SiLU(s_g * (x Q_gate^T)) * (s_u * (x Q_up^T))
    TcParams p{};
    bool ok = true;
    ok &= make_amaps(p.a[0], g.a_perm, R, g.d);
    p.ag = p.a[0][0];
    p.row_src = nullptr;
    p.gather_max = 0;
    ok &= make_map_u8(&p.q0[0], g.w_gate, (int64_t)g.E * g.I, g.d, 128);
    ok &= make_map_u8(&p.q1[0], g.w_up, (int64_t)g.E * g.I, g.d, 128);
    p.sc0[0] = g.s_gate;
    p.sc1[0] = g.s_up;
    if (g.has_shared) {
        ok &= make_amaps(p.a[1], g.a_shared, g.T, g.d);
        ok &= make_map_u8(&p.q0[1], g.ws_gate, g.Is, g.d, 128);
        ok &= make_map_u8(&p.q1[1], g.ws_up, g.Is, g.d, 128);
        p.sc0[1] = g.ss_gate;
        p.sc1[1] = g.ss_up;
    } else {
        for (int b = 0; b < kABoxes; ++b) p.a[1][b] = p.a[0][b];
        p.q0[1] = p.q0[0]; p.q1[1] = p.q1[0];
        p.sc0[1] = p.sc0[0]; p.sc1[1] = p.sc1[0];
    }
    p.qw[0] = p.q0[0]; p.qw[1] = p.q0[1];  // unused by the SWIGLU epilogue
    if (!ok) return cudaErrorInvalidValue;
    p.hdr = hdr;
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
    p.test_stall = test_stall();
    TwoShapes sh(may_pair, st, true);
    cudaError_t e = launch_shapes<EPI_SWIGLU, true>(p, pair_list, single_list, may_pair, sh, true);
    if (e != cudaSuccess) return sh.finish(e);

    // ---- down: y = s_d * (h Q_down^T)
    TcParams q{};
    ok = true;
    ok &= make_amaps(q.a[0], g.h, R, g.I);
    ok &= make_map_u8(&q.qw[0], g.w_down, (int64_t)g.E * g.d, g.I, 256);
    q.sc0[0] = g.s_down;
    if (g.has_shared) {
        ok &= make_amaps(q.a[1], g.h_s, g.T, g.Is);
        ok &= make_map_u8(&q.qw[1], g.ws_down, g.d, g.Is, 256);
        q.sc0[1] = g.ss_down;
    } else {
        for (int b = 0; b < kABoxes; ++b) q.a[1][b] = q.a[0][b];
        q.qw[1] = q.qw[0];
        q.sc0[1] = q.sc0[0];
    }
    q.ag = q.a[0][0];
    // pair tiles load 128 of the n-block's 256 weight rows per CTA (box 128 rows)
    ok &= make_map_u8(&q.q0[0], g.w_down, (int64_t)g.E * g.d, g.I, 128);
    if (g.has_shared) ok &= make_map_u8(&q.q0[1], g.ws_down, g.d, g.Is, 128);
    else q.q0[1] = q.q0[0];
    q.q1[0] = q.q0[0]; q.q1[1] = q.q0[1];
    q.sc1[0] = q.sc0[0]; q.sc1[1] = q.sc0[1];
    if (!ok) return sh.finish(cudaErrorInvalidValue);
    q.hdr = hdr;
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
    q.test_stall = test_stall();
    e = launch_shapes<EPI_STORE_BF16, true>(q, pair_list, single_list, may_pair, sh, sh.side == nullptr);
    return sh.finish(e);
}

// The expert FFN with E4M3 weights AND E4M3 activations (kind::f8f6f4): the
// gate/up GEMM on the quantised rows g.a_perm / g.a_shared (scales
// g.sa_routed / g.sa_shared) writes bf16 h / h_s; the caller quantises those
// in place (codes at the start of each row, 2 * I bytes apart) and runs the
// down GEMM on them (scales g.sa_h / g.sa_hs).  The plan's tiles as in
// launch_ffn_tc: pair tiles (when may_pair) and single-SM tiles.
cudaError_t launch_ffn_tc_a8_gate_up(const FfnGroups& g, const FfnPlanHeader* hdr,
                                     const int4* mtile_list, int max_mtiles, bool may_pair,
                                     DevError* err, cudaStream_t st, int planes) {
    const int64_t R = g.n_routed_rows;
    TcParams p{};
    bool ok = true;
    // activation rows: planes * d codes each (two planes interleaved per 128-code block)
    ok &= make_amaps_u8(p.a[0], g.a_perm, R, planes * g.d, planes * g.d);
    p.ag = p.a[0][0];
    p.row_src = nullptr;
    p.gather_max = 0;
    ok &= make_map_u8(&p.b0[0], g.w_gate, (int64_t)g.E * g.I, g.d, 128);
    ok &= make_map_u8(&p.b1[0], g.w_up, (int64_t)g.E * g.I, g.d, 128);
    ok &= make_map_u8(&p.g64[0], g.w_gate, (int64_t)g.E * g.I, g.d, 64);
    ok &= make_map_u8(&p.u64[0], g.w_up, (int64_t)g.E * g.I, g.d, 64);
    p.half_tiles = half_tiles();
    p.swap_max_rows = g.wblock ? 0 : swap_max_rows(g.max_group_rows);
    p.sc0[0] = g.s_gate;
    p.sc1[0] = g.s_up;
    p.sa[0] = g.sa_routed;
    p.hmax[0] = reinterpret_cast<unsigned int*>(const_cast<float*>(g.sa_h));
    p.hmax[1] = reinterpret_cast<unsigned int*>(const_cast<float*>(g.sa_hs));
    if (g.has_shared) {
        ok &= make_amaps_u8(p.a[1], g.a_shared, g.T, planes * g.d, planes * g.d);
        ok &= make_map_u8(&p.b0[1], g.ws_gate, g.Is, g.d, 128);
        ok &= make_map_u8(&p.b1[1], g.ws_up, g.Is, g.d, 128);
        ok &= make_map_u8(&p.g64[1], g.ws_gate, g.Is, g.d, 64);
        ok &= make_map_u8(&p.u64[1], g.ws_up, g.Is, g.d, 64);
        p.sc0[1] = g.ss_gate;
        p.sc1[1] = g.ss_up;
        p.sa[1] = g.sa_shared;
    } else {
        for (int b = 0; b < kABoxes; ++b) p.a[1][b] = p.a[0][b];
        p.b0[1] = p.b0[0]; p.b1[1] = p.b1[0];
        p.g64[1] = p.g64[0]; p.u64[1] = p.u64[0];
        p.sc0[1] = p.sc0[0]; p.sc1[1] = p.sc1[0];
        p.sa[1] = p.sa[0];
    }
    p.bw[0] = p.b0[0]; p.bw[1] = p.b0[1];  // unused by the SWIGLU epilogue
    if (!ok) return cudaErrorInvalidValue;
    p.hdr = hdr;
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
    p.test_stall = test_stall();
    TwoShapes sh(may_pair, st, true);
    const bool small = g.max_group_rows > 0 && g.max_group_rows <= kSmaRows;
    if (planes == 2 && g.wblock) {  // block-scaled weights: full-height pair tiles only
        p.half_tiles = 0;
        return sh.finish(launch_shapes<EPI_SWIGLU, false, 3>(p, mtile_list + max_mtiles, mtile_list,
                                                             may_pair, sh, true, small));
    }
    if (planes == 2)
        return sh.finish(launch_shapes<EPI_SWIGLU, false, 2>(p, mtile_list + max_mtiles, mtile_list,
                                                             may_pair, sh, true, small));
    if (g.wblock) {  // one plane, block-scaled weights
        p.half_tiles = 0;
        return sh.finish(launch_shapes<EPI_SWIGLU, false, 4>(p, mtile_list + max_mtiles, mtile_list,
                                                             may_pair, sh, true, small));
    }
    return sh.finish(launch_shapes<EPI_SWIGLU, false, 1>(p, mtile_list + max_mtiles, mtile_list,
                                                         may_pair, sh, true, small));
}

cudaError_t launch_ffn_tc_a8_down(const FfnGroups& g, const FfnPlanHeader* hdr,
                                  const int4* mtile_list, int max_mtiles, bool may_pair,
                                  DevError* err, cudaStream_t st, int planes) {
    const int64_t R = g.n_routed_rows;
    TcParams q{};
    bool ok = true;
    // h codes in place: row r at h + r * 2I bytes (I codes, or 2I with two planes)
    ok &= make_amaps_u8(q.a[0], g.h, R, planes * (int64_t)g.I, 2 * (int64_t)g.I);
    ok &= make_map_u8(&q.bw[0], g.w_down, (int64_t)g.E * g.d, g.I, 256);
    ok &= make_map_u8(&q.b0[0], g.w_down, (int64_t)g.E * g.d, g.I, 128);
    q.sc0[0] = g.s_down;
    q.sa[0] = g.sa_h;
    if (g.has_shared) {
        ok &= make_amaps_u8(q.a[1], g.h_s, g.T, planes * (int64_t)g.Is, 2 * (int64_t)g.Is);
        ok &= make_map_u8(&q.bw[1], g.ws_down, g.d, g.Is, 256);
        ok &= make_map_u8(&q.b0[1], g.ws_down, g.d, g.Is, 128);
        q.sc0[1] = g.ss_down;
        q.sa[1] = g.sa_hs;
    } else {
        for (int b = 0; b < kABoxes; ++b) q.a[1][b] = q.a[0][b];
        q.bw[1] = q.bw[0]; q.b0[1] = q.b0[0];
        q.sc0[1] = q.sc0[0];
        q.sa[1] = q.sa[0];
    }
    q.b1[0] = q.b0[0]; q.b1[1] = q.b0[1];
    q.sc1[0] = q.sc0[0]; q.sc1[1] = q.sc0[1];
    q.ag = q.a[0][0];
    q.row_src = nullptr;
    q.half_tiles = half_tiles();
    q.swap_max_rows = g.wblock ? 0 : swap_max_rows(g.max_group_rows);
    if (!ok) return cudaErrorInvalidValue;
    q.hdr = hdr;
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
    q.test_stall = test_stall();
    TwoShapes sh(may_pair, st, true);
    const bool small = g.max_group_rows > 0 && g.max_group_rows <= kSmaRows;
    if (planes == 2 && g.wblock) {
        q.half_tiles = 0;
        return sh.finish(launch_shapes<EPI_STORE_BF16, false, 3>(q, mtile_list + max_mtiles, mtile_list,
                                                                 may_pair, sh, sh.side == nullptr, small));
    }
    if (planes == 2)
        return sh.finish(launch_shapes<EPI_STORE_BF16, false, 2>(q, mtile_list + max_mtiles, mtile_list,
                                                                 may_pair, sh, sh.side == nullptr, small));
    if (g.wblock) {
        q.half_tiles = 0;
        return sh.finish(launch_shapes<EPI_STORE_BF16, false, 4>(q, mtile_list + max_mtiles, mtile_list,
                                                                 may_pair, sh, sh.side == nullptr, small));
    }
    return sh.finish(launch_shapes<EPI_STORE_BF16, false, 1>(q, mtile_list + max_mtiles, mtile_list,
                                                             may_pair, sh, sh.side == nullptr, small));
}

// scores[T][E] (fp32) = x w_g^T on the tensor cores (single tiles)
cudaError_t launch_router_tc(const moe_shape& s, const void* x, const void* w_g, float* scores,
                             DevError* err, cudaStream_t st) {
    TcParams p{};
    bool ok = true;
    ok &= make_amaps(p.a[1], x, s.T, s.d);
    ok &= make_wmaps(p, 1, w_g, s.E, s.d);
    if (!ok) return cudaErrorInvalidValue;
    for (int b = 0; b < kABoxes; ++b) p.a[0][b] = p.a[1][b];
    p.b0[0] = p.b0[1]; p.bw[0] = p.bw[1]; p.b1[0] = p.b0[1]; p.b1[1] = p.b0[1];
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
    p.test_stall = test_stall();
    return launch_tc<EPI_STORE_F32, false>(p, st);
}

}  // namespace moe
