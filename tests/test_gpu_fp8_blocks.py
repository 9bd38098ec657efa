"""Block-scaled 8-bit expert weights (one fp32 scale per 128 x 128 block of each
stacked weight matrix) on the GPU against the oracle.

The block quantiser is integer work decided by fp32 arithmetic that both sides
do in the same precision (the block's amax / 448 and w / scale as IEEE fp32
divisions, round to nearest even): codes and scales must match bit for bit.
The expert FFN and the layer are compared like the row-scaled ones: relative
L2 against the fp64 oracle on the same codes and block scales (the exact
8-bit-weight definition), and, where the tensor cores carry the activations as
two E4M3 planes, against the oracle's two-plane form as well.  The W8A8 calls on
block-scaled weights are compared with the oracle's W8A8 layer on the same
codes (x and h quantised per row on both sides)."""
import numpy as np
import pytest
import torch
from dataclasses import replace

import moe_inputs as mi
import oracle
from tests.gpu_util import (BF16_REL_L2, Layer, assert_routing_on_sample, clean_rows, host,
                            parity_tokens, rel_l2, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _check_rows(y, ref, tol=BF16_REL_L2):
    assert rel_l2(y, ref) <= tol
    for r in range(y.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * tol, r


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols", [(600, 2048), (300, 208), (1, 16), (7168, 256), (129, 7168)])
def test_quantize_blocks_bit_exact(moe, dtype, rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    w = (torch.randn(rows, cols, generator=g) * torch.exp2(torch.rand(rows, 1, generator=g) * 16 - 8)
         * torch.exp2(torch.rand(1, cols, generator=g) * 8 - 4))
    if rows >= 128 and cols >= 128:
        w[:128, :128] = 0.0                              # a block of zeros
    w[rows - 1, cols - 1] = -w.abs().max() * 3           # a negative extreme in the corner block
    w = w.to(mi.torch_dtype(dtype))
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.full(((rows + 127) // 128, (cols + 127) // 128), float("nan"),
                        dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_blocks(w.cuda(), codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_blocks(mi.to_host_array(w), dtype)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_blocks_of_a_3d_weight_stack(moe):
    cfg = replace(mi.CONFIGS["dsv3_decode"], E=3, I=256)
    w = mi.make_weights(cfg, "cuda", only={"w_down"})["w_down"]     # [3][7168][256] bf16
    codes = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(3 * 7168 // 128, 256 // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_blocks(w, codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_blocks(host(w), "bf16")
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def test_quantize_blocks_refuses_unsupported_shapes(moe):
    w = torch.zeros(4, 24, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(4, 24, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, 1, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_quantize_fp8_blocks(w, c, s)              # 24 columns: not a multiple of 16
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED


# ---------------------------------------------------------------- expert FFN

def _expert_ffn_case(moe, counts, d, I, seed=0):
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("fp8b_ffn", T=max(rows, 1), d=d, E=E, K=1, I=I, weights="e4m3b", seed=seed)
    q = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                           "s_down"})
    x_perm = mi.normal((max(rows, 1), d), 1.0, "bf16", "cuda", seed, "x_perm")[:rows]
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    ws = moe.alloc_workspace(s)
    y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_fp8_blocks(s, x_perm, torch.from_numpy(offsets).cuda(),
                                  moe.make_fp8_experts(q), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    qh = {k: host(v) for k, v in q.items()}
    ref = oracle.expert_ffn_fp8(host(x_perm), offsets, qh, dtype="bf16", blocks=True)
    ref2 = oracle.expert_ffn_a2(host(x_perm), offsets, qh, dtype="bf16", blocks=True)
    return to_f64(y), ref, ref2


# groups of <= 8 rows on the GEMV and the rest on single-SM tiles (the default);
# every group on the tensor cores, single-SM tiles only or with CTA-pair tiles
PATHS = {"default": {}, "tc": {"MOE_GEMV8_MAX_ROWS": "0"},
         "tc_pair": {"MOE_GEMV8_MAX_ROWS": "0", "MOE_W8_PAIR": "1"}}


@pytest.mark.parametrize("counts,d,I", [
    ([75, 0, 140, 3, 1, 260, 77, 44], 256, 384),     # ragged groups, one empty; GEMV + tiles
    ([600, 257, 1, 129], 384, 640),                  # pair and single tiles, 5 n-blocks
    ([1, 2, 1, 1, 3, 1, 1, 2], 1024, 256),           # decode-like: every group on the GEMV
    ([8, 9, 0, 7, 16, 17], 128, 128),                # around the GEMV limit, one block per matrix
    ([16, 15, 1, 33], 7168, 256),                    # DeepSeek-width rows, 16-row GEMV passes
    ([2, 1, 5, 3], 640, 640),                        # GEMV rows of one whole 512-code step + a tail
    ([300, 1100], 640, 384),                         # n-block halves past the output (d = 5 x 128)
])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_expert_ffn_fp8_blocks_matches_oracle(moe, counts, d, I, path, monkeypatch):
    """Against the exact block-scaled 8-bit-weight stage (fp64, bf16
    activations) and, for tensor-core groups, the oracle's two-plane form,
    which they compute up to fp32 accumulation and the bf16 storage of h and y."""
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    y, ref, ref2 = _expert_ffn_case(moe, counts, d, I)
    _check_rows(y, ref)
    _check_rows(y, ref2)
    if path != "default":   # every row on the two-plane path: closer to its own form (the
        # rest of the gap is the bf16 storage of h and y, ~1e-3 on either side)
        assert rel_l2(y, ref2) < 0.8 * rel_l2(y, ref)


@pytest.mark.parametrize("rho", [None, "1", "1000000"])
def test_expert_ffn_fp8_blocks_side_by_side_changes_no_bit(moe, rho, monkeypatch):
    """Pair-tile and single-tile groups on two streams at once (the SM split
    pushed to both extremes) give the bits of one launch after the other."""
    counts, d, I = [600, 257, 1, 129, 300, 140], 384, 640
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", "0")
    monkeypatch.setenv("MOE_W8_PAIR", "1")
    monkeypatch.setenv("MOE_CONCURRENT", "0")
    y0, ref, _ = _expert_ffn_case(moe, counts, d, I, seed=4)
    monkeypatch.setenv("MOE_CONCURRENT", "1")
    if rho is not None:
        monkeypatch.setenv("MOE_SPLIT_RHO", rho)
    y1, _, _ = _expert_ffn_case(moe, counts, d, I, seed=4)
    assert np.array_equal(y0, y1)
    assert rel_l2(y0, ref) <= BF16_REL_L2


def test_blocks_with_one_scale_per_row_block_match_the_row_scaled_path(moe, monkeypatch):
    """Block scales equal along each block row describe the same weights as row
    scales repeated over the block's 128 rows: both GPU paths (block-scaled and
    row-scaled, each on the GEMV and on the tensor cores) agree to accumulation
    order."""
    counts, d, I = [3, 200, 7, 90], 512, 384
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("fp8b_rows", T=rows, d=d, E=E, K=1, I=I, weights="e4m3b", seed=9)
    qb = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                            "s_down"})
    qr = dict(qb)
    for sn, w in (("s_gate", "w_gate"), ("s_up", "w_up"), ("s_down", "w_down")):
        col0 = qb[sn][:, :1].contiguous()                          # [rows/128, 1]
        qb[sn] = col0.expand_as(qb[sn]).contiguous()
        qr[sn] = col0.repeat_interleave(128, 0).reshape(qb[w].shape[:-1]).contiguous()
    x_perm = mi.normal((rows, d), 1.0, "bf16", "cuda", 9, "x_perm")
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    off = torch.from_numpy(offsets).cuda()
    for gemv8 in ("8", "0"):
        monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", gemv8)
        yb = torch.empty(rows, d, dtype=torch.bfloat16, device="cuda")
        yr = torch.empty_like(yb)
        ws = moe.alloc_workspace(s)
        moe.moe_expert_ffn_fp8_blocks(s, x_perm, off, moe.make_fp8_experts(qb), yb, ws)
        moe.moe_expert_ffn_fp8(s, x_perm, off, moe.make_fp8_experts(qr), yr, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
        assert rel_l2(to_f64(yb), to_f64(yr)) < 2e-3, gemv8


# ---------------------------------------------------------------- the layer

@pytest.mark.parametrize("router", ["softmax", "sigmoid"])
@pytest.mark.parametrize("gemv8", ["0", "8", "16", "40"])
def test_forward_fp8_blocks_small_layer_all_tokens(moe, router, gemv8, monkeypatch):
    """Groups of ~11 rows and a 45-row shared group: all on the tensor cores
    (limit 0), part of the routed groups on the 8-bit GEMV (8, the default),
    every routed group in one 16-row pass (16), or everything including the
    shared group in passes of 16 rows (40)."""
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", gemv8)
    cfg = mi.LayerConfig("fp8b_small", T=45, d=256, E=12, K=3, I=384, Is=256, router=router,
                         weights="e4m3b")
    L = Layer(cfg)
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


@pytest.mark.parametrize("gemv8", ["0", "8"])
def test_forward_fp8_blocks_decode_full_size(moe, gemv8, monkeypatch):
    """DeepSeek-V3 decode shapes with block-scaled weights: every group on the
    8-bit GEMV (default) or on the tensor cores (limit 0); routing checked too."""
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", gemv8)
    cfg = mi.CONFIGS["dsv3_decode_fp8b"]
    L = Layer(cfg)
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    tokens = np.arange(cfg.T)
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(y, ref["y"])


@pytest.mark.parametrize("name,pair", [("mixtral_prefill_fp8b", "0"), ("mixtral_prefill_fp8b", "1"),
                                       ("dsv3_sweep_fp8b_T512", "0")])
def test_forward_fp8_blocks_sampled_tokens(moe, name, pair, monkeypatch):
    """Mixtral-shaped prefill (~1024-row groups on single-SM tiles, or CTA-pair
    tiles with MOE_W8_PAIR=1) and the DeepSeek-V3 shape at T = 512 (~16-row
    groups): 256 sampled tokens whose routing clears the order margin, routing
    and outputs against the oracle."""
    monkeypatch.setenv("MOE_W8_PAIR", pair)
    cfg = mi.CONFIGS[name]
    L = Layer(cfg)
    y = L.forward(moe)
    tokens, skipped = parity_tokens(L, 256)
    print(f"{cfg.name}: {len(tokens)} sampled tokens checked, {skipped} skipped")
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


def test_forward_fp8_blocks_is_graph_capturable(moe):
    cfg = mi.LayerConfig("fp8b_graph", T=200, d=256, E=8, K=2, I=256, Is=128, weights="e4m3b")
    L = Layer(cfg)
    L.x = clean_rows(L)
    y0 = L.forward(moe)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(L.x)
    W = moe.make_fp8_experts(L.p)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        moe.moe_forward_fp8_blocks(s, L.x, L.p["w_g"], L.bias, W, y, ws, stream=stream)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
        assert torch.equal(y, y0)


def test_forward_fp8_blocks_zero_tokens_is_a_no_op(moe):
    cfg = mi.LayerConfig("fp8b_empty", T=4, d=128, E=4, K=2, I=128, weights="e4m3b")
    L = Layer(cfg)
    s = moe.make_shape(0, 128, 4, 2, 128, 0, "bf16")
    moe.moe_forward_fp8_blocks(s, None, L.p["w_g"], None, moe.make_fp8_experts(L.p), None, None)


def test_fp8_blocks_stalled_copy_times_out_and_the_context_survives(moe, monkeypatch):
    """No tile is ever requested: the MMA's bounded wait runs out, every
    epilogue warp leaves its per-block waits, the kernel records
    MOE_ERR_TIMEOUT and returns; the next call is correct."""
    cfg = mi.LayerConfig("fp8b_stall", T=64, d=256, E=4, K=2, I=256, Is=128, weights="e4m3b")
    L = Layer(cfg)
    monkeypatch.setenv("MOE_TC_TIMEOUT_MS", "50")
    monkeypatch.setenv("MOE_TC_TEST_STALL", "1")
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(L.x)
    moe.moe_forward_fp8_blocks(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_TC_TEST_STALL")
    monkeypatch.delenv("MOE_TC_TIMEOUT_MS")
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    _check_rows(y, L.oracle_tokens(np.arange(cfg.T))["y"])


# ---------------------------------------------------------------- W8A8 on block-scaled weights

def _w8a8_case(moe, counts, d, I, seed=0):
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("w8a8b_ffn", T=max(rows, 1), d=d, E=E, K=1, I=I, weights="e4m3b",
                         acts="e4m3", seed=seed)
    q = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                           "s_down"})
    x_perm = mi.normal((max(rows, 1), d), 1.0, "bf16", "cuda", seed, "x_perm")[:rows]
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    ws = moe.alloc_workspace(s)
    y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_w8a8_blocks(s, x_perm, torch.from_numpy(offsets).cuda(),
                                   moe.make_fp8_experts(q), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    qh = {k: host(v) for k, v in q.items()}
    ref = oracle.expert_ffn_w8a8(host(x_perm), offsets, qh, dtype="bf16", blocks=True)
    return to_f64(y), ref


@pytest.mark.parametrize("counts,d,I", [
    ([75, 0, 140, 3, 1, 260, 77, 44], 256, 384),     # ragged groups, one empty
    ([600, 257, 1, 129], 384, 640),                  # several m-tiles per group, 5 n-blocks
    ([1, 2, 1, 1, 3, 1, 1, 2], 1024, 256),           # a few rows per expert (small-row ring)
    ([16, 15, 1, 33], 7168, 256),                    # DeepSeek-width rows
    ([300, 1100], 640, 384),                         # n-block halves past the output
])
@pytest.mark.parametrize("pair", ["0", "1"])
def test_expert_ffn_w8a8_blocks_matches_oracle(moe, counts, d, I, pair, monkeypatch):
    """Single-SM tiles (the default for block scales) or CTA-pair tiles too
    (MOE_W8_PAIR=1), against the oracle's W8A8 stage on the same block-scaled
    codes (x and h quantised per row on both sides)."""
    monkeypatch.setenv("MOE_W8_PAIR", pair)
    y, ref = _w8a8_case(moe, counts, d, I)
    _check_rows(y, ref)


@pytest.mark.parametrize("router", ["softmax", "sigmoid"])
def test_forward_w8a8_blocks_small_layer_all_tokens(moe, router):
    cfg = mi.LayerConfig("w8a8b_small", T=45, d=256, E=12, K=3, I=384, Is=256, router=router,
                         weights="e4m3b", acts="e4m3")
    L = Layer(cfg)
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


def test_forward_w8a8_blocks_decode_full_size(moe):
    """DeepSeek-V3 decode shapes (every group of <= 8 rows on the small-row
    ring), routing checked too."""
    cfg = mi.CONFIGS["dsv3_decode_w8a8b"]
    L = Layer(cfg)
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    tokens = np.arange(cfg.T)
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(y, ref["y"])


def test_forward_w8a8_blocks_prefill_sampled_tokens(moe):
    cfg = mi.CONFIGS["mixtral_prefill_w8a8b"]
    L = Layer(cfg)
    y = L.forward(moe)
    tokens, skipped = parity_tokens(L, 256)
    print(f"{cfg.name}: {len(tokens)} sampled tokens checked, {skipped} skipped")
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


def test_w8a8_blocks_stalled_copy_times_out_and_the_context_survives(moe, monkeypatch):
    cfg = mi.LayerConfig("w8a8b_stall", T=64, d=256, E=4, K=2, I=256, Is=128, weights="e4m3b",
                         acts="e4m3")
    L = Layer(cfg)
    monkeypatch.setenv("MOE_TC_TIMEOUT_MS", "50")
    monkeypatch.setenv("MOE_TC_TEST_STALL", "1")
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(L.x)
    moe.moe_forward_w8a8_blocks(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_TC_TEST_STALL")
    monkeypatch.delenv("MOE_TC_TIMEOUT_MS")
    L.x = clean_rows(L)
    y = to_f64(L.forward(moe))
    _check_rows(y, L.oracle_tokens(np.arange(cfg.T))["y"])
