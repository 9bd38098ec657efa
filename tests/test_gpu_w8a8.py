"""8-bit weights and 8-bit activations (W8A8) on the GPU against the oracle.

Both sides quantise the same rows with the same fp32 decisions; x is the
same bf16 input on both, so its codes agree bit for bit.  h is computed by
each side in its own precision (fp32 tensor-core sums, fp64 in the oracle) and
rounded to bf16 before it is quantised, so its codes agree except where the
two h values straddle a bf16 rounding boundary: then one element moves by at
most one E4M3 step, or -- when it is the row's largest magnitude -- the row's
scale moves by one bf16 step (2^-8 relative) and ~3% of the row's codes by one
step, about 1% relative on that row's output.  The bf16 tolerances of the
other layer tests (1e-2 relative L2 overall, 2e-2 per row) cover both.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from tests.gpu_util import BF16_REL_L2, Layer, host, rel_l2, to_f64, pair_min_rows
from tests.test_gpu_fp8 import _check_rows, _clean_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


# ---------------------------------------------------------------- expert stage

def _expert_ffn_case(moe, counts, d, I, seed=0):
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("w8a8_ffn", T=max(rows, 1), d=d, E=E, K=1, I=I, weights="e4m3",
                         acts="e4m3", seed=seed)
    q = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                           "s_down"})
    x_perm = mi.normal((max(rows, 1), d), 1.0, "bf16", "cuda", seed, "x_perm")[:rows]
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    ws = moe.alloc_workspace(s)
    y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_w8a8(s, x_perm, torch.from_numpy(offsets).cuda(),
                            moe.make_fp8_experts(q), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    qh = {k: host(v) for k, v in q.items()}
    ref = oracle.expert_ffn_w8a8(host(x_perm), offsets, qh, dtype="bf16")
    return to_f64(y), ref


@pytest.mark.parametrize("counts,d,I", [
    ([75, 0, 140, 3, 1, 260, 77, 44], 256, 384),     # ragged groups, one empty
    ([600, 257, 1, 129], 384, 640),                  # several m-tiles per group, 5 n-blocks
    ([1, 2, 1, 1, 3, 1, 1, 2], 1024, 256),           # a few rows per expert
    ([16, 15, 1, 33], 7168, 256),                    # DeepSeek-width rows
])
@pytest.mark.parametrize("pair_rows", [0, 100000])
def test_expert_ffn_w8a8_matches_oracle(moe, counts, d, I, pair_rows):
    """pair_rows 0: the plan's cost rule picks CTA-pair or single-SM tiles per
    group; 100000: single-SM tiles only."""
    with pair_min_rows(pair_rows):
        y, ref = _expert_ffn_case(moe, counts, d, I)
    _check_rows(y, ref)


@pytest.mark.parametrize("rho", [None, "1", "1000000"])
def test_expert_ffn_w8a8_side_by_side_changes_no_bit(moe, rho, monkeypatch):
    """Groups on CTA-pair tiles and groups on single-SM tiles: both GEMMs run
    their two tile shapes on two streams at once, on the plan's split of the
    SMs (pushed to both extremes through MOE_SPLIT_RHO), with the same bits as
    one after the other (MOE_CONCURRENT=0)."""
    counts, d, I = [600, 257, 1, 129, 300, 140], 384, 640
    monkeypatch.setenv("MOE_CONCURRENT", "0")
    y0, ref = _expert_ffn_case(moe, counts, d, I, seed=4)
    monkeypatch.setenv("MOE_CONCURRENT", "1")
    if rho is not None:
        monkeypatch.setenv("MOE_SPLIT_RHO", rho)
    y1, _ = _expert_ffn_case(moe, counts, d, I, seed=4)
    assert np.array_equal(y0, y1)
    _check_rows(y0, ref)


# ---------------------------------------------------------------- the layer

@pytest.mark.parametrize("router", ["softmax", "sigmoid"])
def test_forward_w8a8_small_layer_all_tokens(moe, router):
    cfg = mi.LayerConfig("w8a8_small", T=45, d=256, E=12, K=3, I=384, Is=256, router=router,
                         weights="e4m3", acts="e4m3")
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


def test_forward_w8a8_without_shared_expert_and_pair_tiles(moe):
    cfg = mi.LayerConfig("w8a8_noshared", T=600, d=512, E=4, K=2, I=256, weights="e4m3",
                         acts="e4m3")
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


def test_forward_w8a8_differs_from_the_8bit_weight_layer(moe):
    """The activations really are quantised: the W8A8 output moves away from
    the W8A16 output of the same weights by the E4M3 noise of x and h (a few
    percent), far more than the parity tolerance of either path."""
    cfg = mi.LayerConfig("w8a8_vs_a16", T=64, d=512, E=8, K=2, I=512, Is=256, weights="e4m3",
                         acts="e4m3")
    L = Layer(cfg)
    L.x = _clean_x(L)
    y8 = to_f64(L.forward(moe))
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y16 = torch.empty_like(L.x)
    moe.moe_forward_fp8(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y16, ws)
    torch.cuda.synchronize()
    d = rel_l2(y8, to_f64(y16))
    assert 2e-2 < d < 0.2, d


@pytest.mark.parametrize("name", ["mixtral_prefill_w8a8", "dsv3_sweep_w8a8_T512", "dsv3_decode_w8a8"])
def test_forward_w8a8_full_size_sampled_tokens(moe, name):
    """Full-size W8A8 layers: 256 sampled tokens that clear the key gap (every
    token, rows re-drawn, for the 8-token decode batch), their routing and
    their layer outputs."""
    from tests.gpu_util import assert_routing_on_sample, parity_tokens
    cfg = mi.CONFIGS[name]
    L = Layer(cfg)
    tokens, skipped = parity_tokens(L, 256)
    print(f"{name}: {len(tokens)} tokens checked, {skipped} skipped")
    y = L.forward(moe)
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


def test_forward_w8a8_zero_tokens_is_a_no_op(moe):
    cfg = mi.LayerConfig("w8a8_empty", T=4, d=128, E=4, K=2, I=128, weights="e4m3",
                         acts="e4m3")
    L = Layer(cfg)
    s = moe.make_shape(0, 128, 4, 2, 128, 0, "bf16")
    moe.moe_forward_w8a8(s, None, L.p["w_g"], None, moe.make_fp8_experts(L.p), None, None)


def test_forward_w8a8_is_deterministic_graph_capturable_and_pdl_neutral(moe, monkeypatch):
    """Repeated calls give identical bits (the row maxima of h are raised with
    integer atomics, whose order does not matter); the call replays from a CUDA
    graph (its memsets and launches are all stream work); programmatic launch
    off gives the same bits."""
    cfg = mi.CONFIGS["dsv3_sweep_w8a8_T512"]
    L = Layer(cfg)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y1 = L.forward(moe, ws=ws)
    y2 = L.forward(moe, ws=ws)
    assert torch.equal(y1, y2)
    monkeypatch.setenv("MOE_PDL", "0")
    assert torch.equal(L.forward(moe, ws=ws), y1)
    monkeypatch.delenv("MOE_PDL")
    W = moe.make_fp8_experts(L.p)
    y3 = torch.empty_like(y1)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        moe.moe_forward_w8a8(s, L.x, L.p["w_g"], L.bias, W, y3, ws, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    y3.zero_()
    with torch.cuda.graph(g, stream=st):
        moe.moe_forward_w8a8(s, L.x, L.p["w_g"], L.bias, W, y3, ws, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y3, y1)


def test_w8a8_stalled_copy_times_out_and_the_context_survives(moe, monkeypatch):
    """No operand tile is ever requested: the MMA's bounded waits run out, the
    kernel records MOE_ERR_TIMEOUT and returns; the next call is correct."""
    cfg = mi.LayerConfig("w8a8_stall", T=300, d=256, E=4, K=2, I=256, Is=128, weights="e4m3",
                         acts="e4m3")
    L = Layer(cfg)
    monkeypatch.setenv("MOE_TC_TIMEOUT_MS", "50")
    monkeypatch.setenv("MOE_TC_TEST_STALL", "1")
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(L.x)
    moe.moe_forward_w8a8(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_TC_TEST_STALL")
    monkeypatch.delenv("MOE_TC_TIMEOUT_MS")
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    _check_rows(y, L.oracle_tokens(np.arange(cfg.T))["y"])


def test_expert_ffn_w8a8_half_pair_tiles_match_full_pair_tiles(moe, monkeypatch):
    """8-bit operands on pair tiles whose last tile has at most 128 rows: M = 128
    (default) or M = 256 (MOE_HALF_TILES=0); both match the oracle."""
    out = {}
    for half in ("0", "1"):
        monkeypatch.setenv("MOE_HALF_TILES", half)
        with pair_min_rows(1):
            y, ref = _expert_ffn_case(moe, [300, 2, 130, 60, 640], 512, 384)
        _check_rows(y, ref)
        out[half] = y
    assert rel_l2(out["1"], out["0"]) <= 1e-3


@pytest.mark.parametrize("T", [1, 8, 32])
def test_forward_w8a8_small_row_ring_changes_no_bit(moe, T, monkeypatch):
    """Batches of at most 32 tokens run their single-SM kind::f8f6f4 tiles on
    the small-row ring (6 stages of 4 KB activation codes + 32 KB weight
    codes); MOE_SMALL_RING=0 keeps the full-size ring: same bits, and parity
    with the oracle."""
    cfg = mi.LayerConfig(f"w8a8_small_ring_T{T}", T=T, d=1024, E=64, K=8, I=256, Is=256,
                         weights="e4m3", acts="e4m3", seed=33)
    L = Layer(cfg)
    L.x = _clean_x(L)
    monkeypatch.setenv("MOE_SMALL_RING", "0")
    y0 = L.forward(moe)
    monkeypatch.setenv("MOE_SMALL_RING", "1")
    y1 = L.forward(moe)
    assert torch.equal(y0, y1)
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(to_f64(y1), ref["y"])


@pytest.mark.parametrize("swap", ["0", "64"])
def test_swapped_w8a8_tiles_match_the_oracle(moe, swap, monkeypatch):
    """W8A8 tiles of at most MOE_SWAP_MAX_ROWS rows beside larger groups run
    with the operands swapped (one E4M3 plane as N columns); 0 keeps them
    unswapped.  Both against the oracle's W8A8 stage."""
    monkeypatch.setenv("MOE_SWAP_MAX_ROWS", swap)
    y, ref = _expert_ffn_case(moe, [300, 1, 7, 16, 17, 33, 64, 65, 0, 130], 384, 640, seed=7)
    _check_rows(y, ref)
