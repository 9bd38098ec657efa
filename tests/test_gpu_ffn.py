"""Stage 3 on the GPU (moe_expert_ffn): both the weight-streaming GEMV path and the
tcgen05 tensor-core grouped GEMM against the oracle's fp64 SwiGLU experts, on
ragged expert groups (empty experts, one-row experts, groups that are not a
multiple of the 128-row tile, one expert holding most rows)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from tests.gpu_util import BF16_REL_L2, F32_MAX_REL_RMS, gemv_limit, host, max_abs_over_rms, rel_l2, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _counts_to_offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _run(moe, counts, d, I, dtype, limit, seed=0):
    E = len(counts)
    offsets = _counts_to_offsets(counts)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("ffn_case", T=rows, d=d, E=E, K=1, I=I, dtype=dtype, seed=seed)
    p = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down"})
    x_perm = mi.normal((rows, d), 1.0, dtype, "cuda", seed, "x_perm")
    s = moe.make_shape(rows, d, E, 1, I, 0, dtype)
    ws = moe.alloc_workspace(s)
    y = torch.full((rows, d), float("nan"), dtype=x_perm.dtype, device="cuda")
    off_d = torch.from_numpy(offsets).cuda()
    with gemv_limit(limit):
        moe.moe_expert_ffn(s, x_perm, off_d, p["w_gate"], p["w_up"], p["w_down"], y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    ref = oracle.expert_ffn(host(x_perm), offsets, host(p["w_gate"]), host(p["w_up"]),
                            host(p["w_down"]), dtype=dtype)
    return to_f64(y), ref


CASES = [
    # counts per expert, d, I
    ([16, 16, 16, 16, 16, 16, 16, 16], 256, 512),
    ([0, 1, 0, 3, 200, 0, 129, 7], 256, 512),
    ([5, 0, 0, 1], 7168, 2048),
    ([300, 2, 130, 0], 1024, 384),
]


@pytest.mark.parametrize("counts,d,I", CASES)
def test_fp32_streaming_path(moe, counts, d, I):
    y, ref = _run(moe, counts, d, I, "f32", limit=1 << 30)
    assert max_abs_over_rms(y, ref) <= F32_MAX_REL_RMS


@pytest.mark.parametrize("counts,d,I", CASES)
@pytest.mark.parametrize("path,limit", [("gemv", 1 << 30), ("tcgen05", 0), ("mixed", 16)])
def test_bf16_paths(moe, counts, d, I, path, limit):
    y, ref = _run(moe, counts, d, I, "bf16", limit=limit)
    assert np.all(np.isfinite(y))
    assert rel_l2(y, ref) <= BF16_REL_L2
    # every row individually, too (a wrong row cannot hide in the total)
    for r in range(y.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r


def test_tcgen05_large_groups_deepseek_shape(moe):
    """Many 128-row tiles per expert, bands of m-tiles, ragged last tiles."""
    counts = [1100, 0, 257, 640, 1, 128, 0, 900]
    y, ref = _run(moe, counts, 7168, 2048, "bf16", limit=0, seed=3)
    assert rel_l2(y, ref) <= BF16_REL_L2
    worst = max(rel_l2(y[r], ref[r]) for r in range(0, y.shape[0], 7))
    assert worst <= 2 * BF16_REL_L2


def test_paths_agree_closely(moe):
    counts = [40, 3, 0, 77]
    y_g, ref = _run(moe, counts, 512, 256, "bf16", limit=1 << 30)
    y_t, _ = _run(moe, counts, 512, 256, "bf16", limit=0)
    assert rel_l2(y_g, y_t) <= 1e-2
    assert rel_l2(y_t, ref) <= BF16_REL_L2


@pytest.mark.parametrize("counts,d,I", CASES + [([1100, 0, 257, 640, 1, 128, 0, 900], 512, 256)])
@pytest.mark.parametrize("pair_min", [1, 1 << 30])
def test_tensor_core_tile_shapes(moe, counts, d, I, pair_min):
    """Every group on 256-row CTA-pair tiles (pair_min=1) or on 128-row single-SM
    tiles (pair_min huge)."""
    from tests.gpu_util import pair_min_rows
    with pair_min_rows(pair_min):
        y, ref = _run(moe, counts, d, I, "bf16", limit=0, seed=5)
    assert rel_l2(y, ref) <= BF16_REL_L2
    for r in range(y.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r


def test_bounded_wait_reports_timeout_and_the_context_survives(moe, monkeypatch):
    """Failure detection without a fault: a test-only flag makes the tcgen05
    producer issue no copy, so the MMA's wait (limited to 50 ms here) runs out.
    The kernel must record MOE_ERR_TIMEOUT in the workspace error word, free its
    tensor memory and return; the next call on the same context must succeed."""
    counts = [40, 3, 0, 77]
    with gemv_limit(0):
        monkeypatch.setenv("MOE_PAIR_MIN_ROWS", str(1 << 30))  # single-SM tiles only
        monkeypatch.setenv("MOE_TC_TIMEOUT_MS", "50")
        monkeypatch.setenv("MOE_TC_TEST_STALL", "1")
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        rows = int(offsets[-1])
        cfg = mi.LayerConfig("stall", T=rows, d=256, E=4, K=1, I=256)
        p = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down"})
        x_perm = mi.normal((rows, 256), 1.0, "bf16", "cuda", 0, "x_perm")
        s = moe.make_shape(rows, 256, 4, 1, 256, 0, "bf16")
        ws = moe.alloc_workspace(s)
        y = torch.zeros((rows, 256), dtype=torch.bfloat16, device="cuda")
        off_d = torch.from_numpy(offsets).cuda()
        moe.moe_expert_ffn(s, x_perm, off_d, p["w_gate"], p["w_up"], p["w_down"], y, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
        monkeypatch.delenv("MOE_TC_TEST_STALL")
        monkeypatch.delenv("MOE_TC_TIMEOUT_MS")
        y_ok, ref = _run(moe, counts, 256, 256, "bf16", limit=0)
    assert rel_l2(y_ok, ref) <= BF16_REL_L2


@pytest.mark.parametrize("counts,d,I", [([1100, 0, 257, 640, 1, 128, 0, 900], 512, 256),
                                        ([300, 2, 130, 60], 1024, 384)])
def test_half_pair_tiles_match_full_pair_tiles(moe, counts, d, I, monkeypatch):
    """Every group on CTA-pair tiles; a group's last tile with at most 128 rows
    runs as an M = 128 MMA (64 rows per CTA; gate/up weight rows loaded in
    alternating 8-row blocks) or, with MOE_HALF_TILES=0, as a full M = 256 tile.
    Both agree with the oracle and with each other."""
    from tests.gpu_util import pair_min_rows
    out = {}
    for half in ("0", "1"):
        monkeypatch.setenv("MOE_HALF_TILES", half)
        with pair_min_rows(1):
            y, ref = _run(moe, counts, d, I, "bf16", limit=0, seed=9)
        assert rel_l2(y, ref) <= BF16_REL_L2
        for r in range(y.shape[0]):
            assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r
        out[half] = y
    assert rel_l2(out["1"], out["0"]) <= 1e-3


# groups the plan sends to CTA-pair tiles next to groups it sends to single-SM tiles
MIXED = [([1100, 0, 257, 640, 1, 128, 0, 900], 512, 256),
         ([300, 2, 130, 60, 700], 1024, 384)]


@pytest.mark.parametrize("counts,d,I", MIXED)
def test_side_by_side_tile_shapes_change_no_bit(moe, counts, d, I, monkeypatch):
    """The pair-tile and single-tile GEMMs of one call run on two streams at
    once, each grid on the plan's share of the SMs (shares pushed to both
    extremes through MOE_SPLIT_RHO), or one after the other on the caller's
    stream (MOE_CONCURRENT=0).  Every tile is computed the same way whichever
    unit takes it: identical bits, and parity with the oracle."""
    outs = []
    for conc, rho in (("0", None), ("1", None), ("1", "1"), ("1", "1000000")):
        monkeypatch.setenv("MOE_CONCURRENT", conc)
        if rho is None:
            monkeypatch.delenv("MOE_SPLIT_RHO", raising=False)
        else:
            monkeypatch.setenv("MOE_SPLIT_RHO", rho)
        y, ref = _run(moe, counts, d, I, "bf16", limit=0, seed=11)
        outs.append(y)
    assert rel_l2(outs[0], ref) <= BF16_REL_L2
    for r in range(ref.shape[0]):
        assert rel_l2(outs[0][r], ref[r]) <= 2 * BF16_REL_L2, r
    for y in outs[1:]:
        assert np.array_equal(y, outs[0])


def test_side_by_side_tile_shapes_in_a_cuda_graph(moe):
    """The fork onto the second stream and the join back are captured into a
    CUDA graph with the kernels; the replay gives the eager call's bits."""
    counts, d, I = MIXED[0]
    E = len(counts)
    offsets = _counts_to_offsets(counts)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("ffn_graph", T=rows, d=d, E=E, K=1, I=I, seed=3)
    p = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down"})
    x_perm = mi.normal((rows, d), 1.0, "bf16", "cuda", 3, "x_perm")
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    ws = moe.alloc_workspace(s)
    off_d = torch.from_numpy(offsets).cuda()
    y1 = torch.zeros((rows, d), dtype=torch.bfloat16, device="cuda")
    y2 = torch.zeros_like(y1)
    st = torch.cuda.Stream()
    with gemv_limit(0):
        with torch.cuda.stream(st):
            moe.moe_expert_ffn(s, x_perm, off_d, p["w_gate"], p["w_up"], p["w_down"], y1, ws,
                               stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            moe.moe_expert_ffn(s, x_perm, off_d, p["w_gate"], p["w_up"], p["w_down"], y2, ws,
                               stream=st)
        g.replay()
        torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(y1, y2)
    ref = oracle.expert_ffn(host(x_perm), offsets, host(p["w_gate"]), host(p["w_up"]),
                            host(p["w_down"]), dtype="bf16")
    assert rel_l2(to_f64(y1), ref) <= BF16_REL_L2


@pytest.mark.parametrize("counts", [[1, 0, 7, 32, 3], [32, 0], [5, 0, 0, 1]])
def test_small_row_ring_expert_stage(moe, counts, monkeypatch):
    """moe_expert_ffn with at most 32 rows in all takes the small-row ring for
    its single-SM tiles: oracle parity and the full-size ring's bits."""
    monkeypatch.setenv("MOE_SMALL_RING", "0")
    y0, ref = _run(moe, counts, 7168 if len(counts) == 4 else 512, 256, "bf16", limit=0, seed=13)
    monkeypatch.setenv("MOE_SMALL_RING", "1")
    y1, _ = _run(moe, counts, 7168 if len(counts) == 4 else 512, 256, "bf16", limit=0, seed=13)
    assert np.array_equal(y0, y1)
    assert rel_l2(y1, ref) <= BF16_REL_L2
    for r in range(ref.shape[0]):
        assert rel_l2(y1[r], ref[r]) <= 2 * BF16_REL_L2, r


# groups of 1 to 64 rows in every activation box height (16, 32, 64), ragged,
# next to single tiles of more rows and a pair-tile group; d = 1088 and I = 320
# leave partial n-blocks (the last gate/up block has 64 of 128 columns, the
# last down block 64 of 256)
SWAP_COUNTS = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 0, 100, 300]


@pytest.mark.parametrize("swap", ["0", "16", "32", "64"])
def test_swapped_small_tiles(moe, swap, monkeypatch):
    """Single tiles of at most MOE_SWAP_MAX_ROWS rows run with the operands
    swapped (the weight rows as the M = 128 operand, the activation rows as
    N = the box height), their products transposed in tensor memory: every
    setting against the oracle, row by row."""
    monkeypatch.setenv("MOE_SWAP_MAX_ROWS", swap)
    y, ref = _run(moe, SWAP_COUNTS, 1088, 320, "bf16", limit=0, seed=17)
    assert np.all(np.isfinite(y))
    assert rel_l2(y, ref) <= BF16_REL_L2
    for r in range(ref.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r
