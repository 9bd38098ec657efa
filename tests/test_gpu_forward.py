"""The whole layer on the GPU (moe_forward) against the oracle, on every workload:
all tokens where the oracle finishes in seconds, a seeded sample of 256 tokens
on the large ones.  A token whose fp64 keys leave a gap below 1e-3 among its K
picks or at the top-K boundary has no unique routing at fp32 precision: the
sampler skips it and draws on until 256 tokens clear the gap (the skip count
is printed), and the small workloads re-draw such rows instead.  On the sample
the library's routing (expert ids in slot order, weights) must equal the
oracle's as well as the layer output."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from tests.gpu_util import (BF16_REL_L2, F32_MAX_REL_RMS, MARGIN, Layer,
                            assert_routing_on_sample, boundary_margin, clean_rows, clean_sample,
                            gemv_limit, host, max_abs_over_rms, rel_l2, to_f64)

pytestmark = pytest.mark.gpu

SAMPLE = 256


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _clean_x(L: Layer):
    return clean_rows(L)


def _check(cfg, y, ref):
    if cfg.dtype == "f32":
        assert max_abs_over_rms(y, ref) <= F32_MAX_REL_RMS
    else:
        assert rel_l2(y, ref) <= BF16_REL_L2
        for r in range(y.shape[0]):
            assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r


@pytest.mark.parametrize("name", ["tiny_f32", "dsv3_decode", "dsv3_sweep_T1", "dsv3_sweep_T8",
                                  "dsv3_sweep_T64"])
def test_forward_all_tokens(moe, name):
    cfg = mi.CONFIGS[name]
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype, bias=L.bias_host())
    assert_routing_on_sample(moe, L, np.arange(cfg.T), ref)
    _check(cfg, y, ref["y"])


@pytest.mark.parametrize("d,I", [(16384, 128), (128, 16384)])
@pytest.mark.parametrize("kind", ["f32", "bf16", "fp8", "w8a8"])
def test_forward_at_the_widest_rows(moe, d, I, kind):
    """d and I (and Is) at their limit, 16384: the widest rows every kernel
    stages -- the fp32 GEMV's shared-memory rows, the 8-bit GEMV's fit check
    (rows this wide go to the tcgen05 path), the per-row activation quantiser
    holding a whole row in registers, the in-place h quantiser -- with a
    160-row shared group on CTA-pair tiles next to routed groups on single
    tiles.  All tokens against the oracle."""
    cfg = mi.LayerConfig(f"wide_{kind}", T=160, d=d, E=4, K=2, I=I, Is=I,
                         dtype="f32" if kind == "f32" else "bf16",
                         weights="e4m3" if kind in ("fp8", "w8a8") else "act",
                         acts="e4m3" if kind == "w8a8" else "act", seed=21)
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check(cfg, y, ref["y"])


@pytest.mark.parametrize("name", ["mixtral_prefill", "dsv3_prefill_zipf", "dsv3_sweep_T512",
                                  "dsv3_sweep_T4096"])
def test_forward_sampled_tokens(moe, name):
    """Full-size workloads: 256 sampled tokens that clear the key gap, their
    routing (ordered expert ids, weights) and their layer outputs."""
    cfg = mi.CONFIGS[name]
    L = Layer(cfg)
    y = L.forward(moe)
    tokens, skipped = clean_sample(L, SAMPLE)
    print(f"{name}: {SAMPLE} sampled tokens checked, {skipped} skipped (key gap < {MARGIN})")
    assert len(tokens) == SAMPLE
    ref = oracle.forward_tokens(tokens, host(L.x), L.hp, cfg.K, dtype=cfg.dtype,
                                bias=L.bias_host())
    err = assert_routing_on_sample(moe, L, tokens, ref)
    print(f"{name}: routing equal on the sample, max |score error| {err:.2e}")
    _check(cfg, to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


def test_forward_small_ragged_shapes_both_paths(moe):
    """Shapes off the workload grid: E=12, K=3, d=192, I=320, Is=128, T=37 (ragged
    tiles everywhere), through the GEMV path and the tensor-core path."""
    cfg = mi.LayerConfig("ragged", T=37, d=192, E=12, K=3, I=320, Is=128)
    L = Layer(cfg)
    L.x = _clean_x(L)
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype)["y"]
    for limit in (1 << 30, 0, 4):
        with gemv_limit(limit):
            y = to_f64(L.forward(moe))
        _check(cfg, y, ref)


def test_forward_K_equals_E_and_single_expert(moe):
    for cfg in (mi.LayerConfig("k_eq_e", T=20, d=128, E=4, K=4, I=128, Is=64),
                mi.LayerConfig("dense", T=300, d=256, E=1, K=1, I=192, Is=0)):
        L = Layer(cfg)
        ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype)["y"]
        _check(cfg, to_f64(L.forward(moe)), ref)


def test_forward_zero_input_and_zero_tokens(moe):
    cfg = mi.LayerConfig("zeros", T=16, d=128, E=8, K=2, I=128, Is=64)
    L = Layer(cfg)
    y = L.forward(moe, x=torch.zeros_like(L.x))
    assert torch.count_nonzero(y).item() == 0
    y0 = L.forward(moe, x=L.x[:0])
    assert y0.shape == (0, cfg.d)


def test_forward_is_deterministic_and_graph_capturable(moe):
    cfg = mi.CONFIGS["dsv3_sweep_T64"]
    L = Layer(cfg)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y1 = L.forward(moe, ws=ws)
    y2 = L.forward(moe, ws=ws)
    assert torch.equal(y1, y2)
    p = L.p
    y3 = torch.empty_like(y1)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        # the first call outside capture sets kernel attributes
        moe.moe_forward(s, L.x, p["w_g"], None, p["w_gate"], p["w_up"], p["w_down"],
                        p["ws_gate"], p["ws_up"], p["ws_down"], y3, ws, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    y3.zero_()
    with torch.cuda.graph(g, stream=st):
        moe.moe_forward(s, L.x, p["w_g"], None, p["w_gate"], p["w_up"], p["w_down"],
                        p["ws_gate"], p["ws_up"], p["ws_down"], y3, ws, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y3, y1)


@pytest.mark.parametrize("name", ["dsv3_decode", "mixtral_prefill", "dsv3_decode_fp8", "tiny_f32"])
def test_programmatic_dependent_launch_changes_no_bit(moe, name, monkeypatch):
    """Every kernel orders itself after its predecessor with griddepcontrol.wait;
    the same call with programmatic launch off (MOE_PDL=0) gives identical bits,
    back to back on one stream (repeated calls overlap only their launch)."""
    cfg = mi.CONFIGS[name]
    L = Layer(cfg)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    monkeypatch.setenv("MOE_PDL", "0")
    ref = L.forward(moe, ws=ws)
    monkeypatch.setenv("MOE_PDL", "1")
    outs = [torch.empty_like(ref) for _ in range(3)]
    for y in outs:  # three calls in a row, no host synchronisation in between
        if cfg.weights == "e4m3":
            moe.moe_forward_fp8(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y, ws)
        else:
            p = L.p
            moe.moe_forward(s, L.x, p["w_g"], L.bias, p["w_gate"], p["w_up"], p["w_down"],
                            p.get("ws_gate"), p.get("ws_up"), p.get("ws_down"), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    for y in outs:
        assert torch.equal(y, ref)


def test_combine_matches_oracle(moe):
    for dtype in ("f32", "bf16"):
        T, d, K = 50, 256, 3
        rng = np.random.default_rng(4)
        yp = mi.normal((T * K, d), 1.0, dtype, "cuda", 1, "yp")
        ys = mi.normal((T, d), 1.0, dtype, "cuda", 1, "ys")
        inv = torch.from_numpy(rng.permutation(T * K).astype(np.int32)).cuda()
        w = torch.from_numpy(rng.random((T, K)).astype(np.float32)).cuda()
        s = moe.make_shape(T, d, 8, K, 64, 0, dtype)
        y = torch.empty_like(ys)
        moe.moe_combine(s, yp, inv, w, ys, y)
        torch.cuda.synchronize()
        ref = oracle.combine(to_f64(yp), inv.cpu().numpy(), w.cpu().numpy().astype(np.float64),
                             to_f64(ys))
        if dtype == "f32":
            assert max_abs_over_rms(to_f64(y), ref) <= 1e-6
        else:
            assert rel_l2(to_f64(y), ref) <= 4e-3


@pytest.mark.parametrize("name,T", [("dsv3_decode", None), ("dsv3_sweep_T4096", None)])
def test_forward_sigmoid_router(moe, name, T):
    """The whole layer with the DeepSeek-V3 router (sigmoid affinities, a
    selection-only bias, weights a / (sum a + 1e-6))."""
    import dataclasses
    cfg = dataclasses.replace(mi.CONFIGS[name], router="sigmoid")
    L = Layer(cfg)
    L.bias = (torch.from_numpy(np.round(np.random.default_rng(9).standard_normal(cfg.E) * 4) / 64)
              .float().cuda())
    if cfg.T <= SAMPLE:
        L.x = _clean_x(L)
        tokens, skipped = np.arange(cfg.T, dtype=np.int32), 0
    else:
        tokens, skipped = clean_sample(L, SAMPLE)
    y = L.forward(moe)
    print(f"{name} (sigmoid): {len(tokens)} tokens checked, {skipped} skipped (key gap < 1e-4)")
    assert len(tokens) == min(SAMPLE, cfg.T)
    ref = oracle.forward_tokens(tokens, host(L.x), L.hp, cfg.K, dtype=cfg.dtype,
                                bias=L.bias_host(), router="sigmoid")
    assert_routing_on_sample(moe, L, tokens, ref)
    _check(cfg, to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


@pytest.mark.parametrize("gather_max,swap", [(0, 64), (0, 0), (32, 64), (128, 64)])
def test_forward_skewed_groups_cover_every_activation_path(moe, monkeypatch, gather_max, swap):
    """Expert groups from a few rows to >1000 rows in one call, on single-SM and
    CTA-pair tiles (pair remainders included), small single tiles swapped or
    not; with the in-GEMM gather enabled, row blocks of <= gather_max rows come
    straight from x (tile::gather4) and larger ones from the permuted copy."""
    monkeypatch.setenv("MOE_GATHER_MAX_ROWS", str(gather_max))
    monkeypatch.setenv("MOE_SWAP_MAX_ROWS", str(swap))
    cfg = mi.LayerConfig("skewed", T=2048, d=256, E=16, K=2, I=256, Is=128, seed=4)
    L = Layer(cfg)
    L.bias = (torch.linspace(2.5, -2.5, cfg.E)).float().cuda()   # expert 0 hot, 15 cold
    L.x = _clean_x(L)
    _, _, keys = oracle.route(host(L.x), L.hp["w_g"], cfg.K, dtype=cfg.dtype, bias=L.bias_host())
    counts = np.bincount(np.argsort(-keys, axis=1, kind="stable")[:, :cfg.K].ravel(),
                         minlength=cfg.E)
    assert counts.max() >= 512 and counts.min() <= 32 and ((counts > 32) & (counts < 512)).any()
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype, bias=L.bias_host())["y"]
    _check(cfg, to_f64(L.forward(moe)), ref)


@pytest.mark.parametrize("name", ["dsv3_decode", "dsv3_sweep_T64", "dsv3_decode_fp8", "tiny_f32",
                                  "w8a8_T64"])
def test_fused_small_dispatch_changes_no_bit(moe, name, monkeypatch):
    """Small batches (T*K <= 1024) run the dispatch and the expert plan as one
    single-block launch; the separate kernels (MOE_FUSED_DISPATCH=0) give the
    same bits."""
    from dataclasses import replace
    cfg = (replace(mi.CONFIGS["dsv3_sweep_fp8_T64"], name="w8a8_T64", acts="e4m3")
           if name == "w8a8_T64" else mi.CONFIGS[name])
    assert cfg.T * cfg.K <= 1024
    L = Layer(cfg)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    monkeypatch.setenv("MOE_FUSED_DISPATCH", "0")
    ref = L.forward(moe, ws=ws)
    monkeypatch.setenv("MOE_FUSED_DISPATCH", "1")
    out = L.forward(moe, ws=ws)
    assert torch.equal(out, ref)


def test_fused_small_dispatch_at_its_limits(moe, monkeypatch):
    """The largest fused case: 1024 slots over 1024 experts (the block's
    per-warp table is 128 KB of shared memory), with a shared expert; the
    outputs match the four-launch path bit for bit and the oracle."""
    cfg = mi.LayerConfig("fused_limits", T=256, d=128, E=1024, K=4, I=128, Is=128)
    L = Layer(cfg)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    monkeypatch.setenv("MOE_FUSED_DISPATCH", "0")
    ref = L.forward(moe, ws=ws)
    monkeypatch.setenv("MOE_FUSED_DISPATCH", "1")
    out = L.forward(moe, ws=ws)
    assert torch.equal(out, ref)
    toks = np.arange(0, cfg.T, 8)
    want = L.oracle_tokens(toks)
    ok = boundary_margin(want["logits"], cfg.K) >= MARGIN
    got = to_f64(out[torch.from_numpy(toks[ok]).long().cuda()])
    assert rel_l2(got, want["y"][ok]) <= BF16_REL_L2


@pytest.mark.parametrize("T", [1, 8, 32, 33])
def test_small_row_ring_changes_no_bit(moe, T, monkeypatch):
    """Batches of at most 32 tokens run their single-SM tiles on the small-row
    ring (6 weight stages of 4 KB activations + 32 KB weights instead of 4 of
    16 + 32 KB); MOE_SMALL_RING=0 keeps the full-size ring.  Same bits, and
    parity with the oracle (T = 33 is past the bound and takes the full ring
    either way)."""
    cfg = mi.LayerConfig(f"small_ring_T{T}", T=T, d=1024, E=64, K=8, I=256, Is=256, seed=31)
    L = Layer(cfg)
    L.x = _clean_x(L)
    monkeypatch.setenv("MOE_SMALL_RING", "0")
    y0 = L.forward(moe)
    monkeypatch.setenv("MOE_SMALL_RING", "1")
    y1 = L.forward(moe)
    assert torch.equal(y0, y1)
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype, bias=L.bias_host())
    _check(cfg, to_f64(y1), ref["y"])


@pytest.mark.parametrize("T,K", [(8, 4), (300, 10), (1030, 4)])
def test_fused_combine(moe, T, K, monkeypatch):
    """With a shared expert the combine runs in the epilogue of the shared
    expert's down projection (one dense launch after the routed down GEMMs:
    single tiles at T = 8, pair tiles with a 6-row half tile at T = 1030; K = 10
    takes the slot loop past its first 8 slots).  Both ways against the oracle,
    and within bf16 rounding of each other (the separate combine adds the shared
    term after rounding it to bf16; the fused one adds its fp32 sum)."""
    cfg = mi.LayerConfig(f"fused_combine_T{T}", T=T, d=512, E=16, K=K, I=256, Is=384, seed=29)
    L = Layer(cfg)
    L.x = _clean_x(L)
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype, bias=L.bias_host())["y"]
    monkeypatch.setenv("MOE_FUSED_COMBINE", "0")
    y0 = to_f64(L.forward(moe))
    monkeypatch.setenv("MOE_FUSED_COMBINE", "1")
    y1 = to_f64(L.forward(moe))
    _check(cfg, y0, ref)
    _check(cfg, y1, ref)
    assert rel_l2(y1, y0) <= 4e-3


@pytest.mark.parametrize("T", [1, 8, 33, 64])
def test_shared_expert_apart_changes_no_bit(moe, T, monkeypatch):
    """Batches of at most 64 tokens run the shared expert in two launches of its
    own on a side stream, beside the routing and dispatch; MOE_SHARED_APART=0
    keeps it in the grouped launches.  Each of its tiles is computed the same
    way either way: identical bits, eager and replayed from a CUDA graph, and
    parity with the oracle."""
    cfg = mi.LayerConfig(f"apart_T{T}", T=T, d=1024, E=64, K=8, I=256, Is=384, seed=37)
    L = Layer(cfg)
    L.x = _clean_x(L)
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    monkeypatch.setenv("MOE_SHARED_APART", "0")
    y0 = L.forward(moe, ws=ws)
    monkeypatch.setenv("MOE_SHARED_APART", "64")
    y1 = L.forward(moe, ws=ws)
    assert torch.equal(y0, y1)
    p = L.p
    y2 = torch.zeros_like(y1)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=st):
        moe.moe_forward(s, L.x, p["w_g"], None, p["w_gate"], p["w_up"], p["w_down"],
                        p["ws_gate"], p["ws_up"], p["ws_down"], y2, ws, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    assert torch.equal(y2, y1)
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype)["y"]
    _check(cfg, to_f64(y1), ref)


@pytest.mark.parametrize("T", [1, 8, 16, 17])
def test_small_batches_gather_inside_the_gemm_with_the_same_bits(moe, T, monkeypatch):
    """Batches of at most 16 tokens load their routed rows straight from x inside
    the GEMM (tile::gather4 through the row -> token map) and make no permuted
    copy; MOE_GATHER_MAX_ROWS=0 forces the copy.  The MMA sees the same rows:
    identical bits, and parity with the oracle (T = 17 takes the copy by
    default)."""
    cfg = mi.LayerConfig(f"gather_T{T}", T=T, d=1024, E=64, K=8, I=256, Is=256, seed=41)
    L = Layer(cfg)
    L.x = _clean_x(L)
    monkeypatch.setenv("MOE_GATHER_MAX_ROWS", "0")
    y0 = L.forward(moe)
    monkeypatch.delenv("MOE_GATHER_MAX_ROWS")
    y1 = L.forward(moe)
    assert torch.equal(y0, y1)
    ref = oracle.forward(host(L.x), L.hp, cfg.K, dtype=cfg.dtype)["y"]
    _check(cfg, to_f64(y1), ref)
