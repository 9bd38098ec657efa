"""8-bit (E4M3) expert weights on the GPU against the oracle.

The row quantiser is integer work decided by fp32 arithmetic that both sides
do in the same precision (amax / 448 and w / scale as IEEE fp32 divisions,
round to nearest even): codes and scales must match bit for bit.  The fp8
expert FFN and the fp8 layer are compared like the bf16 ones (relative L2
against the fp64 oracle on the same codes and scales)."""
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


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols", [(600, 2048), (1, 16), (37, 7168)])
def test_quantize_rows_bit_exact(moe, dtype, rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    w = torch.randn(rows, cols, generator=g) * torch.exp2(torch.rand(rows, 1, generator=g) * 16 - 8)
    if rows > 2:
        w[1] = 0.0                         # a row of zeros
        w[2, 3] = -w[2].abs().max() * 3    # a negative extreme
    w = w.to(mi.torch_dtype(dtype))
    wd = w.cuda()
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(wd, codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_rows(mi.to_host_array(w), dtype)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_rows_of_a_3d_weight_stack(moe):
    cfg = replace(mi.CONFIGS["dsv3_decode"], E=3, I=256)
    w = mi.make_weights(cfg, "cuda", only={"w_down"})["w_down"]     # [3][7168][256] bf16
    codes = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(w.shape[:-1], dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(w, codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_fp8_rows(host(w), "bf16")
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


# ---------------------------------------------------------------- expert FFN

def _expert_ffn_case(moe, counts, d, I, seed=0, with_planes=False):
    E = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    cfg = mi.LayerConfig("fp8_ffn", T=max(rows, 1), d=d, E=E, K=1, I=I, weights="e4m3", seed=seed)
    q = mi.make_weights(cfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                           "s_down"})
    x_perm = mi.normal((max(rows, 1), d), 1.0, "bf16", "cuda", seed, "x_perm")[:rows]
    s = moe.make_shape(rows, d, E, 1, I, 0, "bf16")
    ws = moe.alloc_workspace(s)
    y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    W = moe.make_fp8_experts(q)
    moe.moe_expert_ffn_fp8(s, x_perm, torch.from_numpy(offsets).cuda(), W, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    qh = {k: host(v) for k, v in q.items()}
    ref = oracle.expert_ffn_fp8(host(x_perm), offsets, qh, dtype="bf16")
    if with_planes:
        return to_f64(y), ref, oracle.expert_ffn_a2(host(x_perm), offsets, qh, dtype="bf16")
    return to_f64(y), ref


# the tensor-core groups' activation path: two E4M3 planes on the 8-bit MMA (the
# default), or the codes widened to bf16 in the GEMM on single-SM or pair tiles
PATHS = {"planes": {"MOE_W8_PLANES": "1"},
         "widen": {"MOE_W8_PLANES": "0", "MOE_W8_PAIR": "0"},
         "widen_pair": {"MOE_W8_PLANES": "0", "MOE_W8_PAIR": "1"}}


@pytest.mark.parametrize("counts,d,I", [
    ([75, 0, 140, 3, 1, 260, 77, 44], 256, 384),     # ragged groups, one empty; GEMV + tiles
    ([600, 257, 1, 129], 384, 640),                  # several m-tiles per group, 5 n-blocks
    ([1, 2, 1, 1, 3, 1, 1, 2], 1024, 256),           # decode-like: a few rows per expert (GEMV)
    ([8, 9, 0, 7, 16, 17], 128, 128),                # around the GEMV limit, narrowest shapes
    ([16, 15, 1, 33], 7168, 256),                    # DeepSeek-width rows, 16-row passes
])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_expert_ffn_fp8_matches_oracle(moe, counts, d, I, path, monkeypatch):
    """Every path against the exact 8-bit-weight stage (fp64, bf16 activations);
    the two-plane path also against the oracle's two-plane stage, which it
    computes up to fp32 accumulation and the bf16 storage of h and y."""
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    y, ref, ref2 = _expert_ffn_case(moe, counts, d, I, with_planes=True)
    assert rel_l2(y, ref) <= BF16_REL_L2
    for r in range(y.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r
    if path == "planes":
        assert rel_l2(y, ref2) <= BF16_REL_L2
        for r in range(y.shape[0]):
            assert rel_l2(y[r], ref2[r]) <= 2 * BF16_REL_L2, r


@pytest.mark.parametrize("planes", ["1", "0"])
@pytest.mark.parametrize("rho", [None, "1", "1000000"])
def test_expert_ffn_fp8_side_by_side_changes_no_bit(moe, rho, planes, monkeypatch):
    """Groups on CTA-pair tiles and groups on single-SM tiles: the two tile
    shapes run on two streams at once, on the plan's split of the SMs (pushed
    to both extremes through MOE_SPLIT_RHO), with the same bits as one after
    the other (MOE_CONCURRENT=0)."""
    counts, d, I = [600, 257, 1, 129, 300, 140], 384, 640
    monkeypatch.setenv("MOE_W8_PAIR", "1")
    monkeypatch.setenv("MOE_W8_PLANES", planes)
    monkeypatch.setenv("MOE_CONCURRENT", "0")
    y0, ref = _expert_ffn_case(moe, counts, d, I, seed=4)
    monkeypatch.setenv("MOE_CONCURRENT", "1")
    if rho is not None:
        monkeypatch.setenv("MOE_SPLIT_RHO", rho)
    y1, _ = _expert_ffn_case(moe, counts, d, I, seed=4)
    assert np.array_equal(y0, y1)
    assert rel_l2(y0, ref) <= BF16_REL_L2


# ---------------------------------------------------------------- the layer

def _clean_x(L: Layer):
    return clean_rows(L)


def _check_rows(y, ref):
    assert rel_l2(y, ref) <= BF16_REL_L2
    for r in range(y.shape[0]):
        assert rel_l2(y[r], ref[r]) <= 2 * BF16_REL_L2, r


@pytest.mark.parametrize("router", ["softmax", "sigmoid"])
@pytest.mark.parametrize("gemv8", ["0", "8", "16", "40"])
def test_forward_fp8_small_layer_all_tokens(moe, router, gemv8, monkeypatch):
    """Groups of ~11 rows and a 45-row shared group: all on the tensor cores
    (limit 0), part of the routed groups on the 8-bit GEMV (8, the default),
    every routed group in one 16-row pass of the second list (16), or
    everything including the shared group in passes of 16 rows (40)."""
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", gemv8)
    cfg = mi.LayerConfig("fp8_small", T=45, d=256, E=12, K=3, I=384, Is=256, router=router,
                         weights="e4m3")
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


def test_forward_fp8_without_shared_expert(moe):
    cfg = mi.LayerConfig("fp8_noshared", T=300, d=512, E=8, K=2, I=256, weights="e4m3")
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


@pytest.mark.parametrize("gemv8", ["0", "8"])
def test_forward_fp8_decode_full_size(moe, gemv8, monkeypatch):
    """DeepSeek-V3 decode shapes: every group on the 8-bit GEMV (default) or on
    the tensor cores (limit 0)."""
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", gemv8)
    cfg = mi.CONFIGS["dsv3_decode_fp8"]
    L = Layer(cfg)
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    ref = L.oracle_tokens(np.arange(cfg.T))
    _check_rows(y, ref["y"])


@pytest.mark.parametrize("path", sorted(PATHS))
def test_forward_fp8_prefill_sampled_tokens(moe, path, monkeypatch):
    """Mixtral-shaped prefill: ~1024-row groups with two-plane activations on the
    8-bit MMA (default), or widened to bf16 in the GEMM on single-SM or CTA-pair
    tiles."""
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    cfg = mi.CONFIGS["mixtral_prefill_fp8"]
    L = Layer(cfg)
    y = L.forward(moe)
    tokens, skipped = parity_tokens(L, 256)
    print(f"{cfg.name}: {len(tokens)} sampled tokens checked, {skipped} skipped")
    ref = L.oracle_tokens(tokens)
    assert_routing_on_sample(moe, L, tokens, ref)
    _check_rows(to_f64(y[torch.from_numpy(tokens).long().cuda()]), ref["y"])


@pytest.mark.parametrize("planes,tol", [("0", 2e-3), ("1", BF16_REL_L2)])
def test_forward_fp8_matches_bf16_layer_on_exact_weights(moe, planes, tol, monkeypatch):
    """Power-of-two row scales make every dequantised weight a bf16 value: with
    the codes widened in the GEMM the fp8 layer and the bf16 layer on those
    weights compute the same products, so their outputs agree to accumulation
    order; with two-plane activations, within the planes' 2^-8 reading of x and
    h (the bf16 layer budget)."""
    monkeypatch.setenv("MOE_W8_PLANES", planes)
    cfg = mi.LayerConfig("fp8_exact", T=200, d=256, E=8, K=2, I=256, Is=128, weights="e4m3")
    L = Layer(cfg)
    for k in list(L.p):
        if k.startswith("s") and L.p[k].dtype == torch.float32:
            L.p[k] = torch.exp2(torch.round(torch.log2(L.p[k])))
    y8 = to_f64(L.forward(moe))
    deq = {}
    for n in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        sn = "s" + n[1:] if n.startswith("w_") else "ss" + n[2:]
        v = torch.from_numpy(oracle.e4m3_decode(host(L.p[n]))).cuda()
        deq[n] = (v * L.p[sn].double()[..., None]).to(torch.bfloat16)
    s = L.shape(moe)
    ybf = torch.empty_like(L.x)
    ws = moe.alloc_workspace(s)
    moe.moe_forward(s, L.x, L.p["w_g"], L.bias, deq["w_gate"], deq["w_up"], deq["w_down"],
                    deq["ws_gate"], deq["ws_up"], deq["ws_down"], ybf, ws)
    torch.cuda.synchronize()
    assert rel_l2(y8, to_f64(ybf)) <= tol


def test_forward_fp8_zero_tokens_is_a_no_op(moe):
    cfg = mi.LayerConfig("fp8_empty", T=4, d=128, E=4, K=2, I=128, weights="e4m3")
    L = Layer(cfg)
    s = moe.make_shape(0, 128, 4, 2, 128, 0, "bf16")
    moe.moe_forward_fp8(s, None, L.p["w_g"], None, moe.make_fp8_experts(L.p), None, None)


@pytest.mark.parametrize("planes", ["1", "0"])
def test_fp8_stalled_copy_times_out_and_the_context_survives(moe, planes, monkeypatch):
    """No tile is ever requested: the MMA's bounded waits (and, with the codes
    widened in the GEMM, the converters') run out, the kernel records
    MOE_ERR_TIMEOUT and returns."""
    monkeypatch.setenv("MOE_W8_PLANES", planes)
    cfg = mi.LayerConfig("fp8_stall", T=64, d=256, E=4, K=2, I=256, Is=128, weights="e4m3")
    L = Layer(cfg)
    monkeypatch.setenv("MOE_TC_TIMEOUT_MS", "50")
    monkeypatch.setenv("MOE_TC_TEST_STALL", "1")
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(L.x)
    moe.moe_forward_fp8(s, L.x, L.p["w_g"], L.bias, moe.make_fp8_experts(L.p), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_TC_TEST_STALL")
    monkeypatch.delenv("MOE_TC_TIMEOUT_MS")
    L.x = _clean_x(L)
    y = to_f64(L.forward(moe))
    _check_rows(y, L.oracle_tokens(np.arange(cfg.T))["y"])


@pytest.mark.parametrize("swap", ["0", "16", "64"])
@pytest.mark.parametrize("counts,d,I", [
    ([300, 1, 7, 16, 17, 33, 64, 65, 0, 130], 384, 640),   # small groups beside large ones
    ([2, 40, 600], 7168, 256),                              # DeepSeek-width rows
])
def test_swapped_8bit_tiles_match_the_oracle(moe, counts, d, I, swap, monkeypatch):
    """Groups of at most MOE_SWAP_MAX_ROWS rows beside larger ones run with the
    operands swapped (weights as the M operand, the two activation planes as
    N = 16/32/64 columns); 0 keeps every tile unswapped.  Every setting
    against the exact 8-bit-weight stage and the two-plane stage."""
    monkeypatch.setenv("MOE_SWAP_MAX_ROWS", swap)
    monkeypatch.setenv("MOE_GEMV8_MAX_ROWS", "0")
    y, ref, ref2 = _expert_ffn_case(moe, counts, d, I, seed=7, with_planes=True)
    _check_rows(y, ref)
    _check_rows(y, ref2)
