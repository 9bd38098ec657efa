"""Stage 1 on the GPU (moe_route) against the oracle.

Bit-exact routing: both sides get the same fp32 scores on a 1/512 grid (distinct
values differ by >= 1.95e-3, equal values are decided only by the tie rule).
Scores computed from x . w_g: compared within the fp32 accumulation error; the
picks, in slot order, compared on every token whose fp64 keys leave gaps of at
least 1e-3 among its K picks and at the top-K boundary; the weights within the
bound the score error sets."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from tests.gpu_util import MARGIN, W_RTOL, Layer, clean_rows, host, order_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _route_logits(moe, logits: torch.Tensor, K: int):
    T, E = logits.shape
    s = moe.make_shape(T, 64, E, K, 64, 0, "f32")
    ws = moe.alloc_workspace(s)
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    out = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_route(s, None, None, None, logits.cuda(), out, idx, w, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), logits.cpu())
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,E,K,scale", [
    (64, 8, 2, 512), (8, 256, 8, 512), (4096, 8, 2, 512), (16384, 256, 8, 512),
    (1, 256, 8, 512), (100, 256, 8, 2), (37, 1024, 32, 4), (5, 3, 3, 8), (9, 1, 1, 1),
    (77, 33, 32, 16), (513, 64, 1, 512)])
def test_route_is_bit_exact_from_the_same_scores(moe, T, E, K, scale):
    logits = mi.grid_logits(T, E, seed=101, scale=scale)
    idx, w = _route_logits(moe, logits, K)
    ref_idx, ref_w, _ = oracle.route(None, None, K, logits_in=logits.numpy())
    assert np.array_equal(idx, ref_idx)
    assert np.allclose(w, ref_w, rtol=W_RTOL, atol=0)


def test_route_bit_exact_with_zipf_bias_and_all_ties(moe):
    cfg = mi.CONFIGS["dsv3_prefill_zipf"]
    z = mi.grid_logits(cfg.T, cfg.E, seed=102).double()
    b = mi.make_bias(cfg).double()
    logits = (torch.round((z + b) * 512) / 512).float()
    idx, w = _route_logits(moe, logits, cfg.K)
    ref_idx, ref_w, _ = oracle.route(None, None, cfg.K, logits_in=logits.numpy())
    assert np.array_equal(idx, ref_idx)
    assert np.allclose(w, ref_w, rtol=W_RTOL)
    # every score equal: experts 0..K-1 with weight 1/K; -0.0 ties with +0.0
    zero = torch.zeros(64, 256)
    zero[::2, 5] = -0.0
    idx, w = _route_logits(moe, zero, 8)
    assert np.array_equal(idx, np.tile(np.arange(8), (64, 1)))
    assert np.allclose(w, 1 / 8, rtol=1e-7)


SMALL_E = {f"smallE{E}_{dt}_T{T}": mi.LayerConfig(f"smallE{E}_{dt}", T=T, d=192, E=E, K=min(E, 4),
                                                     I=64, dtype=dt)
           for E, dt, T in [(3, "bf16", 257), (8, "f32", 300), (12, "bf16", 300),
                            (20, "f32", 511), (32, "bf16", 256)]}


@pytest.mark.parametrize("name,T", [("tiny_f32", None), ("dsv3_decode", None),
                                    ("dsv3_prefill_zipf", 512), ("dsv3_sweep_T4096", None),
                                    ("mixtral_prefill", 256), ("mixtral_prefill", 4096),
                                    *[(n, None) for n in SMALL_E]])
def test_route_from_x(moe, name, T):
    """Scores from x . w_g: split-K GEMV router (few tokens), token-major router
    (E <= 32, T >= 256), or the tensor-core router (large bf16 batches, E >= 64)."""
    cfg = SMALL_E[name] if name in SMALL_E else mi.CONFIGS[name]
    if T is not None:
        cfg = cfg.with_T(T)
    L = Layer(cfg, only={"w_g"})
    if cfg.T <= 256:
        L.x = clean_rows(L)  # small batches: every token's routing made unique, all checked
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route(s, L.x, L.p["w_g"], L.bias, None, out, idx, w, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    ref_idx, ref_w, ref_logits = oracle.route(host(L.x), L.hp["w_g"], cfg.K, dtype=cfg.dtype,
                                              bias=L.bias_host())
    got = out.cpu().numpy().astype(np.float64)
    # fp32 accumulation of exact products: error well under 1e-4 of the score scale
    assert np.max(np.abs(got - ref_logits)) <= 1e-4 * max(1.0, np.max(np.abs(ref_logits)))
    # tokens whose picks and slot order are unique at fp32 precision
    ok = order_margin(ref_logits, cfg.K) >= MARGIN
    assert ok.mean() > 0.9 and (cfg.T > 256 or ok.all())
    gi = idx.cpu().numpy()
    assert np.array_equal(gi[ok], ref_idx[ok])  # slot j = the j-th pick
    # a score error delta moves ln w_j by at most 2 max|delta| (softmax over the K)
    gw = w.cpu().numpy().astype(np.float64)
    delta = np.abs(got - ref_logits).max(axis=1, keepdims=True)
    assert np.all(np.abs(gw[ok] - ref_w[ok]) <= (2.0 * delta[ok] + 2e-6) * ref_w[ok])


# ---------------------------------------------------------------- sigmoid router (DeepSeek-V3)

def _route_logits_mode(moe, logits: torch.Tensor, K: int, router: str, bias=None):
    T, E = logits.shape
    s = moe.make_shape(T, 64, E, K, 64, 0, "f32", router)
    ws = moe.alloc_workspace(s)
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    keys = torch.empty((T, E), dtype=torch.float32, device="cuda")
    b = None if bias is None else torch.as_tensor(bias, dtype=torch.float32).cuda()
    moe.moe_route(s, None, None, b, logits.cuda(), keys, idx, w, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), keys.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,E,K,with_bias", [(8, 256, 8, False), (4096, 256, 8, True),
                                             (16384, 256, 8, True), (100, 64, 6, True),
                                             (33, 8, 8, False), (50, 20, 1, True)])
def test_sigmoid_route_matches_oracle(moe, T, E, K, with_bias):
    """Same fp32 scores on both sides.  Without a bias the sigmoid keeps the
    order of the scores, so the selection is bit-exact including ties; with a
    bias (1/32 grid) keys of different experts can nearly coincide, so tokens
    whose fp64 keys leave a gap below 1e-5 among the picks or at the boundary
    are left out."""
    logits = mi.grid_logits(T, E, seed=111, scale=512)
    bias = (np.round(np.random.default_rng(5).standard_normal(E) * 8) / 32) if with_bias else None
    idx, w, keys = _route_logits_mode(moe, logits, K, "sigmoid", bias)
    ref_idx, ref_w, ref_keys = oracle.route(None, None, K, logits_in=logits.numpy(), bias=bias,
                                            router="sigmoid")
    assert np.max(np.abs(keys - ref_keys)) <= 1e-6
    ok = order_margin(ref_keys, K) >= (1e-5 if with_bias else 0.0)
    if with_bias:
        assert ok.mean() >= 0.95
    assert np.array_equal(idx[ok], ref_idx[ok])
    assert np.allclose(w[ok], ref_w[ok], rtol=2e-6, atol=0)


@pytest.mark.parametrize("name,T", [("dsv3_decode", None), ("dsv3_prefill_zipf", 512)])
def test_sigmoid_route_from_x(moe, name, T):
    cfg = mi.CONFIGS[name]
    if T is not None:
        cfg = cfg.with_T(T)
    import dataclasses
    cfg = dataclasses.replace(cfg, router="sigmoid")
    L = Layer(cfg, only={"w_g"})
    bias = None if L.bias is None else (L.bias / 8).contiguous()  # keys live in (0, 1)
    L.bias = bias
    if cfg.T <= 256:
        L.x = clean_rows(L)  # small batches: every token's routing made unique, all checked
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    keys = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route(s, L.x, L.p["w_g"], bias, None, keys, idx, w, ws)
    torch.cuda.synchronize()
    ref_idx, ref_w, ref_keys = oracle.route(host(L.x), L.hp["w_g"], cfg.K, dtype=cfg.dtype,
                                            bias=None if bias is None else bias.double().cpu().numpy(),
                                            router="sigmoid")
    assert np.max(np.abs(keys.cpu().numpy() - ref_keys)) <= 1e-5
    ok = order_margin(ref_keys, cfg.K) >= 1e-4
    assert ok.mean() > 0.9 and (cfg.T > 256 or ok.all())
    gi, gw = idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    assert np.array_equal(gi[ok], ref_idx[ok])  # slot j = the j-th pick
    # the raw scores' error bounds the weights' (d ln sigmoid(s) / ds = 1 - sigmoid(s) <= 1,
    # so |dw| / w <= 2 max|delta|); the raw scores come from the softmax router without bias
    s0 = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype, "softmax")
    raw = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route(s0, L.x, L.p["w_g"], None, None, raw, idx.clone(), w.clone(),
                  moe.alloc_workspace(s0))
    torch.cuda.synchronize()
    _, _, raw_ref = oracle.route(host(L.x), L.hp["w_g"], cfg.K, dtype=cfg.dtype)
    delta = np.abs(raw.cpu().numpy() - raw_ref).max(axis=1, keepdims=True)
    assert np.all(np.abs(gw[ok] - ref_w[ok]) <= (2.0 * delta[ok] + 2e-6) * ref_w[ok])


@pytest.mark.parametrize("T,d,E,K,dtype,router", [
    (1, 7168, 256, 8, "bf16", "softmax"), (8, 7168, 256, 8, "bf16", "sigmoid"),
    (16, 7168, 256, 8, "bf16", "softmax"), (5, 256, 8, 2, "f32", "softmax"),
    (16, 512, 1024, 32, "bf16", "softmax"), (3, 192, 33, 5, "f32", "sigmoid"),
    (17, 7168, 256, 8, "bf16", "softmax")])
def test_fused_router_changes_no_bit(moe, T, d, E, K, dtype, router, monkeypatch):
    """With MOE_FUSED_ROUTER=1 batches of at most 16 tokens score and route in one
    launch (the block that finishes last runs the top-K): the same expert ids,
    weights and keys, bit for bit, as the two launches (the default), on three
    calls in a row on one workspace (the ticket counter must start from zero each
    time) and from a replayed CUDA graph.  T = 17 is past the bound (two launches
    either way)."""
    cfg = mi.LayerConfig("fused_route", T=T, d=d, E=E, K=K, I=64, dtype=dtype, router=router,
                         seed=23)
    L = Layer(cfg, only={"w_g"})
    bias = torch.from_numpy(np.random.default_rng(3).standard_normal(E) / 16).float().cuda()
    s = L.shape(moe)
    ws = moe.alloc_workspace(s)

    def route():
        idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
        w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
        keys = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_route(s, L.x, L.p["w_g"], bias, None, keys, idx, w, ws)
        return idx, w, keys

    monkeypatch.setenv("MOE_FUSED_ROUTER", "0")
    ref = route()
    torch.cuda.synchronize()
    monkeypatch.setenv("MOE_FUSED_ROUTER", "1")
    outs = [route() for _ in range(3)]
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    keys = torch.empty((T, E), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=st):
        moe.moe_route(s, L.x, L.p["w_g"], bias, None, keys, idx, w, ws, stream=st)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    for o in outs + [(idx, w, keys)]:
        for a, b in zip(o, ref):
            assert torch.equal(a, b)
