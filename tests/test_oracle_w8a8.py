"""Pins for the oracle's 8-bit activations (W8A8 experts).

Each step of a W8A8 expert is tied to something other than the oracle:
  - the input row's quantisation: h before rounding equals SiLU(W_gate x_hat) *
    (W_up x_hat) with x_hat made by PyTorch's float8_e4m3fn cast (a library
    round-to-nearest-even encoder) and numpy products;
  - the hidden row's rounding and quantisation: h_hat equals PyTorch's fp32 ->
    bf16 cast followed by its float8_e4m3fn cast of h / s_h, and the bf16
    rounding alone equals PyTorch's cast on ties, infinities and NaN;
  - the down projection: numpy's product of the dequantised weights and h_hat;
  - the whole layer: on a hand-built layer where every activation is already on
    the E4M3 grid with a power-of-two scale, quantising the activations changes
    nothing, so the W8A8 layer must equal the pinned 8-bit-weight layer bit for
    bit (routing, shared expert and combine included).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_fp8 import _bf16_bits, _bits_to_f32, _fp8_layer

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _torch_quant_rows(v32):
    """Per-row E4M3 quantisation of float32 rows with PyTorch's float8 cast:
    scale = amax / 448 (fp32), codes of v / scale (fp32); returns the
    dequantised rows in float64."""
    v32 = np.asarray(v32, np.float32)
    amax = np.abs(v32).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = torch.from_numpy((v32 / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
    return q.to(torch.float64).numpy() * s[:, None].astype(np.float64)


def _torch_bf16(v64):
    """float64 -> float32 -> bf16 (both round to nearest even), as float32."""
    t = torch.from_numpy(np.asarray(v64, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float32).numpy()


def _deq(q, name):
    sn = "s" + name[1:] if name.startswith("w_") else "ss" + name[2:]
    return oracle.e4m3_decode(q[name]) * q[sn][..., None].astype(np.float64)


def _case(seed, rows_per_expert, d=64, I=96):
    rng = np.random.default_rng(seed)
    E = len(rows_per_expert)
    q = _fp8_layer(rng, 1, d, E, I, 0, 12)
    offsets = np.concatenate([[0], np.cumsum(rows_per_expert)]).astype(np.int32)
    R = int(offsets[-1])
    xf = (rng.standard_normal((R, d)) * np.exp2(rng.uniform(-3, 3, (R, 1)))).astype(np.float32)
    if R > 2:
        xf[1] = 0.0                    # a zero row: scale 1, all codes zero
    x = _bf16_bits(xf)
    return q, offsets, x


def test_bf16_rounding_matches_torch_including_ties():
    rng = np.random.default_rng(9)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits[:8000] = (bits[:8000] & 0xFFFF0000) | 0x8000          # exact ties
    bits[8000:9000] = (bits[8000:9000] & 0xFFFF0000) | 0x7FFF  # just below a tie
    v = bits.view(np.float32)
    extra = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.4e38, -3.4e38, 1e-45, -1e-40],
                     np.float32)
    v = np.concatenate([v, extra])
    ours = oracle.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin].view(np.uint32), ref[fin].view(np.uint32))


@pytest.mark.parametrize("seed,rows", [(1, [3, 0, 5, 1]), (2, [7, 2])])
def test_w8a8_expert_matches_library_quantisation_at_every_step(seed, rows):
    q, offsets, x = _case(seed, rows)
    y, h_pre, h_hat = oracle.expert_ffn_w8a8(x, offsets, q, "bf16", taps=True)
    wg, wu, wd = _deq(q, "w_gate"), _deq(q, "w_up"), _deq(q, "w_down")
    xh = _torch_quant_rows(_bits_to_f32(x))
    for e in range(len(rows)):
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        if sl.start == sl.stop:
            continue
        g = xh[sl] @ wg[e].T
        u = xh[sl] @ wu[e].T
        h_ref = g / (1.0 + np.exp(-g)) * u
        tol = 1e-12 * max(np.abs(h_ref).max(), 1e-300)
        assert np.abs(h_pre[sl] - h_ref).max() <= tol
        hh_ref = _torch_quant_rows(_torch_bf16(h_pre[sl]))
        assert np.array_equal(h_hat[sl], hh_ref)
        y_ref = h_hat[sl] @ wd[e].T
        assert np.abs(y[sl] - y_ref).max() <= 1e-12 * max(np.abs(y_ref).max(), 1e-300)


def test_w8a8_quantisation_is_not_a_no_op():
    """On random rows the hidden row really moves onto the E4M3 grid: h_hat
    differs from h, within the format's relative error bound."""
    q, offsets, x = _case(3, [6, 4])
    _, h_pre, h_hat = oracle.expert_ffn_w8a8(x, offsets, q, "bf16", taps=True)
    hb = _torch_bf16(h_pre).astype(np.float64)
    assert (h_hat != hb).mean() > 0.5
    s = np.abs(hb).max(axis=1, keepdims=True) / 448.0
    err = np.abs(h_hat - hb)
    # half a grid step: 2^-4 relative above 2^-6 * s, 2^-10 * s below
    bound = np.maximum(2.0 ** -4 * np.abs(hb), 2.0 ** -10 * s) * (1 + 1e-6)
    assert np.all(err <= bound)


def _exact_layer(T, d, E, K, I, Is, seed):
    """A layer on which every activation quantises exactly (see the module
    docstring): x rows are one-hot at column 0 with value 2^a (a in 0..2);
    gate codes in column 0 are 64, 128 or 256 with unit row scales, so
    g >= 64 and SiLU(g) == g in fp64; up codes in column 0 have magnitudes in
    [2^-4, 448] with power-of-two row scales; row 0 of every gate / up matrix
    holds 256 / 448, the largest product, so the hidden row's scale is a power
    of two and every h lands on the E4M3 grid."""
    rng = np.random.default_rng(seed)

    def codes(*shape):
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        c[(c & 0x7F) == 0x7F] ^= 0x01
        return c

    def gate_up(n_mats, rows):
        g = codes(n_mats, rows, d)
        u = codes(n_mats, rows, d)
        g[:, :, 0] = rng.choice(np.array([0x68, 0x70, 0x78], np.uint8), size=(n_mats, rows))
        mag = rng.integers(0x18, 0x7F, size=(n_mats, rows)).astype(np.uint8)  # 2^-4 .. 448
        u[:, :, 0] = mag | (rng.integers(0, 2, size=(n_mats, rows)).astype(np.uint8) << 7)
        g[:, 0, 0] = 0x78   # 256
        u[:, 0, 0] = 0x7E   # 448
        sg = np.ones((n_mats, rows), np.float32)
        su = np.exp2(rng.integers(-8, -2, size=(n_mats, 1))).repeat(rows, 1).astype(np.float32)
        return g, u, sg, su

    g, u, sg, su = gate_up(E, I)
    q = {"w_gate": g, "w_up": u, "w_down": codes(E, d, I), "s_gate": sg, "s_up": su,
         "s_down": np.exp2(rng.integers(-12, -6, size=(E, d))).astype(np.float32)}
    if Is:
        g, u, sg, su = gate_up(1, Is)
        q.update(ws_gate=g[0], ws_up=u[0], ws_down=codes(d, Is), ss_gate=sg[0], ss_up=su[0],
                 ss_down=np.exp2(rng.integers(-12, -6, size=d)).astype(np.float32))
    xf = np.zeros((T, d), np.float32)
    xf[:, 0] = np.exp2(rng.integers(0, 3, size=T))
    x = _bf16_bits(xf)
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.5).astype(np.float32))
    bias = rng.standard_normal(E) * 0.3
    return q, x, w_g, bias


@pytest.mark.parametrize("router,Is", [("softmax", 32), ("sigmoid", 32), ("softmax", 0)])
def test_w8a8_layer_equals_the_8bit_weight_layer_when_activations_are_exact(router, Is):
    T, d, E, K, I = 11, 32, 5, 2, 48
    q, x, w_g, bias = _exact_layer(T, d, E, K, I, Is, seed=7 + Is)
    toks = np.arange(T)
    ref = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype="bf16", bias=bias, router=router)
    out = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype="bf16", bias=bias, router=router,
                                    act8=True)
    for k in ("topk_idx", "topk_w", "logits"):
        assert np.array_equal(out[k], ref[k]), k
    assert np.array_equal(out["y"], ref["y"])
    assert np.abs(ref["y"]).max() > 0
    # the expert stage alone agrees as well
    counts, offsets, perm, _ = oracle.permute(ref["topk_idx"], E)
    x_perm = np.asarray(x)[perm // K]
    assert np.array_equal(oracle.expert_ffn_w8a8(x_perm, offsets, q),
                          oracle.expert_ffn_fp8(x_perm, offsets, q))


def test_w8a8_token_forward_matches_the_expert_stage():
    """The per-token layer and the grouped expert stage are two code paths of
    the oracle; on random data they agree row for row."""
    rng = np.random.default_rng(5)
    T, d, E, K, I, Is = 7, 64, 4, 2, 64, 32
    q = _fp8_layer(rng, T, d, E, I, Is, 12)
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.2).astype(np.float32))
    out = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, dtype="bf16", act8=True)
    counts, offsets, perm, inv = oracle.permute(out["topk_idx"], E)
    y_perm = oracle.expert_ffn_w8a8(np.asarray(x)[perm // K], offsets, q)
    shared = {"w_gate": q["ws_gate"][None], "w_up": q["ws_up"][None],
              "w_down": q["ws_down"][None], "s_gate": q["ss_gate"][None],
              "s_up": q["ss_up"][None], "s_down": q["ss_down"][None]}
    y_s = oracle.expert_ffn_w8a8(x, np.array([0, T], np.int32), shared)
    y = oracle.combine(y_perm, inv, out["topk_w"], y_s)
    assert np.allclose(y, out["y"], rtol=0, atol=1e-12 * np.abs(y).max())
