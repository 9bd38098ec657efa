"""Pins for the oracle's two-plane activations (the *_a2 functions).

A bf16 row x is carried as two E4M3 codes per element and one fp32 scale per
row: s = amax / 448, q = x / s (fp32), hi = E4M3(q), lo = E4M3(q - value(hi)),
x ~ s * (value(hi) + value(lo)).  Each step is tied to something other than the
oracle:
  - the codes: PyTorch's float8_e4m3fn cast (a library round-to-nearest-even
    encoder) of q and of the fp32 remainder, bit for bit;
  - the reading: within 2^-8 of |x| relative plus 2^-10 s absolute (the
    format's half steps of 2^-4 relative, applied twice), and exact when s is a
    power of two and |x| >= s / 4 (a bf16 value has 8 significant bits);
  - the expert stage: h before rounding equals SiLU(W_gate x~) (W_up x~) with x~
    made from PyTorch's casts and numpy products; h~ equals PyTorch's bf16 cast
    then its two float8 casts; y equals numpy's product with the dequantised
    W_down;
  - the layer: on the hand-built layer of test_oracle_w8a8 every activation is
    already on the E4M3 grid with a power-of-two scale, so the remainder plane
    is zero and the layer equals the pinned 8-bit-weight layer bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_fp8 import _bf16_bits, _bits_to_f32, _fp8_layer
from tests.test_oracle_w8a8 import _case, _deq, _exact_layer, _torch_bf16

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _torch_planes(v32):
    """The two planes of float32 rows with PyTorch's float8 cast: returns (hi,
    lo) as uint8 codes, the fp32 scales, and the rows read back in float64."""
    v32 = np.asarray(v32, np.float32)
    amax = np.abs(v32).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (v32 / s[:, None]).astype(np.float32)
    hi = torch.from_numpy(q).to(torch.float8_e4m3fn)
    r = (q - hi.to(torch.float32).numpy()).astype(np.float32)
    lo = torch.from_numpy(r).to(torch.float8_e4m3fn)
    back = (hi.to(torch.float64).numpy() + lo.to(torch.float64).numpy()) * s[:, None].astype(np.float64)
    return (hi.view(torch.uint8).numpy(), lo.view(torch.uint8).numpy(), s, back)


def _rows(seed, n=64, cols=384):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((n, cols)) * np.exp2(rng.uniform(-12, 12, (n, 1)))
    v[:, ::7] *= np.exp2(rng.uniform(-20, 0, (n, 1)))   # values deep below the row max
    v[3] = 0.0                                          # a zero row
    return _bf16_bits(v.astype(np.float32))


def test_planes_match_torch_float8_casts():
    x = _rows(1)
    hi, lo, s = oracle.split_e4m3_rows(x, "bf16")
    thi, tlo, ts, _ = _torch_planes(_bits_to_f32(x))
    assert np.array_equal(s, ts)
    assert np.array_equal(hi, thi)
    assert np.array_equal(lo, tlo)
    assert np.all(hi[3] == 0) and np.all(lo[3] == 0) and s[3] == 1.0


def test_planes_meet_the_two_step_error_bound_and_are_not_one_plane():
    x = _rows(2)
    hi, lo, s = oracle.split_e4m3_rows(x, "bf16")
    xf = _bits_to_f32(x).astype(np.float64)
    back = (oracle.e4m3_decode(hi) + oracle.e4m3_decode(lo)) * s[:, None].astype(np.float64)
    err = np.abs(back - xf)
    bound = (2.0 ** -8 * np.abs(xf) + 2.0 ** -10 * s[:, None]) * (1 + 1e-9)
    assert np.all(err <= bound)
    # the second plane matters: one plane alone is ~16x worse on random rows
    one = oracle.e4m3_decode(hi) * s[:, None].astype(np.float64)
    assert np.abs(one - xf).sum() > 8 * err.sum()
    assert (lo != 0).mean() > 0.5


def test_planes_are_exact_with_a_power_of_two_scale():
    """amax = 448 * 2^k gives s = 2^k, and every bf16 value of the row with
    |x / s| >= 1/4 is then s * (hi + lo) exactly: hi keeps the top 4 of its 8
    significant bits after rounding, the remainder needs at most 3 more, and its
    lowest bit, 2^-7 of the leading one, is no finer than E4M3's 2^-9 step."""
    rng = np.random.default_rng(3)
    n, cols = 32, 256
    k = rng.integers(-6, 6, size=(n, 1))
    mag = np.exp2(rng.uniform(-2, 8.8, (n, cols)))       # |x / s| in [2^-2, 448)
    v = np.sign(rng.standard_normal((n, cols))) * mag * np.exp2(k)
    v[:, 0] = 448.0 * np.exp2(k[:, 0])
    x = _bf16_bits(v.astype(np.float32))
    hi, lo, s = oracle.split_e4m3_rows(x, "bf16")
    assert np.array_equal(s.astype(np.float64), np.exp2(k[:, 0]).astype(np.float64))
    back = (oracle.e4m3_decode(hi) + oracle.e4m3_decode(lo)) * s[:, None].astype(np.float64)
    assert np.array_equal(back, _bits_to_f32(x).astype(np.float64))


@pytest.mark.parametrize("seed,rows", [(1, [3, 0, 5, 1]), (2, [7, 2])])
def test_a2_expert_matches_library_casts_at_every_step(seed, rows):
    q, offsets, x = _case(seed, rows)
    y, h_pre, h_hat = oracle.expert_ffn_a2(x, offsets, q, "bf16", taps=True)
    wg, wu, wd = _deq(q, "w_gate"), _deq(q, "w_up"), _deq(q, "w_down")
    xt = _torch_planes(_bits_to_f32(x))[3]
    for e in range(len(rows)):
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        if sl.start == sl.stop:
            continue
        g = xt[sl] @ wg[e].T
        u = xt[sl] @ wu[e].T
        h_ref = g / (1.0 + np.exp(-g)) * u
        assert np.abs(h_pre[sl] - h_ref).max() <= 1e-12 * max(np.abs(h_ref).max(), 1e-300)
        assert np.array_equal(h_hat[sl], _torch_planes(_torch_bf16(h_pre[sl]))[3])
        y_ref = h_hat[sl] @ wd[e].T
        assert np.abs(y[sl] - y_ref).max() <= 1e-12 * max(np.abs(y_ref).max(), 1e-300)


def test_a2_expert_is_close_to_the_exact_8bit_weight_expert():
    """Two planes read each activation within 2^-8: the stage stays within the
    bf16 layer's 1e-2 budget of the exact W8A16 stage, far closer than one plane."""
    q, offsets, x = _case(4, [9, 6, 11])
    y2 = oracle.expert_ffn_a2(x, offsets, q, "bf16")
    y16 = oracle.expert_ffn_fp8(x, offsets, q, "bf16")
    y1 = oracle.expert_ffn_w8a8(x, offsets, q, "bf16")
    d2 = np.linalg.norm(y2 - y16) / np.linalg.norm(y16)
    d1 = np.linalg.norm(y1 - y16) / np.linalg.norm(y16)
    assert d2 < 5e-3 and d1 > 4 * d2


@pytest.mark.parametrize("router,Is", [("softmax", 32), ("sigmoid", 0)])
def test_a2_layer_equals_the_8bit_weight_layer_when_activations_are_exact(router, Is):
    T, d, E, K, I = 11, 32, 5, 2, 48
    q, x, w_g, bias = _exact_layer(T, d, E, K, I, Is, seed=11 + Is)
    toks = np.arange(T)
    ref = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype="bf16", bias=bias, router=router)
    out = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype="bf16", bias=bias, router=router,
                                    act8="planes")
    for k in ("topk_idx", "topk_w", "logits", "y"):
        assert np.array_equal(out[k], ref[k]), k
    assert np.abs(ref["y"]).max() > 0


def test_a2_token_forward_matches_the_expert_stage():
    rng = np.random.default_rng(6)
    T, d, E, K, I, Is = 7, 64, 4, 2, 64, 32
    q = _fp8_layer(rng, T, d, E, I, Is, 12)
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.2).astype(np.float32))
    out = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, dtype="bf16", act8="planes")
    counts, offsets, perm, inv = oracle.permute(out["topk_idx"], E)
    y_perm = oracle.expert_ffn_a2(np.asarray(x)[perm // K], offsets, q)
    shared = {"w_gate": q["ws_gate"][None], "w_up": q["ws_up"][None],
              "w_down": q["ws_down"][None], "s_gate": q["ss_gate"][None],
              "s_up": q["ss_up"][None], "s_down": q["ss_down"][None]}
    y_s = oracle.expert_ffn_a2(x, np.array([0, T], np.int32), shared)
    y = oracle.combine(y_perm, inv, out["topk_w"], y_s)
    assert np.allclose(y, out["y"], rtol=0, atol=1e-12 * np.abs(y).max())
