"""Pins for the oracle's 8-bit (E4M3) expert weights.

The codec is tied to PyTorch's float8_e4m3fn dtype (a library decoder and a
round-to-nearest-even encoder), to a brute-force nearest-code search and to
closed-form anchors of the format.  The row quantiser is tied to the format's
error bound and to the amax -> 448 mapping.  The fp8 layer is tied to the
already-pinned bf16/fp32 layer: with scales that make every dequantised weight
exactly representable, both must give bit-identical fp64 results.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _torch_decode(codes):
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


ALL = np.arange(256, dtype=np.uint8)
POS = np.arange(0x7F, dtype=np.uint8)  # +0 .. 448, the finite non-negative codes


# ---------------------------------------------------------------- decode

def test_decode_matches_torch_float8_for_every_code():
    ours, ref = oracle.e4m3_decode(ALL), _torch_decode(ALL)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_decode_closed_form_anchors():
    v = oracle.e4m3_decode(ALL)
    assert v[0x00] == 0.0 and not np.signbit(v[0x00])
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9           # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert v[0x08] == 2.0 ** -6           # smallest normal
    assert v[0x38] == 1.0                 # exponent field 7 = bias
    assert v[0x3F] == 1.875
    assert v[0x40] == 2.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    # the non-negative finite codes are strictly increasing, and the negative
    # codes mirror them
    assert np.all(np.diff(v[POS]) > 0)
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def test_decoded_values_are_exact_in_bf16():
    v = oracle.e4m3_decode(POS).astype(np.float32)
    bf = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(v, bf)


# ---------------------------------------------------------------- encode

def _brute_nearest(v):
    """Nearest non-negative finite code to |v|, ties to the even code, with the
    sign bit of v; magnitudes past 448 clamp."""
    grid = oracle.e4m3_decode(POS)
    out = np.empty(v.shape, np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        a = abs(x)
        dist = np.abs(grid - a)
        best = np.flatnonzero(dist == dist.min())
        code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        out[i] = code | (0x80 if np.signbit(x) else 0)
    return out


def _probe_values(rng):
    grid = oracle.e4m3_decode(POS)
    mids = (grid[1:] + grid[:-1]) / 2
    vals = [grid, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
            np.nextafter(mids.astype(np.float32), np.float32(1000)),
            np.exp2(rng.uniform(-12, 8.8, 3000)),
            rng.uniform(0, 2.0 ** -6, 500)]
    v = np.concatenate([np.asarray(a, np.float64) for a in vals]).astype(np.float32)
    v = v[np.abs(v) < 448]
    sign = np.where(rng.random(v.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    return v * sign


def test_encode_is_the_nearest_code_with_ties_to_even():
    v = _probe_values(np.random.default_rng(11))
    assert np.array_equal(oracle.e4m3_encode(v), _brute_nearest(v))


def test_encode_matches_torch_round_to_nearest_even():
    v = _probe_values(np.random.default_rng(12))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), ref)


def test_encode_saturates_and_keeps_nan():
    big = np.array([448.0, 448.5, 463.9, 464.0, 1e30, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert oracle.e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80


def test_encode_decode_round_trip_on_the_grid():
    v = oracle.e4m3_decode(ALL)
    fin = ~np.isnan(v)
    assert np.array_equal(oracle.e4m3_encode(v[fin].astype(np.float32)), ALL[fin])


# ---------------------------------------------------------------- row quantiser

def _bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantised_rows_meet_the_format_error_bound(dtype):
    rng = np.random.default_rng(21)
    rows, cols = 37, 200
    w = (rng.standard_normal((rows, cols)) * np.exp2(rng.uniform(-8, 6, (rows, 1)))).astype(np.float32)
    w[3] = 0.0                              # a row of zeros
    w[5, 7] = -np.abs(w[5]).max() * 2       # negative extreme
    stored = _bf16_bits(w) if dtype == "bf16" else w
    wv = _bits_to_f32(stored) if dtype == "bf16" else w
    codes, scale = oracle.quantize_fp8_rows(stored, dtype)
    assert codes.shape == (rows, cols) and scale.shape == (rows,)
    amax = np.abs(wv).max(axis=1)
    nz = amax > 0
    # amax maps to the largest finite code: scale = amax / 448 in fp32
    assert np.array_equal(scale[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    assert scale[3] == 1.0 and np.all(codes[3] & 0x7F == 0)
    dec = oracle.e4m3_decode(codes)
    assert not np.isnan(dec).any()
    assert np.all(np.abs(dec[nz]).max(axis=1) == 448.0)
    # rounding error of w / s: half a grid step, i.e. <= 2^-4 relative for
    # normal codes and <= 2^-10 absolute in the subnormal range
    q = wv.astype(np.float64) / scale[:, None].astype(np.float64)
    err = np.abs(dec - q)
    normal = np.abs(q) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(q[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))
    # signs survive
    assert np.all((np.sign(dec) == np.sign(q)) | (dec == 0))


def test_quantise_then_dequantise_keeps_the_row_within_one_sixteenth():
    rng = np.random.default_rng(22)
    w = rng.standard_normal((8, 512)).astype(np.float32)
    codes, scale = oracle.quantize_fp8_rows(w, "f32")
    what = oracle.e4m3_decode(codes) * scale[:, None]
    rel = np.linalg.norm(what - w, axis=1) / np.linalg.norm(w, axis=1)
    assert np.all(rel < 1 / 16)


# ---------------------------------------------------------------- the fp8 layer

def _fp8_layer(rng, T, d, E, I, Is, exact_bits):
    """Random E4M3 codes (no NaN) and per-row scales whose significand has at
    most exact_bits bits, so code * scale is exact in fp32 (<= 20) or bf16
    (0: powers of two)."""
    def codes(*shape):
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        c[(c & 0x7F) == 0x7F] ^= 0x01       # NaN -> +-448 neighbour
        return c

    def scales(*shape):
        e = rng.integers(-12, -4, size=shape)
        m = rng.integers(1 << exact_bits, 2 << exact_bits, size=shape) if exact_bits else 1
        return (np.ldexp(np.float64(1), e) * m / (1 << exact_bits)).astype(np.float32)

    q = {"w_gate": codes(E, I, d), "w_up": codes(E, I, d), "w_down": codes(E, d, I),
         "s_gate": scales(E, I), "s_up": scales(E, I), "s_down": scales(E, d)}
    if Is:
        q.update(ws_gate=codes(Is, d), ws_up=codes(Is, d), ws_down=codes(d, Is),
                 ss_gate=scales(Is), ss_up=scales(Is), ss_down=scales(d))
    return q


def _dequant(q, to):
    """The dequantised weights code * scale[row] as float32 (exact by construction)."""
    out = {}
    for n, sn in (("w_gate", "s_gate"), ("w_up", "s_up"), ("w_down", "s_down"),
                  ("ws_gate", "ss_gate"), ("ws_up", "ss_up"), ("ws_down", "ss_down")):
        if n not in q:
            continue
        v = oracle.e4m3_decode(q[n]) * q[sn][..., None].astype(np.float64)
        v32 = v.astype(np.float32)
        assert np.array_equal(v32.astype(np.float64), v)
        if to == "bf16":
            b = _bf16_bits(v32)
            assert np.array_equal(_bits_to_f32(b), v32)
            out[n] = b
        else:
            out[n] = v32
    return out


@pytest.mark.parametrize("dtype,bits", [("bf16", 0), ("f32", 12)])
def test_fp8_layer_equals_the_layer_on_dequantised_weights(dtype, bits):
    rng = np.random.default_rng(31 + bits)
    T, d, E, K, I, Is = 13, 64, 6, 2, 96, 32
    q = _fp8_layer(rng, T, d, E, I, Is, bits)
    p = _dequant(q, dtype)
    xf = rng.standard_normal((T, d)).astype(np.float32)
    wgf = (rng.standard_normal((E, d)) * d ** -0.5).astype(np.float32)
    x = _bf16_bits(xf) if dtype == "bf16" else xf
    w_g = _bf16_bits(wgf) if dtype == "bf16" else wgf
    p["w_g"] = w_g
    bias = rng.standard_normal(E) * 0.1
    toks = np.arange(T)
    ref = oracle.forward_tokens(toks, x, p, K, dtype=dtype, bias=bias)
    out = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype=dtype, bias=bias)
    for k in ("y", "topk_idx", "topk_w", "logits"):
        assert np.array_equal(out[k], ref[k]), k
    # the expert stage alone, over expert-contiguous rows
    counts, offsets, perm, _ = oracle.permute(ref["topk_idx"], E)
    x_perm = np.asarray(x)[perm // K]
    y_ref = oracle.expert_ffn(x_perm, offsets, p["w_gate"], p["w_up"], p["w_down"], dtype=dtype)
    y_q = oracle.expert_ffn_fp8(x_perm, offsets, q, dtype=dtype)
    assert np.array_equal(y_q, y_ref)


def test_fp8_layer_without_shared_expert():
    rng = np.random.default_rng(41)
    T, d, E, K, I = 9, 64, 5, 3, 128
    q = _fp8_layer(rng, T, d, E, I, 0, 0)
    p = _dequant(q, "bf16")
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    p["w_g"] = _bf16_bits((rng.standard_normal((E, d)) * 0.1).astype(np.float32))
    toks = np.array([0, 4, 8, 4])
    ref = oracle.forward_tokens(toks, x, p, K, dtype="bf16", router="sigmoid")
    out = oracle.forward_tokens_fp8(toks, x, p["w_g"], q, K, dtype="bf16", router="sigmoid")
    assert np.array_equal(out["y"], ref["y"])
