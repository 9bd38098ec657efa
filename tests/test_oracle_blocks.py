"""Pins for the oracle's block-scaled 8-bit weights (the *_blocks functions):
one fp32 scale per 128 x 128 block of the stacked weight matrix, the "per
group" granularity of the "make every byte cheaper" section in the square
blocks of DeepSeek-V3's 8-bit checkpoints.

Each piece is tied to something other than the oracle:
  - the quantiser: per block, PyTorch's float32 amax / 448 and its
    float8_e4m3fn cast of w / scale, bit for bit, including ragged edge blocks;
  - the block accessor: with scales whose products with every code are exact,
    the layer (and the expert stage) on block-scaled codes equals the pinned
    layer on the weights dequantised in numpy (the scale grid expanded with
    np.kron), bit for bit -- a transposed block index, a wrong row length or
    blocks taken per expert instead of over the stacked matrix all change it;
  - the two formats: when every row of a 128-row block has the same amax in
    every 128-column block, row and block quantisation give the same codes and
    scales, and the two layers agree bit for bit;
  - the two-plane form and the W8A8 form (x and h quantised per row): each
    step matches PyTorch's casts and numpy products with the expanded scales.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_a2 import _torch_planes
from tests.test_oracle_fp8 import _bf16_bits, _bits_to_f32
from tests.test_oracle_w8a8 import _torch_bf16

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

B = 128


def _expand(s, rows, cols):
    """The scale of every element of a [rows][cols] matrix from its block grid."""
    return np.kron(np.asarray(s, np.float64), np.ones((B, B)))[:rows, :cols]


def _torch_block_quant(w32):
    """Block quantisation with PyTorch: per block, scale = amax / 448 in float32
    (1 for a block of zeros) and the float8_e4m3fn cast of w / scale."""
    rows, cols = w32.shape
    t = torch.from_numpy(np.ascontiguousarray(w32, np.float32))
    nbr, nbc = -(-rows // B), -(-cols // B)
    codes = np.zeros((rows, cols), np.uint8)
    scales = np.zeros((nbr, nbc), np.float32)
    for br in range(nbr):
        for bc in range(nbc):
            blk = t[br * B:(br + 1) * B, bc * B:(bc + 1) * B]
            amax = blk.abs().max()
            s = amax / 448.0 if amax > 0 else torch.tensor(1.0, dtype=torch.float32)
            codes[br * B:(br + 1) * B, bc * B:(bc + 1) * B] = (
                (blk / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
            scales[br, bc] = s.item()
    return codes, scales


def _matrix(seed, rows, cols):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((rows, cols)) * np.exp2(rng.uniform(-10, 6, (rows, 1)))
    w *= np.exp2(rng.uniform(-4, 4, (1, cols)))
    w[:B, :B] = 0.0                                   # a block of zeros
    w[rows - 1, cols - 1] = -np.abs(w).max() * 3      # a negative extreme in the corner block
    return w.astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(300, 200), (256, 384), (128, 128), (7, 130)])
def test_block_codes_and_scales_match_torch(dtype, shape):
    w = _matrix(sum(shape), *shape)
    stored = _bf16_bits(w) if dtype == "bf16" else w
    wv = _bits_to_f32(stored) if dtype == "bf16" else w
    codes, scales = oracle.quantize_fp8_blocks(stored, dtype)
    tc, ts = _torch_block_quant(wv)
    assert scales.shape == ts.shape
    assert np.array_equal(scales, ts)
    assert np.array_equal(codes, tc)
    if shape[0] >= B and shape[1] >= B:
        assert scales[0, 0] == 1.0 and np.all(codes[:B, :B] & 0x7F == 0)


def test_block_quantiser_meets_the_format_error_bound():
    rows, cols = 384, 320
    w = _matrix(5, rows, cols)
    codes, scales = oracle.quantize_fp8_blocks(w, "f32")
    dec = oracle.e4m3_decode(codes)
    assert not np.isnan(dec).any()
    # every non-zero block reaches the largest finite code exactly once or more
    for br in range(scales.shape[0]):
        for bc in range(scales.shape[1]):
            blk = dec[br * B:(br + 1) * B, bc * B:(bc + 1) * B]
            if scales[br, bc] != 1.0 or np.abs(blk).max() > 0:
                assert np.abs(blk).max() == 448.0
    q = w.astype(np.float64) / _expand(scales, rows, cols)
    err = np.abs(dec - q)
    normal = np.abs(q) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(q[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * (1 + 1e-6))
    # on rows of one range whose column blocks differ in range, a scale per
    # block keeps the small blocks' values off the subnormal steps that a scale
    # per row pushes them onto
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((rows, cols)) *
         np.repeat(np.exp2([0.0, -10.0, -18.0]), B)[:cols]).astype(np.float32)
    bc, bs = oracle.quantize_fp8_blocks(v, "f32")
    rc, rs = oracle.quantize_fp8_rows(v, "f32")
    small = slice(2 * B, cols)
    rel = lambda e: np.linalg.norm(e[:, small]) / np.linalg.norm(v[:, small])  # noqa: E731
    e_blk = oracle.e4m3_decode(bc) * _expand(bs, rows, cols) - v
    e_row = oracle.e4m3_decode(rc) * rs[:, None].astype(np.float64) - v
    assert rel(e_blk) < 2.0 ** -4 < 4 * rel(e_blk) < rel(e_row)


def _codes(rng, *shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] ^= 0x01       # NaN -> a finite neighbour
    return c


def _scales(rng, rows, cols, exact_bits):
    """Block scales whose significands have at most exact_bits bits (0: powers of
    two), so every code * scale is exact in fp32 (<= 20 bits) or bf16 (0)."""
    shape = (-(-rows // B), -(-cols // B))
    e = rng.integers(-12, -4, size=shape)
    m = rng.integers(1 << exact_bits, 2 << exact_bits, size=shape) if exact_bits else 1
    return (np.ldexp(np.float64(1), e) * m / (1 << exact_bits)).astype(np.float32)


def _block_layer(rng, d, E, I, Is, exact_bits):
    q = {"w_gate": _codes(rng, E, I, d), "w_up": _codes(rng, E, I, d), "w_down": _codes(rng, E, d, I),
         "s_gate": _scales(rng, E * I, d, exact_bits), "s_up": _scales(rng, E * I, d, exact_bits),
         "s_down": _scales(rng, E * d, I, exact_bits)}
    if Is:
        q.update(ws_gate=_codes(rng, Is, d), ws_up=_codes(rng, Is, d), ws_down=_codes(rng, d, Is),
                 ss_gate=_scales(rng, Is, d, exact_bits), ss_up=_scales(rng, Is, d, exact_bits),
                 ss_down=_scales(rng, d, Is, exact_bits))
    return q


def _dequant_blocks(q, name):
    """value(code) * its block's scale, computed on the stacked [rows][cols] matrix."""
    sn = "s" + name[1:] if name.startswith("w_") else "ss" + name[2:]
    c = q[name]
    cols = c.shape[-1]
    rows = c.size // cols
    v = oracle.e4m3_decode(c.reshape(rows, cols)) * _expand(q[sn], rows, cols)
    return v.reshape(c.shape)


def _as(v, to):
    v32 = v.astype(np.float32)
    assert np.array_equal(v32.astype(np.float64), v)
    if to == "bf16":
        b = _bf16_bits(v32)
        assert np.array_equal(_bits_to_f32(b), v32)
        return b
    return v32


@pytest.mark.parametrize("dtype,bits,d,I,Is", [
    ("bf16", 0, 256, 384, 128),   # every block inside one expert
    ("f32", 12, 256, 384, 0),
    ("bf16", 0, 192, 320, 64),    # ragged: blocks straddle experts of the stacked matrix
])
def test_block_layer_equals_the_layer_on_dequantised_weights(dtype, bits, d, I, Is):
    rng = np.random.default_rng(50 + bits + d)
    T, E, K = 9, 3, 2
    q = _block_layer(rng, d, E, I, Is, bits)
    p = {n: _as(_dequant_blocks(q, n), dtype) for n in
         ("w_gate", "w_up", "w_down") + (("ws_gate", "ws_up", "ws_down") if Is else ())}
    xf = rng.standard_normal((T, d)).astype(np.float32)
    wgf = (rng.standard_normal((E, d)) * d ** -0.5).astype(np.float32)
    x = _bf16_bits(xf) if dtype == "bf16" else xf
    w_g = _bf16_bits(wgf) if dtype == "bf16" else wgf
    p["w_g"] = w_g
    bias = rng.standard_normal(E) * 0.1
    toks = np.arange(T)
    ref = oracle.forward_tokens(toks, x, p, K, dtype=dtype, bias=bias)
    out = oracle.forward_tokens_fp8(toks, x, w_g, q, K, dtype=dtype, bias=bias, blocks=True)
    for k in ("y", "topk_idx", "topk_w", "logits"):
        assert np.array_equal(out[k], ref[k]), k
    counts, offsets, perm, _ = oracle.permute(ref["topk_idx"], E)
    x_perm = np.asarray(x)[perm // K]
    y_ref = oracle.expert_ffn(x_perm, offsets, p["w_gate"], p["w_up"], p["w_down"], dtype=dtype)
    y_q = oracle.expert_ffn_fp8(x_perm, offsets, q, dtype=dtype, blocks=True)
    assert np.array_equal(y_q, y_ref)


def _one_amax_per_row_block(seed, rows, cols):
    """Weights whose every row, and every 128 x 128 block, has the same largest
    magnitude A_b (one per block of 128 rows, a different one for each)."""
    rng = np.random.default_rng(seed)
    nbr = -(-rows // B)
    A = np.exp2(rng.uniform(-6, 2, nbr)).astype(np.float32)
    w = np.empty((rows, cols), np.float32)
    for r in range(rows):
        a = A[r // B]
        w[r] = rng.uniform(-0.9, 0.9, cols) * a
        for c0 in range(0, cols, B):
            nc = min(B, cols - c0)
            w[r, c0 + r % nc] = a if (r + c0) % 3 else -a
    return w


def test_block_and_row_formats_agree_when_each_row_block_has_one_amax():
    T, d, E, K, I, Is = 6, 256, 2, 2, 256, 128
    rng = np.random.default_rng(61)
    q_row, q_blk = {}, {}
    for n, shape in (("w_gate", (E, I, d)), ("w_up", (E, I, d)), ("w_down", (E, d, I)),
                     ("ws_gate", (Is, d)), ("ws_up", (Is, d)), ("ws_down", (d, Is))):
        rows = int(np.prod(shape[:-1]))
        w = _bf16_bits(_one_amax_per_row_block(len(q_row) + 70, rows, shape[-1]))
        sn = "s" + n[1:] if n.startswith("w_") else "ss" + n[2:]
        rc, rs = oracle.quantize_fp8_rows(w, "bf16")
        bc, bs = oracle.quantize_fp8_blocks(w, "bf16")
        assert np.array_equal(rc, bc)
        assert np.array_equal(_expand(bs, rows, shape[-1]), np.repeat(rs[:, None], shape[-1], 1))
        q_row[n], q_row[sn] = rc.reshape(shape), rs.reshape(shape[:-1])
        q_blk[n], q_blk[sn] = bc.reshape(shape), bs
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.1).astype(np.float32))
    toks = np.arange(T)
    a = oracle.forward_tokens_fp8(toks, x, w_g, q_row, K)
    b = oracle.forward_tokens_fp8(toks, x, w_g, q_blk, K, blocks=True)
    assert np.array_equal(a["y"], b["y"]) and np.abs(a["y"]).max() > 0
    a2 = oracle.forward_tokens_fp8(toks, x, w_g, q_row, K, act8="planes")
    b2 = oracle.forward_tokens_fp8(toks, x, w_g, q_blk, K, act8="planes", blocks=True)
    assert np.array_equal(a2["y"], b2["y"])
    a8 = oracle.forward_tokens_fp8(toks, x, w_g, q_row, K, act8=True)
    b8 = oracle.forward_tokens_fp8(toks, x, w_g, q_blk, K, act8=True, blocks=True)
    assert np.array_equal(a8["y"], b8["y"])


@pytest.mark.parametrize("seed,rows", [(1, [3, 0, 5, 1]), (2, [7, 2])])
def test_a2_blocks_expert_matches_library_casts_at_every_step(seed, rows):
    rng = np.random.default_rng(seed)
    d, I = 256, 384
    E = len(rows)
    q = _block_layer(rng, d, E, I, 0, 12)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(offsets[-1])
    xf = (rng.standard_normal((R, d)) * np.exp2(rng.uniform(-3, 3, (R, 1)))).astype(np.float32)
    x = _bf16_bits(xf)
    y, h_pre, h_hat = oracle.expert_ffn_a2(x, offsets, q, "bf16", taps=True, blocks=True)
    wg, wu, wd = (_dequant_blocks(q, n) for n in ("w_gate", "w_up", "w_down"))
    xt = _torch_planes(_bits_to_f32(x))[3]
    for e in range(E):
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        if sl.start == sl.stop:
            continue
        g = xt[sl] @ wg[e].T
        u = xt[sl] @ wu[e].T
        with np.errstate(over="ignore"):  # exp(-g) = inf for g << 0 gives SiLU(g) = -0
            h_ref = g / (1.0 + np.exp(-g)) * u
        assert np.abs(h_pre[sl] - h_ref).max() <= 1e-12 * max(np.abs(h_ref).max(), 1e-300)
        assert np.array_equal(h_hat[sl], _torch_planes(_torch_bf16(h_pre[sl]))[3])
        y_ref = h_hat[sl] @ wd[e].T
        assert np.abs(y[sl] - y_ref).max() <= 1e-12 * max(np.abs(y_ref).max(), 1e-300)


def test_a2_blocks_token_forward_matches_the_expert_stage():
    rng = np.random.default_rng(7)
    T, d, E, K, I, Is = 7, 256, 3, 2, 256, 128
    q = _block_layer(rng, d, E, I, Is, 12)
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.2).astype(np.float32))
    out = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, act8="planes", blocks=True)
    counts, offsets, perm, inv = oracle.permute(out["topk_idx"], E)
    y_perm = oracle.expert_ffn_a2(np.asarray(x)[perm // K], offsets, q, blocks=True)
    shared = {"w_gate": q["ws_gate"][None], "w_up": q["ws_up"][None],
              "w_down": q["ws_down"][None], "s_gate": q["ss_gate"], "s_up": q["ss_up"],
              "s_down": q["ss_down"]}
    y_s = oracle.expert_ffn_a2(x, np.array([0, T], np.int32), shared, blocks=True)
    y = oracle.combine(y_perm, inv, out["topk_w"], y_s)
    assert np.allclose(y, out["y"], rtol=0, atol=1e-12 * np.abs(y).max())
    # and the exact 8-bit-weight layer is within the two planes' reading of it
    ex = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, blocks=True)
    assert np.linalg.norm(out["y"] - ex["y"]) < 5e-3 * np.linalg.norm(ex["y"])


# ---------------------------------------------------------------- W8A8 on block-scaled weights

@pytest.mark.parametrize("seed,rows", [(3, [3, 0, 5, 1]), (4, [7, 2])])
def test_w8a8_blocks_expert_matches_library_quantisation_at_every_step(seed, rows):
    """x and h quantised per row (torch's float8 cast of v / (amax / 448)), the
    weights dequantised per 128 x 128 block in numpy: h before rounding, h_hat
    and y equal the oracle's taps."""
    from tests.test_oracle_w8a8 import _torch_quant_rows
    rng = np.random.default_rng(seed)
    d, I = 256, 384
    E = len(rows)
    q = _block_layer(rng, d, E, I, 0, 12)
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(offsets[-1])
    xf = (rng.standard_normal((R, d)) * np.exp2(rng.uniform(-3, 3, (R, 1)))).astype(np.float32)
    x = _bf16_bits(xf)
    y, h_pre, h_hat = oracle.expert_ffn_w8a8(x, offsets, q, "bf16", taps=True, blocks=True)
    wg, wu, wd = (_dequant_blocks(q, n) for n in ("w_gate", "w_up", "w_down"))
    xh = _torch_quant_rows(_bits_to_f32(x))
    for e in range(E):
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        if sl.start == sl.stop:
            continue
        g = xh[sl] @ wg[e].T
        u = xh[sl] @ wu[e].T
        with np.errstate(over="ignore"):
            h_ref = g / (1.0 + np.exp(-g)) * u
        assert np.abs(h_pre[sl] - h_ref).max() <= 1e-12 * max(np.abs(h_ref).max(), 1e-300)
        assert np.array_equal(h_hat[sl], _torch_quant_rows(_torch_bf16(h_pre[sl])))
        y_ref = h_hat[sl] @ wd[e].T
        assert np.abs(y[sl] - y_ref).max() <= 1e-12 * max(np.abs(y_ref).max(), 1e-300)


def test_w8a8_blocks_token_forward_matches_the_expert_stage():
    rng = np.random.default_rng(8)
    T, d, E, K, I, Is = 7, 256, 3, 2, 256, 128
    q = _block_layer(rng, d, E, I, Is, 12)
    x = _bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    w_g = _bf16_bits((rng.standard_normal((E, d)) * 0.2).astype(np.float32))
    out = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, act8=True, blocks=True)
    counts, offsets, perm, inv = oracle.permute(out["topk_idx"], E)
    y_perm = oracle.expert_ffn_w8a8(np.asarray(x)[perm // K], offsets, q, blocks=True)
    shared = {"w_gate": q["ws_gate"][None], "w_up": q["ws_up"][None],
              "w_down": q["ws_down"][None], "s_gate": q["ss_gate"], "s_up": q["ss_up"],
              "s_down": q["ss_down"]}
    y_s = oracle.expert_ffn_w8a8(x, np.array([0, T], np.int32), shared, blocks=True)
    y = oracle.combine(y_perm, inv, out["topk_w"], y_s)
    assert np.allclose(y, out["y"], rtol=0, atol=1e-12 * np.abs(y).max())
    # the activations' E4M3 noise moves the output off the exact 8-bit-weight layer
    ex = oracle.forward_tokens_fp8(np.arange(T), x, w_g, q, K, blocks=True)
    assert np.linalg.norm(out["y"] - ex["y"]) > 1e-2 * np.linalg.norm(ex["y"])
