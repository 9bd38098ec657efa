"""Pins for the fp64 oracle: each check ties it to something other than itself.

Brute force (exhaustive stable sort, dense evaluation of every expert masked by
the routing, numpy's stable argsort), closed forms (softmax of all scores when
K = E, hand-built layers whose output has a formula), special cases that reduce
to a dense SwiGLU MLP computed with library matmuls, and invariants the pages
state (selected weights sum to one; every token appears K times).  Shapes are
non-square (d != I != Is) so a transposed operand fails.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _bf16_bits(a):
    return mi.to_host_array(torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16))


def _as_f64(a, dtype):
    """The exact stored values as float64 (bf16 bit patterns widened)."""
    a = np.asarray(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _rand_layer(rng, T, d, E, I, Is, dtype):
    def mk(*shape, std=1.0):
        v = (rng.standard_normal(shape) * std).astype(np.float32)
        return _bf16_bits(v) if dtype == "bf16" else v
    p = {"w_g": mk(E, d, std=d ** -0.5), "w_gate": mk(E, I, d, std=d ** -0.5),
         "w_up": mk(E, I, d, std=d ** -0.5), "w_down": mk(E, d, I, std=I ** -0.5)}
    if Is:
        p.update(ws_gate=mk(Is, d, std=d ** -0.5), ws_up=mk(Is, d, std=d ** -0.5),
                 ws_down=mk(d, Is, std=Is ** -0.5))
    return mk(T, d), p


def _expert_dense(xt, wg, wu, wd):
    """SwiGLU with numpy matmuls: W_down @ (SiLU(W_gate @ x) * (W_up @ x))."""
    return wd @ (_silu(wg @ xt) * (wu @ xt))


# ---------------------------------------------------------------- selection

def _brute_topk(s, K):
    """Full stable sort by (-score, index); first K."""
    order = np.lexsort((np.arange(s.shape[0]), -s))
    return order[:K]


@pytest.mark.parametrize("T,E,K,scale", [(64, 8, 2, 512), (50, 256, 8, 512), (40, 256, 8, 2),
                                         (33, 64, 64, 8), (17, 1024, 32, 4), (9, 1, 1, 8),
                                         (31, 20, 7, 1)])
def test_topk_matches_exhaustive_sort(T, E, K, scale):
    logits = mi.grid_logits(T, E, seed=3, scale=scale).numpy()
    idx, w, used = oracle.route(None, None, K, logits_in=logits)
    assert np.array_equal(used, logits.astype(np.float64))
    for t in range(T):
        s = logits[t].astype(np.float64)
        ref = _brute_topk(s, K)
        assert np.array_equal(idx[t], ref), (t, idx[t], ref)
        # softmax over only the K selected scores (library routine)
        assert np.allclose(w[t], scipy.special.softmax(s[ref]), rtol=1e-14, atol=1e-16)


def test_ties_go_to_lower_index_and_signed_zero_is_a_tie():
    s = np.array([[0.5, -0.0, 0.5, 0.0, 0.25, 0.5]], np.float32)
    idx, w, _ = oracle.route(None, None, 5, logits_in=s)
    assert idx[0].tolist() == [0, 2, 5, 4, 1]      # -0.0 == +0.0 -> index 1 before 3
    idx, _, _ = oracle.route(None, None, 6, logits_in=s)
    assert idx[0].tolist() == [0, 2, 5, 4, 1, 3]


def test_K_equals_E_is_full_softmax():
    logits = mi.grid_logits(12, 16, seed=5, scale=64).numpy()
    idx, w, _ = oracle.route(None, None, 16, logits_in=logits)
    for t in range(12):
        s = logits[t].astype(np.float64)
        # every expert selected; the weight of expert e is softmax(s)[e]
        full = scipy.special.softmax(s)
        assert sorted(idx[t].tolist()) == list(range(16))
        assert np.allclose(w[t], full[idx[t]], rtol=1e-14)


def test_K1_weight_is_one():
    logits = mi.grid_logits(20, 8, seed=7).numpy()
    idx, w, _ = oracle.route(None, None, 1, logits_in=logits)
    assert np.all(w == 1.0)
    assert np.array_equal(idx[:, 0], np.argmax(logits, axis=1))


def test_weights_sum_to_one():
    # explainer section 2.2: the K softmax weights sum to 1
    logits = mi.grid_logits(200, 256, seed=9).numpy()
    _, w, _ = oracle.route(None, None, 8, logits_in=logits)
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-15
    assert np.all(w > 0) and np.all(np.diff(w, axis=1) <= 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_input_ties_everything(dtype):
    T, d, E, K = 6, 32, 12, 4
    rng = np.random.default_rng(0)
    x, p = _rand_layer(rng, T, d, E, 48, 0, dtype)
    x = np.zeros_like(x)
    idx, w, logits = oracle.route(x, p["w_g"], K, dtype=dtype)
    assert np.all(logits == 0.0)
    assert np.array_equal(idx, np.tile(np.arange(K, dtype=np.int32), (T, 1)))
    assert np.allclose(w, 1.0 / K, rtol=0, atol=1e-16)


def test_scores_are_x_times_wg_transposed():
    rng = np.random.default_rng(1)
    for dtype in ("f32", "bf16"):
        x, p = _rand_layer(rng, 7, 40, 9, 16, 0, dtype)
        _, _, logits = oracle.route(x, p["w_g"], 3, dtype=dtype)
        ref = torch.from_numpy(_as_f64(x, dtype)) @ torch.from_numpy(_as_f64(p["w_g"], dtype)).T
        assert np.allclose(logits, ref.numpy(), rtol=1e-13, atol=1e-13)


def test_bias_enters_selection_and_weights():
    s = np.array([[1.0, 0.5, 0.25, 0.0]], np.float32)
    x = np.array([[1.0]], np.float32)
    w_g = s.T.copy()                                   # scores = x . w_g^T = s
    bias = np.array([0.0, 0.0, 2.0, 0.0])
    idx, w, logits = oracle.route(x, w_g, 2, dtype="f32", bias=bias)
    assert np.allclose(logits[0], [1.0, 0.5, 2.25, 0.0])
    assert idx[0].tolist() == [2, 0]
    e = math.exp(1.0 - 2.25)
    assert np.allclose(w[0], [1 / (1 + e), e / (1 + e)], rtol=1e-15)


# ---------------------------------------------------------------- permutation

@pytest.mark.parametrize("T,E,K", [(64, 8, 2), (8, 256, 8), (128, 256, 8), (1, 4, 4),
                                   (0, 5, 2), (37, 3, 3), (300, 1, 1)])
def test_permutation_is_the_stable_expert_order(T, E, K):
    logits = mi.grid_logits(max(T, 1), E, seed=11, scale=4).numpy()[:T]
    idx, _, _ = oracle.route(None, None, K, logits_in=logits.reshape(T, E))
    counts, offsets, perm, inv = oracle.permute(idx, E)
    flat = idx.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[E] == T * K
    assert np.array_equal(np.diff(offsets), counts)
    # numpy's stable sort by expert id gives the same order
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(np.sort(perm), np.arange(T * K))
    assert np.array_equal(inv[perm], np.arange(T * K))
    # every token appears exactly K times
    assert np.array_equal(np.bincount(perm // K, minlength=T) if T else np.zeros(0), np.full(T, K))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ---------------------------------------------------------------- the layer

def _dense_masked(x, p, K, dtype, bias=None):
    """Evaluate every expert on every token and keep the routed ones."""
    xs = _as_f64(x, dtype)
    P = {k: _as_f64(v, dtype) for k, v in p.items()}
    T, d = xs.shape
    E = P["w_g"].shape[0]
    y = np.zeros((T, d))
    for t in range(T):
        s = P["w_g"] @ xs[t] + (0 if bias is None else bias)
        sel = _brute_topk(s, K)
        wsel = scipy.special.softmax(s[sel])
        mask = np.zeros(E)
        mask[sel] = wsel
        acc = np.zeros(d)
        if "ws_gate" in P:
            acc += _expert_dense(xs[t], P["ws_gate"], P["ws_up"], P["ws_down"])
        for e in range(E):
            acc += mask[e] * _expert_dense(xs[t], P["w_gate"][e], P["w_up"][e], P["w_down"][e])
        y[t] = acc
    return y


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,d,E,K,I,Is", [(9, 24, 6, 3, 40, 16), (5, 16, 4, 4, 8, 0),
                                          (12, 32, 7, 1, 24, 56)])
def test_forward_matches_dense_masked_evaluation(dtype, T, d, E, K, I, Is):
    rng = np.random.default_rng(T * 1000 + d)
    x, p = _rand_layer(rng, T, d, E, I, Is, dtype)
    bias = rng.standard_normal(E) * 0.1
    out = oracle.forward(x, p, K, dtype=dtype, bias=bias)
    ref = _dense_masked(x, p, K, dtype, bias=bias)
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(out["y"] - ref)) <= 1e-12 * scale
    tok = oracle.forward_tokens(np.arange(T), x, p, K, dtype=dtype, bias=bias)
    assert np.max(np.abs(tok["y"] - ref)) <= 1e-12 * scale
    assert np.array_equal(tok["topk_idx"], out["topk_idx"])


def test_single_expert_is_a_dense_swiglu_mlp():
    rng = np.random.default_rng(5)
    T, d, I = 11, 48, 80
    x, p = _rand_layer(rng, T, d, 1, I, 0, "f32")
    out = oracle.forward(x, p, 1, dtype="f32")
    X = torch.from_numpy(x.astype(np.float64))
    Wg, Wu, Wd = (torch.from_numpy(p[k][0].astype(np.float64)) for k in ("w_gate", "w_up", "w_down"))
    ref = (torch.nn.functional.silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T
    assert np.allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_identical_experts_make_routing_irrelevant():
    rng = np.random.default_rng(6)
    T, d, E, K, I, Is = 10, 24, 5, 3, 32, 8
    x, p = _rand_layer(rng, T, d, E, I, Is, "f32")
    for k in ("w_gate", "w_up", "w_down"):
        p[k] = np.repeat(p[k][:1], E, axis=0)
    out = oracle.forward(x, p, K, dtype="f32")
    xs = x.astype(np.float64)
    one = np.stack([_expert_dense(xs[t], p["w_gate"][0].astype(np.float64),
                                  p["w_up"][0].astype(np.float64),
                                  p["w_down"][0].astype(np.float64)) for t in range(T)])
    sh = np.stack([_expert_dense(xs[t], p["ws_gate"].astype(np.float64),
                                 p["ws_up"].astype(np.float64),
                                 p["ws_down"].astype(np.float64)) for t in range(T)])
    assert np.allclose(out["y"], one + sh, rtol=1e-12, atol=1e-13)


def test_combine_is_linear_in_the_weights():
    rng = np.random.default_rng(7)
    T, d, K = 6, 10, 3
    y_perm = rng.standard_normal((T * K, d))
    inv = rng.permutation(T * K).astype(np.int32)
    w = rng.random((T, K))
    a = oracle.combine(y_perm, inv, w)
    b = oracle.combine(y_perm, inv, 2.5 * w)
    assert np.allclose(b, 2.5 * a, rtol=1e-14)
    ys = rng.standard_normal((T, d))
    c = oracle.combine(y_perm, inv, w, ys)
    assert np.allclose(c - ys, a, rtol=1e-13, atol=1e-14)
    for t in range(T):
        ref = sum(w[t, j] * y_perm[inv[t * K + j]] for j in range(K))
        assert np.allclose(a[t], ref, rtol=1e-14)


def test_token_order_equivariance():
    rng = np.random.default_rng(8)
    T = 14
    x, p = _rand_layer(rng, T, 16, 6, 24, 12, "bf16")
    q = rng.permutation(T)
    a = oracle.forward(x, p, 2, dtype="bf16")["y"]
    b = oracle.forward(x[q], p, 2, dtype="bf16")["y"]
    assert np.array_equal(a[q], b)


def test_zero_tokens_and_zero_input():
    rng = np.random.default_rng(9)
    x, p = _rand_layer(rng, 4, 16, 5, 24, 8, "f32")
    out = oracle.forward(np.zeros((4, 16), np.float32), p, 2, dtype="f32")
    assert np.all(out["y"] == 0.0)
    empty = oracle.forward(np.zeros((0, 16), np.float32), p, 2, dtype="f32")
    assert empty["y"].shape == (0, 16) and np.all(empty["counts"] == 0)


def test_hand_built_layer_closed_form():
    """d=2, E=3, K=2, I=1: scores (2, 1, 0) select experts 0 and 1 with weights
    e/(1+e) and 1/(1+e); expert e outputs (c_e * SiLU(a_e), 0)."""
    x = np.array([[1.0, 0.0]], np.float32)
    a, c = [1.0, -1.0, 3.0], [1.0, 2.0, 5.0]
    p = {"w_g": np.array([[2.0, 0.0], [1.0, 0.0], [0.0, 0.0]], np.float32),
         "w_gate": np.array([[[ai, 0.0]] for ai in a], np.float32),
         "w_up": np.array([[[1.0, 0.0]] for _ in a], np.float32),
         "w_down": np.array([[[ci], [0.0]] for ci in c], np.float32)}
    out = oracle.forward(x, p, 2, dtype="f32")
    e = math.e
    w0, w1 = e / (1 + e), 1 / (1 + e)
    silu = lambda z: z / (1 + math.exp(-z))  # noqa: E731
    expect = w0 * c[0] * silu(a[0]) + w1 * c[1] * silu(a[1])
    assert out["topk_idx"][0].tolist() == [0, 1]
    assert abs(out["topk_w"][0][0] - w0) < 1e-16 and abs(out["topk_w"][0][1] - w1) < 1e-16
    assert abs(out["y"][0][0] - expect) < 1e-15 and out["y"][0][1] == 0.0
    # with a shared expert (Is=1): adds SiLU(1) * 1 * 1 on column 0
    p.update(ws_gate=np.array([[1.0, 0.0]], np.float32), ws_up=np.array([[1.0, 0.0]], np.float32),
             ws_down=np.array([[1.0], [0.0]], np.float32))
    out = oracle.forward(x, p, 2, dtype="f32")
    assert abs(out["y"][0][0] - (expect + silu(1.0))) < 1e-15


# ---------------------------------------------------------------- sigmoid router (DeepSeek-V3)

def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


@pytest.mark.parametrize("T,E,K,scale", [(50, 256, 8, 512), (40, 64, 6, 4), (9, 8, 8, 8), (20, 5, 1, 2)])
def test_sigmoid_router_matches_brute_force(T, E, K, scale):
    logits = mi.grid_logits(T, E, seed=31, scale=scale).numpy()
    bias = np.round(np.random.default_rng(3).standard_normal(E) * 8) / 32
    idx, w, keys = oracle.route(None, None, K, logits_in=logits, bias=bias, router="sigmoid")
    for t in range(T):
        a = _sigmoid(logits[t].astype(np.float64))
        key = a + bias
        assert np.allclose(keys[t], key, rtol=0, atol=1e-15)
        ref = _brute_topk(key, K)
        assert np.array_equal(idx[t], ref)
        assert np.allclose(w[t], a[ref] / (a[ref].sum() + 1e-6), rtol=1e-14)


def test_sigmoid_bias_steers_selection_but_not_weights():
    s = np.array([[2.0, 1.0, 0.5, -1.0]], np.float32)
    bias = np.array([0.0, 0.0, 0.0, 5.0])
    idx, w, _ = oracle.route(None, None, 2, logits_in=s, bias=bias, router="sigmoid")
    assert idx[0].tolist() == [3, 0]          # the bias lifts expert 3 into the top 2
    a3, a0 = 1 / (1 + math.exp(1.0)), 1 / (1 + math.exp(-2.0))
    assert np.allclose(w[0], [a3 / (a3 + a0 + 1e-6), a0 / (a3 + a0 + 1e-6)], rtol=1e-15)
    assert w[0].sum() < 1.0                   # a / (sum a + 1e-6) sums to just under 1


def test_sigmoid_zero_input_ties_everything():
    rng = np.random.default_rng(12)
    x, p = _rand_layer(rng, 5, 32, 12, 16, 0, "f32")
    idx, w, keys = oracle.route(np.zeros_like(x), p["w_g"], 4, dtype="f32", router="sigmoid")
    assert np.all(keys == 0.5)
    assert np.array_equal(idx, np.tile(np.arange(4, dtype=np.int32), (5, 1)))
    assert np.allclose(w, 0.5 / (4 * 0.5 + 1e-6), rtol=1e-15)


def _dense_masked_sigmoid(x, p, K, dtype, bias):
    xs = _as_f64(x, dtype)
    P = {k: _as_f64(v, dtype) for k, v in p.items()}
    T, d = xs.shape
    E = P["w_g"].shape[0]
    y = np.zeros((T, d))
    for t in range(T):
        a = _sigmoid(P["w_g"] @ xs[t])
        sel = _brute_topk(a + bias, K)
        mask = np.zeros(E)
        mask[sel] = a[sel] / (a[sel].sum() + 1e-6)
        acc = np.zeros(d)
        if "ws_gate" in P:
            acc += _expert_dense(xs[t], P["ws_gate"], P["ws_up"], P["ws_down"])
        for e in range(E):
            acc += mask[e] * _expert_dense(xs[t], P["w_gate"][e], P["w_up"][e], P["w_down"][e])
        y[t] = acc
    return y


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sigmoid_forward_matches_dense_masked_evaluation(dtype):
    rng = np.random.default_rng(13)
    T, d, E, K, I, Is = 9, 24, 6, 3, 40, 16
    x, p = _rand_layer(rng, T, d, E, I, Is, dtype)
    bias = rng.standard_normal(E) * 0.3
    out = oracle.forward(x, p, K, dtype=dtype, bias=bias, router="sigmoid")
    ref = _dense_masked_sigmoid(x, p, K, dtype, bias)
    assert np.max(np.abs(out["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))
    tok = oracle.forward_tokens(np.arange(T), x, p, K, dtype=dtype, bias=bias, router="sigmoid")
    assert np.max(np.abs(tok["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))
