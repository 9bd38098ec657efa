"""Helpers shared by the GPU parity tests (no arithmetic of the layer here)."""
from __future__ import annotations

import os
from contextlib import contextmanager

import numpy as np
import torch

import moe_inputs as mi

MARGIN = 1e-3          # top-K boundary gap below which a token's routing is not unique
BF16_REL_L2 = 1e-2     # bf16 layer outputs vs the fp64 oracle (relative L2)
F32_MAX_REL_RMS = 1e-4 # fp32 layer outputs: max |diff| <= 1e-4 * RMS(reference)
W_RTOL = 1e-6          # routing weights (fp32 on the GPU vs fp64)


def host(t: torch.Tensor):
    return mi.to_host_array(t)


def boundary_margin(logits: np.ndarray, K: int) -> np.ndarray:
    """Gap between the K-th and (K+1)-th largest score of every row (inf if K == E)."""
    E = logits.shape[1]
    if K >= E:
        return np.full(logits.shape[0], np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, K - 1] - s[:, K]


def order_margin(keys: np.ndarray, K: int) -> np.ndarray:
    """Smallest gap between consecutive values among the K+1 largest keys of
    every row: the K picks in slot order and the boundary to the best key left
    out (among the K alone when K == E; inf when K == E == 1).  Where it is at
    least the margin, fp32 keys within half the margin of the fp64 ones select
    the same experts in the same slot order."""
    m = min(K + 1, keys.shape[1])
    if m < 2:
        return np.full(keys.shape[0], np.inf)
    s = -np.sort(-keys, axis=1)[:, :m]
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


def router_margin(cfg) -> float:
    """The key gap a sampled token must clear: 1e-3 on softmax scores; 1e-4 on
    the sigmoid router's keys, which are sigmoid(score) + bias and so squeeze
    score gaps by up to the sigmoid's slope of 1/4 (and more in its tails)."""
    return 1e-4 if getattr(cfg, "router", "softmax") == "sigmoid" else MARGIN


def clean_sample(L, n: int = 256, margin: float | None = None, chunk: int = 256):
    """A seeded sample of n tokens whose routing is unique at fp32 precision.

    Tokens are taken in a seeded random order; a token is kept when the oracle's
    fp64 keys (scores + bias, or sigmoid affinities + bias) clear `margin` in
    order_margin (the picks and their slot order), and skipped otherwise, until
    n are kept.  Returns (tokens sorted int32, skipped count)."""
    import oracle
    cfg = L.cfg
    margin = router_margin(cfg) if margin is None else margin
    order = mi.token_order(cfg.T, cfg.seed).numpy()
    kept, skipped = [], 0
    for c0 in range(0, cfg.T, chunk):
        cand = order[c0:c0 + chunk]
        xs = host(L.x[torch.from_numpy(cand).to(L.x.device)])
        _, _, keys = oracle.route(xs, L.hp["w_g"], cfg.K, dtype=cfg.dtype, bias=L.bias_host(),
                                  router=cfg.router)
        for tok, good in zip(cand.tolist(), (order_margin(keys, cfg.K) >= margin).tolist()):
            if len(kept) == n:
                break
            if good:
                kept.append(tok)
            else:
                skipped += 1
        if len(kept) == n:
            break
    return np.array(sorted(kept), dtype=np.int32), skipped


def clean_rows(L, margin: float | None = None):
    """Re-draw rows of x (deterministically) until every token's fp64 keys clear
    `margin` in order_margin: the small workloads' rule, all tokens checked."""
    import oracle
    cfg = L.cfg
    margin = router_margin(cfg) if margin is None else margin
    x = L.x
    for attempt in range(1, 20):
        _, _, keys = oracle.route(host(x), L.hp["w_g"], cfg.K, dtype=cfg.dtype,
                                  bias=L.bias_host(), router=cfg.router)
        bad = np.nonzero(order_margin(keys, cfg.K) < margin)[0]
        if bad.size == 0:
            return x
        x = mi.redraw_rows(x, bad, cfg, attempt)
    raise AssertionError("could not draw well-separated router scores")


def parity_tokens(L, n: int = 256):
    """The tokens a parity test checks: every token (rows re-drawn until each
    routing is unique; L.x is replaced) when T <= n, else clean_sample's n.
    Returns (tokens sorted int32, skipped count)."""
    if L.cfg.T <= n:
        L.x = clean_rows(L)
        return np.arange(L.cfg.T, dtype=np.int32), 0
    return clean_sample(L, n)


def gpu_route(moe, L, router=None, with_bias=True):
    """moe_route on the whole of L.x through the C ABI.  Returns (topk_idx,
    topk_w, keys) as numpy arrays; keys are the selection keys the library
    wrote to logits_out."""
    cfg = L.cfg
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype,
                       cfg.router if router is None else router)
    ws = moe.alloc_workspace(s)
    idx = torch.full((cfg.T, cfg.K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((cfg.T, cfg.K), -1.0, dtype=torch.float32, device="cuda")
    keys = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    moe.moe_route(s, L.x, L.p["w_g"], L.bias if with_bias else None, None, keys, idx, w, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    return (idx.cpu().numpy(), w.cpu().numpy().astype(np.float64),
            keys.cpu().numpy().astype(np.float64))


def assert_routing_on_sample(moe, L, tokens, ref):
    """The library's routing of the sampled tokens equals the oracle's.

    ref: the oracle's forward_tokens result for `tokens` (topk_idx, topk_w).
    - Expert ids in slot order: bit-exact (the sample clears the key margin).
    - Raw router scores x . w_g^T: within fp32 accumulation error of fp64.
    - Weights: a score error delta moves ln w_j by at most 2 max|delta| (for
      the softmax over the K picks, and for sigmoid(s) / (sum + 1e-6), whose
      log-derivative in s is 1 - sigmoid(s) <= 1), so |dw| / w <= 2 max|delta|
      plus the fp32 evaluation of the weights (2e-6).
    - Weights from the library's own fp32 scores: fed to the oracle as
      logits_in, they give the same picks and weights within 2e-6 relative
      (the routing step alone, scores fixed).
    Returns the largest raw-score error seen."""
    import oracle
    cfg = L.cfg
    tok = np.asarray(tokens, dtype=np.int64)
    idx, w, _ = gpu_route(moe, L)
    assert np.array_equal(idx[tok], ref["topk_idx"]), "expert ids or slot order differ"
    # raw scores: the softmax router without the bias writes x . w_g^T itself
    _, _, raw = gpu_route(moe, L, router="softmax", with_bias=False)
    xs = host(L.x[torch.from_numpy(tok).to(L.x.device)])
    _, _, raw_ref = oracle.route(xs, L.hp["w_g"], cfg.K, dtype=cfg.dtype)
    delta = np.abs(raw[tok] - raw_ref)
    assert np.max(delta) <= 1e-4 * max(1.0, float(np.max(np.abs(raw_ref))))
    tol = 2.0 * delta.max(axis=1, keepdims=True) + 2e-6
    assert np.all(np.abs(w[tok] - ref["topk_w"]) <= tol * ref["topk_w"]), "routing weights differ"
    idx2, w2, _ = oracle.route(None, None, cfg.K, logits_in=raw[tok].astype(np.float32),
                               bias=L.bias_host(), router=cfg.router)
    assert np.array_equal(idx2, idx[tok])
    assert np.allclose(w[tok], w2, rtol=2e-6, atol=0)
    return float(np.max(delta))


def rel_l2(a: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs_over_rms(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return float(np.max(np.abs(a - ref)) / max(rms, 1e-300))


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@contextmanager
def gemv_limit(n: int):
    """Route groups with more than n rows to the tensor-core GEMM (read per call)."""
    old = os.environ.get("MOE_GEMV_MAX_ROWS")
    os.environ["MOE_GEMV_MAX_ROWS"] = str(n)
    try:
        yield
    finally:
        if old is None:
            del os.environ["MOE_GEMV_MAX_ROWS"]
        else:
            os.environ["MOE_GEMV_MAX_ROWS"] = old


class Layer:
    """Seeded inputs of one workload on the GPU, plus host copies for the oracle."""

    def __init__(self, cfg: mi.LayerConfig, device="cuda", x=None, only=None):
        self.cfg = cfg
        self.p = mi.make_weights(cfg, device, only=only)
        self.x = mi.make_x(cfg, device) if x is None else x
        self.bias = mi.make_bias(cfg, device)
        self._host = None

    @property
    def hp(self) -> dict:
        if self._host is None:
            self._host = {k: host(v) for k, v in self.p.items()}
        return self._host

    def bias_host(self):
        return None if self.bias is None else self.bias.double().cpu().numpy()

    def oracle_tokens(self, tokens, x=None):
        """The oracle's per-token layer for these tokens (either weight format)."""
        import oracle
        c = self.cfg
        xh = host(self.x if x is None else x)
        if mi.is_fp8(c):
            return oracle.forward_tokens_fp8(tokens, xh, self.hp["w_g"], self.hp, c.K,
                                             dtype=c.dtype, bias=self.bias_host(),
                                             router=c.router, act8=c.acts == "e4m3",
                                             blocks=c.weights == "e4m3b")
        return oracle.forward_tokens(tokens, xh, self.hp, c.K, dtype=c.dtype,
                                     bias=self.bias_host(), router=c.router)

    def shape(self, moe, T=None):
        c = self.cfg
        return moe.make_shape(c.T if T is None else T, c.d, c.E, c.K, c.I, c.Is, c.dtype, c.router)

    def forward(self, moe, x=None, ws=None):
        x = self.x if x is None else x
        s = self.shape(moe, T=x.shape[0])
        y = torch.empty_like(x)
        ws = moe.alloc_workspace(s) if ws is None else ws
        p = self.p
        if self.cfg.acts == "e4m3" and self.cfg.weights == "e4m3b":
            moe.moe_forward_w8a8_blocks(s, x, p["w_g"], self.bias, moe.make_fp8_experts(p), y, ws)
        elif self.cfg.acts == "e4m3":
            moe.moe_forward_w8a8(s, x, p["w_g"], self.bias, moe.make_fp8_experts(p), y, ws)
        elif self.cfg.weights == "e4m3b":
            moe.moe_forward_fp8_blocks(s, x, p["w_g"], self.bias, moe.make_fp8_experts(p), y, ws)
        elif self.cfg.weights == "e4m3":
            moe.moe_forward_fp8(s, x, p["w_g"], self.bias, moe.make_fp8_experts(p), y, ws)
        else:
            moe.moe_forward(s, x, p["w_g"], self.bias, p["w_gate"], p["w_up"], p["w_down"],
                            p.get("ws_gate"), p.get("ws_up"), p.get("ws_down"), y, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
        return y


@contextmanager
def pair_min_rows(n: int):
    """Groups with at least n rows take the 256-row CTA-pair tiles (read per call)."""
    old = os.environ.get("MOE_PAIR_MIN_ROWS")
    os.environ["MOE_PAIR_MIN_ROWS"] = str(n)
    try:
        yield
    finally:
        if old is None:
            del os.environ["MOE_PAIR_MIN_ROWS"]
        else:
            os.environ["MOE_PAIR_MIN_ROWS"] = old
