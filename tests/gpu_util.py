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
        if c.weights == "e4m3":
            return oracle.forward_tokens_fp8(tokens, xh, self.hp["w_g"], self.hp, c.K,
                                             dtype=c.dtype, bias=self.bias_host(),
                                             router=c.router, act8=c.acts == "e4m3")
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
        if self.cfg.acts == "e4m3":
            moe.moe_forward_w8a8(s, x, p["w_g"], self.bias, moe.make_fp8_experts(p), y, ws)
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
