"""fp64 CPU oracle for one sparse MoE FFN layer forward -- TEST INFRASTRUCTURE.

Only the tests, the package smoke check and the benchmark's CPU-baseline arm may
import this module.  The GPU library never imports, links or calls it, and it
never imports the GPU library: the two share no code.  The arithmetic lives in
``moe_oracle.c`` (plain C, double precision on the exact stored inputs); this
file compiles it with gcc and marshals numpy arrays through ctypes.

Every function here follows the definitions cited in ``moe_oracle.c``:
router scores, top-K with ties to the lower expert index, softmax over the K
selected scores, a stable counting-sort permutation with exclusive offsets, the
SwiGLU expert FFN and the weighted combine plus the shared expert.

Inputs: ``dtype`` is ``"f32"`` (numpy float32 arrays) or ``"bf16"`` (numpy
uint16 arrays holding bf16 bit patterns).  Outputs are float64 / int32 numpy
arrays.  8-bit expert weights are numpy uint8 arrays of E4M3 codes with one
float32 scale per weight row (``*_fp8`` functions); the ``*_w8a8`` functions
also quantise the experts' input and hidden rows to E4M3, one scale per row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {"f32": 0, "bf16": 1}
# router: "softmax" = softmax over the K selected scores (+ bias);
# "sigmoid" = DeepSeek-V3 affinities, bias for selection only, a / (sum a + 1e-6)
_ROUTER = {"softmax": 0, "sigmoid": 1}


def compile_c(src: str, out: str) -> str:
    """gcc, no -ffast-math and no FMA contraction, so results match across x86
    and Arm hosts."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_oracle(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it when it is stale."""
    stale = force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if stale:
        compile_c(_SRC, _LIB_PATH)
    return _LIB_PATH


def bind(lib):
    """Declare the C signatures on a loaded liboracle handle."""
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_default_threads.restype = i32
    lib.oracle_route.argtypes = [i64, i64, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, i32]
    lib.oracle_permute.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
    lib.oracle_expert_ffn.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, vp, i32]
    lib.oracle_combine.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
    lib.oracle_shared_ffn.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp, i32]
    lib.oracle_forward.argtypes = [i64] * 6 + [i32, i32] + [vp] * 16 + [i32]
    lib.oracle_forward_tokens.argtypes = [i64, vp] + [i64] * 6 + [i32, i32] + [vp] * 13 + [i32]
    lib.oracle_expert_ffn_fp8.argtypes = [i64, i64, i64, i32] + [vp] * 9 + [i32]
    lib.oracle_forward_tokens_fp8.argtypes = ([i64, vp] + [i64] * 6 + [i32, i32] + [vp] * 19
                                              + [i32])
    lib.oracle_e4m3_decode.argtypes = [i64, vp, vp]
    lib.oracle_e4m3_encode.argtypes = [i64, vp, vp]
    lib.oracle_quantize_fp8_rows.argtypes = [i64, i64, i32, vp, vp, vp]
    lib.oracle_round_bf16.argtypes = [i64, vp, vp]
    lib.oracle_expert_ffn_w8a8.argtypes = [i64, i64, i64, i32] + [vp] * 11 + [i32]
    lib.oracle_forward_tokens_w8a8.argtypes = ([i64, vp] + [i64] * 6 + [i32, i32] + [vp] * 19
                                               + [i32])
    lib.oracle_forward_tokens_a2.argtypes = lib.oracle_forward_tokens_w8a8.argtypes
    lib.oracle_expert_ffn_a2.argtypes = lib.oracle_expert_ffn_w8a8.argtypes
    lib.oracle_split_e4m3_rows.argtypes = [i64, i64, i32, vp, vp, vp, vp]
    lib.oracle_quantize_fp8_blocks.argtypes = lib.oracle_quantize_fp8_rows.argtypes
    lib.oracle_expert_ffn_fp8_blocks.argtypes = lib.oracle_expert_ffn_fp8.argtypes
    lib.oracle_expert_ffn_a2_blocks.argtypes = lib.oracle_expert_ffn_w8a8.argtypes
    lib.oracle_forward_tokens_fp8_blocks.argtypes = lib.oracle_forward_tokens_fp8.argtypes
    lib.oracle_forward_tokens_a2_blocks.argtypes = lib.oracle_forward_tokens_w8a8.argtypes
    lib.oracle_expert_ffn_w8a8_blocks.argtypes = lib.oracle_expert_ffn_w8a8.argtypes
    lib.oracle_forward_tokens_w8a8_blocks.argtypes = lib.oracle_forward_tokens_w8a8.argtypes
    for f in ("oracle_route", "oracle_permute", "oracle_expert_ffn", "oracle_combine",
              "oracle_shared_ffn", "oracle_forward", "oracle_forward_tokens",
              "oracle_expert_ffn_fp8", "oracle_forward_tokens_fp8", "oracle_e4m3_decode",
              "oracle_e4m3_encode", "oracle_quantize_fp8_rows", "oracle_expert_ffn_w8a8",
              "oracle_forward_tokens_w8a8", "oracle_round_bf16", "oracle_forward_tokens_a2",
              "oracle_expert_ffn_a2", "oracle_split_e4m3_rows", "oracle_quantize_fp8_blocks",
              "oracle_expert_ffn_fp8_blocks", "oracle_expert_ffn_a2_blocks",
              "oracle_forward_tokens_fp8_blocks", "oracle_forward_tokens_a2_blocks",
              "oracle_expert_ffn_w8a8_blocks", "oracle_forward_tokens_w8a8_blocks"):
        getattr(lib, f).restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _arr(a, dtype):
    """Contiguous numpy array of the given dtype (or None)."""
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _in(a, dtype: str):
    if a is None:
        return None
    return _arr(a, np.uint16 if dtype == "bf16" else np.float32)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected its arguments (rc={rc})")


def route(x, w_g, K: int, dtype: str = "f32", bias=None, logits_in=None, threads: int = 0,
          router: str = "softmax"):
    """Top-K routing.  Returns (topk_idx [T,K] int32, topk_w [T,K] f64, keys [T,E] f64),
    keys being the values the selection compares (softmax: score + bias; sigmoid:
    sigmoid(score) + bias).

    With ``logits_in`` (fp32 [T,E]) those raw scores replace x . w_g^T."""
    lib = _load()
    if logits_in is not None:
        logits_in = _arr(logits_in, np.float32)
        T, E = logits_in.shape
        d = 1
        x = w_g = None
    else:
        x, w_g = _in(x, dtype), _in(w_g, dtype)
        T, d = x.shape
        E = w_g.shape[0]
    bias = _arr(bias, np.float64)
    idx = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float64)
    logits = np.zeros((T, E), np.float64)
    _check(lib.oracle_route(T, d, E, K, _DT[dtype], _ROUTER[router], _ptr(x), _ptr(w_g), _ptr(bias),
                            _ptr(logits_in), _ptr(logits), _ptr(idx), _ptr(w), threads),
           "oracle_route")
    return idx, w, logits


def permute(topk_idx, E: int):
    """Returns (counts [E], offsets [E+1], perm [T*K], inv_perm [T*K]) as int32."""
    lib = _load()
    idx = _arr(topk_idx, np.int32)
    T, K = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * K, np.int32)
    inv = np.zeros(T * K, np.int32)
    _check(lib.oracle_permute(T, E, K, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(perm),
                              _ptr(inv)), "oracle_permute")
    return counts, offsets, perm, inv


def expert_ffn(x_perm, offsets, w_gate, w_up, w_down, dtype: str = "f32", threads: int = 0):
    """SwiGLU per expert over expert-contiguous rows.  Returns y_perm [rows, d] f64."""
    lib = _load()
    x_perm = _in(x_perm, dtype)
    offsets = _arr(offsets, np.int32)
    w_gate, w_up, w_down = _in(w_gate, dtype), _in(w_up, dtype), _in(w_down, dtype)
    E, I, d = w_gate.shape
    rows = int(offsets[E])
    y = np.zeros((max(rows, 0), d), np.float64)
    _check(lib.oracle_expert_ffn(d, E, I, _DT[dtype], _ptr(x_perm), _ptr(offsets), _ptr(w_gate),
                                 _ptr(w_up), _ptr(w_down), _ptr(y), threads),
           "oracle_expert_ffn")
    return y


def shared_ffn(x, ws_gate, ws_up, ws_down, dtype: str = "f32", threads: int = 0):
    """The always-on shared expert for every token.  Returns y_s [T, d] f64."""
    lib = _load()
    x = _in(x, dtype)
    ws_gate, ws_up, ws_down = _in(ws_gate, dtype), _in(ws_up, dtype), _in(ws_down, dtype)
    T, d = x.shape
    Is = ws_gate.shape[0]
    y = np.zeros((T, d), np.float64)
    _check(lib.oracle_shared_ffn(T, d, Is, _DT[dtype], _ptr(x), _ptr(ws_gate), _ptr(ws_up),
                                 _ptr(ws_down), _ptr(y), threads), "oracle_shared_ffn")
    return y


def combine(y_perm, inv_perm, topk_w, y_shared=None):
    """y[t] = y_shared[t] + sum_j w[t,j] * y_perm[inv_perm[t*K+j]].  Returns y [T, d] f64."""
    lib = _load()
    y_perm = _arr(y_perm, np.float64)
    inv = _arr(inv_perm, np.int32)
    w = _arr(topk_w, np.float64)
    T, K = w.shape
    d = y_perm.shape[1]
    ys = _arr(y_shared, np.float64)
    y = np.zeros((T, d), np.float64)
    _check(lib.oracle_combine(T, d, K, _ptr(y_perm), _ptr(inv), _ptr(w), _ptr(ys), _ptr(y)),
           "oracle_combine")
    return y


def _weights(p: dict, dtype: str):
    names = ("w_g", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")
    return {n: _in(p.get(n), dtype) for n in names}


def forward(x, params: dict, K: int, dtype: str = "f32", bias=None, threads: int = 0,
            router: str = "softmax"):
    """The whole layer for all T tokens (route, permute, expert FFN, shared, combine).

    ``params`` holds w_g [E,d], w_gate/w_up [E,I,d], w_down [E,d,I] and optionally
    ws_gate/ws_up [Is,d], ws_down [d,Is].  Returns a dict of numpy arrays:
    y, topk_idx, topk_w, counts, offsets, perm, inv_perm."""
    lib = _load()
    x = _in(x, dtype)
    w = _weights(params, dtype)
    T, d = x.shape
    E, I, _ = w["w_gate"].shape
    Is = 0 if w["ws_gate"] is None else w["ws_gate"].shape[0]
    bias = _arr(bias, np.float64)
    out = {
        "y": np.zeros((T, d), np.float64),
        "topk_idx": np.zeros((T, K), np.int32),
        "topk_w": np.zeros((T, K), np.float64),
        "counts": np.zeros(E, np.int32),
        "offsets": np.zeros(E + 1, np.int32),
        "perm": np.zeros(T * K, np.int32),
        "inv_perm": np.zeros(T * K, np.int32),
    }
    _check(lib.oracle_forward(
        T, d, E, K, I, Is, _DT[dtype], _ROUTER[router], _ptr(x), _ptr(w["w_g"]), _ptr(bias),
        _ptr(w["w_gate"]),
        _ptr(w["w_up"]), _ptr(w["w_down"]), _ptr(w["ws_gate"]), _ptr(w["ws_up"]),
        _ptr(w["ws_down"]), _ptr(out["y"]), _ptr(out["topk_idx"]), _ptr(out["topk_w"]),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv_perm"]),
        threads), "oracle_forward")
    return out


def forward_tokens(tokens, x, params: dict, K: int, dtype: str = "f32", bias=None,
                   threads: int = 0, router: str = "softmax"):
    """The layer output for the listed tokens only, from the per-token definition.

    Returns a dict: y [n,d], topk_idx [n,K], topk_w [n,K], logits [n,E]."""
    lib = _load()
    tokens = _arr(tokens, np.int32)
    x = _in(x, dtype)
    w = _weights(params, dtype)
    T, d = x.shape
    E, I, _ = w["w_gate"].shape
    Is = 0 if w["ws_gate"] is None else w["ws_gate"].shape[0]
    n = tokens.shape[0]
    bias = _arr(bias, np.float64)
    out = {
        "y": np.zeros((n, d), np.float64),
        "topk_idx": np.zeros((n, K), np.int32),
        "topk_w": np.zeros((n, K), np.float64),
        "logits": np.zeros((n, E), np.float64),
    }
    _check(lib.oracle_forward_tokens(
        n, _ptr(tokens), T, d, E, K, I, Is, _DT[dtype], _ROUTER[router], _ptr(x), _ptr(w["w_g"]),
        _ptr(bias),
        _ptr(w["w_gate"]), _ptr(w["w_up"]), _ptr(w["w_down"]), _ptr(w["ws_gate"]),
        _ptr(w["ws_up"]), _ptr(w["ws_down"]), _ptr(out["y"]), _ptr(out["topk_idx"]),
        _ptr(out["topk_w"]), _ptr(out["logits"]), threads), "oracle_forward_tokens")
    return out


# ---------------------------------------------------------------- 8-bit weights

def e4m3_decode(codes):
    """The exact value of every E4M3 code (float64; NaN for the NaN codes)."""
    lib = _load()
    c = _arr(codes, np.uint8)
    out = np.zeros(c.shape, np.float64)
    _check(lib.oracle_e4m3_decode(c.size, _ptr(c), _ptr(out)), "oracle_e4m3_decode")
    return out


def e4m3_encode(v):
    """Nearest E4M3 code of each float32 value (ties to even, clamped to +-448)."""
    lib = _load()
    v = _arr(v, np.float32)
    out = np.zeros(v.shape, np.uint8)
    _check(lib.oracle_e4m3_encode(v.size, _ptr(v), _ptr(out)), "oracle_e4m3_encode")
    return out


def quantize_fp8_rows(w, dtype: str = "f32"):
    """Per-row E4M3 quantisation of a [..., cols] matrix: returns (codes uint8 of
    w's shape, scales float32 of w's leading shape)."""
    lib = _load()
    w = _in(w, dtype)
    cols = w.shape[-1]
    rows = w.size // cols
    codes = np.zeros(w.shape, np.uint8)
    scales = np.zeros(w.shape[:-1], np.float32)
    _check(lib.oracle_quantize_fp8_rows(rows, cols, _DT[dtype], _ptr(w), _ptr(codes),
                                        _ptr(scales)), "oracle_quantize_fp8_rows")
    return codes, scales


FP8_BLOCK = 128  # side of a square weight-scale block


def quantize_fp8_blocks(w, dtype: str = "f32"):
    """Block-scaled E4M3 quantisation of a [..., cols] matrix taken as one
    stacked [rows][cols] matrix (rows = the product of the leading sizes): one
    scale per 128 x 128 block.  Returns (codes uint8 of w's shape, scales
    float32 [ceil(rows/128)][ceil(cols/128)])."""
    lib = _load()
    w = _in(w, dtype)
    cols = w.shape[-1]
    rows = w.size // cols
    B = FP8_BLOCK
    codes = np.zeros(w.shape, np.uint8)
    scales = np.zeros(((rows + B - 1) // B, (cols + B - 1) // B), np.float32)
    _check(lib.oracle_quantize_fp8_blocks(rows, cols, _DT[dtype], _ptr(w), _ptr(codes),
                                          _ptr(scales)), "oracle_quantize_fp8_blocks")
    return codes, scales


_FP8_NAMES = ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")


def _fp8_weights(q: dict):
    """Codes (uint8) and row scales (float32) of the expert weights: keys w_gate,
    s_gate, ... as in the C signature (shared ones optional)."""
    out = {}
    for n in _FP8_NAMES:
        out[n] = _arr(q.get(n), np.uint8)
        sn = "s" + n[1:] if n.startswith("w_") else "ss" + n[2:]
        out[sn] = _arr(q.get(sn), np.float32)
    return out


def expert_ffn_fp8(x_perm, offsets, q: dict, dtype: str = "bf16", threads: int = 0,
                   blocks: bool = False):
    """SwiGLU per expert with E4M3 weights (q: w_gate, w_up, w_down codes and
    s_gate, s_up, s_down row scales, or with blocks=True the 128 x 128 block
    scales of quantize_fp8_blocks).  Returns y_perm [rows, d] f64."""
    lib = _load()
    fname = "oracle_expert_ffn_fp8_blocks" if blocks else "oracle_expert_ffn_fp8"
    x_perm = _in(x_perm, dtype)
    offsets = _arr(offsets, np.int32)
    w = _fp8_weights(q)
    E, I, d = w["w_gate"].shape
    rows = int(offsets[E])
    y = np.zeros((max(rows, 0), d), np.float64)
    _check(getattr(lib, fname)(
        d, E, I, _DT[dtype], _ptr(x_perm), _ptr(offsets), _ptr(w["w_gate"]), _ptr(w["w_up"]),
        _ptr(w["w_down"]), _ptr(w["s_gate"]), _ptr(w["s_up"]), _ptr(w["s_down"]), _ptr(y),
        threads), fname)
    return y


def round_bf16(v):
    """float32 -> bf16 (round to nearest even) as the W8A8 experts round h;
    returns float32."""
    lib = _load()
    v = _arr(v, np.float32)
    out = np.zeros(v.shape, np.float32)
    _check(lib.oracle_round_bf16(v.size, _ptr(v), _ptr(out)), "oracle_round_bf16")
    return out


def split_e4m3_rows(x, dtype: str = "bf16"):
    """Two E4M3 planes per row: (hi, lo) uint8 codes [rows, cols] and the fp32
    row scale [rows], with x ~ scale * (value(hi) + value(lo)) (see
    split_vec in moe_oracle.c)."""
    lib = _load()
    x = _in(x, dtype)
    rows, cols = x.shape
    hi = np.zeros((rows, cols), np.uint8)
    lo = np.zeros((rows, cols), np.uint8)
    sc = np.zeros(rows, np.float32)
    _check(lib.oracle_split_e4m3_rows(rows, cols, _DT[dtype], _ptr(x), _ptr(hi), _ptr(lo),
                                      _ptr(sc)), "oracle_split_e4m3_rows")
    return hi, lo, sc


def expert_ffn_a2(x_perm, offsets, q: dict, dtype: str = "bf16", threads: int = 0,
                  taps: bool = False, blocks: bool = False):
    """expert_ffn_fp8 with every x_perm row and every hidden row (after its bf16
    rounding) carried as two E4M3 planes (split_e4m3_rows); blocks=True: the
    weights' 128 x 128 block scales.  Returns as expert_ffn_w8a8."""
    return _expert_ffn_a8(x_perm, offsets, q, dtype, threads, taps,
                          "oracle_expert_ffn_a2_blocks" if blocks else "oracle_expert_ffn_a2")


def expert_ffn_w8a8(x_perm, offsets, q: dict, dtype: str = "bf16", threads: int = 0,
                    taps: bool = False, blocks: bool = False):
    """expert_ffn_fp8 with 8-bit activations: each x_perm row and each hidden row
    (after fp32 -> bf16 rounding) quantised to E4M3 with one scale per row;
    blocks=True: the weights' 128 x 128 block scales.  Returns y_perm [rows, d]
    f64, or (y_perm, h_pre, h_hat) with taps: h before rounding and the
    dequantised quantised h, both [rows, I] f64."""
    return _expert_ffn_a8(x_perm, offsets, q, dtype, threads, taps,
                          "oracle_expert_ffn_w8a8_blocks" if blocks else "oracle_expert_ffn_w8a8")


def _expert_ffn_a8(x_perm, offsets, q, dtype, threads, taps, fname):
    lib = _load()
    x_perm = _in(x_perm, dtype)
    offsets = _arr(offsets, np.int32)
    w = _fp8_weights(q)
    E, I, d = w["w_gate"].shape
    rows = max(int(offsets[E]), 0)
    y = np.zeros((rows, d), np.float64)
    h_pre = np.zeros((rows, I), np.float64) if taps else None
    h_hat = np.zeros((rows, I), np.float64) if taps else None
    _check(getattr(lib, fname)(
        d, E, I, _DT[dtype], _ptr(x_perm), _ptr(offsets), _ptr(w["w_gate"]), _ptr(w["w_up"]),
        _ptr(w["w_down"]), _ptr(w["s_gate"]), _ptr(w["s_up"]), _ptr(w["s_down"]), _ptr(y),
        _ptr(h_pre), _ptr(h_hat), threads), fname)
    return (y, h_pre, h_hat) if taps else y


def forward_tokens_fp8(tokens, x, w_g, q: dict, K: int, dtype: str = "bf16", bias=None,
                       threads: int = 0, router: str = "softmax", act8=False,
                       blocks: bool = False):
    """forward_tokens with E4M3 expert weights (routed and, when present, shared):
    q holds w_gate/w_up/w_down (+ ws_*) codes and s_gate/s_up/s_down (+ ss_*)
    row scales; x and w_g are in dtype.  Returns the same dict as forward_tokens.
    act8: True (or "w8a8") -- every expert runs W8A8 (its input and hidden rows
    quantised per row; see oracle_forward_tokens_w8a8); "planes" -- every
    expert's input and hidden rows carried as two E4M3 planes
    (oracle_forward_tokens_a2).  blocks=True: the scales are the 128 x 128 block
    scales of quantize_fp8_blocks (any act8)."""
    lib = _load()
    tokens = _arr(tokens, np.int32)
    x, w_g = _in(x, dtype), _in(w_g, dtype)
    w = _fp8_weights(q)
    T, d = x.shape
    E, I, _ = w["w_gate"].shape
    Is = 0 if w["ws_gate"] is None else w["ws_gate"].shape[0]
    n = tokens.shape[0]
    bias = _arr(bias, np.float64)
    out = {
        "y": np.zeros((n, d), np.float64),
        "topk_idx": np.zeros((n, K), np.int32),
        "topk_w": np.zeros((n, K), np.float64),
        "logits": np.zeros((n, E), np.float64),
    }
    fname = ("oracle_forward_tokens_a2" if act8 == "planes" else
             "oracle_forward_tokens_w8a8" if act8 else "oracle_forward_tokens_fp8")
    if blocks:
        fname += "_blocks"
    fn = getattr(lib, fname)
    _check(fn(
        n, _ptr(tokens), T, d, E, K, I, Is, _DT[dtype], _ROUTER[router], _ptr(x), _ptr(w_g),
        _ptr(bias), _ptr(w["w_gate"]), _ptr(w["w_up"]), _ptr(w["w_down"]), _ptr(w["s_gate"]),
        _ptr(w["s_up"]), _ptr(w["s_down"]), _ptr(w["ws_gate"]), _ptr(w["ws_up"]),
        _ptr(w["ws_down"]), _ptr(w["ss_gate"]), _ptr(w["ss_up"]), _ptr(w["ss_down"]),
        _ptr(out["y"]), _ptr(out["topk_idx"]), _ptr(out["topk_w"]), _ptr(out["logits"]),
        threads), fname)
    return out
