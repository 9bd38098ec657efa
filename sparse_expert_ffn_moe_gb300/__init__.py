"""Python binding of libmoe, the GB300 (sm_103a) sparse MoE FFN layer forward.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe.so (built from csrc/ by ``_build.build``).  The functions have the names
and argument order of the C ABI in include/moe.h; tensors are torch CUDA
tensors (or None for a NULL pointer), ``stream`` defaults to torch's current
stream.  A non-OK status raises MoeError.  There is no CPU path: importing the
binding without the built library raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_BOUNDS = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTER_SOFTMAX, MOE_ROUTER_SIGMOID = 0, 1

EXPORTED = ("moe_status_string", "moe_workspace_bytes", "moe_route", "moe_permute",
            "moe_permute_noalloc", "moe_expert_ffn", "moe_combine", "moe_forward",
            "moe_quantize_fp8_rows", "moe_expert_ffn_fp8", "moe_forward_fp8",
            "moe_quantize_fp8_blocks", "moe_expert_ffn_fp8_blocks", "moe_forward_fp8_blocks",
            "moe_expert_ffn_w8a8", "moe_forward_w8a8", "moe_expert_ffn_w8a8_blocks",
            "moe_forward_w8a8_blocks", "moe_get_device_error")
FP8_BLOCK = 128  # side of the square weight-scale blocks of the *_fp8_blocks calls


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("inter_shared", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("router", ctypes.c_int32)]


class moe_fp8_experts(ctypes.Structure):
    """E4M3 expert weight codes (uint8) and fp32 scales (per row, or per 128 x 128
    block for the *_fp8_blocks calls): device pointers."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
        "ws_gate", "ws_up", "ws_down", "ss_gate", "ss_up", "ss_down")]


def _load_lib() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libmoe.so is not built ({LIB_PATH}); run sparse_expert_ffn_moe_gb300._build.build() "
            "-- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    sp = ctypes.POINTER(moe_shape)
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_workspace_bytes.argtypes = [sp]
    lib.moe_workspace_bytes.restype = sz
    lib.moe_route.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_permute.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_permute_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_expert_ffn.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_combine.argtypes = [sp, vp, vp, vp, vp, vp, vp]
    lib.moe_forward.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    fp = ctypes.POINTER(moe_fp8_experts)
    lib.moe_quantize_fp8_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, i32, vp, vp, vp, vp]
    lib.moe_expert_ffn_fp8.argtypes = [sp, vp, vp, fp, vp, vp, sz, vp]
    lib.moe_forward_fp8.argtypes = [sp, vp, vp, vp, fp, vp, vp, sz, vp]
    lib.moe_quantize_fp8_blocks.argtypes = lib.moe_quantize_fp8_rows.argtypes
    lib.moe_expert_ffn_fp8_blocks.argtypes = lib.moe_expert_ffn_fp8.argtypes
    lib.moe_forward_fp8_blocks.argtypes = lib.moe_forward_fp8.argtypes
    lib.moe_expert_ffn_w8a8.argtypes = [sp, vp, vp, fp, vp, vp, sz, vp]
    lib.moe_forward_w8a8.argtypes = [sp, vp, vp, vp, fp, vp, vp, sz, vp]
    lib.moe_expert_ffn_w8a8_blocks.argtypes = lib.moe_expert_ffn_w8a8.argtypes
    lib.moe_forward_w8a8_blocks.argtypes = lib.moe_forward_w8a8.argtypes
    lib.moe_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    for f in ("moe_route", "moe_permute", "moe_permute_noalloc", "moe_expert_ffn", "moe_combine",
              "moe_forward", "moe_quantize_fp8_rows", "moe_expert_ffn_fp8", "moe_forward_fp8",
              "moe_quantize_fp8_blocks", "moe_expert_ffn_fp8_blocks", "moe_forward_fp8_blocks",
              "moe_expert_ffn_w8a8", "moe_forward_w8a8", "moe_expert_ffn_w8a8_blocks",
              "moe_forward_w8a8_blocks", "moe_get_device_error"):
        getattr(lib, f).restype = i32
    return lib


_lib = _load_lib()


def library() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def make_shape(T: int, d: int, E: int, K: int, inter: int, inter_shared: int = 0,
               dtype: str | int = "bf16", router: str | int = "softmax") -> moe_shape:
    if isinstance(dtype, str):
        dtype = {"bf16": MOE_BF16, "f32": MOE_F32}[dtype]
    if isinstance(router, str):
        router = {"softmax": MOE_ROUTER_SOFTMAX, "sigmoid": MOE_ROUTER_SIGMOID}[router]
    return moe_shape(T, d, E, K, inter, inter_shared, dtype, router)


def _p(t):
    """Device pointer of a tensor (None -> NULL).  Host tensors are refused."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _p(workspace), workspace.numel() * workspace.element_size()


def moe_workspace_bytes(shape: moe_shape) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(shape)))


def alloc_workspace(shape: moe_shape, device=None) -> torch.Tensor:
    n = moe_workspace_bytes(shape)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def moe_route(shape, x, w_g, bias, logits_in, logits_out, topk_idx, topk_w, workspace,
              stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_route(ctypes.byref(shape), _p(x), _p(w_g), _p(bias), _p(logits_in),
                          _p(logits_out), _p(topk_idx), _p(topk_w), ws, nws, _stream(stream)),
           "moe_route")


def moe_permute(shape, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, workspace,
                stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_permute(ctypes.byref(shape), _p(topk_idx), _p(x), _p(counts), _p(offsets),
                            _p(perm), _p(inv_perm), _p(x_perm), ws, nws, _stream(stream)),
           "moe_permute")


def moe_permute_noalloc(shape, topk_idx, x, counts, offsets, perm, inv_perm, x_perm,
                        stream=None):
    """moe_permute without a workspace: its scratch is a fixed array inside the
    library, for callers that cannot allocate device memory."""
    _check(_lib.moe_permute_noalloc(ctypes.byref(shape), _p(topk_idx), _p(x), _p(counts),
                                    _p(offsets), _p(perm), _p(inv_perm), _p(x_perm),
                                    _stream(stream)), "moe_permute_noalloc")


def moe_expert_ffn(shape, x_perm, offsets, w_gate, w_up, w_down, y_perm, workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_expert_ffn(ctypes.byref(shape), _p(x_perm), _p(offsets), _p(w_gate),
                               _p(w_up), _p(w_down), _p(y_perm), ws, nws, _stream(stream)),
           "moe_expert_ffn")


def moe_combine(shape, y_perm, inv_perm, topk_w, y_shared, y, stream=None):
    _check(_lib.moe_combine(ctypes.byref(shape), _p(y_perm), _p(inv_perm), _p(topk_w),
                            _p(y_shared), _p(y), _stream(stream)), "moe_combine")


def moe_forward(shape, x, w_g, bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y,
                workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_forward(ctypes.byref(shape), _p(x), _p(w_g), _p(bias), _p(w_gate), _p(w_up),
                            _p(w_down), _p(ws_gate), _p(ws_up), _p(ws_down), _p(y), ws, nws,
                            _stream(stream)), "moe_forward")


def moe_quantize_fp8_rows(w, codes, scales, stream=None):
    """Per-row E4M3 quantisation of the last dimension of w (bf16 or fp32):
    codes (uint8, w's shape) and scales (fp32, w's leading shape)."""
    dtype = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}[w.dtype]
    cols = w.shape[-1]
    rows = w.numel() // cols if cols else 0
    _check(_lib.moe_quantize_fp8_rows(rows, cols, dtype, _p(w), _p(codes), _p(scales),
                                      _stream(stream)), "moe_quantize_fp8_rows")


def moe_quantize_fp8_blocks(w, codes, scales, stream=None):
    """Block-scaled E4M3 quantisation of w (bf16 or fp32) taken as one stacked
    [rows][cols] matrix (rows = the product of the leading sizes): codes (uint8,
    w's shape) and scales (fp32, [ceil(rows/128)][ceil(cols/128)])."""
    dtype = {torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}[w.dtype]
    cols = w.shape[-1]
    rows = w.numel() // cols if cols else 0
    _check(_lib.moe_quantize_fp8_blocks(rows, cols, dtype, _p(w), _p(codes), _p(scales),
                                        _stream(stream)), "moe_quantize_fp8_blocks")


def make_fp8_experts(q: dict) -> moe_fp8_experts:
    """A moe_fp8_experts from a dict of device tensors (w_gate, w_up, w_down codes,
    s_gate, s_up, s_down scales; ws_* / ss_* for the shared expert, optional).
    The caller keeps the tensors alive while the struct is in use."""
    return moe_fp8_experts(*[_p(q.get(n)) for n, _ in moe_fp8_experts._fields_])


def moe_expert_ffn_fp8(shape, x_perm, offsets, w: moe_fp8_experts, y_perm, workspace,
                       stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_expert_ffn_fp8(ctypes.byref(shape), _p(x_perm), _p(offsets), ctypes.byref(w),
                                   _p(y_perm), ws, nws, _stream(stream)), "moe_expert_ffn_fp8")


def moe_forward_fp8(shape, x, w_g, bias, w: moe_fp8_experts, y, workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_forward_fp8(ctypes.byref(shape), _p(x), _p(w_g), _p(bias), ctypes.byref(w),
                                _p(y), ws, nws, _stream(stream)), "moe_forward_fp8")


def moe_expert_ffn_fp8_blocks(shape, x_perm, offsets, w: moe_fp8_experts, y_perm, workspace,
                              stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_expert_ffn_fp8_blocks(ctypes.byref(shape), _p(x_perm), _p(offsets),
                                          ctypes.byref(w), _p(y_perm), ws, nws, _stream(stream)),
           "moe_expert_ffn_fp8_blocks")


def moe_forward_fp8_blocks(shape, x, w_g, bias, w: moe_fp8_experts, y, workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_forward_fp8_blocks(ctypes.byref(shape), _p(x), _p(w_g), _p(bias),
                                       ctypes.byref(w), _p(y), ws, nws, _stream(stream)),
           "moe_forward_fp8_blocks")


def moe_expert_ffn_w8a8(shape, x_perm, offsets, w: moe_fp8_experts, y_perm, workspace,
                        stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_expert_ffn_w8a8(ctypes.byref(shape), _p(x_perm), _p(offsets),
                                    ctypes.byref(w), _p(y_perm), ws, nws, _stream(stream)),
           "moe_expert_ffn_w8a8")


def moe_forward_w8a8(shape, x, w_g, bias, w: moe_fp8_experts, y, workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_forward_w8a8(ctypes.byref(shape), _p(x), _p(w_g), _p(bias), ctypes.byref(w),
                                 _p(y), ws, nws, _stream(stream)), "moe_forward_w8a8")


def moe_expert_ffn_w8a8_blocks(shape, x_perm, offsets, w: moe_fp8_experts, y_perm, workspace,
                               stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_expert_ffn_w8a8_blocks(ctypes.byref(shape), _p(x_perm), _p(offsets),
                                           ctypes.byref(w), _p(y_perm), ws, nws, _stream(stream)),
           "moe_expert_ffn_w8a8_blocks")


def moe_forward_w8a8_blocks(shape, x, w_g, bias, w: moe_fp8_experts, y, workspace, stream=None):
    ws, nws = _ws(workspace)
    _check(_lib.moe_forward_w8a8_blocks(ctypes.byref(shape), _p(x), _p(w_g), _p(bias),
                                        ctypes.byref(w), _p(y), ws, nws, _stream(stream)),
           "moe_forward_w8a8_blocks")


def moe_get_device_error(workspace) -> int:
    code = ctypes.c_int32(0)
    _check(_lib.moe_get_device_error(_p(workspace), ctypes.byref(code)), "moe_get_device_error")
    return int(code.value)
