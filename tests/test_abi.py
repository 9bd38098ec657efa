"""The C ABI library builds, loads and exports every symbol include/moe.h declares,
and its host-side argument checks reject bad calls before touching the device
(no GPU needed: nothing here launches work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


@pytest.fixture(scope="module")
def moe(lib):
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_stage_entry_points():
    names = _declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_workspace_bytes", "moe_get_device_error", "moe_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_names_match_the_header(moe):
    assert set(moe.EXPORTED) == set(_declared_functions())
    for n in moe.EXPORTED:
        assert hasattr(moe.library(), n)


def test_status_strings(moe):
    assert moe.status_string(0) == "ok"
    assert "workspace" in moe.status_string(3)
    assert moe.status_string(99) == "unknown status"


def test_workspace_bytes_and_shape_limits(moe):
    s = moe.make_shape(8, 7168, 256, 8, 2048, 2048, "bf16")
    n = moe.moe_workspace_bytes(s)
    # at least the permuted activations, h and y_perm of 64 rows
    assert n >= 64 * 7168 * 2 * 2 + 64 * 2048 * 2
    bad = [moe.make_shape(8, 7168, 256, 9, 2048, 0, "bf16"),     # K > E? no: K=9 ok -> check below
           moe.make_shape(8, 7168, 4, 8, 2048, 0, "bf16"),       # K > E
           moe.make_shape(8, 7100, 256, 8, 2048, 0, "bf16"),     # d not a multiple of 64
           moe.make_shape(8, 7168, 2048, 8, 2048, 0, "bf16"),    # E > 1024
           moe.make_shape(8, 7168, 256, 33, 2048, 0, "bf16"),    # K > 32
           moe.make_shape(-1, 7168, 256, 8, 2048, 0, "bf16"),    # T < 0
           moe.make_shape(8, 7168, 256, 8, 2048, 0, 7)]          # dtype
    assert moe.moe_workspace_bytes(bad[0]) > 0
    for s in bad[1:]:
        assert moe.moe_workspace_bytes(s) == 0


def test_argument_errors_return_before_any_launch(lib, moe):
    """Null/misaligned pointers and a short workspace are refused on the host."""
    s = moe.make_shape(4, 64, 8, 2, 64, 0, "f32")
    sp = ctypes.byref(s)
    lib.moe_forward.restype = ctypes.c_int32
    lib.moe_route.restype = ctypes.c_int32
    lib.moe_combine.restype = ctypes.c_int32
    lib.moe_permute.restype = ctypes.c_int32
    lib.moe_expert_ffn.restype = ctypes.c_int32
    vp = ctypes.c_void_p
    z = ctypes.c_size_t
    fake = vp(1 << 20)          # aligned, never dereferenced: validation fails first
    odd = vp((1 << 20) + 4)     # misaligned
    # null x
    rc = lib.moe_forward(sp, None, fake, None, fake, fake, fake, None, None, None, fake,
                         fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # misaligned weight
    rc = lib.moe_forward(sp, fake, odd, None, fake, fake, fake, None, None, None, fake,
                         fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # shared weights given but inter_shared == 0
    rc = lib.moe_forward(sp, fake, fake, None, fake, fake, fake, fake, fake, fake, fake,
                         fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    rc = lib.moe_forward(sp, fake, fake, None, fake, fake, fake, None, None, None, fake,
                         fake, z(16), None)
    assert rc == moe.MOE_ERR_WORKSPACE
    # no workspace
    rc = lib.moe_route(sp, fake, fake, None, None, None, fake, fake, None, z(0), None)
    assert rc == moe.MOE_ERR_WORKSPACE
    # route without outputs
    rc = lib.moe_route(sp, fake, fake, None, None, None, None, fake, fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # combine without inv_perm
    rc = lib.moe_combine(sp, fake, None, fake, None, fake, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # permute without counts
    rc = lib.moe_permute(sp, fake, None, None, fake, None, None, None, fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # expert ffn with a null weight
    rc = lib.moe_expert_ffn(sp, fake, fake, None, fake, fake, fake, fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # K > E is invalid; K > 32 unsupported
    s2 = moe.make_shape(4, 64, 8, 9, 64, 0, "f32")
    rc = lib.moe_forward(ctypes.byref(s2), fake, fake, None, fake, fake, fake, None, None, None,
                         fake, fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    s3 = moe.make_shape(4, 64, 64, 33, 64, 0, "f32")
    rc = lib.moe_forward(ctypes.byref(s3), fake, fake, None, fake, fake, fake, None, None, None,
                         fake, fake, z(1 << 30), None)
    assert rc == moe.MOE_ERR_UNSUPPORTED


def test_binding_refuses_host_tensors(moe):
    import torch
    s = moe.make_shape(2, 64, 4, 2, 64, 0, "f32")
    x = torch.zeros(2, 64)
    with pytest.raises(ValueError):
        moe.moe_combine(s, x, x, x, None, x, stream=0)


# (layer entry point, stage entry point, quantiser) of each 8-bit-weight form
FP8_FORMS = {"rows": ("moe_forward_fp8", "moe_expert_ffn_fp8", "moe_quantize_fp8_rows"),
             "w8a8": ("moe_forward_w8a8", "moe_expert_ffn_w8a8", "moe_quantize_fp8_rows"),
             "blocks": ("moe_forward_fp8_blocks", "moe_expert_ffn_fp8_blocks",
                        "moe_quantize_fp8_blocks"),
             "w8a8_blocks": ("moe_forward_w8a8_blocks", "moe_expert_ffn_w8a8_blocks",
                             "moe_quantize_fp8_blocks")}


@pytest.mark.parametrize("form", sorted(FP8_FORMS))
def test_fp8_argument_errors_return_before_any_launch(lib, moe, form):
    """The 8-bit entry points (8-bit weights with row or block scales, and
    8-bit weights and activations) refuse bad shapes and pointers on the host."""
    vp, z = ctypes.c_void_p, ctypes.c_size_t
    fake = (1 << 20)
    odd = (1 << 20) + 4
    fwd_name, ffn_name, q_name = FP8_FORMS[form]
    for f in FP8_FORMS[form]:
        getattr(lib, f).restype = ctypes.c_int32
    getattr(lib, q_name).argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                     vp, vp, vp, vp]
    q = getattr(lib, q_name)
    assert q(-1, 64, moe.MOE_BF16, vp(fake), vp(fake), vp(fake), None) == moe.MOE_ERR_INVALID_ARG
    assert q(4, 0, moe.MOE_BF16, vp(fake), vp(fake), vp(fake), None) == moe.MOE_ERR_INVALID_ARG
    assert q(4, 64, 5, vp(fake), vp(fake), vp(fake), None) == moe.MOE_ERR_INVALID_ARG
    assert q(4, 40, moe.MOE_BF16, vp(fake), vp(fake), vp(fake), None) == moe.MOE_ERR_UNSUPPORTED
    assert q(4, 64, moe.MOE_BF16, None, vp(fake), vp(fake), None) == moe.MOE_ERR_INVALID_ARG
    assert q(4, 64, moe.MOE_BF16, vp(fake), vp(odd), vp(fake), None) == moe.MOE_ERR_INVALID_ARG
    assert q(0, 64, moe.MOE_BF16, None, None, None, None) == moe.MOE_OK
    if q_name == "moe_quantize_fp8_blocks":  # more block rows than one launch's grid holds
        assert q(65536 * 128, 64, moe.MOE_BF16, vp(fake), vp(fake), vp(fake),
                 None) == moe.MOE_ERR_UNSUPPORTED

    full = {n: fake for n, _ in moe.moe_fp8_experts._fields_}
    routed = dict(full, ws_gate=None, ws_up=None, ws_down=None, ss_gate=None, ss_up=None,
                  ss_down=None)
    W = moe.moe_fp8_experts(*[routed[n] for n, _ in moe.moe_fp8_experts._fields_])
    s = moe.make_shape(4, 128, 8, 2, 256, 0, "bf16")
    big = z(1 << 30)

    def fwd(shape, w, **kw):
        a = dict(x=vp(fake), w_g=vp(fake), y=vp(fake), ws=vp(fake), n=big)
        a.update(kw)
        f = getattr(lib, fwd_name)
        return f(ctypes.byref(shape), a["x"], a["w_g"], None,
                 ctypes.byref(w) if w is not None else None, a["y"], a["ws"], a["n"], None)

    # activations must be bf16; K extents multiples of 128
    assert fwd(moe.make_shape(4, 128, 8, 2, 256, 0, "f32"), W) == moe.MOE_ERR_UNSUPPORTED
    assert fwd(moe.make_shape(4, 192, 8, 2, 256, 0, "bf16"), W) == moe.MOE_ERR_UNSUPPORTED
    assert fwd(moe.make_shape(4, 128, 8, 2, 320, 0, "bf16"), W) == moe.MOE_ERR_UNSUPPORTED
    assert fwd(moe.make_shape(4, 128, 8, 2, 256, 64, "bf16"), W) == moe.MOE_ERR_UNSUPPORTED
    # null / misaligned pointers, missing or unwanted shared weights, short workspace
    assert fwd(s, None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(s, W, x=None) == moe.MOE_ERR_INVALID_ARG
    assert fwd(s, W, y=vp(odd)) == moe.MOE_ERR_INVALID_ARG
    bad = moe.moe_fp8_experts(*[(odd if n == "s_down" else routed[n])
                                for n, _ in moe.moe_fp8_experts._fields_])
    assert fwd(s, bad) == moe.MOE_ERR_INVALID_ARG
    W_full = moe.moe_fp8_experts(*[full[n] for n, _ in moe.moe_fp8_experts._fields_])
    assert fwd(s, W_full) == moe.MOE_ERR_INVALID_ARG
    assert fwd(moe.make_shape(4, 128, 8, 2, 256, 128, "bf16"), W) == moe.MOE_ERR_INVALID_ARG
    assert fwd(s, W, n=z(16)) == moe.MOE_ERR_WORKSPACE
    assert fwd(moe.make_shape(0, 128, 8, 2, 256, 0, "bf16"), None) == moe.MOE_OK

    e = getattr(lib, ffn_name)
    assert e(ctypes.byref(s), vp(fake), None, ctypes.byref(W), vp(fake), vp(fake), big,
             None) == moe.MOE_ERR_INVALID_ARG
    assert e(ctypes.byref(s), vp(fake), vp(fake), None, vp(fake), vp(fake), big,
             None) == moe.MOE_ERR_INVALID_ARG
    assert e(ctypes.byref(s), vp(fake), vp(fake), ctypes.byref(W), vp(fake), vp(fake), z(16),
             None) == moe.MOE_ERR_WORKSPACE
