"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching the
GPU. CPU only (no compute call needs a device here)."""
import ctypes
import os
import re

import pytest

from route_permute_grouped_gb300 import build as B
from route_permute_grouped_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ops.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "moe_layer_fwd" in names and "moe_layer_bwd" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_workspace_bytes_and_status_strings(lib):
    cfg = ops.make_config(256, 128, 8, 2, 256)
    n_inf = ops.workspace_bytes(cfg, False)
    n_tr = ops.workspace_bytes(cfg, True)
    assert 0 < n_inf < n_tr
    bad = ops.make_config(256, 128, 8, 9, 256)  # k > E
    assert ops.workspace_bytes(bad) == 0
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(5).startswith(b"device")


@pytest.mark.parametrize("over,code", [
    (dict(k=9), 1),                         # k > E
    (dict(H=100), 2),                       # H not a multiple of 64
    (dict(E=6, n_groups=4, topk_groups=2), 2),   # E not divisible by groups
    (dict(E=512, k=8), 2),                  # E > 256
    (dict(score=7), 1),
    (dict(gate_scale=0.0), 1),
    (dict(force_balanced=2), 1),
])
def test_host_rejects_bad_config(lib, over, code):
    d = dict(T=256, H=128, E=8, k=2, F=256)
    d.update(over)
    cfg = ops.make_config(**d)
    fake = ctypes.c_void_p(256)  # never dereferenced: the check fails first
    st = lib.moe_router_topk(ctypes.byref(cfg), fake, fake, None, None, fake, fake, None, None, fake, 1 << 30, None)
    assert st == code


def test_host_rejects_null_and_small_workspace(lib):
    cfg = ops.make_config(256, 128, 8, 2, 256)
    fake = ctypes.c_void_p(256)
    assert lib.moe_router_topk(ctypes.byref(cfg), None, fake, None, None, fake, fake, None, None, fake, 1 << 30,
                               None) == 1
    assert lib.moe_permute(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, 16, None) == 3
    assert lib.moe_layer_fwd(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, None, None, None, fake,
                             None, fake, 16, None) == 3
    misaligned = ctypes.c_void_p(256 + 8)
    assert lib.moe_permute(ctypes.byref(cfg), misaligned, fake, fake, fake, fake, fake, fake, 1 << 30, None) == 1
    # the backward of a layer with a shared expert needs its weights, its saved
    # tensors and its gradient buffers
    sh = ops.make_config(256, 128, 8, 2, 256, F_shared=64)
    sv = ops.MoeFwdSaved(*([256] * 11 + [None, None]))
    args = [fake] * 6
    assert lib.moe_layer_bwd(ctypes.byref(sh), *args, None, None, None, ctypes.byref(sv), fake, fake, fake, fake,
                             fake, None, None, None, None, fake, 1 << 40, None) == 1
    sv_full = ops.MoeFwdSaved(*([256] * 13))
    assert lib.moe_layer_bwd(ctypes.byref(sh), *args, fake, fake, fake, ctypes.byref(sv_full), fake, fake, fake,
                             fake, fake, fake, fake, fake, None, fake, 16, None) == 3


def test_binding_structs_match_the_library(lib):
    lib.moe_abi_struct_bytes.restype = ctypes.c_size_t
    assert lib.moe_abi_struct_bytes(0) == ctypes.sizeof(ops.MoeConfig)
    assert lib.moe_abi_struct_bytes(1) == ctypes.sizeof(ops.MoeFwdSaved)
    assert lib.moe_abi_struct_bytes(2) == 0


def test_low_precision_entry_points_check_on_the_host(lib):
    # shapes the block-scaled GEMMs cannot take: sizes are 0, calls are
    # rejected before any CUDA work (null pointers, bad shapes)
    ok = ops.make_config(256, 256, 8, 2, 256)
    bad_h = ops.make_config(256, 192, 8, 2, 256)      # H not a multiple of 128 / 256
    bad_f = ops.make_config(256, 256, 8, 2, 192)      # F not a multiple of 128 (MXFP8) or 256 (NVFP4)
    shared = ops.make_config(256, 256, 8, 2, 256, F_shared=64)
    for i in range(4):
        assert lib.moe_mx_weight_bytes(ctypes.byref(ok), i) > 0
        assert lib.moe_mx_weight_bytes(ctypes.byref(bad_h), i) == 0
        assert lib.moe_mx_weight_bytes(ctypes.byref(bad_f), i) == 0
    assert lib.moe_mx_workspace_bytes(ctypes.byref(bad_h)) == 0
    for i in range(4):
        assert lib.moe_mx_bwd_weight_bytes(ctypes.byref(ok), i) > 0
        assert lib.moe_mx_bwd_weight_bytes(ctypes.byref(bad_f), i) == 0
    assert lib.moe_mx_bwd_weight_bytes(ctypes.byref(ok), 0) == 8 * 256 * 256
    assert lib.moe_mx_train_workspace_bytes(ctypes.byref(ok)) > lib.moe_mx_workspace_bytes(ctypes.byref(ok))
    assert lib.moe_mx_train_workspace_bytes(ctypes.byref(shared)) == 0      # no shared expert in training
    assert lib.moe_mx_train_workspace_bytes(ctypes.byref(bad_h)) == 0
    for i in range(6):
        assert lib.moe_nv_layer_weight_bytes(ctypes.byref(ok), i) > 0
        assert lib.moe_nv_layer_weight_bytes(ctypes.byref(bad_h), i) == 0
        assert lib.moe_nv_layer_weight_bytes(ctypes.byref(shared), i) == 0   # no shared expert in the NVFP4 layer
    assert lib.moe_nv_workspace_bytes_layer(ctypes.byref(bad_f)) == 0
    assert lib.moe_nv_weight_bytes(4, 256, 8, 0) == 4 * 8 * 128
    assert lib.moe_nv_weight_bytes(257, 256, 8, 0) == 0                      # more than 256 experts
    assert lib.moe_nv_workspace_bytes(4, 10, 100) == 0                       # K not a multiple of 256
    null = ctypes.c_void_p()
    assert lib.moe_layer_fwd_mxfp8(ctypes.byref(ok), null, null, null, null, None, null, null, null, null, null, 0,
                                   null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_fwd_nvfp4(ctypes.byref(ok), null, null, null, null, None, null, null, 0,
                                   null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_nv_grouped_gemm(4, 100, 256, 64, null, null, null, null, null, null, null, 0,
                                   null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_nv_grouped_gemm(4, 100, 200, 64, null, null, null, null, null, null, null, 0,
                                   null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_layer_fwd_mxfp8_train(ctypes.byref(ok), null, null, null, null, None, null, None, null, 0,
                                         null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_fwd_mxfp8_train(ctypes.byref(shared), null, null, null, null, None, null, None, null, 0,
                                         null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_layer_bwd_mxfp8(ctypes.byref(ok), null, null, null, None, None, null, null, null, null, null,
                                   null, 1, null, 0, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize_bwd_weights(ctypes.byref(bad_h), null, null, null, None,
                                           null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_mx_quantize(null, 10, 33, null, null, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_nv_quantize(null, 10, 32, null, null, null, null) == ops.MOE_ERR_INVALID_ARG
    # the NVFP4 training step
    for i in range(6):
        assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(ok), i) > 0
        assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(bad_f), i) == 0
        assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(shared), i) == 0
    assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(ok), 0) == 8 * 256 * 128      # W2 rows along H: [E][F][H/2]
    assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(ok), 3) == 8 * 256 * 256      # [W1 | W3] along 2F: [E][H][F]
    assert lib.moe_nv_bwd_weight_bytes(ctypes.byref(ok), 5) == 4 * 8
    assert lib.moe_nv_train_workspace_bytes(ctypes.byref(ok)) > lib.moe_nv_workspace_bytes_layer(ctypes.byref(ok))
    assert lib.moe_nv_train_workspace_bytes(ctypes.byref(shared)) == 0
    assert lib.moe_layer_fwd_nvfp4_train(ctypes.byref(ok), null, null, null, null, None, null, None, null, 0,
                                         null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_fwd_nvfp4_train(ctypes.byref(bad_f), null, null, null, null, None, null, None, null, 0,
                                         null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_layer_bwd_nvfp4(ctypes.byref(ok), null, null, null, None, None, null, null, null, null, null,
                                   null, null, 0, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_nv_quantize_bwd_weights(ctypes.byref(bad_h), null, null, null, None,
                                           null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_nv_quantize_train_weights(ctypes.byref(bad_h), null, null, null, None, None,
                                             null) == ops.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_nv_quantize_train_weights(ctypes.byref(ok), null, null, null, None, None,
                                             null) == ops.MOE_ERR_INVALID_ARG


def test_read_ceiling_checks_on_the_host(lib):
    # the measurement helpers reject null and misaligned arguments before any
    # CUDA work
    null = ctypes.c_void_p()
    some = ctypes.c_void_p(4096)
    assert lib.moe_read_ceiling(null, 1024, some, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_read_ceiling(some, 1024, null, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_read_ceiling(ctypes.c_void_p(4100), 1024, some, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_read_ceiling(some, 1000, some, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_read_ceiling(some, 1024, ctypes.c_void_p(4100), null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_read_ceiling(some, 0, some, null) == ops.MOE_OK
    assert lib.moe_write_ceiling(null, 1024, 0, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_write_ceiling(ctypes.c_void_p(4100), 1024, 0, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_write_ceiling(some, 1000, 0, null) == ops.MOE_ERR_INVALID_ARG
    assert lib.moe_write_ceiling(some, 0, 0, null) == ops.MOE_OK


def test_default_build_is_not_the_bounds_check_build(lib):
    assert lib.moe_bounds_checked() == 0


def _misaligned_each(call, n_ptrs, structs=()):
    """Run `call(ptrs, structs)` with every pointer 16-byte aligned, then with
    one pointer (or one field of one struct) moved by 8 bytes at a time; yield
    (what was moved, status)."""
    good, bad = 4096, 4096 + 8
    ptrs = [ctypes.c_void_p(good) for _ in range(n_ptrs)]
    mk = [lambda S=S: S(*([good] * len(S._fields_))) for S in structs]
    yield "none", call(ptrs, [m() for m in mk])
    for i in range(n_ptrs):
        p = list(ptrs)
        p[i] = ctypes.c_void_p(bad)
        yield f"pointer {i}", call(p, [m() for m in mk])
    for j, S in enumerate(structs):
        for name, _ in S._fields_:
            st = [m() for m in mk]
            setattr(st[j], name, bad)
            yield f"{S.__name__}.{name}", call(ptrs, st)


def test_every_device_pointer_is_checked_for_alignment(lib):
    """The header's convention (every device pointer 16-byte aligned; the
    kernels reach them with 16-byte vector accesses and TMA copies) is checked
    on each pointer an entry point takes, saved-tensor and weight-struct
    fields included, before anything is enqueued. The workspace size given is
    too small, so a pointer the check missed would show as
    MOE_ERR_WORKSPACE_TOO_SMALL, never as a launch."""
    small = 16
    shared = ops.make_config(256, 256, 8, 2, 256, F_shared=64, aux_coeff=0.01)
    plain = ops.make_config(256, 256, 8, 2, 256, aux_coeff=0.01)
    B = ctypes.byref
    cases = {
        "moe_router_topk": (9, (), lambda p, s: lib.moe_router_topk(B(plain), *p, small, None)),
        "moe_permute": (7, (), lambda p, s: lib.moe_permute(B(plain), *p, small, None)),
        "moe_grouped_swiglu_ffn": (9, (), lambda p, s: lib.moe_grouped_swiglu_ffn(B(plain), *p, small, None)),
        "moe_layer_fwd": (12, (ops.MoeFwdSaved,), lambda p, s: lib.moe_layer_fwd(
            B(shared), *p[:11], B(s[0]), p[11], small, None)),
        "moe_layer_bwd": (19, (ops.MoeFwdSaved,), lambda p, s: lib.moe_layer_bwd(
            B(shared), *p[:9], B(s[0]), *p[9:19], small, None)),
        "moe_layer_fwd_mxfp8": (9, (ops.MoeMxWeights,), lambda p, s: lib.moe_layer_fwd_mxfp8(
            B(shared), *p[:4], B(s[0]), *p[4:9], small, None)),
        "moe_layer_fwd_mxfp8_train": (6, (ops.MoeMxWeights, ops.MoeFwdSaved), lambda p, s: (
            lib.moe_layer_fwd_mxfp8_train(B(plain), *p[:4], B(s[0]), p[4], B(s[1]), p[5], small, None))),
        "moe_layer_bwd_mxfp8": (10, (ops.MoeMxBwdWeights, ops.MoeFwdSaved), lambda p, s: lib.moe_layer_bwd_mxfp8(
            B(plain), *p[:3], B(s[0]), B(s[1]), *p[3:9], 0, p[9], small, None)),
        "moe_layer_fwd_nvfp4": (6, (ops.MoeNvWeights,), lambda p, s: lib.moe_layer_fwd_nvfp4(
            B(plain), *p[:4], B(s[0]), p[4], p[5], small, None)),
        "moe_layer_fwd_nvfp4_train": (6, (ops.MoeNvWeights, ops.MoeFwdSaved), lambda p, s: (
            lib.moe_layer_fwd_nvfp4_train(B(plain), *p[:4], B(s[0]), p[4], B(s[1]), p[5], small, None))),
        "moe_layer_bwd_nvfp4": (10, (ops.MoeNvBwdWeights, ops.MoeFwdSaved), lambda p, s: lib.moe_layer_bwd_nvfp4(
            B(plain), *p[:3], B(s[0]), B(s[1]), *p[3:10], small, None)),
        "moe_nv_grouped_gemm": (7, (), lambda p, s: lib.moe_nv_grouped_gemm(4, 100, 256, 64, *p, small, None)),
    }
    for fn, (n, structs, call) in cases.items():
        for what, st in _misaligned_each(call, n, structs):
            want = ops.MOE_ERR_WORKSPACE_TOO_SMALL if what == "none" else ops.MOE_ERR_INVALID_ARG
            assert st == want, f"{fn}: {what} misaligned -> {st}"


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="entry points without a workspace would launch if a check were missing")
def test_alignment_of_entry_points_without_a_workspace(lib):
    plain = ops.make_config(256, 256, 8, 2, 256)
    B = ctypes.byref
    cases = {
        "moe_unpermute_combine": (5, (), lambda p, s: lib.moe_unpermute_combine(B(plain), *p, None)),
        "moe_permute_noalloc": (6, (), lambda p, s: lib.moe_permute_noalloc(B(plain), *p, None)),
        "moe_mx_quantize": (3, (), lambda p, s: lib.moe_mx_quantize(p[0], 64, 256, p[1], p[2], None)),
        "moe_nv_quantize": (4, (), lambda p, s: lib.moe_nv_quantize(p[0], 64, 256, *p[1:4], None)),
        "moe_nv_quantize_weights": (4, (), lambda p, s: lib.moe_nv_quantize_weights(4, 256, 64, *p, None)),
        "moe_mx_quantize_weights": (3, (ops.MoeMxWeights,), lambda p, s: lib.moe_mx_quantize_weights(
            B(plain), *p, B(s[0]), None)),
        "moe_mx_quantize_bwd_weights": (3, (ops.MoeMxBwdWeights,), lambda p, s: lib.moe_mx_quantize_bwd_weights(
            B(plain), *p, B(s[0]), None)),
        "moe_nv_quantize_layer_weights": (3, (ops.MoeNvWeights,), lambda p, s: lib.moe_nv_quantize_layer_weights(
            B(plain), *p, B(s[0]), None)),
        "moe_nv_quantize_bwd_weights": (3, (ops.MoeNvBwdWeights,), lambda p, s: lib.moe_nv_quantize_bwd_weights(
            B(plain), *p, B(s[0]), None)),
        "moe_nv_quantize_train_weights": (3, (ops.MoeNvWeights, ops.MoeNvBwdWeights),
                                          lambda p, s: lib.moe_nv_quantize_train_weights(B(plain), *p, B(s[0]),
                                                                                         B(s[1]), None)),
    }
    for fn, (n, structs, call) in cases.items():
        for what, st in _misaligned_each(call, n, structs):
            if what != "none":
                assert st == ops.MOE_ERR_INVALID_ARG, f"{fn}: {what} misaligned -> {st}"
