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


def test_binding_structs_match_the_library(lib):
    lib.moe_abi_struct_bytes.restype = ctypes.c_size_t
    assert lib.moe_abi_struct_bytes(0) == ctypes.sizeof(ops.MoeConfig)
    assert lib.moe_abi_struct_bytes(1) == ctypes.sizeof(ops.MoeFwdSaved)
    assert lib.moe_abi_struct_bytes(2) == 0
