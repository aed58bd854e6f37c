"""Python binding of the C ABI in ``include/moe_route_permute.h``.

Argument marshalling only: tensors are allocated with torch on the current CUDA
device, their data pointers and torch's current stream are handed to the
library, and every step of the path runs in the library's kernels. There is no
fallback: if the compiled library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_longlong, c_size_t, c_void_p

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_INDEX = 6
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace too small",
                4: "CUDA error", 5: "device: bounded wait ran out", 6: "device: index out of range"}
SCORE = {"softmax": 0, "sigmoid": 1}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", c_int), ("H", c_int), ("E", c_int), ("k", c_int), ("F", c_int), ("F_shared", c_int),
                ("score", c_int), ("n_groups", c_int), ("topk_groups", c_int), ("gate_scale", c_float),
                ("aux_coeff", c_float), ("out_fp32", c_int), ("inter_fp32", c_int), ("force_balanced", c_int)]


class MoeFwdSaved(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("topk_idx", "topk_gate", "logits", "row_id_map", "counts", "offsets",
                                        "x_perm", "h13", "a", "y_perm", "aux_partials", "h13_shared",
                                        "a_shared")]


_lib = None


def library_path() -> str:
    """The library this process loads: the bounds-check build when the
    environment sets MOE_BOUNDS_CHECK=1, else the default build."""
    return _build.LIB_CHECKED if os.environ.get("MOE_BOUNDS_CHECK") == "1" else _build.LIB


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: run route_permute_grouped_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp = c_void_p
        L.moe_abi_struct_bytes.restype = c_size_t
        L.moe_abi_struct_bytes.argtypes = [c_int]
        if (L.moe_abi_struct_bytes(0) != ctypes.sizeof(MoeConfig)
                or L.moe_abi_struct_bytes(1) != ctypes.sizeof(MoeFwdSaved)):
            raise RuntimeError("moe_config / moe_fwd_saved layout of the binding differs from the library")
        L.moe_workspace_bytes.restype = c_size_t
        L.moe_workspace_bytes.argtypes = [POINTER(MoeConfig), c_int]
        L.moe_router_topk.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        L.moe_permute.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        L.moe_grouped_swiglu_ffn.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        L.moe_unpermute_combine.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp]
        L.moe_layer_fwd.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    POINTER(MoeFwdSaved), vp, c_size_t, vp]
        L.moe_layer_bwd.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, vp, vp, vp, vp, vp, POINTER(MoeFwdSaved),
                                    vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        L.moe_get_device_status.argtypes = [vp, vp, POINTER(c_int)]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [c_int]
        L.moe_debug_set_wait_limit_ns.argtypes = [c_longlong]
        L.moe_debug_set_wait_limit_ns.restype = None
        L.moe_debug_set_fault.argtypes = [c_int]
        L.moe_debug_set_fault.restype = None
        for n in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu_ffn", "moe_unpermute_combine",
                  "moe_layer_fwd", "moe_layer_bwd", "moe_get_device_status"):
            getattr(L, n).restype = c_int
        L.moe_profile_start.argtypes = [c_int]
        L.moe_profile_start.restype = None
        L.moe_profile_stop.argtypes = []
        L.moe_profile_stop.restype = None
        L.moe_profile_read.argtypes = [POINTER(c_int), POINTER(c_float), c_int]
        L.moe_profile_read.restype = c_int
        L.moe_debug_launch_count.argtypes = []
        L.moe_debug_launch_count.restype = ctypes.c_ulonglong
        L.moe_bounds_checked.argtypes = []
        L.moe_bounds_checked.restype = c_int
        L.moe_read_ceiling.argtypes = [vp, c_size_t, vp, vp]
        L.moe_read_ceiling.restype = c_int
        L.moe_write_ceiling.argtypes = [vp, c_size_t, ctypes.c_uint, vp]
        L.moe_write_ceiling.restype = c_int
        L.moe_debug_workspace_offset.argtypes = [POINTER(MoeConfig), c_int, c_int]
        L.moe_debug_workspace_offset.restype = c_size_t
        L.moe_mx_weight_bytes.restype = c_size_t
        L.moe_mx_weight_bytes.argtypes = [POINTER(MoeConfig), c_int]
        L.moe_mx_workspace_bytes.restype = c_size_t
        L.moe_mx_workspace_bytes.argtypes = [POINTER(MoeConfig)]
        L.moe_mx_quantize_weights.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeMxWeights), vp]
        L.moe_mx_quantize.argtypes = [vp, c_longlong, c_int, vp, vp, vp]
        L.moe_layer_fwd_mxfp8.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, POINTER(MoeMxWeights), vp, vp, vp, vp,
                                          vp, c_size_t, vp]
        for n in ("moe_mx_quantize_weights", "moe_mx_quantize", "moe_layer_fwd_mxfp8"):
            getattr(L, n).restype = c_int
        L.moe_mx_bwd_weight_bytes.restype = c_size_t
        L.moe_mx_bwd_weight_bytes.argtypes = [POINTER(MoeConfig), c_int]
        L.moe_mx_train_workspace_bytes.restype = c_size_t
        L.moe_mx_train_workspace_bytes.argtypes = [POINTER(MoeConfig)]
        L.moe_mx_quantize_bwd_weights.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeMxBwdWeights), vp]
        L.moe_layer_fwd_mxfp8_train.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, POINTER(MoeMxWeights), vp,
                                                POINTER(MoeFwdSaved), vp, c_size_t, vp]
        L.moe_layer_bwd_mxfp8.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeMxBwdWeights),
                                          POINTER(MoeFwdSaved), vp, vp, vp, vp, vp, vp, c_int, vp, c_size_t, vp]
        for n in ("moe_mx_quantize_bwd_weights", "moe_layer_fwd_mxfp8_train", "moe_layer_bwd_mxfp8"):
            getattr(L, n).restype = c_int
        L.moe_nv_weight_bytes.restype = c_size_t
        L.moe_nv_weight_bytes.argtypes = [c_int, c_int, c_int, c_int]
        L.moe_nv_workspace_bytes.restype = c_size_t
        L.moe_nv_workspace_bytes.argtypes = [c_int, c_longlong, c_int]
        L.moe_nv_quantize_weights.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp]
        L.moe_nv_quantize.argtypes = [vp, c_longlong, c_int, vp, vp, vp, vp]
        L.moe_nv_grouped_gemm.argtypes = [c_int, c_longlong, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        for n in ("moe_nv_quantize_weights", "moe_nv_quantize", "moe_nv_grouped_gemm"):
            getattr(L, n).restype = c_int
        L.moe_nv_layer_weight_bytes.restype = c_size_t
        L.moe_nv_layer_weight_bytes.argtypes = [POINTER(MoeConfig), c_int]
        L.moe_nv_workspace_bytes_layer.restype = c_size_t
        L.moe_nv_workspace_bytes_layer.argtypes = [POINTER(MoeConfig)]
        L.moe_nv_quantize_layer_weights.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeNvWeights), vp]
        L.moe_layer_fwd_nvfp4.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, POINTER(MoeNvWeights), vp, vp,
                                          c_size_t, vp]
        for n in ("moe_nv_quantize_layer_weights", "moe_layer_fwd_nvfp4"):
            getattr(L, n).restype = c_int
        L.moe_nv_bwd_weight_bytes.restype = c_size_t
        L.moe_nv_bwd_weight_bytes.argtypes = [POINTER(MoeConfig), c_int]
        L.moe_nv_train_workspace_bytes.restype = c_size_t
        L.moe_nv_train_workspace_bytes.argtypes = [POINTER(MoeConfig)]
        L.moe_nv_quantize_bwd_weights.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeNvBwdWeights), vp]
        L.moe_nv_quantize_train_weights.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeNvWeights),
                                                    POINTER(MoeNvBwdWeights), vp]
        L.moe_layer_fwd_nvfp4_train.argtypes = [POINTER(MoeConfig), vp, vp, vp, vp, POINTER(MoeNvWeights), vp,
                                                POINTER(MoeFwdSaved), vp, c_size_t, vp]
        L.moe_layer_bwd_nvfp4.argtypes = [POINTER(MoeConfig), vp, vp, vp, POINTER(MoeNvBwdWeights),
                                          POINTER(MoeFwdSaved), vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
        for n in ("moe_nv_quantize_bwd_weights", "moe_nv_quantize_train_weights", "moe_layer_fwd_nvfp4_train",
                  "moe_layer_bwd_nvfp4"):
            getattr(L, n).restype = c_int
        _lib = L
    return _lib


STAGE_NAMES = {20: "nv_quantize", 21: "nv_gemm", 22: "mx_quantize_tokens", 24: "mx_dgrad_down_swiglu",
               25: "mx_dgrad_gate_up", 26: "shared_dgrad_down_swiglu", 27: "shared_wgrad_down",
               28: "shared_dgrad_gate_up", 29: "shared_wgrad_gate_up", 1: "router", 2: "permute", 3: "ffn1_gate_up", 4: "ffn2_down", 5: "shared_gate_up",
               6: "shared_down", 7: "combine", 10: "combine_bwd", 11: "router_bwd_elem", 12: "dgrad_down_swiglu",
               13: "wgrad_down", 14: "dgrad_gate_up", 15: "wgrad_gate_up", 16: "router_dgrad",
               17: "permute_bwd", 18: "router_wgrad", 19: "aux_loss", 30: "read_ceiling",
               31: "write_ceiling", 32: "nv_dgrad_down", 33: "nv_swiglu_bwd", 34: "nv_dgrad_gate_up"}


def profile_start(capacity: int) -> None:
    lib().moe_profile_start(int(capacity))


def profile_stop() -> None:
    lib().moe_profile_stop()


def profile_read(max_events: int):
    """[(stage name, ms)] for every recorded stage, in order."""
    tags = (c_int * max_events)()
    ms = (c_float * max_events)()
    n = lib().moe_profile_read(tags, ms, max_events)
    if n < 0:
        raise MoeError(4, "moe_profile_read")
    return [(STAGE_NAMES.get(tags[i], str(tags[i])), float(ms[i])) for i in range(n) if tags[i] != 0]


def read_ceiling(buf: torch.Tensor, sink: torch.Tensor) -> None:
    """moe_read_ceiling over the bytes of a contiguous CUDA tensor (a
    measurement helper: one read-only pass; time it with events)."""
    assert buf.is_cuda and buf.is_contiguous() and sink.is_cuda
    nbytes = buf.numel() * buf.element_size() // 16 * 16
    _check(lib().moe_read_ceiling(_p(buf), nbytes, _p(sink), _stream()), "moe_read_ceiling")


def write_ceiling(buf: torch.Tensor, word: int = 0) -> None:
    """moe_write_ceiling over the bytes of a contiguous CUDA tensor (a
    measurement helper: one write-only pass; time it with events)."""
    assert buf.is_cuda and buf.is_contiguous()
    nbytes = buf.numel() * buf.element_size() // 16 * 16
    _check(lib().moe_write_ceiling(_p(buf), nbytes, int(word) & 0xFFFFFFFF, _stream()), "moe_write_ceiling")


def launch_count() -> int:
    return int(lib().moe_debug_launch_count())


WS_TENSORS = {"dy_perm": 0, "dh13": 1, "a": 2, "dx_perm": 3}


def workspace_tensor(ws, cfg, training, name):
    """Test hook: a view of an intermediate the layer keeps in the workspace
    (bf16 dy_perm [R,H], dh13 [R,2F], a [R,F]; dx_perm [R,H], fp32 with
    inter_fp32)."""
    off = int(lib().moe_debug_workspace_offset(ctypes.byref(cfg), int(training), WS_TENSORS[name]))
    if off == ctypes.c_size_t(-1).value:
        raise MoeError(1, "moe_debug_workspace_offset")
    R = cfg.T * cfg.k
    cols = {"dy_perm": cfg.H, "dh13": 2 * cfg.F, "a": cfg.F, "dx_perm": cfg.H}[name]
    dt = torch.float32 if (name == "dx_perm" and cfg.inter_fp32) else torch.bfloat16
    nb = R * cols * (4 if dt == torch.float32 else 2)
    return ws[off:off + nb].view(dt).view(R, cols)


def _p(t):
    if t is None:
        return None
    assert t.is_contiguous(), "tensors must be contiguous"
    return c_void_p(t.data_ptr())


def _stream():
    return c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(st, where):
    if st != MOE_OK:
        raise MoeError(st, where)


def make_config(T, H, E, k, F, F_shared=0, score="softmax", n_groups=1, topk_groups=1, gate_scale=1.0,
                aux_coeff=0.0, out_fp32=False, inter_fp32=False, force_balanced=False) -> MoeConfig:
    return MoeConfig(T, H, E, k, F, F_shared, SCORE[score] if isinstance(score, str) else score, n_groups,
                     topk_groups, gate_scale, aux_coeff, int(out_fp32), int(inter_fp32), int(force_balanced))


def config_from_shape(ls, **over) -> MoeConfig:
    d = dict(T=ls.T, H=ls.H, E=ls.E, k=ls.k, F=ls.F, F_shared=ls.F_shared, score=ls.score, n_groups=ls.n_groups,
             topk_groups=ls.topk_groups, gate_scale=ls.gate_scale, aux_coeff=ls.aux_coeff, out_fp32=ls.out_fp32,
             inter_fp32=ls.inter_fp32, force_balanced=getattr(ls, "force_balanced", False))
    d.update(over)
    return make_config(**d)


def workspace_bytes(cfg: MoeConfig, training: bool = False) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg), int(training)))


def workspace(cfg: MoeConfig, training: bool = False, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg, training)
    if n == 0:
        raise MoeError(1, "moe_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()  # device status word
    return ws


def device_status(ws: torch.Tensor) -> int:
    out = c_int(0)
    _check(lib().moe_get_device_status(_p(ws), _stream(), ctypes.byref(out)), "moe_get_device_status")
    return out.value


def set_wait_limit_ns(ns: int) -> None:
    lib().moe_debug_set_wait_limit_ns(int(ns))


def set_fault(f: int) -> None:
    lib().moe_debug_set_fault(int(f))


def _inter_dtype(cfg):
    return torch.float32 if cfg.inter_fp32 else torch.bfloat16


def _out_dtype(cfg):
    return torch.float32 if cfg.out_fp32 else torch.bfloat16


def router_topk(cfg, x, router_w, expert_bias=None, logit_bias=None, want_logits=False, want_aux=False, ws=None):
    dev = x.device
    T, E, k = cfg.T, cfg.E, cfg.k
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if want_logits else None
    aux = torch.empty((4 * ((T + 127) // 128), E), dtype=torch.float32, device=dev) if want_aux else None
    ws = workspace(cfg, False, dev) if ws is None else ws
    st = lib().moe_router_topk(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias), _p(idx),
                               _p(gate), _p(logits), _p(aux), _p(ws), ws.numel(), _stream())
    _check(st, "moe_router_topk")
    return idx, gate, logits, aux


def permute(cfg, x, topk_idx, ws=None):
    dev = x.device
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    x_perm = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    rows = torch.empty((T, k), dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ws = workspace(cfg, False, dev) if ws is None else ws
    st = lib().moe_permute(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(x_perm), _p(rows), _p(counts), _p(offsets),
                           _p(ws), ws.numel(), _stream())
    _check(st, "moe_permute")
    return x_perm, rows, counts, offsets


def grouped_swiglu_ffn(cfg, x_perm, offsets, W1, W3, W2, save=False, ws=None):
    dev = x_perm.device
    R, H, F = cfg.T * cfg.k, cfg.H, cfg.F
    y_perm = torch.empty((R, H), dtype=_inter_dtype(cfg), device=dev)
    h13 = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev) if save else None
    a = torch.empty((R, F), dtype=torch.bfloat16, device=dev) if save else None
    ws = workspace(cfg, False, dev) if ws is None else ws
    st = lib().moe_grouped_swiglu_ffn(ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(W1), _p(W3), _p(W2), _p(h13),
                                      _p(a), _p(y_perm), _p(ws), ws.numel(), _stream())
    _check(st, "moe_grouped_swiglu_ffn")
    return y_perm, h13, a


def unpermute_combine(cfg, y_perm, row_id_map, topk_gate, shared=None):
    y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=y_perm.device)
    st = lib().moe_unpermute_combine(ctypes.byref(cfg), _p(y_perm), _p(row_id_map), _p(topk_gate), _p(shared),
                                     _p(y), _stream())
    _check(st, "moe_unpermute_combine")
    return y


def alloc_saved(cfg, device="cuda", recompute=False):
    """Tensors the training forward keeps for the backward. ``recompute``:
    the memory-saving mode, which keeps neither ``a`` nor ``y_perm`` (the
    backward recomputes ``a`` from ``h13`` and takes the gate gradient from
    the down-projection dgrad)."""
    T, H, E, k, F = cfg.T, cfg.H, cfg.E, cfg.k, cfg.F
    R = T * k
    f32, i32, bf = torch.float32, torch.int32, torch.bfloat16
    return {
        "topk_idx": torch.empty((T, k), dtype=i32, device=device),
        "topk_gate": torch.empty((T, k), dtype=f32, device=device),
        "logits": torch.empty((T, E), dtype=f32, device=device),
        "row_id_map": torch.empty((T, k), dtype=i32, device=device),
        "counts": torch.empty(E, dtype=i32, device=device),
        "offsets": torch.empty(E + 1, dtype=i32, device=device),
        "x_perm": torch.empty((R, H), dtype=bf, device=device),
        "h13": torch.empty((R, 2 * F), dtype=bf, device=device),
        "a": None if recompute else torch.empty((R, F), dtype=bf, device=device),
        "y_perm": None if recompute else torch.empty((R, H), dtype=_inter_dtype(cfg), device=device),
        "aux_partials": torch.empty((4 * ((T + 127) // 128), E), dtype=f32, device=device) if cfg.aux_coeff else None,
        "h13_shared": torch.empty((T, 2 * cfg.F_shared), dtype=bf, device=device) if cfg.F_shared else None,
        "a_shared": torch.empty((T, cfg.F_shared), dtype=bf, device=device) if cfg.F_shared else None,
    }


def _saved_struct(saved):
    return MoeFwdSaved(*[None if saved.get(n) is None else saved[n].data_ptr() for n, _ in MoeFwdSaved._fields_])


def layer_fwd(cfg, x, router_w, W1, W3, W2, expert_bias=None, logit_bias=None, Ws=None, saved=None, ws=None, y=None):
    """Whole layer forward. ``saved`` (from alloc_saved) makes it a training
    forward that keeps the tensors the backward needs."""
    dev = x.device
    if y is None:
        y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=dev)
    ws = workspace(cfg, saved is not None, dev) if ws is None else ws
    Ws1, Ws3, Ws2 = Ws if Ws is not None else (None, None, None)
    sv = ctypes.byref(_saved_struct(saved)) if saved is not None else None
    st = lib().moe_layer_fwd(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias), _p(W1),
                             _p(W3), _p(W2), _p(Ws1), _p(Ws3), _p(Ws2), _p(y), sv, _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_fwd")
    return y


def alloc_grads(cfg, device="cuda"):
    T, H, E, F, Fs = cfg.T, cfg.H, cfg.E, cfg.F, cfg.F_shared
    f32 = torch.float32
    g = {
        "dx": torch.empty((T, H), dtype=_out_dtype(cfg), device=device),
        "dW_r": torch.empty((E, H), dtype=f32, device=device),
        "dW1": torch.empty((E, H, F), dtype=f32, device=device),
        "dW3": torch.empty((E, H, F), dtype=f32, device=device),
        "dW2": torch.empty((E, F, H), dtype=f32, device=device),
        "aux_loss": torch.zeros(1, dtype=f32, device=device),
    }
    if Fs:  # the shared expert's weight gradients
        g["dWs1"] = torch.empty((H, Fs), dtype=f32, device=device)
        g["dWs3"] = torch.empty((H, Fs), dtype=f32, device=device)
        g["dWs2"] = torch.empty((Fs, H), dtype=f32, device=device)
    return g


def layer_bwd(cfg, dO, x, router_w, W1, W3, W2, saved, ws=None, grads=None, Ws=None):
    """Whole layer backward (``Ws``: the shared expert's weights when
    cfg.F_shared > 0; its gradients land in grads dWs1, dWs3, dWs2)."""
    dev = x.device
    g = alloc_grads(cfg, dev) if grads is None else grads
    ws = workspace(cfg, True, dev) if ws is None else ws
    sv = _saved_struct(saved)
    Ws1, Ws3, Ws2 = Ws if Ws is not None else (None, None, None)
    st = lib().moe_layer_bwd(ctypes.byref(cfg), _p(dO), _p(x), _p(router_w), _p(W1), _p(W3), _p(W2), _p(Ws1),
                             _p(Ws3), _p(Ws2), ctypes.byref(sv), _p(g["dx"]), _p(g["dW_r"]), _p(g["dW1"]),
                             _p(g["dW3"]), _p(g["dW2"]), _p(g.get("dWs1")), _p(g.get("dWs3")), _p(g.get("dWs2")),
                             _p(g["aux_loss"]), _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_bwd")
    return g


# ---------------------------------------------------------------------------
# MXFP8 expert GEMMs (forward)
# ---------------------------------------------------------------------------
class MoeMxWeights(ctypes.Structure):
    """Mirror of moe_mx_weights (four device pointers)."""
    _fields_ = [("w13", c_void_p), ("sf13", c_void_p), ("w2", c_void_p), ("sf2", c_void_p)]


MX_WEIGHT_FIELDS = ("w13", "sf13", "w2", "sf2")


def mx_quantize_weights(cfg, W1, W3, W2):
    """Quantise the bf16 expert weights into new uint8 device tensors (dict
    with keys w13 [E,2,F,H], sf13, w2 [E,H,F], sf2)."""
    dev = W1.device
    out = {}
    for i, n in enumerate(MX_WEIGHT_FIELDS):
        nb = int(lib().moe_mx_weight_bytes(ctypes.byref(cfg), i))
        if nb == 0:
            raise MoeError(2, "moe_mx_weight_bytes")
        out[n] = torch.empty(nb, dtype=torch.uint8, device=dev)
    out["w13"] = out["w13"].view(cfg.E, 2, cfg.F, cfg.H)
    out["w2"] = out["w2"].view(cfg.E, cfg.H, cfg.F)
    st = lib().moe_mx_quantize_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2), ctypes.byref(_mx_struct(out)),
                                       _stream())
    _check(st, "moe_mx_quantize_weights")
    return out


def _mx_struct(w):
    return MoeMxWeights(*[w[n].data_ptr() for n in MX_WEIGHT_FIELDS])


def mx_quantize(x):
    """Row-major MXFP8 quantisation of a bf16 [M, K] tensor: (codes uint8
    [M, K], scales uint8 [M, K/32])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((M, K // 32), dtype=torch.uint8, device=x.device)
    _check(lib().moe_mx_quantize(_p(x), M, K, _p(q), _p(s), _stream()), "moe_mx_quantize")
    return q, s


def mx_workspace(cfg, device="cuda"):
    n = int(lib().moe_mx_workspace_bytes(ctypes.byref(cfg)))
    if n == 0:
        raise MoeError(2, "moe_mx_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def layer_fwd_mxfp8(cfg, x, router_w, mxw, expert_bias=None, logit_bias=None, Ws=None, ws=None, y=None):
    """Whole layer forward with MXFP8 expert GEMMs (``mxw`` from
    mx_quantize_weights)."""
    dev = x.device
    if y is None:
        y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=dev)
    ws = mx_workspace(cfg, dev) if ws is None else ws
    Ws1, Ws3, Ws2 = Ws if Ws is not None else (None, None, None)
    st = lib().moe_layer_fwd_mxfp8(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias),
                                   ctypes.byref(_mx_struct(mxw)), _p(Ws1), _p(Ws3), _p(Ws2), _p(y), _p(ws),
                                   ws.numel(), _stream())
    _check(st, "moe_layer_fwd_mxfp8")
    return y


# ---------------------------------------------------------------------------
# MXFP8 training step (forward saving, backward with MXFP8 data gradients)
# ---------------------------------------------------------------------------
class MoeMxBwdWeights(ctypes.Structure):
    """Mirror of moe_mx_bwd_weights (four device pointers)."""
    _fields_ = [("w2h", c_void_p), ("sf2h", c_void_p), ("w13f", c_void_p), ("sf13f", c_void_p)]


MX_BWD_WEIGHT_FIELDS = ("w2h", "sf2h", "w13f", "sf13f")


def mx_quantize_bwd_weights(cfg, W1, W3, W2):
    """Weights of the MXFP8 data-gradient GEMMs as new uint8 device tensors:
    w2h [E,F,H] (W2 along H), w13f [E,H,2F] (W1 | W3 along F), sf2h, sf13f."""
    dev = W1.device
    out = {}
    for i, n in enumerate(MX_BWD_WEIGHT_FIELDS):
        nb = int(lib().moe_mx_bwd_weight_bytes(ctypes.byref(cfg), i))
        if nb == 0:
            raise MoeError(2, "moe_mx_bwd_weight_bytes")
        out[n] = torch.empty(nb, dtype=torch.uint8, device=dev)
    out["w2h"] = out["w2h"].view(cfg.E, cfg.F, cfg.H)
    out["w13f"] = out["w13f"].view(cfg.E, cfg.H, 2 * cfg.F)
    w = MoeMxBwdWeights(*[out[n].data_ptr() for n in MX_BWD_WEIGHT_FIELDS])
    _check(lib().moe_mx_quantize_bwd_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2), ctypes.byref(w), _stream()),
           "moe_mx_quantize_bwd_weights")
    return out


def mx_train_workspace(cfg, device="cuda"):
    n = int(lib().moe_mx_train_workspace_bytes(ctypes.byref(cfg)))
    if n == 0:
        raise MoeError(2, "moe_mx_train_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def alloc_saved_mxfp8(cfg, device="cuda"):
    """Saved tensors of the MXFP8 training forward (``a`` is not kept: the
    backward recomputes it from ``h13``)."""
    sv = alloc_saved(cfg, device)
    sv["a"] = None
    return sv


def layer_fwd_mxfp8_train(cfg, x, router_w, mxw, saved, expert_bias=None, logit_bias=None, ws=None, y=None):
    """Training forward of the MXFP8 layer (``saved`` from alloc_saved_mxfp8)."""
    dev = x.device
    if y is None:
        y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=dev)
    ws = mx_train_workspace(cfg, dev) if ws is None else ws
    st = lib().moe_layer_fwd_mxfp8_train(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias),
                                         ctypes.byref(_mx_struct(mxw)), _p(y), ctypes.byref(_saved_struct(saved)),
                                         _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_fwd_mxfp8_train")
    return y


def layer_bwd_mxfp8(cfg, dO, x, router_w, mxbw, saved, ws=None, grads=None, mx_wgrad=False):
    """Backward of the MXFP8 training step (``mxbw`` from
    mx_quantize_bwd_weights); gradients as layer_bwd. ``mx_wgrad``: the weight
    gradients in MXFP8 too (operands quantised along each expert's tokens)."""
    dev = x.device
    g = alloc_grads(cfg, dev) if grads is None else grads
    ws = mx_train_workspace(cfg, dev) if ws is None else ws
    w = MoeMxBwdWeights(*[mxbw[n].data_ptr() for n in MX_BWD_WEIGHT_FIELDS])
    st = lib().moe_layer_bwd_mxfp8(ctypes.byref(cfg), _p(dO), _p(x), _p(router_w), ctypes.byref(w),
                                   ctypes.byref(_saved_struct(saved)), _p(g["dx"]), _p(g["dW_r"]), _p(g["dW1"]),
                                   _p(g["dW3"]), _p(g["dW2"]), _p(g["aux_loss"]), int(bool(mx_wgrad)), _p(ws),
                                   ws.numel(), _stream())
    _check(st, "moe_layer_bwd_mxfp8")
    return g


# ---------------------------------------------------------------------------
# NVFP4 grouped expert GEMM
# ---------------------------------------------------------------------------
def nv_quantize_weights(W):
    """Quantise expert weights W [E, K, N] bf16: dict with wq [E, N, K/2]
    (codes, two per byte), sf (tile-ready E4M3 scales), g [E] fp32."""
    E, K, N = W.shape
    nb = [int(lib().moe_nv_weight_bytes(E, K, N, i)) for i in range(3)]
    if 0 in nb:
        raise MoeError(2, "moe_nv_weight_bytes")
    wq = torch.empty((E, N, K // 2), dtype=torch.uint8, device=W.device)
    sf = torch.empty(nb[1], dtype=torch.uint8, device=W.device)
    g = torch.empty(E, dtype=torch.float32, device=W.device)
    _check(lib().moe_nv_quantize_weights(E, K, N, _p(W), _p(wq), _p(sf), _p(g), _stream()), "moe_nv_quantize_weights")
    return {"wq": wq, "sf": sf, "g": g, "E": E, "K": K, "N": N}


def nv_quantize(x):
    """Row-major NVFP4 quantisation of x [M, K] bf16 as one tensor: (codes
    [M, K/2], scales [M, K/16], tensor scale [1])."""
    M, K = x.shape
    q = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    s = torch.empty((M, K // 16), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().moe_nv_quantize(_p(x), M, K, _p(q), _p(s), _p(g), _stream()), "moe_nv_quantize")
    return q, s, g


def nv_workspace(E, R, K, device="cuda"):
    n = int(lib().moe_nv_workspace_bytes(E, R, K))
    if n == 0:
        raise MoeError(2, "moe_nv_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def nv_grouped_gemm(x, offsets, w, ws=None, y=None):
    """y [R, N] bf16 = grouped NVFP4 GEMM of x [R, K] (rows grouped by
    ``offsets``, [E+1] int32 on the device) with quantised weights ``w``."""
    R, K = x.shape
    E, N = w["E"], w["N"]
    if y is None:
        y = torch.empty((R, N), dtype=torch.bfloat16, device=x.device)
    ws = nv_workspace(E, R, K, x.device) if ws is None else ws
    st = lib().moe_nv_grouped_gemm(E, R, K, N, _p(x), _p(offsets), _p(w["wq"]), _p(w["sf"]), _p(w["g"]), _p(y),
                                   _p(ws), ws.numel(), _stream())
    _check(st, "moe_nv_grouped_gemm")
    return y


class MoeNvWeights(ctypes.Structure):
    """Mirror of moe_nv_weights (six device pointers)."""
    _fields_ = [(n, c_void_p) for n in ("w13", "sf13", "g13", "w2", "sf2", "g2")]


def nv_quantize_layer_weights(cfg, W1, W3, W2):
    """NVFP4 weights of the layer (dict of uint8 / fp32 device tensors)."""
    out = {}
    for i, n in enumerate(MoeNvWeights._fields_):
        nb = int(lib().moe_nv_layer_weight_bytes(ctypes.byref(cfg), i))
        if nb == 0:
            raise MoeError(2, "moe_nv_layer_weight_bytes")
        dt = torch.float32 if n[0].startswith("g") else torch.uint8
        out[n[0]] = torch.empty(nb // (4 if dt == torch.float32 else 1), dtype=dt, device=W1.device)
    st = lib().moe_nv_quantize_layer_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2), ctypes.byref(_nv_struct(out)),
                                             _stream())
    _check(st, "moe_nv_quantize_layer_weights")
    return out


def _nv_struct(w):
    return MoeNvWeights(*[w[n[0]].data_ptr() for n in MoeNvWeights._fields_])


def layer_fwd_nvfp4(cfg, x, router_w, nvw, expert_bias=None, logit_bias=None, ws=None, y=None):
    """Whole layer forward with NVFP4 expert GEMMs (``nvw`` from
    nv_quantize_layer_weights)."""
    dev = x.device
    if y is None:
        y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=dev)
    if ws is None:
        n = int(lib().moe_nv_workspace_bytes_layer(ctypes.byref(cfg)))
        if n == 0:
            raise MoeError(2, "moe_nv_workspace_bytes_layer")
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        ws[:256].zero_()
    st = lib().moe_layer_fwd_nvfp4(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias),
                                   ctypes.byref(_nv_struct(nvw)), _p(y), _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_fwd_nvfp4")
    return y


# ---------------------------------------------------------------------------
# NVFP4 training step (forward saving, backward with NVFP4 data gradients)
# ---------------------------------------------------------------------------
class MoeNvBwdWeights(ctypes.Structure):
    """Mirror of moe_nv_bwd_weights (six device pointers)."""
    _fields_ = [(n, c_void_p) for n in ("w2h", "sf2h", "g2h", "w13f", "sf13f", "g13f")]


def nv_quantize_bwd_weights(cfg, W1, W3, W2):
    """Weights of the NVFP4 data-gradient GEMMs as new device tensors: w2h
    [E,F,H/2] (W2 along H), w13f [E,H,F] (W1 | W3 along 2F; codes two per
    byte), their tile-ready scales sf2h, sf13f and tensor scales g2h, g13f [E]."""
    out = {}
    for i, (n, _) in enumerate(MoeNvBwdWeights._fields_):
        nb = int(lib().moe_nv_bwd_weight_bytes(ctypes.byref(cfg), i))
        if nb == 0:
            raise MoeError(2, "moe_nv_bwd_weight_bytes")
        dt = torch.float32 if n.startswith("g") else torch.uint8
        out[n] = torch.empty(nb // (4 if dt == torch.float32 else 1), dtype=dt, device=W1.device)
    out["w2h"] = out["w2h"].view(cfg.E, cfg.F, cfg.H // 2)
    out["w13f"] = out["w13f"].view(cfg.E, cfg.H, cfg.F)
    w = MoeNvBwdWeights(*[out[n].data_ptr() for n, _ in MoeNvBwdWeights._fields_])
    _check(lib().moe_nv_quantize_bwd_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2), ctypes.byref(w), _stream()),
           "moe_nv_quantize_bwd_weights")
    return out


def _nv_alloc(cfg, size_fn, fields, device):
    out = {}
    for i, (n, _) in enumerate(fields):
        nb = int(size_fn(ctypes.byref(cfg), i))
        if nb == 0:
            raise MoeError(2, size_fn.__name__)
        dt = torch.float32 if n.startswith("g") else torch.uint8
        out[n] = torch.empty(nb // (4 if dt == torch.float32 else 1), dtype=dt, device=device)
    return out


def nv_quantize_train_weights(cfg, W1, W3, W2):
    """Both weight copies of the NVFP4 training step in one call (the maxima
    taken once): the dicts nv_quantize_layer_weights and
    nv_quantize_bwd_weights return."""
    fw = _nv_alloc(cfg, lib().moe_nv_layer_weight_bytes, MoeNvWeights._fields_, W1.device)
    bw = _nv_alloc(cfg, lib().moe_nv_bwd_weight_bytes, MoeNvBwdWeights._fields_, W1.device)
    bw["w2h"] = bw["w2h"].view(cfg.E, cfg.F, cfg.H // 2)
    bw["w13f"] = bw["w13f"].view(cfg.E, cfg.H, cfg.F)
    b = MoeNvBwdWeights(*[bw[n].data_ptr() for n, _ in MoeNvBwdWeights._fields_])
    _check(lib().moe_nv_quantize_train_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2),
                                               ctypes.byref(_nv_struct(fw)), ctypes.byref(b), _stream()),
           "moe_nv_quantize_train_weights")
    return fw, bw


def nv_train_workspace(cfg, device="cuda"):
    n = int(lib().moe_nv_train_workspace_bytes(ctypes.byref(cfg)))
    if n == 0:
        raise MoeError(2, "moe_nv_train_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def layer_fwd_nvfp4_train(cfg, x, router_w, nvw, saved, expert_bias=None, logit_bias=None, ws=None, y=None):
    """Training forward of the NVFP4 layer (``nvw`` from
    nv_quantize_layer_weights, ``saved`` from alloc_saved)."""
    dev = x.device
    if y is None:
        y = torch.empty((cfg.T, cfg.H), dtype=_out_dtype(cfg), device=dev)
    ws = nv_train_workspace(cfg, dev) if ws is None else ws
    st = lib().moe_layer_fwd_nvfp4_train(ctypes.byref(cfg), _p(x), _p(router_w), _p(expert_bias), _p(logit_bias),
                                         ctypes.byref(_nv_struct(nvw)), _p(y), ctypes.byref(_saved_struct(saved)),
                                         _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_fwd_nvfp4_train")
    return y


def layer_bwd_nvfp4(cfg, dO, x, router_w, nvbw, saved, ws=None, grads=None):
    """Backward of the NVFP4 training step (``nvbw`` from
    nv_quantize_bwd_weights); gradients as layer_bwd."""
    dev = x.device
    g = alloc_grads(cfg, dev) if grads is None else grads
    ws = nv_train_workspace(cfg, dev) if ws is None else ws
    w = MoeNvBwdWeights(*[nvbw[n].data_ptr() for n, _ in MoeNvBwdWeights._fields_])
    st = lib().moe_layer_bwd_nvfp4(ctypes.byref(cfg), _p(dO), _p(x), _p(router_w), ctypes.byref(w),
                                   ctypes.byref(_saved_struct(saved)), _p(g["dx"]), _p(g["dW_r"]), _p(g["dW1"]),
                                   _p(g["dW3"]), _p(g["dW2"]), _p(g["aux_loss"]), _p(ws), ws.numel(), _stream())
    _check(st, "moe_layer_bwd_nvfp4")
    return g
