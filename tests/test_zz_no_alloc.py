"""moe_permute_noalloc: the permute for callers that cannot allocate device
memory (its scratch is a fixed array inside the library). It must give exactly
the results of moe_permute, which takes a caller-provided workspace, on two
calls in a row (the second call must not see the first call's leftovers).
Collected last so that a failure here never hides another test's result."""
import ctypes

import pytest
import torch

from route_permute_grouped_gb300 import build, ops, synth


def _noalloc(cfg, x, idx):
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    x_perm = torch.full((T * k, H), -1.0, dtype=torch.bfloat16, device=x.device)
    rows = torch.full((T, k), -7, dtype=torch.int32, device=x.device)
    counts = torch.full((E,), -7, dtype=torch.int32, device=x.device)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=x.device)
    L = ops.lib()
    fn = L.moe_permute_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ops.MoeConfig)] + [ctypes.c_void_p] * 7
    st = fn(ctypes.byref(cfg), x.data_ptr(), idx.data_ptr(), x_perm.data_ptr(), rows.data_ptr(),
            counts.data_ptr(), offsets.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"moe_permute_noalloc returned {st}"
    return x_perm, rows, counts, offsets


def test_noalloc_rejects_oversize_before_gpu_work():
    build.build()
    cfg = ops.make_config(65537, 64, 256, 8, 64)  # ceil(T/64)*E = 1025*256 > 262144
    L = ops.lib()
    fn = L.moe_permute_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ops.MoeConfig)] + [ctypes.c_void_p] * 7
    fake = 256
    assert fn(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, None) == 2


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute_twice():
    build.build()
    cases = [(4097, 256, 128, 8, 1.2), (1000, 192, 8, 2, 0.0)]  # larger first, then smaller
    for T, H, E, k, skew in cases:
        cfg = ops.make_config(T, H, E, k, 64)
        idx = synth.synthetic_topk(T, E, k, seed=T, skew=skew, device="cuda")
        x = synth.make_layer(synth.shape("tiny", T=T, H=H, E=E, k=k, F=64), seed=T, device="cuda")["x"]
        ws = ops.workspace(cfg)
        ref = ops.permute(cfg, x, idx, ws)
        got = _noalloc(cfg, x, idx)
        torch.cuda.synchronize()
        assert ops.device_status(ws) == 0
        for name, a, b in zip(("x_perm", "row_id_map", "counts", "offsets"), got, ref):
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"{name} differs (T={T}, E={E}, k={k})"
        assert int(got[2].sum()) == T * k
