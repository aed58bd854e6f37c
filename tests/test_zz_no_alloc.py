"""moe_permute_noalloc: the permute for callers that cannot allocate device
memory (its scratch is a fixed array inside the library). It must give exactly
the results of moe_permute, which takes a caller-provided workspace, on two
calls in a row (the second call must not see the first call's leftovers),
leave the device's free memory unchanged over repeated calls, and report its
device-side errors through moe_noalloc_get_device_status. Collected last so
that a failure here never hides another test's result."""
import ctypes

import pytest
import torch

from route_permute_grouped_gb300 import build, ops, synth


def _outputs(cfg, device):
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    return (torch.full((T * k, H), -1.0, dtype=torch.bfloat16, device=device),
            torch.full((T, k), -7, dtype=torch.int32, device=device),
            torch.full((E,), -7, dtype=torch.int32, device=device),
            torch.full((E + 1,), -7, dtype=torch.int32, device=device))


def _call(cfg, x, idx, out):
    x_perm, rows, counts, offsets = out
    fn = ops.lib().moe_permute_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ops.MoeConfig)] + [ctypes.c_void_p] * 7
    st = fn(ctypes.byref(cfg), x.data_ptr(), idx.data_ptr(), x_perm.data_ptr(), rows.data_ptr(),
            counts.data_ptr(), offsets.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, f"moe_permute_noalloc returned {st}"
    return out


def _noalloc(cfg, x, idx):
    return _call(cfg, x, idx, _outputs(cfg, x.device))


def _status():
    fn = ops.lib().moe_noalloc_get_device_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    out = ctypes.c_int(-1)
    assert fn(torch.cuda.current_stream().cuda_stream, ctypes.byref(out)) == 0
    return out.value


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


@pytest.mark.gpu
def test_noalloc_permute_allocates_nothing_and_reports_device_errors():
    build.build()
    T, H, E, k = 2048, 256, 64, 4
    cfg = ops.make_config(T, H, E, k, 64)
    idx = synth.synthetic_topk(T, E, k, seed=5, device="cuda")
    x = synth.make_layer(synth.shape("tiny", T=T, H=H, E=E, k=k, F=64), seed=5, device="cuda")["x"]
    out = _outputs(cfg, x.device)
    _call(cfg, x, idx, out)  # the first call on the device looks up the array's address
    assert _status() == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        _call(cfg, x, idx, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "moe_permute_noalloc changed the device's free memory"
    # an expert index out of range is skipped and reported; the next clean
    # call reports nothing and gives the workspace permute's results again
    bad = idx.clone()
    bad[7, 2] = E
    _call(cfg, x, bad, out)
    assert _status() == 6  # MOE_ERR_DEVICE_INDEX
    assert int(out[1][7, 2].item()) == -1 and int(out[2].sum().item()) == T * k - 1
    _call(cfg, x, idx, out)
    assert _status() == 0
    ws = ops.workspace(cfg)
    ref = ops.permute(cfg, x, idx, ws)
    torch.cuda.synchronize()
    for name, a, b in zip(("x_perm", "row_id_map", "counts", "offsets"), out, ref):
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{name} differs after an error call"
