"""MXFP8 forward and NVFP4 grouped GEMM at full sizes (GPU), in the kernel
configuration the benchmark times, checked on sampled outputs the oracle
computes one by one: the MXFP8 layer on the Qwen3 expert shape (H=4096,
F=1536, top-8; 32 experts, T=4096) for 48 sampled tokens, and the NVFP4
grouped GEMM on the down projection's full shape (131072 x 1536 x 4096, 128
experts) for the rows of three experts."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def test_mxfp8_layer_qwen3_expert_shape_sampled():
    ls = synth.shape("qwen3_e32")
    d = synth.make_layer(ls, seed=1234, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.mx_workspace(cfg)
    y = ops.layer_fwd_mxfp8(cfg, d["x"], d["router_w"], w, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    tok = np.random.default_rng(3).choice(ls.T, 48, replace=False)
    n = {k: (None if v is None else f64(v)) for k, v in d.items() if k in ("x", "router_w", "W1", "W3", "W2")}
    ref = O.mx_layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, tokens=tok)
    assert_close("y (sampled tokens)", f64(y)[tok], ref["y"][tok])


def test_nvfp4_grouped_gemm_full_shape_sampled():
    E, R, K, N = 128, 131072, 1536, 4096
    offsets = np.arange(0, R + 1, R // E, dtype=np.int32)
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((R, K), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((E, K, N), generator=g, device="cuda") * K ** -0.5).to(torch.bfloat16)
    w = ops.nv_quantize_weights(W)
    ws = ops.nv_workspace(E, R, K)
    y = ops.nv_grouped_gemm(x, torch.from_numpy(offsets).cuda(), w, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    # the tensor maximum from a host copy of the input (exact on bf16 values)
    gx = O.nv_tensor_scale(float(x.cpu().abs().max().float().item()))
    for e in (0, 63, 127):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        xe = f64(x[lo:hi]).astype(np.float32)
        xq = O.nv_roundtrip(xe, axis=1, g=gx)
        We = O.nv_roundtrip(f64(W[e]).astype(np.float32), axis=0)
        ref = O.bf16_rne(xq @ We)
        assert_close(f"y rows of expert {e}", f64(y[lo:hi]), ref, atol=max(2e-2, 2.0 ** -7 * float(np.abs(ref).max())))
