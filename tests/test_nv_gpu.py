"""NVFP4 grouped expert GEMM (GPU) against the NVFP4 oracle: the quantisers
bit for bit (codes, block scales, tensor scales, the tile-ready weight-scale
layout), and the grouped GEMM within the layer's tolerance on expert segments
that span several tiles, end mid-tile, are empty, and a ragged last n tile."""
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


def _unpack(q):
    q = np.asarray(q, np.uint8)
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],), np.uint8)
    out[..., 0::2] = q & 15
    out[..., 1::2] = q >> 4
    return out


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def test_nv_quantize_rows_bit_exact():
    x = _bf16((300, 256), 1.0, 3) * torch.exp(_bf16((300, 1), 1.5, 4).float()).to(torch.bfloat16)
    x[4, 16:32] = 0.0
    x[5, :16] = torch.linspace(-7, 7, 16).to(torch.bfloat16)
    q, s, g = ops.nv_quantize(x.cuda())
    torch.cuda.synchronize()
    rq, rs, rg = O.nv_quantize(f64(x).astype(np.float32), axis=1)
    assert g.item() == float(rg)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(_unpack(q.cpu().numpy()), rq)


def test_nv_quantize_at_e2m1_boundaries():
    # (1) exact ties: with the tensor maximum 2688 * 2^-4 alone in its block,
    # g = 2^-4, and a block whose maximum is 6 * 2^(j-4) has the scale 2^j, so
    # its elements B * 2^(j-4) divide to the E2M1 decision boundaries B exactly
    # (ties to the even code); (2) 4M random elements under random block and
    # row scales, where a few quotients fall within a few fp32 ulps of a
    # boundary: every code and scale as the definition gives them
    bnd = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    base = np.concatenate([[6.0], bnd, -bnd, [0.0]])
    rows = [np.concatenate([[2688.0 * 2.0 ** -4], np.zeros(15)])]
    for j in range(-6, 6):
        rows.append(base * 2.0 ** (j - 4))
    x1 = torch.from_numpy(np.stack(rows).reshape(1, -1).repeat(16, axis=0)).to(torch.bfloat16)
    g = torch.Generator().manual_seed(31)
    x2 = (torch.randn((4096, 1024), generator=g) * torch.exp(torch.randn((4096, 64, 1), generator=g) * 2.0)
          .repeat(1, 1, 16).reshape(4096, 1024)).to(torch.bfloat16)
    for x in (x1, x2):
        q, sc, gg = ops.nv_quantize(x.cuda())
        torch.cuda.synchronize()
        rq, rs, rg = O.nv_quantize(f64(x).astype(np.float32), axis=1)
        assert gg.item() == float(rg)
        assert np.array_equal(sc.cpu().numpy(), rs)
        assert np.array_equal(_unpack(q.cpu().numpy()), rq)


@pytest.mark.parametrize("E,K,N", [(3, 512, 200), (2, 256, 384)])
def test_nv_weight_quantization_bit_exact(E, K, N):
    W = _bf16((E, K, N), K ** -0.5, 11)
    w = ops.nv_quantize_weights(W.cuda())
    torch.cuda.synchronize()
    Wn = f64(W).astype(np.float32)
    nt = -(-N // 192)
    sf = w["sf"].cpu().numpy().reshape(E, nt, K // 256, 2, 4, 32, 4, 4)  # [e][tile][kb][blk][step][r][c][j]
    wq = _unpack(w["wq"].cpu().numpy())
    for e in range(E):
        rq, rs, rg = O.nv_quantize(Wn[e].T, axis=1)  # [N, K] blocks along K
        assert w["g"][e].item() == float(rg)
        assert np.array_equal(wq[e], rq), e
        got = np.zeros((N, K // 16), np.uint8)
        for n in range(N):
            j, b = divmod(n, 192)
            blk, rr = divmod(b, 128)
            c, r = divmod(rr, 32)
            got[n] = sf[e, j, :, blk, :, r, c, :].reshape(-1)
        assert np.array_equal(got, rs), e
        # rows of the last tile past N keep zero scales
        for b in range(N - 192 * (nt - 1), 256):
            blk, rr = divmod(b, 128)
            c, r = divmod(rr, 32)
            assert not sf[e, nt - 1, :, blk, :, r, c, :].any()


@pytest.mark.parametrize("counts,K,N", [([300, 0, 41, 513, 256, 7], 512, 200), ([1000, 24], 256, 384)])
def test_nv_grouped_gemm(counts, K, N):
    E = len(counts)
    R = sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = _bf16((R, K), 1.0, 21)
    W = _bf16((E, K, N), K ** -0.5, 22)
    w = ops.nv_quantize_weights(W.cuda())
    ws = ops.nv_workspace(E, R, K)
    y = ops.nv_grouped_gemm(x.cuda(), torch.from_numpy(offsets).cuda(), w, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    ref = O.nv_grouped_gemm(f64(x).astype(np.float32), offsets, f64(W).astype(np.float32))
    # bf16 outputs: one bf16 ulp of the largest value where the fp32 sum sits
    # at a rounding boundary
    assert_close("y", f64(y), ref, atol=max(2e-2, 2.0 ** -7 * float(np.abs(ref).max())))
    # the NVFP4 GEMM differs from the exact product by FP4 rounding, not more
    exact = np.zeros((R, N))
    for e in range(E):
        exact[offsets[e]:offsets[e + 1]] = f64(x)[offsets[e]:offsets[e + 1]] @ f64(W)[e]
    rel = np.linalg.norm(f64(y) - exact) / np.linalg.norm(exact)
    assert 0.03 < rel < 0.3, rel


def test_nv_rejects_unaligned_shapes():
    assert ops.lib().moe_nv_workspace_bytes(4, 100, 128) == 0   # K not a multiple of 256
    assert ops.lib().moe_nv_weight_bytes(4, 256, 12, 0) == 0     # N not a multiple of 8


NV_LAYER_SHAPES = {
    "tiny": synth.shape("tiny", T=300, H=256, E=8, k=2, F=256),
    "ragged_skew": synth.shape("tiny", T=777, H=512, E=32, k=4, F=256, skew=1.2),
    "sigmoid_groups": synth.shape("tiny", T=333, H=256, E=64, k=8, F=256, score="sigmoid", n_groups=8, topk_groups=4,
                                  gate_scale=2.5, expert_bias_range=0.1),
}


@pytest.mark.parametrize("name", list(NV_LAYER_SHAPES))
def test_layer_fwd_nvfp4(name):
    ls = NV_LAYER_SHAPES[name]
    d = synth.make_layer(ls, seed=1234, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
    y = ops.layer_fwd_nvfp4(cfg, d["x"], d["router_w"], w, d["expert_bias"], d["logit_bias"])
    torch.cuda.synchronize()
    n = {k_: (None if v is None else f64(v)) for k_, v in d.items()}
    ref = O.nv_layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, ls.score, n["expert_bias"],
                         n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale)
    assert_close("y", f64(y), ref["y"], atol=max(2e-2, 2.0 ** -7 * float(np.abs(ref["y"]).max())))
