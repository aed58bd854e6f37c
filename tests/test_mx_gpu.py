"""MXFP8 expert GEMMs (GPU) against the MXFP8 oracle: the quantisers bit for
bit (codes and scales, including the tile-ready scale layout of the expert
weights), and the layer forward within the layer's tolerance on shapes that
span several tiles, ragged tiles, zero-token experts and the group-limited
sigmoid router with a shared expert."""
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


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_mx_quantize_rows_bit_exact():
    g = torch.Generator().manual_seed(21)
    M, K = 333, 256
    x = torch.randn((M, K), generator=g) * torch.exp(2 * torch.randn((M, 1), generator=g))
    x[5, 32:64] = 0.0                        # an all-zero block
    x[6, :32] = 448.0 * 2.0 ** 3             # saturation-free power-of-two block
    x[7, 40] = 1e-30                         # tiny values
    x[8, 64:96] = torch.linspace(-3, 3, 32)  # ties of the E4M3 grid after scaling
    xb = x.to(torch.bfloat16)
    q, s = ops.mx_quantize(xb.cuda())
    torch.cuda.synchronize()
    rq, rs = O.mx_quantize(f64(xb), axis=1)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def _decode_tile_scales(sf, E, ntiles, nkb, rows_of_tile):
    """Scales [E][rows][K/32] from tile-ready blocks; rows_of_tile(j, b) gives
    the matrix row of B row b of tile j (None for unused rows, whose bytes must
    be zero)."""
    sf = sf.reshape(E, ntiles, nkb, 2, 32, 4, 4)  # [e][tile][kb][blk][r][c][s]
    out = {}
    bad = []
    for j in range(ntiles):
        for blk in range(2):
            for c in range(4):
                for r in range(32):
                    b = 128 * blk + 32 * c + r
                    row = rows_of_tile(j, b)
                    vals = sf[:, j, :, blk, r, c, :].reshape(E, nkb * 4)
                    if row is None:
                        if np.any(vals != 0):
                            bad.append((j, b))
                    else:
                        out[row] = vals
    assert not bad, f"unused scale bytes not zero at {bad[:4]}"
    return out


@pytest.mark.parametrize("E,H,F", [(3, 256, 384), (2, 384, 640)])
def test_mx_weight_quantization_bit_exact(E, H, F):
    ls = synth.shape("tiny", T=64, H=H, E=E, k=2, F=F)
    d = synth.make_layer(ls, seed=5, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    torch.cuda.synchronize()
    W1, W3, W2 = f64(d["W1"]), f64(d["W3"]), f64(d["W2"])
    w13 = w["w13"].cpu().numpy()
    w2 = w["w2"].cpu().numpy()
    nt1, nt2 = -(-F // 96), -(-H // 192)
    def rows13(j, b):  # gate/up tile: 96 W1 rows, then 96 W3 rows
        part, f = ("W1", 96 * j + b) if b < 96 else ("W3", 96 * j + b - 96)
        return (part, f) if b < 192 and f < F else None

    s13 = _decode_tile_scales(w["sf13"].cpu().numpy(), E, nt1, H // 128, rows13)
    s2 = _decode_tile_scales(w["sf2"].cpu().numpy(), E, nt2, F // 128,
                             lambda j, b: 192 * j + b if b < 192 and 192 * j + b < H else None)
    for e in range(E):
        for name, W, part in (("W1", W1, 0), ("W3", W3, 1)):
            rq, rs = O.mx_quantize(W[e].T, axis=1)  # [F, H] blocks along H
            assert np.array_equal(w13[e, part], rq), (name, e)
            got = np.stack([s13[(name, f)][e] for f in range(F)])
            assert np.array_equal(got, rs), (name, e)
        rq, rs = O.mx_quantize(W2[e].T, axis=1)  # [H, F] blocks along F
        assert np.array_equal(w2[e], rq), ("W2", e)
        got = np.stack([s2[h][e] for h in range(H)])
        assert np.array_equal(got, rs), ("W2", e)


MX_SHAPES = {
    "tiny": synth.shape("tiny", T=300, H=256, E=8, k=2, F=384),
    # several m tiles per expert, ragged last gate/up tile (F = 640 = 6 x 96 + 64)
    "ragged": synth.shape("tiny", T=1000, H=384, E=8, k=4, F=640),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    # zero-token experts
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=128, skew=1.2),
    # sigmoid + bias + group limit + shared expert (bf16)
    "dsv3_small": synth.shape("dsv3", T=333, H=256, E=64, k=8, F=128, F_shared=192),
}


@pytest.mark.parametrize("name", list(MX_SHAPES))
def test_layer_fwd_mxfp8(name):
    ls = MX_SHAPES[name]
    d = synth.make_layer(ls, seed=1234, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.mx_quantize_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.mx_workspace(cfg)
    Ws = (d["Ws1"], d["Ws3"], d["Ws2"]) if ls.F_shared else None
    y = ops.layer_fwd_mxfp8(cfg, d["x"], d["router_w"], w, d["expert_bias"], d["logit_bias"], Ws=Ws, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = {k_: (None if v is None else f64(v)) for k_, v in d.items()}
    Wsn = (n["Ws1"], n["Ws3"], n["Ws2"]) if ls.F_shared else None
    ref = O.mx_layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, ls.score, n["expert_bias"],
                         n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale, Ws=Wsn)
    assert_close("y", f64(y), ref["y"])
    # the MXFP8 layer differs from the bf16 layer by FP8 rounding, not more
    y16 = ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                        Ws=Ws)
    rel = np.linalg.norm(f64(y) - f64(y16)) / np.linalg.norm(f64(y16))
    assert 1e-3 < rel < 0.1, rel


def test_mxfp8_rejects_unaligned_shapes():
    cfg = ops.make_config(64, 192, 4, 2, 128)  # H not a multiple of 128
    assert ops.lib().moe_mx_workspace_bytes(ctypes_ref(cfg)) == 0
    with pytest.raises(ops.MoeError):
        ops.mx_workspace(cfg)


def ctypes_ref(cfg):
    import ctypes
    return ctypes.byref(cfg)
