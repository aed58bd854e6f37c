"""NVFP4 training step (GPU) against the NVFP4 oracle: the weights of the two
data-gradient GEMMs quantised bit for bit (codes, tile-ready scales, tensor
scales), and the forward output and every gradient (dx, dW_router, dW1, dW3,
dW2, aux loss) within the layer's tolerance, on shapes with several tiles,
ragged N tiles of the data-gradient GEMMs, experts whose row count is not a
multiple of 128 and zero-token experts."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth
from tests._util import MAX_ABS, assert_close, assert_close_but_flips, f64, report_exact, rel_l2, wgrad_atol

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


def _tile_scales(sf, E, N, K):
    """[E, N, K/16] block scales from the tile-ready layout (tile n / 192, B
    row b = n % 192: block b / 128, row b % 128)."""
    nt = -(-N // 192)
    sf = np.asarray(sf).reshape(E, nt, K // 256, 2, 4, 32, 4, 4)  # [e][tile][kb][blk][step][r][c][j]
    out = np.zeros((E, N, K // 16), np.uint8)
    for n in range(N):
        j, b = divmod(n, 192)
        blk, rr = divmod(b, 128)
        c, r = divmod(rr, 32)
        out[:, n] = sf[:, j, :, blk, :, r, c, :].reshape(E, -1)
    return out


@pytest.mark.parametrize("E,H,F", [(3, 256, 512), (2, 512, 256)])
def test_nv_bwd_weight_quantization_bit_exact(E, H, F):
    ls = synth.shape("tiny", T=64, H=H, E=E, k=2, F=F)
    d = synth.make_layer(ls, seed=6, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    w = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    torch.cuda.synchronize()
    W1, W3, W2 = (f64(d[n]).astype(np.float32) for n in ("W1", "W3", "W2"))
    w2h, w13f = _unpack(w["w2h"].cpu().numpy()), _unpack(w["w13f"].cpu().numpy())
    s2 = _tile_scales(w["sf2h"].cpu().numpy(), E, F, H)
    s13 = _tile_scales(w["sf13f"].cpu().numpy(), E, H, 2 * F)
    for e in range(E):
        q, s, g = O.nv_quantize(W2[e], axis=1)                    # [F, H], blocks along H
        assert np.array_equal(w2h[e], q) and np.array_equal(s2[e], s) and w["g2h"][e].item() == float(g), e
        q, s, g = O.nv_quantize(np.concatenate([W1[e], W3[e]], axis=1), axis=1)   # [H, 2F], blocks along 2F
        assert np.array_equal(w13f[e], q) and np.array_equal(s13[e], s) and w["g13f"][e].item() == float(g), e


@pytest.mark.parametrize("E,H,F", [(3, 256, 512), (130, 256, 256)])
def test_nv_train_weights_in_one_call_are_the_two_copies(E, H, F):
    """The combined refresh takes each per-expert maximum once; its codes,
    scales and tensor scales are those of the two separate calls, byte for
    byte (the separate calls being pinned to the oracle above and by the
    forward's weight test)."""
    ls = synth.shape("tiny", T=64, H=H, E=E, k=2, F=F)
    d = synth.make_layer(ls, seed=8, device="cuda", training=False)
    cfg = ops.config_from_shape(ls)
    fw_ref = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
    bw_ref = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    fw, bw = ops.nv_quantize_train_weights(cfg, d["W1"], d["W3"], d["W2"])
    torch.cuda.synchronize()
    for got, ref in ((fw, fw_ref), (bw, bw_ref)):
        assert set(got) == set(ref)
        for n in ref:
            assert torch.equal(got[n].view(torch.uint8).reshape(-1), ref[n].view(torch.uint8).reshape(-1)), n


TRAIN_SHAPES = {
    "tiny": synth.shape("tiny", T=300, H=256, E=8, k=2, F=256),
    # ragged N tiles in both data-gradient GEMMs (F = 512 = 2 x 192 + 128,
    # H = 512), several m tiles per expert
    "ragged": synth.shape("tiny", T=1000, H=512, E=8, k=4, F=512),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    # zero-token experts: their weight gradients are zero
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=256, skew=1.2),
    # the sigmoid router with an expert bias and a group limit (its backward
    # through the sigmoid scores), gates scaled
    "sigmoid_groups": synth.shape("tiny", T=333, H=256, E=64, k=8, F=256, score="sigmoid", n_groups=8, topk_groups=4,
                                  gate_scale=2.5, expert_bias_range=0.1),
}


def _code_flip_atol(want, amax_act, amax_w):
    """Max-abs bound where an NVFP4 code of a routed-row operand may differ:
    its code is decided from a bf16 value that fp32 and fp64 accumulation can
    put on either side of a bf16 rounding boundary, and E2M1 codes are coarse,
    so such a flip (rare) moves the element by one E2M1 step, at most a third
    of its block's largest magnitude (a step of 2 block scales at the top
    binade, the block scale being the block maximum / 6), and each output of
    its GEMM row by at most that step times the other operand's largest
    magnitude. Two flips on one output are admitted, and never less than the
    bf16 bound."""
    return max(wgrad_atol(want), 2.0 * float(amax_act) / 3.0 * float(amax_w))


@pytest.mark.parametrize("name", list(TRAIN_SHAPES))
def test_layer_train_nvfp4(name):
    ls = TRAIN_SHAPES[name]
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    aux = 1e-2 if ls.score == "softmax" else 0.0  # the aux loss applies to the softmax router
    cfg = ops.config_from_shape(ls, aux_coeff=aux, out_fp32=True)
    nvw = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
    nvbw = ops.nv_quantize_bwd_weights(cfg, d["W1"], d["W3"], d["W2"])
    ws = ops.nv_train_workspace(cfg)
    saved = ops.alloc_saved(cfg)
    y = ops.layer_fwd_nvfp4_train(cfg, d["x"], d["router_w"], nvw, saved, d["expert_bias"], d["logit_bias"], ws=ws)
    g = ops.layer_bwd_nvfp4(cfg, d["dO"], d["x"], d["router_w"], nvbw, saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    n = {k_: (None if v is None else f64(v)) for k_, v in d.items()}
    ref = O.nv_layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score,
                         n["expert_bias"], n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale,
                         aux_coeff=aux, prec=O.Precision(y=False, dx=False))
    assert np.array_equal(saved["topk_idx"].cpu().numpy(), ref["topk_idx"]), "routing differs (tie)"
    assert np.array_equal(saved["counts"].cpu().numpy(), ref["counts"])
    # the saved rows and pre-activations are the oracle's stored tensors
    xp = np.zeros((ls.T * ls.k, ls.H))
    xp[ref["row_id_map"].reshape(-1)] = np.repeat(n["x"], ls.k, axis=0)
    assert np.array_equal(f64(saved["x_perm"]), xp)
    E = ls.E
    W13 = np.concatenate([n["W1"], n["W3"]], axis=2)                 # [E, H, 2F]
    ymax = float(np.abs(ref["y"]).max())
    assert_close("y", f64(y), ref["y"], atol=max(MAX_ABS, 2.0 ** -7 * ymax))
    report_exact("nvfp4_train y", f64(y), O.layer_fwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], ls.k, ls.score,
                                                         n["expert_bias"], n["logit_bias"], ls.n_groups,
                                                         ls.topk_groups, ls.gate_scale, prec=O.EXACT)["y"])
    dx_atol = _code_flip_atol(ref["dx"], np.abs(ref["dh13"]).max(), np.abs(W13).max())
    assert_close("dx", f64(g["dx"]), ref["dx"], atol=dx_atol)
    assert_close("dW_r", f64(g["dW_r"]), ref["dW_r"], atol=wgrad_atol(ref["dW_r"]))
    # dy_perm = bf16(g dO) with a gate the router computes in fp32: in rare
    # elements the kernel and the oracle store neighbouring bf16 values, and
    # about one in fifty of those lands on the other side of an E2M1 decision,
    # moving that element's code by a whole step; da, dh13 and the expert's
    # dW1 / dW3 then move by one outer product (see assert_close_but_flips)
    for key in ("dW1", "dW3", "dW2"):
        want = np.stack([ref[key][e] for e in range(E)])
        assert_close_but_flips(key, f64(g[key]), want, atol=wgrad_atol(want))
    if ls.skew:
        empty = np.nonzero(ref["counts"] == 0)[0]
        assert len(empty) > 0
        assert not np.any(f64(g["dW1"])[empty]) and not np.any(f64(g["dW2"])[empty])
    if aux:
        assert abs(float(g["aux_loss"].item()) - ref["aux_loss"]) <= 1e-5 * max(1.0, abs(ref["aux_loss"]))
    # the NVFP4 step differs from the bf16 step by FP4 rounding, not more
    ref16 = O.layer_bwd(n["x"], n["router_w"], n["W1"], n["W3"], n["W2"], n["dO"], ls.k, ls.score,
                        n["expert_bias"], n["logit_bias"], ls.n_groups, ls.topk_groups, ls.gate_scale,
                        aux_coeff=aux, prec=O.Precision(y=False, dx=False))
    r16 = rel_l2(f64(g["dx"]), ref16["dx"])
    assert 1e-2 < r16 < 0.5, r16  # two chained FP4 GEMMs


def test_nv_train_saved_buffers_required():
    ls = TRAIN_SHAPES["tiny"]
    d = synth.make_layer(ls, seed=2, device="cuda", training=True)
    cfg = ops.config_from_shape(ls)
    nvw = ops.nv_quantize_layer_weights(cfg, d["W1"], d["W3"], d["W2"])
    saved = ops.alloc_saved(cfg)
    saved["a"] = None
    with pytest.raises(ops.MoeError):
        ops.layer_fwd_nvfp4_train(cfg, d["x"], d["router_w"], nvw, saved)
