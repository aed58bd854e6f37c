"""The weight-gradient GEMMs of the training step at the layer's literal bar
(GPU).

The backward's weight gradients are GEMMs over each expert's rows (steps b3
and b5 of the path): dW1_e = x_perm_e^T dh1_e, dW3_e = x_perm_e^T dh3_e,
dW2_e = a_e^T dy_perm_e, fp32 out. Evaluated here in fp64 on the very bf16
operands the kernels consumed (x_perm and a from the saved tensors, dh13 and
dy_perm from the workspace), the kernels' outputs must match at max-abs <= 2e-2
and rel-L2 <= 5e-3 with no allowance. The end-to-end comparison with the
oracle (tests/test_parity_*.py) admits one bf16 ulp of the gradient's largest
magnitude on top of 2e-2, for the bf16 rounding flips of the stored
activations; this test shows that allowance covers no GEMM error.
"""
import numpy as np
import pytest
import torch

from route_permute_grouped_gb300 import ops, synth
from tests._util import MAX_ABS, REL_L2, assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def _train(ls, recompute=False):
    d = synth.make_layer(ls, seed=1234, device="cuda", training=True)
    cfg = ops.config_from_shape(ls, aux_coeff=1e-2)
    ws = ops.workspace(cfg, True)
    saved = ops.alloc_saved(cfg, recompute=recompute)
    ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], d["expert_bias"], d["logit_bias"],
                  saved=saved, ws=ws)
    g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    a = saved["a"] if saved["a"] is not None else ops.workspace_tensor(ws, cfg, True, "a")
    ops_in = {"x_perm": saved["x_perm"], "a": a, "dh13": ops.workspace_tensor(ws, cfg, True, "dh13"),
              "dy_perm": ops.workspace_tensor(ws, cfg, True, "dy_perm")}
    return cfg, saved, g, ops_in


def _check_expert(cfg, e, lo, hi, g, t):
    F = cfg.F
    if hi == lo:  # no rows: the gradients are written as zero
        for key in ("dW1", "dW3", "dW2"):
            assert not torch.any(g[key][e]).item(), f"{key}[{e}] of an empty expert is not zero"
        return
    xp = f64(t["x_perm"][lo:hi])
    dh = f64(t["dh13"][lo:hi])
    a = f64(t["a"][lo:hi])
    dy = f64(t["dy_perm"][lo:hi])
    for key, want in (("dW1", xp.T @ dh[:, :F]), ("dW3", xp.T @ dh[:, F:]), ("dW2", a.T @ dy)):
        assert_close(f"{key}[{e}] ({hi - lo} rows)", f64(g[key][e]), want, rel=REL_L2, atol=MAX_ABS)


SMALL = {
    "tiny": synth.shape("tiny"),
    "ragged": synth.shape("tiny", T=1000, H=320, E=8, k=2, F=192),
    "e128_k8": synth.shape("tiny", T=777, H=256, E=128, k=8, F=256, w_std=0.05),
    "skew": synth.shape("tiny", T=900, H=256, E=32, k=4, F=128, skew=1.2),
    "k1": synth.shape("tiny", T=300, H=192, E=3, k=1, F=64),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("recompute", [False, True], ids=["standard", "memory_saving"])
def test_weight_gradient_gemms_on_stored_operands(name, recompute):
    ls = SMALL[name]
    cfg, saved, g, t = _train(ls, recompute)
    offs = saved["offsets"].cpu().numpy()
    for e in range(ls.E):
        _check_expert(cfg, e, int(offs[e]), int(offs[e + 1]), g, t)


@pytest.mark.slow
def test_weight_gradient_gemms_full_skewed_layer():
    """The full Qwen3-shaped training step with Zipf-skewed routing: the hot
    expert (~16K rows), a median expert, the smallest non-empty expert and
    every empty one."""
    ls = synth.shape("qwen3_skew_train")
    cfg, saved, g, t = _train(ls)
    counts = saved["counts"].cpu().numpy()
    offs = saved["offsets"].cpu().numpy()
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    assert counts.max() > 8 * counts.mean() and (counts == 0).sum() >= 1
    for e in sorted({int(order[-1]), int(order[len(order) // 2]), int(order[0])}):
        _check_expert(cfg, e, int(offs[e]), int(offs[e + 1]), g, t)
    for e in np.nonzero(counts == 0)[0]:
        _check_expert(cfg, int(e), int(offs[e]), int(offs[e]), g, t)
