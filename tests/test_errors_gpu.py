"""Device-side error reporting without a GPU fault (GPU): an expert index out
of range is skipped and recorded; a bounded wait that nothing satisfies (a
test hook makes the first scan chunk skip publishing) runs out, records a
timeout and returns, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import oracle as O
from route_permute_grouped_gb300 import ops, synth

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 5
DEVICE_INDEX = 6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


def _inputs(T=512, H=128, E=16, k=2):
    cfg = ops.make_config(T, H, E, k, 64)
    idx = synth.synthetic_topk(T, E, k, seed=9, device="cuda")
    x = synth.make_layer(synth.shape("tiny", T=T, H=H, E=E, k=k, F=64), device="cuda")["x"]
    return cfg, idx, x


def test_out_of_range_expert_index_is_reported():
    cfg, idx, x = _inputs()
    bad = idx.clone()
    bad[5, 1] = cfg.E        # out of range
    bad[300, 0] = -3
    ws = ops.workspace(cfg)
    _, rows, counts, _ = ops.permute(cfg, x, bad, ws)
    assert ops.device_status(ws) == DEVICE_INDEX
    r = rows.cpu().numpy()
    assert r[5, 1] == -1 and r[300, 0] == -1
    assert int(counts.sum()) == cfg.T * cfg.k - 2
    # the status was read and cleared; a clean call reports nothing
    xp, rows, counts, offs = ops.permute(cfg, x, idx, ws)
    assert ops.device_status(ws) == 0
    c_ref, o_ref, r_ref = O.permute_plan(idx.cpu().numpy(), cfg.E)
    assert np.array_equal(rows.cpu().numpy(), r_ref)


def test_bounded_wait_runs_out_and_context_survives():
    cfg, idx, x = _inputs(T=4096)
    ws = ops.workspace(cfg)
    try:
        ops.set_wait_limit_ns(2_000_000)  # 2 ms
        ops.set_fault(1)                  # first chunk never publishes
        ops.permute(cfg, x, idx, ws)
        assert ops.device_status(ws) == DEVICE_TIMEOUT
    finally:
        ops.set_fault(0)
        ops.set_wait_limit_ns(0)
    xp, rows, counts, offs = ops.permute(cfg, x, idx, ws)
    assert ops.device_status(ws) == 0
    _, _, r_ref = O.permute_plan(idx.cpu().numpy(), cfg.E)
    assert np.array_equal(rows.cpu().numpy(), r_ref)
    torch.cuda.synchronize()


def test_combine_skips_slots_the_permute_dropped():
    # moe_permute marks a slot whose expert index is out of range with row -1;
    # the combine then adds only the token's other slots (no read at row -1)
    cfg, idx, x = _inputs()
    bad = idx.clone()
    bad[5, 1] = cfg.E
    ws = ops.workspace(cfg)
    _, rows, _, _ = ops.permute(cfg, x, bad, ws)
    assert ops.device_status(ws) == DEVICE_INDEX
    R = cfg.T * cfg.k
    g = torch.Generator(device="cuda").manual_seed(3)
    y_perm = torch.randn((R, cfg.H), generator=g, device="cuda").to(torch.bfloat16)
    gate = torch.rand((cfg.T, cfg.k), generator=g, device="cuda")
    y = ops.unpermute_combine(cfg, y_perm, rows, gate)
    torch.cuda.synchronize()
    r = rows.cpu().numpy()
    yp = y_perm.float().cpu().numpy().astype(np.float64)
    gt = gate.cpu().numpy().astype(np.float64)
    ref = np.zeros((cfg.T, cfg.H))
    for t in range(cfg.T):
        for i in range(cfg.k):
            if r[t, i] >= 0:
                ref[t] += gt[t, i] * yp[r[t, i]]
    got = y.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= 2e-2 * max(1.0, float(np.abs(ref).max()))
    assert np.allclose(got[5], (gt[5, 0] * yp[r[5, 0]]), rtol=1e-2, atol=1e-2)
