"""The bounds-check build (GPU): compiled with -DMOE_BOUNDS_CHECK, the
element-wise kernels range-check the row indices they read from row_id_map
and record MOE_ERR_DEVICE_INDEX instead of reading or writing out of range.
The scenario runs in a child process that loads that build (MOE_BOUNDS_CHECK=1
selects it in the binding): a training step whose saved row_id_map holds one
index past the routed rows. The tensors that index would reach are padded, so
even an unchecked read or write of it would stay inside their allocations."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch
from route_permute_grouped_gb300 import build, ops, synth
build.build(checked=True)
out = {"checked": int(ops.lib().moe_bounds_checked())}
ls = synth.shape("tiny", T=256, H=128, E=8, k=2, F=64, aux_coeff=1e-2)
d = synth.make_layer(ls, seed=5, device="cuda", training=True)
cfg = ops.config_from_shape(ls)
R = cfg.T * cfg.k
ws = ops.workspace(cfg, True)
saved = ops.alloc_saved(cfg)
pad = torch.zeros((R + 16, cfg.H), dtype=saved["y_perm"].dtype, device="cuda")
saved["y_perm"] = pad[:R]
ops.layer_fwd(cfg, d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved=saved, ws=ws)
torch.cuda.synchronize()
out["fwd_status"] = ops.device_status(ws)
saved["row_id_map"][3, 0] = R + 1
g = ops.layer_bwd(cfg, d["dO"], d["x"], d["router_w"], d["W1"], d["W3"], d["W2"], saved, ws=ws)
torch.cuda.synchronize()
out["bwd_status"] = ops.device_status(ws)
out["pad_untouched"] = bool(torch.count_nonzero(pad[R:]).item() == 0)
print(json.dumps(out))
"""


def test_bounds_check_build_reports_a_row_index_past_the_routed_rows():
    env = dict(os.environ, MOE_BOUNDS_CHECK="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["checked"] == 1
    assert out["fwd_status"] == 0
    assert out["bwd_status"] == 6  # MOE_ERR_DEVICE_INDEX
    assert out["pad_untouched"]
