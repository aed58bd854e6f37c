"""The benchmark's FLOP accounting (CPU): the layer metric counts active FLOPs
only (router 2THE, 6HF per routed (token, expert) pair, 6HFs per token for a
shared expert; the backward twice the forward), checked against the figures
worked out by hand for the named layer shapes (tiny 0.101 GFLOP forward and
0.304 forward + backward; Mixtral-shaped 11.546 TFLOP; Qwen3-shaped 4.965
TFLOP forward, 14.895 training; DeepSeek-V3-shaped 6.524 TFLOP with its
shared expert)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from route_permute_grouped_gb300 import synth  # noqa: E402


# (shape, training, figure, half a unit of its last printed digit)
@pytest.mark.parametrize("name,training,want,half_ulp", [
    ("tiny", False, 0.101e9, 0.0005e9),
    ("tiny", True, 0.304e9, 0.0005e9),
    ("mixtral", False, 11.546e12, 0.0005e12),
    ("qwen3", False, 4.965e12, 0.0005e12),
    ("qwen3_train", True, 14.895e12, 0.0005e12),
    ("dsv3", False, 6.524e12, 0.0005e12),
])
def test_active_flops_of_the_named_shapes(name, training, want, half_ulp):
    got = bench.layer_flops(synth.shape(name), training)
    assert abs(got - want) <= half_ulp, (got, want)


def test_job_throughput_is_the_whole_job():
    # value = FLOPs of all ranks' steps / the slowest rank's time
    assert bench.job_throughput(14.895e12, 10.0, 1) == pytest.approx(1489.5, rel=1e-9)
    assert bench.job_throughput(14.895e12, 10.0, 4) == pytest.approx(4 * 1489.5, rel=1e-9)
