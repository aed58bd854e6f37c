"""moe_read_ceiling (the measurement helper behind the bench's router read
ceiling) on the GPU: a read-only pass that returns MOE_OK, leaves the buffer
unchanged and writes nothing to the sink for data that does not hash to its
marker word (GPU)."""
import pytest
import torch

from route_permute_grouped_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from route_permute_grouped_gb300 import build
    build.build()
    ops.lib()


@pytest.mark.parametrize("nbytes", [16, 4096, (1 << 20) + 48, 64 << 20])
def test_read_ceiling_reads_only(nbytes):
    buf = torch.full((nbytes,), 1, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(4096, dtype=torch.int32, device="cuda")
    before = buf.clone()
    n0 = ops.launch_count()
    ops.read_ceiling(buf, sink)
    torch.cuda.synchronize()
    assert ops.launch_count() == n0 + 1
    assert torch.equal(buf, before)
    assert not torch.any(sink).item()
