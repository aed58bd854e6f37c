"""The bench's measurement helpers on the GPU: moe_read_ceiling (behind the
router's read ceiling) is a read-only pass that returns MOE_OK, leaves the
buffer unchanged and writes nothing to the sink for data that does not hash
to its marker word; moe_write_ceiling (behind the weight gradients' write
ceiling) fills exactly its bytes with the given word (GPU)."""
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


@pytest.mark.parametrize("nbytes", [16, (1 << 20) + 48, 64 << 20])
def test_write_ceiling_fills(nbytes):
    buf = torch.zeros(nbytes + 32, dtype=torch.uint8, device="cuda")
    n0 = ops.launch_count()
    ops.write_ceiling(buf[:nbytes], 0x01020304)
    torch.cuda.synchronize()
    assert ops.launch_count() == n0 + 1
    want = torch.tensor([4, 3, 2, 1], dtype=torch.uint8, device="cuda").repeat(nbytes // 4)
    assert torch.equal(buf[:nbytes], want)
    assert not torch.any(buf[nbytes:]).item()  # nothing past the end
