"""Failure detection on the GPU without a fault: a bounded device wait that
nothing completes expires, the kernel records it in the workspace's status
flags, the host reads them, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


def test_bounded_wait_expiry_sets_timeout_flag(csa):
    dev = torch.device("cuda", 0)
    ws = csa.Workspace(dev)
    assert ws.flags() == 0
    csa.selftest_wait_timeout(ws, 1000)
    assert ws.flags() & 2            # CSA_FLAG_TIMEOUT
    ws.reset()
    assert ws.flags() == 0
    # the context is still usable: a library call after the expiry runs and is exact
    x = torch.ones((1, 8, 512), dtype=torch.bfloat16, device=dev)
    z = torch.zeros((1, 8), dtype=torch.float32, device=dev)
    out = csa.compress_kv(x, z, None, 4, csa.FMT_F32, 0)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.ones((1, 2, 512), dtype=torch.float32, device=dev))
