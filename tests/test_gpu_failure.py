"""Failure detection without a GPU fault: a bounded in-kernel wait on an mbarrier that nothing
completes (the wait every GEMM role uses) gives up at the library's deadline, records
MOK_ERR_TIMEOUT in the caller's status word and returns; the context stays usable, so a layer step
right after it runs clean."""
import time

import pytest
import torch

from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def test_bounded_wait_times_out_and_the_context_survives(mok):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    mok.mok_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert int(status.item()) & 0xFFFFFFFF == 1 << mok.MOK_ERR_TIMEOUT
    assert 1.5 < waited < 60, waited  # the deadline is 2 s

    w = inputs.WORKLOADS["tiny"]
    d = inputs.make(w, seed=0)
    x, ids, s, dY = (d[k].cuda() for k in ("x", "topk_ids", "topk_weights", "dY"))
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, mok.make_config(128, 256))
    weights = mok.weights_struct(*(d[k].cuda() for k in ("Wg", "Wu", "Wd")))
    layer.schedule(ids, s)
    out = layer.forward(x, weights)
    g = layer.backward(dY, weights)
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(layer.sched) == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(g.dx.float()).all()
