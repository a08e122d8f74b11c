"""The layer step (schedule, forward, backward: every launch through the C ABI) captured as one CUDA
graph and replayed on new inputs copied into the captured buffers.  The schedule is rebuilt on the
device from the new routing inside the replay, so every output must equal, bit for bit, an eager
step on the same inputs (BF16 and MXFP8), with a clean device status."""
import pytest
import torch

from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu

KEYS = ("x", "topk_ids", "topk_weights", "dY")


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _outputs(layer):
    g = layer.grads
    return [layer.out, g.dx, g.dw_gate, g.dw_up, g.dw_down, g.d_topk_weights]


CASES = [
    ("bf16", inputs.custom(T=700, H=512, I=384, E=3, K=2), False),
    ("mxfp8", inputs.custom(T=300, H=384, I=256, E=3, K=2), True),
]


@pytest.mark.parametrize("name,w,mx", CASES, ids=[c[0] for c in CASES])
def test_graph_replay_matches_eager(mok, name, w, mx):
    dev = "cuda"
    d0, d1 = inputs.make(w, seed=3), inputs.make(w, seed=4)
    Wg, Wu, Wd = (d0[k].to(dev) for k in ("Wg", "Wu", "Wd"))
    mx_w = mok.quantize_weights(Wg, Wu, Wd) if mx else None  # kept alive: the struct holds raw pointers
    weights = mok.weights_struct(mx=mx_w) if mx else mok.weights_struct(Wg, Wu, Wd)
    cfg = mok.make_config(128, 256, precision=mok.MOK_MXFP8 if mx else mok.MOK_BF16)
    buf = [d0[k].to(dev) for k in KEYS]  # the buffers the graph reads
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    stream = torch.cuda.Stream()

    def step():
        layer.schedule(buf[1], buf[2], stream)
        layer.forward(buf[0], weights, stream)
        layer.backward(buf[3], weights, stream)

    with torch.cuda.stream(stream):
        step()  # eager warm-up on the first inputs
    torch.cuda.synchronize()
    first = [t.clone() for t in _outputs(layer)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for b, k in zip(buf, KEYS):
        b.copy_(d1[k].to(dev))
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(layer.sched) == 0
    got = [t.clone() for t in _outputs(layer)]

    ref = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    ref.schedule(*(d1[k].to(dev) for k in ("topk_ids", "topk_weights")))
    ref.forward(d1["x"].to(dev), weights)
    ref.backward(d1["dY"].to(dev), weights)
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(ref.sched) == 0
    names = ("out", "dx", "dw_gate", "dw_up", "dw_down", "d_topk_weights")
    for n, a, b in zip(names, got, _outputs(ref)):
        assert torch.isfinite(a).all(), n
        assert torch.equal(a, b), n
    assert not torch.equal(got[0], first[0]), "the replay did not recompute the output"

    # a second replay with the first inputs again reproduces the eager warm-up
    for b, k in zip(buf, KEYS):
        b.copy_(d0[k].to(dev))
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    for n, a, b in zip(names, _outputs(layer), first):
        assert torch.equal(a, b), n
