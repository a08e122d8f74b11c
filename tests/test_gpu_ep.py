"""Expert parallelism on one GPU: the group's ranks run one after another on one stream, each with
buffers of its own (its tokens, routing, upstream gradient, workspace, forward context, receive
buffers and its experts' weights and weight gradients), reached by the others only through the
per-rank pointer tables the calls take.  The token rows are pulled by the rank owning the experts;
expert outputs, dX rows and router-weight gradients are pushed back to the rank holding the tokens,
which reduces them in fixed k order.

The group's result must be bitwise the single-rank layer's on the concatenated tokens and experts:
out, dX, d_topk_weights and every expert's weight gradients, for G = 2 and 4 ranks, BF16 and
MXFP8, including a slot with an invalid expert id."""
import pytest
import torch

from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _single(mok, w, d, cfg, mx):
    x, ids, s, dY = (d[k].cuda() for k in ("x", "topk_ids", "topk_weights", "dY"))
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    Wg, Wu, Wd = (d[k].cuda() for k in ("Wg", "Wu", "Wd"))
    mxw = mok.quantize_weights(Wg, Wu, Wd) if mx else None
    weights = mok.weights_struct(mx=mxw) if mx else mok.weights_struct(Wg, Wu, Wd)
    layer.schedule(ids, s)
    out = layer.forward(x, weights).clone()
    g = layer.backward(dY, weights)
    torch.cuda.synchronize()
    status = mok.mok_read_device_status(layer.sched)
    return dict(out=out, dx=g.dx.clone(), ds=g.d_topk_weights.clone(), dwg=g.dw_gate.clone(),
                dwu=g.dw_up.clone(), dwd=g.dw_down.clone()), status


def _group(mok, w, d, cfg, G, mx):
    T, H, I, E, K = w.T, w.H, w.I, w.E, w.K
    Tl, El = T // G, E // G
    bf, f32 = torch.bfloat16, torch.float32
    # every rank's own buffers (separate allocations: each reaches the others only by pointer)
    tok = lambda t, r: t[r * Tl:(r + 1) * Tl].cuda().clone()  # noqa: E731
    x = [tok(d["x"], r) for r in range(G)]
    ids = [tok(d["topk_ids"], r) for r in range(G)]
    wts = [tok(d["topk_weights"], r) for r in range(G)]
    dy = [tok(d["dY"], r) for r in range(G)]
    expw = lambda t, r: t[r * El:(r + 1) * El].cuda().contiguous().clone()  # noqa: E731
    weights, keep = [], []  # the structs hold raw pointers: keep their tensors alive
    for r in range(G):
        Wg, Wu, Wd = expw(d["Wg"], r), expw(d["Wu"], r), expw(d["Wd"], r)
        mxw = mok.quantize_weights(Wg, Wu, Wd) if mx else None
        keep.append((Wg, Wu, Wd, mxw))
        weights.append(mok.weights_struct(mx=mxw) if mx else mok.weights_struct(Wg, Wu, Wd))
    shape = mok.make_shape(T, H, I, El, K)  # the group's tokens, this rank's experts
    ep = [mok.make_ep_group(G, r, Tl) for r in range(G)]
    ws = [mok.alloc_workspace(cfg, shape) for _ in range(G)]
    ctx = [mok.alloc_fwd_ctx(cfg, shape) for _ in range(G)]
    y_recv = [torch.empty((Tl * K, H), dtype=bf, device="cuda") for _ in range(G)]
    dx_recv = [torch.empty((Tl * K, H), dtype=bf, device="cuda") for _ in range(G)]
    ds = [torch.full((Tl, K), float("nan"), dtype=f32, device="cuda") for _ in range(G)]
    out = [torch.empty((Tl, H), dtype=bf, device="cuda") for _ in range(G)]
    dx = [torch.empty((Tl, H), dtype=bf, device="cuda") for _ in range(G)]
    dwg = [torch.empty((El, I, H), dtype=f32, device="cuda") for _ in range(G)]
    dwu = [torch.empty((El, I, H), dtype=f32, device="cuda") for _ in range(G)]
    dwd = [torch.empty((El, H, I), dtype=f32, device="cuda") for _ in range(G)]
    sched = [mok.mok_ep_build_schedule(cfg, shape, ep[r], ids, wts, ws[r]) for r in range(G)]
    for r in range(G):  # every rank's forward (pull dispatch, its experts, push of y rows) ...
        mok.mok_ep_forward(sched[r], ep[r], x, weights[r], y_recv, ctx[r])
    for r in range(G):  # ... then every token owner's fixed-order combine
        mok.mok_ep_combine(shape, ep[r], ids[r], wts[r], y_recv[r], out[r])
    for r in range(G):
        mok.mok_ep_backward(sched[r], ep[r], ctx[r], dy, weights[r], dwg[r], dwu[r], dwd[r], dx_recv, ds)
    for r in range(G):
        mok.mok_ep_combine(shape, ep[r], ids[r], None, dx_recv[r], dx[r])
    torch.cuda.synchronize()
    del keep
    status = [mok.mok_read_device_status(sched[r]) for r in range(G)]
    res = dict(out=torch.cat(out), dx=torch.cat(dx), ds=torch.cat(ds), dwg=torch.cat(dwg), dwu=torch.cat(dwu),
               dwd=torch.cat(dwd))
    return res, status


CASES = [
    ("tiny", 2, False), ("tiny", 4, False), ("bf16_e64", 2, False), ("bf16_e64", 4, False),
    ("sweep_zipf1", 4, False), ("tiny", 2, True), ("mxfp8_ep64_shard", 2, True), ("mxfp8_ep64_shard", 4, True),
]


@pytest.mark.parametrize("name,G,mx", CASES, ids=[f"{n}-G{g}{'-mx' if m else ''}" for n, g, m in CASES])
def test_expert_parallel_group_equals_single_rank_bitwise(mok, name, G, mx):
    w = inputs.WORKLOADS[name]
    d = inputs.make(w, seed=3, weight_device="cuda")
    cfg = mok.make_config(512, 2048, precision=mok.MOK_MXFP8 if mx else mok.MOK_BF16)
    ref, st1 = _single(mok, w, d, cfg, mx)
    got, stg = _group(mok, w, d, cfg, G, mx)
    assert st1 == 0 and stg == [0] * G
    for k in ref:
        assert torch.equal(got[k], ref[k]), k


def test_expert_parallel_invalid_id_matches_single_rank(mok):
    """A slot whose id lies outside the group's experts: skipped in the combine, dS = 0 written by
    its token's own rank, MOK_ERR_BAD_EXPERT_ID in every rank's status (each reads all slots)."""
    w = inputs.custom(T=256, H=256, I=128, E=8, K=2)
    d = inputs.make(w, seed=4)
    ids = d["topk_ids"].clone()
    ids[200, 1] = 8   # == E: invalid, held by rank 1 of 2
    ids[3, 0] = -1    # invalid, held by rank 0
    d["topk_ids"] = ids
    cfg = mok.make_config(128, 256)
    ref, st1 = _single(mok, w, d, cfg, False)
    got, stg = _group(mok, w, d, cfg, 2, False)
    bad = 1 << mok.MOK_ERR_BAD_EXPERT_ID
    assert st1 == bad and stg == [bad, bad]
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    assert float(got["ds"][200, 1]) == 0.0 and float(got["ds"][3, 0]) == 0.0
