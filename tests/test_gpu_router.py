"""GPU router step vs its oracle (oracle/mok_oracle_router.c), through the C ABI.

Bit-exact: the fp32 logits (both sides accumulate over h in ascending order with one fused
multiply-add per step, then add the bias) and therefore the top-k ids.  Tolerances: the
renormalised weights 1e-5 relative (fp32 softmax over K logits); dW_r and d_bias 1e-4 of their
maximum (fp32 sums over at most T rows); dx 4e-3 of its maximum (fp32 sum over K, one bf16
rounding: 2^-8).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import rel_err, to_f64
from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_W, TOL_DW, TOL_DX = 1e-5, 1e-4, 4e-3


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _router_case(T, H, E, K, bias, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((T, H), generator=g) * 1.0).to(torch.bfloat16)
    w = (torch.randn((H, E), generator=g) * 0.05).to(torch.bfloat16)
    b = (torch.randn((E,), generator=g) * 0.5) if bias else None
    d = torch.randn((T, K), generator=g)
    return x, w, b, d


def _run(mok, x, w, b, K, d):
    T, H = x.shape
    E = w.shape[1]
    xc, wc = x.cuda(), w.cuda()
    bc = None if b is None else b.cuda()
    logits, ids, wts = mok.router_forward(xc, wc, bc, K)
    layer = mok.Layer(T, H, 128, E, K, mok.make_config(128, 256))
    layer.schedule(ids, wts)
    dw, db, dx = mok.router_backward(layer.sched, xc, wc, ids, wts, d.cuda(), with_bias=b is not None)
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(layer.sched) == 0
    return [t.cpu() if t is not None else None for t in (logits, ids, wts, dw, db, dx)]


def _check(x, w, b, K, d, got):
    logits, ids, wts, dw, db, dx = got
    xb, wb = inputs.bits(x), inputs.bits(w)
    bn = None if b is None else b.numpy()
    ref_l = oracle.router_logits(xb, wb, bn)
    assert np.array_equal(logits.numpy().view(np.uint32), ref_l.view(np.uint32))  # bit-exact
    ref_ids, ref_w = oracle.router_topk(ref_l, K)
    assert np.array_equal(ids.numpy(), ref_ids)
    assert rel_err(wts.double().numpy(), ref_w) <= TOL_W
    rdw, rdb, rdx = oracle.router_backward(xb, wb, ids.numpy(), wts.numpy(), d.numpy(), b is not None)
    errs = dict(dw=rel_err(dw.double().numpy(), rdw), dx=rel_err(to_f64(dx), rdx))
    if b is not None:
        errs["db"] = rel_err(db.double().numpy(), rdb)
    assert errs["dw"] <= TOL_DW and errs["dx"] <= TOL_DX and errs.get("db", 0.0) <= TOL_DW, errs


@pytest.mark.parametrize("T,H,E,K,bias", [(200, 256, 12, 3, False), (333, 384, 40, 8, True), (64, 128, 1, 1, False),
                                          (50, 256, 32, 32, True), (0, 128, 8, 2, False),
                                          (100, 512, 160, 8, True),  # three expert blocks, the last partial
                                          (64, 1024, 320, 4, False)])  # dW grid of 640 blocks: one row part
def test_router_parity(mok, T, H, E, K, bias):
    x, w, b, d = _router_case(T, H, E, K, bias, seed=T + E)
    got = _run(mok, x, w, b, K, d)
    if T == 0:
        return
    _check(x, w, b, K, d, got)
    if E == K == 1:  # a single expert: weight 1, no gradient through the renormalisation
        assert torch.all(got[2] == 1.0) and not got[3].any()


def test_router_ties_choose_the_lower_expert(mok):
    T, H, E, K = 96, 256, 16, 4
    x, w, b, d = _router_case(T, H, E, K, False, seed=3)
    w[:, 9] = w[:, 2]   # experts 2 and 9 always tie; so do 5, 6, 7
    w[:, 6] = w[:, 5]
    w[:, 7] = w[:, 5]
    got = _run(mok, x, w, b, K, d)
    _check(x, w, b, K, d, got)
    ids = got[1].numpy()
    both = (ids == 2).any(1) & (ids == 9).any(1)
    for r in np.nonzero(both)[0]:
        assert list(ids[r]).index(2) < list(ids[r]).index(9)
    assert not ((ids == 9).any(1) & ~(ids == 2).any(1)).any()  # 9 never chosen without 2


def test_router_accumulates_into_dx_and_is_deterministic(mok):
    T, H, E, K = 120, 256, 24, 4
    x, w, b, d = _router_case(T, H, E, K, True, seed=8)
    xc, wc, bc = x.cuda(), w.cuda(), b.cuda()
    logits, ids, wts = mok.router_forward(xc, wc, bc, K)
    layer = mok.Layer(T, H, 128, E, K, mok.make_config(128, 256))
    layer.schedule(ids, wts)
    dx0 = (torch.randn((T, H), generator=torch.Generator().manual_seed(1)) * 0.01).to(torch.bfloat16).cuda()
    dxa = dx0.clone()
    dw1, db1, _ = mok.router_backward(layer.sched, xc, wc, ids, wts, d.cuda(), with_bias=True, dx=dxa)
    dw2, db2, dxb = mok.router_backward(layer.sched, xc, wc, ids, wts, d.cuda(), with_bias=True)
    torch.cuda.synchronize()
    assert torch.equal(dw1, dw2) and torch.equal(db1, db2)
    _, _, rdx = oracle.router_backward(inputs.bits(x), inputs.bits(w), ids.cpu().numpy(), wts.cpu().numpy(),
                                       d.numpy(), True)
    assert rel_err(to_f64(dxa.cpu()), rdx + to_f64(dx0.cpu())) <= TOL_DX
    # repeat of the forward: same bits
    l2, i2, w2 = mok.router_forward(xc, wc, bc, K)
    assert torch.equal(l2, logits) and torch.equal(i2, ids) and torch.equal(w2, wts)


@pytest.mark.parametrize("name", ["bf16_e64", "dsv3_e256"])
def test_router_full_size(mok, name):
    """The workloads' own router draws (x, W_r, bias): logits and ids bit-exact with the oracle, the
    ids agree with the fp64 routing of the input module except at near-ties, the backward with the
    layer's top-k weight gradient as d."""
    wl = inputs.WORKLOADS[name]
    dd = inputs.make(wl, seed=0, weight_device="cuda")
    x, w, b = dd["x"], dd["Wr"], dd["router_bias"]
    d = torch.randn((wl.T, wl.K), generator=torch.Generator().manual_seed(5))
    got = _run(mok, x, w, b, wl.K, d)
    _check(x, w, b, wl.K, d, got)
    agree = (np.sort(got[1].numpy(), 1) == np.sort(dd["topk_ids"].numpy(), 1)).all(1).mean()
    assert agree >= 0.99, agree
