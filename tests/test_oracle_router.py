"""Pins of the router-step oracle (oracle/mok_oracle_router.c) against what does not depend on it:
exact special cases, the fp32 error bound of the logits, numpy's stable sort and softmax, torch
fp64 autograd and central finite differences."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_build_gb300 import inputs


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return inputs.bits(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16))


def _rand(shape, std, seed):
    return _bf16_bits(np.random.default_rng(seed).normal(0.0, std, shape))


def test_logits_of_one_hot_rows_are_the_weight_rows_exactly():
    H, E = 96, 7
    w = _rand((H, E), 0.5, 1)
    hs = np.array([0, 5, 95, 40])
    x = np.zeros((len(hs), H), dtype=np.float32)
    x[np.arange(len(hs)), hs] = 1.0
    bias = np.linspace(-1, 1, E).astype(np.float32)
    lg = oracle.router_logits(_bf16_bits(x), w, bias)
    want = oracle.bf16_to_f64(w)[hs].astype(np.float32) + bias  # one product, then one fp32 add
    assert np.array_equal(lg, want)


def test_logits_within_the_fp32_sequential_error_bound():
    T, H, E = 16, 2048, 64
    x, w = _rand((T, H), 1.0, 2), _rand((H, E), 0.02, 3)
    bias = np.random.default_rng(4).normal(0, 0.5, E).astype(np.float32)
    lg = oracle.router_logits(x, w, bias).astype(np.float64)
    xd, wd = oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)
    exact = xd @ wd + bias.astype(np.float64)
    # H + 1 roundings of magnitude at most the running sum of |x w| (+ |b|)
    bound = (H + 1) * 2.0 ** -24 * (np.abs(xd) @ np.abs(wd) + np.abs(bias))
    err = np.abs(lg - exact)
    assert (err <= bound).all()
    assert err.max() > 0  # not computed in fp64 by mistake


def test_topk_matches_a_stable_descending_sort_including_ties():
    rng = np.random.default_rng(5)
    T, E, K = 64, 24, 6
    lg = rng.normal(0, 1, (T, E)).astype(np.float32)
    lg[::3, 4] = lg[::3, 9]  # equal logits: the lower id must come first
    lg[1::3, 2:6] = 0.25
    ids, wts = oracle.router_topk(lg, K)
    want = np.argsort(-lg, axis=1, kind="stable")[:, :K]
    assert np.array_equal(ids, want)
    # renormalised weights = numpy's softmax over all E, restricted to the selection and renormalised
    p = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, want, axis=1)
    np.testing.assert_allclose(wts, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(wts.sum(axis=1), 1.0, rtol=1e-12)
    assert (np.diff(wts, axis=1) <= 0).all()


@pytest.mark.parametrize("with_bias", [False, True])
def test_backward_matches_torch_autograd(with_bias):
    rng = np.random.default_rng(6)
    T, H, E, K = 24, 40, 9, 3
    x, w = _rand((T, H), 1.0, 7), _rand((H, E), 0.3, 8)
    bias = rng.normal(0, 0.5, E).astype(np.float32) if with_bias else None
    d = rng.normal(0, 1, (T, K)).astype(np.float32)
    ids, _ = oracle.router_topk(oracle.router_logits(x, w, bias), K)
    xt = torch.tensor(oracle.bf16_to_f64(x), requires_grad=True)
    wt = torch.tensor(oracle.bf16_to_f64(w), requires_grad=True)
    bt = torch.tensor(bias.astype(np.float64) if with_bias else np.zeros(E), requires_grad=True)
    p = torch.softmax(xt @ wt + bt, dim=1)
    sel = torch.gather(p, 1, torch.from_numpy(ids).long())
    wk = sel / sel.sum(dim=1, keepdim=True)
    (wk * torch.from_numpy(d).double()).sum().backward()
    dw, db, dx = oracle.router_backward(x, w, ids, wk.detach().numpy().astype(np.float32), d, with_bias)
    # the oracle takes the fp32 weights: relative 2^-24 in each w_k
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-5, atol=1e-6 * np.abs(wt.grad.numpy()).max())
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-5, atol=1e-6 * np.abs(xt.grad.numpy()).max())
    if with_bias:
        np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-5, atol=1e-6 * np.abs(bt.grad.numpy()).max())


def test_backward_matches_central_differences_of_the_weights():
    # one token, the selected logits moved one at a time: d/dl_j sum_k d_k w_k(l)
    rng = np.random.default_rng(9)
    H, E, K = 1, 8, 4
    lsel = rng.normal(0, 1, K)
    d = rng.normal(0, 1, K).astype(np.float32)

    def f(l):
        e = np.exp(l - l.max())
        return float((e / e.sum()) @ d.astype(np.float64))

    h = 1e-6
    fd = np.array([(f(lsel + h * np.eye(K)[j]) - f(lsel - h * np.eye(K)[j])) / (2 * h) for j in range(K)])
    # x = 1 on a single hidden unit and W row = the logits: dW[0, ids] is then dL/dl
    ids = np.arange(K, dtype=np.int32)[None, :]
    e = np.exp(lsel - lsel.max())
    wts = (e / e.sum()).astype(np.float32)[None, :]
    x = _bf16_bits(np.ones((1, H)))
    w = _bf16_bits(np.zeros((H, E)))
    dw, _, _ = oracle.router_backward(x, w, ids, wts, d[None, :])
    np.testing.assert_allclose(dw[0, :K], fd, rtol=1e-5, atol=1e-7)
    assert not dw[0, K:].any()  # unselected logits get no gradient
