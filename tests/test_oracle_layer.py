"""Pins of the oracle's forward and backward (fp64) of the routed SwiGLU expert layer.

Pages: SwiGLU experts, forward and backward, router-weight gradient computed inside the SwiGLU
backward ("Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary); dispatch and
combine driven by one schedule ("Mixture-of-Kittens(MoK)란? ...", section 4 (1)).

Pins, none of which re-types the oracle's loops:
  * E = 1, K = 1, weight 1 reduces to a dense SwiGLU MLP, computed with numpy matmul;
  * identical experts with renormalised weights reduce to the same dense MLP;
  * linearity in the combine weights and invariance under relabelling experts;
  * gradients against torch CPU fp64 autograd of the layer's loss <out, dY>;
  * central finite differences on the bf16 / fp32 input grids;
  * the two ways of computing the router-weight gradient agree;
  * the sampled (one output at a time) entry points agree with the full ones.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_build_gb300 import inputs


def _np_inputs(w, seed=0):
    d = inputs.make(w, seed=seed)
    return (d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]), inputs.bits(d["Wg"]),
            inputs.bits(d["Wu"]), inputs.bits(d["Wd"]), inputs.bits(d["dY"]))


def _dense_swiglu(xv, wg, wu, wd):
    g = xv @ wg.T
    u = xv @ wu.T
    a = g / (1.0 + np.exp(-g)) * u
    return a @ wd.T


def test_single_expert_top1_is_dense_mlp():
    w = inputs.custom(T=16, H=64, I=32, E=1, K=1)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w)
    s = np.ones_like(s)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    ref = _dense_swiglu(oracle.bf16_to_f64(x), oracle.bf16_to_f64(Wg[0]), oracle.bf16_to_f64(Wu[0]),
                        oracle.bf16_to_f64(Wd[0]))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_identical_experts_renormalised_is_dense_mlp():
    w = inputs.custom(T=32, H=64, I=32, E=4, K=3)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=3)
    Wg = np.repeat(Wg[:1], 4, axis=0)
    Wu = np.repeat(Wu[:1], 4, axis=0)
    Wd = np.repeat(Wd[:1], 4, axis=0)
    s64 = s.astype(np.float64)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    ref = _dense_swiglu(oracle.bf16_to_f64(x), oracle.bf16_to_f64(Wg[0]), oracle.bf16_to_f64(Wu[0]),
                        oracle.bf16_to_f64(Wd[0])) * s64.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    assert np.allclose(s64.sum(axis=1), 1.0, atol=1e-6)  # renormalised routing


def test_linear_in_weights_and_invariant_to_expert_relabelling():
    w = inputs.custom(T=24, H=32, I=16, E=5, K=2)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=4)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    out2 = oracle.forward(ids, (2 * s).astype(np.float32), x, Wg, Wu, Wd)
    assert np.array_equal(out2, 2 * out)
    pi = np.array([3, 0, 4, 1, 2])
    Wg2, Wu2, Wd2 = np.empty_like(Wg), np.empty_like(Wu), np.empty_like(Wd)
    Wg2[pi], Wu2[pi], Wd2[pi] = Wg, Wu, Wd
    out3 = oracle.forward(pi[ids].astype(np.int32), s, x, Wg2, Wu2, Wd2)
    assert np.array_equal(out3, out)
    g1 = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    g3 = oracle.backward(pi[ids].astype(np.int32), s, x, Wg2, Wu2, Wd2, dY)
    assert np.array_equal(g3["dX"], g1["dX"]) and np.array_equal(g3["dS"], g1["dS"])
    assert np.array_equal(g3["dWg"][pi], g1["dWg"]) and np.array_equal(g3["dWd"][pi], g1["dWd"])


def _torch_reference(ids, s, x, Wg, Wu, Wd, dY):
    """Loss <out, dY> in torch fp64 with autograd; gradients come from the library."""
    X = torch.from_numpy(oracle.bf16_to_f64(x)).requires_grad_()
    G = torch.from_numpy(oracle.bf16_to_f64(Wg)).requires_grad_()
    U = torch.from_numpy(oracle.bf16_to_f64(Wu)).requires_grad_()
    D = torch.from_numpy(oracle.bf16_to_f64(Wd)).requires_grad_()
    S = torch.from_numpy(s.astype(np.float64)).requires_grad_()
    idx = torch.from_numpy(ids.astype(np.int64))
    T, K = ids.shape
    xs = X[:, None, :].expand(T, K, X.shape[1])                      # [T,K,H]
    g = torch.einsum("tkh,tkih->tki", xs, G[idx])
    u = torch.einsum("tkh,tkih->tki", xs, U[idx])
    a = torch.nn.functional.silu(g) * u
    y = torch.einsum("tki,tkhi->tkh", a, D[idx])
    out = (S[:, :, None] * y).sum(dim=1)
    loss = (out * torch.from_numpy(oracle.bf16_to_f64(dY))).sum()
    loss.backward()
    return out.detach().numpy(), dict(dX=X.grad.numpy(), dWg=G.grad.numpy(), dWu=U.grad.numpy(),
                                      dWd=D.grad.numpy(), dS=S.grad.numpy())


@pytest.mark.parametrize("T,H,I,E,K,seed", [(40, 64, 32, 6, 2, 0), (17, 32, 64, 3, 3, 1), (8, 16, 16, 1, 1, 2)])
def test_against_torch_autograd(T, H, I, E, K, seed):
    w = inputs.custom(T=T, H=H, I=I, E=E, K=K)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=seed)
    ids[0, :] = ids[0, 0]  # a duplicated expert within one token
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    grads = oracle.backward(ids, s, x, Wg, Wu, Wd, dY, check=True)
    rout, rg = _torch_reference(ids, s, x, Wg, Wu, Wd, dY)
    np.testing.assert_allclose(out, rout, rtol=1e-10, atol=1e-12)
    for k in ("dX", "dWg", "dWu", "dWd", "dS"):
        scale = np.abs(rg[k]).max()
        assert np.abs(grads[k] - rg[k]).max() <= 1e-10 * scale, k
    np.testing.assert_allclose(grads["dS"], grads["dS_check"], rtol=1e-10, atol=1e-12)


def _next_bf16(b, direction):
    """Neighbouring bf16 bit pattern (positive finite values only used here)."""
    return np.uint16(int(b) + direction) if b & 0x8000 == 0 else np.uint16(int(b) - direction)


def test_finite_differences():
    w = inputs.custom(T=4, H=8, I=4, E=3, K=2)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=7)
    dYv = oracle.bf16_to_f64(dY)
    grads = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)

    def loss(ids_, s_, x_, Wg_, Wu_, Wd_):
        return float((oracle.forward(ids_, s_, x_, Wg_, Wu_, Wd_) * dYv).sum())

    def fd_bf16(arr, idx, f):
        up, dn = arr.copy(), arr.copy()
        up[idx] = _next_bf16(arr[idx], +1)
        dn[idx] = _next_bf16(arr[idx], -1)
        hu = oracle.bf16_value(up[idx]) - oracle.bf16_value(arr[idx])
        hd = oracle.bf16_value(arr[idx]) - oracle.bf16_value(dn[idx])
        # non-uniform central difference, second-order accurate
        fu, f0, fdn = f(up), f(arr), f(dn)
        return (hd * hd * (fu - f0) + hu * hu * (f0 - fdn)) / (hu * hd * (hu + hd))

    rng = np.random.default_rng(0)
    for _ in range(6):
        t, h = rng.integers(0, 4), rng.integers(0, 8)
        num = fd_bf16(x, (t, h), lambda a: loss(ids, s, a, Wg, Wu, Wd))
        assert abs(num - grads["dX"][t, h]) <= 2e-3 * (abs(grads["dX"][t, h]) + 1e-3), (t, h)
    used = sorted(set(ids.reshape(-1).tolist()))
    for _ in range(6):
        e = used[rng.integers(0, len(used))]
        i, h = rng.integers(0, 4), rng.integers(0, 8)
        num = fd_bf16(Wg, (e, i, h), lambda a: loss(ids, s, x, a, Wu, Wd))
        assert abs(num - grads["dWg"][e, i, h]) <= 2e-3 * (abs(grads["dWg"][e, i, h]) + 1e-4)
        num = fd_bf16(Wu, (e, i, h), lambda a: loss(ids, s, x, Wg, a, Wd))
        assert abs(num - grads["dWu"][e, i, h]) <= 2e-3 * (abs(grads["dWu"][e, i, h]) + 1e-4)
        num = fd_bf16(Wd, (e, h, i), lambda a: loss(ids, s, x, Wg, Wu, a))
        assert abs(num - grads["dWd"][e, h, i]) <= 2e-3 * (abs(grads["dWd"][e, h, i]) + 1e-4)
    # combine weights are fp32: a small symmetric step is exact on that grid
    for t in range(4):
        for k in range(2):
            hs = np.float32(2.0 ** -12)
            sp, sm = s.copy(), s.copy()
            sp[t, k] += hs
            sm[t, k] -= hs
            num = (loss(ids, sp, x, Wg, Wu, Wd) - loss(ids, sm, x, Wg, Wu, Wd)) / (2 * float(hs))
            assert abs(num - grads["dS"][t, k]) <= 1e-9 * (abs(grads["dS"][t, k]) + 1.0)
    # unused experts have zero gradient
    for e in range(3):
        if e not in used:
            assert not grads["dWg"][e].any() and not grads["dWd"][e].any()


def test_sampled_entry_points_match_full():
    w = inputs.custom(T=50, H=64, I=32, E=7, K=3)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=9)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    g = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    tok = np.array([0, 7, 49, 23])
    np.testing.assert_allclose(oracle.forward_tokens(ids, s, x, Wg, Wu, Wd, tok), out[tok], rtol=1e-12, atol=1e-14)
    dX, dS = oracle.backward_tokens(ids, s, x, Wg, Wu, Wd, dY, tok)
    np.testing.assert_allclose(dX, g["dX"][tok], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dS, g["dS"][tok], rtol=1e-12, atol=1e-14)
    rng = np.random.default_rng(1)
    n = 64
    which = rng.integers(0, 3, n)
    e = rng.integers(0, 7, n)
    m = np.where(which == 2, rng.integers(0, 64, n), rng.integers(0, 32, n))
    c = np.where(which == 2, rng.integers(0, 32, n), rng.integers(0, 64, n))
    val = oracle.dw_entries(ids, s, x, Wg, Wu, Wd, dY, which, e, m, c)
    full = [g["dWg"], g["dWu"], g["dWd"]]
    ref = np.array([full[wh][ee, mm, cc] for wh, ee, mm, cc in zip(which, e, m, c)])
    np.testing.assert_allclose(val, ref, rtol=1e-11, atol=1e-14)
    # the block entry point: one 32-column block of I against sampled hidden columns, every expert
    # (expert 6 may have no slot: exact zeros)
    hs = np.array([0, 5, 63, 31, 32])
    for ee in range(7):
        dwg, dwu, dwd = oracle.dw_block(ids, s, x, Wg, Wu, Wd, dY, ee, 0, hs)
        np.testing.assert_allclose(dwg, g["dWg"][ee, 0:32][:, hs], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(dwu, g["dWu"][ee, 0:32][:, hs], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(dwd, g["dWd"][ee][hs, 0:32], rtol=1e-11, atol=1e-14)
    w2 = inputs.custom(T=30, H=64, I=96, E=3, K=2)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w2, seed=10)
    g = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    dwg, dwu, dwd = oracle.dw_block(ids, s, x, Wg, Wu, Wd, dY, 1, 64, hs)
    np.testing.assert_allclose(dwg, g["dWg"][1, 64:96][:, hs], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dwu, g["dWu"][1, 64:96][:, hs], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dwd, g["dWd"][1][hs, 64:96], rtol=1e-11, atol=1e-14)


def test_intermediates_consistent():
    w = inputs.custom(T=12, H=32, I=16, E=4, K=2)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=11)
    out, it = oracle.forward(ids, s, x, Wg, Wu, Wd, intermediates=True)
    T, K = ids.shape
    ref = (s.astype(np.float64)[:, :, None] * it["y"].reshape(T, K, -1)).sum(axis=1)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-15)
    g, u = it["g"], it["u"]
    np.testing.assert_allclose(it["a"], g / (1 + np.exp(-g)) * u, rtol=1e-13, atol=1e-16)


def test_fp32_timing_build_computes_the_same_layer():
    """The fp32 -O3 build of the layer loops (the timed CPU baseline) computes the same layer as
    the fp64 reference, to fp32 rounding."""
    w = inputs.custom(T=40, H=128, I=64, E=4, K=2)
    ids, s, x, Wg, Wu, Wd, dY = _np_inputs(w, seed=12)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    ref = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    got = oracle.step_f32(ids, s, x, Wg, Wu, Wd, dY)
    assert got["out"].dtype == np.float32
    rel = lambda a, b: np.abs(a.astype(np.float64) - b).max() / np.abs(b).max()  # noqa: E731
    assert rel(got["out"], out) < 1e-5
    for k in ("dX", "dWg", "dWu", "dWd", "dS"):
        assert rel(got[k], ref[k]) < 1e-5, k
        assert not np.array_equal(got[k].astype(np.float64), ref[k]), k  # really computed in fp32
