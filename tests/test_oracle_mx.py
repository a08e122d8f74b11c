"""Pins of the oracle's MXFP8 mode (mok_oracle_mx.c).

The MXFP8 mode is the BF16 layer with MX quantise-dequantise steps at fixed points (x and dY along
H, a and dg/du along I, weights pre-quantised along each GEMM's K).  Pins:
  * the fp64 quantise-dequantise equals the byte-level quantiser (itself pinned against torch's
    float8 conversion) on bf16 inputs, and is idempotent;
  * with quantisation switched off and weights already on the MX grid, the MXFP8 dataflow equals
    the BF16 oracle (pinned against torch autograd and finite differences);
  * with quantisation on, the saved a_q is exactly the quantised SwiGLU output of the BF16 oracle
    run on the quantised inputs;
  * the weight gradients quantise their operands along the routed rows: rebuilt here from the
    expert-grouped row order (numpy stable sort, zero padding to 128 rows, blocks of 32 rows);
  * the forward and data-gradient quantisation points (x and dY along H, a along I, dA' from the
    copy of Wd^T, dS on a_q, dg and du along I into the copies of Wg^T and Wu^T) are rebuilt from
    independent parts: a numpy / torch-float8 quantiser, weights decoded by torch, numpy matmuls
    and torch autograd for the SwiGLU backward; plausible slips (dY left unquantised, a in place
    of a_q, the forward copy of Wd in place of Wd^T's, dg left unquantised) are shown to move the
    result far beyond the tolerance;
  * the sampled entry points agree with the full one.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_build_gb300 import inputs


def _bits(a):
    return inputs.bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def test_fakequant_matches_byte_quantiser_and_is_idempotent():
    rng = np.random.default_rng(0)
    x = _bits(rng.standard_normal((16, 256)) * 2.0 ** rng.integers(-20, 20, size=(16, 1)))
    q, sc = oracle.mxfp8_quantize(x)
    deq = oracle.mxfp8_dequantize(q, sc)
    fq = oracle.mx_fakequant(oracle.bf16_to_f64(x))
    assert np.array_equal(fq, deq)
    assert np.array_equal(oracle.mx_fakequant(fq), fq)
    # fp64 inputs that are not bf16: within half a quantum of the block's top binade (quantum
    # 2^(floor(log2 amax) - 3)), except values beyond 448 * 2^shared, which saturate
    v = rng.standard_normal((4, 64))
    f = oracle.mx_fakequant(v).reshape(4, 2, 32)
    blocks = v.reshape(4, 2, 32)
    _, ex = np.frexp(np.abs(blocks).max(axis=2))
    shared = (ex - 1 - 8)[:, :, None]
    quantum = 2.0 ** (ex - 1 - 3)[:, :, None]
    sat = np.abs(blocks) >= 448.0 * 2.0 ** shared
    assert np.all(np.abs(f - blocks)[~sat] <= (quantum / 2 * np.ones_like(blocks))[~sat])
    assert np.all(np.abs(f[sat]) == (448.0 * 2.0 ** shared * np.ones_like(blocks))[sat])


def _grid_weights(rng, E, I, H):
    """bf16 weights whose values are already on their MX grids along both axes: signed powers of
    two in [2^-9, 2^-3], so any 32-block holds them at most 2^6 below its top, exactly in E4M3."""
    w = rng.standard_normal((E, I, H)) * 0.02
    signs = np.sign(w)
    e = np.clip(np.round(np.log2(np.abs(w) + 1e-30)), -9, -3)
    return _bits(signs * 2.0 ** e)


def test_dataflow_without_quantisation_equals_bf16_oracle():
    rng = np.random.default_rng(1)
    T, H, I, E, K = 24, 64, 64, 3, 2
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    s = rng.random((T, K)).astype(np.float32)
    x = _bits(rng.standard_normal((T, H)))
    dY = _bits(rng.standard_normal((T, H)))
    Wg, Wu = _grid_weights(rng, E, I, H), _grid_weights(rng, E, I, H)
    Wd = _grid_weights(rng, E, H, I)
    mx = oracle.mx_weights(Wg, Wu, Wd)
    # the grid weights decode exactly from every copy
    assert np.array_equal(oracle.mxfp8_dequantize(mx["q_gate"], mx["s_gate"]).reshape(E, I, H),
                          oracle.bf16_to_f64(Wg))
    assert np.array_equal(oracle.mxfp8_dequantize(mx["qt_down"], mx["st_down"]).reshape(E, I, H),
                          oracle.bf16_to_f64(Wd).transpose(0, 2, 1))
    oracle.mx_set_quant(False)
    try:
        r = oracle.layer_mx(ids, s, x, dY, mx, E, I)
    finally:
        oracle.mx_set_quant(True)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    ref = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-14)
    for k in ("dX", "dWg", "dWu", "dWd", "dS"):
        np.testing.assert_allclose(r[k], ref[k], rtol=1e-11, atol=1e-13, err_msg=k)


def test_quantisation_point_of_a():
    rng = np.random.default_rng(2)
    T, H, I, E, K = 16, 64, 64, 2, 1
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    s = np.ones((T, K), np.float32)
    x = _bits(rng.standard_normal((T, H)))
    Wg, Wu = _grid_weights(rng, E, I, H), _grid_weights(rng, E, I, H)
    Wd = _grid_weights(rng, E, H, I)
    mx = oracle.mx_weights(Wg, Wu, Wd)
    r = oracle.layer_mx(ids, s, x, x, mx, E, I, with_aq=True)
    xq = _bits(oracle.mx_fakequant(oracle.bf16_to_f64(x)))  # E4M3 x 2^k values are bf16-exact
    _, it = oracle.forward(ids, s, xq, Wg, Wu, Wd, intermediates=True)
    np.testing.assert_allclose(r["aq"], oracle.mx_fakequant(it["a"]), rtol=0, atol=1e-15)
    assert not np.array_equal(r["aq"], it["a"])  # the quantisation really happened


def test_sampled_entry_points_agree_with_full():
    rng = np.random.default_rng(3)
    w = inputs.custom(T=40, H=128, I=64, E=3, K=2)
    d = inputs.make(w, seed=5)
    args = (d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]), inputs.bits(d["dY"]))
    mx = oracle.mx_weights(inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
    full = oracle.layer_mx(*args, mx, w.E, w.I)
    tok = np.array([0, 11, 39])
    out, dX, dS = oracle.tokens_mx(*args, mx, w.E, w.I, tok)
    np.testing.assert_allclose(out, full["out"][tok], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dX, full["dX"][tok], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dS, full["dS"][tok], rtol=1e-12, atol=1e-14)
    hs = np.array([0, 5, 127, 64])
    for e in range(w.E):
        dwg, dwu, dwd = oracle.dw_block_mx(*args, mx, w.E, w.I, e, 32, hs)
        np.testing.assert_allclose(dwg, full["dWg"][e, 32:64][:, hs], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(dwu, full["dWu"][e, 32:64][:, hs], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(dwd, full["dWd"][e][hs, 32:64], rtol=1e-11, atol=1e-14)


def test_mx_mode_is_close_to_bf16():
    w = inputs.custom(T=32, H=128, I=64, E=4, K=2)
    d = inputs.make(w, seed=6)
    ids, s = d["topk_ids"].numpy(), d["topk_weights"].numpy()
    x, dY = inputs.bits(d["x"]), inputs.bits(d["dY"])
    Wg, Wu, Wd = inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"])
    r = oracle.layer_mx(ids, s, x, dY, oracle.mx_weights(Wg, Wu, Wd), w.E, w.I)
    out = oracle.forward(ids, s, x, Wg, Wu, Wd)
    ref = oracle.backward(ids, s, x, Wg, Wu, Wd, dY)
    rel = lambda a, b: np.abs(a - b).max() / np.abs(b).max()  # noqa: E731
    assert rel(r["out"], out) < 0.15
    for k in ("dX", "dWg", "dWd", "dS"):
        assert rel(r[k], ref[k]) < 0.2, k


def _qr(m):
    """MX quantise-dequantise along rows: every column of m [nrows, ncols] in blocks of 32 rows."""
    out = np.empty_like(m)
    for r0 in range(0, m.shape[0], 32):
        out[r0:r0 + 32] = _q32(np.ascontiguousarray(m[r0:r0 + 32].T)).T
    return out


def test_wgrad_quantised_along_expert_rows():
    rng = np.random.default_rng(4)
    T, H, I, E, K = 100, 64, 64, 3, 2
    ids = rng.integers(0, E - 1, size=(T, K)).astype(np.int32)  # expert E-1 gets no rows
    s = rng.uniform(0.1, 0.9, size=(T, K)).astype(np.float32)
    xf = rng.standard_normal((T, H)) * np.where(np.arange(T) < 30, 2.0 ** 8, 1.0)[:, None]
    x, dY = _bits(xf), _bits(rng.standard_normal((T, H)))
    Wg, Wu, Wd = (_bits(rng.standard_normal(sh) * 0.05) for sh in ((E, I, H), (E, I, H), (E, H, I)))
    mx = oracle.mx_weights(Wg, Wu, Wd)
    r = oracle.layer_mx(ids, s, x, dY, mx, E, I, with_dg=True)
    xv, dyv = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dY)
    flat = ids.reshape(-1)
    for e in range(E):
        slots = np.flatnonzero(flat == e)  # ascending slot order inside the expert
        npad = -(-slots.size // 128) * 128
        def seg(rows):  # noqa: E306
            m = np.zeros((npad, rows.shape[1]))
            m[:slots.size] = rows
            return m
        qdg, qdu = _qr(seg(r["dg"][slots])), _qr(seg(r["du"][slots]))
        qsa = _qr(seg(s.reshape(-1)[slots, None].astype(np.float64) * r["a"][slots]))
        qx, qdy = _qr(seg(xv[slots // K])), _qr(seg(dyv[slots // K]))
        np.testing.assert_allclose(r["dWg"][e], qdg.T @ qx, rtol=1e-11, atol=1e-12, err_msg=f"dWg {e}")
        np.testing.assert_allclose(r["dWu"][e], qdu.T @ qx, rtol=1e-11, atol=1e-12, err_msg=f"dWu {e}")
        np.testing.assert_allclose(r["dWd"][e], qdy.T @ qsa, rtol=1e-11, atol=1e-12, err_msg=f"dWd {e}")
    assert not np.any(r["dWg"][E - 1]) and not np.any(r["dWd"][E - 1])
    # the row blocks matter: quantising x along H instead would give a different dWg
    qx_h = oracle.mx_fakequant(xv)
    slots = np.flatnonzero(flat == 0)
    alt = _qr(np.pad(r["dg"][slots], ((0, -slots.size % 128), (0, 0)))).T @ np.pad(qx_h[slots // K], ((0, -slots.size % 128), (0, 0)))
    assert not np.allclose(alt, r["dWg"][0], rtol=1e-6)


# ------------------------------------------------------------------------------------------------
# Independent rebuild of the forward and data-gradient quantisation points
# ------------------------------------------------------------------------------------------------
def _e4m3_grid():
    """Non-negative finite E4M3 values in code order (codes 0x00 .. 0x7E), decoded by torch."""
    codes = torch.arange(0x7F, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


_GRID = _e4m3_grid()


def _q32(v):
    """MX quantise-dequantise along the last axis in blocks of 32, built without the oracle: the
    shared exponent floor(log2 amax) - 8 from numpy's frexp (clamped to [-127, 127], -127 for an
    all-zero block), then the nearest value of torch's decoded E4M3 grid with ties to the even
    code, saturating at 448."""
    v = np.asarray(v, np.float64)
    blocks = v.reshape(-1, 32)
    amax = np.abs(blocks).max(axis=1)
    _, ex = np.frexp(amax)
    shared = np.where(amax > 0, np.clip(ex - 1 - 8, -127, 127), -127).astype(np.float64)
    scale = 2.0 ** shared[:, None]
    mag = np.minimum(np.abs(blocks) / scale, _GRID[-1])
    hi = np.clip(np.searchsorted(_GRID, mag), 0, _GRID.size - 1)
    lo = np.clip(hi - 1, 0, _GRID.size - 1)
    dlo, dhi = mag - _GRID[lo], _GRID[hi] - mag
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (np.sign(blocks) * _GRID[pick] * scale).reshape(v.shape)


def _decode(q, sc):
    """Value of an MXFP8 matrix from its bytes: torch's float8 decode times 2^(scale - 127)."""
    codes = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes * np.repeat(2.0 ** (sc.astype(np.float64) - 127.0), 32, axis=1)


def _rebuild(ids, s, x, dY, mx, E, I, *, quant_dy=True, ds_on_aq=True, dap_from_wdt=True, quant_dg=True):
    """Forward and data gradients of the MXFP8 mode from the reading of the quantisation points,
    with switches that plant the slips the test must catch."""
    T, K = ids.shape
    H = x.shape[1]
    R = T * K
    e = ids.reshape(-1).astype(np.int64)
    t = np.arange(R) // K
    sv = s.reshape(-1).astype(np.float64)
    Wg = _decode(mx["q_gate"], mx["s_gate"]).reshape(E, I, H)    # along H
    Wu = _decode(mx["q_up"], mx["s_up"]).reshape(E, I, H)
    Wd = _decode(mx["q_down"], mx["s_down"]).reshape(E, H, I)    # along I
    Wgt = _decode(mx["qt_gate"], mx["st_gate"]).reshape(E, H, I)  # Wg^T along I
    Wut = _decode(mx["qt_up"], mx["st_up"]).reshape(E, H, I)
    Wdt = _decode(mx["qt_down"], mx["st_down"]).reshape(E, I, H)  # Wd^T along H
    xq = _q32(oracle.bf16_to_f64(x))
    dy = oracle.bf16_to_f64(dY)
    dyq = _q32(dy) if quant_dy else dy
    g = torch.from_numpy(np.einsum("jih,jh->ji", Wg[e], xq[t])).requires_grad_(True)
    u = torch.from_numpy(np.einsum("jih,jh->ji", Wu[e], xq[t])).requires_grad_(True)
    a_t = torch.nn.functional.silu(g) * u
    a = a_t.detach().numpy()
    aq = _q32(a)
    y = np.einsum("jhi,ji->jh", Wd[e], aq)
    out = np.zeros((T, H))
    np.add.at(out, t, sv[:, None] * y)
    if dap_from_wdt:
        dap = np.einsum("jih,jh->ji", Wdt[e], dyq[t])
    else:  # the forward copy of Wd (quantised along I) read transposed
        dap = np.einsum("jhi,jh->ji", Wd[e], dyq[t])
    dS = np.einsum("ji,ji->j", dap, aq if ds_on_aq else a).reshape(T, K)
    a_t.backward(torch.from_numpy(sv[:, None] * dap))  # SwiGLU backward by autograd
    dg, du = g.grad.numpy(), u.grad.numpy()
    dgq, duq = (_q32(dg), _q32(du)) if quant_dg else (dg, du)
    dX = np.zeros((T, H))
    np.add.at(dX, t, np.einsum("jhi,ji->jh", Wgt[e], dgq) + np.einsum("jhi,ji->jh", Wut[e], duq))
    return dict(out=out, a=a, aq=aq, dS=dS, dg=dg, du=du, dX=dX)


def _mx_case(seed=11):
    rng = np.random.default_rng(seed)
    T, H, I, E, K = 40, 128, 96, 3, 2
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    s = rng.uniform(0.1, 0.9, size=(T, K)).astype(np.float32)
    row_scale = 2.0 ** rng.integers(-6, 7, size=(T, 1))  # spread the block exponents
    x = _bits(rng.standard_normal((T, H)) * row_scale)
    dY = _bits(rng.standard_normal((T, H)) * row_scale[::-1])
    Wg, Wu, Wd = (_bits(rng.standard_normal(sh) * 0.05) for sh in ((E, I, H), (E, I, H), (E, H, I)))
    return ids, s, x, dY, oracle.mx_weights(Wg, Wu, Wd), E, I


def test_quantiser_rebuild_agrees_with_oracle_quantiser():
    """The test's own quantiser (numpy + torch float8 grid) equals the oracle's on fp64 values off
    the bf16 grid, including ties and saturation -- so the rebuild below shares nothing with the
    oracle but agrees with it where they must."""
    rng = np.random.default_rng(12)
    v = rng.standard_normal((64, 96)) * 2.0 ** rng.integers(-30, 30, size=(64, 1))
    v[0, :32] = 0.0
    v[1, :32] = np.linspace(-1, 1, 32) * 448.0 * 1.9  # block whose top values saturate
    # a block with shared = 0 (amax 256) holding exact ties between neighbouring codes
    v[2, :32] = 0.0
    v[2, :6] = [256.0, 1.0625, 1.1875, -1.0625, 3 * 2.0 ** -10, 2.0 ** -10]
    v[3, :32] = 2.0 ** -140 * np.arange(32)  # clamped exponent (-127), subnormal codes
    assert np.array_equal(_q32(v), oracle.mx_fakequant(v))


def test_data_gradient_quantisation_points_rebuilt():
    ids, s, x, dY, mx, E, I = _mx_case()
    r = oracle.layer_mx(ids, s, x, dY, mx, E, I, with_aq=True, with_dg=True)
    ref = _rebuild(ids, s, x, dY, mx, E, I)
    rel = lambda a, b: np.abs(a - b).max() / np.abs(b).max()  # noqa: E731
    for k_or, k_rb in (("out", "out"), ("a", "a"), ("aq", "aq"), ("dS", "dS"), ("dg", "dg"), ("du", "du"),
                       ("dX", "dX")):
        assert rel(r[k_or], ref[k_rb]) <= 1e-11, (k_or, rel(r[k_or], ref[k_rb]))


@pytest.mark.parametrize("slip,keys", [
    (dict(quant_dy=False), ("dS", "dg", "dX")),     # dY not quantised along H
    (dict(ds_on_aq=False), ("dS",)),                # dS formed with a instead of a_q
    (dict(dap_from_wdt=False), ("dS", "dg", "dX")),  # the forward copy of Wd instead of Wd^T's
    (dict(quant_dg=False), ("dX",)),                # dg, du not quantised along I before dgrad2
])
def test_planted_quantisation_slips_are_caught(slip, keys):
    """Each plausible slip moves the affected outputs by far more than the rebuild's 1e-11, so the
    pin above would fail on it."""
    ids, s, x, dY, mx, E, I = _mx_case()
    r = oracle.layer_mx(ids, s, x, dY, mx, E, I, with_aq=True, with_dg=True)
    bad = _rebuild(ids, s, x, dY, mx, E, I, **slip)
    for k in keys:
        assert np.abs(r[k] - bad[k]).max() / np.abs(r[k]).max() > 1e-4, k
