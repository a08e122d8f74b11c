"""GPU MXFP8 mode vs the fp64 MXFP8 oracle (mok_oracle_mx.c), through the C ABI.

Tolerance (MXFP8): max|gpu - oracle| / max|oracle| <= 4e-2 per output tensor.  The pre-quantised
weight bytes the GPU consumes come from mok_mxfp8_quantize and must equal the oracle's own
quantisation bit for bit; activations are quantised inside the library (x, dY in the gather,
along H and along the routed rows; a, dg, du, s*a in the GEMM epilogues) and the oracle mirrors
those points in fp64.
"""
import numpy as np
import pytest
import torch

import fullsize
import oracle
from helpers import rel_err, to_f64
from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_MX = 4e-2


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _run_mx(mok, d, w, cfg, mx_gpu):
    x, ids, s, dY = (d[k].cuda() for k in ("x", "topk_ids", "topk_weights", "dY"))
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    weights = mok.weights_struct(mx=mx_gpu)
    layer.schedule(ids, s)
    out = layer.forward(x, weights)
    g = layer.backward(dY, weights)
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(layer.sched) == 0
    return out, g


def _mx_inputs(mok, d):
    Wg, Wu, Wd = (d[k].cuda() for k in ("Wg", "Wu", "Wd"))
    mx_gpu = mok.quantize_weights(Wg, Wu, Wd)
    torch.cuda.synchronize()
    return mx_gpu


SMALL = [
    ("tiny", inputs.WORKLOADS["tiny"]),
    ("ragged", inputs.custom(T=100, H=256, I=256, E=5, K=3)),
    ("multi_tile", inputs.custom(T=700, H=512, I=384, E=3, K=2)),
    ("h384", inputs.custom(T=300, H=384, I=256, E=3, K=2)),  # H not a multiple of 256: 128-wide tiles
    # H above 4096: the first data-gradient GEMM runs its other epilogue (four warps)
    ("long_h", inputs.custom(T=160, H=4224, I=256, E=3, K=2)),
    # H above 4096 and a multiple of 256: the four-warp first data-gradient epilogue together with
    # the 128 x 256 tiles of the other GEMMs (the EP64 shard's combination, H = 7168)
    ("long_h_wide", inputs.custom(T=160, H=4352, I=256, E=3, K=2)),
    # 2,048 routed rows per expert: the weight gradients run on CTA pairs (128 x 256 tiles per CTA;
    # with H = 384 the gate/up one takes 128-column tiles and the down one stays on single CTAs)
    ("long_experts", inputs.custom(T=4096, H=256, I=256, E=2, K=1)),
    ("long_experts_h384", inputs.custom(T=4096, H=384, I=128, E=2, K=1)),
    # the most experts the library takes: per-expert scale atoms at the limit, most experts short
    ("max_experts", inputs.custom(T=256, H=128, I=128, E=1024, K=8)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[n for n, _ in SMALL])
def test_mxfp8_full_parity(mok, name, w):
    d = inputs.make(w, seed=2)
    mx_gpu = _mx_inputs(mok, d)
    mx_ref = oracle.mx_weights(inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
    for k in oracle.MX_KEYS:  # the weight copies are bit-exact with the oracle's quantisation
        assert np.array_equal(mx_gpu[k].cpu().numpy(), mx_ref[k]), k
    cfg = mok.make_config(128, 256, precision=mok.MOK_MXFP8)
    out, g = _run_mx(mok, d, w, cfg, mx_gpu)
    ref = oracle.layer_mx(d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]),
                          inputs.bits(d["dY"]), mx_ref, w.E, w.I)
    errs = dict(out=rel_err(to_f64(out), ref["out"]), dX=rel_err(to_f64(g.dx), ref["dX"]),
                dWg=rel_err(to_f64(g.dw_gate), ref["dWg"]), dWu=rel_err(to_f64(g.dw_up), ref["dWu"]),
                dWd=rel_err(to_f64(g.dw_down), ref["dWd"]), dS=rel_err(to_f64(g.d_topk_weights), ref["dS"]))
    bad = {k: v for k, v in errs.items() if not v <= TOL_MX}
    assert not bad, errs


def test_mxfp8_ep64_shard_sampled_parity_and_determinism(mok):
    """The per-GPU shard of an EP64 layer: 16,384 routed rows onto 4 experts (Zipf 1.2),
    H=7168, I=2048, top-1: sampled parity (256 rows, dW blocks of the heaviest and the lightest
    expert and of each tensor's peak), ten bitwise-identical repeats, other grids."""
    w = inputs.WORKLOADS["mxfp8_ep64_shard"]
    d = inputs.make(w, seed=0)
    mx_gpu = _mx_inputs(mok, d)
    mx_ref = oracle.mx_weights(inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
    for k in oracle.MX_KEYS:  # the weight copies the GPU reads are the oracle's bytes
        assert np.array_equal(mx_gpu[k].cpu().numpy(), mx_ref[k]), k
    cfg = mok.make_config(512, 2048, precision=mok.MOK_MXFP8)
    r = fullsize.run_layer(mok, w, d, cfg, mx_gpu=mx_gpu, repeats=10)
    errs = fullsize.mx_sampled_errors(d, w, r)
    bad = {k: v for k, v in errs.items() if not v <= TOL_MX}
    assert not bad, errs
    for k, v in r.items():
        assert torch.isfinite(v).all(), k
    # bitwise identical on another grid and minibatch size, and with static tile scheduling
    for cfg in (mok.make_config(256, 512, 37, precision=mok.MOK_MXFP8),
                mok.make_config(512, 2048, 37, precision=mok.MOK_MXFP8, flags=mok.MOK_FLAG_STATIC_TILES)):
        r2 = fullsize.run_layer(mok, w, d, cfg, mx_gpu=mx_gpu)
        for k, v in r2.items():
            assert torch.equal(v, r[k]), k


def _untile_scales(atoms, rows, kg):
    """Row-major [rows, kg] scale bytes from an atom-tiled array (the layout mok.h documents for
    mok_mx_operands_of's row-major copies)."""
    kq = kg // 4
    r = np.arange(rows)[:, None]
    g = np.arange(kg)[None, :]
    off = ((r // 128) * kq + g // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + g % 4
    return atoms[off]


def _untile_scales_t(atoms, nf, rcap, groups):
    """[nf, rcap / 32] scale bytes of a copy quantised along the rows (column f, row block g; atoms
    grouped `groups` at a time), from the layout mok.h documents."""
    kq = rcap // 128
    f = np.arange(nf)[:, None]
    g = np.arange(rcap // 32)[None, :]
    off = (((f // (128 * groups)) * kq + g // 4) * groups + (f // 128) % groups) * 512 + (f % 32) * 16 \
        + ((f // 32) % 4) * 4 + g % 4
    return atoms[off]


def _padded_rows(bits_tc, row_token, rpad):
    """bf16 bit patterns of the expert-grouped padded layout (zero rows for padding)."""
    rt = row_token[:rpad]
    out = np.zeros((rpad, bits_tc.shape[1]), np.uint16)
    out[rt >= 0] = bits_tc[rt[rt >= 0]]
    return out


def _rows_quantised(bits_pad):
    """Oracle bytes of the quantisation along rows (32-row blocks), column-major: codes [n, rpad],
    scales [n, rpad / 32]."""
    rpad, n = bits_pad.shape
    q = np.zeros((n, rpad), np.uint8)
    sc = np.zeros((n, rpad // 32), np.uint8)
    for b in range(rpad // 32):
        qb, sb = oracle.mxfp8_quantize(np.ascontiguousarray(bits_pad[32 * b:32 * b + 32].T))
        q[:, 32 * b:32 * b + 32] = qb
        sc[:, b] = sb[:, 0]
    return q, sc


def _ctx_a(layer, w):
    """bf16 view of the forward context's a (MXFP8 context: xr | its scales | g,u fp32 | a)."""
    up = lambda n: (n + 255) // 256 * 256  # noqa: E731
    rows = layer.sched.c.rpad_max
    rcap = (rows + 127) // 128 * 128
    off = up(w.H * rcap) + up(w.H * rcap // 32) + up(rows * 2 * w.I * 4)
    return layer.ctx.view(torch.uint8)[off:off + rows * w.I * 2].view(torch.bfloat16).view(rows, w.I)


def test_mxfp8_gather_quantises_x_bit_exactly(mok):
    """The quantising gather of x equals the oracle's MX quantisation bit for bit, along H (the
    row-major codes and scales) and along the 32-row blocks of the padded layout (the
    codes and scales the weight gradient reads)."""
    w = inputs.custom(T=200, H=512, I=128, E=4, K=2)
    d = inputs.make(w, seed=4)
    x = d["x"].clone()
    x[3] = x[3] * 1e-30  # tiny block exponents
    x[4] = x[4] * 1e30   # large ones
    x[5, :64] = 0        # zero blocks
    # bit patterns: every finite class at random (subnormals, both signs, every exponent); blocks of
    # bf16 subnormals and tiny normals only (scaled up by 2^127); Inf and NaN blocks; blocks whose
    # small values underflow after scaling and must keep their sign (E4M3 -0 is 0x80)
    rng = np.random.default_rng(11)
    xb = x.view(torch.int16).numpy()
    pat = rng.integers(0, 1 << 16, size=w.H, dtype=np.uint32)
    pat = np.where((pat & 0x7F80) == 0x7F80, pat & 0xBFFF, pat)
    xb[6] = pat.astype(np.uint16).view(np.int16)
    tiny = (rng.integers(0, 3, size=w.H) << 7) | rng.integers(0, 128, size=w.H) | (rng.integers(0, 2, size=w.H) << 15)
    xb[7] = tiny.astype(np.uint16).view(np.int16)
    row8 = np.full(w.H, 0x3F80, np.uint16)
    row8[5], row8[40], row8[70], row8[100] = 0x7F80, 0x7FC1, 0xFF80, 0xFFFF  # +Inf, NaN, -Inf, -NaN
    xb[8] = row8.view(np.int16)
    row9 = np.full(w.H, 0x8001, np.uint16)  # -(smallest subnormal)
    row9[::32] = 0x7100                      # about 6.3e29: the block's maximum
    row9[1::32] = 0xB000                     # -4.7e-10
    xb[9] = row9.view(np.int16)
    d["x"] = x
    mx_gpu = _mx_inputs(mok, d)
    cfg = mok.make_config(128, 256, precision=mok.MOK_MXFP8)
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    layer.schedule(d["topk_ids"].cuda(), d["topk_weights"].cuda())
    layer.forward(x.cuda(), mok.weights_struct(mx=mx_gpu))
    torch.cuda.synchronize()
    t = layer.sched.tables()
    inv = t["inv"].cpu().numpy().astype(np.int64)
    rpad = int(t["meta"][0])
    row_token = t["row_token"].cpu().numpy()
    q_ref, s_ref = oracle.mxfp8_quantize(inputs.bits(x))
    ops = layer.sched.mx_operands(layer.ctx)
    xq = ops["xq"].cpu().numpy()
    xs = _untile_scales(ops["xs"].cpu().numpy(), xq.shape[0], w.H // 32)
    tok = np.arange(w.R) // w.K
    assert np.array_equal(xq[inv], q_ref.reshape(w.T, w.H)[tok])
    assert np.array_equal(xs[inv], s_ref.reshape(w.T, w.H // 32)[tok])
    pad = row_token[:rpad] < 0
    assert pad.any()
    assert not xq[:rpad][pad].any() and not xs[:rpad][pad].any()
    qt_ref, st_ref = _rows_quantised(_padded_rows(inputs.bits(x), row_token, rpad))
    xr = ops["xr"].cpu().numpy()
    xrs = _untile_scales_t(ops["xrs"].cpu().numpy(), w.H, ops["rcap"], ops["xr_groups"])
    assert np.array_equal(xr[:, :rpad], qt_ref)
    assert np.array_equal(xrs[:, :rpad // 32], st_ref)


@pytest.mark.parametrize("name,w", SMALL[1:], ids=[n for n, _ in SMALL[1:]])
def test_mxfp8_operand_copies(mok, name, w):
    """The E4M3 copies the block-scaled GEMMs read:
      * aq (gate/up epilogue) decodes exactly to the context's bf16 a;
      * dY quantised along H and along the routed rows equals the oracle's quantisation bit for bit;
      * dg, du and s*a quantised along the routed rows (dgrad1 epilogue, from fp32 values) match the
        oracle's quantisation of its fp64 values to within one E4M3 step at the block's scale (fp32
        and fp64 may round a value near a code boundary to neighbouring codes)."""
    d = inputs.make(w, seed=7)
    mx_gpu = _mx_inputs(mok, d)
    cfg = mok.make_config(128, 256, precision=mok.MOK_MXFP8)
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    weights = mok.weights_struct(mx=mx_gpu)
    layer.schedule(d["topk_ids"].cuda(), d["topk_weights"].cuda())
    layer.forward(d["x"].cuda(), weights)
    layer.backward(d["dY"].cuda(), weights)
    torch.cuda.synchronize()
    t = layer.sched.tables()
    rpad = int(t["meta"][0])
    row_token = t["row_token"].cpu().numpy()
    perm = t["perm"].cpu().numpy()
    ops = {k: (v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in layer.sched.mx_operands(layer.ctx).items()}
    rows, rcap = ops["rows"], ops["rcap"]
    a_dec = oracle.mxfp8_dequantize(ops["aq"], _untile_scales(ops["as_"], rows, w.I // 32)).reshape(rows, w.I)
    assert np.array_equal(a_dec[:rpad], to_f64(_ctx_a(layer, w)[:rpad]))
    # dY, both axes, bit-exact
    q_ref, s_ref = oracle.mxfp8_quantize(inputs.bits(d["dY"]))
    inv = t["inv"].cpu().numpy().astype(np.int64)
    tok = np.arange(w.R) // w.K
    assert np.array_equal(ops["dyq"][inv], q_ref.reshape(w.T, w.H)[tok])
    assert np.array_equal(_untile_scales(ops["dys"], rows, w.H // 32)[inv], s_ref.reshape(w.T, w.H // 32)[tok])
    qt_ref, st_ref = _rows_quantised(_padded_rows(inputs.bits(d["dY"]), row_token, rpad))
    assert np.array_equal(ops["dyr"][:, :rpad], qt_ref)
    assert np.array_equal(_untile_scales_t(ops["dyrs"], w.H, rcap, 1)[:, :rpad // 32], st_ref)
    # dg, du, s*a along the rows: within one E4M3 step of the oracle's values at the block scale
    mx_ref = oracle.mx_weights(inputs.bits(d["Wg"]), inputs.bits(d["Wu"]), inputs.bits(d["Wd"]))
    ref = oracle.layer_mx(d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]),
                          inputs.bits(d["dY"]), mx_ref, w.E, w.I, with_dg=True)
    sflat = d["topk_weights"].numpy().reshape(-1).astype(np.float64)
    valid = perm[:rpad] >= 0
    slots = perm[:rpad][valid]
    for name_, codes, scales, groups, src in (
            ("dg", ops["dgr"][:w.I], _untile_scales_t(ops["dgrs"], 2 * w.I, rcap, 1)[:w.I], 1, ref["dg"]),
            ("du", ops["dgr"][w.I:], _untile_scales_t(ops["dgrs"], 2 * w.I, rcap, 1)[w.I:], 1, ref["du"]),
            ("sa", ops["sar"], _untile_scales_t(ops["sars"], w.I, rcap, ops["sar_groups"]), ops["sar_groups"],
             sflat[:, None] * ref["a"])):
        dec = oracle.mxfp8_dequantize(np.ascontiguousarray(codes[:, :rpad]),
                                      np.ascontiguousarray(scales[:, :rpad // 32]))  # [features, rpad]
        exact = np.zeros((rpad, src.shape[1]))
        exact[valid] = src[slots]
        refq = oracle.mx_fakequant(np.ascontiguousarray(exact.T))  # along the rows, blocks of 32
        blk = np.abs(exact.T).reshape(src.shape[1], rpad // 32, 32).max(axis=2)
        _, ex = np.frexp(np.where(blk > 0, blk, 1.0))
        step = np.repeat(2.0 ** (ex - 1 - 3), 32, axis=1)  # one E4M3 step in the block's top binade
        err = np.abs(dec - refq)
        assert np.all(err <= step * (1 + 1e-6) + 1e-30), (name_, float((err / step).max()))
        assert not dec[:, ~valid].any(), name_
@pytest.mark.parametrize("name", ["sweep_zipf0_mx", "sweep_zipf1_mx", "sweep_zipf2_mx"])
def test_mxfp8_sweep_sampled_parity_and_determinism(mok, name):
    """T=8192, H=4096, I=1536, E=128, top-8, Zipf-skewed routing, MXFP8: sampled parity and ten
    bitwise-identical repeats.  On the skewed sweeps the sampled tokens are drawn among those routed
    only to the 32 heaviest experts, so the oracle quantises about 35 experts' weights instead of
    128; the dW blocks still cover the lightest expert.  The uniform sweep (s = 0) has no such
    tokens and samples from all of them."""
    w = inputs.WORKLOADS[name]
    d = inputs.make(w, seed=0, weight_device="cuda")
    mx_gpu = _mx_inputs(mok, d)
    r = fullsize.run_layer(mok, w, d, mok.make_config(512, 2048, precision=mok.MOK_MXFP8), mx_gpu=mx_gpu,
                           repeats=10)
    pool = fullsize.tokens_within_heaviest(d, w, 32)
    errs = fullsize.mx_sampled_errors(d, w, r, seed=1, token_pool=pool if pool.size >= 64 else None)
    bad = {k: v for k, v in errs.items() if not v <= TOL_MX}
    assert not bad, errs
    del r, mx_gpu
    torch.cuda.empty_cache()


def test_mxfp8_unused_experts_and_single_row(mok):
    """Experts without rows get exact zero weight gradients (their E4M3 GEMM tiles have no K), and a
    layer with one routed row still matches the oracle (one 32-row block: 1 real row, 31 padding)."""
    w = inputs.custom(T=50, H=256, I=128, E=7, K=2)
    d = inputs.make(w, seed=2)
    ids = d["topk_ids"]
    ids[ids == 3] = 4
    ids[ids == 6] = 0
    d["topk_ids"] = ids
    mx_gpu = _mx_inputs(mok, d)
    out, g = _run_mx(mok, d, w, mok.make_config(128, 256, precision=mok.MOK_MXFP8), mx_gpu)
    for e in (3, 6):
        assert not g.dw_gate[e].any() and not g.dw_up[e].any() and not g.dw_down[e].any()
    assert torch.isfinite(out).all() and torch.isfinite(g.dx).all()
    w1 = inputs.custom(T=1, H=128, I=128, E=3, K=1)
    d1 = inputs.make(w1, seed=3)
    mx1 = _mx_inputs(mok, d1)
    out1, g1 = _run_mx(mok, d1, w1, mok.make_config(128, 128, precision=mok.MOK_MXFP8), mx1)
    mx_ref = oracle.mx_weights(inputs.bits(d1["Wg"]), inputs.bits(d1["Wu"]), inputs.bits(d1["Wd"]))
    ref = oracle.layer_mx(d1["topk_ids"].numpy(), d1["topk_weights"].numpy(), inputs.bits(d1["x"]),
                          inputs.bits(d1["dY"]), mx_ref, w1.E, w1.I)
    errs = dict(out=rel_err(to_f64(out1), ref["out"]), dX=rel_err(to_f64(g1.dx), ref["dX"]),
                dWg=rel_err(to_f64(g1.dw_gate), ref["dWg"]), dWd=rel_err(to_f64(g1.dw_down), ref["dWd"]),
                dS=rel_err(to_f64(g1.d_topk_weights), ref["dS"]))
    assert all(v <= TOL_MX for v in errs.values()), errs


def test_mxfp8_empty_batch(mok):
    w = inputs.custom(T=0, H=128, I=128, E=4, K=2)
    d = inputs.make(w, seed=0)
    mx_gpu = _mx_inputs(mok, d)
    out, g = _run_mx(mok, d, w, mok.make_config(128, 128, precision=mok.MOK_MXFP8), mx_gpu)
    assert out.numel() == 0
    assert not g.dw_gate.any() and not g.dw_up.any() and not g.dw_down.any()
