"""GPU forward / backward of the routed SwiGLU expert layer vs the fp64 oracle.

Tolerance (BF16): max|gpu - oracle| / max|oracle| <= 2e-2 per output tensor; the GPU computes
with bf16 operands, fp32 accumulation and bf16 intermediates (g, u, a, y, dg, du, dX rows), each
rounding contributing about 2^-9 relative.  Small cases compare every element; the full-size
workloads compare sampled tokens and sampled weight-gradient entries the oracle computes one by
one (``fullsize.py``: 256 tokens and at least 4,096 entries of every weight gradient).
Determinism: repeats, grid sizes and minibatch settings must agree bitwise.
"""
import numpy as np
import pytest
import torch

import fullsize
import oracle
from helpers import TOL_BF16, ctx_views, rel_err, to_f64
from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _run(mok, d, w, cfg, dev="cuda"):
    x, ids, s, dY = (d[k].to(dev) for k in ("x", "topk_ids", "topk_weights", "dY"))
    Wg, Wu, Wd = (d[k].to(dev) for k in ("Wg", "Wu", "Wd"))
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    weights = mok.weights_struct(Wg, Wu, Wd)
    layer.schedule(ids, s)
    out = layer.forward(x, weights)
    g = layer.backward(dY, weights)
    torch.cuda.synchronize()
    assert mok.mok_read_device_status(layer.sched) == 0
    return layer, out, g


def _np_args(d):
    return (d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]), inputs.bits(d["Wg"].cpu()),
            inputs.bits(d["Wu"].cpu()), inputs.bits(d["Wd"].cpu()))


SMALL = [
    ("tiny", inputs.WORKLOADS["tiny"]),
    ("ragged", inputs.custom(T=100, H=256, I=256, E=5, K=3)),
    ("multi_tile", inputs.custom(T=700, H=512, I=384, E=3, K=2)),
    ("one_expert", inputs.custom(T=64, H=128, I=128, E=1, K=1)),
    ("wide", inputs.custom(T=96, H=1024, I=512, E=6, K=2)),
    # more than 32 slots per token: the token-order gather takes its slot rows 32 at a time
    ("many_slots", inputs.custom(T=48, H=256, I=128, E=48, K=40)),
    # the most experts the library takes: about two rows each, most padding, 176 experts unused
    ("max_experts", inputs.custom(T=256, H=128, I=128, E=1024, K=8)),
]


@pytest.mark.parametrize("name,w", SMALL, ids=[n for n, _ in SMALL])
def test_forward_backward_full_parity(mok, name, w):
    d = inputs.make(w, seed=1)
    layer, out, g = _run(mok, d, w, mok.make_config(128, 256))
    args = _np_args(d)
    ref_out, it = oracle.forward(*args, intermediates=True)
    ref = oracle.backward(*args, inputs.bits(d["dY"]))
    errs = dict(out=rel_err(to_f64(out), ref_out), dX=rel_err(to_f64(g.dx), ref["dX"]),
                dWg=rel_err(to_f64(g.dw_gate), ref["dWg"]), dWu=rel_err(to_f64(g.dw_up), ref["dWu"]),
                dWd=rel_err(to_f64(g.dw_down), ref["dWd"]), dS=rel_err(to_f64(g.d_topk_weights), ref["dS"]))
    # saved activations in the forward context, row inv[j] <-> slot j
    inv = layer.sched.tables()["inv"].cpu().numpy().astype(np.int64)
    cv = ctx_views(layer.ctx, layer.sched.c.rpad_max, w.H, w.I)
    gu = to_f64(cv["gu"])[inv]
    errs["g"] = rel_err(gu[:, :w.I], it["g"])
    errs["u"] = rel_err(gu[:, w.I:], it["u"])
    errs["a"] = rel_err(to_f64(cv["a"])[inv], it["a"])
    errs["xg"] = rel_err(to_f64(cv["xg"])[inv], oracle.bf16_to_f64(args[2])[np.arange(w.R) // w.K])
    bad = {k: v for k, v in errs.items() if not v <= TOL_BF16}
    assert not bad, errs
    assert errs["xg"] == 0.0  # the gather is a copy


# CTA-pair GEMMs (minibatch tiles of 512 rows): full pairs, and tiles whose last pair has a single
# 128-row block (about 600 rows per expert: 4 + 1 blocks; about 350: 2 + 1)
PAIRED = [
    ("pairs_h256", inputs.custom(T=900, H=256, I=256, E=3, K=2)),
    ("pairs_h384", inputs.custom(T=700, H=384, I=128, E=2, K=1)),
]


@pytest.mark.parametrize("name,w", PAIRED, ids=[n for n, _ in PAIRED])
def test_cta_pair_gemms_full_parity(mok, name, w):
    d = inputs.make(w, seed=5)
    _, out, g = _run(mok, d, w, mok.make_config(512, 2048))
    args = _np_args(d)
    ref_out = oracle.forward(*args)
    ref = oracle.backward(*args, inputs.bits(d["dY"]))
    errs = dict(out=rel_err(to_f64(out), ref_out), dX=rel_err(to_f64(g.dx), ref["dX"]),
                dWg=rel_err(to_f64(g.dw_gate), ref["dWg"]), dWu=rel_err(to_f64(g.dw_up), ref["dWu"]),
                dWd=rel_err(to_f64(g.dw_down), ref["dWd"]), dS=rel_err(to_f64(g.d_topk_weights), ref["dS"]))
    bad = {k: v for k, v in errs.items() if not v <= TOL_BF16}
    assert not bad, errs
    # single-CTA tiles (minibatch 128) give the same bits
    _, out1, g1 = _run(mok, d, w, mok.make_config(128, 256))
    assert torch.equal(out1, out) and torch.equal(g1.dx, g.dx) and torch.equal(g1.d_topk_weights, g.d_topk_weights)
    assert torch.equal(g1.dw_gate, g.dw_gate) and torch.equal(g1.dw_down, g.dw_down)


def test_unused_experts_get_exact_zero_gradients(mok):
    w = inputs.custom(T=50, H=128, I=128, E=7, K=2)
    d = inputs.make(w, seed=2)
    ids = d["topk_ids"]
    ids[ids == 3] = 4
    ids[ids == 6] = 0
    d["topk_ids"] = ids
    _, _, g = _run(mok, d, w, mok.make_config(128, 128))
    for e in (3, 6):
        assert not g.dw_gate[e].any() and not g.dw_up[e].any() and not g.dw_down[e].any()


def test_empty_batch(mok):
    w = inputs.custom(T=0, H=128, I=128, E=4, K=2)
    d = inputs.make(w, seed=0)
    _, out, g = _run(mok, d, w, mok.make_config(128, 128))
    assert out.numel() == 0
    assert not g.dw_gate.any() and not g.dw_down.any()


@pytest.fixture(scope="module")
def full_size(mok):
    """The T=4096, H=2048, I=1024, E=64, top-6 BF16 workload, run once."""
    w = inputs.WORKLOADS["bf16_e64"]
    d = inputs.make(w, seed=0)
    layer, out, g = _run(mok, d, w, mok.make_config(512, 2048))
    res = dict(out=out.clone(), dx=g.dx.clone(), dwg=g.dw_gate.clone(), dwu=g.dw_up.clone(), dwd=g.dw_down.clone(),
               ds=g.d_topk_weights.clone())
    return w, d, res


def test_full_size_sampled_parity(mok, full_size):
    w, d, r = full_size
    errs = fullsize.bf16_sampled_errors(d, w, r)
    bad = {k: v for k, v in errs.items() if not v <= TOL_BF16}
    assert not bad, errs


def test_full_size_properties(full_size):
    w, d, r = full_size
    # every output finite, no expert gradient left unwritten (NaN from uninitialised memory)
    for k, v in r.items():
        assert torch.isfinite(v).all(), k


def test_determinism_repeats_grids_and_minibatches(mok, full_size):
    w, d, r = full_size
    static = mok.MOK_FLAG_STATIC_TILES  # round-robin tiles instead of cluster launch control: same bits
    cfgs = [mok.make_config(512, 2048)] * 9 + [mok.make_config(128, 256, 37), mok.make_config(2048, 4096, 1),
                                                 mok.make_config(256, 256, 300), mok.make_config(0, 0),
                                                 mok.make_config(512, 2048, 0, flags=static),
                                                 mok.make_config(128, 256, 37, flags=static),
                                                 mok.make_config(256, 512, 1, flags=static)]
    for i, cfg in enumerate(cfgs):
        layer, out, g = _run(mok, d, w, cfg)
        if cfg.minibatch_rows == 0:  # automatic granularity: 384 rows per expert -> 512, 2048
            assert (layer.sched.c.config.minibatch_rows, layer.sched.c.config.macrobatch_rows) == (512, 2048)
        for k, v in dict(out=out, dx=g.dx, dwg=g.dw_gate, dwu=g.dw_up, dwd=g.dw_down, ds=g.d_topk_weights).items():
            assert torch.equal(v, r[k]), (i, k)


@pytest.mark.parametrize("name", ["dsv3_e256", "sweep_zipf0", "sweep_zipf1", "sweep_zipf2"])
def test_workload_sampled_parity_and_determinism(mok, name):
    """Full-size workloads (the DeepSeek-V3-style layer with 256 resident experts; the T=8192,
    E=128, top-8 sweep at Zipf s = 0, 1, 2): sampled parity, ten bitwise-identical repeats, and the
    same bits on other grids and at every minibatch size of the granularity sweep."""
    w = inputs.WORKLOADS[name]
    d = inputs.make(w, seed=0, weight_device="cuda")
    r = fullsize.run_layer(mok, w, d, mok.make_config(512, 2048), repeats=10)
    errs = fullsize.bf16_sampled_errors(d, w, r)
    bad = {k: v for k, v in errs.items() if not v <= TOL_BF16}
    assert not bad, errs
    # other grids and every minibatch size of the granularity sweep (128 .. 2048 rows) must give
    # the same bits
    cfgs = [mok.make_config(128, 1024, 61), mok.make_config(512, 2048, 61, flags=mok.MOK_FLAG_STATIC_TILES)]
    if name.startswith("sweep"):
        cfgs += [mok.make_config(mb, 2 * mb) for mb in (256, 1024, 2048)]
    for cfg in cfgs:
        r2 = fullsize.run_layer(mok, w, d, cfg)
        for k, v in r2.items():
            assert torch.equal(v, r[k]), (cfg.minibatch_rows, k)
        del r2
    del r, d
    torch.cuda.empty_cache()
