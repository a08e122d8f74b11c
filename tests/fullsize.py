"""Sampled parity of one full-size GPU run against the oracle, at the sizes the tolerance reading
asks for where the full fp64 oracle would take too long: 256 tokens for out / dX / d_topk_weights,
and for every weight gradient at least 4,096 entries drawn as 32-column blocks of I against 64
hidden columns.  The blocks always cover the heaviest and the lightest expert with rows, a random
used expert, and the entry where each GPU weight-gradient tensor peaks, so a wrong peak cannot hide
behind the denominator.  Errors are max|gpu - oracle| / max|oracle| over the sampled entries of
each tensor.  No layer arithmetic lives here: every expected value comes from the oracle."""
import numpy as np
import torch

import oracle
from helpers import rel_err, to_f64
from mixture_experts_layer_build_gb300 import inputs

N_TOKENS = 256
N_HIDDEN = 64   # hidden columns per 32-column block: 2,048 entries per block and weight


def run_layer(mok, w, d, cfg, mx_gpu=None, repeats=1):
    """Schedule, forward and backward on the GPU; returns the outputs as GPU tensors.  With
    repeats > 1 the same layer object runs again and every output must be bitwise the same."""
    x, ids, s, dY = (d[k].cuda() for k in ("x", "topk_ids", "topk_weights", "dY"))
    layer = mok.Layer(w.T, w.H, w.I, w.E, w.K, cfg)
    weights = mok.weights_struct(mx=mx_gpu) if mx_gpu is not None else \
        mok.weights_struct(d["Wg"].cuda(), d["Wu"].cuda(), d["Wd"].cuda())
    ref = None
    for i in range(repeats):
        layer.schedule(ids, s)
        out = layer.forward(x, weights)
        g = layer.backward(dY, weights)
        torch.cuda.synchronize()
        assert mok.mok_read_device_status(layer.sched) == 0
        cur = dict(out=out, dx=g.dx, dwg=g.dw_gate, dwu=g.dw_up, dwd=g.dw_down, ds=g.d_topk_weights)
        if ref is None:
            ref = {k: v.clone() for k, v in cur.items()}
        else:
            for k, v in cur.items():
                assert torch.equal(v, ref[k]), f"repeat {i}: {k} differs"
    del layer
    return ref


def sample_plan(d, w, r, seed=0, token_pool=None):
    """Tokens and dW blocks to check: (expert, i0, hidden columns) per block."""
    rng = np.random.default_rng(seed)
    ids = d["topk_ids"].numpy()
    pool = np.arange(w.T) if token_pool is None else np.asarray(token_pool)
    tok = np.sort(rng.choice(pool, size=min(N_TOKENS, pool.size), replace=False))
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    used = np.flatnonzero(counts)
    blocks = [(int(np.argmax(counts)), None, None), (int(used[np.argmin(counts[used])]), None, None),
              (int(rng.choice(used)), None, None)]
    # the peak entries: dWg / dWu [e, i, h], dWd [e, h, i]
    for key in ("dwg", "dwu", "dwd"):
        t = r[key]
        pe, pa, pb = (int(v) for v in np.unravel_index(int(t.abs().argmax()), t.shape))
        i, h = (pa, pb) if key != "dwd" else (pb, pa)
        blocks.append((pe, 32 * (i // 32), h))
    plan = []
    for e, i0, h in blocks:
        if i0 is None:
            i0 = 32 * int(rng.integers(0, w.I // 32))
        hs = rng.choice(w.H, size=N_HIDDEN, replace=False)
        if h is not None:
            hs[0] = h
        plan.append((e, i0, np.sort(hs).astype(np.int32)))
    return tok, plan


def compare(r, tok, plan, tokens_fn, block_fn):
    """Errors per tensor: tokens_fn(tok) -> (out, dX, dS); block_fn(e, i0, hs) -> (dwg, dwu, dwd)."""
    tk = torch.from_numpy(tok).cuda()
    ro, rdx, rds = tokens_fn(tok)
    errs = dict(out=rel_err(to_f64(r["out"][tk]), ro), dX=rel_err(to_f64(r["dx"][tk]), rdx),
                dS=rel_err(to_f64(r["ds"][tk]), rds))
    got = {"dWg": [], "dWu": [], "dWd": []}
    ref = {"dWg": [], "dWu": [], "dWd": []}
    for e, i0, hs in plan:
        dwg, dwu, dwd = block_fn(e, i0, hs)
        hk = torch.from_numpy(hs.astype(np.int64)).cuda()
        got["dWg"].append(to_f64(r["dwg"][e, i0:i0 + 32][:, hk]).ravel())
        got["dWu"].append(to_f64(r["dwu"][e, i0:i0 + 32][:, hk]).ravel())
        got["dWd"].append(to_f64(r["dwd"][e][hk, i0:i0 + 32]).ravel())
        ref["dWg"].append(dwg.ravel())
        ref["dWu"].append(dwu.ravel())
        ref["dWd"].append(dwd.ravel())
    for k in got:
        g, o = np.concatenate(got[k]), np.concatenate(ref[k])
        assert g.size >= 4096, (k, g.size)
        errs[k] = rel_err(g, o)
    return errs


def bf16_sampled_errors(d, w, r, seed=0):
    args = (d["topk_ids"].numpy(), d["topk_weights"].numpy(), inputs.bits(d["x"]), inputs.bits(d["Wg"].cpu()),
            inputs.bits(d["Wu"].cpu()), inputs.bits(d["Wd"].cpu()))
    dy = inputs.bits(d["dY"])
    tok, plan = sample_plan(d, w, r, seed)

    def tokens_fn(t):
        out = oracle.forward_tokens(*args, t)
        dX, dS = oracle.backward_tokens(*args, dy, t)
        return out, dX, dS

    return compare(r, tok, plan, tokens_fn, lambda e, i0, hs: oracle.dw_block(*args, dy, e, i0, hs))


def mx_sampled_errors(d, w, r, seed=0, token_pool=None):
    """The oracle quantises only the experts the sampled tokens and blocks touch (the others' bytes
    are never read)."""
    ids = d["topk_ids"].numpy()
    tok, plan = sample_plan(d, w, r, seed, token_pool)
    experts = np.unique(np.concatenate([ids[tok].reshape(-1), [p[0] for p in plan]]))
    mx_ref = oracle.mx_weights(inputs.bits(d["Wg"].cpu()), inputs.bits(d["Wu"].cpu()), inputs.bits(d["Wd"].cpu()),
                               experts=experts)
    args = (ids, d["topk_weights"].numpy(), inputs.bits(d["x"]), inputs.bits(d["dY"]))
    return compare(r, tok, plan, lambda t: oracle.tokens_mx(*args, mx_ref, w.E, w.I, t),
                   lambda e, i0, hs: oracle.dw_block_mx(*args, mx_ref, w.E, w.I, e, i0, hs))


def tokens_within_heaviest(d, w, n_experts):
    """Tokens all of whose K experts are among the n_experts heaviest (bounds the experts the MXFP8
    oracle has to quantise on the 128-expert sweep)."""
    ids = d["topk_ids"].numpy()
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    heavy = np.zeros(w.E, bool)
    heavy[np.argsort(-counts, kind="stable")[:n_experts]] = True
    return np.flatnonzero(heavy[ids].all(axis=1))
