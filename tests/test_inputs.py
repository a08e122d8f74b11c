"""The seeded input recipe, on the CPU: draws are reproducible, routing is valid (K distinct experts
in [0, E) per token, weights as the router defines them), and the Zipf-skewed routers skew as the
sweep workloads rely on (max/mean load growing with the exponent; at exponent 2 expert 0 is in
every token's top-8, i.e. it receives 1/8 of the rows; the top-1 shard's loads fall with the
expert's rank)."""
import pytest
import torch

from mixture_experts_layer_build_gb300 import inputs


def _small(router, zipf=0.0, E=128, K=8, T=2048):
    return inputs.custom(T=T, H=128, I=128, E=E, K=K, router=router, zipf=zipf)


@pytest.mark.parametrize("router", ["softmax", "softmax_bias", "gumbel_max", "gumbel_topk"])
def test_draws_are_reproducible_and_routing_is_valid(router):
    K = 1 if router == "gumbel_max" else 4
    w = _small(router, zipf=1.0, E=16, K=K, T=300)
    a, b, c = inputs.make(w, seed=5), inputs.make(w, seed=5), inputs.make(w, seed=6)
    for k in ("x", "topk_ids", "topk_weights", "Wg", "Wu", "Wd", "dY"):
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["x"], c["x"])
    ids, wts = a["topk_ids"], a["topk_weights"]
    assert ids.dtype == torch.int32 and ids.shape == (w.T, K)
    assert int(ids.min()) >= 0 and int(ids.max()) < w.E
    assert all(len(set(r)) == K for r in ids.tolist())  # K distinct experts per token
    if router == "gumbel_max":
        assert float(wts.min()) >= 0.05 and float(wts.max()) <= 0.30
    else:
        assert torch.allclose(wts.sum(dim=1), torch.ones(w.T), atol=1e-6)
        assert bool((wts[:, :-1] >= wts[:, 1:]).all())  # descending, as the experts were chosen


def test_zipf_skew_of_the_sweep_routers():
    ratios = []
    for z in (0.0, 1.0, 2.0):
        ids = inputs.make(_small("gumbel_topk", zipf=z), seed=0)["topk_ids"]
        ratios.append(inputs.load_stats(ids, 128)["max_over_mean"])
        if z == 2.0:
            assert bool((ids == 0).any(dim=1).all())  # expert 0 in every token's top-8
    assert ratios[0] < 1.5 < ratios[1] < ratios[2] == pytest.approx(16.0)


def test_top1_shard_loads_fall_with_the_expert_rank():
    ids = inputs.make(_small("gumbel_max", zipf=1.2, E=4, K=1), seed=0)["topk_ids"]
    counts = torch.bincount(ids.reshape(-1).long(), minlength=4).tolist()
    assert counts == sorted(counts, reverse=True) and counts[0] > 2 * counts[-1]
