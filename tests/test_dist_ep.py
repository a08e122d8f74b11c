"""The host side of an expert-parallel group on the CPU: two gloo ranks (world size 2, 127.0.0.1).

Each rank holds its shard of a workload's tokens and routing.  The partition, the all-gather of the
routing ids every rank's schedule needs, the dispatch counts and the per-rank buffer sizes must
agree across ranks and with the whole-group schedule of the oracle (its per-expert counts)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from mixture_experts_layer_build_gb300 import ep, inputs, mok
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = inputs.WORKLOADS["bf16_e64"]
    d = inputs.make(inputs.custom(w.T, 128, 128, w.E, w.K, w.router), seed=0, with_dy=False)
    part = ep.partition(w.T, w.E, world, rank)
    ids_local = d["topk_ids"][part.tokens.start:part.tokens.stop].contiguous()
    ids_group = ep.exchange_routing(ids_local)
    counts = ep.dispatch_counts(ids_group.numpy(), part)
    cfg = mok.make_config(512, 2048)
    sizes = ep.buffer_bytes(mok, cfg, mok.make_shape(w.T, w.H, w.I, w.E, w.K), part)
    np.save(os.path.join(out_dir, f"ids{rank}.npy"), ids_group.numpy())
    np.save(os.path.join(out_dir, f"counts{rank}.npy"), counts)
    with open(os.path.join(out_dir, f"sizes{rank}.txt"), "w") as f:
        f.write(" ".join(str(sizes[k]) for k in ("workspace", "fwd_ctx", "y_recv", "dx_recv")))
    # the gathered routing is the whole group's, on every rank
    gathered = [torch.empty_like(ids_group) for _ in range(world)]
    dist.all_gather(gathered, ids_group)
    assert all(torch.equal(g, ids_group) for g in gathered)
    dist.destroy_process_group()


@pytest.mark.timeout(240)
def test_two_gloo_ranks_agree_on_the_group_plan(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    from mixture_experts_layer_build_gb300 import ep, inputs
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    w = inputs.WORKLOADS["bf16_e64"]
    d = inputs.make(inputs.custom(w.T, 128, 128, w.E, w.K, w.router), seed=0, with_dy=False)
    ids = d["topk_ids"].numpy()
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"ids{r}.npy"), ids)
    counts = [np.load(tmp_path / f"counts{r}.npy") for r in range(world)]
    assert np.array_equal(counts[0], counts[1])
    # rows each rank's experts receive = the oracle schedule's counts of its experts; rows each
    # rank's tokens send = its slots
    sch = oracle.schedule(ids, w.E, 512, 2048)
    El = w.E // world
    for r in range(world):
        assert counts[0][:, r].sum() == sch["counts"][r * El:(r + 1) * El].sum()
        assert counts[0][r].sum() == (w.T // world) * w.K
    sizes = [open(tmp_path / f"sizes{r}.txt").read().split() for r in range(world)]
    assert sizes[0] == sizes[1] and all(int(v) > 0 for v in sizes[0])
    assert int(sizes[0][2]) == (w.T // world) * w.K * w.H * 2


def test_partition_rejects_uneven_groups():
    sys.path.insert(0, ROOT)
    from mixture_experts_layer_build_gb300 import ep
    p = ep.partition(4096, 64, 4, 3)
    assert (p.tokens_per_rank, p.experts_per_rank, p.tokens, p.experts) == (1024, 16, range(3072, 4096), range(48, 64))
    for args in ((4096, 63, 4, 0), (4095, 64, 4, 0), (4096, 64, 9, 0), (4096, 64, 2, 2)):
        with pytest.raises(ValueError):
            ep.partition(*args)
    # invalid ids count nowhere in the dispatch plan
    c = ep.dispatch_counts(np.array([[0, 5], [7, -1], [3, 8], [1, 2]]), ep.partition(4, 8, 2, 0))
    assert c.tolist() == [[1, 2], [3, 0]]
