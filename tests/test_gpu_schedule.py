"""GPU schedule vs the oracle, bit-exact (counts, offsets, padded offsets, permutation, inverse,
minibatch tiles, 128-row blocks, per-row token and weight).  Cases span the workloads' routing
shapes, ragged sizes, empty experts, duplicated experts per token and invalid ids."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _gpu_schedule(mok, ids_np, w_np, E, H=128, I=128, mb=128, MB=256):
    T, K = ids_np.shape
    cfg = mok.make_config(mb, MB)
    shp = mok.make_shape(T, H, I, E, K)
    ws = mok.alloc_workspace(cfg, shp)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    s = mok.mok_build_schedule(cfg, shp, ids, w, ws)
    st = mok.mok_read_device_status(s)
    return {k: v.cpu().numpy() for k, v in s.tables().items()}, st


def _compare(ids, w, E, mb, MB, g):
    ref = oracle.schedule(ids, E, mb, MB)
    rp = ref["rpad"]
    assert g["meta"][0] == rp and g["meta"][1] == ref["tiles"].shape[0] and g["meta"][2] == rp // 128
    # block pairs of the CTA-pair GEMMs: per tile, its 128-row blocks two at a time
    blocks = (ref["tiles"][:, 2] + 127) // 128
    assert g["meta"][3] == int(((blocks + 1) // 2).sum())
    assert np.array_equal(g["counts"], ref["counts"])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["poff"], ref["poff"])
    assert np.array_equal(g["perm"][:rp], ref["perm"])
    assert np.array_equal(g["inv"], ref["inv"])
    assert np.array_equal(g["tiles"][:ref["tiles"].shape[0]], ref["tiles"])
    assert np.array_equal(g["mblocks"][:rp // 128], ref["mblocks"])
    K = ids.shape[1]
    perm = ref["perm"]
    tok = np.where(perm >= 0, perm // K, -1)
    assert np.array_equal(g["row_token"][:rp], tok)
    wt = np.where(perm >= 0, w.reshape(-1)[np.maximum(perm, 0)], 0).astype(np.float32)
    assert np.array_equal(g["row_weight"][:rp].view(np.uint32), wt.view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "bf16_e64", "dsv3_e256", "mxfp8_ep64_shard", "sweep_zipf0",
                                  "sweep_zipf1", "sweep_zipf2"])
@pytest.mark.parametrize("mb,MB", [(128, 256), (512, 2048), (2048, 4096)])
def test_schedule_bit_exact_on_workload_routing(mok, name, mb, MB):
    w = inputs.WORKLOADS[name]
    d = inputs.make(inputs.custom(w.T, 128, 128, w.E, w.K, w.router, w.zipf), seed=0, with_dy=False)
    ids, s = d["topk_ids"].numpy(), d["topk_weights"].numpy()
    g, st = _gpu_schedule(mok, ids, s, w.E, mb=mb, MB=MB)
    assert st == 0
    _compare(ids, s, w.E, mb, MB, g)


@pytest.mark.parametrize("T,K,E,seed", [(1, 1, 1, 0), (7, 3, 5, 1), (1000, 2, 3, 2), (513, 6, 64, 3),
                                        (4096, 8, 1024, 4), (300, 4, 17, 5)])
def test_schedule_ragged_and_skewed(mok, T, K, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.minimum(rng.zipf(1.5, size=(T, K)) - 1, E - 1).astype(np.int32)
    if E > 3:
        ids[ids == 2] = 1          # an empty expert
    ids[0, :] = ids[0, 0]          # duplicated expert inside one token
    w = rng.random((T, K)).astype(np.float32)
    g, st = _gpu_schedule(mok, ids, w, E, mb=256, MB=512)
    assert st == 0
    _compare(ids, w, E, 256, 512, g)


def test_schedule_empty_batch(mok):
    ids = np.zeros((0, 2), np.int32)
    g, st = _gpu_schedule(mok, ids, np.zeros((0, 2), np.float32), 4)
    assert st == 0 and g["meta"][0] == 0 and g["meta"][2] == 0
    assert g["counts"].tolist() == [0, 0, 0, 0]


def test_schedule_flags_bad_ids_and_drops_nothing_valid(mok):
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 6, size=(200, 2)).astype(np.int32)
    ids[5, 1] = 6
    ids[17, 0] = -3
    w = rng.random((200, 2)).astype(np.float32)
    g, st = _gpu_schedule(mok, ids, w, 6)
    assert st & (1 << mok.MOK_ERR_BAD_EXPERT_ID)
    good = ids.copy()
    valid = (good >= 0) & (good < 6)
    assert g["counts"].sum() == valid.sum()
    assert g["inv"][5 * 2 + 1] == -1 and g["inv"][17 * 2] == -1
    # every valid slot sits in exactly one row of its expert
    perm = g["perm"][:g["meta"][0]]
    placed = np.sort(perm[perm >= 0])
    assert np.array_equal(placed, np.flatnonzero(valid.reshape(-1)))


def test_schedule_repeat_bitwise(mok):
    w = inputs.WORKLOADS["sweep_zipf2"]
    d = inputs.make(inputs.custom(w.T, 128, 128, w.E, w.K, w.router, w.zipf), seed=1, with_dy=False)
    ids, s = d["topk_ids"].numpy(), d["topk_weights"].numpy()
    first, _ = _gpu_schedule(mok, ids, s, w.E)
    for _ in range(3):
        again, _ = _gpu_schedule(mok, ids, s, w.E)
        for k in first:
            if k in ("perm", "row_token", "row_weight"):
                n = first["meta"][0]
                assert np.array_equal(first[k][:n], again[k][:n]), k
            elif k not in ("tiles", "mblocks"):
                assert np.array_equal(first[k], again[k]), k


def test_schedule_large_batch(mok):
    # 320,000 slots: 625 chunks, so the scan's 32 chunk groups hold up to 20 chunks each
    rng = np.random.default_rng(11)
    T, K, E = 40000, 8, 96
    ids = np.minimum(rng.zipf(1.3, size=(T, K)) - 1, E - 1).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    g, st = _gpu_schedule(mok, ids, w, E, mb=512, MB=2048)
    assert st == 0
    _compare(ids, w, E, 512, 2048, g)
