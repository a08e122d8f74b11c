"""Pins of the oracle's schedule (expert histogram, prefix sums, stable permutation, tiles).

The pages: one schedule table drives dispatch and combine in both passes, and no token is ever
dropped ("Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1) and (3)); the schedule is
built from the top-k expert ids ("Mixture-of-Kittens (MoK)" project card, "Functional API").
The oracle's sort is pinned against numpy's stable argsort (a library routine) and against the
invariants the definition fixes.
"""
import numpy as np
import pytest

import oracle

MT = oracle.MT


def _check_schedule(ids, E, mb, MB, sch):
    T, K = ids.shape
    R = T * K
    flat = ids.reshape(-1)
    counts, offsets, poff, perm, inv = sch["counts"], sch["offsets"], sch["poff"], sch["perm"], sch["inv"]
    # histogram and prefix sums against numpy
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert counts.sum() == R
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    padded = (counts + MT - 1) // MT * MT
    assert np.array_equal(poff, np.concatenate([[0], np.cumsum(padded)]))
    assert sch["rpad"] == poff[-1]
    # stable permutation: the valid rows in padded order equal numpy's stable argsort by expert
    order = np.argsort(flat, kind="stable")
    valid = perm[perm >= 0]
    assert np.array_equal(valid, order)
    # padding rows are -1 and sit at the end of each expert segment
    for e in range(E):
        seg = perm[poff[e]:poff[e + 1]]
        assert np.all(seg[:counts[e]] >= 0) and np.all(seg[counts[e]:] == -1)
        assert np.all(flat[seg[:counts[e]]] == e)
    # inverse
    assert np.array_equal(perm[inv], np.arange(R))
    # tiles: ascending experts, never cross an expert, mb rows each except the last of an expert
    tiles = sch["tiles"]
    assert tiles[:, 2].sum() == R
    exp_tiles = []
    for e in range(E):
        q = 0
        while q < counts[e]:
            exp_tiles.append((e, poff[e] + q, min(mb, counts[e] - q), (poff[e] + q) // MB))
            q += mb
    assert [tuple(t) for t in tiles.tolist()] == exp_tiles
    # Mt-row blocks
    mbk = sch["mblocks"]
    assert mbk.shape[0] == sch["rpad"] // MT
    for b, (e, first, v, t) in enumerate(mbk.tolist()):
        assert first == b * MT and poff[e] <= first < poff[e + 1]
        assert v == min(MT, counts[e] - (first - poff[e]))
        te, tf, tv, _ = tiles[t]
        assert te == e and tf <= first < tf + (tv + MT - 1) // MT * MT


@pytest.mark.parametrize("T,K,E,mb,MB,seed", [
    (128, 2, 8, 128, 256, 0),
    (100, 3, 5, 128, 512, 1),
    (513, 6, 64, 256, 1024, 2),
    (7, 1, 3, 128, 128, 3),
    (300, 8, 16, 512, 2048, 4),
])
def test_schedule_random(T, K, E, mb, MB, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    sch = oracle.schedule(ids, E, mb, MB)
    _check_schedule(ids, E, mb, MB, sch)


def test_schedule_skewed_with_empty_experts_and_duplicates():
    rng = np.random.default_rng(5)
    T, K, E = 400, 4, 12
    ids = np.minimum(rng.zipf(2.0, size=(T, K)) - 1, E - 1).astype(np.int32)
    ids[ids == 3] = 2           # expert 3 empty
    ids[:10, :] = 7             # a token routed to the same expert several times
    sch = oracle.schedule(ids, E, 128, 256)
    _check_schedule(ids, E, 128, 256, sch)
    assert sch["counts"][3] == 0
    assert not np.any(sch["tiles"][:, 0] == 3)


def test_schedule_worked_example():
    # hand-derived from the definition: T=3, K=2, E=3
    ids = np.array([[2, 0], [0, 2], [1, 0]], np.int32)  # slots 0..5 -> experts 2,0,0,2,1,0
    sch = oracle.schedule(ids, 3, 128, 128)
    assert sch["counts"].tolist() == [3, 1, 2]
    assert sch["offsets"].tolist() == [0, 3, 4, 6]
    assert sch["poff"].tolist() == [0, 128, 256, 384]
    assert sch["perm"][:4].tolist() == [1, 2, 5, -1]
    assert sch["perm"][128:130].tolist() == [4, -1]
    assert sch["perm"][256:259].tolist() == [0, 3, -1]
    assert sch["inv"].tolist() == [256, 0, 1, 257, 128, 2]
    assert sch["tiles"].tolist() == [[0, 0, 3, 0], [1, 128, 1, 1], [2, 256, 2, 2]]
    assert sch["mblocks"].tolist() == [[0, 0, 3, 0], [1, 128, 1, 1], [2, 256, 2, 2]]


def test_schedule_empty_batch():
    ids = np.zeros((0, 2), np.int32)
    sch = oracle.schedule(ids, 4, 128, 128)
    assert sch["rpad"] == 0 and sch["tiles"].shape[0] == 0 and sch["mblocks"].shape[0] == 0
    assert sch["counts"].tolist() == [0, 0, 0, 0]


def test_schedule_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.schedule(np.array([[0, 4]], np.int32), 4, 128, 128)
    with pytest.raises(ValueError):
        oracle.schedule(np.array([[-1, 0]], np.int32), 4, 128, 128)


def test_schedule_multi_tile_expert():
    ids = np.zeros((700, 1), np.int32)
    ids[::3] = 1
    sch = oracle.schedule(ids, 2, 256, 512)
    _check_schedule(ids, 2, 256, 512, sch)
    # expert 0 has 466 slots -> tiles of 256, 210 valid rows
    assert sch["tiles"][:2, 2].tolist() == [256, 210]
