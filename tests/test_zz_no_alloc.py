"""mok_build_schedule_noalloc: the schedule build for callers that may not allocate device memory
while they run (a runtime that hands out only fixed, pre-sized buffers, or a hook in which
cudaMalloc is forbidden).  Its scratch lives in a fixed array inside the library, shared by every
call.

Called through the C ABI, its tables must equal, bit for bit (the schedule is integer work, so the
tolerance is zero), both the oracle's schedule and those of mok_build_schedule, on two calls in a
row with different routing, so a stale scratch array would show.  Cases: the empty batch, a shape at
the scratch limit, automatic minibatch sizes with buffers sized from the documented bound, an
MXFP8 config, and out-of-range expert ids.  This file is collected last."""
import ctypes

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


def _caps(T, K, E, mb):
    """Buffer capacities of a shape: mb = 0 (automatic) is sized from the documented bound (the
    resolved minibatch is at least 256 rows)."""
    R = T * K
    rpad_max = R + 127 * E
    tiles_max = -(-R // (mb if mb else 256)) + E
    return rpad_max, tiles_max, rpad_max // 128


def _noalloc(mok, cfg, shp, ids, w, caps=None):
    T, K, E = shp.T, shp.K, shp.E
    R = T * K
    rpad_max, tiles_max, mblocks_max = caps or _caps(T, K, E, cfg.minibatch_rows)
    dev = ids.device
    bufs = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                poff=torch.empty(E + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(rpad_max, dtype=torch.int32, device=dev),
                inv=torch.empty(max(R, 1), dtype=torch.int32, device=dev),
                tiles=torch.empty((max(tiles_max, 1), 4), dtype=torch.int32, device=dev),
                mblocks=torch.empty((max(mblocks_max, 1), 4), dtype=torch.int32, device=dev),
                meta=torch.empty(16, dtype=torch.int32, device=dev),
                row_weight=torch.empty(rpad_max, dtype=torch.float32, device=dev),
                row_token=torch.empty(rpad_max, dtype=torch.int32, device=dev))
    s = mok.mok_schedule()
    for k, v in bufs.items():
        setattr(s, k, v.data_ptr())
    s.rpad_max, s.tiles_max, s.mblocks_max = rpad_max, tiles_max, mblocks_max
    rc = mok._lib.mok_build_schedule_noalloc(ctypes.byref(cfg), ctypes.byref(shp), ids.data_ptr(), w.data_ptr(),
                                             ctypes.byref(s), torch.cuda.current_stream().cuda_stream)
    assert rc == mok.MOK_OK, rc
    torch.cuda.synchronize()
    assert s.rpad_max == R + 127 * E and s.tiles_max <= tiles_max and s.mblocks_max == (R + 127 * E) // 128
    return {k: v.cpu().numpy() for k, v in bufs.items()}, s


def _workspace_schedule(mok, cfg, shp, ids, w):
    ws = mok.alloc_workspace(cfg, shp)
    sch = mok.mok_build_schedule(cfg, shp, ids, w, ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in sch.tables().items()}, sch


def _same(a, b, status_bits=0):
    rp = int(b["meta"][0])
    assert int(a["meta"][0]) == rp and np.array_equal(a["meta"][:3], b["meta"][:3])
    assert a["meta"][15] == b["meta"][15] == status_bits
    for k in ("counts", "offsets", "poff"):
        assert np.array_equal(a[k], b[k]), k
    R = b["inv"].size  # the noalloc buffer holds at least one entry
    assert np.array_equal(a["inv"][:R], b["inv"]), "inv"
    for k in ("perm", "row_token"):
        assert np.array_equal(a[k][:rp], b[k][:rp]), k
    assert np.array_equal(a["row_weight"][:rp].view(np.uint32), b["row_weight"][:rp].view(np.uint32))
    nt = int(b["meta"][1])
    assert np.array_equal(a["tiles"][:nt], b["tiles"][:nt])
    assert np.array_equal(a["mblocks"][:rp // 128], b["mblocks"][:rp // 128])


def _same_as_oracle(a, ids, w, E, mb, MB):
    ref = oracle.schedule(ids, E, mb, MB)
    rp = ref["rpad"]
    assert int(a["meta"][0]) == rp and int(a["meta"][1]) == ref["tiles"].shape[0] and int(a["meta"][2]) == rp // 128
    for k in ("counts", "offsets", "poff"):
        assert np.array_equal(a[k], ref[k]), k
    assert np.array_equal(a["perm"][:rp], ref["perm"])
    assert np.array_equal(a["inv"][:ids.size], ref["inv"])
    assert np.array_equal(a["tiles"][:ref["tiles"].shape[0]], ref["tiles"])
    assert np.array_equal(a["mblocks"][:rp // 128], ref["mblocks"])
    K = ids.shape[1]
    perm = ref["perm"]
    assert np.array_equal(a["row_token"][:rp], np.where(perm >= 0, perm // K, -1))
    wt = np.where(perm >= 0, w.reshape(-1)[np.maximum(perm, 0)], 0).astype(np.float32)
    assert np.array_equal(a["row_weight"][:rp].view(np.uint32), wt.view(np.uint32))


def _routing(T, E, K, name, seed):
    wl = inputs.WORKLOADS[name]
    d = inputs.make(inputs.custom(T, 128, 128, E, K, wl.router, wl.zipf), seed=seed, with_dy=False)
    return d["topk_ids"], d["topk_weights"]


CASES = [
    # (label, T, E, K, routing of, minibatch, macrobatch, precision)
    ("sweep_zipf2", 8192, 128, 8, "sweep_zipf2", 512, 2048, "bf16"),
    ("bf16_e64", 4096, 64, 6, "bf16_e64", 512, 2048, "bf16"),
    ("empty", 0, 16, 4, "bf16_e64", 512, 2048, "bf16"),
    ("automatic", 4096, 64, 6, "bf16_e64", 0, 0, "bf16"),
    ("mxfp8", 16384, 4, 1, "mxfp8_ep64_shard", 512, 2048, "mxfp8"),
    # 512 chunks of 512 slots x (1023 + 1) experts: exactly the 524,288 entries of the scratch
    ("at_limit", 32768, 1023, 8, "sweep_zipf1", 256, 1024, "bf16"),
]


def test_noalloc_schedule_matches_oracle_and_workspace_schedule_on_consecutive_calls(mok):
    for i, (label, T, E, K, route, mb, MB, prec) in enumerate(CASES):
        ids, w = _routing(T, E, K, route, seed=i)
        cfg = mok.make_config(mb, MB, precision=mok.MOK_MXFP8 if prec == "mxfp8" else mok.MOK_BF16)
        shp = mok.make_shape(T, 128, 128, E, K)
        got, s = _noalloc(mok, cfg, shp, ids.cuda(), w.cuda())
        ref, sch = _workspace_schedule(mok, cfg, shp, ids.cuda(), w.cuda())
        _same(got, ref)
        rmb, rMB = s.config.minibatch_rows, s.config.macrobatch_rows  # resolved sizes
        assert (rmb, rMB) == (sch.c.config.minibatch_rows, sch.c.config.macrobatch_rows), label
        _same_as_oracle(got, ids.numpy(), w.numpy(), E, rmb, rMB)
        if label == "at_limit":
            assert -(-T * K // 512) * (E + 1) == 1 << 19


def test_noalloc_out_of_range_ids_match_workspace_schedule(mok):
    ids, w = _routing(600, 8, 2, "bf16_e64", seed=9)
    ids = ids.clone()
    ids[5, 1] = 8    # == E
    ids[77, 0] = -3
    cfg = mok.make_config(128, 256)
    shp = mok.make_shape(600, 128, 128, 8, 2)
    got, _ = _noalloc(mok, cfg, shp, ids.cuda(), w.cuda())
    ref, _ = _workspace_schedule(mok, cfg, shp, ids.cuda(), w.cuda())
    _same(got, ref, status_bits=1 << mok.MOK_ERR_BAD_EXPERT_ID)
    assert got["inv"][5 * 2 + 1] == -1 and got["inv"][77 * 2] == -1


def test_noalloc_rejects_sizes_beyond_its_scratch_and_small_buffers(mok):
    cfg = mok.make_config(512, 2048)
    shp = mok.make_shape(1 << 20, 128, 128, 1024, 2)  # 4096 chunks x 1025 > 524288 entries
    s = mok.mok_schedule()
    for k in ("counts", "offsets", "poff", "perm", "inv", "tiles", "mblocks", "meta", "row_weight", "row_token"):
        setattr(s, k, 256)
    s.rpad_max, s.tiles_max, s.mblocks_max = _caps(1 << 20, 2, 1024, 512)
    rc = mok._lib.mok_build_schedule_noalloc(ctypes.byref(cfg), ctypes.byref(shp), 256, 256, ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_UNSUPPORTED
    # a tiles buffer sized for a larger minibatch than the call resolves is refused, not overrun
    shp = mok.make_shape(4096, 128, 128, 64, 6)
    s.rpad_max, s.tiles_max, s.mblocks_max = _caps(4096, 6, 64, 2048)
    rc = mok._lib.mok_build_schedule_noalloc(ctypes.byref(cfg), ctypes.byref(shp), 256, 256, ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_WORKSPACE_TOO_SMALL
