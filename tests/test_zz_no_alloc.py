"""mok_build_schedule_noalloc: the schedule build for callers that may not allocate device memory
(its scratch lives in a fixed array inside the library).  Called through the C ABI, its tables
must equal those of mok_build_schedule bit for bit -- the schedule is integer work, so the
tolerance is zero -- on two calls in a row with different routing, so a stale scratch array would
show.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _noalloc(mok, cfg, shp, ids, w):
    T, K, E = shp.T, shp.K, shp.E
    R = T * K
    rpad_max = R + 127 * E
    tiles_max = -(-R // cfg.minibatch_rows) + E
    mblocks_max = rpad_max // 128
    dev = ids.device
    bufs = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                poff=torch.empty(E + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(rpad_max, dtype=torch.int32, device=dev),
                inv=torch.empty(max(R, 1), dtype=torch.int32, device=dev),
                tiles=torch.empty((tiles_max, 4), dtype=torch.int32, device=dev),
                mblocks=torch.empty((mblocks_max, 4), dtype=torch.int32, device=dev),
                meta=torch.empty(16, dtype=torch.int32, device=dev),
                row_weight=torch.empty(rpad_max, dtype=torch.float32, device=dev),
                row_token=torch.empty(rpad_max, dtype=torch.int32, device=dev))
    s = mok.mok_schedule()
    for k, v in bufs.items():
        setattr(s, k, v.data_ptr())
    rc = mok._lib.mok_build_schedule_noalloc(ctypes.byref(cfg), ctypes.byref(shp), ids.data_ptr(), w.data_ptr(),
                                             ctypes.byref(s), torch.cuda.current_stream().cuda_stream)
    assert rc == mok.MOK_OK, rc
    torch.cuda.synchronize()
    assert s.rpad_max == rpad_max and s.tiles_max == tiles_max and s.mblocks_max == mblocks_max
    return {k: v.cpu().numpy() for k, v in bufs.items()}, s


def _reference(mok, cfg, shp, ids, w):
    ws = mok.alloc_workspace(cfg, shp)
    sch = mok.mok_build_schedule(cfg, shp, ids, w, ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in sch.tables().items()}


def _same(a, b):
    rp = int(b["meta"][0])
    assert int(a["meta"][0]) == rp and np.array_equal(a["meta"][:3], b["meta"][:3])
    assert a["meta"][15] == b["meta"][15] == 0
    for k in ("counts", "offsets", "poff", "inv"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("perm", "row_token"):
        assert np.array_equal(a[k][:rp], b[k][:rp]), k
    assert np.array_equal(a["row_weight"][:rp].view(np.uint32), b["row_weight"][:rp].view(np.uint32))
    nt = int(b["meta"][1])
    assert np.array_equal(a["tiles"][:nt], b["tiles"][:nt])
    assert np.array_equal(a["mblocks"][:rp // 128], b["mblocks"][:rp // 128])


def test_noalloc_schedule_matches_workspace_schedule_on_consecutive_calls(mok):
    cfg = mok.make_config(512, 2048)
    for name, seed in (("sweep_zipf2", 0), ("bf16_e64", 1)):
        wl = inputs.WORKLOADS[name]
        d = inputs.make(inputs.custom(wl.T, 128, 128, wl.E, wl.K, wl.router, wl.zipf), seed=seed, with_dy=False)
        ids, w = d["topk_ids"].cuda(), d["topk_weights"].cuda()
        shp = mok.make_shape(wl.T, 128, 128, wl.E, wl.K)
        got, _ = _noalloc(mok, cfg, shp, ids, w)
        _same(got, _reference(mok, cfg, shp, ids, w))


def test_noalloc_rejects_sizes_beyond_its_scratch(mok):
    cfg = mok.make_config(512, 2048)
    shp = mok.make_shape(1 << 20, 128, 128, 1024, 2)  # 4096 chunks x 1025 > 524288 entries
    s = mok.mok_schedule()
    for k in ("counts", "offsets", "poff", "perm", "inv", "tiles", "mblocks", "meta", "row_weight", "row_token"):
        setattr(s, k, 256)
    rc = mok._lib.mok_build_schedule_noalloc(ctypes.byref(cfg), ctypes.byref(shp), 256, 256, ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_UNSUPPORTED
