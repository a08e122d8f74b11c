"""The C-ABI library loads and exports every entry point ``include/mok.h`` declares, and its
host-side checks reject bad arguments before any device work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from helpers import ROOT


@pytest.fixture(scope="module")
def mok():
    import __graft_entry__
    __graft_entry__.build_library()
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"MOK_API\s+[\w\s\*]+?\b(mok_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    d = _declared()
    for n in ("mok_mxfp8_quantize", "mok_build_schedule", "mok_forward", "mok_backward"):
        assert n in d


def test_library_exports_every_declared_symbol(mok):
    lib = ctypes.CDLL(mok.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(mok.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", mok.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (mok_\w+)", out))
    assert exported == set(_declared())


def test_version_and_status_strings(mok):
    assert mok.mok_version() == "0.1.0"
    for c in range(8):
        assert mok._lib.mok_status_string(c)


def test_workspace_sizes_and_validation(mok):
    cfg = mok.make_config(512, 2048)
    shp = mok.make_shape(4096, 2048, 1024, 64, 6)
    ws = mok.mok_workspace_bytes(cfg, shp)
    ctx = mok.mok_fwd_ctx_bytes(cfg, shp)
    rpad_max = 4096 * 6 + 64 * 127
    assert ctx >= rpad_max * (2048 + 3 * 1024) * 2
    assert ws >= rpad_max * (2 * 2048 + 3 * 1024) * 2
    bad = [mok.make_shape(16, 100, 128, 4, 2), mok.make_shape(16, 128, 96, 4, 2), mok.make_shape(16, 128, 128, 2, 3),
           mok.make_shape(16, 128, 128, 2000, 2), mok.make_shape(-1, 128, 128, 4, 2)]
    for s in bad:
        with pytest.raises(mok.MokError):
            mok.mok_workspace_bytes(cfg, s)
    for c in (mok.make_config(100, 200), mok.make_config(256, 384), mok.make_config(128, 256, -1)):
        with pytest.raises(mok.MokError):
            mok.mok_workspace_bytes(c, shp)


def test_automatic_granularity_resolves_like_the_documented_rule(mok):
    # minibatch = ceil(T*K/E) rounded up to 128 * 2^k in [256, 2048]; macrobatch = the smallest
    # multiple of it that is >= 4 * minibatch and >= 2048
    for (T, H, I, E, K), mb, MB in [((4096, 2048, 1024, 64, 6), 512, 2048), ((2048, 7168, 2048, 256, 8), 256, 2048),
                                     ((16384, 7168, 2048, 4, 1), 2048, 8192), ((0, 128, 128, 4, 2), 256, 2048),
                                     ((8192, 4096, 1536, 128, 8), 512, 2048)]:
        shp = mok.make_shape(T, H, I, E, K)
        auto = mok.mok_workspace_bytes(mok.make_config(0, 0), shp)
        assert auto == mok.mok_workspace_bytes(mok.make_config(mb, MB), shp), (T, E, K)
        if 0 < T and mb < 2048:  # another minibatch size changes the tile table's bound
            assert auto != mok.mok_workspace_bytes(mok.make_config(2 * mb, max(2 * mb, MB)), shp)
    # an explicit minibatch with an automatic macrobatch
    shp = mok.make_shape(64, 128, 128, 4, 2)
    assert mok.mok_workspace_bytes(mok.make_config(384, 0), shp) == mok.mok_workspace_bytes(
        mok.make_config(384, 2304), shp)


def test_host_rejects_bad_calls_without_touching_the_device(mok):
    cfg = mok.make_config()
    shp = mok.make_shape(16, 128, 128, 4, 2)
    s = mok.mok_schedule()
    # null workspace, null ids, undersized workspace: all refused on the host
    rc = mok._lib.mok_build_schedule(ctypes.byref(cfg), ctypes.byref(shp), None, None, None, 0, ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    rc = mok._lib.mok_build_schedule(ctypes.byref(cfg), ctypes.byref(shp), None, None, 256, 1 << 30,
                                     ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_INVALID_ARG
    rc = mok._lib.mok_build_schedule(ctypes.byref(cfg), ctypes.byref(shp), 256, 256, 256, 16, ctypes.byref(s), None)
    assert rc == mok.MOK_ERR_WORKSPACE_TOO_SMALL
    assert mok._lib.mok_mxfp8_quantize(None, 4, 48, None, None, None) == mok.MOK_ERR_INVALID_ARG
    assert mok._lib.mok_mxfp8_quantize(None, 0, 64, None, None, None) == mok.MOK_OK
    assert mok._lib.mok_forward(None, None, None, None, None, 0, None) == mok.MOK_ERR_INVALID_ARG
    assert mok._lib.mok_backward(None, None, None, None, None, None) == mok.MOK_ERR_INVALID_ARG


def test_product_path_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_layer_build_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "liboracle" not in src and "mok_oracle" not in src, f
