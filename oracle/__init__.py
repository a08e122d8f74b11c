"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle of the routed SwiGLU expert layer.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import this package.  The CUDA library never does, and the two share no code.

This module is argument marshalling over ``mok_oracle.c`` (plain C, fp64 loops), ``mok_oracle_mx.c``
(the MXFP8 mode) and ``mok_oracle_router.c`` (the router step before the layer); every function
cites, in the C source, the page passage it follows.  Arrays cross as numpy arrays:
bf16 tensors as ``uint16`` bit patterns, E4M3 / E8M0 as ``uint8``.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines (numpy / torch CPU float8 / torch autograd) or finite differences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mok_oracle.c")
_SRC_MX = os.path.join(_HERE, "mok_oracle_mx.c")
_SRC_ROUTER = os.path.join(_HERE, "mok_oracle_router.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_LIB32_PATH = os.path.join(_HERE, "liboracle_f32.so")
_lock = threading.Lock()
_lib = None
_lib32 = None

MT = 128  # GEMM row tile used for the padded expert-grouped layout


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fast-math): ``liboracle.so``, the fp64 reference of
    every parity check, and ``liboracle_f32.so``, the same layer loops in fp32 at -O3 -- the timed
    CPU baseline, never a reference."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_MX), os.path.getmtime(_SRC_ROUTER),
                 os.path.getmtime(os.path.abspath(__file__)))
    common = ["-std=c11", "-fopenmp", "-fPIC", "-fno-semantic-interposition", "-shared"]
    jobs = [(_LIB_PATH, ["gcc", "-O2", *common, _SRC, _SRC_MX, _SRC_ROUTER, "-lm"]),
            (_LIB32_PATH, ["gcc", "-O3", *common, "-DORC_REAL=float", "-DORC_TIMING_ONLY", _SRC, "-lm"])]
    for path, cmd in jobs:
        if force or not os.path.exists(path) or os.path.getmtime(path) < newest:
            tmp = path + f".tmp{os.getpid()}"
            subprocess.check_call([*cmd, "-o", tmp])
            os.replace(tmp, path)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            lib.orc_bf16_value.restype = ctypes.c_double
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_e8m0_value.restype = ctypes.c_double
            lib.orc_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.orc_mxfp8_quantize.restype = ctypes.c_int
            lib.orc_mxfp8_quantize.argtypes = [P, i64, i64, P, P]
            lib.orc_rpad_max.restype = i64
            lib.orc_rpad_max.argtypes = [i64, i32, i32, i32]
            lib.orc_schedule.restype = ctypes.c_int
            lib.orc_schedule.argtypes = [i64, i32, i32, P, i32, i32, i32, P, P, P, P, i64, P, P, i64, P, P, i64,
                                         P, P]
            lib.orc_forward.restype = None
            lib.orc_forward.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_backward.restype = None
            lib.orc_backward.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_forward_tokens.restype = None
            lib.orc_forward_tokens.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, i64, P, P]
            lib.orc_backward_tokens.restype = None
            lib.orc_backward_tokens.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, i64, P, P, P]
            lib.orc_dw_entries.restype = None
            lib.orc_dw_entries.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, i64, P, P, P, P, P]
            lib.orc_dw_block.restype = None
            lib.orc_dw_block.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, i32, i32, i64, P, P, P, P]
            lib.orc_mx_set_quant.restype = None
            lib.orc_mx_set_quant.argtypes = [ctypes.c_int]
            lib.orc_mx_fakequant.restype = None
            lib.orc_mx_fakequant.argtypes = [P, i64]
            lib.orc_layer_mx.restype = None
            lib.orc_layer_mx.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_tokens_mx.restype = None
            lib.orc_tokens_mx.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, i64, P, P, P, P]
            lib.orc_dw_block_mx.restype = None
            lib.orc_dw_block_mx.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, i32, i32, i64, P, P, P, P]
            lib.orc_router_logits.restype = None
            lib.orc_router_logits.argtypes = [P, P, P, i64, i32, i32, P]
            lib.orc_router_topk.restype = None
            lib.orc_router_topk.argtypes = [P, i64, i32, i32, P, P]
            lib.orc_router_backward.restype = None
            lib.orc_router_backward.argtypes = [P, P, i64, i32, i32, i32, P, P, P, P, P, P]
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_num_threads.argtypes = []
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def num_threads() -> int:
    return _load().orc_num_threads()


# ----------------------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------------------
def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(int(bits))


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (vectorised form of ``orc_bf16_value``)."""
    with np.errstate(invalid="ignore"):
        return (_u16(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def e8m0_value(b: int) -> float:
    return _load().orc_e8m0_value(int(b))


def mxfp8_quantize(x_bf16: np.ndarray):
    """MXFP8 (E4M3 + one E8M0 scale per 32 along the last axis) of a 2-D bf16 matrix."""
    x = _u16(x_bf16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty((rows, cols // 32), np.uint8)
    rc = _load().orc_mxfp8_quantize(_p(x), rows, cols, _p(q), _p(sc))
    if rc != 0:
        raise ValueError("cols must be a multiple of 32")
    return q, sc


def mxfp8_dequantize(q: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Exact value of an MXFP8 matrix: e4m3 * 2^(e8m0 - 127)."""
    lib = _load()
    lut = np.array([lib.orc_e4m3_value(c) for c in range(256)], np.float64)
    sv = np.array([lib.orc_e8m0_value(b) for b in range(256)], np.float64)
    return lut[q] * np.repeat(sv[sc], 32, axis=1)


# ----------------------------------------------------------------------------------------------
# schedule
# ----------------------------------------------------------------------------------------------
def rpad_max(T: int, K: int, E: int, mt: int = MT) -> int:
    return int(_load().orc_rpad_max(T, K, E, mt))


def schedule(ids: np.ndarray, E: int, mb: int, MB: int, mt: int = MT) -> dict:
    """Expert-grouped schedule of the flat slots of ``ids`` [T, K] (see ``orc_schedule``)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    R = T * K
    cap = rpad_max(T, K, E, mt)
    tcap = (R + mb - 1) // mb + E
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    poff = np.empty(E + 1, np.int32)
    perm = np.empty(cap, np.int32)
    inv = np.empty(max(R, 1), np.int32)
    tiles = np.empty((tcap, 4), np.int32)
    mblocks = np.empty((max(cap // mt, 1), 4), np.int32)
    ntiles = np.zeros(1, np.int64)
    nmb = np.zeros(1, np.int64)
    rp = np.zeros(1, np.int64)
    rc = _load().orc_schedule(T, K, E, _p(ids), mt, mb, MB, _p(counts), _p(offsets), _p(poff), _p(perm), cap,
                              _p(inv), _p(tiles), tcap, _p(ntiles), _p(mblocks), mblocks.shape[0], _p(nmb), _p(rp))
    if rc == 1:
        raise ValueError("expert id out of range")
    if rc == 2:
        raise ValueError("capacity exceeded")
    Rp = int(rp[0])
    return dict(counts=counts, offsets=offsets, poff=poff, perm=perm[:Rp].copy(), inv=inv[:R].copy(),
                tiles=tiles[: int(ntiles[0])].copy(), mblocks=mblocks[: int(nmb[0])].copy(), rpad=Rp)


# ----------------------------------------------------------------------------------------------
# layer forward / backward (fp64)
# ----------------------------------------------------------------------------------------------
def _layer_args(ids, s, x, Wg, Wu, Wd):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    x, Wg, Wu, Wd = _u16(x), _u16(Wg), _u16(Wu), _u16(Wd)
    T, K = ids.shape
    E, I, H = Wg.shape
    assert x.shape == (T, H) and Wu.shape == (E, I, H) and Wd.shape == (E, H, I) and s.shape == (T, K)
    return ids, s, x, Wg, Wu, Wd, T, H, I, E, K


def forward(ids, s, x, Wg, Wu, Wd, intermediates: bool = False):
    """out [T, H] fp64; with ``intermediates`` also g, u, a [R, I] and y [R, H] in slot order."""
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    R = T * K
    out = np.empty((T, H), np.float64)
    if intermediates:
        g, u, a, y = (np.empty((R, I)), np.empty((R, I)), np.empty((R, I)), np.empty((R, H)))
        ptrs = [_p(g), _p(u), _p(a), _p(y)]
    else:
        ptrs = [None] * 4
    _load().orc_forward(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(out), *ptrs)
    if intermediates:
        return out, dict(g=g, u=u, a=a, y=y)
    return out


def backward(ids, s, x, Wg, Wu, Wd, dY, check: bool = False):
    """dict(dX [T,H], dWg, dWu [E,I,H], dWd [E,H,I], dS [T,K]) in fp64 (+ dS_check = <dY, y>)."""
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    dY = _u16(dY)
    assert dY.shape == (T, H)
    dX = np.empty((T, H))
    dWg = np.empty((E, I, H))
    dWu = np.empty((E, I, H))
    dWd = np.empty((E, H, I))
    dS = np.empty((T, K))
    dSc = np.empty((T, K)) if check else None
    _load().orc_backward(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), _p(dX), _p(dWg),
                         _p(dWu), _p(dWd), _p(dS), _p(dSc) if check else None)
    r = dict(dX=dX, dWg=dWg, dWu=dWu, dWd=dWd, dS=dS)
    if check:
        r["dS_check"] = dSc
    return r


def _load32():
    global _lib32
    if _lib32 is None:
        _load()  # builds both libraries
        with _lock:
            lib = ctypes.CDLL(_LIB32_PATH)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            lib.orc_forward.restype = None
            lib.orc_forward.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P]
            lib.orc_backward.restype = None
            lib.orc_backward.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, P]
            _lib32 = lib
    return _lib32


def step_f32(ids, s, x, Wg, Wu, Wd, dY):
    """Forward + backward of the layer loops in fp32 (-O3): the timed CPU baseline.  Returns out,
    dX [T,H], dWg, dWu [E,I,H], dWd [E,H,I], dS [T,K] as float32 arrays."""
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    dY = _u16(dY)
    f = np.float32
    out, dX, dS = np.empty((T, H), f), np.empty((T, H), f), np.empty((T, K), f)
    dWg, dWu, dWd = np.empty((E, I, H), f), np.empty((E, I, H), f), np.empty((E, H, I), f)
    lib = _load32()
    lib.orc_forward(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(out), None, None, None, None)
    lib.orc_backward(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), _p(dX), _p(dWg), _p(dWu),
                     _p(dWd), _p(dS), None)
    return dict(out=out, dX=dX, dWg=dWg, dWu=dWu, dWd=dWd, dS=dS)


def forward_tokens(ids, s, x, Wg, Wu, Wd, tokens):
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    out = np.empty((tok.size, H))
    _load().orc_forward_tokens(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), tok.size, _p(tok),
                               _p(out))
    return out


def backward_tokens(ids, s, x, Wg, Wu, Wd, dY, tokens):
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    dY = _u16(dY)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    dX = np.empty((tok.size, H))
    dS = np.empty((tok.size, K))
    _load().orc_backward_tokens(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), tok.size,
                                _p(tok), _p(dX), _p(dS))
    return dX, dS


def dw_entries(ids, s, x, Wg, Wu, Wd, dY, which, e, m, c):
    """Single entries of dWg (which 0), dWu (1) [e, m<I, c<H] and dWd (2) [e, m<H, c<I]."""
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    dY = _u16(dY)
    which = np.ascontiguousarray(which, np.int32)
    e = np.ascontiguousarray(e, np.int32)
    m = np.ascontiguousarray(m, np.int32)
    c = np.ascontiguousarray(c, np.int32)
    val = np.empty(which.size)
    _load().orc_dw_entries(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), which.size,
                           _p(which), _p(e), _p(m), _p(c), _p(val))
    return val


def dw_block(ids, s, x, Wg, Wu, Wd, dY, e: int, i0: int, hs):
    """dWg, dWu [32, nh] and dWd [nh, 32] of expert e on I columns [i0, i0+32) and hidden columns hs."""
    ids, s, x, Wg, Wu, Wd, T, H, I, E, K = _layer_args(ids, s, x, Wg, Wu, Wd)
    dY = _u16(dY)
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    dwg, dwu, dwd = np.empty((32, hs.size)), np.empty((32, hs.size)), np.empty((hs.size, 32))
    _load().orc_dw_block(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(Wg), _p(Wu), _p(Wd), _p(dY), int(e), int(i0),
                         hs.size, _p(hs), _p(dwg), _p(dwu), _p(dwd))
    return dwg, dwu, dwd


# ----------------------------------------------------------------------------------------------
# MXFP8 mode (mok_oracle_mx.c)
# ----------------------------------------------------------------------------------------------
MX_KEYS = ("q_gate", "s_gate", "q_up", "s_up", "q_down", "s_down",
           "qt_gate", "st_gate", "qt_up", "st_up", "qt_down", "st_down")


def mx_fakequant(v: np.ndarray) -> np.ndarray:
    """MX quantise-dequantise of an fp64 array along its last axis (blocks of 32)."""
    a = np.array(v, dtype=np.float64, copy=True, order="C")
    _load().orc_mx_fakequant(_p(a), a.size)
    return a


def mx_set_quant(on: bool):
    _load().orc_mx_set_quant(1 if on else 0)


def mx_weights(Wg, Wu, Wd, experts=None) -> dict:
    """The pre-quantised weight copies of the MXFP8 mode, from bf16 weights [E,I,H], [E,H,I]:
    forward copies along each GEMM's K (Wg, Wu along H; Wd along I) and backward copies of the
    transposes (Wg^T, Wu^T along I; Wd^T along H).  With ``experts``, only those experts are
    quantised (the others' bytes are zero and must not be read)."""
    Wg, Wu, Wd = _u16(Wg), _u16(Wu), _u16(Wd)
    E, I, H = Wg.shape
    sel = range(E) if experts is None else sorted(set(int(e) for e in np.asarray(experts).reshape(-1)))
    shapes = dict(gate=(I, H), up=(I, H), down=(H, I))
    src = dict(gate=Wg, up=Wu, down=Wd)
    out = {}
    for name, W in src.items():
        r, c = shapes[name]
        q = np.zeros((E * r, c), np.uint8)
        sc = np.zeros((E * r, c // 32), np.uint8)
        qt = np.zeros((E * c, r), np.uint8)
        st = np.zeros((E * c, r // 32), np.uint8)
        for e in sel:
            q[e * r:(e + 1) * r], sc[e * r:(e + 1) * r] = mxfp8_quantize(W[e])
            qt[e * c:(e + 1) * c], st[e * c:(e + 1) * c] = mxfp8_quantize(np.ascontiguousarray(W[e].T))
        out["q_" + name], out["s_" + name], out["qt_" + name], out["st_" + name] = q, sc, qt, st
    return out


def _mx_ptrs(mx: dict):
    arrs = [np.ascontiguousarray(mx[k]) for k in MX_KEYS]
    ptrs = (ctypes.c_void_p * 12)(*[a.ctypes.data for a in arrs])
    return arrs, ptrs


def layer_mx(ids, s, x, dY, mx: dict, E: int, I: int, with_aq: bool = False, with_dg: bool = False) -> dict:
    """Full MXFP8-mode forward + backward (fp64 apart from the quantisation points).  with_aq adds
    a_q [R, I]; with_dg adds the unquantised dg, du, a [R, I] (slot order)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    x, dY = _u16(x), _u16(dY)
    T, K = ids.shape
    H = x.shape[1]
    arrs, ptrs = _mx_ptrs(mx)
    r = dict(out=np.empty((T, H)), dX=np.empty((T, H)), dWg=np.empty((E, I, H)), dWu=np.empty((E, I, H)),
             dWd=np.empty((E, H, I)), dS=np.empty((T, K)))
    aq = np.empty((T * K, I)) if with_aq else None
    dg = np.empty((T * K, I)) if with_dg else None
    du = np.empty((T * K, I)) if with_dg else None
    a = np.empty((T * K, I)) if with_dg else None
    _load().orc_layer_mx(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(dY), ptrs, _p(r["out"]), _p(r["dX"]),
                         _p(r["dWg"]), _p(r["dWu"]), _p(r["dWd"]), _p(r["dS"]), _p(aq) if with_aq else None,
                         _p(dg) if with_dg else None, _p(du) if with_dg else None, _p(a) if with_dg else None)
    if with_aq:
        r["aq"] = aq
    if with_dg:
        r["dg"], r["du"], r["a"] = dg, du, a
    return r


def tokens_mx(ids, s, x, dY, mx: dict, E: int, I: int, tokens):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    x, dY = _u16(x), _u16(dY)
    T, K = ids.shape
    H = x.shape[1]
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    arrs, ptrs = _mx_ptrs(mx)
    out, dX, dS = np.empty((tok.size, H)), np.empty((tok.size, H)), np.empty((tok.size, K))
    _load().orc_tokens_mx(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(dY), ptrs, tok.size, _p(tok), _p(out), _p(dX),
                          _p(dS))
    return out, dX, dS


def dw_block_mx(ids, s, x, dY, mx: dict, E: int, I: int, e: int, i0: int, hs):
    """dWg, dWu [32, nh] and dWd [nh, 32] of expert e on I columns [i0, i0+32) and hidden columns hs."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    x, dY = _u16(x), _u16(dY)
    T, K = ids.shape
    H = x.shape[1]
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    arrs, ptrs = _mx_ptrs(mx)
    dwg, dwu, dwd = np.empty((32, hs.size)), np.empty((32, hs.size)), np.empty((hs.size, 32))
    _load().orc_dw_block_mx(T, H, I, E, K, _p(ids), _p(s), _p(x), _p(dY), ptrs, int(e), int(i0), hs.size, _p(hs),
                            _p(dwg), _p(dwu), _p(dwd))
    return dwg, dwu, dwd


# ---------------------------------------------------------------------------------------------
# router step (mok_oracle_router.c): logits in fp32 as the kernel takes its top-k decision, the
# rest in fp64
# ---------------------------------------------------------------------------------------------
def router_logits(x, w, bias=None) -> np.ndarray:
    """fp32 logits [T,E] of x [T,H] (bf16 bits) and W [H,E] (bf16 bits), + bias [E] fp32."""
    x, w = _u16(x), _u16(w)
    T, H = x.shape
    E = w.shape[1]
    assert w.shape[0] == H
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _load().orc_router_logits(_p(x), _p(w), None if b is None else _p(b), T, H, E, _p(out))
    return out


def router_topk(logits, K: int):
    """Top-K ids [T,K] int32 (descending logit, equal logits in ascending id) and the renormalised
    weights [T,K] fp64."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, K), dtype=np.int32)
    wts = np.empty((T, K))
    _load().orc_router_topk(_p(lg), T, E, K, _p(ids), _p(wts))
    return ids, wts


def router_backward(x, w, ids, weights, d_topk, with_bias: bool = False):
    """dW [H,E], dbias [E] (or None) and dx [T,H], fp64, from the forward's ids / fp32 weights and
    the fp32 top-k weight gradient."""
    x, w = _u16(x), _u16(w)
    T, H = x.shape
    E = w.shape[1]
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    K = ids.shape[1]
    wt = np.ascontiguousarray(weights, dtype=np.float32)
    dt = np.ascontiguousarray(d_topk, dtype=np.float32)
    dw, dx = np.empty((H, E)), np.empty((T, H))
    db = np.empty(E) if with_bias else None
    _load().orc_router_backward(_p(x), _p(w), T, H, E, K, _p(ids), _p(wt), _p(dt), _p(dw),
                                None if db is None else _p(db), _p(dx))
    return dw, db, dx
