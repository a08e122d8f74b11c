"""Thin Python binding of ``libmok.so`` (see ``include/mok.h``): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module only checks tensor
dtypes / devices / contiguity, passes ``data_ptr()``s and the current CUDA stream, and turns
status codes into exceptions.  PyTorch provides device memory and streams.

Importing this module loads the library and raises ``ImportError`` when it is missing: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmok.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libmok.so not found at {LIB_PATH}; build it with __graft_entry__.build() "
                      "(nvcc, sm_103a). There is no CPU fallback.")
_lib = ctypes.CDLL(LIB_PATH)

MOK_OK = 0
MOK_ERR_INVALID_ARG = 1
MOK_ERR_UNSUPPORTED = 2
MOK_ERR_WORKSPACE_TOO_SMALL = 3
MOK_ERR_CUDA = 4
MOK_ERR_BAD_EXPERT_ID = 5
MOK_ERR_CAPACITY = 6
MOK_ERR_TIMEOUT = 7
MOK_BF16 = 0
MOK_MXFP8 = 1


class MokError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.mok_status_string(code).decode()
        super().__init__(f"{where}: {msg} (status {code})")


class mok_config(ctypes.Structure):
    _fields_ = [("minibatch_rows", ctypes.c_int32), ("macrobatch_rows", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("precision", ctypes.c_int32), ("debug_flags", ctypes.c_uint32)]


class mok_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32)]


_P = ctypes.c_void_p


class mok_schedule(ctypes.Structure):
    _fields_ = [("shape", mok_shape), ("config", mok_config), ("rpad_max", ctypes.c_int64),
                ("tiles_max", ctypes.c_int64), ("mblocks_max", ctypes.c_int64), ("counts", _P), ("offsets", _P),
                ("poff", _P), ("perm", _P), ("inv", _P), ("tiles", _P), ("mblocks", _P), ("meta", _P),
                ("row_weight", _P), ("row_token", _P), ("status", _P), ("topk_weights", _P), ("ws", _P),
                ("ws_bytes", ctypes.c_size_t)]


MX_KEYS = ("q_gate", "s_gate", "q_up", "s_up", "q_down", "s_down",
           "qt_gate", "st_gate", "qt_up", "st_up", "qt_down", "st_down")


class mok_weights(ctypes.Structure):
    _fields_ = [("w_gate", _P), ("w_up", _P), ("w_down", _P)] + [(k, _P) for k in MX_KEYS]


class mok_grads(ctypes.Structure):
    _fields_ = [("dx", _P), ("dw_gate", _P), ("dw_up", _P), ("dw_down", _P), ("d_topk_weights", _P)]


_lib.mok_version.restype = ctypes.c_char_p
_lib.mok_version.argtypes = []
_lib.mok_status_string.restype = ctypes.c_char_p
_lib.mok_status_string.argtypes = [ctypes.c_int]
_lib.mok_workspace_bytes.restype = ctypes.c_size_t
_lib.mok_workspace_bytes.argtypes = [ctypes.POINTER(mok_config), ctypes.POINTER(mok_shape)]
_lib.mok_fwd_ctx_bytes.restype = ctypes.c_size_t
_lib.mok_fwd_ctx_bytes.argtypes = [ctypes.POINTER(mok_config), ctypes.POINTER(mok_shape)]
_lib.mok_mxfp8_quantize.restype = ctypes.c_int
_lib.mok_mxfp8_quantize.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, _P, _P, _P]
_lib.mok_build_schedule.restype = ctypes.c_int
_lib.mok_build_schedule.argtypes = [ctypes.POINTER(mok_config), ctypes.POINTER(mok_shape), _P, _P, _P,
                                    ctypes.c_size_t, ctypes.POINTER(mok_schedule), _P]
_lib.mok_forward.restype = ctypes.c_int
_lib.mok_forward.argtypes = [ctypes.POINTER(mok_schedule), _P, ctypes.POINTER(mok_weights), _P, _P,
                             ctypes.c_size_t, _P]
_lib.mok_backward.restype = ctypes.c_int
_lib.mok_backward.argtypes = [ctypes.POINTER(mok_schedule), _P, _P, ctypes.POINTER(mok_weights),
                              ctypes.POINTER(mok_grads), _P]


class mok_trace(ctypes.Structure):
    _fields_ = [("events", ctypes.POINTER(ctypes.c_void_p)), ("kinds", ctypes.POINTER(ctypes.c_int32)),
                ("capacity", ctypes.c_int32), ("count", ctypes.c_int32)]


_lib.mok_set_trace.restype = ctypes.c_int
_lib.mok_set_trace.argtypes = [ctypes.POINTER(mok_trace)]
_lib.mok_kernel_name.restype = ctypes.c_char_p
_lib.mok_kernel_name.argtypes = [ctypes.c_int32]
_lib.mok_read_device_status.restype = ctypes.c_int
_lib.mok_read_device_status.argtypes = [ctypes.POINTER(mok_schedule), ctypes.POINTER(ctypes.c_uint32), _P]
_lib.mok_selftest_wait_timeout.restype = ctypes.c_int
_lib.mok_selftest_wait_timeout.argtypes = [_P, _P]

class mok_mx_operands(ctypes.Structure):
    _fields_ = [(k, _P) for k in ("xq", "xs", "aq", "as_", "dyq", "dys", "dgq", "dgs", "xr", "xrs", "dyr", "dyrs",
                                  "dgr", "dgrs", "sar", "sars")] + \
        [("rows", ctypes.c_int64), ("rcap", ctypes.c_int64), ("xr_groups", ctypes.c_int32),
         ("sar_groups", ctypes.c_int32)]


_lib.mok_mx_operands_of.restype = ctypes.c_int
_lib.mok_mx_operands_of.argtypes = [ctypes.POINTER(mok_schedule), _P, ctypes.POINTER(mok_mx_operands)]

EXPORTED = ("mok_version", "mok_status_string", "mok_workspace_bytes", "mok_fwd_ctx_bytes", "mok_mxfp8_quantize",
            "mok_build_schedule", "mok_forward", "mok_backward", "mok_read_device_status", "mok_set_trace",
            "mok_kernel_name", "mok_build_schedule_noalloc", "mok_mx_operands_of", "mok_router_workspace_bytes",
            "mok_router_forward", "mok_router_backward", "mok_selftest_wait_timeout", "mok_ep_build_schedule",
            "mok_ep_forward", "mok_ep_backward", "mok_ep_combine")
_lib.mok_router_workspace_bytes.restype = ctypes.c_size_t
_lib.mok_router_workspace_bytes.argtypes = [ctypes.POINTER(mok_shape)]
_lib.mok_router_forward.restype = ctypes.c_int
_lib.mok_router_forward.argtypes = [ctypes.POINTER(mok_shape), _P, _P, _P, _P, _P, _P, _P]
_lib.mok_router_backward.restype = ctypes.c_int
_lib.mok_router_backward.argtypes = [ctypes.POINTER(mok_schedule), _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                     _P, ctypes.c_size_t, _P]
_lib.mok_build_schedule_noalloc.restype = ctypes.c_int
_lib.mok_build_schedule_noalloc.argtypes = [ctypes.POINTER(mok_config), ctypes.POINTER(mok_shape), _P, _P,
                                            ctypes.POINTER(mok_schedule), _P]


# ---- expert parallelism ----
MOK_EP_MAX_RANKS = 8


class mok_ep_group(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int32), ("rank", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int64)]


_PT = ctypes.POINTER(_P)
_lib.mok_ep_build_schedule.restype = ctypes.c_int
_lib.mok_ep_build_schedule.argtypes = [ctypes.POINTER(mok_config), ctypes.POINTER(mok_shape),
                                       ctypes.POINTER(mok_ep_group), _PT, _PT, _P, ctypes.c_size_t,
                                       ctypes.POINTER(mok_schedule), _P]
_lib.mok_ep_forward.restype = ctypes.c_int
_lib.mok_ep_forward.argtypes = [ctypes.POINTER(mok_schedule), ctypes.POINTER(mok_ep_group), _PT,
                                ctypes.POINTER(mok_weights), _PT, _P, ctypes.c_size_t, _P]
_lib.mok_ep_backward.restype = ctypes.c_int
_lib.mok_ep_backward.argtypes = [ctypes.POINTER(mok_schedule), ctypes.POINTER(mok_ep_group), _P, _PT,
                                 ctypes.POINTER(mok_weights), _P, _P, _P, _PT, _PT, _P]
_lib.mok_ep_combine.restype = ctypes.c_int
_lib.mok_ep_combine.argtypes = [ctypes.POINTER(mok_shape), ctypes.POINTER(mok_ep_group), _P, _P, _P, _P, _P]


def _check(rc: int, where: str):
    if rc != MOK_OK:
        raise MokError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def mok_version() -> str:
    return _lib.mok_version().decode()


MOK_FLAG_STATIC_TILES = 1  # static round-robin GEMM tile scheduling instead of cluster launch control


def make_config(minibatch_rows=512, macrobatch_rows=2048, num_ctas=0, precision=MOK_BF16, flags=0) -> mok_config:
    return mok_config(minibatch_rows, macrobatch_rows, num_ctas, precision, flags)


def make_shape(T, H, I, E, K) -> mok_shape:
    return mok_shape(T, H, I, E, K)


def mok_workspace_bytes(cfg: mok_config, shape: mok_shape) -> int:
    n = _lib.mok_workspace_bytes(ctypes.byref(cfg), ctypes.byref(shape))
    if n == 0:
        raise MokError(MOK_ERR_INVALID_ARG, "mok_workspace_bytes")
    return n


def mok_fwd_ctx_bytes(cfg: mok_config, shape: mok_shape) -> int:
    n = _lib.mok_fwd_ctx_bytes(ctypes.byref(cfg), ctypes.byref(shape))
    if n == 0:
        raise MokError(MOK_ERR_INVALID_ARG, "mok_fwd_ctx_bytes")
    return n


def mok_mxfp8_quantize(x: torch.Tensor, out_q: torch.Tensor | None = None, out_s: torch.Tensor | None = None,
                       stream=None):
    """MXFP8 of a 2-D bf16 tensor: (E4M3 bytes [rows, cols] uint8, E8M0 scales [rows, cols/32] uint8)."""
    rows, cols = x.shape
    if out_q is None:
        out_q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if out_s is None:
        out_s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    _check(_lib.mok_mxfp8_quantize(_ptr(x, torch.bfloat16, "x"), rows, cols, _ptr(out_q, torch.uint8, "out_q"),
                                   _ptr(out_s, torch.uint8, "out_s"), _stream(stream)), "mok_mxfp8_quantize")
    return out_q, out_s


@dataclass
class Schedule:
    """A built schedule plus the tensors it refers to (kept alive here)."""
    c: mok_schedule
    ws: torch.Tensor
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor

    def _view(self, field, n, dtype=torch.int32):
        """Device tensor view of one schedule table (for tests and inspection)."""
        ptr = getattr(self.c, field)
        base = self.ws.data_ptr()
        off = ptr - base
        esz = torch.tensor([], dtype=dtype).element_size()
        assert off % esz == 0 and off >= 0
        return self.ws.view(torch.uint8)[off:off + n * esz].view(dtype)

    def tables(self) -> dict:
        E = self.c.shape.E
        R = self.c.shape.T * self.c.shape.K
        return dict(counts=self._view("counts", E), offsets=self._view("offsets", E + 1),
                    poff=self._view("poff", E + 1), perm=self._view("perm", self.c.rpad_max),
                    inv=self._view("inv", R), tiles=self._view("tiles", 4 * self.c.tiles_max).view(-1, 4),
                    mblocks=self._view("mblocks", 4 * self.c.mblocks_max).view(-1, 4),
                    meta=self._view("meta", 16), row_weight=self._view("row_weight", self.c.rpad_max, torch.float32),
                    row_token=self._view("row_token", self.c.rpad_max))


    def mx_operands(self, fwd_ctx: torch.Tensor) -> dict:
        """Device views of the MXFP8 operand copies (mok_mx_operands_of): E4M3 codes ([rows, n]
        quantised along each row, transposed [n, rcap] quantised along the rows) and their
        atom-tiled E8M0 scale arrays (flat uint8), plus the layout numbers rows, rcap, xr_groups,
        sar_groups."""
        m = mok_mx_operands()
        _check(_lib.mok_mx_operands_of(ctypes.byref(self.c), _ptr(fwd_ctx, None, "fwd_ctx"), ctypes.byref(m)),
               "mok_mx_operands_of")
        H, I, rows, rcap = self.c.shape.H, self.c.shape.I, m.rows, m.rcap
        rt = (rows + 127) // 128

        def v(ptr, n):
            for buf in (self.ws, fwd_ctx):
                base = buf.data_ptr()
                if base <= ptr < base + buf.numel() * buf.element_size():
                    return buf.view(torch.uint8)[ptr - base:ptr - base + n]
            raise ValueError("pointer outside the workspace and the context")
        return dict(xq=v(m.xq, rows * H).view(rows, H), xs=v(m.xs, rt * 128 * (H // 32)),
                    aq=v(m.aq, rows * I).view(rows, I), as_=v(m.as_, rt * 128 * (I // 32)),
                    dyq=v(m.dyq, rows * H).view(rows, H), dys=v(m.dys, rt * 128 * (H // 32)),
                    dgq=v(m.dgq, rows * 2 * I).view(rows, 2 * I), dgs=v(m.dgs, rt * 128 * (2 * I // 32)),
                    xr=v(m.xr, H * rcap).view(H, rcap), xrs=v(m.xrs, H * rcap // 32),
                    dyr=v(m.dyr, H * rcap).view(H, rcap), dyrs=v(m.dyrs, H * rcap // 32),
                    dgr=v(m.dgr, 2 * I * rcap).view(2 * I, rcap), dgrs=v(m.dgrs, 2 * I * rcap // 32),
                    sar=v(m.sar, I * rcap).view(I, rcap), sars=v(m.sars, I * rcap // 32),
                    rows=rows, rcap=rcap, xr_groups=m.xr_groups, sar_groups=m.sar_groups)


def alloc_workspace(cfg: mok_config, shape: mok_shape, device="cuda") -> torch.Tensor:
    return torch.empty(mok_workspace_bytes(cfg, shape), dtype=torch.uint8, device=device)


def alloc_fwd_ctx(cfg: mok_config, shape: mok_shape, device="cuda") -> torch.Tensor:
    return torch.empty(mok_fwd_ctx_bytes(cfg, shape), dtype=torch.uint8, device=device)


def mok_build_schedule(cfg: mok_config, shape: mok_shape, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                       ws: torch.Tensor, stream=None) -> Schedule:
    s = mok_schedule()
    _check(_lib.mok_build_schedule(ctypes.byref(cfg), ctypes.byref(shape), _ptr(topk_ids, torch.int32, "topk_ids"),
                                   _ptr(topk_weights, torch.float32, "topk_weights"), _ptr(ws, None, "ws"),
                                   ws.numel() * ws.element_size(), ctypes.byref(s), _stream(stream)),
           "mok_build_schedule")
    return Schedule(s, ws, topk_ids, topk_weights)


def weights_struct(Wg=None, Wu=None, Wd=None, mx: dict | None = None) -> mok_weights:
    """bf16 weights for BF16 mode; ``mx`` = the pre-quantised copies (``quantize_weights``) for
    MXFP8 mode.  The struct holds raw pointers: keep the tensors alive while it is used."""
    w = mok_weights()
    w.w_gate = _ptr(Wg, torch.bfloat16, "w_gate")
    w.w_up = _ptr(Wu, torch.bfloat16, "w_up")
    w.w_down = _ptr(Wd, torch.bfloat16, "w_down")
    if mx:
        for k in MX_KEYS:
            setattr(w, k, _ptr(mx.get(k), torch.uint8, k))
    return w


def quantize_weights(Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, stream=None) -> dict:
    """The MXFP8 weight copies of mok_weights, made with mok_mxfp8_quantize on the device: forward
    copies along each GEMM's K and backward copies of the transposes."""
    E, I, H = Wg.shape
    out = {}
    out["q_gate"], out["s_gate"] = mok_mxfp8_quantize(Wg.reshape(E * I, H), stream=stream)
    out["q_up"], out["s_up"] = mok_mxfp8_quantize(Wu.reshape(E * I, H), stream=stream)
    out["q_down"], out["s_down"] = mok_mxfp8_quantize(Wd.reshape(E * H, I), stream=stream)
    out["qt_gate"], out["st_gate"] = mok_mxfp8_quantize(Wg.transpose(1, 2).contiguous().reshape(E * H, I), stream=stream)
    out["qt_up"], out["st_up"] = mok_mxfp8_quantize(Wu.transpose(1, 2).contiguous().reshape(E * H, I), stream=stream)
    out["qt_down"], out["st_down"] = mok_mxfp8_quantize(Wd.transpose(1, 2).contiguous().reshape(E * I, H), stream=stream)
    return out


def mok_forward(sched: Schedule, x: torch.Tensor, weights: mok_weights, out: torch.Tensor, fwd_ctx: torch.Tensor,
                stream=None) -> torch.Tensor:
    _check(_lib.mok_forward(ctypes.byref(sched.c), _ptr(x, torch.bfloat16, "x"), ctypes.byref(weights),
                            _ptr(out, torch.bfloat16, "out"), _ptr(fwd_ctx, None, "fwd_ctx"),
                            fwd_ctx.numel() * fwd_ctx.element_size(), _stream(stream)), "mok_forward")
    return out


@dataclass
class Grads:
    dx: torch.Tensor
    dw_gate: torch.Tensor
    dw_up: torch.Tensor
    dw_down: torch.Tensor
    d_topk_weights: torch.Tensor

    @staticmethod
    def empty(T, H, I, E, K, device="cuda") -> "Grads":
        return Grads(torch.empty((T, H), dtype=torch.bfloat16, device=device),
                     torch.empty((E, I, H), dtype=torch.float32, device=device),
                     torch.empty((E, I, H), dtype=torch.float32, device=device),
                     torch.empty((E, H, I), dtype=torch.float32, device=device),
                     torch.empty((T, K), dtype=torch.float32, device=device))

    def struct(self) -> mok_grads:
        g = mok_grads()
        g.dx = _ptr(self.dx, torch.bfloat16, "dx")
        g.dw_gate = _ptr(self.dw_gate, torch.float32, "dw_gate")
        g.dw_up = _ptr(self.dw_up, torch.float32, "dw_up")
        g.dw_down = _ptr(self.dw_down, torch.float32, "dw_down")
        g.d_topk_weights = _ptr(self.d_topk_weights, torch.float32, "d_topk_weights")
        return g


def mok_backward(sched: Schedule, fwd_ctx: torch.Tensor, dy: torch.Tensor, weights: mok_weights, grads: Grads,
                 stream=None) -> Grads:
    gs = grads.struct()
    _check(_lib.mok_backward(ctypes.byref(sched.c), _ptr(fwd_ctx, None, "fwd_ctx"), _ptr(dy, torch.bfloat16, "dy"),
                             ctypes.byref(weights), ctypes.byref(gs), _stream(stream)), "mok_backward")
    return grads


def make_ep_group(world: int, rank: int, tokens_per_rank: int) -> mok_ep_group:
    return mok_ep_group(world, rank, tokens_per_rank)


def _table(tensors, dtype, name):
    """Host array of per-rank device pointers (one per rank of the group)."""
    if len(tensors) > MOK_EP_MAX_RANKS:
        raise ValueError(f"at most {MOK_EP_MAX_RANKS} ranks")
    arr = (_P * MOK_EP_MAX_RANKS)()
    for r, t in enumerate(tensors):
        arr[r] = _ptr(t, dtype, f"{name}[{r}]")
    return arr


def mok_ep_build_schedule(cfg: mok_config, shape: mok_shape, ep: mok_ep_group, topk_ids: list, topk_weights: list,
                          ws: torch.Tensor, stream=None) -> Schedule:
    """This rank's schedule over the group's slots, from every rank's routing (lists of tensors)."""
    s = mok_schedule()
    ids_t, w_t = _table(topk_ids, torch.int32, "topk_ids"), _table(topk_weights, torch.float32, "topk_weights")
    _check(_lib.mok_ep_build_schedule(ctypes.byref(cfg), ctypes.byref(shape), ctypes.byref(ep), ids_t, w_t,
                                      _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), ctypes.byref(s),
                                      _stream(stream)), "mok_ep_build_schedule")
    return Schedule(s, ws, topk_ids[ep.rank], topk_weights[ep.rank])


def mok_ep_forward(sched: Schedule, ep: mok_ep_group, x: list, weights: mok_weights, y_recv: list,
                   fwd_ctx: torch.Tensor, stream=None) -> None:
    _check(_lib.mok_ep_forward(ctypes.byref(sched.c), ctypes.byref(ep), _table(x, torch.bfloat16, "x"),
                               ctypes.byref(weights), _table(y_recv, torch.bfloat16, "y_recv"),
                               _ptr(fwd_ctx, None, "fwd_ctx"), fwd_ctx.numel() * fwd_ctx.element_size(),
                               _stream(stream)), "mok_ep_forward")


def mok_ep_backward(sched: Schedule, ep: mok_ep_group, fwd_ctx: torch.Tensor, dy: list, weights: mok_weights,
                    dw_gate: torch.Tensor, dw_up: torch.Tensor, dw_down: torch.Tensor, dx_recv: list,
                    d_topk_weights: list, stream=None) -> None:
    _check(_lib.mok_ep_backward(ctypes.byref(sched.c), ctypes.byref(ep), _ptr(fwd_ctx, None, "fwd_ctx"),
                                _table(dy, torch.bfloat16, "dy"), ctypes.byref(weights),
                                _ptr(dw_gate, torch.float32, "dw_gate"), _ptr(dw_up, torch.float32, "dw_up"),
                                _ptr(dw_down, torch.float32, "dw_down"), _table(dx_recv, torch.bfloat16, "dx_recv"),
                                _table(d_topk_weights, torch.float32, "d_topk_weights"), _stream(stream)),
           "mok_ep_backward")


def mok_ep_combine(shape: mok_shape, ep: mok_ep_group, topk_ids: torch.Tensor, topk_weights: torch.Tensor | None,
                   recv: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    _check(_lib.mok_ep_combine(ctypes.byref(shape), ctypes.byref(ep), _ptr(topk_ids, torch.int32, "topk_ids"),
                               _ptr(topk_weights, torch.float32, "topk_weights"), _ptr(recv, torch.bfloat16, "recv"),
                               _ptr(out, torch.bfloat16, "out"), _stream(stream)), "mok_ep_combine")
    return out


def mok_read_device_status(sched: Schedule, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.mok_read_device_status(ctypes.byref(sched.c), ctypes.byref(v), _stream(stream)),
           "mok_read_device_status")
    return v.value


def mok_selftest_wait_timeout(status: torch.Tensor, stream=None) -> None:
    """status: one int32 (bit pattern of a uint32) on the device; the timeout bit is OR-ed in."""
    if status.dtype != torch.int32 or status.numel() != 1 or not status.is_cuda:
        raise ValueError("status must be one int32 on the GPU")
    _check(_lib.mok_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), _stream(stream)),
           "mok_selftest_wait_timeout")


# ---------------------------------------------------------------------------------------------
# router step (before the layer)
# ---------------------------------------------------------------------------------------------
def mok_router_workspace_bytes(shape: mok_shape) -> int:
    n = _lib.mok_router_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise MokError(MOK_ERR_INVALID_ARG, "mok_router_workspace_bytes")
    return n


def mok_router_forward(shape: mok_shape, x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor | None,
                       logits: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, stream=None):
    _check(_lib.mok_router_forward(ctypes.byref(shape), _ptr(x, torch.bfloat16, "x"),
                                   _ptr(w_router, torch.bfloat16, "w_router"), _ptr(bias, torch.float32, "bias"),
                                   _ptr(logits, torch.float32, "logits"), _ptr(topk_ids, torch.int32, "topk_ids"),
                                   _ptr(topk_weights, torch.float32, "topk_weights"), _stream(stream)),
           "mok_router_forward")


def mok_router_backward(sched: Schedule, x: torch.Tensor, w_router: torch.Tensor, topk_ids: torch.Tensor,
                        topk_weights: torch.Tensor, d_topk_weights: torch.Tensor, dw_router: torch.Tensor,
                        d_bias: torch.Tensor | None, dx: torch.Tensor, accumulate_dx: bool, ws: torch.Tensor,
                        stream=None):
    _check(_lib.mok_router_backward(ctypes.byref(sched.c), _ptr(x, torch.bfloat16, "x"),
                                    _ptr(w_router, torch.bfloat16, "w_router"), _ptr(topk_ids, torch.int32, "ids"),
                                    _ptr(topk_weights, torch.float32, "topk_weights"),
                                    _ptr(d_topk_weights, torch.float32, "d_topk_weights"),
                                    _ptr(dw_router, torch.float32, "dw_router"), _ptr(d_bias, torch.float32, "d_bias"),
                                    _ptr(dx, torch.bfloat16, "dx"), 1 if accumulate_dx else 0, _ptr(ws, None, "ws"),
                                    ws.numel() * ws.element_size(), _stream(stream)), "mok_router_backward")


def router_forward(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor | None, K: int, stream=None):
    """Allocating form: returns (logits [T,E] fp32, topk_ids [T,K] int32, topk_weights [T,K] fp32)."""
    T, H = x.shape
    E = w_router.shape[1]
    shape = make_shape(T, H, 128, E, K)
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    ids = torch.empty((T, K), dtype=torch.int32, device=x.device)
    wts = torch.empty((T, K), dtype=torch.float32, device=x.device)
    mok_router_forward(shape, x, w_router, bias, logits, ids, wts, stream)
    return logits, ids, wts


def router_backward(sched: Schedule, x: torch.Tensor, w_router: torch.Tensor, topk_ids: torch.Tensor,
                    topk_weights: torch.Tensor, d_topk_weights: torch.Tensor, with_bias: bool = False,
                    dx: torch.Tensor | None = None, stream=None):
    """Allocating form: returns (dw_router [H,E] fp32, d_bias [E] fp32 or None, dx [T,H] bf16).  A
    given dx receives the router's share added in place."""
    H, E = w_router.shape
    dw = torch.empty((H, E), dtype=torch.float32, device=x.device)
    db = torch.empty((E,), dtype=torch.float32, device=x.device) if with_bias else None
    acc = dx is not None
    if dx is None:
        dx = torch.empty_like(x)
    ws = torch.empty(mok_router_workspace_bytes(sched.c.shape), dtype=torch.uint8, device=x.device)
    mok_router_backward(sched, x, w_router, topk_ids, topk_weights, d_topk_weights, dw, db, dx, acc, ws, stream)
    return dw, db, dx


class Layer:
    """Convenience owner of the workspace and forward context of one (shape, config) pair."""

    def __init__(self, T, H, I, E, K, cfg: mok_config | None = None, device="cuda"):
        self.shape = make_shape(T, H, I, E, K)
        self.cfg = cfg or make_config()
        self.ws = alloc_workspace(self.cfg, self.shape, device)
        self.ctx = alloc_fwd_ctx(self.cfg, self.shape, device)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.grads = Grads.empty(T, H, I, E, K, device)
        self.sched = None

    def schedule(self, topk_ids, topk_weights, stream=None) -> Schedule:
        self.sched = mok_build_schedule(self.cfg, self.shape, topk_ids, topk_weights, self.ws, stream)
        return self.sched

    def forward(self, x, weights: mok_weights, stream=None):
        return mok_forward(self.sched, x, weights, self.out, self.ctx, stream)

    def backward(self, dy, weights: mok_weights, stream=None) -> Grads:
        return mok_backward(self.sched, self.ctx, dy, weights, self.grads, stream)


def mok_kernel_name(kind: int) -> str:
    return _lib.mok_kernel_name(kind).decode()


def mok_set_trace(trace: "mok_trace | None"):
    _check(_lib.mok_set_trace(ctypes.byref(trace) if trace is not None else None), "mok_set_trace")


class Tracer:
    """Records a CUDA event pair around every kernel the library launches while active
    (``with Tracer(n) as tr: ...``), then reports per-launch device times in ms."""

    def __init__(self, capacity: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:
            e.record()  # creates the underlying cudaEvent_t
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self._kinds = (ctypes.c_int32 * capacity)()
        self.trace = mok_trace(self._handles, self._kinds, capacity, 0)

    def __enter__(self):
        self.trace.count = 0
        mok_set_trace(self.trace)
        return self

    def __exit__(self, *exc):
        mok_set_trace(None)
        return False

    def records(self):
        """[(kernel name, ms)] in launch order (synchronises)."""
        torch.cuda.synchronize()
        out = []
        for i in range(self.trace.count):
            out.append((mok_kernel_name(self._kinds[i]),
                        self.events[2 * i].elapsed_time(self.events[2 * i + 1])))
        return out
