"""Shared helpers of the test suite (no layer arithmetic lives here)."""
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerance of the BF16 path: max|gpu - oracle| / max|oracle| per output tensor.
TOL_BF16 = 2e-2
ALIGN = 256


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / den)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy() if t.dtype == torch.bfloat16 else \
        t.detach().cpu().double().numpy()


def ctx_views(ctx: torch.Tensor, rpad_max: int, H: int, I: int) -> dict:
    """Views of the forward context (gathered x, [g | u], a), laid out one after the other with
    256-byte alignment, as the library's header documents for mok_fwd_ctx_bytes."""
    def up(v):
        return (v + ALIGN - 1) // ALIGN * ALIGN
    b = ctx.view(torch.uint8)
    o_xg = 0
    o_gu = up(o_xg + rpad_max * H * 2)
    o_a = up(o_gu + rpad_max * 2 * I * 2)
    return dict(xg=b[o_xg:o_xg + rpad_max * H * 2].view(torch.bfloat16).view(rpad_max, H),
                gu=b[o_gu:o_gu + rpad_max * 2 * I * 2].view(torch.bfloat16).view(rpad_max, 2 * I),
                a=b[o_a:o_a + rpad_max * I * 2].view(torch.bfloat16).view(rpad_max, I))
