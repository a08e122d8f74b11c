"""Seeded synthetic workloads for the routed SwiGLU expert layer.

This module only draws random inputs; it holds none of the layer's arithmetic and imports
neither the CUDA library nor the oracle.  Both sides of every parity check take their inputs
from here.

Routing (logits -> top-k ids and weights) happens upstream of the layer: the layer's schedule
call receives the top-k expert ids and weights as inputs ("Mixture-of-Kittens (MoK)" project
card, "Functional API": ``build_schedule(workspace, config, topk_experts, ...)``).  The routers
below only shape the load distribution of each workload.

Draw order per workload (one torch generator, seed 0 unless stated): x, router draws, Wg, Wu,
Wd, dY.  Normal draws are fp32, scaled, then rounded to bf16 (round to nearest even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens (rows entering the layer)
    H: int            # hidden size
    I: int            # expert intermediate size
    E: int            # experts
    K: int            # top-k
    router: str       # "softmax", "softmax_bias", "gumbel_max", "gumbel_topk"
    zipf: float = 0.0
    precision: str = "bf16"
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.T * self.K

    def flops(self) -> float:
        """Algorithmic flops of one forward + backward: 18 * R * H * I."""
        return 18.0 * self.R * self.H * self.I


WORKLOADS = {
    # tiny layer, BF16 in / fp32 accumulation
    "tiny": Workload("tiny", 128, 256, 128, 8, 2, "softmax"),
    # near-uniform routing, the headline single-GPU shape
    "bf16_e64": Workload("bf16_e64", 4096, 2048, 1024, 64, 6, "softmax"),
    # DeepSeek-V3-style layer shape, every expert resident, mild per-expert bias
    "dsv3_e256": Workload("dsv3_e256", 2048, 7168, 2048, 256, 8, "softmax_bias"),
    # per-GPU shard of an EP64 layer: 2048 tokens x top-8 = 16384 routed rows onto 4 local experts
    "mxfp8_ep64_shard": Workload("mxfp8_ep64_shard", 16384, 7168, 2048, 4, 1, "gumbel_max", zipf=1.2,
                                 precision="mxfp8"),
    # the same shard with a quarter of the rows: a case small enough for multi-pass ncu captures
    "mxfp8_ep64_shard_4k": Workload("mxfp8_ep64_shard_4k", 4096, 7168, 2048, 4, 1, "gumbel_max", zipf=1.2,
                                    precision="mxfp8"),
    # imbalance / granularity sweep
    "sweep_zipf0": Workload("sweep_zipf0", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=0.0),
    "sweep_zipf1": Workload("sweep_zipf1", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=1.0),
    "sweep_zipf2": Workload("sweep_zipf2", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=2.0),
    # the sweep's layer shape and rows per expert (512 on average) with 2048 tokens, 16 experts and
    # top-4: a case small enough for multi-pass ncu captures (about 2 GB on the device)
    "sweep_zipf1_2k": Workload("sweep_zipf1_2k", 2048, 4096, 1536, 16, 4, "gumbel_topk", zipf=1.0),
    "sweep_zipf1_2k_mx": Workload("sweep_zipf1_2k_mx", 2048, 4096, 1536, 16, 4, "gumbel_topk", zipf=1.0,
                                  precision="mxfp8"),
    "sweep_zipf0_mx": Workload("sweep_zipf0_mx", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=0.0,
                               precision="mxfp8"),
    "sweep_zipf1_mx": Workload("sweep_zipf1_mx", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=1.0,
                               precision="mxfp8"),
    "sweep_zipf2_mx": Workload("sweep_zipf2_mx", 8192, 4096, 1536, 128, 8, "gumbel_topk", zipf=2.0,
                               precision="mxfp8"),
}


def custom(T, H, I, E, K, router="softmax", zipf=0.0, name="custom") -> Workload:
    return Workload(name, T, H, I, E, K, router, zipf)


def _normal(gen, shape, std, device):
    return (torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * std).to(torch.bfloat16)


def _topk_desc_low_id(p: torch.Tensor, k: int):
    """Top-k of each row by descending value; equal values keep the lower expert id first."""
    order = torch.sort(p, dim=1, descending=True, stable=True).indices[:, :k]
    return order, torch.gather(p, 1, order)


def make(w: Workload, seed: int = 0, weight_device: str = "cpu", with_dy: bool = True) -> dict:
    """Draw one workload.  Small tensors (x, routing, dY) are always drawn on the CPU; the expert
    weights are drawn on ``weight_device`` (a CUDA generator there, for sizes the CPU would take
    minutes to draw).  Returns torch tensors: x [T,H] bf16, topk_ids [T,K] int32, topk_weights
    [T,K] fp32, Wg/Wu [E,I,H] bf16, Wd [E,H,I] bf16, dY [T,H] bf16."""
    T, H, I, E, K = w.T, w.H, w.I, w.E, w.K
    g = torch.Generator().manual_seed(seed)
    x = _normal(g, (T, H), 1.0, "cpu")
    if w.router in ("softmax", "softmax_bias"):
        Wr = _normal(g, (H, E), 0.02, "cpu")
        logits = x.double() @ Wr.double()
        if w.router == "softmax_bias":
            bias = torch.randn((E,), generator=g, dtype=torch.float32) * 0.5
            logits = logits + bias.double()
        p = torch.softmax(logits, dim=1)
        ids, pk = _topk_desc_low_id(p, K)
        wts = (pk / pk.sum(dim=1, keepdim=True)).float()
    elif w.router == "gumbel_max":
        u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0 - 1e-16)
        prior = -w.zipf * torch.log(torch.arange(1, E + 1, dtype=torch.float64))
        logits = prior[None, :] - torch.log(-torch.log(u))
        ids, _ = _topk_desc_low_id(logits, K)
        wts = (0.05 + 0.25 * torch.rand((T, K), generator=g, dtype=torch.float32))
    elif w.router == "gumbel_topk":
        u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0 - 1e-16)
        prior = -w.zipf * torch.log(torch.arange(1, E + 1, dtype=torch.float64))
        logits = prior[None, :] - torch.log(-torch.log(u))
        ids, lk = _topk_desc_low_id(logits, K)
        wts = torch.softmax(lk, dim=1).float()
    else:
        raise ValueError(w.router)
    if weight_device == "cpu":
        gw = g
    else:
        gw = torch.Generator(device=weight_device).manual_seed(seed * 7919 + 1)
    Wg = _normal(gw, (E, I, H), 0.02, weight_device)
    Wu = _normal(gw, (E, I, H), 0.02, weight_device)
    Wd = _normal(gw, (E, H, I), 0.02, weight_device)
    out = dict(x=x, topk_ids=ids.to(torch.int32).contiguous(), topk_weights=wts.contiguous(), Wg=Wg, Wu=Wu, Wd=Wd)
    if w.router in ("softmax", "softmax_bias"):  # the router's own draws, for the router step
        out["Wr"] = Wr
        out["router_bias"] = bias if w.router == "softmax_bias" else None
    if with_dy:
        out["dY"] = _normal(g, (T, H), 1.0, "cpu")
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def load_stats(ids: torch.Tensor, E: int) -> dict:
    counts = torch.bincount(ids.reshape(-1).long(), minlength=E).double()
    return dict(max_over_mean=float(counts.max() / counts.mean()), min=int(counts.min()), max=int(counts.max()))
