"""Seeded synthetic workloads shared by the tests, the benchmark and the oracle checks.

This module only *draws* inputs: it holds none of the attention, merge or layout arithmetic.
Everything is generated on the CPU with ``torch.Generator`` so that the GPU path and the CPU
oracle see exactly the same bits.

Workloads follow the shapes of the diffusion-transformer attention blocks discussed on
"Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with Multi-Device Inference
Support" (sections "Context parallelism for generative media", "Video generation with NVIDIA
Cosmos 3" -- 44,160 video tokens -- and "Image generation with Flux.1"); the pages' models and
prompts are not available, so N(0, 1) draws of those shapes stand in for them.

Recipe (per workload with index ``i``):
  * seed = 1000 + i; Q, K, V come from three generators seeded ``3*seed + {0, 1, 2}``;
  * each tensor is drawn fp32 N(0, 1) and then rounded to the storage dtype (round to nearest
    even) -- for ``tiny`` the storage dtype is bf16 on the device, and the raw fp32 draw is
    also kept for oracle self-checks;
  * ``stress``: Q is multiplied by 4 and a seeded 1 % of the sequence positions of K
    (floor(0.01 * S) positions, shared by all heads) by 8, in fp32 before rounding, which
    produces large-logit outliers for the merge;
  * ``ulysses``: Q, K, V are drawn directly in the sequence-sharded layout
    [P][B][S/P][H][D] that each context-parallel rank would hold.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Tuple

import torch

__all__ = ["Workload", "WORKLOADS", "draw_qkv", "draw_stress_outlier_rows", "draw_partials"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    S: int
    D: int
    dtype: torch.dtype          # storage dtype on the device
    P: Tuple[int, ...]          # KV-chunk counts (ring) or rank count (Ulysses)
    q_scale: float = 1.0
    k_outlier_frac: float = 0.0
    k_outlier_scale: float = 1.0
    seq_sharded: bool = False   # inputs drawn as [P][B][S/P][H][D]

    @property
    def seed(self) -> int:
        return 1000 + self.index

    def attention_flops(self) -> float:
        """Algorithmic flops of one non-causal forward: 4*B*H*Sq*Skv*D (two GEMMs)."""
        return 4.0 * self.B * self.H * self.S * self.S * self.D


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 0, B=1, H=2, S=256, D=64, dtype=torch.bfloat16, P=(4, 1)),
    "image": Workload("image", 1, B=1, H=24, S=4608, D=128, dtype=torch.bfloat16, P=(1, 2, 4, 8)),
    "video": Workload("video", 2, B=1, H=16, S=44160, D=128, dtype=torch.bfloat16, P=(8,)),
    "stress": Workload("stress", 3, B=1, H=16, S=32768, D=128, dtype=torch.bfloat16, P=(8,),
                       q_scale=4.0, k_outlier_frac=0.01, k_outlier_scale=8.0),
    "ulysses": Workload("ulysses", 4, B=2, H=32, S=16384, D=64, dtype=torch.float16, P=(8,),
                        seq_sharded=True),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def draw_stress_outlier_rows(S: int, frac: float, seed: int) -> torch.Tensor:
    """Sorted sequence positions whose K rows are scaled: floor(frac*S) of them, seeded."""
    n = int(frac * S)
    perm = torch.randperm(S, generator=_gen(3 * seed + 7))
    return torch.sort(perm[:n]).values


def draw_qkv(w: Workload, *, S: int | None = None, H: int | None = None, B: int | None = None,
             keep_fp32: bool = False):
    """Draw (q, k, v) for workload ``w`` (optionally with a smaller S, H or B, same recipe).

    Returns CPU tensors in the storage dtype with shape [B, H, S, D], or [P, B, S/P, H, D] for a
    sequence-sharded workload.  With ``keep_fp32`` also returns the raw fp32 draws.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    S = w.S if S is None else S
    D = w.D
    if w.seq_sharded:
        P = w.P[0]
        assert S % P == 0
        shape = (P, B, S // P, H, D)
    else:
        shape = (B, H, S, D)
    raw = []
    for t in range(3):
        x = torch.randn(shape, generator=_gen(3 * w.seed + t), dtype=torch.float32)
        raw.append(x)
    q, k, v = raw
    if w.q_scale != 1.0:
        q = q * w.q_scale
    if w.k_outlier_frac > 0.0:
        rows = draw_stress_outlier_rows(S, w.k_outlier_frac, w.seed)
        k = k.clone()
        k[:, :, rows, :] *= w.k_outlier_scale
    out = tuple(x.to(w.dtype) for x in (q, k, v))
    if keep_fp32:
        return out, (q, k, v)
    return out


def draw_partials(P: int, B: int, H: int, Sq: int, D: int, dtype: torch.dtype, seed: int,
                  lse_spread: float = 4.0):
    """Random per-chunk partials (O_parts [P,B,H,Sq,D], LSE_parts [P,B,H,Sq] fp32) for testing
    the merge in isolation.  LSE values are N(0, lse_spread^2) plus a per-chunk offset."""
    g = _gen(seed)
    o = torch.randn((P, B, H, Sq, D), generator=g, dtype=torch.float32).to(dtype)
    lse = torch.randn((P, B, H, Sq), generator=g, dtype=torch.float32) * lse_spread
    lse += torch.randn((P, 1, 1, 1), generator=g, dtype=torch.float32) * lse_spread
    return o, lse
