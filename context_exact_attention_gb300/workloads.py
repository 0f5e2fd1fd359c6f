"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random tensors and
describes shapes, so that the CUDA path and the fp64 oracle are fed the very
same values.  Inputs follow the verify script of the juejin ring-attention
debugging page (section 三, ``make_inputs``): a CPU ``torch.Generator`` seeded
once, ``randn`` drawn in the order q, k, v, layout [B, L, H, D]; the values are
then rounded to the compute dtype (round-to-nearest-even for bf16).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    H: int
    D: int
    P: int
    causal: bool
    dtype: torch.dtype = torch.bfloat16
    head_scale: bool = False       # per-head scale s_h ~ U[0.5, 2] on Q and K
    repeats: int = 1               # calls per step (e.g. denoising steps)
    ulysses: bool = False          # seq->head transpose, attention per head group, back
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def shard_len(self) -> int:
        return self.L // self.P


# The five workloads the library is specified against.
TINY = Workload("tiny ring check B1 H2 L256 D64 P4 fp32", 1, 256, 2, 64, 4, False,
                dtype=torch.float32)
DIT = Workload("diffusion-DiT full attention B1 H24 L4096 D128 P4 bf16 x40", 1, 4096, 24, 128, 4,
               False, repeats=40)
LM = Workload("causal LM B1 H32 L32768 D128 P8 bf16", 1, 32768, 32, 128, 8, True, head_scale=True)
ULYSSES = Workload("Ulysses B2 L8192 H32 D128 P8 bf16", 2, 8192, 32, 128, 8, False, ulysses=True)
LONG = Workload("long-context causal B1 H8 L131072 D128 P8 bf16", 1, 131072, 8, 128, 8, True)

ALL = {"tiny": TINY, "dit": DIT, "lm": LM, "ulysses": ULYSSES, "long": LONG}


def make_qkv(B: int, L: int, H: int, D: int, seed: int = 0, dtype=torch.bfloat16,
             head_scale: bool = False, device="cpu"):
    """Draw q, k, v ~ N(0, 1) of shape [B, L, H, D] from one seeded CPU generator.

    With ``head_scale`` one factor s_h ~ U[0.5, 2] per head is drawn after v and
    multiplies both q and k of head h (so score spread grows like s_h**2).
    """
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, H, D, generator=g)
    k = torch.randn(B, L, H, D, generator=g)
    v = torch.randn(B, L, H, D, generator=g)
    if head_scale:
        s = torch.rand(H, generator=g) * 1.5 + 0.5
        q = q * s.view(1, 1, H, 1)
        k = k * s.view(1, 1, H, 1)
    return tuple(t.to(dtype).to(device) for t in (q, k, v))


def make_workload_inputs(w: Workload, seed: int = 0, device="cpu"):
    return make_qkv(w.B, w.L, w.H, w.D, seed=seed, dtype=w.dtype, head_scale=w.head_scale,
                    device=device)


def sample_rows(L: int, P: int, n: int, seed: int = 1):
    """Query rows to check at full size: the first and last row of every shard,
    then distinct rows drawn uniformly (without replacement) from a second
    seeded generator, up to ``n`` rows in total, sorted."""
    Ls = L // P
    fixed = sorted({r * Ls for r in range(P)} | {r * Ls + Ls - 1 for r in range(P)})
    g = torch.Generator().manual_seed(seed)
    need = max(0, n - len(fixed))
    chosen = set(fixed)
    perm = torch.randperm(L, generator=g).tolist()
    for i in perm:
        if need == 0:
            break
        if i not in chosen:
            chosen.add(i)
            need -= 1
    return sorted(chosen)


def visible_pairs(L: int, causal: bool) -> int:
    """Number of (query, key) pairs that enter the softmax for one (batch, head)."""
    return L * (L + 1) // 2 if causal else L * L


def attention_flops(B: int, L: int, H: int, D: int, causal: bool) -> int:
    """Algorithmic forward FLOPs: 2*D for the score dot product plus 2*D for the
    weighted value sum, per visible pair (masked pairs and skipped blocks are not counted)."""
    return 4 * D * B * H * visible_pairs(L, causal)
