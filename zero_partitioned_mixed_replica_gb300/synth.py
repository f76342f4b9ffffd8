"""Seeded synthetic inputs: fp32 master weights and per-rank 16-bit gradient
replicas, standing in for a model's initial weights and each data-parallel
rank's backward output.

This module holds none of the step's arithmetic.  It only draws numbers and
places them at flat offsets that the caller supplies (from whichever layout is
under test), so the oracle and the CUDA path consume the very same values: the
inputs are materialised once, on one device, and copied to the other.

Recipe (seed 1234 by default):
  * master: N(0, master_std) per real element, 0 in padding;
  * gradients of rank r at step s: N(0, grad_std) x (per-tensor scale drawn
    from U(0.1, 10) when the workload asks for it) x loss_scale, converted to
    the 16-bit format by torch, 0 in padding; a fresh stream per (seed, rank,
    step);
  * one +inf can be planted at a given flat index of one rank's replica.
Normal draws come from ``torch.randn`` with an explicit ``torch.Generator``;
values drawn on the CPU and on a GPU differ, which is why each test draws on
one device only.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

TORCH_16 = {0: torch.bfloat16, 1: torch.float16}

_SALT_MASTER = 0x6D61
_SALT_GRAD = 0x6772


def _stream_seed(seed: int, salt: int, rank: int = 0, step: int = 0) -> int:
    return (seed * 1_000_003 + salt * 65_537 + rank * 10_007 + step * 101) % (2 ** 63 - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def tensor_scales(n_tensors: int, seed: int = 1234) -> List[float]:
    """Per-tensor gradient scale factors, U(0.1, 10)."""
    rng = np.random.default_rng(seed)
    return [float(x) for x in rng.uniform(0.1, 10.0, size=n_tensors)]


def master_init(numels: Sequence[int], offsets: Sequence[int], psi_pad: int,
                std: float = 0.02, seed: int = 1234, device="cpu") -> torch.Tensor:
    out = torch.zeros(psi_pad, dtype=torch.float32, device=device)
    gen = _gen(device, _stream_seed(seed, _SALT_MASTER))
    for n, off in zip(numels, offsets):
        out[off:off + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32) * std
    return out


def grad_replica(numels: Sequence[int], offsets: Sequence[int], psi_pad: int, fmt: int,
                 rank: int, step: int, std: float, scales: Optional[Sequence[float]] = None,
                 loss_scale: float = 1.0, seed: int = 1234, device="cpu",
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Rank ``rank``'s 16-bit gradient replica for (1-based) step ``step``."""
    dt = TORCH_16[fmt]
    if out is None:
        out = torch.zeros(psi_pad, dtype=dt, device=device)
    else:
        if out.dtype != dt or out.numel() != psi_pad:
            raise ValueError("out must hold Psi_pad elements of the gradient dtype")
        out.zero_()
    gen = _gen(out.device, _stream_seed(seed, _SALT_GRAD, rank, step))
    for t, (n, off) in enumerate(zip(numels, offsets)):
        k = std * (scales[t] if scales is not None else 1.0) * loss_scale
        x = torch.randn(n, generator=gen, device=out.device, dtype=torch.float32)
        x.mul_(k)
        out[off:off + n] = x.to(dt)
        del x
    return out


def plant_inf(replica: torch.Tensor, index: int) -> None:
    replica[index] = float("inf")


def as_u16(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
