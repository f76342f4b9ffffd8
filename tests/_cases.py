"""Shared test-case builders: seeded inputs for a layout, drawn with the input
generator module on one device (the CPU here) and handed to both sides."""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

from oracle.layout import Layout, make_layout
from zero_partitioned_mixed_replica_gb300 import synth


@dataclass
class Case:
    numels: List[int]
    n_d: int
    stage: int
    fmt: int
    bucket_elems: int = 0
    units: Optional[List[int]] = None
    grad_std: float = 1e-3
    per_tensor_scale: bool = False
    max_norm: float = 0.0
    loss_scale: float = 1.0
    dynamic: bool = False
    growth_interval: int = 2000
    inf_step: Optional[int] = None
    inf_rank: int = 0
    seed: int = 1234
    pad_multiple: int = 0

    def layout(self) -> Layout:
        return make_layout(self.numels, self.n_d, self.stage, bucket_elems=self.bucket_elems,
                           unit_of_tensor=self.units, pad_multiple=self.pad_multiple)

    def master0(self, L: Layout) -> np.ndarray:
        return synth.master_init(L.numels, L.tensor_offsets, L.psi_pad, seed=self.seed).numpy()

    def scales(self):
        return synth.tensor_scales(len(self.numels), self.seed) if self.per_tensor_scale else None

    def grads_torch(self, L: Layout, step: int, loss_scale: float, device="cpu") -> List[torch.Tensor]:
        out = []
        for r in range(self.n_d):
            g = synth.grad_replica(L.numels, L.tensor_offsets, L.psi_pad, self.fmt, r, step,
                                   self.grad_std, self.scales(), loss_scale, self.seed, device)
            if self.inf_step == step and r == self.inf_rank:
                synth.plant_inf(g, L.psi // 2)
            out.append(g)
        return out

    def grads(self, L: Layout, step: int, loss_scale: float) -> List[np.ndarray]:
        return [synth.as_u16(g) for g in self.grads_torch(L, step, loss_scale)]
