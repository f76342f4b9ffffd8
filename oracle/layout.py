"""Oracle: flat-buffer layout, sharding, buckets, ZeRO-3 units, memory and
communication accounting — plain Python integers, no GPU, no numpy.

TEST INFRASTRUCTURE ONLY (tests, the smoke check and the CPU baseline leg of
the benchmark).  Shares no code with the CUDA path.

Sources (page title, then section):
  * Flatten the model's tensors into one contiguous buffer: "ZeRO: Memory
    Optimizations Toward Training Trillion Parameter Models" (reading notes),
    §2.2 "Temporary buffers" and §5.2 "C_B: Constant Size Buffers".
  * Equal 1/N_d split of the optimizer state, gradients and parameters:
    "第 5 课：ZeRO 与 FSDP", §2; the same reading notes, §4.1 P_os.
  * Buckets reduced as backward fills them, last layers first: the mlqm.cn
    data-parallel / ZeRO post, "DDP 的核心优化：梯度桶化"; reading notes §4.1,
    §4.2 ("按 Bucket 异步 ReduceScatter").
  * ZeRO-3 units, one per transformer block plus a root unit for embeddings
    and head: "別再複製本可分片的東西：ZeRO 與 FSDP", "FSDP：同樣的想法，以層為單位".
  * Memory formulas M0..M3 and the FP32-accumulation extras: "第 5 课" §2 and
    its exercise; reading notes §4.1–§4.3.
  * Communication volumes (N_d-1)/N_d * Psi per reduce-scatter / all-gather,
    2 Psi for ZeRO-1/2 and DDP, 3 Psi for ZeRO-3: "第 5 课" §3; reading notes §6.

Readings where the pages are silent (each listed in the design notes):
  * padding: the flat buffer (ZeRO-1/2) or each unit (ZeRO-3) is padded with
    zeros at its tail to a multiple of q = N_d * 128;
  * buckets: contiguous ranges of ``bucket_elems`` elements of the padded flat
    buffer, independent of shard boundaries; ZeRO-3 reduces per unit;
  * ZeRO-3 flat order: unit by unit (unit 0 first), tensors of a unit in
    declaration order; rank r owns slice [r*S_u, (r+1)*S_u) of each unit and
    its shard is the concatenation of those slices in unit order.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from fractions import Fraction
from typing import List, Optional, Sequence, Tuple

VECTOR_QUANTUM = 128  # q = N_d * 128


@dataclass
class Unit:
    """One contiguous, separately padded segment of the flat buffer.

    For ZeRO-1/2 there is exactly one segment: the whole buffer."""
    offset: int        # flat offset of the segment
    real: int          # real (unpadded) element count
    padded: int        # padded element count (multiple of q)
    shard: int         # S_u = padded / N_d
    shard_base: int    # offset of this segment's slice inside every rank's shard


@dataclass
class Layout:
    numels: List[int]
    n_d: int
    stage: int
    q: int
    bucket_elems: int
    psi: int                         # real parameter count
    psi_pad: int                     # padded flat length
    tensor_offsets: List[int]        # flat offset of every tensor
    units: List[Unit]
    shard_len: int                   # per-rank shard length (sum of S_u)
    buckets: List[Tuple[int, int]]   # [begin, end) flat ranges
    unit_of_tensor: Optional[List[int]] = None
    valid_mask_ranges: List[Tuple[int, int]] = field(default_factory=list)

    # ---- element ownership -------------------------------------------------
    def owner(self, i: int) -> Tuple[int, int]:
        """Flat index -> (rank, offset inside that rank's shard)."""
        for u in self.units:
            if u.offset <= i < u.offset + u.padded:
                k = i - u.offset
                r = k // u.shard
                return r, u.shard_base + (k - r * u.shard)
        raise IndexError(i)

    def flat_index(self, r: int, j: int) -> int:
        """(rank, shard offset) -> flat index (inverse of ``owner``)."""
        for u in self.units:
            if u.shard_base <= j < u.shard_base + u.shard:
                return u.offset + r * u.shard + (j - u.shard_base)
        raise IndexError((r, j))

    def is_pad(self, i: int) -> bool:
        for u in self.units:
            if u.offset <= i < u.offset + u.padded:
                return i >= u.offset + u.real
        raise IndexError(i)


def _round_up(x: int, m: int) -> int:
    return ((x + m - 1) // m) * m


def make_layout(numels: Sequence[int], n_d: int, stage: int,
                bucket_elems: int = 0, unit_of_tensor: Optional[Sequence[int]] = None,
                pad_multiple: int = 0) -> Layout:
    """Build the layout.  ``bucket_elems <= 0`` means one bucket for the whole
    buffer.  ``unit_of_tensor`` is required for stage 3 and ignored otherwise;
    for stage 3 it gives each tensor's unit id (units 0..U-1, none empty)."""
    numels = [int(x) for x in numels]
    if n_d <= 0 or stage not in (0, 1, 2, 3) or not numels or min(numels) <= 0:
        raise ValueError("bad layout arguments")
    q = pad_multiple if pad_multiple > 0 else n_d * VECTOR_QUANTUM
    if q % (n_d * VECTOR_QUANTUM) != 0:
        raise ValueError("pad_multiple must be a multiple of n_d*128")
    psi = sum(numels)
    tensor_offsets = [0] * len(numels)
    units: List[Unit] = []
    if stage == 3:
        if unit_of_tensor is None or len(unit_of_tensor) != len(numels):
            raise ValueError("stage 3 needs one unit id per tensor")
        n_units = max(unit_of_tensor) + 1
        members = [[t for t in range(len(numels)) if unit_of_tensor[t] == u]
                   for u in range(n_units)]
        if min(unit_of_tensor) < 0 or any(len(m) == 0 for m in members):
            raise ValueError("unit ids must cover 0..U-1 with no empty unit")
        off = 0
        base = 0
        for u in range(n_units):
            real = 0
            for t in members[u]:
                tensor_offsets[t] = off + real
                real += numels[t]
            padded = _round_up(real, q)
            units.append(Unit(off, real, padded, padded // n_d, base))
            off += padded
            base += padded // n_d
        psi_pad = off
    else:
        off = 0
        for t, n in enumerate(numels):
            tensor_offsets[t] = off
            off += n
        psi_pad = _round_up(psi, q)
        units.append(Unit(0, psi, psi_pad, psi_pad // n_d, 0))
    shard_len = sum(u.shard for u in units)
    if stage == 3:
        buckets = [(u.offset, u.offset + u.padded) for u in units]
    elif bucket_elems <= 0:
        buckets = [(0, psi_pad)]
    else:
        buckets = [(b, min(b + bucket_elems, psi_pad)) for b in range(0, psi_pad, bucket_elems)]
    return Layout(numels=numels, n_d=n_d, stage=stage, q=q, bucket_elems=bucket_elems,
                  psi=psi, psi_pad=psi_pad, tensor_offsets=tensor_offsets, units=units,
                  shard_len=shard_len, buckets=buckets,
                  unit_of_tensor=list(unit_of_tensor) if unit_of_tensor is not None else None,
                  valid_mask_ranges=[(u.offset, u.offset + u.real) for u in units])


# ---------------------------------------------------------------------------
# Memory accounting: "第 5 课：ZeRO 与 FSDP" §2 (M0..M3, k = 12) and the note on
# FP32 gradient accumulation; reading notes §4.1-§4.3.  Exact rationals.
# ---------------------------------------------------------------------------

def memory_formula_bytes(psi, n_d: int, stage: int, k: int = 12,
                         fp32_grad_accum: bool = False) -> Fraction:
    """Per-GPU static model-state bytes: the closed forms M0-M3 of "第 5 课：
    ZeRO 与 FSDP" §2 (also the reading notes §4.1-§4.3: P_os, P_os+g,
    P_os+g+p).  The three model-state terms are 16-bit parameters (2 Psi),
    16-bit gradients (2 Psi) and k bytes of optimizer state per parameter;
    stage s divides the last s of them by N_d:
      M0 = 2Psi + 2Psi + kPsi
      M1 = 2Psi + 2Psi + kPsi/N_d
      M2 = 2Psi + (2Psi + kPsi)/N_d
      M3 = (2Psi + 2Psi + kPsi)/N_d
    FP32 gradient accumulation (the same section's note) adds a full-size fp32
    buffer, 4Psi, while gradients are replicated (stages 0-1) and a 1/N_d
    share of it once they are partitioned (stages 2-3)."""
    psi = Fraction(psi)
    if psi <= 0 or n_d <= 0 or stage not in (0, 1, 2, 3):
        raise ValueError("bad arguments")
    terms = (2 * psi, 2 * psi, k * psi)          # parameters, gradients, optimizer state
    sharded = [i >= 3 - stage for i in range(3)]  # stage s partitions the last s terms
    total = sum((t / n_d if sh else t) for t, sh in zip(terms, sharded))
    if fp32_grad_accum:
        total += 4 * psi / n_d if sharded[1] else 4 * psi
    return total


def layout_memory_bytes(L: Layout) -> dict:
    """Per-rank bytes of this layout (integers, Psi_pad and S from the layout).
    ``formula``: M_stage with Psi -> Psi_pad (per-rank shard S for /N_d terms).
    ``state``: fp32 master + m + v shard (12 S).
    ``gshard``: the fp32 reduced-gradient shard (4 S) — the fused buffers are
    kept in fp32 (reading notes §2.2), so the build holds 4 S where the formula
    counts 2 S of 16-bit gradient.
    ``transient``: ZeRO-3 gathered unit buffer, 2 bytes x the largest padded
    unit, 0 for other stages; ``peak`` = formula + transient."""
    S, P = L.shard_len, L.psi_pad
    if L.stage == 0:
        formula = 16 * P
    elif L.stage == 1:
        formula = 4 * P + 12 * S
    elif L.stage == 2:
        formula = 2 * P + 14 * S
    else:
        formula = 16 * S
    transient = 2 * max(u.padded for u in L.units) if L.stage == 3 else 0
    return {"formula": formula, "state": 12 * S, "gshard": 4 * S,
            "transient": transient, "peak": formula + transient}


# ---------------------------------------------------------------------------
# Communication volume: "第 5 课" §3 and reading notes §6.  Elements moved per
# rank per step, exact (N_d - 1)/N_d forms.
# ---------------------------------------------------------------------------

def comm_volume_elems(psi, n_d: int, stage: int) -> dict:
    """Exact per-rank volumes for a flat buffer of ``psi`` elements (must be a
    multiple of n_d for integer results; any Fraction otherwise)."""
    psi = Fraction(psi)
    one = (n_d - 1) * psi / n_d        # one reduce-scatter or one all-gather
    if stage == 0:
        parts = {"allreduce": 2 * one}
    elif stage in (1, 2):
        parts = {"reduce_scatter": one, "allgather": one}
    elif stage == 3:
        parts = {"allgather_fwd": one, "allgather_bwd": one, "reduce_scatter": one}
    else:
        raise ValueError("stage must be 0..3")
    parts["total"] = sum(parts.values())
    return parts


def comm_volume_micro(psi, n_d: int, stage: int, n_micro: int) -> dict:
    """Per-rank volume of one optimizer step over n_micro micro-batches
    (reading notes §4.1-§4.3): ZeRO-1 needs no extra communication (one
    reduce-scatter and one all-gather per step); ZeRO-2 reduce-scatters every
    micro-batch; ZeRO-3 all-gathers forward and backward and reduce-scatters
    every micro-batch; DDP (stage 0) accumulates locally and all-reduces once."""
    one = comm_volume_elems(psi, n_d, stage)
    parts = {k: v for k, v in one.items() if k != "total"}
    if stage == 2:
        parts["reduce_scatter"] *= n_micro
    elif stage == 3:
        parts = {k: v * n_micro for k, v in parts.items()}
    parts["total"] = sum(parts.values())
    return parts


def layout_comm_elems(L: Layout) -> dict:
    """Integer per-rank counters for this layout: (N_d - 1) * S per collective."""
    one = (L.n_d - 1) * L.shard_len
    if L.stage == 0:
        return {"rs": 0, "ag": 0, "ag_fwd": 0, "ag_bwd": 0, "allreduce": 2 * one, "total": 2 * one}
    if L.stage in (1, 2):
        return {"rs": one, "ag": one, "ag_fwd": 0, "ag_bwd": 0, "allreduce": 0, "total": 2 * one}
    return {"rs": one, "ag": 0, "ag_fwd": one, "ag_bwd": one, "allreduce": 0, "total": 3 * one}
