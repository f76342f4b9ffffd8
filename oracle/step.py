"""Oracle: the ZeRO-DP partitioned mixed-precision AdamW step on the CPU.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path; its arithmetic lives in ``oracle/zero_oracle.c`` (plain C,
one binary32 rounding per operation, no FMA) and the layout in
``oracle/layout.py``.

The plain definition (what ZeRO reaches exactly): DDP — average the N_d
gradient replicas with an all-reduce, then mixed-precision AdamW on the fp32
master and a cast to the 16-bit parameters.  ZeRO-1/2/3 move the same values
through reduce-scatter, a sharded update and all-gathers, with the same
communication volume ("第 5 课：ZeRO 与 FSDP" §3; reading notes "ZeRO: Memory
Optimizations Toward Training Trillion Parameter Models" §6), and the updated
shard is what the next forward gathers ("ZeRO-3 核心流程" §2, step 4).  So this
module runs both forms:

  * :class:`DDPReference`  — all-reduce average over the full buffer, global
    norm, full AdamW, cast;
  * :class:`ZeroSimulation` — literal per-rank ZeRO-1/2/3: bucketed
    reduce-scatter in reverse bucket order, a sharding-aware norm that combines
    every rank's partial sums, per-rank AdamW on its shard, cast, all-gather
    (ZeRO-1/2) or per-unit forward/backward gathers into a transient buffer
    (ZeRO-3).

Step semantics (readings where the pages are silent; all listed in the design
notes):
  * reduce: s = x_0 + ... + x_{N_d-1} in rank order (binary32), g = s / D with
    D = binary32(N_d * loss_scale);
  * overflow: some s is inf/NaN.  Then the step is skipped: master/m/v/params
    unchanged, t not advanced, skipped += 1, the reported norm is +inf, and a
    dynamic loss scale halves (never below 1);
  * global norm: sqrt of the sum over all Psi_pad elements of g^2, with g^2
    exact in binary64, summed in binary64 within consecutive 128-element flat
    chunks, chunk sums added in flat order.  It must be global across shards
    ("ZeRO-3 核心流程", 坑 1: per-shard clipping silently diverges);
  * clip: c = min(1, max_norm / (norm + 1e-6)) in binary64, rounded to
    binary32; max_norm <= 0 disables clipping (c = 1);
  * AdamW: decoupled weight decay, constants computed in binary64 and rounded
    once to binary32 (beta^t by t repeated binary64 multiplications); see
    ``orc_adamw`` in zero_oracle.c for the per-element operation order;
  * cast: round to nearest even to bf16 / fp16 ("第 5 课" §3 step 2 casts the
    updated fp32 shard to BF16 in place);
  * growth: a dynamic loss scale doubles after ``growth_interval`` consecutive
    applied steps.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import build as _build
from .layout import Layout

FMT_BF16 = 0
FMT_FP16 = 1
CLIP_EPS = 1e-6


class _Consts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("decay", "beta1", "beta2", "omb1", "omb2", "eps", "step_size", "sqrt_bc2", "clip")]


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.orc_f32_to_bf16.argtypes = [f32]; L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_f16.argtypes = [f32]; L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_decode_array.argtypes = [i64, P, i32, P]; L.orc_decode_array.restype = None
        L.orc_cast_array.argtypes = [i64, P, i32, P]; L.orc_cast_array.restype = None
        L.orc_reduce.argtypes = [i32, P, i32, i64, f32, P, P]; L.orc_reduce.restype = None
        L.orc_sumsq_chunks128.argtypes = [P, i64, P]; L.orc_sumsq_chunks128.restype = None
        L.orc_sum_sequential.argtypes = [P, i64]; L.orc_sum_sequential.restype = ctypes.c_double
        L.orc_adamw.argtypes = [i64, P, P, P, P, ctypes.POINTER(_Consts)]; L.orc_adamw.restype = None
        L.orc_accumulate.argtypes = [i64, P, i32, P, i32]; L.orc_accumulate.restype = None
        L.orc_reduce_f32.argtypes = [i32, P, i64, f32, P, P]; L.orc_reduce_f32.restype = None
        L.orc_reduce_accumulate.argtypes = [i32, P, i32, i64, P, i32, f32, P]
        L.orc_reduce_accumulate.restype = None
        L.orc_num_threads.argtypes = []; L.orc_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]; L.orc_set_num_threads.restype = None
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------------------
# Elementwise primitives (thin wrappers over the plain C loops)
# ---------------------------------------------------------------------------

def decode16(h: np.ndarray, fmt: int) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_decode_array(h.size, _ptr(h), fmt, _ptr(out))
    return out


def cast16(x: np.ndarray, fmt: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_cast_array(x.size, _ptr(x), fmt, _ptr(out))
    return out


def reduce_grads(reps: Sequence[np.ndarray], fmt: int, D: float) -> Tuple[np.ndarray, bool]:
    """g[i] = (sum over ranks in rank order of decode(reps[r][i])) / D."""
    reps = [np.ascontiguousarray(r, dtype=np.uint16) for r in reps]
    n = reps[0].size
    assert all(r.size == n for r in reps)
    arr = (ctypes.c_void_p * len(reps))(*[_ptr(r) for r in reps])
    g = np.empty(n, np.float32)
    flag = ctypes.c_int32(0)
    lib().orc_reduce(len(reps), arr, fmt, n, float(np.float32(D)), _ptr(g), ctypes.byref(flag))
    return g, bool(flag.value)


def accumulate(x: np.ndarray, fmt: int, acc: np.ndarray, first: bool) -> None:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"] and acc.size == x.size
    lib().orc_accumulate(x.size, _ptr(x), fmt, _ptr(acc), int(first))


def reduce_f32(accs: Sequence[np.ndarray], D: float) -> Tuple[np.ndarray, bool]:
    accs = [np.ascontiguousarray(a, dtype=np.float32) for a in accs]
    n = accs[0].size
    arr = (ctypes.c_void_p * len(accs))(*[_ptr(a) for a in accs])
    g = np.empty(n, np.float32)
    flag = ctypes.c_int32(0)
    lib().orc_reduce_f32(len(accs), arr, n, float(np.float32(D)), _ptr(g), ctypes.byref(flag))
    return g, bool(flag.value)


def reduce_accumulate(reps: Sequence[np.ndarray], fmt: int, acc: np.ndarray, mode: int, D: float) -> bool:
    """mode 1: acc = s; 2: acc += s; 3: acc = (acc + s) / D.  Returns the
    non-finite flag (mode 3 only)."""
    reps = [np.ascontiguousarray(r, dtype=np.uint16) for r in reps]
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"] and acc.size == reps[0].size
    arr = (ctypes.c_void_p * len(reps))(*[_ptr(r) for r in reps])
    flag = ctypes.c_int32(0)
    lib().orc_reduce_accumulate(len(reps), arr, fmt, acc.size, _ptr(acc), mode, float(np.float32(D)),
                                ctypes.byref(flag))
    return bool(flag.value)


def sumsq_chunks(g: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float32)
    assert g.size % 128 == 0
    out = np.empty(g.size // 128, np.float64)
    lib().orc_sumsq_chunks128(_ptr(g), g.size, _ptr(out))
    return out


def sum_sequential(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return float(lib().orc_sum_sequential(_ptr(x), x.size))


# ---------------------------------------------------------------------------
# AdamW hyperparameters and per-step constants
# ---------------------------------------------------------------------------

@dataclass
class AdamWHP:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


def _f32(x: float) -> float:
    return float(np.float32(x))


def beta_pow(beta: float, t: int) -> float:
    """beta^t by t repeated binary64 multiplications."""
    p = 1.0
    for _ in range(t):
        p = p * beta
    return p


def adamw_consts(hp: AdamWHP, t: int, clip: float) -> _Consts:
    """Constants of step t (t >= 1), computed in binary64, rounded once."""
    return _Consts(decay=_f32(1.0 - hp.lr * hp.weight_decay), beta1=_f32(hp.beta1),
                   beta2=_f32(hp.beta2), omb1=_f32(1.0 - hp.beta1), omb2=_f32(1.0 - hp.beta2),
                   eps=_f32(hp.eps), step_size=_f32(hp.lr / (1.0 - beta_pow(hp.beta1, t))),
                   sqrt_bc2=_f32(math.sqrt(1.0 - beta_pow(hp.beta2, t))), clip=_f32(clip))


def adamw_inplace(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray,
                  hp: AdamWHP, t: int, clip: float) -> None:
    for a in (p, m, v, g):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    assert p.size == m.size == v.size == g.size
    k = adamw_consts(hp, t, clip)
    lib().orc_adamw(p.size, _ptr(p), _ptr(m), _ptr(v), _ptr(g), ctypes.byref(k))


# ---------------------------------------------------------------------------
# Step state: loss scale, step counter, skip decision, norm and clip
# ---------------------------------------------------------------------------

def norm_and_clip(sumsq: float, max_norm: float) -> Tuple[float, float]:
    """Global norm and clip coefficient from the global sum of squares.

    The norm is global across shards ("ZeRO-3 核心流程：把参数也切开的那一档",
    坑 1: every rank must clip with the same coefficient).  The coefficient
    follows the common global-norm clipping convention: c = max_norm /
    (norm + 1e-6) in binary64, clamped to at most 1, rounded once to
    binary32; max_norm <= 0 disables clipping (c = 1)."""
    norm = math.sqrt(sumsq)
    clip = _f32(min(1.0, max_norm / (norm + CLIP_EPS))) if max_norm > 0 else 1.0
    return norm, clip


@dataclass
class StepState:
    loss_scale: float = 1.0
    dynamic: bool = False
    growth_interval: int = 2000
    t: int = 0
    skipped: int = 0
    good: int = 0
    history: List[dict] = field(default_factory=list)

    def divisor(self, n_d: int) -> float:
        return _f32(n_d * self.loss_scale)

    def decide(self, nonfinite: bool, sumsq: float, max_norm: float,
               clip_override: Optional[float] = None) -> Tuple[bool, float, float]:
        """Returns (apply, norm, clip) and advances the state.  ``clip_override``
        (tests only) replaces the computed coefficient, to separate the norm's
        summation-order error from the update's arithmetic."""
        if nonfinite:
            norm, clip, apply = math.inf, 1.0, False
            self.skipped += 1
            self.good = 0
            if self.dynamic:
                self.loss_scale = max(1.0, self.loss_scale / 2.0)
        else:
            norm, clip = norm_and_clip(sumsq, max_norm)
            if clip_override is not None:
                clip = _f32(clip_override)
            apply = True
            self.t += 1
            self.good += 1
            if self.dynamic and self.good >= self.growth_interval:
                self.loss_scale = self.loss_scale * 2.0
                self.good = 0
        self.history.append({"overflow": int(nonfinite), "norm": norm, "clip": clip,
                             "t": self.t, "loss_scale": self.loss_scale})
        return apply, norm, clip


# ---------------------------------------------------------------------------
# The plain definition: DDP all-reduce + full AdamW
# ---------------------------------------------------------------------------

class DDPReference:
    """Every rank holds the full state; one all-reduce averages the grads."""

    def __init__(self, L: Layout, master0: np.ndarray, fmt: int, hp: AdamWHP,
                 max_norm: float = 0.0, loss_scale: float = 1.0, dynamic: bool = False,
                 growth_interval: int = 2000):
        assert master0.size == L.psi_pad
        self.L, self.fmt, self.hp, self.max_norm = L, fmt, hp, max_norm
        self.master = master0.astype(np.float32).copy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.params16 = cast16(self.master, fmt)
        self.state = StepState(loss_scale, dynamic, growth_interval)

    def step(self, reps: Sequence[np.ndarray]) -> dict:
        st = self.state
        g, bad = reduce_grads(reps, self.fmt, st.divisor(self.L.n_d))
        sumsq = sum_sequential(sumsq_chunks(g)) if not bad else math.inf
        apply, norm, clip = st.decide(bad, sumsq, self.max_norm)
        if apply:
            adamw_inplace(self.master, self.m, self.v, g, self.hp, st.t, clip)
            self.params16 = cast16(self.master, self.fmt)
        return dict(st.history[-1])


# ---------------------------------------------------------------------------
# Literal ZeRO-1/2/3 simulation with N_d ranks
# ---------------------------------------------------------------------------

class ZeroSimulation:
    """N_d simulated ranks, each with its own shard of master/m/v, its own
    reduced-gradient shard and its own 16-bit parameters (a full replica for
    ZeRO-1/2, a shard for ZeRO-3)."""

    def __init__(self, L: Layout, master0: np.ndarray, fmt: int, hp: AdamWHP,
                 max_norm: float = 0.0, loss_scale: float = 1.0, dynamic: bool = False,
                 growth_interval: int = 2000):
        assert L.stage in (1, 2, 3)
        assert master0.size == L.psi_pad
        self.L, self.fmt, self.hp, self.max_norm = L, fmt, hp, max_norm
        nd, S = L.n_d, L.shard_len
        # Rank r's shard = its slice of every unit, in unit order.
        self.master = [np.empty(S, np.float32) for _ in range(nd)]
        for r in range(nd):
            for u in L.units:
                lo = u.offset + r * u.shard
                self.master[r][u.shard_base:u.shard_base + u.shard] = master0[lo:lo + u.shard]
        self.m = [np.zeros(S, np.float32) for _ in range(nd)]
        self.v = [np.zeros(S, np.float32) for _ in range(nd)]
        self.gshard = [np.zeros(S, np.float32) for _ in range(nd)]
        p16 = [cast16(self.master[r], fmt) for r in range(nd)]
        if L.stage == 3:
            self.shard16 = p16
            self.params16 = None
        else:
            self.shard16 = None
            self.params16 = [np.empty(L.psi_pad, np.uint16) for _ in range(nd)]
            self._allgather(p16)
        self.state = StepState(loss_scale, dynamic, growth_interval)
        self.transients: List[Tuple[str, int, List[np.ndarray]]] = []
        self.record_transients = False

    @classmethod
    def from_flat(cls, L: Layout, master: np.ndarray, m: np.ndarray, v: np.ndarray, fmt: int, hp: AdamWHP,
                  state: StepState, max_norm: float = 0.0) -> "ZeroSimulation":
        """A simulation of layout L whose optimizer state is the given flat
        master/m/v (Psi_pad of L, zero padding) — what loading a sharded
        checkpoint into another layout must reach."""
        zs = cls(L, master, fmt, hp, max_norm=max_norm, loss_scale=state.loss_scale, dynamic=state.dynamic,
                 growth_interval=state.growth_interval)
        for name, flat in (("m", m), ("v", v)):
            dst = getattr(zs, name)
            for r in range(L.n_d):
                for u in L.units:
                    lo = u.offset + r * u.shard
                    dst[r][u.shard_base:u.shard_base + u.shard] = flat[lo:lo + u.shard]
        zs.state = StepState(state.loss_scale, state.dynamic, state.growth_interval, state.t, state.skipped,
                             state.good)
        return zs

    def flat_real(self, which: str) -> np.ndarray:
        """Concatenation of every tensor's values (no padding), in tensor order."""
        flat = self.flat(which)
        return np.concatenate([flat[o:o + n] for o, n in zip(self.L.tensor_offsets, self.L.numels)])

    # -- collectives ---------------------------------------------------------
    def _allgather(self, p16_shards: List[np.ndarray]) -> None:
        """All-gather (ZeRO-1/2): every rank's full replica receives every
        rank's updated 16-bit shard at that shard's flat position."""
        S = self.L.shard_len
        for dst in range(self.L.n_d):
            for src in range(self.L.n_d):
                self.params16[dst][src * S:(src + 1) * S] = p16_shards[src]

    def gather_unit(self, ui: int) -> List[np.ndarray]:
        """ZeRO-3 all-gather of unit ui into each rank's transient buffer:
        concatenate the ranks' 16-bit slices of the unit in rank order and
        drop the unit's tail padding."""
        u = self.L.units[ui]
        full = np.concatenate([self.shard16[r][u.shard_base:u.shard_base + u.shard]
                               for r in range(self.L.n_d)])
        return [full[:u.real].copy() for _ in range(self.L.n_d)]

    def _reduce_scatter(self, begin: int, end: int, reps, D: float) -> bool:
        """Reduce-scatter of flat range [begin, end): each owning rank
        receives the reduced values of its part of the range."""
        L, bad = self.L, False
        for u in L.units:
            lo_u, hi_u = u.offset, u.offset + u.padded
            for r in range(L.n_d):
                lo = max(begin, lo_u + r * u.shard)
                hi = min(end, lo_u + (r + 1) * u.shard)
                if lo >= hi:
                    continue
                g, b = reduce_grads([rep[lo:hi] for rep in reps], self.fmt, D)
                j0 = u.shard_base + (lo - lo_u - r * u.shard)
                self.gshard[r][j0:j0 + (hi - lo)] = g
                bad = bad or b
        return bad

    def _global_sumsq(self) -> float:
        """Sharding-aware norm: every rank contributes the 128-element chunk
        sums of its reduced-gradient shard; the sums are combined in flat
        order (rank slices of a unit are consecutive in the flat buffer)."""
        parts = []
        for u in self.L.units:
            for r in range(self.L.n_d):
                parts.append(sumsq_chunks(self.gshard[r][u.shard_base:u.shard_base + u.shard]))
        return sum_sequential(np.concatenate(parts))

    # -- one step --------------------------------------------------------------
    def step(self, reps: Sequence[np.ndarray], clip_override: Optional[float] = None) -> dict:
        L, st = self.L, self.state
        D = st.divisor(L.n_d)
        bad = False
        if L.stage == 3:
            if self.record_transients:
                self.transients = []
            for ui in range(len(L.units)):                  # forward gathers
                t = self.gather_unit(ui)
                if self.record_transients:
                    self.transients.append(("fwd", ui, t))
            for ui in reversed(range(len(L.units))):        # backward
                t = self.gather_unit(ui)
                if self.record_transients:
                    self.transients.append(("bwd", ui, t))
                u = L.units[ui]
                bad = self._reduce_scatter(u.offset, u.offset + u.padded, reps, D) or bad
        else:
            for (b0, b1) in reversed(L.buckets):           # last bucket first
                bad = self._reduce_scatter(b0, b1, reps, D) or bad
        sumsq = self._global_sumsq() if not bad else math.inf
        apply, norm, clip = st.decide(bad, sumsq, self.max_norm, clip_override)
        if apply:
            for r in range(L.n_d):
                adamw_inplace(self.master[r], self.m[r], self.v[r], self.gshard[r], self.hp, st.t, clip)
            p16 = [cast16(self.master[r], self.fmt) for r in range(L.n_d)]
            if L.stage == 3:
                self.shard16 = p16          # no all-gather at the end of the step
            else:
                self._allgather(p16)
        return dict(st.history[-1])

    # -- gradient accumulation over micro-batches ---------------------------------
    def step_accumulated(self, micro_reps: Sequence[Sequence[np.ndarray]], clip_override=None) -> dict:
        """One optimizer step over M micro-batches (micro_reps[m][r] = rank r's
        16-bit gradient replica of micro-batch m).  Readings of the reading
        notes §4.1-§4.3:
          ZeRO-1 keeps full fp32 accumulators and communicates nothing until
            the last micro-batch: A_r = x_{r,0} + x_{r,1} + ... (per rank),
            then g = (A_0 + A_1 + ...) / (N_d * M * loss_scale);
          ZeRO-2/3 reduce-scatter every micro-batch into the fp32 shard:
            acc = s_0 + s_1 + ... with s_m the rank-order sum of micro-batch
            m, then g = acc / (N_d * M * loss_scale);
          ZeRO-3 also gathers every unit forward and backward per micro-batch.
        M = 1 is the plain step."""
        L, st = self.L, self.state
        M = len(micro_reps)
        if M == 1:
            return self.step(micro_reps[0], clip_override)
        D = _f32(L.n_d * M * st.loss_scale)
        bad = False
        if L.stage == 1:
            accs = [np.empty(L.psi_pad, np.float32) for _ in range(L.n_d)]
            for m, reps in enumerate(micro_reps):
                for r in range(L.n_d):
                    accumulate(reps[r], self.fmt, accs[r], m == 0)
            for (b0, b1) in reversed(L.buckets):
                u = L.units[0]
                for r in range(L.n_d):
                    lo, hi = max(b0, r * u.shard), min(b1, (r + 1) * u.shard)
                    if lo >= hi:
                        continue
                    g, b = reduce_f32([a[lo:hi] for a in accs], D)
                    self.gshard[r][lo - r * u.shard:hi - r * u.shard] = g
                    bad = bad or b
        else:
            for m, reps in enumerate(micro_reps):
                mode = 1 if m == 0 else (3 if m == M - 1 else 2)
                if L.stage == 3:
                    for ui in range(len(L.units)):
                        self.gather_unit(ui)
                    units = list(reversed(range(len(L.units))))
                    ranges = [(L.units[ui].offset, L.units[ui].offset + L.units[ui].padded) for ui in units]
                else:
                    ranges = list(reversed(L.buckets))
                for (b0, b1) in ranges:
                    for u in L.units:
                        for r in range(L.n_d):
                            lo = max(b0, u.offset + r * u.shard)
                            hi = min(b1, u.offset + (r + 1) * u.shard)
                            if lo >= hi:
                                continue
                            j0 = u.shard_base + (lo - u.offset - r * u.shard)
                            acc = self.gshard[r][j0:j0 + (hi - lo)]
                            bad = reduce_accumulate([rep[lo:hi] for rep in reps], self.fmt, acc, mode, D) or bad
        sumsq = self._global_sumsq() if not bad else math.inf
        apply, norm, clip = st.decide(bad, sumsq, self.max_norm, clip_override)
        if apply:
            for r in range(L.n_d):
                adamw_inplace(self.master[r], self.m[r], self.v[r], self.gshard[r], self.hp, st.t, clip)
            p16 = [cast16(self.master[r], self.fmt) for r in range(L.n_d)]
            if L.stage == 3:
                self.shard16 = p16
            else:
                self._allgather(p16)
        return dict(st.history[-1])

    # -- views in flat order -----------------------------------------------------
    def flat(self, which: str) -> np.ndarray:
        """Reassemble master/m/v/gshard (fp32) or shard16 into flat order."""
        L = self.L
        src = {"master": self.master, "m": self.m, "v": self.v, "gshard": self.gshard,
               "shard16": self.shard16}[which]
        out = np.zeros(L.psi_pad, src[0].dtype)
        for u in L.units:
            for r in range(L.n_d):
                lo = u.offset + r * u.shard
                out[lo:lo + u.shard] = src[r][u.shard_base:u.shard_base + u.shard]
        return out


# ---------------------------------------------------------------------------
# Sampled form for buffers too large to simulate whole: every output element
# depends only on its own inputs plus the step's (apply, t, clip).
# ---------------------------------------------------------------------------

class SampledElements:
    """The oracle's per-element update restricted to a set of flat indices,
    driven by step decisions that the caller computes with
    :func:`full_sumsq_blocks` over the whole buffer."""

    def __init__(self, master0_sample: np.ndarray, fmt: int, hp: AdamWHP):
        self.master = master0_sample.astype(np.float32).copy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.fmt, self.hp = fmt, hp
        self.p16 = cast16(self.master, fmt)

    def step(self, rep_samples: Sequence[np.ndarray], D: float, apply: bool, t: int, clip: float) -> None:
        g, _ = reduce_grads(rep_samples, self.fmt, D)
        if apply:
            adamw_inplace(self.master, self.m, self.v, g, self.hp, t, clip)
            self.p16 = cast16(self.master, self.fmt)


class FullSumsq:
    """Accumulates the chunked sum of squares and the overflow flag of a full
    buffer fed block by block in flat order (block lengths multiples of 128)."""

    def __init__(self, fmt: int, D: float):
        self.fmt, self.D = fmt, D
        self.parts: List[np.ndarray] = []
        self.bad = False

    def add(self, rep_blocks: Sequence[np.ndarray]) -> None:
        g, b = reduce_grads(rep_blocks, self.fmt, self.D)
        self.bad = self.bad or b
        if not self.bad:
            self.parts.append(sumsq_chunks(g))

    def result(self) -> Tuple[bool, float]:
        if self.bad:
            return True, math.inf
        return False, sum_sequential(np.concatenate(self.parts))


def num_threads() -> int:
    return int(lib().orc_num_threads())
