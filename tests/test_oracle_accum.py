"""Oracle pins for gradient accumulation over micro-batches: the averaged
gradient against exact rational sums within the sequential-summation bound
(both the ZeRO-1 order and the ZeRO-2/3 order), the orders really differ, the
per-micro-batch communication forms of the reading notes §4.1-§4.3, and the
FP32-accumulation memory extras of "第 5 课：ZeRO 与 FSDP" §2."""
from fractions import Fraction

import numpy as np
import pytest

from oracle.layout import comm_volume_elems, comm_volume_micro, make_layout, memory_formula_bytes
from oracle.step import FMT_BF16, FMT_FP16, AdamWHP, ZeroSimulation, cast16, decode16

U32 = 2.0 ** -24


def _reps(rng, n_micro, nd, n, fmt, scale):
    return [[cast16((rng.standard_normal(n) * scale * (1 + r + m)).astype(np.float32), fmt)
             for r in range(nd)] for m in range(n_micro)]


@pytest.mark.parametrize("stage", [1, 2, 3])
@pytest.mark.parametrize("nd,M", [(2, 3), (4, 2), (3, 5)])
def test_accumulated_gradient_within_exact_bound(stage, nd, M):
    rng = np.random.default_rng(stage * 100 + nd * 10 + M)
    numels = [700, 33]
    L = make_layout(numels, nd, stage, bucket_elems=256 if stage != 3 else 0,
                    unit_of_tensor=[0, 1] if stage == 3 else None)
    fmt, ls = FMT_FP16, 256.0
    reps = _reps(rng, M, nd, L.psi_pad, fmt, 0.5)
    for m in range(M):
        for r in range(nd):
            reps[m][r][L.psi:] = 0 if stage != 3 else reps[m][r][L.psi:]
    if stage == 3:   # zero every unit's padding
        for m in range(M):
            for r in range(nd):
                for u in L.units:
                    reps[m][r][u.offset + u.real:u.offset + u.padded] = 0
    zs = ZeroSimulation(L, np.zeros(L.psi_pad, np.float32), fmt, AdamWHP(), loss_scale=ls)
    zs.step_accumulated(reps)
    g = zs.flat("gshard")
    D = Fraction(nd * M) * Fraction(ls)
    k = nd * M
    gamma = (k - 1) * U32 / (1 - (k - 1) * U32)
    xs = [[decode16(reps[m][r], fmt).astype(np.float64) for r in range(nd)] for m in range(M)]
    for i in range(0, L.psi_pad, 7):
        exact = sum(Fraction(float(xs[m][r][i])) for m in range(M) for r in range(nd)) / D
        absum = sum(abs(float(xs[m][r][i])) for m in range(M) for r in range(nd)) / float(D)
        # summation error, then one rounding of the division (half an ulp of the result)
        bound = Fraction(gamma * absum) + Fraction(abs(float(exact)) * U32) + Fraction(1, 2 ** 149)
        assert abs(Fraction(float(g[i])) - exact) <= bound, i


def test_zero1_and_zero2_orders_differ():
    # two ranks, two micro-batches: ZeRO-1 sums each rank over micro-batches
    # first, ZeRO-2 sums ranks within each micro-batch first
    big, one = np.float32(2.0 ** 25), np.float32(1.0)
    vals = {(0, 0): big, (0, 1): one, (1, 0): -big, (1, 1): one}   # (micro, rank)
    outs = {}
    for stage in (1, 2):
        L = make_layout([128], 2, stage)
        reps = [[cast16(np.full(L.psi_pad, vals[(m, r)], np.float32), FMT_BF16) for r in range(2)]
                for m in range(2)]
        zs = ZeroSimulation(L, np.zeros(L.psi_pad, np.float32), FMT_BF16, AdamWHP())
        zs.step_accumulated(reps)
        outs[stage] = zs.flat("gshard")[0]
    # ZeRO-1 sums ranks' micro-batches first: (2^25 + -2^25) + (1 + 1) = 2 -> g = 2/4;
    # ZeRO-2 sums each micro-batch first: (2^25 + 1 -> 2^25) + (-2^25 + 1 -> -2^25) = 0
    assert outs[1] == np.float32(2.0 / 4) and outs[2] == 0.0


def test_single_micro_batch_is_the_plain_step():
    rng = np.random.default_rng(1)
    L = make_layout([1000], 4, 2, bucket_elems=512)
    reps = _reps(rng, 1, 4, L.psi_pad, FMT_BF16, 1e-3)
    for r in range(4):
        reps[0][r][L.psi:] = 0
    m0 = (rng.standard_normal(L.psi_pad) * 0.02).astype(np.float32)
    m0[L.psi:] = 0
    a = ZeroSimulation(L, m0, FMT_BF16, AdamWHP())
    b = ZeroSimulation(L, m0, FMT_BF16, AdamWHP())
    a.step_accumulated(reps)
    b.step(reps[0])
    assert np.array_equal(a.flat("master"), b.flat("master"))


def test_micro_batch_communication_forms():
    psi, nd = 7 * 10 ** 9, 8
    for M in (1, 2, 4):
        z1, z2, z3 = (comm_volume_micro(psi, nd, s, M) for s in (1, 2, 3))
        one = comm_volume_elems(psi, nd, 1)["reduce_scatter"]
        assert z1["total"] == 2 * one                    # ZeRO-1: no extra communication
        assert z2["total"] == (M + 1) * one              # ZeRO-2: a reduce-scatter per micro-batch
        assert z3["total"] == 3 * M * one                # ZeRO-3: AG + AG + RS per micro-batch
        assert comm_volume_micro(psi, nd, 0, M)["total"] == 2 * one


def test_fp32_accumulation_memory_extras():
    psi, nd = 10 ** 9, 8
    assert memory_formula_bytes(psi, nd, 1, fp32_grad_accum=True) - memory_formula_bytes(psi, nd, 1) == 4 * psi
    assert memory_formula_bytes(psi, nd, 2, fp32_grad_accum=True) - memory_formula_bytes(psi, nd, 2) == \
        Fraction(4 * psi, nd)


def test_zero3_accumulation_equals_zero2():
    rng = np.random.default_rng(4)
    numels = [600, 40]
    L2 = make_layout(numels, 2, 2)
    L3 = make_layout(numels, 2, 3, unit_of_tensor=[0, 0])
    assert L2.psi_pad == L3.psi_pad
    reps = _reps(rng, 3, 2, L2.psi_pad, FMT_BF16, 1e-3)
    for m in range(3):
        for r in range(2):
            reps[m][r][L2.psi:] = 0
    m0 = np.zeros(L2.psi_pad, np.float32)
    a = ZeroSimulation(L2, m0, FMT_BF16, AdamWHP())
    b = ZeroSimulation(L3, m0, FMT_BF16, AdamWHP())
    a.step_accumulated(reps)
    b.step_accumulated(reps)
    assert np.array_equal(a.flat("master"), b.flat("master"))
