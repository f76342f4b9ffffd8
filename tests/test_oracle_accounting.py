"""Oracle pins: memory formulas and communication volumes against the pages'
worked numbers (tests/golden/*.txt, each citing its page and section)."""
import os
from decimal import ROUND_HALF_UP, Decimal
from fractions import Fraction

import pytest

from oracle.layout import (comm_volume_elems, layout_comm_elems, layout_memory_bytes,
                           make_layout, memory_formula_bytes)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GB = Fraction(10 ** 9)


def _kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def _rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    return rows


def _gb(psi, n_d, stage, **kw):
    return memory_formula_bytes(psi, n_d, stage, **kw) / GB


def _printed(x: Fraction, decimals: int) -> float:
    """Decimal rounding half-up, as the pages print (26.25 -> 26.3)."""
    q = Decimal(x.numerator) / Decimal(x.denominator)
    return float(q.quantize(Decimal(1).scaleb(-decimals), rounding=ROUND_HALF_UP))


def test_7b_table_as_printed():
    # The page prints one decimal except 1.75; our exact values must print the same.
    for nd, z0, z1, z2, z3 in _rows("memory_7b_table.txt"):
        nd = int(nd)
        assert _printed(_gb(7 * 10 ** 9, nd, 0), 1) == z0
        assert _printed(_gb(7 * 10 ** 9, nd, 1), 1) == z1
        assert _printed(_gb(7 * 10 ** 9, nd, 2), 1) == z2
        dec = 2 if z3 == 1.75 else 1
        assert _printed(_gb(7 * 10 ** 9, nd, 3), dec) == z3


def test_7b_exact_verification_lines():
    kv = _kv("memory_7b_exact.txt")
    assert _gb(7 * 10 ** 9, 8, 1) == Fraction(kv["Z1_nd8"]).limit_denominator(1000)
    assert _gb(7 * 10 ** 9, 8, 2) == Fraction(kv["Z2_nd8"]).limit_denominator(1000)
    assert _gb(7 * 10 ** 9, 8, 3) == Fraction(kv["Z3_nd8"]).limit_denominator(1000)
    assert _gb(7 * 10 ** 9, 64, 3) == Fraction(kv["Z3_nd64"]).limit_denominator(1000)
    # bytes per parameter at N_d = 64, printed to two decimals
    assert _printed(memory_formula_bytes(1, 64, 1), 2) == kv["Z1_nd64_per_param_approx"]
    assert _printed(memory_formula_bytes(1, 64, 2), 2) == kv["Z2_nd64_per_param_approx"]


def test_7p5b_64gpu_figures():
    kv = _kv("memory_7p5b_64gpu.txt")
    psi = Fraction(75, 10) * 10 ** 9
    assert float(_gb(psi, 64, 0)) == kv["DDP"]
    assert _printed(_gb(psi, 64, 1), 1) == kv["Z1"]
    assert _printed(_gb(psi, 64, 2), 1) == kv["Z2"]
    assert _printed(_gb(psi, 64, 3), 1) == kv["Z3"]
    assert float(2 * psi / GB) == kv["params16"] == kv["grads16"]
    assert float(12 * psi / GB) == kv["optimizer"]


def test_7b_4gpu_figures_including_full_transient():
    kv = _kv("memory_7b_4gpu.txt")
    psi = 7 * 10 ** 9
    assert float(_gb(psi, 4, 0)) == kv["DDP"]
    assert float(_gb(psi, 4, 1)) == kv["Z1"]
    assert float(_gb(psi, 4, 2)) == kv["Z2"]
    assert float(_gb(psi, 4, 3)) == kv["Z3_static_4"]
    # That post counts a transient copy of ALL parameters (2 Psi) on top of the
    # ZeRO-3 static state: our peak formula with a single unit spanning the model.
    assert float(2 * Fraction(psi) / GB) == kv["transient_full_params"]
    for nd, key in ((4, "Z3_peak_4"), (8, "Z3_peak_8"), (16, "Z3_peak_16")):
        peak = memory_formula_bytes(psi, nd, 3) + 2 * psi
        assert float(peak / GB) == kv[key]
        # the layout's peak is the same sum on padded sizes: one unit = the model
        L = make_layout([psi], nd, 3, unit_of_tensor=[0])
        mem = layout_memory_bytes(L)
        assert mem["peak"] == memory_formula_bytes(L.psi_pad, nd, 3) + 2 * L.psi_pad
        assert 0 <= L.psi_pad - psi < nd * 128


def test_gpt2_1p5b_model_states():
    kv = _kv("model_states_gpt2_1p5b.txt")
    psi = Fraction(15, 10) * 10 ** 9
    assert float(_gb(psi, 1, 0)) == kv["total"]
    assert float(2 * psi / GB) == kv["params16"] == kv["grads16"]
    assert float(12 * psi / GB) == kv["optimizer"]
    assert float(4 * psi / GB) == kv["fused_fp32_1p5b"]
    assert float(4 * 3 * 10 ** 9 / GB) == kv["fused_fp32_3b"]


def test_dp1_all_stages_equal():
    # The exercise's own cross-check ("第 5 课" exercise): at dp = 1, Z1 = Z2 = Z3.
    for psi in (1, 10 ** 6, 7 * 10 ** 9, 12345):
        vals = {memory_formula_bytes(psi, 1, s) for s in (0, 1, 2, 3)}
        assert len(vals) == 1
        vals = {memory_formula_bytes(psi, 1, s, fp32_grad_accum=True) for s in (0, 1, 2, 3)}
        assert len(vals) == 1


def test_fp32_grad_accum_extras():
    psi, nd = 10 ** 9, 8
    d1 = memory_formula_bytes(psi, nd, 1, fp32_grad_accum=True) - memory_formula_bytes(psi, nd, 1)
    d2 = memory_formula_bytes(psi, nd, 2, fp32_grad_accum=True) - memory_formula_bytes(psi, nd, 2)
    d3 = memory_formula_bytes(psi, nd, 3, fp32_grad_accum=True) - memory_formula_bytes(psi, nd, 3)
    assert d1 == 4 * psi and d2 == Fraction(4 * psi, nd) and d3 == Fraction(4 * psi, nd)


def test_reduction_factors_limits():
    # Reading notes, "Optimizing Model State Memory": P_os gives a 4x reduction,
    # P_os+g 8x, P_os+g+p N_d x (limits as N_d grows).
    big = 10 ** 9
    assert abs(float(memory_formula_bytes(1, 1, 0) / memory_formula_bytes(1, big, 1)) - 4) < 1e-6
    assert abs(float(memory_formula_bytes(1, 1, 0) / memory_formula_bytes(1, big, 2)) - 8) < 1e-6
    for nd in (2, 8, 64):
        assert memory_formula_bytes(1, 1, 0) / memory_formula_bytes(1, nd, 3) == nd
    # "第 5 课" §1: 70B needs 1120 GB of static state per card under DDP.
    assert memory_formula_bytes(70 * 10 ** 9, 1024, 0) / GB == 1120


def test_comm_volume_forms_and_7b_numbers():
    kv = _kv("comm_7b.txt")
    psi = 7 * 10 ** 9
    for nd in (2, 8, 64, 1000):
        z12 = comm_volume_elems(psi, nd, 1)
        z3 = comm_volume_elems(psi, nd, 3)
        ddp = comm_volume_elems(psi, nd, 0)
        one = Fraction((nd - 1) * psi, nd)
        assert z12["reduce_scatter"] == z12["allgather"] == one
        # RS + AG moves exactly what one all-reduce moves
        assert z12["total"] == ddp["total"] == 2 * one
        assert comm_volume_elems(psi, nd, 2)["total"] == z12["total"]
        assert z3["total"] == 3 * one and z3["total"] / z12["total"] == Fraction(3, 2)
    # N_d -> infinity limits: 2 Psi = 14 G values, 3 Psi = 21 G values
    lim12 = comm_volume_elems(psi, 10 ** 12, 1)["total"] / 10 ** 9
    lim3 = comm_volume_elems(psi, 10 ** 12, 3)["total"] / 10 ** 9
    assert abs(float(lim12) - kv["z12_values_G"]) < 1e-6
    assert abs(float(lim3) - kv["z3_values_G"]) < 1e-6
    assert abs(float(2 * lim12) - kv["z12_bf16_GB"]) < 1e-6
    assert abs(float(2 * lim3) - kv["z3_bf16_GB"]) < 1e-6
    # a single rank communicates nothing
    assert comm_volume_elems(psi, 1, 3)["total"] == 0


def test_layout_counters_match_exact_forms():
    for nd in (1, 2, 3, 8):
        for stage in (1, 2, 3):
            L = make_layout([1000, 7, 300], nd, stage, unit_of_tensor=[0, 1, 1])
            c = layout_comm_elems(L)
            exact = comm_volume_elems(L.psi_pad, nd, stage)
            assert c["total"] == exact["total"]
            assert c["rs"] == exact["reduce_scatter"]


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_layout_memory_is_formula_on_padded_psi(stage):
    L = make_layout([513, 1000, 3], 4, stage, unit_of_tensor=[0, 0, 0])
    mem = layout_memory_bytes(L)
    assert mem["formula"] == memory_formula_bytes(L.psi_pad, 4, stage)
