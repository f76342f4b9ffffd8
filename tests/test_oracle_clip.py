"""Pins of the oracle's clip coefficient (``StepState.decide`` through
``norm_and_clip``) against a library routine that implements the same global-
norm clipping convention: ``torch.nn.utils.clip_grad_norm_`` on CPU binary64
tensors, which scales every gradient by min(1, max_norm / (total_norm + 1e-6)).

The page basis is "ZeRO-3 核心流程：把参数也切开的那一档", 坑 1: the clip
coefficient is computed from the global norm over all shards and is the same
on every rank.  The 1e-6 and the clamp to 1 are the common convention that
the oracle adopts; max_norm <= 0 means "no clipping" (DeepSpeed's
gradient_clipping = 0), where the torch routine would zero the gradients
instead, so that case is checked against its definition.

The torch coefficient is read back exactly: every case has a gradient element
that is a power of two, and scaling a power of two is exact in binary64.
Planted mistakes (a dropped clamp, the 1e-6 moved inside the square root, the
1e-6 dropped, the squared norm used in place of the norm) each fail the pin.
"""
import math

import numpy as np
import pytest
import torch

import oracle.step as S
from oracle.step import StepState, sum_sequential, sumsq_chunks


def _torch_coef(grads64, max_norm: float, probe: tuple) -> float:
    """Scale factor that clip_grad_norm_ applied, read at a power-of-two
    gradient element probe = (tensor index, element index)."""
    params = []
    for g in grads64:
        p = torch.nn.Parameter(torch.zeros(g.shape, dtype=torch.float64))
        p.grad = torch.from_numpy(g.copy())
        params.append(p)
    torch.nn.utils.clip_grad_norm_(params, max_norm, norm_type=2.0, foreach=False)
    ti, ei = probe
    before = float(grads64[ti].reshape(-1)[ei])
    after = float(params[ti].grad.reshape(-1)[ei])
    m, e = math.frexp(before)
    assert m in (0.5, -0.5), "probe must be a power of two"
    return after / before


def _oracle_coef(flat32: np.ndarray, max_norm: float):
    """decide() on the oracle's own binary64 sum of squares of the gradient."""
    n = flat32.size
    padded = np.zeros((n + 127) // 128 * 128, np.float32)
    padded[:n] = flat32
    sumsq = sum_sequential(sumsq_chunks(padded))
    st = StepState()
    apply, norm, clip = st.decide(False, sumsq, max_norm)
    assert apply and st.t == 1
    return norm, clip


def _cases():
    """(gradient tensors as float32 arrays, probe, max_norm, expect_exact)."""
    out = []
    # 3-4-5 gradients: the norm 5a is exact in every summation order
    for a_exp in (-3, -20, 10, 0):
        a = 2.0 ** a_exp
        g = [np.array([3 * a], np.float32), np.array([4 * a], np.float32)]
        norm = 5 * a
        for max_norm in (2 * norm, norm * 1.000001, norm, 0.5 * norm, 1e-6, 1.0, 1e-3, 37.0):
            out.append((g, (1, 0), max_norm, True))
    # random multi-tensor gradients with per-tensor scales, one power-of-two probe
    rng = np.random.default_rng(11)
    for k, n_t in enumerate((1, 3, 7)):
        g = [(rng.standard_normal(int(rng.integers(1, 3000))) * 10.0 ** rng.uniform(-4, 1)).astype(np.float32)
             for _ in range(n_t)]
        g[0][0] = np.float32(2.0 ** -9)
        flat = np.concatenate(g).astype(np.float64)
        norm = float(np.linalg.norm(flat))
        for max_norm in (norm * 4, norm * 0.25, norm * 0.999999, 1e-5):
            out.append((g, (0, 0), max_norm, False))
    return out


def clip_pin_ok() -> bool:
    for g32, probe, max_norm, exact in _cases():
        norm, c = _oracle_coef(np.concatenate(g32), max_norm)
        ct = float(np.float32(_torch_coef([x.astype(np.float64) for x in g32], max_norm, probe)))
        if exact:
            if c != ct:
                return False
        else:
            # torch sums the squares in another order: the binary64 norms differ in the last
            # bits, so the binary32 coefficients may differ by one rounding at most
            if abs(c - ct) > 2.0 ** -23 * abs(ct):
                return False
        if c > 1.0:
            return False
    return True


def test_clip_coefficient_matches_clip_grad_norm():
    assert clip_pin_ok()


def test_clip_clamp_branch_is_exactly_one():
    # max_norm above the norm: c is exactly 1.0 (no scaling); torch leaves the gradient as is
    g = [np.array([3.0], np.float32), np.array([4.0], np.float32)]
    for max_norm in (5.0 * 1.0001, 6.0, 1e6):
        _, c = _oracle_coef(np.concatenate(g), max_norm)
        assert c == 1.0
        assert _torch_coef([x.astype(np.float64) for x in g], max_norm, (1, 0)) == 1.0


def test_clip_at_max_norm_equal_to_norm_is_below_one():
    # norm == max_norm: the 1e-6 makes c = 5 / 5.000001 < 1, one binary32 step below 1 or more
    g = np.array([3.0, 4.0], np.float32)
    _, c = _oracle_coef(g, 5.0)
    assert c == float(np.float32(5.0 / 5.000001)) and c < 1.0


def test_zero_gradient_and_tiny_max_norm():
    # ||g|| = 0: c = min(1, max_norm / 1e-6); both conventions agree
    g = [np.zeros(5, np.float32), np.array([0.0], np.float32)]
    _, c = _oracle_coef(np.concatenate(g), 1e-7)
    assert c == float(np.float32(0.1))
    _, c = _oracle_coef(np.concatenate(g), 1.0)
    assert c == 1.0


@pytest.mark.parametrize("max_norm", [0.0, -1.0])
def test_non_positive_max_norm_disables_clipping(max_norm):
    _, c = _oracle_coef(np.array([3e3, 4e3], np.float32), max_norm)
    assert c == 1.0


def test_overflow_reports_inf_norm_and_no_clip():
    st = StepState(loss_scale=1024.0, dynamic=True)
    apply, norm, clip = st.decide(True, math.inf, 1.0)
    assert not apply and math.isinf(norm) and clip == 1.0
    assert st.t == 0 and st.skipped == 1 and st.loss_scale == 512.0


# ---- planted mistakes: each must fail the pin --------------------------------------------

def _no_clamp(sumsq, max_norm):
    norm = math.sqrt(sumsq)
    return norm, (S._f32(max_norm / (norm + S.CLIP_EPS)) if max_norm > 0 else 1.0)


def _eps_inside_sqrt(sumsq, max_norm):
    norm = math.sqrt(sumsq)
    return norm, (S._f32(min(1.0, max_norm / math.sqrt(sumsq + S.CLIP_EPS))) if max_norm > 0 else 1.0)


def _no_eps(sumsq, max_norm):
    norm = math.sqrt(sumsq)
    return norm, (S._f32(min(1.0, max_norm / norm)) if max_norm > 0 and norm > 0 else 1.0)


def _squared_norm(sumsq, max_norm):
    return math.sqrt(sumsq), (S._f32(min(1.0, max_norm / (sumsq + S.CLIP_EPS))) if max_norm > 0 else 1.0)


@pytest.mark.parametrize("mutant", [_no_clamp, _eps_inside_sqrt, _no_eps, _squared_norm])
def test_clip_mutations_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(S, "norm_and_clip", mutant)
    assert not clip_pin_ok()
