"""Oracle pins for the per-element arithmetic: the gradient reduction against
exact rational sums, AdamW against its closed form under a constant gradient
and against ``torch.optim.AdamW`` (N_d = 1), the float64 evaluation of the same
formulas within binary32 error bounds, and the global norm against closed
forms and exact sums."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.step import (FMT_BF16, FMT_FP16, AdamWHP, adamw_consts, adamw_inplace, cast16,
                         decode16, reduce_grads, sum_sequential, sumsq_chunks)

U32 = 2.0 ** -24


def _rand16(rng, n, fmt, scale):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    return cast16(x, fmt)


@pytest.mark.parametrize("fmt", [FMT_BF16, FMT_FP16])
@pytest.mark.parametrize("nd", [1, 2, 3, 5, 8])
def test_reduce_against_exact_rationals(fmt, nd):
    rng = np.random.default_rng(nd * 10 + fmt)
    n = 2000
    scale = 1e-3 if fmt == FMT_BF16 else 30.0
    reps = [_rand16(rng, n, fmt, scale * (1 + r)) for r in range(nd)]
    D = float(nd * (1 if fmt == FMT_BF16 else 65536))
    g, bad = reduce_grads(reps, fmt, D)
    assert not bad
    xs = [decode16(r, fmt).astype(np.float64) for r in reps]
    gamma = (nd - 1) * U32 / (1 - (nd - 1) * U32)
    for i in range(n):
        exact = sum(Fraction(float(x[i])) for x in xs) / Fraction(D)
        absum = sum(abs(float(x[i])) for x in xs) / D
        # sequential fp32 sum error bound, then an exact power-of-two division
        assert abs(Fraction(float(g[i])) - exact) <= Fraction(gamma * absum) + Fraction(1, 2 ** 149)


def test_reduce_single_rank_is_exact_division():
    rng = np.random.default_rng(3)
    h = _rand16(rng, 5000, FMT_FP16, 100.0)
    g, _ = reduce_grads([h], FMT_FP16, 65536.0)
    assert np.array_equal(g, decode16(h, FMT_FP16) / np.float32(65536.0))


def test_reduce_rank_order_matters_and_is_rank_order():
    # (big + small) - big loses `small`; big - big + small keeps it: sum is in rank order
    big, small = np.float32(2.0 ** 25), np.float32(1.0)
    reps = [cast16(np.array([big], np.float32), FMT_BF16),
            cast16(np.array([small], np.float32), FMT_BF16),
            cast16(np.array([-big], np.float32), FMT_BF16)]
    g, _ = reduce_grads(reps, FMT_BF16, 1.0)
    assert g[0] == 0.0
    g2, _ = reduce_grads([reps[0], reps[2], reps[1]], FMT_BF16, 1.0)
    assert g2[0] == 1.0


def test_nonfinite_detection():
    one = cast16(np.ones(4, np.float32), FMT_FP16)
    inf = one.copy(); inf[2] = 0x7C00
    nan = one.copy(); nan[1] = 0x7E00
    ninf = one.copy(); ninf[2] = 0xFC00
    assert not reduce_grads([one, one], FMT_FP16, 2.0)[1]
    assert reduce_grads([one, inf], FMT_FP16, 2.0)[1]
    assert reduce_grads([nan, one], FMT_FP16, 2.0)[1]
    g, bad = reduce_grads([inf, ninf], FMT_FP16, 2.0)
    assert bad and np.isnan(g[2])
    # finite bf16 inputs whose binary32 sum overflows also count as overflow
    mx = cast16(np.full(2, 3.0e38, np.float32), FMT_BF16)
    assert reduce_grads([mx, mx], FMT_BF16, 2.0)[1]


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------

def test_adamw_closed_form_constant_gradient():
    """With m0 = v0 = 0 and a constant gradient g, bias-corrected moments are
    m_hat = g and v_hat = g^2, so each step is p <- d*p - lr*g/(|g|+eps) and
    p_T = d^T p_0 - lr*g/(|g|+eps) * (1 - d^T)/(1 - d); also
    m_T = (1 - b1^T) g and v_T = (1 - b2^T) g^2."""
    hp = AdamWHP(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    g = np.array([1e-3, -2.5e-2, 3.0, -7e-6, 1e-8, -3e-9, 0.5, 1e-4], np.float32)
    p = np.array([0.02, -0.01, 1.5, 0.0, 0.3, -0.7, 0.0, 2.0], np.float32)
    p0, m, v = p.astype(np.float64), np.zeros_like(p), np.zeros_like(p)
    T = 60
    for t in range(1, T + 1):
        adamw_inplace(p, m, v, g, hp, t, 1.0)
    gd = g.astype(np.float64)
    d = 1.0 - hp.lr * hp.weight_decay
    u = hp.lr * gd / (np.abs(gd) + hp.eps)
    pT = d ** T * p0 - u * (1 - d ** T) / (1 - d)
    mT = (1 - hp.beta1 ** T) * gd
    vT = (1 - hp.beta2 ** T) * gd * gd
    # binary32 rounding accumulated over T steps (a few ulp of |p| + |u| per step)
    tol_p = T * 8 * U32 * (np.abs(pT) + np.abs(u)) + 1e-12
    assert np.all(np.abs(p - pT) <= tol_p), (p, pT)
    assert np.allclose(m, mT, rtol=T * 4 * U32 + 1e-6, atol=0)
    assert np.allclose(v, vT, rtol=T * 6 * U32 + 1e-6, atol=0)


def test_adamw_matches_float64_evaluation_within_fp32_bounds():
    rng = np.random.default_rng(11)
    n = 20000
    hp = AdamWHP()
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = (rng.random(n) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    t, clip = 7, 0.75
    k = adamw_consts(hp, t, clip)
    P, M, V, G = (a.astype(np.float64) for a in (p, m, v, g))
    G = G * k.clip
    P1 = P * k.decay
    M2 = k.beta1 * M + k.omb1 * G
    V2 = k.beta2 * V + k.omb2 * G * G
    den = np.sqrt(V2) / k.sqrt_bc2 + k.eps
    upd = k.step_size * (M2 / den)
    P2 = P1 - upd
    adamw_inplace(p, m, v, g, hp, t, clip)
    assert np.all(np.abs(m - M2) <= 4 * U32 * (k.beta1 * np.abs(M) + k.omb1 * np.abs(G)) + 1e-45)
    assert np.all(np.abs(v - V2) <= 5 * U32 * V2 + 1e-45)
    assert np.all(np.abs(p - P2) <= 12 * U32 * (np.abs(P1) + np.abs(upd)) + 1e-45)


def test_adamw_constants_definition():
    hp = AdamWHP(lr=3e-4, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1)
    k = adamw_consts(hp, 3, 1.0)
    assert k.step_size == pytest.approx(3e-4 / (1 - 0.8 ** 3), rel=1e-7)
    assert k.sqrt_bc2 == pytest.approx(math.sqrt(1 - 0.95 ** 3), rel=1e-7)
    assert k.decay == pytest.approx(1 - 3e-5, rel=1e-7)
    assert k.omb2 == pytest.approx(0.05, rel=1e-7)


def test_adamw_matches_torch_adamw_single_rank():
    """N_d = 1, no clip, no scaler: the step is plain mixed-precision AdamW on
    the fp32 master; torch.optim.AdamW (single-tensor path, fp32, CPU) is a
    library implementation of the same update (it forms m with lerp, so the
    comparison is within binary32 rounding, not bitwise)."""
    rng = np.random.default_rng(5)
    n = 4096
    hp = AdamWHP(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m, v = np.zeros_like(p), np.zeros_like(p)
    tp = torch.nn.Parameter(torch.from_numpy(p.copy()))
    opt = torch.optim.AdamW([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    for t in range(1, 11):
        h = cast16((rng.standard_normal(n) * 1e-3).astype(np.float32), FMT_BF16)
        g, _ = reduce_grads([h], FMT_BF16, 1.0)
        adamw_inplace(p, m, v, g, hp, t, 1.0)
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
    st = opt.state[tp]
    # absolute slack: a few binary32 ulps of the lr-sized update per step
    # (parameters that cancel to ~0 keep the update's absolute rounding)
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-6, atol=10 * 4 * U32 * hp.lr)
    # moments that cancel towards 0 keep the absolute rounding of the terms that
    # form them: (1-b1)|g| ~ 1e-4 for m and (1-b2) g^2 ~ 1e-9 for v, a few ulps
    # per step over 10 steps
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-5, atol=40 * U32 * 1e-4 * 4)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=40 * U32 * 1e-9 * 16)


def test_zero_state_and_zero_grad_keep_padding_zero():
    p = np.zeros(256, np.float32); m = np.zeros_like(p); v = np.zeros_like(p); g = np.zeros_like(p)
    for t in range(1, 6):
        adamw_inplace(p, m, v, g, AdamWHP(), t, 0.5)
    assert not p.any() and not m.any() and not v.any()
    assert not cast16(p, FMT_BF16).any()


# ---------------------------------------------------------------------------
# Norm
# ---------------------------------------------------------------------------

def test_norm_closed_form_constant_gradient():
    for a, psi, pad in ((1e-3, 1000, 24), (-0.37, 12345, 71), (3.0, 128 * 50, 0)):
        g = np.zeros(psi + pad, np.float32)
        g[:psi] = a
        norm = math.sqrt(sum_sequential(sumsq_chunks(g)))
        exact = abs(float(np.float32(a))) * math.sqrt(psi)
        assert norm == pytest.approx(exact, rel=1e-13)


def test_norm_matches_exact_sum_and_numpy():
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(128 * 777) * np.exp(rng.standard_normal(128 * 777) * 3)).astype(np.float32)
    s = sum_sequential(sumsq_chunks(g))
    exact = math.fsum(float(x) * float(x) for x in g.astype(np.float64))
    assert s == pytest.approx(exact, rel=1e-13)
    assert math.sqrt(s) == pytest.approx(float(np.linalg.norm(g.astype(np.float64))), rel=1e-13)


def test_clip_brings_norm_to_max_norm():
    # c = min(1, max_norm / (norm + 1e-6)): the clipped gradient's norm is max_norm
    rng = np.random.default_rng(2)
    g = (rng.standard_normal(128 * 40) * 0.1).astype(np.float32)
    norm = math.sqrt(sum_sequential(sumsq_chunks(g)))
    assert norm > 1.0
    c = float(np.float32(min(1.0, 1.0 / (norm + 1e-6))))
    gc = (g * np.float32(c)).astype(np.float64)
    assert float(np.linalg.norm(gc)) == pytest.approx(1.0, rel=2e-6)
