"""The pins are sensitive: plausible mistakes planted in the oracle (on the
CPU, in a patched copy of its constants or its per-element update) make the
independent checks fail.  Each mutation is applied with monkeypatch and must
be caught by at least one of: the AdamW closed form under a constant
gradient, the binary64 evaluation of the formulas, torch.optim.AdamW at
N_d = 1, the exact-rational reduction bound."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.step as S
from oracle.step import FMT_BF16, AdamWHP, adamw_consts, cast16, decode16

U32 = 2.0 ** -24


def closed_form_ok() -> bool:
    hp = AdamWHP()
    g = np.array([1e-3, -2.5e-2, 3.0, -7e-6, 1e-8], np.float32)
    p = np.array([0.02, -0.01, 1.5, 0.0, 0.3], np.float32)
    p0, m, v = p.astype(np.float64), np.zeros_like(p), np.zeros_like(p)
    T = 20
    for t in range(1, T + 1):
        S.adamw_inplace(p, m, v, g, hp, t, 1.0)
    gd = g.astype(np.float64)
    d = 1.0 - hp.lr * hp.weight_decay
    u = hp.lr * gd / (np.abs(gd) + hp.eps)
    pT = d ** T * p0 - u * (1 - d ** T) / (1 - d)
    return bool(np.all(np.abs(p - pT) <= T * 8 * U32 * (np.abs(pT) + np.abs(u)) + 1e-12)) and \
        bool(np.allclose(m, (1 - hp.beta1 ** T) * gd, rtol=1e-5, atol=0))


def torch_ok() -> bool:
    rng = np.random.default_rng(5)
    n = 1024
    hp = AdamWHP()
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m, v = np.zeros_like(p), np.zeros_like(p)
    tp = torch.nn.Parameter(torch.from_numpy(p.copy()))
    opt = torch.optim.AdamW([tp], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False, fused=False)
    for t in range(1, 6):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        S.adamw_inplace(p, m, v, g, hp, t, 1.0)
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
    return bool(np.allclose(p, tp.detach().numpy(), rtol=1e-6, atol=40 * U32 * hp.lr))


def reduce_ok() -> bool:
    rng = np.random.default_rng(2)
    nd, n = 4, 300
    reps = [cast16((rng.standard_normal(n) * 1e-3 * (r + 1)).astype(np.float32), FMT_BF16) for r in range(nd)]
    g, _ = S.reduce_grads(reps, FMT_BF16, float(nd))
    xs = [decode16(r, FMT_BF16).astype(np.float64) for r in reps]
    gamma = (nd - 1) * U32 / (1 - (nd - 1) * U32)
    for i in range(n):
        exact = sum(Fraction(float(x[i])) for x in xs) / nd
        absum = sum(abs(float(x[i])) for x in xs) / nd
        if abs(Fraction(float(g[i])) - exact) > Fraction(gamma * absum) + Fraction(1, 2 ** 149):
            return False
    return True


def test_unmutated_oracle_passes_every_pin():
    assert closed_form_ok() and torch_ok() and reduce_ok()


def _consts_without_bias_correction(hp, t, clip):
    k = adamw_consts(hp, t, clip)
    k.step_size = np.float32(hp.lr)
    k.sqrt_bc2 = np.float32(1.0)
    return k


def _consts_wrong_decay(hp, t, clip):
    k = adamw_consts(hp, t, clip)
    k.decay = np.float32(1.0 - hp.weight_decay)          # forgot the lr factor
    return k


def _consts_swapped_betas(hp, t, clip):
    k = adamw_consts(hp, t, clip)
    k.beta1, k.beta2 = k.beta2, k.beta1
    k.omb1, k.omb2 = k.omb2, k.omb1
    return k


def _consts_eps_inside_sqrt(hp, t, clip):
    k = adamw_consts(hp, t, clip)
    k.eps = np.float32(math.sqrt(hp.eps))                 # eps applied to v instead of sqrt(v)
    return k


@pytest.mark.parametrize("mutant", [_consts_without_bias_correction, _consts_wrong_decay,
                                    _consts_swapped_betas, _consts_eps_inside_sqrt])
def test_adamw_mutations_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(S, "adamw_consts", mutant)
    assert not (closed_form_ok() and torch_ok())


def test_coupled_weight_decay_is_caught(monkeypatch):
    real = S.adamw_inplace

    def coupled(p, m, v, g, hp, t, clip):       # L2 penalty folded into the gradient
        g2 = (g + np.float32(hp.weight_decay) * p).astype(np.float32)
        hp0 = AdamWHP(hp.lr, hp.beta1, hp.beta2, hp.eps, 0.0)
        real(p, m, v, g2, hp0, t, clip)

    monkeypatch.setattr(S, "adamw_inplace", coupled)
    assert not (closed_form_ok() and torch_ok())


def test_reduction_mutations_are_caught(monkeypatch):
    real = S.reduce_grads

    def drop_last_rank(reps, fmt, D):
        return real(reps[:-1], fmt, D)

    def wrong_divisor(reps, fmt, D):
        return real(reps, fmt, D / len(reps))     # forgot to average over ranks

    for mutant in (drop_last_rank, wrong_divisor):
        monkeypatch.setattr(S, "reduce_grads", mutant)
        assert not reduce_ok()
        monkeypatch.setattr(S, "reduce_grads", real)
