"""Pins of the oracle's sampled form (``SampledElements`` + ``FullSumsq`` +
``StepState``), which checks the full-size GPU runs at sampled indices: on
small layouts it must reproduce the whole-buffer ZeRO simulation bit for bit
at every sampled element and in every step decision.  The simulation itself is
pinned to DDP, the closed forms and torch.optim.AdamW by the other oracle
tests."""
import numpy as np
import pytest

from oracle.step import (AdamWHP, FMT_BF16, FMT_FP16, FullSumsq, SampledElements, StepState,
                         ZeroSimulation)
from tests._cases import Case

HP = AdamWHP()


def _sample(L, rng, n=600):
    idx = set(rng.choice(L.psi_pad, size=min(n, L.psi_pad), replace=False).tolist())
    for u in L.units:                                   # unit edges and the start of their padding
        for e in (u.offset, u.offset + u.real - 1, u.offset + u.real, u.offset + u.padded - 1):
            if 0 <= e < L.psi_pad:
                idx.add(e)
    return np.array(sorted(idx), dtype=np.int64)


CASES = [
    ("fp16 scaler, clip, overflow at step 3", Case([200_000, 1600, 99_999], 8, 2, FMT_FP16, bucket_elems=65_536,
                                                   max_norm=1.0, loss_scale=65536.0, dynamic=True,
                                                   growth_interval=2, per_tensor_scale=True, inf_step=3,
                                                   inf_rank=3)),
    ("bf16 ZeRO-1, no clip", Case([40_000, 33, 77_777, 5], 5, 1, FMT_BF16, bucket_elems=16_384)),
    ("bf16 ZeRO-3 units, clip", Case([30_000, 60_000, 640, 45_000, 7, 20_000, 3], 3, 3, FMT_BF16,
                                     units=[0, 1, 1, 2, 0, 3, 3], max_norm=0.05)),
]


@pytest.mark.parametrize("name,c", CASES, ids=[n for n, _ in CASES])
def test_sampled_form_reproduces_the_simulation(name, c):
    L = c.layout()
    m0 = c.master0(L)
    zs = ZeroSimulation(L, m0, c.fmt, HP, max_norm=c.max_norm, loss_scale=c.loss_scale, dynamic=c.dynamic,
                        growth_interval=c.growth_interval)
    idx = _sample(L, np.random.default_rng(7))
    samp = SampledElements(m0[idx], c.fmt, HP)
    st = StepState(c.loss_scale, c.dynamic, c.growth_interval)
    block = 128 * 97                                    # ragged last block, chunks of 128 kept whole
    for s in range(1, 6):
        reps = c.grads(L, s, st.loss_scale)
        D = st.divisor(c.n_d)
        acc = FullSumsq(c.fmt, D)
        for b in range(0, L.psi_pad, block):
            acc.add([r[b:b + block] for r in reps])
        bad, sumsq = acc.result()
        apply, norm, clip = st.decide(bad, sumsq, c.max_norm)
        samp.step([r[idx] for r in reps], D, apply, st.t, clip)
        o = zs.step(reps)
        assert (o["overflow"], o["t"], o["loss_scale"]) == (int(bad), st.t, st.loss_scale), s
        assert (o["norm"] == norm) or (np.isinf(o["norm"]) and np.isinf(norm)), s
        assert np.float32(o["clip"]) == np.float32(clip), s
        for which, got in (("master", samp.master), ("m", samp.m), ("v", samp.v)):
            assert np.array_equal(zs.flat(which)[idx].view(np.uint32), got.view(np.uint32)), (which, s)
        ref16 = zs.flat("shard16")[idx] if L.stage == 3 else zs.params16[0][idx]
        assert np.array_equal(ref16, samp.p16), s
    if c.inf_step:
        assert st.skipped == 1
