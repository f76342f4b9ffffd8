"""Oracle pins at step level: literal ZeRO-1/2/3 equals the DDP reference bit
for bit (same volume, same semantics: "第 5 课：ZeRO 与 FSDP" §3, reading notes
§6), bucket-size invariance, the fp16 overflow skip, the ZeRO-3 transients are
slices of the DDP parameters ("ZeRO-3 核心流程" §2: the updated shard is what the
next forward gathers), padding stays zero, and the loss-scale schedule."""
import numpy as np
import pytest

from oracle.step import FMT_BF16, FMT_FP16, AdamWHP, DDPReference, ZeroSimulation
from tests._cases import Case

HP = AdamWHP()


def _run(case: Case, steps: int, record=False):
    L = case.layout()
    m0 = case.master0(L)
    kw = dict(max_norm=case.max_norm, loss_scale=case.loss_scale, dynamic=case.dynamic,
              growth_interval=case.growth_interval)
    ddp = DDPReference(L, m0, case.fmt, HP, **kw)
    zs = ZeroSimulation(L, m0, case.fmt, HP, **kw)
    zs.record_transients = record
    hist = []
    for s in range(1, steps + 1):
        assert ddp.state.loss_scale == zs.state.loss_scale
        reps = case.grads(L, s, zs.state.loss_scale)
        a = ddp.step(reps)
        b = zs.step(reps)
        assert a == b
        hist.append(b)
        if record and L.stage == 3:
            for kind, ui, ts in zs.transients:
                u = L.units[ui]
                for t in ts:
                    # before this step's update the transients hold the previous params16
                    assert t.size == u.real
        yield L, ddp, zs, hist


def _assert_same(L, ddp, zs):
    for name in ("master", "m", "v"):
        assert np.array_equal(getattr(ddp, name).view(np.uint32), zs.flat(name).view(np.uint32)), name
    if L.stage == 3:
        assert np.array_equal(ddp.params16, zs.flat("shard16"))
    else:
        for r in range(L.n_d):
            assert np.array_equal(ddp.params16, zs.params16[r])


CASES = {
    "z1_bf16": Case([3000, 17, 5000, 1], 4, 1, FMT_BF16, bucket_elems=1024),
    "z2_bf16_clip": Case([3000, 17, 5000, 1], 3, 2, FMT_BF16, bucket_elems=640, max_norm=0.05),
    "z2_fp16_scaler": Case([4096, 100, 999], 8, 2, FMT_FP16, bucket_elems=2048, max_norm=1.0,
                           loss_scale=65536.0, dynamic=True, per_tensor_scale=True),
    "z3_bf16": Case([300, 2000, 64, 1500, 7], 2, 3, FMT_BF16, units=[0, 1, 1, 2, 0]),
    "z3_fp16_clip": Case([300, 2000, 64, 1500, 7], 5, 3, FMT_FP16, units=[0, 1, 1, 2, 0],
                         max_norm=0.01, loss_scale=1024.0, dynamic=True),
    "nd1": Case([1000, 24], 1, 2, FMT_BF16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_zero_equals_ddp_bitwise(name):
    for L, ddp, zs, hist in _run(CASES[name], 4):
        _assert_same(L, ddp, zs)
        # padding stays exactly zero everywhere
        pad = np.array([L.is_pad(i) for i in range(L.psi_pad)])
        for name_ in ("master", "m", "v"):
            assert not zs.flat(name_)[pad].any()


def test_clipping_is_active_in_the_clip_case():
    *_, (L, ddp, zs, hist) = _run(CASES["z2_bf16_clip"], 2)
    assert all(h["clip"] < 1.0 for h in hist)


def test_bucket_size_invariance():
    base = None
    for bucket in (0, 32, 96, 640, 4096):
        c = Case([3000, 17, 5000, 1], 4, 2, FMT_BF16, bucket_elems=bucket, max_norm=0.05)
        *_, (L, ddp, zs, hist) = _run(c, 3)
        state = [zs.flat(n).copy() for n in ("master", "m", "v")]
        if base is None:
            base = state
        else:
            for a, b in zip(base, state):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_stage1_equals_stage2_equals_stage3_numerically():
    outs = []
    for stage in (1, 2, 3):
        c = Case([3000, 17, 5000, 1], 4, stage, FMT_BF16, units=[0, 0, 0, 0], max_norm=0.05)
        *_, (L, ddp, zs, hist) = _run(c, 3)
        outs.append(ddp.master.copy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_fp16_overflow_skips_step_and_halves_scale():
    c = Case([4096, 100, 999], 4, 2, FMT_FP16, bucket_elems=1024, max_norm=1.0,
             loss_scale=65536.0, dynamic=True, per_tensor_scale=True, inf_step=4, inf_rank=3)
    snaps = {}
    for L, ddp, zs, hist in _run(c, 6):
        s = len(hist)
        snaps[s] = (zs.flat("master").copy(), zs.flat("m").copy(), zs.flat("v").copy(),
                    zs.params16[0].copy(), zs.state.t)
        _assert_same(L, ddp, zs)
    assert [h["overflow"] for h in hist] == [0, 0, 0, 1, 0, 0]
    assert [h["loss_scale"] for h in hist] == [65536.0] * 3 + [32768.0] * 3
    assert hist[3]["norm"] == float("inf")
    for a, b in zip(snaps[3][:4], snaps[4][:4]):
        assert np.array_equal(a, b)
    assert (snaps[3][4], snaps[4][4], snaps[5][4]) == (3, 3, 4)
    assert zs.state.skipped == 1
    assert not np.array_equal(snaps[5][0], snaps[4][0])


def test_dynamic_scale_growth():
    c = Case([2048], 2, 2, FMT_FP16, loss_scale=256.0, dynamic=True, growth_interval=2)
    *_, (L, ddp, zs, hist) = _run(c, 5)
    assert [h["loss_scale"] for h in hist] == [256.0, 512.0, 512.0, 1024.0, 1024.0]


def test_loss_scale_cancels_out():
    # grads drawn x loss_scale then divided by N_d*loss_scale: with scales that
    # keep every value exact, the update does not depend on the loss scale
    outs = []
    for ls in (1.0, 1024.0):
        c = Case([1024], 2, 2, FMT_FP16, grad_std=1e-2, loss_scale=ls)
        *_, (L, ddp, zs, hist) = _run(c, 2)
        outs.append(ddp.master.copy())
    # fp16 rounding of g*ls vs g differs only in subnormal/underflow tails
    assert np.allclose(outs[0], outs[1], rtol=0, atol=5e-6)


def test_zero3_transients_are_previous_parameters():
    c = CASES["z3_bf16"]
    L = c.layout()
    m0 = c.master0(L)
    ddp = DDPReference(L, m0, c.fmt, HP)
    zs = ZeroSimulation(L, m0, c.fmt, HP)
    zs.record_transients = True
    for s in range(1, 4):
        before = ddp.params16.copy()
        reps = c.grads(L, s, 1.0)
        ddp.step(reps)
        zs.step(reps)
        assert len(zs.transients) == 2 * len(L.units)
        kinds = [(k, ui) for k, ui, _ in zs.transients]
        U = len(L.units)
        assert kinds == [("fwd", u) for u in range(U)] + [("bwd", u) for u in reversed(range(U))]
        for kind, ui, ts in zs.transients:
            u = L.units[ui]
            for t in ts:
                assert np.array_equal(t, before[u.offset:u.offset + u.real])


def _random_case(seed: int) -> Case:
    rng = np.random.default_rng(5000 + seed)
    n_d = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    stage = int(rng.integers(1, 4))
    n_t = int(rng.integers(1, 6))
    numels = [int(x) for x in np.exp(rng.uniform(0.0, np.log(6000), n_t)).astype(np.int64) + 1]
    fmt = FMT_FP16 if rng.random() < 0.5 else FMT_BF16
    units = None
    if stage == 3:
        n_u = int(rng.integers(1, n_t + 1))
        units = list(range(n_u)) + [int(x) for x in rng.integers(0, n_u, n_t - n_u)]
        rng.shuffle(units)
    return Case(numels, n_d, stage, fmt, bucket_elems=0 if stage == 3 else 32 * int(rng.integers(1, 200)),
                units=units, max_norm=float(rng.choice([0.0, 1e-3, 10.0])),
                loss_scale=float(2.0 ** int(rng.integers(0, 12))) if fmt == FMT_FP16 else 1.0,
                dynamic=bool(rng.random() < 0.5), growth_interval=2, per_tensor_scale=bool(rng.random() < 0.5),
                inf_step=2 if rng.random() < 0.3 else None, inf_rank=int(rng.integers(0, n_d)),
                seed=int(rng.integers(1, 1 << 30)))


@pytest.mark.parametrize("seed", range(40))
def test_zero_equals_ddp_on_random_layouts(seed):
    # the literal per-rank simulation (shards, reverse-order buckets that straddle shards,
    # per-unit gathers, per-rank AdamW slices, all-gather) against the whole-buffer DDP
    # reference, over 4 steps, on random rank counts, stages, tensor sizes and units
    for L, ddp, zs, hist in _run(_random_case(seed), 4):
        _assert_same(L, ddp, zs)
