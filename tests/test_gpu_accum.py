"""Gradient accumulation over micro-batches on the GPU against the oracle:
ZeRO-1 (local fp32 accumulators, one reduce-scatter), ZeRO-2 and ZeRO-3 (a
reduce-scatter into the fp32 shard every micro-batch), including an fp16 loss
scale with clipping and a generic rank count.  Bit-exact state."""
import numpy as np
import pytest
import torch

from oracle.step import AdamWHP, FMT_BF16, FMT_FP16, ZeroSimulation
from tests._cases import Case

pytestmark = pytest.mark.gpu
HP = AdamWHP()


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _run(c: Case, M: int, steps: int, use_gpu_clip: bool = False, live_units: int = 1):
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    L = c.layout()
    eng = ZeroStep(c.numels, c.n_d, c.stage, c.fmt, c.bucket_elems, c.units,
                   AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay), c.max_norm, c.loss_scale,
                   c.dynamic, c.growth_interval, n_micro=M, live_units=live_units, pad_multiple=c.pad_multiple)
    m0 = c.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, c.fmt, HP, max_norm=c.max_norm, loss_scale=c.loss_scale, dynamic=c.dynamic,
                        growth_interval=c.growth_interval)
    for s in range(1, steps + 1):
        ls = zs.state.loss_scale
        micro = []
        for m in range(M):
            reps = c.grads_torch(L, 100 * s + m, ls)
            micro.append([_u16(g) for g in reps])
            for r, g in enumerate(reps):
                eng.grads[r].copy_(g.cuda())
            eng.micro_step(m)
        g = eng.read_state()
        o = zs.step_accumulated(micro, clip_override=g["clip_coef"] if use_gpu_clip else None)
        assert (g["t"], g["overflow"], g["error"]) == (o["t"], o["overflow"], 0)
        assert g["loss_scale"] == o["loss_scale"]
        if not o["overflow"]:
            assert g["grad_norm"] == pytest.approx(o["norm"], rel=1e-5)
        for name in ("master", "m", "v"):
            assert np.array_equal(eng.flat(name).cpu().numpy().view(np.uint32),
                                  zs.flat(name).view(np.uint32)), (name, s)
        if c.stage == 3:
            assert np.array_equal(_u16(eng.flat("shard16")), zs.flat("shard16"))
        else:
            for r in range(c.n_d):
                assert np.array_equal(_u16(eng.params[r]), zs.params16[r])
    return eng


NUMELS = [120_000, 7, 50_001, 3000]


def test_zero1_local_accumulation():
    _run(Case(NUMELS, 4, 1, FMT_BF16, bucket_elems=32_768), M=3, steps=2)


def test_zero1_generic_rank_count():
    _run(Case(NUMELS, 3, 1, FMT_BF16, bucket_elems=65_536), M=2, steps=2)


def test_zero2_fp16_scaler_clip():
    c = Case(NUMELS, 8, 2, FMT_FP16, bucket_elems=32_768, max_norm=0.5, loss_scale=4096.0, dynamic=True,
             per_tensor_scale=True)
    _run(c, M=4, steps=2, use_gpu_clip=True)


def test_zero2_generic_rank_count():
    _run(Case(NUMELS, 5, 2, FMT_BF16, bucket_elems=32_768), M=2, steps=2)


@pytest.mark.parametrize("live", [1, 2])
def test_zero3_accumulation(live):
    _run(Case(NUMELS, 2, 3, FMT_BF16, units=[0, 1, 1, 2]), M=3, steps=2, live_units=live)


def test_micro_steps_are_traced_per_call():
    # zero_micro_step issues the accumulation's calls: ZeRO-1 accumulates every micro-batch and
    # reduce-scatters once per bucket; ZeRO-2 reduce-scatters every bucket every micro-batch
    from zero_partitioned_mixed_replica_gb300 import binding as B
    for stage, M in ((1, 3), (2, 3)):
        c = Case(NUMELS, 4, stage, FMT_BF16, bucket_elems=8192, max_norm=1.0)
        B.zero_trace_read(reset=True)
        prev = B.zero_trace_enable(True)
        try:
            eng = _run(c, M=M, steps=1)
        finally:
            B.zero_trace_enable(prev)
        t = B.zero_trace_read(reset=True)
        nb = eng.n_buckets
        if stage == 1:
            assert t["accumulate"]["launches"] == M and t["reduce_scatter"]["launches"] == nb
        else:
            assert "accumulate" not in t and t["reduce_scatter"]["launches"] == M * nb
        assert t["grad_norm"]["launches"] == 1 and t["adamw"]["launches"] == 1


def test_zero2_overflow_in_a_middle_micro_batch_skips_the_step():
    c = Case(NUMELS, 4, 2, FMT_FP16, bucket_elems=32_768, loss_scale=1024.0, dynamic=True,
             inf_step=201, inf_rank=2)            # step 2, micro-batch 1 (of 3)
    eng = _run(c, M=3, steps=3)
    st = eng.read_state()
    assert st["skipped"] == 1 and st["t"] == 2 and st["loss_scale"] == 512.0
