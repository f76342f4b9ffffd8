"""Steps whose gradient replicas come from pinned host memory, through the
library's zero_step_from_host (``ZeroStep.step_from_host``): per-bucket
(ZeRO-3: per-unit) copies on the library's two copy streams, each
reduce-scatter or fused update ordered after its own range only, and the
step state copied back to host memory inside the call.  Checked against the
oracle bit for bit, on layouts whose buckets straddle shards, with chunks
smaller than a bucket, and against the device-resident step; steps queued
back to back with overlap_previous, and the cases that must turn it off."""
import numpy as np
import pytest
import torch

from oracle.step import FMT_BF16, FMT_FP16, ZeroSimulation
from tests._cases import Case
from tests.test_gpu_parity import HP, Z3_NUMELS, Z3_UNITS, _engine, _u16, run_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def test_host_input_zero2_fp16_scaler_overflow():
    c = Case([200_000, 1600, 99_999], 8, 2, FMT_FP16, bucket_elems=65_536, max_norm=1.0,
             loss_scale=65536.0, dynamic=True, per_tensor_scale=True, inf_step=2, inf_rank=3)
    _, _, hist = run_parity(c, 3, use_gpu_clip=True, host_input=40_000)   # chunks smaller than a bucket
    assert [g["overflow"] for g, _ in hist] == [0, 1, 0]


def test_host_input_zero1_fused_per_bucket():
    c = Case([40_000, 33, 77_777, 5], 5, 1, FMT_BF16, bucket_elems=16_384, per_tensor_scale=True)
    run_parity(c, 2, host_input=True, per_bucket=False)   # one fused launch after every bucket's copies
    run_parity(c, 2, host_input=True, per_bucket=True)


def test_host_input_garbage_padding():
    c = Case([100_001, 3], 3, 1, FMT_BF16)
    run_parity(c, 2, garbage_pads=True, host_input=True)


@pytest.mark.parametrize("fused,live", [(True, 1), (False, 1), (True, 2), (False, 2)])
def test_host_input_zero3(fused, live):
    c = Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS, max_norm=0.0 if fused else 0.05)
    run_parity(c, 2, host_input=10_000, use_gpu_clip=not fused, live_units=live)


def test_host_input_equals_device_step():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    e1, _, _ = run_parity(c, 2, use_gpu_clip=True, host_input=True)
    e2, _, _ = run_parity(c, 2, use_gpu_clip=True)
    assert torch.equal(e1.master, e2.master) and torch.equal(e1.params, e2.params)
    assert torch.equal(e1.m, e2.m) and torch.equal(e1.v, e2.v)


def test_host_state_read_back_in_the_call():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_FP16, bucket_elems=32_768, max_norm=1.0, loss_scale=1024.0,
             dynamic=True, per_tensor_scale=True)
    L = c.layout()
    eng = _engine(c)
    eng.load_master(torch.from_numpy(c.master0(L)))
    host = torch.empty(tuple(eng.grads.shape), dtype=eng.grads.dtype, pin_memory=True)
    out = torch.zeros(96, dtype=torch.uint8).pin_memory()
    for s in (1, 2):
        for r, g in enumerate(c.grads_torch(L, s, 1024.0)):
            host[r].copy_(g)
        eng.step_from_host(host, state_out=out)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(out, eng.state.cpu())
        assert eng.read_state()["t"] == s


def test_host_input_from_pageable_memory_through_the_c_call():
    # zero_step_from_host accepts pageable host memory too (the copies then stage through the
    # driver); results equal the device-resident step bit for bit
    from zero_partitioned_mixed_replica_gb300 import binding as B
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    L = c.layout()
    a, b = _engine(c), _engine(c)
    m0 = torch.from_numpy(c.master0(L))
    a.load_master(m0)
    b.load_master(m0)
    state = torch.zeros(96, dtype=torch.uint8)              # pageable as well
    for s in (1, 2):
        reps = c.grads_torch(L, s, 1.0)
        host = torch.stack(reps)                            # pageable CPU tensor, N_d x Psi_pad
        B.zero_step_from_host(a.L, a.step_args(), [host[r] for r in range(c.n_d)], 10_000, state)
        for r, g in enumerate(reps):
            b.grads[r].copy_(g.cuda())
        b.step()
        torch.cuda.synchronize()
        assert torch.equal(state, a.state.cpu())
    for name in ("master", "m", "v", "params", "state"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def _queued_case(stage: int, fused: bool) -> Case:
    if stage == 3:
        return Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS, max_norm=0.0 if fused else 0.05)
    return Case([200_000, 1600, 99_999], 4, stage, FMT_BF16 if fused else FMT_FP16, bucket_elems=65_536,
                max_norm=0.0 if fused else 1.0, loss_scale=1.0 if fused else 1024.0, per_tensor_scale=True)


def _pinned_steps(c: Case, L, eng, steps: int):
    """Each step's replicas in a pinned host buffer of its own (a buffer may not be
    rewritten before the stream has passed its step), plus a pinned state buffer."""
    hosts, reps, outs = [], [], []
    for s in range(1, steps + 1):
        reps_t = c.grads_torch(L, s, c.loss_scale)
        h = torch.empty(tuple(eng.grads.shape), dtype=eng.grads.dtype, pin_memory=True)
        for r in range(c.n_d):
            h[r].copy_(reps_t[r])
        hosts.append(h)
        reps.append([_u16(t) for t in reps_t])
        outs.append(torch.zeros(96, dtype=torch.uint8).pin_memory())
    return hosts, reps, outs


def _compare_final(c: Case, eng, zs):
    for name in ("master", "m", "v"):
        got = eng.flat(name).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), zs.flat(name).view(np.uint32)), name
    if c.stage == 3:
        assert np.array_equal(_u16(eng.flat("shard16")), zs.flat("shard16"))
    else:
        for r in range(c.n_d):
            assert np.array_equal(_u16(eng.params[r]), zs.params16[r]), r


def _oracle_step(zs, reps, raw_state):
    from zero_partitioned_mixed_replica_gb300 import binding as B
    st = B.zero_step_state.from_buffer_copy(bytes(raw_state.numpy().tobytes()))
    o = zs.step(reps, clip_override=st.clip_coef)
    assert st.t == o["t"] and st.overflow == o["overflow"] and st.error == 0
    assert st.grad_norm == pytest.approx(o["norm"], rel=1e-5)


@pytest.mark.parametrize("stage,fused,live", [(2, False, 1), (1, True, 1), (3, False, 2), (3, True, 1)])
def test_queued_host_steps_overlap_the_previous_update(stage, fused, live):
    # four host-input steps queued with no synchronisation between them: with overlap_previous,
    # a step's copies overwrite the device replicas while the previous step's norm and update still
    # run; every step's state read-back and the final buffers equal the oracle bit for bit
    c = _queued_case(stage, fused)
    L = c.layout()
    eng = _engine(c, live_units=live) if stage == 3 else _engine(c)
    assert eng.fused == fused
    m0 = c.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, c.fmt, HP, max_norm=c.max_norm, loss_scale=c.loss_scale)
    steps = 4
    hosts, reps, outs = _pinned_steps(c, L, eng, steps)
    for s in range(steps):
        eng.step_from_host(hosts[s], chunk_elems=30_000, state_out=outs[s], overlap_previous=True)
    torch.cuda.synchronize()
    for s in range(steps):
        _oracle_step(zs, reps[s], outs[s])
    _compare_final(c, eng, zs)


def test_other_steps_between_host_steps_turn_the_overlap_off():
    # host step, device-resident step (zero_step), host step, replicas written by upload_grads,
    # host step: the device step and upload_grads touch the device replicas, so the host step
    # after each must wait for all queued work; all queued without synchronisation
    c = _queued_case(2, False)
    L = c.layout()
    eng = _engine(c)
    m0 = c.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, c.fmt, HP, max_norm=c.max_norm, loss_scale=c.loss_scale)
    hosts, reps, outs = _pinned_steps(c, L, eng, 5)
    eng.step_from_host(hosts[0], state_out=outs[0], overlap_previous=True)
    for r in range(c.n_d):                                   # step 2 from device memory, same stream
        eng.grads[r].copy_(hosts[1][r], non_blocking=True)
    eng.step()
    outs[1].copy_(eng.state, non_blocking=True)
    eng.step_from_host(hosts[2], state_out=outs[2], overlap_previous=True)
    eng.upload_grads(hosts[3])                               # step 4: library-external copies
    eng.step()
    outs[3].copy_(eng.state, non_blocking=True)
    eng.step_from_host(hosts[4], state_out=outs[4], overlap_previous=True)
    torch.cuda.synchronize()
    for s in range(5):
        _oracle_step(zs, reps[s], outs[s])
    _compare_final(c, eng, zs)


def test_two_engines_on_two_streams_alternate_overlapped_host_steps():
    # engines A and B (own buffers, own streams) alternate host-input steps with overlap_previous,
    # queued without synchronisation: each call's previous executor call is the other engine's,
    # on another stream with other device replicas, so each must wait for its own stream instead
    # of the other engine's release; both match their oracles bit for bit
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    cases = [_queued_case(2, False), _queued_case(2, False)]
    cases[1].seed = 4321
    engs, sims, data = [], [], []
    for c in cases:
        L = c.layout()
        eng = ZeroStep(c.numels, c.n_d, c.stage, c.fmt, c.bucket_elems, c.units,
                       AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay), c.max_norm, c.loss_scale,
                       c.dynamic, c.growth_interval, stream=torch.cuda.Stream())
        m0 = c.master0(L)
        eng.load_master(torch.from_numpy(m0))
        engs.append(eng)
        sims.append(ZeroSimulation(L, m0, c.fmt, HP, max_norm=c.max_norm, loss_scale=c.loss_scale))
        data.append(_pinned_steps(c, L, eng, 3))
    torch.cuda.synchronize()
    for s in range(3):
        for k in (0, 1):
            hosts, _, outs = data[k]
            engs[k].step_from_host(hosts[s], chunk_elems=30_000, state_out=outs[s], overlap_previous=True)
    torch.cuda.synchronize()
    for k in (0, 1):
        _, reps, outs = data[k]
        for s in range(3):
            _oracle_step(sims[k], reps[s], outs[s])
        _compare_final(cases[k], engs[k], sims[k])
