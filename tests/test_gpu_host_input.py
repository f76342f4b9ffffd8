"""Steps whose gradient replicas come from pinned host memory, through the
library's zero_step_from_host (``ZeroStep.step_from_host``): per-bucket
(ZeRO-3: per-unit) copies on the library's two copy streams, each
reduce-scatter or fused update ordered after its own range only, and the
step state copied back to host memory inside the call.  Checked against the
oracle bit for bit, on layouts whose buckets straddle shards, with chunks
smaller than a bucket, and against the device-resident step."""
import pytest
import torch

from oracle.step import FMT_BF16, FMT_FP16
from tests._cases import Case
from tests.test_gpu_parity import Z3_NUMELS, Z3_UNITS, run_parity

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
    from tests.test_gpu_parity import _engine
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
    from tests.test_gpu_parity import _engine
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
