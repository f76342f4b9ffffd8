"""The allocation-free entry point (zero_fused_step_noalloc) against the
regular one.

Callers that cannot allocate device memory when they run (a plug-in whose
host owns all device memory, a loop that may not risk a synchronising
cudaMalloc) call zero_fused_step_noalloc, which keeps the norm scratch in a
fixed array inside the library instead of a caller workspace.  This test runs
it through the C ABI twice in a row and checks every output against
zero_fused_step + zero_grad_norm(AFTER_FUSED) on identical inputs.  Both run
the same kernels on the same inputs, so master/m/v, the 16-bit outputs and
the norm must be bit-identical (a unit skipped in the ZeRO-3 loop, or a stale
partial left in the shared array by an earlier, larger call, would show).
It lives in its own file, collected last, and works alone in a fresh process
as well as after the other tests."""
import pytest
import torch

from tests._cases import Case
from oracle.step import FMT_BF16, FMT_FP16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _engine(case):
    from zero_partitioned_mixed_replica_gb300.engine import ZeroStep
    return ZeroStep(case.numels, case.n_d, case.stage, case.fmt, case.bucket_elems, case.units,
                    fused=True, per_bucket=False)


def _same_bits(a: torch.Tensor, b: torch.Tensor, what: str):
    assert a.shape == b.shape and a.dtype == b.dtype, what
    ai = a.contiguous().view(torch.int32 if a.element_size() == 4 else torch.int16)
    bi = b.contiguous().view(torch.int32 if b.element_size() == 4 else torch.int16)
    n = int((ai != bi).sum())
    assert n == 0, "%s: %d elements differ" % (what, n)


@pytest.mark.parametrize("case", [
    Case([1000 * 512, 512, 487 * 1000, 2491], 4, 2, FMT_BF16),
    Case([200_000, 1600, 99_999], 8, 1, FMT_FP16, per_tensor_scale=True),
    Case([30_000, 60_000, 640, 45_000, 7, 20_000, 3], 2, 3, FMT_BF16, units=[0, 1, 1, 2, 0, 3, 3]),
], ids=["zero2_bf16", "zero1_fp16", "zero3_bf16"])
def test_noalloc_matches_workspace_entry_point(case):
    from zero_partitioned_mixed_replica_gb300 import binding as B
    L = case.layout()
    ref, new = _engine(case), _engine(case)
    m0 = torch.from_numpy(case.master0(L))
    ref.load_master(m0)
    new.load_master(m0)
    out = new.shard16_rows if case.stage == 3 else new.param_rows
    kind = B.ZERO_OUT_SHARDS if case.stage == 3 else B.ZERO_OUT_FULL_REPLICAS
    for step in (1, 2):                      # two calls in a row
        for r, g in enumerate(case.grads_torch(L, step, 1.0)):
            ref.grads[r].copy_(g.cuda())
            new.grads[r].copy_(g.cuda())
        ref.step()
        B.zero_fused_step_noalloc(new.L, new.hp, new.grad_rows, new.master_rows, new.m_rows, new.v_rows,
                                  new.state, out, kind)
        a, b = new.read_state(), ref.read_state()
        assert (a["t"], a["overflow"], a["error"]) == (b["t"], b["overflow"], b["error"]) == (step, 0, 0)
        assert a["grad_norm"] == b["grad_norm"] and a["grad_norm"] > 0
        for name in ("master", "m", "v"):
            _same_bits(getattr(new, name), getattr(ref, name), "%s step %d" % (name, step))
        if case.stage == 3:
            _same_bits(new.shard16, ref.shard16, "shard16 step %d" % step)
        else:
            _same_bits(new.params, ref.params, "params step %d" % step)


def test_noalloc_rejects_buffers_above_its_limit():
    from zero_partitioned_mixed_replica_gb300 import binding as B
    L = B.zero_layout_init([B.ZERO_NOALLOC_MAX_ELEMS + 1], None, 1, 2, 0, 0, B.ZERO_BF16)
    fake = [1 << 40]            # never dereferenced: the size check comes first
    with pytest.raises(B.ZeroError) as e:
        B.zero_fused_step_noalloc(L, B.zero_adamw_hp(lr=1e-3, eps=1e-8, weight_decay=0.0), fake, fake, fake,
                                  fake, 1 << 40, fake, B.ZERO_OUT_FULL_REPLICAS, 0)
    assert e.value.status == B.ZERO_ERR_INVALID
    assert "limit" in B.zero_last_error()
