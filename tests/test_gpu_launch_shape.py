"""Launch-shape invariance: every kernel of the step grid-strides over fixed
element positions and writes its norm partials to fixed 32-element slots, so
the results (master/m/v, 16-bit parameters, norm, flags) are bit-identical
whatever grid the launchers pick: the default per-kernel choice, or a cap of
1, 7, 152 or 304 CTAs set through zero_set_max_ctas."""
import pytest
import torch

from oracle.step import AdamWHP, FMT_BF16, FMT_FP16
from tests._cases import Case

pytestmark = pytest.mark.gpu
HP = AdamWHP()
CAPS = [0, 1, 7, 152, 304]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _run(c: Case, cap: int, steps: int = 2, **kw):
    from zero_partitioned_mixed_replica_gb300 import binding as B
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    L = c.layout()
    eng = ZeroStep(c.numels, c.n_d, c.stage, c.fmt, c.bucket_elems, c.units,
                   AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay), c.max_norm, c.loss_scale,
                   c.dynamic, c.growth_interval, **kw)
    eng.load_master(torch.from_numpy(c.master0(L)))
    old = B.zero_set_max_ctas(cap)
    try:
        for s in range(1, steps + 1):
            for r, g in enumerate(c.grads_torch(L, s, eng.read_state()["loss_scale"])):
                eng.grads[r].copy_(g.cuda())
            eng.step()
        torch.cuda.synchronize()
    finally:
        B.zero_set_max_ctas(old)
    out = {n: getattr(eng, n).clone() for n in ("master", "m", "v", "state")}
    out["p16"] = (eng.shard16 if c.stage == 3 else eng.params).clone()
    return out


def _same(a, b):
    for k in a:
        assert torch.equal(a[k].view(torch.uint8) if a[k].dtype != torch.uint8 else a[k],
                           b[k].view(torch.uint8) if b[k].dtype != torch.uint8 else b[k]), k


CASES = [
    ("Z1 fused, N_d=8, buckets", Case([300_000, 7, 180_001], 8, 1, FMT_BF16, bucket_elems=65_536), {}),
    ("Z1 fused whole buffer, N_d=8", Case([300_000, 7, 180_001], 8, 1, FMT_BF16), dict(per_bucket=False)),
    ("Z2 split fp16 clip, N_d=8", Case([300_000, 1600, 99_999], 8, 2, FMT_FP16, bucket_elems=65_536, max_norm=0.5,
                                       loss_scale=1024.0, dynamic=True), {}),
    ("Z2 split clip, N_d=2 (LDG AdamW)", Case([300_000, 7, 50_001], 2, 2, FMT_BF16, max_norm=0.05), {}),
    ("Z2 split clip, N_d=5 (runtime N_d)", Case([300_000, 7, 50_001], 5, 2, FMT_BF16, max_norm=0.05), {}),
    ("Z3 fused, N_d=2", Case([30_000, 60_000, 640, 45_000, 7, 20_000, 3], 2, 3, FMT_BF16,
                             units=[0, 1, 1, 2, 0, 3, 3]), {}),
    ("Z3 split clip, N_d=8", Case([30_000, 60_000, 640, 45_000, 7, 20_000, 3], 8, 3, FMT_BF16,
                                  units=[0, 1, 1, 2, 0, 3, 3], max_norm=0.05), {}),
]


@pytest.mark.parametrize("name,c,kw", CASES, ids=[n for n, _, _ in CASES])
def test_results_do_not_depend_on_the_grid(name, c, kw):
    ref = _run(c, 0, **kw)
    for cap in CAPS[1:]:
        _same(ref, _run(c, cap, **kw))
