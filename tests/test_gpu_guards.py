"""Out-of-bounds writes: every device buffer handed to the library sits inside
a larger allocation whose guard bands (before and after, 256-byte aligned)
hold a sentinel pattern; after several steps of every kind of launch the
guards must be untouched.  Shapes are ragged (odd tensor sizes, buckets that
straddle shards, units of different sizes)."""
import pytest
import torch

from oracle.step import FMT_BF16, FMT_FP16
from tests._cases import Case

pytestmark = pytest.mark.gpu
GUARD = 4096  # bytes on each side


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


class Guarded:
    """A device buffer of n elements of dtype with sentinel guard bands."""

    def __init__(self, n, dtype, fill=0):
        es = torch.tensor([], dtype=dtype).element_size()
        g = GUARD // es
        self.raw = torch.empty(n + 2 * g, dtype=dtype, device="cuda")
        self.raw.view(torch.uint8).fill_(0xA5)
        self.g, self.n = g, n
        self.t = self.raw[g:g + n]
        self.t.zero_()
        if fill:
            self.t.fill_(fill)

    def guards_intact(self):
        b = self.raw.view(torch.uint8)
        gb = self.g * self.raw.element_size()
        return bool((b[:gb] == 0xA5).all()) and bool((b[-gb:] == 0xA5).all())


def _run(c: Case, steps: int, split: bool, micro: int = 1):
    from zero_partitioned_mixed_replica_gb300 import binding as B
    L = c.layout()
    CL = B.zero_layout_init(c.numels, c.units, c.n_d, c.stage, 0, c.bucket_elems if c.stage != 3 else 0, c.fmt)
    info = B.zero_layout_query(CL)
    P, S = info.psi_pad, info.shard_len
    dt16 = torch.bfloat16 if c.fmt == FMT_BF16 else torch.float16
    nd = c.n_d
    grads = [Guarded(P, dt16) for _ in range(nd)]
    master = [Guarded(S, torch.float32, 0.01) for _ in range(nd)]
    m = [Guarded(S, torch.float32) for _ in range(nd)]
    v = [Guarded(S, torch.float32) for _ in range(nd)]
    gsh = [Guarded(S, torch.float32) for _ in range(nd)]
    out = [Guarded(S if c.stage == 3 else P, dt16) for _ in range(nd)]
    shard16 = [Guarded(S, dt16) for _ in range(nd)]
    maxu = max(B.zero_layout_unit(CL, u).real for u in range(info.n_units))
    trans = [Guarded(maxu, dt16) for _ in range(nd)]
    acc = [Guarded(P, torch.float32) for _ in range(nd)] if (micro > 1 and c.stage == 1) else []
    ws = Guarded(info.workspace_bytes, torch.uint8)
    st = Guarded(96, torch.uint8)
    T = lambda xs: [x.t for x in xs]
    B.zero_state_init(st.t, 0.9, 0.999, c.loss_scale, c.dynamic, 2000)
    hp = B.zero_adamw_hp(lr=1e-3, eps=1e-8, weight_decay=0.01)
    kind = B.ZERO_OUT_SHARDS if c.stage == 3 else B.ZERO_OUT_FULL_REPLICAS
    for s in range(1, steps + 1):
        for mb in range(micro):
            for r, g in enumerate(c.grads_torch(L, 10 * s + mb, c.loss_scale)):
                grads[r].t.copy_(g.cuda())
            if c.stage == 3:
                for u in range(info.n_units):
                    B.zero_stage3_gather_layer(CL, u, T(out), T(trans))
            if micro > 1:
                if c.stage == 1:
                    B.zero_accumulate_grads(CL, mb, T(grads), T(acc))
                    if mb == micro - 1:
                        for b in range(info.n_buckets):
                            B.zero_reduce_scatter_accumulated(CL, b, T(acc), T(gsh), micro, st.t, ws.t)
                else:
                    for b in range(info.n_buckets):
                        B.zero_reduce_scatter_micro(CL, b, mb, micro, T(grads), T(gsh), st.t, ws.t)
            elif split:
                for b in reversed(range(info.n_buckets)):
                    B.zero_reduce_scatter(CL, b, T(grads), T(gsh), st.t, ws.t)
            else:
                for b in reversed(range(info.n_buckets)):
                    B.zero_fused_step(CL, b, hp, T(grads), T(master), T(m), T(v), st.t, T(out), kind, ws.t)
        if split or micro > 1:
            B.zero_grad_norm(CL, c.max_norm, B.ZERO_NORM_DECIDE, st.t, ws.t)
            if c.stage == 3:
                B.zero_adamw_shard_step(CL, hp, T(master), T(m), T(v), T(gsh), st.t, T(out), kind)
            else:
                B.zero_adamw_shard_step(CL, hp, T(master), T(m), T(v), T(gsh), st.t, T(shard16),
                                        B.ZERO_OUT_SHARDS)
                B.zero_allgather_params(CL, T(shard16), T(out))
        else:
            B.zero_grad_norm(CL, 0.0, B.ZERO_NORM_AFTER_FUSED, st.t, ws.t)
    torch.cuda.synchronize()
    everything = grads + master + m + v + gsh + out + shard16 + trans + acc + [ws, st]
    bad = [i for i, x in enumerate(everything) if not x.guards_intact()]
    assert not bad, "guard bands overwritten: %s" % bad
    assert not torch.isnan(torch.stack([x.t.float().sum() for x in master])).any()


RAGGED = [50_001, 7, 30_000, 333]


@pytest.mark.parametrize("nd", [1, 2, 3, 8, 64])
def test_guards_fused_zero2(nd):
    _run(Case(RAGGED, nd, 2, FMT_BF16, bucket_elems=4096 + 32), 2, split=False)


@pytest.mark.parametrize("nd", [2, 5, 8, 64])
def test_guards_split_clip_fp16_unfused_allgather(nd):
    _run(Case(RAGGED, nd, 2, FMT_FP16, bucket_elems=8192, max_norm=0.1, loss_scale=1024.0, dynamic=True),
         2, split=True)


@pytest.mark.parametrize("nd", [2, 4, 7])
def test_guards_zero3(nd):
    c = Case(RAGGED, nd, 3, FMT_BF16, units=[0, 1, 1, 2])
    _run(c, 2, split=False)
    _run(c, 2, split=True)


def test_guards_accumulation():
    _run(Case(RAGGED, 4, 1, FMT_BF16, bucket_elems=8192), 2, split=True, micro=3)
    _run(Case(RAGGED, 4, 2, FMT_BF16, bucket_elems=8192), 2, split=True, micro=3)
