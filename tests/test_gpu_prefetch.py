"""ZeRO-3 prefetch/overlap on the GPU: with the unit gathers on a second
stream overlapping a stand-in layer compute, the step's results equal the
sequential step and the oracle's ZeRO-3 simulation bit for bit, and every
compute saw exactly the unit's previous 16-bit parameters (integer checksums
of the transient buffers against the oracle), for 1, 2 and 3 live units."""
import numpy as np
import pytest
import torch

from oracle.step import AdamWHP, FMT_BF16, ZeroSimulation
from tests._cases import Case

pytestmark = pytest.mark.gpu
HP = AdamWHP()


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _engine(c):
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    return ZeroStep(c.numels, c.n_d, c.stage, c.fmt, 0, c.units,
                    AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay))


@pytest.mark.parametrize("live,ctas", [(1, 0), (2, 0), (3, 0), (2, 40)])
def test_overlapped_equals_sequential_and_sees_previous_params(live, ctas):
    c = Case([300_000, 200_000, 7, 150_000, 64_000, 3], 2, 3, FMT_BF16, units=[0, 1, 1, 2, 3, 0])
    L = c.layout()
    m0 = torch.from_numpy(c.master0(L))
    seq, ovl = _engine(c), _engine(c)
    seq.load_master(m0)
    ovl.load_master(m0)
    zs = ZeroSimulation(L, m0.numpy(), c.fmt, HP)
    U = len(L.units)
    for s in range(1, 3):
        reps = c.grads_torch(L, s, 1.0)
        for r, g in enumerate(reps):
            seq.grads[r].copy_(g.cuda())
            ovl.grads[r].copy_(g.cuda())
        sums = torch.zeros(2 * U, c.n_d, dtype=torch.int64, device="cuda")
        order = {}

        def compute(kind, u, rows):
            k = len(order)
            order[k] = (kind, u)
            real = L.units[u].real
            for r in range(c.n_d):
                # stand-in layer work on the current stream: read the gathered unit
                sums[k, r] = rows[r][:real].view(torch.int16).to(torch.int64).sum()

        prev16 = zs.flat("shard16").astype(np.int16).astype(np.int64)
        seq.step()
        ovl.step_overlapped(compute, max_live_units=live, comm_ctas=ctas)
        zs.step([g.contiguous().view(torch.int16).numpy().view(np.uint16) for g in reps])
        torch.cuda.synchronize()
        assert [order[k] for k in range(2 * U)] == [("fwd", u) for u in range(U)] + \
            [("bwd", u) for u in reversed(range(U))]
        got = sums.cpu().numpy()
        for k in range(2 * U):
            u = L.units[order[k][1]]
            want = int(prev16[u.offset:u.offset + u.real].sum())
            assert all(int(x) == want for x in got[k]), (k, order[k])
        for name in ("master", "m", "v", "shard16"):
            assert torch.equal(getattr(ovl, name), getattr(seq, name)), (name, s)
        assert torch.equal(ovl.state, seq.state)
        # and against the oracle, not only against the sequential engine
        for name in ("master", "m", "v"):
            assert np.array_equal(ovl.flat(name).cpu().numpy().view(np.uint32), zs.flat(name).view(np.uint32)), \
                (name, s)
        assert np.array_equal(ovl.flat("shard16").view(torch.int16).cpu().numpy().view(np.uint16),
                              zs.flat("shard16")), s
        st, o = ovl.read_state(), zs.state.history[-1]
        assert (st["t"], st["overflow"]) == (o["t"], o["overflow"])
        assert abs(st["grad_norm"] - o["norm"]) <= 1e-9 * o["norm"]
