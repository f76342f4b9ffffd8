"""Sharded checkpoints on the GPU: every simulated rank writes its own shard;
loading into the same layout continues bit for bit like an uninterrupted run,
and loading into another N_d / stage / unit split continues exactly like the
oracle started from the same flat optimizer state."""
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


def _engine(c, **kw):
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    return ZeroStep(c.numels, c.n_d, c.stage, c.fmt, c.bucket_elems, c.units,
                    AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay), c.max_norm, c.loss_scale,
                    c.dynamic, c.growth_interval, **kw)


def _u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _steps(eng, c, L, first, last, loss_scales=None):
    for s in range(first, last + 1):
        ls = eng.read_state()["loss_scale"]
        for r, g in enumerate(c.grads_torch(L, s, ls)):
            eng.grads[r].copy_(g.cuda())
        eng.step()


NUMELS = [120_000, 7, 50_001, 3000]


def test_same_layout_roundtrip_is_bit_exact(tmp_path):
    c = Case(NUMELS, 4, 2, FMT_FP16, bucket_elems=32_768, max_norm=0.05, loss_scale=1024.0, dynamic=True)
    L = c.layout()
    m0 = torch.from_numpy(c.master0(L))
    ref = _engine(c)
    ref.load_master(m0)
    _steps(ref, c, L, 1, 4)
    a = _engine(c)
    a.load_master(m0)
    _steps(a, c, L, 1, 2)
    a.save_checkpoint(str(tmp_path))
    b = _engine(c)
    info = b.load_checkpoint(str(tmp_path))
    assert info["segments"] == 4
    assert torch.equal(b.state, a.state)
    _steps(b, c, L, 3, 4)
    for name in ("master", "m", "v", "params"):
        assert torch.equal(getattr(b, name), getattr(ref, name)), name
    assert torch.equal(b.state, ref.state)


@pytest.mark.parametrize("dst", [dict(n_d=2, stage=3, units=[0, 1, 1, 2]), dict(n_d=8, stage=1, units=None),
                                 dict(n_d=3, stage=2, units=None)])
def test_reshard_continues_like_the_oracle(tmp_path, dst):
    src_c = Case(NUMELS, 4, 2, FMT_BF16, bucket_elems=32_768)
    Ls = src_c.layout()
    m0 = src_c.master0(Ls)
    a = _engine(src_c)
    a.load_master(torch.from_numpy(m0))
    _steps(a, src_c, Ls, 1, 2)
    a.save_checkpoint(str(tmp_path))
    zs = ZeroSimulation(Ls, m0, FMT_BF16, HP)
    for s in (1, 2):
        zs.step([_u16(g) for g in src_c.grads_torch(Ls, s, 1.0)])
    dst_c = Case(NUMELS, dst["n_d"], dst["stage"], FMT_BF16, units=dst["units"],
                 bucket_elems=0 if dst["stage"] == 3 else 65_536)
    Ld = dst_c.layout()
    b = _engine(dst_c)
    b.load_checkpoint(str(tmp_path))
    assert b.read_state()["t"] == 2
    # the oracle restarted from the same flat state in the new layout
    def to_flat(name):
        real = zs.flat_real(name)
        out = np.zeros(Ld.psi_pad, np.float32)
        pos = 0
        for off, n in zip(Ld.tensor_offsets, Ld.numels):
            out[off:off + n] = real[pos:pos + n]
            pos += n
        return out
    zd = ZeroSimulation.from_flat(Ld, to_flat("master"), to_flat("m"), to_flat("v"), FMT_BF16, HP, zs.state)
    for name in ("master", "m", "v"):
        assert np.array_equal(b.flat(name).cpu().numpy(), zd.flat(name))
    for s in (3, 4):
        reps = dst_c.grads_torch(Ld, s, 1.0)
        for r, g in enumerate(reps):
            b.grads[r].copy_(g.cuda())
        b.step()
        zd.step([_u16(g) for g in reps])
    assert b.read_state()["t"] == zd.state.t == 4
    for name in ("master", "m", "v"):
        assert np.array_equal(b.flat(name).cpu().numpy().view(np.uint32), zd.flat(name).view(np.uint32)), name
    if dst["stage"] == 3:
        assert np.array_equal(_u16(b.flat("shard16")), zd.flat("shard16"))
    else:
        for r in range(dst["n_d"]):
            assert np.array_equal(_u16(b.params[r]), zd.params16[r])


def test_damaged_checkpoints_are_refused(tmp_path):
    import json
    import os
    c = Case(NUMELS, 4, 2, FMT_BF16)
    L = c.layout()
    a = _engine(c)
    a.load_master(torch.from_numpy(c.master0(L)))
    _steps(a, c, L, 1, 1)
    a.save_checkpoint(str(tmp_path))
    fn = os.path.join(str(tmp_path), "rank002.bin")
    with open(fn, "r+b") as f:                      # a truncated rank file
        f.truncate(os.path.getsize(fn) - 4)
    with pytest.raises(ValueError, match="rank002.bin"):
        _engine(c).load_checkpoint(str(tmp_path))
    a.save_checkpoint(str(tmp_path))
    meta_fn = os.path.join(str(tmp_path), "meta.json")
    meta = json.load(open(meta_fn))
    meta["shard_len"] += 128                        # metadata that contradicts its own layout
    json.dump(meta, open(meta_fn, "w"))
    with pytest.raises(ValueError, match="shard_len"):
        _engine(c).load_checkpoint(str(tmp_path))
