"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element, on the same seeded inputs (drawn on the CPU, copied to the GPU).

Sizes span many CTAs and grid-stride rounds with ragged tails (padding inside
the last vector, buckets that straddle shards, units of different sizes).
The bar: step flags, counters and loss scale bit-exact; fp32 master/m/v within
1e-6 relative (|x| < 1e-30 absolutely within 1e-36); 16-bit parameters within
1 ulp; the global norm within 1e-5 relative (and within 2^-25, the rounding of
the binary32 partials).  Bitwise equality of the state is
also asserted wherever GPU and oracle used the same clip coefficient (always,
when the oracle is re-run with the GPU's coefficient)."""
import math
from dataclasses import dataclass

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


def _engine(case: Case, **kw):
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    return ZeroStep(case.numels, case.n_d, case.stage, case.fmt, case.bucket_elems, case.units,
                    AdamW(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay), case.max_norm,
                    case.loss_scale, case.dynamic, case.growth_interval, pad_multiple=case.pad_multiple, **kw)


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_key(h: np.ndarray) -> np.ndarray:
    h = h.astype(np.int64)
    return np.where(h & 0x8000, -(h & 0x7FFF), h)


def assert_state_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    assert gpu.shape == ref.shape
    d = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    big = np.abs(ref) >= 1e-30
    bad = np.flatnonzero((big & (d > 1e-6 * np.abs(ref))) | (~big & (d > 1e-36)))
    assert bad.size == 0, "%s: %d elements out of tolerance, e.g. idx %s gpu %s ref %s" % (
        what, bad.size, bad[:3], gpu[bad[:3]], ref[bad[:3]])


def assert_p16_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    dist = np.abs(_ulp_key(gpu) - _ulp_key(ref))
    assert dist.max(initial=0) <= 1, "%s: max ulp distance %d" % (what, dist.max())


def run_parity(case: Case, steps: int, garbage_pads: bool = False, use_gpu_clip: bool = False,
               expect_bitwise: bool = True, host_input: bool = False, **engine_kw):
    L = case.layout()
    eng = _engine(case, **engine_kw)
    m0 = case.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, case.fmt, HP, max_norm=case.max_norm, loss_scale=case.loss_scale,
                        dynamic=case.dynamic, growth_interval=case.growth_interval)
    pad = np.zeros(L.psi_pad, bool)
    for u in L.units:
        pad[u.offset + u.real:u.offset + u.padded] = True
    hist = []
    for s in range(1, steps + 1):
        reps_t = case.grads_torch(L, s, zs.state.loss_scale)
        reps = [_u16(t) for t in reps_t]
        if host_input:      # the replicas come from pinned host memory inside the step
            host = torch.empty(tuple(eng.grads.shape), dtype=eng.grads.dtype, pin_memory=True)
            for r in range(case.n_d):
                host[r].copy_(reps_t[r])
                if garbage_pads and pad.any():
                    host[r].view(torch.int16)[torch.from_numpy(np.flatnonzero(pad))] = 0x7F81 if r % 2 else 0x7C00
            eng.step_from_host(host, chunk_elems=host_input if host_input is not True else 1 << 27)
        else:
            for r in range(case.n_d):
                eng.grads[r].copy_(reps_t[r].to(eng.device))
                if garbage_pads and pad.any():
                    idx = torch.from_numpy(np.flatnonzero(pad)).to(eng.device)
                    eng.grads[r].view(torch.int16)[idx] = 0x7F81 if r % 2 else 0x7C00   # NaN / inf bits
            eng.step()
        g = eng.read_state()
        o = zs.step(reps, clip_override=g["clip_coef"] if use_gpu_clip else None)
        hist.append((g, o))
        assert g["overflow"] == o["overflow"], s
        assert g["t"] == o["t"] and g["skipped"] == zs.state.skipped, s
        assert g["loss_scale"] == o["loss_scale"], s
        assert g["error"] == 0 and g["nonfinite"] == 0
        if o["overflow"]:
            assert math.isinf(g["grad_norm"])
        else:
            assert g["grad_norm"] == pytest.approx(o["norm"], rel=1e-5, abs=1e-30)
            # far inside the bar: each 32-element partial is one binary32 (relative error <= 2^-24
            # on the sum of squares, 2^-25 on the norm); with many partials the errors average out
            # (<= 1e-9 measured), with one partial (Psi = 1) the whole 2^-25 can show
            assert abs(g["grad_norm"] - o["norm"]) <= 2.0 ** -25 * (1 + 1e-6) * o["norm"] + 1e-30
        same_clip = np.float32(g["clip_coef"]) == np.float32(o["clip"])
        for name in ("master", "m", "v"):
            gpu = eng.flat(name).cpu().numpy()
            ref = zs.flat(name)
            assert_state_close(gpu, ref, "%s step %d" % (name, s))
            if expect_bitwise and same_clip:
                assert np.array_equal(gpu.view(np.uint32), ref.view(np.uint32)), "%s step %d bitwise" % (name, s)
            assert not gpu[pad].any(), "padding of %s must stay 0" % name
        if case.stage == 3:
            gp, rp = _u16(eng.flat("shard16")), zs.flat("shard16")
            assert_p16_close(gp, rp, "shard16 step %d" % s)
            if expect_bitwise and same_clip:
                assert np.array_equal(gp, rp)
        else:
            for r in range(case.n_d):
                gp = _u16(eng.params[r])
                assert_p16_close(gp, zs.params16[r], "params16[%d] step %d" % (r, s))
                if expect_bitwise and same_clip:
                    assert np.array_equal(gp, zs.params16[r])
    return eng, zs, hist


def test_tiny_fused_zero2():
    # Psi = 1,002,003 (4 tensors), N_d = 4, ZeRO-2, bf16, one bucket, 3 steps
    c = Case([1000 * 512, 512, 487 * 1000, 2491], 4, 2, FMT_BF16)
    run_parity(c, 3)


def test_tiny_fused_per_bucket_equals_whole_buffer():
    c = Case([1000 * 512, 512, 487 * 1000, 2491], 4, 2, FMT_BF16, bucket_elems=4096 * 7 + 32)
    e1, _, _ = run_parity(c, 2, per_bucket=True)
    e2, _, _ = run_parity(c, 2, per_bucket=False)
    assert torch.equal(e1.master, e2.master) and torch.equal(e1.params, e2.params)


@pytest.mark.parametrize("n_d", [1, 2, 3, 5, 8, 16])
def test_zero1_fused_all_rank_counts(n_d):
    c = Case([40_000, 33, 77_777, 5], n_d, 1, FMT_BF16, bucket_elems=65_536, per_tensor_scale=True)
    run_parity(c, 2)


@pytest.mark.parametrize("n_d", [2, 3, 8])
def test_zero2_split_clip_bf16(n_d):
    c = Case([120_000, 7, 50_001], n_d, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05,
             per_tensor_scale=True)
    _, _, hist = run_parity(c, 3, use_gpu_clip=True)
    assert all(g["clip_coef"] < 1.0 for g, _ in hist)


def test_zero2_split_clip_independent_coefficient():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05, per_tensor_scale=True)
    run_parity(c, 3, use_gpu_clip=False)


def test_zero2_fp16_scaler_overflow_skip():
    # like the GPT-2 1.5B run: fp16 grads x 2^16, dynamic scale, clip 1.0, +inf in rank 3 at step 4
    c = Case([200_000, 1600, 99_999], 8, 2, FMT_FP16, bucket_elems=65_536, max_norm=1.0,
             loss_scale=65536.0, dynamic=True, per_tensor_scale=True, inf_step=4, inf_rank=3)
    eng, zs, hist = run_parity(c, 6, use_gpu_clip=True)
    assert [g["overflow"] for g, _ in hist] == [0, 0, 0, 1, 0, 0]
    assert [g["loss_scale"] for g, _ in hist] == [65536.0] * 3 + [32768.0] * 3
    assert [g["t"] for g, _ in hist] == [1, 2, 3, 3, 4, 5]


def test_scale_growth_on_gpu():
    c = Case([30_000], 2, 2, FMT_FP16, loss_scale=256.0, dynamic=True, growth_interval=2)
    _, _, hist = run_parity(c, 5)
    assert [g["loss_scale"] for g, _ in hist] == [256.0, 512.0, 512.0, 1024.0, 1024.0]


def test_garbage_in_gradient_padding_is_ignored():
    c = Case([1000 * 512, 512, 487 * 1000, 2491], 4, 2, FMT_BF16, max_norm=0.5)
    run_parity(c, 2, garbage_pads=True, use_gpu_clip=True)
    c = Case([100_001, 3], 3, 1, FMT_BF16)
    run_parity(c, 2, garbage_pads=True)


def test_unfused_allgather_equals_fused():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    e1, _, _ = run_parity(c, 2, use_gpu_clip=True, fuse_allgather=False)
    e2, _, _ = run_parity(c, 2, use_gpu_clip=True, fuse_allgather=True)
    assert torch.equal(e1.params, e2.params) and torch.equal(e1.master, e2.master)


def test_split_equals_fused_without_clip():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768)
    e1, _, _ = run_parity(c, 2, fused=False)
    e2, _, _ = run_parity(c, 2, fused=True)
    assert torch.equal(e1.master, e2.master) and torch.equal(e1.params, e2.params)


Z3_NUMELS = [30_000, 60_000, 640, 45_000, 7, 20_000, 3]
Z3_UNITS = [0, 1, 1, 2, 0, 3, 3]


@pytest.mark.parametrize("n_d", [1, 2, 5])
def test_zero3_fused_with_transients(n_d):
    c = Case(Z3_NUMELS, n_d, 3, FMT_BF16, units=Z3_UNITS)
    L = c.layout()
    seen = []

    def hook(kind, u, rows):
        torch.cuda.synchronize()
        unit = L.units[u]
        seen.append((kind, u, [_u16(r[:unit.real]) for r in rows]))

    eng = _engine(c)
    eng.transient_hook = hook
    m0 = c.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, c.fmt, HP)
    zs.record_transients = True
    for s in range(1, 4):
        seen.clear()
        reps_t = c.grads_torch(L, s, 1.0)
        for r in range(n_d):
            eng.grads[r].copy_(reps_t[r].cuda())
        eng.step()
        zs.step([_u16(t) for t in reps_t])
        assert [(k, u) for k, u, _ in seen] == [(k, u) for k, u, _ in zs.transients]
        for (k, u, gts), (_, _, ots) in zip(seen, zs.transients):
            for a, b in zip(gts, ots):
                assert np.array_equal(a, b), (k, u)
        assert np.array_equal(_u16(eng.flat("shard16")), zs.flat("shard16"))
        for name in ("master", "m", "v"):
            assert np.array_equal(eng.flat(name).cpu().numpy().view(np.uint32), zs.flat(name).view(np.uint32))


def test_zero3_split_fp16_clip_scaler():
    c = Case(Z3_NUMELS, 4, 3, FMT_FP16, units=Z3_UNITS, max_norm=0.01, loss_scale=1024.0, dynamic=True,
             inf_step=2, inf_rank=1)
    _, _, hist = run_parity(c, 4, use_gpu_clip=True)
    assert [g["overflow"] for g, _ in hist] == [0, 1, 0, 0]


def test_zero3_garbage_pads():
    c = Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS)
    run_parity(c, 2, garbage_pads=True)


def test_bucket_size_invariance_on_gpu():
    outs = []
    for bucket in (0, 32, 4096, 65_536 + 32):
        c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=bucket, max_norm=0.05)
        L = c.layout()
        eng = _engine(c)
        eng.load_master(torch.from_numpy(c.master0(L)))
        for s in range(1, 3):
            for r, t in enumerate(c.grads_torch(L, s, 1.0)):
                eng.grads[r].copy_(t.cuda())
            eng.step()
        st = eng.read_state()
        outs.append((st["grad_norm"], st["clip_coef"], eng.master.clone(), eng.params.clone()))
    for o in outs[1:]:
        assert o[0] == outs[0][0] and o[1] == outs[0][1]
        assert torch.equal(o[2], outs[0][2]) and torch.equal(o[3], outs[0][3])


def test_cuda_graph_replay_equals_eager():
    c = Case([120_000, 7, 50_001], 4, 2, FMT_FP16, bucket_elems=32_768, max_norm=1.0, loss_scale=65536.0,
             dynamic=True)
    L = c.layout()
    res = []
    for graph in (False, True):
        eng = _engine(c)
        eng.load_master(torch.from_numpy(c.master0(L)))
        for r, t in enumerate(c.grads_torch(L, 1, 65536.0)):
            eng.grads[r].copy_(t.cuda())
        if graph:
            g = eng.capture()
            eng.reset_state()
            eng.load_master(torch.from_numpy(c.master0(L)))
            for _ in range(3):
                g.replay()
        else:
            for _ in range(3):
                eng.step()
        res.append((eng.read_state(), eng.master.clone(), eng.params.clone()))
    assert res[0][0]["t"] == res[1][0]["t"] == 3
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])


def test_deterministic_rerun():
    c = Case([120_000, 7, 50_001], 8, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    a, _, ha = run_parity(c, 2, use_gpu_clip=True)
    b, _, hb = run_parity(c, 2, use_gpu_clip=True)
    assert [g["grad_norm"] for g, _ in ha] == [g["grad_norm"] for g, _ in hb]
    assert torch.equal(a.master, b.master) and torch.equal(a.params, b.params)


def test_launch_count_of_a_split_step():
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    eng = _engine(c)
    Bd.zero_launch_count(reset=True)
    eng.step()
    torch.cuda.synchronize()
    # one reduce-scatter per bucket, two norm passes, one AdamW
    assert Bd.zero_launch_count() == eng.n_buckets + 3


def test_nan_gradient_skips_split_step_and_is_reported_by_fused_step():
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=1.0)
    L = c.layout()
    for fused in (False, True):
        cc = Case(c.numels, c.n_d, c.stage, c.fmt, c.bucket_elems, max_norm=0.0 if fused else 1.0)
        eng = _engine(cc)
        eng.load_master(torch.from_numpy(cc.master0(L)))
        before = eng.master.clone()
        for r, g in enumerate(cc.grads_torch(L, 1, 1.0)):
            eng.grads[r].copy_(g.cuda())
        eng.grads[1].view(torch.int16)[L.psi // 3] = 0x7FC1          # NaN in a real element
        eng.step()
        st = eng.read_state()
        assert st["overflow"] == 1 and st["nonfinite"] == 0
        if fused:   # no global decision before the update: the step ran and t advanced
            assert st["t"] == 1
        else:
            assert st["t"] == 0 and st["skipped"] == 1 and torch.equal(eng.master, before)


def test_zero_gradients_apply_weight_decay_only():
    c = Case([120_000, 7, 50_001], 3, 2, FMT_BF16, bucket_elems=32_768, grad_std=0.0)
    eng, zs, _ = run_parity(c, 2)
    assert float(eng.read_state()["grad_norm"]) == 0.0
    assert not eng.m.any() and not eng.v.any()


@dataclass
class _ZeroRegions(Case):
    """Tensors in `zero_tensors` get zero gradients of both signs on every rank
    at every step, so their g, m and v stay zero: the update kernels' short path
    for all-zero elements (and, where a 4- or 8-element group straddles a
    tensor edge, the plain update on a mixed group).  Half of their master
    weights start at +0 or -0, so the zero signs of p1 - step_size * m matter."""
    zero_tensors: tuple = ()

    def master0(self, L):
        m = super().master0(L).copy()
        for t in self.zero_tensors:
            o, n = L.tensor_offsets[t], L.numels[t]
            m[o:o + n // 4] = 0.0
            m[o + n // 4:o + n // 2] = -0.0
        return m

    def grads_torch(self, L, step, loss_scale, device="cpu"):
        out = super().grads_torch(L, step, loss_scale, device)
        for r, g in enumerate(out):
            for t in self.zero_tensors:
                o, n = L.tensor_offsets[t], L.numels[t]
                bits = torch.zeros(n, dtype=torch.int16)
                bits[(torch.arange(n) + r + step) % 3 == 0] = -0x8000      # -0 in fp16 and bf16
                g.view(torch.int16)[o:o + n] = bits
        return out


@pytest.mark.parametrize("n_d,stage,max_norm,fmt", [
    (4, 2, 1.0, FMT_FP16),    # split step: the TMA update
    (4, 1, 1.0, FMT_BF16),    # split step: the TMA update
    (2, 2, 1.0, FMT_BF16),    # N_d = 2: the LDG update
    (4, 3, 1.0, FMT_FP16),    # 16-bit shards: the LDG update
    (4, 2, 0.0, FMT_FP16),    # fused per-bucket update
    (3, 3, 0.0, FMT_BF16),    # fused update into 16-bit shards
])
def test_zero_state_regions_in_every_update_kernel(n_d, stage, max_norm, fmt):
    # a 300k-element zero tensor spans ~150 TMA tiles; the 33- and 5-element ones sit between dense
    # tensors, so groups straddle zero and non-zero elements
    c = _ZeroRegions([70_001, 300_000, 33, 90_000, 5, 40_000], n_d, stage, fmt, bucket_elems=65_536,
                     max_norm=max_norm, loss_scale=1024.0 if fmt == FMT_FP16 else 1.0,
                     units=[0, 0, 1, 1, 2, 2] if stage == 3 else None, zero_tensors=(1, 2, 4))
    eng, zs, _ = run_parity(c, 3)
    L = c.layout()
    for name in ("m", "v"):
        flat = zs.flat(name)
        for t in c.zero_tensors:
            o = L.tensor_offsets[t]
            assert not flat[o:o + L.numels[t]].any(), (name, t)   # the case does exercise zero state


def test_units_smaller_than_a_rank_slice():
    # 3- and 5-element units with N_d = 4: most ranks own only padding of them
    c = Case([3, 5000, 5, 70_000], 4, 3, FMT_BF16, units=[0, 1, 2, 3])
    run_parity(c, 2)
    c = Case([3, 5000, 5, 70_000], 4, 3, FMT_FP16, units=[0, 1, 2, 3], max_norm=0.1, loss_scale=512.0,
             dynamic=True)
    run_parity(c, 2, use_gpu_clip=True)


@pytest.mark.parametrize("stage,units", [(2, None), (3, [0, 1, 1, 2])])
def test_user_pad_multiple(stage, units):
    # a pad quantum of 4 N_d 128 (a DeepSpeed-style alignment knob): more padding, same results
    c = Case([120_000, 7, 50_001, 3000], 3, stage, FMT_BF16, bucket_elems=32_768 if stage != 3 else 0,
             units=units, max_norm=0.05, pad_multiple=4 * 3 * 128)
    eng, zs, _ = run_parity(c, 2, use_gpu_clip=True)
    assert eng.info.q == 4 * 3 * 128 and eng.info.psi_pad % (4 * 3 * 128) == 0


@pytest.mark.parametrize("n_d,stage", [(64, 2), (64, 1), (16, 2), (64, 3)])
def test_split_clip_at_the_rank_limit(n_d, stage):
    # ZERO_MAX_RANKS = 64: the runtime-N_d reduce-scatter, the TMA AdamW's 64 bulk stores per
    # tile (ZeRO-1/2) or the shard-output update (ZeRO-3); fp16 with a dynamic scale and clip
    units = [0, 1, 1, 2] if stage == 3 else None
    c = Case([200_000, 7, 50_001, 3000], n_d, stage, FMT_FP16, bucket_elems=65_536 if stage != 3 else 0,
             units=units, max_norm=0.05, loss_scale=1024.0, dynamic=True, per_tensor_scale=True)
    _, _, hist = run_parity(c, 2, use_gpu_clip=True)
    assert all(g["clip_coef"] < 1.0 for g, _ in hist)


@pytest.mark.parametrize("stage,fmt,loss_scale", [(2, FMT_BF16, 1.0), (2, FMT_FP16, 65536.0),
                                                  (3, FMT_FP16, 1024.0)])
def test_split_clip_clamp_branch_equals_unclipped(stage, fmt, loss_scale):
    # max_norm far above the global norm ("ZeRO-3 核心流程", 坑 1: one coefficient on every rank):
    # the clamp gives c = 1.0 exactly, on the GPU and in the oracle's own decision, and the step
    # equals the same step without clipping, bit for bit
    units = Z3_UNITS if stage == 3 else None
    numels = Z3_NUMELS if stage == 3 else [120_000, 7, 50_001]
    kw = dict(bucket_elems=32_768 if stage != 3 else 0, units=units, loss_scale=loss_scale,
              dynamic=loss_scale != 1.0, per_tensor_scale=True)
    c = Case(numels, 4, stage, fmt, max_norm=1e3, **kw)
    e1, _, hist = run_parity(c, 3, use_gpu_clip=False)
    assert all(g["clip_coef"] == 1.0 and o["clip"] == 1.0 and o["norm"] < 1e3 for g, o in hist)
    assert all(0.0 < g["grad_norm"] for g, _ in hist)
    c0 = Case(numels, 4, stage, fmt, max_norm=0.0, **kw)
    e0, _, _ = run_parity(c0, 3)
    for name in ("master", "m", "v"):
        assert torch.equal(getattr(e1, name), getattr(e0, name)), name
    if stage == 3:
        assert torch.equal(e1.shard16, e0.shard16)
    else:
        assert torch.equal(e1.params, e0.params)


@pytest.mark.parametrize("n_d,stage,fmt", [(3, 2, FMT_BF16), (8, 1, FMT_FP16), (5, 3, FMT_FP16), (64, 2, FMT_BF16)])
def test_cast_params_matches_oracle_cast(n_d, stage, fmt):
    # zero_cast_params: the RNE cast of the master ("第 5 课" §3 step 2) into every replica (ZeRO-1/2,
    # with the all-gather of step 3) or the rank's shard (ZeRO-3), against the oracle's encoder;
    # the master holds fp16 subnormals, values at and beyond 65504, RNE midpoints and signed zeros
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    units = [0, 1, 1, 2] if stage == 3 else None
    c = Case([40_000, 7, 33_001, 999], n_d, stage, fmt, units=units)
    L = c.layout()
    m0 = c.master0(L)
    rng = np.random.default_rng(3)
    special = np.array([6e-8, -6e-8, 5.96e-8, 1e-5, -3.1e-5, 65504.0, 65519.0, 65520.0, -7e4, 1e30, -0.0,
                        1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    real = np.concatenate([np.arange(o, o + n) for o, n in zip(L.tensor_offsets, L.numels)])
    idx = rng.choice(real, size=special.size * 40, replace=False)
    m0[idx] = np.tile(special, 40)
    eng = _engine(c)
    Bd.zero_launch_count(reset=True)
    eng.load_master(torch.from_numpy(m0))
    torch.cuda.synchronize()
    assert Bd.zero_launch_count() == 1
    zs = ZeroSimulation(L, m0, c.fmt, HP)
    if stage == 3:
        assert np.array_equal(_u16(eng.flat("shard16")), zs.flat("shard16"))
    else:
        for r in range(n_d):
            assert np.array_equal(_u16(eng.params[r]), zs.params16[r]), r
    # the layout's padding casts to +0
    pad = np.ones(L.psi_pad, bool)
    pad[real] = False
    if stage != 3:
        assert not _u16(eng.params[0])[pad].any()


def _issue_step_calls(eng, s=None):
    """The step's calls issued one by one through the C ABI, in the pages' order
    as the test restates it: ZeRO-1/2 reduce-scatter (or fused step) per bucket,
    last bucket first, then the norm and, split, AdamW (fused or unfused
    all-gather); ZeRO-3 forward gathers, then per unit in reverse a gather and a
    fused step or reduce-scatter, then the norm (and, split, the shard update)."""
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    L = eng.L
    s = s or torch.cuda.current_stream()
    if eng.stage == 3:
        U = len(eng.units)
        for u in list(range(U)) + list(reversed(range(U))):
            Bd.zero_stage3_gather_layer(L, u, eng.shard16_rows, eng.transient_rows, s)
        for u in reversed(range(U)):
            if eng.fused:
                Bd.zero_fused_step(L, u, eng.hp, eng.grad_rows, eng.master_rows, eng.m_rows, eng.v_rows, eng.state,
                                   eng.shard16_rows, Bd.ZERO_OUT_SHARDS, eng.workspace, s)
            else:
                Bd.zero_reduce_scatter(L, u, eng.grad_rows, eng.gshard_rows, eng.state, eng.workspace, s)
        if eng.fused:
            Bd.zero_grad_norm(L, 0.0, Bd.ZERO_NORM_AFTER_FUSED, eng.state, eng.workspace, s)
        else:
            Bd.zero_grad_norm(L, eng.max_norm, Bd.ZERO_NORM_DECIDE, eng.state, eng.workspace, s)
            Bd.zero_adamw_shard_step(L, eng.hp, eng.master_rows, eng.m_rows, eng.v_rows, eng.gshard_rows,
                                     eng.state, eng.shard16_rows, Bd.ZERO_OUT_SHARDS, s)
        return
    if eng.fused:
        for b in (reversed(range(eng.n_buckets)) if eng.per_bucket else [-1]):
            Bd.zero_fused_step(L, b, eng.hp, eng.grad_rows, eng.master_rows, eng.m_rows, eng.v_rows, eng.state,
                               eng.param_rows, Bd.ZERO_OUT_FULL_REPLICAS, eng.workspace, s)
        Bd.zero_grad_norm(L, 0.0, Bd.ZERO_NORM_AFTER_FUSED, eng.state, eng.workspace, s)
        return
    for b in reversed(range(eng.n_buckets)):
        Bd.zero_reduce_scatter(L, b, eng.grad_rows, eng.gshard_rows, eng.state, eng.workspace, s)
    Bd.zero_grad_norm(L, eng.max_norm, Bd.ZERO_NORM_DECIDE, eng.state, eng.workspace, s)
    if eng.fuse_allgather:
        Bd.zero_adamw_shard_step(L, eng.hp, eng.master_rows, eng.m_rows, eng.v_rows, eng.gshard_rows, eng.state,
                                 eng.param_rows, Bd.ZERO_OUT_FULL_REPLICAS, s)
    else:
        Bd.zero_adamw_shard_step(L, eng.hp, eng.master_rows, eng.m_rows, eng.v_rows, eng.gshard_rows, eng.state,
                                 eng.shard16_rows, Bd.ZERO_OUT_SHARDS, s)
        Bd.zero_allgather_params(L, eng.shard16_rows, eng.param_rows, s)


@pytest.mark.parametrize("mode", ["z2_fused_bucket", "z2_fused_whole", "z2_split_clip_fp16", "z1_split_unfused_ag",
                                  "z3_fused", "z3_split_fp16", "z3_fused_two_live"])
def test_native_executor_equals_call_by_call(mode):
    # zero_step (the library issues the step's calls: alternating bucket streams, two live units)
    # against the same calls issued one by one on one stream: bit-identical state after 3 steps
    kw = {"z2_fused_bucket": dict(n_d=4, stage=2, fmt=FMT_BF16, eng=dict(per_bucket=True)),
          "z2_fused_whole": dict(n_d=4, stage=2, fmt=FMT_BF16, eng=dict(per_bucket=False)),
          "z2_split_clip_fp16": dict(n_d=8, stage=2, fmt=FMT_FP16, max_norm=0.05, loss_scale=4096.0, dynamic=True,
                                     inf_step=2, inf_rank=5, eng={}),
          "z1_split_unfused_ag": dict(n_d=3, stage=1, fmt=FMT_BF16, max_norm=0.05, eng=dict(fuse_allgather=False)),
          "z3_fused": dict(n_d=2, stage=3, fmt=FMT_BF16, eng={}),
          "z3_split_fp16": dict(n_d=4, stage=3, fmt=FMT_FP16, max_norm=0.01, loss_scale=256.0, dynamic=True,
                                eng={}),
          "z3_fused_two_live": dict(n_d=2, stage=3, fmt=FMT_BF16, eng=dict(live_units=2))}[mode]
    ekw = kw.pop("eng")
    n_d, stage, fmt = kw.pop("n_d"), kw.pop("stage"), kw.pop("fmt")
    z3 = stage == 3
    c = Case(Z3_NUMELS if z3 else [120_000, 7, 50_001], n_d, stage, fmt, bucket_elems=0 if z3 else 32_768,
             units=Z3_UNITS if z3 else None, per_tensor_scale=True, **kw)
    L = c.layout()
    a, b = _engine(c, **ekw), _engine(c, **ekw)
    m0 = torch.from_numpy(c.master0(L))
    a.load_master(m0)
    b.load_master(m0)
    for s in range(1, 4):
        reps = c.grads_torch(L, s, a.read_state()["loss_scale"])
        for r, g in enumerate(reps):
            a.grads[r].copy_(g.cuda())
            b.grads[r].copy_(g.cuda())
        a.step()
        _issue_step_calls(b)
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "state"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.shard16, b.shard16) if z3 else torch.equal(a.params, b.params)
    if mode == "z2_split_clip_fp16":
        assert a.read_state()["skipped"] == 1


@pytest.mark.parametrize("live", [1, 2])
def test_unit_hook_sees_every_gather_in_order(live):
    # the executor's unit hook runs after each gather is issued, forward then backward, with the
    # buffers that gather wrote; each holds the unit's previous parameters (the oracle's)
    c = Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS)
    L = c.layout()
    eng = _engine(c, live_units=live)
    m0 = c.master0(L)
    eng.load_master(torch.from_numpy(m0))
    zs = ZeroSimulation(L, m0, c.fmt, HP)
    seen = []

    def hook(kind, u, rows):
        torch.cuda.current_stream().synchronize()
        torch.cuda.synchronize()
        seen.append((kind, u, rows[0].data_ptr(), [_u16(r[:L.units[u].real]) for r in rows]))

    eng.transient_hook = hook
    for s in (1, 2):
        seen.clear()
        prev = zs.flat("shard16")
        reps = c.grads_torch(L, s, 1.0)
        for r, g in enumerate(reps):
            eng.grads[r].copy_(g.cuda())
        eng.step()
        zs.step([_u16(t) for t in reps])
        U = len(L.units)
        assert [(k, u) for k, u, _, _ in seen] == [("fwd", u) for u in range(U)] + \
            [("bwd", u) for u in reversed(range(U))]
        for k, u, _, rows in seen:
            want = prev[L.units[u].offset:L.units[u].offset + L.units[u].real]
            for row in rows:
                assert np.array_equal(row, want), (k, u)
        bufs = {p for _, _, p, _ in seen}
        assert len(bufs) == live


def test_launch_tracing_counts_every_call_of_the_executor():
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768, max_norm=0.05)
    L = c.layout()
    eng = _engine(c)
    eng.load_master(torch.from_numpy(c.master0(L)))
    for r, g in enumerate(c.grads_torch(L, 1, 1.0)):
        eng.grads[r].copy_(g.cuda())
    Bd.zero_trace_read(reset=True)
    prev = Bd.zero_trace_enable(True)
    try:
        for _ in range(3):
            eng.step()
    finally:
        Bd.zero_trace_enable(prev)
    t = Bd.zero_trace_read(reset=True)
    assert t["reduce_scatter"]["launches"] == 3 * eng.n_buckets
    assert t["grad_norm"]["launches"] == 3 and t["adamw"]["launches"] == 3
    for k in t.values():
        assert 0 < k["busy_ms"] <= k["total_ms"] * (1 + 1e-6)
    eng.step()                                   # tracing off: nothing recorded
    assert Bd.zero_trace_read(reset=True) == {}
    f = _engine(Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=32_768))
    Bd.zero_trace_enable(True)
    try:
        f.step()
    finally:
        Bd.zero_trace_enable(False)
    t = Bd.zero_trace_read(reset=True)
    assert t["fused_step"]["launches"] == f.n_buckets and t["grad_norm"]["launches"] == 1


@pytest.mark.parametrize("fused,fmt", [(True, FMT_BF16), (False, FMT_FP16)])
def test_zero3_two_live_units_equal_one(fused, fmt):
    # zero_step with a second transient set (units alternate buffers and streams) against one buffer
    # and against the oracle, bit for bit
    kw = {} if fused else dict(max_norm=0.01, loss_scale=512.0, dynamic=True)
    c = Case(Z3_NUMELS, 4, 3, fmt, units=Z3_UNITS, per_tensor_scale=True, **kw)
    e2, zs, _ = run_parity(c, 3, live_units=2)
    assert e2.transient2 is not None
    e1, _, _ = run_parity(c, 3)
    for name in ("master", "m", "v", "shard16", "state"):
        assert torch.equal(getattr(e1, name), getattr(e2, name)), name


@pytest.mark.parametrize("n_d,stage,fmt,max_norm", [(1, 2, FMT_BF16, 0.0), (1, 1, FMT_FP16, 1e-4), (3, 2, FMT_BF16, 0.0),
                                                    (64, 2, FMT_FP16, 1e-4), (64, 3, FMT_BF16, 0.0),
                                                    (2, 3, FMT_FP16, 1e-4)])
def test_single_parameter_buffers(n_d, stage, fmt, max_norm):
    # Psi = 1: one real element and q - 1 padding elements; every rank but rank 0 owns only padding
    units = [0] if stage == 3 else None
    c = Case([1], n_d, stage, fmt, units=units, max_norm=max_norm, loss_scale=2.0 ** 10 if fmt == FMT_FP16 else 1.0,
             dynamic=fmt == FMT_FP16)
    eng, zs, hist = run_parity(c, 3, garbage_pads=True)
    assert eng.info.psi == 1 and eng.info.psi_pad == n_d * 128
    if max_norm > 0:    # the coefficients agree to one binary32 rounding (the norm's partial, above)
        assert all(0 < g["clip_coef"] <= 1 and abs(g["clip_coef"] - o["clip"]) <= 2.0 ** -23 * o["clip"]
                   for g, o in hist if not g["overflow"])


def test_tracing_is_off_inside_a_graph_capture():
    # traced calls record no events while their stream is being captured; the replayed graph
    # equals eager steps, and tracing resumes for eager calls afterwards
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    c = Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=4096)    # 43 buckets: two streams
    L = c.layout()
    a, b = _engine(c), _engine(c)
    for e in (a, b):
        e.load_master(torch.from_numpy(c.master0(L)))
        for r, g in enumerate(c.grads_torch(L, 1, 1.0)):
            e.grads[r].copy_(g.cuda())
    Bd.zero_trace_read(reset=True)
    prev = Bd.zero_trace_enable(True)
    try:
        graph = a.capture()
        assert Bd.zero_trace_read(reset=True) == {}
        a.reset_state()
        a.load_master(torch.from_numpy(c.master0(L)))
        for _ in range(2):
            graph.replay()
            b.step()
        torch.cuda.synchronize()
        t = Bd.zero_trace_read(reset=True)
        assert t["fused_step"]["launches"] == 2 * b.n_buckets        # the eager steps only
    finally:
        Bd.zero_trace_enable(prev)
    for name in ("master", "m", "v", "params"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_unit_hook_exceptions_reach_the_caller():
    # an exception cannot cross the executor's C frames; the binding re-raises the hook's first one
    c = Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS)
    eng = _engine(c)
    calls = []

    def hook(kind, u, rows):
        calls.append((kind, u))
        if (kind, u) == ("fwd", 1):
            raise ValueError("planted in the hook")

    eng.transient_hook = hook
    with pytest.raises(ValueError, match="planted in the hook"):
        eng.step()
    assert calls[:2] == [("fwd", 0), ("fwd", 1)] and len(calls) == 2     # later calls are skipped
    eng.transient_hook = None
    eng.step()                                                            # the engine stays usable
    assert eng.read_state()["error"] == 0


def test_two_host_threads_share_the_executor():
    # two engines stepped from two host threads at once, each on its own stream: the executor's
    # per-device lock serialises their issue; results equal the same engines stepped one by one
    import threading
    cases = [Case([120_000, 7, 50_001], 4, 2, FMT_BF16, bucket_elems=4096, per_tensor_scale=True),
             Case(Z3_NUMELS, 2, 3, FMT_FP16, units=Z3_UNITS, max_norm=0.01, loss_scale=256.0, dynamic=True)]
    kws = [{}, dict(live_units=2)]

    def make():
        out = []
        for c, kw in zip(cases, kws):
            L = c.layout()
            e = _engine(c, **kw)
            e.load_master(torch.from_numpy(c.master0(L)))
            for r, g in enumerate(c.grads_torch(L, 1, c.loss_scale)):
                e.grads[r].copy_(g.cuda())
            out.append(e)
        torch.cuda.synchronize()
        return out

    seq = make()
    for e in seq:
        for _ in range(5):
            e.step()
    torch.cuda.synchronize()
    par = make()
    errors = []

    def worker(e):
        try:
            s = torch.cuda.Stream()
            e.stream = s
            for _ in range(5):
                e.step()
            s.synchronize()
        except BaseException as ex:      # noqa: BLE001 (reported below)
            errors.append(ex)

    threads = [threading.Thread(target=worker, args=(e,)) for e in par]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for a, b in zip(seq, par):
        for name in ("master", "m", "v", "state"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("stage", [1, 2, 3])
def test_fp16_subnormal_gradients(stage):
    # fp16 gradients of std 2e-6 without loss scaling: most are fp16 subnormals (below 6.1e-5), so
    # the reduce decodes them (and the cast writes subnormal parameters where the update makes them)
    units = Z3_UNITS if stage == 3 else None
    numels = Z3_NUMELS if stage == 3 else [120_000, 7, 50_001]
    c = Case(numels, 4, stage, FMT_FP16, bucket_elems=32_768 if stage != 3 else 0, units=units, grad_std=2e-6,
             max_norm=1e-4)
    L = c.layout()
    reps = c.grads(L, 1, 1.0)
    h = np.concatenate(reps)
    sub = ((h & 0x7C00) == 0) & ((h & 0x03FF) != 0)
    assert sub.mean() > 0.5
    run_parity(c, 3)


def test_zero3_two_live_units_replay_from_a_graph():
    # the executor's forks and joins between its streams capture into a CUDA graph; replays equal
    # eager steps bit for bit
    c = Case(Z3_NUMELS, 2, 3, FMT_BF16, units=Z3_UNITS, per_tensor_scale=True)
    L = c.layout()
    a, b = _engine(c, live_units=2), _engine(c, live_units=2)
    for e in (a, b):
        e.load_master(torch.from_numpy(c.master0(L)))
        for r, g in enumerate(c.grads_torch(L, 1, 1.0)):
            e.grads[r].copy_(g.cuda())
    g = a.capture()
    a.reset_state()
    a.load_master(torch.from_numpy(c.master0(L)))
    for _ in range(3):
        g.replay()
        b.step()
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "shard16", "state"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert a.read_state()["t"] == 3


def test_long_run_with_natural_overflows():
    # 200 steps, fp16 x a dynamic scale that doubles every 20 good steps from 2^16: once the scaled
    # gradients pass 65504 they overflow on their own, the step is skipped and the scale halves, then
    # grows again.  Flags, counters, scale, norm and state match the oracle at every step (beta^t
    # after ~190 applied steps included); several buckets, rotating over the executor's streams.
    c = Case([1000 * 512, 512, 487 * 1000, 2491], 4, 2, FMT_FP16, bucket_elems=4096 * 7 + 32, max_norm=1.0,
             loss_scale=65536.0, dynamic=True, growth_interval=20, per_tensor_scale=True)
    _, _, hist = run_parity(c, 200)
    over = [g["overflow"] for g, _ in hist]
    scales = [g["loss_scale"] for g, _ in hist]
    assert sum(over) >= 2, over
    assert max(scales) > 65536.0 and any(b < a for a, b in zip(scales, scales[1:]))
    assert hist[-1][0]["t"] == 200 - sum(over)


def test_trace_timeline_of_a_step():
    # the executor's per-call timeline: one record per library call, each on the stream it was
    # issued on; a ZeRO-1 step of short buckets spreads its bucket launches over several streams
    from zero_partitioned_mixed_replica_gb300 import binding as Bd
    c = Case([200_000, 1600, 99_999, 333], 8, 1, FMT_BF16, bucket_elems=32_768)
    eng = _engine(c)
    eng.load_master(torch.from_numpy(c.master0(c.layout())))
    eng.step()
    torch.cuda.synchronize()
    Bd.zero_trace_read(reset=True)
    Bd.zero_trace_enable(True)
    try:
        Bd.zero_launch_count(reset=True)
        eng.step()
        eng.step()
        torch.cuda.synchronize()
        launches = Bd.zero_launch_count()
        tl = Bd.zero_trace_timeline()
        totals = Bd.zero_trace_read(reset=True)
    finally:
        Bd.zero_trace_enable(False)
    assert len(tl) == sum(v["launches"] for v in totals.values())     # one record per library call
    assert {r["kind"] for r in tl} == {"fused_step", "grad_norm"}
    assert launches == len(tl) + sum(r["kind"] == "grad_norm" for r in tl)   # the norm call is two kernels
    assert all(r["end_ms"] >= r["start_ms"] >= 0.0 for r in tl)
    buckets = eng.n_buckets
    assert sum(r["kind"] == "fused_step" for r in tl) == 2 * buckets
    assert len({r["stream"] for r in tl if r["kind"] == "fused_step"}) >= 2
    norm = [r for r in tl if r["kind"] == "grad_norm"]
    fused = [r for r in tl if r["kind"] == "fused_step"]
    # each step's norm starts after that step's last bucket launch has ended (the lanes join first)
    assert norm[0]["start_ms"] >= max(r["end_ms"] for r in fused[:buckets]) - 1e-3
