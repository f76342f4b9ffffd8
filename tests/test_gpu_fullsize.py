"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (ZeroStep with the workload's settings).

* GPT-2 small (124M, N_d = 8, ZeRO-1, bucket 5e6, 10 steps): the whole buffer
  against the literal ZeRO simulation of the oracle, every element.
* GPT-2 1.5B (N_d = 8, ZeRO-2, fp16 x 2^16 dynamic scale, clip 1.0, +inf in
  rank 3 at step 4; all 10 steps): step flags, counters and loss scale exact;
  the global norm against the oracle's own sum over every gradient element;
  master/m/v and every 16-bit replica, every element, against the oracle's
  per-element update driven by its own decisions.  The buffers are streamed
  through the oracle in contiguous shard pieces of at most 64M elements.
* Llama-style 7B (N_d = 2, ZeRO-3, 33 units; 3 steps): every element of the
  rank shards and 16-bit shards, the reported norm against the oracle's sum,
  and every forward and backward transient of all 33 units against the
  oracle's previous parameters.
* GPT-2 medium 350M + 1 sweep points (odd Psi, N_d up to 64): sampled
  outputs and the norm against the oracle's sum over every element.

Inputs are drawn on the GPU by the input generator and copied to the host for
the oracle; no expected value comes from the CUDA path.  Comparisons of whole
buffers run on the device, against the oracle's values copied there."""
import bisect
import math

import numpy as np
import pytest
import torch

from oracle.layout import make_layout
from oracle.step import AdamWHP, FullSumsq, SampledElements, StepState, ZeroSimulation

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_key(h):
    h = h.astype(np.int64)
    return np.where(h & 0x8000, -(h & 0x7FFF), h)


def assert_state_close(gpu, ref, what):
    d = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    big = np.abs(ref) >= 1e-30
    bad = np.flatnonzero((big & (d > 1e-6 * np.abs(ref))) | (~big & (d > 1e-36)))
    assert bad.size == 0, "%s: %d out of tolerance, e.g. %s vs %s" % (what, bad.size, gpu[bad[:3]], ref[bad[:3]])


def assert_p16_close(gpu, ref, what):
    dist = np.abs(_ulp_key(gpu) - _ulp_key(ref))
    assert dist.max(initial=0) <= 1, "%s: %d ulp" % (what, dist.max())


def _engine(w):
    from zero_partitioned_mixed_replica_gb300.engine import AdamW, ZeroStep
    return ZeroStep(w.numels, w.n_d, w.stage, w.dtype, w.bucket_elems if w.stage != 3 else 0,
                    w.unit_of_tensor if w.stage == 3 else None,
                    AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay), w.max_norm, w.loss_scale,
                    w.dynamic_scale, w.growth_interval)


def _hp(w):
    return AdamWHP(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)


def _oracle_layout(w):
    return make_layout(w.numels, w.n_d, w.stage, bucket_elems=w.bucket_elems if w.stage != 3 else 0,
                       unit_of_tensor=w.unit_of_tensor if w.stage == 3 else None)


def _fill_grads(eng, w, step, loss_scale):
    from zero_partitioned_mixed_replica_gb300 import synth
    scales = synth.tensor_scales(len(w.numels)) if w.per_tensor_scale else None
    for r in range(w.n_d):
        synth.grad_replica(w.numels, eng.tensor_offsets, eng.info.psi_pad, w.dtype, r, step, w.grad_std, scales,
                           loss_scale, device=eng.device, out=eng.grads[r])
        if w.inf_step == step and r == w.inf_rank:
            synth.plant_inf(eng.grads[r], w.psi // 2)


def _sample_indices(L, n_random=40_000, seed=5):
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, L.psi_pad, size=n_random).tolist())
    edges = set()
    for b0, b1 in L.buckets:
        edges.update([b0, b1])
    for u in L.units:
        for r in range(L.n_d + 1):
            edges.add(u.offset + r * u.shard)
        edges.update([u.offset + u.real, u.offset + u.padded])
    for off in L.tensor_offsets[:64] + L.tensor_offsets[-64:]:
        edges.add(off)
    for e in edges:
        for d in (-2, -1, 0, 1, 2):
            if 0 <= e + d < L.psi_pad:
                idx.add(e + d)
    return np.array(sorted(idx), dtype=np.int64)


def _owners(L, idx):
    """Flat indices -> (rank, shard offset) arrays."""
    offs = [u.offset for u in L.units]
    r = np.empty(idx.size, np.int64)
    j = np.empty(idx.size, np.int64)
    for n, i in enumerate(idx.tolist()):
        u = L.units[bisect.bisect_right(offs, i) - 1]
        k = i - u.offset
        r[n] = k // u.shard
        j[n] = u.shard_base + k - r[n] * u.shard
    return r, j


def _full_sumsq(eng, w, D, block=None):
    # at most ~1 GB of host copies per block, whatever N_d
    block = block or max(1 << 20, (1 << 29) // w.n_d // 128 * 128)
    acc = FullSumsq(w.dtype, D)
    P = eng.info.psi_pad
    for b in range(0, P, block):
        e = min(P, b + block)
        acc.add([_u16(eng.grads[r, b:e]) for r in range(w.n_d)])
    return acc.result()


def _pieces(L, block=1 << 26):
    """The flat buffer as contiguous pieces (lo, hi, rank, shard offset) that
    are also contiguous in one rank's shard: every unit's rank slices, split
    into blocks of at most ``block`` elements (multiples of 128)."""
    out = []
    for u in L.units:
        for r in range(L.n_d):
            lo0 = u.offset + r * u.shard
            for lo in range(lo0, lo0 + u.shard, block):
                hi = min(lo0 + u.shard, lo + block)
                out.append((lo, hi, r, u.shard_base + lo - lo0))
    return out


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int32) if a.element_size() == 4 else a.view(torch.int16),
                       b.view(torch.int32) if b.element_size() == 4 else b.view(torch.int16))


def _close_on_device(gpu: torch.Tensor, ref: torch.Tensor, what: str):
    d = (gpu.double() - ref.double()).abs()
    big = ref.abs() >= 1e-30
    bad = int(((big & (d > 1e-6 * ref.double().abs())) | (~big & (d > 1e-36))).sum())
    assert bad == 0, "%s: %d elements out of tolerance" % (what, bad)


def _p16_close_on_device(gpu: torch.Tensor, ref: torch.Tensor, what: str):
    def key(h):
        h = h.view(torch.int16).to(torch.int32) & 0xFFFF
        return torch.where(h >= 0x8000, -(h & 0x7FFF), h)
    dist = int((key(gpu) - key(ref)).abs().max()) if gpu.numel() else 0
    assert dist <= 1, "%s: %d ulp" % (what, dist)


def _whole_buffer_run(w, steps, check_transients=False):
    """Every element of the step's outputs against the oracle, streamed in
    shard pieces; every ZeRO-3 transient against the oracle's previous
    parameters."""
    from zero_partitioned_mixed_replica_gb300 import synth
    L = _oracle_layout(w)
    eng = _engine(w)
    dev = eng.device
    assert eng.tensor_offsets == L.tensor_offsets and eng.info.psi_pad == L.psi_pad
    m0 = synth.master_init(w.numels, eng.tensor_offsets, L.psi_pad, w.master_std, device=dev)
    eng.load_master(m0)
    pieces = _pieces(L)
    samp = [SampledElements(m0[lo:hi].cpu().numpy(), w.dtype, _hp(w)) for lo, hi, _, _ in pieces]
    del m0
    st = StepState(w.loss_scale, w.dynamic_scale, w.growth_interval)
    seen, prev_cache = [], {}
    if check_transients:
        by_unit = {}
        for k, (lo, hi, r, j0) in enumerate(pieces):
            for ui, u in enumerate(L.units):
                if u.offset <= lo < u.offset + u.padded:
                    by_unit.setdefault(ui, []).append(k)

        def hook(kind, ui, rows):
            # the oracle's previous 16-bit parameters of the unit: its pieces in flat order
            # (unchanged during the GPU step: the forward and backward gathers share one device copy)
            u = L.units[ui]
            if ui not in prev_cache:
                prev = np.concatenate([samp[k].p16 for k in sorted(by_unit[ui], key=lambda k: pieces[k][0])])
                prev_cache[ui] = torch.from_numpy(prev[:u.real].view(np.int16)).to(dev)
            ref = prev_cache[ui]
            for q, row in enumerate(rows):
                assert _same_bits(row[:u.real], ref), (kind, ui, q)
            seen.append((kind, ui))
        eng.transient_hook = hook
    hist = []
    for s in range(1, steps + 1):
        _fill_grads(eng, w, s, st.loss_scale)
        D = st.divisor(w.n_d)
        bad, sumsq = _full_sumsq(eng, w, D)
        seen.clear()
        prev_cache.clear()
        eng.step()
        g = eng.read_state()
        apply, norm, clip = st.decide(bad, sumsq, w.max_norm)
        hist.append(g)
        assert (g["overflow"], g["t"], g["skipped"], g["error"]) == (int(bad), st.t, st.skipped, 0), s
        assert g["loss_scale"] == st.loss_scale
        if bad:
            assert math.isinf(g["grad_norm"])
        else:
            assert g["grad_norm"] == pytest.approx(norm, rel=1e-5)
            assert abs(g["grad_norm"] - norm) <= 1e-9 * norm
        if check_transients:
            U = len(L.units)
            assert seen == [("fwd", u) for u in range(U)] + [("bwd", u) for u in reversed(range(U))]
        same_clip = np.float32(g["clip_coef"]) == np.float32(clip)
        for k, (lo, hi, r, j0) in enumerate(pieces):
            sp = samp[k]
            sp.step([_u16(eng.grads[q, lo:hi]) for q in range(w.n_d)], D, apply, st.t, clip)
            n = hi - lo
            for name, ref in (("master", sp.master), ("m", sp.m), ("v", sp.v)):
                gpu = getattr(eng, name)[r, j0:j0 + n]
                tref = torch.from_numpy(ref).to(dev)
                if same_clip:
                    assert _same_bits(gpu, tref), "%s step %d piece %d" % (name, s, k)
                else:
                    _close_on_device(gpu, tref, "%s step %d piece %d" % (name, s, k))
            p16 = torch.from_numpy(sp.p16.view(np.int16)).to(dev)
            outs = [eng.shard16[r, j0:j0 + n]] if w.stage == 3 else [eng.params[q, lo:hi] for q in range(w.n_d)]
            for q, o in enumerate(outs):
                if same_clip:
                    assert _same_bits(o, p16), "16-bit output %d step %d piece %d" % (q, s, k)
                else:
                    _p16_close_on_device(o, p16, "16-bit output %d step %d piece %d" % (q, s, k))
    return hist


def test_gpt2_small_whole_buffer_against_simulation():
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.gpt2_small()
    L = _oracle_layout(w)
    eng = _engine(w)
    assert eng.tensor_offsets == L.tensor_offsets and eng.info.psi_pad == L.psi_pad
    from zero_partitioned_mixed_replica_gb300 import synth
    m0 = synth.master_init(w.numels, eng.tensor_offsets, L.psi_pad, w.master_std, device=eng.device)
    eng.load_master(m0)
    zs = ZeroSimulation(L, m0.cpu().numpy(), w.dtype, _hp(w))
    for s in range(1, w.steps + 1):
        _fill_grads(eng, w, s, 1.0)
        reps = [_u16(eng.grads[r]) for r in range(w.n_d)]
        eng.step()
        g = eng.read_state()
        o = zs.step(reps)
        assert (g["t"], g["overflow"], g["error"]) == (o["t"], 0, 0)
        assert g["grad_norm"] == pytest.approx(o["norm"], rel=1e-5)
        for name in ("master", "m", "v"):
            gpu, ref = eng.flat(name).cpu().numpy(), zs.flat(name)
            assert_state_close(gpu, ref, "%s step %d" % (name, s))
            assert np.array_equal(gpu.view(np.uint32), ref.view(np.uint32)), "%s step %d" % (name, s)
    for r in range(w.n_d):
        assert np.array_equal(_u16(eng.params[r]), zs.params16[r])


def _sampled_run(w, steps, check_transients=(), check_norm=True):
    from zero_partitioned_mixed_replica_gb300 import synth
    L = _oracle_layout(w)
    eng = _engine(w)
    assert eng.tensor_offsets == L.tensor_offsets and eng.info.psi_pad == L.psi_pad
    m0 = synth.master_init(w.numels, eng.tensor_offsets, L.psi_pad, w.master_std, device=eng.device)
    eng.load_master(m0)
    idx = _sample_indices(L)
    r_idx, j_idx = _owners(L, idx)
    tr, tj = torch.from_numpy(r_idx).to(eng.device), torch.from_numpy(j_idx).to(eng.device)
    ti = torch.from_numpy(idx).to(eng.device)
    samp = SampledElements(m0[ti].cpu().numpy(), w.dtype, _hp(w))
    del m0
    st = StepState(w.loss_scale, w.dynamic_scale, w.growth_interval)
    seen = {}
    if check_transients:
        units = {u: L.units[u] for u in check_transients}

        def hook(kind, u, rows):
            if u in units:
                torch.cuda.synchronize()
                lo = units[u].offset
                pos = idx[(idx >= lo) & (idx < lo + units[u].real)] - lo
                tp = torch.from_numpy(pos).to(eng.device)
                seen[(kind, u)] = (pos, [_u16(row[tp]) for row in rows])
        eng.transient_hook = hook
    hist = []
    for s in range(1, steps + 1):
        _fill_grads(eng, w, s, st.loss_scale)
        D = st.divisor(w.n_d)
        if check_norm:
            bad, sumsq = _full_sumsq(eng, w, D)
        else:   # no clipping and no scaler: the update needs no norm; nothing non-finite is planted
            bad, sumsq = False, 0.0
        reps = [_u16(eng.grads[r][ti]) for r in range(w.n_d)]
        p16_before = samp.p16.copy()
        seen.clear()
        eng.step()
        g = eng.read_state()
        apply, norm, clip = st.decide(bad, sumsq, w.max_norm)
        samp.step(reps, D, apply, st.t, clip)
        hist.append(g)
        assert (g["overflow"], g["t"], g["skipped"], g["error"]) == (int(bad), st.t, st.skipped, 0), s
        assert g["loss_scale"] == st.loss_scale
        if bad:
            assert math.isinf(g["grad_norm"])
        elif check_norm:
            assert g["grad_norm"] == pytest.approx(norm, rel=1e-5)
        for name, ref in (("master", samp.master), ("m", samp.m), ("v", samp.v)):
            gpu = getattr(eng, name)[tr, tj].cpu().numpy()
            assert_state_close(gpu, ref, "%s step %d" % (name, s))
            if np.float32(g["clip_coef"]) == np.float32(clip):
                assert np.array_equal(gpu.view(np.uint32), ref.view(np.uint32)), "%s step %d" % (name, s)
        if w.stage == 3:
            assert_p16_close(_u16(eng.shard16[tr, tj]), samp.p16, "shard16 step %d" % s)
        else:
            for r in range(w.n_d):
                assert_p16_close(_u16(eng.params[r][ti]), samp.p16, "params[%d] step %d" % (r, s))
        for (kind, u), (pos, rows) in seen.items():
            lo = L.units[u].offset
            sel = np.searchsorted(idx, pos + lo)
            for row in rows:
                assert np.array_equal(row, p16_before[sel]), (kind, u, s)
    return hist


def test_gpt2_xl_fp16_overflow_and_clip_every_element():
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.gpt2_xl()
    hist = _whole_buffer_run(w, w.steps)
    assert [g["overflow"] for g in hist] == [0, 0, 0, 1] + [0] * (w.steps - 4)
    assert [g["loss_scale"] for g in hist] == [65536.0] * 3 + [32768.0] * (w.steps - 3)
    assert [g["t"] for g in hist] == [1, 2, 3, 3] + list(range(4, w.steps))
    assert all(g["clip_coef"] < 1.0 for g in hist if not g["overflow"])


def test_llama7b_zero3_every_element_and_every_transient():
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.llama7b()
    hist = _whole_buffer_run(w, 3, check_transients=True)
    assert [g["t"] for g in hist] == [1, 2, 3]


@pytest.mark.parametrize("n_d,stage,bucket", [(64, 2, 100_000), (16, 3, 0), (2, 1, 50_000_000)])
def test_gpt2_medium_sweep_points_sampled(n_d, stage, bucket):
    # sampled outputs; the norm against the oracle's sum over every element, N_d = 64 included
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.gpt2_medium_odd(n_d=n_d, stage=stage, bucket_elems=bucket)
    assert w.psi % 2 == 1
    _sampled_run(w, 2, check_norm=True)
