"""Seeded random layouts through the library's host layout code (C ABI)
against the oracle's, with no GPU: 400 valid layouts (N_d 1-64, stages 0-3,
1-12 tensors of 1 to ~1M elements, buckets, pad multiples, ZeRO-3 unit ids in
any order) must give identical sizes, buckets, units, tensor offsets, memory
and volume accounting; 200 invalid ones must be rejected by both sides (or by
the library alone for the limits only it has); and reshard plans between 40
random pairs of layouts of the same tensors must move every real element
exactly once to where the oracle's target layout owns it."""
import numpy as np
import pytest

from oracle.layout import layout_comm_elems, layout_memory_bytes, make_layout
from zero_partitioned_mixed_replica_gb300 import binding as B
from zero_partitioned_mixed_replica_gb300 import build as zbuild


@pytest.fixture(scope="module", autouse=True)
def _built():
    zbuild.build()


def _valid(rng, max_elems=1_000_000, max_tensors=12):
    n_d = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 16, 33, 64]))
    stage = int(rng.integers(0, 4))
    n_t = int(rng.integers(1, max_tensors + 1))
    numels = [int(x) for x in np.exp(rng.uniform(0.0, np.log(max_elems), n_t)).astype(np.int64) + 1]
    bucket = 0 if rng.random() < 0.3 else 32 * int(np.exp(rng.uniform(0.0, np.log(200_000))))
    pad = 0 if rng.random() < 0.6 else n_d * 128 * int(rng.integers(1, 5))
    units = None
    if stage == 3:
        n_u = int(rng.integers(1, n_t + 1))
        units = list(range(n_u)) + [int(x) for x in rng.integers(0, n_u, n_t - n_u)]
        rng.shuffle(units)
    return numels, n_d, stage, bucket, pad, units


def _compare(numels, n_d, stage, bucket, pad, units):
    L = B.zero_layout_init(numels, units, n_d, stage, pad, bucket, B.ZERO_BF16)
    O = make_layout(numels, n_d, stage, bucket_elems=bucket, unit_of_tensor=units, pad_multiple=pad)
    info = B.zero_layout_query(L)
    assert (info.psi, info.psi_pad, info.shard_len, info.q) == (O.psi, O.psi_pad, O.shard_len, O.q)
    assert info.n_buckets == len(O.buckets) and info.n_units == len(O.units)
    assert [B.zero_layout_bucket(L, b) for b in range(info.n_buckets)] == O.buckets
    for u in range(info.n_units):
        ui, ou = B.zero_layout_unit(L, u), O.units[u]
        assert (ui.offset, ui.real, ui.padded, ui.shard, ui.shard_base) == \
               (ou.offset, ou.real, ou.padded, ou.shard, ou.shard_base)
    assert [B.zero_layout_tensor_offset(L, t) for t in range(len(numels))] == O.tensor_offsets
    mem, comm = layout_memory_bytes(O), layout_comm_elems(O)
    assert (info.mem_formula, info.mem_state, info.mem_gshard, info.mem_transient, info.mem_peak) == \
           (mem["formula"], mem["state"], mem["gshard"], mem["transient"], mem["peak"])
    assert (info.comm_rs, info.comm_ag, info.comm_ag_fwd, info.comm_ag_bwd, info.comm_allreduce,
            info.comm_total) == (comm["rs"], comm["ag"], comm["ag_fwd"], comm["ag_bwd"], comm["allreduce"],
                                 comm["total"])


@pytest.mark.parametrize("chunk", range(8))
def test_random_layouts_match_the_oracle(chunk):
    rng = np.random.default_rng(7000 + chunk)
    for _ in range(50):
        _compare(*_valid(rng))


def _invalid(rng):
    """A valid layout with one thing broken; returns (args, oracle_rejects_too)."""
    numels, n_d, stage, bucket, pad, units = _valid(rng, 100_000, 8)
    kind = int(rng.integers(0, 7))
    if kind == 0:
        numels[int(rng.integers(0, len(numels)))] = 0                  # an empty tensor
        return (numels, n_d, stage, bucket, pad, units), True
    if kind == 1:
        pad = n_d * 128 * int(rng.integers(1, 4)) + int(rng.integers(1, n_d * 128))   # not a multiple of q
        return (numels, n_d, stage, bucket, pad, units), True
    if kind == 2:
        n_d = 0
        return (numels, n_d, stage, bucket, 0, units), True
    if kind == 3:                                                      # ZeRO-3 with a unit id skipped
        numels = numels + [int(rng.integers(1, 1000))]
        units = [0] * (len(numels) - 1) + [2]
        return (numels, n_d, 3, 0, pad, units), True
    if kind == 4:                                                      # ZeRO-3 without unit ids
        return (numels, n_d, 3, 0, pad, None), True
    if kind == 5:
        n_d = int(rng.integers(65, 200))                               # above the library's rank limit
        return (numels, n_d, stage, bucket, 0, units), False
    bucket = 32 * int(rng.integers(1, 1000)) + int(rng.integers(1, 32))    # not a multiple of 32
    return (numels, n_d, stage, bucket, pad, units), False


def test_random_invalid_layouts_are_rejected():
    rng = np.random.default_rng(8000)
    for _ in range(200):
        (numels, n_d, stage, bucket, pad, units), both = _invalid(rng)
        with pytest.raises(B.ZeroError) as e:
            B.zero_layout_init(numels, units, n_d, stage, pad, bucket, B.ZERO_BF16)
        assert e.value.status == B.ZERO_ERR_INVALID
        if both:
            with pytest.raises(ValueError):
                make_layout(numels, n_d, stage, bucket_elems=bucket, unit_of_tensor=units, pad_multiple=pad)


def _tags(L):
    """Per-rank shards holding 1 + the element's index among all real
    elements (tensors concatenated) at every real element, 0 in padding."""
    shards = [np.zeros(L.shard_len, np.int64) for _ in range(L.n_d)]
    base = 1
    for off, n in zip(L.tensor_offsets, L.numels):
        for e in range(n):
            r, j = L.owner(off + e)
            shards[r][j] = base + e
        base += n
    return shards


def test_random_reshard_plans_move_every_element():
    rng = np.random.default_rng(9000)
    for _ in range(40):
        a = _valid(rng, 3000, 6)
        numels = a[0]
        b = _valid(rng, 3000, 6)
        n_t = len(numels)
        # the second layout holds the same tensors: redraw its unit ids for their count
        nd_b, st_b, bk_b, pd_b = b[1], max(1, b[2]), b[3], b[4]
        ub = None
        if st_b == 3:
            n_u = int(rng.integers(1, n_t + 1))
            ub = list(range(n_u)) + [int(x) for x in rng.integers(0, n_u, n_t - n_u)]
            rng.shuffle(ub)
        st_a = max(1, a[2])
        ua = a[5] if st_a == 3 and a[5] is not None else (list(range(n_t)) if st_a == 3 else None)
        La = make_layout(numels, a[1], st_a, bucket_elems=a[3], unit_of_tensor=ua, pad_multiple=a[4])
        Lb = make_layout(numels, nd_b, st_b, bucket_elems=bk_b, unit_of_tensor=ub, pad_multiple=pd_b)
        ca = B.zero_layout_init(numels, ua, a[1], st_a, a[4], a[3], B.ZERO_BF16)
        cb = B.zero_layout_init(numels, ub, nd_b, st_b, pd_b, bk_b, B.ZERO_BF16)
        src = _tags(La)
        dst = [np.zeros(Lb.shard_len, np.int64) for _ in range(nd_b)]
        moved = 0
        for sr, so, dr, do, n in B.zero_reshard_plan(ca, cb):
            assert n > 0
            assert not dst[dr][do:do + n].any(), "an element is written twice"
            dst[dr][do:do + n] = src[sr][so:so + n]
            moved += n
        assert moved == sum(numels)
        want = _tags(Lb)
        for r in range(nd_b):
            assert np.array_equal(dst[r], want[r])
