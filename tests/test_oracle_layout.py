"""Oracle pins: the flat layout by brute force on tiny inputs, and the model
parameter counts of the workloads (public figures of the named models)."""
import pytest

from oracle.layout import make_layout
from zero_partitioned_mixed_replica_gb300 import workloads


@pytest.mark.parametrize("n_d", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("stage", [1, 2, 3])
def test_every_index_has_exactly_one_owner(n_d, stage):
    for numels in ([1], [7], [64], [5, 9, 1], [128 * n_d], [128 * n_d + 1, 3]):
        units = [i % 2 for i in range(len(numels))] if len(numels) > 1 else [0]
        if stage == 3 and len(numels) > 1 and len(set(units)) < 2:
            continue
        L = make_layout(numels, n_d, stage, unit_of_tensor=units)
        assert L.psi == sum(numels)
        assert L.psi_pad % (n_d * 128) == 0 or stage == 3
        seen = {}
        for i in range(L.psi_pad):
            r, j = L.owner(i)
            assert 0 <= r < n_d and 0 <= j < L.shard_len
            assert (r, j) not in seen
            seen[(r, j)] = i
            assert L.flat_index(r, j) == i
        assert len(seen) == n_d * L.shard_len == L.psi_pad
        # tensors are back to back inside their segment and never overlap pads
        covered = set()
        for t, (n, off) in enumerate(zip(L.numels, L.tensor_offsets)):
            rng = set(range(off, off + n))
            assert not (rng & covered)
            covered |= rng
            assert not any(L.is_pad(i) for i in rng)
        pads = {i for i in range(L.psi_pad) if L.is_pad(i)}
        assert covered | pads == set(range(L.psi_pad)) and not (covered & pads)


def test_zero12_shards_are_contiguous_ranges():
    L = make_layout([1000, 24], 4, 2, bucket_elems=96)
    S = L.psi_pad // 4
    assert L.shard_len == S == 256
    for i in range(L.psi_pad):
        assert L.owner(i) == (i // S, i % S)
    # buckets tile the padded buffer in order, independent of shard boundaries
    assert L.buckets[0] == (0, 96) and L.buckets[-1][1] == L.psi_pad
    assert all(a[1] == b[0] for a, b in zip(L.buckets, L.buckets[1:]))
    assert sum(e - b for b, e in L.buckets) == L.psi_pad


def test_zero3_units_padded_separately():
    L = make_layout([10, 20, 300, 5], 2, 3, unit_of_tensor=[1, 0, 1, 2])
    # flat order is unit by unit; inside a unit tensors keep declaration order
    u0, u1, u2 = L.units
    assert (u0.offset, u0.real, u0.padded) == (0, 20, 256)
    assert (u1.offset, u1.real, u1.padded) == (256, 310, 512)
    assert (u2.offset, u2.real, u2.padded) == (768, 5, 256)
    assert L.tensor_offsets == [256, 0, 266, 768]
    assert [u.shard for u in L.units] == [128, 256, 128]
    assert [u.shard_base for u in L.units] == [0, 128, 384]
    assert L.shard_len == 512 and L.psi_pad == 1024
    assert L.buckets == [(0, 256), (256, 768), (768, 1024)]


def test_pad_multiple_override():
    L = make_layout([1000], 2, 1, pad_multiple=1024)
    assert L.psi_pad == 1024
    with pytest.raises(ValueError):
        make_layout([1000], 2, 1, pad_multiple=100)


def test_bad_arguments_rejected():
    for args in (([], 2, 1), ([0], 2, 1), ([5], 0, 1), ([5], 2, 4), ([5, 6], 2, 3)):
        with pytest.raises(ValueError):
            make_layout(*args)
    with pytest.raises(ValueError):
        make_layout([5, 6], 2, 3, unit_of_tensor=[0, 2])   # unit 1 empty


def test_workload_parameter_counts():
    # Public parameter counts of the named architectures.
    assert workloads.gpt2_small().psi == 124_439_808
    assert workloads.gpt2_xl().psi == 1_557_611_200
    assert workloads.llama7b().psi == 6_738_415_616
    assert workloads.gpt2_medium_odd().psi == 354_823_168 + 1
    assert workloads.tiny().psi == 1_002_003


def test_workload_layout_sizes():
    w = workloads.gpt2_xl()
    L = make_layout(w.numels, w.n_d, w.stage, bucket_elems=w.bucket_elems)
    assert (L.psi_pad, L.shard_len, len(L.buckets)) == (1_557_611_520, 194_701_440, 4)
    w = workloads.gpt2_small()
    L = make_layout(w.numels, w.n_d, w.stage, bucket_elems=w.bucket_elems)
    assert (L.psi_pad, L.shard_len, len(L.buckets)) == (124_440_576, 15_555_072, 25)
    assert L.buckets[-1][1] - L.buckets[-1][0] == 4_440_576
    w = workloads.llama7b()
    L = make_layout(w.numels, w.n_d, w.stage, unit_of_tensor=w.unit_of_tensor)
    assert len(L.units) == 33
    assert L.units[0].real == L.units[0].padded == 262_148_096
    assert all(u.real == u.padded == 202_383_360 for u in L.units[1:])
    assert L.psi_pad == w.psi
    w = workloads.tiny()
    L = make_layout(w.numels, w.n_d, w.stage)
    assert (L.psi_pad, L.shard_len) == (1_002_496, 250_624)
    w = workloads.gpt2_medium_odd(n_d=64)
    L = make_layout(w.numels, 64, 2, bucket_elems=100_000)
    assert L.psi_pad == 354_828_288 and len(L.buckets) == 3549
