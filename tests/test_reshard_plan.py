"""The reshard plan (host C ABI) against the oracle's layouts: moving a
tagged copy of every source shard through the plan must put each real
element exactly where the oracle's target layout owns it, and touch no
padding."""
import itertools

import numpy as np
import pytest

from oracle.layout import make_layout
from zero_partitioned_mixed_replica_gb300 import binding as B
from zero_partitioned_mixed_replica_gb300 import build as zbuild


@pytest.fixture(scope="module", autouse=True)
def _built():
    zbuild.build()


NUMELS = [1000, 24, 300, 7, 4096, 1]
UNITS_A = [0, 1, 1, 2, 2, 0]
UNITS_B = [0, 0, 1, 1, 2, 3]
LAYOUTS = [(4, 2, None, 0), (2, 3, UNITS_A, 0), (3, 1, None, 640), (8, 3, UNITS_B, 0), (1, 2, None, 0),
           (5, 2, None, 96)]


def _tags(L):
    """Per-rank shards holding, at every real element, 1 + its index in the
    concatenation of all tensors; 0 in padding."""
    shards = [np.zeros(L.shard_len, np.int64) for _ in range(L.n_d)]
    base = 1
    for off, n in zip(L.tensor_offsets, L.numels):
        for e in range(n):
            r, j = L.owner(off + e)
            shards[r][j] = base + e
        base += n
    return shards


@pytest.mark.parametrize("a,b", list(itertools.permutations(range(len(LAYOUTS)), 2)))
def test_plan_moves_every_element_to_its_owner(a, b):
    (nda, sa, ua, ba), (ndb, sb, ub, bb) = LAYOUTS[a], LAYOUTS[b]
    La = make_layout(NUMELS, nda, sa, bucket_elems=ba, unit_of_tensor=ua)
    Lb = make_layout(NUMELS, ndb, sb, bucket_elems=bb, unit_of_tensor=ub)
    ca = B.zero_layout_init(NUMELS, ua, nda, sa, 0, ba, B.ZERO_BF16)
    cb = B.zero_layout_init(NUMELS, ub, ndb, sb, 0, bb, B.ZERO_BF16)
    plan = B.zero_reshard_plan(ca, cb)
    src = _tags(La)
    dst = [np.zeros(Lb.shard_len, np.int64) for _ in range(ndb)]
    moved = 0
    for sr, so, dr, do, n in plan:
        assert n > 0
        assert not dst[dr][do:do + n].any(), "an element is written twice"
        dst[dr][do:do + n] = src[sr][so:so + n]
        moved += n
    assert moved == sum(NUMELS)
    want = _tags(Lb)
    for r in range(ndb):
        assert np.array_equal(dst[r], want[r])


def test_plan_is_maximal_for_same_split():
    L = B.zero_layout_init(NUMELS, None, 4, 2, 0, 0, B.ZERO_BF16)
    L1 = B.zero_layout_init(NUMELS, None, 4, 1, 0, 512, B.ZERO_BF16)
    plan = B.zero_reshard_plan(L, L1)
    # tensors are back to back in both ZeRO-1/2 layouts: one segment per rank piece
    assert len(plan) == 4 and all(sr == dr and so == do for sr, so, dr, do, n in plan)


def test_plan_rejects_different_tensors():
    a = B.zero_layout_init([10, 20], None, 2, 2, 0, 0, B.ZERO_BF16)
    b = B.zero_layout_init([10, 21], None, 2, 2, 0, 0, B.ZERO_BF16)
    with pytest.raises(B.ZeroError) as e:
        B.zero_reshard_plan(a, b)
    assert e.value.status == B.ZERO_ERR_INVALID
