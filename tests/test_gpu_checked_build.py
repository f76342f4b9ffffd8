"""The bounds-checked build (libzero_checked.so, -DZK_CHECKED): every global
access of every kernel is tested against the extent the layout gives its
buffer, and one outside is skipped and counted instead of made.  It stands in
for a memory checker: the GPU parity, random-layout, host-input,
accumulation, guard-band and launch-shape suites run again against it, and
after each test the count must be zero (tests/conftest.py).  A positive
control shortens every checked extent (the build's test hook) so that each
kind of launch reports the accesses it skipped, with the buffers whole and
no fault."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    return build.build(checked=True)


def _env(lib):
    env = dict(os.environ)
    env["ZERO_LIB"] = lib
    return env


def test_suites_run_inside_their_buffers(checked_lib):
    files = ["tests/test_gpu_parity.py", "tests/test_gpu_random_layouts.py", "tests/test_gpu_host_input.py",
             "tests/test_gpu_accum.py", "tests/test_gpu_guards.py", "tests/test_gpu_launch_shape.py"]
    p = subprocess.run([sys.executable, "-m", "pytest", *files, "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=_env(checked_lib), capture_output=True, text=True, timeout=1500)
    assert p.returncode == 0, p.stdout[-4000:] + p.stderr[-2000:]
    assert " passed" in p.stdout


CONTROL = r"""
import sys, torch
from zero_partitioned_mixed_replica_gb300 import binding as B, synth
from zero_partitioned_mixed_replica_gb300.engine import ZeroStep
assert B.zero_checked_build()
numels = [40000, 333, 70001, 5]
res = {}
for name, kw in (("z2_split", dict(n_d=8, stage=2, bucket_elems=16384, max_norm=1.0)),
                 ("z2_fused", dict(n_d=4, stage=2, bucket_elems=16384)),
                 ("z2_ldg", dict(n_d=2, stage=2, max_norm=1.0)),
                 ("z1_unfused_ag", dict(n_d=8, stage=1, max_norm=1.0, fuse_allgather=False)),
                 ("z3_split", dict(n_d=4, stage=3, unit_of_tensor=[0, 1, 1, 2], max_norm=1.0)),
                 ("z3_fused", dict(n_d=2, stage=3, unit_of_tensor=[0, 1, 1, 2])),
                 ("z1_accum", dict(n_d=4, stage=1, bucket_elems=16384, n_micro=2))):
    eng = ZeroStep(numels, **kw)
    m0 = synth.master_init(numels, eng.tensor_offsets, eng.info.psi_pad, device=eng.device)
    eng.load_master(m0)
    for r in range(eng.n_d):
        synth.grad_replica(numels, eng.tensor_offsets, eng.info.psi_pad, eng.dtype, r, 1, 1e-3, out=eng.grads[r])
    run = (lambda: [eng.micro_step(m) for m in range(2)]) if kw.get("n_micro") else eng.step
    run()
    assert B.zero_bounds_violations(reset=True) == 0, name           # exact extents: nothing skipped
    B.zero_checked_set_slack(64)
    eng.load_master(m0)                                                # the cast kernel too
    cast_hits = B.zero_bounds_violations(reset=True)
    run()
    hits = B.zero_bounds_violations(reset=True)
    assert cast_hits > 0, name
    B.zero_checked_set_slack(0)
    run()
    torch.cuda.synchronize()
    assert B.zero_bounds_violations(reset=True) == 0, name
    assert eng.read_state()["error"] == 0, name                        # the empty TMA tiles did not time out
    res[name] = hits
print(res)
assert all(v > 0 for v in res.values()), res
"""


def test_checks_fire_when_the_extents_are_short(checked_lib):
    p = subprocess.run([sys.executable, "-c", CONTROL], cwd=ROOT, env=_env(checked_lib), capture_output=True,
                       text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-3000:] + p.stderr[-3000:]
