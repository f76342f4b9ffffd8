"""Failure detection on the GPU without a fault: the library's bounded
mbarrier wait (`mbar_wait_bounded`, used by the TMA-staged AdamW on every
tile) is run by a test program on a barrier that nothing completes.  It must
give up after about its 1 s limit, report the timeout to the host, and leave
the CUDA context usable: no trap, no fault, no hang."""
import os
import re
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounded_wait_gives_up_and_reports(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = str(tmp_path / "wait_timeout")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "zero_partitioned_mixed_replica_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "wait_timeout.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    m = re.search(r"wait_ok=(-?\d+) elapsed_ns=(\d+) err1=(-?\d+) err2=(-?\d+) counted=(-?\d+)", p.stdout)
    assert m, p.stdout + p.stderr
    ok, ns, e1, e2, n = (int(x) for x in m.groups())
    assert p.returncode == 0 and (ok, e1, e2, n) == (0, 0, 0, 64), p.stdout
    assert 0.9e9 <= ns <= 10e9, ns            # the 1 s limit, checked every 64 polls
