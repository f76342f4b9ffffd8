"""A plain C caller of the library (tests/native/c_step.c): built with gcc
against include/zero.h, linked to libzero.so and the CUDA runtime only, it
allocates its own device buffers with cudaMalloc and runs whole steps through
zero_step.  Its outputs are compared with the oracle's ZeRO-2 simulation bit
for bit: the header and the library stand on their own, without Python, torch
or the binding."""
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle.step import AdamWHP, FMT_BF16, ZeroSimulation
from tests._cases import Case

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def _cuda_lib_dir():
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
              "/usr/local/cuda/targets/x86_64-linux/lib"):
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    pytest.skip("libcudart.so not found")


def test_plain_c_caller_matches_the_oracle(tmp_path):
    pkg = os.path.join(ROOT, "zero_partitioned_mixed_replica_gb300")
    exe = str(tmp_path / "c_step")
    cudalib = _cuda_lib_dir()
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", "/usr/local/cuda/include", os.path.join(ROOT, "tests", "native", "c_step.c"),
                    "-L", pkg, "-lzero", "-L", cudalib, "-lcudart", "-Wl,-rpath," + pkg + ":" + cudalib,
                    "-o", exe], check=True, capture_output=True, timeout=300)
    c = Case([40_000, 33, 77_777, 5], 4, 2, FMT_BF16, per_tensor_scale=True)
    L = c.layout()
    m0 = c.master0(L).astype(np.float32)
    reps = c.grads(L, 1, 1.0)
    m0.tofile(str(tmp_path / "master.bin"))
    np.stack(reps).astype(np.uint16).tofile(str(tmp_path / "grads.bin"))
    steps = 3
    p = subprocess.run([exe, str(tmp_path), str(c.n_d), str(len(c.numels))] + [str(n) for n in c.numels] +
                       [str(steps)], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "c_step ok: t=%d" % steps in p.stdout
    zs = ZeroSimulation(L, m0, c.fmt, AdamWHP())
    for _ in range(steps):
        o = zs.step(reps)
    P = L.psi_pad
    for name in ("master", "m", "v"):
        got = np.fromfile(str(tmp_path / ("out_%s.bin" % name)), dtype=np.float32)
        assert got.size == P
        assert np.array_equal(got.view(np.uint32), zs.flat(name).view(np.uint32)), name
    params = np.fromfile(str(tmp_path / "out_params.bin"), dtype=np.uint16).reshape(c.n_d, P)
    for r in range(c.n_d):
        assert np.array_equal(params[r], zs.params16[r]), r
    from zero_partitioned_mixed_replica_gb300 import binding as B
    raw = (tmp_path / "out_state.bin").read_bytes()
    st = B.zero_step_state.from_buffer_copy(raw)
    assert st.t == steps and st.error == 0 and st.overflow == 0
    assert abs(st.grad_norm - o["norm"]) <= 2.0 ** -25 * (1 + 1e-6) * o["norm"]
