"""Seeded random layouts through the step executor, against the oracle bit for
bit: N_d from 1 to 64, ZeRO-1/2/3, one to seven tensors of 1 to ~300k
elements, bucket sizes from 32 elements to the whole buffer, bf16 and fp16
(with a loss scale, sometimes dynamic), clipping that does and does not bite,
an overflow planted in one rank at step 2 on the split path, the fused and
split paths, per-bucket and whole-buffer fused launches, an unfused
all-gather, random ZeRO-3 unit groupings with one or two live units, and
larger pad multiples; a third of the cases again with the replicas in pinned
host memory (zero_step_from_host, chunks of random size), and another third
accumulated over 2-4 micro-batches (zero_micro_step).  Each case's
parameters come from its seed alone, and the case id names them."""
import numpy as np
import pytest
import torch

from oracle.step import FMT_BF16, FMT_FP16
from tests._cases import Case
from tests.test_gpu_parity import run_parity

pytestmark = pytest.mark.gpu

N_CASES = 96


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from zero_partitioned_mixed_replica_gb300 import build
    build.build()


def draw_case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    n_d = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 33, 64]))
    stage = int(rng.integers(1, 4))
    n_t = int(rng.integers(1, 8))
    numels = [int(x) for x in np.exp(rng.uniform(0.0, np.log(300_000), n_t)).astype(np.int64) + 1]
    fmt = FMT_FP16 if rng.random() < 0.5 else FMT_BF16
    q = n_d * 128
    pad_multiple = q * int(rng.choice([1, 1, 1, 3])) if rng.random() < 0.3 else 0
    kind = rng.choice(["fused", "clip", "noclip_split", "scaler"])
    max_norm = {"fused": 0.0, "clip": 1e-4, "noclip_split": 1e3, "scaler": float(rng.choice([0.0, 1e-4]))}[kind]
    loss_scale, dynamic = 1.0, False
    if kind == "scaler" or (fmt == FMT_FP16 and kind != "fused"):
        loss_scale = float(2.0 ** int(rng.integers(0, 14)))
        dynamic = bool(rng.random() < 0.5)
    split = not (max_norm <= 0 and loss_scale == 1.0 and not dynamic)
    inf_step = 2 if split and rng.random() < 0.3 else None
    kw = {}
    units = None
    bucket = 0
    if stage == 3:
        cuts = sorted(set(int(x) for x in rng.integers(1, n_t, int(rng.integers(0, n_t)))) if n_t > 1 else [])
        units, u = [], 0
        for t in range(n_t):
            if t in cuts:
                u += 1
            units.append(u)
        kw["live_units"] = int(rng.integers(1, 3))
    else:
        bucket = int(rng.choice([0, 32 * int(rng.integers(1, 64)), 32 * int(rng.integers(64, 20_000))]))
        if not split:
            kw["per_bucket"] = bool(rng.random() < 0.7)
        elif rng.random() < 0.3:
            kw["fuse_allgather"] = False
    c = Case(numels, n_d, stage, fmt, bucket_elems=bucket, units=units, max_norm=max_norm, loss_scale=loss_scale,
             dynamic=dynamic, growth_interval=1, per_tensor_scale=bool(rng.random() < 0.5), inf_step=inf_step,
             inf_rank=int(rng.integers(0, n_d)), seed=int(rng.integers(1, 1 << 30)), pad_multiple=pad_multiple)
    return c, kw


def _id(seed: int) -> str:
    c, kw = draw_case(seed)
    return "s%d-nd%d-z%d-%s-t%d-b%d-mn%g-ls%g%s%s" % (
        seed, c.n_d, c.stage, "fp16" if c.fmt == FMT_FP16 else "bf16", len(c.numels), c.bucket_elems, c.max_norm,
        c.loss_scale, "-dyn" if c.dynamic else "", "-inf" if c.inf_step else "")


@pytest.mark.parametrize("seed", range(N_CASES), ids=[_id(s) for s in range(N_CASES)])
def test_random_layout_matches_the_oracle(seed):
    c, kw = draw_case(seed)
    _, _, hist = run_parity(c, 3, use_gpu_clip=True, **kw)
    if c.inf_step is not None:
        assert [g["overflow"] for g, _ in hist] == [0, 1, 0]


@pytest.mark.parametrize("seed", range(0, N_CASES, 3), ids=[_id(s) for s in range(0, N_CASES, 3)])
def test_random_layout_from_host_memory_matches_the_oracle(seed):
    # the same layouts with the replicas coming from pinned host memory through
    # zero_step_from_host, in chunks of a random size (a multiple of 8 elements)
    c, kw = draw_case(seed)
    chunk = 8 * int(np.random.default_rng(seed).integers(1, 40_000))
    _, _, hist = run_parity(c, 3, use_gpu_clip=True, host_input=chunk, **kw)
    if c.inf_step is not None:
        assert [g["overflow"] for g, _ in hist] == [0, 1, 0]


@pytest.mark.parametrize("seed", range(1, N_CASES, 3), ids=[_id(s) for s in range(1, N_CASES, 3)])
def test_random_layout_with_gradient_accumulation_matches_the_oracle(seed):
    # the same layouts accumulated over 2-4 micro-batches (zero_micro_step; the split step),
    # against the oracle's accumulation order for the stage
    from tests.test_gpu_accum import _run
    c, kw = draw_case(seed)
    M = int(np.random.default_rng(seed).integers(2, 5))
    _run(c, M=M, steps=2, use_gpu_clip=True, live_units=kw.get("live_units", 1))
