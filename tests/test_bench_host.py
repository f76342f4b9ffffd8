"""bench.py host logic without a GPU: the max-over-ranks timing of a
multi-rank run (two gloo ranks on the CPU, rendezvous on 127.0.0.1), the
reference arm's JSON line, and non-zero ranks of the reference arm exiting
without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    dist.barrier()
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True,
                          text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_json_line():
    import time
    t0 = time.perf_counter()
    p = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
              "--cpu-seconds", "0.5"])
    wall = time.perf_counter() - t0
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "params/s"
    assert (d["steps"], d["warmup"]) == (2, 1)        # exactly K timed and W untimed oracle steps
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]
    # every step is the whole workload and ms_per_step is measured: K steps fit in the run's wall time
    assert d["ms_per_step"] * d["steps"] / 1e3 <= wall
    assert "sample" not in d["config"] and "the whole layout" in d["cpu_baseline"]["sample"]
    assert d["value"] == pytest.approx(d["config"]["psi"] / (d["ms_per_step"] / 1e3), rel=1e-9)


def test_oracle_samples_are_whole_tensors_of_the_workload():
    import bench
    from zero_partitioned_mixed_replica_gb300 import synth, workloads
    w = workloads.gpt2_xl()
    numels, units, scales, desc = bench.oracle_sample(w, 2)
    assert len(numels) == 24 and units == [0] * 12 + [1] * 12
    assert numels == w.numels[2:26]                          # block 1 and block 2, after wte and wpe
    assert scales == synth.tensor_scales(len(w.numels))[2:26]  # each tensor keeps its own scale
    full = bench.oracle_sample(w, None)
    assert full[0] == w.numels and "whole layout" in full[3]
    gb = 10 ** 9
    assert bench.oracle_blocks_that_fit(w, 199 * gb) is None      # the 1.5B oracle state fits a 199 GB host
    k = bench.oracle_blocks_that_fit(w, 62 * gb)
    assert 1 <= k < 48
    assert bench.oracle_bytes(w, sum(bench.oracle_sample(w, k)[0])) <= 0.6 * 62 * gb


def test_reference_arm_nonzero_rank_exits_quietly():
    p = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0 and p.stdout.strip() == ""


@pytest.mark.parametrize("name,micro", [("gpt2_xl", 1), ("gpt2_small", 1), ("llama7b", 1), ("gpt2_xl", 4),
                                        ("gpt2_small", 4), ("llama7b", 2), ("tiny", 3)])
def test_per_kernel_bytes_add_up_to_the_step(name, micro):
    # the per-kernel byte model behind the JSON line's "gbs" and roofline equals the per-step model
    import bench
    from oracle.layout import make_layout
    from zero_partitioned_mixed_replica_gb300 import workloads
    w = workloads.ALL[name]()
    L = make_layout(w.numels, w.n_d, w.stage, bucket_elems=w.bucket_elems if w.stage != 3 else 0,
                    unit_of_tensor=w.unit_of_tensor if w.stage == 3 else None)
    fused = w.fused() and micro == 1
    nb, U, M = len(L.buckets), len(L.units), micro
    if w.stage == 3:
        launches = {"stage3_gather": 2 * U * M, ("fused_step" if fused else "reduce_scatter"): U * M}
    elif fused:
        launches = {"fused_step": nb}
    else:
        launches = {"reduce_scatter": nb * (M if w.stage == 2 else 1)}
        if w.stage == 1 and M > 1:
            launches["accumulate"] = M
    if not fused:
        launches["adamw"] = 1
    total = sum(n * bench.kernel_bytes(k, w, bench.elems_per_launch(k, w, L.psi_pad, n, M), M)
                for k, n in launches.items())
    expect = bench.bytes_per_param(w, fused, M) * L.psi_pad
    gathered_pad = 2 * (2 + 2 * w.n_d) * M * (L.psi_pad - w.psi) if w.stage == 3 else 0   # gathers skip padding
    assert abs(total + gathered_pad - expect) <= 1e-9 * expect, (total, expect)


def test_e2e_skips_when_pinned_copies_would_crowd_the_host():
    import bench
    assert bench.host_mem_available() is None or bench.host_mem_available() > 0
    gb = 10 ** 9
    assert bench.e2e_fits(25 * gb, 1, 199 * gb)          # 1.5B at N = 1 on a 199 GB host
    assert bench.e2e_fits(25 * gb, 2, 199 * gb)
    assert not bench.e2e_fits(25 * gb, 8, 199 * gb)      # 8 ranks would pin 200 GB
    assert bench.e2e_fits(25 * gb, 8, None)              # unknown: no guard


def test_timeline_summary_gaps_and_overlap():
    import bench
    recs = [  # stream 1: 0-1 ms, stream 2: 0.5-2 ms (overlaps), gap, stream 1: 2.5-3 ms, gap, 3.2-4 ms
        {"kind": "fused_step", "device": 0, "stream": 1, "start_ms": 0.0, "end_ms": 1.0},
        {"kind": "fused_step", "device": 0, "stream": 2, "start_ms": 0.5, "end_ms": 2.0},
        {"kind": "grad_norm", "device": 0, "stream": 1, "start_ms": 2.5, "end_ms": 3.0},
        {"kind": "grad_norm", "device": 0, "stream": 1, "start_ms": 3.2, "end_ms": 4.0},
    ]
    s = bench.timeline_summary(list(reversed(recs)))
    assert s["records"] == 4 and s["streams"] == 2 and s["overlapped_starts"] == 1
    assert abs(s["span_ms"] - 4.0) < 1e-12 and abs(s["busy_ms"] - 3.3) < 1e-12
    assert s["gaps"] == 2 and abs(s["mean_gap_us"] - 350.0) < 1e-9 and abs(s["max_gap_us"] - 500.0) < 1e-9
    assert abs(s["idle_frac"] - 0.7 / 4.0) < 1e-12
    assert bench.timeline_summary([]) == {"records": 0}


def test_timeline_file_is_a_chrome_trace(tmp_path):
    import bench
    recs = [{"kind": "reduce_scatter", "device": 0, "stream": 77, "start_ms": 0.25, "end_ms": 1.25},
            {"kind": "adamw", "device": 0, "stream": 78, "start_ms": 1.5, "end_ms": 3.0}]
    out = bench.write_timeline(recs, str(tmp_path / "t.json"))
    d = json.load(open(out["file"]))
    ev = d["traceEvents"]
    assert [e["name"] for e in ev] == ["reduce_scatter", "adamw"] and [e["tid"] for e in ev] == [0, 1]
    assert ev[0]["ph"] == "X" and ev[0]["ts"] == 250.0 and ev[0]["dur"] == 1000.0
    assert out["records"] == 2 and out["gaps"] == 1
