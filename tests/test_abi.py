"""C ABI checks that need no GPU: libzero.so loads, exports every entry point
that include/zero.h declares, its host-side layout and accounting equal the
oracle's bit for bit, and argument validation fails before any launch.

Only argument errors that the library rejects before touching the device are
exercised here (NULL, misaligned, out-of-range, wrong stage)."""
import ctypes
import os
import re

import pytest

from oracle.layout import layout_comm_elems, layout_memory_bytes, make_layout
from zero_partitioned_mixed_replica_gb300 import binding as B
from zero_partitioned_mixed_replica_gb300 import build as zbuild
from zero_partitioned_mixed_replica_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    zbuild.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "zero.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "zero_reduce_scatter" in names and "zero_stage3_gather_layer" in names
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTED) == names


def _layout_pair(numels, n_d, stage, bucket=0, units=None):
    L = B.zero_layout_init(numels, units, n_d, stage, 0, bucket, B.ZERO_BF16)
    O = make_layout(numels, n_d, stage, bucket_elems=bucket, unit_of_tensor=units)
    return L, O


CASES = [
    ([1000 * 512, 512, 487 * 1000, 2491], 4, 2, 0, None),
    ([3000, 17, 5000, 1], 3, 1, 640, None),
    ([300, 2000, 64, 1500, 7], 5, 3, 0, [0, 1, 1, 2, 0]),
    ([1], 1, 2, 32, None),
    ([7, 9, 11], 64, 2, 96, None),
    ([10, 20, 300, 5], 2, 3, 0, [1, 0, 1, 2]),
    ([5, 6, 7], 8, 0, 0, None),
]


@pytest.mark.parametrize("numels,n_d,stage,bucket,units", CASES)
def test_layout_matches_oracle(numels, n_d, stage, bucket, units):
    L, O = _layout_pair(numels, n_d, stage, bucket, units)
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
    assert info.workspace_bytes >= info.psi_pad // 32 * 4 + 1024 * 8


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_xl", "llama7b"])
def test_workload_layouts_match_oracle(name):
    w = workloads.ALL[name]()
    units = w.unit_of_tensor if w.stage == 3 else None
    L, O = _layout_pair(w.numels, w.n_d, w.stage, w.bucket_elems if w.stage != 3 else 0, units)
    info = B.zero_layout_query(L)
    assert (info.psi_pad, info.shard_len, info.n_buckets) == (O.psi_pad, O.shard_len, len(O.buckets))
    assert [B.zero_layout_tensor_offset(L, t) for t in range(len(w.numels))] == O.tensor_offsets


@pytest.mark.parametrize("args,status", [
    (([], None, 2, 1, 0, 0, 0), B.ZERO_ERR_INVALID),
    (([5], None, 0, 1, 0, 0, 0), B.ZERO_ERR_INVALID),
    (([5], None, 65, 1, 0, 0, 0), B.ZERO_ERR_INVALID),
    (([5], None, 2, 4, 0, 0, 0), B.ZERO_ERR_INVALID),
    (([5], None, 2, 3, 0, 0, 0), B.ZERO_ERR_INVALID),          # stage 3 without units
    (([5, 6], [0, 2], 2, 3, 0, 0, 0), B.ZERO_ERR_INVALID),      # empty unit 1
    (([5], None, 2, 1, 100, 0, 0), B.ZERO_ERR_INVALID),         # pad not a multiple of n_d*128
    (([5], None, 2, 1, 0, 48, 0), B.ZERO_ERR_INVALID),          # bucket not a multiple of 32
    (([5], None, 2, 1, 0, 0, 7), B.ZERO_ERR_INVALID),           # dtype
    (([0, 5], None, 2, 1, 0, 0, 0), B.ZERO_ERR_INVALID),        # empty tensor
    (([5, 6], [0, (1 << 31) - 1], 2, 3, 0, 0, 0), B.ZERO_ERR_INVALID),   # unit id >= tensor count
    (([1 << 62, 1 << 62], None, 2, 1, 0, 0, 0), B.ZERO_ERR_INVALID),   # Psi would overflow int64
    (([5], None, 2, 1, 256 << 40, 0, 0), B.ZERO_ERR_INVALID),          # pad quantum above 2^34
])
def test_layout_init_rejects(args, status):
    with pytest.raises(B.ZeroError) as e:
        B.zero_layout_init(*args)
    assert e.value.status == status
    assert B.zero_last_error()


FAKE = 1 << 40          # 256-aligned host-side stand-in, never dereferenced: every
MIS = FAKE + 16         # call below is rejected by validation before any launch


def test_step_calls_validate_before_launch():
    L = B.zero_layout_init([1000, 24], None, 2, 2, 0, 0, B.ZERO_BF16)
    L3 = B.zero_layout_init([1000, 24], [0, 1], 2, 3, 0, 0, B.ZERO_BF16)
    L0 = B.zero_layout_init([1000, 24], None, 2, 0, 0, 0, B.ZERO_BF16)
    two = [FAKE, FAKE]
    hp = B.zero_adamw_hp(lr=1e-3, eps=1e-8, weight_decay=0.0)

    def status(fn, *a):
        with pytest.raises(B.ZeroError) as e:
            fn(*a)
        return e.value.status

    assert status(B.zero_reduce_scatter, L, 5, two, two, FAKE, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_reduce_scatter, L, 0, [FAKE, MIS], two, FAKE, FAKE, 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_reduce_scatter, L, 0, [FAKE, 0], two, FAKE, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_reduce_scatter, L, 0, two, two, MIS, FAKE, 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_reduce_scatter, L0, 0, two, two, FAKE, FAKE, 0) == B.ZERO_ERR_STATE
    assert status(B.zero_grad_norm, L, 1.0, 7, FAKE, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_grad_norm, L, float("nan"), 0, FAKE, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_grad_norm, L, 1.0, 0, FAKE, 0, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_adamw_shard_step, L3, hp, two, two, two, two, FAKE, two,
                  B.ZERO_OUT_FULL_REPLICAS, 0) == B.ZERO_ERR_STATE
    assert status(B.zero_adamw_shard_step, L, hp, two, two, two, two, FAKE, two, 9, 0) == B.ZERO_ERR_INVALID
    for eps in (0.0, 2.0 ** -150, -1e-8, float("nan")):   # 2^-150 rounds to a binary32 zero
        bad_hp = B.zero_adamw_hp(lr=1e-3, eps=eps, weight_decay=0.0)
        assert status(B.zero_adamw_shard_step, L, bad_hp, two, two, two, two, FAKE, two,
                      B.ZERO_OUT_SHARDS, 0) == B.ZERO_ERR_INVALID, eps
    assert status(B.zero_allgather_params, L3, two, two, 0) == B.ZERO_ERR_STATE
    assert status(B.zero_stage3_gather_layer, L, 0, two, two, 0) == B.ZERO_ERR_STATE
    assert status(B.zero_stage3_gather_layer, L3, 2, two, two, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_fused_step, L, 3, hp, two, two, two, two, FAKE, two,
                  B.ZERO_OUT_FULL_REPLICAS, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_fused_step, L3, -1, hp, two, two, two, two, FAKE, two,
                  B.ZERO_OUT_SHARDS, FAKE, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_state_init, MIS, 0.9, 0.999, 1.0, False, 10, 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_state_init, FAKE, 1.0, 0.999, 1.0, False, 10, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_state_init, FAKE, 0.9, 0.999, 0.5, False, 10, 0) == B.ZERO_ERR_INVALID


def test_layout_rejects_psi_pad_at_the_vector_counter_limit():
    # Psi_pad / 8 must stay below 2^31 (32-bit grid-stride counters)
    with pytest.raises(B.ZeroError) as e:
        B.zero_layout_init([1 << 34], None, 1, 2, 0, 0, B.ZERO_BF16)
    assert e.value.status == B.ZERO_ERR_INVALID
    L = B.zero_layout_init([(1 << 34) - 1024], None, 1, 2, 0, 0, B.ZERO_BF16)
    assert B.zero_layout_query(L).psi_pad == (1 << 34) - 1024


def test_bucket_larger_than_buffer_is_one_bucket():
    L = B.zero_layout_init([1000, 24], None, 2, 1, 0, (1 << 62) - 32 * 3, B.ZERO_BF16)
    info = B.zero_layout_query(L)
    assert info.n_buckets == 1 and B.zero_layout_bucket(L, 0) == (0, info.psi_pad)


def test_binding_refuses_pointer_lists_of_the_wrong_length():
    # the library reads exactly N_d pointers; a shorter host list would be read past its end
    L = B.zero_layout_init([1000, 24], None, 4, 2, 0, 0, B.ZERO_BF16)
    for xs in ([FAKE], [FAKE] * 5):
        with pytest.raises(B.ZeroError) as e:
            B.zero_reduce_scatter(L, 0, xs, [FAKE] * 4, FAKE, FAKE, 0)
        assert e.value.status == B.ZERO_ERR_INVALID
    with pytest.raises(B.ZeroError) as e:      # NULL array: rejected by the library itself
        B.zero_allgather_params(L, None, [FAKE] * 4, 0)
    assert e.value.status == B.ZERO_ERR_INVALID


def test_executor_and_cast_validate_before_launch():
    L = B.zero_layout_init([1000, 24], None, 2, 2, 0, 0, B.ZERO_BF16)
    L3 = B.zero_layout_init([1000, 24], [0, 1], 2, 3, 0, 0, B.ZERO_BF16)
    L0 = B.zero_layout_init([1000, 24], None, 2, 0, 0, 0, B.ZERO_BF16)
    two = [FAKE, FAKE]
    hp = B.zero_adamw_hp(lr=1e-3, eps=1e-8, weight_decay=0.0)

    def status(fn, *a):
        with pytest.raises(B.ZeroError) as e:
            fn(*a)
        return e.value.status

    def args(Lx, fused, max_norm=0.0, gshard=two, full=two, shards=None, transient=None, grads=two):
        return B.StepArgs(Lx, hp, max_norm, fused, True, grads, two, two, two, gshard, full, shards, transient,
                          FAKE, FAKE)

    assert status(B.zero_step, L, args(L, True, max_norm=1.0), 0) == B.ZERO_ERR_INVALID     # fused cannot clip
    assert status(B.zero_step, L, args(L, False, gshard=None), 0) == B.ZERO_ERR_INVALID    # split needs shards
    assert status(B.zero_step, L, args(L, False, full=None), 0) == B.ZERO_ERR_INVALID      # ZeRO-2 needs replicas
    assert status(B.zero_step, L, args(L, True, shards=two), 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_step, L3, args(L3, True, full=None, shards=two), 0) == B.ZERO_ERR_INVALID  # no transient
    assert status(B.zero_step, L3, args(L3, True, full=None, transient=two), 0) == B.ZERO_ERR_INVALID  # no shards
    assert status(B.zero_step, L0, args(L0, False), 0) == B.ZERO_ERR_STATE
    # every pointer is validated before the executor touches the device
    assert status(B.zero_step, L, args(L, False, grads=[FAKE, MIS]), 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_step, L, args(L, False, gshard=[0, FAKE]), 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_step_from_host, L, args(L, False), None, 0, None, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_step_from_host, L, args(L, False), [FAKE, 0], 0, None, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_step_from_host, L, args(L, True, max_norm=0.5), two, 0, None, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_step_from_host, L, args(L, False, full=[FAKE, MIS]), two, 0, None, 0) == B.ZERO_ERR_ALIGN
    bad_flag = args(L, False)
    bad_flag.args.overlap_previous = 2
    assert status(B.zero_step, L, bad_flag, 0) == B.ZERO_ERR_INVALID                  # the flag is 0 or 1
    assert B.lib().zero_trace_read(None, 0) == B.ZERO_ERR_INVALID
    assert B.zero_trace_read() == {}             # nothing traced: no kind reported
    L1 = B.zero_layout_init([1000, 24], None, 2, 1, 0, 0, B.ZERO_BF16)
    assert status(B.zero_micro_step, L, args(L, False), 2, 2, None, 0) == B.ZERO_ERR_INVALID      # micro >= n_micro
    assert status(B.zero_micro_step, L, args(L, False), -1, 2, None, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_micro_step, L, args(L, True, gshard=None), 0, 2, None, 0) == B.ZERO_ERR_INVALID  # fused
    assert status(B.zero_micro_step, L1, args(L1, False), 0, 2, None, 0) == B.ZERO_ERR_INVALID    # no accumulators
    assert status(B.zero_micro_step, L1, args(L1, False), 0, 2, [FAKE, MIS], 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_cast_params, L3, two, two, B.ZERO_OUT_FULL_REPLICAS, 0) == B.ZERO_ERR_STATE
    assert status(B.zero_cast_params, L, two, two, 5, 0) == B.ZERO_ERR_INVALID
    assert status(B.zero_cast_params, L, [FAKE, MIS], two, B.ZERO_OUT_SHARDS, 0) == B.ZERO_ERR_ALIGN
    assert status(B.zero_cast_params, L0, two, two, B.ZERO_OUT_SHARDS, 0) == B.ZERO_ERR_STATE


def test_ctypes_structs_match_the_header(tmp_path):
    # every struct the binding mirrors has the header's size and field offsets (plain C compiler)
    import subprocess
    structs = {"zero_step_args": B.zero_step_args, "zero_step_state": B.zero_step_state,
               "zero_trace_totals": B.zero_trace_totals, "zero_layout_info": B.zero_layout_info,
               "zero_unit_info": B.zero_unit_info, "zero_adamw_hp": B.zero_adamw_hp,
               "zero_copy_segment": B.zero_copy_segment, "zero_trace_record": B.zero_trace_record}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "zero.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (name, name))
        for f in cls._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (name, f[0], name, f[0]))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for f in cls._fields_:
            assert int(got["%s.%s" % (name, f[0])]) == getattr(cls, f[0]).offset, (name, f[0])


def test_unit_hook_trampoline_keeps_the_first_exception():
    # the executor calls the hook through a C function pointer; an exception cannot cross the C
    # frames, so the binding keeps the first one and re-raises it after the call
    L3 = B.zero_layout_init([1000, 24], [0, 1], 2, 3, 0, 0, B.ZERO_BF16)
    hp = B.zero_adamw_hp(lr=1e-3, eps=1e-8, weight_decay=0.0)
    two = [FAKE, FAKE]
    a = B.StepArgs(L3, hp, 0.0, True, True, two, two, two, two, None, None, two, two, FAKE, FAKE)
    seen = []

    def hook(pass_, unit, addresses, stream):
        seen.append((pass_, unit, addresses))
        raise KeyError("planted")

    a.set_unit_hook(hook)
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE + 256)
    for unit in (0, 1):          # call the C function pointer the way the executor does
        a.args.unit_hook(None, 0, unit, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), None)
    assert seen == [(0, 0, [FAKE, FAKE + 256])]      # the second call is skipped after the error
    with pytest.raises(KeyError, match="planted"):
        B._raise_hook_error(a)
    B._raise_hook_error(a)                              # cleared once raised
    a.set_unit_hook(None)
    assert not a.args.unit_hook


def test_normal_build_reports_no_checks():
    # the bounds checks are compiled out of the normal build: it says so, counts nothing and
    # refuses the checked build's test hook
    if os.environ.get("ZERO_LIB"):
        pytest.skip("another build of the library is loaded")
    assert not B.zero_checked_build()
    assert B.zero_bounds_violations() == 0
    with pytest.raises(B.ZeroError) as e:
        B.zero_checked_set_slack(8)
    assert e.value.status == B.ZERO_ERR_STATE
    assert B.lib().zero_bounds_violations(None, 0) == B.ZERO_ERR_INVALID


def test_trace_timeline_validates_and_is_empty_without_records():
    import ctypes
    n = ctypes.c_int64(-1)
    assert B.lib().zero_trace_timeline(None, 0, None, 0) == B.ZERO_ERR_INVALID
    assert B.lib().zero_trace_timeline(None, 4, ctypes.byref(n), 0) == B.ZERO_ERR_INVALID
    assert B.lib().zero_trace_timeline(None, -1, ctypes.byref(n), 0) == B.ZERO_ERR_INVALID
    assert B.zero_trace_timeline() == []
