"""ctypes binding of libzero (``include/zero.h``): same entry-point names,
argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; nothing here computes.

Device buffers are passed as torch tensors (their ``data_ptr()``) or raw
integer addresses; pointer arrays as Python sequences of those.  Streams are
``torch.cuda.Stream`` objects, raw handles, or ``None`` for torch's current
stream.  A non-zero status raises :class:`ZeroError` with the library's
message.  If ``libzero.so`` has not been built the first call raises — there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
# ZERO_LIB names another build of the library to load (the bounds-checked
# libzero_checked.so); the in-tree libzero.so otherwise.
LIB_PATH = os.environ.get("ZERO_LIB") or os.path.join(PKG, "libzero.so")

ZERO_OK = 0
ZERO_ERR_INVALID = -1
ZERO_ERR_ALIGN = -2
ZERO_ERR_CUDA = -3
ZERO_ERR_STATE = -4
ZERO_ERR_TIMEOUT = -5
ZERO_ERR_NOMEM = -6
ZERO_BF16 = 0
ZERO_FP16 = 1
ZERO_MAX_RANKS = 64
ZERO_OUT_FULL_REPLICAS = 0
ZERO_OUT_SHARDS = 1
ZERO_NORM_DECIDE = 0
ZERO_NORM_AFTER_FUSED = 1

EXPORTED = ["zero_layout_init", "zero_layout_query", "zero_layout_bucket", "zero_layout_unit",
            "zero_layout_tensor_offset", "zero_layout_destroy", "zero_state_init",
            "zero_reduce_scatter", "zero_grad_norm", "zero_adamw_shard_step",
            "zero_allgather_params", "zero_cast_params", "zero_stage3_gather_layer", "zero_fused_step",
            "zero_fused_step_noalloc", "zero_reshard_plan", "zero_accumulate_grads",
            "zero_reduce_scatter_accumulated", "zero_reduce_scatter_micro", "zero_step", "zero_micro_step", "zero_step_from_host",
            "zero_trace_enable", "zero_trace_read", "zero_trace_timeline", "zero_set_max_ctas",
            "zero_last_error", "zero_launch_count", "zero_checked_build", "zero_bounds_violations",
            "zero_checked_set_slack"]
ZERO_NOALLOC_MAX_ELEMS = 67108864


class ZeroError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("libzero status %d: %s" % (status, msg))
        self.status = status


class zero_layout_info(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int32) for n in ("n_d", "stage", "dtype", "n_tensors", "n_buckets",
                                               "n_units", "reserved0", "reserved1")] +
                [(n, ctypes.c_int64) for n in ("psi", "psi_pad", "q", "bucket_elems", "shard_len",
                                               "max_unit_padded", "mem_formula", "mem_state",
                                               "mem_gshard", "mem_transient", "mem_peak", "comm_rs",
                                               "comm_ag", "comm_ag_fwd", "comm_ag_bwd",
                                               "comm_allreduce", "comm_total", "workspace_bytes")])


class zero_unit_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("offset", "real", "padded", "shard", "shard_base")]


class zero_step_state(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_double) for n in ("beta1", "beta2", "beta1_pow", "beta2_pow", "grad_norm")] +
                [("loss_scale", ctypes.c_float), ("clip_coef", ctypes.c_float)] +
                [(n, ctypes.c_int32) for n in ("t", "skipped", "good_steps", "growth_interval",
                                               "dynamic_scale", "nonfinite", "overflow", "apply",
                                               "error")] +
                [("reserved", ctypes.c_int32 * 3)])


class zero_copy_segment(ctypes.Structure):
    _fields_ = [("src_rank", ctypes.c_int32), ("dst_rank", ctypes.c_int32), ("src_off", ctypes.c_int64),
                ("dst_off", ctypes.c_int64), ("len", ctypes.c_int64)]


class zero_adamw_hp(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


ZERO_CALL_NAMES = ["reduce_scatter", "grad_norm", "adamw", "fused_step", "stage3_gather", "allgather", "accumulate"]


class zero_trace_totals(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_int64 * 8), ("total_ms", ctypes.c_double * 8), ("busy_ms", ctypes.c_double * 8)]


class zero_trace_record(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("device", ctypes.c_int32), ("stream", ctypes.c_uint64),
                ("start_ms", ctypes.c_double), ("end_ms", ctypes.c_double)]


ZERO_UNIT_HOOK = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p)


class zero_step_args(ctypes.Structure):
    _fields_ = [("hp", ctypes.POINTER(zero_adamw_hp)), ("max_norm", ctypes.c_double),
                ("fused", ctypes.c_int32), ("per_bucket", ctypes.c_int32)] + \
               [(n, ctypes.POINTER(ctypes.c_void_p)) for n in
                ("grad_replicas", "master", "m", "v", "grad_shards", "param16_full", "param16_shards",
                 "transient")] + \
               [("state", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("transient2", ctypes.POINTER(ctypes.c_void_p)), ("unit_hook", ZERO_UNIT_HOOK),
                ("hook_user", ctypes.c_void_p), ("overlap_previous", ctypes.c_int32)]


class StepArgs:
    """A filled ``zero_step_args`` that keeps its pointer arrays and
    hyperparameters alive as long as it lives."""

    def __init__(self, L: "Layout", hp: zero_adamw_hp, max_norm: float, fused: bool, per_bucket: bool,
                 grad_replicas, master, m, v, grad_shards, param16_full, param16_shards, transient, st,
                 workspace, transient2=None):
        self._keep = [hp]
        self.args = zero_step_args(hp=ctypes.pointer(hp), max_norm=float(max_norm), fused=int(bool(fused)),
                                   per_bucket=int(bool(per_bucket)), state=_addr(st), workspace=_addr(workspace))
        for name, xs in (("grad_replicas", grad_replicas), ("master", master), ("m", m), ("v", v),
                         ("grad_shards", grad_shards), ("param16_full", param16_full),
                         ("param16_shards", param16_shards), ("transient", transient),
                         ("transient2", transient2)):
            arr = _ptrs(xs, L)
            if arr is not None:
                self._keep.append(arr)
                setattr(self.args, name, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)))
        self._n_d = L.n_d
        self._hook = None
        self.hook_error = None      # first exception raised by the unit hook during a call

    def set_unit_hook(self, fn) -> None:
        """fn(pass_, unit, transient_addresses, stream_handle) or None: called
        by the executor after it issues each ZeRO-3 unit gather (pass_ 0:
        forward, 1: backward)."""
        if fn is None:
            self._hook = None
            self.args.unit_hook = ZERO_UNIT_HOOK()
            return
        n_d = self._n_d

        def trampoline(user, pass_, unit, transient, stream):
            # an exception cannot cross the C frames: keep the first one for the caller to re-raise
            if self.hook_error is not None:
                return
            try:
                fn(int(pass_), int(unit), [transient[i] for i in range(n_d)], stream)
            except BaseException as ex:     # noqa: BLE001 (re-raised by zero_step)
                self.hook_error = ex

        self._hook = ZERO_UNIT_HOOK(trampoline)
        self.args.unit_hook = self._hook


assert ctypes.sizeof(zero_step_state) == 96

_lib = None


def lib():
    """Load libzero.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libzero.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, dbl, flt = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_float
    PP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "zero_layout_init": [ctypes.POINTER(i64), i32, ctypes.POINTER(i32), i32, i32, i64, i64, i32,
                             ctypes.POINTER(P)],
        "zero_layout_query": [P, ctypes.POINTER(zero_layout_info)],
        "zero_layout_bucket": [P, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)],
        "zero_layout_unit": [P, i32, ctypes.POINTER(zero_unit_info)],
        "zero_layout_tensor_offset": [P, i32, ctypes.POINTER(i64)],
        "zero_state_init": [P, dbl, dbl, flt, i32, i32, P],
        "zero_reduce_scatter": [P, i32, PP, PP, P, P, P],
        "zero_grad_norm": [P, dbl, i32, P, P, P],
        "zero_adamw_shard_step": [P, ctypes.POINTER(zero_adamw_hp), PP, PP, PP, PP, P, PP, i32, P],
        "zero_allgather_params": [P, PP, PP, P],
        "zero_cast_params": [P, PP, PP, i32, P],
        "zero_stage3_gather_layer": [P, i32, PP, PP, P],
        "zero_fused_step": [P, i32, ctypes.POINTER(zero_adamw_hp), PP, PP, PP, PP, P, PP, i32, P, P],
        "zero_fused_step_noalloc": [P, ctypes.POINTER(zero_adamw_hp), PP, PP, PP, PP, P, PP, i32, P],
        "zero_reshard_plan": [P, P, ctypes.POINTER(zero_copy_segment), i64, ctypes.POINTER(i64)],
        "zero_accumulate_grads": [P, i32, PP, PP, P],
        "zero_reduce_scatter_accumulated": [P, i32, PP, PP, i32, P, P, P],
        "zero_reduce_scatter_micro": [P, i32, i32, i32, PP, PP, P, P, P],
        "zero_step": [P, ctypes.POINTER(zero_step_args), P],
        "zero_step_from_host": [P, ctypes.POINTER(zero_step_args), PP, i64, P, P],
        "zero_micro_step": [P, ctypes.POINTER(zero_step_args), i32, i32, PP, P],
        "zero_trace_read": [ctypes.POINTER(zero_trace_totals), i32],
        "zero_trace_timeline": [ctypes.POINTER(zero_trace_record), i64, ctypes.POINTER(i64), i32],
        "zero_bounds_violations": [ctypes.POINTER(i64), i32],
        "zero_checked_set_slack": [i64],
        "zero_checked_build": [],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = i32
    L.zero_layout_destroy.argtypes = [P]
    L.zero_layout_destroy.restype = None
    L.zero_last_error.argtypes = []
    L.zero_last_error.restype = ctypes.c_char_p
    L.zero_launch_count.argtypes = [i32]
    L.zero_launch_count.restype = i64
    L.zero_trace_enable.argtypes = [i32]
    L.zero_trace_enable.restype = i32
    L.zero_set_max_ctas.argtypes = [i32]
    L.zero_set_max_ctas.restype = i32
    _lib = L
    return L


def _check(status: int) -> None:
    if status != ZERO_OK:
        raise ZeroError(status, lib().zero_last_error().decode())


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptrs(xs: Optional[Sequence], L: "Layout"):
    """Host array of one device pointer per rank.  The library reads exactly
    N_d entries, so a list of another length is refused here (a shorter one
    would be read past its end); None passes NULL, which the library rejects."""
    if xs is None:
        return None
    if len(xs) != L.n_d:
        raise ZeroError(ZERO_ERR_INVALID, "expected %d pointers (one per rank), got %d" % (L.n_d, len(xs)))
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


class Layout:
    """Owns a ``zero_layout*``; destroyed with the object."""

    def __init__(self, handle: int, n_d: int):
        self.handle = ctypes.c_void_p(handle)
        self.n_d = n_d

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.zero_layout_destroy(h)

    @property
    def _as_parameter_(self):
        return self.handle


def zero_layout_init(numels: Sequence[int], unit_of_tensor: Optional[Sequence[int]], n_d: int, stage: int,
                     pad_multiple: int = 0, bucket_elems: int = 0, dtype: int = ZERO_BF16) -> Layout:
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*numels)
    units = (ctypes.c_int32 * n)(*unit_of_tensor) if unit_of_tensor is not None else None
    out = ctypes.c_void_p()
    _check(lib().zero_layout_init(arr, n, units, n_d, stage, pad_multiple, bucket_elems, dtype,
                                  ctypes.byref(out)))
    return Layout(out.value, n_d)


def zero_layout_query(L: Layout) -> zero_layout_info:
    info = zero_layout_info()
    _check(lib().zero_layout_query(L, ctypes.byref(info)))
    return info


def zero_layout_bucket(L: Layout, b: int):
    b0, b1 = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_layout_bucket(L, b, ctypes.byref(b0), ctypes.byref(b1)))
    return b0.value, b1.value


def zero_layout_unit(L: Layout, u: int) -> zero_unit_info:
    info = zero_unit_info()
    _check(lib().zero_layout_unit(L, u, ctypes.byref(info)))
    return info


def zero_layout_tensor_offset(L: Layout, t: int) -> int:
    off = ctypes.c_int64()
    _check(lib().zero_layout_tensor_offset(L, t, ctypes.byref(off)))
    return off.value


def zero_layout_destroy(L: Layout) -> None:
    h, L.handle = L.handle, None
    if h:
        lib().zero_layout_destroy(h)


def zero_state_init(st, beta1: float, beta2: float, loss_scale: float = 1.0, dynamic_scale: bool = False,
                    growth_interval: int = 2000, stream=None) -> None:
    _check(lib().zero_state_init(_addr(st), beta1, beta2, loss_scale, int(dynamic_scale), growth_interval,
                                 _stream(stream)))


def zero_reduce_scatter(L: Layout, bucket_or_unit: int, grad_replicas, grad_shards, st, workspace,
                        stream=None) -> None:
    _check(lib().zero_reduce_scatter(L, bucket_or_unit, _ptrs(grad_replicas, L), _ptrs(grad_shards, L), _addr(st),
                                     _addr(workspace), _stream(stream)))


def zero_grad_norm(L: Layout, max_norm: float, flags: int, st, workspace, stream=None) -> None:
    _check(lib().zero_grad_norm(L, max_norm, flags, _addr(st), _addr(workspace), _stream(stream)))


def _hp(lr, eps, weight_decay) -> zero_adamw_hp:
    return zero_adamw_hp(lr=lr, eps=eps, weight_decay=weight_decay)


def zero_adamw_shard_step(L: Layout, hp: zero_adamw_hp, master, m, v, grad_shards, st, param16_out,
                          out_kind: int, stream=None) -> None:
    _check(lib().zero_adamw_shard_step(L, ctypes.byref(hp), _ptrs(master, L), _ptrs(m, L), _ptrs(v, L),
                                       _ptrs(grad_shards, L), _addr(st), _ptrs(param16_out, L), out_kind,
                                       _stream(stream)))


def zero_allgather_params(L: Layout, param16_shards, param16_full, stream=None) -> None:
    _check(lib().zero_allgather_params(L, _ptrs(param16_shards, L), _ptrs(param16_full, L), _stream(stream)))


def zero_cast_params(L: Layout, master, param16_out, out_kind: int, stream=None) -> None:
    _check(lib().zero_cast_params(L, _ptrs(master, L), _ptrs(param16_out, L), out_kind, _stream(stream)))


def zero_stage3_gather_layer(L: Layout, unit: int, param16_shards, transient, stream=None) -> None:
    _check(lib().zero_stage3_gather_layer(L, unit, _ptrs(param16_shards, L), _ptrs(transient, L), _stream(stream)))


def zero_fused_step(L: Layout, bucket_or_unit: int, hp: zero_adamw_hp, grad_replicas, master, m, v, st,
                    param16_out, out_kind: int, workspace, stream=None) -> None:
    _check(lib().zero_fused_step(L, bucket_or_unit, ctypes.byref(hp), _ptrs(grad_replicas, L), _ptrs(master, L),
                                 _ptrs(m, L), _ptrs(v, L), _addr(st), _ptrs(param16_out, L), out_kind,
                                 _addr(workspace), _stream(stream)))


def zero_fused_step_noalloc(L: Layout, hp: zero_adamw_hp, grad_replicas, master, m, v, st, param16_out,
                            out_kind: int, stream=None) -> None:
    """Whole fused step without a caller workspace (see include/zero.h)."""
    _check(lib().zero_fused_step_noalloc(L, ctypes.byref(hp), _ptrs(grad_replicas, L), _ptrs(master, L), _ptrs(m, L),
                                         _ptrs(v, L), _addr(st), _ptrs(param16_out, L), out_kind, _stream(stream)))


def zero_reshard_plan(src: Layout, dst: Layout):
    """List of (src_rank, src_off, dst_rank, dst_off, len) copy segments."""
    n = ctypes.c_int64()
    _check(lib().zero_reshard_plan(src, dst, None, 0, ctypes.byref(n)))
    arr = (zero_copy_segment * max(1, n.value))()
    _check(lib().zero_reshard_plan(src, dst, arr, n.value, ctypes.byref(n)))
    return [(g.src_rank, g.src_off, g.dst_rank, g.dst_off, g.len) for g in arr[:n.value]]


def zero_accumulate_grads(L: Layout, micro: int, grad_replicas, acc_replicas, stream=None) -> None:
    _check(lib().zero_accumulate_grads(L, micro, _ptrs(grad_replicas, L), _ptrs(acc_replicas, L), _stream(stream)))


def zero_reduce_scatter_accumulated(L: Layout, bucket: int, acc_replicas, grad_shards, n_micro: int, st, workspace,
                                    stream=None) -> None:
    _check(lib().zero_reduce_scatter_accumulated(L, bucket, _ptrs(acc_replicas, L), _ptrs(grad_shards, L), n_micro,
                                                 _addr(st), _addr(workspace), _stream(stream)))


def zero_reduce_scatter_micro(L: Layout, bucket_or_unit: int, micro: int, n_micro: int, grad_replicas, acc_shards,
                              st, workspace, stream=None) -> None:
    _check(lib().zero_reduce_scatter_micro(L, bucket_or_unit, micro, n_micro, _ptrs(grad_replicas, L),
                                           _ptrs(acc_shards, L), _addr(st), _addr(workspace), _stream(stream)))


def _raise_hook_error(args: StepArgs) -> None:
    ex, args.hook_error = args.hook_error, None
    if ex is not None:
        raise ex


def zero_step(L: Layout, args: StepArgs, stream=None) -> None:
    """One step; an exception raised by the unit hook is re-raised here,
    after the call (the executor has issued the whole step by then)."""
    args.hook_error = None
    status = lib().zero_step(L, ctypes.byref(args.args), _stream(stream))
    _raise_hook_error(args)
    _check(status)


def zero_micro_step(L: Layout, args: StepArgs, micro: int, n_micro: int, acc_replicas=None, stream=None) -> None:
    args.hook_error = None
    status = lib().zero_micro_step(L, ctypes.byref(args.args), int(micro), int(n_micro),
                                   _ptrs(acc_replicas, L), _stream(stream))
    _raise_hook_error(args)
    _check(status)


def zero_step_from_host(L: Layout, args: StepArgs, host_grads, chunk_elems: int = 0, host_state=None,
                        stream=None, overlap_previous: bool = False) -> None:
    """host_grads: one host pointer (or CPU tensor) per rank; host_state: a
    CPU tensor / address of 96 bytes, or None; overlap_previous sets the
    field of the same name in ``args`` for this call."""
    args.args.overlap_previous = int(bool(overlap_previous))
    args.hook_error = None
    status = lib().zero_step_from_host(L, ctypes.byref(args.args), _ptrs(host_grads, L), int(chunk_elems),
                                       _addr(host_state), _stream(stream))
    _raise_hook_error(args)
    _check(status)


def zero_trace_enable(on: bool) -> bool:
    return bool(lib().zero_trace_enable(int(bool(on))))


def zero_trace_read(reset: bool = True) -> dict:
    """{call name: {"launches": n, "total_ms": t, "busy_ms": b, "avg_ms": b / n}}
    for every kind of call traced since the last reset.  ``busy_ms`` is the
    time with at least one call of the kind in flight; ``avg_ms`` divides it
    by the calls (equal to total / n when no two calls of the kind overlapped)."""
    t = zero_trace_totals()
    _check(lib().zero_trace_read(ctypes.byref(t), int(bool(reset))))
    return {name: {"launches": int(t.calls[k]), "total_ms": float(t.total_ms[k]), "busy_ms": float(t.busy_ms[k]),
                   "avg_ms": float(t.busy_ms[k]) / int(t.calls[k])}
            for k, name in enumerate(ZERO_CALL_NAMES) if t.calls[k] > 0}


def zero_trace_timeline(reset: bool = False) -> list:
    """Every call traced since the last reset, in issue order:
    [{"kind": name, "device": d, "stream": id, "start_ms": a, "end_ms": b}];
    times on one axis per device, from its first traced event."""
    n = ctypes.c_int64(0)
    _check(lib().zero_trace_timeline(None, 0, ctypes.byref(n), 0))
    buf = (zero_trace_record * max(1, n.value))()
    _check(lib().zero_trace_timeline(buf, n.value, ctypes.byref(n), int(bool(reset))))
    names = ZERO_CALL_NAMES
    return [{"kind": names[r.kind] if 0 <= r.kind < len(names) else str(r.kind), "device": int(r.device),
             "stream": int(r.stream), "start_ms": float(r.start_ms), "end_ms": float(r.end_ms)}
            for r in buf[:min(n.value, len(buf))]]


def zero_set_max_ctas(n: int) -> int:
    return int(lib().zero_set_max_ctas(int(n)))


def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def zero_launch_count(reset: bool = False) -> int:
    return int(lib().zero_launch_count(int(reset)))


def zero_checked_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().zero_checked_build())


def zero_bounds_violations(reset: bool = False) -> int:
    """Accesses the bounds-checked build skipped on the current device (0 in
    a normal build); synchronises the device."""
    n = ctypes.c_int64(0)
    _check(lib().zero_bounds_violations(ctypes.byref(n), int(reset)))
    return int(n.value)


def zero_checked_set_slack(elems: int) -> None:
    """Test hook of the bounds-checked build: every checked extent is
    ``elems`` short of the real one."""
    _check(lib().zero_checked_set_slack(int(elems)))
