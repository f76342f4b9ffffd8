"""Step sequencer over the C ABI: one GPU, N_d simulated data-parallel ranks.

:class:`ZeroStep` allocates every buffer once (torch is the allocator, in the
spirit of the pre-allocated contiguous blocks of "ZeRO: Memory Optimizations
Toward Training Trillion Parameter Models" reading notes §3.2.3/§5.3) and
runs a step as one call of the library's step executor (``zero_step``, or
``zero_step_from_host`` for gradients in host memory), which issues the
library calls in the order the pages give:

* ZeRO-1/2, split (clipping or a loss scaler active): reduce-scatter bucket by
  bucket, last bucket first (backward produces the last layers first; mlqm.cn
  post "梯度桶化", reading notes §4.1-§4.2) -> global norm and step decision ->
  sharded AdamW with the all-gather fused into its epilogue ("第 5 课：ZeRO 与
  FSDP" §3).
* ZeRO-1/2, fused (neither): reduce-scatter + AdamW + cast + all-gather in one
  pass per bucket (or one pass for the whole buffer), then the norm report.
* ZeRO-3: forward gathers unit by unit into the transient buffer; backward
  walks the units in reverse, re-gathers each, reduce-scatters it and (fused)
  updates its shard; no all-gather at the end of the step ("第 5 课" Fig. 5-1,
  reading notes §3.1 and §4.3, "ZeRO-3 核心流程" §2).  With clipping or a scaler
  the shard updates wait for the global decision.

Gradient accumulation (``micro_step``) is one ``zero_micro_step`` call per
micro-batch.  Only the ZeRO-3 prefetch under a caller's compute
(``step_overlapped``) issues its calls from here.  Every arithmetic step runs
inside libzero's kernels; this module only owns memory, orders calls and
reads back the 96-byte step state.
"""
from __future__ import annotations

import json
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import binding as B

TORCH_16 = {B.ZERO_BF16: torch.bfloat16, B.ZERO_FP16: torch.float16}


@dataclass
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


class ZeroStep:
    def __init__(self, numels: Sequence[int], n_d: int, stage: int, dtype: int = B.ZERO_BF16,
                 bucket_elems: int = 0, unit_of_tensor: Optional[Sequence[int]] = None,
                 adamw: AdamW = AdamW(), max_norm: float = 0.0, loss_scale: float = 1.0,
                 dynamic_scale: bool = False, growth_interval: int = 2000,
                 fused: Optional[bool] = None, per_bucket: bool = True, fuse_allgather: bool = True,
                 n_micro: int = 1, device: str = "cuda", stream: Optional[torch.cuda.Stream] = None,
                 pad_multiple: int = 0, live_units: int = 1):
        if stage not in (1, 2, 3):
            raise ValueError("ZeroStep runs ZeRO stages 1, 2 and 3")
        self.pad_multiple = pad_multiple    # 0: N_d * 128; else a multiple of it
        self.L = B.zero_layout_init(list(numels), list(unit_of_tensor) if unit_of_tensor is not None else None,
                                    n_d, stage, pad_multiple, bucket_elems, dtype)
        self.info = B.zero_layout_query(self.L)
        self.n_d, self.stage, self.dtype = n_d, stage, dtype
        self.adamw = adamw
        self.max_norm = float(max_norm)
        self.loss_scale0 = float(loss_scale)
        self.dynamic, self.growth_interval = bool(dynamic_scale), int(growth_interval)
        no_scaler = (not dynamic_scale) and loss_scale == 1.0
        self.n_micro = int(n_micro)
        if self.n_micro < 1:
            raise ValueError("n_micro must be >= 1")
        self.fused = (self.max_norm <= 0 and no_scaler and self.n_micro == 1) if fused is None else bool(fused)
        if self.fused and self.n_micro > 1:
            raise ValueError("gradient accumulation uses the split step")
        if self.fused and not (self.max_norm <= 0 and no_scaler):
            raise ValueError("the fused step cannot clip or skip: use the split step")
        self.per_bucket = per_bucket
        # ZeRO-1/2 split step only: False writes 16-bit shards, then all-gathers them
        self.fuse_allgather = fuse_allgather or stage == 3 or self.fused
        self.device = torch.device(device)
        self.stream = stream
        dt16 = TORCH_16[dtype]
        P, S = self.info.psi_pad, self.info.shard_len
        dev = self.device
        self.n_buckets = self.info.n_buckets
        self.units = [B.zero_layout_unit(self.L, u) for u in range(self.info.n_units)]
        self.tensor_offsets = [B.zero_layout_tensor_offset(self.L, t) for t in range(len(numels))]
        self.numels = list(numels)
        self.unit_of_tensor = list(unit_of_tensor) if unit_of_tensor is not None else None
        # rank-major 2-D allocations; row r is rank r's buffer (rows stay 256-byte aligned)
        self.grads = torch.zeros(n_d, P, dtype=dt16, device=dev)
        self.master = torch.zeros(n_d, S, dtype=torch.float32, device=dev)
        self.m = torch.zeros(n_d, S, dtype=torch.float32, device=dev)
        self.v = torch.zeros(n_d, S, dtype=torch.float32, device=dev)
        self.gshard = None if self.fused else torch.zeros(n_d, S, dtype=torch.float32, device=dev)
        # ZeRO-1 accumulates each rank's full gradient in fp32 ("第 5 课" §2: + 4 Psi per rank);
        # ZeRO-2/3 accumulate in the fp32 shard itself (+ 4 Psi / N_d, already held)
        self.acc = (torch.zeros(n_d, P, dtype=torch.float32, device=dev)
                    if (self.n_micro > 1 and stage == 1) else None)
        if stage == 3:
            self.params = None
            self.shard16 = torch.zeros(n_d, S, dtype=dt16, device=dev)
            max_real = max(u.real for u in self.units)
            self.transient = torch.zeros(n_d, (max_real + 127) // 128 * 128, dtype=dt16, device=dev)
            # live_units = 2: a second transient per rank, so that zero_step gathers the next unit
            # while the previous one is reduced and updated ("第 5 课" §4 prefetch, two live units)
            self.transient2 = torch.zeros_like(self.transient) if live_units >= 2 else None
        else:
            self.params = torch.zeros(n_d, P, dtype=dt16, device=dev)
            self.shard16 = None if self.fuse_allgather else torch.zeros(n_d, S, dtype=dt16, device=dev)
            self.transient = None
            self.transient2 = None
        self.workspace = torch.zeros(self.info.workspace_bytes, dtype=torch.uint8, device=dev)
        self.state = torch.zeros(96, dtype=torch.uint8, device=dev)
        self._rows()
        self.hp = B.zero_adamw_hp(lr=adamw.lr, eps=adamw.eps, weight_decay=adamw.weight_decay)
        self.transient_hook = None  # called as hook(kind, unit, transient_rows) after each ZeRO-3 gather
        self.reset_state()

    def set_bucket_elems(self, bucket_elems: int) -> None:
        """Re-lay the same buffers with another bucket size (ZeRO-1/2): the
        padded length and shards do not depend on it, so nothing moves (the
        step arguments stay valid)."""
        if self.stage == 3:
            raise ValueError("ZeRO-3 reduces per unit")
        L = B.zero_layout_init(self.numels, None, self.n_d, self.stage, self.pad_multiple, bucket_elems, self.dtype)
        info = B.zero_layout_query(L)
        if info.psi_pad != self.info.psi_pad or info.shard_len != self.info.shard_len:   # cannot happen: padding ignores buckets
            raise RuntimeError("re-bucketed layout changed the padded length")
        self.L, self.info, self.n_buckets = L, info, info.n_buckets

    # -- pointer lists ---------------------------------------------------------
    def _rows(self):
        rows = lambda t: [t[r] for r in range(self.n_d)] if t is not None else None
        self.grad_rows = rows(self.grads)
        self.master_rows, self.m_rows, self.v_rows = rows(self.master), rows(self.m), rows(self.v)
        self.gshard_rows = rows(self.gshard)
        self.param_rows = rows(self.params)
        self.shard16_rows = rows(self.shard16)
        self.transient_rows = rows(self.transient)
        self.transient2_rows = rows(self.transient2)
        self.acc_rows = rows(getattr(self, "acc", None))

    def _s(self):
        return self.stream if self.stream is not None else torch.cuda.current_stream(self.device)

    # -- initialisation (plumbing, not part of the step) -------------------------
    def reset_state(self):
        # after the work on the current stream (the buffers' zero fill, at construction), when
        # the engine runs on a stream of its own
        self._s().wait_stream(torch.cuda.current_stream(self.device))
        B.zero_state_init(self.state, self.adamw.beta1, self.adamw.beta2, self.loss_scale0, self.dynamic,
                          self.growth_interval, self._s())

    def load_master(self, flat_master: torch.Tensor) -> None:
        """Scatter a flat fp32 master (Psi_pad, zero padding) into the rank
        shards, zero m and v, and set the 16-bit parameters to its
        round-to-nearest-even cast (the library's zero_cast_params: into the
        16-bit shards and/or every full replica)."""
        if flat_master.numel() != self.info.psi_pad:
            raise ValueError("load_master needs Psi_pad = %d elements, got %d" % (self.info.psi_pad, flat_master.numel()))
        if flat_master.dtype != torch.float32:
            raise ValueError("load_master takes the fp32 master, got %s" % flat_master.dtype)
        fm = flat_master.to(self.device)
        for u in self.units:
            for r in range(self.n_d):
                lo = u.offset + r * u.shard
                self.master[r, u.shard_base:u.shard_base + u.shard].copy_(fm[lo:lo + u.shard])
        self.m.zero_()
        self.v.zero_()
        s = self._s()
        s.wait_stream(torch.cuda.current_stream(self.device))   # the copies above ran on the current stream
        if self.shard16 is not None:
            B.zero_cast_params(self.L, self.master_rows, self.shard16_rows, B.ZERO_OUT_SHARDS, s)
        if self.params is not None:
            B.zero_cast_params(self.L, self.master_rows, self.param_rows, B.ZERO_OUT_FULL_REPLICAS, s)

    # -- the step ------------------------------------------------------------------
    def step_args(self) -> B.StepArgs:
        """This engine's buffers and settings as the library's zero_step_args
        (built once, as the buffers never move; built again if ``hp`` is
        replaced by another object), with ``transient_hook`` installed as the
        executor's unit hook."""
        if getattr(self, "_args", None) is None or self._args_hp is not self.hp:
            self._args_hp = self.hp
            self._args_hook = None
            stage3 = self.stage == 3
            self._args = B.StepArgs(
                self.L, self.hp, self.max_norm if not self.fused else 0.0, self.fused, self.per_bucket,
                self.grad_rows, self.master_rows, self.m_rows, self.v_rows,
                None if self.fused else self.gshard_rows, None if stage3 else self.param_rows,
                self.shard16_rows if (stage3 or not self.fuse_allgather) else None,
                self.transient_rows if stage3 else None, self.state, self.workspace,
                self.transient2_rows if stage3 else None)
        if self._args_hook is not self.transient_hook:
            self._args_hook = self.transient_hook
            self._args.set_unit_hook(self._unit_hook if self.transient_hook is not None else None)
        return self._args

    def _unit_hook(self, pass_: int, unit: int, addresses, stream) -> None:
        """The executor's unit hook: hand the gathered unit's transient rows to
        ``transient_hook(kind, unit, rows)``."""
        first = addresses[0]
        buf = self.transient
        if self.transient2 is not None and first == self.transient2[0].data_ptr():
            buf = self.transient2
        self.transient_hook("fwd" if pass_ == 0 else "bwd", unit, [buf[r] for r in range(self.n_d)])

    def step(self) -> None:
        """One step: one call of the library's step executor (zero_step), which
        issues the step's calls in the pages' order (see ``zero.h``).  A
        ``transient_hook(kind, unit, rows)`` set on the engine is called after
        each ZeRO-3 unit gather is issued, where a layer's compute would be
        enqueued."""
        B.zero_step(self.L, self.step_args(), self._s())

    # -- ZeRO-3 prefetch: gathers on a second stream overlap the layers' compute -------
    def step_overlapped(self, compute, max_live_units: int = 2, comm_ctas: int = 0) -> None:
        """ZeRO-3 step whose unit gathers run on a communication stream while
        ``compute(kind, unit, transient_rows)`` — the caller's stand-in for
        the layer's forward ("fwd") or backward ("bwd") work, launched on the
        current stream — uses the previous unit ("第 5 课：ZeRO 与 FSDP" §4:
        gather layer l+1 in forward and l-1 in backward while layer l
        computes; "ZeRO-3 核心流程" §3; reading notes §4.3).  In backward the
        unit's reduce-scatter and update follow its compute on the
        communication stream.  ``max_live_units`` transient buffers are in
        flight (1 = no prefetch: every gather waits for the previous
        compute).  ``comm_ctas`` > 0 caps the CTAs of the library's launches
        in this step, leaving SMs to the concurrent compute.  Results are
        identical to :meth:`step`."""
        if self.stage != 3 or not self.fused:
            raise ValueError("step_overlapped runs the fused ZeRO-3 step")
        nb = max(1, int(max_live_units))
        if getattr(self, "_bufs", None) is None or len(self._bufs) < nb:
            self._bufs = [self.transient] + [torch.zeros_like(self.transient) for _ in range(nb - 1)]
            self._comm = torch.cuda.Stream(self.device)
        comp = self._s()
        comm = self._comm
        L, U = self.L, len(self.units)
        uses = [("fwd", u) for u in range(U)] + [("bwd", u) for u in reversed(range(U))]
        gathered = [torch.cuda.Event() for _ in uses]
        used = [torch.cuda.Event() for _ in uses]
        rows = [[b[r] for r in range(self.n_d)] for b in self._bufs[:nb]]
        comm.wait_stream(comp)
        prev_cap = B.zero_set_max_ctas(comm_ctas) if comm_ctas > 0 else None

        def gather(i):
            kind, u = uses[i]
            if i >= nb:
                comm.wait_event(used[i - nb])       # its buffer's previous user is done
            B.zero_stage3_gather_layer(L, u, self.shard16_rows, rows[i % nb], comm)
            gathered[i].record(comm)

        try:
            gather(0)
            for i, (kind, u) in enumerate(uses):
                if i + 1 < len(uses) and nb > 1:
                    gather(i + 1)                        # prefetch the next unit
                comp.wait_event(gathered[i])
                compute(kind, u, rows[i % nb])
                used[i].record(comp)
                if nb == 1 and i + 1 < len(uses):
                    gather(i + 1)
                if kind == "bwd":
                    comm.wait_event(used[i])             # the unit's gradients exist after its backward
                    B.zero_fused_step(L, u, self.hp, self.grad_rows, self.master_rows, self.m_rows, self.v_rows,
                                      self.state, self.shard16_rows, B.ZERO_OUT_SHARDS, self.workspace, comm)
            B.zero_grad_norm(L, 0.0, B.ZERO_NORM_AFTER_FUSED, self.state, self.workspace, comm)
        finally:
            comp.wait_stream(comm)
            if prev_cap is not None:                     # the cap is process-wide: always put it back
                B.zero_set_max_ctas(prev_cap)

    # -- gradient accumulation over micro-batches ------------------------------------
    def micro_step(self, micro: int) -> None:
        """Process micro-batch ``micro`` (0-based) of ``n_micro``, whose 16-bit
        gradients are in ``grads``; the last one finishes the optimizer step.
        One zero_micro_step call: ZeRO-1 accumulates locally in fp32 and
        reduce-scatters once (reading notes §4.1); ZeRO-2 reduce-scatters
        every micro-batch into the fp32 shard (§4.2); ZeRO-3 also gathers
        every unit forward and backward for every micro-batch (§4.3)."""
        M = self.n_micro
        if M == 1:
            self.step()
            return
        if not 0 <= micro < M:
            raise ValueError("micro out of range")
        B.zero_micro_step(self.L, self.step_args(), micro, M, self.acc_rows, self._s())

    # -- CUDA graph of one step -------------------------------------------------------
    def capture(self) -> torch.cuda.CUDAGraph:
        """Record one step into a CUDA graph (the step allocates nothing and
        never synchronises, so it captures as is).  Replaying the graph runs
        one step."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        side.wait_stream(self._s())          # and the engine's own stream, if it has one
        old = self.stream
        try:
            with torch.cuda.stream(side):
                self.stream = side
                with torch.cuda.graph(g, stream=side):
                    self.step()
        finally:
            self.stream = old
        torch.cuda.current_stream(self.device).wait_stream(side)
        return g

    # -- host input ----------------------------------------------------------------------
    def _check_host(self, host: torch.Tensor, need_pinned: bool) -> None:
        if tuple(host.shape) != tuple(self.grads.shape) or host.dtype != self.grads.dtype:
            raise ValueError("host gradients must be %s %s, got %s %s"
                             % (tuple(self.grads.shape), self.grads.dtype, tuple(host.shape), host.dtype))
        if need_pinned and not host.is_pinned():
            raise ValueError("overlapped host copies need pinned host memory")

    def step_from_host(self, host: torch.Tensor, chunk_elems: int = 1 << 27,
                       state_out: Optional[torch.Tensor] = None, overlap_previous: bool = False) -> None:
        """One step whose N_d gradient replicas come from pinned host memory,
        through the library's zero_step_from_host: each bucket's range
        (ZeRO-3: each unit's) is copied on the library's two copy streams in
        the order the step consumes them, and each bucket's reduce-scatter or
        fused update waits only for its own range, so later buckets cross the
        host link while earlier ones are reduced (reading notes "ZeRO: Memory
        Optimizations Toward Training Trillion Parameter Models" §4.1-§4.2: a
        bucket is reduced as soon as backward has filled it; the host link
        stands in for backward).  ``state_out`` (96 bytes of host memory,
        pinned for an asynchronous copy) receives the step state at the end
        of the step.  The result is identical to ``upload_grads(host)`` then
        ``step()``.

        ``overlap_previous``: when the previous library step of this device
        was also a host-input step, this step's copies start as soon as that
        step has reduced its replicas, so its norm and update overlap them.
        The device replicas (``grads``) must then not be touched in between;
        ``upload_grads`` since the last host-input step turns the overlap off
        for the next one."""
        self._check_host(host, True)
        if state_out is not None and (state_out.device.type != "cpu" or state_out.numel() * state_out.element_size()
                                      < self.state.numel()):
            raise ValueError("state_out must be a host tensor of at least 96 bytes")
        overlap = overlap_previous and not getattr(self, "_grads_written", False)
        self._grads_written = False
        B.zero_step_from_host(self.L, self.step_args(), [host[r] for r in range(self.n_d)], chunk_elems,
                              state_out, self._s(), overlap_previous=overlap)

    def upload_grads(self, host: torch.Tensor, chunk_elems: int = 1 << 27) -> None:
        """Copy the N_d gradient replicas from (pinned) host memory, in chunks
        alternating over two copy streams (faster than one large copy on this
        part), ordered before the next library call on the step's stream."""
        self._check_host(host, False)
        self._grads_written = True
        if getattr(self, "_copy_streams", None) is None:
            self._copy_streams = [torch.cuda.Stream(self.device) for _ in range(2)]
        cur = self._s()
        flat_h, flat_d = host.view(-1), self.grads.view(-1)
        for s in self._copy_streams:
            s.wait_stream(cur)
        for i, off in enumerate(range(0, flat_h.numel(), chunk_elems)):
            with torch.cuda.stream(self._copy_streams[i % 2]):
                flat_d[off:off + chunk_elems].copy_(flat_h[off:off + chunk_elems], non_blocking=True)
        for s in self._copy_streams:
            cur.wait_stream(s)

    # -- sharded checkpoints ("別再複製本可分片的東西：ZeRO 與 FSDP": each rank dumps
    #    its own shard in parallel) ---------------------------------------------------
    def _shard16_rows_view(self):
        if self.shard16 is not None:
            return [self.shard16[r] for r in range(self.n_d)]
        S = self.info.shard_len     # ZeRO-1/2 fused all-gather: rank r's slice of its replica
        return [self.params[r, r * S:(r + 1) * S] for r in range(self.n_d)]

    def save_checkpoint(self, path: str) -> dict:
        """Write one file per simulated rank (its fp32 master/m/v shard and
        16-bit parameter shard), in parallel, plus meta.json with the layout
        and the 96-byte step state.  Returns the bytes written."""
        os.makedirs(path, exist_ok=True)
        torch.cuda.synchronize(self.device)
        p16 = self._shard16_rows_view()

        chunk = 64 << 20                       # bytes per staged device-to-host copy

        def dump(r):
            # one pinned staging buffer per writer; the file gets the staged bytes as they are
            stage = torch.empty(chunk, dtype=torch.uint8, pin_memory=True)
            view = stage.numpy()
            stream = torch.cuda.Stream(self.device)
            with open(os.path.join(path, "rank%03d.bin" % r), "wb") as f, torch.cuda.stream(stream):
                for t in (self.master[r], self.m[r], self.v[r], p16[r].contiguous()):
                    flat = t.view(torch.uint8)
                    for off in range(0, flat.numel(), chunk):
                        n = min(chunk, flat.numel() - off)
                        stage[:n].copy_(flat[off:off + n], non_blocking=True)
                        stream.synchronize()
                        f.write(memoryview(view[:n]))
            return 14 * self.info.shard_len

        with ThreadPoolExecutor(max_workers=min(16, self.n_d)) as ex:
            nbytes = sum(ex.map(dump, range(self.n_d)))
        meta = {"format": "zero-shard-v1", "numels": self.numels,
                "unit_of_tensor": self.unit_of_tensor, "n_d": self.n_d, "stage": self.stage,
                "dtype": self.dtype, "bucket_elems": int(self.info.bucket_elems),
                "psi_pad": int(self.info.psi_pad), "shard_len": int(self.info.shard_len),
                "state": bytes(self.state.cpu().numpy().tobytes()).hex()}
        with open(os.path.join(path, "meta.json"), "w") as f:
            json.dump(meta, f)
        return {"bytes": nbytes}

    def load_checkpoint(self, path: str) -> dict:
        """Load a checkpoint written by any layout of the same tensors (other
        N_d, stage or unit split): the library's reshard plan maps every real
        element to its shard here; each of this layout's ranks is assembled on
        the host and uploaded once per array.  The 16-bit replicas of ZeRO-1/2
        are rebuilt from the shards by the all-gather kernel."""
        with open(os.path.join(path, "meta.json")) as f:
            meta = json.load(f)
        if meta.get("format") != "zero-shard-v1":
            raise ValueError("not a zero-shard-v1 checkpoint")
        src = B.zero_layout_init(meta["numels"], meta["unit_of_tensor"] if meta["stage"] == 3 else None,
                                 meta["n_d"], meta["stage"], 0, meta["bucket_elems"], meta["dtype"])
        if meta["dtype"] != self.dtype:
            raise ValueError("checkpoint dtype differs")
        plan = B.zero_reshard_plan(src, self.L)
        S0, S = meta["shard_len"], self.info.shard_len
        if B.zero_layout_query(src).shard_len != S0:
            raise ValueError("checkpoint shard_len %d does not match its own layout" % S0)
        st = bytes.fromhex(meta["state"])
        if len(st) != self.state.numel():
            raise ValueError("checkpoint step state has %d bytes, expected %d" % (len(st), self.state.numel()))
        files = []
        for r in range(meta["n_d"]):
            fn = os.path.join(path, "rank%03d.bin" % r)
            if os.path.getsize(fn) != 14 * S0:      # fp32 master, m, v + 16-bit parameters per element
                raise ValueError("%s holds %d bytes, expected %d" % (fn, os.path.getsize(fn), 14 * S0))
            files.append(np.memmap(fn, dtype=np.uint8, mode="r"))
        views = []
        for mm in files:
            f32 = mm[:12 * S0].view(np.float32)
            views.append((f32[:S0], f32[S0:2 * S0], f32[2 * S0:3 * S0], mm[12 * S0:14 * S0].view(np.uint16)))
        by_dst = {r: [] for r in range(self.n_d)}
        for seg in plan:
            by_dst[seg[2]].append(seg)
        p16_rows = self._shard16_rows_view()

        def assemble(r):
            host = [np.zeros(S, np.float32) for _ in range(3)] + [np.zeros(S, np.uint16)]
            for sr, so, dr, do, n in by_dst[r]:
                for k in range(4):
                    host[k][do:do + n] = views[sr][k][so:so + n]
            return r, host

        with ThreadPoolExecutor(max_workers=min(16, self.n_d)) as ex:
            for r, host in ex.map(assemble, range(self.n_d)):
                self.master[r].copy_(torch.from_numpy(host[0]))
                self.m[r].copy_(torch.from_numpy(host[1]))
                self.v[r].copy_(torch.from_numpy(host[2]))
                p16_rows[r].view(torch.int16).copy_(torch.from_numpy(host[3].view(np.int16)))
        self.state.copy_(torch.frombuffer(bytearray(st), dtype=torch.uint8))
        self._s().wait_stream(torch.cuda.current_stream(self.device))   # the uploads ran on the current stream
        if self.stage != 3:
            if self.shard16 is None:
                shards = torch.stack([t.clone() for t in p16_rows])
                self._s().wait_stream(torch.cuda.current_stream(self.device))
                B.zero_allgather_params(self.L, [shards[r] for r in range(self.n_d)], self.param_rows, self._s())
                torch.cuda.synchronize(self.device)
                del shards
            else:
                B.zero_allgather_params(self.L, self.shard16_rows, self.param_rows, self._s())
        torch.cuda.synchronize(self.device)
        return {"segments": len(plan), "bytes": 14 * S * self.n_d}

    # -- readback -------------------------------------------------------------------
    def read_state(self) -> dict:
        torch.cuda.synchronize(self.device)
        raw = bytes(self.state.cpu().numpy().tobytes())
        st = B.zero_step_state.from_buffer_copy(raw)
        return {"t": st.t, "skipped": st.skipped, "overflow": st.overflow, "apply": st.apply,
                "grad_norm": st.grad_norm, "clip_coef": st.clip_coef, "loss_scale": st.loss_scale,
                "good_steps": st.good_steps, "nonfinite": st.nonfinite, "error": st.error,
                "beta1_pow": st.beta1_pow, "beta2_pow": st.beta2_pow}

    def flat(self, which: str) -> torch.Tensor:
        """Reassemble master/m/v (fp32) or shard16 (ZeRO-3) into flat order."""
        src = {"master": self.master, "m": self.m, "v": self.v, "shard16": self.shard16,
               "gshard": self.gshard}[which]
        # the copies below run on the current stream: after the engine's own stream
        torch.cuda.current_stream(self.device).wait_stream(self._s())
        out = torch.zeros(self.info.psi_pad, dtype=src.dtype, device=src.device)
        for u in self.units:
            for r in range(self.n_d):
                lo = u.offset + r * u.shard
                out[lo:lo + u.shard].copy_(src[r, u.shard_base:u.shard_base + u.shard])
        return out
