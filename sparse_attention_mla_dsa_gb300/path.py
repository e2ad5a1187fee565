"""Device-resident state and one decode step of the DSA hot path.

``DeviceWorkload`` uploads a synthetic workload (key arena, gate, paged FP8
latent pool, per-row metadata and queries) once and runs the four C-ABI calls
in stream order -- S0 latent write (when the workload writes new rows), S1
index scores, S2 top-k, S3 gather-attend -- without any host synchronisation.

``DsaDecoder`` is the host-facing form: per step it copies that step's inputs
(queries, head weights, the new latent rows, row metadata) from one pinned
host staging buffer to the device in one copy, runs the same four calls, and
the gather-attend writes the attention output straight into pinned host memory.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api


def _dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceWorkload:
    """All inputs of a workload resident on one CUDA device, plus outputs."""

    def __init__(self, wl, device: str | torch.device = "cuda", pool: torch.Tensor | None = None,
                 _clone_of: "DeviceWorkload | None" = None):
        self.wl = wl
        if _clone_of is not None:
            self._init_clone(_clone_of)
            return
        self.device = torch.device(device)
        d = self.device
        self.seq_lens = _dev(wl.seq_lens.astype(np.int32), d)
        self.positions = _dev(wl.positions.astype(np.int32), d)
        self.slots = _dev(wl.slots.astype(np.int64), d)
        self.block_table = _dev(wl.block_table.astype(np.int32), d)
        self.pool = pool if pool is not None else _dev(wl.pool, d)
        self.idx_k = _dev(wl.idx_k, d)
        self.idx_gate = _dev(wl.idx_gate, d)
        self.idx_base = _dev(wl.idx_base.astype(np.int64), d)
        self.q_idx = _dev(wl.q_idx, d)
        self.head_w = _dev(wl.head_w, d)
        self.Q = _dev(wl.Q, d)
        self.kv_a = _dev(wl.kv_a, d) if wl.kv_a is not None else None
        self.norm_w = _dev(wl.norm_w, d) if wl.norm_w is not None else None
        R, H = wl.rows, wl.heads
        self.max_len = max(1, wl.max_len)
        self.scores = torch.empty((R, self.max_len), dtype=torch.float32, device=d)
        self.sel = torch.empty((R, wl.topk), dtype=torch.int32, device=d)
        self.out = torch.empty((R, H, 512), dtype=torch.int16, device=d)
        self.lse = torch.empty((R, H), dtype=torch.float32, device=d)
        nbytes = api.dsa_workspace_bytes(R, H, wl.topk)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=d)
        self.out_target = None      # where S3 writes; None = self.out
        self.rows = api.make_rows(self.seq_lens, self.block_table, wl.block_size, self.slots,
                                  self.positions, shared_table=(wl.bt_stride == 0))

    def _init_clone(self, src: "DeviceWorkload"):
        self.device = src.device
        for name in ("seq_lens", "positions", "slots", "block_table", "pool", "idx_k", "idx_gate",
                     "idx_base", "q_idx", "head_w", "Q", "kv_a", "norm_w", "scores", "sel", "out",
                     "lse", "workspace"):
            t = getattr(src, name)
            setattr(self, name, None if t is None else t.clone())
        self.max_len = src.max_len
        self.out_target = None
        wl = self.wl
        self.rows = api.make_rows(self.seq_lens, self.block_table, wl.block_size, self.slots,
                                  self.positions, shared_table=(wl.bt_stride == 0))

    def clone(self) -> "DeviceWorkload":
        """An independent copy at new device addresses (for cold-cache rotation)."""
        return DeviceWorkload(self.wl, _clone_of=self)

    def input_bytes(self) -> int:
        return sum(getattr(self, n).numel() * getattr(self, n).element_size()
                   for n in ("pool", "idx_k", "idx_gate", "Q", "q_idx"))

    # ---- the four steps
    def latent_write(self, stream=None):
        wl = self.wl
        api.dsa_latent_write(self.rows, self.kv_a, self.norm_w, self.pool, wl.eps, wl.kv_scale,
                             stream)

    def index_scores(self, stream=None, inputs_early: bool = False):
        """S1.  ``inputs_early``: the indexer's inputs (resident here, or
        uploaded before the step) were complete before the kernel issued just
        before this call started, so the indexer may load and score them
        before its dependency wait (its stores still wait)."""
        api.dsa_index_scores(self.rows, self.q_idx, self.head_w, self.idx_k, self.idx_gate,
                             self.idx_base, self.wl.group_rows, self.max_len, self.scores,
                             stream=stream, inputs_early=inputs_early)

    def select_topk(self, stream=None):
        api.dsa_select_topk(self.rows, self.scores, self.max_len, self.wl.topk, self.sel, stream)

    def mla_decode(self, stream=None, q_early: bool = False):
        """S3.  ``q_early``: the call follows this workload's top-k on the same
        stream (Q was uploaded before the step), so the attend may convert Q
        before its dependency wait.  The split plan is the workload's
        (``long_splits``)."""
        wl = self.wl
        out = self.out if self.out_target is None else self.out_target
        api.dsa_mla_decode_fp8(self.rows, self.Q, self.pool, self.sel, wl.topk, wl.kv_scale,
                               wl.sm_scale, out, self.lse, self.workspace, stream, q_early=q_early,
                               long_splits=wl.long_splits)

    def step(self, stream=None):
        """One pass of the whole hot path (S0 when the workload writes, S1-S3)."""
        if self.kv_a is not None:
            self.latent_write(stream)
        self.index_scores(stream, inputs_early=True)  # no kernel of the step writes its inputs
        self.select_topk(stream)
        self.mla_decode(stream, q_early=True)  # right after this workload's top-k

    # ---- host views of the results
    def out_f32(self) -> np.ndarray:
        return self.out.view(torch.bfloat16).float().cpu().numpy()


class DsaDecoder:
    """Host-facing decode: resident caches, per-step host inputs and outputs.

    The caches (key arena, gate, FP8 latent pool) live on the device; each
    ``decode`` call copies the step's inputs from pinned host memory to the
    device, runs S0-S3, and the gather-attend writes the attention output into
    pinned host memory.  The per-step
    inputs (queries, head weights, the new latent rows, row metadata) sit in
    one pinned staging buffer mirrored by one device buffer per cache replica,
    whose views the kernels read, so a step moves its inputs in one copy.
    With ``graphs=True`` (the default) the whole sequence -- the host-to-device
    copy and the four calls -- is captured once per
    cache replica as a CUDA graph and replayed, so a step costs one launch;
    the buffers keep their addresses, so each replay moves the current
    contents of the pinned inputs."""

    _INPUTS = ("q_idx", "head_w", "Q", "seq_lens", "positions", "slots", "block_table",
               "idx_base")

    def __init__(self, wl, device: str | torch.device = "cuda", replicas: int = 1,
                 graphs: bool = True):
        first = DeviceWorkload(wl, device)
        self.replicas = [first] + [first.clone() for _ in range(replicas - 1)]
        self._next = 0
        self._graphs = [None] * len(self.replicas) if graphs else None
        names = self._INPUTS + (("kv_a",) if first.kv_a is not None else ())
        layout, off = [], 0
        for name in names:
            t = getattr(first, name)
            nbytes = t.numel() * t.element_size()
            layout.append((name, off, nbytes, t.dtype, tuple(t.shape)))
            off = (off + nbytes + 255) // 256 * 256
        self._stage_bytes = off
        self._host = torch.empty(off, dtype=torch.uint8, pin_memory=True)
        self._host_in = {name: self._host[o:o + n].view(dt).view(shape)
                         for name, o, n, dt, shape in layout}
        for dw in self.replicas:
            buf = torch.empty(off, dtype=torch.uint8, device=first.device)
            for name, o, n, dt, shape in layout:
                view = buf[o:o + n].view(dt).view(shape)
                view.copy_(getattr(dw, name))
                setattr(dw, name, view)
            dw.stage_buf = buf
            dw.rows = api.make_rows(dw.seq_lens, dw.block_table, wl.block_size, dw.slots,
                                    dw.positions, shared_table=(wl.bt_stride == 0))
        # Pinned host memory is mapped into the device's address space: the
        # gather-attend (or its merge) stores the output there directly, so no
        # device-to-host copy follows the step.
        self.host_out = torch.empty(first.out.shape, dtype=first.out.dtype, pin_memory=True)
        for dw in self.replicas:
            dw.out_target = self.host_out

    @property
    def h2d_bytes(self) -> int:
        return self._stage_bytes

    @property
    def d2h_bytes(self) -> int:
        return self.host_out.numel() * self.host_out.element_size()

    def stage(self, wl) -> None:
        """Fill the pinned input buffers from a workload's per-step arrays."""
        src = {"q_idx": wl.q_idx, "head_w": wl.head_w, "Q": wl.Q.view(np.int16),
               "seq_lens": wl.seq_lens.astype(np.int32), "positions": wl.positions.astype(np.int32),
               "slots": wl.slots.astype(np.int64), "block_table": wl.block_table.astype(np.int32),
               "idx_base": wl.idx_base.astype(np.int64)}
        if "kv_a" in self._host_in:
            src["kv_a"] = wl.kv_a.view(np.int16)
        for k, t in self._host_in.items():
            t.copy_(torch.from_numpy(np.ascontiguousarray(src[k])))

    def _run(self, dw, stream=None) -> None:
        dw.stage_buf.copy_(self._host, non_blocking=True)
        dw.step(stream)                       # S3 writes straight into host_out

    def decode(self, stream=None) -> torch.Tensor:
        """Copy staged inputs in, run the path, copy the output out (async on
        the current stream; synchronise before reading ``host_out``).
        Successive calls rotate over the resident cache replicas."""
        i = self._next
        dw = self.replicas[i]
        self._next = (self._next + 1) % len(self.replicas)
        if self._graphs is None:
            self._run(dw, stream)
            return self.host_out
        if self._graphs[i] is None:
            self._run(dw, stream)              # first use of this replica runs eagerly
            torch.cuda.current_stream().synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._run(dw)
            self._graphs[i] = g
            return self.host_out
        self._graphs[i].replay()
        return self.host_out
