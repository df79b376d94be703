"""One step of the whole hot path on device-resident buffers.

A step is what one tensor-parallel layer boundary does, with the P ranks
standing in as P slabs in one GPU's HBM:

* quantized formats (INT8 / INT4): sender-side group quantization of all P
  slabs (one launch), then the fused two-step reduce + residual add +
  RMSNorm (one launch) that also writes the requantized all-gather payload;
* BF16: the fused reduce + residual add + RMSNorm on the bf16 slabs;
* BF16_TAGGED: the producers pack every slab into epoch-tagged blocks with a
  fresh epoch (one launch for all slabs), then the consumer validates and reduces
  them.

With ``splits`` > 1 (BF16_TAGGED, INT8, INT4) the token rows are split into
that many subsets whose fused calls run on their own streams (TokenWeave's
token splitting), at even or wave-aware boundaries.

All device memory is allocated here by torch at construction; ``step()``
only launches libfcomm kernels.  ``alg_bytes()`` gives the bytes the method
must move per step (intermediates kept on chip are not counted).
"""
from __future__ import annotations

import numpy as np
import torch

from . import fcomm as fc
from .synth import (FMT_BF16, FMT_BF16_TAGGED, FMT_INT4_ASYM, FMT_INT8_SYM, QTAGGED, Workload,
                    base_format)


def _bf16_dev(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def qs_bytes(w: Workload, E: int) -> int:
    """Bytes of one quantized slab of E elements: codes + scales (+ zeros)."""
    ng = E // w.group
    fmt = base_format(w.fmt)
    if fmt == FMT_INT8_SYM:
        return E + 4 * ng
    if fmt == FMT_INT4_ASYM:
        return E // 2 + 8 * ng
    raise ValueError(w.fmt)


class Pipeline:
    def __init__(self, w: Workload, inputs: dict, device="cuda", with_payload=True,
                 split: str = "even"):
        self.w = w
        self.device = device
        self.spec = fc.QSpec(w.fmt, w.group)
        T, H = w.T, w.H
        self.x = [_bf16_dev(s, device) for s in inputs["slabs"]]
        self.residual = _bf16_dev(inputs["residual"], device)
        self.gamma = _bf16_dev(inputs["gamma"], device)
        self.residual_out = torch.empty_like(self.residual)
        self.y = torch.empty_like(self.residual)
        self.epoch = 0
        self.status = None
        self.payload = None
        if w.fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
            self.codes = [fc.alloc_qtensor(self.spec, T, H, device) for _ in range(w.P)]
            if with_payload:
                self.payload = fc.alloc_qtensor(self.spec, T, H, device)
        elif w.fmt in QTAGGED:
            self.blocks = [torch.empty(fc.codes_bytes(self.spec, T, H), dtype=torch.uint8,
                                       device=device) for _ in range(w.P)]
            self.status = torch.zeros(1, 2, dtype=torch.int32, device=device)
            if with_payload:
                self.payload = fc.alloc_qtensor(fc.QSpec(base_format(w.fmt), w.group), T, H, device)
        elif w.fmt == FMT_BF16_TAGGED:
            self.blocks = [torch.empty(fc.tagged_bytes(T, H), dtype=torch.uint8, device=device)
                           for _ in range(w.P)]
            self.status = torch.zeros(max(1, w.splits), 2, dtype=torch.int32, device=device)
        if max(1, w.splits) > 1:
            self.streams = [torch.cuda.Stream(device=device) for _ in range(w.splits)]
        # token-subset boundaries: even, or wave-aware (the first subset is
        # whole waves of the fused kernel on this GPU)
        n = max(1, w.splits)
        if split == "wave" and n == 2:
            first, self.wave_rows = fc.token_split(self.spec, w.P, w.T, w.H)
            self.bounds = [0, first, w.T]
        else:
            self.wave_rows = None
            self.bounds = [w.T * i // n for i in range(n + 1)]
        self.launches_per_step = self._launches()
        self.graph = None
        self._bind()

    def _bind(self):
        """Marshal every launch of a step once (fcomm.Bound): a step then
        spends no host time converting arguments."""
        w = self.w
        self._send, self._fuse, self._split = None, None, []
        if w.fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
            self._send = fc.bind_group_quantize_multi(self.x, self.spec, self.codes)
            if max(1, w.splits) == 1:
                self._fuse = fc.bind_allreduce_residual_rmsnorm(
                    self.codes, self.spec, w.T, w.H, self.residual, self.residual_out, self.gamma,
                    w.eps, self.y, requant_out=self.payload)
            else:  # token subsets: each a fused call over its rows' codes, scales, zeros
                for i in range(w.splits):
                    r0, r1 = self.bounds[i], self.bounds[i + 1]
                    rows = lambda q: None if q is None else q[self._qoff(q, r0):self._qoff(q, r1)]
                    sub = lambda qt: tuple(rows(q) for q in qt)
                    self._split.append(fc.bind_allreduce_residual_rmsnorm(
                        [sub(c) for c in self.codes], self.spec, r1 - r0, w.H,
                        self.residual[r0:r1], self.residual_out[r0:r1], self.gamma, w.eps,
                        self.y[r0:r1],
                        requant_out=None if self.payload is None else sub(self.payload)))
        elif w.fmt in QTAGGED:
            self._send = fc.bind_group_quantize_tagged(self.x, self.spec, self.epoch, self.blocks)
            self._fuse = fc.bind_allreduce_residual_rmsnorm(
                self.blocks, self.spec, w.T, w.H, self.residual, self.residual_out, self.gamma,
                w.eps, self.y, requant_out=self.payload, expected_epoch=self.epoch,
                d_status=self.status[0])
        elif w.fmt == FMT_BF16:
            self._fuse = fc.bind_allreduce_residual_rmsnorm(
                self.x, self.spec, w.T, w.H, self.residual, self.residual_out, self.gamma, w.eps,
                self.y)
        else:
            self._send = fc.bind_pack_tagged_multi(self.x, self.epoch, self.blocks)
            bpr = fc.tagged_bytes(1, w.H)
            for i in range(max(1, w.splits)):
                r0, r1 = self.bounds[i], self.bounds[i + 1]
                self._split.append(fc.bind_allreduce_residual_rmsnorm(
                    [b[r0 * bpr:r1 * bpr] for b in self.blocks], self.spec, r1 - r0, w.H,
                    self.residual[r0:r1], self.residual_out[r0:r1], self.gamma, w.eps,
                    self.y[r0:r1], expected_epoch=self.epoch, d_status=self.status[i]))

    def _qoff(self, q, r: int) -> int:
        """Index of row r's first entry in a flat codes, scales or zeros tensor."""
        return r * (q.numel() // self.w.T)

    # ------------------------------------------------------------------
    def _launches(self) -> int:
        """Kernels launched per step: the sender, the consumer call(s), and for
        each consumer call that takes a status word the one-thread kernel
        that resets it."""
        w = self.w
        if w.fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
            return 1 + max(1, w.splits)
        if w.fmt in QTAGGED:
            return 1 + 2
        if w.fmt == FMT_BF16:
            return 1
        return 1 + 2 * max(1, w.splits)

    def step(self, stream=None):
        """Launch one pass of the hot path on `stream` (default: current)."""
        st = stream or torch.cuda.current_stream(self.device)
        self.sender(st)
        self.consumer(st)

    def capture(self):
        """Capture one step into a CUDA graph; replay() then issues the whole
        step with one host call (the launches keep their programmatic
        dependent launch edges inside the graph).  Untagged formats only: a
        tagged step packs a fresh epoch every time, which a graph would fix
        at the captured value."""
        w = self.w
        if w.fmt in QTAGGED or w.fmt == FMT_BF16_TAGGED:
            raise ValueError("graph capture is for untagged formats (the epoch changes per step)")
        cur = torch.cuda.current_stream(self.device)
        s = torch.cuda.Stream(self.device)
        s.wait_stream(cur)
        self.step(s)  # every launch shape resolved before capture
        cur.wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.step(s)
        self.graph = g
        return g

    def replay(self, stream=None):
        """Launch the captured step (capture() first) on `stream` (default: current)."""
        st = stream or torch.cuda.current_stream(self.device)
        if st != torch.cuda.current_stream(self.device):
            with torch.cuda.stream(st):
                self.graph.replay()
        else:
            self.graph.replay()

    def step_marked(self, stream, marks):
        """step() with CUDA events marks[0], marks[1], marks[2] recorded before
        the sender stage, between the stages and after the fused stage."""
        marks[0].record(stream)
        self.sender(stream)
        marks[1].record(stream)
        self.consumer(stream)
        marks[2].record(stream)

    def sender(self, st):
        """Sender side: group-quantize (INT8/INT4) or pack with a fresh epoch (tagged)."""
        w = self.w
        if w.fmt in QTAGGED or w.fmt == FMT_BF16_TAGGED:
            self.epoch = (self.epoch + 1) & 0xFFFFFFFF
            self._send.epoch = self.epoch
        if self._send is not None:
            self._send(st)

    def consumer(self, st):
        """Receiver side: the fused reduce + residual add + RMSNorm."""
        if self._fuse is not None:
            self._fuse.epoch = self.epoch
            self._fuse(st)
        else:
            self._split_consume(st)

    def _split_consume(self, st):
        fork = torch.cuda.Event()
        fork.record(st)
        joins = []
        for call, s in zip(self._split, self.streams):
            s.wait_event(fork)
            if self.w.fmt == FMT_BF16_TAGGED:
                call.epoch = self.epoch
            call(s)
            ev = torch.cuda.Event()
            ev.record(s)
            joins.append(ev)
        for ev in joins:
            st.wait_event(ev)

    # ------------------------------------------------------------------
    def alg_bytes(self) -> dict:
        """Algorithmic bytes per step, by stage: {'sender': .., 'fused': ..}."""
        w = self.w
        E, H, P = w.T * w.H, w.H, w.P
        if w.fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
            qs = qs_bytes(w, E)
            return {"sender": P * 2 * E + P * qs,
                    "fused": P * qs + 2 * E + max(1, w.splits) * 2 * H
                    + (qs if self.payload is not None else 0) + 4 * E}
        if w.fmt in QTAGGED:
            tb = fc.codes_bytes(self.spec, w.T, w.H)
            qs = qs_bytes(w, E)
            return {"sender": P * 2 * E + P * tb,
                    "fused": P * tb + 2 * E + 2 * H + (qs if self.payload is not None else 0)
                    + 4 * E}
        if w.fmt == FMT_BF16:
            return {"sender": 0, "fused": P * 2 * E + 2 * E + 2 * H + 4 * E}
        tb = fc.tagged_bytes(w.T, w.H)
        return {"sender": P * 2 * E + P * tb,
                "fused": P * tb + 2 * E + max(1, w.splits) * 2 * H + 4 * E}

    def outputs(self) -> dict:
        """Host copies (uint16 bf16 bits etc.) of the step's outputs."""
        torch.cuda.synchronize(self.device)
        out = dict(h=self.residual_out.view(torch.int16).cpu().numpy().view(np.uint16),
                   y=self.y.view(torch.int16).cpu().numpy().view(np.uint16))
        if self.payload is not None:
            out.update(codes=self.payload[0].cpu().numpy(), scales=self.payload[1].cpu().numpy(),
                       zeros=None if self.payload[2] is None else self.payload[2].cpu().numpy())
        if self.status is not None:
            out["status"] = self.status.cpu().numpy()
        return out
