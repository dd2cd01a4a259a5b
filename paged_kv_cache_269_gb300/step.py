"""A decode step for a continuously batched set of sequences, replayable as a
CUDA graph.

Each step the caller hands over, for up to `max_seqs` running sequences, the
new token's q, k and v, the slot the KV block manager gave that token, and the
block tables and context lengths.  The step copies them to the device in one
host-to-device copy (they are packed into one pinned staging buffer), stores
the new K/V with reshape_and_cache and runs decode.  Rows past the batch are
padding: slot -1 (skipped by reshape_and_cache) and context length 0 (a zero
output row), so the launch shapes never change and the three operations can
be captured once as a CUDA graph and replayed every step.  Copy-on-write
copies reported by the manager are made eagerly, before the step, with
copy_blocks.

With max_groups > 0 the step decodes with decode_shared_prefix: the caller
also hands over the groups of adjacent rows that share prompt blocks (e.g.
KVManager.prefix_groups of the batch), staged with the other inputs; unused
group slots are empty, so the shapes still never change.

PipelinedDecodeStep runs two such steps in turn, each with its own staging
buffers, so that step k + 1's host-to-device copy (on a copy stream) overlaps
step k's kernels and the host reads step k's output after step k + 1 has been
launched.  The kernels of successive steps still run in order on one stream:
each step's reshape_and_cache writes the cache the next step's decode reads.

This module only orchestrates calls into libpa; all arithmetic runs in its
kernels.
"""
from __future__ import annotations

import numpy as np

from . import (copy_blocks, decode, decode_counters_bytes, decode_shared_prefix,
               decode_shared_prefix_counters_bytes, decode_shared_prefix_workspace_bytes,
               decode_workspace_bytes, reshape_and_cache)


class DecodeStep:
    def __init__(self, k_cache, v_cache, max_seqs, max_blocks_per_seq, scale, use_graph=True,
                 partition_tokens=0, stream=None, host_out=False, max_groups=0,
                 upload_stream=None):
        """upload_stream: None keeps the host-to-device copy in the step (in
        its graph); a stream moves it there, ordered by events: the copy waits
        until this step's previous kernels stopped reading the device buffer,
        and the kernels wait for the copy."""
        import torch
        self.torch = torch
        self.k_cache, self.v_cache = k_cache, v_cache
        N, H, B, D = k_cache.shape
        self.S, self.H, self.D, self.MB = max_seqs, H, D, max_blocks_per_seq
        self.scale, self.partition_tokens = float(scale), partition_tokens
        self.dev = k_cache.device
        self.dtype = k_cache.dtype
        self.stream = stream or torch.cuda.Stream(self.dev)
        self.upload_stream = upload_stream
        self.upload_done = torch.cuda.Event() if upload_stream is not None else None
        self.compute_done = torch.cuda.Event() if upload_stream is not None else None
        self.launched = False
        self.use_graph = use_graph
        self.graph = None
        self.G = int(max_groups)
        S, MB = max_seqs, max_blocks_per_seq
        # packed layout: name -> (offset, shape, numpy dtype, torch dtype), 256-byte aligned
        el = np.float16 if self.dtype == torch.float16 else np.uint16
        fields = [("q", (S, H, D), el, self.dtype), ("k_new", (S, H, D), el, self.dtype),
                  ("v_new", (S, H, D), el, self.dtype), ("slots", (S,), np.int32, torch.int32),
                  ("tables", (S, MB), np.int32, torch.int32),
                  ("lens", (S,), np.int32, torch.int32)]
        if self.G > 0:
            fields += [("gstart", (self.G + 1,), np.int32, torch.int32),
                       ("gpre", (self.G,), np.int32, torch.int32)]
        self.layout, off = {}, 0
        for name, shape, nd, td in fields:
            nbytes = int(np.prod(shape)) * np.dtype(nd).itemsize
            self.layout[name] = (off, shape, nd, td, nbytes)
            off += (nbytes + 255) // 256 * 256
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.devbuf = torch.empty(off, dtype=torch.uint8, device=self.dev)
        hb = self.host.numpy()
        self.h = {n: hb[o:o + nb].view(nd).reshape(shape) for n, (o, shape, nd, td, nb)
                  in self.layout.items()}
        self.d = {n: self.devbuf[o:o + nb].view(td).view(shape) for n, (o, shape, nd, td, nb)
                  in self.layout.items()}
        self.out = torch.zeros((S, H, D), dtype=self.dtype, device=self.dev)
        # with host_out, the decode writes its output straight into pinned
        # host memory over the host link (no separate copy); read it after
        # the stream reaches the end of the step
        self.out_host = (torch.empty((S, H, D), dtype=self.dtype).pin_memory()
                         if host_out else None)
        self.dst = self.out_host if host_out else self.out
        dt = 1 if self.dtype == torch.bfloat16 else 0
        if self.G > 0:
            ws = decode_shared_prefix_workspace_bytes(S, H, D, B, N, MB, partition_tokens, dtype=dt)
            ctr = decode_shared_prefix_counters_bytes(S, H, D, B, N)
        else:
            ws = decode_workspace_bytes(S, H, D, B, N, MB, partition_tokens, dtype=dt)
            ctr = decode_counters_bytes(S, H, D, B, N)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=self.dev)
        self.counters = torch.zeros(ctr // 4, dtype=torch.int32, device=self.dev)
        self.h["slots"][:] = -1
        self.h["lens"][:] = 0
        self.h["tables"][:] = -1
        if self.G > 0:
            self.h["gstart"][:] = 0
            self.h["gpre"][:] = 0

    def prepare(self, q, k_new, v_new, slots, tables, lens, groups=None):
        """Stage one step's inputs (numpy; n <= max_seqs rows) into the pinned
        buffer; rows n .. max_seqs-1 become padding.  groups (with
        max_groups > 0): (group_start [G + 1], group_prefix_blocks [G]) over
        the n rows, G <= max_groups; None shares nothing.  Waits first for
        the previous copy out of the same pinned buffer (the previous step)."""
        if self.upload_stream is None:
            self.stream.synchronize()
        elif self.launched:
            self.upload_done.synchronize()
        n = len(lens)
        if n > self.S:
            raise ValueError("more sequences than max_seqs")
        h = self.h
        for name, val in (("q", q), ("k_new", k_new), ("v_new", v_new)):
            h[name][:n] = val
        h["slots"][:n] = slots
        h["slots"][n:] = -1
        h["tables"][:n] = tables[:, :self.MB]
        h["tables"][n:] = -1
        h["lens"][:n] = lens
        h["lens"][n:] = 0
        if self.G > 0:
            gs, gp = groups if groups is not None else (np.zeros(1, np.int32), np.zeros(0, np.int32))
            g = len(gp)
            if g > self.G or len(gs) != g + 1:
                raise ValueError("more groups than max_groups, or inconsistent group arrays")
            h["gstart"][:g + 1] = gs
            h["gstart"][g + 1:] = gs[-1]
            h["gpre"][:g] = gp
            h["gpre"][g:] = 0
        elif groups is not None:
            raise ValueError("groups need a step built with max_groups > 0")

    def _body(self):
        d = self.d
        if self.upload_stream is None:
            self.devbuf.copy_(self.host, non_blocking=True)
        reshape_and_cache(d["k_new"], d["v_new"], self.k_cache, self.v_cache, d["slots"])
        if self.G > 0:
            decode_shared_prefix(self.dst, d["q"], self.k_cache, self.v_cache, d["tables"],
                                 d["lens"], self.scale, d["gstart"], d["gpre"],
                                 max_group_size=self.S, partition_tokens=self.partition_tokens,
                                 workspace=self.workspace, counters=self.counters)
        else:
            decode(self.dst, d["q"], self.k_cache, self.v_cache, d["tables"], d["lens"],
                   self.scale, partition_tokens=self.partition_tokens, workspace=self.workspace,
                   counters=self.counters)

    def copy_on_write(self, pairs):
        """Make the manager's copy-on-write copies ((src, dst) rows) before the step."""
        if len(pairs):
            with self.torch.cuda.stream(self.stream):
                t = self.torch.as_tensor(np.asarray(pairs, np.int32).reshape(-1, 2),
                                         device=self.dev)
                copy_blocks(self.k_cache, self.v_cache, self.k_cache, self.v_cache, t)

    def _upload(self):
        """With an upload stream: copy the staged inputs there once this
        step's previous kernels are done with the device buffer, and make the
        step's stream wait for the copy."""
        torch = self.torch
        if self.upload_stream is None:
            return
        with torch.cuda.stream(self.upload_stream):
            if self.launched:
                self.upload_stream.wait_event(self.compute_done)
            self.devbuf.copy_(self.host, non_blocking=True)
            self.upload_done.record(self.upload_stream)
        self.stream.wait_event(self.upload_done)

    def launch(self):
        """Enqueue the staged step on self.stream; returns the output tensor
        (valid once the stream reaches this point) -- the pinned host copy
        when the step was built with host_out."""
        torch = self.torch
        self._upload()
        if not self.use_graph:
            with torch.cuda.stream(self.stream):
                self._body()
            self._done()
            return self.out if self.out_host is None else self.out_host
        if self.graph is None:
            with torch.cuda.stream(self.stream):
                self._body()                        # warm-up: kernels set up outside capture
            self.stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self._body()
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        self._done()
        return self.out if self.out_host is None else self.out_host

    def _done(self):
        self.launched = True
        if self.compute_done is not None:
            self.compute_done.record(self.stream)

    def synchronize(self):
        """Wait until this step's last launch has finished (its output is then
        readable)."""
        if self.compute_done is not None and self.launched:
            self.compute_done.synchronize()
        else:
            self.stream.synchronize()


class PipelinedDecodeStep:
    """Two DecodeSteps used in turn: step k + 1's inputs are copied to the
    device on a copy stream while step k's kernels run, and step k's output
    is read after step k + 1 has been launched.

    submit(...) stages one step's inputs (as DecodeStep.prepare) into the next
    slot and launches it, returning a ticket; result(ticket) waits for that
    step and returns its output (a pinned host tensor with host_out).  The
    output buffer of a slot is rewritten by the step submitted two tickets
    later, so read a result before submitting the step after next.
    prepare() / launch() split submit for callers that relaunch staged
    inputs."""

    def __init__(self, k_cache, v_cache, max_seqs, max_blocks_per_seq, scale, use_graph=True,
                 partition_tokens=0, stream=None, host_out=False, max_groups=0, depth=2):
        import torch
        self.stream = stream or torch.cuda.Stream(k_cache.device)
        self.upload_stream = torch.cuda.Stream(k_cache.device)
        self.steps = [DecodeStep(k_cache, v_cache, max_seqs, max_blocks_per_seq, scale,
                                 use_graph=use_graph, partition_tokens=partition_tokens,
                                 stream=self.stream, host_out=host_out, max_groups=max_groups,
                                 upload_stream=self.upload_stream) for _ in range(depth)]
        self.next = 0

    def prepare(self, *args, **kw):
        """Stage inputs into the slot the next launch() uses."""
        self.steps[self.next % len(self.steps)].prepare(*args, **kw)

    def launch(self):
        """Launch the next slot's staged inputs; returns its ticket."""
        t = self.next
        self.steps[t % len(self.steps)].launch()
        self.next += 1
        return t

    def submit(self, *args, **kw):
        self.prepare(*args, **kw)
        return self.launch()

    def result(self, ticket):
        if not self.next - len(self.steps) <= ticket < self.next:
            raise ValueError("not one of the last steps submitted (a later step has "
                             "rewritten its output, or it was never submitted)")
        st = self.steps[ticket % len(self.steps)]
        st.synchronize()
        return st.out if st.out_host is None else st.out_host

    def copy_on_write(self, pairs):
        """Make copy-on-write copies before the next step (on the step stream)."""
        self.steps[0].copy_on_write(pairs)
