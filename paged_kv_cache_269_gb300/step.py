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
                 partition_tokens=0, stream=None, host_out=False, max_groups=0):
        import torch
        self.torch = torch
        self.k_cache, self.v_cache = k_cache, v_cache
        N, H, B, D = k_cache.shape
        self.S, self.H, self.D, self.MB = max_seqs, H, D, max_blocks_per_seq
        self.scale, self.partition_tokens = float(scale), partition_tokens
        self.dev = k_cache.device
        self.dtype = k_cache.dtype
        self.stream = stream or torch.cuda.Stream(self.dev)
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
        the n rows, G <= max_groups; None shares nothing.  Waits for the
        previous step first, whose copy reads the same pinned buffer."""
        self.stream.synchronize()
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

    def launch(self):
        """Enqueue the staged step on self.stream; returns the output tensor
        (valid once the stream reaches this point) -- the pinned host copy
        when the step was built with host_out."""
        torch = self.torch
        if not self.use_graph:
            with torch.cuda.stream(self.stream):
                self._body()
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
        return self.out if self.out_host is None else self.out_host
