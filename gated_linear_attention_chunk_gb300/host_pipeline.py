"""Prefill from pinned host memory with the copies overlapped (plumbing, no arithmetic).

``HostPrefill`` runs ``kda_chunk_fwd`` over a packed batch whose inputs live in
pinned host memory and whose outputs go back to pinned host memory.  The batch
is cut into pieces: runs of whole sequences, and, for a sequence much longer
than a piece's share of the tokens, parts of that sequence cut at chunk
(64-token) boundaries.  Piece i's inputs travel host -> device on one stream
while piece i-1 computes on a second stream and piece i-2's outputs travel
device -> host on a third, so the host link, the kernels and the return copies
work at the same time instead of one after the other; the more pieces, the
shorter the pipeline's fill and drain.  Every piece is an ordinary
``kda_chunk_fwd`` call on a contiguous token range (the packed layout keeps a
sequence's tokens contiguous), with the full workspace of that call.  The parts
of one sequence run one after the other: the fp32 state at a part's end stays
in device memory and is the next part's initial state (updated in place), which
is how the chunked kernel carries its state from chunk to chunk inside one
call.  Each piece takes whatever path ``kda_chunk_fwd`` picks for its shape (a
piece of few chains may take the T-segment split) and carries that call's
accuracy.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch

from . import kda as _kda


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t if t.is_pinned() else t.pin_memory()


def plan_groups(cu: List[int], groups: int) -> List[Tuple[int, int]]:
    """Cuts N sequences (token offsets ``cu``, N + 1 of them) into at most ``groups`` runs of
    whole sequences [a, b) with about the same number of tokens each: boundary i is the
    sequence offset nearest to i / groups of the tokens, kept strictly increasing so that no
    group is empty (lengths of zero are allowed and go with their neighbours)."""
    N = len(cu) - 1
    groups = max(1, min(int(groups), N))
    T = cu[N] - cu[0]
    bounds: List[int] = [0]
    for i in range(1, groups):
        target = cu[0] + T * i / groups
        bounds.append(min(range(bounds[-1] + 1, N - (groups - i) + 1), key=lambda m: abs(cu[m] - target)))
    bounds.append(N)
    return [(bounds[i], bounds[i + 1]) for i in range(groups) if bounds[i + 1] > bounds[i]]


def plan_pieces(cu: List[int], pieces: int, align: int = 64) -> List[Tuple[int, int, int, int]]:
    """Pieces (a, b, t0, t1) of the batch: sequences [a, b) and their tokens [t0, t1).

    The sequence groups of ``plan_groups(cu, pieces)`` come first.  A group that is a
    single sequence longer than 1.5 x the share T / pieces is then cut into about
    length / share parts at multiples of ``align`` tokens from the sequence's start (so
    that every part but the last holds whole chunks); such a part has b == a + 1 and a
    token range inside the sequence.  The result may hold a few more pieces than asked
    for; the pieces cover every token once, in order."""
    N = len(cu) - 1
    T = cu[N] - cu[0]
    share = max(1, -(-T // max(1, int(pieces))))
    out: List[Tuple[int, int, int, int]] = []
    for a, b in plan_groups(cu, pieces):
        L = cu[b] - cu[a]
        if b == a + 1 and 2 * L > 3 * share and L > align:
            k = -(-L // share)
            cuts = sorted({round(L * i / k / align) * align for i in range(1, k)})
            ends = [0] + [x for x in cuts if 0 < x < L] + [L]
            out.extend((a, b, cu[a] + s0, cu[a] + s1) for s0, s1 in zip(ends, ends[1:]))
        else:
            out.append((a, b, cu[a], cu[b]))
    return out


class HostPrefill:
    """Pipelined host -> device -> host prefill of one packed batch.

    Inputs (CPU tensors, pinned or made pinned once here): q, k, g [T, H, dk], v [T, H, dv],
    beta [T, H], cu_seqlens [N + 1] int32, init_state [N, H, dk, dv] fp32 or None.
    ``groups`` is about the number of pieces (``plan_pieces``).  ``run()`` copies the inputs
    in, computes, and leaves o and final_state in the pinned host tensors ``host_o`` and
    ``host_final_state``; it returns once the last copy has been issued (synchronize the
    device, or ``self.done``, before reading them).

    With ``graph=True`` the pass is issued once more under CUDA-graph capture (on the second
    ``run()``; the first runs as usual) and every later ``run()`` replays that graph: the
    copies read the same pinned host tensors, so new inputs written into ``self.host`` (and
    ``host_s0``) in place are picked up, while the host no longer issues each copy and call
    of every piece in every pass.
    """

    def __init__(self, q, k, v, g, beta, cu_seqlens, init_state=None, scale: float = 1.0,
                 groups: int = 4, device="cuda", graph: bool = False):
        self.device = torch.device(device)
        self.host = {n: _pinned(x) for n, x in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}
        self.host_s0 = None if init_state is None else _pinned(init_state)
        cu = [int(x) for x in cu_seqlens.tolist()]
        N = len(cu) - 1
        T, H, dk = q.shape
        dv = v.shape[2]
        self.scale = float(scale)
        self.groups = plan_pieces(cu, groups)
        # per-piece cu_seqlens, rebased to the piece's first token (host side, pinned)
        self.host_cu = [_pinned(torch.tensor([0, t1 - t0] if self._part(a, b, t0, t1, cu) else
                                             [c - cu[a] for c in cu[a:b + 1]], dtype=torch.int32))
                        for a, b, t0, t1 in self.groups]
        self.cu = cu
        dev = self.device
        self.dev = {n: torch.empty_like(x, device=dev) for n, x in self.host.items()}
        self.dev_cu = [torch.empty_like(c, device=dev) for c in self.host_cu]
        self.dev_s0 = None if self.host_s0 is None else torch.empty_like(self.host_s0, device=dev)
        self.o = torch.empty(T, H, dv, dtype=q.dtype, device=dev)
        self.final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
        self.host_o = torch.empty(T, H, dv, dtype=q.dtype).pin_memory()
        self.host_final_state = torch.empty(N, H, dk, dv, dtype=torch.float32).pin_memory()
        # the running state of every sequence that is cut into parts, between its parts
        self.carry = {a: torch.empty(1, H, dk, dv, dtype=torch.float32, device=dev)
                      for a, b, t0, t1 in self.groups if self._part(a, b, t0, t1, cu)}
        # one workspace per piece, so that every piece's device status survives the pass
        self.workspaces = [_kda.new_workspace(_kda.kda_chunk_fwd_workspace_size(b - a, t1 - t0, H, dk, dv), dev)
                           for a, b, t0, t1 in self.groups]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_run = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.done: Optional[torch.cuda.Event] = None
        self.use_graph = bool(graph)
        self._graph = None
        self._passes = 0
        self.h2d_bytes = sum(x.numel() * x.element_size() for x in self.host.values())
        self.h2d_bytes += sum(c.numel() * 4 for c in self.host_cu)
        if self.host_s0 is not None:
            self.h2d_bytes += self.host_s0.numel() * 4
        self.d2h_bytes = self.host_o.numel() * self.host_o.element_size() + self.host_final_state.numel() * 4

    @staticmethod
    def _part(a: int, b: int, t0: int, t1: int, cu: List[int]) -> bool:
        """True for a piece that is part of one sequence, not the whole of it."""
        return b == a + 1 and (t0, t1) != (cu[a], cu[b])

    def run(self) -> None:
        if not self.use_graph or (self._graph is None and self._passes == 0):
            self._passes += 1
            self._issue()
            return
        if self._graph is None:
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize(self.device)
            with torch.cuda.graph(g):
                self._issue()
            self._graph = g
        self._passes += 1
        self._graph.replay()
        cur = torch.cuda.current_stream(self.device)
        self.done = torch.cuda.Event()
        self.done.record(cur)

    def _issue(self) -> None:
        """One pass, issued piece by piece on the three streams."""
        cu = self.cu
        cur = torch.cuda.current_stream(self.device)
        # the previous pass (and anything queued before it on the caller's stream) comes first
        for s in (self.s_in, self.s_run, self.s_out):
            s.wait_stream(cur)
        for i, (a, b, t0, t1) in enumerate(self.groups):
            first, last = t0 == cu[a], t1 == cu[b]  # both for runs of whole sequences
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(self.s_in):
                for n in ("q", "k", "v", "g", "beta"):
                    self.dev[n][t0:t1].copy_(self.host[n][t0:t1], non_blocking=True)
                self.dev_cu[i].copy_(self.host_cu[i], non_blocking=True)
                if self.dev_s0 is not None and first:
                    self.dev_s0[a:b].copy_(self.host_s0[a:b], non_blocking=True)
                ev_in.record(self.s_in)
            # a later part of a sequence starts from the carried state (updated in place)
            s0 = (None if self.dev_s0 is None else self.dev_s0[a:b]) if first else self.carry[a]
            s1 = self.final_state[a:b] if last else self.carry[a]
            ev_run = torch.cuda.Event()
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(ev_in)
                d = self.dev
                _kda.kda_chunk_fwd(d["q"][t0:t1], d["k"][t0:t1], d["v"][t0:t1], d["g"][t0:t1], d["beta"][t0:t1],
                                   cu_seqlens=self.dev_cu[i], init_state=s0, scale=self.scale, o=self.o[t0:t1],
                                   final_state=s1, workspace=self.workspaces[i], stream=self.s_run)
                ev_run.record(self.s_run)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_run)
                self.host_o[t0:t1].copy_(self.o[t0:t1], non_blocking=True)
                if last:
                    self.host_final_state[a:b].copy_(self.final_state[a:b], non_blocking=True)
        self.done = torch.cuda.Event()
        self.done.record(self.s_out)
        cur.wait_stream(self.s_out)
        cur.wait_stream(self.s_in)
        cur.wait_stream(self.s_run)

    def status(self) -> int:
        """Device status of the last pass: the first group's error, or KDA_OK (synchronizes)."""
        for ws in self.workspaces:
            st = _kda.kda_device_status(ws)
            if st != _kda.KDA_OK:
                return st
        return _kda.KDA_OK
