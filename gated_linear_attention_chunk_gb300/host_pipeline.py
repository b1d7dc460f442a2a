"""Prefill from pinned host memory with the copies overlapped (plumbing, no arithmetic).

``HostPrefill`` runs ``kda_chunk_fwd`` over a packed batch whose inputs live in
pinned host memory and whose outputs go back to pinned host memory.  The batch
is cut into groups of whole sequences.  Group i's inputs travel host -> device
on one stream while group i-1 computes on a second stream and group i-2's
outputs travel device -> host on a third, so the host link, the kernels and the
return copies work at the same time instead of one after the other.  Every
group is an ordinary ``kda_chunk_fwd`` call on a contiguous token range (the
packed layout keeps a sequence group's tokens contiguous), with the full
workspace of that call, so each group takes whatever path ``kda_chunk_fwd``
picks for its shape (a group of few chains may take the T-segment split) and
carries that call's accuracy.
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


class HostPrefill:
    """Pipelined host -> device -> host prefill of one packed batch.

    Inputs (CPU tensors, pinned or made pinned once here): q, k, g [T, H, dk], v [T, H, dv],
    beta [T, H], cu_seqlens [N + 1] int32, init_state [N, H, dk, dv] fp32 or None.
    ``groups`` is the number of sequence groups (at most N).  ``run()`` copies the inputs in,
    computes, and leaves o and final_state in the pinned host tensors ``host_o`` and
    ``host_final_state``; it returns once the last copy has been issued (synchronize the
    device, or ``self.done``, before reading them).
    """

    def __init__(self, q, k, v, g, beta, cu_seqlens, init_state=None, scale: float = 1.0,
                 groups: int = 4, device="cuda"):
        self.device = torch.device(device)
        self.host = {n: _pinned(x) for n, x in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}
        self.host_s0 = None if init_state is None else _pinned(init_state)
        cu = [int(x) for x in cu_seqlens.tolist()]
        N = len(cu) - 1
        T, H, dk = q.shape
        dv = v.shape[2]
        self.scale = float(scale)
        self.groups = plan_groups(cu, groups)
        # per-group cu_seqlens, rebased to the group's first token (host side, pinned)
        self.host_cu = [_pinned(torch.tensor([c - cu[a] for c in cu[a:b + 1]], dtype=torch.int32))
                        for a, b in self.groups]
        self.cu = cu
        dev = self.device
        self.dev = {n: torch.empty_like(x, device=dev) for n, x in self.host.items()}
        self.dev_cu = [torch.empty_like(c, device=dev) for c in self.host_cu]
        self.dev_s0 = None if self.host_s0 is None else torch.empty_like(self.host_s0, device=dev)
        self.o = torch.empty(T, H, dv, dtype=q.dtype, device=dev)
        self.final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
        self.host_o = torch.empty(T, H, dv, dtype=q.dtype).pin_memory()
        self.host_final_state = torch.empty(N, H, dk, dv, dtype=torch.float32).pin_memory()
        # one workspace per group, so that every group's device status survives the pass
        self.workspaces = [_kda.new_workspace(_kda.kda_chunk_fwd_workspace_size(b - a, cu[b] - cu[a], H, dk, dv),
                                              dev) for a, b in self.groups]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_run = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.done: Optional[torch.cuda.Event] = None
        self.h2d_bytes = sum(x.numel() * x.element_size() for x in self.host.values())
        self.h2d_bytes += sum(c.numel() * 4 for c in self.host_cu)
        if self.host_s0 is not None:
            self.h2d_bytes += self.host_s0.numel() * 4
        self.d2h_bytes = self.host_o.numel() * self.host_o.element_size() + self.host_final_state.numel() * 4

    def run(self) -> None:
        cu = self.cu
        cur = torch.cuda.current_stream(self.device)
        # the previous pass (and anything queued before it on the caller's stream) comes first
        for s in (self.s_in, self.s_run, self.s_out):
            s.wait_stream(cur)
        for i, (a, b) in enumerate(self.groups):
            t0, t1 = cu[a], cu[b]
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(self.s_in):
                for n in ("q", "k", "v", "g", "beta"):
                    self.dev[n][t0:t1].copy_(self.host[n][t0:t1], non_blocking=True)
                self.dev_cu[i].copy_(self.host_cu[i], non_blocking=True)
                if self.dev_s0 is not None:
                    self.dev_s0[a:b].copy_(self.host_s0[a:b], non_blocking=True)
                ev_in.record(self.s_in)
            ev_run = torch.cuda.Event()
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(ev_in)
                d = self.dev
                _kda.kda_chunk_fwd(d["q"][t0:t1], d["k"][t0:t1], d["v"][t0:t1], d["g"][t0:t1], d["beta"][t0:t1],
                                   cu_seqlens=self.dev_cu[i],
                                   init_state=None if self.dev_s0 is None else self.dev_s0[a:b],
                                   scale=self.scale, o=self.o[t0:t1], final_state=self.final_state[a:b],
                                   workspace=self.workspaces[i], stream=self.s_run)
                ev_run.record(self.s_run)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_run)
                self.host_o[t0:t1].copy_(self.o[t0:t1], non_blocking=True)
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
