"""Seeded synthetic inputs for the KDA forward (prefill, decode, replay).

This module only draws random inputs; it holds none of the recurrence's
arithmetic.  Both the fp64 oracle and the CUDA library consume the tensors it
returns, so the two sides always see the same bytes.

Input recipe (the KDA paragraph of "Kimi K3 on Fireworks: Fast RL at frontier
scale" gives no shapes or distributions; the recipe below is the one this
library standardises on):

* q, k, v ~ N(0, 1) drawn in fp32; k is L2-normalised per (token, head); q is
  multiplied by 1/sqrt(dk); then everything is rounded (RNE) to the storage
  dtype.
* g = logsigmoid(x), x ~ N(g_mu, 1) per channel (g_mu = 3, or 4 for the
  slow-decay long-context case), so alpha = exp(g) lies in (0, 1).
* beta = sigmoid(N(0, 1)), one scalar per (token, head).
* initial states ~ N(0, 0.02^2) in fp32 (or absent = zeros).
* draw order: lengths, q, k, v, x_g, x_beta, initial state.
* raw cases (``raw=True``, for the fused preprocessing): the same draws, but q
  and k are left un-normalised and unscaled, g holds x_g and beta holds x_beta
  (the library's preprocessing flags turn them into L2-normalised rows,
  alpha = sigmoid(x_g) and beta = sigmoid(x_beta)); the caller passes
  scale = 1/sqrt(dk).

All draws use a CPU ``torch.Generator`` seeded with the case seed, so the oracle
and the library see the same bytes.  ``device="cuda"`` draws the same recipe with
a CUDA generator seeded the same way (other bytes, same distributions): the
benchmark uses it for its large timing-only workloads, where no oracle compares.
Sequence lengths and accept lengths are always drawn on the CPU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

__all__ = ["KdaCase", "make_case", "NAMED_WORKLOADS", "named_case", "varlen_lengths",
           "make_decode_tokens", "make_accept_lengths"]


@dataclasses.dataclass
class KdaCase:
    """One packed variable-length KDA prefill problem (token-major layout)."""
    q: torch.Tensor            # [T_total, H, dk]
    k: torch.Tensor            # [T_total, H, dk]
    v: torch.Tensor            # [T_total, H, dv]
    g: torch.Tensor            # [T_total, H, dk]  log-gates (<= 0)
    beta: torch.Tensor         # [T_total, H]
    cu_seqlens: torch.Tensor   # [N + 1] int32
    init_state: Optional[torch.Tensor]  # [N, H, dk, dv] fp32 or None
    scale: float
    lengths: List[int]

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def T_total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def dk(self) -> int:
        return self.q.shape[2]

    @property
    def dv(self) -> int:
        return self.v.shape[2]

    def nbytes_inputs(self) -> int:
        n = sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v, self.g, self.beta))
        n += self.cu_seqlens.numel() * 4
        if self.init_state is not None:
            n += self.init_state.numel() * 4
        return n


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def varlen_lengths(n_seq: int, median: int, sigma: float, lo: int, hi: int, gen: torch.Generator) -> List[int]:
    """Log-normal lengths round(exp(N(ln median, sigma))) clipped to [lo, hi]."""
    z = torch.randn(n_seq, generator=gen, dtype=torch.float64)
    lens = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return [int(x) for x in lens.tolist()]


def _draw_tokens(T: int, H: int, dk: int, dv: int, dtype: torch.dtype, gen: torch.Generator,
                 g_mu: float, q_scale: bool = True, raw: bool = False):
    dev = gen.device
    q = torch.randn(T, H, dk, generator=gen, dtype=torch.float32, device=dev)
    k = torch.randn(T, H, dk, generator=gen, dtype=torch.float32, device=dev)
    v = torch.randn(T, H, dv, generator=gen, dtype=torch.float32, device=dev)
    xg = torch.randn(T, H, dk, generator=gen, dtype=torch.float32, device=dev) + g_mu
    xb = torch.randn(T, H, generator=gen, dtype=torch.float32, device=dev)
    if raw:
        return (q.to(dtype), k.to(dtype), v.to(dtype), xg.to(dtype), xb.to(dtype))
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    if q_scale:
        q = q * (1.0 / math.sqrt(dk))
    g = torch.nn.functional.logsigmoid(xg)
    beta = torch.sigmoid(xb)
    return (q.to(dtype), k.to(dtype), v.to(dtype), g.to(dtype), beta.to(dtype))


def make_case(lengths: List[int], H: int, dk: int, dv: int, dtype: torch.dtype = torch.bfloat16,
              seed: int = 0, init: bool = True, g_mu: float = 3.0, init_std: float = 0.02,
              q_scale: bool = True, scale: float = 1.0, raw: bool = False, device="cpu") -> KdaCase:
    """Packed varlen case with the given per-sequence lengths.

    ``q_scale`` folds 1/sqrt(dk) into q (then ``scale`` is normally 1.0);
    ``q_scale=False`` leaves q raw so the caller passes ``scale=1/sqrt(dk)``.
    ``raw`` returns the un-preprocessed draws (see the module docstring).
    ``device`` is where the draws are made and kept (see the module docstring).
    """
    gen = _gen(seed, device)
    T = int(sum(lengths))
    q, k, v, g, beta = _draw_tokens(T, H, dk, dv, dtype, gen, g_mu, q_scale, raw)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if lengths:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    cu = cu.to(device)
    s0 = None
    if init:
        s0 = (torch.randn(len(lengths), H, dk, dv, generator=gen, dtype=torch.float32, device=gen.device)
              * init_std)
    return KdaCase(q, k, v, g, beta, cu, s0, float(scale), list(lengths))


# Named workloads.  Sizes follow the 4K-128K-token range the KDA paragraph
# quotes its forward speedup over; every one is synthetic.
NAMED_WORKLOADS = {
    "tiny_fp32": dict(desc="B=1 T=256 H=2 dk=dv=64 fp32, zero initial state, seed 0",
                      lengths=[256], H=2, dk=64, dv=64, dtype="f32", init=False, g_mu=3.0, seed=0),
    "prefill_1k": dict(desc="B=4 T=1024 H=32 dk=dv=128 bf16, N(0,0.02) initial state (small profiling case,"
                            " inputs just above L2)",
                       lengths=[1024] * 4, H=32, dk=128, dv=128, dtype="bf16", init=True, g_mu=3.0, seed=5),
    "prefill_4k": dict(desc="B=4 T=4096 H=32 dk=dv=128 bf16, N(0,0.02) initial state",
                       lengths=[4096] * 4, H=32, dk=128, dv=128, dtype="bf16", init=True, g_mu=3.0, seed=1),
    "prefill_4k_d64": dict(desc="B=4 T=4096 H=32 dk=dv=64 bf16, N(0,0.02) initial state (config 1 with"
                                " 64-wide heads)",
                           lengths=[4096] * 4, H=32, dk=64, dv=64, dtype="bf16", init=True, g_mu=3.0, seed=6),
    "prefill_4k_fp32": dict(desc="B=4 T=4096 H=32 dk=dv=128 fp32, N(0,0.02) initial state (config 1 with fp32"
                                 " inputs: the token-sequential kernel)",
                            lengths=[4096] * 4, H=32, dk=128, dv=128, dtype="f32", init=True, g_mu=3.0, seed=7),
    "varlen_64": dict(desc="64 sequences, log-normal lengths (median 4096, sigma 0.5, clipped to"
                           " [1024, 20480]), H=32 dk=dv=128 bf16, random initial states",
                      lengths="lognormal", H=32, dk=128, dv=128, dtype="bf16", init=True, g_mu=3.0, seed=2),
    "long_128k": dict(desc="B=1 T=131072 H=32 dk=dv=128 bf16, slow decay g=logsigmoid(N(4,1)), zero state",
                      lengths=[131072], H=32, dk=128, dv=128, dtype="bf16", init=False, g_mu=4.0, seed=3),
    "spec_rollout": dict(desc="128 sequences: 2048-token prefill, then 64 x (4-token verify + replay of"
                              " U{1..4} accepted tokens), H=32 dk=dv=128 bf16",
                         lengths=[2048] * 128, H=32, dk=128, dv=128, dtype="bf16", init=False, g_mu=3.0,
                         seed=4),
}


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def named_case(name: str, lengths_override: Optional[List[int]] = None, raw: bool = False,
               device="cpu") -> KdaCase:
    """Build one of ``NAMED_WORKLOADS`` (the prefill part for ``spec_rollout``); ``raw``
    gives the same draws before preprocessing, with scale = 1/sqrt(dk); ``device`` as in
    ``make_case``."""
    w = NAMED_WORKLOADS[name]
    seed = w["seed"]
    if lengths_override is not None:
        lengths = list(lengths_override)
    elif w["lengths"] == "lognormal":
        lengths = varlen_lengths(64, 4096, 0.5, 1024, 20480, _gen(seed + 1000))
    else:
        lengths = list(w["lengths"])
    return make_case(lengths, w["H"], w["dk"], w["dv"], _torch_dtype(w["dtype"]), seed=seed,
                     init=w["init"], g_mu=w["g_mu"], q_scale=not raw, scale=w["dk"] ** -0.5 if raw else 1.0,
                     raw=raw, device=device)


def make_decode_tokens(n_tok: int, H: int, dk: int, dv: int, dtype: torch.dtype, seed: int,
                       g_mu: float = 3.0, raw: bool = False, device="cpu"):
    """Per-token inputs (q, k, v, g, beta) for ``n_tok`` decode/verify tokens."""
    return _draw_tokens(n_tok, H, dk, dv, dtype, _gen(seed, device), g_mu, True, raw)


def make_accept_lengths(n_steps: int, n_seq: int, max_accept: int, seed: int) -> torch.Tensor:
    """Accepted-token counts, uniform in {1..max_accept}, drawn up front: [n_steps, n_seq]."""
    return torch.randint(1, max_accept + 1, (n_steps, n_seq), generator=_gen(seed), dtype=torch.int32)
