"""fp64 CPU oracle for the KDA forward, decode step and replay.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package.  It shares no code with the CUDA
library and never imports it.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by
token).  This module compiles it with gcc on first use, converts inputs to
float64 (an exact upcast of bf16/fp32 data) and exposes:

* ``forward``  -- packed varlen prefill: o and final state.
* ``decode``   -- one token per sequence on a slot-indexed state pool.
* ``replay``   -- accepted tokens re-applied to committed states (no output).
* ``conv``     -- the short causal convolution (+ SiLU) of the input projections,
  with the convolution state carried across calls.
* ``backward`` -- gradients of a loss with respect to every input, given its
  gradients with respect to o and the final states (reverse mode of the same
  token-by-token recurrence).

Decode and replay are the same recurrence as ``forward`` (the speculative-
decoding paragraph of "Kimi K3 on Fireworks: Fast RL at frontier scale" replays
the accepted tokens' update inputs from a committed checkpoint), so they are
written as calls of ``forward`` on the gathered states.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``_build/libkda_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64),
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_double, ctypes.c_int, dp, dp,
                                               ctypes.c_int]
            lib.kda_oracle_prep.restype = ctypes.c_int
            lib.kda_oracle_prep.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_double, ctypes.c_int]
            lib.kda_oracle_backward.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64),
                                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_double, ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, dp,
                                                ctypes.c_int]
            lib.kda_oracle_conv.restype = ctypes.c_int
            lib.kda_oracle_conv.argtypes = [dp, dp, dp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, dp, dp]
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


PREP_L2NORM_Q, PREP_L2NORM_K, PREP_SIGMOID_GATE, PREP_SIGMOID_BETA = 1, 2, 4, 8


def prep(q, k, g, beta, flags: int, eps: float = 1e-6):
    """fp64 copies of the inputs with the preprocessing of ``flags`` applied
    (kda_oracle_prep: L2 normalisation of q / k rows, alpha = sigmoid(x_g),
    beta = sigmoid(x_beta)).  q may be None when flags has no PREP_L2NORM_Q."""
    lib = _load()
    k64, g64, b64 = _f64(k).copy(), _f64(g).copy(), _f64(beta).copy()
    q64 = None if q is None else _f64(q).copy()
    T, H, dk = k64.shape
    rc = lib.kda_oracle_prep(_ptr(q64), _ptr(k64), _ptr(g64), _ptr(b64), T, H, dk, float(eps), int(flags))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_prep failed with code {rc}")
    return q64, k64, g64, b64


def forward(q, k, v, g, beta, cu_seqlens, init_state=None, scale: float = 1.0,
            gate_is_alpha: bool = False, want_o: bool = True, threads: int = 1, prep_flags: int = 0,
            prep_eps: float = 1e-6):
    """Packed variable-length KDA forward in fp64.

    Shapes: q, k, g [T, H, dk]; v [T, H, dv]; beta [T, H]; cu_seqlens [N+1];
    init_state [N, H, dk, dv] or None.  Returns ``(o, final_state)`` as float64
    numpy arrays (``o`` is None when ``want_o`` is False).  ``prep_flags`` applies
    the input preprocessing first (see ``prep``); with PREP_SIGMOID_GATE, g holds
    the raw gate x and alpha = sigmoid(x).
    """
    if prep_flags:
        q, k, g, beta = prep(q if want_o else None, k, g, beta, prep_flags, prep_eps)
        gate_is_alpha = bool(prep_flags & PREP_SIGMOID_GATE) or gate_is_alpha
    lib = _load()
    k64, v64, g64, b64 = _f64(k), _f64(v), _f64(g), _f64(beta)
    q64 = _f64(q) if want_o else None
    cu = np.ascontiguousarray(np.asarray(_f64(cu_seqlens), dtype=np.int64))
    T, H, dk = k64.shape
    dv = v64.shape[2]
    N = cu.shape[0] - 1
    s0 = _f64(init_state)
    if s0 is not None and s0.shape != (N, H, dk, dv):
        raise ValueError(f"init_state shape {s0.shape} != {(N, H, dk, dv)}")
    o = np.zeros((T, H, dv), dtype=np.float64) if want_o else None
    fs = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = lib.kda_oracle_forward(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(b64), _ptr(s0),
                                cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk, dv,
                                float(scale), int(bool(gate_is_alpha)), _ptr(o), _ptr(fs),
                                int(threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_forward failed with code {rc}")
    return o, fs


def decode(q, k, v, g, beta, state_pool, slots=None, scale: float = 1.0, threads: int = 1, prep_flags: int = 0,
           prep_eps: float = 1e-6):
    """One decode step per sequence on a slot-indexed pool.

    q, k, g [N, H, dk]; v [N, H, dv]; beta [N, H]; state_pool [S, H, dk, dv];
    slots [N] (None: sequence n uses slot n).  Returns ``(o, new_pool)``.
    """
    pool = _f64(state_pool).copy()
    N = np.asarray(_f64(k)).shape[0]
    sl = np.arange(N) if slots is None else np.asarray(_f64(slots), dtype=np.int64)
    cu = np.arange(N + 1, dtype=np.int64)
    o, fs = forward(q, k, v, g, beta, cu, pool[sl], scale=scale, threads=threads, prep_flags=prep_flags,
                    prep_eps=prep_eps)
    pool[sl] = fs
    return o, pool


def replay(k, v, g, beta, cu_accept, state_pool, slots=None, threads: int = 1, prep_flags: int = 0,
           prep_eps: float = 1e-6):
    """Apply each sequence's accepted tokens to its committed state in the pool.

    k, g [A, H, dk]; v [A, H, dv]; beta [A, H]; cu_accept [N+1].  Returns the
    new pool.
    """
    pool = _f64(state_pool).copy()
    cu = np.asarray(_f64(cu_accept), dtype=np.int64)
    N = cu.shape[0] - 1
    sl = np.arange(N) if slots is None else np.asarray(_f64(slots), dtype=np.int64)
    _, fs = forward(None, k, v, g, beta, cu, pool[sl], want_o=False, threads=threads,
                    prep_flags=prep_flags & ~PREP_L2NORM_Q, prep_eps=prep_eps)
    pool[sl] = fs
    return pool


def backward(q, k, v, g, beta, cu_seqlens, init_state, d_o, d_final=None, scale: float = 1.0,
             gate_is_alpha: bool = False, threads: int = 1, prep_flags: int = 0, prep_eps: float = 1e-6):
    """Reverse mode of ``forward`` in fp64 (kda_oracle_backward).

    Given dL/do [T, H, dv] and dL/d(final_state) [N, H, dk, dv] (None = 0), returns a
    dict of float64 arrays: dq, dk, dg [T, H, dk] (dg with respect to the log-gates,
    or to alpha with ``gate_is_alpha``), dv [T, H, dv], dbeta [T, H] and d_init
    [N, H, dk, dv].  With ``prep_flags`` the inputs are raw (see ``prep``) and the
    gradients are taken with respect to them: the recurrence's gradients are carried
    back through the L2 normalisation (dx = r (dxn - xn (xn . dxn)), r = (sum x^2 +
    eps)^-1/2, xn = r x), alpha = sigmoid(x_g) (dx = dalpha alpha (1 - alpha)) and
    beta = sigmoid(x_beta) (dx = dbeta beta (1 - beta)).
    """
    if prep_flags:
        qn, kn, gn, bn = prep(q, k, g, beta, prep_flags, prep_eps)
        sig_gate = bool(prep_flags & PREP_SIGMOID_GATE)
        G = backward(qn, kn, v, gn, bn, cu_seqlens, init_state, d_o, d_final, scale=scale,
                     gate_is_alpha=sig_gate or gate_is_alpha, threads=threads)
        for flag, name, raw, xn in ((PREP_L2NORM_Q, "dq", q, qn), (PREP_L2NORM_K, "dk", k, kn)):
            if prep_flags & flag:
                x = _f64(raw)
                r = 1.0 / np.sqrt((x * x).sum(-1, keepdims=True) + prep_eps)
                dxn = G[name]
                G[name] = r * (dxn - xn * (xn * dxn).sum(-1, keepdims=True))
        if sig_gate:
            G["dg"] = G["dg"] * gn * (1.0 - gn)
        if prep_flags & PREP_SIGMOID_BETA:
            G["dbeta"] = G["dbeta"] * bn * (1.0 - bn)
        return G
    lib = _load()
    q64, k64, v64, g64, b64 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    cu = np.ascontiguousarray(np.asarray(_f64(cu_seqlens), dtype=np.int64))
    T, H, dk = k64.shape
    dv = v64.shape[2]
    N = cu.shape[0] - 1
    s0, do64, df64 = _f64(init_state), _f64(d_o), _f64(d_final)
    out = {"dq": np.zeros((T, H, dk)), "dk": np.zeros((T, H, dk)), "dv": np.zeros((T, H, dv)),
           "dg": np.zeros((T, H, dk)), "dbeta": np.zeros((T, H)), "d_init": np.zeros((N, H, dk, dv))}
    rc = lib.kda_oracle_backward(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(b64), _ptr(s0),
                                 cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk, dv, float(scale),
                                 int(bool(gate_is_alpha)), _ptr(do64), _ptr(df64), _ptr(out["dq"]),
                                 _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                                 _ptr(out["d_init"]), int(threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_backward failed with code {rc}")
    return out


def conv(x, w, cu_seqlens, state_in=None):
    """Short causal depthwise convolution + SiLU (kda_oracle_conv).

    x [T, H, C]; w [H, C, W]; state_in [N, W-1, H, C] (previous inputs, oldest first) or
    None.  Returns ``(y [T, H, C], state_out [N, W-1, H, C])`` as float64 arrays."""
    lib = _load()
    x64, w64, s64 = _f64(x), _f64(w), _f64(state_in)
    cu = np.ascontiguousarray(np.asarray(_f64(cu_seqlens), dtype=np.int64))
    T, H, C = x64.shape
    W = w64.shape[2]
    N = cu.shape[0] - 1
    y = np.zeros((T, H, C))
    so = np.zeros((N, max(W - 1, 0), H, C))
    rc = lib.kda_oracle_conv(_ptr(x64), _ptr(w64), _ptr(s64), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                             N, H, C, W, _ptr(y), _ptr(so) if W > 1 else None)
    if rc != 0:
        raise RuntimeError(f"kda_oracle_conv failed with code {rc}")
    return y, so
