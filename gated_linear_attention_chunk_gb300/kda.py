"""Python binding of libkda (ctypes).  Argument marshalling only.

Each function takes torch CUDA tensors, checks dtypes/shapes/contiguity,
allocates outputs the caller did not pass (torch is the device allocator and
stream provider), and calls the C entry point of the same name in
``_lib/libkda.so`` on the current CUDA stream.  All arithmetic runs in the CUDA
kernels; there is no fallback path: if the library is missing, importing the
binding raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkda.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "kda.h")

KDA_OK = 0
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_GATE_RANGE = 5
KDA_ERR_TIMEOUT = 6
KDA_ERR_BAD_SEQLENS = 7
KDA_ERR_BAD_SLOT = 8
KDA_BF16 = 0
KDA_F32 = 1
KDA_WS_HEADER_BYTES = 256
KDA_PREP_L2NORM_Q = 1
KDA_PREP_L2NORM_K = 2
KDA_PREP_SIGMOID_GATE = 4
KDA_PREP_SIGMOID_BETA = 8
KDA_CONV_WIDTH = 4

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_SIGS = {
    "kda_chunk_fwd_workspace_size": (ctypes.c_size_t, [_int, _i64, _int, _int, _int]),
    "kda_chunk_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int,
                             ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_decode_step": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _i64, _vp, _int, _int, _int, _int,
                               ctypes.c_float, _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_replay": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _int, _i64, _int, _int, _int,
                          _vp, ctypes.c_size_t, _vp]),
    "kda_chunk_fwd_prep": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int,
                                  ctypes.c_float, ctypes.c_uint32, ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t,
                                  _vp]),
    "kda_decode_step_prep": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _i64, _vp, _int, _int, _int, _int,
                                    ctypes.c_float, ctypes.c_uint32, ctypes.c_float, _vp, _vp, ctypes.c_size_t,
                                    _vp]),
    "kda_replay_prep": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _int, _i64, _int, _int, _int,
                               ctypes.c_uint32, ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
    "kda_chunk_bwd_workspace_size": (ctypes.c_size_t, [_int, _i64, _int, _int, _int]),
    "kda_chunk_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int, ctypes.c_float,
                             _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_conv_fwd": (_int, [_vp, _vp, _vp, _int, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int, _vp, _vp, _vp,
                            _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_decode_step_conv": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _i64, _vp, _int, _int, _int, _int,
                                    ctypes.c_float, _vp, _int, _vp, ctypes.c_uint32, ctypes.c_float, _vp, _vp,
                                    ctypes.c_size_t, _vp]),
    "kda_replay_conv": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _int, _vp, _int, _i64, _int, _int, _int,
                               _vp, _int, _vp, ctypes.c_uint32, ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
    "kda_chunk_bwd_prep": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int,
                                  ctypes.c_float, ctypes.c_uint32, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_device_status": (_int, [_vp, _vp]),
    "kda_status_string": (ctypes.c_char_p, [_int]),
    "kda_version": (_int, []),
    "kda_chunk_fwd_uses_tensor_cores": (_int, [_int, _int, _int]),
    "kda_chunk_fwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _int, _i64, _int, _int, _int,
                                     ctypes.c_float, _vp, _vp, ctypes.POINTER(ctypes.c_void_p), _vp]),
    "kda_state_fork": (_int, [_vp, _i64, _vp, _vp, _int, _int, _int, _int, _vp, ctypes.c_size_t, _vp]),
    "kda_state_offload": (_int, [_vp, _i64, _vp, _int, _int, _int, _int, _vp, _vp, ctypes.c_size_t, _vp]),
    "kda_state_restore": (_int, [_vp, _i64, _vp, _int, _int, _int, _int, _vp, _vp, ctypes.c_size_t, _vp]),
}

_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {kda_status_string(code)}")


def load_library():
    """Load ``libkda.so`` (raises ImportError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkda.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_functions():
    """Names of the functions declared in include/kda.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kda_[a-z_0-9]+)\s*\(", text, re.M)))


def kda_status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def kda_version() -> int:
    return int(load_library().kda_version())


def _check(code: int, where: str):
    if code != KDA_OK:
        raise KdaError(code, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kda_chunk_fwd_uses_tensor_cores(dk: int, dv: int, dtype) -> bool:
    """Whether kda_chunk_fwd runs full chunks on the tcgen05 kernel for this shape/dtype."""
    code = dtype if isinstance(dtype, int) else (KDA_BF16 if dtype == torch.bfloat16 else KDA_F32)
    return bool(load_library().kda_chunk_fwd_uses_tensor_cores(int(dk), int(dv), code))


def kda_chunk_fwd_workspace_size(N: int, T_total: int, H: int, dk: int, dv: int) -> int:
    return int(load_library().kda_chunk_fwd_workspace_size(N, T_total, H, dk, dv))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace buffer (uint8, 256-byte aligned by the caching allocator)."""
    return torch.empty(max(int(nbytes), KDA_WS_HEADER_BYTES), dtype=torch.uint8, device=device)


def kda_chunk_fwd(q, k, v, g, beta, cu_seqlens=None, init_state=None, scale: float = 1.0,
                  output_final_state: bool = True, o=None, final_state=None, workspace=None,
                  stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Packed varlen KDA prefill.  Returns ``(o, final_state)``.

    q, k, g [T, H, dk]; v [T, H, dv]; beta [T, H] (bf16 or fp32, one dtype);
    cu_seqlens [N+1] int32 CUDA (None: one sequence of length T);
    init_state [N, H, dk, dv] fp32 or None.  ``final_state`` may be passed (and
    may be ``init_state`` itself for an in-place update).
    """
    return _chunk_fwd(q, k, v, g, beta, cu_seqlens, init_state, scale, output_final_state, o, final_state,
                      workspace, stream, None, 0.0)


def kda_chunk_fwd_prep(q, k, v, g, beta, prep: int, l2_eps: float = 1e-6, cu_seqlens=None, init_state=None,
                       scale: float = 1.0, output_final_state: bool = True, o=None, final_state=None,
                       workspace=None, stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """kda_chunk_fwd on raw inputs: ``prep`` is a set of KDA_PREP_* flags (L2-normalised
    q / k rows with ``l2_eps``, g as raw gates with alpha = sigmoid(g), beta <- sigmoid(beta)),
    applied inside the kernels."""
    return _chunk_fwd(q, k, v, g, beta, cu_seqlens, init_state, scale, output_final_state, o, final_state,
                      workspace, stream, int(prep), float(l2_eps))


def _chunk_fwd(q, k, v, g, beta, cu_seqlens, init_state, scale, output_final_state, o, final_state, workspace,
               stream, prep, l2_eps):
    lib = load_library()
    dt = q.dtype
    T, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv)),
                         ("g", g, (T, H, dk)), ("beta", beta, (T, H))):
        _need(t, name, dt, shp)
    if cu_seqlens is None:
        N = 1
    else:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, (N, H, dk, dv))
    if o is None:
        o = torch.empty(T, H, dv, dtype=dt, device=q.device)
    _need(o, "o", dt, (T, H, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, dk, dv))
    need = kda_chunk_fwd_workspace_size(N, T, H, dk, dv)  # the size that enables every path
    if workspace is None:
        workspace = new_workspace(need, q.device)
    common = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype_code(q), _ptr(init_state),
              _ptr(cu_seqlens), N, T, H, dk, dv, float(scale))
    tail = (_ptr(o), _ptr(final_state), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    if prep is None:
        _check(lib.kda_chunk_fwd(*common, *tail), "kda_chunk_fwd")
    else:
        _check(lib.kda_chunk_fwd_prep(*common, prep, l2_eps, *tail), "kda_chunk_fwd_prep")
    return o, final_state


def kda_chunk_fwd_noalloc(q, k, v, g, beta, o, cu_seqlens=None, init_state=None, final_state=None,
                          scale: float = 1.0, stream=None) -> int:
    """kda_chunk_fwd without a workspace: the library's fixed device scratch is used
    instead, for callers that cannot allocate.  ``o`` (and ``final_state`` when wanted)
    must be passed in.  Returns the scratch's device address, which
    ``kda_device_status`` accepts."""
    lib = load_library()
    dt = q.dtype
    T, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv)),
                         ("g", g, (T, H, dk)), ("beta", beta, (T, H)), ("o", o, (T, H, dv))):
        _need(t, name, dt, shp)
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, (N, H, dk, dv))
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, dk, dv))
    ws = ctypes.c_void_p()
    # the library's scratch and the default stream are those of the current device
    with torch.cuda.device(q.device):
        rc = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype_code(q),
                                       _ptr(init_state), _ptr(cu_seqlens), N, T, H, dk, dv, float(scale), _ptr(o),
                                       _ptr(final_state), ctypes.byref(ws), _stream_handle(stream))
    _check(rc, "kda_chunk_fwd_noalloc")
    return int(ws.value)


def kda_decode_step(q, k, v, g, beta, state_pool, slots=None, scale: float = 1.0, o=None, workspace=None,
                    stream=None) -> torch.Tensor:
    """One token per sequence; updates ``state_pool`` [S, H, dk, dv] in place.  Returns o [N, H, dv]."""
    return _decode_step(q, k, v, g, beta, state_pool, slots, scale, o, workspace, stream, None, 0.0)


def kda_decode_step_prep(q, k, v, g, beta, state_pool, prep: int, l2_eps: float = 1e-6, slots=None,
                         scale: float = 1.0, o=None, workspace=None, stream=None) -> torch.Tensor:
    """kda_decode_step on raw inputs (KDA_PREP_* flags, see kda_chunk_fwd_prep)."""
    return _decode_step(q, k, v, g, beta, state_pool, slots, scale, o, workspace, stream, int(prep),
                        float(l2_eps))


def _decode_step(q, k, v, g, beta, state_pool, slots, scale, o, workspace, stream, prep, l2_eps):
    lib = load_library()
    dt = q.dtype
    N, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("v", v, (N, H, dv)),
                         ("g", g, (N, H, dk)), ("beta", beta, (N, H))):
        _need(t, name, dt, shp)
    _need(state_pool, "state_pool", torch.float32)
    if tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [S, {H}, {dk}, {dv}]")
    if slots is not None:
        _need(slots, "slots", torch.int32, (N,))
    if o is None:
        o = torch.empty(N, H, dv, dtype=dt, device=q.device)
    _need(o, "o", dt, (N, H, dv))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, q.device)
    common = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype_code(q), _ptr(state_pool),
              state_pool.shape[0], _ptr(slots), N, H, dk, dv, float(scale))
    tail = (_ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if prep is None:
        _check(lib.kda_decode_step(*common, *tail), "kda_decode_step")
    else:
        _check(lib.kda_decode_step_prep(*common, prep, l2_eps, *tail), "kda_decode_step_prep")
    return o


def kda_replay(state_pool, k, v, g, beta, cu_accept, slots=None, workspace=None, stream=None) -> None:
    """Apply accepted tokens [A, H, .] to the pool states in place (cu_accept [N+1] int32)."""
    _replay(state_pool, k, v, g, beta, cu_accept, slots, workspace, stream, None, 0.0)


def kda_replay_prep(state_pool, k, v, g, beta, cu_accept, prep: int, l2_eps: float = 1e-6, slots=None,
                    workspace=None, stream=None) -> None:
    """kda_replay on raw inputs (KDA_PREP_* flags; KDA_PREP_L2NORM_Q has no effect)."""
    _replay(state_pool, k, v, g, beta, cu_accept, slots, workspace, stream, int(prep), float(l2_eps))


def _replay(state_pool, k, v, g, beta, cu_accept, slots, workspace, stream, prep, l2_eps):
    lib = load_library()
    dt = k.dtype
    A, H, dk = k.shape
    dv = v.shape[2]
    for name, t, shp in (("k", k, (A, H, dk)), ("v", v, (A, H, dv)), ("g", g, (A, H, dk)),
                         ("beta", beta, (A, H))):
        _need(t, name, dt, shp)
    _need(cu_accept, "cu_accept", torch.int32)
    N = cu_accept.numel() - 1
    _need(state_pool, "state_pool", torch.float32)
    if tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [S, {H}, {dk}, {dv}]")
    if slots is not None:
        _need(slots, "slots", torch.int32, (N,))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, k.device)
    common = (_ptr(state_pool), state_pool.shape[0], _ptr(slots), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
              _dtype_code(k), _ptr(cu_accept), N, A, H, dk, dv)
    tail = (_ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if prep is None:
        _check(lib.kda_replay(*common, *tail), "kda_replay")
    else:
        _check(lib.kda_replay_prep(*common, prep, l2_eps, *tail), "kda_replay_prep")


def kda_chunk_bwd_workspace_size(N: int, T_total: int, H: int, dk: int, dv: int) -> int:
    return int(load_library().kda_chunk_bwd_workspace_size(N, T_total, H, dk, dv))


def kda_chunk_bwd(q, k, v, g, beta, d_o, cu_seqlens=None, init_state=None, d_final_state=None,
                  scale: float = 1.0, want_d_init: bool = True, workspace=None, stream=None) -> dict:
    """Backward of kda_chunk_fwd: returns a dict with dq, dk, dg [T, H, dk], dv [T, H, dv],
    dbeta [T, H] (input dtype) and d_init [N, H, dk, dv] fp32 (None unless ``want_d_init``),
    given d_o [T, H, dv] and d_final_state [N, H, dk, dv] fp32 (None = zero)."""
    return _chunk_bwd(q, k, v, g, beta, d_o, cu_seqlens, init_state, d_final_state, scale, want_d_init,
                      workspace, stream, None, 0.0)


def kda_chunk_bwd_prep(q, k, v, g, beta, d_o, prep: int, l2_eps: float = 1e-6, cu_seqlens=None, init_state=None,
                       d_final_state=None, scale: float = 1.0, want_d_init: bool = True, workspace=None,
                       stream=None) -> dict:
    """kda_chunk_bwd for a forward taken with kda_chunk_fwd_prep (raw inputs, same flags):
    the gradients are with respect to the raw inputs."""
    return _chunk_bwd(q, k, v, g, beta, d_o, cu_seqlens, init_state, d_final_state, scale, want_d_init,
                      workspace, stream, int(prep), float(l2_eps))


def _chunk_bwd(q, k, v, g, beta, d_o, cu_seqlens, init_state, d_final_state, scale, want_d_init, workspace,
               stream, prep, l2_eps):
    lib = load_library()
    dt = q.dtype
    T, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv)),
                         ("g", g, (T, H, dk)), ("beta", beta, (T, H)), ("d_o", d_o, (T, H, dv))):
        _need(t, name, dt, shp)
    if cu_seqlens is None:
        N = 1
    else:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, (N, H, dk, dv))
    if d_final_state is not None:
        _need(d_final_state, "d_final_state", torch.float32, (N, H, dk, dv))
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
           "dg": torch.empty_like(g), "dbeta": torch.empty_like(beta),
           "d_init": torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device) if want_d_init else None}
    need = kda_chunk_bwd_workspace_size(N, T, H, dk, dv)
    if workspace is None:
        workspace = new_workspace(need, q.device)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype_code(q), _ptr(init_state), _ptr(cu_seqlens), N,
            T, H, dk, dv, float(scale))
    tail = (_ptr(d_o), _ptr(d_final_state), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
            _ptr(out["dbeta"]), _ptr(out["d_init"]), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    if prep is None:
        _check(lib.kda_chunk_bwd(*head, *tail), "kda_chunk_bwd")
    else:
        _check(lib.kda_chunk_bwd_prep(*head, prep, l2_eps, *tail), "kda_chunk_bwd_prep")
    return out


def _conv_check(conv_weight, H, dk, dv):
    _need(conv_weight, "conv_weight", torch.float32, (H, 2 * dk + dv, KDA_CONV_WIDTH))


def kda_conv_fwd(q, k, v, conv_weight, cu_seqlens=None, conv_state_in=None, conv_state_out=None,
                 want_state: bool = True, workspace=None, stream=None):
    """Short causal convolution (width 4) + SiLU of the raw projections q, k, v [T, H, d].
    conv_weight [H, 2dk+dv, 4] fp32 (channels q | k | v); conv_state_in / out [N, 3, H, 2dk+dv]
    fp32.  Returns ``(q_out, k_out, v_out, conv_state_out)``."""
    lib = load_library()
    dt = q.dtype
    T, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("v", v, (T, H, dv))):
        _need(t, name, dt, shp)
    _conv_check(conv_weight, H, dk, dv)
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
    cs = (N, KDA_CONV_WIDTH - 1, H, 2 * dk + dv)
    if conv_state_in is not None:
        _need(conv_state_in, "conv_state_in", torch.float32, cs)
    if conv_state_out is None and want_state:
        conv_state_out = torch.empty(cs, dtype=torch.float32, device=q.device)
    if conv_state_out is not None:
        _need(conv_state_out, "conv_state_out", torch.float32, cs)
    qo, ko, vo = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, q.device)
    rc = lib.kda_conv_fwd(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(conv_weight), KDA_CONV_WIDTH,
                          _ptr(conv_state_in), _ptr(cu_seqlens), N, T, H, dk, dv, _ptr(qo), _ptr(ko), _ptr(vo),
                          _ptr(conv_state_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream_handle(stream))
    _check(rc, "kda_conv_fwd")
    return qo, ko, vo, conv_state_out


def kda_decode_step_conv(q, k, v, g, beta, state_pool, conv_weight, conv_pool, prep: int = 0,
                         l2_eps: float = 1e-6, slots=None, scale: float = 1.0, o=None, workspace=None,
                         stream=None) -> torch.Tensor:
    """kda_decode_step on raw projections with the short convolution fused (conv_pool
    [S, 3, H, 2dk+dv] fp32, advanced in place) and optional KDA_PREP_* flags."""
    lib = load_library()
    dt = q.dtype
    N, H, dk = q.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("v", v, (N, H, dv)),
                         ("g", g, (N, H, dk)), ("beta", beta, (N, H))):
        _need(t, name, dt, shp)
    _need(state_pool, "state_pool", torch.float32)
    if tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [S, {H}, {dk}, {dv}]")
    _conv_check(conv_weight, H, dk, dv)
    _need(conv_pool, "conv_pool", torch.float32, (state_pool.shape[0], KDA_CONV_WIDTH - 1, H, 2 * dk + dv))
    if slots is not None:
        _need(slots, "slots", torch.int32, (N,))
    if o is None:
        o = torch.empty(N, H, dv, dtype=dt, device=q.device)
    _need(o, "o", dt, (N, H, dv))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, q.device)
    rc = lib.kda_decode_step_conv(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dtype_code(q), _ptr(state_pool),
                                  state_pool.shape[0], _ptr(slots), N, H, dk, dv, float(scale), _ptr(conv_weight),
                                  KDA_CONV_WIDTH, _ptr(conv_pool), int(prep), float(l2_eps), _ptr(o),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    _check(rc, "kda_decode_step_conv")
    return o


def kda_replay_conv(state_pool, q, k, v, g, beta, cu_accept, conv_weight, conv_pool, prep: int = 0,
                    l2_eps: float = 1e-6, slots=None, workspace=None, stream=None) -> None:
    """kda_replay on raw projections with the short convolution fused: the accepted
    tokens' q, k, v advance conv_pool and their convolved k, v the recurrent states."""
    lib = load_library()
    dt = k.dtype
    A, H, dk = k.shape
    dv = v.shape[2]
    for name, t, shp in (("q", q, (A, H, dk)), ("k", k, (A, H, dk)), ("v", v, (A, H, dv)),
                         ("g", g, (A, H, dk)), ("beta", beta, (A, H))):
        _need(t, name, dt, shp)
    _need(cu_accept, "cu_accept", torch.int32)
    N = cu_accept.numel() - 1
    _need(state_pool, "state_pool", torch.float32)
    if tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state_pool shape {tuple(state_pool.shape)} != [S, {H}, {dk}, {dv}]")
    _conv_check(conv_weight, H, dk, dv)
    _need(conv_pool, "conv_pool", torch.float32, (state_pool.shape[0], KDA_CONV_WIDTH - 1, H, 2 * dk + dv))
    if slots is not None:
        _need(slots, "slots", torch.int32, (N,))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, k.device)
    rc = lib.kda_replay_conv(_ptr(state_pool), state_pool.shape[0], _ptr(slots), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(beta), _dtype_code(k), _ptr(cu_accept), N, A, H, dk, dv, _ptr(conv_weight),
                             KDA_CONV_WIDTH, _ptr(conv_pool), int(prep), float(l2_eps), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "kda_replay_conv")


def _pool_shape(state_pool):
    _need(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4:
        raise ValueError(f"state_pool must be [S, H, dk, dv], got {tuple(state_pool.shape)}")
    S, H, dk, dv = state_pool.shape
    return S, H, dk, dv


def kda_state_fork(state_pool, src_slots, dst_slots, workspace=None, stream=None) -> None:
    """state_pool[dst_slots[i]] = state_pool[src_slots[i]] (int32 CUDA slot arrays), bit for bit."""
    lib = load_library()
    S, H, dk, dv = _pool_shape(state_pool)
    n = src_slots.numel()
    _need(src_slots, "src_slots", torch.int32, (n,))
    _need(dst_slots, "dst_slots", torch.int32, (n,))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, state_pool.device)
    rc = lib.kda_state_fork(_ptr(state_pool), S, _ptr(src_slots), _ptr(dst_slots), n, H, dk, dv, _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "kda_state_fork")


def kda_state_offload(state_pool, slots, host_states, workspace=None, stream=None) -> None:
    """host_states[i] = state_pool[slots[i]]; host_states is a pinned CPU fp32 tensor [n, H, dk, dv]
    (slots None: slot i).  Asynchronous: synchronize the stream before reading host_states."""
    lib = load_library()
    S, H, dk, dv = _pool_shape(state_pool)
    if host_states.device.type != "cpu" or not host_states.is_pinned() or not host_states.is_contiguous():
        raise ValueError("host_states must be a contiguous pinned CPU tensor")
    n = host_states.shape[0]
    if tuple(host_states.shape) != (n, H, dk, dv) or host_states.dtype != torch.float32:
        raise ValueError(f"host_states must be float32 [n, {H}, {dk}, {dv}]")
    if slots is not None:
        _need(slots, "slots", torch.int32, (n,))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, state_pool.device)
    rc = lib.kda_state_offload(_ptr(state_pool), S, _ptr(slots), n, H, dk, dv, host_states.data_ptr(),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "kda_state_offload")


def kda_state_restore(state_pool, slots, host_states, workspace=None, stream=None) -> None:
    """state_pool[slots[i]] = host_states[i]; host_states a pinned CPU fp32 tensor [n, H, dk, dv]."""
    lib = load_library()
    S, H, dk, dv = _pool_shape(state_pool)
    if host_states.device.type != "cpu" or not host_states.is_pinned() or not host_states.is_contiguous():
        raise ValueError("host_states must be a contiguous pinned CPU tensor")
    n = host_states.shape[0]
    if tuple(host_states.shape) != (n, H, dk, dv) or host_states.dtype != torch.float32:
        raise ValueError(f"host_states must be float32 [n, {H}, {dk}, {dv}]")
    if slots is not None:
        _need(slots, "slots", torch.int32, (n,))
    if workspace is None:
        workspace = new_workspace(KDA_WS_HEADER_BYTES, state_pool.device)
    rc = lib.kda_state_restore(_ptr(state_pool), S, _ptr(slots), n, H, dk, dv, host_states.data_ptr(),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "kda_state_restore")


def kda_device_status(workspace, stream=None) -> int:
    """Synchronize the stream and return the device status code of the last call on ``workspace``
    (a tensor, or a raw device address such as the one kda_chunk_fwd_noalloc returns)."""
    ptr = ctypes.c_void_p(workspace) if isinstance(workspace, int) else _ptr(workspace)
    return int(load_library().kda_device_status(ptr, _stream_handle(stream)))
