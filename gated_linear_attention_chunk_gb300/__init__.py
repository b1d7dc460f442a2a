"""libkda: Kimi Delta Attention forward (prefill, decode, replay, state-pool ops) on GB300.

The compute path is the CUDA library ``_lib/libkda.so`` (C ABI, declared in
``include/kda.h``); this package is its ctypes binding.  Importing the package
loads the library and raises ImportError if it has not been built (run
``__graft_entry__.build()`` or ``python gated_linear_attention_chunk_gb300/build.py``).
"""
from .kda import (KDA_BF16, KDA_ERR_BAD_SEQLENS, KDA_ERR_BAD_SLOT, KDA_ERR_CUDA, KDA_ERR_GATE_RANGE,
                  KDA_ERR_INVALID_ARGUMENT, KDA_ERR_TIMEOUT, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_F32,
                  KDA_CONV_WIDTH, KDA_OK, KDA_PREP_L2NORM_K, KDA_PREP_L2NORM_Q, KDA_PREP_SIGMOID_BETA, KDA_PREP_SIGMOID_GATE,
                  KDA_WS_HEADER_BYTES, KdaError, kda_chunk_bwd, kda_chunk_bwd_prep, kda_chunk_bwd_workspace_size, kda_chunk_fwd,
                  kda_chunk_fwd_noalloc, kda_chunk_fwd_prep,
                  kda_chunk_fwd_uses_tensor_cores, kda_chunk_fwd_workspace_size, kda_conv_fwd, kda_decode_step, kda_decode_step_conv,
                  kda_decode_step_prep, kda_device_status, kda_replay, kda_replay_conv, kda_replay_prep, kda_state_fork,
                  kda_state_offload, kda_state_restore, kda_status_string, kda_version, load_library,
                  new_workspace)

load_library()

__all__ = [
    "kda_chunk_fwd", "kda_chunk_bwd", "kda_chunk_bwd_prep", "kda_chunk_bwd_workspace_size", "kda_chunk_fwd_prep", "kda_chunk_fwd_noalloc", "kda_chunk_fwd_workspace_size",
    "kda_chunk_fwd_uses_tensor_cores", "kda_decode_step", "kda_decode_step_prep", "kda_replay", "kda_replay_prep",
    "kda_conv_fwd", "kda_decode_step_conv", "kda_replay_conv", "KDA_CONV_WIDTH",
    "kda_state_fork", "kda_state_offload", "kda_state_restore", "kda_device_status", "kda_status_string",
    "kda_version", "new_workspace", "KdaError", "KDA_OK", "KDA_BF16", "KDA_F32", "KDA_WS_HEADER_BYTES",
    "KDA_PREP_L2NORM_Q", "KDA_PREP_L2NORM_K", "KDA_PREP_SIGMOID_GATE", "KDA_PREP_SIGMOID_BETA",
    "KDA_ERR_INVALID_ARGUMENT", "KDA_ERR_UNSUPPORTED", "KDA_ERR_WORKSPACE", "KDA_ERR_CUDA", "KDA_ERR_GATE_RANGE",
    "KDA_ERR_TIMEOUT", "KDA_ERR_BAD_SEQLENS", "KDA_ERR_BAD_SLOT",
]
