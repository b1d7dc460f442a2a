"""The C-ABI library: it loads without a GPU, exports every declared symbol, and
rejects bad arguments on the host (before any CUDA call)."""
import ctypes

import pytest

from tests._helpers import ensure_built


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from gated_linear_attention_chunk_gb300 import kda
    return kda.load_library()


def test_exports_every_declared_symbol(lib):
    from gated_linear_attention_chunk_gb300 import kda
    names = kda.header_functions()
    assert {"kda_chunk_fwd", "kda_decode_step", "kda_replay", "kda_device_status",
            "kda_chunk_fwd_workspace_size", "kda_status_string", "kda_version", "kda_chunk_fwd_prep",
            "kda_decode_step_prep", "kda_replay_prep", "kda_state_fork", "kda_state_offload",
            "kda_state_restore", "kda_chunk_fwd_noalloc", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size", "kda_conv_fwd", "kda_decode_step_conv",
            "kda_replay_conv"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    from gated_linear_attention_chunk_gb300 import kda
    assert kda.kda_status_string(0) == "KDA_OK"
    assert kda.kda_status_string(7) == "KDA_ERR_BAD_SEQLENS"
    assert kda.kda_status_string(99) == "KDA_ERR_UNKNOWN"
    assert kda.kda_version() >= 10000


def test_workspace_size(lib):
    from gated_linear_attention_chunk_gb300 import kda
    fb = lambda N, H: (N * H + 15) // 16 * 16  # strong-decay fallback flags, one byte per chain
    assert kda.kda_chunk_fwd_workspace_size(4, 16384, 32, 128, 128) == 256 + 4 * 32 * 128 * 128 * 4 + fb(4, 32)
    # few chains and long sequences: room for the T-segment split (three state sets + bf16 outputs)
    assert kda.kda_chunk_fwd_workspace_size(1, 131072, 32, 128, 128) == \
        256 + 3 * 32 * 65536 + 131072 * 32 * 256 + fb(1, 32)
    assert kda.kda_chunk_fwd_workspace_size(6, 4096, 8, 128, 128) == 256 + 3 * 48 * 65536 + 4096 * 8 * 256 + fb(6, 8)
    assert kda.kda_chunk_fwd_workspace_size(7, 4096, 7, 128, 128) == 256 + 49 * 65536 + fb(7, 7)  # 49 chains: no split
    assert kda.kda_chunk_fwd_workspace_size(1, 4095, 2, 128, 128) == 256 + 2 * 65536 + fb(1, 2)  # too short: no split
    assert kda.kda_chunk_fwd_workspace_size(1, 8192, 2, 64, 64) == 256 + 2 * 16384 + fb(1, 2)  # d = 64: no split
    assert kda.kda_chunk_fwd_workspace_size(0, 0, 1, 64, 64) == 256
    # more chains than one wave of CTAs: room for the launch order (N int32, 16-byte rounded)
    assert kda.kda_chunk_fwd_workspace_size(64, 300000, 32, 128, 128) == 256 + 64 * 32 * 65536 + 256 + fb(64, 32)
    assert kda.kda_chunk_fwd_workspace_size(39, 5000, 4, 64, 64) == 256 + 39 * 4 * 16384 + 160 + fb(39, 4)
    assert kda.kda_chunk_fwd_workspace_size(38, 5000, 4, 64, 64) == 256 + 38 * 4 * 16384 + fb(38, 4)  # one wave
    assert kda.kda_chunk_fwd_workspace_size(1, 10, 2, 96, 128) == 0
    assert kda.kda_chunk_fwd_workspace_size(-1, 10, 2, 64, 128) == 0


FAKE = 0x10000  # a 16-byte aligned non-null value; never dereferenced (the checks fail first)


def _chunk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, dtype=0, init=None, cu=None, N=1, T=64, H=2,
             dk=128, dv=128, scale=1.0, o=FAKE, fs=FAKE, ws=FAKE, wsb=256, stream=None)
    a.update(kw)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["dtype"], a["init"], a["cu"], a["N"],
                             a["T"], a["H"], a["dk"], a["dv"], a["scale"], a["o"], a["fs"], a["ws"], a["wsb"],
                             a["stream"])


def test_chunk_fwd_host_errors(lib):
    assert _chunk(lib, dk=96) == 2                       # UNSUPPORTED
    assert _chunk(lib, dv=32) == 2
    assert _chunk(lib, dtype=7) == 2
    assert _chunk(lib, H=0) == 1                         # INVALID_ARGUMENT
    assert _chunk(lib, N=-1) == 1
    assert _chunk(lib, q=None) == 1
    assert _chunk(lib, o=None) == 1
    assert _chunk(lib, k=FAKE + 4) == 1                  # misaligned
    assert _chunk(lib, beta=FAKE + 1) == 1               # bf16 beta must be 2-byte aligned
    assert _chunk(lib, N=3, T=64) == 1                   # equal lengths need N | T
    assert _chunk(lib, ws=None) == 3                     # WORKSPACE
    assert _chunk(lib, wsb=255) == 3
    assert _chunk(lib, fs=None, wsb=256) == 3            # no final_state: staging space needed
    assert _chunk(lib, init=FAKE + 8) == 1


def test_decode_and_replay_host_errors(lib):
    d = lib.kda_decode_step
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 96, 1.0, FAKE, FAKE, 256, None) == 2
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, 4, None, 2, 2, 128, 128, 1.0, FAKE, FAKE, 256, None) == 1
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, None, 2, 2, 128, 128, 1.0, FAKE, FAKE, 256, None) == 1
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 128, 1.0, FAKE, FAKE, 100, None) == 3
    r = lib.kda_replay
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 0, None, 2, 8, 2, 128, 128, FAKE, 256, None) == 1
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 2, 8, 2, 64, 48, FAKE, 256, None) == 2
    assert r(FAKE, 1, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, FAKE, 256, None) == 1
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, None, 256, None) == 3


def test_state_pool_host_errors(lib):
    """Host-detectable errors of the state-pool calls return before any CUDA work."""
    import ctypes
    ws = ctypes.c_void_p(4096)          # never dereferenced on these paths
    fake = ctypes.c_void_p(1 << 20)     # aligned stand-in for a device pointer
    assert lib.kda_state_fork(fake, 8, fake, fake, 1, 2, 96, 128, ws, 256, None) == 2   # UNSUPPORTED dk
    assert lib.kda_state_fork(fake, 8, fake, fake, -1, 2, 128, 128, ws, 256, None) == 1  # negative n
    assert lib.kda_state_fork(fake, 8, None, fake, 1, 2, 128, 128, ws, 256, None) == 1   # NULL slots
    assert lib.kda_state_fork(fake, 8, fake, fake, 1, 2, 128, 128, None, 256, None) == 3  # no workspace
    assert lib.kda_state_offload(fake, 8, None, 1, 2, 128, 128, None, ws, 256, None) == 1  # NULL host
    assert lib.kda_state_restore(fake, 8, None, 1, 0, 128, 128, fake, ws, 256, None) == 1  # H = 0
    assert lib.kda_state_offload(fake, 8, None, 1, 2, 128, 128, fake, ws, 16, None) == 3   # small workspace


def test_prep_flag_host_errors(lib):
    """Unknown preprocessing flags and a bad epsilon are rejected on the host; the
    plain calls are the _prep calls with no flags (same checks, same codes)."""
    c = lib.kda_chunk_fwd_prep
    args = lambda prep, eps, **kw: (FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("dtype", 0), None, None, 1, 64, 2,
                                    kw.get("dk", 128), 128, 1.0, prep, eps, FAKE, FAKE, FAKE, kw.get("wsb", 256),
                                    None)
    assert c(*args(16, 1e-6)) == 1                      # unknown flag
    assert c(*args(0x80000000, 1e-6)) == 1
    assert c(*args(2, -1e-6)) == 1                       # negative eps
    assert c(*args(2, float("nan"))) == 1
    assert c(*args(2, float("inf"))) == 1
    assert c(*args(2, 1e-6, dk=96)) == 2                 # shape checks come first
    assert c(*args(15, 1e-6, wsb=255)) == 3              # valid flags: falls through to the workspace check
    d = lib.kda_decode_step_prep
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 128, 1.0, 32, 1e-6, FAKE, FAKE, 256,
             None) == 1
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 128, 1.0, 15, 1e-6, FAKE, FAKE, 100,
             None) == 3
    r = lib.kda_replay_prep
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, 64, 1e-6, FAKE, 256, None) == 1
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, 15, -2.0, FAKE, 256, None) == 1
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, 15, 1e-6, None, 256, None) == 3


def test_bwd_workspace_size_and_host_errors(lib):
    """Backward workspace: header, checkpoints and records per (64-token slot, head),
    staging states and the persistent-CTA scratch; host-detectable errors return early."""
    from gated_linear_attention_chunk_gb300 import kda
    small = kda.kda_chunk_bwd_workspace_size(1, 64, 1, 64, 64)
    big = kda.kda_chunk_bwd_workspace_size(1, 6400, 1, 64, 64)
    assert small > 256 and big > small
    # 99 more slots, each a 64x64 checkpoint (16 KiB) and a record of the same size per slot
    per_slot = (big - small) // 99
    assert (big - small) % 99 == 0 and per_slot > 64 * 64 * 4
    assert kda.kda_chunk_bwd_workspace_size(1, 64, 1, 96, 64) == 0
    assert kda.kda_chunk_bwd_workspace_size(-1, 64, 1, 64, 64) == 0
    b = lib.kda_chunk_bwd
    args = lambda **kw: tuple(kw.get(n, d) for n, d in (
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("g", FAKE), ("beta", FAKE), ("dtype", 0), ("init", None),
        ("cu", None), ("N", 1), ("T", 64), ("H", 1), ("dk", 64), ("dv", 64), ("scale", 1.0), ("d_o", FAKE),
        ("d_fin", None), ("dq", FAKE), ("dkk", FAKE), ("dvv", FAKE), ("dg", FAKE), ("db", FAKE), ("dinit", None),
        ("ws", FAKE), ("wsb", small), ("stream", None)))
    assert b(*args(dk=96)) == 2                   # UNSUPPORTED
    assert b(*args(dtype=5)) == 2
    assert b(*args(H=0)) == 1                     # INVALID_ARGUMENT
    assert b(*args(d_o=None)) == 1
    assert b(*args(dg=None)) == 1
    assert b(*args(k=FAKE + 4)) == 1              # misaligned
    assert b(*args(N=3, wsb=big)) == 1            # equal lengths need N | T
    assert b(*args(ws=None)) == 3                 # WORKSPACE
    assert b(*args(wsb=small - 1)) == 3


def test_conv_host_errors(lib):
    """The convolution calls reject a width other than KDA_CONV_WIDTH and missing weights on the host."""
    c = lib.kda_conv_fwd
    base = dict(q=FAKE, k=FAKE, v=FAKE, dtype=0, w=FAKE, width=4, sin=None, cu=None, N=1, T=8, H=1, dk=64, dv=64,
                qo=FAKE, ko=FAKE, vo=FAKE, sout=None, ws=FAKE, wsb=256, stream=None)
    call = lambda **kw: c(*({**base, **kw}).values())
    assert call(width=3) == 2                    # UNSUPPORTED
    assert call(dk=96) == 2
    assert call(w=None) == 1                     # INVALID_ARGUMENT
    assert call(qo=None) == 1
    assert call(N=3) == 1                        # equal lengths need N | T
    assert call(ws=None) == 3                    # WORKSPACE
    d = lib.kda_decode_step_conv
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 128, 1.0, FAKE, 5, FAKE, 0, 0.0, FAKE,
             FAKE, 256, None) == 2
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 4, None, 2, 2, 128, 128, 1.0, None, 4, FAKE, 0, 0.0, FAKE,
             FAKE, 256, None) == 1
    r = lib.kda_replay_conv
    assert r(FAKE, 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, FAKE, 4, None, 0, 0.0, FAKE,
             256, None) == 1
    assert r(FAKE, 4, None, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 2, 128, 128, FAKE, 4, FAKE, 0, 0.0, FAKE,
             256, None) == 1                     # the accepted tokens' q is needed for the convolution state
