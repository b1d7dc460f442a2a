"""kda_chunk_fwd_noalloc: the allocation-free prefill entry point, called through the C ABI.

Callers that cannot allocate device memory (hosts that plan every device byte and
give plug-in kernels no workspace, latency-critical loops that may not call
cudaMalloc) use this entry point; it runs on a fixed scratch array the library
owns.  The test compares it with kda_chunk_fwd on the same inputs, twice in a
row (the second call reuses the shared scratch left by the first), and checks
that requests too large for the scratch are refused.  It sits in its own file,
collected last, and needs nothing from the other tests.
"""
import ctypes

import pytest
import torch

import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from gated_linear_attention_chunk_gb300 import kda as binding
    return binding.load_library()


def _call_noalloc(lib, d, case, o, final_state):
    ws = ctypes.c_void_p()
    rc = lib.kda_chunk_fwd_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                                   d["beta"].data_ptr(), 0, d["init_state"].data_ptr(),
                                   d["cu_seqlens"].data_ptr(), case.N, case.T_total, case.H, case.dk, case.dv,
                                   case.scale, o.data_ptr(),
                                   None if final_state is None else final_state.data_ptr(), ctypes.byref(ws),
                                   torch.cuda.current_stream().cuda_stream)
    return rc, ws.value


def test_noalloc_matches_chunk_fwd_on_two_calls(lib):
    from gated_linear_attention_chunk_gb300 import kda as binding
    # full chunks (tensor-core kernel) plus partial tails, so the staged states are exercised
    case = workloads.make_case([200, 70, 64, 5], H=2, dk=128, dv=128, seed=909)
    d = to_dev(case)
    o_ref, fs_ref = binding.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                          init_state=d["init_state"])
    torch.cuda.synchronize()
    ref_o = o_ref.double().cpu().numpy()
    ref_fs = fs_ref.double().cpu().numpy()

    # call 1: no final_state, so the states are staged in the library's scratch
    o1 = torch.full_like(o_ref, float("nan"))
    rc, ws = _call_noalloc(lib, d, case, o1, None)
    assert rc == binding.KDA_OK
    assert ws
    assert binding.kda_device_status(ws) == binding.KDA_OK
    assert_close(o1, ref_o, "noalloc call 1: o")

    # call 2: same inputs again, with final_state; the scratch still holds call 1's contents
    o2 = torch.full_like(o_ref, float("nan"))
    fs2 = torch.full_like(fs_ref, float("nan"))
    rc, ws2 = _call_noalloc(lib, d, case, o2, fs2)
    assert rc == binding.KDA_OK and ws2 == ws
    assert binding.kda_device_status(ws2) == binding.KDA_OK
    assert_close(o2, ref_o, "noalloc call 2: o")
    assert_close(fs2, ref_fs, "noalloc call 2: final_state")


def test_noalloc_refuses_requests_beyond_its_scratch(lib):
    from gated_linear_attention_chunk_gb300 import kda as binding
    # 129 states of 128 x 128 fp32 to stage: one more than the 8 MiB scratch holds
    N, H, T = 129, 1, 129
    q = torch.zeros(T, H, 128, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    ws = ctypes.c_void_p()
    rc = lib.kda_chunk_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), b.data_ptr(), 0, None,
                                   cu.data_ptr(), N, T, H, 128, 128, 1.0, o.data_ptr(), None, ctypes.byref(ws),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == binding.KDA_ERR_WORKSPACE
    # with final_state given only the status header is needed, so the same batch is accepted
    fs = torch.empty(N, H, 128, 128, dtype=torch.float32, device="cuda")
    rc = lib.kda_chunk_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), b.data_ptr(), 0, None,
                                   cu.data_ptr(), N, T, H, 128, 128, 1.0, o.data_ptr(), fs.data_ptr(),
                                   ctypes.byref(ws), torch.cuda.current_stream().cuda_stream)
    assert rc == binding.KDA_OK
    assert binding.kda_device_status(ws.value) == binding.KDA_OK
