"""HostPrefill: a packed prefill from pinned host memory, cut into pieces (runs of whole
sequences, and chunk-aligned parts of a long sequence whose state carries from part to part)
whose host->device copies, kernels and device->host copies overlap on three streams.  Checked
against the fp64 oracle and, bit for bit, against one kda_chunk_fwd call over the whole
batch where every piece takes the same path as that call (no T-segment split): a part of a
sequence continues from the fp32 state of the previous part exactly as the kernel continues
from chunk to chunk."""
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    return m


@pytest.mark.parametrize("groups", [1, 3, 5])
def test_host_prefill_matches_oracle_and_single_call(kda, groups):
    from gated_linear_attention_chunk_gb300.host_pipeline import HostPrefill
    case = workloads.make_case([300, 64, 1000, 5, 129], H=4, dk=128, dv=128, seed=31)
    pipe = HostPrefill(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                       scale=case.scale, groups=groups, device="cuda")
    parts = [pc for pc in pipe.groups if pc[1] == pc[0] + 1 and (pc[2], pc[3]) != (int(case.cu_seqlens[pc[0]]),
                                                                                  int(case.cu_seqlens[pc[1]]))]
    assert (len(parts) > 0) == (groups > 1)  # the 1000-token sequence is cut when its share is smaller
    for _ in range(2):  # the second pass reuses every buffer
        pipe.host_o.fill_(float("nan"))
        pipe.run()
        torch.cuda.synchronize()
        assert pipe.status() == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    assert_close(pipe.host_o, o_ref, f"host pipeline ({groups} groups) o")
    assert_close(pipe.host_final_state, fs_ref, f"host pipeline ({groups} groups) final_state")
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(pipe.host_o, o.cpu())
    assert torch.equal(pipe.host_final_state, fs.cpu())


def test_host_prefill_parts_without_initial_state(kda):
    """Long sequences cut into many parts, no initial state (the first part starts from zero)."""
    from gated_linear_attention_chunk_gb300.host_pipeline import HostPrefill
    case = workloads.make_case([1500, 70, 2100, 64], H=3, dk=128, dv=128, seed=32)
    pipe = HostPrefill(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, None,
                       scale=case.scale, groups=9, device="cuda")
    assert len(pipe.groups) >= 9
    pipe.run()
    torch.cuda.synchronize()
    assert pipe.status() == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, None, threads=0)
    assert_close(pipe.host_o, o_ref, "host pipeline parts o")
    assert_close(pipe.host_final_state, fs_ref, "host pipeline parts final_state")
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=None, scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(pipe.host_o, o.cpu())
    assert torch.equal(pipe.host_final_state, fs.cpu())


def test_host_prefill_graph_replay_matches_eager(kda):
    """graph=True: the second pass is captured and later passes replay it; the replays give the
    eager pipeline's bits, and inputs rewritten in place in the pinned host tensors are read."""
    from gated_linear_attention_chunk_gb300.host_pipeline import HostPrefill
    case = workloads.make_case([700, 64, 1300, 3], H=2, dk=128, dv=128, seed=33)
    args = (case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state)
    eager = HostPrefill(*args, scale=case.scale, groups=5, device="cuda")
    graph = HostPrefill(*args, scale=case.scale, groups=5, device="cuda", graph=True)
    assert graph.groups == eager.groups
    for it in range(4):
        if it == 3:  # new values for v in place: the replay must copy them in
            for pipe in (eager, graph):
                pipe.host["v"].mul_(-0.5)
        for pipe in (eager, graph):
            pipe.host_o.fill_(float("nan"))
            pipe.run()
        torch.cuda.synchronize()
        assert eager.status() == kda.KDA_OK and graph.status() == kda.KDA_OK
        assert torch.equal(graph.host_o, eager.host_o), f"pass {it}"
        assert torch.equal(graph.host_final_state, eager.host_final_state), f"pass {it}"
    assert graph._graph is not None
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v * -0.5, case.g, case.beta, case.cu_seqlens,
                                   case.init_state, threads=0)
    assert_close(graph.host_o, o_ref, "graph replay o")
    assert_close(graph.host_final_state, fs_ref, "graph replay final_state")


@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 128, 128), (torch.bfloat16, 64, 64), (torch.bfloat16, 64, 128)])
def test_host_prefill_parts_other_dtypes_and_head_dims(kda, dtype, dk, dv):
    """Parts of a sequence continue bit for bit on the token-sequential path (fp32 inputs) and on
    the 64-wide tensor-core instances, as within one call."""
    from gated_linear_attention_chunk_gb300.host_pipeline import HostPrefill
    case = workloads.make_case([1100, 40, 700], H=2, dk=dk, dv=dv, dtype=dtype, seed=34 + dk + dv)
    pipe = HostPrefill(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                       scale=case.scale, groups=6, device="cuda")
    assert any(b == a + 1 and (t0, t1) != (int(case.cu_seqlens[a]), int(case.cu_seqlens[b]))
               for a, b, t0, t1 in pipe.groups)
    pipe.run()
    torch.cuda.synchronize()
    assert pipe.status() == kda.KDA_OK
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(pipe.host_o, o.cpu())
    assert torch.equal(pipe.host_final_state, fs.cpu())
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    assert_close(pipe.host_o, o_ref, f"parts {dtype} {dk}x{dv} o")
    assert_close(pipe.host_final_state, fs_ref, f"parts {dtype} {dk}x{dv} final_state")
