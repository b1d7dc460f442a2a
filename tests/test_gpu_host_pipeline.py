"""HostPrefill: a packed prefill from pinned host memory, cut into sequence groups whose
host->device copies, kernels and device->host copies overlap on three streams.  Checked
against the fp64 oracle and, bit for bit, against one kda_chunk_fwd call over the whole
batch where every group takes the same path as that call (no T-segment split)."""
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
    assert len(pipe.groups) == min(groups, case.N)
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
