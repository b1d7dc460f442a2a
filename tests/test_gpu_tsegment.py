"""T-segment split of the chunked prefill (few (sequence, head) chains, long sequences).

With N*H <= 48 and T_total >= 4096 (dk = dv = 128) and the full workspace,
kda_chunk_fwd cuts each sequence's full chunks in two and merges the halves
exactly; with a workspace that is only large enough for the plain path it runs
unsplit.  Both are checked against the fp64 oracle, including a sequence too
short to have a second segment and sequences with a partial-chunk tail.
"""
import pytest

import oracle
import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    return m


def _run(kda, case, split):
    d = to_dev(case)
    N, H = case.N, case.H
    T = int(case.cu_seqlens[-1])
    full = kda.kda_chunk_fwd_workspace_size(N, T, H, 128, 128)
    plain = kda.KDA_WS_HEADER_BYTES + N * H * 128 * 128 * 4
    assert full > plain  # the shape qualifies for the split
    ws = kda.new_workspace(full if split else plain, "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    return o, fs


@pytest.mark.parametrize("lengths,H", [([4497], 2), ([3000, 70, 1500], 2), ([2048, 2048, 64], 4)])
@pytest.mark.parametrize("split", [True, False])
def test_split_and_plain_match_oracle(kda, lengths, H, split):
    case = workloads.make_case(lengths, H=H, dk=128, dv=128, seed=len(lengths) * 31 + H)
    o, fs = _run(kda, case, split)
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    tag = "split" if split else "plain"
    assert_close(o, o_ref, f"{tag} o")
    assert_close(fs, fs_ref, f"{tag} final_state")


def test_split_in_place_state(kda):
    """init_state aliasing final_state: segment 0 reads it before the merge overwrites it."""
    case = workloads.make_case([4160], H=2, dk=128, dv=128, seed=5)
    d = to_dev(case)
    st = d["init_state"].clone()
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(case.N, 4160, case.H, 128, 128), "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=st, final_state=st, scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    assert_close(o, o_ref, "in-place split o")
    assert_close(st, fs_ref, "in-place split final_state")
