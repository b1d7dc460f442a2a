"""Strong decay on the chunked path: a 64-token chunk whose decay product falls below the range
the factored (WY) form supports, or a gate of exactly zero (g = -inf), sends its (sequence, head)
chain to the token-sequential kernel, which recomputes it from the initial state; the call
succeeds and every chain matches the fp64 oracle.  Without room in the workspace for the
per-chain flags the call still reports KDA_ERR_GATE_RANGE (test_gpu_workloads)."""
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


def _run_and_check(kda, case, g=None, what=""):
    d = to_dev(case)
    if g is not None:
        d["g"] = g.cuda()
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(case.N, case.T_total, case.H, case.dk, case.dv), "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g if g is None else g, case.beta,
                                   case.cu_seqlens, case.init_state, threads=0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(fs).all()
    assert_close(o, o_ref, f"{what} o")
    assert_close(fs, fs_ref, f"{what} final_state")


def test_strong_decay_everywhere(kda):
    """g = logsigmoid(N(-1, 1)): a 64-token chunk decays by about e^-84, below 2^-100, in nearly every
    channel, so every chain is recomputed token by token."""
    case = workloads.make_case([4096, 1000, 70], H=4, dk=128, dv=128, seed=21, g_mu=-1.0)
    _run_and_check(kda, case, what="strong decay")


def test_strong_decay_in_one_chain_only(kda):
    """Only head 2 of sequence 1 decays strongly; every other chain stays on the chunked path."""
    case = workloads.make_case([640, 1300, 64], H=4, dk=128, dv=128, seed=22)
    g = case.g.clone()
    b, e = int(case.cu_seqlens[1]), int(case.cu_seqlens[2])
    g[b + 200:b + 264, 2, :] = -3.0
    _run_and_check(kda, case, g=g, what="one strong chain")


def test_zero_gate_inside_a_chunk(kda):
    """g = -inf (alpha = 0, the state is erased) on one token in the middle of a full chunk, in some
    channels of one head and in every channel of another."""
    case = workloads.make_case([512, 300], H=3, dk=128, dv=128, seed=23)
    g = case.g.clone()
    g[100, 0, 5:40] = float("-inf")
    g[390, 1, :] = float("-inf")
    _run_and_check(kda, case, g=g, what="zero gate")


def test_strong_decay_with_the_t_segment_split(kda):
    """A batch of few long chains takes the T-segment split; a flagged chain is still recomputed."""
    case = workloads.make_case([4096 + 37], H=4, dk=128, dv=128, seed=24)
    assert case.N * case.H <= 48
    g = case.g.clone()
    g[3000:3064, 1, 7] = -3.5
    _run_and_check(kda, case, g=g, what="split path")


def test_strong_decay_with_the_launch_order(kda):
    """More chains than one wave: sequences are ordered longest first; a flagged chain is recomputed."""
    lengths = [200 + 37 * i for i in range(40)]
    case = workloads.make_case(lengths, H=4, dk=128, dv=128, seed=25)
    assert case.N * case.H > 152
    g = case.g.clone()
    b = int(case.cu_seqlens[33])
    g[b + 64:b + 128, 3, :] = -2.5
    _run_and_check(kda, case, g=g, what="ordered path")
