"""Head dims of 64 on the chunked tensor-core path (bf16).  The kernel works on 128-wide tiles;
with dk or dv = 64 its tensor maps cover 64 channels, TMA fills the second 64-channel box with
zeros, and the state and output stores skip the columns beyond dv.  Zero channels and columns
leave the d = 64 result unchanged, so every check is the usual one: the fp64 oracle within the
tolerance, and the bit-exact contracts with the token-sequential kernel (the partial-chunk
tail continues from the chunked state)."""
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (64, 128), (128, 64)]


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    return m


def _bits(t):
    return t.detach().cpu().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def _oracle(case, prep=0, eps=1e-6):
    return oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                          scale=case.scale, threads=0, prep_flags=prep, prep_eps=eps)


def test_tensor_core_path_covers_head_dims_64(kda):
    for dk, dv in DIMS + [(128, 128)]:
        assert kda.kda_chunk_fwd_uses_tensor_cores(dk, dv, torch.bfloat16)
        assert not kda.kda_chunk_fwd_uses_tensor_cores(dk, dv, torch.float32)


@pytest.mark.parametrize("dk,dv", DIMS)
def test_many_chunks_match_oracle(kda, dk, dv):
    """Several full chunks per sequence, ragged tails, an empty sequence, initial states."""
    case = workloads.make_case([1000, 300, 0, 64, 129, 5], H=4, dk=dk, dv=dv, seed=90 + dk + dv)
    d = to_dev(case)
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(case.N, case.T_total, case.H, dk, dv), "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    o_ref, fs_ref = _oracle(case)
    assert_close(o, o_ref, f"d={dk}x{dv} o")
    assert_close(fs, fs_ref, f"d={dk}x{dv} final_state")


@pytest.mark.parametrize("dk,dv", DIMS)
@pytest.mark.parametrize("r", [1, 63])
def test_prefill_tail_is_bit_exact_with_decode_steps(kda, dk, dv, r):
    """chunk_fwd over 128 + r tokens == chunk_fwd over 128 tokens, then r decode steps."""
    H, P = 2, 128
    L = P + r
    case = workloads.make_case([L], H=H, dk=dk, dv=dv, seed=100 + r + dk)
    d = to_dev(case)
    o_full, fs_full = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                        init_state=d["init_state"])
    cu_p = torch.tensor([0, P], dtype=torch.int32, device="cuda")
    sl = slice(0, P)
    o_p, state = kda.kda_chunk_fwd(d["q"][sl], d["k"][sl], d["v"][sl], d["g"][sl], d["beta"][sl],
                                   cu_seqlens=cu_p, init_state=d["init_state"])
    outs = [o_p]
    for t in range(P, L):
        ts = slice(t, t + 1)
        outs.append(kda.kda_decode_step(d["q"][ts], d["k"][ts], d["v"][ts], d["g"][ts], d["beta"][ts], state))
    torch.cuda.synchronize()
    assert torch.equal(_bits(torch.cat(outs)), _bits(o_full))
    assert torch.equal(_bits(state), _bits(fs_full))
    o_ref, fs_ref = _oracle(case)
    assert_close(o_full, o_ref, "o")
    assert_close(fs_full, fs_ref, "final_state")


def test_preprocessing_flags_with_head_dim_64(kda):
    """Raw inputs, every flag (row norms, sigmoid gate, sigmoid beta): the zero channels add
    nothing to the norms, and their sigmoid gate of 1/2 only scales zero state rows."""
    flags, eps = 15, 1e-6
    case = workloads.make_case([700, 65, 128], H=3, dk=64, dv=64, seed=110, q_scale=False, scale=64 ** -0.5,
                               raw=True)
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], flags, eps,
                                   cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], scale=case.scale)
    torch.cuda.synchronize()
    o_ref, fs_ref = _oracle(case, flags, eps)
    assert_close(o, o_ref, "prep o")
    assert_close(fs, fs_ref, "prep final_state")


def test_launch_order_and_strong_decay_with_head_dim_64(kda):
    """More chains than one wave (launch order) and one chain whose gates decay too strongly
    for the chunked form (recomputed token by token)."""
    lengths = [150 + 29 * i for i in range(48)]
    case = workloads.make_case(lengths, H=4, dk=64, dv=64, seed=111)
    assert case.N * case.H > 152
    g = case.g.clone()
    b = int(case.cu_seqlens[20])
    g[b + 64:b + 128, 1, :] = -3.0
    d = to_dev(case)
    d["g"] = g.cuda()
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(case.N, case.T_total, case.H, 64, 64), "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, g, case.beta, case.cu_seqlens, case.init_state,
                                   scale=case.scale, threads=0)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


def test_in_place_state_with_head_dim_64(kda):
    """final_state may be init_state (dk x dv, row stride dv)."""
    case = workloads.make_case([300, 64, 1], H=2, dk=64, dv=128, seed=112)
    d = to_dev(case)
    st = d["init_state"].clone()
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=st, final_state=st, scale=case.scale)
    torch.cuda.synchronize()
    o_ref, fs_ref = _oracle(case)
    assert fs.data_ptr() == st.data_ptr()
    assert_close(o, o_ref, "o")
    assert_close(st, fs_ref, "final_state in place")
