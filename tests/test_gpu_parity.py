"""GPU parity of kda_chunk_fwd / kda_decode_step / kda_replay against the fp64 oracle,
and the bit-exact contracts between them.  Every call goes through the C ABI."""
import numpy as np
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


def _run_chunk(kda, case, **kw):
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, **kw)
    torch.cuda.synchronize()
    return o, fs


def _oracle(case):
    return oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                          scale=case.scale, threads=0)


LENGTHS = [1, 63, 64, 65, 130, 0, 200, 128, 7]


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_chunk_fwd_varlen_matches_oracle(kda, dk, dv, dtype):
    case = workloads.make_case(LENGTHS, H=3, dk=dk, dv=dv, dtype=dtype, seed=dk + dv + (dtype == torch.float32))
    o, fs = _run_chunk(kda, case)
    o_ref, fs_ref = _oracle(case)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


def test_tiny_fp32_named_workload(kda):
    case = workloads.named_case("tiny_fp32")
    o, fs = _run_chunk(kda, case)
    o_ref, fs_ref = _oracle(case)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


def test_raw_query_with_scale_argument(kda):
    case = workloads.make_case([150, 70], H=2, dk=128, dv=128, q_scale=False, scale=128 ** -0.5, seed=5)
    o, fs = _run_chunk(kda, case)
    o_ref, fs_ref = _oracle(case)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


def test_no_init_state_and_no_final_state(kda):
    case = workloads.make_case([70, 64, 3], H=2, dk=128, dv=128, init=False, seed=6)
    o, fs = _run_chunk(kda, case, output_final_state=False)
    assert fs is None
    o_ref, _ = _oracle(case)
    assert_close(o, o_ref, "o")


def test_in_place_state_update(kda):
    case = workloads.make_case([100, 64, 1], H=2, dk=128, dv=128, seed=7)
    d = to_dev(case)
    state = d["init_state"].clone()
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"], init_state=state,
                      final_state=state)
    torch.cuda.synchronize()
    _, fs_ref = _oracle(case)
    assert_close(state, fs_ref, "final_state (in place)")


def test_equal_length_batch_without_cu_seqlens(kda):
    case = workloads.make_case([96, 96], H=2, dk=64, dv=64, seed=8)
    d = to_dev(case)
    q, k, v, g, b = d["q"], d["k"], d["v"], d["g"], d["beta"]
    # cu_seqlens=None means one sequence in the binding; go through the C ABI with N=2 explicitly
    from gated_linear_attention_chunk_gb300 import kda as binding
    lib = binding.load_library()
    o = torch.empty_like(v)
    fs = torch.empty(2, 2, 64, 64, dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(256, "cuda")
    rc = lib.kda_chunk_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), b.data_ptr(), 0,
                           d["init_state"].data_ptr(), None, 2, 192, 2, 64, 64, 1.0, o.data_ptr(), fs.data_ptr(),
                           ws.data_ptr(), 256, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert binding.kda_device_status(ws) == 0
    o_ref, fs_ref = _oracle(case)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


# ------------------------------------------------------------------------------------------------
# Bit-exact contracts
# ------------------------------------------------------------------------------------------------

def _bits(t):
    return t.detach().cpu().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_is_bit_exact_with_one_token_chunk_fwd(kda, dtype):
    N, H, dk, dv = 5, 4, 128, 128
    q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(N, H, dk, dv, dtype, seed=11))
    pool = (torch.randn(N + 2, H, dk, dv, generator=torch.Generator().manual_seed(1)) * 0.3).cuda()
    slots = torch.tensor([3, 0, 6, 2, 5], dtype=torch.int32, device="cuda")
    init = pool[slots.long()].clone()
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    o_chunk, fs_chunk = kda.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=cu, init_state=init, scale=0.5)
    pool2 = pool.clone()
    o_dec = kda.kda_decode_step(q, k, v, g, b, pool2, slots=slots, scale=0.5)
    torch.cuda.synchronize()
    assert torch.equal(_bits(o_dec), _bits(o_chunk))
    assert torch.equal(_bits(pool2[slots.long()]), _bits(fs_chunk))
    untouched = torch.tensor([1, 4], device="cuda")
    assert torch.equal(pool2[untouched], pool[untouched])
    # and both match the oracle
    o_ref, pool_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), g.cpu(), b.cpu(), pool.cpu(), slots.cpu(),
                                    scale=0.5)
    assert_close(o_dec, o_ref, "decode o")
    assert_close(pool2, pool_ref, "decode pool")


def test_replay_is_bit_exact_with_chunk_fwd_final_state(kda):
    H, dk, dv = 4, 128, 128
    acc = [1, 4, 0, 3, 2, 4]
    N = len(acc)
    A = sum(acc)
    q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(A, H, dk, dv, torch.bfloat16, seed=12))
    pool = (torch.randn(N, H, dk, dv, generator=torch.Generator().manual_seed(2)) * 0.3).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(acc)]), dtype=torch.int32, device="cuda")
    _, fs = kda.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=cu, init_state=pool)
    pool2 = pool.clone()
    kda.kda_replay(pool2, k, v, g, b, cu)
    torch.cuda.synchronize()
    assert torch.equal(_bits(pool2), _bits(fs))
    ref = oracle.replay(k.cpu(), v.cpu(), g.cpu(), b.cpu(), cu.cpu(), pool.cpu())
    assert_close(pool2, ref, "replay pool")


@pytest.mark.parametrize("r", [1, 17, 63])
def test_prefill_tail_is_bit_exact_with_decode_steps(kda, r):
    """chunk_fwd over 64m + r tokens == chunk_fwd over 64m tokens, then r decode steps."""
    H, dk, dv, m = 2, 128, 128, 2
    L = 64 * m + r
    case = workloads.make_case([L], H=H, dk=dk, dv=dv, seed=20 + r)
    d = to_dev(case)
    o_full, fs_full = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                        init_state=d["init_state"])
    P = 64 * m
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


def test_run_to_run_determinism_and_batch_invariance(kda):
    H, dk, dv = 2, 128, 128
    case = workloads.make_case([200, 70, 64], H=H, dk=dk, dv=dv, seed=30)
    o1, f1 = _run_chunk(kda, case)
    o2, f2 = _run_chunk(kda, case)
    assert torch.equal(_bits(o1), _bits(o2)) and torch.equal(_bits(f1), _bits(f2))
    # the second sequence alone gives the same bits as inside the batch
    d = to_dev(case)
    sl = slice(200, 270)
    o_a, f_a = kda.kda_chunk_fwd(d["q"][sl], d["k"][sl], d["v"][sl], d["g"][sl], d["beta"][sl],
                                 cu_seqlens=torch.tensor([0, 70], dtype=torch.int32, device="cuda"),
                                 init_state=d["init_state"][1:2].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(_bits(o_a), _bits(o1[sl]))
    assert torch.equal(_bits(f_a), _bits(f1[1:2]))


def test_split_invariance_at_chunk_boundary(kda):
    """[0, 128) then [128, 300) with the carried state equals [0, 300): bitwise at a 64-aligned split."""
    case = workloads.make_case([300], H=2, dk=128, dv=128, seed=31)
    d = to_dev(case)
    o_full, f_full = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                       init_state=d["init_state"])
    s1, s2 = slice(0, 128), slice(128, 300)
    cu1 = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    cu2 = torch.tensor([0, 172], dtype=torch.int32, device="cuda")
    o1, f1 = kda.kda_chunk_fwd(d["q"][s1], d["k"][s1], d["v"][s1], d["g"][s1], d["beta"][s1], cu_seqlens=cu1,
                               init_state=d["init_state"])
    o2, f2 = kda.kda_chunk_fwd(d["q"][s2], d["k"][s2], d["v"][s2], d["g"][s2], d["beta"][s2], cu_seqlens=cu2,
                               init_state=f1)
    torch.cuda.synchronize()
    assert torch.equal(_bits(torch.cat([o1, o2])), _bits(o_full))
    assert torch.equal(_bits(f2), _bits(f_full))


def test_split_invariance_off_boundary_within_tolerance(kda):
    case = workloads.make_case([300], H=2, dk=128, dv=128, seed=32)
    d = to_dev(case)
    o_full, f_full = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                       init_state=d["init_state"])
    s1, s2 = slice(0, 100), slice(100, 300)
    o1, f1 = kda.kda_chunk_fwd(d["q"][s1], d["k"][s1], d["v"][s1], d["g"][s1], d["beta"][s1],
                               cu_seqlens=torch.tensor([0, 100], dtype=torch.int32, device="cuda"),
                               init_state=d["init_state"])
    o2, f2 = kda.kda_chunk_fwd(d["q"][s2], d["k"][s2], d["v"][s2], d["g"][s2], d["beta"][s2],
                               cu_seqlens=torch.tensor([0, 200], dtype=torch.int32, device="cuda"),
                               init_state=f1)
    torch.cuda.synchronize()
    assert_close(torch.cat([o1, o2]), o_full.double().cpu().numpy(), "split o")
    assert_close(f2, f_full.double().cpu().numpy(), "split state")


# ------------------------------------------------------------------------------------------------
# Device-detected errors (no GPU fault: the kernel skips the work item and sets a status bit)
# ------------------------------------------------------------------------------------------------

def test_bad_cu_seqlens_reported(kda):
    case = workloads.make_case([10, 20], H=2, dk=64, dv=64, seed=40)
    d = to_dev(case)
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")  # decreasing
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(2, 30, 2, 64, 64), "cuda")
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=bad, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SEQLENS
    bad2 = torch.tensor([0, 10, 31], dtype=torch.int32, device="cuda")  # beyond T_total
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=bad2, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SEQLENS
    # a valid call on the same workspace clears the word
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"], workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK


def test_bad_slot_reported(kda):
    q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(2, 2, 64, 64, torch.bfloat16, seed=41))
    pool = torch.zeros(3, 2, 64, 64, device="cuda")
    ws = kda.new_workspace(256, "cuda")
    kda.kda_decode_step(q, k, v, g, b, pool, slots=torch.tensor([0, 3], dtype=torch.int32, device="cuda"),
                        workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SLOT
    cu = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    kda.kda_replay(pool, k, v, g, b, cu, slots=torch.tensor([-1, 0], dtype=torch.int32, device="cuda"),
                   workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SLOT


def test_empty_sequences_copy_state(kda):
    case = workloads.make_case([0, 5, 0], H=2, dk=128, dv=128, seed=42)
    o, fs = _run_chunk(kda, case)
    assert torch.equal(fs[0].cpu(), case.init_state[0]) and torch.equal(fs[2].cpu(), case.init_state[2])
    o_ref, fs_ref = _oracle(case)
    assert_close(fs, fs_ref, "final_state")


def test_launch_order_for_many_chains_is_bit_identical(kda):
    """More chains than one wave (40 x 4 = 160): with the full workspace the call starts the
    longest sequences first; the results equal the oracle and, bit for bit, the same call
    with the minimum workspace (natural order)."""
    gen = torch.Generator().manual_seed(9)
    lengths = [int(x) for x in torch.randint(1, 400, (40,), generator=gen)]
    lengths[3], lengths[17] = 0, 64
    case = workloads.make_case(lengths, H=4, dk=128, dv=128, seed=75)
    d = to_dev(case)
    N, T = case.N, case.T_total
    full = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(N, T, 4, 128, 128), "cuda")
    o1, fs1 = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                init_state=d["init_state"], workspace=full)
    small = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, "cuda")
    o2, fs2 = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                init_state=d["init_state"], workspace=small)
    torch.cuda.synchronize()
    assert kda.kda_device_status(full) == kda.KDA_OK and kda.kda_device_status(small) == kda.KDA_OK
    assert torch.equal(_bits(o1), _bits(o2)) and torch.equal(_bits(fs1), _bits(fs2))
    o_ref, fs_ref = _oracle(case)
    assert_close(o1, o_ref, "o")
    assert_close(fs1, fs_ref, "final_state")
