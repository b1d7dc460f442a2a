"""GPU parity of the fused input preprocessing (kda_chunk_fwd_prep, kda_decode_step_prep,
kda_replay_prep) against the fp64 oracle on raw inputs, and the bit-exact contracts
between the three calls with preprocessing on.  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu

ALL = 15          # L2NORM_Q | L2NORM_K | SIGMOID_GATE | SIGMOID_BETA
EPS = 1e-6


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    assert m.KDA_PREP_L2NORM_Q | m.KDA_PREP_L2NORM_K | m.KDA_PREP_SIGMOID_GATE | m.KDA_PREP_SIGMOID_BETA == ALL
    return m


def _bits(t):
    return t.detach().cpu().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def _raw_case(lengths, H=2, dk=128, dv=128, dtype=torch.bfloat16, seed=0, init=True):
    return workloads.make_case(lengths, H=H, dk=dk, dv=dv, dtype=dtype, seed=seed, init=init, q_scale=False,
                               scale=dk ** -0.5, raw=True)


def _run(kda, case, prep, eps=EPS, **kw):
    d = to_dev(case)
    o, fs = kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], prep, eps,
                                   cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], scale=case.scale, **kw)
    torch.cuda.synchronize()
    return o, fs


def _oracle(case, prep, eps=EPS):
    return oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                          scale=case.scale, threads=0, prep_flags=prep, prep_eps=eps)


LENGTHS = [1, 63, 64, 65, 130, 0, 200, 128, 7]


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_chunk_fwd_prep_all_flags_matches_oracle(kda, dk, dv, dtype):
    """Tensor-core chunks (bf16, 128 x 128), the token-sequential kernel and the ragged tails."""
    case = _raw_case(LENGTHS, H=3, dk=dk, dv=dv, dtype=dtype, seed=40 + dk + dv)
    o, fs = _run(kda, case, ALL)
    o_ref, fs_ref = _oracle(case, ALL)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


@pytest.mark.parametrize("flag", [1, 2, 4, 8, 3, 12])
def test_chunk_fwd_prep_each_flag(kda, flag):
    """One flag at a time: a flag left off uses that input as given, so the raw case is
    first made valid for the flags that are off (unit-norm k, log-gates, beta in (0, 1))."""
    case = _raw_case([256, 100, 64], H=2, seed=50 + flag)
    if not flag & 2:
        case.k = (case.k.float() / case.k.float().norm(dim=-1, keepdim=True)).to(case.k.dtype)
    if not flag & 4:
        case.g = torch.nn.functional.logsigmoid(case.g.float()).to(case.g.dtype)
    if not flag & 8:
        case.beta = torch.sigmoid(case.beta.float()).to(case.beta.dtype)
    o, fs = _run(kda, case, flag)
    o_ref, fs_ref = _oracle(case, flag)
    assert_close(o, o_ref, f"o (flags {flag})")
    assert_close(fs, fs_ref, f"final_state (flags {flag})")


def test_prep_zero_is_the_plain_call(kda):
    """The _prep call with no flags is bit for bit the plain call (both kernels)."""
    case = workloads.make_case([200, 64, 9], H=2, dk=128, dv=128, seed=60)
    d = to_dev(case)
    o1, fs1 = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                init_state=d["init_state"])
    o2, fs2 = kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], 0, 0.0,
                                     cu_seqlens=d["cu_seqlens"], init_state=d["init_state"])
    torch.cuda.synchronize()
    assert torch.equal(_bits(o1), _bits(o2))
    assert torch.equal(_bits(fs1), _bits(fs2))


def test_chunk_fwd_prep_eps_matters(kda):
    """A large eps changes the result the way the oracle says (eps sits under the root)."""
    case = _raw_case([130], H=2, seed=61)
    o, fs = _run(kda, case, ALL, eps=64.0)
    o_ref, fs_ref = _oracle(case, ALL, eps=64.0)
    assert_close(o, o_ref, "o (eps 64)")
    assert_close(fs, fs_ref, "final_state (eps 64)")


def test_chunk_fwd_prep_t_segment_split(kda):
    """Few long sequences take the T-segment split; the preprocessing applies in every
    segment run (including the transition run)."""
    case = _raw_case([8192], H=2, seed=62, init=True)
    o, fs = _run(kda, case, ALL)
    o_ref, fs_ref = _oracle(case, ALL)
    assert_close(o, o_ref, "o (split)")
    assert_close(fs, fs_ref, "final_state (split)")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_prep_is_bit_exact_with_one_token_chunk_fwd_prep(kda, dtype):
    N, H, dk, dv = 5, 4, 128, 128
    q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(N, H, dk, dv, dtype, seed=63, raw=True))
    pool = (torch.randn(N + 2, H, dk, dv, generator=torch.Generator().manual_seed(3)) * 0.3).cuda()
    slots = torch.tensor([3, 0, 6, 2, 5], dtype=torch.int32, device="cuda")
    init = pool[slots.long()].clone()
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    o_chunk, fs_chunk = kda.kda_chunk_fwd_prep(q, k, v, g, b, ALL, EPS, cu_seqlens=cu, init_state=init,
                                               scale=dk ** -0.5)
    pool2 = pool.clone()
    o_dec = kda.kda_decode_step_prep(q, k, v, g, b, pool2, ALL, EPS, slots=slots, scale=dk ** -0.5)
    torch.cuda.synchronize()
    assert torch.equal(_bits(o_dec), _bits(o_chunk))
    assert torch.equal(_bits(pool2[slots.long()]), _bits(fs_chunk))
    o_ref, pool_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), g.cpu(), b.cpu(), pool.cpu(), slots.cpu(),
                                    scale=dk ** -0.5, prep_flags=ALL, prep_eps=EPS)
    assert_close(o_dec, o_ref, "decode o")
    assert_close(pool2, pool_ref, "decode pool")


def test_replay_prep_is_bit_exact_with_chunk_fwd_prep_final_state(kda):
    H, dk, dv = 4, 128, 128
    acc = [1, 4, 0, 3, 2, 4]
    N, A = len(acc), sum(acc)
    q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(A, H, dk, dv, torch.bfloat16, seed=64,
                                                                     raw=True))
    pool = (torch.randn(N, H, dk, dv, generator=torch.Generator().manual_seed(4)) * 0.3).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(acc)]), dtype=torch.int32, device="cuda")
    _, fs = kda.kda_chunk_fwd_prep(q, k, v, g, b, ALL, EPS, cu_seqlens=cu, init_state=pool)
    pool2 = pool.clone()
    kda.kda_replay_prep(pool2, k, v, g, b, cu, ALL, EPS)
    torch.cuda.synchronize()
    assert torch.equal(_bits(pool2), _bits(fs))
    ref = oracle.replay(k.cpu(), v.cpu(), g.cpu(), b.cpu(), cu.cpu(), pool.cpu(), prep_flags=ALL, prep_eps=EPS)
    assert_close(pool2, ref, "replay pool")


@pytest.mark.parametrize("r", [1, 40])
def test_prefill_prep_tail_is_bit_exact_with_decode_prep_steps(kda, r):
    H, dk, dv, m = 2, 128, 128, 2
    L = 64 * m + r
    case = _raw_case([L], H=H, seed=65 + r)
    d = to_dev(case)
    sc = case.scale
    o_full, fs_full = kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], ALL, EPS,
                                             cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], scale=sc)
    P = 64 * m
    cu_p = torch.tensor([0, P], dtype=torch.int32, device="cuda")
    sl = slice(0, P)
    o_p, state = kda.kda_chunk_fwd_prep(d["q"][sl], d["k"][sl], d["v"][sl], d["g"][sl], d["beta"][sl], ALL, EPS,
                                        cu_seqlens=cu_p, init_state=d["init_state"], scale=sc)
    outs = [o_p]
    for t in range(P, L):
        ts = slice(t, t + 1)
        outs.append(kda.kda_decode_step_prep(d["q"][ts], d["k"][ts], d["v"][ts], d["g"][ts], d["beta"][ts], state,
                                             ALL, EPS, scale=sc))
    torch.cuda.synchronize()
    assert torch.equal(_bits(torch.cat(outs)), _bits(o_full))
    assert torch.equal(_bits(state), _bits(fs_full))


def test_sigmoid_gate_beyond_the_chunked_range(kda):
    """A raw gate so negative that a chunk's decay product falls below the range the chunked
    kernel factors (sigmoid(-6)^64 is about 2^-222): with the full workspace the chain is
    recomputed token by token and matches the oracle; with only the status header the call
    reports KDA_ERR_GATE_RANGE, as with log-gates."""
    case = _raw_case([128], H=1, seed=66)
    case.g = torch.full_like(case.g, -6.0)
    d = to_dev(case)
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(1, 128, 1, 128, 128), "cuda")
    o, fs = kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], ALL, EPS, cu_seqlens=d["cu_seqlens"],
                                   init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   scale=case.scale, prep_flags=ALL, prep_eps=EPS)
    assert_close(o, o_ref, "o (strong sigmoid gate, recomputed)")
    assert_close(fs, fs_ref, "final_state (strong sigmoid gate, recomputed)")
    small = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, "cuda")
    kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], ALL, EPS, cu_seqlens=d["cu_seqlens"],
                           init_state=d["init_state"], scale=case.scale, workspace=small)
    assert kda.kda_device_status(small) == kda.KDA_ERR_GATE_RANGE
    case.g = torch.full_like(case.g, 2.0)
    d = to_dev(case)
    kda.kda_chunk_fwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], ALL, EPS, cu_seqlens=d["cu_seqlens"],
                           init_state=d["init_state"], scale=case.scale, workspace=small)
    assert kda.kda_device_status(small) == kda.KDA_OK
