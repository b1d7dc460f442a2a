"""GPU parity of the short convolution of the input projections (kda_conv_fwd for the
prefill, fused into kda_decode_step_conv and kda_replay_conv) against the fp64 oracle,
and the bit-exact contracts between decode and replay.  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_close, ensure_built

pytestmark = pytest.mark.gpu

W = 4
ALL = 15
EPS = 1e-6


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    assert m.KDA_CONV_WIDTH == W
    return m


def _bits(t):
    return t.detach().cpu().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def _weights(H, dk, dv, seed):
    return torch.randn(H, 2 * dk + dv, W, generator=torch.Generator().manual_seed(seed)) * 0.5


def _oracle_conv(q, k, v, w, cu, state):
    dk = q.shape[2]
    x = np.concatenate([np.asarray(t.float()) for t in (q, k, v)], axis=-1)
    y, so = oracle.conv(x, w, cu, state)
    return y[..., :dk], y[..., dk:2 * dk], y[..., 2 * dk:], so


LENGTHS = [1, 63, 64, 65, 130, 0, 200, 7]


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv_fwd_matches_oracle(kda, dk, dv, dtype, with_state):
    case = workloads.make_case(LENGTHS, H=2, dk=dk, dv=dv, dtype=dtype, seed=80 + dk + dv, raw=True)
    w = _weights(2, dk, dv, seed=dk)
    N = case.N
    st = (torch.randn(N, W - 1, 2, 2 * dk + dv, generator=torch.Generator().manual_seed(3))
          if with_state else None)
    dev = lambda t: None if t is None else t.cuda()
    qo, ko, vo, so = kda.kda_conv_fwd(dev(case.q), dev(case.k), dev(case.v), w.cuda(),
                                      cu_seqlens=dev(case.cu_seqlens), conv_state_in=dev(st))
    torch.cuda.synchronize()
    rq, rk, rv, rs = _oracle_conv(case.q, case.k, case.v, w.numpy(), case.cu_seqlens.numpy(),
                                  None if st is None else st.numpy())
    assert_close(qo, rq, "q conv")
    assert_close(ko, rk, "k conv")
    assert_close(vo, rv, "v conv")
    # the new state holds copies of inputs (or of the old state): exact
    assert np.array_equal(so.cpu().numpy().astype(np.float64), rs)


def test_conv_fwd_state_in_place(kda):
    case = workloads.make_case([5, 2, 9], H=2, dk=64, dv=64, seed=90, raw=True)
    w = _weights(2, 64, 64, seed=9)
    st = torch.randn(3, W - 1, 2, 192, generator=torch.Generator().manual_seed(4))
    ref = _oracle_conv(case.q, case.k, case.v, w.numpy(), case.cu_seqlens.numpy(), st.numpy())
    buf = st.clone().cuda()
    kda.kda_conv_fwd(case.q.cuda(), case.k.cuda(), case.v.cuda(), w.cuda(), cu_seqlens=case.cu_seqlens.cuda(),
                     conv_state_in=buf, conv_state_out=buf)
    torch.cuda.synchronize()
    assert np.array_equal(buf.cpu().numpy().astype(np.float64), ref[3])


@pytest.mark.parametrize("prep", [ALL, 0])
def test_prefill_then_fused_decode_match_oracle(kda, prep):
    """Raw projections of one 150-token sequence per head pair: the first 130 through
    kda_conv_fwd + kda_chunk_fwd_prep, the last 20 through kda_decode_step_conv (one
    token per call); o and both states against the oracle's convolution, preprocessing
    and recurrence over the whole sequence."""
    H, dk, dv, L, P = 2, 128, 128, 150, 130
    case = workloads.make_case([L], H=H, dk=dk, dv=dv, seed=91, raw=True, init=True, q_scale=False,
                               scale=dk ** -0.5)
    if not prep:  # without the flags the inputs must already be valid (unit k, log-gates, beta in (0, 1))
        case.g = torch.nn.functional.logsigmoid(case.g.float()).to(case.g.dtype)
        case.beta = torch.sigmoid(case.beta.float()).to(case.beta.dtype)
        case.q, case.k, case.v = (t * 0.3 for t in (case.q, case.k, case.v))
    w = _weights(H, dk, dv, seed=11)
    # oracle over the whole sequence
    rq, rk, rv, rs = _oracle_conv(case.q, case.k, case.v, w.numpy(), np.array([0, L]), None)
    o_ref, fs_ref = oracle.forward(rq, rk, rv, case.g, case.beta, np.array([0, L]), case.init_state,
                                   scale=case.scale, prep_flags=prep, prep_eps=EPS)
    d = {n: getattr(case, n).cuda() for n in ("q", "k", "v", "g", "beta")}
    sl = slice(0, P)
    qo, ko, vo, cstate = kda.kda_conv_fwd(d["q"][sl], d["k"][sl], d["v"][sl], w.cuda())
    o_p, state = kda.kda_chunk_fwd_prep(qo, ko, vo, d["g"][sl], d["beta"][sl], prep, EPS,
                                        init_state=case.init_state.cuda(), scale=case.scale)
    outs = [o_p]
    for t in range(P, L):
        ts = slice(t, t + 1)
        outs.append(kda.kda_decode_step_conv(d["q"][ts], d["k"][ts], d["v"][ts], d["g"][ts], d["beta"][ts], state,
                                             w.cuda(), cstate, prep, EPS, scale=case.scale))
    torch.cuda.synchronize()
    assert_close(torch.cat(outs), o_ref, "o (prefill + fused decode)")
    assert_close(state, fs_ref, "final state")
    x = np.concatenate([np.asarray(t.float()) for t in (case.q, case.k, case.v)], axis=-1)
    assert np.array_equal(cstate.cpu().numpy().astype(np.float64)[0], x[L - (W - 1):])


def test_replay_conv_matches_oracle_and_decode_bits(kda):
    """Accepted tokens replayed onto committed recurrent and convolution states equal the
    oracle, and bit for bit the same tokens applied by fused decode steps."""
    H, dk, dv = 2, 128, 128
    acc = [1, 4, 0, 3]
    N, A = len(acc), sum(acc)
    q, k, v, g, b = workloads.make_decode_tokens(A, H, dk, dv, torch.bfloat16, seed=92, raw=True)
    w = _weights(H, dk, dv, seed=12)
    gen = torch.Generator().manual_seed(6)
    pool = torch.randn(N, H, dk, dv, generator=gen) * 0.1
    cpool = torch.randn(N, W - 1, H, 2 * dk + dv, generator=gen)
    cu = np.concatenate([[0], np.cumsum(acc)]).astype(np.int64)
    # oracle: convolution from each committed state, then the recurrence
    rq, rk, rv, rs = _oracle_conv(q, k, v, w.numpy(), cu, cpool.numpy())
    ref_pool = oracle.replay(rk, rv, g, b, cu, pool, prep_flags=ALL, prep_eps=EPS)
    p1, c1 = pool.clone().cuda(), cpool.clone().cuda()
    kda.kda_replay_conv(p1, q.cuda(), k.cuda(), v.cuda(), g.cuda(), b.cuda(),
                        torch.tensor(cu, dtype=torch.int32, device="cuda"), w.cuda(), c1, ALL, EPS)
    torch.cuda.synchronize()
    assert_close(p1, ref_pool, "replay pool")
    assert np.array_equal(c1.cpu().numpy().astype(np.float64), rs)
    # the same tokens as decode steps, sequence by sequence (slot = sequence)
    p2, c2 = pool.clone().cuda(), cpool.clone().cuda()
    for n in range(N):
        for t in range(cu[n], cu[n + 1]):
            ts = slice(t, t + 1)
            kda.kda_decode_step_conv(q[ts].cuda(), k[ts].cuda(), v[ts].cuda(), g[ts].cuda(), b[ts].cuda(), p2,
                                     w.cuda(), c2, ALL, EPS,
                                     slots=torch.tensor([n], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(_bits(p2), _bits(p1))
    assert torch.equal(_bits(c2), _bits(c1))
