"""GPU parity of kda_chunk_bwd (the backward of the packed prefill) against the fp64
oracle's reverse mode, through the C ABI.

Tolerance: the gradients are accumulated in fp32 and stored in the input dtype, so
besides the relative L2 bound of the forward (5e-3) the max-abs bound is taken
relative to each tensor's largest reference entry (1e-2 of it; bf16 storage alone
costs up to 2^-9 of an entry)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_close, ensure_built, to_dev

pytestmark = pytest.mark.gpu

REL = 5e-3
MAB_REL = 1e-2


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    return m


def _grads_out(case, seed, with_final=True, dtype=None):
    gen = torch.Generator().manual_seed(seed)
    dtype = dtype or case.q.dtype
    T, H, dv = case.T_total, case.H, case.dv
    d_o = torch.randn(T, H, dv, generator=gen).to(dtype)
    d_fin = (torch.randn(case.N, H, case.dk, dv, generator=gen) * 0.1) if with_final else None
    return d_o, d_fin


def _check(out, ref, what=""):
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        r = ref[key]
        assert_close(out[key], r, f"{key}{what}", rel=REL, mab=MAB_REL * max(1.0, float(np.abs(r).max())))
    if out["d_init"] is not None:
        r = ref["d_init"]
        assert_close(out["d_init"], r, f"d_init{what}", rel=REL, mab=MAB_REL * max(1.0, float(np.abs(r).max())))


def _run(kda, case, d_o, d_fin, **kw):
    d = to_dev(case)
    out = kda.kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o.cuda(), cu_seqlens=d["cu_seqlens"],
                            init_state=d["init_state"], d_final_state=None if d_fin is None else d_fin.cuda(),
                            scale=case.scale, **kw)
    torch.cuda.synchronize()
    return out


def _oracle(case, d_o, d_fin):
    return oracle.backward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state, d_o,
                           d_fin, scale=case.scale, threads=0)


LENGTHS = [1, 63, 64, 65, 130, 0, 200, 128, 7]


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bwd_varlen_matches_oracle(kda, dk, dv, dtype):
    case = workloads.make_case(LENGTHS, H=2, dk=dk, dv=dv, dtype=dtype, seed=70 + dk + dv)
    d_o, d_fin = _grads_out(case, seed=1)
    out = _run(kda, case, d_o, d_fin)
    _check(out, _oracle(case, d_o, d_fin), f" ({dk}x{dv} {dtype})")


def test_bwd_without_initial_state_or_final_gradient(kda):
    case = workloads.make_case([150, 64, 3], H=2, dk=128, dv=128, init=False, seed=71)
    d_o, _ = _grads_out(case, seed=2, with_final=False)
    out = _run(kda, case, d_o, None)
    _check(out, _oracle(case, d_o, None))


def test_bwd_raw_query_with_scale(kda):
    case = workloads.make_case([130, 70], H=2, dk=128, dv=128, q_scale=False, scale=128 ** -0.5, seed=72)
    d_o, d_fin = _grads_out(case, seed=3)
    out = _run(kda, case, d_o, d_fin)
    _check(out, _oracle(case, d_o, d_fin))


def test_bwd_single_sequence_without_cu_seqlens(kda):
    case = workloads.make_case([200], H=2, dk=64, dv=64, seed=73)
    d_o, d_fin = _grads_out(case, seed=4)
    d = to_dev(case)
    out = kda.kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o.cuda(), cu_seqlens=None,
                            init_state=d["init_state"], d_final_state=d_fin.cuda(), scale=case.scale)
    torch.cuda.synchronize()
    _check(out, _oracle(case, d_o, d_fin))


def test_bwd_empty_sequence_passes_final_gradient_through(kda):
    case = workloads.make_case([0, 5, 0], H=2, dk=128, dv=128, seed=74)
    d_o, d_fin = _grads_out(case, seed=5)
    out = _run(kda, case, d_o, d_fin)
    assert torch.equal(out["d_init"][0].cpu(), d_fin[0]) and torch.equal(out["d_init"][2].cpu(), d_fin[2])
    _check(out, _oracle(case, d_o, d_fin))


def test_bwd_full_size_prefill_4k_sampled_heads(kda):
    """The 4 x 4096-token, 32-head workload through one call; the oracle checks two
    heads of the first and of the last sequence (heads are independent chains)."""
    case = workloads.named_case("prefill_4k")
    d_o, d_fin = _grads_out(case, seed=6)
    out = _run(kda, case, d_o, d_fin)
    cu = case.cu_seqlens.tolist()
    for n, heads in ((0, slice(0, 2)), (3, slice(30, 32))):
        ts = slice(cu[n], cu[n + 1])
        sub = dict(q=case.q[ts, heads], k=case.k[ts, heads], v=case.v[ts, heads], g=case.g[ts, heads],
                   beta=case.beta[ts, heads])
        ref = oracle.backward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], np.array([0, cu[n + 1] - cu[n]]),
                              case.init_state[n:n + 1, heads], d_o[ts, heads], d_fin[n:n + 1, heads],
                              scale=case.scale, threads=2)
        got = {key: out[key][ts, heads] for key in ("dq", "dk", "dv", "dg", "dbeta")}
        got["d_init"] = out["d_init"][n:n + 1, heads]
        _check(got, ref, f" (sequence {n})")


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, torch.bfloat16), (64, 64, torch.bfloat16), (64, 64, torch.float32)])
def test_bwd_prep_matches_oracle(kda, dk, dv, dtype):
    """Raw inputs with every preprocessing flag: the gradients with respect to the raw
    q, k, gate and beta logits (and v, the initial state) equal the oracle's."""
    case = workloads.make_case(LENGTHS, H=2, dk=dk, dv=dv, dtype=dtype, seed=76 + dk, raw=True, q_scale=False,
                               scale=dk ** -0.5)
    d_o, d_fin = _grads_out(case, seed=7)
    d = to_dev(case)
    out = kda.kda_chunk_bwd_prep(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o.cuda(), 15, 1e-6,
                                 cu_seqlens=d["cu_seqlens"], init_state=d["init_state"],
                                 d_final_state=d_fin.cuda(), scale=case.scale)
    torch.cuda.synchronize()
    ref = oracle.backward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state, d_o, d_fin,
                          scale=case.scale, threads=0, prep_flags=15, prep_eps=1e-6)
    _check(out, ref, f" (prep, {dk}x{dv} {dtype})")


def test_bwd_prep_zero_is_the_plain_call(kda):
    case = workloads.make_case([150, 64, 9], H=2, dk=128, dv=128, seed=77)
    d_o, d_fin = _grads_out(case, seed=8)
    d = to_dev(case)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d_o.cuda())
    kw = dict(cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], d_final_state=d_fin.cuda())
    a = kda.kda_chunk_bwd(*args, **kw)
    b = kda.kda_chunk_bwd_prep(*args, 0, 0.0, **kw)
    torch.cuda.synchronize()
    for key in ("dq", "dk", "dv", "dg", "dbeta", "d_init"):
        assert torch.equal(a[key], b[key]), key


def test_bwd_strong_decay_reports_gate_range(kda):
    """A chunk whose decay leaves the chunked form's range: the backward has no token-by-token
    fallback, so it reports KDA_ERR_GATE_RANGE through the device status (and returns)."""
    case = workloads.make_case([300, 130], H=2, dk=128, dv=128, seed=88)
    g = case.g.clone()
    g[70:134, 1, :] = -3.0  # a whole chunk of sequence 0, head 1: decay e^-192
    d_o, d_fin = _grads_out(case, seed=9)
    d = to_dev(case)
    ws = kda.new_workspace(kda.kda_chunk_bwd_workspace_size(case.N, case.T_total, case.H, case.dk, case.dv), "cuda")
    kda.kda_chunk_bwd(d["q"], d["k"], d["v"], g.cuda(), d["beta"], d_o.cuda(), cu_seqlens=d["cu_seqlens"],
                      init_state=d["init_state"], d_final_state=d_fin.cuda(), scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_GATE_RANGE
    # the same call on in-range gates is clean with the same workspace
    kda.kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d_o.cuda(), cu_seqlens=d["cu_seqlens"],
                      init_state=d["init_state"], d_final_state=d_fin.cuda(), scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
