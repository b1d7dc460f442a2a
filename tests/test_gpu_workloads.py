"""GPU parity at the benchmark workloads' full sizes, in the launch configuration the
benchmark times, checked against the fp64 oracle on sampled (sequence, head) chains
(each chain is an independent recurrence, so a sampled chain is checked exactly),
plus multi-chunk edge cases of the chunked tensor-core path."""
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


def _chain_oracle(case, n, h):
    """fp64 oracle for one (sequence, head) chain of a packed case."""
    return _chains_oracle(case, [(n, h)])[(n, h)]


def _chains_oracle(case, chains, threads=8):
    """fp64 oracle for several (sequence, head) chains in one call: each chain becomes a
    sequence of a one-head packed batch, so the oracle runs them on parallel threads."""
    cu = case.cu_seqlens.tolist()
    parts = {name: [] for name in ("q", "k", "v", "g", "beta")}
    bounds, s0 = [0], []
    for n, h in chains:
        b, e = int(cu[n]), int(cu[n + 1])
        for name in parts:
            t = getattr(case, name)
            parts[name].append(t[b:e, h:h + 1])
        bounds.append(bounds[-1] + e - b)
        if case.init_state is not None:
            s0.append(case.init_state[n:n + 1, h:h + 1])
    cat = {name: torch.cat(x) for name, x in parts.items()}
    o, fs = oracle.forward(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"], np.array(bounds),
                           torch.cat(s0) if s0 else None, scale=case.scale, threads=threads)
    return {c: (o[bounds[i]:bounds[i + 1], 0], fs[i, 0]) for i, c in enumerate(chains)}


def _check_chains(case, o, fs, chains, tag):
    refs = _chains_oracle(case, chains)
    for n, h in chains:
        o_ref, fs_ref = refs[(n, h)]
        b, e = int(case.cu_seqlens[n]), int(case.cu_seqlens[n + 1])
        assert_close(o[b:e, h].float().cpu(), o_ref, f"{tag} o chain ({n},{h})")
        assert_close(fs[n, h].cpu(), fs_ref, f"{tag} final_state chain ({n},{h})")


def _run(kda, case):
    """kda_chunk_fwd with the full workspace, as the benchmark calls it."""
    d = to_dev(case)
    ws = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(case.N, case.T_total, case.H, case.dk, case.dv),
                           "cuda")
    o, fs = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                              init_state=d["init_state"], scale=case.scale, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    return o, fs


def test_tensor_core_path_is_used(kda):
    assert kda.kda_chunk_fwd_uses_tensor_cores(128, 128, torch.bfloat16)


@pytest.mark.parametrize("lengths", [[1024, 700, 64, 191, 5], [4096], [128, 129, 127, 63, 65]])
def test_multi_chunk_varlen(kda, lengths):
    case = workloads.make_case(lengths, H=4, dk=128, dv=128, seed=sum(lengths) % 1000)
    o, fs = _run(kda, case)
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


@pytest.mark.parametrize("lengths", [
    [4] * 17 + [64] + [4] * 10 + [130, 70] + [4] * 9 + [200],   # verify-like: few full chunks among short sequences
    [64, 0, 64] + [0] * 48 + [64],                              # exactly floor(T / 64) sequences with a full chunk
    [3] * 60,                                                   # no full chunk at all (T >= 64)
    [1] * 50,                                                   # T < 64
])
def test_many_short_sequences_launch_only_needed_ctas(kda, lengths):
    """With more chains than one wave the sequences are ordered longest first and chunked CTAs are
    launched only for the first floor(T / 64) ranks; every sequence still matches the oracle."""
    case = workloads.make_case(lengths, H=4, dk=128, dv=128, seed=len(lengths))
    assert case.N * case.H > 152
    o, fs = _run(kda, case)
    o_ref, fs_ref = oracle.forward(case.q, case.k, case.v, case.g, case.beta, case.cu_seqlens, case.init_state,
                                   threads=0)
    assert_close(o, o_ref, "o")
    assert_close(fs, fs_ref, "final_state")


def test_prefill_4k_full_size_sampled(kda):
    """Eight chains of the 4 x 4096 benchmark batch, the first and the last (sequence, head) among them."""
    case = workloads.named_case("prefill_4k")
    o, fs = _run(kda, case)
    assert torch.isfinite(o.float()).all() and torch.isfinite(fs).all()
    _check_chains(case, o, fs, [(0, 0), (0, 31), (1, 7), (1, 16), (2, 19), (2, 2), (3, 0), (3, 31)], "prefill_4k")


def test_prefill_4k_fp32_full_size_sampled(kda):
    """The 4 x 4096 batch with fp32 inputs (token-sequential kernel), four chains checked."""
    case = workloads.named_case("prefill_4k_fp32")
    assert not kda.kda_chunk_fwd_uses_tensor_cores(case.dk, case.dv, case.q.dtype)
    o, fs = _run(kda, case)
    _check_chains(case, o, fs, [(0, 0), (1, 13), (2, 22), (3, 31)], "prefill_4k_fp32")


def test_varlen_64_full_size_sampled(kda):
    case = workloads.named_case("varlen_64")
    o, fs = _run(kda, case)
    lens = np.diff(case.cu_seqlens.numpy())
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    _check_chains(case, o, fs, [(longest, 3), (longest, 31), (shortest, 30), (17, 12), (0, 0), (63, 31)],
                  "varlen_64")


def test_long_128k_full_size_sampled(kda):
    """Eight of the 32 chains of 131072 tokens (T-segment split path), head 31 among them."""
    case = workloads.named_case("long_128k")
    o, fs = _run(kda, case)
    _check_chains(case, o, fs, [(0, h) for h in (0, 5, 9, 14, 21, 26, 30, 31)], "long_128k")


def test_spec_rollout_committed_states(kda):
    """The rollout workload in full: a 2048-token prefill of 128 sequences, then 64 x (4-token
    verify from the committed states + replay of the accepted prefix, U{1..4} tokens).  Verify
    outputs and committed states are checked against the oracle on sampled chains at every step."""
    steps = 64
    case = workloads.named_case("spec_rollout")
    d = to_dev(case)
    N, H, dk, dv = case.N, case.H, case.dk, case.dv
    pool = torch.zeros(N, H, dk, dv, dtype=torch.float32, device="cuda")
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"], final_state=pool)
    acc = workloads.make_accept_lengths(steps, N, 4, seed=404)
    sample = [(0, 0), (31, 31), (57, 13), (64, 1), (100, 22), (127, 31)]
    prefill_refs = _chains_oracle(case, sample)
    ref = {c: prefill_refs[c][1] for c in sample}
    for c in sample:
        assert_close(pool[c[0], c[1]].cpu(), ref[c], f"spec_rollout prefill state chain {c}")
    cu4 = torch.arange(0, 4 * N + 1, 4, dtype=torch.int32, device="cuda")
    ws_v = kda.new_workspace(kda.kda_chunk_fwd_workspace_size(N, 4 * N, H, dk, dv), "cuda")
    for s in range(steps):
        q, k, v, g, b = (t.cuda() for t in workloads.make_decode_tokens(4 * N, H, dk, dv, torch.bfloat16,
                                                                         seed=1000 + s))
        o_v, _ = kda.kda_chunk_fwd(q, k, v, g, b, cu_seqlens=cu4, init_state=pool, output_final_state=False,
                                   workspace=ws_v)
        a = acc[s]
        sel = torch.cat([torch.arange(4 * i, 4 * i + int(a[i])) for i in range(N)]).cuda()
        cu_a = torch.zeros(N + 1, dtype=torch.int32)
        cu_a[1:] = torch.cumsum(a, 0)
        kda.kda_replay(pool, k[sel].contiguous(), v[sel].contiguous(), g[sel].contiguous(), b[sel].contiguous(),
                       cu_a.cuda())
        torch.cuda.synchronize()
        for n, h in sample:
            sl = slice(4 * n, 4 * n + 4)
            pk = lambda x: x[sl, h:h + 1].cpu()
            o_ref, _ = oracle.forward(pk(q), pk(k), pk(v), pk(g), b[sl, h:h + 1].cpu(), np.array([0, 4]),
                                      ref[(n, h)][None, None])
            assert_close(o_v[sl, h].float().cpu(), o_ref[:, 0], f"spec_rollout verify o step {s} chain ({n},{h})")
            na = int(a[n])
            _, fs = oracle.forward(None, pk(k)[:na], pk(v)[:na], pk(g)[:na], b[sl, h:h + 1].cpu()[:na],
                                   np.array([0, na]), ref[(n, h)][None, None], want_o=False)
            ref[(n, h)] = fs[0, 0]
            assert_close(pool[n, h].cpu(), ref[(n, h)], f"spec_rollout committed state step {s} chain ({n},{h})")


def test_gate_range_violation_is_reported(kda):
    """A chunk whose cumulative decay leaves the supported range sets KDA_ERR_GATE_RANGE
    (no NaN-producing silent result, no fault)."""
    case = workloads.make_case([192], H=2, dk=128, dv=128, seed=77)
    g = case.g.clone()
    g[64:128, 1, 5] = -3.0   # 64 tokens x 3 = 192 nats > 100 ln 2 in one chunk, channel 5 of head 1
    d = to_dev(case)
    ws = kda.new_workspace(256, "cuda")
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], g.cuda(), d["beta"], cu_seqlens=d["cu_seqlens"],
                      init_state=d["init_state"], workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_GATE_RANGE
    # the library stays usable afterwards
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                      init_state=d["init_state"], workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
