"""Host logic of HostPrefill (CPU): the sequence groups cover every sequence once, in order,
none is empty, and their token counts are close to equal where the lengths allow it; the
pieces cover every token once, in order, and cut a sequence only at multiples of 64 tokens
from its start."""
import random

from gated_linear_attention_chunk_gb300.host_pipeline import plan_groups, plan_pieces


def _cu(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


def _check_cover(groups, N):
    assert groups[0][0] == 0 and groups[-1][1] == N
    for (a, b), (c, d) in zip(groups, groups[1:]):
        assert b == c
    assert all(b > a for a, b in groups)


def test_groups_cover_every_sequence_once():
    rng = random.Random(3)
    for _ in range(200):
        N = rng.randint(1, 40)
        lengths = [rng.choice([0, 1, 5, 64, 300, 4096]) for _ in range(N)]
        for g in (1, 2, 3, 4, 7, 64):
            groups = plan_groups(_cu(lengths), g)
            assert 1 <= len(groups) <= min(g, N)
            _check_cover(groups, N)


def test_equal_lengths_split_evenly():
    groups = plan_groups(_cu([4096] * 8), 4)
    assert groups == [(0, 2), (2, 4), (4, 6), (6, 8)]


def test_token_balance_within_one_sequence():
    """Each boundary lands within one sequence length of its ideal token offset."""
    rng = random.Random(5)
    lengths = [rng.randint(1000, 20000) for _ in range(64)]
    cu = _cu(lengths)
    groups = plan_groups(cu, 4)
    assert len(groups) == 4
    for i, (a, _) in enumerate(groups[1:], start=1):
        assert abs(cu[a] - cu[-1] * i / 4) <= max(lengths)


def test_more_groups_than_sequences():
    assert plan_groups(_cu([10, 20]), 5) == [(0, 1), (1, 2)]
    assert plan_groups(_cu([0]), 3) == [(0, 1)]


def _check_pieces(pieces, cu):
    N = len(cu) - 1
    assert pieces[0][2] == cu[0] and pieces[-1][3] == cu[N]
    for (a, b, t0, t1), (c, d, u0, u1) in zip(pieces, pieces[1:]):
        assert t1 == u0 and c in (b, a)  # the next piece starts where this one ends
    for a, b, t0, t1 in pieces:
        assert cu[a] <= t0 <= t1 <= cu[b]
        if (t0, t1) != (cu[a], cu[b]):  # a part of one sequence
            assert b == a + 1 and t1 > t0
            assert (t0 - cu[a]) % 64 == 0  # every part but the last holds whole chunks
            assert t1 == cu[b] or (t1 - cu[a]) % 64 == 0
    # every sequence is covered: whole, or by consecutive parts from its start to its end
    covered = {}
    for a, b, t0, t1 in pieces:
        for n in range(a, b):
            covered.setdefault(n, []).append((max(t0, cu[n]), min(t1, cu[n + 1])))
    for n in range(N):
        spans = covered[n]
        assert spans[0][0] == cu[n] and spans[-1][1] == cu[n + 1]
        assert all(x[1] == y[0] for x, y in zip(spans, spans[1:]))


def test_pieces_cover_every_token_once():
    rng = random.Random(7)
    for _ in range(200):
        N = rng.randint(1, 12)
        lengths = [rng.choice([0, 1, 5, 64, 65, 300, 1000, 4096, 9000]) for _ in range(N)]
        for g in (1, 2, 3, 4, 9, 16, 64):
            _check_pieces(plan_pieces(_cu(lengths), g), _cu(lengths))


def test_long_sequences_are_cut_into_whole_chunks():
    pieces = plan_pieces(_cu([4096] * 4), 16)
    assert len(pieces) == 16
    assert all(t1 - t0 == 1024 for _, _, t0, t1 in pieces)
    assert plan_pieces(_cu([300, 64, 1000, 5, 129]), 1) == [(0, 5, 0, 1498)]
    pieces = plan_pieces(_cu([100, 100, 100, 4000]), 4)
    assert [p[:2] for p in pieces[:3]] == [(0, 1), (1, 2), (2, 3)] and len(pieces) > 4
