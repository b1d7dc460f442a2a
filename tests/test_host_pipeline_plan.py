"""Host logic of HostPrefill (CPU): the sequence groups cover every sequence once, in order,
none is empty, and their token counts are close to equal where the lengths allow it."""
import random

from gated_linear_attention_chunk_gb300.host_pipeline import plan_groups


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
