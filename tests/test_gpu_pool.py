"""State-pool operations (fork / offload / restore), called through the C ABI.

Copies are exact, so every check is bit-for-bit: forked slots equal their
sources, an offload / restore round trip returns the same bits, out-of-range
slots are reported and skipped, and a forked branch continues exactly like its
source under the same decode token.
"""
import pytest
import torch

import workloads
from tests._helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    import gated_linear_attention_chunk_gb300 as m
    return m


def _pool(S, H, d, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(S, H, d, d, generator=g) * 0.02).cuda()


@pytest.mark.parametrize("d", [128, 64])
def test_fork_copies_exactly(kda, d):
    pool = _pool(16, 4, d, seed=1)
    before = pool.clone()
    src = torch.tensor([3, 5, 5, 7], dtype=torch.int32, device="cuda")
    dst = torch.tensor([10, 11, 12, 7], dtype=torch.int32, device="cuda")  # 7 -> 7: onto itself
    ws = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, "cuda")
    kda.kda_state_fork(pool, src, dst, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    for s, t in [(3, 10), (5, 11), (5, 12), (7, 7)]:
        assert torch.equal(pool[t], before[s])
    untouched = [i for i in range(16) if i not in (10, 11, 12)]
    assert torch.equal(pool[untouched], before[untouched])


def test_offload_restore_round_trip(kda):
    pool = _pool(12, 4, 128, seed=2)
    before = pool.clone()
    slots = torch.tensor([7, 2, 9], dtype=torch.int32, device="cuda")
    host = torch.empty(3, 4, 128, 128, dtype=torch.float32).pin_memory()
    ws = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, "cuda")
    kda.kda_state_offload(pool, slots, host, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK  # synchronizes the stream
    for i, s in enumerate([7, 2, 9]):
        assert torch.equal(host[i], before[s].cpu())
    pool.zero_()
    back = torch.tensor([0, 1, 11], dtype=torch.int32, device="cuda")
    kda.kda_state_restore(pool, back, host, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    for i, s in enumerate([0, 1, 11]):
        assert torch.equal(pool[s], before[[7, 2, 9][i]])
    assert int(torch.count_nonzero(pool[[3, 4, 5, 6, 7, 8, 9, 10]])) == 0
    # slots None: slot i <-> host row i
    host2 = torch.empty(2, 4, 128, 128, dtype=torch.float32).pin_memory()
    kda.kda_state_offload(pool, None, host2, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_OK
    assert torch.equal(host2[0], before[7].cpu()) and torch.equal(host2[1], before[2].cpu())


def test_bad_slot_is_reported_and_skipped(kda):
    pool = _pool(8, 2, 128, seed=3)
    before = pool.clone()
    src = torch.tensor([1, 99], dtype=torch.int32, device="cuda")
    dst = torch.tensor([2, 3], dtype=torch.int32, device="cuda")
    ws = kda.new_workspace(kda.KDA_WS_HEADER_BYTES, "cuda")
    kda.kda_state_fork(pool, src, dst, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SLOT
    assert torch.equal(pool[2], before[1])          # the valid item ran
    assert torch.equal(pool[3], before[3])          # the invalid one wrote nothing
    host = torch.empty(1, 2, 128, 128, dtype=torch.float32).pin_memory()
    kda.kda_state_restore(pool, torch.tensor([-1], dtype=torch.int32, device="cuda"), host, workspace=ws)
    assert kda.kda_device_status(ws) == kda.KDA_ERR_BAD_SLOT


def test_unpinned_host_buffer_is_refused(kda):
    pool = _pool(4, 2, 128, seed=4)
    host = torch.empty(1, 2, 128, 128, dtype=torch.float32)  # pageable
    with pytest.raises(ValueError):
        kda.kda_state_offload(pool, None, host)


def test_forked_branch_continues_like_its_source(kda):
    """Fork a committed state, then decode the same token on both: identical bits."""
    H, d = 4, 128
    pool = _pool(6, H, d, seed=5)
    kda.kda_state_fork(pool, torch.tensor([1], dtype=torch.int32, device="cuda"),
                       torch.tensor([4], dtype=torch.int32, device="cuda"))
    q, k, v, g, b = (x.cuda() for x in workloads.make_decode_tokens(1, H, d, d, torch.bfloat16, seed=6))
    q2, k2, v2, g2, b2 = (torch.cat([x, x]) for x in (q, k, v, g, b))
    slots = torch.tensor([1, 4], dtype=torch.int32, device="cuda")
    o = kda.kda_decode_step(q2, k2, v2, g2, b2, pool, slots=slots)
    torch.cuda.synchronize()
    assert torch.equal(o[0], o[1])
    assert torch.equal(pool[1], pool[4])
