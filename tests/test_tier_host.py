"""The expert tier's residency logic (moe_slot_cache_*), host only, against the
oracle's restatement of its rules (oracle_tier_step) and hand-built traces.

The policy under test ("Distributed MoE" (tenzro docs), expert-residency
paragraph: a bounded least-recently-used tier with readahead of the experts
the routing decision selected; "Module expert_store" (ferrox-core docs),
design list: leased entries are never evicted, and a step whose experts do not
fit still succeeds): hits first, pinned for pass 0; a miss takes the lowest
free slot, else the least recently used slot not pinned by the current pass
(lowest index on ties); when every slot is pinned a new pass starts and the
pins are dropped.
"""
import numpy as np
import pytest

import oracle
from expert_dispatch_gb300 import moe


def test_create_rejects_bad_sizes():
    for n_slots, n_exp in ((0, 4), (5, 4), (1, 0), (-1, 3)):
        with pytest.raises(moe.MoeError) as ei:
            moe.SlotCache(n_slots, n_exp)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG


def test_first_use_misses_then_hits():
    c = moe.SlotCache(4, 10)
    slot, load, pas, npass = c.assign([3, 1, 4])
    assert list(load) == [1, 1, 1] and list(pas) == [0, 0, 0] and npass == 1
    assert list(slot) == [0, 1, 2]  # lowest free slots, in request order
    slot2, load2, pas2, npass2 = c.assign([1, 5])
    assert list(slot2) == [1, 3] and list(load2) == [0, 1] and npass2 == 1
    st = c.stats()
    assert (st["steps"], st["hits"], st["misses"], st["evictions"]) == (2, 1, 4, 0)
    assert st["resident"] == 4 and st["n_slots"] == 4 and st["bytes_loaded"] == 0
    assert [c.slot_of(e) for e in (3, 1, 4, 5, 0)] == [0, 1, 2, 3, -1]


def test_least_recently_used_is_evicted():
    c = moe.SlotCache(3, 10)
    c.assign([0, 1, 2])      # slots 0, 1, 2
    c.assign([0])            # 0 used again: 1 and 2 are older
    c.assign([2])            # now 1 is the least recently used
    slot, load, _, _ = c.assign([7])
    assert slot[0] == 1 and load[0] == 1
    assert c.slot_of(1) == -1 and c.slot_of(7) == 1
    assert c.stats()["evictions"] == 1


def test_hits_of_a_step_are_never_evicted_by_its_misses():
    c = moe.SlotCache(3, 10)
    c.assign([0, 1, 2])
    slot, load, pas, npass = c.assign([0, 1, 5])   # one slot left to evict: 2's
    assert npass == 1 and list(load) == [0, 0, 1] and slot[2] == 2
    assert c.slot_of(0) == 0 and c.slot_of(1) == 1


def test_overflow_runs_in_passes_with_bounded_slots():
    c = moe.SlotCache(2, 10)
    experts = [4, 0, 9, 3, 7]
    slot, load, pas, npass = c.assign(experts)
    assert npass == 3
    assert sorted(pas.tolist()) == [0, 0, 1, 1, 2]
    for p in range(npass):  # within a pass, distinct slots
        s = slot[pas == p]
        assert len(set(s.tolist())) == len(s)
    assert all(0 <= s < 2 for s in slot) and all(load == 1)
    st = c.stats()
    assert st["extra_passes"] == 2 and st["misses"] == 5 and st["evictions"] == 3
    assert st["resident"] == 2


def test_bad_requests_leave_the_cache_unchanged():
    c = moe.SlotCache(3, 6)
    c.assign([1, 2])
    before = c.stats(), [c.slot_of(e) for e in range(6)]
    for bad in ([1, 1], [0, 6], [-1], [5, 2, 5]):
        with pytest.raises(moe.MoeError) as ei:
            c.assign(bad)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    assert (c.stats(), [c.slot_of(e) for e in range(6)]) == before
    assert c.assign([])[3] == 0


@pytest.mark.parametrize("n_slots,n_experts,seed", [(1, 5, 0), (3, 8, 1), (5, 40, 2),
                                                    (16, 64, 3), (8, 8, 4), (64, 385, 5),
                                                    (192, 385, 6)])
def test_matches_the_tier_oracle(n_slots, n_experts, seed):
    """moe_slot_cache_assign against the oracle's restatement of the tier's
    rules (oracle_tier_step), step by step: slots, loads, passes, counters and
    the resident set, bit for bit."""
    rng = np.random.default_rng(seed)
    c = moe.SlotCache(n_slots, n_experts)
    o = oracle.TierOracle(n_slots, n_experts)
    p = 1.0 / np.arange(1, n_experts + 1) ** 1.1  # skewed, so some experts recur often
    for _ in range(60):
        n = int(rng.integers(0, min(n_experts, 2 * n_slots + 3) + 1))
        experts = rng.choice(n_experts, size=n, replace=False, p=p / p.sum())
        if rng.integers(0, 2):
            experts = np.sort(experts)  # the tier's forward asks in ascending expert order
        slot, load, pas, npass = c.assign(experts.tolist())
        os_, ol, op, on = o.step(experts)
        assert np.array_equal(slot, os_) and np.array_equal(load, ol)
        assert np.array_equal(pas, op) and npass == on
        assert [c.slot_of(e) for e in range(n_experts)] == [o.slot_of(e)
                                                            for e in range(n_experts)]
    st, ost = c.stats(), o.stats()
    for key in ("steps", "hits", "misses", "evictions", "extra_passes", "resident"):
        assert st[key] == ost[key], key
