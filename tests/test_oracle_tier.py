"""Pins of the expert tier's oracle (oracle_tier_step), CPU only.

The rules it restates: "Distributed MoE" (tenzro docs), expert-residency
paragraph (a bounded tier with least-recently-used eviction; the experts a
routing decision selected are read ahead before the forward); "Module
expert_store" (ferrox-core docs), design list (a leased entry is never
evicted; a request that does not fit is still served, at the cost of more
transfers).  Each pin below is fixed by something outside the oracle: a
textbook result, a library-backed brute force, or a closed form.
"""
from collections import OrderedDict

import numpy as np
import pytest

import oracle

# The reference string of the classic page-replacement example (Silberschatz,
# Galvin and Gagne, "Operating System Concepts", chapter on virtual memory):
# with three frames, LRU replacement takes 12 page faults.
TEXTBOOK_REFS = [7, 0, 1, 2, 0, 3, 0, 4, 2, 3, 0, 3, 2, 1, 2, 0, 1, 7, 0, 1]


def test_textbook_lru_fault_count():
    o = oracle.TierOracle(3, 8)
    for e in TEXTBOOK_REFS:
        o.step([e])
    st = o.stats()
    assert st["misses"] == 12 and st["hits"] == 8
    assert st["evictions"] == 12 - 3 and st["extra_passes"] == 0
    # the last three distinct pages used stay resident: 1, 0, 7
    assert sorted(int(e) for e in o.holder) == [0, 1, 7]


def _lru_brute(n_slots, refs):
    """Single-expert steps through an OrderedDict LRU (most recent last)."""
    cache, misses, order = OrderedDict(), 0, []
    for e in refs:
        if e in cache:
            cache.move_to_end(e)
        else:
            misses += 1
            if len(cache) == n_slots:
                cache.popitem(last=False)
            cache[e] = True
        order.append(sorted(cache))
    return misses, order


@pytest.mark.parametrize("n_slots,n_experts,seed", [(1, 4, 0), (2, 6, 1), (4, 12, 2), (7, 9, 3),
                                                    (16, 40, 4)])
def test_single_expert_steps_match_a_plain_lru(n_slots, n_experts, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, n_experts + 1) ** 1.2
    refs = rng.choice(n_experts, size=300, p=p / p.sum()).tolist()
    misses, order = _lru_brute(n_slots, refs)
    o = oracle.TierOracle(n_slots, n_experts)
    for i, e in enumerate(refs):
        o.step([e])
        assert sorted(int(h) for h in o.holder if h >= 0) == order[i]
    assert o.stats()["misses"] == misses


def test_a_leased_slot_is_never_evicted():
    o = oracle.TierOracle(3, 10)
    o.step([0, 1, 2])            # slots 0, 1, 2 (0 and 1 are the least recently used)
    o.step([2])
    slot, load, pas, npass = o.step([0, 1, 5])
    # 0 and 1 are hits and leased by this step; only expert 2's slot may go
    assert npass == 1 and load.tolist() == [0, 0, 1] and slot.tolist() == [0, 1, 2]
    assert o.slot_of(2) == -1 and o.slot_of(5) == 2


def test_least_recently_used_goes_first_and_empty_slots_before_any():
    o = oracle.TierOracle(4, 10)
    o.step([3])
    o.step([1])
    o.step([4])                  # slots 0:3 1:1 2:4, slot 3 empty
    slot, load, _, _ = o.step([9])
    assert slot.tolist() == [3] and load.tolist() == [1]     # the empty slot
    slot, _, _, _ = o.step([8])
    assert slot.tolist() == [0] and o.slot_of(3) == -1        # then the oldest (expert 3)
    o.step([1])
    slot, _, _, _ = o.step([7])
    assert slot.tolist() == [2] and o.slot_of(4) == -1        # 4 is older than 9, 8, 1


def test_one_slot_means_one_pass_per_expert():
    o = oracle.TierOracle(1, 6)
    slot, load, pas, npass = o.step([5, 2, 0, 3])
    assert npass == 4 and pas.tolist() == [0, 1, 2, 3]
    assert slot.tolist() == [0, 0, 0, 0] and load.tolist() == [1, 1, 1, 1]
    assert o.stats()["extra_passes"] == 3
    slot, load, pas, npass = o.step([4, 3])     # 3 stayed: served first, as a hit
    assert load.tolist() == [1, 0] and pas.tolist() == [1, 0] and npass == 2


@pytest.mark.parametrize("n_slots,n_experts,seed", [(3, 20, 5), (8, 64, 6), (5, 5, 7)])
def test_pass_count_and_conservation(n_slots, n_experts, seed):
    """Passes = ceil(requested / slots); within a pass the slots are distinct;
    hits + misses = requests; loads = misses."""
    rng = np.random.default_rng(seed)
    o = oracle.TierOracle(n_slots, n_experts)
    total = 0
    for _ in range(80):
        n = int(rng.integers(0, n_experts + 1))
        req = rng.choice(n_experts, size=n, replace=False)
        slot, load, pas, npass = o.step(req)
        total += n
        assert npass == -(-n // n_slots)
        for p in range(npass):
            s = slot[pas == p]
            assert len(s) > 0 and len(set(s.tolist())) == len(s)
        assert (pas >= 0).all() and (slot >= 0).all() and (slot < n_slots).all()
        # the last pass's experts are resident afterwards
        for e, s, p in zip(req, slot, pas):
            if p == npass - 1:
                assert o.slot_of(int(e)) == int(s)
    st = o.stats()
    assert st["hits"] + st["misses"] == total


def test_bad_requests_are_refused_and_change_nothing():
    o = oracle.TierOracle(3, 6)
    o.step([1, 2])
    before = (o.holder.copy(), o.last_use.copy(), o.clock.copy(), o.counters.copy())
    for bad in ([1, 1], [0, 6], [-1], [5, 2, 5]):
        with pytest.raises(RuntimeError):
            o.step(bad)
    after = (o.holder, o.last_use, o.clock, o.counters)
    assert all(np.array_equal(a, b) for a, b in zip(before, after))
    assert o.step([])[3] == 0
