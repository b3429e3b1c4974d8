"""The expert slot cache's policy (moe_cache_*, host code of the library) on
CPU: hand-worked sequences from the rules of the pages (section "Load and
ownership": least frequently used eviction, recency breaking ties), the oracle
(oracle/cache_oracle.py) pinned by the same sequences, and the library against
the oracle on long uniform and Zipf-skewed selection streams."""
import numpy as np
import pytest

import bit_affine_quantized_gb300 as bq
from oracle.cache_oracle import SlotCache


def _lib_cache(n_layers, n_slots):
    bq.build_library()
    return bq.ExpertCache(n_layers, n_slots)


# Worked by hand from the rules (3 slots, k <= 3):
#  1 [4,7]   empty slots 0,1                          -> [0,1]  fills (0,4) (1,7)
#  2 [7,9]   7 hit (uses 2); 9 -> empty slot 2        -> [1,2]  fill (2,9)
#  3 [4,5]   4 hit (uses 2); 5: slot 2 has the fewest uses (1) -> [0,2]  fill (2,5)
#  4 [9,7]   7 hit; 9: slot 0 (uses 2) vs slot 2 (uses 1)      -> [2,1]  fill (2,9)
#  5 [1,2]   1: slots 0 (2 uses, step 3), 1 (3 uses), 2 (1 use) -> slot 2;
#            2: slots 0 (2 uses) and 1 (3 uses)                -> slot 0;  [2,0]
#  6 [7,1,2] all hits                                           -> [1,2,0]
#  7 [3]     slot 0 (2 uses, step 6), slot 1 (4 uses), slot 2 (2 uses, step 6):
#            equal uses and recency -> the lower slot 0          -> [0]
HAND = [
    ([4, 7], [0, 1], [(0, 4), (1, 7)]),
    ([7, 9], [1, 2], [(2, 9)]),
    ([4, 5], [0, 2], [(2, 5)]),
    ([9, 7], [2, 1], [(2, 9)]),
    ([1, 2], [2, 0], [(2, 1), (0, 2)]),
    ([7, 1, 2], [1, 2, 0], []),
    ([3], [0], [(0, 3)]),
]
# recency breaks a tie of uses (2 slots): 1 and 2 used once each, 1 longer ago
RECENCY = [([1], [0], [(0, 1)]), ([2], [1], [(1, 2)]), ([3], [0], [(0, 3)]), ([1], [1], [(1, 1)])]
# frequency beats recency (2 slots): 1 used twice, 2 once but more recently
FREQUENCY = [([1], [0], [(0, 1)]), ([1], [0], []), ([2], [1], [(1, 2)]), ([3], [1], [(1, 3)])]


@pytest.mark.parametrize("n_slots,seq", [(3, HAND), (2, RECENCY), (2, FREQUENCY)], ids=["hand", "recency", "frequency"])
def test_hand_worked(n_slots, seq):
    ref = SlotCache(n_slots)
    lib = _lib_cache(1, n_slots)
    for ids, want_slots, want_loads in seq:
        assert ref.step(ids) == (want_slots, want_loads), f"oracle at {ids}"
        assert lib.lookup(0, ids) == (want_slots, want_loads), f"library at {ids}"
    hits = sum(len(set(ids)) for ids, _, _ in seq) - sum(len(l) for _, _, l in seq)
    assert lib.stats(0) == (hits, sum(len(l) for _, _, l in seq)) == (ref.hits, ref.misses)
    lib.close()


def _streams(E, k, steps, seed):
    rng = np.random.default_rng(seed)
    uniform = [rng.choice(E, size=k, replace=False).tolist() for _ in range(steps)]
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    perm = rng.permutation(E)
    zipf = [perm[rng.choice(E, size=k, replace=False, p=p)].tolist() for _ in range(steps)]
    return {"uniform": uniform, "zipf": zipf}


@pytest.mark.parametrize("n_slots", [8, 16, 24])
@pytest.mark.parametrize("kind", ["uniform", "zipf"])
def test_library_matches_oracle(n_slots, kind):
    stream = _streams(128, 8, 1500, 5 + n_slots)[kind]
    ref = SlotCache(n_slots)
    lib = _lib_cache(2, n_slots)
    for ids in stream:
        got = lib.lookup(1, ids)
        want = ref.step(ids)
        assert got == want, f"step with {ids}"
        # the step's experts are all resident, each in its own slot
        held = [lib.slot_expert(1, s) for s in range(n_slots)]
        assert all(held[s] == e for s, e in zip(got[0], ids))
        assert len(set(got[0])) == len(set(ids))
    assert lib.stats(1) == (ref.hits, ref.misses)
    assert lib.stats(0) == (0, 0)  # the other layer untouched
    if kind == "zipf" and n_slots >= 16:
        assert ref.hits > ref.misses  # with room to spare, skewed routing keeps its favourites
    lib.close()


def test_errors():
    lib = _lib_cache(1, 4)
    with pytest.raises(bq.MoeError) as e:
        lib.lookup(0, [1, 2, 3, 4, 5])
    assert e.value.status == bq.MOE_ERR_UNSUPPORTED
    with pytest.raises(bq.MoeError) as e:
        lib.lookup(0, [1, -2])
    assert e.value.status == bq.MOE_ERR_BAD_EXPERT_ID
    with pytest.raises(bq.MoeError) as e:
        lib.lookup(3, [1])
    assert e.value.status == bq.MOE_ERR_INVALID_ARG
    # a repeated id takes one slot and one fill
    assert lib.lookup(0, [6, 6, 7]) == ([0, 0, 1], [(0, 6), (1, 7)])
    lib.close()
    with pytest.raises(bq.MoeError):
        bq.ExpertCache(1, 0)
    with pytest.raises(bq.MoeError):
        bq.ExpertCache(1, 65)


def _mutants():
    """Plausible slips in the oracle's rules, each of which the hand-worked
    sequences must catch."""
    def lru_only(self, s):  # recency alone, frequency ignored
        return (self.last[s], s)

    def most_used(self, s):  # evicts the most used
        return (-self.uses[s], self.last[s], s)

    def most_recent_tie(self, s):  # ties to the most recent
        return (self.uses[s], -self.last[s], s)

    return {"lru": lru_only, "most-used": most_used, "recent-tie": most_recent_tie}


@pytest.mark.parametrize("name", sorted(_mutants()))
def test_pins_catch_mutated_rules(name, monkeypatch):
    key = _mutants()[name]

    def step(self, ids):
        wanted = list(dict.fromkeys(ids))
        self.step_no += 1
        where = {}
        for e in wanted:
            if e in self.expert:
                s = self.expert.index(e)
                self.uses[s] += 1
                self.last[s] = self.step_no
                where[e] = s
        busy = set(where.values())
        loads = []
        for e in wanted:
            if e in where:
                continue
            empty = [s for s in range(self.n_slots) if self.expert[s] is None and s not in busy]
            victim = empty[0] if empty else min((s for s in range(self.n_slots) if s not in busy),
                                                key=lambda s: key(self, s))
            self.expert[victim], self.uses[victim], self.last[victim] = e, 1, self.step_no
            busy.add(victim)
            where[e] = victim
            loads.append((victim, e))
        return [where[e] for e in ids], loads

    monkeypatch.setattr(SlotCache, "step", step)
    caught = False
    for n_slots, seq in ((3, HAND), (2, RECENCY), (2, FREQUENCY)):
        ref = SlotCache(n_slots)
        for ids, want_slots, want_loads in seq:
            if ref.step(ids) != (want_slots, want_loads):
                caught = True
    assert caught, f"mutant {name} passes every pin"
