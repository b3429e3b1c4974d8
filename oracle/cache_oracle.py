"""Oracle of the expert slot cache (test infrastructure only: tests and the
bench's reference arm may import it; the product path never does).

Page "TurboFieldfare - System design", sections "Resource split" (16
routed-expert slots per opened layer) and "Load and ownership" (the cache
records which expert occupies each slot; least-frequently-used eviction with
recency as the tie-breaker; a hit reuses the buffer, a miss assigns an
evictable slot and reads the expert into it).  The readings the pages leave
open, stated once here and used as written:

  * an expert's use count starts at 1 when it enters a slot, grows by 1 at
    every step that selects it, and is forgotten when it is evicted;
  * recency = the step at which the slot's expert was last selected;
  * an empty slot is taken before any eviction, lowest slot first;
  * the experts a step selects are not evictable during that step;
  * among equally frequent and equally recent candidates, the lower slot.

A step is one token's selection (its k expert ids); the result of a step is
the slot of every selected id and the list of (slot, expert) fills."""


class SlotCache:
    """One layer's slots, written as plainly as the rules above."""

    def __init__(self, n_slots: int):
        self.n_slots = n_slots
        self.expert = [None] * n_slots  # expert id held by each slot, None when empty
        self.uses = [0] * n_slots
        self.last = [0] * n_slots
        self.step_no = 0
        self.hits = 0
        self.misses = 0

    def step(self, ids):
        if any(e < 0 for e in ids):
            raise ValueError("negative expert id")
        wanted = list(dict.fromkeys(ids))  # distinct, in selection order
        if len(wanted) > self.n_slots:
            raise ValueError("more distinct experts than slots")
        self.step_no += 1
        where = {}
        # hits
        for e in wanted:
            if e in self.expert:
                s = self.expert.index(e)
                self.uses[s] += 1
                self.last[s] = self.step_no
                self.hits += 1
                where[e] = s
        busy = set(where.values())
        loads = []
        # misses, in selection order
        for e in wanted:
            if e in where:
                continue
            empty = [s for s in range(self.n_slots) if self.expert[s] is None and s not in busy]
            if empty:
                victim = empty[0]
            else:
                candidates = [s for s in range(self.n_slots) if s not in busy]
                victim = min(candidates, key=lambda s: (self.uses[s], self.last[s], s))
            self.expert[victim] = e
            self.uses[victim] = 1
            self.last[victim] = self.step_no
            self.misses += 1
            busy.add(victim)
            where[e] = victim
            loads.append((victim, e))
        return [where[e] for e in ids], loads
