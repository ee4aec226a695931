"""Brute-force simulator of the adopt policy (LRU whose staged calls end holding
their most-used experts), written from the rule text with plain lists:

  * single-stage calls: exactly the per-layer LRU rule;
  * a call with more distinct experts than slots: rank its experts by picks in
    the call (more first), then by expert id (lower first); take the misses
    lowest rank first; stage 0 is the hits plus the first S - |hits| misses on
    the LRU victims (empty slots by index, then the least recently used slots
    whose expert the call does not pick);
  * m misses remain: LRU would need G = ceil(m / S) more stages; stream them
    through C = ceil(m / G) slots: keep the S - C slots whose stage-0 expert
    ranks highest, and put the i-th remaining miss into the (i mod C)-th of the
    other slots (ascending index) at stage 1 + i // C;
  * every slot the call used gets the call's tick.

Independent of the oracle (which is C) and of the GPU plan kernel.
"""
import math


class BruteAdopt:
    def __init__(self, S, E):
        self.S, self.E = S, E
        self.holder = [None] * S
        self.used_at = [0] * S
        self.tick = 0

    def call(self, tokens):
        S = self.S
        self.tick += 1
        now = self.tick
        picks = [e for tok in tokens for e in tok]
        count = {}
        for e in picks:
            count[e] = count.get(e, 0) + 1
        wanted = sorted(count)
        where = {e: s for s, e in enumerate(self.holder) if e is not None}
        hits = [e for e in wanted if e in where]
        misses = [e for e in wanted if e not in where]
        staged = len(wanted) > S

        def rank(e):           # smaller is better
            return (-count[e], e)

        if staged:
            misses.sort(key=rank, reverse=True)   # lowest rank first
        first = len(misses) if not staged else S - len(hits)

        placed = {}
        for e in hits:
            s = where[e]
            self.used_at[s] = now
            placed[e] = (s, 0)
        records = []
        evictions = 0

        empty = [s for s in range(S) if self.holder[s] is None]
        stale = [s for s in range(S) if self.holder[s] is not None and self.holder[s] not in count]
        stale.sort(key=lambda s: (self.used_at[s], s))
        for e, s in zip(misses[:first], empty + stale):
            old = self.holder[s]
            evictions += old is not None
            self.holder[s] = e
            self.used_at[s] = now
            placed[e] = (s, 0)
            records.append((e, s, -1 if old is None else old, 0))

        rest = misses[first:]
        n_stages = 1
        if rest:
            m = len(rest)
            G = math.ceil(m / S)
            C = math.ceil(m / G)
            by_rank = sorted(range(S), key=lambda s: rank(self.holder[s]))
            kept = set(by_rank[:S - C])
            stream = [s for s in range(S) if s not in kept]
            for i, e in enumerate(rest):
                s, j = stream[i % C], 1 + i // C
                old = self.holder[s]
                evictions += 1
                self.holder[s] = e
                self.used_at[s] = now
                placed[e] = (s, j)
                records.append((e, s, old, j))
                n_stages = max(n_stages, j + 1)

        pick_hits = sum(1 for e in picks if e in where)
        return {
            "gpu_slot": [[placed[e][0] for e in tok] for tok in tokens],
            "stage": [[placed[e][1] for e in tok] for tok in tokens],
            "misses": records,
            "n_unique": len(wanted), "n_hits": len(hits), "n_miss": len(misses),
            "n_stages": n_stages, "n_evict": evictions,
            "pick_hits": pick_hits, "pick_misses": len(picks) - pick_hits,
        }

    def state(self):
        expert_slot = [-1] * self.E
        for s, e in enumerate(self.holder):
            if e is not None:
                expert_slot[e] = s
        return {"slot_expert": [-1 if e is None else e for e in self.holder],
                "expert_slot": expert_slot, "slot_stamp": list(self.used_at), "clock": self.tick}
