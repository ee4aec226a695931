"""Brute-force simulator of the per-layer slot map, written from the rule text.

Rule (plain reading of "Longhaul MoE loading": per-layer LRU with a fixed budget;
experts planned as a batch, the batch's experts protected from eviction,
duplicates loaded once; more experts than slots -> stages whose partial results
are summed):

  * one clock tick per call; every slot used by the call gets the call's tick;
  * distinct picked experts U, ascending; hits are those already in a slot;
  * |U| <= S: a single stage; else stage 0 is the hits plus the first S - |hits|
    misses and each further stage takes the next S misses;
  * stage 0 evicts empty slots first (lowest index first), then the least
    recently used slots whose expert the call does not pick (ties: lowest index);
  * a later stage evicts slots used by this call's earlier stages, least
    recently used first (all share the tick, so lowest index first);
  * misses are placed in ascending expert order onto the victims in order.

Written with plain lists and dictionaries, independently of the oracle.
"""


class BruteLRU:
    def __init__(self, S, E):
        self.S, self.E = S, E
        self.holder = [None] * S      # expert in each slot
        self.used_at = [0] * S        # tick of last use
        self.tick = 0

    def call(self, tokens):
        """tokens: list of per-token pick lists.  Returns a dict like the oracle's plan."""
        S = self.S
        self.tick += 1
        now = self.tick
        wanted = sorted({e for tok in tokens for e in tok})
        where = {}
        for s, e in enumerate(self.holder):
            if e is not None:
                where[e] = s
        hits = [e for e in wanted if e in where]
        misses = [e for e in wanted if e not in where]

        if len(wanted) <= S:
            groups = [misses]
        else:
            first = S - len(hits)
            groups = [misses[:first]]
            rest = misses[first:]
            while rest:
                groups.append(rest[:S])
                rest = rest[S:]

        placed = {}                   # expert -> (slot, stage)
        mine = set()                  # slots holding this call's experts
        for e in hits:
            s = where[e]
            self.used_at[s] = now
            placed[e] = (s, 0)
            mine.add(s)

        records = []
        evictions = 0
        for j, grp in enumerate(groups):
            if j == 0:
                empty = [s for s in range(S) if self.holder[s] is None]
                stale = [s for s in range(S)
                         if self.holder[s] is not None and self.holder[s] not in wanted]
                stale.sort(key=lambda s: (self.used_at[s], s))
                order = empty + stale
            else:
                order = sorted(mine, key=lambda s: (self.used_at[s], s))
            assert len(order) >= len(grp)
            for e, s in zip(grp, order):
                old = self.holder[s]
                if old is not None:
                    evictions += 1
                self.holder[s] = e
                self.used_at[s] = now
                placed[e] = (s, j)
                mine.add(s)
                records.append((e, s, -1 if old is None else old, j))

        pick_hits = sum(1 for tok in tokens for e in tok if e in hits)
        return {
            "gpu_slot": [[placed[e][0] for e in tok] for tok in tokens],
            "stage": [[placed[e][1] for e in tok] for tok in tokens],
            "misses": records,
            "n_unique": len(wanted), "n_hits": len(hits), "n_miss": len(misses),
            "n_stages": len(groups), "n_evict": evictions,
            "pick_hits": pick_hits,
            "pick_misses": sum(len(tok) for tok in tokens) - pick_hits,
        }

    def state(self):
        expert_slot = [-1] * self.E
        for s, e in enumerate(self.holder):
            if e is not None:
                expert_slot[e] = s
        return {"slot_expert": [-1 if e is None else e for e in self.holder],
                "expert_slot": expert_slot, "slot_stamp": list(self.used_at), "clock": self.tick}
