"""Brute-force simulator of the decayed-score admission policy, written from
the rule text, independently of the oracle.

Rule (plain reading of "Keeping the cache fresh": a decayed usage score per
expert, x0.9 per token; a missed expert that scores higher than the weakest
slot is promoted, up to a budget of copies; every miss is still computed):

  * one clock tick per call; token by token every score is multiplied by 0.9
    and each picked expert gains 1, in single precision (each operation
    rounded to float32);
  * distinct picked experts U; hits keep their slots and get the tick; the call
    must fit one stage (|U| <= S);
  * misses are considered strongest first (score descending, then lower id);
  * while the budget lasts (0 = no limit), a miss takes an empty slot (lowest
    index first) if there is one, else the weakest slot whose expert the call
    does not pick (score ascending, then lowest index) if its own score is
    strictly higher; otherwise it is bypassed (no slot, nothing evicted);
  * every admission uses one unit of the budget;
  * sticky share (per mille, "never evict the most-used share of each layer's
    slots"): after the scores of the call are updated, the floor(share x S /
    1000) occupied slots with the highest scores (ties: lower index) are not
    evictable in this call.

Plain lists and dictionaries.
"""
import numpy as np


class BruteScore:
    def __init__(self, S, E, budget=0, sticky=0):
        self.S, self.E, self.budget, self.sticky = S, E, budget, sticky
        self.holder = [None] * S
        self.used_at = [0] * S
        self.tick = 0
        self.score = [np.float32(0.0)] * E

    def call(self, tokens):
        S = self.S
        wanted = sorted({e for tok in tokens for e in tok})
        assert len(wanted) <= S
        self.tick += 1
        now = self.tick
        for tok in tokens:
            self.score = [np.float32(v * np.float32(0.9)) for v in self.score]
            for e in tok:
                self.score[e] = np.float32(self.score[e] + np.float32(1.0))
        where = {e: s for s, e in enumerate(self.holder) if e is not None}
        hits = [e for e in wanted if e in where]
        misses = [e for e in wanted if e not in where]
        for e in hits:
            self.used_at[where[e]] = now
        empty = [s for s in range(S) if self.holder[s] is None]
        occupied = sorted((s for s in range(S) if self.holder[s] is not None),
                          key=lambda s: (-self.score[self.holder[s]], s))
        protected = set(occupied[:self.sticky * S // 1000])
        weak = [s for s in range(S) if self.holder[s] is not None and self.holder[s] not in wanted
                and s not in protected]
        weak.sort(key=lambda s: (self.score[self.holder[s]], s))
        left = self.budget if self.budget > 0 else S + 1
        slot_of = {e: where[e] for e in hits}
        evicted_by = {}
        evictions = bypass = 0
        for m in sorted(misses, key=lambda e: (-self.score[e], e)):
            s, old = None, None
            if left > 0:
                if empty:
                    s = empty.pop(0)
                elif weak and self.score[m] > self.score[self.holder[weak[0]]]:
                    s = weak.pop(0)
                    old = self.holder[s]
            if s is None:
                bypass += 1
                slot_of[m] = -1
                evicted_by[m] = -1
                continue
            left -= 1
            if old is not None:
                evictions += 1
            self.holder[s] = m
            self.used_at[s] = now
            slot_of[m] = s
            evicted_by[m] = -1 if old is None else old
        picks = [e for tok in tokens for e in tok]
        return {
            "gpu_slot": [[slot_of[e] for e in tok] for tok in tokens],
            "misses": [(m, slot_of[m], evicted_by[m], 0) for m in misses],
            "n_unique": len(wanted), "n_hits": len(hits), "n_miss": len(misses), "n_stages": 1,
            "n_evict": evictions, "n_bypass": bypass,
            "pick_hits": sum(1 for e in picks if e in where),
            "pick_misses": sum(1 for e in picks if e not in where),
        }

    def state(self):
        es = [-1] * self.E
        for s, e in enumerate(self.holder):
            if e is not None:
                es[e] = s
        return {"slot_expert": [-1 if e is None else e for e in self.holder], "expert_slot": es,
                "slot_stamp": list(self.used_at), "clock": self.tick}
