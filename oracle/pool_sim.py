"""Brute-force simulator of the bounded pool's slot policy (TEST INFRASTRUCTURE).

Written as plainly as possible: full scans, no sets, no incremental bookkeeping. The rule
(the pages give only "bounded pool, LFU + recency eviction"; paotong.dev commentary on Swiftlet):
one pool over all layers keyed by (layer, expert); each lookup call advances a tick; a hit adds one
use and stamps the tick; a miss fills the lowest free slot, else evicts the unpinned slot with the
smallest (uses, last tick, slot index); a new entry has one use and the current tick; everything
looked up or loaded since the last release is pinned.
"""


class PoolSim:
    def __init__(self, n_slots):
        self.owner = [None] * n_slots
        self.uses = [0] * n_slots
        self.last = [0] * n_slots
        self.pinned = [False] * n_slots
        self.tick = 0

    def slot_of(self, key):
        for s, o in enumerate(self.owner):
            if o == key:
                return s
        return -1

    def lookup(self, layer, experts):
        self.tick += 1
        out = []
        for e in experts:
            s = self.slot_of((layer, e))
            if s >= 0:
                self.uses[s] += 1
                self.last[s] = self.tick
                self.pinned[s] = True
            out.append(s)
        return out

    def load(self, layer, expert):
        s = self.slot_of((layer, expert))
        if s >= 0:
            self.lookup(layer, [expert])
            return s
        free = [s for s in range(len(self.owner)) if self.owner[s] is None]
        if free:
            s = min(free)
        else:
            cand = [(self.uses[s], self.last[s], s) for s in range(len(self.owner)) if not self.pinned[s]]
            if not cand:
                return None
            s = min(cand)[2]
        self.owner[s] = (layer, expert)
        self.uses[s] = 1
        self.last[s] = self.tick
        self.pinned[s] = True
        return s

    def release(self):
        self.pinned = [False] * len(self.owner)
