"""Oracle for the slot replacement of the expert cache.  TEST INFRASTRUCTURE
ONLY.

The Strata 4090 post (section 5, second paragraph) keeps the hottest experts
in a least-recently-used set of VRAM slots (1,300-1,600 of them on its card)
in front of slower tiers, fetching one layer ahead; the DeepSeek-V4.1-Flash
field report (section 3B) runs 4288 expert slots.  Here the slot pool in HBM
is the cache, the host's pinned memory the tier behind it, and the per-layer
slot tables the indirection.

Readings where the pages are silent (also in the design notes):
  * every slot has a fixed format (its size); an expert goes only into a slot
    of its own format;
  * a plan is one layer's request (its experts, duplicates allowed); each
    plan has a sequence number c = 0, 1, ...;
  * a requested expert already in a slot is a hit and marks the slot used at
    c; otherwise it takes, among the slots of its format not used by this
    plan or the previous one (those may still be read by a kernel in
    flight), the one used longest ago (never-used slots first, then the lower
    slot index), evicting what it held;
  * no such slot: the plan fails (nothing changes).
"""
from __future__ import annotations


class LruCache:
    def __init__(self, n_layers: int, n_experts: int, slot_fmt, expert_fmt):
        self.L, self.E = n_layers, n_experts
        self.slot_fmt = list(slot_fmt)
        self.expert_fmt = list(expert_fmt)  # (layer * E + expert) -> format
        self.holder = [-1] * len(self.slot_fmt)  # slot -> key or -1
        self.where = {}  # key -> slot
        self.used = [-1] * len(self.slot_fmt)  # slot -> last plan that used it
        self.c = 0

    def plan(self, layer: int, experts):
        """Returns [(slot, miss, evicted key or -1)] per request, or None when
        some miss finds no slot (state unchanged then)."""
        saved = (list(self.holder), dict(self.where), list(self.used))
        c = self.c
        out = []
        for e in experts:
            key = layer * self.E + e
            if key in self.where:
                s = self.where[key]
                self.used[s] = c
                out.append((s, False, -1))
                continue
            fmt = self.expert_fmt[key]
            best = -1
            for s in range(len(self.slot_fmt)):
                if self.slot_fmt[s] != fmt or (self.used[s] >= 0 and self.used[s] >= c - 1):
                    continue
                if best < 0 or self.used[s] < self.used[best]:
                    best = s
            if best < 0:
                self.holder, self.where, self.used = saved
                return None
            old = self.holder[best]
            if old >= 0:
                del self.where[old]
            self.holder[best] = key
            self.where[key] = best
            self.used[best] = c
            out.append((best, True, old))
        self.c += 1
        return out
