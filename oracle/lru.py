"""Oracle of the VRAM expert-slot cache's replacement policy (plain Python).

TEST INFRASTRUCTURE ONLY.

The page "8GB 笔记本 39.3 tok/s、单卡跑 753B：FreeToken 把 frontier MoE 拉回本地"
(section 设计核心, second principle) keeps a global LRU cache of experts in
VRAM: adjacent tokens route to overlapping experts, so most routed accesses
hit and only misses are filled from host memory.  It does not fix the
details, so this oracle states them:

* one cache per layer with ``slots`` slots, initially empty;
* a token's k experts are visited in ascending expert id;
* a hit sets the expert's last-use stamp to the current step;
* a miss takes the lowest-index free slot if there is one, otherwise evicts
  the slot with the oldest stamp among experts the current token does not
  select, the lower slot index winning a tie; the new expert's stamp is the
  current step.

The page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算" (paragraph on
bandwidth-aware storage) predicts the experts the next steps will need from the
gate outputs and fetches them asynchronously, so that transfer and compute
overlap.  How a prediction enters the cache is not said; this oracle reads it
as: predicted ids in ascending order, repeats ignored; one already resident is
left as it is (a prediction is not a use); otherwise it takes the lowest free
slot, else the slot with the oldest stamp older than the current step (lower
slot on a tie) whose expert is not among the predicted ones, so neither the
current token's experts nor a predicted one are displaced; no slot, no fetch.  A fetched expert gets
stamp step - 1.  A later access that finds a
fetched expert before it left the cache counts as a used prediction.

The same page (section 设计核心, third mechanism) resizes and rebuilds the cache
at safe points from free VRAM without a reload.  Which experts survive is not
said; this oracle reads it as: all resident experts when they fit, else the
``slots`` most recently used ones (the lower old slot on equal stamps); they
keep their stamps and take slots 0, 1, ... in the order of their old slots.
"""
from __future__ import annotations


class LayerLRU:
    def __init__(self, slots: int):
        if slots <= 0:
            raise ValueError("slots must be positive")
        self.slots = slots
        self.expert_of = [-1] * slots   # slot -> expert, -1 when free
        self.stamp = [-1] * slots       # slot -> step of last use
        self.slot_of = {}               # expert -> slot
        self.fetched = [False] * slots  # slot -> installed by a prefetch and not used since
        self.prefetched = 0             # experts installed by prefetches
        self.prefetch_used = 0          # ... of which a later access found

    def access(self, step: int, ids):
        """Process one token's expert ids; returns (slots, misses) in the order of ``ids``.

        ``misses`` is the list of (expert, slot) pairs the caller must fill,
        in ascending expert order.
        """
        ids = [int(e) for e in ids]
        if len(set(ids)) != len(ids):
            raise ValueError("a token selects each expert at most once")
        if len(ids) > self.slots:
            raise ValueError("more experts per token than slots")
        current = set(ids)
        result = {}
        misses = []
        for e in sorted(ids):
            if e in self.slot_of:
                s = self.slot_of[e]
                self.stamp[s] = step
                if self.fetched[s]:
                    self.fetched[s] = False
                    self.prefetch_used += 1
                result[e] = s
                continue
            free = [s for s in range(self.slots) if self.expert_of[s] < 0]
            if free:
                s = free[0]
            else:
                cands = [s for s in range(self.slots) if self.expert_of[s] not in current]
                s = min(cands, key=lambda q: (self.stamp[q], q))
                del self.slot_of[self.expert_of[s]]
            self.expert_of[s] = e
            self.stamp[s] = step
            self.slot_of[e] = s
            self.fetched[s] = False
            result[e] = s
            misses.append((e, s))
        return [result[e] for e in ids], misses

    def prefetch(self, step: int, ids):
        """Install predicted experts ahead of the token that uses them; returns the (expert, slot) fills, ascending."""
        fills = []
        want = sorted(set(int(i) for i in ids))
        for e in want:
            if e in self.slot_of:
                continue
            free = [s for s in range(self.slots) if self.expert_of[s] < 0]
            if free:
                s = free[0]
            else:
                older = [s for s in range(self.slots) if self.stamp[s] < step and self.expert_of[s] not in want]
                if not older:
                    continue
                s = min(older, key=lambda q: (self.stamp[q], q))
                del self.slot_of[self.expert_of[s]]
            self.expert_of[s] = e
            self.stamp[s] = step - 1
            self.slot_of[e] = s
            self.fetched[s] = True
            self.prefetched += 1
            fills.append((e, s))
        return fills

    def resize(self, slots: int):
        """Resize to ``slots`` slots; returns, for each new slot, the old slot whose expert moves there (-1: free)."""
        if slots <= 0:
            raise ValueError("slots must be positive")
        resident = [q for q in range(self.slots) if self.expert_of[q] >= 0]
        if len(resident) > slots:
            newest_first = sorted(resident, key=lambda q: (-self.stamp[q], q))
            resident = sorted(newest_first[:slots])
        moves = resident + [-1] * (slots - len(resident))
        self.expert_of = [self.expert_of[q] if q >= 0 else -1 for q in moves]
        self.stamp = [self.stamp[q] if q >= 0 else -1 for q in moves]
        self.fetched = [self.fetched[q] if q >= 0 else False for q in moves]
        self.slot_of = {e: s for s, e in enumerate(self.expert_of) if e >= 0}
        self.slots = slots
        return moves
