"""Slot-pool simulator with the asynchronous prefetch protocol of SeqMoE.

Oracle; test infrastructure only.  Sources:
  * SeqMoE "Mechanism" and "notes": the device owns the prediction and the
    cache metadata; the only host thread reads a mapped control region and
    copies on a stream the compute never waits on; a monotonically increasing
    tag per slot is the only synchronisation — the device commits a prefetched
    expert into the cache only when the tag written back by the host matches
    the tag the device assigned, so a stale or superseded copy is never
    committed.
  * HybriMoE "Mechanism": prefetch candidates in priority order — routing
    score first, and the copy volume already committed to the layer.
  * MoE-CORE "Mechanism": a prefetch goes into a slot the cache can give up,
    and its count is capped.

Readings taken where the pages are silent (each is listed in the design notes):
  * At the end of layer l's plan, once its own misses have their slots, the
    device issues up to (per_step - misses of this step) prefetches for layer
    l: the experts of layer l that this step does not need, that are neither
    resident nor already prefetched when this phase starts (an expert one of
    these prefetches evicts is not a candidate), in descending order of this
    step's router score s_e(t) (ties to the lower id).  Each takes the lowest free
    slot, else the lowest-eviction-score slot of layer l that holds an expert
    this step does not need (ties to the lower slot); with no such slot no more
    prefetches are issued.  The slot's occupant is evicted, the slot becomes
    pending for the expert (owner -2 - (l * E + e): not resident, never a
    victim) and its tag grows by one; the request carries that tag.
  * After that, every pending slot whose written-back tag equals its own tag is
    committed (owner and table point at the expert), in request order.
  * A step that needs a pending expert counts it as a miss; its slot is the
    miss's slot (no eviction), committed at once with the tag grown by one, and
    the demand copy goes into it.  Until the prefetch's own tag has been
    written back, that slot is never a victim (its late copy would overwrite a
    new occupant).
  * The host writes back a request's tag once its copy has landed.  drain()
    stands for "every request issued so far has landed" (the GPU tests wait
    for the host thread between calls); corrupt(n) makes the next n
    write-backs carry a wrong tag, and such a slot is never committed.
"""
import numpy as np

from .cache import F32, SlotPoolSim

def pending_owner(flat):
    """Owner value of a slot holding a pending prefetch of expert l * E + e."""
    return -2 - int(flat)


class PrefetchSim(SlotPoolSim):
    def __init__(self, L, E, S, policy, window=16, ema_decay=0.9, core_w=(0.25, 0.25, 0.25, 0.25), per_step=1):
        super().__init__(L, E, S, policy, window, ema_decay, core_w)
        self.per_step = per_step
        self.pf_expert = np.full(S, -1, np.int64)        # l * E + e pending in the slot, or -1
        self.pf_tag = np.zeros(S, np.uint32)             # tag of the slot's last prefetch
        self.landed = np.zeros(S, np.uint32)             # tag the host wrote back for the slot
        self.queue = []                                  # requests not yet written back: (slot, tag)
        self.pending = []                                # pending slots, in request order
        self._corrupt = 0
        self.pf_issued = self.pf_committed = self.pf_demanded = 0

    def set_lut(self, lut):
        super().set_lut(lut)
        self.pf_expert[:] = -1
        self.pending = []
        self.queue = []
        self.landed[:] = self.pf_tag

    # ------------------------------------------------------------ host side
    def corrupt(self, n):
        self._corrupt += n

    def drain(self):
        """Every request issued so far has landed and its tag was written back."""
        for slot, tag in self.queue:
            if self._corrupt > 0:
                self._corrupt -= 1
                self.landed[slot] = np.uint32(tag + 0x5A5A0000)
            else:
                self.landed[slot] = tag
        self.queue = []

    # ---------------------------------------------------------- device side
    def plan(self, l, ids, s=None):
        """Layer l's step: table, misses, victims (as SlotPoolSim.plan, pending slots excluded),
        then prefetches for layer l by the router score s [E] of this step, then commits."""
        E = self.E
        U = sorted(set(int(e) for e in np.asarray(ids).reshape(-1)))
        protected = set(int(self.lut[l, e]) for e in U if self.lut[l, e] >= 0)
        hits = sum(1 for e in U if self.lut[l, e] >= 0)
        n_miss = n_bypass = 0
        for e in U:
            if self.lut[l, e] >= 0:
                continue
            n_miss += 1
            pend = [q for q in self.pending if self.pf_expert[q] == l * E + e]
            if pend:
                # the expert's prefetch has not been committed: its slot takes the demand copy
                v = pend[0]
                self.pending.remove(v)
                self.pf_expert[v] = -1
                self.owner[v] = l * E + e
                self.lut[l, e] = v
                self.tag[v] += 1
                protected.add(v)
                self.pf_demanded += 1
                continue
            victim = self._victim(l, protected, other_layers=True)
            if victim < 0:
                n_bypass += 1
                continue
            self._install(l, e, victim)
            protected.add(victim)
        self.hits += hits
        self.misses += n_miss
        self.bypass += n_bypass
        # prefetches for this layer
        budget = self.per_step - n_miss
        if budget > 0 and s is not None:
            s = np.asarray(s, F32)
            need = set(U)
            pending_e = set(int(self.pf_expert[q]) for q in self.pending)
            cands = [e for e in range(E) if e not in need and self.lut[l, e] < 0 and l * E + e not in pending_e]
            cands.sort(key=lambda e: (-float(s[e]), e))
            for e in cands[:budget]:
                victim = self._victim(l, protected, other_layers=False)
                if victim < 0:
                    break
                old = int(self.owner[victim])
                if old >= 0:
                    self.lut[old // E, old % E] = -1
                    self.evictions += 1
                self.owner[victim] = pending_owner(l * E + e)
                self.pf_expert[victim] = l * E + e
                self.tag[victim] += 1
                self.pf_tag[victim] = self.tag[victim]
                self.pending.append(victim)
                self.queue.append((victim, self.tag[victim]))
                self.pf_issued += 1
        # commits: every pending slot whose written-back tag matches
        for q in list(self.pending):
            if self.landed[q] == self.pf_tag[q]:
                x = int(self.pf_expert[q])
                self.owner[q] = x
                self.lut[x // E, x % E] = q
                self.pf_expert[q] = -1
                self.pending.remove(q)
                self.pf_committed += 1
        return {"U": U, "misses": n_miss, "hits": hits, "bypass": n_bypass,
                "slot_of": {e: int(self.lut[l, e]) for e in U}}

    # -------------------------------------------------------------- helpers
    def _victim(self, l, protected, other_layers):
        E = self.E
        free = np.nonzero(self.owner == -1)[0]
        if free.size:
            return int(free[0])
        best = None
        for q in range(self.S):
            o = int(self.owner[q])
            if o >= 0 and o // E == l and q not in protected and not self._busy(q):
                sc = self.score[o // E, o % E]
                if best is None or sc < best[0]:
                    best = (sc, q)
        if best is None and other_layers:
            for q in range(self.S):
                o = int(self.owner[q])
                if o >= 0 and o // E != l and not self._busy(q):
                    sc = self.score[o // E, o % E]
                    if best is None or sc < best[0]:
                        best = (sc, q)
        return -1 if best is None else best[1]

    def _busy(self, q):
        """A prefetch copy into slot q may still be in flight: its tag is not yet written back."""
        return self.pf_tag[q] != self.landed[q]

    def _install(self, l, e, victim):
        E = self.E
        old = int(self.owner[victim])
        if old >= 0:
            self.lut[old // E, old % E] = -1
            self.evictions += 1
        self.owner[victim] = l * E + e
        self.lut[l, e] = victim
        self.tag[victim] += 1
