"""Slot-pool simulator: LUT, residency, victims, eviction scores, permutation.

Oracle; test infrastructure only.  Sources:
  * SeqMoE "Mechanism": one pool of cache slots shared by every MoE layer at a
    fixed base, a table rewriting expert_id to slot_id, misses copied into a
    slot by the device from a pinned, mapped host pool, a per-slot tag that
    grows on every new occupant.
  * MoE-CORE "Mechanism": a per-layer decode cache; its routing-history score
    combines, with nonnegative weights, the selection count over a window W,
    an EMA of selections, the current router score and the age since the last
    selection, each normalised across the layer; the lowest score is evicted.
  * HybriMoE "Mechanism": Minus Recent Score — the routing scores of the recent
    steps added up, minus the most recent one.
  * RapidMoE §4.3: for several tokens in a step, the router score is the
    token-averaged gate probability.

Readings taken where the pages are silent (each is listed in the design notes):
  * s_e(t) = (sum over tokens of the full softmax / sigmoid probability) / T,
    the sum taken in ascending token order.  sel_e(t) = 1 if any token
    selected e.
  * History lives per (layer, expert) for all E experts and is not reset on
    eviction; ring buffers of W steps start at zero.  Each layer counts its own
    steps t = 0, 1, 2, ...
  * MRS_e = (sum of s_e over the W most recent steps, oldest first) - s_e(t).
  * MoE-CORE: c = sum of sel over the window; m <- lam*m + (1-lam)*sel;
    g = s_e(t); age a = t - last_sel (t+1 if never selected).  Each of c, m, g
    is divided by its maximum over the layer's E experts (0 when that maximum
    is 0); age enters as recency r = 1 - a / max a (1 when max a is 0) so that
    all four weights stay nonnegative; score = ((w0 c^ + w1 m^) + w2 g^) + w3 r.
  * LRU (the baseline both pages compare against): score = last selection step.
  * The history of layer l is updated before layer l's victims are chosen in
    the same step.  Victims: misses in ascending expert id; the lowest free
    slot first; else the lowest-score slot of layer l that holds no expert
    needed in this step; else the lowest-score slot of any other layer; ties to
    the lowest slot id.  If no slot can be freed (every slot holds an expert
    this step needs) the miss is served straight from the host pool for this
    step and the table is left as it is ("bypass").
All score arithmetic is float32, one rounding per operation, in the order
written, because it decides integer victim choices.
"""
import numpy as np

EVICT_CORE, EVICT_MRS, EVICT_LRU = 0, 1, 2

F32 = np.float32


class SlotPoolSim:
    def __init__(self, L, E, S, policy=EVICT_CORE, window=16, ema_decay=0.9,
                 core_w=(0.25, 0.25, 0.25, 0.25)):
        self.L, self.E, self.S, self.W = L, E, S, window
        self.policy = policy
        self.lam = F32(ema_decay)
        self.one_minus_lam = F32(F32(1.0) - self.lam)
        self.core_w = [F32(v) for v in core_w]
        self.lut = np.full((L, E), -1, np.int32)
        self.owner = np.full(S, -1, np.int32)          # l * E + e, or -1 for free
        self.tag = np.zeros(S, np.uint32)
        self.step = np.zeros(L, np.int64)
        self.hist_s = np.zeros((L, window, E), F32)
        self.hist_sel = np.zeros((L, window, E), np.uint8)
        self.ema = np.zeros((L, E), F32)
        self.last_sel = np.full((L, E), -1, np.int64)
        self.score = np.zeros((L, E), F32)
        self.hits = self.misses = self.evictions = self.bypass = 0

    # ---------------------------------------------------------------- table
    def set_lut(self, lut):
        lut = np.asarray(lut, np.int32).reshape(self.L, self.E)
        used = lut[lut >= 0]
        if used.size and (used.max() >= self.S or np.unique(used).size != used.size):
            raise ValueError("lut must map experts to distinct slots in [0, S)")
        if (lut < -1).any():
            raise ValueError("lut entries must be a slot id or -1")
        self.lut = lut.copy()
        self.owner[:] = -1
        for l in range(self.L):
            for e in range(self.E):
                s = lut[l, e]
                if s >= 0:
                    self.owner[s] = l * self.E + e
                    self.tag[s] += 1

    def load_slot(self, l, e, slot):
        """Place expert (l, e) in `slot`, evicting its occupant; a previous slot of (l, e) becomes free."""
        prev = self.lut[l, e]
        if prev == slot:
            return
        if prev >= 0:
            self.owner[prev] = -1
        occ = self.owner[slot]
        if occ >= 0:
            self.lut[occ // self.E, occ % self.E] = -1
        self.owner[slot] = l * self.E + e
        self.lut[l, e] = slot
        self.tag[slot] += 1

    # --------------------------------------------------------------- scores
    def update_scores(self, l, ids, probs32):
        """One history step of layer l from ids [T, k] and float32 probs [T, E]."""
        ids = np.asarray(ids)
        p = np.asarray(probs32, F32)
        T = p.shape[0]
        E, W = self.E, self.W
        t = int(self.step[l])
        s = np.zeros(E, F32)
        for tt in range(T):                       # ascending token order
            s = s + p[tt]
        s = s / F32(T)
        sel = np.zeros(E, np.uint8)
        sel[ids.reshape(-1)] = 1
        slot = t % W
        self.hist_s[l, slot] = s
        self.hist_sel[l, slot] = sel
        self.ema[l] = self.lam * self.ema[l] + self.one_minus_lam * sel.astype(F32)
        self.last_sel[l, sel == 1] = t
        count = self.hist_sel[l].astype(np.int64).sum(axis=0)
        age = t - self.last_sel[l]                 # never selected: t - (-1) = t + 1

        if self.policy == EVICT_MRS:
            acc = np.zeros(E, F32)
            for j in range(W - 1, -1, -1):         # oldest step of the window first
                acc = acc + self.hist_s[l, (t - j) % W]
            self.score[l] = acc - s
        elif self.policy == EVICT_CORE:
            w0, w1, w2, w3 = self.core_w
            c = count.astype(F32)
            a = age.astype(F32)
            m = self.ema[l]
            cmax, mmax, smax, amax = c.max(), m.max(), s.max(), a.max()
            c_hat = c / cmax if cmax > 0 else np.zeros(E, F32)
            m_hat = m / mmax if mmax > 0 else np.zeros(E, F32)
            g_hat = s / smax if smax > 0 else np.zeros(E, F32)
            r_hat = F32(1.0) - a / amax if amax > 0 else np.ones(E, F32)
            self.score[l] = ((w0 * c_hat + w1 * m_hat) + w2 * g_hat) + w3 * r_hat
        else:
            self.score[l] = self.last_sel[l].astype(F32)
        self.step[l] = t + 1
        return s

    # -------------------------------------------------------- miss handling
    def _slot_score(self, slot):
        o = int(self.owner[slot])
        return self.score[o // self.E, o % self.E]

    def plan(self, l, ids):
        """LUT rewrite, miss detection and victim choice for layer l's step.

        Returns dict: U (ascending needed experts), slot_of (expert -> slot, -1 = bypass),
        events (list of (expert, slot, evicted owner or -1)), hits, misses, bypass.
        """
        E = self.E
        U = sorted(set(int(e) for e in np.asarray(ids).reshape(-1)))
        protected = set(int(self.lut[l, e]) for e in U if self.lut[l, e] >= 0)
        hits = sum(1 for e in U if self.lut[l, e] >= 0)
        events, n_miss, n_bypass = [], 0, 0
        for e in U:
            if self.lut[l, e] >= 0:
                continue
            n_miss += 1
            victim = -1
            free = np.nonzero(self.owner < 0)[0]
            if free.size:
                victim = int(free[0])
            else:
                best = None
                for s in range(self.S):            # own layer, not needed this step
                    if self.owner[s] // E == l and s not in protected:
                        sc = self._slot_score(s)
                        if best is None or sc < best[0]:
                            best = (sc, s)
                if best is None:
                    for s in range(self.S):        # any other layer
                        if self.owner[s] // E != l:
                            sc = self._slot_score(s)
                            if best is None or sc < best[0]:
                                best = (sc, s)
                if best is not None:
                    victim = best[1]
            if victim < 0:
                n_bypass += 1
                events.append((e, -1, -1))
                continue
            old = int(self.owner[victim])
            if old >= 0:
                self.lut[old // E, old % E] = -1
                self.evictions += 1
            self.owner[victim] = l * E + e
            self.lut[l, e] = victim
            self.tag[victim] += 1
            protected.add(victim)
            events.append((e, victim, old))
        self.hits += hits
        self.misses += n_miss
        self.bypass += n_bypass
        slot_of = {e: int(self.lut[l, e]) for e in U}
        return {"U": U, "slot_of": slot_of, "events": events, "hits": hits,
                "misses": n_miss, "bypass": n_bypass}


def permute(ids, E):
    """Rows (t, j) grouped by expert, stable in (t, j): counts [E], offs [E+1], perm [T*k], inv [T*k].

    perm[r] is the flat entry index t*k + j placed at sorted row r; inv is its inverse.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.zeros(E, np.int64)
    for e in flat:
        counts[e] += 1
    offs = np.zeros(E + 1, np.int64)
    for e in range(E):
        offs[e + 1] = offs[e] + counts[e]
    fill = offs[:-1].copy()
    perm = np.empty(T * k, np.int64)
    for i in range(T * k):                      # entries in (t, j) order: stable
        e = flat[i]
        perm[fill[e]] = i
        fill[e] += 1
    inv = np.empty(T * k, np.int64)
    inv[perm] = np.arange(T * k)
    return counts, offs, perm, inv
