"""Offline cache shaping of MoE-CORE: per-layer hit-rate curves and nonuniform slot quotas.

Oracle; test infrastructure only.  Source: MoE-CORE "Mechanism" — a fixed
decode-cache budget is not split evenly over the layers; an offline replay of
hit-rate curves moves slots in steps of delta-K from layers whose hit rate
stays above the median and barely drops when shrunk, to layers at least
tau_low below the median whose hit rate rises the most when grown; the cache
starts from a domain profile, each layer's K_l experts of highest mean router
score on a profiling set.  The same page's transfer notes add that slots move
only when the receiver gains more than the donor loses.

Readings taken where the page is silent (each is listed in the design notes):
  * Hit-rate curve h_l(K): a cache of K slots holding layer l's experts only,
    filled first with the K experts of highest mean probability over the
    trace (ties to the lower id), then run over the trace's steps with the
    pool's own history score and victim rule (the simulator of cache.py with
    one layer and K slots).  h_l(K) = hits / (hits + misses); the denominator,
    the experts the steps need, does not depend on K.  h_l(0) = 0.
  * Start: the uniform split, floor(S/L) slots and one more for the first
    S mod L layers, each capped at E.
  * One move per round: the median is that of the L current hit rates (the
    mean of the two middle values when L is even).  A donor has
    h_l(K_l - dK) >= median (it stays at or above the median when shrunk) and
    K_l - dK >= 1; among donors the smallest drop h_l(K_l) - h_l(K_l - dK)
    gives.  A receiver has h_l(K_l) <= median - tau_low and K_l + dK <= E;
    among receivers the largest gain h_l(K_l + dK) - h_l(K_l) takes.  Ties go
    to the lower layer index.  The move is made only if gain > drop; otherwise,
    or with no donor or receiver, the plan is final.  Every move raises the sum
    of the hit rates, so the rounds end.
Hit rates are float64 ratios of integer counts, compared in float64.
"""
import numpy as np

from .cache import SlotPoolSim


def profile_order(probs_l):
    """Experts of one layer by descending mean probability over the trace, ties to the lower id.

    probs_l: float32 [steps, T, E].  The mean is taken as the float64 sum over every
    (step, token), in that order, divided by their count.
    """
    p = np.asarray(probs_l, np.float64)
    steps, T, E = p.shape
    total = np.zeros(E)
    for s in range(steps):
        for t in range(T):
            total = total + p[s, t]
    mean = total / (steps * T)
    return sorted(range(E), key=lambda e: (-mean[e], e))


def layer_hit_rate(ids_l, probs_l, E, K, policy, window, ema_decay, core_w):
    """h_l(K) and its counts: (hits, needed) over the trace of one layer.

    ids_l: int [steps, T, k]; probs_l: float32 [steps, T, E].
    """
    ids_l = np.asarray(ids_l)
    needed = sum(len(set(int(e) for e in ids_l[s].reshape(-1))) for s in range(ids_l.shape[0]))
    if K <= 0:
        return 0.0, 0, needed
    sim = SlotPoolSim(1, E, K, policy, window, ema_decay, core_w)
    lut = np.full((1, E), -1, np.int32)
    for slot, e in enumerate(profile_order(probs_l)[:K]):
        lut[0, e] = slot
    sim.set_lut(lut)
    for s in range(ids_l.shape[0]):
        sim.update_scores(0, ids_l[s], np.asarray(probs_l[s], np.float32))
        sim.plan(0, ids_l[s])
    return sim.hits / needed if needed else 0.0, sim.hits, needed


def plan_quotas(ids, probs, E, budget, delta_k, tau_low, policy, window=16, ema_decay=0.9,
                core_w=(0.25, 0.25, 0.25, 0.25)):
    """Nonuniform per-layer quotas for a budget of `budget` slots.

    ids: int [steps, L, T, k]; probs: float32 [steps, L, T, E].
    Returns (quotas [L] int, hit rates at those quotas [L] float64, moves made).
    """
    ids = np.asarray(ids)
    probs = np.asarray(probs, np.float32)
    L = ids.shape[1]
    base, extra = divmod(budget, L)
    K = [min(E, base + (1 if l < extra else 0)) for l in range(L)]
    memo = {}

    def h(l, k):
        if (l, k) not in memo:
            memo[(l, k)] = layer_hit_rate(ids[:, l], probs[:, l], E, k, policy, window, ema_decay, core_w)[0]
        return memo[(l, k)]

    moves = 0
    while True:
        cur = [h(l, K[l]) for l in range(L)]
        srt = sorted(cur)
        med = srt[L // 2] if L % 2 else (srt[L // 2 - 1] + srt[L // 2]) / 2.0
        donor, drop = None, None
        for l in range(L):
            if K[l] - delta_k >= 1 and h(l, K[l] - delta_k) >= med:
                d = cur[l] - h(l, K[l] - delta_k)
                if drop is None or d < drop:
                    donor, drop = l, d
        recv, gain = None, None
        for l in range(L):
            if l != donor and cur[l] <= med - tau_low and K[l] + delta_k <= E:
                g = h(l, K[l] + delta_k) - cur[l]
                if gain is None or g > gain:
                    recv, gain = l, g
        if donor is None or recv is None or not gain > drop:
            break
        K[donor] -= delta_k
        K[recv] += delta_k
        moves += 1
    return np.array(K, np.int32), np.array([h(l, K[l]) for l in range(L)]), moves


def profile_lut(probs, quotas, E):
    """The initial table from a domain profile: layer l's quota[l] experts of highest mean
    probability, slots handed out layer by layer in that order.  probs: float32 [steps, L, T, E]."""
    probs = np.asarray(probs, np.float32)
    L = probs.shape[1]
    lut = np.full((L, E), -1, np.int32)
    nxt = 0
    for l in range(L):
        for e in profile_order(probs[:, l])[:int(quotas[l])]:
            lut[l, e] = nxt
            nxt += 1
    return lut
