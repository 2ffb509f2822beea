"""Approximate expert substitution (AES) of MoE-CORE, as a rewrite of one step's routing.

Oracle; test infrastructure only.  Source: MoE-CORE "Mechanism" — an optional
approximate path, off in the main numbers, substitutes a resident unselected
expert for a low-score miss whose score is within alpha of the rank-(k+1)
boundary, keeping the missed expert's routing coefficient; high-score misses
still take the exact host-to-device copy.

Readings taken where the page is silent (each is listed in the design notes):
  * Per token.  The "score" is the router logit z (the quantity the top-k
    ranks); a selected expert is a low-score miss when it is not resident at
    the start of the step and z_e - z_(k+1) <= alpha in float32, z_(k+1) being
    the largest logit the token did not select.  k = E leaves nothing to
    substitute.
  * The token's low-score misses, in rank order, take the token's resident
    unselected experts in rank order (highest logit first, ties to the lower
    id), one each, while any remain.  The substitute takes the miss's position
    in the token's top-k, so it keeps the missed expert's renormalised weight;
    the weights are not recomputed.
  * Everything after the gate sees the rewritten routing: the history counts the
    substitutes as selected, the table and misses use them, the combine sums
    over them (in ascending expert id, as for any routing).
"""
import numpy as np


def rank_order(z_row):
    """Experts of one token by descending float32 logit, ties to the lower id."""
    z = np.asarray(z_row, np.float32)
    return sorted(range(z.size), key=lambda e: (-float(z[e]), e))


def aes_substitute(z, ids, resident, alpha):
    """Rewrite ids [T, k] (each row in rank order) for the resident mask [E] (start of the step).

    z: logits [T, E] (any float type, compared in float32); alpha: float32 bound.
    Returns (new ids [T, k] int32, number of substitutions).
    """
    z = np.asarray(z, np.float32)
    ids = np.array(ids, np.int32, copy=True)
    resident = np.asarray(resident, bool)
    a = np.float32(alpha)
    T, k = ids.shape
    E = z.shape[1]
    n = 0
    if k >= E:
        return ids, 0
    for t in range(T):
        order = rank_order(z[t])
        assert order[:k] == ids[t].tolist(), "ids must be the token's top-k in rank order"
        boundary = z[t, order[k]]
        subs = [e for e in order[k:] if resident[e]]
        nxt = 0
        for r in range(k):
            e = int(ids[t, r])
            if resident[e] or not (z[t, e] - boundary <= a):
                continue
            if nxt >= len(subs):
                break
            ids[t, r] = subs[nxt]
            nxt += 1
            n += 1
    return ids, n
