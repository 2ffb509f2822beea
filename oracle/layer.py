"""Top-k gated MoE layer with SwiGLU experts (oracle; test infrastructure only).

Definitions followed:
  * RapidMoE §2.1 ("Mixture of Experts and Reasoning Models"): the gate is a
    linear projection of the token followed by a softmax; the k experts with the
    highest logits are activated; the layer output is the gate-weighted sum of
    the activated experts' outputs.
  * CAP §II-A, Eq. 1: MoE(x) = sum over the k selected experts of
    Gate_i(x) * Expert_i(x), Gate_i being the *normalised* routing weight — so
    the weights of the k selected experts sum to 1.
  * RapidMoE §4.5, Eq. 7: the expert is W_down · (SiLU(W_gate x) ⊙ (W_up x)).
    The §4.4 sentence that prints SiLU(W_gate x ⊙ W_up x) is read as an
    extraction error; Eq. 7 puts SiLU on the gate projection only.
  * RapidMoE Table 2: the DeepSeek-V3 shape adds one shared expert to every
    token; it is added with weight 1 after the routed sum.

Gating forms: "softmax-renorm" (softmax over all E logits, renormalised over the
top-k, equal to exp(z_j - z_max) / sum_{i in top-k} exp(z_i - z_max)) and
"sigmoid-renorm" (sigma(z_j) / sum_{i in top-k} sigma(z_i)).  The router bias is
part of the logit for both selection and weights.

Arithmetic is float64 throughout.  The top-k *order* is decided on the logits
rounded to float32, the precision the kernels take that decision in; ties go to
the lower expert index.  The combine sums the selected experts in ascending
expert id.
"""
import numpy as np

from .numerics import decode_act, decode_weight

GATE_SOFTMAX_RENORM = 0
GATE_SIGMOID_RENORM = 1


def router_logits(x: np.ndarray, w_r: np.ndarray, b: np.ndarray) -> np.ndarray:
    """z[t, e] = sum_h x[t, h] * W_r[e, h] + b[e]   (float64)."""
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T + np.asarray(b, np.float64)[None, :]


def topk_ids(z: np.ndarray, k: int):
    """Top-k by descending float32 logit, ties to the lower index.

    Returns (ids [T, k] int32, gap [T] float64) where gap is the float32 logit of
    the k-th selected expert minus that of the best unselected one (inf if k == E).
    """
    z32 = np.asarray(z, np.float64).astype(np.float32)
    T, E = z32.shape
    ids = np.empty((T, k), np.int32)
    gap = np.full(T, np.inf)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(z32[t, e]), e))
        ids[t] = order[:k]
        if k < E:
            gap[t] = float(z32[t, order[k - 1]]) - float(z32[t, order[k]])
    return ids, gap


def gate_probs(z: np.ndarray, gating: int) -> np.ndarray:
    """Per-expert router probability used for the history score: softmax over all E, or sigmoid."""
    z = np.asarray(z, np.float64)
    if gating == GATE_SOFTMAX_RENORM:
        m = z.max(axis=1, keepdims=True)
        ez = np.exp(z - m)
        return ez / ez.sum(axis=1, keepdims=True)
    return 1.0 / (1.0 + np.exp(-z))


def gate_weights(z: np.ndarray, ids: np.ndarray, gating: int) -> np.ndarray:
    """Normalised routing weights of the selected experts (CAP Eq. 1), [T, k] float64."""
    z = np.asarray(z, np.float64)
    T, k = ids.shape
    w = np.empty((T, k))
    for t in range(T):
        zt = z[t, ids[t]]
        if gating == GATE_SOFTMAX_RENORM:
            num = np.exp(zt - z[t].max())
        else:
            num = 1.0 / (1.0 + np.exp(-zt))
        w[t] = num / num.sum()
    return w


def route(x, w_r, b, k: int, gating: int):
    """Router + gate: returns dict(z, ids, w, probs, gap)."""
    z = router_logits(x, w_r, b)
    ids, gap = topk_ids(z, k)
    return {"z": z, "ids": ids, "w": gate_weights(z, ids, gating),
            "probs": gate_probs(z, gating), "gap": gap}


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a / (1 + exp(-a))."""
    return a / (1.0 + np.exp(-a))


def swiglu_expert(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """RapidMoE Eq. 7 without the residual split: W_down (SiLU(W_gate x) ⊙ W_up x), rows of x are tokens."""
    x = np.asarray(x, np.float64)
    g = x @ w_gate.T
    u = x @ w_up.T
    return (silu(g) * u) @ w_down.T


def expert_mats(stored, weight_dtype: int, I: int):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) in float64 from one stored expert (w13 = [gate; up])."""
    w13 = decode_weight(stored, "w13", weight_dtype)
    w2 = decode_weight(stored, "w2", weight_dtype)
    return w13[:I], w13[I:], w2


def moe_layer(x, routing, experts, shared=None):
    """Sparse layer: out[t] = sum over selected e, ascending e, of w_e * E_e(x_t)  (+ shared(x_t)).

    experts: callable e -> (W_gate, W_up, W_down) float64, or a dict of them.
    routing: the dict from route().  Returns float64 [T, H].
    """
    x = np.asarray(x, np.float64)
    ids, w = routing["ids"], routing["w"]
    T = x.shape[0]
    get = experts if callable(experts) else experts.__getitem__
    out = np.zeros_like(x)
    cache = {}
    for t in range(T):
        for j in np.argsort(ids[t], kind="stable"):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = get(e)
            y = swiglu_expert(x[t:t + 1], *cache[e])[0]
            out[t] = out[t] + w[t, j] * y
        if shared is not None:
            out[t] = out[t] + swiglu_expert(x[t:t + 1], *shared)[0]
    return out


def moe_layer_dense_masked(x, routing, experts, E: int, shared=None):
    """Brute force: evaluate every expert on every token, multiply by a mask weight (0 if unselected).

    Summed in ascending e, this must be bit-identical to moe_layer (adding 0 * y changes nothing).
    """
    x = np.asarray(x, np.float64)
    ids, w = routing["ids"], routing["w"]
    T = x.shape[0]
    get = experts if callable(experts) else experts.__getitem__
    gate = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            gate[t, ids[t, j]] = w[t, j]
    out = np.zeros_like(x)
    for e in range(E):
        mats = get(e)
        for t in range(T):
            # one token per call, as in moe_layer, so both see the same library rounding
            out[t] = out[t] + gate[t, e] * swiglu_expert(x[t:t + 1], *mats)[0]
    if shared is not None:
        for t in range(T):
            out[t] = out[t] + swiglu_expert(x[t:t + 1], *shared)[0]
    return out


def layer_from_stored(x_stored, act_dtype, w_r_stored, b, experts_stored, weight_dtype, I, k, gating,
                      shared_stored=None):
    """Convenience: decode everything stored, route and run the sparse layer. Returns (out, routing)."""
    x = decode_act(x_stored, act_dtype)
    w_r = decode_act(w_r_stored, act_dtype)
    routing = route(x, w_r, b, k, gating)
    getter = experts_stored if callable(experts_stored) else experts_stored.__getitem__

    def experts(e):
        return expert_mats(getter(e), weight_dtype, I)

    shared = expert_mats(shared_stored, weight_dtype, I) if shared_stored is not None else None
    return moe_layer(x, routing, experts, shared), routing
