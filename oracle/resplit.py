"""Residual-split experts and the UMIA critical set of RapidMoE (oracle; test infrastructure only).

Sources:
  * RapidMoE §4.4, Alg. 3 (residual-split representation): W^Q = Quantize(W, b_q),
    W^R = Quantize(W - W^Q, b_r); the high-precision weight is W^H = W^Q + W^R
    and the low-precision one W^L = W^Q.  Because of the SwiGLU nonlinearity
    the residual is used for gate_proj and up_proj only; down_proj is stored
    twice, W^L_down = Quantize(W_down, b_q) and W^H_down = Quantize(W_down,
    b_q + b_r).
  * RapidMoE §4.3, Eq. 3-4 (UMIA): a multiplicatively separable threshold
    Theta(l, t) = Theta * beta(l) * gamma(t) per layer l and phase t; the
    critical set is the experts whose router score g reaches it; for several
    tokens the score is the token-averaged g.

Readings taken where the page is silent (each is listed in the design notes):
  * Codec (the page's GGUF formats are third-party, so this one is defined
    here): b_q = b_r = 4 and b_q + b_r = 8; symmetric integer codes per
    128-column group along the input dimension, scale = group amax / (2^(b-1)
    - 1); stored as described in synth.gen.resplit_encode.
  * Routing is the layer's usual top-k; UMIA decides only the precision of the
    selected experts.  g is the step's token-averaged router probability s_e
    (the routing-history score); an expert is critical when s_e >= Theta(l, t),
    computed in float32 as (Theta * beta(l)) * gamma(t).  Critical experts run
    W^Q + W^R for gate/up and W^H_down, the others W^Q and W^L_down.  A shared
    expert, when there is one, is critical.
"""
import numpy as np

F32 = np.float32


def dequant_groups(codes, scales):
    """W[i, j] = codes[i, j] * scales[i, j // 128]  (float64, exact)."""
    c = np.asarray(codes, np.int64).astype(np.float64)
    s = np.asarray(scales, np.float32).astype(np.float64)
    return c * np.repeat(s, 128, axis=1)[:, :c.shape[1]]


def resplit_mats(stored, I, critical):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) in float64 at the precision UMIA chose."""
    w13 = dequant_groups(stored["q13"], stored["sq13"])
    if critical:
        w13 = w13 + dequant_groups(stored["r13"], stored["sr13"])
        w2 = dequant_groups(stored["h2"], stored["sh2"])
    else:
        w2 = dequant_groups(stored["l2"], stored["sl2"])
    return w13[:I], w13[I:], w2


def umia_threshold(theta, beta_l, gamma):
    """Theta(l, t) = (Theta * beta(l)) * gamma(t), float32."""
    return F32(F32(F32(theta) * F32(beta_l)) * F32(gamma))


def umia_critical(s, theta, beta_l, gamma):
    """Critical mask over the experts from the step's token-averaged router probability s [E] (float32)."""
    return np.asarray(s, F32) >= umia_threshold(theta, beta_l, gamma)
