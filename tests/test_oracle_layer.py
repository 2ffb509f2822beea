"""Pins for the oracle's MoE layer (CPU only).

Each check ties the oracle to something other than itself: a library routine
for a special case (torch / scipy), a hand-worked fixture, a closed form
evaluated in arbitrary precision, or a brute-force evaluation.
"""
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

mpmath = pytest.importorskip("mpmath")

from oracle.layer import (GATE_SIGMOID_RENORM, GATE_SOFTMAX_RENORM, gate_probs, gate_weights,
                          moe_layer, moe_layer_dense_masked, route, router_logits, silu, swiglu_expert,
                          topk_ids, layer_from_stored)
from synth import get_workload, gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_gate():
    d = {}
    with open(os.path.join(GOLDEN, "gate_worked.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, vals = ln.split(":", 1)
            d[key.strip()] = [float(v) for v in vals.split()]
    return d


def test_gate_worked_example():
    g = _golden_gate()
    z = np.array([g["z"]])
    k = int(g["k"][0])
    ids, gap = topk_ids(z, k)
    assert list(ids[0]) == [int(v) for v in g["ids"]]
    np.testing.assert_allclose(gate_weights(z, ids, GATE_SOFTMAX_RENORM)[0], g["softmax_w"], rtol=1e-15)
    np.testing.assert_allclose(gate_weights(z, ids, GATE_SIGMOID_RENORM)[0], g["sigmoid_w"], rtol=1e-15)
    np.testing.assert_allclose(gate_probs(z, GATE_SOFTMAX_RENORM)[0], g["softmax_probs"], rtol=1e-15)
    np.testing.assert_allclose(gate_probs(z, GATE_SIGMOID_RENORM)[0], g["sigmoid_probs"], rtol=1e-15)
    # gap is taken on float32 logits
    assert abs(gap[0] - g["gap"][0]) < 1e-7


def test_router_logits_match_library_linear():
    rng = np.random.default_rng(0)
    x, w, b = rng.standard_normal((5, 64)), rng.standard_normal((12, 64)), rng.standard_normal(12)
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(router_logits(x, w, b), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("gating", [GATE_SOFTMAX_RENORM, GATE_SIGMOID_RENORM])
def test_weights_renormalise_to_one(gating):
    rng = np.random.default_rng(1)
    z = rng.standard_normal((64, 32)) * 3
    for k in (1, 2, 8, 32):
        ids, _ = topk_ids(z, k)
        w = gate_weights(z, ids, gating)
        assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12
        assert np.all(w > 0)


def test_k_equals_E_is_library_softmax_and_k1_is_one():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((16, 8)) * 4
    ids, gap = topk_ids(z, 8)
    w = gate_weights(z, ids, GATE_SOFTMAX_RENORM)
    sm = scipy.special.softmax(z, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(sm, ids, axis=1), rtol=1e-13)
    assert np.all(np.isinf(gap))
    ws = gate_weights(z, ids, GATE_SIGMOID_RENORM)
    ex = scipy.special.expit(z)
    np.testing.assert_allclose(ws, np.take_along_axis(ex / ex.sum(1, keepdims=True), ids, axis=1), rtol=1e-13)
    ids1, _ = topk_ids(z, 1)
    assert np.all(gate_weights(z, ids1, GATE_SOFTMAX_RENORM) == 1.0)
    assert np.all(gate_weights(z, ids1, GATE_SIGMOID_RENORM) == 1.0)


def test_softmax_is_shift_safe_for_large_logits():
    z = np.array([[1000.0, 999.0, -1000.0]])
    ids, _ = topk_ids(z, 2)
    w = gate_weights(z, ids, GATE_SOFTMAX_RENORM)[0]
    e = np.exp(-1.0)
    np.testing.assert_allclose(w, [1 / (1 + e), e / (1 + e)], rtol=1e-14)


def test_topk_matches_torch_topk_away_from_ties():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((200, 128))
    ids, gap = topk_ids(z, 8)
    tv, ti = torch.topk(torch.from_numpy(z.astype(np.float32)), 8, dim=1)
    ok = gap >= 1e-4
    assert ok.sum() > 150
    np.testing.assert_array_equal(ids[ok], ti.numpy()[ok])
    # gap is the k-th minus the (k+1)-th float32 logit
    t9 = torch.topk(torch.from_numpy(z.astype(np.float32)), 9, dim=1).values.numpy().astype(np.float64)
    np.testing.assert_array_equal(gap, t9[:, 7] - t9[:, 8])


def test_topk_ties_go_to_lower_index():
    z = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]])
    ids, gap = topk_ids(z, 2)
    assert list(ids[0]) == [1, 2] and gap[0] == 0.0


def test_silu_closed_form_arbitrary_precision():
    mpmath.mp.dps = 40
    for a in (-20.0, -3.5, -1e-3, 0.0, 0.7, 2.0, 15.0):
        ref = mpmath.mpf(a) / (1 + mpmath.exp(-mpmath.mpf(a)))
        assert abs(silu(np.float64(a)) - float(ref)) <= 2e-16 * max(1.0, abs(float(ref)))


def test_swiglu_scalar_closed_form():
    # H = I = 1: y = c * SiLU(a x) * (b x); x=2, a=1, b=3, c=0.5 -> 0.5 * 2/(1+e^-2) * 6
    mpmath.mp.dps = 40
    ref = mpmath.mpf("0.5") * (2 / (1 + mpmath.exp(-2))) * 6
    y = swiglu_expert(np.array([[2.0]]), np.array([[1.0]]), np.array([[3.0]]), np.array([[0.5]]))
    assert abs(y[0, 0] - float(ref)) < 1e-15
    # silu on the gate only (Eq. 7): swapping gate and up changes the value
    y2 = swiglu_expert(np.array([[2.0]]), np.array([[3.0]]), np.array([[1.0]]), np.array([[0.5]]))
    assert abs(y2[0, 0] - y[0, 0]) > 0.1


def test_swiglu_matches_library_composition():
    rng = np.random.default_rng(4)
    H, I = 48, 20
    x = rng.standard_normal((3, H))
    wg, wu, wd = rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I))
    t = lambda a: torch.from_numpy(a)
    ref = F.linear(F.silu(F.linear(t(x), t(wg))) * F.linear(t(x), t(wu)), t(wd)).numpy()
    np.testing.assert_allclose(swiglu_expert(x, wg, wu, wd), ref, rtol=1e-12, atol=1e-12)


def _tiny_problem(seed=5, E=6, H=32, I=16, T=5, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    w_r = rng.standard_normal((E, H)) * 0.2
    b = rng.standard_normal(E) * 0.3
    experts = {e: (rng.standard_normal((I, H)) * 0.1, rng.standard_normal((I, H)) * 0.1,
                   rng.standard_normal((H, I)) * 0.1) for e in range(E)}
    shared = (rng.standard_normal((I, H)) * 0.1, rng.standard_normal((I, H)) * 0.1, rng.standard_normal((H, I)) * 0.1)
    return x, w_r, b, experts, shared, k


@pytest.mark.parametrize("gating", [GATE_SOFTMAX_RENORM, GATE_SIGMOID_RENORM])
@pytest.mark.parametrize("with_shared", [False, True])
def test_sparse_equals_dense_masked_bitwise(gating, with_shared):
    x, w_r, b, experts, shared, k = _tiny_problem()
    r = route(x, w_r, b, k, gating)
    sh = shared if with_shared else None
    sparse = moe_layer(x, r, experts, sh)
    dense = moe_layer_dense_masked(x, r, experts, len(experts), sh)
    np.testing.assert_array_equal(sparse, dense)


def test_E1_k1_is_textbook_swiglu_ffn():
    x, w_r, b, experts, _, _ = _tiny_problem(E=1, k=1)
    r = route(x, w_r, b, 1, GATE_SOFTMAX_RENORM)
    out = moe_layer(x, r, experts)
    t = lambda a: torch.from_numpy(a)
    wg, wu, wd = experts[0]
    ref = F.linear(F.silu(F.linear(t(x), t(wg))) * F.linear(t(x), t(wu)), t(wd)).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_layer_matches_library_composition():
    """Whole layer vs. torch: linear -> softmax -> topk -> renorm -> per-token expert sum."""
    x, w_r, b, experts, shared, k = _tiny_problem(seed=9, E=8, T=7, k=3)
    r = route(x, w_r, b, k, GATE_SOFTMAX_RENORM)
    out = moe_layer(x, r, experts, shared)
    t = lambda a: torch.from_numpy(a)
    logits = F.linear(t(x), t(w_r), t(b))
    p = torch.softmax(logits, dim=-1)
    tw, ti = torch.topk(p, k, dim=-1)
    tw = tw / tw.sum(-1, keepdim=True)
    ref = torch.zeros_like(t(x))
    for tt in range(x.shape[0]):
        for j in range(k):
            wg, wu, wd = (t(m) for m in experts[int(ti[tt, j])])
            ref[tt] += tw[tt, j] * F.linear(F.silu(F.linear(t(x[tt]), wg)) * F.linear(t(x[tt]), wu), wd)
        wg, wu, wd = (t(m) for m in shared)
        ref[tt] += F.linear(F.silu(F.linear(t(x[tt]), wg)) * F.linear(t(x[tt]), wu), wd)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_tiny_workload_from_stored_inputs_runs_and_is_sparse():
    wl = get_workload("tiny")
    w_r, b = gen.router_stored(wl, 0)
    x = gen.store_act(wl, gen.decode_hidden(wl, 0, 4, 1)[0])
    experts = {e: gen.expert_stored(wl, 0, e) for e in range(wl.E)}
    out, r = layer_from_stored(x, wl.act_dtype, w_r, b, experts, wl.weight_dtype, wl.I, wl.k, wl.gating)
    assert out.shape == (4, wl.H) and np.isfinite(out).all()
    # changing an unselected expert's weights leaves the output unchanged
    unused = sorted(set(range(wl.E)) - set(r["ids"].ravel().tolist()))
    assert unused
    experts2 = dict(experts)
    experts2[unused[0]] = {kk: np.zeros_like(v) for kk, v in experts[unused[0]].items()}
    out2, _ = layer_from_stored(x, wl.act_dtype, w_r, b, experts2, wl.weight_dtype, wl.I, wl.k, wl.gating)
    np.testing.assert_array_equal(out, out2)
