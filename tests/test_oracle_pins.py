"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

No page prints a worked numeric example of the layer, so the oracle is pinned
by closed forms, special cases that reduce to a library routine (numpy,
scipy), brute force on tiny inputs, invariants the pages state, and the one
printed plan record.  Each test names what it pins; together they are chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t):
    return t.double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _swiglu_np(x, Wg, Wu, Wd):
    """Plain SwiGLU MLP with numpy matmuls: Wd @ (silu(Wg @ x) * (Wu @ x))."""
    g = x @ Wg.T
    u = x @ Wu.T
    h = scipy.special.expit(g) * g * u
    return h @ Wd.T


def _identity_router(scores):
    """x = scores, Wr = I so that logit[t, e] == scores[t, e] exactly."""
    T, E = scores.shape
    return np.ascontiguousarray(scores, np.float64), np.eye(E, dtype=np.float64)


# ---------------------------------------------------------------- bf16 reader
def test_bf16_widening_matches_torch():
    """The oracle's own bf16 decoder equals torch's bf16 -> fp64 conversion."""
    g = torch.Generator().manual_seed(3)
    a = (torch.randn(4096, generator=g) * 37).to(torch.bfloat16)
    a[:4] = torch.tensor([0.0, -0.0, 1e-40, -3.0e38]).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.widen(a), a.double().numpy())


# ---------------------------------------------------------------- top-k
@pytest.mark.parametrize("E,k", [(4, 2), (6, 3), (5, 1), (6, 6)])
def test_topk_exhaustive(E, k):
    """Top-k set = the k-subset with the largest score sum (unique for distinct scores),
    found by enumerating every subset; the ids come out in descending score."""
    rng = np.random.default_rng(E * 10 + k)
    scores = rng.standard_normal((40, E))
    x, Wr = _identity_router(scores)
    ids, _ = oracle.route(x, Wr, k, oracle.GATE_SOFTMAX)
    for t in range(scores.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda c: scores[t, list(c)].sum())
        assert set(ids[t].tolist()) == set(best)
        assert np.all(np.diff(scores[t, ids[t]]) < 0)


def test_topk_matches_stable_argsort():
    """Against numpy's stable argsort of the negated scores, including exact ties
    (ties go to the lower expert index)."""
    rng = np.random.default_rng(1)
    scores = np.round(rng.standard_normal((200, 40)), 1)  # many exact ties
    x, Wr = _identity_router(scores)
    ids, _ = oracle.route(x, Wr, 7, oracle.GATE_SOFTMAX)
    ref = np.argsort(-scores, axis=1, kind="stable")[:, :7]
    np.testing.assert_array_equal(ids, ref)


def test_sigmoid_selection_uses_bias_but_weights_do_not():
    """Sigmoid family: selection on sigmoid(l) + b; weights from the unbiased sigmoid."""
    rng = np.random.default_rng(2)
    T, E, k = 64, 12, 4
    logits = rng.standard_normal((T, E))
    bias = rng.uniform(-0.3, 0.3, E)
    x, Wr = _identity_router(logits)
    ids, w = oracle.route(x, Wr, k, oracle.GATE_SIGMOID, norm_topk=0, routed_scaling=1.0,
                          sel_bias=bias)
    s = scipy.special.expit(logits)
    ref_ids = np.argsort(-(s + bias), axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, np.take_along_axis(s, ref_ids, 1), rtol=1e-14, atol=0)


def test_sigmoid_forced_selection():
    """A +10 selection bias on expert e puts e first for every token."""
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((32, 9))
    bias = np.zeros(9)
    bias[5] = 10.0
    x, Wr = _identity_router(logits)
    ids, _ = oracle.route(x, Wr, 3, oracle.GATE_SIGMOID, sel_bias=bias)
    assert np.all(ids[:, 0] == 5)


# ---------------------------------------------------------------- gate weights
def test_softmax_weights_are_softmax_probabilities():
    """Softmax family, no renormalisation: w_j = softmax(l)[id_j] (scipy); with k = E
    the weights sum to one (closed form)."""
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 8)) * 3
    x, Wr = _identity_router(logits)
    ids, w = oracle.route(x, Wr, 3, oracle.GATE_SOFTMAX)
    p = scipy.special.softmax(logits, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13, atol=0)
    ids8, w8 = oracle.route(x, Wr, 8, oracle.GATE_SOFTMAX)
    np.testing.assert_allclose(w8.sum(1), 1.0, rtol=0, atol=1e-14)


def test_softmax_logit_bias_enters_selection_and_weights():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((40, 10))
    lb = rng.standard_normal(10)
    x, Wr = _identity_router(logits)
    ids, w = oracle.route(x, Wr, 4, oracle.GATE_SOFTMAX, logit_bias=lb)
    l2 = logits + lb
    p = scipy.special.softmax(l2, axis=1)
    np.testing.assert_array_equal(ids, np.argsort(-l2, axis=1, kind="stable")[:, :4])
    np.testing.assert_allclose(w, np.take_along_axis(p, ids, 1), rtol=1e-13, atol=0)


def test_sigmoid_normalised_weights_sum_to_routed_scaling():
    """norm_topk=1: weights are s_j / sum(s_sel) * rs, so they sum to rs (closed form)."""
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((64, 16))
    x, Wr = _identity_router(logits)
    ids, w = oracle.route(x, Wr, 5, oracle.GATE_SIGMOID, norm_topk=1, routed_scaling=2.5,
                          sel_bias=rng.uniform(-0.1, 0.1, 16))
    np.testing.assert_allclose(w.sum(1), 2.5, rtol=0, atol=1e-12)
    s = scipy.special.expit(np.take_along_axis(logits, ids, 1))
    np.testing.assert_allclose(w, 2.5 * s / s.sum(1, keepdims=True), rtol=1e-13, atol=0)


def test_router_logits_are_x_times_router_transpose():
    """Router logits = x @ Wr^T (+ logit bias) with a library matmul; bf16 inputs read
    exactly as stored."""
    cfg = LayerConfig("t", T=33, d=64, E=12, I=32, k=3)
    inp = make_inputs(cfg, seed=11)
    lb = np.linspace(-1, 1, 12)
    logits, scores = oracle.router_scores(inp["x"], inp["Wr"], oracle.GATE_SOFTMAX, logit_bias=lb)
    ref = _f64(inp["x"]) @ _f64(inp["Wr"]).T + lb
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(scores, logits)
    sb = np.linspace(-0.1, 0.1, 12)
    l2, s2 = oracle.router_scores(inp["x"], inp["Wr"], oracle.GATE_SIGMOID, sel_bias=sb)
    np.testing.assert_allclose(s2, scipy.special.expit(l2) + sb, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- dispatch plan
def _plan_invariants(ids, E, S, p):
    T, k = ids.shape
    ks = k + S
    off, tok, sr = p["expert_offsets"], p["token_indices"], p["slot_row"]
    assert off[0] == 0 and off[-1] == T * ks and np.all(np.diff(off) >= 0)
    # each (token, slot) pair is in exactly one batch row: slot_row is a bijection
    assert sorted(sr.ravel().tolist()) == list(range(T * ks))
    for t in range(T):
        for j in range(ks):
            pos = sr[t, j]
            e = ids[t, j] if j < k else E + (j - k)
            assert tok[pos] == t
            assert off[e] <= pos < off[e + 1]
    for e in range(E + S):
        b = tok[off[e]:off[e + 1]]
        assert np.all(np.diff(b) > 0)  # ascending, each token once per expert
    for s in range(S):
        np.testing.assert_array_equal(tok[off[E + s]:off[E + s + 1]], np.arange(T))
    counts = np.diff(off)
    np.testing.assert_array_equal(p["active_ids"], np.nonzero(counts)[0])


@pytest.mark.parametrize("T,E,k,S", [(1, 4, 2, 0), (17, 8, 3, 1), (64, 16, 2, 0), (50, 40, 8, 2)])
def test_plan_partitions_routing(T, E, k, S):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = oracle.plan(ids, E, S)
    _plan_invariants(ids, E, S, p)
    # the batches are a stable sort of the token-major pair list by expert id (numpy)
    flat_e = np.concatenate([ids, np.tile(E + np.arange(S), (T, 1))], 1).ravel()
    order = np.argsort(flat_e, kind="stable")
    np.testing.assert_array_equal(p["token_indices"], order // (k + S))


def test_plan_empty_batch_and_no_tokens():
    ids = np.array([[0, 2], [2, 0]], np.int32)
    p = oracle.plan(ids, 5, 0)
    assert list(p["expert_offsets"]) == [0, 2, 2, 4, 4, 4]
    assert list(p["active_ids"]) == [0, 2]
    p0 = oracle.plan(np.zeros((0, 3), np.int32), 4, 1)
    assert list(p0["expert_offsets"]) == [0] * 6 and p0["n_active"] == 0


def test_plan_rejects_out_of_range_ids():
    with pytest.raises(RuntimeError):
        oracle.plan(np.array([[0, 4]], np.int32), 4, 0)
    with pytest.raises(RuntimeError):
        oracle.plan(np.array([[-1, 1]], np.int32), 4, 0)


def test_plan_matches_printed_example():
    """The dispatch-plan record printed on the tenzro page: expert 1 of layer 0 gets the
    batch token_indices [0, 1, 4, 9]; token 0's assignment lists its slots."""
    with open(os.path.join(GOLDEN, "plan_dispatch_example.json")) as f:
        ex = json.load(f)
    ids = np.array(ex["routings"], np.int32)
    p = oracle.plan(ids, ex["E"], 0)
    off, tok = p["expert_offsets"], p["token_indices"]
    e = ex["expert"]
    assert tok[off[e]:off[e + 1]].tolist() == ex["token_indices"]
    # token 0's slots point at rows of the batches of the experts it selected
    for j, ej in enumerate(ids[0]):
        assert off[ej] <= p["slot_row"][0, j] < off[ej + 1]


# ---------------------------------------------------------------- FFN and combine
def _tiny(seed=0, T=9, d=16, E=5, I=8, k=2, S=0, gate=oracle.GATE_SOFTMAX, dtype="f32"):
    cfg = LayerConfig("t", T=T, d=d, E=E, I=I, k=k, S=S, gate=gate, dtype=dtype)
    return cfg, make_inputs(cfg, seed=seed)


def test_single_expert_is_plain_swiglu_mlp():
    """E = 1, k = 1, softmax => w = 1, so y is a SwiGLU MLP (numpy matmuls)."""
    cfg, inp = _tiny(E=1, k=1, T=7)
    y, ids, w = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 1,
                               oracle.GATE_SOFTMAX)
    assert np.all(ids == 0) and np.all(w == 1.0)
    ref = _swiglu_np(_f64(inp["x"]), _f64(inp["Wg"][0]), _f64(inp["Wu"][0]), _f64(inp["Wd"][0]))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_k_equals_E_is_dense_softmax_mixture():
    """k = E => y = sum_e softmax(l)_e * FFN_e(x): a dense mixture (numpy einsum)."""
    cfg, inp = _tiny(E=4, k=4, T=6)
    x = _f64(inp["x"])
    y, _, _ = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 4,
                             oracle.GATE_SOFTMAX)
    p = scipy.special.softmax(x @ _f64(inp["Wr"]).T, axis=1)
    Wg, Wu, Wd = _f64(inp["Wg"]), _f64(inp["Wu"]), _f64(inp["Wd"])
    g = np.einsum("td,eid->tei", x, Wg)
    u = np.einsum("td,eid->tei", x, Wu)
    h = g * scipy.special.expit(g) * u
    ref = np.einsum("te,tei,edi->td", p, h, Wd)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_shared_expert_has_weight_one():
    """Zero the routed experts' down projections => y is exactly the shared expert's
    SwiGLU output (weight 1.0); zero the shared one => y is the routed part alone."""
    cfg, inp = _tiny(E=6, k=2, S=1, gate=oracle.GATE_SIGMOID, T=11)
    Wd0 = inp["Wd"].clone()
    Wd0[:6] = 0
    y, _, _ = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], Wd0, 2,
                             oracle.GATE_SIGMOID, S=1, norm_topk=1, routed_scaling=2.0)
    ref = _swiglu_np(_f64(inp["x"]), _f64(inp["Wg"][6]), _f64(inp["Wu"][6]), _f64(inp["Wd"][6]))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    Wd1 = inp["Wd"].clone()
    Wd1[6] = 0
    y1, _, _ = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], Wd1, 2,
                              oracle.GATE_SIGMOID, S=1, norm_topk=1, routed_scaling=2.0)
    y0, _, _ = oracle.forward(inp["x"], inp["Wr"], inp["Wg"][:6], inp["Wu"][:6], inp["Wd"][:6],
                              2, oracle.GATE_SIGMOID, S=0, norm_topk=1, routed_scaling=2.0)
    np.testing.assert_allclose(y1, y0, rtol=1e-13, atol=1e-14)
    # and the routed part is the gate-weighted sum of the selected experts (numpy)
    x = _f64(inp["x"])
    _, ids, w = oracle.forward(inp["x"], inp["Wr"], inp["Wg"][:6], inp["Wu"][:6], inp["Wd"][:6],
                               2, oracle.GATE_SIGMOID, norm_topk=1, routed_scaling=2.0)
    ref0 = np.zeros_like(y0)
    for t in range(x.shape[0]):
        for j in range(2):
            e = ids[t, j]
            ref0[t] += w[t, j] * _swiglu_np(x[t], _f64(inp["Wg"][e]), _f64(inp["Wu"][e]),
                                            _f64(inp["Wd"][e]))
    np.testing.assert_allclose(y0, ref0, rtol=1e-12, atol=1e-13)


def test_expert_contribution_is_linear_in_its_down_projection():
    """Doubling Wd_e doubles expert e's share of y and leaves routing unchanged."""
    cfg, inp = _tiny(E=5, k=2, T=10)
    args = (inp["x"], inp["Wr"], inp["Wg"], inp["Wu"])
    y, ids, w = oracle.forward(*args, inp["Wd"], 2, oracle.GATE_SOFTMAX)
    Wd2 = inp["Wd"].clone()
    Wd2[3] *= 2
    y2, ids2, w2 = oracle.forward(*args, Wd2, 2, oracle.GATE_SOFTMAX)
    np.testing.assert_array_equal(ids, ids2)
    Wd3 = torch.zeros_like(inp["Wd"])
    Wd3[3] = inp["Wd"][3]
    y3, _, _ = oracle.forward(*args, Wd3, 2, oracle.GATE_SOFTMAX)  # expert 3's share alone
    np.testing.assert_allclose(y2 - y, y3, rtol=1e-11, atol=1e-13)
    assert np.abs(y3).max() > 0


def test_token_and_expert_permutation():
    """Permuting tokens permutes y; relabelling experts (router rows, biases and expert
    weights together) leaves y unchanged."""
    cfg, inp = _tiny(E=7, k=3, S=1, gate=oracle.GATE_SIGMOID, T=12, seed=5)
    sb = np.linspace(-0.05, 0.05, 7)
    kw = dict(S=1, norm_topk=1, routed_scaling=1.5, sel_bias=sb)
    y, _, _ = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 3,
                             oracle.GATE_SIGMOID, **kw)
    tp = np.random.default_rng(0).permutation(12)
    yt, _, _ = oracle.forward(inp["x"][tp], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 3,
                              oracle.GATE_SIGMOID, **kw)
    np.testing.assert_allclose(yt, y[tp], rtol=1e-13, atol=1e-14)
    ep = np.random.default_rng(1).permutation(7)
    full = np.concatenate([ep, [7]])
    kw2 = dict(kw, sel_bias=sb[ep])
    ye, _, _ = oracle.forward(inp["x"], inp["Wr"][ep], inp["Wg"][full], inp["Wu"][full],
                              inp["Wd"][full], 3, oracle.GATE_SIGMOID, **kw2)
    np.testing.assert_allclose(ye, y, rtol=1e-12, atol=1e-13)


def test_residual_is_added():
    cfg, inp = _tiny(T=8)
    res = np.random.default_rng(0).standard_normal((8, 16))
    args = (inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 2, oracle.GATE_SOFTMAX)
    y, _, _ = oracle.forward(*args)
    yr, _, _ = oracle.forward(*args, residual=res)
    np.testing.assert_allclose(yr, y + res, rtol=1e-14, atol=1e-14)


def test_sample_rows_equal_full_rows():
    cfg, inp = _tiny(T=20, E=6, k=2)
    args = (inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 2, oracle.GATE_SOFTMAX)
    y, ids, w = oracle.forward(*args)
    sample = np.array([19, 0, 7, 7], np.int32)
    ys, ids_s, w_s = oracle.forward(*args, tokens=sample)
    np.testing.assert_array_equal(ys, y[sample])
    np.testing.assert_array_equal(ids_s, ids[sample])
    # experts no sampled token uses may be left out
    used = set(ids_s.ravel().tolist())
    Wg_l = [inp["Wg"][e] if e in used else None for e in range(6)]
    Wu_l = [inp["Wu"][e] if e in used else None for e in range(6)]
    Wd_l = [inp["Wd"][e] if e in used else None for e in range(6)]
    ys2, _, _ = oracle.forward(inp["x"], inp["Wr"], Wg_l, Wu_l, Wd_l, 2, oracle.GATE_SOFTMAX,
                               tokens=sample)
    np.testing.assert_array_equal(ys2, ys)


def test_bf16_storage_is_read_exactly():
    """bf16 weights give bit-identical results to the same values stored as fp32."""
    cfg, inp = _tiny(T=9, E=5, k=2, dtype="bf16", S=1, gate=oracle.GATE_SIGMOID)
    kw = dict(S=1, norm_topk=1, routed_scaling=2.0)
    y, ids, w = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 2,
                               oracle.GATE_SIGMOID, **kw)
    f = lambda t: t.float()
    y2, ids2, w2 = oracle.forward(f(inp["x"]), f(inp["Wr"]), f(inp["Wg"]), f(inp["Wu"]),
                                  f(inp["Wd"]), 2, oracle.GATE_SIGMOID, **kw)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(ids, ids2)


# ---------------------------------------------------------------- exactness of sharding
@pytest.mark.parametrize("gate,S", [(oracle.GATE_SOFTMAX, 0), (oracle.GATE_SIGMOID, 1)])
def test_sharded_equals_monolithic(gate, S):
    """Grouping the work by expert is an exact regrouping: the pages report
    max|delta| = 3.6e-12; in fp64 the two orders agree to rounding (<= 1e-12 of max|y|)."""
    cfg = LayerConfig("t", T=40, d=32, E=8, I=16, k=3, S=S, gate=gate)
    inp = make_inputs(cfg, seed=2)
    kw = dict(S=S, norm_topk=1 if gate else 0, routed_scaling=2.5 if gate else 1.0,
              sel_bias=np.linspace(-0.1, 0.1, 8) if gate else None)
    args = (inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 3, gate)
    y, ids, w = oracle.forward(*args, **kw)
    ys, ids_s, w_s = oracle.forward_sharded(*args, **kw)
    np.testing.assert_array_equal(ids, ids_s)
    np.testing.assert_array_equal(w, w_s)
    assert np.abs(ys - y).max() <= 1e-12 * np.abs(y).max()


def test_each_pair_computed_once():
    """Each selected (token, expert) pair is computed exactly once: zeroing every
    expert but one leaves, per token, w * FFN_e(x) if the token selected e and zero
    otherwise (no double counting, no missing pair)."""
    cfg, inp = _tiny(T=30, E=6, k=3, seed=9)
    x = _f64(inp["x"])
    for e in range(6):
        Wd = torch.zeros_like(inp["Wd"])
        Wd[e] = inp["Wd"][e]
        y, ids, w = oracle.forward_sharded(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], Wd, 3,
                                           oracle.GATE_SOFTMAX)
        fe = _swiglu_np(x, _f64(inp["Wg"][e]), _f64(inp["Wu"][e]), _f64(inp["Wd"][e]))
        weight = np.where(ids == e, w, 0.0).sum(1)
        np.testing.assert_allclose(y, weight[:, None] * fe, rtol=1e-12, atol=1e-13)


def test_errors_are_reported():
    cfg, inp = _tiny()
    with pytest.raises(RuntimeError):  # k > E
        oracle.route(inp["x"], inp["Wr"], 6, oracle.GATE_SOFTMAX)
    with pytest.raises(RuntimeError):  # selection bias belongs to the sigmoid family
        oracle.route(inp["x"], inp["Wr"], 2, oracle.GATE_SOFTMAX, sel_bias=np.zeros(5))


# ---------------------------------------------------------------- per-call pieces
def test_expert_rows_is_swiglu_on_gathered_rows():
    """One expert over a token list = the numpy SwiGLU MLP of the gathered rows."""
    cfg, inp = _tiny(T=12, E=3, k=1, d=24, I=40)
    toks = np.array([11, 0, 5, 5, 3], np.int32)
    out = oracle.expert_rows(inp["x"], inp["Wg"][2], inp["Wu"][2], inp["Wd"][2], toks)
    ref = _swiglu_np(_f64(inp["x"])[toks], _f64(inp["Wg"][2]), _f64(inp["Wu"][2]),
                     _f64(inp["Wd"][2]))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_combine_is_weighted_gather():
    """Combine = weighted gather-sum of batch rows (numpy einsum), shared rows weight 1;
    with k = 1, w = 1, S = 0 it is a plain row gather (exact)."""
    rng = np.random.default_rng(12)
    T, d, k, S = 9, 16, 3, 1
    P = T * (k + S)
    rows = rng.standard_normal((P, d))
    slot_row = rng.permutation(P).astype(np.int32).reshape(T, k + S)
    w = rng.uniform(0, 1, (T, k))
    res = rng.standard_normal((T, d))
    y = oracle.combine(rows, slot_row, k, S, w=w, residual=res)
    wfull = np.concatenate([w, np.ones((T, S))], 1)
    ref = np.einsum("tj,tjd->td", wfull, rows[slot_row]) + res
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)
    sr1 = rng.permutation(T).astype(np.int32).reshape(T, 1)
    np.testing.assert_array_equal(oracle.combine(rows[:T], sr1, 1, 0), rows[:T][sr1[:, 0]])
    # unweighted form equals weights of one
    np.testing.assert_allclose(oracle.combine(rows, slot_row, k, S),
                               oracle.combine(rows, slot_row, k, S, w=np.ones((T, k))),
                               rtol=0, atol=0)


def test_sharded_pieces_compose_to_forward():
    """route -> plan -> expert_rows per batch -> combine reproduces forward()."""
    cfg, inp = _tiny(T=21, E=6, k=2, S=1, gate=oracle.GATE_SIGMOID, seed=4)
    kw = dict(norm_topk=1, routed_scaling=2.5, sel_bias=np.linspace(-0.1, 0.1, 6))
    y, ids, w = oracle.forward(inp["x"], inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"], 2,
                               oracle.GATE_SIGMOID, S=1, **kw)
    ids2, w2 = oracle.route(inp["x"], inp["Wr"], 2, oracle.GATE_SIGMOID, **kw)
    p = oracle.plan(ids2, 6, 1)
    off, tok = p["expert_offsets"], p["token_indices"]
    rows = np.zeros((21 * 3, 16))
    for e in range(7):
        if off[e + 1] > off[e]:
            rows[off[e]:off[e + 1]] = oracle.expert_rows(inp["x"], inp["Wg"][e], inp["Wu"][e],
                                                         inp["Wd"][e], tok[off[e]:off[e + 1]])
    y2 = oracle.combine(rows, p["slot_row"], 2, 1, w=w2)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- partial combine
def _partial_case(seed=3, T=12, k=3, S=1, E=6):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.05, 1.0, (T, k))
    p = oracle.plan(ids, E, S)
    return rng, ids, w, p


def test_partial_combine_with_everyone_responding_is_the_plain_combine():
    rng, ids, w, p = _partial_case()
    rows = rng.standard_normal((12 * 4, 10))
    y, missing = oracle.combine_partial(rows, p["slot_row"], ids, w, np.ones(7), 3, 1, 6)
    np.testing.assert_array_equal(y, oracle.combine(rows, p["slot_row"], 3, 1, w=w))
    assert missing.sum() == 0


def test_partial_combine_effective_weights():
    """Unit-vector rows expose every slot's effective weight: unavailable slots
    weigh 0, responding routed slots w * mass / resp (numpy), so the routed mass
    sum_j w_j is kept; an unavailable shared expert drops out."""
    rng, ids, w, p = _partial_case(T=10)
    P = 10 * 4
    avail = np.ones(7, np.int32)
    avail[[1, 4, 6]] = 0  # two routed experts and the shared one are down
    y, missing = oracle.combine_partial(np.eye(P), p["slot_row"], ids, w, avail, 3, 1, 6)
    sr = p["slot_row"]
    for t in range(10):
        ok = avail[ids[t]] == 1
        eff = y[t, sr[t, :3]]
        if ok.any():
            np.testing.assert_allclose(eff, np.where(ok, w[t] * w[t].sum() / w[t][ok].sum(), 0),
                                       rtol=1e-14, atol=0)
            np.testing.assert_allclose(eff.sum(), w[t].sum(), rtol=1e-14)
        else:
            assert np.all(eff == 0)
        assert y[t, sr[t, 3]] == 0.0  # shared expert down
        np.testing.assert_array_equal(missing[t], np.r_[~ok, True].astype(np.int32))


def test_partial_combine_is_a_reduced_top_k():
    """With the sigmoid family's normalised weights, renormalising over the
    responding experts gives rs * s_j / sum over responding s (scipy), i.e. the
    weights of the same routing with the missing experts left out."""
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((20, 9))
    x = np.ascontiguousarray(logits)
    ids, w = oracle.route(x, np.eye(9), 4, oracle.GATE_SIGMOID, norm_topk=1, routed_scaling=2.5)
    p = oracle.plan(ids, 9, 0)
    avail = np.ones(9, np.int32)
    avail[[0, 5]] = 0
    y, _ = oracle.combine_partial(np.eye(20 * 4), p["slot_row"], ids, w, avail, 4, 0, 9)
    s = scipy.special.expit(np.take_along_axis(logits, ids, 1))
    ok = avail[ids] == 1
    for t in range(20):
        if not ok[t].any():
            continue
        ref = np.where(ok[t], 2.5 * s[t] / s[t][ok[t]].sum(), 0.0)
        np.testing.assert_allclose(y[t, p["slot_row"][t]], ref, rtol=1e-13, atol=1e-15)


def test_missing_pairs_hand_example():
    """Three tokens, top-2 of four experts plus one shared expert (index 4);
    expert 2 and the shared expert are down."""
    ids = np.array([[0, 2], [3, 1], [2, 0]], np.int32)
    avail = np.array([1, 1, 0, 1, 0], np.int32)
    pairs = oracle.missing_pairs(ids, avail, k=2, S=1, E=4)
    assert pairs.tolist() == [[2, 0], [4, 0], [4, 1], [2, 2], [4, 2]]
    assert oracle.missing_pairs(ids, np.ones(5, np.int32), 2, 1, 4).shape == (0, 2)


def test_missing_pairs_list_the_flagged_slots():
    """The list is the partial combine's missing mask read in row-major order
    (numpy argwhere), each slot mapped to its expert."""
    rng, ids, w, p = _partial_case(seed=5, T=30)
    avail = (rng.uniform(size=7) < 0.6).astype(np.int32)
    _, missing = oracle.combine_partial(np.eye(30 * 4), p["slot_row"], ids, w, avail, 3, 1, 6)
    experts = np.concatenate([ids, np.full((30, 1), 6, np.int32)], axis=1)
    want = [[int(experts[t, j]), int(t)] for t, j in np.argwhere(missing == 1)]
    assert oracle.missing_pairs(ids, avail, 3, 1, 6).tolist() == want


# ---------------------------------------------------------------- Q8_0 weights
def test_q8_0_rounds_exact_halves_away_from_zero():
    """A block whose largest magnitude is 127 has d = 1 and 1/d = 1 exactly, so
    each code is round(w) of the stored value itself; the halves settle the
    rounding rule of the reading taken (round half away from zero, as GGUF's
    encoder does), which round-half-to-even would break on 0.5, 2.5 and -0.5."""
    import torch
    w = torch.zeros((1, 1, 32), dtype=torch.float32)
    vals = [127.0, 0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 3.5, 126.5, -126.5, 0.25, -0.75]
    w[0, 0, :len(vals)] = torch.tensor(vals)
    for dt in (torch.float32, torch.bfloat16):
        q, s = oracle.quantize_q8_0(w.to(dt))
        assert s[0, 0, 0] == 0x3C00  # f16(1.0)
        want = [127, 1, -1, 2, -2, 3, -3, 4, 127, -127, 0, -1]
        assert q[0, 0, :len(vals)].tolist() == want
        assert (q[0, 0, len(vals):] == 0).all()


def test_q8_0_round_trip_is_exact_on_representable_blocks():
    """Blocks of the form s * q (s an f16 value, integer codes with max |q| = 127)
    quantize back to exactly those codes and that scale."""
    rng = np.random.default_rng(0)
    n, R, K = 2, 5, 96
    q0 = rng.integers(-127, 128, size=(n, R, K)).astype(np.int8)
    q0[..., ::32] = 127 * rng.choice([-1, 1], size=(n, R, K // 32))  # a code of |127| per block
    s0 = rng.uniform(1e-3, 5e-2, size=(n, K // 32, R)).astype(np.float16)
    w = (s0.astype(np.float64).transpose(0, 2, 1).repeat(32, axis=2) * q0).astype(np.float32)
    q, s = oracle.quantize_q8_0(torch.from_numpy(w))
    np.testing.assert_array_equal(q, q0)
    np.testing.assert_array_equal(s, s0.view(np.uint16))
    np.testing.assert_array_equal(oracle.dequantize_q8_0(q, s), w.astype(np.float64))


def test_q8_0_error_bound_and_special_blocks():
    """|w - scale*q| <= d/2 + 127 |d - f16(d)| (d = amax/127) elementwise; max |q| is
    127 in every nonzero block; an all-zero block has scale 0 and codes 0; negating
    the input negates the codes; the scale is the f16 nearest to amax/127."""
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(3, 7, 128, generator=g) * 0.02).to(torch.bfloat16)
    w[1, 2, 32:64] = 0
    q, s = oracle.quantize_q8_0(w)
    wf = w.double().numpy()
    blocks = wf.reshape(3, 7, 4, 32)
    d = np.abs(blocks).max(-1) / 127.0                       # [3, 7, 4]
    sd = s.view(np.float16).astype(np.float64).transpose(0, 2, 1)  # [3, 7, 4]
    err = np.abs(wf - oracle.dequantize_q8_0(q, s)).reshape(3, 7, 4, 32)
    bound = d / 2 + 127 * np.abs(d - sd) + 1e-12
    assert np.all(err <= bound[..., None])
    qb = np.abs(q.astype(np.int32)).reshape(3, 7, 4, 32).max(-1)
    nz = d > 0
    assert np.all(qb[nz] == 127) and np.all(qb[~nz] == 0) and np.all(sd[~nz] == 0)
    ulp = np.spacing(np.abs(d).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(sd - d) <= ulp / 2 + 1e-18)
    qn, sn = oracle.quantize_q8_0(-w)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)
    # 32 int8 codes + one f16 scale per block: 8.5 bits per weight
    assert (q.nbytes + s.nbytes) * 8 / q.size == 8.5
