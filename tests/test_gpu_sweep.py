"""A randomized sweep of whole-layer shapes against the oracle: bf16 and fp32
layers, and the same bf16 layers with Q8_0 experts.  Shapes range from decode
sized batches (one token, top-32 of 64 experts) to batches of several hundred
rows per expert, which take the SM-pair and 256-row GEMM paths; up to two
shared experts, both gate families.  Routing must match bit for bit, gate
weights within 1e-4, outputs within the layer tolerance (Q8_0: within 1e-2 of
the oracle on the dequantized weights); the four layer calls made one by one
must give the fused call's result bit for bit.  A draw whose top-(k+1) scores cannot
be separated by the routing margin (many sigmoid scores at large k) is skipped."""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs
from tests.helpers import check_weights, host, make_case, rel_err, y_tol

DEV = "cuda"


def _draw(seed):
    rng = np.random.default_rng(50000 + seed)
    f32 = rng.random() < 0.25
    if rng.random() < 0.4:  # large batches: few experts, many rows each
        E = int(rng.integers(4, 17))
        k = int(rng.integers(1, min(E, 4) + 1))
        T = int(rng.integers(100, 601))
    else:
        E = int(rng.integers(4, 65))
        k = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.integers(1, 81))
    S = int(rng.integers(0, 3))
    gate = int(rng.integers(0, 2))
    norm = int(rng.integers(0, 2)) if gate == 0 else 1
    if f32:
        d, I = 8 * int(rng.integers(2, 33)), 4 * int(rng.integers(2, 65))
    else:
        d, I = 64 * int(rng.integers(1, 7)), 64 * int(rng.integers(1, 7))
        while (E + S) * min(d, I) < 128:
            d, I = d + 64, I + 64
    return LayerConfig("sweep_%d" % seed, T=T, d=d, E=E, I=I, k=k, S=S, gate=gate,
                       norm_topk=norm, routed_scaling=2.5 if gate else 1.0,
                       sel_bias_range=0.1 if gate else 0.0, dtype="f32" if f32 else "bf16")


def _deq(W):
    q, s = oracle.quantize_q8_0(host(W))
    return oracle.dequantize_q8_0(q, s)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(60))
def test_layer_random_sweep(seed):
    cfg = _draw(seed)
    try:
        inp = make_case(cfg, seed=seed, device=DEV)
    except RuntimeError as e:
        pytest.skip(str(e))
    kw = dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
              logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    desc = moe.desc_from_config(cfg)
    layer = moe.MoeLayer(desc, inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"],
                         logit_bias=inp["logit_bias"], sel_bias=inp["sel_bias"])
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    y = layer.forward(inp["x"], topk_ids=ids, topk_w=w)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate, **kw)
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    check_weights(host(w).numpy(), w_ref, inp, cfg)
    y_ref, _, _ = oracle.forward(host(inp["x"]), host(inp["Wr"]), host(inp["Wg"]),
                                 host(inp["Wu"]), host(inp["Wd"]), cfg.k, cfg.gate, S=cfg.S,
                                 **kw)
    assert rel_err(host(y).double().numpy(), y_ref) <= y_tol(cfg), cfg
    # the four layer calls one by one give the fused call's routing and output
    # bit for bit (the FFN call gathers rows by token_indices where the fused
    # call scatters them by slot_row; both leave the gate weights to the combine)
    P, i32 = cfg.T * (cfg.k + cfg.S), torch.int32
    ws2 = moe.alloc_workspace(desc)
    ids2, w2 = torch.empty_like(ids), torch.empty_like(w)
    moe.moe_route(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"], ids2, w2, ws2)
    off = torch.empty((cfg.E + cfg.S + 1,), dtype=i32, device=DEV)
    tok = torch.empty((P,), dtype=i32, device=DEV)
    sr = torch.empty((cfg.T, cfg.k + cfg.S), dtype=i32, device=DEV)
    moe.moe_plan_dispatch(desc, ids2, None, off, tok, sr, None, None, None, ws2)
    y_perm = torch.empty((P, cfg.d), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn(desc, inp["x"], off, tok, None, inp["Wg"], inp["Wu"], inp["Wd"], y_perm,
                       ws2)
    y2 = torch.empty_like(y)
    moe.moe_combine(desc, y_perm, sr, w2, None, y2)
    assert moe.moe_get_device_status(ws2) == moe.MOE_OK
    assert torch.equal(ids2, ids) and torch.equal(w2, w) and torch.equal(y2, y), cfg
    if cfg.dtype != "bf16":
        return
    Wq = [moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd")]
    lq = moe.MoeLayer(desc, inp["Wr"], *Wq, logit_bias=inp["logit_bias"],
                      sel_bias=inp["sel_bias"])
    yq = lq.forward(inp["x"])
    assert moe.moe_get_device_status(lq.ws) == moe.MOE_OK
    yq_ref, _, _ = oracle.forward(host(inp["x"]), oracle.widen(host(inp["Wr"])), _deq(inp["Wg"]),
                                  _deq(inp["Wu"]), _deq(inp["Wd"]), cfg.k, cfg.gate, S=cfg.S,
                                  **kw)
    assert rel_err(host(yq).double().numpy(), yq_ref) <= 1e-2, cfg


def _host_copy(t):
    h = moe.host_empty(t.shape, t.dtype)
    h.copy_(t)
    return h


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(24))
def test_tier_random_sweep_equals_resident(seed):
    """The expert tier (experts in host memory, a random number of HBM slots,
    down to one) gives the resident layer's output and routing bit for bit."""
    rng = np.random.default_rng(70000 + seed)
    big = rng.random() < 0.3
    E = int(rng.integers(4, 13)) if big else int(rng.integers(4, 49))
    k = int(rng.integers(1, min(E, 4 if big else 8) + 1))
    T = int(rng.integers(100, 401)) if big else int(rng.integers(1, 65))
    S = int(rng.integers(0, 3))
    gate = int(rng.integers(0, 2))
    d, I = 64 * int(rng.integers(1, 5)), 64 * int(rng.integers(1, 5))
    while (E + S) * min(d, I) < 128:
        d, I = d + 64, I + 64
    cfg = LayerConfig("tier_sweep_%d" % seed, T=T, d=d, E=E, I=I, k=k, S=S, gate=gate,
                      norm_topk=gate, routed_scaling=2.5 if gate else 1.0,
                      sel_bias_range=0.1 if gate else 0.0)
    slots = int(rng.integers(1, E + S + 1))
    inp = make_inputs(cfg, seed=seed, device=DEV)
    desc = moe.desc_from_config(cfg)
    layer = moe.MoeLayer(desc, inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"],
                         logit_bias=inp["logit_bias"], sel_bias=inp["sel_bias"])
    tier = moe.ExpertTier(desc, inp["Wr"], *(_host_copy(inp[n]) for n in ("Wg", "Wu", "Wd")),
                          slots * 3 * I * d * 2, logit_bias=inp["logit_bias"],
                          sel_bias=inp["sel_bias"])
    try:
        g = torch.Generator(device=DEV).manual_seed(seed)
        for _ in range(3):
            x = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
            ids_ref = torch.empty((T, k), dtype=torch.int32, device=DEV)
            y_ref = layer.forward(x, topk_ids=ids_ref).clone()
            ids = torch.empty_like(ids_ref)
            y = tier.forward(x, topk_ids=ids)
            assert moe.moe_get_device_status(tier.ws) == moe.MOE_OK
            assert torch.equal(ids, ids_ref) and torch.equal(y, y_ref), (cfg, slots)
        st = tier.stats()
        assert st["steps"] == 3 and st["resident"] <= st["n_slots"] == min(slots, E + S)
        assert st["bytes_loaded"] == st["misses"] * 3 * I * d * 2
    finally:
        tier.close()


def _skewed_ids(T, E, k, rng):
    """Distinct expert ids per token: the top k of Gumbel-perturbed Zipf(s)
    log-weights (s = 0 is uniform), so some experts get large batches and
    others none."""
    s = float(rng.choice([0.0, 0.8, 1.5]))
    logw = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logw[None, :] + rng.gumbel(size=(T, E))
    ids = np.argpartition(-keys, k - 1, axis=1)[:, :k]
    order = np.argsort(-np.take_along_axis(keys, ids, 1), axis=1)  # descending score
    return np.take_along_axis(ids, order, 1).astype(np.int32)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(40))
def test_plan_random_sweep(seed):
    """moe_plan_dispatch against the oracle's plan, bit for bit, over random
    sizes: the one-block plan and the three-kernel plan (large T x E)."""
    rng = np.random.default_rng(90000 + seed)
    E = int(np.exp(rng.uniform(0, np.log(1024))))
    k = int(rng.integers(1, min(E, 32) + 1))
    S = int(rng.integers(0, 5))
    T = int(np.exp(rng.uniform(0, np.log(20000))))
    T = max(1, min(T, 4_000_000 // E))
    ids = _skewed_ids(T, E, k, rng)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    # the plan does not depend on the layer's dtype; an fp32 record admits E + S = 1
    desc = moe.make_desc(T, 64, E, k, 64, S, dtype=moe.MOE_F32)
    ws = moe.alloc_workspace(desc)
    P = T * (k + S)
    off = torch.full((E + S + 1,), -1, dtype=torch.int32, device=DEV)
    tok = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    sr = torch.full((T, k + S), -1, dtype=torch.int32, device=DEV)
    act = torch.full((E + S,), -1, dtype=torch.int32, device=DEV)
    na = torch.zeros((1,), dtype=torch.int32, device=DEV)
    sw = torch.zeros((P,), dtype=torch.float32, device=DEV)
    moe.moe_plan_dispatch(desc, torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV), off,
                          tok, sr, act, na, sw, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    ref = oracle.plan(ids, E, S)
    np.testing.assert_array_equal(host(off).numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(host(tok).numpy(), ref["token_indices"])
    np.testing.assert_array_equal(host(sr).numpy(), ref["slot_row"])
    n = int(host(na)[0])
    assert n == ref["n_active"]
    np.testing.assert_array_equal(host(act).numpy()[:n], ref["active_ids"])
    wfull = np.concatenate([w, np.ones((T, S), np.float32)], 1)
    exp = np.empty(P, np.float32)
    exp[ref["slot_row"].ravel()] = wfull.ravel()
    np.testing.assert_array_equal(host(sw).numpy(), exp)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(30))
def test_combine_partial_random_sweep(seed):
    """moe_combine_partial against the oracle over random sizes and random
    availability (from every expert available to none); with every expert
    available it equals moe_combine bit for bit; the list of unserved pairs
    (moe_partial_missing_pairs) equals the oracle's."""
    rng = np.random.default_rng(110000 + seed)
    f32 = rng.random() < 0.3
    E = int(rng.integers(2, 65))
    k = int(rng.integers(1, min(E, 16) + 1))
    S = int(rng.integers(0, 3))
    T = int(rng.integers(1, 301))
    d = 8 * int(rng.integers(1, 65)) if f32 else 64 * int(rng.integers(1, 9))
    desc = moe.make_desc(T, d, E, k, 128, S, dtype=moe.MOE_F32 if f32 else moe.MOE_BF16)
    dt = torch.float32 if f32 else torch.bfloat16
    ids = _skewed_ids(T, E, k, rng)
    w = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    plan = oracle.plan(ids, E, S)
    P = T * (k + S)
    g = torch.Generator(device=DEV).manual_seed(seed)
    y_perm = torch.randn((P, d), generator=g, device=DEV).to(dt)
    sr = torch.from_numpy(plan["slot_row"]).to(DEV)
    g_ids, g_w = torch.from_numpy(ids).to(DEV), torch.from_numpy(w).to(DEV)
    y = torch.empty((T, d), dtype=torch.float32, device=DEV)
    miss = torch.full((T, k + S), 7, dtype=torch.int32, device=DEV)
    everyone = torch.ones((E + S,), dtype=torch.int32, device=DEV)
    moe.moe_combine_partial(desc, y_perm, sr, g_ids, g_w, everyone, None, y, miss)
    y_full = torch.empty_like(y)
    moe.moe_combine(desc, y_perm, sr, g_w, None, y_full)
    assert torch.equal(y, y_full) and int(miss.sum()) == 0
    p_avail = float(rng.choice([0.0, 0.3, 0.7, 1.0]))
    avail = (rng.random(E + S) < p_avail).astype(np.int32)
    res = torch.randn((T, d), generator=g, device=DEV) if rng.random() < 0.5 else None
    moe.moe_combine_partial(desc, y_perm, sr, g_ids, g_w, torch.from_numpy(avail).to(DEV), res,
                            y, miss)
    y_ref, miss_ref = oracle.combine_partial(host(y_perm).double().numpy(), plan["slot_row"], ids,
                                             w, avail, k, S, E, residual=host(res))
    np.testing.assert_array_equal(host(miss).numpy(), miss_ref)
    scale = max(float(np.abs(y_ref).max()), 1e-30)
    assert float(np.abs(host(y).double().numpy() - y_ref).max()) / scale <= 1e-6
    pairs = torch.full((P, 2), -9, dtype=torch.int32, device=DEV)
    n_pairs = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    moe.moe_partial_missing_pairs(desc, g_ids, miss, pairs, n_pairs)
    want = oracle.missing_pairs(ids, avail, k, S, E)
    n = int(host(n_pairs)[0])
    assert n == len(want)
    np.testing.assert_array_equal(host(pairs).numpy()[:n], want)


def _draw_medium(seed):
    """Medium layers: K of 512-1024 (the large-tile kernels at longer reductions
    than the small draws reach), 256-2048 tokens, one or two tile heights of
    rows per expert, skewed or uniform routing."""
    rng = np.random.default_rng(70000 + seed)
    E = int(rng.integers(4, 9)) if rng.random() < 0.35 else int(rng.integers(8, 65))
    k = int(rng.integers(2, min(E, 8) + 1))
    S = int(rng.integers(0, 2))
    T = int(rng.integers(256, 2049))
    gate = int(rng.integers(0, 2))
    d, I = 64 * int(rng.integers(8, 17)), 64 * int(rng.integers(8, 17))
    return LayerConfig("medium_%d" % seed, T=T, d=d, E=E, I=I, k=k, S=S, gate=gate,
                       norm_topk=gate, routed_scaling=2.5 if gate else 1.0,
                       sel_bias_range=0.1 if gate else 0.0,
                       zipf_s=1.2 if rng.random() < 0.5 else 0.0)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(6))
def test_layer_medium_sweep_every_token(seed):
    """Medium layers, bf16 and Q8_0 experts: routing bit-exact and every token's
    output against the oracle (Q8_0: the oracle on its own dequantization of the
    same weights)."""
    from tests.helpers import check_all_tokens
    cfg = _draw_medium(seed)
    try:
        inp = make_case(cfg, seed=seed, device=DEV)
    except RuntimeError as e:
        pytest.skip(str(e))
    kw = dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
              logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    desc = moe.desc_from_config(cfg)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate, **kw)
    for q8 in (False, True):
        Wg, Wu, Wd = inp["Wg"], inp["Wu"], inp["Wd"]
        if q8:
            Wg, Wu, Wd = (moe.quantize_q8_0(W) for W in (Wg, Wu, Wd))
        layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd, logit_bias=inp["logit_bias"],
                             sel_bias=inp["sel_bias"])
        ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
        w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
        y = layer.forward(inp["x"], topk_ids=ids, topk_w=w)
        assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
        np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
        check_weights(host(w).numpy(), w_ref, inp, cfg)
        if q8:
            ref_w = [list(_deq(inp[n])) for n in ("Wg", "Wu", "Wd")]
            y_ref, _, _ = oracle.forward(host(inp["x"]), oracle.widen(host(inp["Wr"])), *ref_w,
                                         cfg.k, cfg.gate, S=cfg.S, **kw)
        else:
            y_ref, _, _ = oracle.forward(host(inp["x"]), host(inp["Wr"]), host(inp["Wg"]),
                                         host(inp["Wu"]), host(inp["Wd"]), cfg.k, cfg.gate,
                                         S=cfg.S, **kw)
        check_all_tokens(host(y).double().numpy(), y_ref, ids_ref, cfg, 1e-2)
