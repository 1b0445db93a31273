"""A randomized sweep of whole-layer shapes against the oracle: bf16 and fp32
layers, and the same bf16 layers with Q8_0 experts.  Shapes range from decode
sized batches (one token, top-32 of 64 experts) to batches of several hundred
rows per expert, which take the SM-pair and 256-row GEMM paths; up to two
shared experts, both gate families.  Routing must match bit for bit, gate
weights within 1e-4, outputs within the layer tolerance (Q8_0: within 1e-2 of
the oracle on the dequantized weights).  A draw whose top-(k+1) scores cannot
be separated by the routing margin (many sigmoid scores at large k) is skipped."""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs
from tests.helpers import W_RTOL, host, make_case, rel_err, y_tol

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
    np.testing.assert_allclose(host(w).numpy(), w_ref, rtol=W_RTOL, atol=0)
    y_ref, _, _ = oracle.forward(host(inp["x"]), host(inp["Wr"]), host(inp["Wg"]),
                                 host(inp["Wu"]), host(inp["Wd"]), cfg.k, cfg.gate, S=cfg.S,
                                 **kw)
    assert rel_err(host(y).double().numpy(), y_ref) <= y_tol(cfg), cfg
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
