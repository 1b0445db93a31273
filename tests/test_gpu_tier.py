"""GPU: the expert tier (moe_tier_*) -- experts in host memory, a bounded pool of
HBM slots -- gives moe_layer_forward's result bit for bit, whatever the budget
("Module expert_store" (ferrox-core docs): the cached path proven bit-identical
to the resident one at generous and at smaller-than-one-step budgets); its
output matches the fp64 oracle's layer forward, and its hit / miss / eviction
/ extra-pass counters match the oracle's restatement of the tier's rules
(oracle_tier_step) replayed on the oracle's routing of the same steps."""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import KIMI_DECODE, LayerConfig, make_inputs
from tests.helpers import enforce_margins, host, rel_err, y_tol

pytestmark = pytest.mark.gpu

DEV = "cuda"

# a Kimi-layout layer, scaled down: sigmoid + selection bias, one shared expert
SMALL = LayerConfig("tier_small", T=24, d=512, E=48, I=256, k=6, S=1, gate=1, norm_topk=1,
                    routed_scaling=2.5, sel_bias_range=0.1)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from expert_dispatch_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def _host_weights(inp):
    out = []
    for n in ("Wg", "Wu", "Wd"):
        h = moe.host_empty(inp[n].shape, inp[n].dtype)
        h.copy_(inp[n])
        out.append(h)
    return tuple(out)


def _resident(cfg, inp, x):
    layer = moe.MoeLayer(moe.desc_from_config(cfg), inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"],
                         logit_bias=inp["logit_bias"], sel_bias=inp["sel_bias"])
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    y = layer.forward(x, topk_ids=ids)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    return y, ids


def _tier(cfg, inp, slots):
    expert_bytes = 3 * cfg.I * cfg.d * 2
    return moe.ExpertTier(moe.desc_from_config(cfg), inp["Wr"], *_host_weights(inp),
                          slots * expert_bytes, logit_bias=inp["logit_bias"],
                          sel_bias=inp["sel_bias"])


def _xs(cfg, n, seed, inp=None):
    """n token batches; with the layer's inputs given, each batch keeps every
    routing decision clear of near-ties (so that routing is comparable with the
    oracle's bit for bit)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    xs = [torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
          for _ in range(n)]
    if inp is not None:
        for i, x in enumerate(xs):
            enforce_margins(dict(inp, x=x), cfg, seed * 100 + i)
    return xs


def _oracle_kw(cfg, inp):
    return dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
                logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))


def _check_against_oracle(cfg, inp, xs, ys, slots):
    """Every step's output against the oracle's forward, and the tier's counters
    against the oracle's tier fed the same steps (each step asks for its active
    experts in ascending order, the shared experts included)."""
    nE = cfg.E + cfg.S
    tier_o = oracle.TierOracle(min(slots, nE), nE)
    Wg, Wu, Wd = (host(inp[n]) for n in ("Wg", "Wu", "Wd"))
    for x, y in zip(xs, ys):
        y_ref, ids_ref, _ = oracle.forward(host(x), host(inp["Wr"]), Wg, Wu, Wd, cfg.k,
                                           cfg.gate, S=cfg.S, **_oracle_kw(cfg, inp))
        err = rel_err(host(y).double().numpy(), y_ref)
        assert err <= y_tol(cfg), err
        active = sorted(set(ids_ref.flatten().tolist()) | set(range(cfg.E, nE)))
        tier_o.step(active)
    return tier_o.stats()


@pytest.mark.parametrize("slots", [49, 20, 7, 2, 1])
def test_tier_equals_resident_layer(slots):
    cfg = SMALL
    inp = make_inputs(cfg, seed=3, device=DEV)
    tier = _tier(cfg, inp, slots)
    assert tier.stats()["n_slots"] == min(slots, cfg.E + cfg.S)
    xs, ys = _xs(cfg, 5, seed=slots, inp=inp), []
    for x in xs:
        y_ref, ids_ref = _resident(cfg, inp, x)
        ids = torch.empty_like(ids_ref)
        y = tier.forward(x, topk_ids=ids)
        assert moe.moe_get_device_status(tier.ws) == moe.MOE_OK
        assert torch.equal(ids, ids_ref)
        assert torch.equal(y, y_ref)
        ys.append(y.clone())
    st = tier.stats()
    ost = _check_against_oracle(cfg, inp, xs, ys, slots)
    for key in ("hits", "misses", "evictions", "extra_passes", "resident"):
        assert st[key] == ost[key], (key, st[key], ost[key])
    assert st["steps"] == 5 and st["resident"] <= st["n_slots"]
    assert st["bytes_loaded"] == st["misses"] * 3 * cfg.I * cfg.d * 2
    if slots < 10:  # a step's experts (up to 24 * 6 routed + 1 shared) exceed the slots
        assert st["extra_passes"] > 0
    tier.close()


def test_repeat_step_hits_and_loads_nothing():
    cfg = SMALL
    inp = make_inputs(cfg, seed=4, device=DEV)
    tier = _tier(cfg, inp, cfg.E + cfg.S)
    x = _xs(cfg, 1, seed=1)[0]
    y1 = tier.forward(x).clone()
    s1 = tier.stats()
    assert s1["hits"] == 0 and s1["misses"] > 0
    y2 = tier.forward(x)
    s2 = tier.stats()
    assert s2["misses"] == s1["misses"] and s2["bytes_loaded"] == s1["bytes_loaded"]
    assert s2["hits"] == s1["misses"]  # every expert of the step is now resident
    assert torch.equal(y1, y2)
    tier.close()


def test_prefetch_makes_the_next_step_hit():
    cfg = SMALL
    inp = make_inputs(cfg, seed=5, device=DEV)
    x = _xs(cfg, 1, seed=2)[0]
    _, ids = _resident(cfg, inp, x)
    needed = sorted(set(ids.flatten().tolist()) | {cfg.E})  # routed + the shared expert
    tier = _tier(cfg, inp, len(needed))
    tier.prefetch(needed)
    s0 = tier.stats()
    assert s0["misses"] == len(needed) and s0["resident"] == len(needed)
    tier.forward(x)
    s1 = tier.stats()
    assert s1["misses"] == s0["misses"] and s1["hits"] == len(needed)
    tier.close()


def test_host_memory_for_the_tier():
    h = moe.host_empty((3, 5, 64), torch.bfloat16)
    assert h.device.type == "cpu" and h.is_contiguous() and bool((h == 0).all())
    v = h[1]
    del h
    v.fill_(2.0)  # the block outlives the tensor it was made for while a view exists
    assert bool((v == 2.0).all())
    with pytest.raises(moe.MoeError):
        moe._check(moe.lib().moe_host_free(moe.ctypes.c_void_p(12345)), "moe_host_free")


def test_tier_rejects_bad_arguments():
    cfg = SMALL
    inp = make_inputs(cfg, seed=6, device=DEV)
    desc = moe.desc_from_config(cfg)
    hw = _host_weights(inp)
    with pytest.raises(moe.MoeError) as ei:  # budget below one expert
        moe.ExpertTier(desc, inp["Wr"], *hw, 3 * cfg.I * cfg.d * 2 - 1)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    f32 = moe.make_desc(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.S, dtype=moe.MOE_F32)
    with pytest.raises((moe.MoeError, TypeError)):
        moe.ExpertTier(f32, inp["Wr"], *(w.float() for w in hw), 1 << 30)


def test_tier_full_size_kimi_decode():
    """Kimi layout at T=64 with room for a quarter of the experts."""
    cfg = KIMI_DECODE.with_T(64)
    inp = make_inputs(cfg, seed=0, device=DEV)
    nE = cfg.E + cfg.S
    tier = _tier(cfg, inp, nE // 4)
    xs, ys = _xs(cfg, 3, seed=0, inp=inp), []
    for x in xs:
        y_ref, ids_ref = _resident(cfg, inp, x)
        ids = torch.empty_like(ids_ref)
        y = tier.forward(x, topk_ids=ids)
        assert moe.moe_get_device_status(tier.ws) == moe.MOE_OK
        assert torch.equal(ids, ids_ref) and torch.equal(y, y_ref)
        ys.append(y.clone())
    st = tier.stats()
    assert st["n_slots"] == nE // 4 and st["extra_passes"] > 0
    ost = _check_against_oracle(cfg, inp, xs, ys, nE // 4)
    for key in ("hits", "misses", "evictions", "extra_passes", "resident"):
        assert st[key] == ost[key], (key, st[key], ost[key])
    tier.close()
    del inp
    torch.cuda.empty_cache()


def test_load_launches_are_profiled_with_their_bytes():
    """moe_profile_list gives each load launch of the tier with the bytes it
    moved; they add up to the tier's bytes_loaded counter."""
    cfg = SMALL
    inp = make_inputs(cfg, seed=8, device=DEV)
    tier = _tier(cfg, inp, 7)
    s0 = tier.stats()
    moe.moe_profile_enable(True)
    for x in _xs(cfg, 3, seed=4):
        tier.forward(x)
    torch.cuda.synchronize()
    ms, nbytes = moe.moe_profile_list("load_experts")
    g_ms, g_bytes = moe.moe_profile_list("ffn_gateup_tc")
    moe.moe_profile_enable(False)
    s1 = tier.stats()
    assert len(ms) > 0 and all(t > 0 for t in ms)
    assert sum(nbytes) == s1["bytes_loaded"] - s0["bytes_loaded"]
    assert all(b % (3 * cfg.I * cfg.d * 2) == 0 for b in nbytes)
    assert len(g_ms) >= 3 and all(b == 0 for b in g_bytes)
    tier.close()
