"""GPU: the expert tier (moe_tier_*) -- experts in host memory, a bounded pool of
HBM slots -- gives moe_layer_forward's result bit for bit, whatever the budget
("Module expert_store" (ferrox-core docs): the cached path proven bit-identical
to the resident one at generous and at smaller-than-one-step budgets)."""
import numpy as np
import pytest
import torch

from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import KIMI_DECODE, LayerConfig, make_inputs

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


def _xs(cfg, n, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return [torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
            for _ in range(n)]


@pytest.mark.parametrize("slots", [49, 20, 7, 2, 1])
def test_tier_equals_resident_layer(slots):
    cfg = SMALL
    inp = make_inputs(cfg, seed=3, device=DEV)
    tier = _tier(cfg, inp, slots)
    assert tier.stats()["n_slots"] == min(slots, cfg.E + cfg.S)
    for x in _xs(cfg, 5, seed=slots):
        y_ref, ids_ref = _resident(cfg, inp, x)
        ids = torch.empty_like(ids_ref)
        y = tier.forward(x, topk_ids=ids)
        assert moe.moe_get_device_status(tier.ws) == moe.MOE_OK
        assert torch.equal(ids, ids_ref)
        assert torch.equal(y, y_ref)
    st = tier.stats()
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
    for x in _xs(cfg, 3, seed=0):
        y_ref, ids_ref = _resident(cfg, inp, x)
        ids = torch.empty_like(ids_ref)
        y = tier.forward(x, topk_ids=ids)
        assert moe.moe_get_device_status(tier.ws) == moe.MOE_OK
        assert torch.equal(ids, ids_ref) and torch.equal(y, y_ref)
    st = tier.stats()
    assert st["n_slots"] == nE // 4 and st["extra_passes"] > 0
    tier.close()
    del inp
    torch.cuda.empty_cache()
