"""Q8_0 expert weights on the GPU against the fp64 oracle.

The quantizer's integer codes and f16 scales must match the oracle's bit for
bit (both decide in fp32).  The FFN and the layer forward on Q8_0 weights are
compared with the oracle run on its own dequantization of the same bf16
weights (exact scale * q in fp64); the GPU rounds each dequantized weight to
bf16 before the tensor cores, which the 1e-2 output tolerance covers.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import CONFIGS, KIMI_DECODE, LayerConfig, make_inputs
from tests.helpers import check_all_tokens, enforce_margins, host, rel_err

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from expert_dispatch_gb300 import build
    build.build()


def _oracle_deq(W):
    """Host copy of W [n, R, K] -> the oracle's Q8_0 codes -> exact fp64 weights."""
    q, s = oracle.quantize_q8_0(host(W))
    return oracle.dequantize_q8_0(q, s)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_matches_oracle_bit_for_bit(dtype):
    g = torch.Generator(device=DEV).manual_seed(17)
    w = (torch.randn((5, 192, 256), generator=g, device=DEV) * 0.03).to(dtype)
    w[1, 3, 64:96] = 0                      # an all-zero block
    w[2, 7, :32] *= 1000                    # a large block
    w[4, :, 128:160] = -w[4, :, 128:160].abs()
    # a block whose codes are exact halves (max 127 -> d = 1): the rounding rule decides
    ties = torch.tensor([127.0, 0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 3.5, 126.5, -126.5] + [0.0] * 22)
    w[3, 5, 32:64] = ties.to(dtype).to(DEV)
    qw = moe.quantize_q8_0(w)
    q_ref, s_ref = oracle.quantize_q8_0(host(w))
    np.testing.assert_array_equal(host(qw.q).numpy(), q_ref)
    np.testing.assert_array_equal(host(qw.scale).numpy().view(np.uint16), s_ref)


Q8_CASES = [
    LayerConfig("q_small_tiles", T=67, d=128, E=8, I=192, k=2, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    LayerConfig("q_mid_tiles", T=300, d=192, E=8, I=320, k=2, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    LayerConfig("q_large_tiles", T=600, d=256, E=4, I=320, k=2),
    LayerConfig("q_hot_expert", T=2000, d=128, E=8, I=128, k=2, zipf_s=1.2),
    LayerConfig("q_one_token", T=1, d=512, E=32, I=256, k=4, S=1, gate=1, norm_topk=1,
                routed_scaling=2.8, sel_bias_range=0.1),
]


@pytest.mark.parametrize("cfg", Q8_CASES, ids=lambda c: c.name)
def test_expert_ffn_q8_parity(cfg):
    inp = enforce_margins(make_inputs(cfg, seed=23, device=DEV), cfg, 23)
    ids, _ = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                          norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
                          logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    plan = oracle.plan(ids, cfg.E, cfg.S)
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    P = cfg.T * (cfg.k + cfg.S)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    y_perm = torch.zeros((P, cfg.d), dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn_q8(desc, inp["x"], torch.from_numpy(plan["expert_offsets"]).to(DEV),
                          torch.from_numpy(plan["token_indices"]).to(DEV), None, Wg, Wu, Wd,
                          y_perm, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    dg, du, dd = (_oracle_deq(inp[n]) for n in ("Wg", "Wu", "Wd"))
    o, tok = plan["expert_offsets"], plan["token_indices"]
    ref = np.zeros((P, cfg.d))
    for e in range(cfg.E + cfg.S):
        if o[e + 1] > o[e]:
            ref[o[e]:o[e + 1]] = oracle.expert_rows(host(inp["x"]), dg[e], du[e], dd[e],
                                                    tok[o[e]:o[e + 1]])
    got = host(y_perm).double().numpy()
    assert rel_err(got, ref) <= 1e-2, rel_err(got, ref)


@pytest.mark.parametrize("cfg", [KIMI_DECODE.with_T(1), KIMI_DECODE.with_T(8),
                                 KIMI_DECODE.with_T(64), CONFIGS["qwen_t512"]],
                         ids=["kimi_decode_T1", "kimi_decode_T8", "kimi_decode_T64", "qwen_t512"])
def test_layer_forward_q8_full_size(cfg):
    """Every token of the layer on Q8_0 experts against the oracle.  The oracle
    side is the grouped form of the same definition ("Expert-Sharded Swarm
    Inference: The Design", exactness paragraph): each active expert's
    dequantized projections run over its batch of token rows
    (oracle.expert_rows), and the rows are combined per token with the oracle's
    gate weights (oracle.combine).  One expert's fp64 weights are held at a
    time."""
    inp = enforce_margins(make_inputs(cfg, seed=0, device=DEV), cfg, 0)
    desc = moe.desc_from_config(cfg)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd, logit_bias=inp["logit_bias"],
                         sel_bias=inp["sel_bias"])
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    y = layer.forward(inp["x"], topk_ids=ids)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    y_host = host(y).double().numpy()
    del layer, Wg, Wu, Wd, y
    torch.cuda.empty_cache()
    kw = dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
              logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate, **kw)
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    plan = oracle.plan(ids_ref, cfg.E, cfg.S)
    o, tok = plan["expert_offsets"], plan["token_indices"]
    x_host = host(inp["x"])
    rows = np.zeros((cfg.T * (cfg.k + cfg.S), cfg.d))
    for e in range(cfg.E + cfg.S):
        if o[e + 1] == o[e]:
            continue
        dg, du, dd = (_oracle_deq(inp[n][e:e + 1])[0] for n in ("Wg", "Wu", "Wd"))
        rows[o[e]:o[e + 1]] = oracle.expert_rows(x_host, dg, du, dd, tok[o[e]:o[e + 1]])
    y_ref = oracle.combine(rows, plan["slot_row"], cfg.k, cfg.S, w=w_ref)
    check_all_tokens(y_host, y_ref, ids_ref, cfg, 1e-2)


def test_layer_forward_q8_max_groups():
    """The largest layer record on Q8_0 experts: 1024 routed experts, top-32 and
    4 shared experts (1028 expert batches, the kernels' schedule limit), every
    token against the oracle on the dequantized weights."""
    cfg = LayerConfig("q_max_groups", T=40, d=128, E=1024, I=64, k=32, S=4, norm_topk=1)
    inp = enforce_margins(make_inputs(cfg, seed=7, device=DEV), cfg, 7)
    desc = moe.desc_from_config(cfg)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    y = layer.forward(inp["x"], topk_ids=ids)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    kw = dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling)
    ids_ref, _ = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate, **kw)
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    deq = [list(_oracle_deq(inp[n])) for n in ("Wg", "Wu", "Wd")]
    y_ref, _, _ = oracle.forward(host(inp["x"]), oracle.widen(host(inp["Wr"])), *deq, cfg.k,
                                 cfg.gate, S=cfg.S, **kw)
    check_all_tokens(host(y).double().numpy(), y_ref, ids_ref, cfg, 1e-2)


def tile_covering_tokens(plan, tile_rows, rng):
    """Tokens such that every tile of every expert's batch, for each tile height
    in tile_rows, holds at least one of their rows (one random row per tile)."""
    o, tok = plan["expert_offsets"], plan["token_indices"]
    picked = set()
    for e in range(len(o) - 1):
        cnt = int(o[e + 1] - o[e])
        for bt in tile_rows:
            for s0 in range(0, cnt, bt):
                picked.add(int(tok[o[e] + s0 + rng.integers(0, min(bt, cnt - s0))]))
    return np.array(sorted(picked), np.int32)


@pytest.mark.parametrize("name", ["deepseek_prefill", "skewed_zipf"])
def test_layer_forward_q8_full_size_prefill(name):
    """The prefill workloads at full size on Q8_0 experts (the 192-token gate/up
    and 256-token down variants), checked on a token sample that puts at least
    one checked row in every tile of every expert's batch at both tile heights.
    Oracle side: per active expert, its dequantized projections over the sampled
    tokens' rows of its batch (oracle.expert_rows), combined per token with the
    oracle's gate weights -- one expert's fp64 weights in memory at a time."""
    cfg = CONFIGS[name]
    inp = enforce_margins(make_inputs(cfg, seed=0, device=DEV), cfg, 0)
    desc = moe.desc_from_config(cfg)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd, logit_bias=inp["logit_bias"],
                         sel_bias=inp["sel_bias"])
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    y = layer.forward(inp["x"], topk_ids=ids)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    y_host = host(y).double().numpy()
    del layer, Wg, Wu, Wd, y
    torch.cuda.empty_cache()
    kw = dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
              logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate, **kw)
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    plan = oracle.plan(ids_ref, cfg.E, cfg.S)
    tokens = tile_covering_tokens(plan, (192, 256), np.random.default_rng(3))
    o, tok = plan["expert_offsets"], plan["token_indices"]
    want = np.zeros(cfg.T, bool)
    want[tokens] = True
    P = cfg.T * (cfg.k + cfg.S)
    rows = np.zeros((P, cfg.d))
    x_host = host(inp["x"])
    for e in range(cfg.E + cfg.S):
        r = np.arange(o[e], o[e + 1])
        r = r[want[tok[r]]]  # the batch rows of sampled tokens
        if len(r) == 0:
            continue
        dg, du, dd = (_oracle_deq(inp[n][e:e + 1])[0] for n in ("Wg", "Wu", "Wd"))
        rows[r] = oracle.expert_rows(x_host, dg, du, dd, tok[r])
    sr = plan["slot_row"][tokens]
    y_ref = oracle.combine(rows, sr, cfg.k, cfg.S, w=w_ref[tokens])
    check_all_tokens(y_host[tokens], y_ref, ids_ref[tokens], cfg, 1e-2)


# Batch sizes on the tile edges of the Q8_0 kernels: 32-token tiles with
# several issuers (mean batch <= 48 rows), and the large-batch variants
# (192-token gate/up, 256-token down), with weight blocks that end inside a
# matrix (I = 320, d = 192) and K of an odd number of 64-wide blocks (two-block
# weight stages with a half-empty last stage).
Q8_TILE_EDGE_CASES = [
    ("small", LayerConfig("q8_edges_small", T=136, d=192, E=10, I=320, k=2),
     [1, 15, 16, 17, 31, 32, 33, 63, 64, 0]),
    ("large", LayerConfig("q8_edges_large", T=1498, d=192, E=12, I=320, k=2),
     [1, 31, 33, 191, 192, 193, 255, 256, 257, 384, 500, 703]),
]


@pytest.mark.parametrize("name,cfg,sizes", Q8_TILE_EDGE_CASES,
                         ids=[c[0] for c in Q8_TILE_EDGE_CASES])
def test_expert_ffn_q8_tile_edges(name, cfg, sizes):
    P = cfg.T * cfg.k
    assert sum(sizes) == P and len(sizes) == cfg.E
    inp = make_inputs(cfg, seed=29, device=DEV)
    rng = np.random.default_rng(29)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    tok = rng.integers(0, cfg.T, size=P).astype(np.int32)
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    y_perm = torch.full((P, cfg.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn_q8(desc, inp["x"], torch.from_numpy(off).to(DEV),
                          torch.from_numpy(tok).to(DEV), None, Wg, Wu, Wd, y_perm, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    dg, du, dd = (_oracle_deq(inp[n]) for n in ("Wg", "Wu", "Wd"))
    got = host(y_perm).double().numpy()
    for e in range(cfg.E):
        if sizes[e] == 0:
            continue
        ref = oracle.expert_rows(host(inp["x"]), dg[e], du[e], dd[e], tok[off[e]:off[e + 1]])
        err = rel_err(got[off[e]:off[e + 1]], ref)
        assert err <= 1e-2, (e, sizes[e], err)


def test_layer_forward_q8_host_buffers():
    cfg = Q8_CASES[0]
    inp = enforce_margins(make_inputs(cfg, seed=31, device=DEV), cfg, 31)
    desc = moe.desc_from_config(cfg)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd, logit_bias=inp["logit_bias"],
                         sel_bias=inp["sel_bias"])
    y_dev = layer.forward(inp["x"])
    x_host = host(inp["x"]).pin_memory()
    y_host = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32).pin_memory()
    layer.forward_host(x_host, y_host)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    assert torch.equal(y_host, host(y_dev))


def test_layer_forward_q8_host_pipelined():
    cfg = Q8_CASES[0]
    inp = enforce_margins(make_inputs(cfg, seed=37, device=DEV), cfg, 37)
    desc = moe.desc_from_config(cfg)
    Wg, Wu, Wd = (moe.quantize_q8_0(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = moe.MoeLayer(desc, inp["Wr"], Wg, Wu, Wd, logit_bias=inp["logit_bias"],
                         sel_bias=inp["sel_bias"])
    xa, xb = inp["x"], torch.roll(inp["x"], shifts=5, dims=0)
    want = [host(layer.forward(x)) for x in (xa, xb, xa)]
    xa_host, xb_host = host(xa).pin_memory(), host(xb).pin_memory()
    x_hosts = [xa_host, xb_host, xa_host]  # an input buffer may repeat
    y_hosts = [torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32).pin_memory()
               for _ in range(3)]
    layer.forward_host_pipelined(x_hosts, y_hosts)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    for i in range(3):
        assert torch.equal(y_hosts[i], want[i]), i
