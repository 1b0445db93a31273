"""GPU parity: every C-ABI call against the fp64 oracle on the same seeded inputs.

Routing (ids) and the dispatch plan must match bit-exactly; gate weights within
the fp32-accumulation bound; layer outputs within max|dy|/max|y| <= 1e-5 (fp32
layer) or 1e-2 (bf16 layer).  Small cases span several tiles and ragged tails;
the five workloads run at full size with every token checked against the
per-token oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import (CONFIGS, DECODE_TS, KIMI_DECODE, LayerConfig,
                                          make_inputs)
from tests.helpers import (check_all_tokens, check_weights, enforce_margins, host, rel_err,
                           y_tol)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from expert_dispatch_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def _case(cfg, seed=0):
    inp = make_inputs(cfg, seed=seed, device=DEV)
    return enforce_margins(inp, cfg, seed)


def _oracle_kw(cfg, inp):
    return dict(norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
                logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))


def _gpu_layer(cfg, inp, residual=None):
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    y = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32, device=DEV)
    ids = torch.full((cfg.T, cfg.k), -7, dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    moe.moe_layer_forward(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"],
                          inp["Wg"], inp["Wu"], inp["Wd"], residual, y, ids, w, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    return y, ids, w, ws


def _experts_on_host(inp, needed, nE):
    lists = []
    for name in ("Wg", "Wu", "Wd"):
        W = inp[name]
        lists.append([host(W[e]) if e in needed else None for e in range(nE)])
    return lists


def _oracle_forward(cfg, inp, tokens, ids_ref, residual=None):
    needed = set(np.unique(ids_ref[tokens]).tolist()) | set(range(cfg.E, cfg.E + cfg.S))
    Wg, Wu, Wd = _experts_on_host(inp, needed, cfg.E + cfg.S)
    y, ids, w = oracle.forward(host(inp["x"]), host(inp["Wr"]), Wg, Wu, Wd, cfg.k, cfg.gate,
                               S=cfg.S, residual=host(residual), tokens=tokens,
                               **_oracle_kw(cfg, inp))
    return y, ids, w


# ---------------------------------------------------------------- router
ROUTER_CASES = [
    LayerConfig("r_fp32", T=64, d=256, E=16, I=128, k=2, dtype="f32"),
    LayerConfig("r_bf16_simt", T=45, d=128, E=40, I=64, k=6, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    LayerConfig("r_bf16_tc", T=300, d=192, E=130, I=64, k=8, zipf_s=1.2),
    LayerConfig("r_bf16_tc_sig", T=517, d=256, E=256, I=64, k=8, S=1, gate=1, norm_topk=1,
                routed_scaling=2.827, sel_bias_range=0.1),
    # CUDA-core router over several token runs per expert row (the last one ragged)
    LayerConfig("r_bf16_simt_runs", T=600, d=320, E=40, I=64, k=4),
    # every expert selected (k = E): the weights are the whole softmax / the normalised scores
    LayerConfig("r_k_equals_E_softmax", T=33, d=128, E=8, I=64, k=8),
    LayerConfig("r_k_equals_E_sigmoid", T=33, d=128, E=8, I=64, k=8, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
]


@pytest.mark.parametrize("cfg", ROUTER_CASES, ids=lambda c: c.name)
def test_route_parity(cfg):
    inp = _case(cfg, seed=3)
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    moe.moe_route(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"], ids, w, ws)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                                  **_oracle_kw(cfg, inp))
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    check_weights(host(w).numpy(), w_ref, inp, cfg)


# ---------------------------------------------------------------- planner
PLAN_CASES = [(1, 4, 2, 0), (5, 8, 3, 1), (33, 40, 8, 0), (1000, 256, 8, 1), (4099, 64, 6, 2),
              (2, 1024, 32, 0)]


def _random_ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=k, replace=False)
    return ids


@pytest.mark.parametrize("T,E,k,S", PLAN_CASES)
def test_plan_parity(T, E, k, S):
    ids = _random_ids(T, E, k, seed=T + E)
    w = np.random.default_rng(1).uniform(0, 1, (T, k)).astype(np.float32)
    desc = moe.make_desc(T, 64, E, k, 64, S, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(desc)
    P = T * (k + S)
    g_ids = torch.from_numpy(ids).to(DEV)
    g_w = torch.from_numpy(w).to(DEV)
    off = torch.full((E + S + 1,), -1, dtype=torch.int32, device=DEV)
    tok = torch.full((P,), -1, dtype=torch.int32, device=DEV)
    sr = torch.full((T, k + S), -1, dtype=torch.int32, device=DEV)
    act = torch.full((E + S,), -1, dtype=torch.int32, device=DEV)
    na = torch.zeros((1,), dtype=torch.int32, device=DEV)
    sw = torch.zeros((P,), dtype=torch.float32, device=DEV)
    for _ in range(2):  # a second call on the same workspace gives the same plan
        moe.moe_plan_dispatch(desc, g_ids, g_w, off, tok, sr, act, na, sw, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        ref = oracle.plan(ids, E, S)
        np.testing.assert_array_equal(host(off).numpy(), ref["expert_offsets"])
        np.testing.assert_array_equal(host(tok).numpy(), ref["token_indices"])
        np.testing.assert_array_equal(host(sr).numpy(), ref["slot_row"])
        n = int(host(na)[0])
        assert n == ref["n_active"]
        np.testing.assert_array_equal(host(act).numpy()[:n], ref["active_ids"])
    # slot weights follow the rows: routed pairs carry their gate weight, shared rows 1.0
    wfull = np.concatenate([w, np.ones((T, S), np.float32)], 1)
    exp = np.empty(P, np.float32)
    exp[ref["slot_row"].ravel()] = wfull.ravel()
    np.testing.assert_array_equal(host(sw).numpy(), exp)


def test_plan_flags_out_of_range_ids():
    T, E, k = 6, 8, 2
    ids = _random_ids(T, E, k, 5)
    ids[2, 1] = E + 3
    ids[4, 0] = -1
    desc = moe.make_desc(T, 64, E, k, 64, 0, dtype=moe.MOE_BF16)
    ws = moe.alloc_workspace(desc)
    off = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    tok = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    sr = torch.empty((T, k), dtype=torch.int32, device=DEV)
    moe.moe_plan_dispatch(desc, torch.from_numpy(ids).to(DEV), None, off, tok, sr, None, None,
                          None, ws)
    assert moe.moe_get_device_status(ws, clear=True) == moe.MOE_ERR_DEVICE_INPUT
    s = host(sr).numpy()
    assert s[2, 1] == -1 and s[4, 0] == -1
    assert int(host(off)[-1]) == T * k - 2  # the bad pairs are dropped
    assert moe.moe_get_device_status(ws) == moe.MOE_OK  # cleared


# ---------------------------------------------------------------- expert FFN
FFN_CASES = [
    LayerConfig("f_fp32", T=64, d=256, E=16, I=128, k=2, dtype="f32"),
    LayerConfig("f_fp32_ragged", T=37, d=72, E=5, I=36, k=3, S=1, dtype="f32", gate=1,
                norm_topk=1, routed_scaling=2.0, sel_bias_range=0.1),
    LayerConfig("f_bf16_small_tiles", T=67, d=128, E=8, I=192, k=2, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    LayerConfig("f_bf16_large_tiles", T=600, d=256, E=4, I=320, k=2),
    LayerConfig("f_bf16_skewed", T=700, d=192, E=12, I=128, k=3, zipf_s=1.2),
    LayerConfig("f_bf16_one_token", T=1, d=512, E=32, I=256, k=4, S=1, gate=1, norm_topk=1,
                routed_scaling=2.8, sel_bias_range=0.1),
    # ~100 rows per batch: 128-token tiles, shared batch of 300 rows in 3 tiles
    LayerConfig("f_bf16_mid_tiles", T=300, d=192, E=8, I=320, k=2, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    # a hot expert with more than four 256-token tiles (weight-block-minor order)
    LayerConfig("f_bf16_hot_expert", T=2000, d=128, E=8, I=128, k=2, zipf_s=1.2),
]


@pytest.mark.parametrize("cfg", FFN_CASES, ids=lambda c: c.name)
def test_expert_ffn_and_combine_parity(cfg):
    inp = _case(cfg, seed=5)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                                  **_oracle_kw(cfg, inp))
    ref = oracle.plan(ids_ref, cfg.E, cfg.S)
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    P = cfg.T * (cfg.k + cfg.S)
    off = torch.from_numpy(ref["expert_offsets"]).to(DEV)
    tok = torch.from_numpy(ref["token_indices"]).to(DEV)
    y_perm = torch.zeros((P, cfg.d), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn(desc, inp["x"], off, tok, None, inp["Wg"], inp["Wu"], inp["Wd"], y_perm,
                       ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    # oracle: each batch through its expert
    x_h = host(inp["x"])
    rows = np.zeros((P, cfg.d))
    o = ref["expert_offsets"]
    for e in range(cfg.E + cfg.S):
        if o[e + 1] > o[e]:
            rows[o[e]:o[e + 1]] = oracle.expert_rows(x_h, host(inp["Wg"][e]), host(inp["Wu"][e]),
                                                     host(inp["Wd"][e]), ref["token_indices"][o[e]:o[e + 1]])
    got = host(y_perm).double().numpy()
    assert rel_err(got, rows) <= y_tol(cfg), rel_err(got, rows)
    # per-expert check too: no batch may be silently wrong inside the global max
    for e in range(cfg.E + cfg.S):
        if o[e + 1] > o[e]:
            assert rel_err(got[o[e]:o[e + 1]], rows[o[e]:o[e + 1]]) <= 4 * y_tol(cfg)
    # combine of the GPU rows against the oracle combine of the same rows
    res = torch.randn((cfg.T, cfg.d), generator=torch.Generator(device=DEV).manual_seed(2),
                      device=DEV)
    g_w = torch.from_numpy(w_ref.astype(np.float32)).to(DEV)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=DEV)
    sr = torch.from_numpy(ref["slot_row"]).to(DEV)
    moe.moe_combine(desc, y_perm, sr, g_w, res, y)
    ref_y = oracle.combine(got, ref["slot_row"], cfg.k, cfg.S, w=w_ref.astype(np.float32),
                           residual=host(res))
    assert rel_err(host(y).numpy(), ref_y) <= 1e-6


# Batch sizes chosen to land on every tile edge of the large-tile paths: 32-row
# MMA widths (pair halves of 16 rows), 160-row tiles (SM-pair gate/up), 256-row
# tiles (SM-pair down, one-SM gate/up), several tiles per batch, and weight
# blocks of 256 rows that end inside a matrix (I = 320, d = 192).
TILE_EDGE_CASES = [
    ("pair160", LayerConfig("edges_pair160", T=689, d=256, E=10, I=320, k=2),
     [1, 15, 16, 17, 33, 159, 160, 161, 300, 516]),
    ("onesm256", LayerConfig("edges_onesm256", T=1216, d=192, E=8, I=320, k=2),
     [1, 255, 256, 257, 600, 1000, 31, 32]),
]


@pytest.mark.parametrize("name,cfg,sizes", TILE_EDGE_CASES, ids=[c[0] for c in TILE_EDGE_CASES])
def test_expert_ffn_tile_edges(name, cfg, sizes):
    P = cfg.T * cfg.k
    assert sum(sizes) == P and len(sizes) == cfg.E
    inp = make_inputs(cfg, seed=11, device=DEV)
    rng = np.random.default_rng(11)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    tok = rng.integers(0, cfg.T, size=P).astype(np.int32)
    desc = moe.desc_from_config(cfg)
    ws = moe.alloc_workspace(desc)
    y_perm = torch.full((P, cfg.d), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn(desc, inp["x"], torch.from_numpy(off).to(DEV),
                       torch.from_numpy(tok).to(DEV), None, inp["Wg"], inp["Wu"], inp["Wd"],
                       y_perm, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    got = host(y_perm).double().numpy()
    x_h = host(inp["x"])
    for e in range(cfg.E):
        ref = oracle.expert_rows(x_h, host(inp["Wg"][e]), host(inp["Wu"][e]), host(inp["Wd"][e]),
                                 tok[off[e]:off[e + 1]])
        err = rel_err(got[off[e]:off[e + 1]], ref)
        assert err <= y_tol(cfg), (e, sizes[e], err)


# The routing inside a layer call equals the separate router call bit for bit
# (ids and gate weights), and a second layer call on the same workspace
# repeats the first exactly.
ROUTE_REPEAT_CASES = [
    LayerConfig("fr_one_token", T=1, d=512, E=32, I=64, k=4, S=1, gate=1, norm_topk=1,
                routed_scaling=2.8, sel_bias_range=0.1),
    LayerConfig("fr_fp32_ragged", T=37, d=72, E=5, I=36, k=3, S=1, dtype="f32", gate=1,
                norm_topk=1, routed_scaling=2.0, sel_bias_range=0.1),
    LayerConfig("fr_max_experts", T=40, d=128, E=1024, I=64, k=32, S=4, norm_topk=1),
]


@pytest.mark.parametrize("cfg", ROUTE_REPEAT_CASES, ids=lambda c: c.name)
def test_layer_routing_matches_router_call_and_repeats(cfg):
    inp = _case(cfg, seed=13)
    y, ids, w, ws = _gpu_layer(cfg, inp)
    ids2 = torch.full_like(ids, -5)
    w2 = torch.full_like(w, float("nan"))
    desc = moe.desc_from_config(cfg)
    moe.moe_route(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"], ids2, w2, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(ids, ids2)
    assert torch.equal(w, w2)
    # a second layer call on the same workspace agrees bit for bit
    y3 = torch.full_like(y, float("nan"))
    ids3 = torch.full_like(ids, -7)
    w3 = torch.empty_like(w)
    moe.moe_layer_forward(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"],
                          inp["Wg"], inp["Wu"], inp["Wd"], None, y3, ids3, w3, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(ids, ids3) and torch.equal(w, w3) and torch.equal(y, y3)


# The layer call with host buffers equals the device call bit for bit.
@pytest.mark.parametrize("cfg", [FFN_CASES[0], FFN_CASES[5], FFN_CASES[6]],
                         ids=lambda c: c.name)
def test_layer_forward_host_buffers(cfg):
    inp = _case(cfg, seed=17)
    desc = moe.desc_from_config(cfg)
    layer = moe.MoeLayer(desc, inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"],
                         logit_bias=inp["logit_bias"], sel_bias=inp["sel_bias"])
    y_dev = layer.forward(inp["x"])
    x_host = host(inp["x"]).pin_memory()
    y_host = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32).pin_memory()
    layer.forward_host(x_host, y_host)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    assert torch.equal(y_host, host(y_dev))


# The pipelined call with host buffers: every step equals the device call on
# its input bit for bit.  Step 0's input reaches its host buffer through a copy
# enqueued on the stream just before the call, behind a device sleep, so an
# upload that did not wait for the stream would read NaNs; the last output is
# read back by a copy enqueued after the call.
def _step_inputs(x, n):
    return [torch.roll(x, shifts=3 * i, dims=0) * (1.0 - 0.25 * (i % 3)) for i in range(n)]


@pytest.mark.parametrize("n_steps", [1, 2, 5])
@pytest.mark.parametrize("cfg", [FFN_CASES[0], FFN_CASES[6]], ids=lambda c: c.name)
def test_layer_forward_host_pipelined(cfg, n_steps):
    inp = _case(cfg, seed=23)
    desc = moe.desc_from_config(cfg)
    layer = moe.MoeLayer(desc, inp["Wr"], inp["Wg"], inp["Wu"], inp["Wd"],
                         logit_bias=inp["logit_bias"], sel_bias=inp["sel_bias"])
    xs = _step_inputs(inp["x"], n_steps)
    want = [host(layer.forward(x)) for x in xs]
    torch.cuda.synchronize()
    x_hosts = [host(x).pin_memory() for x in xs]
    x_hosts[0].fill_(float("nan"))
    y_hosts = [torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32).pin_memory()
               for _ in range(n_steps)]
    torch.cuda._sleep(2_000_000)  # ~1 ms of device time ahead of the copy below
    x_hosts[0].copy_(xs[0], non_blocking=True)
    layer.forward_host_pipelined(x_hosts, y_hosts)
    y_last = y_hosts[-1].to(DEV, non_blocking=True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    for i in range(n_steps):
        assert torch.equal(y_hosts[i], want[i]), i
    assert torch.equal(host(y_last), want[-1])


# ---------------------------------------------------------------- whole layer, small
# the largest shape the layer record admits: E=1024 routed + 4 shared experts
# (1028 groups, the grouped GEMM's limit), top-32; softmax scores, whose gaps
# among the top 33 of 1024 stay wide enough for the routing margin
MAX_GROUPS = LayerConfig("l_max_groups", T=40, d=128, E=1024, I=64, k=32, S=4, norm_topk=1)
LAYER_CASES = FFN_CASES + [ROUTER_CASES[2], ROUTER_CASES[3], MAX_GROUPS] + [
    c for c in ROUTER_CASES if c.name.startswith("r_k_equals_E")]


@pytest.mark.parametrize("cfg", LAYER_CASES, ids=lambda c: c.name)
def test_layer_forward_parity_small(cfg):
    inp = _case(cfg, seed=7)
    residual = torch.randn((cfg.T, cfg.d), generator=torch.Generator(device=DEV).manual_seed(9),
                           device=DEV)
    y, ids, w, _ = _gpu_layer(cfg, inp, residual=residual)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                                  **_oracle_kw(cfg, inp))
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    check_weights(host(w).numpy(), w_ref, inp, cfg)
    y_ref, _, _ = _oracle_forward(cfg, inp, np.arange(cfg.T, dtype=np.int32), ids_ref,
                                  residual=residual)
    # the residual is exact in fp32; compare the MoE part against its own scale
    moe_part = host(y).double().numpy() - host(residual).double().numpy()
    moe_ref = y_ref - host(residual).double().numpy()
    assert rel_err(moe_part, moe_ref) <= y_tol(cfg), rel_err(moe_part, moe_ref)


# Seeded random tiny shapes across the whole layer (both dtypes, both gate
# families, with and without a shared expert): T in 1..67, E in 4..40, k in
# 1..min(E, 8); d and I multiples of 64 (bf16) or of 8 / 4 (fp32).
def _random_tiny_config(seed):
    rng = np.random.default_rng(1000 + seed)
    f32 = seed % 3 == 0
    E = int(rng.integers(4, 41))
    k = int(rng.integers(1, min(E, 32) + 1))  # the library's whole k range
    S = int(rng.integers(0, 2))
    gate = int(rng.integers(0, 2))
    if f32:
        d, I = 8 * int(rng.integers(2, 33)), 4 * int(rng.integers(2, 65))
    else:
        d, I = 64 * int(rng.integers(1, 5)), 64 * int(rng.integers(1, 5))
        while (E + S) * min(d, I) < 128:
            d, I = d + 64, I + 64
    return LayerConfig("tiny_%d" % seed, T=int(rng.integers(1, 68)), d=d, E=E, I=I, k=k, S=S,
                       gate=gate, norm_topk=gate, routed_scaling=2.0 if gate else 1.0,
                       sel_bias_range=0.1 if gate else 0.0, dtype="f32" if f32 else "bf16")


@pytest.mark.parametrize("seed", range(16))
def test_layer_forward_random_tiny_shapes(seed):
    cfg = _random_tiny_config(seed)
    inp = _case(cfg, seed=seed)
    y, ids, w, _ = _gpu_layer(cfg, inp)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                                  **_oracle_kw(cfg, inp))
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    check_weights(host(w).numpy(), w_ref, inp, cfg)
    y_ref, _, _ = _oracle_forward(cfg, inp, np.arange(cfg.T, dtype=np.int32), ids_ref)
    assert rel_err(host(y).double().numpy(), y_ref) <= y_tol(cfg), (cfg, rel_err(host(y).double().numpy(), y_ref))


def test_layer_forward_with_no_tokens_is_a_no_op():
    cfg = FFN_CASES[4]
    inp = _case(cfg, seed=2)
    desc = moe.desc_from_config(cfg, T=0)
    ws = torch.zeros((16,), dtype=torch.uint8, device=DEV)
    y = torch.full((1, cfg.d), 7.0, dtype=torch.float32, device=DEV)
    c0 = moe.moe_launch_count()
    moe.moe_layer_forward(desc, inp["x"][:0], inp["Wr"], inp["logit_bias"], inp["sel_bias"],
                          inp["Wg"], inp["Wu"], inp["Wd"], None, y[:0], None, None, ws)
    torch.cuda.synchronize()
    assert moe.moe_launch_count() == c0 and bool((y == 7.0).all())


def test_layer_forward_is_deterministic():
    cfg = FFN_CASES[4]
    inp = _case(cfg, seed=11)
    y1, ids1, w1, _ = _gpu_layer(cfg, inp)
    y2, ids2, w2, _ = _gpu_layer(cfg, inp)
    assert torch.equal(ids1, ids2) and torch.equal(w1, w2) and torch.equal(y1, y2)


# ---------------------------------------------------------------- the five workloads, full size
def _full_size(cfg, seed=0):
    """The workload at full size: routing and plan bit-exact on all tokens, and
    every token's output against the per-token oracle."""
    inp = _case(cfg, seed=seed)
    y, ids, w, ws = _gpu_layer(cfg, inp)
    ids_ref, w_ref = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                                  **_oracle_kw(cfg, inp))
    np.testing.assert_array_equal(host(ids).numpy(), ids_ref)
    check_weights(host(w).numpy(), w_ref, inp, cfg)
    # the plan of the full routing, bit-exact
    desc = moe.desc_from_config(cfg)
    P = cfg.T * (cfg.k + cfg.S)
    off = torch.empty((cfg.E + cfg.S + 1,), dtype=torch.int32, device=DEV)
    tok = torch.empty((P,), dtype=torch.int32, device=DEV)
    sr = torch.empty((cfg.T, cfg.k + cfg.S), dtype=torch.int32, device=DEV)
    moe.moe_plan_dispatch(desc, ids, None, off, tok, sr, None, None, None, ws)
    ref = oracle.plan(ids_ref, cfg.E, cfg.S)
    np.testing.assert_array_equal(host(off).numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(host(tok).numpy(), ref["token_indices"])
    np.testing.assert_array_equal(host(sr).numpy(), ref["slot_row"])
    y_host = host(y).double().numpy()
    del y, ws
    torch.cuda.empty_cache()
    # every token through the oracle, one by one
    y_ref, ids_o, _ = _oracle_forward(cfg, inp, np.arange(cfg.T, dtype=np.int32), ids_ref)
    np.testing.assert_array_equal(ids_o, ids_ref)
    check_all_tokens(y_host, y_ref, ids_ref, cfg, y_tol(cfg))
    del inp
    torch.cuda.empty_cache()


def test_full_tiny_fp32():
    _full_size(CONFIGS["tiny_fp32"])


def test_full_qwen_t512():
    _full_size(CONFIGS["qwen_t512"])


def test_full_deepseek_prefill():
    _full_size(CONFIGS["deepseek_prefill"])


def test_full_skewed_zipf():
    _full_size(CONFIGS["skewed_zipf"])


@pytest.mark.parametrize("T", DECODE_TS)
def test_full_kimi_decode(T):
    _full_size(KIMI_DECODE.with_T(T))


# ---------------------------------------------------------------- partial combine
@pytest.mark.parametrize("cfg", [FFN_CASES[2], FFN_CASES[1], ROUTER_CASES[3]],
                         ids=lambda c: c.name)
def test_combine_partial_parity(cfg):
    """The partial combine against the oracle, with routed experts (and, where
    present, the shared expert) unavailable; all available = moe_combine exactly."""
    inp = _case(cfg, seed=21)
    ids, w = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                          **_oracle_kw(cfg, inp))
    plan = oracle.plan(ids, cfg.E, cfg.S)
    desc = moe.desc_from_config(cfg)
    P = cfg.T * (cfg.k + cfg.S)
    g = torch.Generator(device=DEV).manual_seed(4)
    y_perm = torch.randn((P, cfg.d), generator=g, device=DEV).to(cfg.torch_dtype)
    rows = host(y_perm).double().numpy()
    sr = torch.from_numpy(plan["slot_row"]).to(DEV)
    g_ids = torch.from_numpy(ids).to(DEV)
    w32 = w.astype(np.float32)
    g_w = torch.from_numpy(w32).to(DEV)
    avail = np.ones(cfg.E + cfg.S, np.int32)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device=DEV)
    y_ref_full = torch.empty_like(y)
    miss = torch.full((cfg.T, cfg.k + cfg.S), 7, dtype=torch.int32, device=DEV)
    moe.moe_combine_partial(desc, y_perm, sr, g_ids, g_w, torch.from_numpy(avail).to(DEV), None,
                            y, miss)
    moe.moe_combine(desc, y_perm, sr, g_w, None, y_ref_full)
    assert torch.equal(y, y_ref_full) and int(miss.sum()) == 0
    rng = np.random.default_rng(1)
    avail[rng.choice(cfg.E, size=max(1, cfg.E // 3), replace=False)] = 0
    if cfg.S:
        avail[cfg.E] = 0
    res = torch.randn((cfg.T, cfg.d), generator=g, device=DEV)
    moe.moe_combine_partial(desc, y_perm, sr, g_ids, g_w, torch.from_numpy(avail).to(DEV), res,
                            y, miss)
    y_ref, miss_ref = oracle.combine_partial(rows, plan["slot_row"], ids, w32, avail, cfg.k,
                                             cfg.S, cfg.E, residual=host(res))
    np.testing.assert_array_equal(host(miss).numpy(), miss_ref)
    assert rel_err(host(y).numpy(), y_ref) <= 1e-6
    # the unserved (expert, token) pairs as a list
    pairs = torch.full((P, 2), -9, dtype=torch.int32, device=DEV)
    n_pairs = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    moe.moe_partial_missing_pairs(desc, g_ids, miss, pairs, n_pairs)
    want = oracle.missing_pairs(ids, avail, cfg.k, cfg.S, cfg.E)
    n = int(host(n_pairs)[0])
    assert n == len(want) > 0
    np.testing.assert_array_equal(host(pairs).numpy()[:n], want)
    assert bool((pairs[n:] == -9).all())
