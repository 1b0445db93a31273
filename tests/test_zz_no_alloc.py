"""moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate
device memory (their host application owns it all, or they must never call
cudaMalloc).  It must give exactly the rows of moe_expert_ffn, which runs the
same kernels with a caller workspace, call after call -- also after a call for
another layer has left its own data in the one fixed array inside the library
that every call reuses -- and those rows must match the oracle's per-expert
FFN.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs
from tests.helpers import enforce_margins, host, rel_err, y_tol

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [
    LayerConfig("na_bf16_small_tiles", T=67, d=128, E=8, I=192, k=2, S=1, gate=1, norm_topk=1,
                routed_scaling=2.5, sel_bias_range=0.1),
    LayerConfig("na_bf16_large_tiles", T=600, d=256, E=4, I=320, k=2),
    LayerConfig("na_fp32", T=37, d=72, E=5, I=36, k=3, S=1, dtype="f32", gate=1, norm_topk=1,
                routed_scaling=2.0, sel_bias_range=0.1),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from expert_dispatch_gb300 import build
    build.build()


def _layer(cfg, seed):
    """A layer's inputs and the oracle's dispatch plan of its routing."""
    inp = enforce_margins(make_inputs(cfg, seed=seed, device=DEV), cfg, seed)
    ids, _ = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                          norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
                          logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    plan = oracle.plan(ids, cfg.E, cfg.S)
    off = torch.from_numpy(plan["expert_offsets"]).to(DEV)
    tok = torch.from_numpy(plan["token_indices"]).to(DEV)
    return inp, plan, off, tok


def _noalloc(cfg, inp, off, tok):
    P = cfg.T * (cfg.k + cfg.S)
    y = torch.full((P, cfg.d), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn_noalloc(moe.desc_from_config(cfg), inp["x"], off, tok, None, inp["Wg"],
                               inp["Wu"], inp["Wd"], y)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    inp, plan, off, tok = _layer(cfg, 13)
    desc = moe.desc_from_config(cfg)
    P = cfg.T * (cfg.k + cfg.S)
    # the existing entry point, with a workspace
    ws = moe.alloc_workspace(desc)
    y_ws = torch.zeros((P, cfg.d), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn(desc, inp["x"], off, tok, None, inp["Wg"], inp["Wu"], inp["Wd"], y_ws, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    # both run the same kernels on the same plan: the rows must be identical
    y1 = _noalloc(cfg, inp, off, tok)
    assert torch.equal(y1, y_ws)
    # another layer in between leaves different data in the shared scratch;
    # the next call must not depend on it
    other = CASES[(CASES.index(cfg) + 1) % len(CASES)]
    o_inp, _, o_off, o_tok = _layer(other, 14)
    _noalloc(other, o_inp, o_off, o_tok)
    y2 = _noalloc(cfg, inp, off, tok)
    assert torch.equal(y2, y_ws)
    # and the rows against the oracle's per-expert FFN
    o, t = plan["expert_offsets"], plan["token_indices"]
    ref = np.zeros((P, cfg.d))
    for e in range(cfg.E + cfg.S):
        if o[e + 1] > o[e]:
            ref[o[e]:o[e + 1]] = oracle.expert_rows(host(inp["x"]), host(inp["Wg"][e]),
                                                    host(inp["Wu"][e]), host(inp["Wd"][e]),
                                                    t[o[e]:o[e + 1]])
    err = rel_err(host(y2).double().numpy(), ref)
    assert err <= y_tol(cfg), err


def test_noalloc_rejects_layers_beyond_its_scratch():
    """The DeepSeek-layout prefill batch needs ~680 MB of scratch: refused up front."""
    desc = moe.make_desc(4096, 7168, 256, 8, 2048, 1, gate=moe.MOE_GATE_SIGMOID_BIAS,
                         norm_topk=1, routed_scaling=2.5, dtype=moe.MOE_BF16)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    st = moe.lib().moe_expert_ffn_noalloc(ctypes.byref(desc), fake, fake, fake, None, fake, fake,
                                          fake, fake, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
