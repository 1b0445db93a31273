"""moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate
device memory (their host application owns it all, or they must never call
cudaMalloc).  It must give the results of moe_expert_ffn, which uses a caller
workspace, call after call, although its scratch is one fixed array inside the
library that every call reuses.  This file is collected last on purpose."""
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


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    inp = enforce_margins(make_inputs(cfg, seed=13, device=DEV), cfg, 13)
    ids, _ = oracle.route(host(inp["x"]), host(inp["Wr"]), cfg.k, cfg.gate,
                          norm_topk=cfg.norm_topk, routed_scaling=cfg.routed_scaling,
                          logit_bias=host(inp["logit_bias"]), sel_bias=host(inp["sel_bias"]))
    plan = oracle.plan(ids, cfg.E, cfg.S)
    off = torch.from_numpy(plan["expert_offsets"]).to(DEV)
    tok = torch.from_numpy(plan["token_indices"]).to(DEV)
    desc = moe.desc_from_config(cfg)
    P = cfg.T * (cfg.k + cfg.S)
    # the existing entry point, with a workspace
    ws = moe.alloc_workspace(desc)
    y_ws = torch.zeros((P, cfg.d), dtype=cfg.torch_dtype, device=DEV)
    moe.moe_expert_ffn(desc, inp["x"], off, tok, None, inp["Wg"], inp["Wu"], inp["Wd"], y_ws, ws)
    torch.cuda.synchronize()
    ref = host(y_ws).double().numpy()
    assert np.isfinite(ref).all() and np.abs(ref).max() > 0
    # the allocation-free one, twice in a row (the second call reuses the scratch)
    for _ in range(2):
        y_na = torch.full((P, cfg.d), float("nan"), dtype=cfg.torch_dtype, device=DEV)
        moe.moe_expert_ffn_noalloc(desc, inp["x"], off, tok, None, inp["Wg"], inp["Wu"],
                                   inp["Wd"], y_na)
        torch.cuda.synchronize()
        got = host(y_na).double().numpy()
        assert rel_err(got, ref) <= y_tol(cfg), rel_err(got, ref)


def test_noalloc_rejects_layers_beyond_its_scratch():
    """The DeepSeek-layout prefill batch needs ~680 MB of scratch: refused up front."""
    desc = moe.make_desc(4096, 7168, 256, 8, 2048, 1, gate=moe.MOE_GATE_SIGMOID_BIAS,
                         norm_topk=1, routed_scaling=2.5, dtype=moe.MOE_BF16)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    st = moe.lib().moe_expert_ffn_noalloc(ctypes.byref(desc), fake, fake, fake, None, fake, fake,
                                          fake, fake, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
