"""Failure detection on the GPU without a fault: every bounded wait in the
library's kernels gives up after about a second, records MOE_ERR_TIMEOUT in the
workspace's device flag and lets its kernel end.  Each case here waits on an
mbarrier that nothing completes, checks the status the host reads, and then runs
a layer forward on the same context and workspace against the oracle, which
shows the context stayed usable.
"""
import time

import pytest
import torch

import oracle
from expert_dispatch_gb300 import moe
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs
from tests.helpers import enforce_margins, host, rel_err, y_tol

pytestmark = pytest.mark.gpu

DEV = "cuda"
CFG = LayerConfig("after_timeout", T=67, d=128, E=8, I=192, k=2, S=1, gate=1, norm_topk=1,
                  routed_scaling=2.5, sel_bias_range=0.1)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from expert_dispatch_gb300 import build
    build.build()
    yield
    torch.cuda.synchronize()


def _forward_matches_oracle(ws):
    inp = enforce_margins(make_inputs(CFG, seed=3, device=DEV), CFG, 3)
    desc = moe.desc_from_config(CFG)
    y = torch.full((CFG.T, CFG.d), float("nan"), dtype=torch.float32, device=DEV)
    ids = torch.empty((CFG.T, CFG.k), dtype=torch.int32, device=DEV)
    w = torch.empty((CFG.T, CFG.k), dtype=torch.float32, device=DEV)
    moe.moe_layer_forward(desc, inp["x"], inp["Wr"], inp["logit_bias"], inp["sel_bias"],
                          inp["Wg"], inp["Wu"], inp["Wd"], None, y, ids, w, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    nE = CFG.E + CFG.S
    Ws = [[host(inp[n][e]) for e in range(nE)] for n in ("Wg", "Wu", "Wd")]
    y_ref, ids_ref, _ = oracle.forward(host(inp["x"]), host(inp["Wr"]), *Ws, CFG.k, CFG.gate,
                                       S=CFG.S, norm_topk=CFG.norm_topk,
                                       routed_scaling=CFG.routed_scaling,
                                       logit_bias=host(inp["logit_bias"]),
                                       sel_bias=host(inp["sel_bias"]))
    assert (host(ids).numpy() == ids_ref).all()
    assert rel_err(host(y).numpy(), y_ref) <= y_tol(CFG)


@pytest.mark.parametrize("which", [0, 1, 2, 3],
                         ids=["thread_wait", "warp_wait", "drain_wait", "shared_abort"])
def test_bounded_wait_expires_and_context_stays_usable(which):
    desc = moe.desc_from_config(CFG)
    ws = moe.alloc_workspace(desc)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_check_bounded_wait(ws, which)
    status = moe.moe_get_device_status(ws, clear=True)
    waited = time.perf_counter() - t0
    assert status == moe.MOE_ERR_TIMEOUT
    assert 0.9 <= waited <= 10.0  # the limit is one second of device time
    assert moe.moe_get_device_status(ws) == moe.MOE_OK  # cleared
    _forward_matches_oracle(ws)


def test_bounded_wait_check_rejects_bad_arguments():
    desc = moe.desc_from_config(CFG)
    ws = moe.alloc_workspace(desc)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_check_bounded_wait(ws, 4)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_check_bounded_wait(ws[:8], 0)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    assert moe.moe_get_device_status(ws) == moe.MOE_OK  # nothing was launched
