"""Host-side checks of the C ABI that need no GPU: the library builds, exports
every entry point include/moe.h declares, sizes workspaces, and rejects bad
arguments synchronously before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from expert_dispatch_gb300 import build as moe_build
from expert_dispatch_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_five_layer_calls():
    names = declared_functions()
    for f in ("moe_route", "moe_plan_dispatch", "moe_expert_ffn", "moe_combine",
              "moe_layer_forward", "moe_workspace_size", "moe_status_string"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_[a-z0-9_]+)$", out, flags=re.M))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    assert set(moe.EXPORTED) == set(declared_functions())


def test_desc_layout_matches_header(L):
    assert ctypes.sizeof(moe.LayerDesc) == 11 * 4


def _desc(**kw):
    base = dict(T=64, d=256, E=16, k=2, I=128, S=0, gate=0, norm_topk=0, routed_scaling=1.0,
                dtype=moe.MOE_F32)
    base.update(kw)
    return moe.make_desc(**base)


def _ws_size(L, desc):
    n = ctypes.c_size_t(0)
    st = L.moe_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    return st, n.value


def test_workspace_size(L):
    st, n = _ws_size(L, _desc())
    assert st == moe.MOE_OK and n > 0 and n % 256 == 0
    st, n0 = _ws_size(L, _desc(T=0))
    assert st == moe.MOE_OK and n0 == 0
    # grows with T
    _, n2 = _ws_size(L, _desc(T=640))
    assert n2 > n


@pytest.mark.parametrize("bad,status", [
    (dict(k=17), moe.MOE_ERR_INVALID_ARG),           # k > E
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(E=2000, k=2), moe.MOE_ERR_INVALID_ARG),    # E > 1024
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(S=5), moe.MOE_ERR_INVALID_ARG),
    (dict(gate=7), moe.MOE_ERR_INVALID_ARG),
    (dict(norm_topk=2), moe.MOE_ERR_INVALID_ARG),
    (dict(routed_scaling=float("nan")), moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=9), moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=moe.MOE_BF16, d=96), moe.MOE_ERR_UNSUPPORTED),   # d % 64
    (dict(dtype=moe.MOE_BF16, I=100), moe.MOE_ERR_UNSUPPORTED),  # I % 64
    (dict(d=12), moe.MOE_ERR_UNSUPPORTED),                       # fp32 d % 8
])
def test_bad_descriptors_rejected(L, bad, status):
    st, _ = _ws_size(L, _desc(**bad))
    assert st == status


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def test_null_and_misaligned_pointers_rejected(L):
    d = _desc()
    _, n = _ws_size(L, d)
    ws = FAKE
    assert L.moe_route(ctypes.byref(d), None, FAKE, None, None, FAKE, FAKE, ws, n, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_route(ctypes.byref(d), ctypes.c_void_p(0x10004), FAKE, None, None, FAKE, FAKE,
                       ws, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward(ctypes.byref(d), FAKE, FAKE, None, None, FAKE, FAKE, None, None,
                               FAKE, None, None, ws, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(d), FAKE, None, None, None, FAKE, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_selection_bias_needs_sigmoid_family(L):
    d = _desc(gate=moe.MOE_GATE_SOFTMAX_TOPK)
    _, n = _ws_size(L, d)
    st = L.moe_route(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, n, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_workspace_too_small_rejected(L):
    d = _desc()
    _, n = _ws_size(L, d)
    st = L.moe_route(ctypes.byref(d), FAKE, FAKE, None, None, FAKE, FAKE, FAKE, n - 256, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = L.moe_plan_dispatch(ctypes.byref(d), FAKE, None, FAKE, FAKE, FAKE, None, None, None,
                             None, n, None)
    assert st == moe.MOE_ERR_WORKSPACE


def test_zero_tokens_is_a_noop(L):
    d = _desc(T=0)
    # nothing is launched, so no device is needed
    assert L.moe_layer_forward(ctypes.byref(d), None, None, None, None, None, None, None, None,
                               None, None, None, None, 0, None) == moe.MOE_OK


def test_status_strings(L):
    for s in range(7):
        assert moe.moe_status_string(s).startswith("MOE_")
    assert "unknown" in moe.moe_status_string(42)


def test_pipelined_host_call_argument_checks(L):
    d = _desc()
    _, n = _ws_size(L, d)
    two = (ctypes.c_void_p * 2)(FAKE.value, FAKE.value)
    holed = (ctypes.c_void_p * 2)(FAKE.value, None)
    as_vp = lambda a: ctypes.cast(a, ctypes.c_void_p)
    for fn in (L.moe_layer_forward_host_pipelined, L.moe_layer_forward_q8_host_pipelined):
        q8 = fn is L.moe_layer_forward_q8_host_pipelined
        dd = _desc(dtype=moe.MOE_BF16) if q8 else d
        _, nn = _ws_size(L, dd)
        w = None  # weights are not reached: argument checks fail first
        call = lambda steps, xs, ys, ws_bytes: fn(ctypes.byref(dd), steps, xs, FAKE, None, None,
                                                  w, w, w, ys, FAKE, ws_bytes, None)
        # no steps (or no tokens): nothing is enqueued, no device is needed
        assert call(0, None, None, nn) == moe.MOE_OK
        assert call(-1, as_vp(two), as_vp(two), nn) == moe.MOE_ERR_INVALID_ARG
        assert call(2, None, as_vp(two), nn) == moe.MOE_ERR_INVALID_ARG
        assert call(2, as_vp(two), None, nn) == moe.MOE_ERR_INVALID_ARG
        assert call(2, as_vp(holed), as_vp(two), nn) == moe.MOE_ERR_INVALID_ARG
        assert call(2, as_vp(two), as_vp(holed), nn) == moe.MOE_ERR_INVALID_ARG
        assert call(2, as_vp(two), as_vp(two), nn - 256) == moe.MOE_ERR_WORKSPACE


def test_missing_pairs_argument_checks(L):
    d = _desc()
    fn = L.moe_partial_missing_pairs
    assert fn(ctypes.byref(d), FAKE, FAKE, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(d), None, FAKE, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(d), FAKE, None, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(d), FAKE, FAKE, None, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(d), FAKE, FAKE, ctypes.c_void_p(0x10004), FAKE, None) == \
        moe.MOE_ERR_INVALID_ARG
    bad = _desc(k=0)
    assert fn(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
