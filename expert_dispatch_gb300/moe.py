"""Thin Python binding of libmoe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch tensors (PyTorch supplies device memory and
streams); each function checks device, dtype, shape and contiguity, passes raw
pointers and the current CUDA stream, and raises ``MoeError`` on a non-OK
status.  There is no fallback: if libmoe.so is missing, every call raises.

Entry points carry the C names: moe_workspace_size, moe_workspace_init,
moe_route, moe_plan_dispatch, moe_expert_ffn, moe_combine, moe_layer_forward,
moe_get_device_status, moe_status_string, moe_launch_count,
moe_profile_enable, moe_profile_query, moe_profile_list, the Q8_0 and no-alloc variants, the
slot cache (moe_slot_cache_*) and the expert tier (moe_tier_*).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_INPUT = 6

MOE_GATE_SOFTMAX_TOPK = 0
MOE_GATE_SIGMOID_BIAS = 1
MOE_F32 = 0
MOE_BF16 = 1

EXPORTED = ("moe_workspace_size", "moe_workspace_init", "moe_route", "moe_plan_dispatch",
            "moe_expert_ffn", "moe_combine", "moe_layer_forward", "moe_get_device_status",
            "moe_status_string", "moe_launch_count", "moe_profile_enable", "moe_profile_query",
            "moe_expert_ffn_noalloc", "moe_combine_partial", "moe_partial_missing_pairs",
            "moe_profile_list",
            "moe_quantize_q8_0",
            "moe_expert_ffn_q8", "moe_layer_forward_q8", "moe_slot_cache_create",
            "moe_slot_cache_destroy", "moe_slot_cache_assign", "moe_slot_cache_slot_of",
            "moe_slot_cache_get_stats", "moe_tier_create", "moe_tier_destroy",
            "moe_tier_prefetch", "moe_tier_forward", "moe_tier_get_stats", "moe_host_alloc",
            "moe_host_free", "moe_check_bounded_wait", "moe_layer_forward_host",
            "moe_layer_forward_q8_host", "moe_layer_forward_host_pipelined",
            "moe_layer_forward_q8_host_pipelined")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, moe_status_string(status)))


class LayerDesc(ctypes.Structure):
    """moe_layer_desc"""
    _fields_ = [("layer", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("I", ctypes.c_int32),
                ("S", ctypes.c_int32), ("gate", ctypes.c_int32), ("norm_topk", ctypes.c_int32),
                ("routed_scaling", ctypes.c_float), ("dtype", ctypes.c_int32)]


class Q8WeightStruct(ctypes.Structure):
    """moe_q8_weight"""
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class TierStats(ctypes.Structure):
    """moe_tier_stats"""
    _fields_ = [("steps", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("extra_passes", ctypes.c_uint64),
                ("bytes_loaded", ctypes.c_uint64), ("n_slots", ctypes.c_int32),
                ("resident", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def make_desc(T, d, E, k, I, S=0, gate=MOE_GATE_SOFTMAX_TOPK, norm_topk=0, routed_scaling=1.0,
              dtype=MOE_BF16, layer=0) -> LayerDesc:
    return LayerDesc(layer, T, d, E, k, I, S, gate, norm_topk, routed_scaling, dtype)


def desc_from_config(cfg, T=None) -> LayerDesc:
    """Layer record of a workload config (expert_dispatch_gb300.inputs.LayerConfig)."""
    return make_desc(cfg.T if T is None else T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.S, cfg.gate,
                     cfg.norm_topk, cfg.routed_scaling,
                     MOE_F32 if cfg.dtype == "f32" else MOE_BF16)


_lib = None


def lib():
    """Open libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libmoe.so is not built (run python -m expert_dispatch_gb300.build); "
                           "this package has no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(LayerDesc)
    L.moe_workspace_size.argtypes = [D, ctypes.POINTER(sz)]
    L.moe_workspace_init.argtypes = [vp, sz, vp]
    L.moe_route.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_plan_dispatch.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_expert_ffn.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_combine.argtypes = [D, vp, vp, vp, vp, vp, vp]
    L.moe_layer_forward.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_get_device_status.argtypes = [vp, sz, i32, vp]
    L.moe_check_bounded_wait.argtypes = [vp, sz, i32, vp]
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_launch_count.argtypes = []
    L.moe_launch_count.restype = ctypes.c_int64
    L.moe_expert_ffn_noalloc.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_combine_partial.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_partial_missing_pairs.argtypes = [D, vp, vp, vp, vp, vp]
    Q = ctypes.POINTER(Q8WeightStruct)
    L.moe_quantize_q8_0.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
    L.moe_expert_ffn_q8.argtypes = [D, vp, vp, vp, vp, Q, Q, Q, vp, vp, sz, vp]
    L.moe_layer_forward_q8.argtypes = [D, vp, vp, vp, vp, Q, Q, Q, vp, vp, vp, vp, vp, sz, vp]
    L.moe_layer_forward_host.argtypes = [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_layer_forward_q8_host.argtypes = [D, vp, vp, vp, vp, Q, Q, Q, vp, vp, vp, vp, vp, sz,
                                            vp]
    L.moe_layer_forward_host_pipelined.argtypes = [D, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                                   vp]
    L.moe_layer_forward_q8_host_pipelined.argtypes = [D, i32, vp, vp, vp, vp, Q, Q, Q, vp, vp, sz,
                                                      vp]
    vpp = ctypes.POINTER(ctypes.c_void_p)
    ip = ctypes.POINTER(ctypes.c_int32)
    TS = ctypes.POINTER(TierStats)
    L.moe_slot_cache_create.argtypes = [i32, i32, vpp]
    L.moe_slot_cache_destroy.argtypes = [vp]
    L.moe_slot_cache_assign.argtypes = [vp, vp, i32, vp, vp, vp, ip]
    L.moe_slot_cache_slot_of.argtypes = [vp, i32, ip]
    L.moe_slot_cache_get_stats.argtypes = [vp, TS]
    L.moe_tier_create.argtypes = [D, vp, vp, vp, sz, vpp]
    L.moe_tier_destroy.argtypes = [vp]
    L.moe_tier_prefetch.argtypes = [vp, vp, i32, vp]
    L.moe_tier_forward.argtypes = [vp, D, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_tier_get_stats.argtypes = [vp, TS]
    L.moe_host_alloc.argtypes = [sz, vpp]
    L.moe_host_free.argtypes = [vp]
    L.moe_profile_enable.argtypes = [i32]
    L.moe_profile_query.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_float)]
    L.moe_profile_list.argtypes = [ctypes.c_char_p, ctypes.c_int32, vp, vp,
                                   ctypes.POINTER(ctypes.c_int32)]
    for f in EXPORTED:
        if f not in ("moe_status_string", "moe_launch_count"):
            getattr(L, f).restype = ctypes.c_int
    _lib = L
    return L


# ---------------------------------------------------------------- marshalling helpers
def _p(t, dtype=None, what="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _act_dtype(desc):
    return torch.float32 if desc.dtype == MOE_F32 else torch.bfloat16


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def _need(t, shape, what):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))


# ---------------------------------------------------------------- entry points
def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_workspace_size(desc: LayerDesc) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def alloc_workspace(desc: LayerDesc, device="cuda") -> torch.Tensor:
    """A uint8 device buffer of moe_workspace_size(desc) bytes, flag cleared."""
    ws = torch.empty(max(moe_workspace_size(desc), 256), dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_workspace_init(ws, stream=None):
    _check(lib().moe_workspace_init(_p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)),
           "moe_workspace_init")


def moe_route(desc, x, Wr, logit_bias, sel_bias, topk_ids, topk_w, ws, stream=None):
    dt = _act_dtype(desc)
    _need(x, (desc.T, desc.d), "x")
    _need(Wr, (desc.E, desc.d), "Wr")
    _need(topk_ids, (desc.T, desc.k), "topk_ids")
    _need(topk_w, (desc.T, desc.k), "topk_w")
    st = lib().moe_route(ctypes.byref(desc), _p(x, dt, "x"), _p(Wr, dt, "Wr"),
                         _p(logit_bias, torch.float32, "logit_bias"),
                         _p(sel_bias, torch.float32, "sel_bias"),
                         _p(topk_ids, torch.int32, "topk_ids"), _p(topk_w, torch.float32, "topk_w"),
                         _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream))
    _check(st, "moe_route")


def moe_plan_dispatch(desc, topk_ids, topk_w, expert_offsets, token_indices, slot_row,
                      active_ids, n_active, slot_w, ws, stream=None):
    P = desc.T * (desc.k + desc.S)
    _need(topk_ids, (desc.T, desc.k), "topk_ids")
    _need(expert_offsets, (desc.E + desc.S + 1,), "expert_offsets")
    _need(token_indices, (P,), "token_indices")
    _need(slot_row, (desc.T, desc.k + desc.S), "slot_row")
    st = lib().moe_plan_dispatch(
        ctypes.byref(desc), _p(topk_ids, torch.int32, "topk_ids"),
        _p(topk_w, torch.float32, "topk_w"), _p(expert_offsets, torch.int32, "expert_offsets"),
        _p(token_indices, torch.int32, "token_indices"), _p(slot_row, torch.int32, "slot_row"),
        _p(active_ids, torch.int32, "active_ids"), _p(n_active, torch.int32, "n_active"),
        _p(slot_w, torch.float32, "slot_w"), _p(ws, torch.uint8, "workspace"), ws.numel(),
        _stream(stream))
    _check(st, "moe_plan_dispatch")


def moe_expert_ffn(desc, x, expert_offsets, token_indices, slot_w, Wg, Wu, Wd, y_perm, ws,
                   stream=None):
    dt = _act_dtype(desc)
    nE = desc.E + desc.S
    _need(x, (desc.T, desc.d), "x")
    _need(Wg, (nE, desc.I, desc.d), "Wg")
    _need(Wu, (nE, desc.I, desc.d), "Wu")
    _need(Wd, (nE, desc.d, desc.I), "Wd")
    _need(y_perm, (desc.T * (desc.k + desc.S), desc.d), "y_perm")
    st = lib().moe_expert_ffn(
        ctypes.byref(desc), _p(x, dt, "x"), _p(expert_offsets, torch.int32, "expert_offsets"),
        _p(token_indices, torch.int32, "token_indices"), _p(slot_w, torch.float32, "slot_w"),
        _p(Wg, dt, "Wg"), _p(Wu, dt, "Wu"), _p(Wd, dt, "Wd"), _p(y_perm, dt, "y_perm"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream))
    _check(st, "moe_expert_ffn")


def moe_expert_ffn_noalloc(desc, x, expert_offsets, token_indices, slot_w, Wg, Wu, Wd, y_perm,
                           stream=None):
    """moe_expert_ffn without a workspace, for callers that cannot allocate device
    memory (their host application owns it all, or they must never call cudaMalloc).
    The scratch is a fixed 64 MiB array inside the library, shared by every call on
    a device: calls must not overlap on the GPU.  Larger layers raise
    MoeError(MOE_ERR_UNSUPPORTED)."""
    dt = _act_dtype(desc)
    nE = desc.E + desc.S
    _need(x, (desc.T, desc.d), "x")
    _need(Wg, (nE, desc.I, desc.d), "Wg")
    _need(Wu, (nE, desc.I, desc.d), "Wu")
    _need(Wd, (nE, desc.d, desc.I), "Wd")
    _need(y_perm, (desc.T * (desc.k + desc.S), desc.d), "y_perm")
    st = lib().moe_expert_ffn_noalloc(
        ctypes.byref(desc), _p(x, dt, "x"), _p(expert_offsets, torch.int32, "expert_offsets"),
        _p(token_indices, torch.int32, "token_indices"), _p(slot_w, torch.float32, "slot_w"),
        _p(Wg, dt, "Wg"), _p(Wu, dt, "Wu"), _p(Wd, dt, "Wd"), _p(y_perm, dt, "y_perm"),
        _stream(stream))
    _check(st, "moe_expert_ffn_noalloc")


def moe_combine(desc, y_perm, slot_row, topk_w, residual, y, stream=None):
    dt = _act_dtype(desc)
    _need(y_perm, (desc.T * (desc.k + desc.S), desc.d), "y_perm")
    _need(slot_row, (desc.T, desc.k + desc.S), "slot_row")
    _need(y, (desc.T, desc.d), "y")
    st = lib().moe_combine(ctypes.byref(desc), _p(y_perm, dt, "y_perm"),
                           _p(slot_row, torch.int32, "slot_row"),
                           _p(topk_w, torch.float32, "topk_w"),
                           _p(residual, torch.float32, "residual"), _p(y, torch.float32, "y"),
                           _stream(stream))
    _check(st, "moe_combine")


def moe_combine_partial(desc, y_perm, slot_row, topk_ids, topk_w, expert_available, residual, y,
                        missing=None, stream=None):
    """Combine when some experts did not respond (expert_available[E+S] int32):
    weights renormalised over the responding routed experts, unserved slots
    reported in missing[T, k+S]."""
    dt = _act_dtype(desc)
    ks = desc.k + desc.S
    _need(y_perm, (desc.T * ks, desc.d), "y_perm")
    _need(slot_row, (desc.T, ks), "slot_row")
    _need(topk_ids, (desc.T, desc.k), "topk_ids")
    _need(topk_w, (desc.T, desc.k), "topk_w")
    _need(expert_available, (desc.E + desc.S,), "expert_available")
    _need(y, (desc.T, desc.d), "y")
    if missing is not None:
        _need(missing, (desc.T, ks), "missing")
    st = lib().moe_combine_partial(
        ctypes.byref(desc), _p(y_perm, dt, "y_perm"), _p(slot_row, torch.int32, "slot_row"),
        _p(topk_ids, torch.int32, "topk_ids"), _p(topk_w, torch.float32, "topk_w"),
        _p(expert_available, torch.int32, "expert_available"),
        _p(residual, torch.float32, "residual"), _p(y, torch.float32, "y"),
        _p(missing, torch.int32, "missing"), _stream(stream))
    _check(st, "moe_combine_partial")


def moe_partial_missing_pairs(desc, topk_ids, missing, pairs, n_pairs, stream=None):
    """The (expert, token) pairs flagged in a partial combine's missing mask,
    written to pairs[T*(k+S), 2] in token, then slot order; n_pairs[1] gets the
    count."""
    ks = desc.k + desc.S
    _need(topk_ids, (desc.T, desc.k), "topk_ids")
    _need(missing, (desc.T, ks), "missing")
    _need(pairs, (desc.T * ks, 2), "pairs")
    _need(n_pairs, (1,), "n_pairs")
    st = lib().moe_partial_missing_pairs(
        ctypes.byref(desc), _p(topk_ids, torch.int32, "topk_ids"),
        _p(missing, torch.int32, "missing"), _p(pairs, torch.int32, "pairs"),
        _p(n_pairs, torch.int32, "n_pairs"), _stream(stream))
    _check(st, "moe_partial_missing_pairs")


def moe_layer_forward(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, residual, y, topk_ids_out,
                      topk_w_out, ws, stream=None):
    dt = _act_dtype(desc)
    nE = desc.E + desc.S
    _need(x, (desc.T, desc.d), "x")
    _need(Wr, (desc.E, desc.d), "Wr")
    _need(Wg, (nE, desc.I, desc.d), "Wg")
    _need(Wu, (nE, desc.I, desc.d), "Wu")
    _need(Wd, (nE, desc.d, desc.I), "Wd")
    _need(y, (desc.T, desc.d), "y")
    st = lib().moe_layer_forward(
        ctypes.byref(desc), _p(x, dt, "x"), _p(Wr, dt, "Wr"),
        _p(logit_bias, torch.float32, "logit_bias"), _p(sel_bias, torch.float32, "sel_bias"),
        _p(Wg, dt, "Wg"), _p(Wu, dt, "Wu"), _p(Wd, dt, "Wd"),
        _p(residual, torch.float32, "residual"), _p(y, torch.float32, "y"),
        _p(topk_ids_out, torch.int32, "topk_ids_out"), _p(topk_w_out, torch.float32, "topk_w_out"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream))
    _check(st, "moe_layer_forward")


# ---------------------------------------------------------------- Q8_0 expert weights
class Q8Weight:
    """A Q8_0 projection on the device: int8 codes [n, rows, K] and the f16 scale
    bit patterns (held as int16) [n, K/32, rows]."""

    def __init__(self, q: torch.Tensor, scale: torch.Tensor):
        if q.dtype != torch.int8 or scale.dtype != torch.int16:
            raise TypeError("Q8_0 codes must be int8 and scales int16 (f16 bits)")
        n, rows, K = q.shape
        if tuple(scale.shape) != (n, K // 32, rows):
            raise ValueError("scale shape %s, expected %s" % (tuple(scale.shape), (n, K // 32, rows)))
        self.q, self.scale = q, scale

    def struct(self):
        return Q8WeightStruct(_p(self.q, torch.int8, "q"), _p(self.scale, torch.int16, "scale"))

    @property
    def shape(self):
        return tuple(self.q.shape)


def moe_quantize_q8_0(w, q, scale, stream=None):
    """Q8_0 codes and scales of w [n, rows, K] (fp32 or bf16, on the device)."""
    n, rows, K = w.shape
    dt = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}.get(w.dtype)
    if dt is None:
        raise TypeError("w must be fp32 or bf16")
    _need(q, (n, rows, K), "q")
    _need(scale, (n, K // 32, rows), "scale")
    st = lib().moe_quantize_q8_0(n, rows, K, dt, _p(w, w.dtype, "w"), _p(q, torch.int8, "q"),
                                 _p(scale, torch.int16, "scale"), _stream(stream))
    _check(st, "moe_quantize_q8_0")


def quantize_q8_0(w, stream=None) -> Q8Weight:
    n, rows, K = w.shape
    q = torch.empty((n, rows, K), dtype=torch.int8, device=w.device)
    s = torch.empty((n, K // 32, rows), dtype=torch.int16, device=w.device)
    moe_quantize_q8_0(w, q, s, stream)
    return Q8Weight(q, s)


def _q8_check(desc, Wg, Wu, Wd):
    nE = desc.E + desc.S
    for name, W, shape in (("Wg", Wg, (nE, desc.I, desc.d)), ("Wu", Wu, (nE, desc.I, desc.d)),
                           ("Wd", Wd, (nE, desc.d, desc.I))):
        if not isinstance(W, Q8Weight) or W.shape != shape:
            raise ValueError("%s must be a Q8Weight of shape %s" % (name, shape))


def moe_expert_ffn_q8(desc, x, expert_offsets, token_indices, slot_w, Wg, Wu, Wd, y_perm, ws,
                      stream=None):
    _q8_check(desc, Wg, Wu, Wd)
    _need(x, (desc.T, desc.d), "x")
    _need(y_perm, (desc.T * (desc.k + desc.S), desc.d), "y_perm")
    g, u, d = Wg.struct(), Wu.struct(), Wd.struct()
    st = lib().moe_expert_ffn_q8(
        ctypes.byref(desc), _p(x, torch.bfloat16, "x"),
        _p(expert_offsets, torch.int32, "expert_offsets"),
        _p(token_indices, torch.int32, "token_indices"), _p(slot_w, torch.float32, "slot_w"),
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), _p(y_perm, torch.bfloat16, "y_perm"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream))
    _check(st, "moe_expert_ffn_q8")


def moe_layer_forward_q8(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, residual, y,
                         topk_ids_out, topk_w_out, ws, stream=None):
    _q8_check(desc, Wg, Wu, Wd)
    _need(x, (desc.T, desc.d), "x")
    _need(Wr, (desc.E, desc.d), "Wr")
    _need(y, (desc.T, desc.d), "y")
    g, u, d = Wg.struct(), Wu.struct(), Wd.struct()
    st = lib().moe_layer_forward_q8(
        ctypes.byref(desc), _p(x, torch.bfloat16, "x"), _p(Wr, torch.bfloat16, "Wr"),
        _p(logit_bias, torch.float32, "logit_bias"), _p(sel_bias, torch.float32, "sel_bias"),
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
        _p(residual, torch.float32, "residual"), _p(y, torch.float32, "y"),
        _p(topk_ids_out, torch.int32, "topk_ids_out"), _p(topk_w_out, torch.float32, "topk_w_out"),
        _p(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream))
    _check(st, "moe_layer_forward_q8")


def moe_get_device_status(ws, clear=False, stream=None) -> int:
    """Synchronizes the stream and returns the workspace's sticky device status."""
    return lib().moe_get_device_status(_p(ws, torch.uint8, "workspace"), ws.numel(),
                                       1 if clear else 0, _stream(stream))


def moe_check_bounded_wait(ws, which, stream=None):
    """Enqueues the bounded-wait self-check (see include/moe.h); afterwards
    moe_get_device_status(ws) reports MOE_ERR_TIMEOUT."""
    _check(lib().moe_check_bounded_wait(_p(ws, torch.uint8, "workspace"), ws.numel(), which,
                                        _stream(stream)), "moe_check_bounded_wait")


def moe_launch_count() -> int:
    return lib().moe_launch_count()


def moe_profile_enable(on):
    """True / 1: record every launch; 2: only launches that state their bytes
    (the expert tier's loads); False / 0: stop."""
    mode = 2 if on == 2 else (1 if on else 0)
    _check(lib().moe_profile_enable(mode), "moe_profile_enable")


def moe_profile_query(kernel: str):
    """(launches, total_ms) recorded for one kernel name since profiling was enabled."""
    n = ctypes.c_int32(0)
    ms = ctypes.c_float(0.0)
    _check(lib().moe_profile_query(kernel.encode(), ctypes.byref(n), ctypes.byref(ms)),
           "moe_profile_query")
    return n.value, ms.value


def moe_profile_list(kernel: str):
    """The named kernel's recorded launches in launch order: (ms list, bytes list)."""
    n = ctypes.c_int32(0)
    _check(lib().moe_profile_list(kernel.encode(), 0, None, None, ctypes.byref(n)),
           "moe_profile_list")
    if n.value == 0:
        return [], []
    ms = (ctypes.c_float * n.value)()
    by = (ctypes.c_uint64 * n.value)()
    _check(lib().moe_profile_list(kernel.encode(), n.value, ctypes.cast(ms, ctypes.c_void_p),
                                  ctypes.cast(by, ctypes.c_void_p), ctypes.byref(n)),
           "moe_profile_list")
    return list(ms), list(by)


# ---------------------------------------------------------------- slot cache and expert tier
class SlotCache:
    """moe_slot_cache: expert residency over n_slots slots (host only)."""

    def __init__(self, n_slots: int, n_experts: int):
        h = ctypes.c_void_p()
        _check(lib().moe_slot_cache_create(n_slots, n_experts, ctypes.byref(h)),
               "moe_slot_cache_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_slot_cache_destroy(self._h)
            self._h = None

    __del__ = close

    def assign(self, experts):
        """(slot, load, pass, n_passes) for one step's distinct experts."""
        import numpy as np
        e = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
        n = e.size
        slot, load, pas = (np.empty(n, np.int32) for _ in range(3))
        npass = ctypes.c_int32(0)
        ptr = lambda a: a.ctypes.data if n else None
        _check(lib().moe_slot_cache_assign(self._h, ptr(e), n, ptr(slot), ptr(load), ptr(pas),
                                           ctypes.byref(npass)), "moe_slot_cache_assign")
        return slot, load, pas, npass.value

    def slot_of(self, expert: int) -> int:
        s = ctypes.c_int32(0)
        _check(lib().moe_slot_cache_slot_of(self._h, expert, ctypes.byref(s)),
               "moe_slot_cache_slot_of")
        return s.value

    def stats(self) -> dict:
        st = TierStats()
        _check(lib().moe_slot_cache_get_stats(self._h, ctypes.byref(st)),
               "moe_slot_cache_get_stats")
        return st.as_dict()


class _HostBlock:
    """Owner of one moe_host_alloc block; frees it when the last view is gone."""

    def __init__(self, nbytes):
        p = ctypes.c_void_p()
        _check(lib().moe_host_alloc(nbytes, ctypes.byref(p)), "moe_host_alloc")
        self.ptr, self.nbytes = p.value, nbytes

    def __del__(self):
        if getattr(self, "ptr", None):
            lib().moe_host_free(ctypes.c_void_p(self.ptr))
            self.ptr = None


def host_empty(shape, dtype=torch.bfloat16) -> torch.Tensor:
    """A CPU tensor in moe_host_alloc memory (page-locked, huge-page backed, zeroed):
    the fast home for an expert tier's projections."""
    import numpy as np
    n = 1
    for v in shape:
        n *= int(v)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    block = _HostBlock(max(nbytes, 1))
    buf = (ctypes.c_uint8 * nbytes).from_address(block.ptr)
    buf._owner = block  # tensor -> numpy array -> this buffer -> the block
    arr = np.frombuffer(buf, dtype=np.uint8)
    return torch.from_numpy(arr).view(dtype).view(*shape)


def _host_p(t, dtype, what):
    """Pointer of a contiguous host (CPU) tensor."""
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError("%s must be a CPU tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    return t.data_ptr()


class ExpertTier:
    """moe_expert_tier: expert projections kept in host memory (Wg/Wu/Wd CPU bf16
    tensors, kept alive here), a bounded pool of expert slots in HBM, and a
    forward() that calls moe_tier_forward.  Wr and the biases are device tensors."""

    def __init__(self, desc: LayerDesc, Wr, Wg_host, Wu_host, Wd_host, hbm_budget_bytes: int,
                 logit_bias=None, sel_bias=None):
        nE = desc.E + desc.S
        for name, W, shape in (("Wg", Wg_host, (nE, desc.I, desc.d)),
                               ("Wu", Wu_host, (nE, desc.I, desc.d)),
                               ("Wd", Wd_host, (nE, desc.d, desc.I))):
            _need(W, shape, name)
        self.desc = desc
        self.host = (Wg_host, Wu_host, Wd_host)
        self.Wr, self.logit_bias, self.sel_bias = Wr, logit_bias, sel_bias
        h = ctypes.c_void_p()
        _check(lib().moe_tier_create(
            ctypes.byref(desc), _host_p(Wg_host, torch.bfloat16, "Wg"),
            _host_p(Wu_host, torch.bfloat16, "Wu"), _host_p(Wd_host, torch.bfloat16, "Wd"),
            int(hbm_budget_bytes), ctypes.byref(h)), "moe_tier_create")
        self._h = h
        self.ws = alloc_workspace(desc, device=Wr.device)

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_tier_destroy(self._h)
            self._h = None

    __del__ = close

    def prefetch(self, experts, stream=None):
        import numpy as np
        e = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
        _check(lib().moe_tier_prefetch(self._h, e.ctypes.data if e.size else None, e.size,
                                       _stream(stream)), "moe_tier_prefetch")

    def forward(self, x, residual=None, y=None, topk_ids=None, topk_w=None, desc=None,
                stream=None):
        d = desc if desc is not None else self.desc
        if d.T > self.desc.T:  # the workspace is sized for the tier's T
            raise ValueError("T %d exceeds the tier's %d" % (d.T, self.desc.T))
        _need(x, (d.T, d.d), "x")
        if y is None:
            y = torch.empty((d.T, d.d), dtype=torch.float32, device=x.device)
        _need(y, (d.T, d.d), "y")
        st = lib().moe_tier_forward(
            self._h, ctypes.byref(d), _p(x, torch.bfloat16, "x"),
            _p(self.Wr, torch.bfloat16, "Wr"), _p(self.logit_bias, torch.float32, "logit_bias"),
            _p(self.sel_bias, torch.float32, "sel_bias"), _p(residual, torch.float32, "residual"),
            _p(y, torch.float32, "y"), _p(topk_ids, torch.int32, "topk_ids_out"),
            _p(topk_w, torch.float32, "topk_w_out"), _p(self.ws, torch.uint8, "workspace"),
            self.ws.numel(), _stream(stream))
        _check(st, "moe_tier_forward")
        return y

    def stats(self) -> dict:
        st = TierStats()
        _check(lib().moe_tier_get_stats(self._h, ctypes.byref(st)), "moe_tier_get_stats")
        return st.as_dict()


# ---------------------------------------------------------------- convenience
class MoeLayer:
    """A layer's weights and workspace on the device, with a forward() that calls
    moe_layer_forward.  Weights are used in place (no copies)."""

    def __init__(self, desc: LayerDesc, Wr, Wg, Wu, Wd, logit_bias=None, sel_bias=None):
        """Wg/Wu/Wd are bf16/fp32 tensors, or Q8Weight (Q8_0 experts, bf16 layers)."""
        self.desc = desc
        self.Wr, self.Wg, self.Wu, self.Wd = Wr, Wg, Wu, Wd
        self.q8 = isinstance(Wg, Q8Weight)
        self.logit_bias, self.sel_bias = logit_bias, sel_bias
        self.ws = alloc_workspace(desc, device=Wr.device)

    def forward(self, x, residual=None, y=None, topk_ids=None, topk_w=None, stream=None):
        d = self.desc
        if y is None:
            y = torch.empty((d.T, d.d), dtype=torch.float32, device=x.device)
        fwd = moe_layer_forward_q8 if self.q8 else moe_layer_forward
        fwd(d, x, self.Wr, self.logit_bias, self.sel_bias, self.Wg, self.Wu, self.Wd, residual, y,
            topk_ids, topk_w, self.ws, stream)
        return y

    def forward_host(self, x_host, y_host, residual=None, stream=None):
        """The layer call with host buffers (moe_layer_forward_host): x_host and
        y_host are CPU tensors (page-locked for asynchronous copies); the library
        copies x in, runs the layer and copies y out, all on the stream."""
        d = self.desc
        _need(x_host, (d.T, d.d), "x_host")
        _need(y_host, (d.T, d.d), "y_host")
        if x_host.is_cuda or y_host.is_cuda:
            raise ValueError("forward_host takes host (CPU) tensors")
        if x_host.dtype != _act_dtype(d) or y_host.dtype != torch.float32:
            raise TypeError("x_host must be %s and y_host float32" % _act_dtype(d))
        if not (x_host.is_contiguous() and y_host.is_contiguous()):
            raise ValueError("forward_host takes contiguous host tensors")
        common = (ctypes.byref(d), ctypes.c_void_p(x_host.data_ptr()),
                  _p(self.Wr, None, "Wr"), _p(self.logit_bias, torch.float32, "logit_bias"),
                  _p(self.sel_bias, torch.float32, "sel_bias"))
        tail = (_p(residual, torch.float32, "residual"), ctypes.c_void_p(y_host.data_ptr()),
                None, None, _p(self.ws, torch.uint8, "workspace"), self.ws.numel(),
                _stream(stream))
        if self.q8:
            g, u, w = self.Wg.struct(), self.Wu.struct(), self.Wd.struct()
            st = lib().moe_layer_forward_q8_host(*common, ctypes.byref(g), ctypes.byref(u),
                                                 ctypes.byref(w), *tail)
            _check(st, "moe_layer_forward_q8_host")
        else:
            st = lib().moe_layer_forward_host(*common, _p(self.Wg, None, "Wg"),
                                              _p(self.Wu, None, "Wu"), _p(self.Wd, None, "Wd"),
                                              *tail)
            _check(st, "moe_layer_forward_host")
        return y_host

    def forward_host_pipelined(self, x_hosts, y_hosts, stream=None):
        """A run of layer calls on host buffers with the copies overlapped
        (moe_layer_forward_host_pipelined): step i reads x_hosts[i] and writes
        y_hosts[i] (CPU tensors, page-locked for asynchronous copies); no
        residual.  The run is ordered on the stream like a single call."""
        d = self.desc
        if len(x_hosts) != len(y_hosts):
            raise ValueError("one output buffer per input buffer")
        for x_host, y_host in zip(x_hosts, y_hosts):
            _need(x_host, (d.T, d.d), "x_host")
            _need(y_host, (d.T, d.d), "y_host")
            if x_host.is_cuda or y_host.is_cuda:
                raise ValueError("forward_host_pipelined takes host (CPU) tensors")
            if x_host.dtype != _act_dtype(d) or y_host.dtype != torch.float32:
                raise TypeError("x_host must be %s and y_host float32" % _act_dtype(d))
            if not (x_host.is_contiguous() and y_host.is_contiguous()):
                raise ValueError("forward_host_pipelined takes contiguous host tensors")
        n = len(x_hosts)
        xs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in x_hosts])
        ys = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in y_hosts])
        head = (ctypes.byref(d), n, ctypes.cast(xs, ctypes.c_void_p), _p(self.Wr, None, "Wr"),
                _p(self.logit_bias, torch.float32, "logit_bias"),
                _p(self.sel_bias, torch.float32, "sel_bias"))
        tail = (ctypes.cast(ys, ctypes.c_void_p), _p(self.ws, torch.uint8, "workspace"),
                self.ws.numel(), _stream(stream))
        if self.q8:
            g, u, w = self.Wg.struct(), self.Wu.struct(), self.Wd.struct()
            st = lib().moe_layer_forward_q8_host_pipelined(*head, ctypes.byref(g),
                                                           ctypes.byref(u), ctypes.byref(w),
                                                           *tail)
            _check(st, "moe_layer_forward_q8_host_pipelined")
        else:
            st = lib().moe_layer_forward_host_pipelined(*head, _p(self.Wg, None, "Wg"),
                                                        _p(self.Wu, None, "Wu"),
                                                        _p(self.Wd, None, "Wd"), *tail)
            _check(st, "moe_layer_forward_host_pipelined")
        return y_hosts
