"""fp64 CPU oracle of the MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches them: the two share
no code.  The arithmetic lives in ``oracle.c`` (plain loops, fp64); this module
only marshals arrays into it with ``ctypes``.

Functions (each follows the passage cited in ``oracle.c``):
  router_scores  logits and selection scores, [T, E] fp64
  route          top-k expert ids [T, k] and gate weights [T, k] fp64
  plan           dispatch plan (CSR batches per expert + per-token slots)
  forward        monolithic per-token layer forward, optionally on a sample
  forward_sharded  the same layer grouped by expert (the workers' regrouping)
  expert_rows    one expert's SwiGLU FFN over a list of token rows
  combine        gate-weighted sum of batch rows per token plus shared rows
  combine_partial  the combine with unavailable experts (allow_partial)
  missing_pairs  the unserved (expert, token) pairs of a partial combine
  quantize_q8_0 / dequantize_q8_0  Q8_0 blocks of the expert projections
  TierOracle     the expert tier's slot assignment, step by step
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

GATE_SOFTMAX = 0
GATE_SIGMOID = 1

F32, BF16, F64 = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_router_scores.argtypes = [i32, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, i32]
    lib.oracle_route.argtypes = [i32, i32, i32, i32, i32, i32, f64, i32, vp, i32, vp, vp, vp,
                                 vp, vp, i32]
    lib.oracle_plan.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_forward.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, f64, i32, vp, i32, vp,
                                   vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, i32]
    lib.oracle_forward_sharded.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, f64, i32, vp,
                                           i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32]
    lib.oracle_widen.argtypes = [vp, i32, ctypes.c_size_t, vp]
    lib.oracle_expert_rows.argtypes = [i32, i32, i32, vp, i32, vp, vp, vp, i32, vp, vp, i32]
    lib.oracle_combine.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.oracle_combine_partial.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                           vp]
    lib.oracle_combine_partial.restype = ctypes.c_int
    lib.oracle_quantize_q8_0.argtypes = [i32, i32, i32, i32, vp, vp, vp]
    lib.oracle_quantize_q8_0.restype = ctypes.c_int
    lib.oracle_dequantize_q8_0.argtypes = [i32, i32, i32, vp, vp, vp]
    lib.oracle_dequantize_q8_0.restype = ctypes.c_int
    lib.oracle_missing_pairs.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
    lib.oracle_missing_pairs.restype = ctypes.c_int
    lib.oracle_tier_step.argtypes = [i32, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.oracle_tier_step.restype = ctypes.c_int
    for f in ("oracle_router_scores", "oracle_route", "oracle_plan", "oracle_forward",
              "oracle_forward_sharded", "oracle_max_threads", "oracle_expert_rows",
              "oracle_combine"):
        getattr(lib, f).restype = ctypes.c_int
    lib.oracle_widen.restype = None
    _lib = lib
    return lib


def max_threads() -> int:
    return _load().oracle_max_threads()


# --------------------------------------------------------------------------
# array marshalling: torch CPU tensors (fp32 / bf16) or numpy (fp32 / fp64)
# --------------------------------------------------------------------------
class _Arr:
    """Keeps a contiguous host buffer alive and reports its pointer and dtype code."""

    def __init__(self, a):
        self.keep = a
        try:
            import torch
        except ImportError:  # pragma: no cover
            torch = None
        if torch is not None and isinstance(a, torch.Tensor):
            if a.device.type != "cpu":
                raise ValueError("oracle inputs must be host tensors")
            a = a.contiguous()
            self.keep = a
            codes = {torch.float32: F32, torch.bfloat16: BF16, torch.float64: F64}
            if a.dtype not in codes:
                raise TypeError("unsupported dtype %s" % a.dtype)
            self.dt = codes[a.dtype]
            self.ptr = a.data_ptr()
            self.shape = tuple(a.shape)
            self.elsize = a.element_size()
        else:
            a = np.ascontiguousarray(a)
            if a.dtype == np.float32:
                self.dt = F32
            elif a.dtype == np.float64:
                self.dt = F64
            else:
                raise TypeError("unsupported dtype %s" % a.dtype)
            self.keep = a
            self.ptr = a.ctypes.data
            self.shape = a.shape
            self.elsize = a.itemsize


def _f64(a):
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed with code %d" % (what, rc))


def _expert_ptrs(W, n_experts):
    """Per-expert base pointers from a [E+S, r, c] tensor or a list (None allowed)."""
    keep = []
    ptrs = (ctypes.c_void_p * n_experts)()
    dt = None
    if isinstance(W, (list, tuple)):
        if len(W) != n_experts:
            raise ValueError("expected %d expert tensors" % n_experts)
        for e, w in enumerate(W):
            if w is None:
                ptrs[e] = None
                continue
            a = _Arr(w)
            keep.append(a)
            ptrs[e] = a.ptr
            dt = a.dt if dt is None else dt
            if a.dt != dt:
                raise TypeError("mixed expert dtypes")
    else:
        a = _Arr(W)
        keep.append(a)
        if a.shape[0] != n_experts:
            raise ValueError("weight tensor has %d experts, expected %d" % (a.shape[0], n_experts))
        per = int(np.prod(a.shape[1:])) * a.elsize
        for e in range(n_experts):
            ptrs[e] = a.ptr + e * per
        dt = a.dt
    return ptrs, dt, keep


def router_scores(x, Wr, gate, logit_bias=None, sel_bias=None, nthreads=0):
    """Router logits [T, E] and selection scores [T, E], fp64."""
    lib = _load()
    xa, wa = _Arr(x), _Arr(Wr)
    T, d = xa.shape
    E = wa.shape[0]
    lb, sb = _f64(logit_bias), _f64(sel_bias)
    logits = np.empty((T, E), np.float64)
    scores = np.empty((T, E), np.float64)
    rc = lib.oracle_router_scores(T, d, E, gate, xa.dt, xa.ptr, wa.dt, wa.ptr, _ptr(lb), _ptr(sb),
                                  logits.ctypes.data, scores.ctypes.data, nthreads)
    _check(rc, "oracle_router_scores")
    return logits, scores


def route(x, Wr, k, gate, norm_topk=0, routed_scaling=1.0, logit_bias=None, sel_bias=None,
          nthreads=0):
    """Top-k ids [T, k] int32 (descending score) and gate weights [T, k] fp64."""
    lib = _load()
    xa, wa = _Arr(x), _Arr(Wr)
    T, d = xa.shape
    E = wa.shape[0]
    lb, sb = _f64(logit_bias), _f64(sel_bias)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = lib.oracle_route(T, d, E, k, gate, int(norm_topk), float(routed_scaling), xa.dt, xa.ptr,
                          wa.dt, wa.ptr, _ptr(lb), _ptr(sb), ids.ctypes.data, w.ctypes.data,
                          nthreads)
    _check(rc, "oracle_route")
    return ids, w


def plan(ids, E, S=0):
    """Dispatch plan of a routing ids[T, k]; returns a dict of int32 arrays."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    P = T * (k + S)
    offsets = np.empty(E + S + 1, np.int32)
    tok = np.empty(max(P, 1), np.int32)
    slot_row = np.empty(max(P, 1), np.int32)
    active = np.empty(E + S, np.int32)
    n_active = np.zeros(1, np.int32)
    rc = lib.oracle_plan(T, E, k, S, ids.ctypes.data, offsets.ctypes.data, tok.ctypes.data,
                         slot_row.ctypes.data, active.ctypes.data, n_active.ctypes.data)
    _check(rc, "oracle_plan")
    na = int(n_active[0])
    return {"expert_offsets": offsets, "token_indices": tok[:P],
            "slot_row": slot_row[:P].reshape(T, k + S), "active_ids": active[:na].copy(),
            "n_active": na}


def forward(x, Wr, Wg, Wu, Wd, k, gate, S=0, norm_topk=0, routed_scaling=1.0, logit_bias=None,
            sel_bias=None, residual=None, tokens=None, nthreads=0):
    """Monolithic per-token forward.  Returns (y [n, d], ids [n, k], w [n, k]) in fp64.

    ``tokens`` selects a sample of token indices (all tokens when None).  Wg/Wu
    /Wd are [E+S, I, d] / [E+S, I, d] / [E+S, d, I] host tensors, or lists of
    per-expert tensors in which experts that no sampled token uses may be None.
    """
    lib = _load()
    xa, wra = _Arr(x), _Arr(Wr)
    T, d = xa.shape
    E = wra.shape[0]
    gp, gdt, k1 = _expert_ptrs(Wg, E + S)
    up, udt, k2 = _expert_ptrs(Wu, E + S)
    dp, ddt, k3 = _expert_ptrs(Wd, E + S)
    if not (gdt == udt == ddt == wra.dt):
        raise TypeError("router and expert weights must share one dtype")
    I = _infer_I(Wg)
    lb, sb, res = _f64(logit_bias), _f64(sel_bias), _f64(residual)
    if tokens is None:
        n = T
        tl = None
    else:
        tl = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tl.shape[0]
    y = np.empty((n, d), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    rc = lib.oracle_forward(T, d, E, k, I, S, gate, int(norm_topk), float(routed_scaling), xa.dt,
                            xa.ptr, wra.dt, wra.ptr, _ptr(lb), _ptr(sb), gp, up, dp, _ptr(res), n,
                            _ptr(tl), y.ctypes.data, ids.ctypes.data, w.ctypes.data, nthreads)
    del k1, k2, k3
    _check(rc, "oracle_forward")
    return y, ids, w


def forward_sharded(x, Wr, Wg, Wu, Wd, k, gate, S=0, norm_topk=0, routed_scaling=1.0,
                    logit_bias=None, sel_bias=None, residual=None, nthreads=0):
    """Grouped-by-expert forward of all T tokens.  Returns (y [T, d], ids, w)."""
    lib = _load()
    xa, wra = _Arr(x), _Arr(Wr)
    T, d = xa.shape
    E = wra.shape[0]
    gp, gdt, k1 = _expert_ptrs(Wg, E + S)
    up, udt, k2 = _expert_ptrs(Wu, E + S)
    dp, ddt, k3 = _expert_ptrs(Wd, E + S)
    if not (gdt == udt == ddt == wra.dt):
        raise TypeError("router and expert weights must share one dtype")
    I = _infer_I(Wg)
    lb, sb, res = _f64(logit_bias), _f64(sel_bias), _f64(residual)
    y = np.empty((T, d), np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    rc = lib.oracle_forward_sharded(T, d, E, k, I, S, gate, int(norm_topk), float(routed_scaling),
                                    xa.dt, xa.ptr, wra.dt, wra.ptr, _ptr(lb), _ptr(sb), gp, up, dp,
                                    _ptr(res), y.ctypes.data, ids.ctypes.data, w.ctypes.data,
                                    nthreads)
    del k1, k2, k3
    _check(rc, "oracle_forward_sharded")
    return y, ids, w


def expert_rows(x, Wg_e, Wu_e, Wd_e, tokens, nthreads=0):
    """FFN of one expert (weights [I, d], [I, d], [d, I]) on rows x[tokens]; [n, d] fp64."""
    lib = _load()
    xa, ga, ua, da = _Arr(x), _Arr(Wg_e), _Arr(Wu_e), _Arr(Wd_e)
    if not (ga.dt == ua.dt == da.dt):
        raise TypeError("expert weights must share one dtype")
    d = xa.shape[1]
    I = ga.shape[0]
    tl = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty((tl.shape[0], d), np.float64)
    rc = lib.oracle_expert_rows(d, I, xa.dt, xa.ptr, ga.dt, ga.ptr, ua.ptr, da.ptr, tl.shape[0],
                                tl.ctypes.data, out.ctypes.data, nthreads)
    _check(rc, "oracle_expert_rows")
    return out


def combine(rows, slot_row, k, S, w=None, residual=None):
    """y[t] = sum_j w[t, j] rows[slot_row[t, j]] + shared rows (+ residual), fp64."""
    lib = _load()
    rows = _f64(rows)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    T = sr.shape[0]
    d = rows.shape[1]
    wv, res = _f64(w), _f64(residual)
    y = np.empty((T, d), np.float64)
    rc = lib.oracle_combine(T, d, k, S, rows.ctypes.data, sr.ctypes.data, _ptr(wv), _ptr(res),
                            y.ctypes.data)
    _check(rc, "oracle_combine")
    return y


def combine_partial(rows, slot_row, ids, w, avail, k, S, E, residual=None):
    """Combine with unavailable experts: (y [T, d] fp64, missing [T, k+S] int32).

    avail[e] (e < E+S) is nonzero for experts that responded; responding routed
    slots keep the token's routed gate mass (w * mass / resp), unavailable slots
    and shared experts drop out and are reported in `missing`."""
    lib = _load()
    rows = _f64(rows)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    idv = np.ascontiguousarray(ids, dtype=np.int32)
    wv = _f64(w)
    av = np.ascontiguousarray(avail, dtype=np.int32)
    res = _f64(residual)
    T = sr.shape[0]
    d = rows.shape[1]
    y = np.empty((T, d), np.float64)
    missing = np.empty((T, k + S), np.int32)
    rc = lib.oracle_combine_partial(T, d, k, S, E, rows.ctypes.data, sr.ctypes.data,
                                    idv.ctypes.data, wv.ctypes.data, av.ctypes.data, _ptr(res),
                                    y.ctypes.data, missing.ctypes.data)
    _check(rc, "oracle_combine_partial")
    return y, missing


def missing_pairs(ids, avail, k, S, E):
    """(expert, token) of every slot whose expert did not respond, [n, 2] int32,
    ordered by token, then slot."""
    lib = _load()
    idv = np.ascontiguousarray(ids, dtype=np.int32)
    av = np.ascontiguousarray(avail, dtype=np.int32)
    T = idv.shape[0]
    pairs = np.empty((max(T * (k + S), 1), 2), np.int32)
    n = np.zeros(1, np.int32)
    _check(lib.oracle_missing_pairs(T, k, S, E, idv.ctypes.data, av.ctypes.data,
                                    pairs.ctypes.data, n.ctypes.data), "oracle_missing_pairs")
    return pairs[:int(n[0])].copy()


def quantize_q8_0(w):
    """Q8_0 codes and scales of w [n_mats, R, K] (fp32 or bf16 host tensor):
    (q int8 [n_mats, R, K], scales uint16 (f16 bits) [n_mats, K/32, R])."""
    lib = _load()
    wa = _Arr(w)
    n, R, K = wa.shape
    q = np.empty((n, R, K), np.int8)
    s = np.empty((n, K // 32, R), np.uint16)
    _check(lib.oracle_quantize_q8_0(n, R, K, wa.dt, wa.ptr, q.ctypes.data, s.ctypes.data),
           "oracle_quantize_q8_0")
    return q, s


def dequantize_q8_0(q, scales):
    """scale * q in fp64, [n_mats, R, K] (exact)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    n, R, K = q.shape
    out = np.empty((n, R, K), np.float64)
    _check(lib.oracle_dequantize_q8_0(n, R, K, q.ctypes.data, s.ctypes.data, out.ctypes.data),
           "oracle_dequantize_q8_0")
    return out


class TierOracle:
    """The expert tier's residency rules (oracle_tier_step in oracle.c): a
    bounded set of slots, least-recently-used eviction, leased slots never
    evicted, extra passes when a step's experts do not fit."""

    def __init__(self, n_slots, n_experts):
        self.n_slots, self.n_experts = int(n_slots), int(n_experts)
        self.holder = np.full(self.n_slots, -1, np.int32)
        self.last_use = np.zeros(self.n_slots, np.int64)
        self.clock = np.zeros(1, np.int64)
        self.counters = np.zeros(4, np.int64)  # hits, misses, evictions, extra passes

    def step(self, experts):
        """(slot, load, pass, n_passes) of one step's requested experts."""
        lib = _load()
        req = np.ascontiguousarray(experts, dtype=np.int32)
        n = int(req.shape[0])
        slot = np.full(max(n, 1), -1, np.int32)
        load = np.zeros(max(n, 1), np.int32)
        pas = np.full(max(n, 1), -1, np.int32)
        npass = np.zeros(1, np.int32)
        rc = lib.oracle_tier_step(self.n_slots, self.n_experts, self.holder.ctypes.data,
                                  self.last_use.ctypes.data, self.clock.ctypes.data,
                                  self.counters.ctypes.data, req.ctypes.data, n,
                                  slot.ctypes.data, load.ctypes.data, pas.ctypes.data,
                                  npass.ctypes.data)
        _check(rc, "oracle_tier_step")
        return slot[:n], load[:n], pas[:n], int(npass[0])

    def slot_of(self, expert):
        hit = np.nonzero(self.holder == expert)[0]
        return int(hit[0]) if len(hit) else -1

    def stats(self):
        h, m, ev, ex = (int(v) for v in self.counters)
        return {"steps": int(self.clock[0]), "hits": h, "misses": m, "evictions": ev,
                "extra_passes": ex, "resident": int((self.holder >= 0).sum())}


def widen(a):
    """Stored fp32/bf16 values as fp64, decoded by the oracle's own bf16 reader."""
    lib = _load()
    aa = _Arr(a)
    n = int(np.prod(aa.shape))
    out = np.empty(n, np.float64)
    lib.oracle_widen(aa.ptr, aa.dt, n, out.ctypes.data)
    return out.reshape(aa.shape)


def _infer_I(Wg):
    if isinstance(Wg, (list, tuple)):
        for w in Wg:
            if w is not None:
                return int(w.shape[0])
        raise ValueError("no expert weights given")
    return int(Wg.shape[1])
