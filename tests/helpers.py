"""Shared test utilities: margin-enforced inputs and error metrics.

Margins: routing must match the oracle bit-exactly, so inputs are redrawn
until every token's top-(k+1) selection scores (computed by the fp64 oracle)
are separated by at least 1e-3.  fp32 router arithmetic is many orders of
magnitude more accurate than that, so no decision is a near-tie.
"""
import numpy as np
import torch

import oracle
from expert_dispatch_gb300.inputs import LayerConfig, make_inputs, redraw_rows

MARGIN = 1e-3


def host(t):
    return None if t is None else t.detach().cpu()


def bad_margin_rows(x, Wr, cfg, logit_bias, sel_bias, rows=None):
    xs = x if rows is None else x[torch.as_tensor(rows, dtype=torch.long, device=x.device)]
    _, scores = oracle.router_scores(host(xs), host(Wr), cfg.gate, logit_bias=host(logit_bias),
                                     sel_bias=host(sel_bias))
    n = min(cfg.k + 1, cfg.E)
    top = -np.sort(-scores, axis=1)[:, :n]
    gaps = top[:, :-1] - top[:, 1:]
    bad = np.nonzero(gaps.min(axis=1) < MARGIN)[0] if n > 1 else np.zeros(0, np.int64)
    if rows is not None:
        bad = np.asarray(rows)[bad]
    return bad


def enforce_margins(inp, cfg, seed, max_rounds=40):
    """Redraw x rows (in place) until all top-(k+1) score gaps are >= MARGIN."""
    x = inp["x"]
    bad = bad_margin_rows(x, inp["Wr"], cfg, inp["logit_bias"], inp["sel_bias"])
    for rnd in range(max_rounds):
        if len(bad) == 0:
            return inp
        redraw_rows(x, bad, seed, rnd)
        bad = bad_margin_rows(x, inp["Wr"], cfg, inp["logit_bias"], inp["sel_bias"], rows=bad)
    raise RuntimeError("could not enforce routing margins")


def make_case(cfg: LayerConfig, seed=0, device="cpu"):
    inp = make_inputs(cfg, seed=seed, device=device)
    return enforce_margins(inp, cfg, seed)


def rel_err(y, ref):
    """max |y - ref| / max |ref| -- the layer's tolerance metric."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-300))


# Output tolerances: fp32 layer 1e-5, bf16 layer 1e-2 (max|dy| / max|y|).
def y_tol(cfg):
    return 1e-5 if cfg.dtype == "f32" else 1e-2


# Gate weights: fp32 accumulation of a d-term router dot product; the
# probabilistic error bound sqrt(d) * 2^-24 * sum|x_i w_i| is ~1e-5 .. 1e-4
# relative for these shapes, far above the typical 1e-6.
W_RTOL = 1e-4
