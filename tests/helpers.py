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


def worst_experts(err_tok, ids, tol, S, E, n=5):
    """Where the output errors sit: the worst tokens with their experts, and the
    experts that every token above the tolerance shares (a bad tile of one
    expert's batch shows up as that expert in all of them)."""
    order = np.argsort(-err_tok)[:n]
    worst = [(int(t), float(err_tok[t]), ids[t].tolist()) for t in order]
    bad = np.nonzero(err_tok > tol)[0]
    common = None
    if len(bad):
        common = set(ids[bad[0]].tolist()) | set(range(E, E + S))
        for t in bad[1:]:
            common &= set(ids[t].tolist()) | set(range(E, E + S))
    return {"worst_tokens": worst, "n_tokens_over": int(len(bad)),
            "experts_shared_by_all_over": sorted(common) if common is not None else None}


def check_all_tokens(y, y_ref, ids_ref, cfg, tol):
    """Every output element of every token against the oracle: max|dy|/max|y|."""
    got = np.asarray(y, np.float64)
    assert got.shape == y_ref.shape and np.isfinite(got).all()
    scale = max(np.abs(y_ref).max(), 1e-300)
    err_tok = np.abs(got - y_ref).max(axis=1) / scale
    err = float(err_tok.max())
    assert err <= tol, (err, worst_experts(err_tok, ids_ref, tol, cfg.S, cfg.E))
    return err


# Output tolerances: fp32 layer 1e-5, bf16 layer 1e-2 (max|dy| / max|y|).
def y_tol(cfg):
    return 1e-5 if cfg.dtype == "f32" else 1e-2


# Gate weights.  The GPU scores in fp32: a router logit is an fp32 sum of d
# products (exact for bf16 operands), and the weights are formed from the
# logits with expf, one division or reciprocal per weight and a sum over the
# normalising set (all E experts for softmax, the k selected for sigmoid with
# norm_topk).  Rule-of-thumb (root-n) error of a d-term fp32 sum:
#     eps_l(t) = (sqrt(d) + 1) * u * s(t),  s(t) = max_e sum_i |x_ti * Wr_ei| (+ |lb|),
# u = 2^-24 (the + 1 covers the rounding of fp32 products).  A logit error
# of eps moves log w_j by at most 2*eps (its own term and the normaliser);
# the argument of expf, l_e - max l, is rounded with an error of at most
# u * 2 s(t); the normaliser's own sum adds at most n_norm * u, and expf,
# the reciprocal and the division a few u more.  So
#     |dw_j| / w_j <= 2 * eps_l(t) + 2 * u * s(t) + (n_norm + 8) * u.
U32 = 2.0 ** -24


def weight_rtol(x, Wr, cfg, logit_bias=None):
    """Per-token relative tolerance of the gate weights, [T] (see above)."""
    xa = np.abs(oracle.widen(host(x)))
    wa = np.abs(oracle.widen(host(Wr)))
    s = (xa @ wa.T).max(axis=1)  # max_e sum_i |x_ti Wr_ei|
    if logit_bias is not None:
        s = s + np.abs(oracle.widen(host(logit_bias))).max()
    n_norm = cfg.E if cfg.gate == 0 else cfg.k
    return (2.0 * (np.sqrt(cfg.d) + 1.0) + 2.0) * U32 * s + (n_norm + 8) * U32


def check_weights(w, w_ref, inp, cfg):
    """Gate weights against the oracle within the derived per-token bound."""
    w = np.asarray(w, np.float64)
    tol = weight_rtol(inp["x"], inp["Wr"], cfg, inp.get("logit_bias"))
    rel = np.abs(w - w_ref) / np.maximum(np.abs(w_ref), 1e-300)
    ratio = rel / tol[:, None]
    assert ratio.max() <= 1.0, ("gate weight error above the derived bound", float(rel.max()),
                                float(ratio.max()))
    return float(rel.max())
