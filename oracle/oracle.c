/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: it is an independent restatement of what the pages
 * define, written so that a reader can check it against them line by line.
 *
 * What is computed, and where it is stated:
 *   - gating, two families (softmax top-k; sigmoid scoring with a per-expert
 *     selection bias and a routed scaling factor), plus the shared expert as
 *     one extra slot of weight 1.0 per token:
 *       "Distributed MoE" (tenzro docs), paragraph on the two router families;
 *       "Expert-Sharded Swarm Inference: The Design" (kvasir), layer pseudocode;
 *   - the dispatch plan (per-expert batches of token_indices, per-token slot
 *     assignments): "Distributed MoE", tenzro_moePlanDispatch request and
 *     response records;
 *   - the expert FFN: SwiGLU over gate/up/down projections, every projection
 *     applied as Y = X * W^T with W stored [out, in]:
 *       "Distributed MoE", expert-host-runtime and compute-seam paragraphs;
 *   - the combine: per-token sum of gate-weighted expert outputs plus the
 *     shared expert: "Distributed MoE", expert-host-runtime paragraph;
 *       "Expert-Sharded Swarm Inference: The Design", layer pseudocode;
 *   - sharded (grouped by expert) == monolithic (per token) up to rounding:
 *       "Expert-Sharded Swarm Inference: The Design", exactness paragraph;
 *       "Expert-sharding" (kvasir wiki), section "Gemeten, niet beloofd".
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - softmax family: no renormalisation of the top-k probabilities unless
 *     norm_topk != 0 (the pseudocode keeps softmax(...) as is);
 *   - sigmoid family: the selection bias only chooses experts; the weights are
 *     the unbiased sigmoid scores, divided by their sum over the selected set
 *     when norm_topk != 0, then multiplied by routed_scaling;
 *   - an optional per-expert logit bias lb[e] is added to the router logit
 *     before either family's scoring (used to make skewed workloads);
 *   - top-k ties go to the lower expert index; a token's routed slots are in
 *     descending selection score; shared slots follow them;
 *   - batches are in ascending expert index, token_indices ascending inside
 *     each batch (the printed example is ascending);
 *   - silu(z) = z / (1 + exp(-z)); SwiGLU h = silu(gate) * up.
 *
 * Numbers: every input is read exactly as stored (fp32 or bf16) and widened to
 * fp64; all arithmetic is fp64.  Parallelism: OpenMP over tokens only; each
 * token's arithmetic is the sequential loop written below.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2

#define OR_GATE_SOFTMAX 0
#define OR_GATE_SIGMOID 1

#define OR_OK 0
#define OR_EINVAL -1
#define OR_ENOMEM -2
#define OR_EMISSING -3

/* widen element i of an fp32 / bf16 / fp64 array to double (exact) */
static double widen(const void* p, int dt, size_t i) {
  if (dt == OR_F32) return (double)((const float*)p)[i];
  if (dt == OR_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16; /* bf16 = top half of fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return ((const double*)p)[i];
}

/* copy n elements starting at element `off` into an fp64 row */
static void widen_row(double* dst, const void* src, int dt, size_t off, int n) {
  for (int i = 0; i < n; ++i) dst[i] = widen(src, dt, off + (size_t)i);
}

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* -------------------------------------------------------------------------
 * Router: logits and selection scores of one token.
 *   logit[e] = x_t . Wr[e] (+ lb[e])          (router weights stored [E, d])
 *   softmax family : selection score = logit (softmax is monotone in it)
 *   sigmoid family : selection score = sigmoid(logit) + sel_bias[e]
 * ------------------------------------------------------------------------- */
static void router_one(int d, int E, int gate, const double* xt, const void* Wr, int w_dt,
                       const double* lb, const double* sb, double* logit, double* score,
                       double* rowbuf) {
  for (int e = 0; e < E; ++e) {
    widen_row(rowbuf, Wr, w_dt, (size_t)e * d, d);
    double l = dot(xt, rowbuf, d);
    if (lb) l += lb[e];
    logit[e] = l;
    if (gate == OR_GATE_SOFTMAX)
      score[e] = l;
    else
      score[e] = sigmoid(l) + (sb ? sb[e] : 0.0);
  }
}

/* k largest selection scores, in descending order; ties to the lower index */
static void topk_desc(const double* score, int E, int k, int32_t* sel, unsigned char* taken) {
  memset(taken, 0, (size_t)E);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || score[e] > score[best]) best = e;
    }
    taken[best] = 1;
    sel[j] = best;
  }
}

/* gate weights of the selected experts */
static void gate_weights(int E, int k, int gate, int norm_topk, double rs, const double* logit,
                         const int32_t* sel, double* w) {
  if (gate == OR_GATE_SOFTMAX) {
    double m = logit[0];
    for (int e = 1; e < E; ++e)
      if (logit[e] > m) m = logit[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp(logit[e] - m);
    for (int j = 0; j < k; ++j) w[j] = exp(logit[sel[j]] - m) / z;
  } else {
    for (int j = 0; j < k; ++j) w[j] = sigmoid(logit[sel[j]]);
  }
  if (norm_topk) {
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += w[j];
    for (int j = 0; j < k; ++j) w[j] = w[j] / s;
  }
  for (int j = 0; j < k; ++j) w[j] = rs * w[j];
}

/* -------------------------------------------------------------------------
 * Expert FFN of one token row:  out = Wd * (silu(Wg * v) (.) (Wu * v))
 * Wg, Wu stored [I, d]; Wd stored [d, I]  (Y = X * W^T, W is [out, in]).
 * ------------------------------------------------------------------------- */
static void ffn_one(int d, int I, const double* v, const void* Wg, const void* Wu, const void* Wd,
                    int w_dt, double* out, double* h, double* rowbuf) {
  for (int n = 0; n < I; ++n) {
    widen_row(rowbuf, Wg, w_dt, (size_t)n * d, d);
    double g = dot(rowbuf, v, d);
    widen_row(rowbuf, Wu, w_dt, (size_t)n * d, d);
    double u = dot(rowbuf, v, d);
    h[n] = silu(g) * u;
  }
  for (int m = 0; m < d; ++m) {
    widen_row(rowbuf, Wd, w_dt, (size_t)m * I, I);
    out[m] = dot(rowbuf, h, I);
  }
}

static int check_common(int T, int d, int E, int k, int S, int gate) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || S < 0) return OR_EINVAL;
  if (gate != OR_GATE_SOFTMAX && gate != OR_GATE_SIGMOID) return OR_EINVAL;
  return OR_OK;
}

static void set_threads(int nthreads) {
  if (nthreads > 0) omp_set_num_threads(nthreads);
}

/* Router logits and selection scores for all T tokens ([T, E] each). */
int oracle_router_scores(int T, int d, int E, int gate, int x_dt, const void* x, int w_dt,
                         const void* Wr, const double* lb, const double* sb, double* logits,
                         double* scores, int nthreads) {
  if (check_common(T, d, E, 1, 0, gate) != OR_OK) return OR_EINVAL;
  if (gate == OR_GATE_SOFTMAX && sb) return OR_EINVAL;
  set_threads(nthreads);
  int err = OR_OK;
#pragma omp parallel
  {
    double* xt = malloc(sizeof(double) * (size_t)d);
    double* rowbuf = malloc(sizeof(double) * (size_t)d);
    if (!xt || !rowbuf) {
#pragma omp atomic write
      err = OR_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int t = 0; t < T; ++t) {
        widen_row(xt, x, x_dt, (size_t)t * d, d);
        router_one(d, E, gate, xt, Wr, w_dt, lb, sb, logits + (size_t)t * E,
                   scores + (size_t)t * E, rowbuf);
      }
    }
    free(xt);
    free(rowbuf);
  }
  return err;
}

/* Routing of T tokens: ids[T, k] (descending score) and gate weights w[T, k]. */
int oracle_route(int T, int d, int E, int k, int gate, int norm_topk, double rs, int x_dt,
                 const void* x, int w_dt, const void* Wr, const double* lb, const double* sb,
                 int32_t* ids, double* w, int nthreads) {
  if (check_common(T, d, E, k, 0, gate) != OR_OK) return OR_EINVAL;
  if (gate == OR_GATE_SOFTMAX && sb) return OR_EINVAL;
  set_threads(nthreads);
  int err = OR_OK;
#pragma omp parallel
  {
    double* xt = malloc(sizeof(double) * (size_t)d);
    double* rowbuf = malloc(sizeof(double) * (size_t)d);
    double* logit = malloc(sizeof(double) * (size_t)E);
    double* score = malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = malloc((size_t)E);
    if (!xt || !rowbuf || !logit || !score || !taken) {
#pragma omp atomic write
      err = OR_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int t = 0; t < T; ++t) {
        widen_row(xt, x, x_dt, (size_t)t * d, d);
        router_one(d, E, gate, xt, Wr, w_dt, lb, sb, logit, score, rowbuf);
        topk_desc(score, E, k, ids + (size_t)t * k, taken);
        gate_weights(E, k, gate, norm_topk, rs, logit, ids + (size_t)t * k, w + (size_t)t * k);
      }
    }
    free(xt);
    free(rowbuf);
    free(logit);
    free(score);
    free(taken);
  }
  return err;
}

/* -------------------------------------------------------------------------
 * Dispatch plan: invert token -> experts into expert -> tokens.
 * The T*(k+S) (token, slot) pairs are visited in token-major order; slot j < k
 * is routed expert ids[t, j], slot k + s is shared expert E + s.  Each pair
 * lands in its expert's batch behind the earlier pairs of that expert, so
 * token_indices are ascending inside each batch (a counting sort).
 *   offsets[E+S+1]         : batch e is token_indices[offsets[e] .. offsets[e+1])
 *   token_indices[T*(k+S)] : token of each batch row
 *   slot_row[T*(k+S)]      : batch row of pair (t, j)  -- the token assignments
 *   active_ids[E+S], n_active : experts with a non-empty batch, ascending
 * ------------------------------------------------------------------------- */
int oracle_plan(int T, int E, int k, int S, const int32_t* ids, int32_t* offsets,
                int32_t* token_indices, int32_t* slot_row, int32_t* active_ids,
                int32_t* n_active) {
  if (T < 0 || E <= 0 || k <= 0 || S < 0) return OR_EINVAL;
  const int nE = E + S, ks = k + S;
  for (size_t i = 0; i < (size_t)T * k; ++i)
    if (ids[i] < 0 || ids[i] >= E) return OR_EINVAL;
  int64_t* count = calloc((size_t)nE, sizeof(int64_t));
  int64_t* fill = calloc((size_t)nE, sizeof(int64_t));
  if (!count || !fill) {
    free(count);
    free(fill);
    return OR_ENOMEM;
  }
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < ks; ++j) {
      int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
      count[e] += 1;
    }
  offsets[0] = 0;
  for (int e = 0; e < nE; ++e) offsets[e + 1] = offsets[e] + (int32_t)count[e];
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < ks; ++j) {
      int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
      int32_t pos = offsets[e] + (int32_t)fill[e];
      fill[e] += 1;
      token_indices[pos] = t;
      slot_row[(size_t)t * ks + j] = pos;
    }
  int na = 0;
  for (int e = 0; e < nE; ++e)
    if (count[e] > 0) active_ids[na++] = e;
  *n_active = na;
  free(count);
  free(fill);
  return OR_OK;
}

/* -------------------------------------------------------------------------
 * Monolithic forward, token by token (the layer pseudocode):
 *   y_t = sum_{j<k} w_tj * FFN(ids_tj, x_t) + sum_{s<S} 1.0 * FFN(E+s, x_t)
 *         (+ residual_t when given)
 * Only the tokens in token_list (n_list of them; all T when token_list is
 * NULL) are computed; row i of y / ids / w belongs to token token_list[i].
 * Expert weights come as per-expert base pointers Wg[e] ([I, d]), Wu[e]
 * ([I, d]), Wd[e] ([d, I]) for e in 0..E+S-1; an expert that no computed
 * token uses may be NULL.
 * ------------------------------------------------------------------------- */
int oracle_forward(int T, int d, int E, int k, int I, int S, int gate, int norm_topk, double rs,
                   int x_dt, const void* x, int w_dt, const void* Wr, const double* lb,
                   const double* sb, const void* const* Wg, const void* const* Wu,
                   const void* const* Wd, const double* residual, int n_list,
                   const int32_t* token_list, double* y, int32_t* ids, double* w, int nthreads) {
  if (check_common(T, d, E, k, S, gate) != OR_OK || I <= 0) return OR_EINVAL;
  if (gate == OR_GATE_SOFTMAX && sb) return OR_EINVAL;
  const int n = token_list ? n_list : T;
  for (int i = 0; i < n && token_list; ++i)
    if (token_list[i] < 0 || token_list[i] >= T) return OR_EINVAL;
  set_threads(nthreads);
  int err = OR_OK;
  const int rowlen = d > I ? d : I;
#pragma omp parallel
  {
    double* xt = malloc(sizeof(double) * (size_t)d);
    double* rowbuf = malloc(sizeof(double) * (size_t)rowlen);
    double* logit = malloc(sizeof(double) * (size_t)E);
    double* score = malloc(sizeof(double) * (size_t)E);
    double* h = malloc(sizeof(double) * (size_t)I);
    double* out = malloc(sizeof(double) * (size_t)d);
    unsigned char* taken = malloc((size_t)E);
    if (!xt || !rowbuf || !logit || !score || !h || !out || !taken) {
#pragma omp atomic write
      err = OR_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < n; ++i) {
        const int t = token_list ? token_list[i] : i;
        int32_t* sel = ids + (size_t)i * k;
        double* wt = w + (size_t)i * k;
        double* yt = y + (size_t)i * d;
        widen_row(xt, x, x_dt, (size_t)t * d, d);
        router_one(d, E, gate, xt, Wr, w_dt, lb, sb, logit, score, rowbuf);
        topk_desc(score, E, k, sel, taken);
        gate_weights(E, k, gate, norm_topk, rs, logit, sel, wt);
        for (int m = 0; m < d; ++m) yt[m] = 0.0;
        for (int j = 0; j < k + S; ++j) {
          const int e = j < k ? sel[j] : E + (j - k);
          const double we = j < k ? wt[j] : 1.0;
          if (!Wg[e] || !Wu[e] || !Wd[e]) {
#pragma omp atomic write
            err = OR_EMISSING;
            continue;
          }
          ffn_one(d, I, xt, Wg[e], Wu[e], Wd[e], w_dt, out, h, rowbuf);
          for (int m = 0; m < d; ++m) yt[m] += we * out[m];
        }
        if (residual)
          for (int m = 0; m < d; ++m) yt[m] += residual[(size_t)t * d + m];
      }
    }
    free(xt);
    free(rowbuf);
    free(logit);
    free(score);
    free(h);
    free(out);
    free(taken);
  }
  return err;
}

/* -------------------------------------------------------------------------
 * Sharded forward: the same layer computed the way the pages' workers do it.
 * Route every token once, build the dispatch plan, then run each expert over
 * its batch of token rows (experts in ascending order) and add each row's
 * gate-weighted output into its token's y.  The pages report that this
 * regrouping equals the monolithic result up to rounding.
 * y is [T, d]; ids / w ([T, k]) receive the routing.
 * ------------------------------------------------------------------------- */
int oracle_forward_sharded(int T, int d, int E, int k, int I, int S, int gate, int norm_topk,
                           double rs, int x_dt, const void* x, int w_dt, const void* Wr,
                           const double* lb, const double* sb, const void* const* Wg,
                           const void* const* Wu, const void* const* Wd, const double* residual,
                           double* y, int32_t* ids, double* w, int nthreads) {
  if (check_common(T, d, E, k, S, gate) != OR_OK || I <= 0) return OR_EINVAL;
  int rc = oracle_route(T, d, E, k, gate, norm_topk, rs, x_dt, x, w_dt, Wr, lb, sb, ids, w,
                        nthreads);
  if (rc != OR_OK) return rc;
  const int nE = E + S, ks = k + S;
  const size_t P = (size_t)T * ks;
  int32_t* offsets = malloc(sizeof(int32_t) * (size_t)(nE + 1));
  int32_t* tok = malloc(sizeof(int32_t) * (P ? P : 1));
  int32_t* slot_row = malloc(sizeof(int32_t) * (P ? P : 1));
  int32_t* active = malloc(sizeof(int32_t) * (size_t)nE);
  double* wrow = malloc(sizeof(double) * (P ? P : 1));
  int32_t na = 0;
  if (!offsets || !tok || !slot_row || !active || !wrow) {
    rc = OR_ENOMEM;
    goto done;
  }
  rc = oracle_plan(T, E, k, S, ids, offsets, tok, slot_row, active, &na);
  if (rc != OR_OK) goto done;
  /* weight of each batch row: routed pair -> its gate weight, shared -> 1.0 */
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < ks; ++j)
      wrow[slot_row[(size_t)t * ks + j]] = j < k ? w[(size_t)t * k + j] : 1.0;
  for (size_t i = 0; i < (size_t)T * d; ++i) y[i] = 0.0;
  set_threads(nthreads);
  const int rowlen = d > I ? d : I;
  for (int e = 0; e < nE && rc == OR_OK; ++e) {
    const int32_t b0 = offsets[e], b1 = offsets[e + 1];
    if (b1 == b0) continue;
    if (!Wg[e] || !Wu[e] || !Wd[e]) {
      rc = OR_EMISSING;
      break;
    }
    /* rows of one batch belong to distinct tokens, so they may run in parallel */
#pragma omp parallel
    {
      double* xt = malloc(sizeof(double) * (size_t)d);
      double* rowbuf = malloc(sizeof(double) * (size_t)rowlen);
      double* h = malloc(sizeof(double) * (size_t)I);
      double* out = malloc(sizeof(double) * (size_t)d);
      if (!xt || !rowbuf || !h || !out) {
#pragma omp atomic write
        rc = OR_ENOMEM;
      } else {
#pragma omp for schedule(dynamic, 1)
        for (int32_t pos = b0; pos < b1; ++pos) {
          const int t = tok[pos];
          widen_row(xt, x, x_dt, (size_t)t * d, d);
          ffn_one(d, I, xt, Wg[e], Wu[e], Wd[e], w_dt, out, h, rowbuf);
          for (int m = 0; m < d; ++m) y[(size_t)t * d + m] += wrow[pos] * out[m];
        }
      }
      free(xt);
      free(rowbuf);
      free(h);
      free(out);
    }
  }
  if (rc == OR_OK && residual)
    for (size_t i = 0; i < (size_t)T * d; ++i) y[i] += residual[i];
done:
  free(offsets);
  free(tok);
  free(slot_row);
  free(active);
  free(wrow);
  return rc;
}

/* -------------------------------------------------------------------------
 * One expert over a list of token rows (what a worker computes for one
 * expert of its slice): out[i] = FFN(e, x[tokens[i]]), [n_rows, d].
 * ------------------------------------------------------------------------- */
int oracle_expert_rows(int d, int I, int x_dt, const void* x, int w_dt, const void* Wg,
                       const void* Wu, const void* Wd, int n_rows, const int32_t* tokens,
                       double* out, int nthreads) {
  if (d <= 0 || I <= 0 || n_rows < 0 || !Wg || !Wu || !Wd) return OR_EINVAL;
  set_threads(nthreads);
  int err = OR_OK;
  const int rowlen = d > I ? d : I;
#pragma omp parallel
  {
    double* xt = malloc(sizeof(double) * (size_t)d);
    double* rowbuf = malloc(sizeof(double) * (size_t)rowlen);
    double* h = malloc(sizeof(double) * (size_t)I);
    if (!xt || !rowbuf || !h) {
#pragma omp atomic write
      err = OR_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < n_rows; ++i) {
        widen_row(xt, x, x_dt, (size_t)tokens[i] * d, d);
        ffn_one(d, I, xt, Wg, Wu, Wd, w_dt, out + (size_t)i * d, h, rowbuf);
      }
    }
    free(xt);
    free(rowbuf);
    free(h);
  }
  return err;
}

/* -------------------------------------------------------------------------
 * Combine: y_t = sum_{j<k} w_tj * rows[slot_row[t, j]]
 *                + sum_{s<S} rows[slot_row[t, k+s]]  (+ residual_t)
 * w NULL means every routed weight is 1 (rows already weighted).
 * ------------------------------------------------------------------------- */
int oracle_combine(int T, int d, int k, int S, const double* rows, const int32_t* slot_row,
                   const double* w, const double* residual, double* y) {
  if (T < 0 || d <= 0 || k <= 0 || S < 0) return OR_EINVAL;
  const int ks = k + S;
  for (int t = 0; t < T; ++t) {
    double* yt = y + (size_t)t * d;
    for (int m = 0; m < d; ++m) yt[m] = 0.0;
    for (int j = 0; j < ks; ++j) {
      const int32_t r = slot_row[(size_t)t * ks + j];
      const double wj = (j < k && w) ? w[(size_t)t * k + j] : 1.0;
      for (int m = 0; m < d; ++m) yt[m] += wj * rows[(size_t)r * d + m];
    }
    if (residual)
      for (int m = 0; m < d; ++m) yt[m] += residual[(size_t)t * d + m];
  }
  return OR_OK;
}

/* -------------------------------------------------------------------------
 * Partial combine ("Distributed MoE", failover paragraph: with allow_partial
 * a forward that cannot cover every (expert, token) pair renormalises the
 * gate weights over the experts that responded and reports the unserved
 * pairs as missing -- a reduced top-k).
 * Reading taken: avail[e] (e < E+S) says whether expert e responded.  For
 * token t, with mass = sum_{j<k} w_tj and resp = sum_{j<k, avail} w_tj, each
 * responding routed slot gets w_tj * mass / resp (the token keeps its routed
 * gate mass; nothing missing => the plain combine); a token none of whose
 * routed experts responded gets no routed term.  A shared expert that did
 * not respond is dropped (weight 0).  missing[t, j] = 1 for every slot whose
 * expert did not respond, else 0.
 * ------------------------------------------------------------------------- */
int oracle_combine_partial(int T, int d, int k, int S, int E, const double* rows,
                           const int32_t* slot_row, const int32_t* ids, const double* w,
                           const int32_t* avail, const double* residual, double* y,
                           int32_t* missing) {
  if (T < 0 || d <= 0 || k <= 0 || S < 0 || E <= 0 || !w || !ids || !avail) return OR_EINVAL;
  const int ks = k + S;
  for (int t = 0; t < T; ++t) {
    double mass = 0.0, resp = 0.0;
    for (int j = 0; j < k; ++j) {
      const double wj = w[(size_t)t * k + j];
      mass += wj;
      if (avail[ids[(size_t)t * k + j]]) resp += wj;
    }
    double* yt = y + (size_t)t * d;
    for (int m = 0; m < d; ++m) yt[m] = 0.0;
    for (int j = 0; j < ks; ++j) {
      const int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
      const int ok = avail[e] != 0;
      if (missing) missing[(size_t)t * ks + j] = ok ? 0 : 1;
      if (!ok) continue;
      const double wj = j < k ? w[(size_t)t * k + j] * (mass / resp) : 1.0;
      const int32_t r = slot_row[(size_t)t * ks + j];
      for (int m = 0; m < d; ++m) yt[m] += wj * rows[(size_t)r * d + m];
    }
    if (residual)
      for (int m = 0; m < d; ++m) yt[m] += residual[(size_t)t * d + m];
  }
  return OR_OK;
}

/* The unserved (expert, token) pairs of a partial combine, as a list
 * ("Distributed MoE", failover paragraph: the pairs that could not be served
 * are reported under `missing`).  Reading taken: token by token, slot by slot
 * (routed slots in the routing's order, then the shared experts E+s), every
 * pair whose expert did not respond is listed as (expert, token).
 * pairs[2 * i], pairs[2 * i + 1] = expert, token of the i-th pair; *n = count. */
int oracle_missing_pairs(int T, int k, int S, int E, const int32_t* ids, const int32_t* avail,
                         int32_t* pairs, int32_t* n) {
  if (T < 0 || k <= 0 || S < 0 || E <= 0 || !n || (T > 0 && (!ids || !avail || !pairs)))
    return OR_EINVAL;
  int32_t count = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k + S; ++j) {
      const int e = j < k ? ids[(size_t)t * k + j] : E + (j - k);
      if (avail[e]) continue;
      pairs[2 * (size_t)count] = e;
      pairs[2 * (size_t)count + 1] = t;
      count += 1;
    }
  *n = count;
  return OR_OK;
}

/* -------------------------------------------------------------------------
 * Q8_0 block quantization ("Distributed MoE", quantization table: 32-element
 * blocks with one f16 scale, about 8.5 bits per weight; the prepare job
 * block-quantizes each expert projection).
 * For every block of 32 consecutive elements along K of a row:
 *   amax = max |w|;  d = amax / 127 (fp32);  id = d != 0 ? 1 / d : 0 (fp32);
 *   q[i] = round-half-away(w[i] * id) (fp32 product);  scale = f16(d) (to nearest even).
 * The block represents scale * q[i].  Codes keep the weight's layout
 * q[m][r][k]; scales are stored transposed per matrix, s[m][k/32][r].
 * (Reading: the codes are decided in fp32 from the unrounded d, and f16(d)
 * is what is stored, as GGUF-style encoders do.)
 * ------------------------------------------------------------------------- */
int oracle_quantize_q8_0(int n_mats, int R, int K, int w_dt, const void* w, int8_t* q,
                         uint16_t* scales) {
  if (n_mats < 0 || R <= 0 || K <= 0 || K % 32) return OR_EINVAL;
  const int nb = K / 32;
  for (int m = 0; m < n_mats; ++m)
    for (int r = 0; r < R; ++r)
      for (int b = 0; b < nb; ++b) {
        const size_t base = ((size_t)m * R + r) * K + (size_t)b * 32;
        float v[32];
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
          v[i] = (float)widen(w, w_dt, base + (size_t)i);
          const float a = fabsf(v[i]);
          if (a > amax) amax = a;
        }
        const float d = amax / 127.0f;
        const float id = d != 0.0f ? 1.0f / d : 0.0f;
        for (int i = 0; i < 32; ++i) {
          const float prod = v[i] * id;
          q[base + (size_t)i] = (int8_t)roundf(prod);
        }
        const _Float16 dh = (_Float16)d;
        uint16_t bits;
        memcpy(&bits, &dh, sizeof bits);
        scales[((size_t)m * nb + b) * R + r] = bits;
      }
  return OR_OK;
}

/* scale * q as fp64 (exact), out[m][r][k] */
int oracle_dequantize_q8_0(int n_mats, int R, int K, const int8_t* q, const uint16_t* scales,
                           double* out) {
  if (n_mats < 0 || R <= 0 || K <= 0 || K % 32) return OR_EINVAL;
  const int nb = K / 32;
  for (int m = 0; m < n_mats; ++m)
    for (int r = 0; r < R; ++r)
      for (int k = 0; k < K; ++k) {
        _Float16 dh;
        const uint16_t bits = scales[((size_t)m * nb + k / 32) * R + r];
        memcpy(&dh, &bits, sizeof dh);
        const size_t i = ((size_t)m * R + r) * K + k;
        out[i] = (double)(float)dh * (double)q[i];
      }
  return OR_OK;
}

/* Widen a whole fp32/bf16 array to fp64 (used by the tests to read stored values). */
void oracle_widen(const void* src, int dt, size_t n, double* dst) {
  for (size_t i = 0; i < n; ++i) dst[i] = widen(src, dt, i);
}

int oracle_max_threads(void) { return omp_get_max_threads(); }

/* -------------------------------------------------------------------------
 * Expert tier: which of a bounded set of device slots serves each expert a
 * step needs, and which experts must be copied in.
 *   "Distributed MoE" (tenzro docs), expert-residency paragraph: experts live
 *     in a byte-bounded tier with least-recently-used eviction above a colder
 *     one, and before a forward is dispatched the experts that its routing
 *     decision selected are read ahead into the tier;
 *   "Module expert_store" (ferrox-core docs), design list: an entry held by a
 *     lease is never evicted, and when what a request needs does not fit, the
 *     request is still served (by a pass-through copy): capacity pressure
 *     costs extra transfers, never a wrong answer or a deadlock.
 * Readings taken: one slot holds one expert's three projections (the byte
 * budget divided by an expert's bytes); the work of a step leases every slot
 * it reads until that work is done; when every slot is leased by the work
 * gathered so far, that work forms a pass that runs first, its leases end,
 * and the remaining experts form the next pass (the pass-through copy, done
 * in slots); the experts already resident are served first (they cost no
 * copy), then the others in request order; an expert that is missing takes
 * an empty slot if there is one (lowest slot number), else the slot whose
 * expert was used least recently among those not leased (lowest slot number
 * on equal recency); recency is the step in which a slot was last used.
 * State (owned by the caller, updated in place): holder[n_slots] (expert in
 * each slot, -1 = empty), last_use[n_slots], clock[1] (steps so far) and
 * counters[4] = hits, misses, evictions, extra passes.
 * Out, per request i: slot[i], load[i] (1 = copied in this step), pass[i];
 * *n_passes = number of passes (0 for an empty request).  A request that
 * names an expert twice or one outside 0..n_experts-1 is refused and leaves
 * the state unchanged.
 * ------------------------------------------------------------------------- */
static int tier_choose_slot(int n_slots, const int32_t* holder, const int64_t* last_use,
                            const unsigned char* leased) {
  for (int s = 0; s < n_slots; ++s)
    if (!leased[s] && holder[s] < 0) return s; /* an empty slot */
  int victim = -1;
  for (int s = 0; s < n_slots; ++s) {
    if (leased[s]) continue;
    if (victim < 0 || last_use[s] < last_use[victim]) victim = s; /* least recently used */
  }
  return victim; /* -1: every slot is leased */
}

int oracle_tier_step(int n_slots, int n_experts, int32_t* holder, int64_t* last_use,
                     int64_t* clock, int64_t* counters, const int32_t* req, int n,
                     int32_t* slot, int32_t* load, int32_t* pass, int32_t* n_passes) {
  if (n_slots <= 0 || n_experts <= 0 || n < 0 || !holder || !last_use || !clock || !counters ||
      !n_passes)
    return OR_EINVAL;
  for (int i = 0; i < n; ++i) {
    if (req[i] < 0 || req[i] >= n_experts) return OR_EINVAL;
    for (int j = 0; j < i; ++j)
      if (req[j] == req[i]) return OR_EINVAL;
  }
  unsigned char* leased = calloc((size_t)n_slots, 1);
  unsigned char* served = calloc((size_t)(n ? n : 1), 1);
  if (!leased || !served) {
    free(leased);
    free(served);
    return OR_ENOMEM;
  }
  *clock += 1;
  /* the experts already resident: no copy, leased for the first pass */
  for (int i = 0; i < n; ++i)
    for (int s = 0; s < n_slots; ++s)
      if (holder[s] == req[i]) {
        slot[i] = s;
        load[i] = 0;
        pass[i] = 0;
        leased[s] = 1;
        last_use[s] = *clock;
        served[i] = 1;
        counters[0] += 1;
      }
  /* the others, in request order, each copied into a slot */
  int p = 0;
  for (int i = 0; i < n; ++i) {
    if (served[i]) continue;
    int s = tier_choose_slot(n_slots, holder, last_use, leased);
    if (s < 0) { /* everything leased: the pass so far runs, its leases end */
      p += 1;
      counters[3] += 1;
      memset(leased, 0, (size_t)n_slots);
      s = tier_choose_slot(n_slots, holder, last_use, leased);
    }
    if (holder[s] >= 0) counters[2] += 1;
    holder[s] = req[i];
    last_use[s] = *clock;
    leased[s] = 1;
    slot[i] = s;
    load[i] = 1;
    pass[i] = p;
    counters[1] += 1;
  }
  *n_passes = n > 0 ? p + 1 : 0;
  free(leased);
  free(served);
  return OR_OK;
}
