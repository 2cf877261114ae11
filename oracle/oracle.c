/*
 * oracle.c -- plain, slow float64 CPU oracle for draft-token verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Sources restated here (cited by page title and section):
 *   [EIN]  Edge Inference Notes, post on speculative decoding and EAGLE-3,
 *          sections "The core idea: draft, then check", "Why it changes
 *          nothing about the output" and "One decode round, end to end".
 *   [TGTG] "Towards Green Text Generation: Memory-Based Speculative
 *          Decoding", section 2.4 "Verifier and Acceptance", section 5.1
 *          "The Verifier Cost Model" (equation 1).
 *   [SDSC] "Speculative Decoding Speedup Calculator", steps 1-3.
 *
 * Every step is written the plain way: a full stable sort to rank tokens,
 * sequential sums in float64, a left-to-right scan.  No blocking, no fusion.
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of the repository):
 *   - temperature first, then top-k, then top-p on the renormalised top-k
 *     distribution, applied identically to the target and draft rows;
 *   - ties are ranked by (value descending, index ascending); top-k keeps
 *     exactly top_k tokens; top-p keeps a token iff the mass ranked strictly
 *     before it is below top_p (so the first token is always kept);
 *   - the accept test is  u * q(x) < p(x)  with u in [0, 1);
 *   - the inverse CDF picks the smallest index j whose running sum (in
 *     ascending index order) exceeds u * S;
 *   - a residual of total mass 0 after a rejection (reachable only through
 *     rounding) is replaced by the target row itself;
 *   - token trees (sampling): the children of a node are tried in ascending
 *     node order, each rejected child replaces the residual r by
 *     max(0, r - q) renormalised (q unchanged), the next child is tested
 *     against it, and the node where the walk stops draws from its current
 *     residual; temperature only (scalar or per tree), no top-k / top-p.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Per-sequence flags written by oracle_verify_sample. */
#define OFLAG_ACCEPT_BOUNDARY 1u  /* an accept test had |u - p/q| < 1e-6     */
#define OFLAG_DRAW_BOUNDARY 2u    /* the draw had u*S within 1e-6*S of an edge */
#define OFLAG_DEGENERATE 4u       /* residual mass was exactly zero           */
#define OFLAG_CUT_BOUNDARY 8u     /* a consulted row's top-p cut is within 1e-6
                                     and the other decision changes the outcome */
#define OFLAG_BAD_TOKEN 16u       /* a draft token outside [0, V)             */
#define OFLAG_BAD_ROW 32u         /* a row with NaN/+inf or no finite entry   */
#define OFLAG_BAD_PARENT 64u      /* tree: parents[0] != -1 or a parent outside [0, j) */
#define OFLAG_DEPTH 128u          /* tree: the walk stopped at depth max_depth on a
                                     node that has children                    */

#define BOUNDARY_EPS 1e-6

/* bf16 stores the upper 16 bits of an IEEE float32; widening is exact. */
static double read_logit(const void* base, int dtype, size_t i) {
  if (dtype == ORACLE_BF16) {
    uint16_t h = ((const uint16_t*)base)[i];
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

typedef struct {
  double z;
  int idx;
} ranked_t;

/* Rank order: larger value first, lower index first among equal values. */
static int rank_cmp(const void* a, const void* b) {
  const ranked_t* x = (const ranked_t*)a;
  const ranked_t* y = (const ranked_t*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/*
 * One row of the target or the draft turned into the distribution the accept
 * test uses ([EIN] "Why it changes nothing about the output": temperature,
 * top-k or nucleus adjust both distributions before the test).
 *
 *   z_t  = l_t / T
 *   rank every token by (z desc, index asc)
 *   top-k: keep rank < top_k                      (top_k <= 0: keep all)
 *   top-p: over the top-k set, p'_t = exp(z_t - m) / Z_k; walk in rank order
 *          and keep t iff the mass ranked before t is < top_p (top_p >= 1: off)
 *   p_t  = exp(z_t - m) / sum over kept of exp(z - m)  on kept, else 0
 *
 * `adjust` is 0 for the rule above.  For the boundary check only, -1 keeps one
 * token fewer and +1 one token more than the top-p rule (the neighbouring
 * decision at the cut).
 * probs[V] receives p.  *cut_margin receives the distance |before - top_p| of
 * the last kept and the first dropped token (the smaller one); +inf when no
 * top-p cut was made.  *cut_lo / *cut_hi receive those two token ids (-1 if
 * none); *near_lo / *near_hi tell whether each is within BOUNDARY_EPS.
 * Returns 0, or -1 for a row with NaN, +inf or no finite entry.
 */
static int row_probs_adj(const void* row, int dtype, int V, double temperature, int top_k,
                         double top_p, int adjust, double* probs, double* cut_margin,
                         int* cut_lo, int* cut_hi, int* near_lo, int* near_hi) {
  ranked_t* r = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)V);
  char* kept = (char*)calloc((size_t)V, 1);
  int t, n_topk, rc = 0;
  double m, zk, zkept, before;
  if (cut_margin) *cut_margin = INFINITY;
  if (cut_lo) *cut_lo = -1;
  if (cut_hi) *cut_hi = -1;
  if (near_lo) *near_lo = 0;
  if (near_hi) *near_hi = 0;
  for (t = 0; t < V; ++t) {
    double l = read_logit(row, dtype, (size_t)t);
    if (isnan(l) || (isinf(l) && l > 0)) rc = -1;
    r[t].z = l / temperature;
    r[t].idx = t;
  }
  if (rc == 0) {
    qsort(r, (size_t)V, sizeof(ranked_t), rank_cmp);
    m = r[0].z;
    if (isinf(m)) rc = -1; /* every entry is -inf */
  }
  if (rc != 0) {
    for (t = 0; t < V; ++t) probs[t] = 0.0;
    free(r);
    free(kept);
    return -1;
  }
  n_topk = (top_k > 0 && top_k < V) ? top_k : V;
  zk = 0.0;
  for (t = 0; t < n_topk; ++t) zk += exp(r[t].z - m);
  if (top_p < 1.0) {
    int last_kept = 0, n_keep;
    before = 0.0;
    for (t = 0; t < n_topk; ++t) {
      if (!(before < top_p)) break;
      last_kept = t;
      before += exp(r[t].z - m) / zk;
    }
    {
      /* margins of the last kept and the first dropped token */
      double b_last = 0.0, margin;
      int s;
      for (s = 0; s < last_kept; ++s) b_last += exp(r[s].z - m) / zk;
      margin = fabs(top_p - b_last);
      if (cut_lo) *cut_lo = r[last_kept].idx;
      if (near_lo) *near_lo = last_kept > 0 && margin < BOUNDARY_EPS;
      if (last_kept + 1 < n_topk) {
        double b_next = b_last + exp(r[last_kept].z - m) / zk;
        if (near_hi) *near_hi = fabs(b_next - top_p) < BOUNDARY_EPS;
        if (fabs(b_next - top_p) < margin) margin = fabs(b_next - top_p);
        if (cut_hi) *cut_hi = r[last_kept + 1].idx;
      }
      if (cut_margin) *cut_margin = margin;
    }
    n_keep = last_kept + 1 + adjust;
    if (n_keep < 1) n_keep = 1;
    if (n_keep > n_topk) n_keep = n_topk;
    for (t = 0; t < n_keep; ++t) kept[r[t].idx] = 1;
  } else {
    for (t = 0; t < n_topk; ++t) kept[r[t].idx] = 1;
  }
  zkept = 0.0;
  for (t = 0; t < V; ++t)
    if (kept[t]) zkept += exp(read_logit(row, dtype, (size_t)t) / temperature - m);
  for (t = 0; t < V; ++t)
    probs[t] = kept[t] ? exp(read_logit(row, dtype, (size_t)t) / temperature - m) / zkept : 0.0;
  free(r);
  free(kept);
  return 0;
}

int oracle_row_probs(const void* row, int dtype, int V, double temperature,
                     int top_k, double top_p, double* probs, double* cut_margin,
                     int* cut_lo, int* cut_hi) {
  return row_probs_adj(row, dtype, V, temperature, top_k, top_p, 0, probs, cut_margin, cut_lo,
                       cut_hi, NULL, NULL);
}

/*
 * Inverse CDF in ascending index order: the smallest j with
 * sum_{t<=j} w_t > u * S, S = sum_t w_t.  *margin receives the distance of
 * u*S to the nearer edge of j's interval, divided by S.
 */
static int inverse_cdf(const double* w, int V, double u, double* margin) {
  double s = 0.0, target, c = 0.0;
  int t, last_pos = -1;
  for (t = 0; t < V; ++t) s += w[t];
  target = u * s;
  for (t = 0; t < V; ++t) {
    double prev = c;
    if (w[t] > 0.0) last_pos = t;
    c += w[t];
    if (c > target) {
      double a = fabs(target - prev), b = fabs(c - target);
      if (margin) *margin = (a < b ? a : b) / s;
      return t;
    }
  }
  if (margin) *margin = 0.0; /* unreachable for u < 1 and S > 0 */
  return last_pos;
}

/* The rows of one sequence, turned into distributions on first use. */
typedef struct {
  const void* target; /* this sequence's [k+1][V] */
  const void* draft;  /* this sequence's [k][V]   */
  int dtype, k, V, top_k;
  double T, top_p;
  double* probs[2 * 32 + 1]; /* row id: target i -> i, draft i -> k+1+i */
  int ok[2 * 32 + 1];
  double margin[2 * 32 + 1];
  int near_lo[2 * 32 + 1], near_hi[2 * 32 + 1];
} seq_rows_t;

static const double* seq_row(seq_rows_t* s, int id) {
  if (!s->probs[id]) {
    size_t es = (s->dtype == ORACLE_BF16) ? 2 : 4;
    const char* base = id <= s->k ? (const char*)s->target + (size_t)id * s->V * es
                                  : (const char*)s->draft + (size_t)(id - s->k - 1) * s->V * es;
    s->probs[id] = (double*)malloc(sizeof(double) * (size_t)s->V);
    s->ok[id] = row_probs_adj(base, s->dtype, s->V, s->T, s->top_k, s->top_p, 0, s->probs[id],
                              &s->margin[id], NULL, NULL, &s->near_lo[id], &s->near_hi[id]) == 0;
  }
  return s->probs[id];
}

static double* alt_row(seq_rows_t* s, int id, int adjust) {
  size_t es = (s->dtype == ORACLE_BF16) ? 2 : 4;
  const char* base = id <= s->k ? (const char*)s->target + (size_t)id * s->V * es
                                : (const char*)s->draft + (size_t)(id - s->k - 1) * s->V * es;
  double* p = (double*)malloc(sizeof(double) * (size_t)s->V);
  row_probs_adj(base, s->dtype, s->V, s->T, s->top_k, s->top_p, adjust, p, NULL, NULL, NULL, NULL,
                NULL);
  return p;
}

typedef struct {
  int n, drawn;
  int tokens[33];
  uint32_t flags;      /* accept / draw / degenerate / bad-token / bad-row bits */
  double min_margin;
  int consulted[2 * 32 + 1];
  int n_consulted;
} outcome_t;

/*
 * The left-to-right scan of [EIN] "The core idea: draft, then check", step 3,
 * for one sequence.  Row `alt_id` (if >= 0) is replaced by `alt_probs`.
 */
static void scan_sequence(seq_rows_t* s, const int32_t* x, const float* u, int alt_id,
                          const double* alt_probs, double* w, outcome_t* o) {
  const int k = s->k, V = s->V;
  int i, t;
  o->flags = 0;
  o->min_margin = INFINITY;
  o->n_consulted = 0;
  o->drawn = -1;
#define ROW(id) ((id) == alt_id ? alt_probs : seq_row(s, (id)))
  for (i = 0; i < k; ++i) {
    const double* p = ROW(i);
    const double* q = ROW(k + 1 + i);
    const int ok = s->ok[i] && s->ok[k + 1 + i];
    const int in_range = x[i] >= 0 && x[i] < V;
    const double px = in_range ? p[x[i]] : 0.0, qx = in_range ? q[x[i]] : 0.0;
    o->consulted[o->n_consulted++] = i;
    o->consulted[o->n_consulted++] = k + 1 + i;
    if (!in_range) o->flags |= OFLAG_BAD_TOKEN;
    if (!ok) o->flags |= OFLAG_BAD_ROW;
    if (qx > 0.0 && px < qx) {
      double mg = fabs((double)u[i] - px / qx);
      if (mg < o->min_margin) o->min_margin = mg;
      if (mg < BOUNDARY_EPS) o->flags |= OFLAG_ACCEPT_BOUNDARY;
    }
    if (in_range && ok && (double)u[i] * qx < px) {
      o->tokens[i] = x[i];
      continue;
    }
    /* first rejection: resample from max(0, p - q) */
    o->n = i;
    if (ok) {
      double sum = 0.0, mg = 0.0;
      for (t = 0; t < V; ++t) {
        double d = p[t] - q[t];
        w[t] = d > 0.0 ? d : 0.0;
        sum += w[t];
      }
      if (!(sum > 0.0)) {
        o->flags |= OFLAG_DEGENERATE;
        o->drawn = inverse_cdf(p, V, (double)u[k + 1], &mg);
      } else {
        o->drawn = inverse_cdf(w, V, (double)u[k + 1], &mg);
      }
      if (mg < BOUNDARY_EPS) o->flags |= OFLAG_DRAW_BOUNDARY;
      if (mg < o->min_margin) o->min_margin = mg;
    }
    o->tokens[i] = o->drawn;
    return;
  }
  /* every draft accepted: bonus token from the last target row */
  {
    const double* p = ROW(k);
    double mg = 0.0;
    o->consulted[o->n_consulted++] = k;
    o->n = k;
    if (!s->ok[k]) {
      o->flags |= OFLAG_BAD_ROW;
    } else {
      o->drawn = inverse_cdf(p, V, (double)u[k], &mg);
      if (mg < BOUNDARY_EPS) o->flags |= OFLAG_DRAW_BOUNDARY;
      if (mg < o->min_margin) o->min_margin = mg;
    }
    o->tokens[k] = o->drawn;
  }
#undef ROW
}

/*
 * Speculative sampling verification ([EIN] "The core idea: draft, then
 * check", step 3 "Accept or correct"):
 *
 *   for i = 0 .. k-1, left to right:
 *     accept draft x_i iff u_i * q_i(x_i) < p_i(x_i)   (probability min(1, p/q))
 *     at the first rejection stop: n = i
 *   if n < k: draw one token from the normalised residual max(0, p_n - q_n)
 *             with u_{k+1}
 *   else    : draw the bonus token from p_k with u_k
 *   commit x_0 .. x_{n-1} and the drawn token (1 .. k+1 tokens per pass).
 *
 * Layouts: target [B][k+1][V], draft [B][k][V], tokens [B][k],
 * uniforms [B][k+2] (u_0..u_{k-1} accept tests, u_k bonus, u_{k+1} resample),
 * temperature_per_seq [B] or NULL; k <= 32.
 * Outputs: out_tokens [B][k+1] (-1 padded), out_n [B], out_p / out_q [B][k]
 * (p_i(x_i), q_i(x_i); NaN where not computed), out_flags [B] (OFLAG_*),
 * out_margin [B] (smallest accept / draw margin met; may be NULL).
 * all_rows != 0 computes p_i(x_i), q_i(x_i) for every i, not only the rows
 * the scan consults.
 *
 * Boundary flags: a decision is "within 1e-6 of its edge" when an accept test
 * has |u - p/q| < 1e-6, when the draw has u*S within 1e-6*S of an edge of the
 * chosen token's interval, or when a consulted row's top-p cut has a margin
 * below 1e-6 AND taking the neighbouring cut decision for that row changes
 * the committed tokens.
 */
int oracle_verify_sample(const void* target, const void* draft, int dtype,
                         const int32_t* tokens, const float* uniforms, int B, int k,
                         int V, double temperature, const float* temperature_per_seq,
                         int top_k, double top_p, int all_rows, int32_t* out_tokens,
                         int32_t* out_n, double* out_p, double* out_q,
                         uint32_t* out_flags, double* out_margin) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int b, i, j;
  if (k < 1 || k > 32) {
    free(w);
    return -1;
  }
  for (b = 0; b < B; ++b) {
    seq_rows_t s;
    outcome_t o, alt;
    const int32_t* x = tokens + (size_t)b * k;
    const float* u = uniforms + (size_t)b * (size_t)(k + 2);
    memset(&s, 0, sizeof s);
    s.target = (const char*)target + (size_t)b * (k + 1) * (size_t)V * es;
    s.draft = (const char*)draft + (size_t)b * k * (size_t)V * es;
    s.dtype = dtype;
    s.k = k;
    s.V = V;
    s.top_k = top_k;
    s.T = temperature_per_seq ? (double)temperature_per_seq[b] : temperature;
    s.top_p = top_p;
    scan_sequence(&s, x, u, -1, NULL, w, &o);
    /* top-p cuts within 1e-6 of top_p: does the neighbouring decision matter? */
    for (j = 0; j < o.n_consulted; ++j) {
      int id = o.consulted[j], adj;
      for (adj = -1; adj <= 1; adj += 2) {
        double* ap;
        int differs;
        if (!(adj < 0 ? s.near_lo[id] : s.near_hi[id])) continue;
        ap = alt_row(&s, id, adj);
        scan_sequence(&s, x, u, id, ap, w, &alt);
        differs = alt.n != o.n;
        for (i = 0; i <= o.n && !differs; ++i) differs = alt.tokens[i] != o.tokens[i];
        if (differs) o.flags |= OFLAG_CUT_BOUNDARY;
        free(ap);
      }
    }
    for (i = 0; i <= k; ++i) out_tokens[(size_t)b * (k + 1) + i] = i <= o.n ? o.tokens[i] : -1;
    out_n[b] = o.n;
    out_flags[b] = o.flags;
    if (out_margin) out_margin[b] = o.min_margin;
    for (i = 0; i < k; ++i) {
      int have = s.probs[i] && s.probs[k + 1 + i];
      double px = NAN, qx = NAN;
      if (all_rows || have) {
        const double* p = seq_row(&s, i);
        const double* q = seq_row(&s, k + 1 + i);
        int in_range = x[i] >= 0 && x[i] < V;
        px = in_range ? p[x[i]] : 0.0;
        qx = in_range ? q[x[i]] : 0.0;
      }
      out_p[(size_t)b * k + i] = px;
      out_q[(size_t)b * k + i] = qx;
    }
    for (i = 0; i < 2 * 32 + 1; ++i) free(s.probs[i]);
  }
  free(w);
  return 0;
}

/* Index of the largest entry of a raw logit row; the lowest index wins ties. */
static int row_argmax(const void* row, int dtype, int V) {
  int t, best = 0;
  double bv = read_logit(row, dtype, 0);
  for (t = 1; t < V; ++t) {
    double v = read_logit(row, dtype, (size_t)t);
    if (v > bv) {
      bv = v;
      best = t;
    }
  }
  return best;
}

/*
 * Greedy chain verification ([TGTG] section 2.4): the k+1 target rows are
 * compared greedily with the k drafts; the longest prefix that equals the
 * target's argmax is accepted and the target's own choice at the first
 * disagreement (or after the last draft) is appended.
 * target [B][k+1][V], tokens [B][k]; out_tokens [B][k+1] (-1 padded), out_n [B].
 */
int oracle_verify_greedy(const void* target, int dtype, const int32_t* tokens, int B,
                         int k, int V, int32_t* out_tokens, int32_t* out_n) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  int b, i;
  for (b = 0; b < B; ++b) {
    int n = k;
    for (i = 0; i <= k; ++i) out_tokens[(size_t)b * (k + 1) + i] = -1;
    for (i = 0; i <= k; ++i) {
      const char* row = (const char*)target + ((size_t)b * (k + 1) + i) * (size_t)V * es;
      int a = row_argmax(row, dtype, V);
      if (i == k || tokens[(size_t)b * k + i] != a) {
        out_tokens[(size_t)b * (k + 1) + i] = a;
        n = i;
        break;
      }
      out_tokens[(size_t)b * (k + 1) + i] = a;
    }
    out_n[b] = n;
  }
  return 0;
}

/*
 * The rejection fast path ([TGTG] section 2.4, KV-cached regime): the first
 * draft token is checked against the previous step's logits, already
 * computed; the k-token pass is needed only when it is accepted.  For every
 * sequence b: a = argmax of prev_rows[b] (lowest index on ties);
 * out_accept[b] = 1 iff draft0[b] == a; out_argmax[b] = a (the token to
 * commit when draft 0 is rejected).
 */
int oracle_first_draft_check(const void* prev_rows, int dtype, const int32_t* draft0, int B, int V,
                             int32_t* out_accept, int32_t* out_argmax) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  int b;
  for (b = 0; b < B; ++b) {
    const char* row = (const char*)prev_rows + (size_t)b * (size_t)V * es;
    int a = row_argmax(row, dtype, V);
    out_argmax[b] = a;
    out_accept[b] = draft0[b] == a ? 1 : 0;
  }
  return 0;
}

/*
 * Greedy token-tree verification ([EIN] "One decode round, end to end"):
 * node j's row is the target's distribution for the token after node j
 * (node 0 is the root, the last committed token).  A node is on an agreed
 * path iff its parent is and its token equals the parent's argmax.  The
 * deepest agreed node d* (lowest index among equally deep ones) is committed
 * with its path (root excluded) and the correction token argmax(row d*).
 *
 * logits [B][N][V], node_tokens [B][N], parents [B][N] (parents[0] = -1,
 * 0 <= parents[j] < j).  out_tokens, out_path [B][max_depth+1] (-1 padded),
 * out_n [B] = depth of d*.  out_flags [B]: 1 = malformed parent array,
 * 2 = an agreed node deeper than max_depth (ignored).  Nodes with a bad
 * parent are treated as not agreed.
 */
int oracle_verify_tree_greedy(const void* logits, int dtype, const int32_t* node_tokens,
                              const int32_t* parents, int B, int N, int V, int max_depth,
                              int32_t* out_tokens, int32_t* out_path, int32_t* out_n,
                              uint32_t* out_flags) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  int* am = (int*)malloc(sizeof(int) * (size_t)N);
  int* depth = (int*)malloc(sizeof(int) * (size_t)N);
  char* agreed = (char*)malloc((size_t)N);
  int* chain = (int*)malloc(sizeof(int) * (size_t)(N + 1));
  int b, j;
  for (b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * N;
    const int32_t* tok = node_tokens + (size_t)b * N;
    uint32_t flags = 0;
    int best = 0, len = 0, c;
    for (j = 0; j < N; ++j) {
      const char* row = (const char*)logits + ((size_t)b * N + j) * (size_t)V * es;
      am[j] = row_argmax(row, dtype, V);
    }
    agreed[0] = 1;
    depth[0] = 0;
    if (par[0] != -1) flags |= 1u;
    for (j = 1; j < N; ++j) {
      int pj = par[j];
      agreed[j] = 0;
      depth[j] = 0;
      if (pj < 0 || pj >= j) {
        flags |= 1u;
        continue;
      }
      depth[j] = depth[pj] + 1;
      agreed[j] = agreed[pj] && tok[j] == am[pj];
      if (agreed[j] && depth[j] > max_depth) {
        flags |= 2u;
        agreed[j] = 0;
      }
    }
    for (j = 1; j < N; ++j)
      if (agreed[j] && depth[j] > depth[best]) best = j;
    for (j = 0; j <= max_depth; ++j) {
      out_tokens[(size_t)b * (max_depth + 1) + j] = -1;
      out_path[(size_t)b * (max_depth + 1) + j] = -1;
    }
    for (c = best; c != 0; c = par[c]) chain[len++] = c;
    for (j = 0; j < len; ++j) {
      int node = chain[len - 1 - j];
      out_path[(size_t)b * (max_depth + 1) + j] = node;
      out_tokens[(size_t)b * (max_depth + 1) + j] = tok[node];
    }
    out_tokens[(size_t)b * (max_depth + 1) + len] = am[best];
    out_n[b] = len;
    out_flags[b] = flags;
  }
  free(am);
  free(depth);
  free(agreed);
  free(chain);
  return 0;
}

/*
 * Token-tree sampling verification ([EIN] "One decode round, end to end": the
 * accept-or-correct rule of "The core idea: draft, then check" applied down
 * the branches of the draft tree).  Per tree b, starting at the root (node 0):
 *
 *   p = softmax(node_logits[v] / T), q = softmax(draft_logits[v] / T)
 *   r = p
 *   for each child j of v (parents[j] == v), in ascending node order:
 *     skip j if its token is outside [0, V) or depth(v) == max_depth
 *     accept j iff u_j * q(x_j) < r(x_j)   (probability min(1, r/q))
 *       -> commit x_j, move to v = j, start again
 *     else r <- max(0, r - q) / sum(max(0, r - q))   (q is unchanged)
 *          a residual of total mass 0 is replaced by p
 *   no child accepted: draw one token from r with u_0 (inverse CDF,
 *   ascending index order) and stop.
 *
 * The pages state the rule for a chain and say only that it is applied down
 * the branches.  The sibling rule taken here (each rejected sibling removes
 * its draft mass from the residual, the next sibling is tested against the
 * renormalised residual) keeps the output distributed as p when the children
 * of a node are drawn independently from q; the tests check that property.
 *
 * Layouts: node_logits, draft_logits [B][N][V] (draft row v is the draft
 * distribution the children of v were drawn from), node_tokens, parents
 * [B][N], uniforms [B][N] (u_0 the final draw, u_j the test of node j).
 * Outputs: out_tokens [B][max_depth+1] (path tokens, the drawn token, then
 * -1), out_path [B][max_depth+1] (path node ids, root excluded, -1 padded),
 * out_n [B] (accepted nodes), out_flags [B] (OFLAG_*), out_margin [B] (the
 * smallest accept / draw margin met; may be NULL).  temperature_per_tree [B]
 * (or NULL for the scalar temperature) gives every tree its own T; a T that
 * is not finite and positive ends that tree's walk at the root (drawn -1).
 * A node whose parent entry is malformed is never a child of anything; a
 * non-finite row at a visited node ends the walk there with drawn token -1.
 */
int oracle_verify_tree_sample(const void* node_logits, const void* draft_logits, int dtype,
                              const int32_t* node_tokens, const int32_t* parents,
                              const float* uniforms, int B, int N, int V, int max_depth,
                              double temperature, const float* temperature_per_tree,
                              int32_t* out_tokens, int32_t* out_path,
                              int32_t* out_n, uint32_t* out_flags, double* out_margin) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  int b, j, t;
  if (N < 1 || max_depth < 1 || (!temperature_per_tree && !(temperature > 0.0))) {
    free(p);
    free(q);
    free(r);
    return -1;
  }
  for (b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * N;
    const int32_t* tok = node_tokens + (size_t)b * N;
    const float* u = uniforms + (size_t)b * N;
    const size_t D = (size_t)max_depth + 1;
    uint32_t flags = 0;
    double margin = INFINITY;
    int v = 0, n = 0, drawn = -1;
    const double T = temperature_per_tree ? (double)temperature_per_tree[b] : temperature;
    if (par[0] != -1) flags |= OFLAG_BAD_PARENT;
    for (j = 1; j < N; ++j) {
      if (par[j] < 0 || par[j] >= j) flags |= OFLAG_BAD_PARENT;
      if (tok[j] < 0 || tok[j] >= V) flags |= OFLAG_BAD_TOKEN;
    }
    for (j = 0; j < (int)D; ++j) {
      out_tokens[(size_t)b * D + j] = -1;
      out_path[(size_t)b * D + j] = -1;
    }
    for (;;) {
      const char* prow = (const char*)node_logits + ((size_t)b * N + v) * (size_t)V * es;
      if (!(T > 0.0) || isinf(T)) { /* a temperature that gives no distribution */
        flags |= OFLAG_BAD_ROW;
        break;
      }
      const char* qrow = (const char*)draft_logits + ((size_t)b * N + v) * (size_t)V * es;
      int has_child = 0, n_test = 0, accepted = -1;
      for (j = v + 1; j < N; ++j)
        if (par[j] == v) {
          has_child = 1;
          if (tok[j] >= 0 && tok[j] < V && n < max_depth) ++n_test;
        }
      if (has_child && n >= max_depth) flags |= OFLAG_DEPTH;
      if (row_probs_adj(prow, dtype, V, T, 0, 1.0, 0, p, NULL, NULL, NULL, NULL, NULL) != 0) {
        flags |= OFLAG_BAD_ROW;
        break;
      }
      if (n_test > 0 &&
          row_probs_adj(qrow, dtype, V, T, 0, 1.0, 0, q, NULL, NULL, NULL, NULL, NULL) != 0) {
        flags |= OFLAG_BAD_ROW;
        break;
      }
      for (t = 0; t < V; ++t) r[t] = p[t];
      for (j = v + 1; j < N && n_test > 0; ++j) {
        int x = tok[j];
        double s;
        if (par[j] != v || x < 0 || x >= V) continue;
        if (q[x] > 0.0 && r[x] < q[x]) {
          double mg = fabs((double)u[j] - r[x] / q[x]);
          if (mg < margin) margin = mg;
          if (mg < BOUNDARY_EPS) flags |= OFLAG_ACCEPT_BOUNDARY;
        }
        if ((double)u[j] * q[x] < r[x]) {
          accepted = j;
          break;
        }
        s = 0.0;
        for (t = 0; t < V; ++t) {
          double d = r[t] - q[t];
          r[t] = d > 0.0 ? d : 0.0;
          s += r[t];
        }
        if (s > 0.0) {
          for (t = 0; t < V; ++t) r[t] /= s;
        } else {
          flags |= OFLAG_DEGENERATE;
          for (t = 0; t < V; ++t) r[t] = p[t];
        }
      }
      if (accepted >= 0) {
        out_path[(size_t)b * D + n] = accepted;
        out_tokens[(size_t)b * D + n] = tok[accepted];
        ++n;
        v = accepted;
        continue;
      }
      {
        double mg = 0.0;
        drawn = inverse_cdf(r, V, (double)u[0], &mg);
        if (mg < margin) margin = mg;
        if (mg < BOUNDARY_EPS) flags |= OFLAG_DRAW_BOUNDARY;
      }
      break;
    }
    out_tokens[(size_t)b * D + n] = drawn;
    out_n[b] = n;
    out_flags[b] = flags;
    if (out_margin) out_margin[b] = margin;
  }
  free(p);
  free(q);
  free(r);
  return 0;
}

/* [SDSC] step 1: expected tokens per pass, as the geometric series. */
double oracle_expected_tokens_series(double alpha, int gamma) {
  double e = 0.0, a = 1.0;
  int i;
  for (i = 0; i <= gamma; ++i) {
    e += a;
    a *= alpha;
  }
  return e;
}

/* [SDSC] step 1: the closed form (1 - alpha^(gamma+1)) / (1 - alpha). */
double oracle_expected_tokens_closed(double alpha, int gamma) {
  return (1.0 - pow(alpha, (double)(gamma + 1))) / (1.0 - alpha);
}

/* [SDSC] steps 2-3: cost gamma*c + 1 and speedup E / (gamma*c + 1). */
double oracle_improvement_factor(double alpha, int gamma, double c) {
  return oracle_expected_tokens_series(alpha, gamma) / ((double)gamma * c + 1.0);
}

/* [TGTG] section 5.1, equation 1: break-even acceptance k / (k + 1). */
double oracle_break_even(int k) { return (double)k / (double)(k + 1); }

/*
 * [SDSC] the draft length scan: the gamma in 1..gamma_max with the largest
 * speedup E / (gamma*c + 1) (the first one on ties), its speedup in *best.
 */
int oracle_best_gamma(double alpha, double c, int gamma_max, double* best) {
  int g, arg = 1;
  double top = oracle_improvement_factor(alpha, 1, c);
  for (g = 2; g <= gamma_max; ++g) {
    double f = oracle_improvement_factor(alpha, g, c);
    if (f > top) {
      top = f;
      arg = g;
    }
  }
  if (best) *best = top;
  return arg;
}
