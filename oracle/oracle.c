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
 *     rounding) is replaced by the target row itself.
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
#define OFLAG_CUT_BOUNDARY 8u     /* a token that decided the outcome sits at a
                                     top-p cut whose margin is below 1e-6    */
#define OFLAG_BAD_TOKEN 16u       /* a draft token outside [0, V)             */
#define OFLAG_BAD_ROW 32u         /* a row with NaN/+inf or no finite entry   */

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
 * probs[V] receives p.  *cut_margin receives the distance |before - top_p| of
 * the last kept and the first dropped token (the smaller one); +inf when no
 * top-p cut was made.  *cut_lo / *cut_hi receive those two token ids (-1 if
 * none).  Returns 0, or -1 for a row with NaN, +inf or no finite entry.
 */
int oracle_row_probs(const void* row, int dtype, int V, double temperature,
                     int top_k, double top_p, double* probs, double* cut_margin,
                     int* cut_lo, int* cut_hi) {
  ranked_t* r = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)V);
  char* kept = (char*)calloc((size_t)V, 1);
  int t, n_topk, rc = 0;
  double m, zk, zkept, before;
  if (cut_margin) *cut_margin = INFINITY;
  if (cut_lo) *cut_lo = -1;
  if (cut_hi) *cut_hi = -1;
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
    int last_kept = 0;
    before = 0.0;
    for (t = 0; t < n_topk; ++t) {
      if (!(before < top_p)) break;
      kept[r[t].idx] = 1;
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
      if (last_kept + 1 < n_topk) {
        double b_next = b_last + exp(r[last_kept].z - m) / zk;
        if (fabs(b_next - top_p) < margin) margin = fabs(b_next - top_p);
        if (cut_hi) *cut_hi = r[last_kept + 1].idx;
      }
      if (cut_margin) *cut_margin = margin;
    }
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
 * temperature_per_seq [B] or NULL.
 * Outputs: out_tokens [B][k+1] (-1 padded), out_n [B], out_p / out_q [B][k]
 * (p_i(x_i), q_i(x_i); NaN where not computed), out_flags [B] (OFLAG_*),
 * out_margin [B] (smallest decision margin met; may be NULL).
 * all_rows != 0 computes p_i(x_i), q_i(x_i) for every i, not only the rows
 * the scan consults.
 */
int oracle_verify_sample(const void* target, const void* draft, int dtype,
                         const int32_t* tokens, const float* uniforms, int B, int k,
                         int V, double temperature, const float* temperature_per_seq,
                         int top_k, double top_p, int all_rows, int32_t* out_tokens,
                         int32_t* out_n, double* out_p, double* out_q,
                         uint32_t* out_flags, double* out_margin) {
  size_t es = (dtype == ORACLE_BF16) ? 2 : 4;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int b, i, t;
  for (b = 0; b < B; ++b) {
    double T = temperature_per_seq ? (double)temperature_per_seq[b] : temperature;
    const float* u = uniforms + (size_t)b * (size_t)(k + 2);
    uint32_t flags = 0;
    double min_margin = INFINITY;
    int n = k, drawn = -1;
    int decided = 0;
    for (i = 0; i <= k; ++i) out_tokens[(size_t)b * (k + 1) + i] = -1;
    for (i = 0; i < k; ++i) {
      out_p[(size_t)b * k + i] = NAN;
      out_q[(size_t)b * k + i] = NAN;
    }
    for (i = 0; i < k; ++i) {
      const char* trow = (const char*)target + ((size_t)b * (k + 1) + i) * (size_t)V * es;
      const char* drow = (const char*)draft + ((size_t)b * k + i) * (size_t)V * es;
      double mp, mq, px, qx;
      int x = tokens[(size_t)b * k + i];
      int lo_p, hi_p, lo_q, hi_q, okp, okq;
      if (decided && !all_rows) break;
      okp = oracle_row_probs(trow, dtype, V, T, top_k, top_p, p, &mp, &lo_p, &hi_p);
      okq = oracle_row_probs(drow, dtype, V, T, top_k, top_p, q, &mq, &lo_q, &hi_q);
      if (x < 0 || x >= V) {
        if (!decided) flags |= OFLAG_BAD_TOKEN;
        px = 0.0;
        qx = 0.0;
      } else {
        px = p[x];
        qx = q[x];
      }
      if (okp != 0 || okq != 0) {
        if (!decided) flags |= OFLAG_BAD_ROW;
      }
      out_p[(size_t)b * k + i] = px;
      out_q[(size_t)b * k + i] = qx;
      if (decided) continue;
      {
        int accept = (x >= 0 && x < V && okp == 0 && okq == 0) &&
                     ((double)u[i] * qx < px);
        if (qx > 0.0 && px < qx) {
          double mg = fabs((double)u[i] - px / qx);
          if (mg < min_margin) min_margin = mg;
          if (mg < BOUNDARY_EPS) flags |= OFLAG_ACCEPT_BOUNDARY;
        }
        if ((x == lo_p || x == hi_p) && mp < BOUNDARY_EPS) flags |= OFLAG_CUT_BOUNDARY;
        if ((x == lo_q || x == hi_q) && mq < BOUNDARY_EPS) flags |= OFLAG_CUT_BOUNDARY;
        if (mp < min_margin && (x == lo_p || x == hi_p)) min_margin = mp;
        if (mq < min_margin && (x == lo_q || x == hi_q)) min_margin = mq;
        if (accept) {
          out_tokens[(size_t)b * (k + 1) + i] = x;
          continue;
        }
        /* first rejection: resample from max(0, p - q) */
        n = i;
        decided = 1;
        if (okp == 0 && okq == 0) {
          double s = 0.0, mg = 0.0;
          for (t = 0; t < V; ++t) {
            double d = p[t] - q[t];
            w[t] = d > 0.0 ? d : 0.0;
            s += w[t];
          }
          if (!(s > 0.0)) {
            flags |= OFLAG_DEGENERATE;
            drawn = inverse_cdf(p, V, (double)u[k + 1], &mg);
          } else {
            drawn = inverse_cdf(w, V, (double)u[k + 1], &mg);
          }
          if (mg < BOUNDARY_EPS) flags |= OFLAG_DRAW_BOUNDARY;
          if (mg < min_margin) min_margin = mg;
          if ((drawn == lo_p || drawn == hi_p) && mp < BOUNDARY_EPS) flags |= OFLAG_CUT_BOUNDARY;
          if ((drawn == lo_q || drawn == hi_q) && mq < BOUNDARY_EPS) flags |= OFLAG_CUT_BOUNDARY;
        }
        out_tokens[(size_t)b * (k + 1) + i] = drawn;
      }
    }
    if (!decided) {
      /* every draft accepted: bonus token from the last target row */
      const char* trow = (const char*)target + ((size_t)b * (k + 1) + k) * (size_t)V * es;
      double mp, mg = 0.0;
      int lo_p, hi_p;
      if (oracle_row_probs(trow, dtype, V, T, top_k, top_p, p, &mp, &lo_p, &hi_p) != 0) {
        flags |= OFLAG_BAD_ROW;
        drawn = -1;
      } else {
        drawn = inverse_cdf(p, V, (double)u[k], &mg);
        if (mg < BOUNDARY_EPS) flags |= OFLAG_DRAW_BOUNDARY;
        if (mg < min_margin) min_margin = mg;
        if ((drawn == lo_p || drawn == hi_p) && mp < BOUNDARY_EPS) flags |= OFLAG_CUT_BOUNDARY;
      }
      n = k;
      out_tokens[(size_t)b * (k + 1) + k] = drawn;
    }
    out_n[b] = n;
    out_flags[b] = flags;
    if (out_margin) out_margin[b] = min_margin;
  }
  free(p);
  free(q);
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
