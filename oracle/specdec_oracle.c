/*
 * specdec_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of the target-side verify step of
 * speculative decoding.  It exists to check the CUDA path: only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code, header or constant table with the CUDA library; the status values
 * below are restated here from the interface description on purpose.
 *
 * Source of every step: "Chapter 15: Decoding acceleration" of the LLM edge
 * inference notes (zsc.github.io, llm_edge_inference/chapter15), section
 * 15.1.2 "mathematical framework of speculative decoding":
 *   step 2 "parallel verification": one target row per drafted position,
 *          p_i = softmax(logits row), read at the drafted token;
 *   step 3 "accept/reject": for i = 1..gamma, accept x~_i iff
 *          u_i <= min(1, p_i / q_i); stop at the first rejection;
 *   step 4 "distribution correction": at the rejected position sample from
 *          r(x) = max(0, p(x) - q(x)) / sum_x' r(x');
 *   the section's theorem (output law = p) and Lemma 1 are what the tests pin.
 * The bonus draw from the last target row when every draft is accepted is
 * implied by section 15.1.3's expected token count (1 - a^(g+1)) / (1 - a).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - temperature: p = softmax(l / T); T = 0 means greedy, i.e. the T -> 0
 *     limit: p is one-hot at the first maximal logit; other valid T lie in
 *     [2^-20, 2^20];
 *   - accept compare is "u <= min(1, p/q)" (the chapter's pseudo-code);
 *   - a draw from weights w with uniform U picks the smallest v whose
 *     running sum C_v = w_0 + ... + w_v exceeds U * Z, Z = sum w (strict);
 *   - if the residual mass Z is 0 (only reachable by rounding) the draw
 *     falls back to p itself;
 *   - q is used exactly as stored: no renormalisation;
 *   - token tree: children of a node are tried in ascending node index; a
 *     rejected sibling replaces the current distribution P by
 *     max(0, P - q_parent) / sum(...) (literal renormalisation), a leaf
 *     draws its bonus from its own target row;
 *   - a malformed request gets a status bitmask and sentinel outputs.
 *
 * The uniforms the method draws (section 15.1.2 step 3: u ~ U(0,1)) are an
 * input of both sides.  For generating them on the device, the library has a
 * Philox4x64-10 generator; its statement here (specdec_oracle_philox_*) follows
 * the generator's published definition (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11) and is pinned against NumPy's
 * Philox bit generator, an independent implementation of the same definition.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no fast-math: IEEE double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_DT_F32 0
#define OR_DT_BF16 1

#define OR_ROW_BAD_TOKEN 1
#define OR_ROW_BAD_Q 2
#define OR_ROW_NONFINITE 4
#define OR_ROW_BAD_TEMP 8
#define OR_ROW_BAD_TREE 16

/* ------------------------------------------------------------------------ */
/* element access                                                             */
/* ------------------------------------------------------------------------ */

static double load_elem(const void *base, int dtype, size_t idx) {
  if (dtype == OR_DT_F32) return (double)((const float *)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Valid temperatures: 0 (greedy) or 2^-20 <= T <= 2^20. */
static int temperature_valid(float T) {
  return T == 0.0f || (T >= 0x1p-20f && T <= 0x1p20f);
}

/* A target row is unusable when it holds a NaN or +Inf, when no value is
 * finite, or when its largest logit exceeds 2^100 (so l / T stays far inside
 * the float range for every valid temperature). */
static int row_nonfinite(const void *base, int dtype, size_t off, int V) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = load_elem(base, dtype, off + (size_t)v);
    if (isnan(x) || x == INFINITY) return 1;
    if (x > mx) mx = x;
  }
  return mx == -INFINITY || mx > 0x1p100;
}

/* Target distribution of one row (section 15.1.2 step 2 with temperature):
 * T > 0: p_v = exp(z_v - m) / sum_u exp(z_u - m), z = l / T, m = max z.
 * T = 0: one-hot at the first index of the largest logit. */
static void target_probs(const void *logits, int dtype, size_t off, int V, double T,
                         double *p) {
  if (T == 0.0) {
    int a = 0;
    double best = load_elem(logits, dtype, off);
    for (int v = 1; v < V; ++v) {
      double x = load_elem(logits, dtype, off + (size_t)v);
      if (x > best) { best = x; a = v; }
    }
    for (int v = 0; v < V; ++v) p[v] = 0.0;
    p[a] = 1.0;
    return;
  }
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = load_elem(logits, dtype, off + (size_t)v) / T;
    if (z > m) m = z;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    double e = exp(load_elem(logits, dtype, off + (size_t)v) / T - m);
    p[v] = e;
    S += e;
  }
  for (int v = 0; v < V; ++v) p[v] /= S;
}

/* Inverse-CDF draw: smallest v with C_v > U * Z.  Reports the distance of
 * U * Z to the two CDF boundaries around the chosen v, relative to Z, and Z
 * itself (the weights' total). */
static int cdf_draw(const double *w, int V, double U, double *margin, double *total) {
  double Z = 0.0;
  for (int v = 0; v < V; ++v) Z += w[v];
  *total = Z;
  double t = U * Z;
  double C = 0.0, prev = 0.0;
  for (int v = 0; v < V; ++v) {
    prev = C;
    C += w[v];
    if (C > t) {
      if (margin) {
        double a = fabs(t - prev), b = fabs(C - t);
        *margin = (a < b ? a : b) / Z;
      }
      return v;
    }
  }
  /* only reachable by rounding: the last index with positive weight */
  for (int v = V - 1; v >= 0; --v)
    if (w[v] > 0.0) {
      if (margin) *margin = 0.0;
      return v;
    }
  if (margin) *margin = 0.0;
  return V - 1;
}

/* ------------------------------------------------------------------------ */
/* linear verify                                                              */
/* ------------------------------------------------------------------------ */

/* All arrays are host arrays, row-major:
 *   logits [B, gamma+1, V], q [B, gamma, V] (dtype 0 = float32, 1 = bf16 bits),
 *   draft_tokens int32 [B, gamma], temperature float32 [B],
 *   uniforms float32 [B, gamma+1] (slot i = test of draft i, slot gamma = draw).
 * Outputs: n_accepted [B], out_tokens [B, gamma+1] (-1 padded),
 *   final_token [B], is_bonus [B], row_status [B].
 * Optional diagnostics (NULL to skip):
 *   p_draft [B, gamma]    target probability of each drafted token;
 *   ratio   [B, gamma]    min(1, p/q) of each drafted token;
 *   final_margin [B]      distance of U*Z to the nearest CDF boundary / Z;
 *   row_diag [B, gamma, 2] per drafted row: sum_x min(p,q), sum_x max(0,p-q);
 *   final_mass [B]        Z, the total of the final draw's weights: the mass of
 *                         max(0, p_k - q_k) after a rejection at k, of p_gamma
 *                         for the bonus draw (NaN for a malformed request).
 * Returns 0, or -1 on a bad argument. */
/* Candidate set of the top-k residual (the chapter's implementation note:
 * precompute the residual probabilities of the top-k candidates instead of
 * the whole vocabulary): the k tokens of largest target probability, ties to
 * the lower index.  in_k[v] = 1 for them. */
static const double *g_sort_p; /* comparator context (one sort per thread at a time) */
#pragma omp threadprivate(g_sort_p)
static int by_p_desc(const void *a, const void *b) {
  const int i = *(const int *)a, j = *(const int *)b;
  if (g_sort_p[i] > g_sort_p[j]) return -1;
  if (g_sort_p[i] < g_sort_p[j]) return 1;
  return (i > j) - (i < j);
}

static void topk_candidates(const double *p, int V, int k, unsigned char *in_k) {
  int *idx = (int *)malloc(sizeof(int) * (size_t)V);
  for (int v = 0; v < V; ++v) {
    idx[v] = v;
    in_k[v] = 0;
  }
  g_sort_p = p;
  qsort(idx, (size_t)V, sizeof(int), by_p_desc);
  for (int j = 0; j < k && j < V; ++j) in_k[idx[j]] = 1;
  free(idx);
}

static int verify_linear_impl(const void *logits, const void *q, int dtype,
                              const int32_t *draft_tokens, const float *temperature,
                              const float *uniforms, int B, int gamma, int V, int topk,
                              int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                              uint8_t *is_bonus, int32_t *row_status, double *p_draft,
                              double *ratio, double *final_margin, double *row_diag,
                              double *tv, double *final_mass);

int specdec_oracle_verify_linear(const void *logits, const void *q, int dtype,
                                 const int32_t *draft_tokens, const float *temperature,
                                 const float *uniforms, int B, int gamma, int V,
                                 int32_t *n_accepted, int32_t *out_tokens,
                                 int32_t *final_token, uint8_t *is_bonus,
                                 int32_t *row_status, double *p_draft, double *ratio,
                                 double *final_margin, double *row_diag, double *final_mass) {
  return verify_linear_impl(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                            0, n_accepted, out_tokens, final_token, is_bonus, row_status,
                            p_draft, ratio, final_margin, row_diag, NULL, final_mass);
}

/* The linear step with the top-k residual (an approximation: the law of the
 * correction token is no longer max(0, p - q) / Z).  At a rejection the
 * residual is restricted to the top-k candidates of p and renormalised; if
 * it has no mass there, the draw uses p restricted to the candidates.  The
 * bonus draw is unchanged.  tv[b] (NULL to skip) = total-variation distance
 * between the exact residual law and the one drawn from = 1 - Z_K / Z for a
 * rejected request whose exact residual has mass (Z_K the residual mass on
 * the candidates), else NaN. */
int specdec_oracle_verify_linear_topk(const void *logits, const void *q, int dtype,
                                      const int32_t *draft_tokens, const float *temperature,
                                      const float *uniforms, int B, int gamma, int V, int topk,
                                      int32_t *n_accepted, int32_t *out_tokens,
                                      int32_t *final_token, uint8_t *is_bonus,
                                      int32_t *row_status, double *p_draft, double *ratio,
                                      double *final_margin, double *tv, double *final_mass) {
  if (topk < 1) return -1;
  return verify_linear_impl(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                            topk, n_accepted, out_tokens, final_token, is_bonus, row_status,
                            p_draft, ratio, final_margin, NULL, tv, final_mass);
}

static int verify_linear_impl(const void *logits, const void *q, int dtype,
                              const int32_t *draft_tokens, const float *temperature,
                              const float *uniforms, int B, int gamma, int V, int topk,
                              int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                              uint8_t *is_bonus, int32_t *row_status, double *p_draft,
                              double *ratio, double *final_margin, double *row_diag,
                              double *tv, double *final_mass) {
  if (B < 0 || gamma < 1 || V < 1 || (dtype != OR_DT_F32 && dtype != OR_DT_BF16)) return -1;
  const int R = gamma + 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    const float Tf = temperature[b];
    const int32_t *tok = draft_tokens + (size_t)b * gamma;
    const float *u = uniforms + (size_t)b * R;
    const size_t lbase = (size_t)b * R * V;
    const size_t qbase = (size_t)b * gamma * V;
    int status = 0;

    if (!temperature_valid(Tf)) status |= OR_ROW_BAD_TEMP;
    for (int i = 0; i < gamma; ++i)
      if (tok[i] < 0 || tok[i] >= V) status |= OR_ROW_BAD_TOKEN;
    for (int i = 0; i < gamma; ++i) {
      if (tok[i] < 0 || tok[i] >= V) continue;
      double qx = load_elem(q, dtype, qbase + (size_t)i * V + tok[i]);
      if (!(qx > 0.0) || isinf(qx)) status |= OR_ROW_BAD_Q;
    }
    for (int i = 0; i < R; ++i)
      if (row_nonfinite(logits, dtype, lbase + (size_t)i * V, V)) status |= OR_ROW_NONFINITE;

    row_status[b] = status;
    if (status) {
      n_accepted[b] = 0;
      for (int j = 0; j < R; ++j) out_tokens[(size_t)b * R + j] = -1;
      final_token[b] = -1;
      is_bonus[b] = 0;
      if (p_draft) for (int i = 0; i < gamma; ++i) p_draft[(size_t)b * gamma + i] = NAN;
      if (ratio) for (int i = 0; i < gamma; ++i) ratio[(size_t)b * gamma + i] = NAN;
      if (final_margin) final_margin[b] = NAN;
      if (tv) tv[b] = NAN;
      if (final_mass) final_mass[b] = NAN;
      continue;
    }

    /* step 2: every target row's distribution (computed in parallel by the
     * target model; here one after the other). */
    double *P = (double *)malloc(sizeof(double) * (size_t)R * V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    for (int i = 0; i < R; ++i)
      target_probs(logits, dtype, lbase + (size_t)i * V, V, (double)Tf, P + (size_t)i * V);

    for (int i = 0; i < gamma; ++i) {
      double px = P[(size_t)i * V + tok[i]];
      double qx = load_elem(q, dtype, qbase + (size_t)i * V + tok[i]);
      double r = px / qx;
      if (r > 1.0) r = 1.0;
      if (p_draft) p_draft[(size_t)b * gamma + i] = px;
      if (ratio) ratio[(size_t)b * gamma + i] = r;
      if (row_diag) {
        double smin = 0.0, sres = 0.0;
        for (int v = 0; v < V; ++v) {
          double pv = P[(size_t)i * V + v];
          double qv = load_elem(q, dtype, qbase + (size_t)i * V + v);
          smin += (pv < qv ? pv : qv);
          sres += (pv > qv ? pv - qv : 0.0);
        }
        row_diag[((size_t)b * gamma + i) * 2 + 0] = smin;
        row_diag[((size_t)b * gamma + i) * 2 + 1] = sres;
      }
    }

    /* step 3: sequential accept test, early stop at the first rejection */
    int k = gamma;
    for (int i = 0; i < gamma; ++i) {
      double px = P[(size_t)i * V + tok[i]];
      double qx = load_elem(q, dtype, qbase + (size_t)i * V + tok[i]);
      double r = px / qx;
      if (r > 1.0) r = 1.0;
      if ((double)u[i] <= r) continue;
      k = i;
      break;
    }

    /* step 4: residual at the rejected row, or the bonus row */
    const double *Pk = P + (size_t)k * V;
    double Z = 0.0;
    if (tv) tv[b] = NAN;
    if (k < gamma) {
      for (int v = 0; v < V; ++v) {
        double d = Pk[v] - load_elem(q, dtype, qbase + (size_t)k * V + v);
        w[v] = d > 0.0 ? d : 0.0;
        Z += w[v];
      }
      if (topk > 0) {
        /* top-k residual: keep the candidates' weights only */
        unsigned char *in_k = (unsigned char *)malloc((size_t)V);
        topk_candidates(Pk, V, topk, in_k);
        double ZK = 0.0;
        for (int v = 0; v < V; ++v) {
          if (!in_k[v]) w[v] = 0.0;
          ZK += w[v];
        }
        if (tv && Z > 0.0) tv[b] = 1.0 - ZK / Z;
        if (!(ZK > 0.0))
          for (int v = 0; v < V; ++v) w[v] = in_k[v] ? Pk[v] : 0.0;
        free(in_k);
      } else if (!(Z > 0.0)) {
        for (int v = 0; v < V; ++v) w[v] = Pk[v];
      }
    } else {
      for (int v = 0; v < V; ++v) w[v] = Pk[v];
    }
    double margin = 0.0, mass = 0.0;
    int fin = cdf_draw(w, V, (double)u[gamma], &margin, &mass);

    n_accepted[b] = k;
    for (int j = 0; j < R; ++j) {
      int32_t t = -1;
      if (j < k) t = tok[j];
      else if (j == k) t = fin;
      out_tokens[(size_t)b * R + j] = t;
    }
    final_token[b] = fin;
    is_bonus[b] = (uint8_t)(k == gamma);
    if (final_margin) final_margin[b] = margin;
    if (final_mass) final_mass[b] = mass;
    free(P);
    free(w);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* token-tree verify                                                          */
/* ------------------------------------------------------------------------ */

/* Arrays, row-major:
 *   logits [B, N, V]: row n is the target distribution after the path to n;
 *   q      [B, N, V]: row n is the draft distribution node n's children were
 *                     drawn from (i.i.d.);
 *   node_tokens int32 [B, N] (entry 0 unused), parent int32 [B, N]
 *   (parent[0] = -1, 0 <= parent[n] < n), temperature [B],
 *   uniforms [B, N] (slot 0 = final draw, slot n = test of node n).
 * Outputs: n_accepted [B]; path_nodes [B, max_depth+1] = 0 then the accepted
 *   nodes, -1 padded; out_tokens [B, max_depth+1] = accepted tokens then the
 *   final token, -1 padded; final_token, is_bonus, row_status [B].
 * Diagnostics (NULL to skip): p_node [B, N] = target probability of node n's
 *   token under its parent's row (before any renormalisation; NaN for n = 0);
 *   test_margin [B] = min |u - r| over the sibling tests that ran (+inf if
 *   none); final_margin [B] as in the linear form; final_mass [B] = the mass
 *   of the final node's residual relative to its target row: the product of
 *   the normalisers of its rejected siblings' renormalisations (1 when none)
 *   times the total of the drawn weights (NaN for a malformed request). */
int specdec_oracle_verify_tree(const void *logits, const void *q, int dtype,
                               const int32_t *node_tokens, const int32_t *parent,
                               const float *temperature, const float *uniforms, int B,
                               int N, int V, int max_depth, int32_t *n_accepted,
                               int32_t *path_nodes, int32_t *out_tokens,
                               int32_t *final_token, uint8_t *is_bonus,
                               int32_t *row_status, double *p_node, double *test_margin,
                               double *final_margin, double *final_mass) {
  if (B < 0 || N < 1 || V < 1 || max_depth < 0 ||
      (dtype != OR_DT_F32 && dtype != OR_DT_BF16))
    return -1;
  const int D1 = max_depth + 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    const float Tf = temperature[b];
    const int32_t *tok = node_tokens + (size_t)b * N;
    const int32_t *par = parent + (size_t)b * N;
    const float *u = uniforms + (size_t)b * N;
    const size_t base = (size_t)b * N * V;
    int status = 0;

    if (!temperature_valid(Tf)) status |= OR_ROW_BAD_TEMP;
    int *depth = (int *)malloc(sizeof(int) * (size_t)N);
    if (par[0] != -1) status |= OR_ROW_BAD_TREE;
    depth[0] = 0;
    for (int n = 1; n < N; ++n) {
      if (par[n] < 0 || par[n] >= n) {
        status |= OR_ROW_BAD_TREE;
        depth[n] = 0;
        continue;
      }
      depth[n] = depth[par[n]] + 1;
      if (depth[n] > max_depth) status |= OR_ROW_BAD_TREE;
    }
    for (int n = 1; n < N; ++n)
      if (tok[n] < 0 || tok[n] >= V) status |= OR_ROW_BAD_TOKEN;
    for (int n = 1; n < N; ++n) {
      if (tok[n] < 0 || tok[n] >= V || par[n] < 0 || par[n] >= n) continue;
      double qx = load_elem(q, dtype, base + (size_t)par[n] * V + tok[n]);
      if (!(qx > 0.0) || isinf(qx)) status |= OR_ROW_BAD_Q;
    }
    for (int n = 0; n < N; ++n)
      if (row_nonfinite(logits, dtype, base + (size_t)n * V, V)) status |= OR_ROW_NONFINITE;
    free(depth);

    row_status[b] = status;
    if (status) {
      n_accepted[b] = 0;
      for (int j = 0; j < D1; ++j) {
        path_nodes[(size_t)b * D1 + j] = -1;
        out_tokens[(size_t)b * D1 + j] = -1;
      }
      final_token[b] = -1;
      is_bonus[b] = 0;
      if (p_node) for (int n = 0; n < N; ++n) p_node[(size_t)b * N + n] = NAN;
      if (test_margin) test_margin[b] = NAN;
      if (final_margin) final_margin[b] = NAN;
      if (final_mass) final_mass[b] = NAN;
      continue;
    }

    double *P = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);

    if (p_node) {
      p_node[(size_t)b * N] = NAN;
      for (int n = 1; n < N; ++n) {
        target_probs(logits, dtype, base + (size_t)par[n] * V, V, (double)Tf, P);
        p_node[(size_t)b * N + n] = P[tok[n]];
      }
    }

    int cur = 0, nacc = 0, bonus = 0;
    /* the tree was checked to be no deeper than max_depth, so the path fits */
    int *path = (int *)malloc(sizeof(int) * (size_t)D1);
    path[0] = 0;
    double tmin = INFINITY;
    double node_mass = 1.0; /* product of the renormalisations at the current node */
    target_probs(logits, dtype, base, V, (double)Tf, P);
    for (;;) {
      int has_child = 0, accepted = -1;
      for (int n = cur + 1; n < N; ++n) {
        if (par[n] != cur) continue;
        has_child = 1;
        const size_t qrow = base + (size_t)cur * V;
        double qt = load_elem(q, dtype, qrow + tok[n]);
        double r = P[tok[n]] / qt;
        if (r > 1.0) r = 1.0;
        double d = fabs((double)u[n] - r);
        if (d < tmin) tmin = d;
        if ((double)u[n] <= r) {
          accepted = n;
          break;
        }
        /* rejected sibling: P <- max(0, P - q_cur) / sum (kept if sum = 0) */
        double Z = 0.0;
        for (int v = 0; v < V; ++v) {
          double x = P[v] - load_elem(q, dtype, qrow + (size_t)v);
          w[v] = x > 0.0 ? x : 0.0;
          Z += w[v];
        }
        if (Z > 0.0) {
          for (int v = 0; v < V; ++v) P[v] = w[v] / Z;
          node_mass *= Z;
        }
      }
      if (accepted >= 0) {
        cur = accepted;
        ++nacc;
        path[nacc] = cur;
        target_probs(logits, dtype, base + (size_t)cur * V, V, (double)Tf, P);
        node_mass = 1.0;
        continue;
      }
      bonus = !has_child;
      break;
    }
    double margin = 0.0, total = 0.0;
    int fin = cdf_draw(P, V, (double)u[0], &margin, &total);

    n_accepted[b] = nacc;
    for (int j = 0; j < D1; ++j) {
      path_nodes[(size_t)b * D1 + j] = (j <= nacc) ? path[j] : -1;
      int32_t t = -1;
      if (j < nacc) t = tok[path[j + 1]];
      else if (j == nacc) t = fin;
      out_tokens[(size_t)b * D1 + j] = t;
    }
    final_token[b] = fin;
    is_bonus[b] = (uint8_t)bonus;
    if (test_margin) test_margin[b] = tmin;
    if (final_margin) final_margin[b] = margin;
    if (final_mass) final_mass[b] = node_mass * total;
    free(P);
    free(w);
    free(path);
  }
  return 0;
}

/* Number of OpenMP threads a parallel region of this library uses. */
/* Threads of the oracle's parallel loops from now on (n >= 1); no effect
 * without OpenMP. */
void specdec_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int specdec_oracle_num_threads(void) {
  int n = 1;
#ifdef _OPENMP
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
#endif
  return n;
}

/* ------------------------------------------------------------------------
 * Philox4x64-10 (SC'11 paper above).  One round maps the counter block
 * (x0, x1, x2, x3) with key (k0, k1) to
 *     (hi(M1 x2) ^ x1 ^ k0,  lo(M1 x2),  hi(M0 x0) ^ x3 ^ k1,  lo(M0 x0))
 * where hi/lo are the halves of the 128-bit product; the key is bumped by the
 * Weyl constants (W0, W1) between rounds; ten rounds.  Word i of a stream
 * that starts from counter c is word i mod 4 of the block for counter
 * c + floor(i / 4) + 1 (256-bit little-endian words; the counter is advanced
 * before each block, as NumPy's Philox does).  Uniform: u = ((w >> 41) + 0.5)
 * * 2^-23, exact in float32, in (0, 1).
 * ------------------------------------------------------------------------ */
static const uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;
static const uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
static const uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull;
static const uint64_t kPhiloxW1 = 0xBB67AE8584CAA73Bull;

static void philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const unsigned __int128 p0 = (unsigned __int128)kPhiloxM0 * x0;
    const unsigned __int128 p1 = (unsigned __int128)kPhiloxM1 * x2;
    const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* counter + add (256-bit, little-endian 64-bit words) */
static void counter_add(const uint64_t c[4], uint64_t add, uint64_t out[4]) {
  uint64_t carry = add;
  for (int i = 0; i < 4; ++i) {
    const uint64_t v = c[i] + carry;
    carry = (v < c[i]) ? 1 : 0;
    out[i] = v;
  }
}

/* Raw words [first, first + n) of the stream (key, counter). */
void specdec_oracle_philox_words(const uint64_t *key, const uint64_t *counter, uint64_t first,
                                 int64_t n, uint64_t *out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t w = first + (uint64_t)i;
    uint64_t c[4], blk[4];
    /* block floor(w / 4) uses counter + floor(w / 4) + 1: add in two steps so
     * that a block index of 2^64 - 1 carries correctly */
    counter_add(counter, w / 4, c);
    counter_add(c, 1, c);
    philox4x64_10(c, key, blk);
    out[i] = blk[w % 4];
  }
}

/* Uniforms of the words [first, first + n). */
void specdec_oracle_philox_uniforms(const uint64_t *key, const uint64_t *counter, uint64_t first,
                                    int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) {
    uint64_t w;
    specdec_oracle_philox_words(key, counter, first + (uint64_t)i, 1, &w);
    out[i] = (float)(((double)(w >> 41) + 0.5) * 0x1p-23);
  }
}

/* ------------------------------------------------------------------------
 * Per-row entropy and path log-probability (the adaptive-draft-length and
 * path-probability passages of the same chapter: entropy = -sum p log p of
 * the target distribution, and log P(path) = sum_i log p(x_i | prefix_i)).
 * ------------------------------------------------------------------------ */

/* entropy[b * R + i] = -sum_v p log p of target row (b, i), natural log;
 * 0 for greedy rows (one-hot), NaN for an invalid temperature or an unusable
 * row. */
void specdec_oracle_row_entropy(const void *logits, int dtype, const float *temperature, int B,
                                int R, int V, double *entropy) {
#pragma omp parallel
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
#pragma omp for schedule(dynamic, 1)
    for (long long row = 0; row < (long long)B * R; ++row) {
      const int b = (int)(row / R);
      const float T = temperature[b];
      const size_t off = (size_t)row * (size_t)V;
      if (!temperature_valid(T) || row_nonfinite(logits, dtype, off, V)) {
        entropy[row] = NAN;
        continue;
      }
      target_probs(logits, dtype, off, V, (double)T, p);
      double h = 0.0;
      for (int v = 0; v < V; ++v)
        if (p[v] > 0.0) h -= p[v] * log(p[v]);
      entropy[row] = h;
    }
    free(p);
  }
}

/* alpha[b * gamma + i] = sum_v min(p_i(v), q_i(v)) for the drafted rows
 * i < gamma of request b: the probability that the speculative sampling test
 * accepts one token drawn from q_i (the first term of Lemma 1 in "Chapter 15:
 * Decoding acceleration", section 15.1.2), the per-position acceptance rate
 * the chapter's adaptive draft length averages.  p_i as in the verify step
 * (one-hot at the first arg-max for a greedy row); q_i as stored, not
 * renormalised.  NaN for an invalid temperature or an unusable target row. */
void specdec_oracle_row_alpha(const void *logits, const void *q, int dtype,
                              const float *temperature, int B, int gamma, int V,
                              double *alpha) {
  const int R = gamma + 1;
#pragma omp parallel
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
#pragma omp for schedule(dynamic, 1)
    for (long long j = 0; j < (long long)B * gamma; ++j) {
      const int b = (int)(j / gamma), i = (int)(j % gamma);
      const float T = temperature[b];
      const size_t loff = ((size_t)b * R + (size_t)i) * (size_t)V;
      const size_t qoff = (size_t)j * (size_t)V;
      if (!temperature_valid(T) || row_nonfinite(logits, dtype, loff, V)) {
        alpha[j] = NAN;
        continue;
      }
      target_probs(logits, dtype, loff, V, (double)T, p);
      double a = 0.0;
      for (int v = 0; v < V; ++v) {
        const double qv = load_elem(q, dtype, qoff + (size_t)v);
        a += (p[v] < qv) ? p[v] : qv;
      }
      alpha[j] = a;
    }
    free(p);
  }
}

/* logprob[b] = sum_{j=0..n_accepted[b]} log p_{row_j}(out_tokens[b, j]) with
 * row_j = j (path_nodes NULL, linear form) or path_nodes[b, j] (tree form);
 * out_tokens and path_nodes have rows of path_len entries.  NaN for a
 * request with a nonzero status, an invalid temperature, an unusable row or
 * a token or node out of range; -inf where a token has probability 0. */
void specdec_oracle_path_logprob(const void *logits, int dtype, const float *temperature,
                                 const int32_t *out_tokens, const int32_t *n_accepted,
                                 const int32_t *path_nodes, const int32_t *row_status, int B,
                                 int R, int V, int path_len, double *logprob) {
#pragma omp parallel
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
      const float T = temperature[b];
      const int k = n_accepted[b];
      double s = 0.0;
      int bad = (row_status && row_status[b] != 0) || !temperature_valid(T) || k < 0 ||
                k >= path_len;
      for (int j = 0; !bad && j <= k; ++j) {
        const int row = path_nodes ? path_nodes[(size_t)b * path_len + j] : j;
        const int tok = out_tokens[(size_t)b * path_len + j];
        if (row < 0 || row >= R || tok < 0 || tok >= V) {
          bad = 1;
          break;
        }
        const size_t off = ((size_t)b * R + (size_t)row) * (size_t)V;
        if (row_nonfinite(logits, dtype, off, V)) {
          bad = 1;
          break;
        }
        target_probs(logits, dtype, off, V, (double)T, p);
        s += log(p[tok]);
      }
      logprob[b] = bad ? NAN : s;
    }
    free(p);
  }
}
