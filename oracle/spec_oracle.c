/*
 * spec_oracle.c -- plain fp64 CPU oracle of the batched draft-verification
 * sampler used in speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library to check and to time the CUDA path; the
 * product path never links, loads or calls it.  It shares no code, header,
 * table or constant with the CUDA sources: every rule below is restated here
 * from the pages it cites.
 *
 * Pages cited (by title, then section):
 *   [DVC] "Speculative Decoding: Draft, Verify, and Correct"
 *   [SMB] "Speculative Decoding: How a Small Model Speeds Up a Big One Without
 *          Changing Its Output"
 *   [CRS] "Speculative decoding: why correcting a rejection is not resampling
 *          from the target"
 *   [MNW] "Margins, Not Windows: Training-Free Per-Step Lossy Speculative
 *          Decoding" (AdaptiveSpec)
 *
 * Style: every step is written the slow, obvious way -- fp64 throughout,
 * sequential sums in vocabulary order, no blocking, no fusion.  OpenMP only
 * splits independent batch rows across threads; each row is computed by one
 * thread exactly as the single-threaded loop would.
 *
 * Row status codes (same meaning as the library contract):
 *   0 ok, 1 non-finite logit (NaN or +inf), 2 token id outside [0,V),
 *   3 uniform outside [0,1), 4 bad parent index, 5 a row with no finite logit,
 *   7 temperature not finite and > 0.  When several apply the smallest code
 *   is reported.  Failed rows get accepted_len = -1, num_emitted = 0 and
 *   all-(-1) token outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { O_F32 = 0, O_BF16 = 1 };
enum { O_STOCHASTIC = 0, O_GREEDY = 1 };
enum {
  O_ROW_OK = 0,
  O_ROW_NONFINITE = 1,
  O_ROW_BAD_TOKEN = 2,
  O_ROW_BAD_UNIFORM = 3,
  O_ROW_BAD_PARENT = 4,
  O_ROW_EMPTY = 5,
  O_ROW_BAD_TEMPERATURE = 7
};

/* ---------------------------------------------------------------- inputs */

/* One logit as a double.  bf16 is the upper half of an IEEE binary32. */
static double logit_at(const void *base, int dtype, size_t idx) {
  if (dtype == O_F32) return (double)((const float *)base)[idx];
  uint32_t w = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Flags of one logit row: NaN or +inf anywhere -> bit O_ROW_NONFINITE; every
 * entry -inf (or V == 0) -> bit O_ROW_EMPTY.  -inf alone is a legal mask
 * ([CRS] section 2: a masked event has zero probability). */
static unsigned row_flags(const void *base, int dtype, size_t off, int V) {
  unsigned f = 0;
  int any_finite = 0;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(base, dtype, off + (size_t)v);
    if (isnan(x) || x == INFINITY) f |= 1u << O_ROW_NONFINITE;
    else if (x != -INFINITY) any_finite = 1;
  }
  if (!any_finite) f |= 1u << O_ROW_EMPTY;
  return f;
}

static int lowest_code(unsigned flags) {
  for (int c = 1; c < 32; ++c)
    if (flags & (1u << c)) return c;
  return O_ROW_OK;
}

static int uniform_ok(float u) { return u >= 0.0f && u < 1.0f; }

/* --------------------------------------------------------- distributions */

/* p = softmax(l / T) in fp64: [DVC] "Preserve the distribution you actually
 * intend" and [CRS] section 1 -- the sampling law after temperature and
 * masks, never raw logits.  x = l/T, m = max x, S = sum exp(x - m) summed
 * sequentially in vocabulary order, p_v = exp(x_v - m) / S. */
static void softmax_row(const void *base, int dtype, size_t off, int V,
                        double T, double *p) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(base, dtype, off + (size_t)v) / T;
    if (x > m) m = x;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(base, dtype, off + (size_t)v) / T;
    p[v] = exp(x - m);
    S += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] /= S;
}

/* Inverse CDF of the non-negative weights w at fraction u in [0,1):
 * t = u * total, the token is the smallest v with C_v > t where
 * C_v = w_0 + ... + w_v summed in vocabulary order.  If rounding leaves no
 * such v, the last v with w_v > 0 is taken.  *gap receives the distance of t
 * to the nearer edge of the chosen interval, relative to the total (0 when
 * clamped) -- how far the draw is from choosing a neighbour. */
static int inverse_cdf(const double *w, int V, double u, double *gap) {
  double total = 0.0;
  for (int v = 0; v < V; ++v) total += w[v];
  double t = u * total;
  double c = 0.0;
  for (int v = 0; v < V; ++v) {
    double prev = c;
    c += w[v];
    if (c > t) {
      double g = fmin(t - prev, c - t);
      if (gap) *gap = total > 0.0 ? g / total : 0.0;
      return v;
    }
  }
  if (gap) *gap = 0.0;
  for (int v = V - 1; v >= 0; --v)
    if (w[v] > 0.0) return v;
  return -1;
}

/* Top-k / top-p truncation of a distribution already computed by
 * softmax_row ([DVC] "Preserve the distribution you actually intend": when
 * top-p filtering (or top-k) defines the sampling law, acceptance and
 * correction both use the truncated p, and q must be the truncated law that
 * produced the draft).  Order: temperature (already in p), then top-k, then
 * top-p.
 *   top-k (1 <= k < V): keep the tokens whose logit is >= the k-th largest
 *     logit (ties at the boundary are kept).
 *   top-p (0 < top_p < 1): over the kept tokens, renormalised, take whole
 *     groups of equal logits in descending order until the cumulative mass
 *     reaches top_p; keep the tokens of those groups.
 * p is zeroed outside the kept set and renormalised.  *gap (if not NULL) is
 * lowered to the distance of top_p to the cumulative masses on either side
 * of the chosen boundary -- the margin of the one floating-point decision. */
typedef struct {
  double l;
  double w;
} lw_pair;

static int by_logit_desc(const void *a, const void *b) {
  const double x = ((const lw_pair *)a)->l, y = ((const lw_pair *)b)->l;
  return (x < y) - (x > y);
}

static void truncate_dist(const void *base, int dtype, size_t off, int V, int top_k,
                          double top_p, double *p, lw_pair *tmp, double *gap) {
  const int use_k = top_k >= 1 && top_k < V;
  const int use_p = top_p > 0.0 && top_p < 1.0;
  if (!use_k && !use_p) return;
  for (int v = 0; v < V; ++v) {
    tmp[v].l = logit_at(base, dtype, off + (size_t)v);
    tmp[v].w = p[v];
  }
  qsort(tmp, (size_t)V, sizeof(lw_pair), by_logit_desc);
  double theta = tmp[V - 1].l; /* keep everything */
  int n = V;                   /* kept tokens, a prefix of the sorted list */
  if (use_k) {
    theta = tmp[top_k - 1].l;
    n = top_k;
    while (n < V && tmp[n].l == theta) ++n;
  }
  if (use_p) {
    double mass = 0.0;
    for (int i = 0; i < n; ++i) mass += tmp[i].w;
    double cum = 0.0;
    int i = 0;
    while (i < n) {
      int e = i; /* the group of logits equal to tmp[i].l */
      double g = 0.0;
      while (e < n && tmp[e].l == tmp[i].l) g += tmp[e++].w;
      const double before = cum;
      cum += g / mass;
      if (cum >= top_p || e == n) {
        theta = tmp[i].l;
        if (gap) {
          const double m = fmin(cum - top_p, top_p - before);
          if (m < *gap) *gap = m > 0.0 ? m : 0.0;
        }
        break;
      }
      i = e;
    }
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    if (logit_at(base, dtype, off + (size_t)v) >= theta) S += p[v];
    else p[v] = 0.0;
  }
  for (int v = 0; v < V; ++v) p[v] /= S;
}

/* Lowest index of the largest logit (ties -> lowest index).  Greedy rule of
 * [SMB] "The Guarantee Behind Rejection Sampling": keep the draft iff it is
 * the target's argmax.  Temperature does not move an argmax. */
static int argmax_row(const void *base, int dtype, size_t off, int V,
                      double *best_out) {
  double best = -INFINITY;
  int idx = -1;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(base, dtype, off + (size_t)v);
    if (x > best) {
      best = x;
      idx = v;
    }
  }
  if (best_out) *best_out = best;
  return idx;
}

/* Margin rule of [MNW] section 3 "Margin-based Lossy Verification": promote a
 * mismatched draft when p_t(draft) / p_t(top1) exceeds kappa.  With
 * p_t = softmax(l / T) the ratio is exp((l_d - l_top) / T), so the test is
 * l_d - l_top > T * ln(kappa), evaluated in fp64 (kappa <= 0 disables it). */
static int margin_promotes(double l_d, double l_top, double T, float kappa) {
  if (!(kappa > 0.0f)) return 0;
  return (l_d - l_top) > T * log((double)kappa);
}

/* ------------------------------------------------------------ chain mode */

/*
 * so_verify_chain: one verification step for B independent rows.
 *
 * target [B, K+1, V] and draft [B, K, V] logits (dtype f32 or bf16), row-major.
 * draft_tokens [B, K]; temperature [B] or NULL (=1); u_accept [B, K];
 * u_sample [B, K+1]; kappa: margin threshold for GREEDY (<= 0: strict).
 *
 * STOCHASTIC ([DVC] "Name the two distributions at one prefix", "Verify several
 * proposed tokens in one target pass"; [SMB] "Seeing It in Code"; [CRS]
 * section 2): at position j, y = draft_tokens[b,j], ratio = p_j(y) / q_j(y);
 * accept iff ratio >= 1 or u_accept[b,j] < ratio (the min(1, p/q) test with a
 * strict '<').  Walk j = 0, 1, ... and stop at the first rejection; there the
 * correction is the inverse CDF of r = [p_j - q_j]_+ at u_sample[b,j] (if the
 * residual sums to 0 in fp64 the target law p_j is used instead).  If every
 * draft is accepted, the bonus token is the inverse CDF of p_K at
 * u_sample[b,K] ([DVC] "Verify several ..."; [CRS] section 5).
 *
 * GREEDY ([SMB] "The Guarantee Behind Rejection Sampling" and the greedy step
 * in "Seeing It in Code"; [MNW] section 3): accept iff y == argmax target_j,
 * or the margin rule promotes it; at the first failure emit argmax target_j;
 * if all pass, emit argmax target_K.  draft may be NULL.
 *
 * Outputs: accepted_len [B], out_tokens [B, K+1] (accepted drafts, then the
 * correction or bonus, then -1), num_emitted [B] = accepted_len + 1,
 * row_status [B].  Optional (NULL to skip), STOCHASTIC only, every j < K
 * independent of the walk: p_at_draft, q_at_draft, ratio [B,K]; resid_mass
 * [B,K] = sum_v [p_j - q_j]_+ at the position where the walk stops on a
 * rejection (the residual that is sampled), 0 at every other position.
 * Band bookkeeping (optional): accept_margin [B,K] = |u - min(1, ratio)|;
 * row_margin [B] = smallest decision margin met by the walk (accept margins
 * of positions 0..stop and the sampling gap at the stop; +inf for greedy).
 */
/* so_verify_chain_trunc: so_verify_chain with per-row top-k (top_k[b] <= 0
 * or >= V: off) and top-p (top_p[b] >= 1: off) applied to every p and q of
 * the stochastic walk (see truncate_dist); NULL arrays turn each off.  The
 * top-p boundary margins of the positions the walk reads join row_margin.
 * Greedy mode is unaffected (truncation keeps the argmax). */
void so_verify_chain_trunc(int B, int K, int V, int dtype, int mode,
                           const void *target, const void *draft,
                           const int32_t *draft_tokens, const float *temperature,
                           const float *u_accept, const float *u_sample, float kappa,
                           const int32_t *top_k, const float *top_p,
                           int32_t *accepted_len, int32_t *out_tokens,
                           int32_t *num_emitted, int32_t *row_status,
                           double *p_at_draft, double *q_at_draft, double *ratio_out,
                           double *resid_mass, double *accept_margin,
                           double *row_margin, int nthreads);

void so_verify_chain(int B, int K, int V, int dtype, int mode,
                     const void *target, const void *draft,
                     const int32_t *draft_tokens, const float *temperature,
                     const float *u_accept, const float *u_sample, float kappa,
                     int32_t *accepted_len, int32_t *out_tokens,
                     int32_t *num_emitted, int32_t *row_status,
                     double *p_at_draft, double *q_at_draft, double *ratio_out,
                     double *resid_mass, double *accept_margin,
                     double *row_margin, int nthreads) {
  so_verify_chain_trunc(B, K, V, dtype, mode, target, draft, draft_tokens, temperature,
                        u_accept, u_sample, kappa, NULL, NULL, accepted_len, out_tokens,
                        num_emitted, row_status, p_at_draft, q_at_draft, ratio_out,
                        resid_mass, accept_margin, row_margin, nthreads);
}

void so_verify_chain_trunc(int B, int K, int V, int dtype, int mode,
                           const void *target, const void *draft,
                           const int32_t *draft_tokens, const float *temperature,
                           const float *u_accept, const float *u_sample, float kappa,
                           const int32_t *top_k, const float *top_p,
                           int32_t *accepted_len, int32_t *out_tokens,
                           int32_t *num_emitted, int32_t *row_status,
                           double *p_at_draft, double *q_at_draft, double *ratio_out,
                           double *resid_mass, double *accept_margin,
                           double *row_margin, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double *q = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double *r = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    lw_pair *tmp = (lw_pair *)malloc(sizeof(lw_pair) * (size_t)(V > 0 ? V : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int b = 0; b < B; ++b) {
      const int tk = top_k ? top_k[b] : 0;
      const double tp = top_p ? (double)top_p[b] : 1.0;
      const size_t trow0 = (size_t)b * (size_t)(K + 1);
      const size_t drow0 = (size_t)b * (size_t)K;
      double T = temperature ? (double)temperature[b] : 1.0;
      unsigned flags = 0;
      int T_used = (mode == O_STOCHASTIC) || (kappa > 0.0f);
      if (T_used && !(T > 0.0 && isfinite(T)))
        flags |= 1u << O_ROW_BAD_TEMPERATURE;
      for (int j = 0; j <= K; ++j)
        flags |= row_flags(target, dtype, (trow0 + j) * (size_t)V, V);
      if (mode == O_STOCHASTIC)
        for (int j = 0; j < K; ++j)
          flags |= row_flags(draft, dtype, (drow0 + j) * (size_t)V, V);
      for (int j = 0; j < K; ++j) {
        int32_t y = draft_tokens[drow0 + j];
        if (y < 0 || y >= V) flags |= 1u << O_ROW_BAD_TOKEN;
      }
      if (mode == O_STOCHASTIC) {
        for (int j = 0; j < K; ++j)
          if (!uniform_ok(u_accept[drow0 + j])) flags |= 1u << O_ROW_BAD_UNIFORM;
        for (int j = 0; j <= K; ++j)
          if (!uniform_ok(u_sample[trow0 + j])) flags |= 1u << O_ROW_BAD_UNIFORM;
      }

      for (int j = 0; j <= K; ++j) out_tokens[trow0 + j] = -1;
      if (row_margin) row_margin[b] = INFINITY;
      if (flags) {
        row_status[b] = lowest_code(flags);
        accepted_len[b] = -1;
        num_emitted[b] = 0;
        continue;
      }
      row_status[b] = O_ROW_OK;

      if (mode == O_GREEDY) {
        int stop = K, token = -1;
        for (int j = 0; j < K; ++j) {
          double l_top;
          size_t off = (trow0 + j) * (size_t)V;
          int top = argmax_row(target, dtype, off, V, &l_top);
          int32_t y = draft_tokens[drow0 + j];
          double l_y = logit_at(target, dtype, off + (size_t)y);
          if (y == top || margin_promotes(l_y, l_top, T, kappa)) continue;
          stop = j;
          token = top;
          break;
        }
        if (stop == K)
          token = argmax_row(target, dtype, (trow0 + K) * (size_t)V, V, NULL);
        for (int j = 0; j < stop; ++j) out_tokens[trow0 + j] = draft_tokens[drow0 + j];
        out_tokens[trow0 + stop] = token;
        accepted_len[b] = stop;
        num_emitted[b] = stop + 1;
        continue;
      }

      /* STOCHASTIC: every position's test is evaluated (diagnostics), the
       * walk stops at the first rejection. */
      int stop = -1, token = -1;
      double margin = INFINITY;
      for (int j = 0; j < K; ++j) {
        double tgap = INFINITY; /* top-p boundary margins of this position */
        softmax_row(target, dtype, (trow0 + j) * (size_t)V, V, T, p);
        softmax_row(draft, dtype, (drow0 + j) * (size_t)V, V, T, q);
        truncate_dist(target, dtype, (trow0 + j) * (size_t)V, V, tk, tp, p, tmp, &tgap);
        truncate_dist(draft, dtype, (drow0 + j) * (size_t)V, V, tk, tp, q, tmp, &tgap);
        int32_t y = draft_tokens[drow0 + j];
        double ratio = p[y] / q[y];
        float u = u_accept[drow0 + j];
        int accept = (ratio >= 1.0) || ((double)u < ratio);
        double m_acc = isnan(ratio) ? INFINITY : fabs((double)u - fmin(1.0, ratio));
        double Z = 0.0;
        for (int v = 0; v < V; ++v) {
          r[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
          Z += r[v];
        }
        size_t o = drow0 + j;
        if (p_at_draft) p_at_draft[o] = p[y];
        if (q_at_draft) q_at_draft[o] = q[y];
        if (ratio_out) ratio_out[o] = ratio;
        if (resid_mass) resid_mass[o] = 0.0;
        if (accept_margin) accept_margin[o] = m_acc;
        if (stop >= 0) continue; /* walk already stopped: diagnostics only */
        if (m_acc < margin) margin = m_acc;
        if (tgap < margin) margin = tgap;
        if (!accept) {
          double gap;
          stop = j;
          if (resid_mass) resid_mass[o] = Z;
          token = Z > 0.0 ? inverse_cdf(r, V, (double)u_sample[trow0 + j], &gap)
                          : inverse_cdf(p, V, (double)u_sample[trow0 + j], &gap);
          if (gap < margin) margin = gap;
        }
      }
      if (stop < 0) {
        double gap;
        stop = K;
        softmax_row(target, dtype, (trow0 + K) * (size_t)V, V, T, p);
        double tgap = INFINITY;
        truncate_dist(target, dtype, (trow0 + K) * (size_t)V, V, tk, tp, p, tmp, &tgap);
        if (tgap < margin) margin = tgap;
        token = inverse_cdf(p, V, (double)u_sample[trow0 + K], &gap);
        if (gap < margin) margin = gap;
      }
      for (int j = 0; j < stop; ++j) out_tokens[trow0 + j] = draft_tokens[drow0 + j];
      out_tokens[trow0 + stop] = token;
      accepted_len[b] = stop;
      num_emitted[b] = stop + 1;
      if (row_margin) row_margin[b] = margin;
    }
    free(p);
    free(q);
    free(r);
    free(tmp);
  }
}

/* ------------------------------------------------------------- tree mode */

/*
 * so_verify_tree: greedy (+ margin) verification of a parent-indexed draft
 * tree per row ([SMB] "Beyond Two Models: The EAGLE Line": all branches are
 * verified in one pass and the best branch is kept; [MNW] section 3).
 *
 * target [B, N, V]: row i is the target's next-token logits after node i
 * (node 0 = the root, i.e. the last committed token).  parent [B, N] with
 * parent[b,0] = -1 and 0 <= parent[b,i] < i; node_tokens [B, N] (entry 0
 * ignored).  Node i >= 1 is accepted iff its parent is accepted and its token
 * is argmax target[parent] or the margin rule promotes it.  The kept branch
 * is the deepest accepted node (depth = edges from the root; ties -> lowest
 * node index).  Emitted: the tokens along that root path, then argmax of the
 * target row of the deepest node.
 *
 * Outputs: accepted_len [B] (depth), path_nodes [B, N] (node ids of the path
 * without the root, -1 padded), out_tokens [B, N], num_emitted [B],
 * row_status [B].
 */
void so_verify_tree(int B, int N, int V, int dtype, const void *target,
                    const int32_t *parent, const int32_t *node_tokens,
                    const float *temperature, float kappa,
                    int32_t *accepted_len, int32_t *path_nodes,
                    int32_t *out_tokens, int32_t *num_emitted,
                    int32_t *row_status, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    int *top = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    double *l_top = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    char *acc = (char *)malloc((size_t)(N > 0 ? N : 1));
    int *depth = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int b = 0; b < B; ++b) {
      const size_t row0 = (size_t)b * (size_t)N;
      double T = temperature ? (double)temperature[b] : 1.0;
      unsigned flags = 0;
      if (kappa > 0.0f && !(T > 0.0 && isfinite(T)))
        flags |= 1u << O_ROW_BAD_TEMPERATURE;
      for (int i = 0; i < N; ++i)
        flags |= row_flags(target, dtype, (row0 + i) * (size_t)V, V);
      if (N > 0 && parent[row0] != -1) flags |= 1u << O_ROW_BAD_PARENT;
      for (int i = 1; i < N; ++i) {
        int32_t pa = parent[row0 + i];
        if (pa < 0 || pa >= i) flags |= 1u << O_ROW_BAD_PARENT;
        int32_t t = node_tokens[row0 + i];
        if (t < 0 || t >= V) flags |= 1u << O_ROW_BAD_TOKEN;
      }
      for (int i = 0; i < N; ++i) {
        path_nodes[row0 + i] = -1;
        out_tokens[row0 + i] = -1;
      }
      if (flags || N == 0) {
        row_status[b] = N == 0 ? O_ROW_EMPTY : lowest_code(flags);
        accepted_len[b] = -1;
        num_emitted[b] = 0;
        continue;
      }
      row_status[b] = O_ROW_OK;
      for (int i = 0; i < N; ++i)
        top[i] = argmax_row(target, dtype, (row0 + i) * (size_t)V, V, &l_top[i]);
      acc[0] = 1;
      depth[0] = 0;
      int best = 0;
      for (int i = 1; i < N; ++i) {
        int pa = parent[row0 + i];
        int t = node_tokens[row0 + i];
        double l_t = logit_at(target, dtype, (row0 + pa) * (size_t)V + (size_t)t);
        int ok = (t == top[pa]) || margin_promotes(l_t, l_top[pa], T, kappa);
        acc[i] = acc[pa] && ok;
        depth[i] = depth[pa] + 1;
        if (acc[i] && depth[i] > depth[best]) best = i;
      }
      int d = depth[best];
      for (int n = best, k = d - 1; k >= 0; n = parent[row0 + n], --k) {
        path_nodes[row0 + k] = n;
        out_tokens[row0 + k] = node_tokens[row0 + n];
      }
      out_tokens[row0 + d] = top[best];
      accepted_len[b] = d;
      num_emitted[b] = d + 1;
    }
    free(top);
    free(l_top);
    free(acc);
    free(depth);
  }
}

/* ------------------------------------------------------------- rollback */

/*
 * so_rollback_lengths: KV-cache lengths that agree with the emitted tokens
 * ([DVC] "Speculation needs cache rollback"; [SMB] "Where Speculative
 * Decoding Disappoints"; [CRS] section 5).
 *
 * kv_len_in[b] counts the cache entries before the verify pass.  The pass fed
 * the last emitted token and the drafts, so the entries of the last token and
 * of every accepted draft are valid; the new correction/bonus token has no
 * entry yet.  Emission is cut after the first eos_id (kept) and so that the
 * sequence (kv_len_in + 1 tokens before the step) does not exceed max_len[b]
 * (NULL: no limit).  With n tokens kept and a accepted drafts:
 * committed = kv_len_in + 1 + min(n, a).  Rows with accepted_len < 0 (a failed
 * verify) keep kv_len_in and emit nothing.
 */
void so_rollback_lengths(int B, int max_emit, const int32_t *kv_len_in,
                         const int32_t *accepted_len, const int32_t *num_emitted_in,
                         const int32_t *out_tokens, int32_t eos_id,
                         const int32_t *max_len, int32_t *committed_kv_len,
                         int32_t *num_emitted_out) {
  for (int b = 0; b < B; ++b) {
    int a = accepted_len[b];
    if (a < 0) {
      committed_kv_len[b] = kv_len_in[b];
      num_emitted_out[b] = 0;
      continue;
    }
    int n = num_emitted_in[b];
    if (n > max_emit) n = max_emit;
    if (eos_id >= 0)
      for (int e = 0; e < n; ++e)
        if (out_tokens[(size_t)b * (size_t)max_emit + e] == eos_id) {
          n = e + 1;
          break;
        }
    if (max_len) {
      long room = (long)max_len[b] - ((long)kv_len_in[b] + 1);
      if (room < 0) room = 0;
      if (n > room) n = (int)room;
    }
    committed_kv_len[b] = kv_len_in[b] + 1 + (n < a ? n : a);
    num_emitted_out[b] = n;
  }
}

/* -------------------------------------------------- DRIFT residuals */

/*
 * so_drift_residuals: the free supervision signal of [DRIFT] "DRIFT:
 * Gradient-Free Draft Recalibration From Verification Feedback" (the residual
 * paragraph): at every drafted position j < K of row b, restrict the target
 * and draft distributions to a shared support of m tokens and take the
 * target log-probability minus the draft log-probability there.
 * Reading: the support is the m tokens of highest target probability (ties
 * to the lower index), listed in that order; the log-probabilities are those
 * of the full temperature-scaled distributions, natural log.  A draft
 * probability of 0 (a masked logit) gives +inf.  Rows failing the input
 * checks (status 1, 5 or 7, as in verification) get support -1 and NaN.
 * support [B*K*m] int32, residual [B*K*m] float, row_status [B].
 */
void so_drift_residuals(int B, int K, int V, int dtype, const void *target, const void *draft,
                        const float *temperature, int m, int32_t *support, float *residual,
                        int32_t *row_status, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int b = 0; b < B; ++b) {
    const double T = temperature ? (double)temperature[b] : 1.0;
    unsigned flags = 0;
    if (!(T > 0.0) || isinf(T)) flags |= 1u << O_ROW_BAD_TEMPERATURE;
    for (int j = 0; j < K; ++j) {
      flags |= row_flags(target, dtype, ((size_t)b * (K + 1) + j) * (size_t)V, V);
      flags |= row_flags(draft, dtype, ((size_t)b * K + j) * (size_t)V, V);
    }
    row_status[b] = lowest_code(flags);
    unsigned char *taken = (unsigned char *)calloc((size_t)V, 1);
    double *lp = (double *)malloc(sizeof(double) * (size_t)V);
    double *lq = (double *)malloc(sizeof(double) * (size_t)V);
    for (int j = 0; j < K; ++j) {
      int32_t *sup = support + ((size_t)b * K + j) * (size_t)m;
      float *res = residual + ((size_t)b * K + j) * (size_t)m;
      if (flags) {
        for (int i = 0; i < m; ++i) {
          sup[i] = -1;
          res[i] = NAN;
        }
        continue;
      }
      const size_t to = ((size_t)b * (K + 1) + j) * (size_t)V;
      const size_t dof = ((size_t)b * K + j) * (size_t)V;
      /* log-softmax of l / T, each: x = l / T, m = max x, log S = log sum exp(x - m) */
      for (int pass = 0; pass < 2; ++pass) {
        const void *base = pass == 0 ? target : draft;
        const size_t off = pass == 0 ? to : dof;
        double *out = pass == 0 ? lp : lq;
        double mx = -INFINITY;
        for (int v = 0; v < V; ++v) {
          const double xs = logit_at(base, dtype, off + (size_t)v) / T;
          if (xs > mx) mx = xs;
        }
        double S = 0.0;
        for (int v = 0; v < V; ++v) {
          const double xs = logit_at(base, dtype, off + (size_t)v) / T;
          if (xs != -INFINITY) S += exp(xs - mx);
        }
        const double lS = log(S);
        for (int v = 0; v < V; ++v) {
          const double xs = logit_at(base, dtype, off + (size_t)v) / T;
          out[v] = xs == -INFINITY ? -INFINITY : (xs - mx) - lS;
        }
      }
      /* the m largest target logits, one scan per rank, lower index first */
      memset(taken, 0, (size_t)V);
      for (int i = 0; i < m; ++i) {
        int best = -1;
        double bv = 0.0;
        for (int v = 0; v < V; ++v) {
          if (taken[v]) continue;
          const double x = logit_at(target, dtype, to + (size_t)v);
          if (best < 0 || x > bv) {
            best = v;
            bv = x;
          }
        }
        if (best < 0) { /* m > V */
          sup[i] = -1;
          res[i] = NAN;
          continue;
        }
        taken[best] = 1;
        sup[i] = best;
        res[i] = (float)(lp[best] - lq[best]);
      }
    }
    free(taken);
    free(lp);
    free(lq);
  }
}

/* ------------------------------------------------------ KV compaction */

/*
 * so_kv_compact_tree: keep the KV entries of the accepted root path of a
 * verified draft tree ([DVC] "Speculation needs cache rollback": keep the
 * cache for the accepted prefix; [SMB] "Where Speculative Decoding
 * Disappoints": rejected drafts' keys and values must be rewound).
 *
 * Cache layout (bytes): entry (plane p, row b, token slot s) starts at
 * p*plane_stride + b*row_stride + s*tok_stride and is E bytes long.  The
 * verify pass wrote tree node i of row b at slot kv_len_in[b] + i (node 0 is
 * the root, the last committed token).  With a = accepted_len[b] and root
 * path nodes path[b][0..a-1], the entry of path[b][k] moves to slot
 * kv_len_in[b] + 1 + k.  Defined out of place: all sources are read before
 * any destination is written.  A row whose path is not strictly increasing
 * within [1, N), or whose slots leave [0, S_max), is left untouched and gets
 * status 4; a < 0 (a failed verify) is a no-op with status 0.
 */
void so_kv_compact_tree(int B, int N, int planes, long long S_max, long long E,
                        unsigned char *kv, long long plane_stride, long long row_stride,
                        long long tok_stride, const int32_t *kv_len_in,
                        const int32_t *accepted_len, const int32_t *path_nodes,
                        int32_t *row_status) {
  unsigned char *tmp = (unsigned char *)malloc((size_t)(E > 0 ? E : 1) * (size_t)(N > 0 ? N : 1));
  for (int b = 0; b < B; ++b) {
    const int a = accepted_len[b];
    const long long base = kv_len_in[b];
    int ok = 1;
    if (a > 0) {
      if (a > N - 1 || base < 0 || base + N > S_max) ok = 0;
      int prev = 0;
      for (int k = 0; ok && k < a; ++k) {
        const int n = path_nodes[(size_t)b * N + k];
        if (n <= prev || n >= N) ok = 0;
        prev = n;
      }
    }
    row_status[b] = ok ? 0 : 4;
    if (!ok || a <= 0) continue;
    for (int p = 0; p < planes; ++p) {
      unsigned char *row = kv + (size_t)p * plane_stride + (size_t)b * row_stride;
      for (int k = 0; k < a; ++k)
        memcpy(tmp + (size_t)k * E, row + (size_t)(base + path_nodes[(size_t)b * N + k]) * tok_stride, (size_t)E);
      for (int k = 0; k < a; ++k)
        memcpy(row + (size_t)(base + 1 + k) * tok_stride, tmp + (size_t)k * E, (size_t)E);
    }
  }
  free(tmp);
}

/* ------------------------------------------------- AdaptiveSpec tree policy */

/*
 * so_adaptive_policy: one step of the per-sequence draft-tree shape policy of
 * [MNW] "Method", dynamic draft tree-shaping.  For each row:
 *   a       = accepted_len / depth (0 when depth <= 0; clamped to [0, 1]):
 *             the fraction of the verified draft depth that was accepted
 *   ema     = alpha * a + (1 - alpha) * ema            (rolling acceptance)
 *   zero    = accepted_len == 0 ? zero + 1 : 0
 *   if zero >= breaker: shape = start, ema = ema0, zero = 0  (circuit breaker)
 *   else: dcs = clamp(p1 * ema / divisor, 0, 1)    (draft confidence score;
 *         p1 = the draft's top-1 probability, clamped to [0, 1], NaN -> 0)
 *         shape[i] = floor(lo[i] + dcs * (hi[i] - lo[i]) + 0.5)
 *   with shape = (nsteps, top-k, ndt), lo = the shallow-wide end and hi = the
 *   deep-narrow end ((3, 4, 4) and (7, 1, 8) on the page): depth and draft
 *   tokens grow with dcs, branching with 1 - dcs.
 * fp64, each operation rounded separately in the order written.
 */
void so_adaptive_policy(int B, double alpha, double divisor, const int32_t *lo,
                        const int32_t *hi, const int32_t *start, double ema0, int breaker,
                        const int32_t *accepted_len, const int32_t *depth,
                        const float *draft_top1, double *ema, int32_t *zero_run,
                        int32_t *shape) {
  for (int b = 0; b < B; ++b) {
    double a = 0.0;
    if (depth[b] > 0) a = (double)accepted_len[b] / (double)depth[b];
    if (!(a >= 0.0)) a = 0.0;
    if (a > 1.0) a = 1.0;
    const double e = alpha * a + (1.0 - alpha) * ema[b];
    int32_t z = accepted_len[b] == 0 ? zero_run[b] + 1 : 0;
    if (z >= breaker) {
      ema[b] = ema0;
      zero_run[b] = 0;
      for (int i = 0; i < 3; ++i) shape[(size_t)b * 3 + i] = start[i];
      continue;
    }
    ema[b] = e;
    zero_run[b] = z;
    double p1 = (double)draft_top1[b];
    if (!(p1 >= 0.0)) p1 = 0.0;
    if (p1 > 1.0) p1 = 1.0;
    double dcs = p1 * e / divisor;
    if (!(dcs >= 0.0)) dcs = 0.0;
    if (dcs > 1.0) dcs = 1.0;
    for (int i = 0; i < 3; ++i)
      shape[(size_t)b * 3 + i] = (int32_t)floor((double)lo[i] + dcs * (double)(hi[i] - lo[i]) + 0.5);
  }
}

/* ----------------------------------------------------------- cost model */

/* Expected tokens per verification cycle under a constant acceptance rate
 * alpha and gamma drafts: the sum of the tail probabilities
 * P(at least i retained) = alpha^i for i = 0..gamma ([CRS] section 6; the
 * same 1 + a + ... + a^k of [DVC] "When is drafting worth it?"). */
double so_expected_tokens(double alpha, int gamma) {
  double E = 0.0, a = 1.0;
  for (int i = 0; i <= gamma; ++i) {
    E += a;
    a *= alpha;
  }
  return E;
}

/* Speedup of [CRS] sections 6-7: E / (g + c * gamma), g = verification cost
 * in target steps (1 in the simple model), c = cost of one draft token. */
double so_speedup(double alpha, int gamma, double c, double g) {
  return so_expected_tokens(alpha, gamma) / (g + c * (double)gamma);
}

int so_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
