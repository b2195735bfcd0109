/*
 * spec_oracle.c -- plain, slow, double-precision CPU oracle for batched
 * speculative-decoding verification (the Leviathan/Chen accept/reject rule).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Every function follows the definition on the pages directly, with scalar
 * loops in increasing index order and no blocking, fusion or reordering:
 *
 *   [SDE]  "Speculative decoding and EAGLE" (aiengineeringfromscratch.com,
 *          Phase 10 lesson 25): section "The concept" (the K-draft / K+1-verify
 *          step, accept the longest matching prefix, bonus when all match),
 *          section "The exactness rule" (accept x_t if r < p(x_t)/q(x_t), else
 *          sample the residual (p - q)+ / ||(p - q)+||_1 and stop; greedy case
 *          at temperature 0: accept iff argmax(p) == x_t, else emit argmax(p)),
 *          section "Tree attention verification" (verify a candidate tree in one
 *          pass, keep the longest accepted branch), and the worked step function
 *          in section "Make it" (softmax(logits / temperature) for draft and
 *          target rows, one uniform per accept test, a separate draw for the
 *          replacement and for the bonus).
 *   [DVR]  "Speculative decoding: draft, verify, repeat" (Phase 07 lesson 16):
 *          step 1 accept_or_reject (a zero draft probability is accepted),
 *          step 2 residual_dist (max(0, p - q) over the whole row, renormalised),
 *          step 3 the bonus token after all drafts are accepted.
 *   [SOTA] "Speculative Decoding: from idea to SOTA" (mountainai.tech), section 3
 *          "Mathematics": acceptance alpha(x) = min(1, p(x)/q(x)); resampling
 *          p'(x) = max(0, p(x) - q(x)) / sum_x' max(0, p(x') - q(x')); the
 *          theorem P(output = x) = min(p, q) + max(0, p - q) = p.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - uniforms[b,t,0] drives the accept test at position t, uniforms[b,t,1]
 *     the replacement sample at the stopping position (residual if t < K,
 *     bonus if t == K); uniforms[b,K,0] is unused.
 *   - sampling from a weight vector w with total R by a given uniform u is the
 *     inverse CDF in vocabulary order: the smallest v whose running sum
 *     C_v = w_0 + ... + w_v exceeds u*R; if rounding leaves none, the largest
 *     v with w_v > 0.
 *   - residual mass R == 0 at a rejected position falls back to sampling p_t.
 *   - draft probabilities (not logits) are used exactly as given.
 *   - argmax ties go to the lowest index (numpy's argmax, which the pages use).
 *   - tree: the deepest accepted node wins, ties to the smallest node index.
 *   - a sequence whose verification reads an invalid row (NaN, +inf or no
 *     finite entry for a softmax row; NaN for an argmax row) or that has a draft
 *     token outside [0, V) is reported with num_accepted = -1 and all -1 tokens.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* Exact widening of one element (float32 or bfloat16 bits) to double. */
static double orc_elem(const void *base, int dtype, size_t i) {
  if (dtype == ORC_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[i];
}

void orc_widen_row(const void *base, int dtype, size_t offset, int V, double *out) {
  for (int v = 0; v < V; ++v) out[v] = orc_elem(base, dtype, offset + (size_t)v);
}

/* Temperature softmax p_v = exp((z_v - M)/T) / sum_w exp((z_w - M)/T), M = max z
 * ([SDE] "Make it": softmax(logits / temperature)).  Subtracting M changes
 * nothing mathematically; it only keeps exp in range.  Returns 0 on success,
 * 1 if the row contains NaN or +inf or has no finite entry (p is then unset). */
int orc_softmax(const double *z, int V, double T, double *p) {
  double M = -INFINITY;
  for (int v = 0; v < V; ++v) {
    if (isnan(z[v]) || z[v] == INFINITY) return 1;
    if (z[v] > M) M = z[v];
  }
  if (M == -INFINITY) return 1;
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    p[v] = exp((z[v] - M) / T);
    S += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] = p[v] / S;
  return 0;
}

/* Residual weights w_v = max(0, p_v - q_v) over the whole row and their total
 * R = sum_v w_v ([SOTA] section 3, resampling rule; [DVR] step 2). */
double orc_residual(const double *p, const double *q, int V, double *w) {
  double R = 0.0;
  for (int v = 0; v < V; ++v) {
    double d = p[v] - q[v];
    w[v] = d > 0.0 ? d : 0.0;
    R += w[v];
  }
  return R;
}

/* Inverse-CDF draw from weights w (total R) with uniform u: the smallest v with
 * C_v > u*R, C_v the running sum in increasing v.  *gap receives the distance
 * of u*R to the nearer of the two CDF values bracketing the choice, divided by
 * R (how close the draw came to picking a neighbour).  Returns -1 if no weight
 * is positive. */
int orc_icdf(const double *w, int V, double R, double u, double *gap) {
  double target = u * R;
  double C = 0.0, Cprev = 0.0;
  int last_pos = -1;
  for (int v = 0; v < V; ++v) {
    Cprev = C;
    C += w[v];
    if (w[v] > 0.0) last_pos = v;
    if (C > target) {
      if (gap) {
        double a = target - Cprev, b = C - target;
        *gap = (a < b ? a : b) / R;
      }
      return v;
    }
  }
  if (gap) *gap = 0.0;
  return last_pos;
}

/* Accept test at one position ([SDE] "The exactness rule": r < p/q; [DVR]
 * step 1: a zero draft probability is accepted; [SOTA] section 3:
 * alpha = min(1, p/q), and since u < 1 the min is redundant). */
int orc_accept(double a, double c, double u) {
  if (c == 0.0) return 1;
  return u < a / c;
}

/* Index of the first maximum of a row (ties to the lowest index).  Returns -1
 * if the row contains NaN. */
int orc_argmax(const double *z, int V) {
  int best = 0;
  for (int v = 0; v < V; ++v) {
    if (isnan(z[v])) return -1;
    if (z[v] > z[best]) best = v;
  }
  return best;
}

static void orc_fill_invalid(int32_t *out_tokens, int32_t *num_accepted, int width, int b) {
  for (int j = 0; j < width; ++j) out_tokens[(size_t)b * width + j] = -1;
  num_accepted[b] = -1;
}

/* Greedy chain verification ([SDE] "The exactness rule", greedy case):
 * g_t = argmax of target row t; accept x_t while g_t == x_t; at the first
 * mismatch emit g_t and stop; if all K match, emit g_K. */
int orc_verify_greedy(const void *target, int dtype, const int32_t *tokens,
                      int B, int K, int V, int32_t *out_tokens, int32_t *num_accepted) {
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  if (!z) return 2;
  const int W = K + 1;
  for (int b = 0; b < B; ++b) {
    int bad = 0;
    for (int t = 0; t < K; ++t) {
      int x = tokens[(size_t)b * K + t];
      if (x < 0 || x >= V) bad = 1;
    }
    if (bad) { orc_fill_invalid(out_tokens, num_accepted, W, b); continue; }
    for (int j = 0; j < W; ++j) out_tokens[(size_t)b * W + j] = -1;
    int n = 0;
    for (int t = 0; t <= K; ++t) {
      orc_widen_row(target, dtype, ((size_t)b * W + t) * (size_t)V, V, z);
      int g = orc_argmax(z, V);
      if (g < 0) { bad = 1; break; }
      if (t < K && g == tokens[(size_t)b * K + t]) {
        out_tokens[(size_t)b * W + t] = g;
        n = t + 1;
        continue;
      }
      out_tokens[(size_t)b * W + t] = g;
      n = t;
      break;
    }
    if (bad) { orc_fill_invalid(out_tokens, num_accepted, W, b); continue; }
    num_accepted[b] = n;
  }
  free(z);
  return 0;
}

/* Sampling-mode chain verification, one step per sequence ([SDE] "The
 * exactness rule" and "Make it"; [DVR] steps 1-3; [SOTA] section 3).
 *
 * For t = 0..K-1: a = p_t(x_t), c = q_t(x_t); accept iff c == 0 or
 * u[b,t,0] < a/c.  At the first rejection: w = (p_t - q_t)+, R = sum w (R == 0
 * falls back to w = p_t), emit icdf(w, R, u[b,t,1]), num_accepted = t.  If all
 * K are accepted: emit icdf(p_K, sum p_K, u[b,K,1]), num_accepted = K.
 *
 * Diagnostics (optional, may be NULL): near_accept[b] = first t whose accept
 * test had |u - a/c| < tol (else -1); near_cdf[b] = 1 if the replacement draw
 * had a CDF gap below tol; ratio[b*K + t] = a/c at evaluated positions (NaN
 * elsewhere, +inf when c == 0).  Temperature 0 means the greedy rule. */
int orc_verify_sample(const void *target, int target_dtype, const void *draft, int draft_dtype,
                      int draft_is_probs, const int32_t *tokens, const float *uniforms,
                      double T, int B, int K, int V, int32_t *out_tokens, int32_t *num_accepted,
                      int32_t *near_accept, int32_t *near_cdf, double tol, double *ratio) {
  if (T == 0.0) {
    if (near_accept) for (int b = 0; b < B; ++b) near_accept[b] = -1;
    if (near_cdf) for (int b = 0; b < B; ++b) near_cdf[b] = 0;
    return orc_verify_greedy(target, target_dtype, tokens, B, K, V, out_tokens, num_accepted);
  }
  const int W = K + 1;
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  if (!z || !p || !q || !w) { free(z); free(p); free(q); free(w); return 2; }
  for (int b = 0; b < B; ++b) {
    if (near_accept) near_accept[b] = -1;
    if (near_cdf) near_cdf[b] = 0;
    if (ratio) for (int t = 0; t < K; ++t) ratio[(size_t)b * K + t] = NAN;
    int bad = 0;
    for (int t = 0; t < K; ++t) {
      int x = tokens[(size_t)b * K + t];
      if (x < 0 || x >= V) bad = 1;
    }
    if (bad) { orc_fill_invalid(out_tokens, num_accepted, W, b); continue; }
    for (int j = 0; j < W; ++j) out_tokens[(size_t)b * W + j] = -1;
    const float *u = uniforms + (size_t)b * W * 2;
    int stop = K;
    for (int t = 0; t < K; ++t) {
      int x = tokens[(size_t)b * K + t];
      orc_widen_row(target, target_dtype, ((size_t)b * W + t) * (size_t)V, V, z);
      if (orc_softmax(z, V, T, p)) { bad = 1; break; }
      if (draft_is_probs) {
        orc_widen_row(draft, ORC_F32, ((size_t)b * K + t) * (size_t)V, V, q);
        if (isnan(q[x]) || q[x] < 0.0) { bad = 1; break; }
      } else {
        orc_widen_row(draft, draft_dtype, ((size_t)b * K + t) * (size_t)V, V, z);
        if (orc_softmax(z, V, T, q)) { bad = 1; break; }
      }
      double a = p[x], c = q[x];
      double r = (c == 0.0) ? INFINITY : a / c;
      if (ratio) ratio[(size_t)b * K + t] = r;
      if (near_accept && near_accept[b] < 0 && c != 0.0 && fabs((double)u[2 * t] - r) < tol)
        near_accept[b] = t;
      if (orc_accept(a, c, (double)u[2 * t])) {
        out_tokens[(size_t)b * W + t] = x;
        continue;
      }
      double R = orc_residual(p, q, V, w);
      double gap = 1.0;
      int v;
      if (R > 0.0) {
        v = orc_icdf(w, V, R, (double)u[2 * t + 1], &gap);
      } else {
        double S = 0.0;
        for (int i = 0; i < V; ++i) S += p[i];
        v = orc_icdf(p, V, S, (double)u[2 * t + 1], &gap);
      }
      out_tokens[(size_t)b * W + t] = v;
      if (near_cdf && gap < tol) near_cdf[b] = 1;
      stop = t;
      break;
    }
    if (!bad && stop == K) {
      orc_widen_row(target, target_dtype, ((size_t)b * W + K) * (size_t)V, V, z);
      if (orc_softmax(z, V, T, p)) {
        bad = 1;
      } else {
        double S = 0.0, gap = 1.0;
        for (int i = 0; i < V; ++i) S += p[i];
        out_tokens[(size_t)b * W + K] = orc_icdf(p, V, S, (double)u[2 * K + 1], &gap);
        if (near_cdf && gap < tol) near_cdf[b] = 1;
      }
    }
    if (bad) { orc_fill_invalid(out_tokens, num_accepted, W, b); continue; }
    num_accepted[b] = stop;
  }
  free(z); free(p); free(q); free(w);
  return 0;
}

/* The normalised residual row w/R at (b, t) as the sampling rule would build it
 * on a rejection there, and its mass R (R == 0 gives p_t and R = sum p_t).
 * Returns 0, or 1 if a needed row is invalid. */
int orc_residual_row(const void *target, int target_dtype, const void *draft, int draft_dtype,
                     int draft_is_probs, double T, int K, int V, int b, int t,
                     double *out_row, double *out_mass) {
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  int rc = 0;
  if (!z || !p || !q) { rc = 2; goto done; }
  orc_widen_row(target, target_dtype, ((size_t)b * (K + 1) + t) * (size_t)V, V, z);
  if (orc_softmax(z, V, T, p)) { rc = 1; goto done; }
  if (t < K) {
    if (draft_is_probs) {
      orc_widen_row(draft, ORC_F32, ((size_t)b * K + t) * (size_t)V, V, q);
    } else {
      orc_widen_row(draft, draft_dtype, ((size_t)b * K + t) * (size_t)V, V, z);
      if (orc_softmax(z, V, T, q)) { rc = 1; goto done; }
    }
  } else {
    for (int v = 0; v < V; ++v) q[v] = 0.0;
  }
  double R = orc_residual(p, q, V, out_row);
  if (R == 0.0) {
    for (int v = 0; v < V; ++v) { out_row[v] = p[v]; R += p[v]; }
  }
  for (int v = 0; v < V; ++v) out_row[v] = out_row[v] / R;
  *out_mass = R;
done:
  free(z); free(p); free(q);
  return rc;
}

/* Greedy tree verification ([SDE] "Tree attention verification": one target
 * pass over a candidate tree, keep the longest accepted branch; the greedy
 * rule per node).  Node 0 (the root) is accepted; node i >= 1 is accepted iff
 * its parent is accepted and node_tokens[i] == argmax of the parent's row.
 * The deepest accepted node i* (ties to the smallest index) wins; the output
 * is the tokens of the path root -> i* (root excluded), then argmax of i*'s
 * row; num_accepted = depth(i*); out_path lists the node ids of that path
 * (root excluded).  Only accepted nodes' rows are read: a NaN in one makes the
 * sequence invalid.  A node token outside [0, V) never matches.  A malformed
 * topology (parents[0] != -1, parents[i] outside [0, i), depth > max_depth)
 * makes every sequence invalid. */
int orc_verify_tree_greedy(const void *target, int dtype, const int32_t *parents,
                           const int32_t *node_tokens, int B, int N, int V, int max_depth,
                           int32_t *out_tokens, int32_t *num_accepted, int32_t *out_path) {
  const int W = max_depth + 1;
  int *depth = (int *)malloc(sizeof(int) * (size_t)N);
  int *acc = (int *)malloc(sizeof(int) * (size_t)N);
  int *g = (int *)malloc(sizeof(int) * (size_t)N);
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  if (!depth || !acc || !g || !z) { free(depth); free(acc); free(g); free(z); return 2; }
  int topo_ok = (N >= 1 && parents[0] == -1);
  if (topo_ok) depth[0] = 0;
  for (int i = 1; topo_ok && i < N; ++i) {
    if (parents[i] < 0 || parents[i] >= i) { topo_ok = 0; break; }
    depth[i] = depth[parents[i]] + 1;
    if (depth[i] > max_depth) topo_ok = 0;
  }
  for (int b = 0; b < B; ++b) {
    if (!topo_ok) {
      orc_fill_invalid(out_tokens, num_accepted, W, b);
      if (out_path) for (int j = 0; j < W; ++j) out_path[(size_t)b * W + j] = -1;
      continue;
    }
    int bad = 0;
    for (int i = 0; i < N; ++i) { acc[i] = 0; g[i] = -1; }
    acc[0] = 1;
    for (int i = 0; i < N; ++i) {
      if (i > 0) {
        int par = parents[i];
        acc[i] = acc[par] && node_tokens[(size_t)b * N + i] == g[par];
      }
      if (acc[i]) {
        orc_widen_row(target, dtype, ((size_t)b * N + i) * (size_t)V, V, z);
        g[i] = orc_argmax(z, V);
        if (g[i] < 0) { bad = 1; break; }
      }
    }
    if (bad) {
      orc_fill_invalid(out_tokens, num_accepted, W, b);
      if (out_path) for (int j = 0; j < W; ++j) out_path[(size_t)b * W + j] = -1;
      continue;
    }
    int best = 0;
    for (int i = 1; i < N; ++i)
      if (acc[i] && depth[i] > depth[best]) best = i;
    int d = depth[best];
    for (int j = 0; j < W; ++j) out_tokens[(size_t)b * W + j] = -1;
    if (out_path) for (int j = 0; j < W; ++j) out_path[(size_t)b * W + j] = -1;
    int node = best;
    for (int j = d - 1; j >= 0; --j) {
      out_tokens[(size_t)b * W + j] = node_tokens[(size_t)b * N + node];
      if (out_path) out_path[(size_t)b * W + j] = node;
      node = parents[node];
    }
    out_tokens[(size_t)b * W + d] = g[best];
    num_accepted[b] = d;
  }
  free(depth); free(acc); free(g); free(z);
  return 0;
}

/* Tree attention mask ([SDE] "Tree attention verification"; [SOTA] section 6):
 * when the draft proposes a tree, the target checks every node in one pass
 * with a causal mask that follows the tree instead of a line: a node sees only
 * its ancestors (and itself).
 *
 * parents [B, N] (one tree per sequence; parents[b, 0] = -1 and
 * 0 <= parents[b, i] < i), out [B, N, NW] uint32 with NW = ceil(N / 32):
 * bit j % 32 of word j / 32 of row i is 1 iff node j is node i or one of its
 * ancestors.  Computed by walking from i up to the root.  A sequence whose
 * parents break the rule gets status -1 and an all-zero mask; status 0
 * otherwise. */
void orc_tree_mask(const int32_t *parents, int B, int N, uint32_t *out, int32_t *status) {
  const int NW = (N + 31) / 32;
  for (int b = 0; b < B; ++b) {
    const int32_t *par = parents + (size_t)b * N;
    uint32_t *mb = out + (size_t)b * N * NW;
    for (size_t k = 0; k < (size_t)N * NW; ++k) mb[k] = 0u;
    int ok = (N >= 1 && par[0] == -1);
    for (int i = 1; ok && i < N; ++i)
      if (par[i] < 0 || par[i] >= i) ok = 0;
    status[b] = ok ? 0 : -1;
    if (!ok) continue;
    for (int i = 0; i < N; ++i) {
      int node = i;
      while (node >= 0) {
        mb[(size_t)i * NW + node / 32] |= 1u << (node % 32);
        node = par[node];
      }
    }
  }
}

/* Commit on accept ([DVR] "KV rollback": verification writes the drafts'
 * entries to a scratch buffer first and commits only what was accepted, so a
 * rejection rolls the cache back to the accepted length).
 *
 * cache [B, Lmax, E] bytes, lengths [B], scratch [B, N, E] bytes, path [B, W]
 * (the scratch slots to append, in order) or NULL for slots 0, 1, 2, ...,
 * count [B] entries to append.  For each sequence: if count < 0 nothing is
 * appended and new_lengths = lengths; if count > W (with a path), a slot is
 * outside [0, N), or lengths + count > Lmax, nothing is appended and
 * new_lengths = -1; otherwise entry j goes to position lengths + j and
 * new_lengths = lengths + count.  Entries are copied byte for byte. */
void orc_kv_commit(uint8_t *cache, const int32_t *lengths, const uint8_t *scratch, const int32_t *path,
                   const int32_t *count, int B, int Lmax, int N, int W, size_t E, int32_t *new_lengths) {
  for (int b = 0; b < B; ++b) {
    const int n = count[b], L = lengths[b];
    if (n < 0) { new_lengths[b] = L; continue; }
    int ok = (L >= 0 && (long long)L + n <= Lmax && (path == NULL || n <= W));
    for (int j = 0; ok && j < n; ++j) {
      const int s = path ? path[(size_t)b * W + j] : j;
      if (s < 0 || s >= N) ok = 0;
    }
    if (!ok) { new_lengths[b] = -1; continue; }
    for (int j = 0; j < n; ++j) {
      const int s = path ? path[(size_t)b * W + j] : j;
      const uint8_t *src = scratch + ((size_t)b * N + (size_t)s) * E;
      uint8_t *dst = cache + ((size_t)b * Lmax + (size_t)L + (size_t)j) * E;
      for (size_t k = 0; k < E; ++k) dst[k] = src[k];
    }
    new_lengths[b] = L + n;
  }
}

/* Acceptance statistics of a draft against its target, per drafted position
 * ([DVR] step 4: acceptance rate against the divergence between draft and
 * verifier; [SOTA] section 3: a draft token is accepted with probability
 * min(1, p/q), so position t is accepted with probability
 * alpha_t = sum_v min(p_t(v), q_t(v))).
 *
 * For t = 0..K-1 of each sequence, with p_t = softmax(target[b,t]/T) and q_t
 * the draft distribution (softmax(draft[b,t]/T), or the given probabilities):
 *   alpha[b,t] = sum_v min(p, q)
 *   kl[b,t]    = KL(q || p) = sum_{v: q > 0} q log(q / p)   (+inf if some p = 0 < q)
 *   tv[b,t]    = 1/2 sum_v |p - q|
 * Rows that are invalid (NaN, +inf, no finite entry; NaN or negative
 * probabilities) give NaN in all three. */
int orc_row_stats(const void *target, int target_dtype, const void *draft, int draft_dtype, int draft_is_probs,
                  double T, int B, int K, int V, double *alpha, double *kl, double *tv) {
  const int W = K + 1;
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  if (!z || !p || !q) { free(z); free(p); free(q); return 2; }
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < K; ++t) {
      const size_t o = (size_t)b * K + t;
      int bad = 0;
      orc_widen_row(target, target_dtype, ((size_t)b * W + t) * (size_t)V, V, z);
      if (orc_softmax(z, V, T, p)) bad = 1;
      if (draft_is_probs) {
        orc_widen_row(draft, ORC_F32, o * (size_t)V, V, q);
        for (int v = 0; v < V; ++v)
          if (isnan(q[v]) || q[v] < 0.0) bad = 1;
      } else {
        orc_widen_row(draft, draft_dtype, o * (size_t)V, V, z);
        if (orc_softmax(z, V, T, q)) bad = 1;
      }
      if (bad) { alpha[o] = kl[o] = tv[o] = NAN; continue; }
      double a = 0.0, k = 0.0, d = 0.0;
      for (int v = 0; v < V; ++v) {
        a += (p[v] < q[v]) ? p[v] : q[v];
        d += fabs(p[v] - q[v]);
        if (q[v] > 0.0) k += (p[v] > 0.0) ? q[v] * log(q[v] / p[v]) : INFINITY;
      }
      alpha[o] = a;
      kl[o] = k;
      tv[o] = 0.5 * d;
    }
  }
  free(z); free(p); free(q);
  return 0;
}

/* Top-k tree drafting ([SDE] "Make it": an EAGLE-style drafter builds a tree of
 * depth K whose branches are the top-k tokens at each node; exercise 4: the
 * top-3 branches at each depth instead of a chain; [SDE] "EAGLE": K = 4-8
 * candidates per depth).
 *
 * draft [B, N, V]: one draft logit row per tree node; row p is the draft's
 * distribution for the token after node p.  parents [N] (parents[0] = -1,
 * 0 <= parents[i] < i).  The children of node p, taken in increasing index
 * order, receive the tokens of row p in decreasing logit order (equal logits:
 * the smaller vocabulary index first): child r gets the r-th largest.
 * node_logq[b, i] = log q(token) with q = softmax(row p / T), the draft
 * probability of the child's token.  Node 0 gets token -1 and log q 0.  A
 * child whose rank is >= V gets -1 / NaN; so do the children of an invalid row
 * (NaN, +inf, or no finite entry).  A malformed topology (or a node with more
 * than max_children children, the caller's stated bound) gives -1 / NaN for
 * every node of every sequence and returns 1. */
int orc_tree_draft(const void *draft, int dtype, const int32_t *parents, int B, int N, int V, double T,
                   int max_children, int32_t *node_tokens, double *node_logq) {
  int ok = (N >= 1 && parents[0] == -1);
  for (int i = 1; ok && i < N; ++i)
    if (parents[i] < 0 || parents[i] >= i) ok = 0;
  for (int par = 0; ok && par < N; ++par) {   /* the caller's bound on children per node */
    int nchild = 0;
    for (int i = par + 1; i < N; ++i)
      if (parents[i] == par) ++nchild;
    if (nchild > max_children) ok = 0;
  }
  if (!ok) {
    for (size_t k = 0; k < (size_t)B * N; ++k) { node_tokens[k] = -1; node_logq[k] = NAN; }
    return 1;
  }
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  char *taken = (char *)malloc((size_t)V);
  if (!z || !p || !taken) { free(z); free(p); free(taken); return 2; }
  for (int b = 0; b < B; ++b) {
    int32_t *tok = node_tokens + (size_t)b * N;
    double *lq = node_logq + (size_t)b * N;
    tok[0] = -1;
    lq[0] = 0.0;
    for (int par = 0; par < N; ++par) {
      int nchild = 0;
      for (int i = par + 1; i < N; ++i)
        if (parents[i] == par) ++nchild;
      if (nchild == 0) continue;
      orc_widen_row(draft, dtype, ((size_t)b * N + (size_t)par) * (size_t)V, V, z);
      const int bad = orc_softmax(z, V, T, p);
      for (int v = 0; v < V; ++v) taken[v] = 0;
      int r = 0;
      for (int i = par + 1; i < N; ++i) {
        if (parents[i] != par) continue;
        int best = -1;
        if (!bad && r < V) {
          /* the r-th largest: the largest logit not taken yet, smallest index on ties */
          for (int v = 0; v < V; ++v)
            if (!taken[v] && (best < 0 || z[v] > z[best])) best = v;
          if (best >= 0) taken[best] = 1;
        }
        tok[i] = best;
        lq[i] = best < 0 ? NAN : log(p[best]);
        ++r;
      }
    }
  }
  free(z); free(p); free(taken);
  return 0;
}
