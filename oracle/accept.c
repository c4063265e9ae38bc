/*
 * accept.c -- rejection-sampling acceptance along the temporal order.
 * TEST INFRASTRUCTURE ONLY (see simsd_oracle.h).
 *
 * SimSD (gist.science, paper 2606.02544), "Speculative Decoding Pipeline",
 * acceptance: standard rejection sampling is applied along the temporal
 * order the draft induced, and the longest accepted prefix is committed.
 * "Standard" is read as the textbook speculative-sampling rule:
 *   p = softmax(target logits), q = softmax(draft logits) of the same slot;
 *   step t (t = 1..B) tests the slot k whose label tau(k) = t;
 *   the draft token x is accepted with probability min(1, p(x)/q(x)),
 *   i.e. iff u * q(x) < p(x) for a uniform u in [0,1);
 *   at the first rejection a token is drawn from norm(max(0, p - q)) by
 *   inverse CDF, and the walk stops.
 * Readings: no bonus token when every step is accepted (the layout has no
 * slot after D~_B); u[t-1] tests step t and u[B] draws the residual; the
 * accept comparison is made in fp32 (the kernel's precision) on p(x), q(x)
 * computed in fp64 and rounded to fp32, with u the given fp32 value.
 */
#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include "simsd_oracle.h"

/* log(sum_v exp(x_v)), fp64, max-shifted. */
static double log_sum_exp(const double *x, int V) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (x[v] > m) m = x[v];
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(x[v] - m);
  return m + log(s);
}

double oracle_residual(int V, const double *tl, const double *dl, double *r) {
  const double lse_p = log_sum_exp(tl, V);
  const double lse_q = log_sum_exp(dl, V);
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    double pv = exp(tl[v] - lse_p), qv = exp(dl[v] - lse_q);
    r[v] = pv > qv ? pv - qv : 0.0;
    S += r[v];
  }
  if (S == 0.0) { /* p == q: the residual is empty, draw from p itself */
    for (int v = 0; v < V; ++v) { r[v] = exp(tl[v] - lse_p); S += r[v]; }
  }
  return S;
}

static int accept_one(int B, int first, int V, const double *target, const double *draft,
                      const int *draft_tokens, const int *tau, const float *u,
                      int *n_accept, int *token, int *pos,
                      double *accept_margin, double *resample_margin) {
  int *slot_of_step = (int *)malloc(sizeof(int) * (size_t)B);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  if (!slot_of_step || !r) { free(slot_of_step); free(r); return ORACLE_ERR_ARG; }
  for (int k = 0; k < B; ++k) slot_of_step[tau[k] - 1] = k;
  for (int k = 0; k < B; ++k)
    if (accept_margin) accept_margin[k] = -1.0;
  if (resample_margin) *resample_margin = -1.0;

  *n_accept = B;
  *token = -1;
  *pos = -1;
  /* steps before `first` belong to positions decided in earlier passes of
     the block: counted as accepted, not tested again */
  for (int t = first; t <= B; ++t) {
    const int k = slot_of_step[t - 1];
    const double *tl = target + (size_t)k * V;
    const double *dl = draft + (size_t)k * V;
    const int x = draft_tokens[k];
    const double lse_p = log_sum_exp(tl, V);
    const double lse_q = log_sum_exp(dl, V);
    const double px = exp(tl[x] - lse_p);
    const double qx = exp(dl[x] - lse_q);
    const float uf = u[t - 1];
    const int accepted = (uf * (float)qx) < (float)px;
    if (accept_margin)
      accept_margin[k] = px > 0.0 ? fabs((double)uf * qx - px) / px
                                  : ((double)uf * qx > 0.0 ? INFINITY : 0.0);
    if (accepted) continue;

    /* first rejection: draw from norm(max(0, p - q)) with u[B] */
    *n_accept = t - 1;
    *pos = k;
    const double S = oracle_residual(V, tl, dl, r);
    const double U = (double)u[B] * S;
    int chosen = -1;
    double below = 0.0, c = 0.0;
    for (int v = 0; v < V; ++v) {
      below = c;
      c += r[v];
      if (c > U) { chosen = v; break; }
    }
    if (chosen < 0) { /* rounding left U past the total: last positive bin */
      for (int v = V - 1; v >= 0; --v)
        if (r[v] > 0.0) { chosen = v; break; }
      below = U;
      c = U;
    }
    *token = chosen;
    if (resample_margin) {
      double d1 = U - below, d2 = c - U;
      *resample_margin = (d1 < d2 ? d1 : d2) / S;
    }
    break;
  }
  free(slot_of_step);
  free(r);
  return ORACLE_OK;
}

/* First step of sequence b's walk: first_step[b], or 1 without the array. */
static int first_of(const int *first_step, int b) { return first_step ? first_step[b] : 1; }

int oracle_accept(int batch, int V, const int *cu_B, const double *target,
                  const double *draft, const int *draft_tokens,
                  const int *tau, const float *uniforms, int u_stride,
                  const int *first_step, int *n_accept, int *token, int *pos,
                  double *accept_margin, double *resample_margin,
                  int n_threads) {
  if (batch < 0 || V < 1 || !cu_B || !target || !draft || !draft_tokens ||
      !tau || !uniforms || !n_accept || !token || !pos)
    return ORACLE_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    int B = cu_B[b + 1] - cu_B[b];
    if (B < 1 || u_stride < B + 1) return ORACLE_ERR_ARG;
    if (first_of(first_step, b) < 1 || first_of(first_step, b) > B + 1) return ORACLE_ERR_ARG;
    if (!oracle_tau_is_permutation(B, tau + cu_B[b])) return ORACLE_ERR_TAU;
    for (int k = 0; k < B; ++k) {
      int x = draft_tokens[cu_B[b] + k];
      if (x < 0 || x >= V) return ORACLE_ERR_ARG;
    }
  }
  int rc = ORACLE_OK;
  const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt) reduction(max : rc)
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_B[b];
    const int B = cu_B[b + 1] - s0;
    int r = accept_one(B, first_of(first_step, b), V, target + (size_t)s0 * V,
                       draft + (size_t)s0 * V,
                       draft_tokens + s0, tau + s0,
                       uniforms + (size_t)b * u_stride, &n_accept[b], &token[b],
                       &pos[b], accept_margin ? accept_margin + s0 : NULL,
                       resample_margin ? resample_margin + b : NULL);
    if (r > rc) rc = r;
  }
  return rc;
}

/* Greedy verification (the acceptance variant with temperature -> 0): step t
 * tests slot k = tau^-1(t) and accepts iff its draft token equals the
 * target's most likely token a_k = argmax_v target_k(v) (the smallest index
 * among equal maxima).  At the first rejection the token is a_k and the walk
 * stops; no uniform is read and the draft logits play no part. */
int oracle_accept_greedy(int batch, int V, const int *cu_B, const double *target,
                         const int *draft_tokens, const int *tau, const int *first_step,
                         int *n_accept, int *token, int *pos) {
  if (batch < 0 || V < 1 || !cu_B || !target || !draft_tokens || !tau || !n_accept ||
      !token || !pos)
    return ORACLE_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_B[b], B = cu_B[b + 1] - s0;
    if (B < 1) return ORACLE_ERR_ARG;
    if (first_of(first_step, b) < 1 || first_of(first_step, b) > B + 1) return ORACLE_ERR_ARG;
    if (!oracle_tau_is_permutation(B, tau + s0)) return ORACLE_ERR_TAU;
    n_accept[b] = B;
    token[b] = -1;
    pos[b] = -1;
    for (int t = first_of(first_step, b); t <= B; ++t) {
      int k = 0;
      while (tau[s0 + k] != t) ++k;
      const double *row = target + (size_t)(s0 + k) * V;
      int a = 0;
      for (int v = 1; v < V; ++v)
        if (row[v] > row[a]) a = v;
      if (draft_tokens[s0 + k] == a) continue;
      n_accept[b] = t - 1;
      token[b] = a;
      pos[b] = k;
      break;
    }
  }
  return ORACLE_OK;
}

/* Sample matching (Spiffy's verification, read for one slot per step): step
 * t draws the target's own token y_t from p_k by inverse CDF with u[t-1] (the
 * smallest v whose running mass exceeds u[t-1]; the last v with p > 0 if
 * rounding leaves none) and accepts iff y_t equals the draft token; the
 * first rejection emits y_t and stops.  Every emitted token is a sample of
 * p_k; a step accepts with probability p_k(x).  u[B] is not used. */
int oracle_accept_match(int batch, int V, const int *cu_B, const double *target,
                        const int *draft_tokens, const int *tau, const float *uniforms,
                        int u_stride, const int *first_step, int *n_accept, int *token,
                        int *pos) {
  if (batch < 0 || V < 1 || !cu_B || !target || !draft_tokens || !tau || !uniforms ||
      !n_accept || !token || !pos)
    return ORACLE_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_B[b], B = cu_B[b + 1] - s0;
    if (B < 1 || u_stride < B) return ORACLE_ERR_ARG;
    if (first_of(first_step, b) < 1 || first_of(first_step, b) > B + 1) return ORACLE_ERR_ARG;
    if (!oracle_tau_is_permutation(B, tau + s0)) return ORACLE_ERR_TAU;
    n_accept[b] = B;
    token[b] = -1;
    pos[b] = -1;
    for (int t = first_of(first_step, b); t <= B; ++t) {
      int k = 0;
      while (tau[s0 + k] != t) ++k;
      const double *row = target + (size_t)(s0 + k) * V;
      const double lse = log_sum_exp(row, V);
      const double U = (double)uniforms[(size_t)b * u_stride + t - 1];
      int y = -1, last = -1;
      double c = 0.0;
      for (int v = 0; v < V; ++v) {
        const double pv = exp(row[v] - lse);
        if (pv > 0.0) last = v;
        c += pv;
        if (y < 0 && c > U) y = v;
      }
      if (y < 0) y = last;
      if (draft_tokens[s0 + k] == y) continue;
      n_accept[b] = t - 1;
      token[b] = y;
      pos[b] = k;
      break;
    }
  }
  return ORACLE_OK;
}

/* The draft-side step (the step before the layout): each open slot k of a
 * sequence samples its draft token x_k from q_k = softmax(draft row k) by
 * inverse CDF with u[k] (the smallest v whose running mass exceeds u[k];
 * the last v with q > 0 if rounding leaves none), and the step labels order
 * the open slots by the draft's confidence in each row, max_v q_k(v), most
 * confident first, equal confidences in position order.  The pages leave
 * the ordering rule open.  The confidence is the row's, not the sampled
 * token's: an order chosen on the samples would make the token tested at
 * a step no longer a draw from q, and the walk's rejection sampling would
 * stop reproducing the target's distribution.
 * Within a block (the blockwise loop), the first decided[b] steps belong to
 * positions decided in earlier passes: a slot k with tau_prev(k) <=
 * decided[b] keeps its token (draft_tokens is read there) and its label;
 * the open slots take the labels decided[b]+1 .. B in confidence order.
 * decided == NULL: every slot is open (tau_prev is then not read).
 * confidence[k] is -1 for a decided slot. */
int oracle_draft_step(int batch, int V, const int *cu_B, const double *draft,
                      const float *uniforms, int u_stride, const int *decided,
                      const int *tau_prev, int *draft_tokens, int *tau, double *confidence) {
  if (batch < 0 || V < 1 || !cu_B || !draft || !uniforms || !draft_tokens || !tau ||
      !confidence || (decided && !tau_prev))
    return ORACLE_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_B[b], B = cu_B[b + 1] - s0;
    const int d = decided ? decided[b] : 0;
    if (B < 1 || u_stride < B || d < 0 || d > B) return ORACLE_ERR_ARG;
    if (decided && !oracle_tau_is_permutation(B, tau_prev + s0)) return ORACLE_ERR_TAU;
    for (int k = 0; k < B; ++k) {
      if (decided && tau_prev[s0 + k] <= d) {   /* decided: keep token and label */
        tau[s0 + k] = tau_prev[s0 + k];
        confidence[s0 + k] = -1.0;
        continue;
      }
      const double *row = draft + (size_t)(s0 + k) * V;
      const double lse = log_sum_exp(row, V);
      const double U = (double)uniforms[(size_t)b * u_stride + k];
      int y = -1, last = -1;
      double c = 0.0, qmax = 0.0;
      for (int v = 0; v < V; ++v) {
        const double qv = exp(row[v] - lse);
        if (qv > 0.0) last = v;
        if (qv > qmax) qmax = qv;
        c += qv;
        if (y < 0 && c > U) y = v;
      }
      if (y < 0) y = last;
      draft_tokens[s0 + k] = y;
      confidence[s0 + k] = qmax;
    }
    /* an open slot's label: d + 1 + the number of open slots before it */
    for (int k = 0; k < B; ++k) {
      if (confidence[s0 + k] < 0.0) continue;
      int before = 0;
      for (int j = 0; j < B; ++j) {
        const double cj = confidence[s0 + j], ck = confidence[s0 + k];
        if (cj < 0.0) continue;
        if (cj > ck || (cj == ck && j < k)) ++before;
      }
      tau[s0 + k] = d + before + 1;
    }
  }
  return ORACLE_OK;
}

/* Commit after a pass of the blockwise loop (SimSD "Speculative Decoding
 * Pipeline": the longest accepted prefix is committed and the process
 * repeats; "Contributions": KV cache and blockwise decoding).  For sequence
 * b with the pass's walk (n_accept, token, pos):
 *   - the positions with tau <= n_accept are decided with the tokens the
 *     pass's data section held (block_tokens);
 *   - a rejection (pos >= 0) decides position pos with the drawn token,
 *     written into block_tokens[pos]; it holds the next label, n_accept+1;
 *   - decided[b] = the number of decided positions (the next pass's walk
 *     starts at step decided[b] + 1);
 *   - when every position is decided AND the pass drew nothing, the data
 *     section's keys and values in the cache are those of the final tokens:
 *     the block is done, lens[b] += B and decided[b] = 0 (the next block
 *     starts); a block completed by a draw is not done yet (the cache holds
 *     the draft's token at pos), so it takes one more pass in which every
 *     step is decided and nothing is tested.
 * done[b] = 1 when the block closed in this commit. */
int oracle_commit(int batch, const int *cu_B, const int *tau, const int *n_accept,
                  const int *token, const int *pos, int *block_tokens, int *decided,
                  int *lens, int *done) {
  if (batch < 0 || !cu_B || !tau || !n_accept || !token || !pos || !block_tokens ||
      !decided || !lens || !done)
    return ORACLE_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    const int s0 = cu_B[b], B = cu_B[b + 1] - s0;
    const int n = n_accept[b];
    if (B < 1 || n < 0 || n > B || (pos[b] >= 0 && (pos[b] >= B || n == B)) ||
        (pos[b] < 0 && n != B))
      return ORACLE_ERR_ARG;
    if (!oracle_tau_is_permutation(B, tau + s0)) return ORACLE_ERR_TAU;
    done[b] = 0;
    if (pos[b] >= 0) {
      if (tau[s0 + pos[b]] != n + 1) return ORACLE_ERR_ARG;   /* the walk's next step */
      block_tokens[s0 + pos[b]] = token[b];
      decided[b] = n + 1;
    } else if (n == B) {
      decided[b] = 0;
      lens[b] += B;
      done[b] = 1;
    }
  }
  return ORACLE_OK;
}
