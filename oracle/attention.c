/*
 * attention.c -- RoPE and the masked verification attention, fp64.
 * TEST INFRASTRUCTURE ONLY (see simsd_oracle.h).
 *
 * SimSD (gist.science, paper 2606.02544):
 *  - "Speculative Decoding Pipeline", verification: one forward pass over
 *    [prompt | D | D~] under the temporal causal mask;
 *  - "Position Encoding Alignment": D~_k is rotated with D_k's index.
 * Attention itself is the textbook definition: for each row, scores
 * s_c = sm_scale * q.k_c over the visible columns c, softmax, o = sum p_c v_c.
 * Grouped-query heads: query head h reads KV head h / (Hq/Hkv).
 */
#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include "simsd_oracle.h"

void oracle_rope(const double *x, int n_tok, int n_heads, int hd,
                 const int *pos, double base, double *out) {
  const int half = hd / 2;
  for (int t = 0; t < n_tok; ++t) {
    for (int h = 0; h < n_heads; ++h) {
      const double *xi = x + ((size_t)t * n_heads + h) * hd;
      double *yo = out + ((size_t)t * n_heads + h) * hd;
      for (int d = 0; d < half; ++d) {
        double inv_freq = pow(base, -2.0 * (double)d / (double)hd);
        double theta = (double)pos[t] * inv_freq;
        double c = cos(theta), s = sin(theta);
        double x1 = xi[d], x2 = xi[d + half];
        yo[d] = x1 * c - x2 * s;
        yo[d + half] = x2 * c + x1 * s;
      }
    }
  }
}

/* One output row: softmax over the visible keys of row r for query vector qr
 * (already rotated), KV head g.  keys(c) / vals(c) come from the prompt for
 * c < P and from the rotated new keys / raw new values after it. */
static void attend_row(int P, int B, int Hkv, int hd, double sm_scale,
                       const int *tau, int r, int g, const double *qr,
                       const double *k_prompt, const double *v_prompt,
                       const double *k_new_rot, const double *v_new,
                       double *score, double *out) {
  const int L = P + 2 * B;
  double m = -INFINITY;
  for (int c = 0; c < L; ++c) {
    if (!oracle_mask_entry(P, B, tau, r, c)) { score[c] = -INFINITY; continue; }
    const double *kc = (c < P) ? k_prompt + ((size_t)c * Hkv + g) * hd
                               : k_new_rot + ((size_t)(c - P) * Hkv + g) * hd;
    double s = 0.0;
    for (int d = 0; d < hd; ++d) s += qr[d] * kc[d];
    s *= sm_scale;
    score[c] = s;
    if (s > m) m = s;
  }
  double denom = 0.0;
  for (int c = 0; c < L; ++c)
    if (score[c] != -INFINITY) denom += exp(score[c] - m);
  for (int d = 0; d < hd; ++d) out[d] = 0.0;
  for (int c = 0; c < L; ++c) {
    if (score[c] == -INFINITY) continue;
    double w = exp(score[c] - m) / denom;
    const double *vc = (c < P) ? v_prompt + ((size_t)c * Hkv + g) * hd
                               : v_new + ((size_t)(c - P) * Hkv + g) * hd;
    for (int d = 0; d < hd; ++d) out[d] += w * vc[d];
  }
}

int oracle_verify_attn_seq(int P, int B, int Hq, int Hkv, int hd,
                           double rope_base, double sm_scale, int pos_offset,
                           const int *tau, const double *q,
                           const double *k_prompt, const double *v_prompt,
                           const double *k_new, const double *v_new,
                           int n_rows, const int *row_tok, const int *row_head,
                           double *out) {
  if (P < 0 || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || hd < 2 ||
      hd % 2 != 0 || q == NULL || k_new == NULL || v_new == NULL || out == NULL ||
      (P > 0 && (k_prompt == NULL || v_prompt == NULL)))
    return ORACLE_ERR_ARG;
  if (n_rows >= 0 && n_rows > 0 && (row_tok == NULL || row_head == NULL))
    return ORACLE_ERR_ARG;
  const int L = P + 2 * B;
  const int G = Hq / Hkv;
  int *positions = (int *)malloc(sizeof(int) * (size_t)L);
  double *k_new_rot = (double *)malloc(sizeof(double) * (size_t)2 * B * Hkv * hd);
  double *qr = (double *)malloc(sizeof(double) * (size_t)hd);
  double *score = (double *)malloc(sizeof(double) * (size_t)L);
  int rc = ORACLE_OK;
  if (!positions || !k_new_rot || !qr || !score) { rc = ORACLE_ERR_ARG; goto done; }
  rc = oracle_layout(P, B, tau, positions, NULL);
  if (rc != ORACLE_OK) goto done;
  int *new_pos = positions + P;             /* positions of the 2B new tokens */
  for (int t = 0; t < 2 * B; ++t) new_pos[t] += pos_offset;
  oracle_rope(k_new, 2 * B, Hkv, hd, new_pos, rope_base, k_new_rot);

  const int total = (n_rows < 0) ? 2 * B * Hq : n_rows;
  for (int i = 0; i < total; ++i) {
    int t = (n_rows < 0) ? i / Hq : row_tok[i];
    int h = (n_rows < 0) ? i % Hq : row_head[i];
    if (t < 0 || t >= 2 * B || h < 0 || h >= Hq) { rc = ORACLE_ERR_ARG; goto done; }
    const double *qi = q + ((size_t)t * Hq + h) * hd;
    oracle_rope(qi, 1, 1, hd, &new_pos[t], rope_base, qr);
    attend_row(P, B, Hkv, hd, sm_scale, tau, t, h / G, qr, k_prompt, v_prompt,
               k_new_rot, v_new, score, out + (size_t)i * hd);
  }
done:
  free(positions);
  free(k_new_rot);
  free(qr);
  free(score);
  return rc;
}

int oracle_verify_attn(int batch, const int *lens, const int *cu_B, int Hq,
                       int Hkv, int hd, double rope_base, double sm_scale,
                       const int *tau, const double *q,
                       const double *k_prompt, const double *v_prompt,
                       const double *k_new, const double *v_new,
                       double *out, int n_threads) {
  if (batch < 0 || lens == NULL || cu_B == NULL) return ORACLE_ERR_ARG;
  size_t *prompt_off = (size_t *)malloc(sizeof(size_t) * ((size_t)batch + 1));
  if (prompt_off == NULL) return ORACLE_ERR_ARG;
  prompt_off[0] = 0;
  for (int b = 0; b < batch; ++b) prompt_off[b + 1] = prompt_off[b] + (size_t)lens[b];
  int rc = ORACLE_OK;
  const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(max : rc)
  for (int b = 0; b < batch; ++b) {
    int B = cu_B[b + 1] - cu_B[b];
    size_t tok0 = 2 * (size_t)cu_B[b];
    int r = oracle_verify_attn_seq(
        lens[b], B, Hq, Hkv, hd, rope_base, sm_scale, 0, tau + cu_B[b],
        q + tok0 * Hq * hd, k_prompt + prompt_off[b] * Hkv * hd,
        v_prompt + prompt_off[b] * Hkv * hd, k_new + tok0 * Hkv * hd,
        v_new + tok0 * Hkv * hd, -1, NULL, NULL, out + tok0 * Hq * hd);
    if (r > rc) rc = r;
  }
  free(prompt_off);
  return rc;
}

/* ------------------------------------------------------------------------
 * Spiffy (gist.science, paper 2509.18085), "Metodologia: Spiffy": draft
 * states form a directed graph (a block at timestep t_a is a parent of one
 * at t_b = t_a - 1 whose unmasked tokens are a superset of its own), and
 * verification evaluates several draft candidates in parallel under a
 * custom blockwise attention mask.  Reading taken: each node of the graph
 * is a complete candidate state of the block (node_size tokens, unmasked
 * or [MASK]); the section holds n_nodes such copies after the prompt; a
 * row of node n attends to the whole prompt and to every token of node n
 * (a dLLM attends bidirectionally within its block), and to no token of
 * another node -- a child already holds its parent's unmasked tokens, so
 * the parent set orders the acceptance walk, not the mask.  Every node's
 * token k sits at position P + k (each node is a copy of the block). */
int oracle_graph_mask_entry(int P, int n_nodes, int node_size, int r, int c) {
  if (r < 0 || r >= n_nodes * node_size || c < 0 || c >= P + n_nodes * node_size) return 0;
  if (c < P) return 1;
  return (c - P) / node_size == r / node_size;
}

int oracle_verify_attn_graph_seq(int P, int n_nodes, int node_size, int Hq, int Hkv, int hd,
                                 double rope_base, double sm_scale, const double *q,
                                 const double *k_prompt, const double *v_prompt,
                                 const double *k_new, const double *v_new, double *out) {
  if (P < 0 || n_nodes < 1 || node_size < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
      hd < 2 || hd % 2 != 0 || !q || !k_new || !v_new || !out ||
      (P > 0 && (!k_prompt || !v_prompt)))
    return ORACLE_ERR_ARG;
  const int T = n_nodes * node_size, L = P + T, G = Hq / Hkv;
  int *pos = (int *)malloc(sizeof(int) * (size_t)T);
  double *k_rot = (double *)malloc(sizeof(double) * (size_t)T * Hkv * hd);
  double *qr = (double *)malloc(sizeof(double) * (size_t)hd);
  double *score = (double *)malloc(sizeof(double) * (size_t)L);
  if (!pos || !k_rot || !qr || !score) {
    free(pos); free(k_rot); free(qr); free(score);
    return ORACLE_ERR_ARG;
  }
  for (int j = 0; j < T; ++j) pos[j] = P + j % node_size;
  oracle_rope(k_new, T, Hkv, hd, pos, rope_base, k_rot);
  for (int r = 0; r < T; ++r) {
    for (int h = 0; h < Hq; ++h) {
      const int g = h / G;
      oracle_rope(q + ((size_t)r * Hq + h) * hd, 1, 1, hd, &pos[r], rope_base, qr);
      double m = -INFINITY;
      for (int c = 0; c < L; ++c) {
        if (!oracle_graph_mask_entry(P, n_nodes, node_size, r, c)) { score[c] = -INFINITY; continue; }
        const double *kc = (c < P) ? k_prompt + ((size_t)c * Hkv + g) * hd
                                   : k_rot + ((size_t)(c - P) * Hkv + g) * hd;
        double sc = 0.0;
        for (int d = 0; d < hd; ++d) sc += qr[d] * kc[d];
        score[c] = sc * sm_scale;
        if (score[c] > m) m = score[c];
      }
      double denom = 0.0;
      for (int c = 0; c < L; ++c)
        if (score[c] != -INFINITY) denom += exp(score[c] - m);
      double *o = out + ((size_t)r * Hq + h) * hd;
      for (int d = 0; d < hd; ++d) o[d] = 0.0;
      for (int c = 0; c < L; ++c) {
        if (score[c] == -INFINITY) continue;
        const double w = exp(score[c] - m) / denom;
        const double *vc = (c < P) ? v_prompt + ((size_t)c * Hkv + g) * hd
                                   : v_new + ((size_t)(c - P) * Hkv + g) * hd;
        for (int d = 0; d < hd; ++d) o[d] += w * vc[d];
      }
    }
  }
  free(pos); free(k_rot); free(qr); free(score);
  return ORACLE_OK;
}
