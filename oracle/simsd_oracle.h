/*
 * simsd_oracle.h -- plain fp64 CPU oracle for the SimSD verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this code: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through seeded synthetic inputs.
 *
 * Source: "SimSD: Simple Speculative Decoding in Diffusion Language Models"
 * (technical summaries on gist.science, paper 2606.02544, Dutch and French
 * pages), sections "Input Layout" (1), "Temporal Attention Mask" (2),
 * "Position Encoding Alignment" (3) and "Speculative Decoding Pipeline" (4).
 *
 * Every routine is written for a reader to check by eye against those
 * sections: the mask is materialised from its definition, attention is a
 * two-pass softmax over explicitly listed visible keys, acceptance walks the
 * temporal order one step at a time.  No blocking, fusion or reordering.
 *
 * Parity unpinned (no pin exists on the pages):
 *   - the RoPE pairing convention (rotate-half is a reading; the pages say
 *     only "RoPE copy");
 *   - the softmax scale (an argument; the pages give none).
 */
#ifndef SIMSD_ORACLE_H
#define SIMSD_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,   /* a size or pointer is invalid                  */
  ORACLE_ERR_TAU = 2    /* tau is not a permutation of 1..B              */
};

/* 1 if tau[0..B) is a permutation of 1..B, else 0. */
int oracle_tau_is_permutation(int B, const int *tau);

/* One entry of the temporal causal mask for the 2B new rows.
 * Row r in [0,2B): r < B is data token D_{r+1}, r >= B is mask slot
 * D~_{r-B+1}.  Column c in [0, P+2B): c < P is a prompt token, then the B
 * data tokens, then the B mask slots.  Returns 1 when the row may attend. */
int oracle_mask_entry(int P, int B, const int *tau, int r, int c);

/* Paired layout: positions[P+2B] (prompt j -> j, D_k and D~_k -> P+k-1) and,
 * when mask != NULL, the explicit mask[2B][P+2B] of the new rows.
 * Returns ORACLE_OK, ORACLE_ERR_ARG or ORACLE_ERR_TAU. */
int oracle_layout(int P, int B, const int *tau, int *positions,
                  unsigned char *mask);

/* Rotary position embedding (rotate-half pairing), fp64.
 * x, out: [n_tok][n_heads][hd]; pos: [n_tok].  For d < hd/2 with
 * theta = pos * base^(-2d/hd):
 *   out[d]        = x[d]        cos(theta) - x[d+hd/2] sin(theta)
 *   out[d+hd/2]   = x[d+hd/2]   cos(theta) + x[d]      sin(theta)
 * out may alias x. */
void oracle_rope(const double *x, int n_tok, int n_heads, int hd,
                 const int *pos, double base, double *out);

/* Verification attention for ONE sequence, fp64.
 *   q       [2B][Hq][hd]   raw (pre-RoPE) queries of D_1..D_B, D~_1..D~_B
 *   k_prompt[P][Hkv][hd]   prompt keys, already rotated at positions
 *                          pos_offset + 0 .. pos_offset + P-1
 *   v_prompt[P][Hkv][hd]
 *   k_new, v_new [2B][Hkv][hd]  raw keys/values of the new tokens
 *   tau[B]  step labels, a permutation of 1..B
 * New tokens are rotated at pos_offset + their layout position.  Query head
 * h reads KV head h / (Hq/Hkv).
 * Rows: n_rows >= 0 selects (row_tok[i], row_head[i]) pairs, out[n_rows][hd];
 * n_rows < 0 computes every row, out[2B][Hq][hd].
 * Returns ORACLE_OK or an error code. */
int oracle_verify_attn_seq(int P, int B, int Hq, int Hkv, int hd,
                           double rope_base, double sm_scale, int pos_offset,
                           const int *tau, const double *q,
                           const double *k_prompt, const double *v_prompt,
                           const double *k_new, const double *v_new,
                           int n_rows, const int *row_tok, const int *row_head,
                           double *out);

/* Whole batch, every row: sequences are laid out back to back.
 *   lens[b] = P_b, cu_B[batch+1] prefix sums of B_b.
 *   q, out:        [sum 2B_b][Hq][hd]
 *   k_new, v_new:  [sum 2B_b][Hkv][hd]
 *   k_prompt, v_prompt: [sum P_b][Hkv][hd]
 *   tau: [sum B_b]
 * Runs sequences in parallel on n_threads OpenMP threads (<= 0: default). */
int oracle_verify_attn(int batch, const int *lens, const int *cu_B, int Hq,
                       int Hkv, int hd, double rope_base, double sm_scale,
                       const int *tau, const double *q,
                       const double *k_prompt, const double *v_prompt,
                       const double *k_new, const double *v_new,
                       double *out, int n_threads);

/* Spiffy's draft-graph verification (reading: each node a complete
 * candidate state of the block).  Mask entry for new row r (node r /
 * node_size) and column c: 1 for every prompt column and for the columns
 * of the same node, else 0. */
int oracle_graph_mask_entry(int P, int n_nodes, int node_size, int r, int c);

/* Attention of one sequence's n_nodes x node_size new rows under that mask,
 * fp64.  q [T][Hq][hd], k_new / v_new [T][Hkv][hd] raw (T = n_nodes *
 * node_size, node-major); k_prompt / v_prompt [P][Hkv][hd] with the keys
 * rotated; every node's token k is rotated at position P + k.
 * out [T][Hq][hd]. */
int oracle_verify_attn_graph_seq(int P, int n_nodes, int node_size, int Hq, int Hkv, int hd,
                                 double rope_base, double sm_scale, const double *q,
                                 const double *k_prompt, const double *v_prompt,
                                 const double *k_new, const double *v_new, double *out);

/* Residual of one slot: r[v] = max(0, p(v) - q(v)) with p, q the softmax of
 * the target and draft logit rows (p itself when that is empty); returns
 * S = sum r.  The acceptance walk draws its token from r / S. */
double oracle_residual(int V, const double *target, const double *draft, double *r);

/* Rejection-sampling acceptance along the temporal order, fp64.
 *   target, draft: [sum B_b][V] logits; row k of sequence b is response
 *                  position k (the logits read at D~_k).
 *   draft_tokens:  [sum B_b], tau: [sum B_b]
 *   uniforms:      [batch][u_stride] in [0,1): u[t-1] tests step t,
 *                  u[B_b] draws the residual token.
 *   first_step:    [batch] or NULL (1): the walk starts at this step
 *                  (1..B_b+1); earlier steps are positions decided in
 *                  earlier passes of the block, counted as accepted.
 * Outputs per sequence: n_accept (accepted prefix length in temporal
 * order), token (resampled token at the first rejection, -1 if all were
 * accepted), pos (response position of that rejection, -1 if none).
 * accept_margin[sum B_b] (optional): |u q(x) - p(x)| / p(x) of every tested
 *   step, stored at the tested slot; -1 for slots never tested.
 * resample_margin[batch] (optional): distance of u*S to the nearest CDF
 *   boundary of the chosen token, relative to S; -1 when nothing was drawn.
 * n_threads <= 0: OpenMP default.  Returns ORACLE_OK or an error code. */
int oracle_accept(int batch, int V, const int *cu_B, const double *target,
                  const double *draft, const int *draft_tokens,
                  const int *tau, const float *uniforms, int u_stride,
                  const int *first_step, int *n_accept, int *token, int *pos,
                  double *accept_margin, double *resample_margin,
                  int n_threads);

/* Greedy verification: step t accepts iff its draft token is the target's
 * argmax (smallest index among equal maxima); the first rejection emits that
 * argmax.  Uniforms and draft logits are not used.  first_step as above. */
int oracle_accept_greedy(int batch, int V, const int *cu_B, const double *target,
                         const int *draft_tokens, const int *tau, const int *first_step,
                         int *n_accept, int *token, int *pos);

/* Sample matching: step t draws y_t from p by inverse CDF with u[t-1] and
 * accepts iff y_t is the draft token; the first rejection emits y_t.
 * first_step as above. */
int oracle_accept_match(int batch, int V, const int *cu_B, const double *target,
                        const int *draft_tokens, const int *tau, const float *uniforms,
                        int u_stride, const int *first_step, int *n_accept, int *token,
                        int *pos);

/* The draft-side step: each open slot samples its token from the draft
 * softmax by inverse CDF with u[k]; tau orders the open slots by the row's
 * largest draft probability (most confident first, ties in position order)
 * after the decided[b] steps decided in earlier passes of the block, which
 * keep their tokens and labels (from tau_prev).  decided == NULL: all open. */
int oracle_draft_step(int batch, int V, const int *cu_B, const double *draft,
                      const float *uniforms, int u_stride, const int *decided,
                      const int *tau_prev, int *draft_tokens, int *tau, double *confidence);

/* Commit after a pass of the blockwise loop: the drawn token goes to
 * block_tokens at pos, decided[b] becomes the count of decided positions,
 * and a block whose positions are all decided by a pass that drew nothing
 * closes (lens[b] += B_b, decided[b] = 0, done[b] = 1). */
int oracle_commit(int batch, const int *cu_B, const int *tau, const int *n_accept,
                  const int *token, const int *pos, int *block_tokens, int *decided,
                  int *lens, int *done);

#ifdef __cplusplus
}
#endif
#endif /* SIMSD_ORACLE_H */
