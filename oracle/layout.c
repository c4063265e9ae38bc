/*
 * layout.c -- paired input layout, positions and the explicit temporal mask.
 * TEST INFRASTRUCTURE ONLY (see simsd_oracle.h).
 *
 * SimSD (gist.science, paper 2606.02544):
 *  - "Input Layout": two sections of length B follow the prompt, the data
 *    section D (reference tokens) and the mask section D~ (prediction slots);
 *    (D_k, D~_k) share one response position.
 *  - "Temporal Attention Mask": a step map assigns each response position a
 *    label tau in {1..B}; a mask slot D~_i may attend to D_j when
 *    tau(j) < tau(i) and to D~_j when tau(j) >= tau(i); never to data tokens
 *    not yet revealed.  The logits are conditioned like a prefix in
 *    autoregressive verification, so the whole prompt is visible.
 *  - Rows of D (a reading: only the slot logits are consumed) see the prompt
 *    and the data tokens with tau(j) <= tau(i), and no mask slot.
 *  - "Position Encoding Alignment": D~_k reuses the RoPE index of D_k.
 */
#include <stdlib.h>
#include "simsd_oracle.h"

int oracle_tau_is_permutation(int B, const int *tau) {
  if (B < 1 || tau == NULL) return 0;
  char *seen = (char *)calloc((size_t)B + 1, 1);
  if (seen == NULL) return 0;
  int ok = 1;
  for (int k = 0; k < B; ++k) {
    int t = tau[k];
    if (t < 1 || t > B || seen[t]) { ok = 0; break; }
    seen[t] = 1;
  }
  free(seen);
  return ok;
}

int oracle_mask_entry(int P, int B, const int *tau, int r, int c) {
  if (c < P) return 1;                 /* the whole prompt is visible       */
  int col = c - P;                     /* 0..2B-1 over [D | D~]             */
  int row_is_slot = (r >= B);
  int col_is_slot = (col >= B);
  int i = row_is_slot ? r - B : r;     /* response index of the row         */
  int j = col_is_slot ? col - B : col; /* response index of the column      */
  if (row_is_slot) {
    if (!col_is_slot) return tau[j] < tau[i];  /* earlier data tokens       */
    return tau[j] >= tau[i];                   /* current/later slots       */
  }
  if (!col_is_slot) return tau[j] <= tau[i];   /* data row: revealed data   */
  return 0;                                    /* data rows see no slot     */
}

int oracle_layout(int P, int B, const int *tau, int *positions,
                  unsigned char *mask) {
  if (P < 0 || B < 1 || tau == NULL || positions == NULL) return ORACLE_ERR_ARG;
  if (!oracle_tau_is_permutation(B, tau)) return ORACLE_ERR_TAU;
  const int L = P + 2 * B;
  for (int j = 0; j < P; ++j) positions[j] = j;
  for (int k = 0; k < B; ++k) {
    positions[P + k] = P + k;       /* D_{k+1}                              */
    positions[P + B + k] = P + k;   /* D~_{k+1} copies D_{k+1}'s RoPE index */
  }
  if (mask != NULL) {
    for (int r = 0; r < 2 * B; ++r)
      for (int c = 0; c < L; ++c)
        mask[(size_t)r * L + c] = (unsigned char)oracle_mask_entry(P, B, tau, r, c);
  }
  return ORACLE_OK;
}
