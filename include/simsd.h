/*
 * simsd.h -- C ABI of libsimsd.so: the SimSD speculative-verification step
 * for diffusion language models on one NVIDIA GB300 (sm_103a).
 *
 * Method: "SimSD: Simple Speculative Decoding in Diffusion Language Models"
 * (gist.science technical summaries of paper 2606.02544):
 *   section 1 "Input Layout"            -- prompt | D (B reference tokens) |
 *                                          D~ (B [MASK] prediction slots);
 *   section 2 "Temporal Attention Mask" -- step map tau, mask A_ij;
 *   section 3 "Position Encoding Alignment" -- D~_k reuses D_k's RoPE index;
 *   section 4 "Speculative Decoding Pipeline" -- one verification forward,
 *                                          rejection sampling along tau.
 *
 * Conventions shared by every call
 *   - Plain C types only.  "device" pointers are CUDA device memory of the
 *     current device; "host" pointers are ordinary host memory.
 *   - All memory is owned by the caller.  The device calls never allocate:
 *     scratch lives in a caller-provided workspace whose size the matching
 *     *_workspace_size function returns (256-byte aligned pointer required).
 *   - Device calls are asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).  They never
 *     synchronise the host.
 *   - Argument errors are detected on the host and returned before anything
 *     is launched.  A launch failure returns SIMSD_ERR_CUDA.  Kernels never
 *     trap: a bounded wait that runs out, or device arrays that disagree
 *     with the limits, set a bit in the workspace's status word (its first
 *     4 bytes).  The bits stay set across calls until simsd_read_status()
 *     reads and clears them (no call clears it on the hot path), so a new
 *     workspace must start zero-filled (or be passed to simsd_read_status
 *     once).
 *   - Token order inside a sequence with section length B is
 *     D_1..D_B, D~_1..D~_B (2B tokens); sequences are back to back, so
 *     sequence b's tokens start at row 2*cu_B[b].
 *   - Limits: head_dim in {64, 128}; num_q_heads % num_kv_heads == 0;
 *     1 <= B_b <= 32; page_size == 16; batch >= 1; one new token's raw
 *     q, k and v rows together at most 196,608 bytes
 *     ((num_q_heads + 2 num_kv_heads) * head_dim * element size).
 *   - Every device array of q, k, v, cache or output values starts on a
 *     16-byte boundary (SIMSD_ERR_ALIGN otherwise); logits may be unaligned
 *     (slower element-wise loads).
 *   - The library is stateless and re-entrant.  Calls on different streams
 *     must not share a workspace or write the same cache pages.
 */
#ifndef SIMSD_H
#define SIMSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SIMSD_OK = 0,
  SIMSD_ERR_NULL = 1,      /* a required pointer is NULL                    */
  SIMSD_ERR_SHAPE = 2,     /* a size is out of range or inconsistent        */
  SIMSD_ERR_TAU = 3,       /* tau is not a permutation of 1..B              */
  SIMSD_ERR_DTYPE = 4,     /* unsupported dtype                             */
  SIMSD_ERR_WORKSPACE = 5, /* workspace missing, misaligned or too small    */
  SIMSD_ERR_CUDA = 6,      /* a CUDA runtime call or launch failed          */
  SIMSD_ERR_TIMEOUT = 7,   /* a device-side bounded wait ran out            */
  SIMSD_ERR_ALIGN = 8      /* a device array is not 16-byte aligned         */
} simsd_status;

typedef enum { SIMSD_F32 = 0, SIMSD_BF16 = 1 } simsd_dtype;

/* Static text for a status code; never NULL. */
const char *simsd_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int simsd_version(void);

/* ------------------------------------------------------------------------
 * simsd_layout -- host only.  Sections 1-3: paired layout, positions, mask.
 *   prompt_len  P >= 0
 *   B           1..32 (section length; also the draft length gamma)
 *   tau         host int32[B], tau[k] = step label of response position k+1
 *   positions   host int32[P+2B] out: prompt j -> j; D_k -> P+k-1;
 *               D~_k -> P+k-1 (copied RoPE index)
 *   mask        host uint8[2B][P+2B] out, may be NULL.  Row r < B is D_{r+1},
 *               row B+i is D~_{i+1}; column c < P is prompt token c, then D,
 *               then D~.  1 = may attend.  Slot rows: whole prompt, D_j with
 *               tau(j) < tau(i), D~_j with tau(j) >= tau(i).  Data rows (a
 *               convention: their outputs feed later layers, their logits
 *               are not consumed): prompt and D_j with tau(j) <= tau(i).
 * Errors: SIMSD_ERR_NULL, SIMSD_ERR_SHAPE, SIMSD_ERR_TAU.
 * ---------------------------------------------------------------------- */
simsd_status simsd_layout(int32_t prompt_len, int32_t B, const int32_t *tau,
                          int32_t *positions, uint8_t *mask);

/* ------------------------------------------------------------------------
 * simsd_verify_attn -- sections 2-4: one attention layer of the verification
 * forward over [prompt KV cache | D | D~] for a batch of sequences.
 *
 * Kernel sequence on `stream`:
 *   K1  rotate q (all query heads) and k_new at the layout positions (D~_k
 *       uses D_k's), write rotated k and raw v of the 2B new tokens into
 *       cache slots [lens[b], lens[b]+2B_b) of sequence b;
 *   K2  attention of all 2B_b x Hq query rows of a sequence and KV head
 *       against the cache, the temporal mask evaluated on the fly; a
 *       (sequence, KV head) unit runs whole or in key splits (every unit
 *       when the block-table width makes one unit long, or only the units
 *       of the last partial wave of CTAs, so that wave takes a split's
 *       time instead of a unit's);
 *   K3  merge of the split units' partial softmax states (launched only
 *       when some unit is split).
 * lens[] is NOT advanced: rolling back a rejected draft costs nothing, and
 * committing accepted tokens is the caller's business.
 *
 * Layouts (row-major, innermost last):
 *   q            device [T][Hq][hd]   raw queries, T = 2 * total_B
 *   k_new, v_new device [T][Hkv][hd]  raw keys / values of the new tokens
 *   k_cache, v_cache device [num_pages][Hkv][page_size][hd]; prompt slots
 *                hold keys already rotated at their own positions
 *   block_table  device int32[batch][max_pages_per_seq]; entries
 *                0 .. ceil((lens[b]+2B_b)/16)-1 of row b must be valid page
 *                ids < num_pages (the rest are never read)
 *   tau          device int32[total_B]; sequence b's labels at cu_B[b]..
 *   lens         device int32[batch]   prompt KV length P_b >= 0
 *   cu_B         device int32[batch+1] prefix sums of B_b (cu_B[0] = 0)
 *   out          device [T][Hq][hd]    attention output of every new row
 * dtype applies to q, k/v (new and cache) and out.
 * Host-side fields (total_B, B_max, max_pages_per_seq) must agree with the
 * device arrays.  A sequence whose device arrays disagree with them (cu_B
 * not within 0..total_B, B_b outside 1..B_max, lens[b]+2B_b beyond the
 * table row, a page id outside the cache) sets the status word's bad-input
 * bit (2) and is skipped: nothing is read or written out of range for it.
 * tau is trusted: a wrong tau gives a wrong mask, never an out-of-bounds
 * access.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t batch;
  int32_t num_q_heads;        /* Hq                                         */
  int32_t num_kv_heads;       /* Hkv                                        */
  int32_t head_dim;           /* hd: 64 or 128                              */
  int32_t page_size;          /* 16                                         */
  int32_t num_pages;          /* pages in each cache array                  */
  int32_t max_pages_per_seq;  /* row stride of block_table                  */
  int32_t total_B;            /* sum_b B_b (host copy)                      */
  int32_t B_max;              /* max_b B_b (host copy), 1..32               */
  simsd_dtype dtype;
  float rope_base;            /* RoPE base (e.g. 1e6)                       */
  float sm_scale;             /* score = sm_scale * q.k; finite, > 0        */
  const void *q;
  void *k_cache;
  void *v_cache;
  const int32_t *block_table;
  const void *k_new;
  const void *v_new;
  const int32_t *tau;
  const int32_t *lens;
  const int32_t *cu_B;
  void *out;
  void *workspace;            /* device, 256-byte aligned                   */
  size_t workspace_bytes;
  int32_t wait_polls;         /* polls a kernel's bounded wait makes before
                                 it gives up: 0 (a zero-filled descriptor)
                                 selects the default 2^24; a negative value
                                 gives up at once, which runs the timeout
                                 path (status bit 0, nothing written to the
                                 cache; out undefined) -- for tests        */
  int32_t node_size;          /* 0: SimSD's paired layout under the temporal
                                 mask (above).  > 0: Spiffy's draft-graph
                                 verification: a sequence's 2B_b new tokens
                                 are 2B_b / node_size candidate states of the
                                 block (nodes of node_size <= 32 tokens, node
                                 after node); token k of every node sits at
                                 position lens[b] + k; a row attends to the
                                 whole prompt and to every token of its own
                                 node, nothing of another node; tau is not
                                 read (may be NULL).  A sequence whose 2B_b
                                 is not a multiple of node_size sets the
                                 bad-input bit and is skipped                */
} simsd_verify_desc;

/* Bytes of workspace simsd_verify_attn needs for these sizes (reads only
 * the host-side fields).  Returns 0 if the sizes are invalid.  The size
 * follows the key-split plan, which depends on the current device's SM
 * count (152 when no device is visible): query it with the device that
 * will run the call current. */
size_t simsd_verify_workspace_size(const simsd_verify_desc *d);
simsd_status simsd_verify_attn(const simsd_verify_desc *d, void *stream);

/* Same as simsd_verify_attn, and records caller-created CUDA events (each a
 * cudaEvent_t, or NULL to skip) on `stream` at the kernel boundaries:
 * events[0] before K1, [1] after K1, [2] after K2, [3] after K3 (recorded
 * even when K3 is not needed).  For per-kernel timing; the events are not
 * waited on or destroyed. */
simsd_status simsd_verify_attn_timed(const simsd_verify_desc *d, void *stream,
                                     void *const events[4]);

/* ------------------------------------------------------------------------
 * simsd_prompt_append -- K1 on plain positions: rotate n_b raw keys of
 * sequence b at positions start[b] .. start[b]+n_b-1 and write them (and
 * the raw values) into the same cache slots.  Fills a prompt's cache, or
 * commits tokens after acceptance.
 *   k, v     device [sum n_b][Hkv][hd]   raw keys / values
 *   start    device int32[batch]         first slot (= position) per seq
 *   cu_n     device int32[batch+1]       prefix sums of n_b
 *   total_n  host: sum n_b
 *   block_table as above; every slot written must be covered.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
  int32_t total_n;
  simsd_dtype dtype;
  float rope_base;
  const void *k;
  const void *v;
  const int32_t *start;
  const int32_t *cu_n;
  void *k_cache;
  void *v_cache;
  const int32_t *block_table;
} simsd_append_desc;

simsd_status simsd_prompt_append(const simsd_append_desc *d, void *stream);

/* ------------------------------------------------------------------------
 * simsd_accept -- section 4, acceptance: standard rejection sampling along
 * the temporal order tau.  For sequence b and steps t = 1..B_b, slot
 * k = tau^-1(t) with draft token x = draft_tokens[k]:
 *   p = softmax(target row k / T), q = softmax(draft row k / T) (fp32
 *   math; T = temperature, 1 by default);
 *   accept iff u[t-1] * q(x) < p(x);
 *   at the first rejection draw a token from max(0, p - q) normalised (p
 *   itself if that is empty) by inverse CDF with u[B_b], and stop.
 * Variant rule SIMSD_ACCEPT_GREEDY (the temperature -> 0 limit): step t
 * accepts iff x is the target row's argmax (the smallest index among equal
 * maxima); the first rejection emits that argmax.  It reads neither the
 * draft logits nor the uniforms (they may be NULL).
 * Variant rule SIMSD_ACCEPT_MATCH (sample matching, Spiffy's verification):
 * step t draws the target's own token y from p (at temperature T) by
 * inverse CDF with u[t-1] and accepts iff y = x; the first rejection emits
 * y (u[B_b] unused, draft logits not read and may be NULL).
 * Kernels: K4a, a chunk pass over (row, 32 KB chunk) items on every SM
 * (for the sampling rule's small batches a pass that loads each part
 * directly, a warp per part), writes per eighth of a chunk (a "part") its
 * maximum and sum of
 * exponentials -- of both rows of every slot for the sampling rule; of the
 * target rows and the mass below the draft token for sample matching; the
 * largest value and its index for the greedy rule -- and the logits at the
 * draft tokens, to the workspace.  K4b: sampling, up to two CTAs per SM
 * over the batch, each owning a range of a sequence's chunks: every CTA of
 * a sequence merges its slots' parts and walks the steps alike, computes
 * the residual masses of its chunks of the rejected slot's two rows, and
 * the last CTA of the sequence draws from them; greedy and matching, one
 * CTA per sequence merging each slot's parts (matching: a slot that
 * rejects draws its token from the part holding u S) and walking the
 * steps.  With a workspace smaller than simsd_accept_workspace_size, or
 * with `decided` (the blockwise loop: decided slots' rows are not read),
 * each rule's thread-block cluster kernel (C <= 16 CTAs per sequence, each
 * owning 1/C of the vocabulary) streams the rows itself in one launch.
 *   target_logits, draft_logits device [total_B][vocab] (dtype); row k of
 *                sequence b (at cu_B[b]+k) holds the logits read at D~_k
 *   draft_tokens device int32[total_B] in [0, vocab); a token outside
 *                sets the status word's bad-input bit and its step rejects
 * A sequence whose cu_B entries fall outside 0..total_B, whose B_b is
 * outside 1..B_max, or whose tau is not a permutation of 1..B_b sets the
 * bad-input bit and gets n_accept = 0, token = -1, pos = -1 without reading
 * its logits.  Logits must not be NaN (-inf is allowed; the greedy rule
 * gives index 0 for a row with no larger entry).
 *   tau, cu_B    device, as for simsd_verify_attn
 *   uniforms     device float32[batch][B_max+1], values in [0, 1)
 *   n_accept     device int32[batch] out: accepted prefix length (0..B_b)
 *   token        device int32[batch] out: token drawn at the rejection,
 *                -1 when every step was accepted (no bonus token: the
 *                layout has no slot after D~_B)
 *   pos          device int32[batch] out: response position (0-based k) of
 *                the rejected slot, -1 when none
 * Limits: 1 <= vocab <= 2^21; batch <= 65535.  Rows whose byte length is
 * a multiple of 16 (and 16-byte aligned logits) are streamed by bulk
 * copies; other vocabularies take a slower element-wise copy.
 * Workspace: simsd_accept_workspace_size returns the size of the
 * two-kernel path, with C = ceil(vocab / E) chunks of E = 16384 entries
 * (bf16) or 8192 (fp32) and each term rounded up to a multiple of 256:
 * sampling, 256 + 2 total_B C * 64 + 2 total_B * 4 + batch * 4 +
 * batch C * 256 bytes; greedy and matching, 256 + total_B C * 128 +
 * total_B * 4.  Any workspace of at least 256 bytes is accepted; one smaller
 * than that size runs the single-launch path.  A wait of the chunk pass
 * that gives up leaves every sequence of the call with n_accept = 0,
 * token = -1, pos = -1 (and the timeout bit set).
 * Errors: SIMSD_ERR_NULL, SIMSD_ERR_SHAPE (also: an unknown rule, or a
 * temperature that is negative or not finite), SIMSD_ERR_DTYPE,
 * SIMSD_ERR_WORKSPACE, SIMSD_ERR_CUDA.
 * ---------------------------------------------------------------------- */
typedef enum {
  SIMSD_ACCEPT_SAMPLE = 0,    /* rejection sampling at temperature T         */
  SIMSD_ACCEPT_GREEDY = 1,    /* accept iff x = argmax of the target row      */
  SIMSD_ACCEPT_MATCH = 2      /* accept iff x = the target's own sample       */
} simsd_accept_rule;

typedef struct {
  int32_t batch;
  int32_t vocab;
  int32_t total_B;            /* host copy                                  */
  int32_t B_max;              /* host copy, 1..32                           */
  simsd_dtype dtype;          /* of the logits                              */
  const void *target_logits;
  const void *draft_logits;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  void *workspace;            /* device, 256-byte aligned                   */
  size_t workspace_bytes;
  simsd_accept_rule rule;     /* 0 (a zero-filled descriptor): sampling      */
  float temperature;          /* > 0; 0 selects 1 (a zero-filled descriptor
                                 keeps the standard rule); the logits are
                                 divided by this float's exact value         */
  int32_t wait_polls;         /* as in simsd_verify_desc; a sequence whose
                                 wait gave up gets n_accept = 0, token = -1,
                                 pos = -1 (the sampling rule's chunk pass for
                                 small batches and the finishing kernels have
                                 no waits)                                   */
  const int32_t *decided;     /* device int32[batch] or NULL (all 0): steps
                                 1..decided[b] belong to positions decided
                                 in earlier passes of the block (the
                                 blockwise loop, simsd_commit); the walk
                                 starts at step decided[b]+1 and counts the
                                 earlier ones as accepted (0..B_b; B_b: no
                                 step is tested, n_accept = B_b)             */
} simsd_accept_desc;

size_t simsd_accept_workspace_size(const simsd_accept_desc *d);
simsd_status simsd_accept(const simsd_accept_desc *d, void *stream);

/* Same as simsd_accept, recording events (cudaEvent_t or NULL) on `stream`:
 * events[0] before K4, [1] after K4a (the chunk pass; recorded right after
 * [0] on the single-launch path), [2] after K4b. */
simsd_status simsd_accept_timed(const simsd_accept_desc *d, void *stream,
                                void *const events[3]);

/* ------------------------------------------------------------------------
 * simsd_draft_step -- section 4, drafting: the draft proposes the section's
 * tokens and their temporal order.  For each open slot k of sequence b
 * (every slot when decided is NULL; else those with tau_prev[k] >
 * decided[b]): q = softmax(draft row k / T); the token is the smallest v
 * whose running mass exceeds u[k] (inverse CDF; the last v with q > 0 if
 * rounding leaves none); the open slots take the step labels
 * decided[b]+1 .. B_b in order of the row's largest probability, max_v q(v)
 * (most confident first, equal ones in position order).  The order depends
 * on the draft rows only, not on the drawn tokens, which keeps the walk's
 * rejection sampling exact.  Decided slots keep their token and label.
 *   draft_logits device [total_B][vocab] (dtype)
 *   uniforms     device float32[batch][B_max], values in [0, 1): u[k]
 *                draws slot k
 *   decided      device int32[batch] or NULL
 *   tau_prev     device int32[total_B], read when decided is not NULL: the
 *                block's labels so far (decided slots: 1..decided[b])
 *   tokens       device int32[total_B] in/out: decided slots are kept,
 *                open slots get their drawn token
 *   tau          device int32[total_B] out (may be tau_prev itself)
 *   confidence   device float32[total_B] out or NULL: max_v q(v) of open
 *                slots, -1 at decided ones
 * Kernels: with a workspace of simsd_draft_workspace_size bytes and no
 * decided slots, a chunk pass over (row, 32 KB chunk) items on every SM
 * (per eighth of a chunk: maximum, sum of exponentials, largest logit),
 * then one CTA per sequence: a warp per slot merges its row's parts, finds
 * the part holding u*S and scans it; a wait of the chunk pass that gives
 * up sets the timeout bit and leaves every tokens and tau entry of the
 * call unwritten.  Otherwise one thread-block cluster per sequence (as
 * simsd_accept's rules): one pass over every open row for its normaliser,
 * then each slot's inverse-CDF scan in the vocabulary slice holding u*S.
 * Errors: as simsd_accept (SIMSD_ERR_SHAPE also for a negative or
 * non-finite temperature).  Bad device arrays (cu_B, decided outside
 * 0..B_b, tau_prev not a permutation) set the bad-input bit and leave the
 * sequence's tokens and tau unwritten.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t batch;
  int32_t vocab;
  int32_t total_B;            /* host copy                                  */
  int32_t B_max;              /* host copy, 1..32                           */
  simsd_dtype dtype;          /* of the logits                              */
  float temperature;          /* > 0; 0 selects 1                           */
  const void *draft_logits;
  const int32_t *cu_B;
  const float *uniforms;
  const int32_t *decided;
  const int32_t *tau_prev;
  int32_t *tokens;
  int32_t *tau;
  float *confidence;
  void *workspace;            /* device, 256-byte aligned: the status word,
                                 or simsd_draft_workspace_size bytes (256 +
                                 total_B ceil(vocab / E) * 128 rounded up to
                                 a multiple of 256, E as in simsd_accept)
                                 for the chunked path                      */
  size_t workspace_bytes;
} simsd_draft_desc;

size_t simsd_draft_workspace_size(const simsd_draft_desc *d);
simsd_status simsd_draft_step(const simsd_draft_desc *d, void *stream);

/* ------------------------------------------------------------------------
 * simsd_commit -- section 4: "the longest accepted prefix is committed, and
 * the process is repeated", with the KV cache and blockwise decoding
 * (section "Contributions").  One pass of the blockwise loop is
 * simsd_draft_step -> simsd_verify_attn -> simsd_accept (decided) ->
 * simsd_commit.  For sequence b, with the walk's n_accept, token, pos:
 *   - positions with tau <= n_accept stay decided with their tokens;
 *   - a rejection (pos >= 0) decides position pos with the drawn token
 *     (written to tokens[pos]); it holds label n_accept + 1, so
 *     decided[b] = n_accept + 1;
 *   - every position decided by a pass that drew nothing (n_accept = B_b,
 *     pos = -1): the cache slots [lens, lens+B_b) written by that pass's
 *     verification hold the final tokens' keys and values, so the block
 *     closes: lens[b] += B_b, decided[b] = 0, done[b] = 1 (the mask-slot
 *     slots past them are free again).  A block whose last position was
 *     decided by a draw stays open with decided[b] = B_b: its next pass
 *     tests nothing, rewrites the section's keys and values from the final
 *     tokens, and closes it.
 *   tau, cu_B, n_accept, token, pos  device, as written by simsd_accept
 *   tokens   device int32[total_B] in/out (the pass's data-section tokens)
 *   decided  device int32[batch] in/out
 *   lens     device int32[batch] in/out
 *   done     device int32[batch] out
 * A sequence whose arrays are inconsistent (cu_B outside 0..total_B, B_b
 * outside 1..B_max, a walk that does not fit its tau) sets the bad-input
 * bit and is left unchanged (done = 0).  One thread per sequence.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t batch;
  int32_t total_B;            /* host copy                                  */
  int32_t B_max;              /* host copy, 1..32                           */
  const int32_t *cu_B;
  const int32_t *tau;
  const int32_t *n_accept;
  const int32_t *token;
  const int32_t *pos;
  int32_t *tokens;
  int32_t *decided;
  int32_t *lens;
  int32_t *done;
  void *workspace;            /* device, 256-byte aligned (status word)     */
  size_t workspace_bytes;
} simsd_commit_desc;

size_t simsd_commit_workspace_size(const simsd_commit_desc *d);
simsd_status simsd_commit(const simsd_commit_desc *d, void *stream);

/* ------------------------------------------------------------------------
 * simsd_accept_noalloc -- simsd_accept for callers that cannot allocate
 * device memory.  (No counterpart in the SimSD paper: it is a deployment
 * convenience.)  Some callers never get to call cudaMalloc: a serving loop
 * that runs the acceptance step under a fixed memory budget and must not
 * allocate per request (an allocation can fail under memory pressure, or
 * stall the device mid-request), or a plugin whose host framework owns all
 * device memory and hands it only the input and output tensors.  This entry
 * point takes the same descriptor, ignores its workspace fields, and keeps
 * its scratch in a static device array of SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES
 * bytes that every GPU loading the library holds until the process exits.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - It runs the two-kernel path where its chunk partials (which grow
 *     with total_B and vocab) fit the array, and the single-launch path,
 *     whose scratch is one status word for every size, otherwise; a
 *     scratch need beyond the array would be rejected with
 *     SIMSD_ERR_WORKSPACE before any launch.
 *   - The first call on each device looks up the array's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the one array per device (zero at load time) and it
 *     keeps the previous call's contents.  Calls that
 *     overlap on the GPU -- on different streams, or from several host
 *     threads -- race on it: serialise them.
 *   - The kernels' status word lives in that array, so simsd_read_status
 *     cannot read it; device-detected input errors are not reported here.
 *   - The address is cached per device ordinal for the life of the process:
 *     it assumes the device's primary context (the one the CUDA runtime
 *     uses) and no cudaDeviceReset in between.
 * ---------------------------------------------------------------------- */
#define SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES ((size_t)4096)
simsd_status simsd_accept_noalloc(const simsd_accept_desc *d, void *stream);

/* ------------------------------------------------------------------------
 * simsd_read_status -- synchronise `stream`, copy the device status word of
 * a workspace used by simsd_verify_attn / simsd_accept to *word_out (bit 0:
 * a bounded wait ran out) and clear it, together with the chunk pass's
 * control words (bytes 128..139 of a workspace, zero between calls).  Returns SIMSD_ERR_TIMEOUT when a
 * bit was set, SIMSD_OK otherwise, SIMSD_ERR_CUDA on a CUDA error.
 * ---------------------------------------------------------------------- */
simsd_status simsd_read_status(void *workspace, void *stream,
                               uint32_t *word_out);

#ifdef __cplusplus
}
#endif
#endif /* SIMSD_H */
