// internal.h -- host-side plan and kernel launchers of libsimsd (not ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/simsd.h"

namespace simsd {

constexpr int kBlockKeys = 128;   // keys per pipeline stage of the attention
constexpr int kPageTokens = 16;  // tokens per KV-cache page (ABI page_size)
constexpr int kMaxB = 32;
constexpr size_t kMaxRowBytes = 192 * 1024;   // raw q + k + v of one new token (staged in smem)

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
constexpr size_t kAlign = 256;
// The first kAlign bytes of every workspace: the status word at offset 0
// and, for the chunked acceptance and draft paths, the chunk pass's three
// control words at this fixed offset (the same place for every size, so a
// workspace reused at another size never finds partials there);
// simsd_read_status clears both.
constexpr size_t kClaimOffset = 128;
constexpr size_t kClaimBytes = 3 * sizeof(int);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Everything simsd_verify_attn derives on the host from the descriptor.
struct VerifyPlan {
  int T;             // new tokens, 2 * total_B
  int G;             // query heads per KV head
  int M_max;         // max query rows per (sequence, KV head): 2 * B_max * G
  int rows_per_tile; // query rows one CTA owns
  int row_tiles;     // CTAs per (sequence, KV head, split) along the rows
  int key_splits;    // warps sharing one stage's keys (mma path)
  int chunk;         // keys per split (multiple of kBlockKeys)
  int n_splits;      // most splits of any unit (partials buffers)
  // Units (sequence, KV head, row tile): the first tail_from run whole,
  // each later one in s_tail splits of chunk_tail keys (tail_from = 0:
  // every unit split; tail_from = units: none).  The split units' CTAs are
  // launched after the whole ones, or before them when tail_first.
  int tail_from, s_tail, chunk_tail, grid;
  int tail_first;
  // the split merge's rows: the last merge_rows of the T * Hq rows (the
  // split units' sequences are the last ones; all rows when every unit is
  // split)
  int64_t merge_rows;
  size_t esize;      // bytes per q/k/v/out element
  // workspace carve-up (byte offsets)
  size_t off_status, off_qrot, off_tokinfo, off_opart, off_ml, total;
};

// Fills *plan; returns SIMSD_OK or the first argument error.
simsd_status verify_plan(const simsd_verify_desc *d, VerifyPlan *plan);

// RoPE inverse frequencies base^(-2d/hd), d < hd/2, computed in double on
// the host and passed both as double and as a pair of floats hi + lo.
struct RopeTable {
  double inv_freq[64];
  float hi[64], lo[64];
};
void make_rope_table(float base, int hd, RopeTable *t);   // cached per (base, hd)

// Parameters every attention kernel reads.
struct AttnParams {
  const void *q;              // [T][Hq][hd], raw (the bf16 kernel rotates it)
  const void *q_rot;          // [T][Hq][hd], rotated by K1 (fp32 path)
  void *out;                  // [T][Hq][hd]
  float *o_part;              // [n_splits][T][Hq][hd]
  float2 *ml_part;            // [n_splits][T][Hq]  (running max, sum)
  const int32_t *tau;
  const int32_t *lens;
  const int32_t *cu_B;
  const int32_t *block_table;
  const void *k_cache;        // fp32 path reads the cache directly
  const void *v_cache;
  uint32_t *status;
  int max_pages_per_seq;
  int num_pages;
  int batch;
  int Hq, Hkv, G, T;
  int total_B, B_max;         // host copies: a sequence's cu_B and B must fit them
  int node_size;              // 0: SimSD's temporal layout; > 0: draft-graph nodes
  int chunk, rows_per_tile;
  int tail_from, s_tail, chunk_tail;   // as in VerifyPlan
  int tail_first;             // as in VerifyPlan
  int row_tiles;
  uint32_t polls;             // bounded-wait polls (wait_polls_of the descriptor)
  float sm_scale;
  RopeTable tab;              // angles of the query rotation (bf16 kernel)
};

// K1: rotate q and k_new at the layout positions, append k/v to the cache.
cudaError_t launch_rope_verify(const simsd_verify_desc *d, const VerifyPlan &p,
                               void *q_rot, int4 *tok_info, uint32_t *status,
                               cudaStream_t stream);
cudaError_t launch_rope_append(const simsd_append_desc *d, cudaStream_t stream);

// K2: split-KV masked attention (tcgen05 for bf16, CUDA cores for fp32).
cudaError_t launch_attn_tc(const simsd_verify_desc *d, const VerifyPlan &p,
                           const AttnParams &a, cudaStream_t stream);
cudaError_t launch_attn_f32(const simsd_verify_desc *d, const VerifyPlan &p,
                            const AttnParams &a, cudaStream_t stream);

// K3: merge split partials.
cudaError_t launch_combine(const simsd_verify_desc *d, const VerifyPlan &p,
                           const AttnParams &a, const int4 *tok_info,
                           cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// TMA descriptor of a paged bf16 cache [num_pages][Hkv][16][hd] as the 4-D
// tensor (hd, slot, head, page); one box = one page of one head, 64 columns
// (128 bytes) wide, 128-byte swizzle.  False if the CUDA driver's tensor-map
// encoding fails.  Descriptors are cached per (device, pointer, sizes):
// repeated calls on the same cache encode nothing.
bool make_cache_map(CUtensorMap *m, void *ptr, int num_pages, int Hkv, int hd);

// Records `event` (a cudaEvent_t, may be NULL) on `stream`; under stream
// capture it becomes an event-record node of the graph, so a replayed graph
// still yields per-kernel times.
bool record_event(void *event, cudaStream_t stream);

// Current device, or -1.
int current_device();

// Launch `kern` with programmatic stream serialisation: it may begin while
// the previous kernel on `stream` still runs, and waits for it on the device
// (grid_dep_wait) before reading its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}


// The draft-side step's chunk pass over the draft rows (accept.cu): per
// (row, 32 KB chunk, consumer warp) the reference, the sum of 2^(l ls -
// reference) and the part's largest logit, into part4 [total_B][nchunks][8].
// claim[0..2] must be zero; the finishing kernel zeroes them again.
int draft_chunk_entries(int esize);
cudaError_t launch_draft_chunks(const simsd_draft_desc *d, float4 *part4, int *claim,
                                uint32_t *status, int nchunks, cudaStream_t stream);

}  // namespace simsd
