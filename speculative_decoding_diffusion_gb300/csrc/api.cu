// api.cu -- host side of the C ABI: argument checks, planning, launches.
//
// simsd_layout follows SimSD sections 1-3 (paired layout, temporal mask,
// RoPE copy); simsd_verify_attn and simsd_prompt_append plan and launch the
// kernels K1-K3; the acceptance entry points live in accept.cu.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace simsd {

// SMs of the current device (a GB300's 152 when no device is visible, so
// that workspace sizes queried on a host without a GPU match the plan one
// would make on it)
int device_sm_count() {
  constexpr int kDefaultSms = 152;
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return kDefaultSms;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = kDefaultSms;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

}  // namespace

static bool encode_cache_map(CUtensorMap *m, void *ptr, int num_pages, int Hkv, int hd) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)kPageTokens, (cuuint64_t)Hkv,
                        (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)kPageTokens * hd * 2,
                           (cuuint64_t)Hkv * kPageTokens * hd * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kPageTokens, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


int current_device() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

bool make_cache_map(CUtensorMap *m, void *ptr, int num_pages, int Hkv, int hd) {
  struct Entry {
    int dev, num_pages, Hkv, hd;
    void *ptr;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int used = 0, next = 0;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    const Entry &e = cache[i];
    if (e.dev == dev && e.ptr == ptr && e.num_pages == num_pages && e.Hkv == Hkv && e.hd == hd) {
      *m = e.map;
      return true;
    }
  }
  if (!encode_cache_map(m, ptr, num_pages, Hkv, hd)) return false;
  Entry &e = cache[next];
  e.dev = dev; e.ptr = ptr; e.num_pages = num_pages; e.Hkv = Hkv; e.hd = hd; e.map = *m;
  next = (next + 1) % 16;
  if (used < 16) ++used;
  return true;
}

bool record_event(void *event, cudaStream_t stream) {
  if (event == nullptr) return true;
  return cudaEventRecordWithFlags((cudaEvent_t)event, stream, cudaEventRecordExternal) ==
         cudaSuccess;
}

static void fill_rope_table(float base, int hd, RopeTable *t) {
  memset(t, 0, sizeof(*t));
  for (int d = 0; d < hd / 2 && d < 64; ++d) {
    t->inv_freq[d] = pow((double)base, -2.0 * (double)d / (double)hd);
    t->hi[d] = (float)t->inv_freq[d];
    t->lo[d] = (float)(t->inv_freq[d] - (double)t->hi[d]);
  }
}

void make_rope_table(float base, int hd, RopeTable *t) {
  static std::mutex mu;
  static float last_base = 0.f;
  static int last_hd = 0;
  static RopeTable last;
  std::lock_guard<std::mutex> lock(mu);
  if (last_hd != hd || last_base != base) {
    fill_rope_table(base, hd, &last);
    last_base = base;
    last_hd = hd;
  }
  *t = last;
}

static bool valid_dtype(simsd_dtype t) { return t == SIMSD_F32 || t == SIMSD_BF16; }

simsd_status verify_plan(const simsd_verify_desc *d, VerifyPlan *p) {
  if (d == nullptr || p == nullptr) return SIMSD_ERR_NULL;
  if (!valid_dtype(d->dtype)) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 ||
      d->num_q_heads % d->num_kv_heads != 0 ||
      (d->head_dim != 64 && d->head_dim != 128) || d->page_size != kPageTokens ||
      d->num_pages < 1 || d->max_pages_per_seq < 1 || d->B_max < 1 ||
      d->B_max > kMaxB || d->total_B < d->batch ||
      (int64_t)d->total_B > (int64_t)d->batch * d->B_max)
    return SIMSD_ERR_SHAPE;
  if (!(d->sm_scale > 0.0f) || !(d->sm_scale < INFINITY) || !(d->rope_base > 1.0f) ||
      d->node_size < 0 || d->node_size > kMaxB)
    return SIMSD_ERR_SHAPE;
  memset(p, 0, sizeof(*p));
  p->T = 2 * d->total_B;
  p->G = d->num_q_heads / d->num_kv_heads;
  p->M_max = 2 * d->B_max * p->G;
  p->esize = d->dtype == SIMSD_BF16 ? 2 : 4;
  if ((size_t)(d->num_q_heads + 2 * d->num_kv_heads) * d->head_dim * p->esize > kMaxRowBytes)
    return SIMSD_ERR_SHAPE;
  if (d->dtype == SIMSD_BF16) {
    p->rows_per_tile = 128;   // the tensor-core tile's M; smaller tiles are padded
    p->key_splits = 1;
  } else {
    p->rows_per_tile = p->M_max;
    p->key_splits = 1;
  }
  p->row_tiles = (p->M_max + p->rows_per_tile - 1) / p->rows_per_tile;
  // Split each sequence's keys into `splits` ranges of whole 128-key blocks.
  // Cost model in block-times (one 128-key block per SM with every SM
  // streaming at the DRAM-bound rate; one CTA per SM): a wave of n CTAs of
  // `per` blocks takes per * max(n / sms, kRho) -- DRAM-bound while at
  // least kRho of the SMs stream, each SM at its own rate below that (kRho
  // = K2's best GPU-wide rate, ~6.5 TB/s, over 152 SMs' own ~50 GB/s) --
  // plus kRamp per wave (a CTA's setup and first copies, ~4.5 us) and, when
  // split, the merge's read of the partials.  The longest possible sequence
  // (the block-table width) stands for every sequence.  (On the 8 x 32768
  // workload this picks 2 splits, one wave of 128 CTAs: K2 204 -> 188 us
  // against the 7 splits in 3 waves an earlier model chose.)
  const int64_t max_keys = (int64_t)d->max_pages_per_seq * kPageTokens;
  const int64_t max_blocks = (max_keys + kBlockKeys - 1) / kBlockKeys;
  const int64_t pairs = (int64_t)d->batch * d->num_kv_heads * p->row_tiles;
  const int64_t sms = device_sm_count();
  constexpr double kRho = 0.85, kRamp = 3.0;
  int64_t splits = 1;
  double best = 1e300;
  for (int64_t s = 1; s <= max_blocks && s <= 64; ++s) {
    const int64_t per = (max_blocks + s - 1) / s;
    if (s > 1 && (max_blocks + per - 1) / per < s) continue;   // same split as a smaller s
    const int64_t ctas = pairs * s, full = ctas / sms, rest = ctas % sms;
    double cost = (double)(full * per) + kRamp * (double)full;
    if (rest > 0) cost += (double)per * std::max((double)rest / (double)sms, kRho) + kRamp;
    if (s > 1) cost += (double)ctas / (double)sms;
    if (cost < best - 1e-9) { best = cost; splits = s; }
  }
  int64_t blocks_per_split = (max_blocks + splits - 1) / splits;
  p->chunk = (int)(blocks_per_split * kBlockKeys);
  p->n_splits = (int)((max_keys + p->chunk - 1) / p->chunk);
  // every unit split alike, or none
  p->tail_from = p->n_splits > 1 ? 0 : (int)pairs;
  p->tail_first = 0;
  p->s_tail = p->n_splits;
  p->chunk_tail = p->chunk;
  p->grid = (int)(pairs * p->n_splits);
  p->merge_rows = (int64_t)p->T * d->num_q_heads;
  if (d->dtype == SIMSD_BF16 && p->n_splits == 1 && pairs > sms && pairs % sms != 0) {
    // Whole units in full waves, then the last partial wave's r units in
    // s = sms / r splits each: that wave takes a split's time instead of a
    // unit's (same block-time model, plus the split merge's read).
    const int64_t W = pairs / sms, r = pairs - W * sms;
    const int64_t s = std::min<int64_t>(sms / r, max_blocks);
    if (s >= 2) {
      const int64_t per = (max_blocks + s - 1) / s;
      const double whole = (double)(W + 1) * ((double)max_blocks + 1.5);
      const double tail = (double)W * ((double)max_blocks + 1.5) + ((double)per + 2.5) +
                          (double)(r * s) / (double)sms;
      if (tail < whole - 1e-9) {
        p->tail_from = (int)(W * sms);
        // With few full waves the split units go first: the SMs that ran
        // them then run whole units offset by a split, so the wave
        // boundaries' ramps no longer coincide (64 x 4096: K2 208 -> 201
        // us).  With many waves they go last, where they even out the end
        // of a ragged batch (ragged 256: first, 716 -> 730 us).
        p->tail_first = W <= 4;
        p->s_tail = (int)s;
        p->chunk_tail = (int)(per * kBlockKeys);
        p->n_splits = (int)((max_keys + p->chunk_tail - 1) / p->chunk_tail);
        p->grid = (int)(W * sms + r * s);
        // the split units belong to the last ceil(r / units per sequence)
        // (+1 for a sequence cut by the boundary) sequences, whose tokens
        // are the last ones
        const int64_t per_seq = (int64_t)d->num_kv_heads * p->row_tiles;
        const int64_t seqs = std::min<int64_t>(d->batch, (r + per_seq - 1) / per_seq + 1);
        p->merge_rows = std::min<int64_t>(p->merge_rows, seqs * 2 * d->B_max * d->num_q_heads);
      }
    }
  }
  // workspace
  size_t off = 0;
  p->off_status = off;  off = align_up(off + sizeof(uint32_t), kAlign);
  p->off_qrot = off;    // rotated queries: the fp32 path only (the bf16 kernel rotates its own)
  if (d->dtype == SIMSD_F32)
    off = align_up(off + (size_t)p->T * d->num_q_heads * d->head_dim * p->esize, kAlign);
  p->off_tokinfo = off;  off = align_up(off + (size_t)p->T * sizeof(int4), kAlign);
  p->off_opart = off;
  if (p->n_splits > 1) {
    off = align_up(off + (size_t)p->n_splits * p->T * d->num_q_heads * d->head_dim * sizeof(float), kAlign);
    p->off_ml = off;
    off = align_up(off + (size_t)p->n_splits * p->T * d->num_q_heads * sizeof(float2), kAlign);
  } else {
    p->off_ml = off;
  }
  p->total = off;
  return SIMSD_OK;
}

}  // namespace simsd

using namespace simsd;

extern "C" {

const char *simsd_status_string(int status) {
  switch (status) {
    case SIMSD_OK: return "ok";
    case SIMSD_ERR_NULL: return "a required pointer is NULL";
    case SIMSD_ERR_SHAPE: return "a size is out of range or inconsistent";
    case SIMSD_ERR_TAU: return "tau is not a permutation of 1..B";
    case SIMSD_ERR_DTYPE: return "unsupported dtype";
    case SIMSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SIMSD_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case SIMSD_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case SIMSD_ERR_ALIGN: return "a device array is not 16-byte aligned";
    default: return "unknown status";
  }
}

int simsd_version(void) { return 100; }

simsd_status simsd_layout(int32_t P, int32_t B, const int32_t *tau,
                          int32_t *positions, uint8_t *mask) {
  if (tau == nullptr || positions == nullptr) return SIMSD_ERR_NULL;
  if (P < 0 || B < 1 || B > kMaxB) return SIMSD_ERR_SHAPE;
  // tau must label the B response positions with the steps 1..B, each once
  uint32_t seen = 0;
  for (int k = 0; k < B; ++k) {
    const int t = tau[k];
    if (t < 1 || t > B || (seen >> (t - 1)) & 1u) return SIMSD_ERR_TAU;
    seen |= 1u << (t - 1);
  }
  for (int j = 0; j < P; ++j) positions[j] = j;
  for (int k = 0; k < B; ++k) {
    positions[P + k] = P + k;      // data token D_{k+1}
    positions[P + B + k] = P + k;  // slot D~_{k+1}: RoPE index copied
  }
  if (mask != nullptr) {
    const int64_t L = (int64_t)P + 2 * B;
    for (int r = 0; r < 2 * B; ++r) {
      uint8_t *row = mask + (int64_t)r * L;
      memset(row, 1, (size_t)P);
      const bool slot_row = r >= B;
      const int ti = tau[slot_row ? r - B : r];
      for (int j = 0; j < B; ++j) {
        const int tj = tau[j];
        // data columns: slots see strictly earlier steps, data rows see
        // their own step and earlier ones
        row[P + j] = slot_row ? (tj < ti) : (tj <= ti);
        // slot columns: slots see their own and later steps, data rows none
        row[P + B + j] = slot_row ? (tj >= ti) : 0;
      }
    }
  }
  return SIMSD_OK;
}

size_t simsd_verify_workspace_size(const simsd_verify_desc *d) {
  VerifyPlan p;
  if (verify_plan(d, &p) != SIMSD_OK) return 0;
  return p.total;
}

simsd_status simsd_verify_attn(const simsd_verify_desc *d, void *stream_ptr) {
  return simsd_verify_attn_timed(d, stream_ptr, nullptr);
}

static bool mark(void *const *events, int i, cudaStream_t stream) {
  return events == nullptr || record_event(events[i], stream);
}

simsd_status simsd_verify_attn_timed(const simsd_verify_desc *d, void *stream_ptr,
                                     void *const events[4]) {
  VerifyPlan p;
  simsd_status st = verify_plan(d, &p);
  if (st != SIMSD_OK) return st;
  if (!d->q || !d->k_cache || !d->v_cache || !d->block_table || !d->k_new ||
      !d->v_new || (d->node_size == 0 && !d->tau) || !d->lens || !d->cu_B || !d->out)
    return SIMSD_ERR_NULL;
  if (!aligned16(d->q) || !aligned16(d->k_cache) || !aligned16(d->v_cache) ||
      !aligned16(d->k_new) || !aligned16(d->v_new) || !aligned16(d->out))
    return SIMSD_ERR_ALIGN;
  if (d->workspace == nullptr || ((uintptr_t)d->workspace % kAlign) != 0 ||
      d->workspace_bytes < p.total)
    return SIMSD_ERR_WORKSPACE;
  cudaStream_t stream = (cudaStream_t)stream_ptr;
  char *ws = (char *)d->workspace;
  uint32_t *status = (uint32_t *)(ws + p.off_status);
  void *q_rot = ws + p.off_qrot;
  int4 *tok_info = (int4 *)(ws + p.off_tokinfo);
  if (!mark(events, 0, stream) ||
      launch_rope_verify(d, p, q_rot, tok_info, status, stream) != cudaSuccess ||
      !mark(events, 1, stream))
    return SIMSD_ERR_CUDA;
  AttnParams a;
  memset(&a, 0, sizeof(a));
  a.q = d->q;
  a.q_rot = q_rot;
  make_rope_table(d->rope_base, d->head_dim, &a.tab);
  a.out = d->out;
  a.o_part = (float *)(ws + p.off_opart);
  a.ml_part = (float2 *)(ws + p.off_ml);
  a.tau = d->tau;
  a.lens = d->lens;
  a.cu_B = d->cu_B;
  a.block_table = d->block_table;
  a.k_cache = d->k_cache;
  a.v_cache = d->v_cache;
  a.status = status;
  a.max_pages_per_seq = d->max_pages_per_seq;
  a.num_pages = d->num_pages;
  a.batch = d->batch;
  a.Hq = d->num_q_heads;
  a.Hkv = d->num_kv_heads;
  a.G = p.G;
  a.T = p.T;
  a.total_B = d->total_B;
  a.B_max = d->B_max;
  a.polls = wait_polls_of(d->wait_polls);
  a.node_size = d->node_size;
  a.chunk = p.chunk;
  a.tail_from = p.tail_from;
  a.s_tail = p.s_tail;
  a.chunk_tail = p.chunk_tail;
  a.tail_first = p.tail_first;
  a.row_tiles = p.row_tiles;
  a.rows_per_tile = p.rows_per_tile;
  a.sm_scale = d->sm_scale;
  cudaError_t e = d->dtype == SIMSD_BF16 ? launch_attn_tc(d, p, a, stream)
                                         : launch_attn_f32(d, p, a, stream);
  if (e != cudaSuccess || !mark(events, 2, stream)) return SIMSD_ERR_CUDA;
  if (p.n_splits > 1 && launch_combine(d, p, a, tok_info, stream) != cudaSuccess)
    return SIMSD_ERR_CUDA;
  return mark(events, 3, stream) ? SIMSD_OK : SIMSD_ERR_CUDA;
}

simsd_status simsd_prompt_append(const simsd_append_desc *d, void *stream_ptr) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (!valid_dtype(d->dtype)) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->num_kv_heads < 1 ||
      (d->head_dim != 64 && d->head_dim != 128) || d->page_size != kPageTokens ||
      d->num_pages < 1 || d->max_pages_per_seq < 1 || d->total_n < 0 ||
      !(d->rope_base > 1.0f))
    return SIMSD_ERR_SHAPE;
  if (!d->k || !d->v || !d->start || !d->cu_n || !d->k_cache || !d->v_cache ||
      !d->block_table)
    return SIMSD_ERR_NULL;
  if (!aligned16(d->k) || !aligned16(d->v) || !aligned16(d->k_cache) || !aligned16(d->v_cache))
    return SIMSD_ERR_ALIGN;
  if (d->total_n == 0) return SIMSD_OK;
  return launch_rope_append(d, (cudaStream_t)stream_ptr) == cudaSuccess ? SIMSD_OK
                                                                        : SIMSD_ERR_CUDA;
}

simsd_status simsd_read_status(void *workspace, void *stream_ptr, uint32_t *word_out) {
  if (workspace == nullptr) return SIMSD_ERR_NULL;
  cudaStream_t stream = (cudaStream_t)stream_ptr;
  uint32_t w = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SIMSD_ERR_CUDA;
  if (cudaMemcpy(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SIMSD_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(w)) != cudaSuccess ||
      cudaMemset((char *)workspace + kClaimOffset, 0, kClaimBytes) != cudaSuccess)
    return SIMSD_ERR_CUDA;
  if (word_out) *word_out = w;
  return w ? SIMSD_ERR_TIMEOUT : SIMSD_OK;
}

}  // extern "C"
