// rope_append.cu -- K1: RoPE-copy rotation and paged KV append.
//
// SimSD section 3 "Position Encoding Alignment": each mask slot D~_k reuses
// the RoPE index of its data token D_k, so both new tokens of response
// position k (1-based) of a sequence with prompt length P rotate at P+k-1.
// Section 1 "Input Layout": the 2B new tokens occupy layout indices
// P .. P+2B-1 (D_1..D_B then D~_1..D~_B); those are the cache slots written.
//
// One CTA per new token; angles from rope.cuh (float-pair product and
// Cody-Waite reduction), the rotation in fp32.  The bf16 attention kernel
// rotates its own query tile, so the queries are rotated here only for the
// fp32 path.
// Rotate-half pairing: element d pairs with d + hd/2.  16-byte vector I/O.
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "rope.cuh"

namespace simsd {
namespace {

constexpr int kThreads = 128;

// Angles for one position into smem: cs[d] = (cos, sin) of frequency d.
__device__ __forceinline__ void angles(const RopeTable &tab, int hd, int pos, float2 *cs) {
  for (int d = threadIdx.x; d < hd / 2; d += blockDim.x) cs[d] = rope_cs(tab, d, pos);
}

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  using V = float4;
  static __device__ __forceinline__ void unpack(const V &v, float *f) {
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  static __device__ __forceinline__ V pack(const float *f) {
    return make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  using V = uint4;
  static __device__ __forceinline__ void unpack(const V &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ V pack(const float *f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
};

// Rotate `heads` rows of hd elements from src into dst (row h at h*hd; dst
// rows at dst_stride apart) with the angles in cs.  Each thread loads a
// batch of its vectors before storing any, so global loads are in flight
// together rather than serialised behind possibly aliasing stores (a
// source in shared memory takes BATCH 1: fewer registers, more CTAs).
template <typename T, int BATCH>
__device__ __forceinline__ void rotate_rows(const T *__restrict__ src, T *__restrict__ dst,
                                            int heads, int hd, long dst_stride,
                                            const float2 *cs) {
  using VT = Vec<T>;
  constexpr int N = VT::N;
  const int half = hd / 2;
  const int per_head = half / N;  // vector pairs per head
  const int items = heads * per_head;
  for (int i0 = threadIdx.x; i0 < items; i0 += BATCH * blockDim.x) {
    typename VT::V va[BATCH], vb[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < items) {
        const T *x = src + (long)(i / per_head) * hd + (i % per_head) * N;
        va[u] = *reinterpret_cast<const typename VT::V *>(x);
        vb[u] = *reinterpret_cast<const typename VT::V *>(x + half);
      }
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i >= items) break;
      const int h = i / per_head, d0 = (i % per_head) * N;
      float x1[N], x2[N], y1[N], y2[N];
      VT::unpack(va[u], x1);
      VT::unpack(vb[u], x2);
#pragma unroll
      for (int j = 0; j < N; ++j) {
        const float c = cs[d0 + j].x, sn = cs[d0 + j].y;
        y1[j] = x1[j] * c - x2[j] * sn;
        y2[j] = x2[j] * c + x1[j] * sn;
      }
      T *y = dst + (long)h * dst_stride;
      *reinterpret_cast<typename VT::V *>(y + d0) = VT::pack(y1);
      *reinterpret_cast<typename VT::V *>(y + d0 + half) = VT::pack(y2);
    }
  }
}

template <typename T, int BATCH>
__device__ __forceinline__ void copy_rows(const T *__restrict__ src, T *__restrict__ dst,
                                          int heads, int hd, long dst_stride) {
  using VT = Vec<T>;
  constexpr int N = VT::N;
  const int per_head = hd / N;
  const int items = heads * per_head;
  for (int i0 = threadIdx.x; i0 < items; i0 += BATCH * blockDim.x) {
    typename VT::V v[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < items)
        v[u] = *reinterpret_cast<const typename VT::V *>(src + (long)(i / per_head) * hd +
                                                         (i % per_head) * N);
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i >= items) break;
      *reinterpret_cast<typename VT::V *>(dst + (long)(i / per_head) * dst_stride +
                                          (i % per_head) * N) = v[u];
    }
  }
}

struct RopeVerifyArgs {
  RopeTable tab;
  const void *q;
  const void *k_new;
  const void *v_new;
  void *q_rot;
  void *k_cache;
  void *v_cache;
  const int32_t *block_table;
  const int32_t *lens;
  const int32_t *cu_B;
  int4 *tok_info;       // [T]: (keys of the sequence or 0 if malformed, its first
                        // unit, the token's index in the section, -)
  uint32_t *status;
  int batch, Hq, Hkv, hd, max_pages, num_pages;
  int row_tiles;        // row tiles per (sequence, KV head) of the attention kernel
  int total_B, B_max;   // host copies: a sequence's cu_B and B must fit them
  uint32_t polls;       // bounded-wait polls
  int node_size;        // 0: SimSD's paired layout; > 0: draft-graph nodes
  int rotate_q;         // write rotated queries to q_rot (fp32 path)
};

// sequences whose cu_B / lens are staged in shared memory; kept small so
// the attention kernel's CTAs (launched early, programmatic dependent
// launch) fit on the same SMs as this kernel's
constexpr int kStageSeqs = 512;

// 16 CTAs (2048 threads) per SM at bf16 (32 registers, no spills): a batch
// of a few thousand new tokens runs in about one wave of CTAs
template <typename T>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 16 : 12)
rope_verify_kernel(const __grid_constant__ RopeVerifyArgs a) {
  extern __shared__ __align__(16) uint8_t rows_s[];   // raw q | k | v rows of the token
  __shared__ float2 cs[64];
  __shared__ int32_t cu_s[kStageSeqs + 1], lens_s[kStageSeqs];
  __shared__ __align__(8) uint64_t bar_s;
  grid_dep_launch();                         // the attention kernel may start its prologue
  const int r = blockIdx.x;                  // new-token row
  const uint32_t qbytes = a.rotate_q ? (uint32_t)(a.Hq * a.hd * sizeof(T)) : 0u;
  const uint32_t kvbytes = (uint32_t)(a.Hkv * a.hd * sizeof(T));
  const uint32_t bar = smem_u32(&bar_s), rows = smem_u32(rows_s);
  // the token's raw rows are needed whatever its sequence: one thread starts
  // three bulk copies into shared memory before anything else
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, qbytes + 2 * kvbytes);
    if (qbytes) bulk_load(rows, (const char *)a.q + (long)r * qbytes, qbytes, bar);
    bulk_load(rows + qbytes, (const char *)a.k_new + (long)r * kvbytes, kvbytes, bar);
    bulk_load(rows + qbytes + kvbytes, (const char *)a.v_new + (long)r * kvbytes, kvbytes, bar);
  }
  // sequence of the token: cu_B (and lens) staged once, searched in smem
  int b, c0, B, P;
  if (a.batch <= kStageSeqs) {
    // every load is issued before the first store to shared memory, so the
    // staging costs one round trip, not one per loop step
    constexpr int kCu = (kStageSeqs + 1 + kThreads - 1) / kThreads, kLen = kStageSeqs / kThreads;
    int cu_v[kCu], len_v[kLen];
#pragma unroll
    for (int u = 0; u < kCu; ++u) {
      const int i = threadIdx.x + u * kThreads;
      cu_v[u] = i <= a.batch ? __ldg(a.cu_B + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kLen; ++u) {
      const int i = threadIdx.x + u * kThreads;
      len_v[u] = i < a.batch ? __ldg(a.lens + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kCu; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i <= a.batch) cu_s[i] = cu_v[u];
    }
#pragma unroll
    for (int u = 0; u < kLen; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i < a.batch) lens_s[i] = len_v[u];
    }
    __syncthreads();
    b = find_seq_smem(cu_s, a.batch, r >> 1);
    c0 = cu_s[b];
    B = cu_s[b + 1] - c0;
    P = lens_s[b];
  } else {
    b = find_seq(a.cu_B, a.batch, r >> 1);
    c0 = __ldg(a.cu_B + b);
    B = __ldg(a.cu_B + b + 1) - c0;
    P = __ldg(a.lens + b);
  }
  const int j = r - 2 * c0;                  // 0..2B-1 within the sequence
  // response index (0-based): D~_k copies D_k's position; in the
  // draft-graph layout every node's token k sits at the same position
  const int k = a.node_size > 0 ? j % a.node_size : (j < B ? j : j - B);
  const int pos = P + k;
  const int slot = P + j;                    // layout index = cache slot
  bool ok = !(B < 1 || B > kMaxSection || B > a.B_max || c0 < 0 || c0 + B > a.total_B ||
              j < 0 || j >= 2 * B || P < 0 || (long)P + 2 * B > (long)a.max_pages * kPage ||
              (a.node_size > 0 && (2 * B) % a.node_size != 0));
  const int page = ok ? __ldg(a.block_table + (long)b * a.max_pages + slot / kPage) : -1;
  // the angles need only the position: computed while the page is loaded
  if (ok) angles(a.tab, a.hd, pos, cs);
  ok = ok && page >= 0 && page < a.num_pages;   // cu_B or block table out of range
  // the split merge reads it: which of its rows were split, without a search
  if (threadIdx.x == 0) a.tok_info[r] = make_int4(ok ? P + 2 * B : 0, b * a.Hkv * a.row_tiles, j, 0);
  if (!ok && threadIdx.x == 0) raise_status(a.status, kStatusBadInput);
  __syncthreads();
  // every exit waits for the copies into this CTA's shared memory (the
  // drain after a wait that gave up takes the default limit)
  if (!mbar_wait(bar, 0, a.polls)) {
    if (threadIdx.x == 0) raise_status(a.status, kStatusTimeout);
    (void)mbar_wait(bar, 0);
    return;
  }
  if (!ok) return;                           // malformed sequence: write nothing
  const T *qs = reinterpret_cast<const T *>(rows_s);
  const T *ks = reinterpret_cast<const T *>(rows_s + qbytes);
  const T *vs = reinterpret_cast<const T *>(rows_s + qbytes + kvbytes);
  if (a.rotate_q) rotate_rows<T, 1>(qs, (T *)a.q_rot + (long)r * a.Hq * a.hd, a.Hq, a.hd, a.hd, cs);
  const long base = ((long)page * a.Hkv * kPage + slot % kPage) * a.hd;
  const long stride = (long)kPage * a.hd;    // next KV head, same slot
  rotate_rows<T, 1>(ks, (T *)a.k_cache + base, a.Hkv, a.hd, stride, cs);
  copy_rows<T, 1>(vs, (T *)a.v_cache + base, a.Hkv, a.hd, stride);
}

struct RopeAppendArgs {
  RopeTable tab;
  const void *k;
  const void *v;
  void *k_cache;
  void *v_cache;
  const int32_t *block_table;
  const int32_t *start;
  const int32_t *cu_n;
  int batch, Hkv, hd, max_pages, num_pages;
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
rope_append_kernel(const __grid_constant__ RopeAppendArgs a) {
  __shared__ float2 cs[64];
  const int r = blockIdx.x;
  const int b = find_seq(a.cu_n, a.batch, r);
  const int pos = __ldg(a.start + b) + (r - __ldg(a.cu_n + b));
  if (pos < 0 || pos >= a.max_pages * kPage) return;   // outside the table row
  const int page = __ldg(a.block_table + (long)b * a.max_pages + pos / kPage);
  if (page < 0 || page >= a.num_pages) return;
  angles(a.tab, a.hd, pos, cs);
  __syncthreads();
  const long base = ((long)page * a.Hkv * kPage + pos % kPage) * a.hd;
  const long stride = (long)kPage * a.hd;
  rotate_rows<T, 4>((const T *)a.k + (long)r * a.Hkv * a.hd, (T *)a.k_cache + base,
                    a.Hkv, a.hd, stride, cs);
  copy_rows<T, 4>((const T *)a.v + (long)r * a.Hkv * a.hd, (T *)a.v_cache + base,
                  a.Hkv, a.hd, stride);
}

}  // namespace

cudaError_t launch_rope_verify(const simsd_verify_desc *d, const VerifyPlan &p,
                               void *q_rot, int4 *tok_info, uint32_t *status,
                               cudaStream_t stream) {
  RopeVerifyArgs a;
  make_rope_table(d->rope_base, d->head_dim, &a.tab);
  a.q = d->q;
  a.k_new = d->k_new;
  a.v_new = d->v_new;
  a.q_rot = q_rot;
  a.k_cache = d->k_cache;
  a.v_cache = d->v_cache;
  a.block_table = d->block_table;
  a.lens = d->lens;
  a.cu_B = d->cu_B;
  a.tok_info = tok_info;
  a.row_tiles = p.row_tiles;
  a.status = status;
  a.num_pages = d->num_pages;
  a.batch = d->batch;
  a.Hq = d->num_q_heads;
  a.Hkv = d->num_kv_heads;
  a.hd = d->head_dim;
  a.max_pages = d->max_pages_per_seq;
  a.total_B = d->total_B;
  a.B_max = d->B_max;
  a.polls = wait_polls_of(d->wait_polls);
  a.node_size = d->node_size;
  a.rotate_q = d->dtype == SIMSD_F32;
  const size_t smem = (size_t)((a.rotate_q ? a.Hq : 0) + 2 * a.Hkv) * a.hd * p.esize;   // <= kMaxRowBytes
  const void *kern = d->dtype == SIMSD_BF16 ? (const void *)rope_verify_kernel<__nv_bfloat16>
                                            : (const void *)rope_verify_kernel<float>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  {
    // the SMs running this kernel keep the largest shared-memory split, so
    // the attention kernel's CTAs (programmatic dependent launch) can start
    // beside it instead of waiting for the SM to drain (set once per device
    // and dtype)
    static std::atomic<uint64_t> carved[2];
    const int dev = current_device();
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    std::atomic<uint64_t> &flag = carved[d->dtype == SIMSD_BF16 ? 1 : 0];
    if (!bit || !(flag.load() & bit)) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      flag.fetch_or(bit);
    }
  }
  if (d->dtype == SIMSD_BF16)
    rope_verify_kernel<__nv_bfloat16><<<p.T, kThreads, smem, stream>>>(a);
  else
    rope_verify_kernel<float><<<p.T, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_append(const simsd_append_desc *d, cudaStream_t stream) {
  RopeAppendArgs a;
  make_rope_table(d->rope_base, d->head_dim, &a.tab);
  a.k = d->k;
  a.v = d->v;
  a.k_cache = d->k_cache;
  a.v_cache = d->v_cache;
  a.block_table = d->block_table;
  a.start = d->start;
  a.cu_n = d->cu_n;
  a.batch = d->batch;
  a.Hkv = d->num_kv_heads;
  a.hd = d->head_dim;
  a.max_pages = d->max_pages_per_seq;
  a.num_pages = d->num_pages;
  if (d->dtype == SIMSD_BF16)
    rope_append_kernel<__nv_bfloat16><<<d->total_n, kThreads, 0, stream>>>(a);
  else
    rope_append_kernel<float><<<d->total_n, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace simsd
