// attn_f32.cu -- K2 (fp32 I/O) and K3: split-KV masked attention on CUDA
// cores for fp32 caches, and the merge of split partials for both dtypes.
//
// SimSD section 2 "Temporal Attention Mask": every new row sees the whole
// prompt; slot D~_i sees D_j with tau(j) < tau(i) and D~_j with
// tau(j) >= tau(i); data row D_i (convention) sees D_j with tau(j) <= tau(i).
//
// The fp32 path keeps full fp32 arithmetic (no tensor-core rounding of the
// operands), for small fp32 workloads that need 1e-4 agreement.  One CTA per
// (split, KV head, sequence); each warp takes one query row at a time, lanes
// stride over keys for the scores and over head dimensions for P.V.  The
// softmax runs online in the log2 domain, like the bf16 kernel, so both
// produce partials K3 can merge.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace simsd {
namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Visibility of key index `key` (0..P+2B-1) for a new row with token index
// `tok` (0..2B-1), tau of the new tokens in tau_s[0..2B); node_size > 0:
// the draft-graph layout (the row's own node).
__device__ __forceinline__ bool visible(int P, int B, const int *tau_s, int tok, int key,
                                        int node_size) {
  if (key < P) return true;
  const int j = key - P;
  if (node_size > 0) return j / node_size == tok / node_size;
  const int ti = tau_s[tok], tj = tau_s[j];
  const bool row_slot = tok >= B, key_slot = j >= B;
  if (row_slot) return key_slot ? tj >= ti : tj < ti;
  return !key_slot && tj <= ti;
}

template <int HD>
__global__ void __launch_bounds__(kWarps * 32)
attn_f32_kernel(const __grid_constant__ AttnParams a) {
  constexpr int PER = HD / 32;
  __shared__ int tau_s[2 * kMaxB];
  __shared__ float q_s[kWarps][HD];
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int P = __ldg(a.lens + b);
  const int Lk = P + 2 * B;
  const int M = 2 * B * a.G;
  const int k_begin = split * a.chunk;
  if (B < 1 || B > kMaxSection || B > a.B_max || c0 < 0 || c0 + B > a.total_B || P < 0 ||
      (long)Lk > (long)a.max_pages_per_seq * kPage ||
      (a.node_size > 0 && (2 * B) % a.node_size != 0)) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) raise_status(a.status, kStatusBadInput);
    return;
  }
  if (k_begin >= Lk) return;
  const int k_end = min(Lk, k_begin + a.chunk);
  const int n_splits_b = (Lk + a.chunk - 1) / a.chunk;
  if (a.node_size == 0)
    for (int j = threadIdx.x; j < 2 * B; j += blockDim.x)
      tau_s[j] = __ldg(a.tau + c0 + (j < B ? j : j - B));
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *qr = (const float *)a.q_rot;
  const float *kc = (const float *)a.k_cache;
  const float *vc = (const float *)a.v_cache;
  const int32_t *bt = a.block_table + (long)b * a.max_pages_per_seq;
  const float scale = a.sm_scale * kLog2e;
  for (int r = warp; r < M; r += kWarps) {
    const int tok = r / a.G;
    const int head = kvh * a.G + r % a.G;
    const long row = (2L * c0 + tok) * a.Hq + head;
    for (int d = lane; d < HD; d += 32) q_s[warp][d] = qr[row * HD + d];
    __syncwarp();
    float m = -INFINITY, l = 0.f, o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = 0.f;
    for (int base = k_begin; base < k_end; base += 32) {
      const int key = base + lane;
      float s = -INFINITY;
      const int kpage = key < k_end ? __ldg(bt + key / kPage) : -1;
      if (kpage >= 0 && kpage < a.num_pages && visible(P, B, tau_s, tok, key, a.node_size)) {
        const int page = kpage;
        const float *kr = kc + (((long)page * a.Hkv + kvh) * kPage + key % kPage) * HD;
        float acc = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) acc = fmaf(q_s[warp][d], kr[d], acc);
        s = acc * scale;
      }
      float cm = s;
#pragma unroll
      for (int w = 16; w > 0; w >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, w));
      const float m_new = fmaxf(m, cm);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m - m_use);
      const float p = exp2f(s - m_use);
      float ps = p;
#pragma unroll
      for (int w = 16; w > 0; w >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, w);
      l = l * alpha + ps;
#pragma unroll
      for (int i = 0; i < PER; ++i) o[i] *= alpha;
      for (int j = 0; j < 32; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
        if (pj == 0.f) continue;            // masked or past the end
        const int kj = base + j;
        const int page = __ldg(bt + kj / kPage);
        const float *vr = vc + (((long)page * a.Hkv + kvh) * kPage + kj % kPage) * HD;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = fmaf(pj, vr[lane + 32 * i], o[i]);
      }
      m = m_new;
    }
    if (n_splits_b == 1) {
      float *out = (float *)a.out + row * HD;
#pragma unroll
      for (int i = 0; i < PER; ++i) out[lane + 32 * i] = o[i] / l;
    } else {
      const long prow = (long)split * a.T * a.Hq + row;
#pragma unroll
      for (int i = 0; i < PER; ++i) a.o_part[prow * HD + lane + 32 * i] = o[i];
      if (lane == 0) a.ml_part[prow] = make_float2(m, l);
    }
    __syncwarp();
  }
}

// K3: O = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*) l_s, one warp per
// (token, query head) row, each lane a contiguous hd/32 columns (8- or
// 16-byte loads); rows of units that ran whole were finished by the
// attention kernel.  The partials of the first kMergeBatch splits are
// requested before the row's split count is known (the buffer holds every
// split of every row, so the reads stay in it; the extra ones are
// dropped), so a merge of up to kMergeBatch splits costs one round trip.
// Whether a row's unit was split comes from the append kernel's per-token
// record.
constexpr int kMergeBatch = 8;
constexpr int kMergeThreads = 256;
constexpr int kMergeRowsPerCta = kMergeThreads / 32;

// four CTAs (32 rows) per SM without spills: lane s keeps split s's
// (max, sum) and its weight is broadcast when the partials are summed
template <typename T, int HD>
__global__ void __launch_bounds__(kMergeThreads, 4)
combine_kernel(const __grid_constant__ AttnParams a, const int4 *tok_info, long row0, int max_splits) {
  constexpr int PER = HD / 32;               // 4 or 2 columns per lane
  using V = typename std::conditional<PER == 4, float4, float2>::type;
  grid_dep_wait();                           // partials come from the attention kernel
  const long row = row0 + (long)blockIdx.x * kMergeRowsPerCta + threadIdx.x / 32;
  const int lane = threadIdx.x % 32, col = lane * PER;
  if (row >= (long)a.T * a.Hq) return;
  const long stride = (long)a.T * a.Hq;
  auto load_batch = [&](int s0, int n, V *v, float2 &ml) {
#pragma unroll
    for (int s = 0; s < kMergeBatch; ++s)
      if (s < n) v[s] = __ldcg(reinterpret_cast<const V *>(a.o_part + ((s0 + s) * stride + row) * HD + col));
    ml = lane < n ? __ldcg(a.ml_part + (s0 + lane) * stride + row) : make_float2(-INFINITY, 0.f);
  };
  // the first batch, requested with the row's record
  V v[kMergeBatch];
  float2 ml;
  load_batch(0, min(kMergeBatch, max_splits), v, ml);
  // the row's unit (sequence, KV head, row tile) and whether it was split
  const int4 ti = __ldg(tok_info + row / a.Hq);   // keys 0: a malformed sequence (skipped)
  const int hq = (int)(row % a.Hq);
  const int rtile = (ti.z * a.G + hq % a.G) / a.rows_per_tile;
  const int unit = ti.y + rtile * a.Hkv + hq / a.G;
  const int ns = unit >= a.tail_from ? (ti.x + a.chunk_tail - 1) / a.chunk_tail : 1;
  if (ns <= 1) return;
  float mstar = -INFINITY, den = 0.f, o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kMergeBatch) {
    const int n = min(kMergeBatch, ns - s0);
    if (s0 > 0) load_batch(s0, n, v, ml);
    if (lane >= n) ml = make_float2(-INFINITY, 0.f);   // splits past the row's own
    float mb = ml.x;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, m));
    mb = fmaxf(mb, mstar);
    if (mb > mstar && mstar != -INFINITY) {  // a later batch raised the reference
      const float r = exp2f(mstar - mb);
      den *= r;
#pragma unroll
      for (int i = 0; i < PER; ++i) o[i] *= r;
    }
    mstar = mb;
    const float mu = mstar == -INFINITY ? 0.f : mstar;
    const float wl = lane < n ? exp2f(ml.x - mu) : 0.f;   // lane s: split s's weight
    float dl = wl * ml.y;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, m);
    den += dl;
#pragma unroll
    for (int s = 0; s < kMergeBatch; ++s) {
      const float w = __shfl_sync(0xffffffffu, wl, s);
      if (s < n) {
        const float *vf = reinterpret_cast<const float *>(&v[s]);
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = fmaf(w, vf[i], o[i]);
      }
    }
  }
  const float inv = 1.f / den;
  T *out = (T *)a.out + row * HD + col;
#pragma unroll
  for (int i = 0; i < PER; ++i) Elem<T>::store(out + i, o[i] * inv);
}

}  // namespace

cudaError_t launch_attn_f32(const simsd_verify_desc *d, const VerifyPlan &p,
                            const AttnParams &a, cudaStream_t stream) {
  dim3 grid(p.n_splits, d->num_kv_heads, d->batch);
  if (d->head_dim == 128)
    attn_f32_kernel<128><<<grid, kWarps * 32, 0, stream>>>(a);
  else
    attn_f32_kernel<64><<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const simsd_verify_desc *d, const VerifyPlan &p,
                           const AttnParams &a, const int4 *tok_info,
                           cudaStream_t stream) {
  const long rows = (long)p.merge_rows;
  const long row0 = (long)p.T * d->num_q_heads - rows;
  const unsigned blocks = (unsigned)((rows + kMergeRowsPerCta - 1) / kMergeRowsPerCta);
  const int4 *ts = tok_info;
  if (d->dtype == SIMSD_BF16)
    return d->head_dim == 128
               ? launch_pdl(combine_kernel<__nv_bfloat16, 128>, dim3(blocks), dim3(kMergeThreads), 0, stream, a, ts, row0, p.n_splits)
               : launch_pdl(combine_kernel<__nv_bfloat16, 64>, dim3(blocks), dim3(kMergeThreads), 0, stream, a, ts, row0, p.n_splits);
  return d->head_dim == 128
             ? launch_pdl(combine_kernel<float, 128>, dim3(blocks), dim3(kMergeThreads), 0, stream, a, ts, row0, p.n_splits)
             : launch_pdl(combine_kernel<float, 64>, dim3(blocks), dim3(kMergeThreads), 0, stream, a, ts, row0, p.n_splits);
}

}  // namespace simsd
