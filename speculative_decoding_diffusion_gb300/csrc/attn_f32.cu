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
// attention kernel.  The grid is (token, group of kMergeRowsPerCta heads),
// so a row needs no division to find its token.  The partials of the first
// MB splits (MB = 2, 4 or 8: the plan's split count rounded up, at most 8)
// are requested before the row's split count is known (the buffer holds
// every split of every row, so the reads stay in it; the extra ones are
// dropped), so a merge of up to MB splits costs one round trip, and the
// max and sum reductions run over MB lanes only.  Whether a row's unit was
// split comes from the append kernel's per-token record.
constexpr int kMergeThreads = 256;
constexpr int kMergeRowsPerCta = kMergeThreads / 32;

template <typename T, int PER> struct MergeOut;
template <> struct MergeOut<float, 4> {
  static __device__ __forceinline__ void store(float *p, const float *o) {
    *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct MergeOut<float, 2> {
  static __device__ __forceinline__ void store(float *p, const float *o) {
    *reinterpret_cast<float2 *>(p) = make_float2(o[0], o[1]);
  }
};
template <> struct MergeOut<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *o) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
  }
};
template <> struct MergeOut<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *o) {
    *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(o[0], o[1]);
  }
};

// four CTAs (32 rows) per SM without spills, eight (64 rows: 9728 rows in
// one wave) for batches of two splits: lane s keeps split s's (max, sum)
// and its weight is broadcast when the partials are summed
template <typename T, int HD, int MB>
__global__ void __launch_bounds__(kMergeThreads, MB <= 2 ? 8 : 4)
combine_kernel(const __grid_constant__ AttnParams a, const int4 *tok_info, int tok0, int max_splits) {
  constexpr int PER = HD / 32;               // 4 or 2 columns per lane
  using V = typename std::conditional<PER == 4, float4, float2>::type;
  grid_dep_wait();                           // partials come from the attention kernel
  const int hq = blockIdx.y * kMergeRowsPerCta + threadIdx.x / 32;
  if (hq >= a.Hq) return;
  const int tok = tok0 + (int)blockIdx.x, lane = threadIdx.x % 32;
  const size_t stride = (size_t)a.T * a.Hq;  // rows per split
  const size_t row = (size_t)tok * a.Hq + hq;
  const V *src = reinterpret_cast<const V *>(a.o_part + row * HD) + lane;
  const float2 *ml_src = a.ml_part + row;
  const size_t vstep = stride * (HD / PER);  // one split, in V units
  auto load_batch = [&](int s0, int n, V *v, float2 &ml) {
#pragma unroll
    for (int s = 0; s < MB; ++s)
      if (s < n) v[s] = __ldcg(src + (size_t)(s0 + s) * vstep);
    ml = lane < n ? __ldcg(ml_src + (size_t)(s0 + lane) * stride) : make_float2(-INFINITY, 0.f);
  };
  // the first batch, requested with the row's record
  V v[MB];
  float2 ml;
  load_batch(0, min(MB, max_splits), v, ml);
  // the row's unit (sequence, KV head, row tile) and whether it was split
  const int4 ti = __ldg(tok_info + tok);     // keys 0: a malformed sequence (skipped)
  const int g = hq / a.G;
  const int rtile = (ti.z * a.G + (hq - g * a.G)) / a.rows_per_tile;
  const int unit = ti.y + rtile * a.Hkv + g;
  const int ns = unit >= a.tail_from ? (ti.x + a.chunk_tail - 1) / a.chunk_tail : 1;
  if (ns <= 1) return;
  float mstar = -INFINITY, den = 0.f, o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += MB) {
    const int n = min(MB, ns - s0);
    if (s0 > 0) load_batch(s0, n, v, ml);
    if (lane >= n) ml = make_float2(-INFINITY, 0.f);   // splits past the row's own
    // lanes [0, MB) hold the batch: reduce within groups of MB lanes and
    // take lane 0's
    float mb = ml.x;
#pragma unroll
    for (int m = MB / 2; m > 0; m >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, m));
    mb = fmaxf(__shfl_sync(0xffffffffu, mb, 0), mstar);
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
    for (int m = MB / 2; m > 0; m >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, m);
    den += __shfl_sync(0xffffffffu, dl, 0);
#pragma unroll
    for (int s = 0; s < MB; ++s) {
      const float w = __shfl_sync(0xffffffffu, wl, s);
      if (s < n) {
        const float *vf = reinterpret_cast<const float *>(&v[s]);
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = fmaf(w, vf[i], o[i]);
      }
    }
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] *= inv;
  MergeOut<T, PER>::store((T *)a.out + row * HD + lane * PER, o);
}

template <typename T, int HD>
cudaError_t launch_combine_t(dim3 grid, cudaStream_t stream, const AttnParams &a,
                             const int4 *ts, int tok0, int n_splits) {
  if (n_splits <= 2)
    return launch_pdl(combine_kernel<T, HD, 2>, grid, dim3(kMergeThreads), 0, stream, a, ts, tok0, n_splits);
  if (n_splits <= 4)
    return launch_pdl(combine_kernel<T, HD, 4>, grid, dim3(kMergeThreads), 0, stream, a, ts, tok0, n_splits);
  return launch_pdl(combine_kernel<T, HD, 8>, grid, dim3(kMergeThreads), 0, stream, a, ts, tok0, n_splits);
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
  // merge_rows is a whole number of tokens (the last ones)
  const int tokens = (int)(p.merge_rows / d->num_q_heads);
  const int tok0 = p.T - tokens;
  const dim3 grid((unsigned)tokens, (unsigned)((d->num_q_heads + kMergeRowsPerCta - 1) / kMergeRowsPerCta));
  if (tokens == 0) return cudaSuccess;
  if (d->dtype == SIMSD_BF16)
    return d->head_dim == 128
               ? launch_combine_t<__nv_bfloat16, 128>(grid, stream, a, tok_info, tok0, p.n_splits)
               : launch_combine_t<__nv_bfloat16, 64>(grid, stream, a, tok_info, tok0, p.n_splits);
  return d->head_dim == 128
             ? launch_combine_t<float, 128>(grid, stream, a, tok_info, tok0, p.n_splits)
             : launch_combine_t<float, 64>(grid, stream, a, tok_info, tok0, p.n_splits);
}

}  // namespace simsd
