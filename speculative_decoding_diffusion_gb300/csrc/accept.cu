// accept.cu -- K4: rejection-sampling acceptance along the temporal order.
//
// SimSD section 4 "Speculative Decoding Pipeline", acceptance: standard
// rejection sampling along the draft-induced temporal order; the longest
// accepted prefix is committed.  For sequence b, step t = 1..B tests the
// slot k = tau^-1(t) with draft token x: p = softmax(target row k),
// q = softmax(draft row k); accept iff u[t-1] * q(x) < p(x) (fp32).  At the
// first rejection a token is drawn from max(0, p - q) normalised (p itself
// when that is empty) by inverse CDF with u[B].
//
// Numerics: every exponential is taken relative to a row maximum M in logit
// units, 2^((x - M) log2 e): x - M is exact for bf16 logits, so only the
// product and exp2f round (~2e-7 relative on the entries that carry mass).
// Cross-thread sums, the normaliser and every running CDF are fp64 (a few
// hundred additions per CTA); per-thread partial sums of <= 16 entries stay
// fp32.  The residual CDF is then within ~1e-6 (absolute, probability mass)
// of the exact one.
//
// Four launches, all sized to the data rather than to the batch:
//   K4a  grid (vocab chunk, slot): max and sum of exponentials of the target
//        and draft rows of every slot (the dominant HBM stream);
//   K4b  one CTA per sequence: merge chunk partials, p(x), q(x), the walk;
//   K4c  grid (residual chunk, sequence): per-chunk sums of max(0, p - q)
//        (and of p) of the rejected slot only;
//   K4d  one CTA per sequence with a rejection: prefix over chunk sums,
//        inverse CDF inside the selected chunk.  Within a chunk the running
//        sum never decreases (thread totals prefixed sequentially), so the
//        chosen token always has positive mass.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace simsd {
namespace {

constexpr int kThreads = 256;
constexpr int kLseChunk = 4096;   // K4a vocabulary chunk
constexpr int kResPer = 8;        // residual entries per thread
constexpr int kResChunk = kThreads * kResPer;
constexpr float kLog2e = 1.4426950408889634f;

// Per sequence, after the walk: rejected slot (-1: none) and the row maxima
// and normalisers of that slot.
struct WalkState {
  int rej;
  float Mt, Md;
  double St, Sd;
};

struct AcceptWs {
  size_t off_status, off_lse, off_state, off_res, total;
  int lse_chunks, res_chunks;
};

AcceptWs accept_ws(const simsd_accept_desc *d) {
  AcceptWs w;
  w.lse_chunks = (d->vocab + kLseChunk - 1) / kLseChunk;
  w.res_chunks = (d->vocab + kResChunk - 1) / kResChunk;
  size_t off = 0;
  w.off_status = off; off = align_up(off + sizeof(uint32_t), kAlign);
  w.off_lse = off;    off = align_up(off + (size_t)d->total_B * w.lse_chunks * sizeof(float4), kAlign);
  w.off_state = off;  off = align_up(off + (size_t)d->batch * sizeof(WalkState), kAlign);
  w.off_res = off;    off = align_up(off + (size_t)d->batch * w.res_chunks * sizeof(double2), kAlign);
  w.total = off;
  return w;
}

struct AcceptArgs {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  float4 *lse_part;     // [total_B][lse_chunks]: (M_t, s_t, M_d, s_d)
  WalkState *state;     // [batch]
  double2 *res_part;    // [batch][res_chunks]: (sum r, sum p)
  uint32_t *status;
  int batch, vocab, B_max, lse_chunks, res_chunks, vec_ok;
};

// (M, s) with s = sum 2^((x - M) log2 e): merge two partial states.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) { m = mm; s = 0.f; return; }
  s = s * exp2f((m - mm) * kLog2e) + s2 * exp2f((m2 - mm) * kLog2e);
  m = mm;
}

__device__ __forceinline__ void accum(float &m, float &s, const float *x, int n) {
  float mx = -INFINITY;
  for (int i = 0; i < n; ++i) mx = fmaxf(mx, x[i]);
  if (mx > m) { s *= exp2f((m - mx) * kLog2e); m = mx; }
  if (m == -INFINITY) return;
  for (int i = 0; i < n; ++i) s += exp2f((x[i] - m) * kLog2e);
}

template <typename T> struct Ld;
template <> struct Ld<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void vec(const float *p, float *f) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  static __device__ __forceinline__ float one(const float *p) { return __ldg(p); }
};
template <> struct Ld<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void vec(const __nv_bfloat16 *p, float *f) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ float one(const __nv_bfloat16 *p) {
    return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
  }
};

// Block-wide (M, s) merge: warps in fp32, across warps in fp64 relative to
// the block maximum.  Result in thread 0.
__device__ __forceinline__ void block_lse(float &m, float &s, float2 *scratch) {
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, w);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, w);
    lse_merge(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = make_float2(m, s);
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int i = 0; i < kThreads / 32; ++i) M = fmaxf(M, scratch[i].x);
    double S = 0.0;
    if (M != -INFINITY)
      for (int i = 0; i < kThreads / 32; ++i)
        S += (double)scratch[i].y * (double)exp2f((scratch[i].x - M) * kLog2e);
    m = M;
    s = (float)S;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- K4a
template <typename T>
__global__ void __launch_bounds__(kThreads)
lse_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ float2 scratch[2][kThreads / 32];
  const int chunk = blockIdx.x, slot = blockIdx.y;
  const long row = (long)slot * a.vocab;
  const int v0 = chunk * kLseChunk;
  const int v1 = min(a.vocab, v0 + kLseChunk);
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
  constexpr int N = Ld<T>::N;
  int tail0 = v0;
  if (a.vec_ok) {
    for (int v = v0 + threadIdx.x * N; v + N <= v1; v += kThreads * N) {
      float xt[N], xd[N];
      Ld<T>::vec(tr + v, xt);
      Ld<T>::vec(dr + v, xd);
      accum(mt, st, xt, N);
      accum(md, sd, xd, N);
    }
    tail0 = v0 + ((v1 - v0) / N) * N;   // ragged end (last chunk only)
  }
  for (int v = tail0 + threadIdx.x; v < v1; v += kThreads) {
    float xt = Ld<T>::one(tr + v), xd = Ld<T>::one(dr + v);
    accum(mt, st, &xt, 1);
    accum(md, sd, &xd, 1);
  }
  block_lse(mt, st, scratch[0]);
  block_lse(md, sd, scratch[1]);
  if (threadIdx.x == 0) a.lse_part[(long)slot * a.lse_chunks + chunk] = make_float4(mt, st, md, sd);
}

// Row maximum and normaliser of one slot from its chunk partials (one warp).
__device__ __forceinline__ void row_norm(const float4 *pp, int chunks, int lane,
                                         float &Mt, double &St, float &Md, double &Sd) {
  float mt = -INFINITY, md = -INFINITY;
  for (int c = lane; c < chunks; c += 32) { mt = fmaxf(mt, pp[c].x); md = fmaxf(md, pp[c].z); }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, w));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, w));
  }
  double st = 0.0, sd = 0.0;
  for (int c = lane; c < chunks; c += 32) {
    const float4 v = pp[c];
    if (v.y > 0.f) st += (double)v.y * (double)exp2f((v.x - mt) * kLog2e);
    if (v.w > 0.f) sd += (double)v.w * (double)exp2f((v.z - md) * kLog2e);
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    st += __shfl_xor_sync(0xffffffffu, st, w);
    sd += __shfl_xor_sync(0xffffffffu, sd, w);
  }
  Mt = mt; St = st; Md = md; Sd = sd;
}

// ---------------------------------------------------------------- K4b
template <typename T>
__global__ void __launch_bounds__(kThreads)
walk_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ float px_s[kMaxB], qx_s[kMaxB], mt_s[kMaxB], md_s[kMaxB];
  __shared__ double st_s[kMaxB], sd_s[kMaxB];
  const int b = blockIdx.x;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  if (B < 1 || B > kMaxB) {                  // malformed sequence: no walk
    if (threadIdx.x == 0) {
      a.n_accept[b] = 0; a.token[b] = -1; a.pos[b] = -1;
      a.state[b] = WalkState{-1, 0.f, 0.f, 0.0, 0.0};
      raise_status(a.status, kStatusBadInput);
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = warp; k < B; k += kThreads / 32) {
    float Mt, Md;
    double St, Sd;
    row_norm(a.lse_part + (long)(c0 + k) * a.lse_chunks, a.lse_chunks, lane, Mt, St, Md, Sd);
    if (lane == 0) {
      const long row = (long)(c0 + k) * a.vocab;
      int x = __ldg(a.draft_tokens + c0 + k);
      if (x < 0 || x >= a.vocab) { raise_status(a.status, kStatusBadInput); x = 0; }
      const float tx = Ld<T>::one((const T *)a.target + row + x);
      const float dx = Ld<T>::one((const T *)a.draft + row + x);
      px_s[k] = (float)((double)exp2f((tx - Mt) * kLog2e) / St);
      qx_s[k] = (float)((double)exp2f((dx - Md) * kLog2e) / Sd);
      mt_s[k] = Mt; md_s[k] = Md; st_s[k] = St; sd_s[k] = Sd;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int slot_of_step[kMaxB];
    for (int k = 0; k < kMaxB; ++k) slot_of_step[k] = 0;
    for (int k = 0; k < B; ++k) {
      const int t = __ldg(a.tau + c0 + k);   // a label outside 1..B is ignored
      if (t >= 1 && t <= B) slot_of_step[t - 1] = k;
    }
    const float *u = a.uniforms + (long)b * (a.B_max + 1);
    int n = B, rej = -1;
    for (int t = 1; t <= B; ++t) {
      const int k = slot_of_step[t - 1];
      if (!(__ldg(u + t - 1) * qx_s[k] < px_s[k])) { n = t - 1; rej = k; break; }
    }
    a.n_accept[b] = n;
    a.pos[b] = rej;
    if (rej < 0) {
      a.token[b] = -1;
      a.state[b] = WalkState{-1, 0.f, 0.f, 0.0, 0.0};
    } else {
      a.state[b] = WalkState{rej, mt_s[rej], md_s[rej], st_s[rej], sd_s[rej]};
    }
  }
}

// Residual mass r = max(0, p - q) and target mass p of one entry.
__device__ __forceinline__ void res_pair(float t, float d, const WalkState &st,
                                         float inv_st, float inv_sd, float &r, float &p) {
  p = exp2f((t - st.Mt) * kLog2e) * inv_st;
  const float q = exp2f((d - st.Md) * kLog2e) * inv_sd;
  r = fmaxf(p - q, 0.f);
}

// ---------------------------------------------------------------- K4c
template <typename T>
__global__ void __launch_bounds__(kThreads)
residual_sum_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ double2 scratch[kThreads / 32];
  const int chunk = blockIdx.x, b = blockIdx.y;
  const WalkState st = a.state[b];
  if (st.rej < 0) return;
  const float inv_st = (float)(1.0 / st.St), inv_sd = (float)(1.0 / st.Sd);
  const long row = (long)(__ldg(a.cu_B + b) + st.rej) * a.vocab;
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  const int v0 = chunk * kResChunk + threadIdx.x * kResPer;
  float sr = 0.f, sp = 0.f;
  for (int i = 0; i < kResPer; ++i) {
    const int v = v0 + i;
    if (v >= a.vocab) break;
    float r, p;
    res_pair(Ld<T>::one(tr + v), Ld<T>::one(dr + v), st, inv_st, inv_sd, r, p);
    sr += r;
    sp += p;
  }
  double dr_ = sr, dp = sp;
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    dr_ += __shfl_xor_sync(0xffffffffu, dr_, w);
    dp += __shfl_xor_sync(0xffffffffu, dp, w);
  }
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = make_double2(dr_, dp);
  __syncthreads();
  if (threadIdx.x == 0) {
    double2 tot = scratch[0];
    for (int i = 1; i < kThreads / 32; ++i) { tot.x += scratch[i].x; tot.y += scratch[i].y; }
    a.res_part[(long)b * a.res_chunks + chunk] = tot;
  }
}

// ---------------------------------------------------------------- K4d
template <typename T>
__global__ void __launch_bounds__(kThreads)
residual_draw_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ double wsum[kThreads];
  __shared__ int sel_chunk, use_p_s, best_s, last_pos_s;
  __shared__ double base_s, U_s;
  const int b = blockIdx.x;
  const WalkState st = a.state[b];
  if (st.rej < 0) return;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const double2 *rp = a.res_part + (long)b * a.res_chunks;
  if (threadIdx.x == 0) {
    double S = 0.0;
    for (int c = 0; c < a.res_chunks; ++c) S += rp[c].x;
    const int use_p = !(S > 0.0);            // empty residual: draw from p
    double tot = 0.0;
    if (use_p) for (int c = 0; c < a.res_chunks; ++c) tot += rp[c].y;
    else tot = S;
    const double U = (double)__ldg(a.uniforms + (long)b * (a.B_max + 1) + B) * tot;
    // chunk c with T[c] <= U < T[c+1] (T: running sum of chunk masses); if
    // rounding leaves U at or past the total, the last non-empty chunk
    double T0 = 0.0, sel_base = 0.0, last_base = 0.0;
    int sel = -1, last_nz = 0;
    for (int c = 0; c < a.res_chunks; ++c) {
      const double m = use_p ? rp[c].y : rp[c].x;
      const double T1 = T0 + m;
      if (m > 0.0) { last_nz = c; last_base = T0; }
      if (sel < 0 && U < T1 && m > 0.0) { sel = c; sel_base = T0; }
      T0 = T1;
    }
    if (sel < 0) { sel = last_nz; sel_base = last_base; }
    sel_chunk = sel;
    base_s = sel_base;
    U_s = U;
    use_p_s = use_p;
    best_s = 0x7fffffff;
    last_pos_s = -1;
  }
  __syncthreads();
  const int use_p = use_p_s;
  const float inv_st = (float)(1.0 / st.St), inv_sd = (float)(1.0 / st.Sd);
  const long row = (long)(c0 + st.rej) * a.vocab;
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  const int v0 = sel_chunk * kResChunk + threadIdx.x * kResPer;
  float m[kResPer];
  float local = 0.f;
#pragma unroll
  for (int i = 0; i < kResPer; ++i) {
    const int v = v0 + i;
    float r = 0.f, p = 0.f;
    if (v < a.vocab) res_pair(Ld<T>::one(tr + v), Ld<T>::one(dr + v), st, inv_st, inv_sd, r, p);
    m[i] = use_p ? p : r;
    local += m[i];
  }
  wsum[threadIdx.x] = (double)local;
  __syncthreads();
  if (threadIdx.x == 0) {   // exclusive prefix of thread totals, in order
    double run = 0.0;
    for (int i = 0; i < kThreads; ++i) { const double x = wsum[i]; wsum[i] = run; run += x; }
  }
  __syncthreads();
  const double U = U_s, base = base_s + wsum[threadIdx.x];
  float lp = 0.f;
  int first = 0x7fffffff, last_pos = -1;
#pragma unroll
  for (int i = 0; i < kResPer; ++i) {
    lp += m[i];
    if (m[i] > 0.f) {
      last_pos = v0 + i;
      if (first == 0x7fffffff && base + (double)lp > U) first = v0 + i;
    }
  }
  if (first != 0x7fffffff) atomicMin(&best_s, first);
  if (last_pos >= 0) atomicMax(&last_pos_s, last_pos);
  __syncthreads();
  if (threadIdx.x == 0) a.token[b] = best_s != 0x7fffffff ? best_s : last_pos_s;
}

void mark(void *const *events, int i, cudaStream_t stream) {
  if (events != nullptr && events[i] != nullptr) cudaEventRecord((cudaEvent_t)events[i], stream);
}

template <typename T>
cudaError_t launch_all(const AcceptArgs &a, int total_B, cudaStream_t stream,
                       void *const *events) {
  mark(events, 0, stream);
  lse_kernel<T><<<dim3(a.lse_chunks, total_B), kThreads, 0, stream>>>(a);
  mark(events, 1, stream);
  walk_kernel<T><<<a.batch, kThreads, 0, stream>>>(a);
  mark(events, 2, stream);
  residual_sum_kernel<T><<<dim3(a.res_chunks, a.batch), kThreads, 0, stream>>>(a);
  mark(events, 3, stream);
  residual_draw_kernel<T><<<a.batch, kThreads, 0, stream>>>(a);
  mark(events, 4, stream);
  return cudaGetLastError();
}

simsd_status accept_check(const simsd_accept_desc *d) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (d->dtype != SIMSD_F32 && d->dtype != SIMSD_BF16) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->batch > 65535 || d->vocab < 1 || d->B_max < 1 ||
      d->B_max > kMaxB || d->total_B < d->batch ||
      (int64_t)d->total_B > (int64_t)d->batch * d->B_max || d->total_B > 65535 ||
      (int64_t)d->vocab > (int64_t)kLseChunk * 65535)
    return SIMSD_ERR_SHAPE;
  return SIMSD_OK;
}

// Scratch of simsd_accept_noalloc: one static array per device, alive until
// the process exits.  Host code may not take its address directly (the
// name is a host-side stand-in there); static_scratch() looks the device
// address up once per device.
constexpr int kMaxDevices = 64;
static_assert(SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES % kAlign == 0, "scratch size");
static __device__ __align__(256) unsigned char g_accept_scratch[SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES];

cudaError_t static_scratch(char **out) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = (char *)addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace simsd

using namespace simsd;

extern "C" {

size_t simsd_accept_workspace_size(const simsd_accept_desc *d) {
  if (accept_check(d) != SIMSD_OK) return 0;
  return accept_ws(d).total;
}

simsd_status simsd_accept(const simsd_accept_desc *d, void *stream_ptr) {
  return simsd_accept_timed(d, stream_ptr, nullptr);
}

simsd_status simsd_accept_timed(const simsd_accept_desc *d, void *stream_ptr,
                                void *const events[5]) {
  simsd_status st = accept_check(d);
  if (st != SIMSD_OK) return st;
  if (!d->target_logits || !d->draft_logits || !d->draft_tokens || !d->tau ||
      !d->cu_B || !d->uniforms || !d->n_accept || !d->token || !d->pos)
    return SIMSD_ERR_NULL;
  const AcceptWs w = accept_ws(d);
  if (d->workspace == nullptr || ((uintptr_t)d->workspace % kAlign) != 0 ||
      d->workspace_bytes < w.total)
    return SIMSD_ERR_WORKSPACE;
  cudaStream_t stream = (cudaStream_t)stream_ptr;
  char *ws = (char *)d->workspace;
  if (cudaMemsetAsync(ws + w.off_status, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return SIMSD_ERR_CUDA;
  AcceptArgs a;
  a.target = d->target_logits;
  a.draft = d->draft_logits;
  a.draft_tokens = d->draft_tokens;
  a.tau = d->tau;
  a.cu_B = d->cu_B;
  a.uniforms = d->uniforms;
  a.n_accept = d->n_accept;
  a.token = d->token;
  a.pos = d->pos;
  a.lse_part = (float4 *)(ws + w.off_lse);
  a.state = (WalkState *)(ws + w.off_state);
  a.res_part = (double2 *)(ws + w.off_res);
  a.status = (uint32_t *)(ws + w.off_status);
  a.batch = d->batch;
  a.vocab = d->vocab;
  a.B_max = d->B_max;
  a.lse_chunks = w.lse_chunks;
  a.res_chunks = w.res_chunks;
  const size_t es = d->dtype == SIMSD_BF16 ? 2 : 4;
  a.vec_ok = ((size_t)d->vocab * es) % 16 == 0 &&
             ((uintptr_t)d->target_logits % 16) == 0 &&
             ((uintptr_t)d->draft_logits % 16) == 0;
  cudaError_t e = d->dtype == SIMSD_BF16
                      ? launch_all<__nv_bfloat16>(a, d->total_B, stream, events)
                      : launch_all<float>(a, d->total_B, stream, events);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

// Same kernels and arguments as simsd_accept; scratch from the static
// array instead of a caller workspace (see simsd.h for who needs this).
simsd_status simsd_accept_noalloc(const simsd_accept_desc *d, void *stream_ptr) {
  simsd_status st = accept_check(d);
  if (st != SIMSD_OK) return st;
  if (!d->target_logits || !d->draft_logits || !d->draft_tokens || !d->tau ||
      !d->cu_B || !d->uniforms || !d->n_accept || !d->token || !d->pos)
    return SIMSD_ERR_NULL;
  const AcceptWs w = accept_ws(d);
  if (w.total > SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES) return SIMSD_ERR_WORKSPACE;
  char *ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return SIMSD_ERR_CUDA;
  cudaStream_t stream = (cudaStream_t)stream_ptr;
  if (cudaMemsetAsync(ws + w.off_status, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return SIMSD_ERR_CUDA;
  AcceptArgs a;
  a.target = d->target_logits;
  a.draft = d->draft_logits;
  a.draft_tokens = d->draft_tokens;
  a.tau = d->tau;
  a.cu_B = d->cu_B;
  a.uniforms = d->uniforms;
  a.n_accept = d->n_accept;
  a.token = d->token;
  a.pos = d->pos;
  a.lse_part = (float4 *)(ws + w.off_lse);
  a.state = (WalkState *)(ws + w.off_state);
  a.res_part = (double2 *)(ws + w.off_res);
  a.status = (uint32_t *)(ws + w.off_status);
  a.batch = d->batch;
  a.vocab = d->vocab;
  a.B_max = d->B_max;
  a.lse_chunks = w.lse_chunks;
  a.res_chunks = w.res_chunks;
  const size_t es = d->dtype == SIMSD_BF16 ? 2 : 4;
  a.vec_ok = ((size_t)d->vocab * es) % 16 == 0 &&
             ((uintptr_t)d->target_logits % 16) == 0 &&
             ((uintptr_t)d->draft_logits % 16) == 0;
  cudaError_t e = d->dtype == SIMSD_BF16
                      ? launch_all<__nv_bfloat16>(a, d->total_B, stream, nullptr)
                      : launch_all<float>(a, d->total_B, stream, nullptr);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

}  // extern "C"
