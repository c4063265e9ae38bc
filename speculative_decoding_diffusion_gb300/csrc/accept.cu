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
// Two launches:
//   K4a  grid (vocab chunk, slot): max and sum of exponentials of the target
//        and draft rows (the dominant HBM stream).  The last CTA to finish a
//        sequence (a wait-free counter, no spinning) merges that sequence's
//        partials and walks its steps in tau order.
//   K4b  grid (residual chunk, sequence): per-chunk residual mass of the
//        rejected slot only; the last CTA of a sequence takes the prefix over
//        chunks and draws the token inside the selected chunk.
// Numerics: a partial state is (R, s) with R a reference in log2 units (the
// maximum of x log2 e seen so far, rounded once) and s = sum 2^(x log2 e - R),
// each exponent argument formed by one fma (a single rounding, small for
// the entries near the maximum that carry the mass) and exponentiated by
// the MUFU ex2 instruction; references of different partials differ by
// exactly representable amounts.  Normalisers, chunk sums and running CDFs
// are compensated fp32 pairs (two-sum), never fp64 (GB300's fp64 rate is a
// small fraction of its fp32 rate).  The residual CDF is then within ~1e-6
// (absolute probability mass) of the exact one.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace simsd {
namespace {

constexpr int kThreads = 256;
constexpr int kVecs = 2;                          // 16-byte loads per row per thread
constexpr float kLog2e = 1.4426950408889634f;

// Vocabulary chunk of one CTA (both kernels): kThreads x kVecs 16-byte
// vectors per row -- 4096 bf16 or 2048 fp32 entries.
constexpr int chunk_entries(simsd_dtype t) { return kThreads * kVecs * (t == SIMSD_BF16 ? 8 : 4); }

// ------------------------------------------------------------ two-sum pairs
// value = hi + lo with |lo| <= ulp(hi)/2 (Knuth's two-sum; Dekker's
// fast-two-sum for the renormalisation).
struct Ff {
  float hi, lo;
};
__device__ __forceinline__ Ff ff_add(Ff a, Ff b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float err = (a.hi - (s - bb)) + (b.hi - bb);
  const float lo = err + a.lo + b.lo;
  const float hi = s + lo;
  return Ff{hi, lo - (hi - s)};
}
__device__ __forceinline__ Ff ff_of(float x) { return Ff{x, 0.f}; }
__device__ __forceinline__ Ff ff_shfl_xor(Ff a, int m) {
  return Ff{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}
__device__ __forceinline__ Ff ff_shfl_up(Ff a, int d) {
  return Ff{__shfl_up_sync(0xffffffffu, a.hi, d), __shfl_up_sync(0xffffffffu, a.lo, d)};
}
// a > u where u is a pair: compare the exact sums' signs
__device__ __forceinline__ bool ff_gt(Ff a, Ff u) {
  const Ff d = ff_add(a, Ff{-u.hi, -u.lo});
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

// Per sequence, after the walk: the rejected slot's logit row (-1: none),
// its references (log2 units), reciprocal normalisers and the residual
// draw's uniform.
struct __align__(16) WalkState {
  int row;
  float Mt, Md, inv_st, inv_sd, u;
  int pad0, pad1;
};

struct AcceptWs {
  size_t off_status, status_bytes, off_lse, off_x, off_state, off_res, total;
  int chunks;
};

// status word, then two per-sequence arrival counters; the whole head is
// cleared at the start of every call.
AcceptWs accept_ws(const simsd_accept_desc *d) {
  AcceptWs w;
  const int ce = chunk_entries(d->dtype);
  w.chunks = (d->vocab + ce - 1) / ce;
  size_t off = 0;
  w.off_status = off;
  w.status_bytes = sizeof(uint32_t) * (1 + 2 * (size_t)d->batch);
  off = align_up(off + w.status_bytes, kAlign);
  w.off_lse = off;    off = align_up(off + (size_t)d->total_B * w.chunks * sizeof(float4), kAlign);
  w.off_x = off;      off = align_up(off + (size_t)d->total_B * sizeof(float2), kAlign);
  w.off_state = off;  off = align_up(off + (size_t)d->batch * sizeof(WalkState), kAlign);
  w.off_res = off;    off = align_up(off + (size_t)d->batch * w.chunks * sizeof(float4), kAlign);
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
  float4 *lse_part;     // [total_B][chunks]: (R_t, s_t, R_d, s_d)
  float2 *xval;         // [total_B]: target and draft logit at the draft token
  WalkState *state;     // [batch]
  float4 *res_part;     // [batch][chunks]: residual pair, target-mass pair
  uint32_t *status;     // [0]: status word; [1..batch]: K4a counters; then K4b's
  int batch, vocab, B_max, chunks, vec_ok;
};

// 2^x on the MUFU (approximate, ~2 ulp; subnormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^(x log2 e - R): the argument rounded once.
__device__ __forceinline__ float rel_exp(float x, float R) { return ex2(fmaf(x, kLog2e, -R)); }

// (R, s) with s = sum 2^(x log2 e - R): merge two partial states.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) { m = mm; s = 0.f; return; }
  s = s * ex2(m - mm) + s2 * ex2(m2 - mm);
  m = mm;
}

// Raw 16-byte vectors of logits: loads, unpacking, lane-wise maximum.
template <typename T> struct Ld;
template <> struct Ld<float> {
  static constexpr int N = 4;
  static constexpr uint32_t kNegInf = 0xff800000u;
  static __device__ __forceinline__ uint4 raw(const float *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
  }
  static __device__ __forceinline__ uint32_t one_raw(const float *p) {
    return __float_as_uint(__ldg(p));
  }
  static __device__ __forceinline__ uint4 gather(const float *row, int v, int v1) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = v + e < v1 ? one_raw(row + v + e) : kNegInf;
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ float vmax(const uint4 *w, int n) {
    float m0 = -INFINITY, m1 = -INFINITY;
    for (int i = 0; i < n; ++i) {
      m0 = fmaxf(m0, fmaxf(__uint_as_float(w[i].x), __uint_as_float(w[i].y)));
      m1 = fmaxf(m1, fmaxf(__uint_as_float(w[i].z), __uint_as_float(w[i].w)));
    }
    return fmaxf(m0, m1);
  }
};
template <> struct Ld<__nv_bfloat16> {
  static constexpr int N = 8;
  static constexpr uint32_t kNegInf = 0xff80u;
  static __device__ __forceinline__ uint4 raw(const __nv_bfloat16 *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
  }
  static __device__ __forceinline__ uint32_t one_raw(const __nv_bfloat16 *p) {
    return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p));
  }
  static __device__ __forceinline__ uint4 gather(const __nv_bfloat16 *row, int v, int v1) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t lo = v + 2 * e < v1 ? one_raw(row + v + 2 * e) : kNegInf;
      const uint32_t hi = v + 2 * e + 1 < v1 ? one_raw(row + v + 2 * e + 1) : kNegInf;
      w[e] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  // packed maximum of the bf16 pairs (exact), then of the two halves
  static __device__ __forceinline__ float vmax(const uint4 *w, int n) {
    uint32_t m = 0xff80ff80u;
    for (int i = 0; i < n; ++i) m = max2(m, max2(max2(w[i].x, w[i].y), max2(w[i].z, w[i].w)));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
};

// Entries [v0, v1) of a row: thread t's vector i holds entries
// v0 + (i * kThreads + t) * N ... + N - 1 (coalesced; order within the
// chunk does not matter to the sums).  Entries past v1 read as -inf.
template <typename T>
__device__ __forceinline__ void load_strided(const T *row, int v0, int v1, bool vec, uint4 *w) {
  constexpr int N = Ld<T>::N;
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const int v = v0 + (i * kThreads + threadIdx.x) * N;
    w[i] = vec && v + N <= v1 ? Ld<T>::raw(row + v) : Ld<T>::gather(row, v, v1);
  }
}

// Entries [v0, v1) of a row, thread t holding the kVecs * N consecutive
// entries from v0 + t * kVecs * N (vocabulary order follows thread order).
template <typename T>
__device__ __forceinline__ void load_contig(const T *row, int v0, int v1, bool vec, uint4 *w) {
  constexpr int N = Ld<T>::N;
#pragma unroll
  for (int i = 0; i < kVecs; ++i) {
    const int v = v0 + (threadIdx.x * kVecs + i) * N;
    w[i] = vec && v + N <= v1 ? Ld<T>::raw(row + v) : Ld<T>::gather(row, v, v1);
  }
}

// (R, s) of the loaded entries: R = max * log2 e (rounded once), then
// s = sum 2^(x log2 e - R), one fma and the MUFU per entry.
template <typename T>
__device__ __forceinline__ void thread_lse(const uint4 *w, float &R, float &s) {
  constexpr int N = Ld<T>::N;
  const float mx = Ld<T>::vmax(w, kVecs);
  R = mx * kLog2e;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  if (mx != -INFINITY) {
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      float x[N];
      Ld<T>::unpack(w[i], x);
#pragma unroll
      for (int e = 0; e < N; ++e) a[e & 3] += rel_exp(x[e], R);
    }
  }
  s = (a[0] + a[1]) + (a[2] + a[3]);
}

// Block-wide merge of the (R, s) pairs of both rows; result in thread 0.
// Warps reduce by shuffles, then warp 0 merges the warps' partials (sums as
// two-sum pairs relative to the block reference): one barrier per CTA.
__device__ __forceinline__ void block_lse2(float &mt, float &st, float &md, float &sd,
                                           float4 *scratch) {
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    lse_merge(mt, st, __shfl_xor_sync(0xffffffffu, mt, w), __shfl_xor_sync(0xffffffffu, st, w));
    lse_merge(md, sd, __shfl_xor_sync(0xffffffffu, md, w), __shfl_xor_sync(0xffffffffu, sd, w));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = make_float4(mt, st, md, sd);
  __syncthreads();
  if (warp == 0) {
    constexpr int W = kThreads / 32;
    const float4 v = lane < W ? scratch[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    float Mt = v.x, Md = v.z;
#pragma unroll
    for (int w = W / 2; w > 0; w >>= 1) {
      Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, w));
      Md = fmaxf(Md, __shfl_xor_sync(0xffffffffu, Md, w));
    }
    Ff St = ff_of(v.y > 0.f ? v.y * ex2(v.x - Mt) : 0.f);
    Ff Sd = ff_of(v.w > 0.f ? v.w * ex2(v.z - Md) : 0.f);
#pragma unroll
    for (int w = W / 2; w > 0; w >>= 1) {
      St = ff_add(St, ff_shfl_xor(St, w));
      Sd = ff_add(Sd, ff_shfl_xor(Sd, w));
    }
    mt = Mt; st = St.hi + St.lo; md = Md; sd = Sd.hi + Sd.lo;
  }
}

// Row maximum and normaliser of one slot from its chunk partials (one warp;
// the first kNormRegs * 32 partials are read once and kept in registers).
constexpr int kNormRegs = 4;
__device__ __forceinline__ void row_norm(const float4 *pp, int chunks, int lane,
                                         float &Mt, float &St, float &Md, float &Sd) {
  float4 c4[kNormRegs];
#pragma unroll
  for (int j = 0; j < kNormRegs; ++j) {
    const int c = lane + 32 * j;
    c4[j] = c < chunks ? __ldcg(pp + c) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  }
  float mt = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int j = 0; j < kNormRegs; ++j) { mt = fmaxf(mt, c4[j].x); md = fmaxf(md, c4[j].z); }
  for (int c = lane + 32 * kNormRegs; c < chunks; c += 32) {
    const float4 v = __ldcg(pp + c);
    mt = fmaxf(mt, v.x);
    md = fmaxf(md, v.z);
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, w));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, w));
  }
  Ff st = ff_of(0.f), sd = ff_of(0.f);
#pragma unroll
  for (int j = 0; j < kNormRegs; ++j) {
    if (c4[j].y > 0.f) st = ff_add(st, ff_of(c4[j].y * ex2(c4[j].x - mt)));
    if (c4[j].w > 0.f) sd = ff_add(sd, ff_of(c4[j].w * ex2(c4[j].z - md)));
  }
  for (int c = lane + 32 * kNormRegs; c < chunks; c += 32) {
    const float4 v = __ldcg(pp + c);
    if (v.y > 0.f) st = ff_add(st, ff_of(v.y * ex2(v.x - mt)));
    if (v.w > 0.f) sd = ff_add(sd, ff_of(v.w * ex2(v.z - md)));
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    st = ff_add(st, ff_shfl_xor(st, w));
    sd = ff_add(sd, ff_shfl_xor(sd, w));
  }
  Mt = mt; St = st.hi + st.lo; Md = md; Sd = sd.hi + sd.lo;
}

// The walk of sequence b (whole CTA).  Every global read it needs -- labels,
// uniforms, draft tokens, logits at the draft tokens, chunk partials -- is
// issued before any result is used; then p(x), q(x) per slot; then thread 0
// takes the steps in tau order from shared memory and writes the outputs
// and the walk state.
__device__ void walk(const AcceptArgs &a, int b, int c0, int B) {
  __shared__ float px_s[kMaxB], qx_s[kMaxB], u_s[kMaxB + 1];
  __shared__ int tau_s[kMaxB], slot_of_step[kMaxB];
  __shared__ WalkState ws_s[kMaxB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = threadIdx.x;
  if (t < B) tau_s[t] = __ldg(a.tau + c0 + t);
  if (t <= B) u_s[t] = __ldg(a.uniforms + (long)b * (a.B_max + 1) + t);
  for (int k = warp; k < B; k += kThreads / 32) {
    int x = 0;
    float2 xv = make_float2(0.f, 0.f);
    if (lane == 0) {
      x = __ldg(a.draft_tokens + c0 + k);
      xv = __ldcg(a.xval + c0 + k);          // written by the CTA holding x
    }
    float Mt, Md, St, Sd;
    row_norm(a.lse_part + (long)(c0 + k) * a.chunks, a.chunks, lane, Mt, St, Md, Sd);
    if (lane == 0) {
      if (x < 0 || x >= a.vocab) {           // no CTA captured a logit: reject here
        px_s[k] = 0.f;
        qx_s[k] = 0.f;
      } else {
        px_s[k] = rel_exp(xv.x, Mt) / St;
        qx_s[k] = rel_exp(xv.y, Md) / Sd;
      }
      ws_s[k] = WalkState{c0 + k, Mt, Md, 1.f / St, 1.f / Sd, 0.f, 0, 0};
    }
  }
  __syncthreads();
  if (t == 0) {
    for (int k = 0; k < kMaxB; ++k) slot_of_step[k] = 0;
    for (int k = 0; k < B; ++k) {
      const int tk = tau_s[k];               // a label outside 1..B is ignored
      if (tk >= 1 && tk <= B) slot_of_step[tk - 1] = k;
    }
    int n = B, rej = -1;
    for (int s = 1; s <= B; ++s) {
      const int k = slot_of_step[s - 1];
      if (!(u_s[s - 1] * qx_s[k] < px_s[k])) { n = s - 1; rej = k; break; }
    }
    a.n_accept[b] = n;
    a.pos[b] = rej;
    if (rej < 0) {
      a.token[b] = -1;
      a.state[b] = WalkState{-1, 0.f, 0.f, 1.f, 1.f, 0.f, 0, 0};
    } else {
      WalkState w = ws_s[rej];
      w.u = u_s[B];
      a.state[b] = w;
    }
  }
}

// ---------------------------------------------------------------- K4a
constexpr int kStageSeqs = 2048;   // sequences whose cu_B fits the smem stage

template <typename T>
__global__ void __launch_bounds__(kThreads, 6)
lse_walk_kernel(const __grid_constant__ AcceptArgs a) {
  constexpr int N = Ld<T>::N, CE = kThreads * kVecs * N;
  __shared__ float4 scratch[kThreads / 32];
  __shared__ int last_s;
  __shared__ int32_t cu_s[kStageSeqs + 1];
  const int chunk = blockIdx.x, slot = blockIdx.y;
  grid_dep_launch();                         // the residual kernel may be scheduled
  const long row = (long)slot * a.vocab;
  const int v0 = chunk * CE;
  const int v1 = min(a.vocab, v0 + CE);
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  // every load of the CTA goes out first: both rows' entries, the draft
  // token, cu_B (for the sequence lookup at the end)
  uint4 wt[kVecs], wd[kVecs];
  load_strided<T>(tr, v0, v1, a.vec_ok, wt);
  load_strided<T>(dr, v0, v1, a.vec_ok, wd);
  const int x = __ldg(a.draft_tokens + slot);
  if (a.batch <= kStageSeqs)
    for (int i = threadIdx.x; i <= a.batch; i += kThreads) cu_s[i] = __ldg(a.cu_B + i);
  float mt, st, md, sd;
  thread_lse<T>(wt, mt, st);
  thread_lse<T>(wd, md, sd);
  if (x >= v0 && x < v1) {                   // this chunk holds the draft token
    const int off = x - v0;
    if (threadIdx.x == (off / N) % kThreads) {
      const int i = off / (kThreads * N), e = off % N;
      uint4 ut = wt[0], ud = wd[0];
#pragma unroll
      for (int ii = 1; ii < kVecs; ++ii)
        if (i == ii) { ut = wt[ii]; ud = wd[ii]; }
      float ft[N], fd[N];
      Ld<T>::unpack(ut, ft);
      Ld<T>::unpack(ud, fd);
      float vt = ft[0], vd = fd[0];
#pragma unroll
      for (int ee = 1; ee < N; ++ee)
        if (e == ee) { vt = ft[ee]; vd = fd[ee]; }
      a.xval[slot] = make_float2(vt, vd);
      __threadfence();                       // before this CTA's arrival below
    }
  } else if (chunk == 0 && threadIdx.x == 0 && (x < 0 || x >= a.vocab)) {
    raise_status(a.status, kStatusBadInput);
  }
  block_lse2(mt, st, md, sd, scratch);       // (its barrier also publishes cu_s, xval)
  // the sequence this slot belongs to, and whether this CTA finishes it
  int b, c0, B;
  if (a.batch <= kStageSeqs) {
    b = find_seq_smem(cu_s, a.batch, slot);
    c0 = cu_s[b];
    B = cu_s[b + 1] - c0;
  } else {
    b = find_seq(a.cu_B, a.batch, slot);
    c0 = __ldg(a.cu_B + b);
    B = __ldg(a.cu_B + b + 1) - c0;
  }
  if (threadIdx.x == 0) {
    a.lse_part[(long)slot * a.chunks + chunk] = make_float4(mt, st, md, sd);
    __threadfence();
    const unsigned total = (unsigned)B * a.chunks;
    last_s = atomicAdd(a.status + 1 + b, 1u) + 1 == total;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  if (B < 1 || B > kMaxB) {                  // malformed sequence: no walk
    if (threadIdx.x == 0) {
      a.n_accept[b] = 0; a.token[b] = -1; a.pos[b] = -1;
      a.state[b] = WalkState{-1, 0.f, 0.f, 1.f, 1.f, 0.f, 0, 0};
      raise_status(a.status, kStatusBadInput);
    }
    return;
  }
  walk(a, b, c0, B);
}

// Residual mass r = max(0, p - q) and target mass p of one entry.
__device__ __forceinline__ void res_pair(float t, float d, const WalkState &st, float &r,
                                         float &p) {
  p = rel_exp(t, st.Mt) * st.inv_st;
  const float q = rel_exp(d, st.Md) * st.inv_sd;
  r = fmaxf(p - q, 0.f);
}

// Inclusive block scan of two-sum pairs in thread order; returns the
// exclusive prefix of this thread and the block total (in all threads).
__device__ __forceinline__ Ff block_excl_scan(Ff x, Ff *warp_tot, Ff &total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ff inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Ff y = ff_shfl_up(inc, d);
    if (lane >= d) inc = ff_add(y, inc);
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  Ff base = ff_of(0.f), tot = ff_of(0.f);
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w == warp) base = tot;
    tot = ff_add(tot, warp_tot[w]);
  }
  total = tot;
  const Ff excl_in_warp = ff_add(inc, Ff{-x.hi, -x.lo});
  return ff_add(base, excl_in_warp);
}

// Sum of a thread's entries' residual and target masses (pairwise, so the
// rounding grows with log2 of the count).
template <int N>
__device__ __forceinline__ void tree_sum(float *v) {
#pragma unroll
  for (int h = N / 2; h > 0; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i) v[i] += v[i + h];
}

// ---------------------------------------------------------------- K4b
constexpr int kStageChunks = 1024;   // chunk sums staged in shared memory

template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
residual_kernel(const __grid_constant__ AcceptArgs a) {
  constexpr int N = Ld<T>::N, E = kVecs * N, CE = kThreads * E;
  __shared__ Ff warp_a[kThreads / 32], warp_b[kThreads / 32];
  __shared__ float4 chunk_s[kStageChunks];
  __shared__ int last_s, use_p_s, sel_s, best_s, lastpos_s;
  __shared__ Ff base_s, U_s, tot_s[2];
  const int chunk = blockIdx.x, b = blockIdx.y;
  grid_dep_wait();                           // the walk state comes from K4a
  WalkState st;
  {
    const uint4 *sp = reinterpret_cast<const uint4 *>(a.state + b);
    const uint4 s0 = __ldcg(sp), s1 = __ldcg(sp + 1);
    st.row = (int)s0.x; st.Mt = __uint_as_float(s0.y); st.Md = __uint_as_float(s0.z);
    st.inv_st = __uint_as_float(s0.w); st.inv_sd = __uint_as_float(s1.x);
    st.u = __uint_as_float(s1.y);
  }
  if (st.row < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long row = (long)st.row * a.vocab;
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  {
    const int v0 = chunk * CE, v1 = min(a.vocab, v0 + CE);
    uint4 wt[kVecs], wd[kVecs];
    load_strided<T>(tr, v0, v1, a.vec_ok, wt);
    load_strided<T>(dr, v0, v1, a.vec_ok, wd);
    float r[E], p[E];
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      float xt[N], xd[N];
      Ld<T>::unpack(wt[i], xt);
      Ld<T>::unpack(wd[i], xd);
#pragma unroll
      for (int e = 0; e < N; ++e) res_pair(xt[e], xd[e], st, r[i * N + e], p[i * N + e]);
    }
    tree_sum<E>(r);
    tree_sum<E>(p);
    Ff fr = ff_of(r[0]), fp = ff_of(p[0]);
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
      fr = ff_add(fr, ff_shfl_xor(fr, w));
      fp = ff_add(fp, ff_shfl_xor(fp, w));
    }
    if (lane == 0) { warp_a[warp] = fr; warp_b[warp] = fp; }
    __syncthreads();
    if (threadIdx.x == 0) {
      Ff tr_ = warp_a[0], tp = warp_b[0];
      for (int i = 1; i < kThreads / 32; ++i) { tr_ = ff_add(tr_, warp_a[i]); tp = ff_add(tp, warp_b[i]); }
      a.res_part[(long)b * a.chunks + chunk] = make_float4(tr_.hi, tr_.lo, tp.hi, tp.lo);
      __threadfence();
      last_s = atomicAdd(a.status + 1 + a.batch + b, 1u) + 1 == (unsigned)a.chunks;
    }
    __syncthreads();
  }
  if (!last_s) return;
  __threadfence();
  // -- the last CTA of sequence b draws the token.  (1) All chunk sums,
  // read once (staged in shared memory), give the totals S (residual) and
  // Sp (target); U = u * S, or u * Sp when the residual is empty (draw from
  // p).  (2) Warp 0 scans the chunk masses 32 at a time for the chunk whose
  // running sum first exceeds U.  (3) The block rescans that chunk in
  // vocabulary order.
  const float4 *rp = a.res_part + (long)b * a.chunks;
  {
    Ff S = ff_of(0.f), Sp = ff_of(0.f);
    for (int c = threadIdx.x; c < a.chunks; c += kThreads) {
      const float4 v = __ldcg(rp + c);
      if (c < kStageChunks) chunk_s[c] = v;
      S = ff_add(S, Ff{v.x, v.y});
      Sp = ff_add(Sp, Ff{v.z, v.w});
    }
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
      S = ff_add(S, ff_shfl_xor(S, w));
      Sp = ff_add(Sp, ff_shfl_xor(Sp, w));
    }
    __syncthreads();                         // warp_a / warp_b are free again
    if (lane == 0) { warp_a[warp] = S; warp_b[warp] = Sp; }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < kThreads / 32; ++i) { S = ff_add(S, warp_a[i]); Sp = ff_add(Sp, warp_b[i]); }
      tot_s[0] = S;
      tot_s[1] = Sp;
    }
    __syncthreads();
  }
  if (warp == 0) {
    const Ff S = tot_s[0];
    const int use_p = !(S.hi > 0.f);         // empty residual: draw from p
    const Ff tot = use_p ? tot_s[1] : S;
    // U = u * tot as a pair (u exact in fp32; the product's error by fma)
    const float u = st.u;
    const float uh = u * tot.hi;
    const Ff U = ff_add(Ff{uh, fmaf(u, tot.hi, -uh)}, ff_of(u * tot.lo));
    Ff carry = ff_of(0.f), last_base = ff_of(0.f), sel_base = ff_of(0.f);
    int sel = -1, last_nz = 0;
    for (int g = 0; g < a.chunks && sel < 0; g += 32) {
      const int c = g + lane;
      Ff m = ff_of(0.f);
      if (c < a.chunks) {
        const float4 v = c < kStageChunks ? chunk_s[c] : __ldcg(rp + c);
        m = use_p ? Ff{v.z, v.w} : Ff{v.x, v.y};
      }
      Ff inc = m;                             // inclusive scan over the lanes
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const Ff y = ff_shfl_up(inc, d);
        if (lane >= d) inc = ff_add(y, inc);
      }
      const Ff T1 = ff_add(carry, inc);
      const Ff T0 = ff_add(T1, Ff{-m.hi, -m.lo});
      const unsigned cross = __ballot_sync(0xffffffffu, m.hi > 0.f && ff_gt(T1, U));
      const unsigned nz = __ballot_sync(0xffffffffu, m.hi > 0.f);
      if (nz) {
        const int hl = 31 - __clz(nz);
        last_nz = g + hl;
        last_base = Ff{__shfl_sync(0xffffffffu, T0.hi, hl), __shfl_sync(0xffffffffu, T0.lo, hl)};
      }
      if (cross) {
        const int fl = __ffs(cross) - 1;
        sel = g + fl;
        sel_base = Ff{__shfl_sync(0xffffffffu, T0.hi, fl), __shfl_sync(0xffffffffu, T0.lo, fl)};
      }
      carry = Ff{__shfl_sync(0xffffffffu, T1.hi, 31), __shfl_sync(0xffffffffu, T1.lo, 31)};
    }
    if (lane == 0) {
      if (sel < 0) { sel = last_nz; sel_base = last_base; }
      sel_s = sel;
      base_s = sel_base;
      U_s = U;
      use_p_s = use_p;
      best_s = 0x7fffffff;
      lastpos_s = -1;
    }
  }
  __syncthreads();
  const bool use_p = use_p_s != 0;
  const int v0 = sel_s * CE, v1 = min(a.vocab, v0 + CE);
  float m[E];
  {
    uint4 wt[kVecs], wd[kVecs];
    load_contig<T>(tr, v0, v1, a.vec_ok, wt);
    load_contig<T>(dr, v0, v1, a.vec_ok, wd);
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      float xt[N], xd[N];
      Ld<T>::unpack(wt[i], xt);
      Ld<T>::unpack(wd[i], xd);
#pragma unroll
      for (int e = 0; e < N; ++e) {
        float r, p;
        res_pair(xt[e], xd[e], st, r, p);
        m[i * N + e] = use_p ? p : r;
      }
    }
  }
  Ff local = ff_of(0.f);
#pragma unroll
  for (int i = 0; i < E; ++i) local = ff_add(local, ff_of(m[i]));
  Ff total;
  const Ff excl = block_excl_scan(local, warp_a, total);
  const Ff U = U_s;
  Ff run = ff_add(base_s, excl);
  const int vt = v0 + threadIdx.x * E;
  int first = 0x7fffffff, last_pos = -1;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    run = ff_add(run, ff_of(m[i]));
    if (m[i] > 0.f) {
      last_pos = vt + i;
      if (first == 0x7fffffff && ff_gt(run, U)) first = vt + i;
    }
  }
  if (first != 0x7fffffff) atomicMin(&best_s, first);
  if (last_pos >= 0) atomicMax(&lastpos_s, last_pos);
  __syncthreads();
  if (threadIdx.x == 0) a.token[b] = best_s != 0x7fffffff ? best_s : lastpos_s;
}

void mark(void *const *events, int i, cudaStream_t stream) {
  if (events != nullptr) record_event(events[i], stream);
}

template <typename T>
cudaError_t launch_all(const AcceptArgs &a, int total_B, cudaStream_t stream,
                       void *const *events) {
  mark(events, 0, stream);
  lse_walk_kernel<T><<<dim3(a.chunks, total_B), kThreads, 0, stream>>>(a);
  mark(events, 1, stream);
  cudaError_t e = launch_pdl(residual_kernel<T>, dim3(a.chunks, a.batch), dim3(kThreads), 0,
                             stream, a);
  mark(events, 2, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

simsd_status accept_check(const simsd_accept_desc *d) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (d->dtype != SIMSD_F32 && d->dtype != SIMSD_BF16) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->batch > 65535 || d->vocab < 1 || d->B_max < 1 ||
      d->B_max > kMaxB || d->total_B < d->batch ||
      (int64_t)d->total_B > (int64_t)d->batch * d->B_max || d->total_B > 65535 ||
      d->vocab > (1 << 30))
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

// Clears the status head of the workspace and launches K4a and K4b.
simsd_status run_accept(const simsd_accept_desc *d, const AcceptWs &w, char *ws,
                        cudaStream_t stream, void *const *events) {
  if (cudaMemsetAsync(ws + w.off_status, 0, w.status_bytes, stream) != cudaSuccess)
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
  a.xval = (float2 *)(ws + w.off_x);
  a.state = (WalkState *)(ws + w.off_state);
  a.res_part = (float4 *)(ws + w.off_res);
  a.status = (uint32_t *)(ws + w.off_status);
  a.batch = d->batch;
  a.vocab = d->vocab;
  a.B_max = d->B_max;
  a.chunks = w.chunks;
  const size_t es = d->dtype == SIMSD_BF16 ? 2 : 4;
  a.vec_ok = ((size_t)d->vocab * es) % 16 == 0 &&
             ((uintptr_t)d->target_logits % 16) == 0 &&
             ((uintptr_t)d->draft_logits % 16) == 0;
  cudaError_t e = d->dtype == SIMSD_BF16
                      ? launch_all<__nv_bfloat16>(a, d->total_B, stream, events)
                      : launch_all<float>(a, d->total_B, stream, events);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
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
                                void *const events[3]) {
  simsd_status st = accept_check(d);
  if (st != SIMSD_OK) return st;
  if (!d->target_logits || !d->draft_logits || !d->draft_tokens || !d->tau ||
      !d->cu_B || !d->uniforms || !d->n_accept || !d->token || !d->pos)
    return SIMSD_ERR_NULL;
  const AcceptWs w = accept_ws(d);
  if (d->workspace == nullptr || ((uintptr_t)d->workspace % kAlign) != 0 ||
      d->workspace_bytes < w.total)
    return SIMSD_ERR_WORKSPACE;
  return run_accept(d, w, (char *)d->workspace, (cudaStream_t)stream_ptr, events);
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
  return run_accept(d, w, ws, (cudaStream_t)stream_ptr, nullptr);
}

}  // extern "C"
