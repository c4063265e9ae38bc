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
constexpr int kLseVec = 2;                        // 16-byte loads per row per thread per pass
constexpr int kLseChunk = 8192;                   // K4a vocabulary chunk
constexpr int kResPer = 8;                        // residual entries per thread
constexpr int kResChunk = kThreads * kResPer;     // 2048
constexpr float kLog2e = 1.4426950408889634f;

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

// Per sequence, after the walk: rejected slot (-1: none), that slot's
// references (log2 units) and normalisers.
struct WalkState {
  int rej;
  float Mt, Md, St, Sd;
};

struct AcceptWs {
  size_t off_status, status_bytes, off_lse, off_x, off_state, off_res, total;
  int lse_chunks, res_chunks;
};

// status word, then two per-sequence arrival counters; the whole head is
// cleared at the start of every call.
AcceptWs accept_ws(const simsd_accept_desc *d) {
  AcceptWs w;
  w.lse_chunks = (d->vocab + kLseChunk - 1) / kLseChunk;
  w.res_chunks = (d->vocab + kResChunk - 1) / kResChunk;
  size_t off = 0;
  w.off_status = off;
  w.status_bytes = sizeof(uint32_t) * (1 + 2 * (size_t)d->batch);
  off = align_up(off + w.status_bytes, kAlign);
  w.off_lse = off;    off = align_up(off + (size_t)d->total_B * w.lse_chunks * sizeof(float4), kAlign);
  w.off_x = off;      off = align_up(off + (size_t)d->total_B * sizeof(float2), kAlign);
  w.off_state = off;  off = align_up(off + (size_t)d->batch * sizeof(WalkState), kAlign);
  w.off_res = off;    off = align_up(off + (size_t)d->batch * w.res_chunks * sizeof(float4), kAlign);
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
  float4 *lse_part;     // [total_B][lse_chunks]: (R_t, s_t, R_d, s_d)
  float2 *xval;         // [total_B]: target and draft logit at the draft token
  WalkState *state;     // [batch]
  float4 *res_part;     // [batch][res_chunks]: residual pair, target-mass pair
  uint32_t *status;     // [0]: status word; [1..batch]: K4a counters; then K4b's
  int batch, vocab, B_max, lse_chunks, res_chunks, vec_ok;
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

// Fold n logits into (R, s); R moves to the new maximum (in log2 units).
__device__ __forceinline__ void accum(float &m, float &s, const float *x, int n) {
  float mx = -INFINITY;
  for (int i = 0; i < n; ++i) mx = fmaxf(mx, x[i]);
  const float R = mx * kLog2e;
  if (R > m) { s *= ex2(m - R); m = R; }
  if (m == -INFINITY) return;
  for (int i = 0; i < n; ++i) s += rel_exp(x[i], m);
}

template <typename T> struct Ld;
template <> struct Ld<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ uint4 raw(const float *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
  }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ float one(const float *p) { return __ldg(p); }
};
template <> struct Ld<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ uint4 raw(const __nv_bfloat16 *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
  }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
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

// Row maximum and normaliser of one slot from its chunk partials (one warp).
__device__ __forceinline__ void row_norm(const float4 *pp, int chunks, int lane,
                                         float &Mt, float &St, float &Md, float &Sd) {
  float mt = -INFINITY, md = -INFINITY;
  for (int c = lane; c < chunks; c += 32) {
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
  for (int c = lane; c < chunks; c += 32) {
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

// The walk of sequence b (whole CTA): p(x), q(x) per slot, then steps in tau
// order; writes the outputs and the walk state.
template <typename T>
__device__ void walk(const AcceptArgs &a, int b, int c0, int B) {
  __shared__ float px_s[kMaxB], qx_s[kMaxB];
  __shared__ WalkState ws_s[kMaxB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = warp; k < B; k += kThreads / 32) {
    float Mt, Md, St, Sd;
    row_norm(a.lse_part + (long)(c0 + k) * a.lse_chunks, a.lse_chunks, lane, Mt, St, Md, Sd);
    if (lane == 0) {
      const long row = (long)(c0 + k) * a.vocab;
      const int x = __ldg(a.draft_tokens + c0 + k);
      float tx, dx;
      if (x < 0 || x >= a.vocab) {
        raise_status(a.status, kStatusBadInput);
        tx = Ld<T>::one((const T *)a.target + row);
        dx = Ld<T>::one((const T *)a.draft + row);
      } else {
        const float2 xv = __ldcg(a.xval + c0 + k);   // captured by K4a
        tx = xv.x;
        dx = xv.y;
      }
      px_s[k] = rel_exp(tx, Mt) / St;
      qx_s[k] = rel_exp(dx, Md) / Sd;
      ws_s[k] = WalkState{k, Mt, Md, St, Sd};
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
      a.state[b] = WalkState{-1, 0.f, 0.f, 1.f, 1.f};
    } else {
      a.state[b] = ws_s[rej];
    }
  }
}

// ---------------------------------------------------------------- K4a
constexpr int kStageSeqs = 2048;   // sequences whose cu_B fits the smem stage

template <typename T>
__global__ void __launch_bounds__(kThreads, 8)
lse_walk_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ float4 scratch[kThreads / 32];
  __shared__ int last_s;
  __shared__ int32_t cu_s[kStageSeqs + 1];
  const int chunk = blockIdx.x, slot = blockIdx.y;
  grid_dep_launch();                         // the residual kernel may be scheduled
  // independent of the stream below: the draft token and cu_B (for the
  // sequence lookup at the end) are requested first
  int x = -1;
  if (threadIdx.x == 0) x = __ldg(a.draft_tokens + slot);
  if (a.batch <= kStageSeqs)
    for (int i = threadIdx.x; i <= a.batch; i += kThreads) cu_s[i] = __ldg(a.cu_B + i);
  const long row = (long)slot * a.vocab;
  const int v0 = chunk * kLseChunk;
  const int v1 = min(a.vocab, v0 + kLseChunk);
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
  constexpr int N = Ld<T>::N;
  int tail0 = v0;
  if (a.vec_ok) {
    // kLseVec independent 16-byte loads per row in flight per thread
    constexpr int STEP = kThreads * N;
    int v = v0 + threadIdx.x * N;
    for (; v + (kLseVec - 1) * STEP + N <= v1; v += kLseVec * STEP) {
      uint4 rt[kLseVec], rd[kLseVec];
#pragma unroll
      for (int i = 0; i < kLseVec; ++i) { rt[i] = Ld<T>::raw(tr + v + i * STEP); rd[i] = Ld<T>::raw(dr + v + i * STEP); }
#pragma unroll
      for (int i = 0; i < kLseVec; ++i) {
        float xt[N], xd[N];
        Ld<T>::unpack(rt[i], xt);
        Ld<T>::unpack(rd[i], xd);
        accum(mt, st, xt, N);
        accum(md, sd, xd, N);
      }
    }
    for (; v + N <= v1; v += STEP) {
      float xt[N], xd[N];
      Ld<T>::unpack(Ld<T>::raw(tr + v), xt);
      Ld<T>::unpack(Ld<T>::raw(dr + v), xd);
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
  block_lse2(mt, st, md, sd, scratch);       // (its barrier also publishes cu_s)
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
    if (x >= v0 && x < v1)                   // this chunk holds the draft token
      a.xval[slot] = make_float2(Ld<T>::one(tr + x), Ld<T>::one(dr + x));
    a.lse_part[(long)slot * a.lse_chunks + chunk] = make_float4(mt, st, md, sd);
    __threadfence();
    const unsigned total = (unsigned)B * a.lse_chunks;
    last_s = atomicAdd(a.status + 1 + b, 1u) + 1 == total;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  if (B < 1 || B > kMaxB) {                  // malformed sequence: no walk
    if (threadIdx.x == 0) {
      a.n_accept[b] = 0; a.token[b] = -1; a.pos[b] = -1;
      a.state[b] = WalkState{-1, 0.f, 0.f, 1.f, 1.f};
      raise_status(a.status, kStatusBadInput);
    }
    return;
  }
  walk<T>(a, b, c0, B);
}

// Residual mass r = max(0, p - q) and target mass p of one entry.
__device__ __forceinline__ void res_pair(float t, float d, const WalkState &st,
                                         float inv_st, float inv_sd, float &r, float &p) {
  p = rel_exp(t, st.Mt) * inv_st;
  const float q = rel_exp(d, st.Md) * inv_sd;
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

// ---------------------------------------------------------------- K4b
// The 8 residual / target masses of entries v0..v0+7 of the rejected row.
template <typename T>
__device__ __forceinline__ void res_block(const T *tr, const T *dr, int v0, int vocab, bool vec,
                                          const WalkState &st, float inv_st, float inv_sd,
                                          float *r, float *p) {
  constexpr int N = Ld<T>::N;
  if (vec && v0 + kResPer <= vocab) {
    float xt[kResPer], xd[kResPer];
#pragma unroll
    for (int h = 0; h < kResPer / N; ++h) {
      Ld<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(tr + v0 + h * N)), xt + h * N);
      Ld<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(dr + v0 + h * N)), xd + h * N);
    }
#pragma unroll
    for (int i = 0; i < kResPer; ++i) res_pair(xt[i], xd[i], st, inv_st, inv_sd, r[i], p[i]);
  } else {
#pragma unroll
    for (int i = 0; i < kResPer; ++i) {
      r[i] = p[i] = 0.f;
      if (v0 + i < vocab)
        res_pair(Ld<T>::one(tr + v0 + i), Ld<T>::one(dr + v0 + i), st, inv_st, inv_sd, r[i], p[i]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
residual_kernel(const __grid_constant__ AcceptArgs a) {
  __shared__ Ff warp_tot[kThreads / 32], rs[kThreads / 32], ps[kThreads / 32];
  __shared__ int last_s, sel_s, use_p_s, best_s, lastpos_s;
  __shared__ Ff base_s, U_s;
  const int chunk = blockIdx.x, b = blockIdx.y;
  grid_dep_wait();                           // the walk state comes from K4a
  const WalkState st = a.state[b];
  if (st.rej < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_st = 1.f / st.St, inv_sd = 1.f / st.Sd;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const long row = (long)(c0 + st.rej) * a.vocab;
  const T *tr = (const T *)a.target + row;
  const T *dr = (const T *)a.draft + row;
  {
    float r[kResPer], p[kResPer];
    res_block<T>(tr, dr, chunk * kResChunk + threadIdx.x * kResPer, a.vocab, a.vec_ok, st,
                 inv_st, inv_sd, r, p);
    float sr = 0.f, sp = 0.f;
#pragma unroll
    for (int i = 0; i < kResPer; ++i) { sr += r[i]; sp += p[i]; }
    Ff fr = ff_of(sr), fp = ff_of(sp);
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
      fr = ff_add(fr, ff_shfl_xor(fr, w));
      fp = ff_add(fp, ff_shfl_xor(fp, w));
    }
    if (lane == 0) { rs[warp] = fr; ps[warp] = fp; }
    __syncthreads();
    if (threadIdx.x == 0) {
      Ff tr_ = rs[0], tp = ps[0];
      for (int i = 1; i < kThreads / 32; ++i) { tr_ = ff_add(tr_, rs[i]); tp = ff_add(tp, ps[i]); }
      a.res_part[(long)b * a.res_chunks + chunk] = make_float4(tr_.hi, tr_.lo, tp.hi, tp.lo);
      __threadfence();
      last_s = atomicAdd(a.status + 1 + a.batch + b, 1u) + 1 == (unsigned)a.res_chunks;
    }
    __syncthreads();
  }
  if (!last_s) return;
  __threadfence();
  // -- the last CTA of sequence b draws the token.  Warp 0 scans the chunk
  // masses 32 at a time for the chunk whose running sum first exceeds U.
  const float4 *rp = a.res_part + (long)b * a.res_chunks;
  if (warp == 0) {
    Ff S = ff_of(0.f), Sp = ff_of(0.f);
    for (int c = lane; c < a.res_chunks; c += 32) {
      const float4 v = __ldcg(rp + c);
      S = ff_add(S, Ff{v.x, v.y});
      Sp = ff_add(Sp, Ff{v.z, v.w});
    }
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
      S = ff_add(S, ff_shfl_xor(S, w));
      Sp = ff_add(Sp, ff_shfl_xor(Sp, w));
    }
    const int use_p = !(S.hi > 0.f);         // empty residual: draw from p
    const Ff tot = use_p ? Sp : S;
    // U = u * tot as a pair (u exact in fp32; the product's error by fma)
    const float u = __ldg(a.uniforms + (long)b * (a.B_max + 1) + B);
    const float uh = u * tot.hi;
    const Ff U = ff_add(Ff{uh, fmaf(u, tot.hi, -uh)}, ff_of(u * tot.lo));
    Ff carry = ff_of(0.f), last_base = ff_of(0.f), sel_base = ff_of(0.f);
    int sel = -1, last_nz = 0;
    for (int c0_ = 0; c0_ < a.res_chunks && sel < 0; c0_ += 32) {
      const int c = c0_ + lane;
      Ff m = ff_of(0.f);
      if (c < a.res_chunks) {
        const float4 v = __ldcg(rp + c);
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
        last_nz = c0_ + hl;
        last_base = Ff{__shfl_sync(0xffffffffu, T0.hi, hl), __shfl_sync(0xffffffffu, T0.lo, hl)};
      }
      if (cross) {
        const int fl = __ffs(cross) - 1;
        sel = c0_ + fl;
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
  const int v0 = sel_s * kResChunk + threadIdx.x * kResPer;
  float m[kResPer];
  {
    float r[kResPer], p[kResPer];
    res_block<T>(tr, dr, v0, a.vocab, a.vec_ok, st, inv_st, inv_sd, r, p);
#pragma unroll
    for (int i = 0; i < kResPer; ++i) m[i] = use_p_s ? p[i] : r[i];
  }
  float local = 0.f;
#pragma unroll
  for (int i = 0; i < kResPer; ++i) local += m[i];
  Ff total;
  const Ff excl = block_excl_scan(ff_of(local), warp_tot, total);
  const Ff base = ff_add(base_s, excl);
  const Ff U = U_s;
  float lp = 0.f;
  int first = 0x7fffffff, last_pos = -1;
#pragma unroll
  for (int i = 0; i < kResPer; ++i) {
    lp += m[i];
    if (m[i] > 0.f) {
      last_pos = v0 + i;
      if (first == 0x7fffffff && ff_gt(ff_add(base, ff_of(lp)), U)) first = v0 + i;
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
  lse_walk_kernel<T><<<dim3(a.lse_chunks, total_B), kThreads, 0, stream>>>(a);
  mark(events, 1, stream);
  cudaError_t e = launch_pdl(residual_kernel<T>, dim3(a.res_chunks, a.batch), dim3(kThreads), 0,
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
