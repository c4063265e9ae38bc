// vocab.cuh -- device helpers of the kernels that sweep vocabulary rows
// (the acceptance rules and the draft-side step): compensated fp32 pairs,
// 2^x on the MUFU, thread-block-cluster barriers and distributed shared
// memory, and 16-byte vectors of bf16 or fp32 logits.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace simsd {
namespace vocab {

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
__device__ __forceinline__ Ff ff_neg(Ff a) { return Ff{-a.hi, -a.lo}; }
__device__ __forceinline__ Ff ff_shfl_xor(Ff a, int m) {
  return Ff{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}
__device__ __forceinline__ Ff ff_shfl_up(Ff a, int d) {
  return Ff{__shfl_up_sync(0xffffffffu, a.hi, d), __shfl_up_sync(0xffffffffu, a.lo, d)};
}
__device__ __forceinline__ Ff ff_shfl(Ff a, int l) {
  return Ff{__shfl_sync(0xffffffffu, a.hi, l), __shfl_sync(0xffffffffu, a.lo, l)};
}
// a > u where u is a pair: compare the exact sums' signs
__device__ __forceinline__ bool ff_gt(Ff a, Ff u) {
  const Ff d = ff_add(a, ff_neg(u));
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

// 2^x on the MUFU (approximate, ~2 ulp; subnormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The logits' scale into log2 units, log2(e) / temperature, as an
// unevaluated float pair hi + lo (from double on the host): a single float
// would act like a temperature off by up to 2^-24 relative, which shifts
// the whole distribution's shape consistently (an error that does not
// average out over the vocabulary, unlike per-entry rounding).
// hi is the float just below the exact scale, so lo > 0: a -inf logit then
// gives -inf + (-inf) in the argument (mass 0), never -inf + inf (NaN).
struct Scale {
  float hi, lo;
};
inline Scale scale_of(double temperature) {
  const double l = 1.4426950408889634074 / temperature;
  float hi = (float)l;
  if ((double)hi >= l) hi = nextafterf(hi, 0.f);
  return Scale{hi, (float)(l - (double)hi)};
}

// 2^(x (hi + lo) - R): x hi - R exact before one rounding, then x lo added
// with one more (the rounding is at the scale of the result's argument).
__device__ __forceinline__ float rel_exp(float x, float R, Scale ls) {
  return ex2(fmaf(x, ls.lo, fmaf(x, ls.hi, -R)));
}

// References (the R above) are whole numbers: ceil(max * hi) for a set of
// logits whose largest is max, so every entry's argument is at most ~0.
// Partial sums taken against different references then combine through
// exact powers of two (exp2_int), and a hierarchy of partial masses
// (slices, pieces, ranges) adds up to exactly what a scan of the entries
// against the final reference sees, up to the sums' own rounding.
__device__ __forceinline__ float ref_of(float mx, Scale ls) { return ceilf(mx * ls.hi); }

// 2^d for a whole number d (0 below the normal range, -inf included).
__device__ __forceinline__ float exp2_int(float d) {
  return d < -126.f ? 0.f : d > 127.f ? INFINITY : __int_as_float(((int)d + 127) << 23);
}

// a / b for pairs (Dekker's division: quotient, remainder by fma, one
// correction term); a / a is exactly (1, 0).
__device__ __forceinline__ Ff ff_div(Ff a, Ff b) {
  const float q1 = a.hi / b.hi;
  const float r = fmaf(-q1, b.hi, a.hi) + a.lo - q1 * b.lo;
  const float q2 = r / b.hi;
  const float hi = q1 + q2;
  return Ff{hi, q2 - (hi - q1)};
}


__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem(const void *p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_dsmem2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_dsmem_i32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------- logits
// Raw 16-byte vectors of logits: unpacking, lane-wise maximum, the -inf fill.
template <typename T> struct Ld;
template <> struct Ld<float> {
  static constexpr int N = 4;
  static constexpr uint32_t kNegInf = 0xff800000u;
  static __device__ __forceinline__ uint4 neg_inf() { return make_uint4(kNegInf, kNegInf, kNegInf, kNegInf); }
  static __device__ __forceinline__ float value(float v) { return v; }
  static __device__ __forceinline__ float neg_inf_elem() { return -INFINITY; }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  // the vector at p (16-byte aligned if `aligned`): entries past `valid`
  // (which may be <= 0) read as -inf
  static __device__ __forceinline__ uint4 load(const float *p, int valid, bool aligned) {
    if (aligned && valid >= N) return *reinterpret_cast<const uint4 *>(p);
    uint32_t r[N];
#pragma unroll
    for (int e = 0; e < N; ++e) r[e] = e < valid ? __float_as_uint(p[e]) : kNegInf;
    return make_uint4(r[0], r[1], r[2], r[3]);
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
  static constexpr uint32_t kNegInf2 = 0xff80ff80u;
  static __device__ __forceinline__ uint4 neg_inf() { return make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2); }
  static __device__ __forceinline__ float value(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 neg_inf_elem() { return __ushort_as_bfloat16(0xff80); }
  static __device__ __forceinline__ void unpack(uint4 v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint4 load(const __nv_bfloat16 *p, int valid, bool aligned) {
    if (aligned && valid >= N) return *reinterpret_cast<const uint4 *>(p);
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = 2 * i < valid ? __bfloat16_as_ushort(p[2 * i]) : 0xff80u;
      const uint32_t hi = 2 * i + 1 < valid ? __bfloat16_as_ushort(p[2 * i + 1]) : 0xff80u;
      r[i] = lo | (hi << 16);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
  }
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  // packed maximum of the bf16 pairs (exact), then of the two halves
  static __device__ __forceinline__ float vmax(const uint4 *w, int n) {
    uint32_t m = kNegInf2;
    for (int i = 0; i < n; ++i) m = max2(m, max2(max2(w[i].x, w[i].y), max2(w[i].z, w[i].w)));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
};

// Element e (dynamic) of the N entries held in vector w.
template <typename T>
__device__ __forceinline__ float pick(uint4 w, int e) {
  float f[Ld<T>::N];
  Ld<T>::unpack(w, f);
  float v = f[0];
#pragma unroll
  for (int i = 1; i < Ld<T>::N; ++i)
    if (e == i) v = f[i];
  return v;
}

// ------------------------------------------------------------ acceptance
// The residual in target-mass units: with e_t = 2^(x ls - Mt) (so p =
// e_t / St) and e_d = 2^(y ls - Md) (q = e_d / Sd), S_t max(0, p - q) =
// max(0, e_t - rho e_d), rho = St / Sd (a pair).  The draw is the same in
// any common unit, so no normaliser is rounded into the entries.  rho e_d
// takes a product and one fused multiply-add, the difference its own
// rounding (no contraction), so identical target and draft rows (rho
// exactly 1) give an exactly empty residual, and the residual pass and the
// draw compute the same values.
__device__ __forceinline__ float draft_mass(float y, float Md, Ff rho, Scale ls) {
  const float e = rel_exp(y, Md, ls);
  return __fmaf_rn(e, rho.lo, __fmul_rn(e, rho.hi));
}
__device__ __forceinline__ float residual(float et, float ed) { return fmaxf(__fsub_rn(et, ed), 0.f); }


// Producer warp: one piece of a row slice into a ring stage, completion on
// `full` (bulk copy with a byte count, or element copies by the whole warp
// and a plain arrival; those fill the rest of the last 16-byte vector with
// -inf, since consumers read whole vectors).
template <typename T>
__device__ __noinline__ void copy_piece(uint8_t *dst, uint32_t dst_s, const T *src, int n,
                                           uint32_t full, bool bulk, int lane) {
  if (bulk) {
    if (lane == 0) {
      mbar_arrive_expect_tx(full, (uint32_t)(n * sizeof(T)));
      bulk_load(dst_s, src, (uint32_t)(n * sizeof(T)), full);
    }
  } else {
    constexpr int N = 16 / (int)sizeof(T);
    T *d = reinterpret_cast<T *>(dst);
    for (int e = lane; e < n; e += 32) d[e] = src[e];
    for (int e = n + lane; e < (n + N - 1) / N * N; e += 32) d[e] = Ld<T>::neg_inf_elem();
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
  }
}

// Warp-wide choice among up to 32 consecutive ranges: lane i holds the
// mass m of range i (0 for lanes without one), the ranges start at `base`.
// Returns the first range whose running total exceeds U (else the last one
// with mass, else 0), and in *start the running total before it.
static __device__ __noinline__ int warp_pick(Ff m, Ff base, Ff U, Ff *start) {
  const int lane = threadIdx.x & 31;
  Ff inc = m;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Ff y = ff_shfl_up(inc, d);
    if (lane >= d) inc = ff_add(y, inc);
  }
  const Ff run = ff_add(base, inc);
  const unsigned cross = __ballot_sync(0xffffffffu, m.hi > 0.f && ff_gt(run, U));
  const unsigned nz = __ballot_sync(0xffffffffu, m.hi > 0.f);
  const int ch = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : 0);
  *start = ff_shfl(ff_add(base, ff_add(inc, ff_neg(m))), ch);
  return ch;
}

// ------------------------------------------------------------ part draws
// Inverse-CDF draws from one row after a chunk pass, which left per part
// (1/8 of a 32 KB chunk, contiguous in the vocabulary; parts in (chunk,
// part) order are in vocabulary order) what the part's mass is made of.
// All 32 lanes call these; every lane gets the result.
//
// locate_part: lane l holds parts l + 32 i (i < HELD) in h, the rest are
// read from pr; mass_of(part) gives a part's mass (pairs, in the units of
// U).  Returns the part whose running mass first exceeds U, else the last
// part with mass (0 if none), and in *start the mass before it.
template <int HELD, typename P, typename MassOf>
__device__ int locate_part(const P *pr, const P (&h)[HELD], int n_ent, Ff U, MassOf mass_of, int lane,
                           Ff *start_out) {
  Ff base = ff_of(0.f), last_start = ff_of(0.f);
  int sel = -1, last_nz = 0;
  auto group = [&](int g0, const P &v) {            // parts g0 .. g0 + 31
    const Ff m = g0 + lane < n_ent ? mass_of(v) : ff_of(0.f);
    Ff inc = m;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const Ff y = ff_shfl_up(inc, d);
      if (lane >= d) inc = ff_add(y, inc);
    }
    const Ff run = ff_add(base, inc);
    const Ff start = ff_add(base, ff_add(inc, ff_neg(m)));
    const unsigned cross = __ballot_sync(0xffffffffu, m.hi > 0.f && ff_gt(run, U));
    const unsigned nz = __ballot_sync(0xffffffffu, m.hi > 0.f);
    if (cross) {
      const int l = __ffs(cross) - 1;
      sel = g0 + l;
      base = ff_shfl(start, l);
    } else {
      if (nz) {
        const int l = 31 - __clz(nz);
        last_nz = g0 + l;
        last_start = ff_shfl(start, l);
      }
      base = ff_shfl(run, 31);
    }
  };
#pragma unroll
  for (int i = 0; i < HELD; ++i)
    if (sel < 0 && 32 * i < n_ent) group(32 * i, h[i]);
  for (int g0 = 32 * HELD; g0 < n_ent && sel < 0; g0 += 32) {
    const P v = g0 + lane < n_ent ? __ldcg(pr + g0 + lane) : P{};
    group(g0, v);
  }
  if (sel < 0) {
    sel = last_nz;
    base = last_start;
  }
  *start_out = base;
  return sel;
}

// scan_part: the entries [p0, p0 + n) of ROWS rows (rows[r] + p0 is the
// part's first entry in row r), column by column in vocabulary order
// (lane l: vector l of each column of 32 vectors), with entry_mass(f, m)
// turning the ROWS rows' values of a vector into its N masses.  The loads
// of kBatch columns are issued together (a part of a 32 KB chunk is 8
// columns: one round for one row, two for two).  Running masses are fp32 relative to the part's
// start; dd is U minus the mass before the part.  Returns the first entry
// whose running mass exceeds dd, else the last entry with mass (-1: none).
template <typename T, int ROWS, typename EntryMass>
__device__ int scan_part(const T *const (&rows)[ROWS], int p0, int n, int part_vecs, float dd, bool bulk,
                         int lane, EntryMass entry_mass) {
  constexpr int N = Ld<T>::N;
  constexpr int kBatch = 8 / ROWS;
  float col_base = 0.f;
  int first = 0x7fffffff, last_pos = -1;
#pragma unroll 1
  for (int c0 = 0; c0 * 32 < part_vecs && first == 0x7fffffff; c0 += kBatch) {
    uint4 w[kBatch][ROWS];
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {
      const int e0 = ((c0 + c) * 32 + lane) * N;
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
        w[c][r] = (c0 + c) * 32 < part_vecs ? Ld<T>::load(rows[r] + p0 + e0, n - e0, bulk) : Ld<T>::neg_inf();
    }
#pragma unroll
    for (int c = 0; c < kBatch; ++c) {
      if (first != 0x7fffffff || (c0 + c) * 32 >= part_vecs) break;   // warp-uniform
      const int e0 = ((c0 + c) * 32 + lane) * N;
      float f[ROWS][N], m[N];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) Ld<T>::unpack(w[c][r], f[r]);
      entry_mass(f, m);
      float lane_mass = 0.f;
#pragma unroll
      for (int e = 0; e < N; ++e) {
        lane_mass += m[e];
        if (m[e] > 0.f) last_pos = p0 + e0 + e;
      }
      float inc = lane_mass;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += y;
      }
      const float prev = __shfl_up_sync(0xffffffffu, inc, 1);
      const float start = col_base + (lane ? prev : 0.f);
      if (dd < col_base + inc) {
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          run += m[e];
          if (first == 0x7fffffff && m[e] > 0.f && start + run > dd) first = p0 + e0 + e;
        }
      }
      first = __reduce_min_sync(0xffffffffu, first);
      col_base += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
  last_pos = __reduce_max_sync(0xffffffffu, last_pos);
  return first != 0x7fffffff ? first : last_pos;
}

// part_draw: a draw from one row's softmax after a chunk pass that left
// per part its reference (.x) and sum of 2^(l ls - reference) (.y); M is the
// row's reference and U the draw point, both in units of 2^M.
template <typename T, int HELD>
__device__ int part_draw(const float4 *pr, const float4 (&h)[HELD], int n_ent, float M, Ff U,
                         const T *row, int vocab, int chunk, bool bulk, Scale ls, int lane) {
  constexpr int N = Ld<T>::N;
  constexpr int kParts = 8;
  const int part_len = chunk / kParts;
  auto mass_of = [&](const float4 &v) {
    const float w = (M != -INFINITY && v.x != -INFINITY) ? exp2_int(v.x - M) : 0.f;
    return ff_of(v.y > 0.f ? v.y * w : 0.f);
  };
  Ff base;
  const int sel = locate_part<HELD>(pr, h, n_ent, U, mass_of, lane, &base);
  const int p0 = (sel / kParts) * chunk + (sel % kParts) * part_len;
  const Ff D0 = ff_add(U, ff_neg(base));
  const T *const rows[1] = {row};
  return scan_part<T, 1>(rows, p0, min(part_len, vocab - p0), part_len / N, D0.hi + D0.lo, bulk, lane,
                         [&](const float (&f)[1][N], float (&m)[N]) {
#pragma unroll
                           for (int e = 0; e < N; ++e) m[e] = rel_exp(f[0][e], M, ls);
                         });
}

// ------------------------------------------------- chunk pass control words
// claim[0]: the chunk pass's item counter; claim[1]: set when one of its
// waits gave up (its partials are then incomplete); claim[2]: how many CTAs
// of the kernel reading the partials have read claim[1].  One thread per
// CTA calls chunk_flag_read after grid_dep_wait (the chunk pass has
// finished, its writes visible): it returns claim[1] and the CTA's ticket
// (its place in the count).  The CTA whose ticket is the last calls
// chunk_flag_reset before it exits -- every CTA has read the flag by then
// -- so the next call starts from zeros.  The ticket is compared only at
// the end, so the atomic's round trip overlaps the CTA's work.
__device__ __forceinline__ int chunk_flag_read(int *claim, int *ticket) {
  const int fail = *(volatile int *)(claim + 1);
  __threadfence();                               // the read precedes the count
  *ticket = atomicAdd(claim + 2, 1);
  return fail;
}
__device__ __forceinline__ void chunk_flag_reset(int *claim, int ticket, int ctas) {
  if (ticket != ctas - 1) return;
  __threadfence();
  claim[0] = 0;
  claim[1] = 0;
  claim[2] = 0;
}

}  // namespace vocab
}  // namespace simsd
