// accept.cu -- K4: rejection-sampling acceptance along the temporal order.
//
// SimSD section 4 "Speculative Decoding Pipeline", acceptance: standard
// rejection sampling along the draft-induced temporal order; the longest
// accepted prefix is committed.  For sequence b, step t = 1..B tests the
// slot k = tau^-1(t) with draft token x: p = softmax(target row k / T),
// q = softmax(draft row k / T) at temperature T (1 by default); accept iff
// u[t-1] * q(x) < p(x) (fp32).  At the first rejection a token is drawn
// from max(0, p - q) normalised (p itself when that is empty) by inverse
// CDF with u[B].  The greedy rule and sample matching have their own,
// simpler kernels at the end of this file.
//
// One launch; one thread-block cluster of C CTAs per sequence (C <= 16, from
// a makespan estimate over the resident-cluster waves: 8-16 for small
// batches, 1-2 for large ones), CTA r owning the vocabulary slice
// [r * per, (r + 1) * per) of every row of the sequence.  Each CTA streams
// its slices of the 2B rows (target and draft of every slot) in pieces of
// equal size (at most 32 KB) through a 6-stage shared-memory ring filled by
// bulk copies (one producer warp); two groups of 8 consumer warps take
// alternate pieces, so one group's waits and reductions overlap the other's
// exponentials:
//   1. per (slot, row): maximum and sum of exponentials of the slice;
//   2. cluster barrier; every CTA merges the C slices' partials through
//      distributed shared memory, evaluates p(x), q(x) and walks the steps
//      (identically: same inputs, same order; CTA 0 writes the outputs);
//   3. on a rejection every CTA streams its slices of the rejected slot's
//      two rows again (from L2) for the residual and target masses of 16
//      contiguous vocabulary ranges of each piece;
//   4. cluster barrier; every CTA reads the C slice totals, so all agree on
//      the CTA whose slice holds u * S; one warp of that CTA narrows down to
//      the piece, then the range (warp scans of the stored masses), then
//      rereads that range (64 B of each row per lane; from the ring when the
//      piece is still there) and finds the entry by a warp scan in
//      vocabulary order.
// No global atomics, no partial results in global memory, no second launch.
// Numerics: a partial state is (R, s) with R a reference in log2 units (the
// maximum of x log2 e seen so far, rounded once) and s = sum 2^(x log2 e - R),
// each exponent argument formed by one fma (a single rounding, small for
// the entries near the maximum that carry the mass) and exponentiated by
// the MUFU ex2 instruction.  Normalisers, masses and running CDFs are
// compensated fp32 pairs (two-sum), never fp64 (GB300's fp64 rate is a
// small fraction of its fp32 rate).  The residual CDF is then within ~1e-6
// (absolute probability mass) of the exact one.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace simsd {
namespace {

constexpr int kMaxCluster = 16;                    // CTAs per sequence, at most (over 8: non-portable)
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;          // + the producer warp
constexpr int kGroupWarps = kConsumerWarps / 2;    // two groups take alternate pieces
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kStages = 6;
constexpr int kStageBytes = 32768;                 // at most one piece of one row slice
constexpr int kVecs = kStageBytes / 16 / kGroupThreads;   // 16-byte vectors per thread per piece
constexpr int kRanges = kConsumerWarps;           // vocabulary ranges per piece (residual sums)
constexpr int kRangeVecs = kStageBytes / 16 / kRanges;
constexpr int kMaxPieces = 32;                     // pieces per row slice
static_assert(kMaxPieces <= 32 && kRanges <= 32 && kMaxCluster <= 32,
              "the draw picks pieces, ranges and slices one per lane");
static_assert(kVecs % 2 == 0 && kRangeVecs % 32 == 0, "a range is whole vectors per lane");
static_assert(kRanges * kRangeVecs * 16 == kStageBytes, "the ranges tile a stage");
static_assert(kConsumers % kMaxCluster == 0 && 32 % kMaxCluster == 0,
              "whole groups of consumer threads per pair");
// the main pass's 8 accumulators see the same slots in both rolled halves:
// (kVecs / 2) vectors of N >= 4 entries are a multiple of 8 entries
static_assert((kVecs / 2) * 4 % 8 == 0, "accumulator slots repeat every half");
constexpr int kMaxPairs = 2 * kMaxB;               // (slot, row) pairs per sequence
constexpr int kMaxVocab = 1 << 21;                 // 8 slices of kMaxPieces pieces of 8192 fp32 entries
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

// 2^(x log2 e - R): the argument rounded once.
// (ls = log2(e) / temperature: the logits' scale into log2 units)
__device__ __forceinline__ float rel_exp(float x, float R, float ls) { return ex2(fmaf(x, ls, -R)); }

// p(v) = 2^(x log2 e - M) / S with the reciprocal normaliser, and the
// residual max(0, p - q): separately rounded (no fused multiply-subtract),
// so identical target and draft rows give p == q and an exactly empty
// residual, and the residual pass and the draw compute the same values.
__device__ __forceinline__ float prob(float x, float M, float inv_s, float ls) {
  return __fmul_rn(rel_exp(x, M, ls), inv_s);
}
__device__ __forceinline__ float residual(float p, float q) { return fmaxf(__fsub_rn(p, q), 0.f); }

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void consumers_sync() { named_sync(1, kConsumers); }

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

// ---------------------------------------------------------------- state
struct __align__(16) WalkInfo {
  int slot;              // rejected slot (0-based within the sequence), -1: none
  float Mt, Md;          // its references (log2 units)
  float inv_st, inv_sd;  // reciprocal normalisers
  float u;               // the residual draw's uniform
  int pad0, pad1;
};

struct __align__(16) AccShared {
  uint64_t full[kStages], empty[kStages];
  float2 part_w[kMaxPairs][kConsumerWarps];   // per warp: (R, s) of each (slot, row)
  float2 cpart[kMaxPairs];                    // this CTA's slice: (R, s)
  float2 norm[kMaxPairs];                     // CTA 0: merged (M, S) of each row
  float2 xv[kMaxB];                           // logits at the draft token, if in this slice
  float px[kMaxB], qx[kMaxB], u[kMaxB + 1];
  int tau[kMaxB], x[kMaxB], slot_of_step[kMaxB];
  float4 piece_w[kMaxPieces][kRanges];        // residual pass: per range (r pair, p pair)
  float4 piece_s[kMaxPieces];
  float4 tot;                                 // this slice's residual and target mass
  WalkInfo walk;                              // CTA 0's result, read by every CTA
  int flag;
};

struct AcceptParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int batch, vocab, B_max, total_B;
  int csize;   // CTAs per cluster (one cluster per sequence)
  int per;     // entries per CTA slice (a multiple of 16 bytes' worth)
  int piece;   // entries per ring stage
  int bulk;    // rows 16-byte aligned: bulk copies; else element copies
  float ls;    // log2(e) / temperature
};

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
__device__ __noinline__ int warp_pick(Ff m, Ff base, Ff U, Ff *start) {
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

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
accept_kernel(const __grid_constant__ AcceptParams a) {
  constexpr int N = Ld<T>::N;
  extern __shared__ __align__(128) uint8_t smem[];
  AccShared &S = *reinterpret_cast<AccShared *>(smem + kStages * kStageBytes);
  const uint32_t ring = smem_u32(smem);
  const int rank = blockIdx.x;               // the cluster spans x: rank = blockIdx.x
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const bool producer = warp == kConsumerWarps;
  const float ls = a.ls;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= kMaxB;  // the same in every CTA of the cluster
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  const int npieces = (len + a.piece - 1) / a.piece;
  auto piece_len = [&](int pc) { return min(a.piece, len - pc * a.piece); };
  auto row_ptr = [&](int k, int row) {
    return (const T *)(row ? a.draft : a.target) + (long)(c0 + k) * a.vocab + s0;
  };
  if (t == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&S.full[i]), 1);
      mbar_init(smem_u32(&S.empty[i]), kConsumerWarps);
    }
    S.flag = 0;
    fence_barrier_init();
  }
  __syncthreads();                           // the ring's barriers are ready
  if (valid && !producer) {                  // (the producer starts streaming meanwhile)
    if (t < B) {
      S.tau[t] = __ldg(a.tau + c0 + t);
      S.x[t] = __ldg(a.draft_tokens + c0 + t);
      S.xv[t] = make_float2(0.f, 0.f);
    }
    if (t <= B) S.u[t] = __ldg(a.uniforms + (long)b * (a.B_max + 1) + t);
    consumers_sync();                        // the sequence's labels, tokens, uniforms
  }

  int issued = 0;                            // producer: stages started so far
  int g = 0;                                 // stage counter (producer and consumers)
  if (valid) {
    // ---------------------------------------------------- 1. row slices
    const int J = 2 * B * npieces;
    if (producer) {
      for (int pair = 0, pc = 0; g < J; ++g) {
        const int s = g % kStages;
        if (g >= kStages && !mbar_wait_warp(smem_u32(&S.empty[s]), ((g / kStages) - 1) & 1)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); }
          break;
        }
        copy_piece<T>(smem + s * kStageBytes, ring + s * kStageBytes,
                      row_ptr(pair >> 1, pair & 1) + pc * a.piece, piece_len(pc),
                      smem_u32(&S.full[s]), a.bulk, lane);
        issued = g + 1;
        if (++pc == npieces) { pc = 0; ++pair; }
      }
    } else {
      // The two consumer groups (warps 0-7, 8-15) take alternate chunks of
      // stages -- whole (slot, row) pairs when a slice is at most two
      // pieces (one warp merge per pair), else single pieces -- so one
      // group's barrier waits, loads and merges overlap the other's
      // exponentials instead of all warps moving in step.
      const int grp = warp / kGroupWarps, gtid = t % kGroupThreads;
      const int v0 = (warp % kGroupWarps) * 32;
      const int chunk = npieces == 2 ? 2 : 1;
      if (lane == 0)                         // pairs this warp may see no piece of
        for (int q = 0; q < 2 * B; ++q) S.part_w[q][warp] = make_float2(-INFINITY, 0.f);
      float R = -INFINITY, sum = 0.f;
      int gg = grp * chunk, pair = 0, pc = gg;
      if (npieces > 0)
        while (pc >= npieces) { pc -= npieces; ++pair; }
      while (gg < J) {
        const int s = gg % kStages;
        const int n = piece_len(pc);
        if (!mbar_wait_warp(smem_u32(&S.full[s]), (gg / kStages) & 1)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); }
          break;
        }
        const uint4 *sv = reinterpret_cast<const uint4 *>(smem + s * kStageBytes);
        uint4 w[kVecs];
#pragma unroll
        for (int i = 0; i < kVecs; ++i) {
          const int idx = i * kGroupThreads + gtid;
          w[i] = idx * N < n ? sv[idx] : Ld<T>::neg_inf();
        }
        // the logit at the slot's draft token, if this piece holds it
        if (gtid == 0) {
          const int off = S.x[pair >> 1] - (s0 + pc * a.piece);
          if (off >= 0 && off < n) {
            const float v = pick<T>(sv[off / N], off % N);
            if (pair & 1) S.xv[pair >> 1].y = v; else S.xv[pair >> 1].x = v;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_n(smem_u32(&S.empty[s]), 2);
        const float mx = Ld<T>::vmax(w, kVecs);
        const float Rn = mx * ls;
        if (Rn > R) {
          sum = R == -INFINITY ? 0.f : sum * ex2(R - Rn);
          R = Rn;
        }
        if (R != -INFINITY) {
          // vectors past the piece's end hold -inf (adding their zeros
          // changes nothing): a warp skips those of a short piece.  Two
          // rolled halves of four vectors (the code stays small: it is
          // often fetched cold, after other kernels ran).
          const int nvec = (n + N - 1) / N;
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int i = 0; i < kVecs / 2; ++i) {
              if ((h * kVecs / 2 + i) * kGroupThreads + v0 >= nvec) break;
              float f[N];
              Ld<T>::unpack(w[i], f);
#pragma unroll
              for (int e = 0; e < N; ++e) acc[(i * N + e) & 7] += rel_exp(f[e], R, ls);
            }
#pragma unroll
            for (int i = 0; i < kVecs / 2; ++i) w[i] = w[i + kVecs / 2];
          }
          sum += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        }
        // this group's next stage
        const int gn = (gg + 1) % chunk != 0 ? gg + 1 : gg + chunk + 1;
        const int pair_now = pair;
        pc += gn - gg;
        while (pc >= npieces) { pc -= npieces; ++pair; }
        gg = gn;
        if (pair != pair_now || gg >= J) {
          // the group's part of the pair is done: warp merge to the warp's
          // largest reference (an order-preserving integer maximum), one
          // rescale per lane, one sum
          const uint32_t ru = __float_as_uint(R);
          const uint32_t km = __reduce_max_sync(0xffffffffu, (ru & 0x80000000u) ? ~ru : (ru | 0x80000000u));
          const float Rm = __uint_as_float((km & 0x80000000u) ? (km & 0x7fffffffu) : ~km);
          float sc = Rm == -INFINITY ? 0.f : sum * ex2(R - Rm);
#pragma unroll
          for (int m = 16; m > 0; m >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, m);
          if (lane == 0) S.part_w[pair_now][warp] = make_float2(Rm, sc);
          R = -INFINITY;
          sum = 0.f;
        }
      }
      consumers_sync();
      if (t < 2 * B) {                       // this CTA's slice of pair t
        float2 c = make_float2(-INFINITY, 0.f);
        if (npieces > 0 && !*(volatile int *)&S.flag) {
          float M = -INFINITY;
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, S.part_w[t][w].x);
          Ff sm = ff_of(0.f);
          if (M != -INFINITY)
#pragma unroll 1
            for (int w = 0; w < kConsumerWarps; ++w) {
              const float2 v = S.part_w[t][w];
              if (v.y > 0.f) sm = ff_add(sm, ff_of(v.y * ex2(v.x - M)));
            }
          c = make_float2(M, sm.hi + sm.lo);
        }
        S.cpart[t] = c;
      }
    }
    cluster_sync();                          // B1: every slice's partials are in place

    // ---------------------------------------------------- 2. the walk
    // every CTA merges the slices' partials and walks the steps itself (the
    // same inputs in the same order give the same decisions everywhere), so
    // no barrier is needed before the residual pass; CTA 0 writes outputs
    if (!producer) {
      // thread (pair q, slice r) reads one slice's partial; groups of gs
      // lanes (8, or 16 for clusters over 8) merge them (pair q: slot q / 2,
      // row q % 2)
      const int lg = a.csize > 8 ? 4 : 3, gs = 1 << lg;
      for (int q0 = 0; q0 < 2 * B; q0 += kConsumers >> lg) {
      if (warp * 32 < (2 * B - q0) << lg) {  // whole warps: the shuffles need every lane
        const int q = q0 + (t >> lg), r = t & (gs - 1);
        const bool mine = q < 2 * B;
        const int k = q >> 1, row = q & 1, x = mine ? S.x[k] : -1;
        const bool xin = x >= 0 && x < a.vocab;
        const float2 xl = r == 0 && xin ? ld_dsmem2(dsmem(&S.xv[k], x / a.per)) : make_float2(0.f, 0.f);
        const float2 v = mine && r < a.csize ? ld_dsmem2(dsmem(&S.cpart[q], r)) : make_float2(-INFINITY, 0.f);
        float M = v.x;
#pragma unroll 1
        for (int m = gs / 2; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
        Ff sm = ff_of(M != -INFINITY && v.y > 0.f ? v.y * ex2(v.x - M) : 0.f);
#pragma unroll 1
        for (int m = gs / 2; m > 0; m >>= 1) sm = ff_add(sm, ff_shfl_xor(sm, m));
        if (mine && r == 0) {
          S.norm[q] = make_float2(M, sm.hi + sm.lo);
          // p(x) (row 0) or q(x) (row 1); a token no slice holds rejects
          const float pr = xin ? rel_exp(row ? xl.y : xl.x, M, ls) / (sm.hi + sm.lo) : 0.f;
          if (row) S.qx[k] = pr; else S.px[k] = pr;
          if (!xin && row == 0 && rank == 0) raise_status(a.status, kStatusBadInput);
        }
      }
      }
      consumers_sync();
      if (t == 0) {
        for (int k = 0; k < kMaxB; ++k) S.slot_of_step[k] = 0;
        for (int k = 0; k < B; ++k) {
          const int tk = S.tau[k];           // a label outside 1..B is ignored
          if (tk >= 1 && tk <= B) S.slot_of_step[tk - 1] = k;
        }
        int n = B, rej = -1;
        for (int st = 1; st <= B; ++st) {
          const int k = S.slot_of_step[st - 1];
          if (!(S.u[st - 1] * S.qx[k] < S.px[k])) { n = st - 1; rej = k; break; }
        }
        if (rank == 0) {
          a.n_accept[b] = n;
          a.pos[b] = rej;
          if (rej < 0) a.token[b] = -1;
        }
        WalkInfo w{-1, 0.f, 0.f, 1.f, 1.f, 0.f, 0, 0};
        if (rej >= 0) {
          w.slot = rej;
          w.Mt = S.norm[2 * rej].x;
          w.Md = S.norm[2 * rej + 1].x;
          w.inv_st = 1.f / S.norm[2 * rej].y;
          w.inv_sd = 1.f / S.norm[2 * rej + 1].y;
          w.u = S.u[B];
        }
        S.walk = w;
      }
    }
    __syncthreads();                         // the walk's result, for the producer too
    const WalkInfo w = S.walk;

    if (w.slot >= 0) {
      // -------------------------------------------------- 3. residual masses
      const int J2 = J + 2 * npieces;
      if (producer) {
        for (; g < J2 && !*(volatile int *)&S.flag; ++g) {
          const int s = g % kStages, pc = (g - J) >> 1, row = (g - J) & 1;
          if (g >= kStages && !mbar_wait_warp(smem_u32(&S.empty[s]), ((g / kStages) - 1) & 1)) {
            if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); }
            break;
          }
          copy_piece<T>(smem + s * kStageBytes, ring + s * kStageBytes,
                        row_ptr(w.slot, row) + pc * a.piece, piece_len(pc),
                        smem_u32(&S.full[s]), a.bulk, lane);
          issued = g + 1;
        }
      } else {
        // every warp takes part in every piece: warp w reads range w, the
        // contiguous vectors [w * kRangeVecs, (w + 1) * kRangeVecs) of the
        // piece (lane-interleaved), whose masses the draw narrows down to
        for (int pc = 0; pc < npieces && !*(volatile int *)&S.flag; ++pc) {
          const int gt = J + 2 * pc, gd = gt + 1;
          const int st = gt % kStages, sd = gd % kStages;
          const int n = piece_len(pc);
          if (!mbar_wait_warp(smem_u32(&S.full[st]), (gt / kStages) & 1) ||
              !mbar_wait_warp(smem_u32(&S.full[sd]), (gd / kStages) & 1)) {
            if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); }
            break;
          }
          const uint4 *tv = reinterpret_cast<const uint4 *>(smem + st * kStageBytes);
          const uint4 *dv = reinterpret_cast<const uint4 *>(smem + sd * kStageBytes);
          const int nvec = (n + N - 1) / N;
          float rs[4] = {0.f, 0.f, 0.f, 0.f}, ps[4] = {0.f, 0.f, 0.f, 0.f};
          if (warp * kRangeVecs < nvec) {
#pragma unroll
            for (int i = 0; i < kRangeVecs / 32; ++i) {
              const int idx = warp * kRangeVecs + i * 32 + lane;
              const bool in = idx < nvec;
              float ft[N], fd[N];
              Ld<T>::unpack(in ? tv[idx] : Ld<T>::neg_inf(), ft);
              Ld<T>::unpack(in ? dv[idx] : Ld<T>::neg_inf(), fd);
#pragma unroll
              for (int e = 0; e < N; ++e) {
                const float p = prob(ft[e], w.Mt, w.inv_st, ls);
                const float q = prob(fd[e], w.Md, w.inv_sd, ls);
                rs[e & 3] += residual(p, q);
                ps[e & 3] += p;
              }
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&S.empty[st]));
            mbar_arrive(smem_u32(&S.empty[sd]));
          }
          Ff fr = ff_add(ff_of(rs[0] + rs[1]), ff_of(rs[2] + rs[3]));
          Ff fp = ff_add(ff_of(ps[0] + ps[1]), ff_of(ps[2] + ps[3]));
#pragma unroll 1
          for (int m = 16; m > 0; m >>= 1) {
            fr = ff_add(fr, ff_shfl_xor(fr, m));
            fp = ff_add(fp, ff_shfl_xor(fp, m));
          }
          if (lane == 0) S.piece_w[pc][warp] = make_float4(fr.hi, fr.lo, fp.hi, fp.lo);
        }
        consumers_sync();
        if (warp == 0) {                     // lane i: piece i (npieces <= 32)
          const bool failed = *(volatile int *)&S.flag != 0;
          Ff r = ff_of(0.f), p = ff_of(0.f);
          if (lane < npieces && !failed)
#pragma unroll 1
            for (int ww = 0; ww < kRanges; ++ww) {
              const float4 v = S.piece_w[lane][ww];
              r = ff_add(r, Ff{v.x, v.y});
              p = ff_add(p, Ff{v.z, v.w});
            }
          if (lane < npieces) S.piece_s[lane] = make_float4(r.hi, r.lo, p.hi, p.lo);
#pragma unroll 1
          for (int m = 16; m > 0; m >>= 1) {
            r = ff_add(r, ff_shfl_xor(r, m));
            p = ff_add(p, ff_shfl_xor(p, m));
          }
          if (lane == 0) S.tot = make_float4(r.hi, r.lo, p.hi, p.lo);
        }
      }
      cluster_sync();                        // B3: every slice's masses are in place

      // -------------------------------------------------- 4. the draw
      // U = u * S (u * Sp when the residual is empty).  Every CTA makes the
      // same choice from the same C slice totals (in rank order): the first
      // slice whose running mass exceeds U, else the last with mass.  Warp 0
      // of that CTA narrows down the same way to a piece, then to one warp's
      // vocabulary range of the piece, then to the entry.
      if (warp == 0) {
        const float4 v = lane < a.csize ? ld_dsmem4(dsmem(&S.tot, lane)) : make_float4(0.f, 0.f, 0.f, 0.f);
        Ff Sr{v.x, v.y}, Sp{v.z, v.w};
#pragma unroll 1
        for (int m = 16; m > 0; m >>= 1) {
          Sr = ff_add(Sr, ff_shfl_xor(Sr, m));
          Sp = ff_add(Sp, ff_shfl_xor(Sp, m));
        }
        cluster_arrive();                    // B4: this CTA's remote reads are done (used above)
        const bool use_p = !(Sr.hi > 0.f);
        const Ff tot = use_p ? Sp : Sr;
        const float uh = w.u * tot.hi;
        const Ff U = ff_add(Ff{uh, fmaf(w.u, tot.hi, -uh)}, ff_of(w.u * tot.lo));
        auto mass_of = [&](float4 q) { return use_p ? Ff{q.z, q.w} : Ff{q.x, q.y}; };
        Ff base;
        const int ch = warp_pick(mass_of(v), ff_of(0.f), U, &base);
        if (ch == rank && !*(volatile int *)&S.flag) {
          const float4 vp = lane < npieces ? S.piece_s[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
          const int sel = warp_pick(mass_of(vp), base, U, &base);
          const float4 vw = lane < kRanges ? S.piece_w[sel][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
          const int ws = warp_pick(mass_of(vw), base, U, &base);
          // The range's 128 vectors as 4 columns of 32 (lane l: vectors
          // l, l + 32, l + 64, l + 96), read from the ring if the piece is
          // among the residual pass's last kStages stages, else from L2.
          // Column by column in vocabulary order: the lanes' masses, their
          // inclusive scan (fp32, relative to the range start: small, so the
          // rounding stays far below the residual tie zone); the lane whose
          // span holds U claims its first entry with mass whose running
          // total exceeds U; else the last entry with mass.
          const int n = npieces > 0 ? piece_len(sel) : 0;
          const int gsel = J + 2 * sel;
          const bool in_ring = gsel >= J + 2 * npieces - kStages;
          const T *tr = in_ring ? reinterpret_cast<const T *>(smem + (gsel % kStages) * kStageBytes)
                                : row_ptr(w.slot, 0) + sel * a.piece;
          const T *dr = in_ring ? reinterpret_cast<const T *>(smem + ((gsel + 1) % kStages) * kStageBytes)
                                : row_ptr(w.slot, 1) + sel * a.piece;
          constexpr int kCols = kRangeVecs / 32;
          const Ff D0 = ff_add(U, ff_neg(base));
          const float d = D0.hi + D0.lo;     // U - the range's start
          float col_base = 0.f;
          int first = 0x7fffffff, last_pos = -1;
#pragma unroll 1
          for (int i = 0; i < kCols && first == 0x7fffffff; ++i) {
            const int e0 = (ws * kRangeVecs + i * 32 + lane) * N;  // the vector's first entry
            const int vbase = s0 + sel * a.piece + e0;
            float ft[N], fd[N], m[N];
            Ld<T>::unpack(Ld<T>::load(tr + e0, n - e0, a.bulk != 0), ft);
            Ld<T>::unpack(Ld<T>::load(dr + e0, n - e0, a.bulk != 0), fd);
            float lane_mass = 0.f;
#pragma unroll
            for (int e = 0; e < N; ++e) {
              const float p = prob(ft[e], w.Mt, w.inv_st, ls);
              const float q = prob(fd[e], w.Md, w.inv_sd, ls);
              m[e] = use_p ? p : residual(p, q);
              lane_mass += m[e];
              if (m[e] > 0.f) last_pos = vbase + e;
            }
            float inc = lane_mass;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, inc, dd);
              if (lane >= dd) inc += y;
            }
            const float prev = __shfl_up_sync(0xffffffffu, inc, 1);
            const float start = col_base + (lane ? prev : 0.f);
            if (d < col_base + inc) {
              float run = 0.f;
#pragma unroll
              for (int e = 0; e < N; ++e) {
                run += m[e];
                if (first == 0x7fffffff && m[e] > 0.f && start + run > d) first = vbase + e;
              }
            }
            first = __reduce_min_sync(0xffffffffu, first);
            col_base += __shfl_sync(0xffffffffu, inc, 31);
          }
          last_pos = __reduce_max_sync(0xffffffffu, last_pos);
          if (lane == 0) a.token[b] = first != 0x7fffffff ? first : last_pos;
        }
      } else {
        cluster_arrive();                    // B4
      }
    } else {
      cluster_arrive();                      // B4
    }
  } else {
    if (rank == 0 && t == 0) {               // malformed sequence: no walk
      a.n_accept[b] = 0;
      a.token[b] = -1;
      a.pos[b] = -1;
      raise_status(a.status, kStatusBadInput);
    }
    cluster_arrive();                        // B4
  }
  // copies still in flight after a timeout land before the CTA can exit
  if (producer && *(volatile int *)&S.flag)
    for (int j = max(0, issued - kStages); j < issued; ++j)
      (void)mbar_wait_warp(smem_u32(&S.full[j % kStages]), (j / kStages) & 1);
  cluster_wait();                            // B4: no CTA leaves while others read it
}

constexpr size_t kSmemBytes = kStages * kStageBytes + sizeof(AccShared);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

void mark(void *const *events, int i, cudaStream_t stream) {
  if (events != nullptr) record_event(events[i], stream);
}

cudaLaunchConfig_t launch_config(int csize, int batch, cudaStream_t stream,
                                 cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Per device and cluster size 1..kMaxCluster: clusters of this kernel
// resident at once (queried once; the answer depends on the device only;
// -1 for a size the device cannot place).
template <typename T>
cudaError_t max_active_clusters(int dev, int csize, int *out) {
  static std::mutex mu;
  static int cache[64][kMaxCluster + 1] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][0] == 0) {
    cudaError_t e = cudaFuncSetAttribute(accept_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    // sizes over 8 are optional: without the attribute they are skipped
    if (cudaFuncSetAttribute(accept_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      (void)cudaGetLastError();
    cache[dev][0] = 1;
  }
  if (cache[dev][csize] == 0) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(csize, csize, nullptr, attr);
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, accept_kernel<T>, &cfg);
    if (e != cudaSuccess) {
      if (csize <= 8) return e;
      (void)cudaGetLastError();              // a non-portable size this device refuses
      n = 0;
    }
    cache[dev][csize] = n > 0 ? n : -1;
  }
  *out = cache[dev][csize];
  return cudaSuccess;
}

template <typename T>
cudaError_t launch(AcceptParams a, cudaStream_t stream) {
  const int dev = current_device();
  // Cluster size by a makespan estimate: clusters run in waves of the
  // resident count; a CTA's time is its share of the sequence's exponentials
  // at 16 per clock per SM (a round figure: the MUFU alone sustains ~24, the
  // whole streaming loop fewer) plus the fixed cost of the walk, residual
  // and draw phases.  Small batches get large clusters (every SM busy),
  // large batches small ones (fewer waves).  Never so small that a slice
  // needs more pieces than the kernel tracks.
  const int piece = kStageBytes / (int)sizeof(T), vec = 16 / (int)sizeof(T);
  const int64_t max_slice = (int64_t)kMaxPieces * piece;
  const double per_seq = (2.0 * a.total_B / a.batch + 2.0) * a.vocab;   // exponentials
  constexpr double kPhaseCycles = 20000.0;
  int csize = kMaxCluster;
  double best = 1e300;
  for (int c = kMaxCluster; c >= 1; --c) {
    if (((int64_t)a.vocab + c - 1) / c > max_slice) break;
    int n = 0;
    cudaError_t e = max_active_clusters<T>(dev, c, &n);
    if (e != cudaSuccess) return e;
    if (n <= 0) continue;
    const double waves = (double)((a.batch + n - 1) / n);
    const double cost = waves * (per_seq / c / 16.0 + kPhaseCycles);
    if (cost < best * (1.0 - 1e-9)) { best = cost; csize = c; }
  }
  a.csize = csize;
  a.per = ((a.vocab + csize - 1) / csize + vec - 1) / vec * vec;
  // pieces of equal size (whole vectors, at most one stage) per slice
  const int np = (a.per + piece - 1) / piece;
  a.piece = ((a.per + np - 1) / np + vec - 1) / vec * vec;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = launch_config(csize, a.batch, stream, attr);
  return cudaLaunchKernelEx(&cfg, accept_kernel<T>, a);
}

// ---------------------------------------------------------------- greedy
// The greedy rule: per slot the target row's argmax (the largest value, the
// smallest index among equal values), then the walk.  One cluster of C CTAs
// per sequence, CTA r scanning vocabulary slice r of every target row with
// 16-byte loads; CTA 0 merges the slices' candidates through distributed
// shared memory and walks the steps.  Neither the draft logits nor the
// uniforms are read.
constexpr int kGreedyThreads = 512;
constexpr int kGreedyUnroll = 8;
constexpr int kGreedyCluster = 8;

struct GreedyParams {
  const void *target;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int vocab, csize, per, bulk;
};

// candidate (v, i) beats (w, j): a larger value, or an equal one at a
// smaller index (-inf entries still win over "none", index 2^31 - 1)
__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

template <typename T>
__global__ void __launch_bounds__(kGreedyThreads)
accept_greedy_kernel(const __grid_constant__ GreedyParams a) {
  constexpr int N = Ld<T>::N;
  __shared__ float2 cand[kMaxB];                    // per slot: (value, index bits)
  __shared__ float2 wbest[kGreedyThreads / 32];
  const int rank = blockIdx.x, b = blockIdx.y;    // the cluster spans x
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= kMaxB;
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  if (valid) {
    for (int k = 0; k < B; ++k) {
      const T *row = (const T *)a.target + (long)(c0 + k) * a.vocab + s0;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      if (a.bulk) {                                 // len is whole vectors here
        // kGreedyUnroll independent 16-byte loads in flight per thread
        const uint4 *rv = reinterpret_cast<const uint4 *>(row);
        const int nv = len / N;
        for (int i0 = t; i0 < nv; i0 += kGreedyUnroll * kGreedyThreads) {
          uint4 w[kGreedyUnroll];
#pragma unroll
          for (int u = 0; u < kGreedyUnroll; ++u) {
            const int i = i0 + u * kGreedyThreads;
            w[u] = i < nv ? __ldg(rv + i) : Ld<T>::neg_inf();
          }
#pragma unroll
          for (int u = 0; u < kGreedyUnroll; ++u) {
            const int i = i0 + u * kGreedyThreads;
            float f[N];
            Ld<T>::unpack(w[u], f);
#pragma unroll
            for (int e = 0; e < N; ++e)
              if (i < nv && beats(f[e], s0 + i * N + e, bv, bi)) { bv = f[e]; bi = s0 + i * N + e; }
          }
        }
      } else {
        for (int e = t; e < len; e += kGreedyThreads) {
          const float v = Ld<T>::value(row[e]);
          if (beats(v, s0 + e, bv, bi)) { bv = v; bi = s0 + e; }
        }
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, m);
        if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) wbest[warp] = make_float2(bv, __int_as_float(bi));
      __syncthreads();
      if (t == 0) {
        float v = -INFINITY;
        int i = 0x7fffffff;
        for (int w = 0; w < kGreedyThreads / 32; ++w) {
          const float2 c = wbest[w];
          if (beats(c.x, __float_as_int(c.y), v, i)) { v = c.x; i = __float_as_int(c.y); }
        }
        cand[k] = make_float2(v, __int_as_float(i));
      }
      __syncthreads();
    }
  }
  cluster_sync();                                   // every slice's candidates are in place
  if (rank == 0 && t == 0) {
    if (!valid) {                                   // malformed sequence: no walk
      a.n_accept[b] = 0;
      a.token[b] = -1;
      a.pos[b] = -1;
      raise_status(a.status, kStatusBadInput);
    } else {
      int slot_of_step[kMaxB];
      for (int k = 0; k < B; ++k) slot_of_step[k] = 0;
      for (int k = 0; k < B; ++k) {
        const int tk = __ldg(a.tau + c0 + k);     // a label outside 1..B is ignored
        if (tk >= 1 && tk <= B) slot_of_step[tk - 1] = k;
      }
      int n = B, tok = -1, ps = -1;
      for (int st = 1; st <= B; ++st) {
        const int k = slot_of_step[st - 1];
        float v = -INFINITY;
        int am = 0x7fffffff;
        for (int r = 0; r < a.csize; ++r) {
          const float2 c = ld_dsmem2(dsmem(&cand[k], r));
          if (beats(c.x, __float_as_int(c.y), v, am)) { v = c.x; am = __float_as_int(c.y); }
        }
        const int x = __ldg(a.draft_tokens + c0 + k);
        if (x < 0 || x >= a.vocab) raise_status(a.status, kStatusBadInput);
        if (x != am) { n = st - 1; tok = am; ps = k; break; }
      }
      a.n_accept[b] = n;
      a.token[b] = tok;
      a.pos[b] = ps;
    }
  }
  cluster_sync();                                   // no CTA leaves while CTA 0 reads it
}

template <typename T>
cudaError_t launch_greedy(GreedyParams a, int batch, cudaStream_t stream) {
  // about one CTA per SM across the batch, at most kGreedyCluster per sequence
  const int vec = 16 / (int)sizeof(T);
  a.csize = max(1, min(kGreedyCluster, device_sm_count() / max(1, batch)));
  a.per = ((a.vocab + a.csize - 1) / a.csize + vec - 1) / vec * vec;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.csize, batch);
  cfg.blockDim = dim3(kGreedyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_greedy_kernel<T>, a);
}

// ---------------------------------------------------------------- match
// Sample matching: step t draws the target's own token y_t from p by inverse
// CDF with u[t-1] and accepts iff y_t is the draft token; the first
// rejection emits y_t.  In mass units of S = sum_v 2^(l_v ls - M): the step
// accepts iff Pre(x) <= u S < Pre(x) + 2^(l_x ls - M), Pre(x) the mass of
// the entries below x.  One cluster of C CTAs per sequence; CTA r streams
// slice r of every target row once for (reference, mass, mass below x, l_x);
// every CTA merges the C slices' partials through distributed shared memory
// and walks the steps identically; at a rejection the CTA whose slice holds
// u S finds y_t by a block scan of its slice in vocabulary order.
constexpr int kMatchThreads = 512;
constexpr int kMatchWarps = kMatchThreads / 32;
constexpr int kMatchUnroll = 8;

struct MatchParams {
  const void *target;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int vocab, B_max, csize, per, bulk;
  float ls;
};

struct __align__(16) MatchSlot {
  float R, xl;       // the slice's reference (log2 units) and l_x if x lies in it
  Ff s, pre;         // sum of 2^(l ls - R) over the slice, and over its entries below x
};

// (R, s, pre) += (R2, s2, pre2): both sums to the larger reference
__device__ __forceinline__ void match_merge(float &R, Ff &s, Ff &pre, float R2, Ff s2, Ff pre2) {
  const float M = fmaxf(R, R2);
  if (M == -INFINITY) return;
  const float a = ex2(R - M), b = ex2(R2 - M);
  s = ff_add(Ff{s.hi * a, s.lo * a}, Ff{s2.hi * b, s2.lo * b});
  pre = ff_add(Ff{pre.hi * a, pre.lo * a}, Ff{pre2.hi * b, pre2.lo * b});
  R = M;
}

template <typename T>
__global__ void __launch_bounds__(kMatchThreads)
accept_match_kernel(const __grid_constant__ MatchParams a) {
  constexpr int N = Ld<T>::N;
  __shared__ MatchSlot slot[kMaxB];
  __shared__ MatchSlot wpart[kMatchWarps];
  __shared__ Ff wsum[kMatchWarps];
  __shared__ int s_ch, s_best, s_last, s_k;
  __shared__ Ff s_U, s_base;
  __shared__ float s_M;
  const int rank = blockIdx.x, b = blockIdx.y;    // the cluster spans x
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const float ls = a.ls;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= kMaxB;
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  auto value_at = [&](const T *row, int e) { return Ld<T>::value(row[e]); };
  if (valid) {
    for (int k = 0; k < B; ++k) {
      const T *row = (const T *)a.target + (long)(c0 + k) * a.vocab + s0;
      const int x = __ldg(a.draft_tokens + c0 + k);
      const int xo = x - s0;                        // x's offset in this slice
      float R = -INFINITY, sm = 0.f, pr = 0.f, xl = -INFINITY;
      // one group of kMatchUnroll entries (vectors in the bulk case) per round
      const int unit = a.bulk ? N : 1;
      const int nu = a.bulk ? len / N : len;
      for (int i0 = t; i0 < nu; i0 += kMatchUnroll * kMatchThreads) {
        float f[kMatchUnroll][N];
#pragma unroll
        for (int u = 0; u < kMatchUnroll; ++u) {
          const int i = i0 + u * kMatchThreads;
          if (a.bulk) {
            Ld<T>::unpack(i < nu ? __ldg(reinterpret_cast<const uint4 *>(row) + i) : Ld<T>::neg_inf(), f[u]);
          } else {
#pragma unroll
            for (int e = 0; e < N; ++e) f[u][e] = (e == 0 && i < nu) ? value_at(row, i) : -INFINITY;
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kMatchUnroll; ++u)
#pragma unroll
          for (int e = 0; e < N; ++e) mx = fmaxf(mx, f[u][e]);
        const float Rn = mx * ls;
        if (Rn > R) {
          const float c = R == -INFINITY ? 0.f : ex2(R - Rn);
          sm *= c;
          pr *= c;
          R = Rn;
        }
        if (R == -INFINITY) continue;
#pragma unroll
        for (int u = 0; u < kMatchUnroll; ++u) {
          const int base_e = (i0 + u * kMatchThreads) * unit;
#pragma unroll
          for (int e = 0; e < N; ++e) {
            const float m = rel_exp(f[u][e], R, ls);
            sm += m;
            if (base_e + e < xo) pr += m;
            if (base_e + e == xo) xl = f[u][e];
          }
        }
      }
      // warp, then block: to the largest reference, sums as pairs
      Ff s2 = ff_of(sm), p2 = ff_of(pr);
      float Rw = R;
#pragma unroll 1
      for (int m = 16; m > 0; m >>= 1) {
        const float R2 = __shfl_xor_sync(0xffffffffu, Rw, m);
        const Ff so = ff_shfl_xor(s2, m), po = ff_shfl_xor(p2, m);
        match_merge(Rw, s2, p2, R2, so, po);
        xl = fmaxf(xl, __shfl_xor_sync(0xffffffffu, xl, m));
      }
      if (lane == 0) wpart[warp] = MatchSlot{Rw, xl, s2, p2};
      __syncthreads();
      if (t == 0) {
        MatchSlot c = wpart[0];
        for (int w = 1; w < kMatchWarps; ++w) {
          const MatchSlot o = wpart[w];
          match_merge(c.R, c.s, c.pre, o.R, o.s, o.pre);
          c.xl = fmaxf(c.xl, o.xl);
        }
        slot[k] = c;
      }
      __syncthreads();
    }
  }
  cluster_sync();                                   // B1: every slice's partials are in place
  if (t == 0) {
    s_ch = -1;
    s_k = -1;
    if (valid) {
      int slot_of_step[kMaxB];
      for (int k = 0; k < B; ++k) slot_of_step[k] = 0;
      for (int k = 0; k < B; ++k) {
        const int tk = __ldg(a.tau + c0 + k);     // a label outside 1..B is ignored
        if (tk >= 1 && tk <= B) slot_of_step[tk - 1] = k;
      }
      int n = B, rej = -1;
      for (int st = 1; st <= B; ++st) {
        const int k = slot_of_step[st - 1];
        // the slices' partials in rank order, merged to the largest reference
        float M = -INFINITY, xl = -INFINITY;
        for (int r = 0; r < a.csize; ++r) {
          const float4 h = ld_dsmem4(dsmem(&slot[k], r));
          M = fmaxf(M, h.x);
          xl = fmaxf(xl, h.y);
        }
        Ff S = ff_of(0.f), Pre = ff_of(0.f);
        if (M != -INFINITY)
          for (int r = 0; r < a.csize; ++r) {
            const float4 h = ld_dsmem4(dsmem(&slot[k], r));
            const float4 q = ld_dsmem4(dsmem(reinterpret_cast<const float4 *>(&slot[k]) + 1, r));
            if (h.x == -INFINITY) continue;
            const float w = ex2(h.x - M);
            S = ff_add(S, Ff{h.z * w, h.w * w});
            Pre = ff_add(Pre, Ff{q.x * w, q.y * w});
          }
        const int x = __ldg(a.draft_tokens + c0 + k);
        if (x < 0 || x >= a.vocab) raise_status(a.status, kStatusBadInput);
        const float u = __ldg(a.uniforms + (long)b * (a.B_max + 1) + st - 1);
        const float uh = u * S.hi;
        const Ff U = ff_add(Ff{uh, fmaf(u, S.hi, -uh)}, ff_of(u * S.lo));
        const float px = (x >= 0 && x < a.vocab) ? ex2(fmaf(xl, ls, -M)) : 0.f;   // mass of x
        const bool acc = px > 0.f && !ff_gt(Pre, U) && ff_gt(ff_add(Pre, ff_of(px)), U);
        if (acc) continue;
        n = st - 1;
        rej = k;
        // the slice holding U: the first whose running total exceeds it,
        // else the last with mass
        Ff run = ff_of(0.f), base = ff_of(0.f);
        int ch = -1, lastnz = 0;
        Ff lastbase = ff_of(0.f);
        for (int r = 0; r < a.csize; ++r) {
          const float4 h = ld_dsmem4(dsmem(&slot[k], r));
          const float w = h.x == -INFINITY ? 0.f : ex2(h.x - M);
          const Ff m = Ff{h.z * w, h.w * w};
          const Ff nx = ff_add(run, m);
          if (m.hi > 0.f) {
            lastnz = r;
            lastbase = run;
            if (ff_gt(nx, U)) { ch = r; base = run; break; }
          }
          run = nx;
        }
        if (ch < 0) { ch = lastnz; base = lastbase; }
        s_ch = ch;
        s_k = k;
        s_U = U;
        s_base = base;
        s_best = 0x7fffffff;
        s_last = -1;
        s_M = M;
        break;
      }
      if (rank == 0) {
        a.n_accept[b] = n;
        a.pos[b] = rej;
        if (rej < 0) a.token[b] = -1;
      }
    } else if (rank == 0) {                         // malformed sequence: no walk
      a.n_accept[b] = 0;
      a.token[b] = -1;
      a.pos[b] = -1;
      raise_status(a.status, kStatusBadInput);
    }
  }
  __syncthreads();
  if (s_ch == rank && s_k >= 0) {
    // block scan of this slice of row k in vocabulary order: thread t holds
    // the contiguous chunk [t * chunk, (t + 1) * chunk)
    const int k = s_k;
    const float M = s_M;
    const T *row = (const T *)a.target + (long)(c0 + k) * a.vocab + s0;
    const int chunk = (len + kMatchThreads - 1) / kMatchThreads;
    const int e0 = min(len, t * chunk), e1 = min(len, e0 + chunk);
    float part = 0.f;
    int last = -1;
    for (int e = e0; e < e1; ++e) {
      const float m = rel_exp(value_at(row, e), M, ls);
      part += m;
      if (m > 0.f) last = s0 + e;
    }
    // exclusive prefix of the chunk masses (pairs) over the block
    Ff inc = ff_of(part);
#pragma unroll 1
    for (int d = 1; d < 32; d <<= 1) {
      const Ff y = ff_shfl_up(inc, d);
      if (lane >= d) inc = ff_add(y, inc);
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    Ff start = s_base;
    for (int w = 0; w < warp; ++w) start = ff_add(start, wsum[w]);
    start = ff_add(start, ff_add(inc, ff_of(-part)));
    const Ff D = ff_add(s_U, ff_neg(start));
    const float dd = D.hi + D.lo;                   // U - this chunk's start
    int first = 0x7fffffff;
    if (dd < part) {
      float run = 0.f;
      for (int e = e0; e < e1; ++e) {
        const float m = rel_exp(value_at(row, e), M, ls);
        run += m;
        if (m > 0.f && run > dd) { first = s0 + e; break; }
      }
    }
    if (first != 0x7fffffff) atomicMin(&s_best, first);
    if (last >= 0) atomicMax(&s_last, last);
    __syncthreads();
    if (t == 0) a.token[b] = s_best != 0x7fffffff ? s_best : s_last;
  }
  cluster_sync();                                   // B2: no CTA leaves while others read it
}

template <typename T>
cudaError_t launch_match(MatchParams a, int batch, cudaStream_t stream) {
  const int vec = 16 / (int)sizeof(T);
  a.csize = max(1, min(kGreedyCluster, device_sm_count() / max(1, batch)));
  a.per = ((a.vocab + a.csize - 1) / a.csize + vec - 1) / vec * vec;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.csize, batch);
  cfg.blockDim = dim3(kMatchThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_match_kernel<T>, a);
}

simsd_status accept_check(const simsd_accept_desc *d) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (d->dtype != SIMSD_F32 && d->dtype != SIMSD_BF16) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->batch > 65535 || d->vocab < 1 || d->vocab > kMaxVocab ||
      d->B_max < 1 || d->B_max > kMaxB || d->total_B < d->batch ||
      (int64_t)d->total_B > (int64_t)d->batch * d->B_max)
    return SIMSD_ERR_SHAPE;
  if ((d->rule != SIMSD_ACCEPT_SAMPLE && d->rule != SIMSD_ACCEPT_GREEDY &&
       d->rule != SIMSD_ACCEPT_MATCH) ||
      !(d->temperature >= 0.f && d->temperature <= 3.0e38f))   // negative, NaN or inf
    return SIMSD_ERR_SHAPE;
  return SIMSD_OK;
}

// The pointers each rule reads (greedy: no draft logits, no uniforms;
// sample matching: no draft logits).
bool accept_pointers_ok(const simsd_accept_desc *d) {
  const bool draft = d->rule == SIMSD_ACCEPT_SAMPLE;
  const bool uni = d->rule != SIMSD_ACCEPT_GREEDY;
  return d->target_logits && d->draft_tokens && d->tau && d->cu_B && d->n_accept &&
         d->token && d->pos && (!draft || d->draft_logits) && (!uni || d->uniforms);
}

// The workspace holds the status word only (everything else stays on chip).
constexpr size_t kAcceptWorkspace = kAlign;

// Scratch of simsd_accept_noalloc: one static array per device, alive until
// the process exits.  Host code may not take its address directly (the
// name is a host-side stand-in there); static_scratch() looks the device
// address up once per device.
constexpr int kMaxDevices = 64;
static_assert(SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES % kAlign == 0, "scratch size");
static_assert(SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES >= kAcceptWorkspace, "scratch size");
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

// Launches K4 (the status word is not cleared here: its bits stay set until
// simsd_read_status reads them).
simsd_status run_accept(const simsd_accept_desc *d, char *ws, cudaStream_t stream,
                        void *const *events) {
  const int es = d->dtype == SIMSD_BF16 ? 2 : 4;
  if (d->rule == SIMSD_ACCEPT_GREEDY) {
    GreedyParams g;
    g.target = d->target_logits;
    g.draft_tokens = d->draft_tokens;
    g.tau = d->tau;
    g.cu_B = d->cu_B;
    g.n_accept = d->n_accept;
    g.token = d->token;
    g.pos = d->pos;
    g.status = (uint32_t *)ws;
    g.vocab = d->vocab;
    g.csize = 1;
    g.per = 0;
    g.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits);
    mark(events, 0, stream);
    const cudaError_t e = d->dtype == SIMSD_BF16 ? launch_greedy<__nv_bfloat16>(g, d->batch, stream)
                                                 : launch_greedy<float>(g, d->batch, stream);
    mark(events, 1, stream);
    mark(events, 2, stream);
    return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
  }
  if (d->rule == SIMSD_ACCEPT_MATCH) {
    MatchParams m;
    m.target = d->target_logits;
    m.draft_tokens = d->draft_tokens;
    m.tau = d->tau;
    m.cu_B = d->cu_B;
    m.uniforms = d->uniforms;
    m.n_accept = d->n_accept;
    m.token = d->token;
    m.pos = d->pos;
    m.status = (uint32_t *)ws;
    m.vocab = d->vocab;
    m.B_max = d->B_max;
    m.csize = 1;
    m.per = 0;
    m.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits);
    m.ls = kLog2e / (d->temperature > 0.f ? d->temperature : 1.f);
    mark(events, 0, stream);
    const cudaError_t e = d->dtype == SIMSD_BF16 ? launch_match<__nv_bfloat16>(m, d->batch, stream)
                                                 : launch_match<float>(m, d->batch, stream);
    mark(events, 1, stream);
    mark(events, 2, stream);
    return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
  }
  AcceptParams a;
  a.target = d->target_logits;
  a.draft = d->draft_logits;
  a.draft_tokens = d->draft_tokens;
  a.tau = d->tau;
  a.cu_B = d->cu_B;
  a.uniforms = d->uniforms;
  a.n_accept = d->n_accept;
  a.token = d->token;
  a.pos = d->pos;
  a.status = (uint32_t *)ws;
  a.batch = d->batch;
  a.vocab = d->vocab;
  a.B_max = d->B_max;
  a.total_B = d->total_B;
  a.ls = kLog2e / (d->temperature > 0.f ? d->temperature : 1.f);
  // slices of whole 16-byte vectors (set with the cluster size at launch);
  // a piece is one ring stage
  a.csize = kMaxCluster;
  a.per = 0;
  a.piece = 0;
  a.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits) &&
           aligned16(d->draft_logits);
  mark(events, 0, stream);
  const cudaError_t e = d->dtype == SIMSD_BF16 ? launch<__nv_bfloat16>(a, stream)
                                               : launch<float>(a, stream);
  mark(events, 1, stream);
  mark(events, 2, stream);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

}  // namespace
}  // namespace simsd

using namespace simsd;

extern "C" {

size_t simsd_accept_workspace_size(const simsd_accept_desc *d) {
  if (accept_check(d) != SIMSD_OK) return 0;
  return kAcceptWorkspace;
}

simsd_status simsd_accept(const simsd_accept_desc *d, void *stream_ptr) {
  return simsd_accept_timed(d, stream_ptr, nullptr);
}

simsd_status simsd_accept_timed(const simsd_accept_desc *d, void *stream_ptr,
                                void *const events[3]) {
  simsd_status st = accept_check(d);
  if (st != SIMSD_OK) return st;
  if (!accept_pointers_ok(d)) return SIMSD_ERR_NULL;
  if (d->workspace == nullptr || ((uintptr_t)d->workspace % kAlign) != 0 ||
      d->workspace_bytes < kAcceptWorkspace)
    return SIMSD_ERR_WORKSPACE;
  return run_accept(d, (char *)d->workspace, (cudaStream_t)stream_ptr, events);
}

// Same kernel and arguments as simsd_accept; scratch from the static array
// instead of a caller workspace (see simsd.h for who needs this).
simsd_status simsd_accept_noalloc(const simsd_accept_desc *d, void *stream_ptr) {
  simsd_status st = accept_check(d);
  if (st != SIMSD_OK) return st;
  if (!accept_pointers_ok(d)) return SIMSD_ERR_NULL;
  if (kAcceptWorkspace > SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES) return SIMSD_ERR_WORKSPACE;
  char *ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return SIMSD_ERR_CUDA;
  return run_accept(d, ws, (cudaStream_t)stream_ptr, nullptr);
}

}  // extern "C"
