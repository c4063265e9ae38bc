// accept.cu -- K4: rejection-sampling acceptance along the temporal order.
//
// SimSD section 4 "Speculative Decoding Pipeline", acceptance: standard
// rejection sampling along the draft-induced temporal order; the longest
// accepted prefix is committed.  For sequence b, step t = 1..B tests the
// slot k = tau^-1(t) with draft token x: p = softmax(target row k / T),
// q = softmax(draft row k / T) at temperature T (1 by default); accept iff
// u[t-1] * q(x) < p(x) (fp32).  At the first rejection a token is drawn
// from max(0, p - q) normalised (p itself when that is empty) by inverse
// CDF with u[B].  The greedy rule and sample matching (Spiffy's
// verification) share the machinery below.
//
// Two paths.  The chunked path (a workspace of simsd_accept_workspace_size
// bytes, no decided steps) runs K4a, the chunk pass: every SM streams
// (row, 32 KB chunk) items through a bulk-copy ring and writes, per eighth
// of a chunk (a "part"), what the rule needs (reference and sum of
// exponentials; the largest value and its index; the mass below the draft
// token), plus the logits at the draft tokens.  K4b then finishes from
// those partials -- for sampling, CTAs per (sequence, chunk range) that
// each repeat the sequence's walk, compute their chunks' residual masses and
// let the last of them draw; for greedy and matching, a CTA per sequence.
// The single-launch path (a workspace of just the status word, or decided
// steps) is one thread-block cluster of C CTAs per sequence (C <= 16, from
// a makespan estimate over the resident-cluster waves), CTA r owning the
// vocabulary slice [r * per, (r + 1) * per) of every row of the sequence;
// it streams its slices of the 2B rows in pieces of at most 32 KB through a
// 6-stage shared-memory ring (one producer warp, two groups of 8 consumer
// warps taking alternate pieces):
//   1. per (slot, row): maximum and sum of exponentials of the slice;
//   2. cluster barrier; every CTA merges the C slices' partials through
//      distributed shared memory, evaluates p(x), q(x) and walks the steps
//      (identically: same inputs, same order; CTA 0 writes the outputs);
//   3. on a rejection every CTA streams its slices of the rejected slot's
//      two rows again (from L2) for the residual and target masses of 16
//      contiguous vocabulary ranges of each piece;
//   4. cluster barrier; every CTA reads the C slice totals, so all agree on
//      the CTA whose slice holds u * S; one warp of that CTA narrows down to
//      the piece, then the range, then rereads that range and finds the
//      entry by a warp scan in vocabulary order.
// Numerics: a partial state is (R, s) with R a reference in log2 units (the
// maximum of x log2 e seen so far, rounded once) and s = sum 2^(x log2 e - R),
// each exponent argument formed by one fma (a single rounding, small for
// the entries near the maximum that carry the mass) and exponentiated by
// the MUFU ex2 instruction.  Normalisers, masses and running CDFs across
// parts are compensated fp32 pairs (two-sum), never fp64 (GB300's fp64
// rate is a small fraction of its fp32 rate); within a part or range the
// running mass is fp32 relative to its start.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "vocab.cuh"

namespace simsd {
namespace {

using namespace vocab;

constexpr int kMaxCluster = 16;                    // CTAs per sequence, at most (over 8: non-portable)
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
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
// the chunk pass (K4a) of the two-kernel path
// a chunk is one ring stage: kStageBytes / sizeof(T) entries (and a K4b piece)
constexpr int kAStages = 3;
constexpr int kAConsumerWarps = 8;
constexpr int kAConsumers = kAConsumerWarps * 32;
constexpr int kAThreads = kAConsumers + 32;
constexpr int kMaxPairs = 2 * kMaxB;               // (slot, row) pairs per sequence
constexpr int kMaxVocab = 1 << 21;                 // 8 slices of kMaxPieces pieces of 8192 fp32 entries

// ---------------------------------------------------------------- state
struct __align__(16) WalkInfo {
  int slot;              // rejected slot (0-based within the sequence), -1: none
  float Mt, Md;          // its references (log2 units)
  Ff rho;                // St / Sd
  float u;               // the residual draw's uniform
  int pad0, pad1;
};

template <int NW>                             // consumer warps
struct __align__(16) AccSharedT {
  uint64_t full[kStages], empty[kStages];
  float2 part_w[kMaxPairs][NW];               // per warp: (R, s) of each (slot, row)
  float2 cpart[kMaxPairs];                    // this CTA's slice: (R, s)
  float4 norm[kMaxPairs];                     // merged (M, S.hi, S.lo) of each (slot, row)
  float2 xv[kMaxB];                           // logits at the draft token, if in this slice
  float px[kMaxB], qx[kMaxB], u[kMaxB + 1];
  int tau[kMaxB], x[kMaxB], slot_of_step[kMaxB];
  float4 piece_w[kMaxPieces][kRanges];        // residual pass: per range (r pair, p pair)
  float4 piece_s[kMaxPieces];
  float4 tot;                                 // this slice's residual and target mass
  WalkInfo walk;                              // CTA 0's result, read by every CTA
  int flag;                                   // any wait of this CTA gave up
  int fail1, fail3;                           // ... in phase 1 / phase 3 (read remotely
                                              // after the barrier closing that phase)
};

struct AcceptParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  const int32_t *decided;   // steps decided in earlier passes (NULL: none)
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int batch, vocab, B_max, total_B;
  uint32_t polls;  // bounded-wait polls
  int csize;   // CTAs per cluster (one cluster per sequence)
  int per;     // entries per CTA slice (a multiple of 16 bytes' worth)
  int piece;   // entries per ring stage
  int bulk;    // rows 16-byte aligned: bulk copies; else element copies
  Scale ls;    // log2(e) / temperature
};

// NW consumer warps (two groups) and an NS-stage ring: one CTA per SM.
template <typename T, int NW, int NS>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
accept_kernel(const __grid_constant__ AcceptParams a) {
  constexpr int N = Ld<T>::N;
  constexpr int kConsumerWarps = NW, kConsumers = NW * 32, kStages = NS;
  constexpr int kGroupWarps = NW / 2, kGroupThreads = kGroupWarps * 32;
  constexpr int kVecs = kStageBytes / 16 / kGroupThreads;   // phase 1
  constexpr int kRangesPerWarp = kRanges / NW;
  static_assert(kRangesPerWarp * NW == kRanges, "whole ranges per warp");
  using AccShared = AccSharedT<NW>;
  auto consumers_sync = [] { named_sync(1, kConsumers); };
  extern __shared__ __align__(128) uint8_t smem[];
  AccShared &S = *reinterpret_cast<AccShared *>(smem + kStages * kStageBytes);
  const uint32_t ring = smem_u32(smem);
  const int rank = blockIdx.x;               // the cluster spans x: rank = blockIdx.x
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  const bool producer = warp == kConsumerWarps;
  const Scale ls = a.ls;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int dcd = a.decided ? __ldg(a.decided + b) : 0;   // the walk starts at step dcd + 1
  // the same in every CTA of the cluster; rows c0 .. c0+B-1 exist
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B && dcd >= 0 &&
                     dcd <= B;
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
    S.fail1 = 0;
    S.fail3 = 0;
    fence_barrier_init();
  }
  __syncthreads();                           // the ring's barriers are ready
  if (valid && !producer) {                  // (the producer starts streaming meanwhile)
    if (t < B) {
      S.tau[t] = __ldg(a.tau + c0 + t);
      S.x[t] = __ldg(a.draft_tokens + c0 + t);
    }
    if (t < B) S.xv[t] = make_float2(0.f, 0.f);
    if (t <= B) S.u[t] = __ldg(a.uniforms + (long)b * (a.B_max + 1) + t);
    consumers_sync();                        // the sequence's labels, tokens, uniforms
  }
  // the open slots (labels above dcd): only their rows are streamed; open
  // pair q is (open slot number q / 2, row q % 2)
  uint32_t open = 0;
  if (valid) {
    if (a.decided == nullptr) {
      open = B == 32 ? 0xffffffffu : (1u << B) - 1u;
    } else if (producer) {
      open = __ballot_sync(0xffffffffu, lane < B && __ldg(a.tau + c0 + lane) > dcd);
    } else {
      for (int k = 0; k < B; ++k)
        if (S.tau[k] > dcd) open |= 1u << k;
    }
  }
  const int n_open = __popc(open);
  auto slot_of = [&](int i) { return (int)__fns(open, 0, i + 1); };   // open slot number i

  int issued = 0;                            // producer: stages started so far
  int g = 0;                                 // stage counter (producer and consumers)
  if (valid) {
    // ---------------------------------------------------- 1. row slices
    const int J = 2 * n_open * npieces;
    if (producer) {
      for (int pair = 0, pc = 0; g < J; ++g) {
        const int s = g % kStages;
        if (g >= kStages && !mbar_wait_warp(smem_u32(&S.empty[s]), ((g / kStages) - 1) & 1, a.polls)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); atomicOr(&S.fail1, 1); }
          break;
        }
        copy_piece<T>(smem + s * kStageBytes, ring + s * kStageBytes,
                      row_ptr(slot_of(pair >> 1), pair & 1) + pc * a.piece, piece_len(pc),
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
        for (int q = 0; q < 2 * n_open; ++q) S.part_w[q][warp] = make_float2(-INFINITY, 0.f);
      float R = -INFINITY, sum = 0.f;
      int gg = grp * chunk, pair = 0, pc = gg;
      if (npieces > 0)
        while (pc >= npieces) { pc -= npieces; ++pair; }
      while (gg < J) {
        const int s = gg % kStages;
        const int n = piece_len(pc);
        if (!mbar_wait_warp(smem_u32(&S.full[s]), (gg / kStages) & 1, a.polls)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); atomicOr(&S.fail1, 1); }
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
          const int ks = slot_of(pair >> 1);
          const int off = S.x[ks] - (s0 + pc * a.piece);
          if (off >= 0 && off < n) {
            const float v = pick<T>(sv[off / N], off % N);
            if (pair & 1) S.xv[ks].y = v; else S.xv[ks].x = v;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_n(smem_u32(&S.empty[s]), 2);
        const float mx = Ld<T>::vmax(w, kVecs);
        const float Rn = ref_of(mx, ls);
        if (Rn > R) {
          sum = R == -INFINITY ? 0.f : sum * exp2_int(R - Rn);
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
          float sc = Rm == -INFINITY ? 0.f : sum * exp2_int(R - Rm);
#pragma unroll
          for (int m = 16; m > 0; m >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, m);
          if (lane == 0) S.part_w[pair_now][warp] = make_float2(Rm, sc);
          R = -INFINITY;
          sum = 0.f;
        }
      }
      consumers_sync();
      if (t < 2 * n_open) {                // this CTA's slice of open pair t
        float2 c = make_float2(-INFINITY, 0.f);
        if (npieces > 0 && !*(volatile int *)&S.flag) {
          float M = -INFINITY;
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, S.part_w[t][w].x);
          Ff sm = ff_of(0.f);
          if (M != -INFINITY)
#pragma unroll 1
            for (int w = 0; w < kConsumerWarps; ++w) {
              const float2 v = S.part_w[t][w];
              if (v.y > 0.f) sm = ff_add(sm, ff_of(v.y * exp2_int(v.x - M)));
            }
          c = make_float2(M, sm.hi + sm.lo);
        }
        S.cpart[t] = c;
      }
    }
    cluster_sync();                        // B1: every slice's partials are in place

    // ---------------------------------------------------- 2. the walk
    // every CTA merges the slices' partials and walks the steps itself (the
    // same inputs in the same order give the same decisions everywhere), so
    // no barrier is needed before the residual pass; CTA 0 writes outputs
    if (!producer) {
      // thread (pair q, slice r) reads one slice's partial; groups of gs
      // lanes (8, or 16 for clusters over 8) merge them (pair q: slot q / 2,
      // row q % 2)
      const int lg = a.csize > 8 ? 4 : 3, gs = 1 << lg;
      for (int q0 = 0; q0 < 2 * n_open; q0 += kConsumers >> lg) {
      if (warp * 32 < (2 * n_open - q0) << lg) {  // whole warps: the shuffles need every lane
        const int q = q0 + (t >> lg), r = t & (gs - 1);
        const bool mine = q < 2 * n_open;
        const int k = mine ? slot_of(q >> 1) : 0, row = q & 1, x = mine ? S.x[k] : -1;
        const bool xin = x >= 0 && x < a.vocab;
        // the logits at x: from the slice that holds x (every CTA has them
        // in partials mode)
        const float2 xl = r == 0 && xin ? ld_dsmem2(dsmem(&S.xv[k], x / a.per)) : make_float2(0.f, 0.f);
        const float2 v = mine && r < a.csize ? ld_dsmem2(dsmem(&S.cpart[q], r)) : make_float2(-INFINITY, 0.f);
        float M = v.x;
#pragma unroll 1
        for (int m = gs / 2; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
        Ff sm = ff_of(M != -INFINITY && v.y > 0.f ? v.y * exp2_int(v.x - M) : 0.f);
#pragma unroll 1
        for (int m = gs / 2; m > 0; m >>= 1) sm = ff_add(sm, ff_shfl_xor(sm, m));
        if (mine && r == 0) {
          S.norm[2 * k + row] = make_float4(M, sm.hi, sm.lo, 0.f);
          // p(x) (row 0) or q(x) (row 1); a token no slice holds rejects
          const float pr = xin ? rel_exp(row ? xl.y : xl.x, M, ls) / (sm.hi + sm.lo) : 0.f;
          if (row) S.qx[k] = pr; else S.px[k] = pr;
          if (!xin && row == 0 && rank == 0) raise_status(a.status, kStatusBadInput);
        }
      }
      }
    }
    if (!producer) {
      consumers_sync();
      if (t == 0) {
        for (int k = 0; k < kMaxB; ++k) S.slot_of_step[k] = 0;
        uint32_t seen = 0;
        for (int k = 0; k < B; ++k) {
          const int tk = S.tau[k];
          if (tk >= 1 && tk <= B) {
            seen |= 1u << (tk - 1);
            S.slot_of_step[tk - 1] = k;
          }
        }
        // a tau that is not a permutation of 1..B, or a wait in any CTA of
        // the cluster that gave up in phase 1 (the snapshots are final
        // after B1, so every CTA decides alike): no walk
        bool any_fail = false;
        for (int r = 0; r < a.csize; ++r) any_fail |= ld_dsmem_i32(dsmem(&S.fail1, r)) != 0;
        const bool perm = seen == (B == 32 ? 0xffffffffu : (1u << B) - 1u);
        int n = B, rej = -1;
        if (!perm || any_fail) {
          n = 0;
          if (!perm && rank == 0) raise_status(a.status, kStatusBadInput);
        } else {
          for (int st = dcd + 1; st <= B; ++st) {
            const int k = S.slot_of_step[st - 1];
            if (!(S.u[st - 1] * S.qx[k] < S.px[k])) { n = st - 1; rej = k; break; }
          }
        }
        if (rank == 0) {
          a.n_accept[b] = n;
          a.pos[b] = rej;
          if (rej < 0) a.token[b] = -1;
        }
        WalkInfo w{-1, 0.f, 0.f, Ff{1.f, 0.f}, 0.f, 0, 0};
        if (rej >= 0) {
          const float4 nt = S.norm[2 * rej], nd = S.norm[2 * rej + 1];
          w.slot = rej;
          w.Mt = nt.x;
          w.Md = nd.x;
          w.rho = ff_div(Ff{nt.y, nt.z}, Ff{nd.y, nd.z});
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
          if (g >= kStages && !mbar_wait_warp(smem_u32(&S.empty[s]), ((g / kStages) - 1) & 1, a.polls)) {
            if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); atomicOr(&S.fail3, 1); }
            break;
          }
          copy_piece<T>(smem + s * kStageBytes, ring + s * kStageBytes,
                        row_ptr(w.slot, row) + pc * a.piece, piece_len(pc),
                        smem_u32(&S.full[s]), a.bulk, lane);
          issued = g + 1;
        }
      } else {
        // every warp takes part in every piece: warp w reads ranges w,
        // w + NW, ..., each the contiguous vectors [r * kRangeVecs,
        // (r + 1) * kRangeVecs) of the piece (lane-interleaved), whose
        // masses the draw narrows down to
        for (int pc = 0; pc < npieces && !*(volatile int *)&S.flag; ++pc) {
          const int gt = J + 2 * pc, gd = gt + 1;
          const int st = gt % kStages, sd = gd % kStages;
          const int n = piece_len(pc);
          if (!mbar_wait_warp(smem_u32(&S.full[st]), (gt / kStages) & 1, a.polls) ||
              !mbar_wait_warp(smem_u32(&S.full[sd]), (gd / kStages) & 1, a.polls)) {
            if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(&S.flag, 1); atomicOr(&S.fail3, 1); }
            break;
          }
          const uint4 *tv = reinterpret_cast<const uint4 *>(smem + st * kStageBytes);
          const uint4 *dv = reinterpret_cast<const uint4 *>(smem + sd * kStageBytes);
          const int nvec = (n + N - 1) / N;
          float rs[kRangesPerWarp][4], ps[kRangesPerWarp][4];
#pragma unroll
          for (int k = 0; k < kRangesPerWarp; ++k) {
            const int r = warp + k * NW;
#pragma unroll
            for (int e = 0; e < 4; ++e) rs[k][e] = ps[k][e] = 0.f;
            if (r * kRangeVecs < nvec) {
#pragma unroll
              for (int i = 0; i < kRangeVecs / 32; ++i) {
                const int idx = r * kRangeVecs + i * 32 + lane;
                const bool in = idx < nvec;
                float ft[N], fd[N];
                Ld<T>::unpack(in ? tv[idx] : Ld<T>::neg_inf(), ft);
                Ld<T>::unpack(in ? dv[idx] : Ld<T>::neg_inf(), fd);
#pragma unroll
                for (int e = 0; e < N; ++e) {
                  const float et = rel_exp(ft[e], w.Mt, ls);
                  rs[k][e & 3] += residual(et, draft_mass(fd[e], w.Md, w.rho, ls));
                  ps[k][e & 3] += et;
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&S.empty[st]));
            mbar_arrive(smem_u32(&S.empty[sd]));
          }
#pragma unroll
          for (int k = 0; k < kRangesPerWarp; ++k) {
            Ff fr = ff_add(ff_of(rs[k][0] + rs[k][1]), ff_of(rs[k][2] + rs[k][3]));
            Ff fp = ff_add(ff_of(ps[k][0] + ps[k][1]), ff_of(ps[k][2] + ps[k][3]));
#pragma unroll 1
            for (int m = 16; m > 0; m >>= 1) {
              fr = ff_add(fr, ff_shfl_xor(fr, m));
              fp = ff_add(fp, ff_shfl_xor(fp, m));
            }
            if (lane == 0) S.piece_w[pc][warp + k * NW] = make_float4(fr.hi, fr.lo, fp.hi, fp.lo);
          }
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
        // a wait that gave up in any CTA's residual pass (snapshots final
        // after B3): every CTA skips the draw, CTA 0 reports no walk
        const bool any_fail =
            __any_sync(0xffffffffu, lane < a.csize && ld_dsmem_i32(dsmem(&S.fail3, lane)) != 0);
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
        if (any_fail && rank == 0 && lane == 0) {
          a.n_accept[b] = 0;
          a.token[b] = -1;
          a.pos[b] = -1;
        }
        if (!any_fail && ch == rank && !*(volatile int *)&S.flag) {
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
              const float et = rel_exp(ft[e], w.Mt, ls);
              m[e] = use_p ? et : residual(et, draft_mass(fd[e], w.Md, w.rho, ls));
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

// ---------------------------------------------------------------- chunk pass
// K4a of the two-kernel path: every SM streams (row, chunk) items -- rows
// are the target and draft rows of every slot, chunks kChunk entries --
// through a bulk-copy ring.  Each consumer warp takes its own 1/8 of every
// item (kV 16-byte vectors per lane), reduces it against its own
// whole-number reference and writes (reference, sum) for (row, chunk,
// warp); the warp whose part holds the slot's draft token also writes that
// logit.  Warps never wait for one another -- only for the ring -- so a
// warp can be on the next item while another finishes this one.  No item
// depends on another, so the grid is as many CTAs as the SMs hold (two per
// SM for bf16) and every SM streams until the items run out; the
// per-sequence walk and residual draw (K4b, the cluster kernel in partials
// mode) then read only these partials and the rejected slots' rows.

// candidate (v, i) beats (w, j): a larger value, or an equal one at a
// smaller index (-inf entries still win over "none", index 2^31 - 1)
__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

struct ChunkParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  float2 *part;       // [2 total_B][nchunks][kAConsumerWarps]: (reference, sum of 2^(l ls - ref))
  float *xlogit;      // [2 total_B]
  float4 *part4;      // draft rows only: [total_B][nchunks][kAConsumerWarps]: (reference,
                      // sum, the part's largest logit, -)
  int *claim;         // [0] item counter, [1] give-up flag, [2] readers' count (zero at
                      // launch; the kernel reading the partials zeroes them again)
  int *zero;          // n_zero ints the pass zeroes for the kernel after it (or NULL)
  int n_zero;
  uint32_t *status;
  int vocab, total_B, nchunks, bulk;
  uint32_t polls;
  Scale ls;
};

template <typename T>
__host__ __device__ constexpr int chunk_stage_bytes() { return kStageBytes; }
template <typename T>
__host__ __device__ constexpr int chunk_entries() { return kStageBytes / (int)sizeof(T); }
template <typename T>
constexpr size_t chunk_smem_bytes() { return (size_t)kAStages * chunk_stage_bytes<T>() + 256; }

// Modes: the sampling rule (target and draft rows in pairs; per part
// (reference, sum); the logit at the slot's draft token); the draft-side
// step (draft rows; per part (reference, sum, largest logit)); sample
// matching (target rows; per part (reference, sum, the sum over the
// entries below the draft token x when x is in the part); the logit at x);
// the greedy rule (target rows; per part the largest value and its
// smallest index).
enum : int { kModeSample = 0, kModeDraft = 1, kModeMatch = 2, kModeGreedy = 3 };

template <typename T, int MODE>
__global__ void __launch_bounds__(kAThreads)
vocab_chunk_kernel(const __grid_constant__ ChunkParams a) {
  constexpr bool kPairs = MODE == kModeSample;
  constexpr bool kToken = MODE == kModeSample || MODE == kModeMatch;
  constexpr int N = Ld<T>::N;
  constexpr int kStage = chunk_stage_bytes<T>();
  constexpr int kChunk = chunk_entries<T>();
  constexpr int kWarpVecs = kStage / 16 / kAConsumerWarps;   // a warp's part of an item
  constexpr int kV = kWarpVecs / 32;                         // 16-byte vectors per lane
  static_assert(kV * 32 * kAConsumerWarps * 16 == kStage, "the warps' parts tile an item");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kAStages * kStage);
  uint64_t *empty = full + kAStages;
  int *stage_x = reinterpret_cast<int *>(empty + kAStages);   // [kAStages]: the item's draft token
  int *stage_i = stage_x + kAStages;                          // [kAStages]: the item, -1: the end
  int *flag = stage_i + kAStages;                             // a wait gave up (the drain)
  const uint32_t ring = smem_u32(smem);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const bool producer = warp == kAConsumerWarps;
  grid_dep_launch();                           // the kernel after it may be scheduled
  const long items = (kPairs ? 2L : 1L) * a.total_B * a.nchunks;
  if (a.zero != nullptr)                       // counters the kernel after it starts from
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero; i += gridDim.x * blockDim.x)
      a.zero[i] = 0;
  if (t == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kAConsumerWarps);
    }
    *flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  long issued = 0;
  bool ended = false;
  if (producer) {
    // Items: a CTA's first 2 kAStages items are static (blockIdx.x + k
    // grid), the rest come from the workspace counter (first_dyn + c), so
    // CTAs that stream faster take more.  Lane 0 keeps, per ring slot u,
    // the slot's next item and its draft token (requested a ring ahead)
    // and a claim one more ring ahead (its latency overlaps a ring of
    // copies); the loop is unrolled by kAStages, so these stay in
    // registers and none is moved while its load is in flight.
    const long grid = gridDim.x, first_dyn = 2L * kAStages * grid;
    auto token_of = [&](long i) {
      return !kToken || i < 0 ? 0 : __ldg(a.draft_tokens + (kPairs ? i / a.nchunks >> 1 : i / a.nchunks));
    };
    long it[kAStages], ahead[kAStages];
    int xs[kAStages];
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < kAStages; ++u) {
        const long i0 = blockIdx.x + u * grid, i1 = blockIdx.x + (kAStages + u) * grid;
        it[u] = i0 < items ? i0 : -1;
        ahead[u] = i1 < items ? i1 : -1;
        xs[u] = token_of(it[u]);
      }
    }
    bool ok = true;
    for (long j0 = 0; ok && !ended; j0 += kAStages) {
#pragma unroll
      for (int u = 0; u < kAStages; ++u) {
        const long j = j0 + u;
        const int s = u;                            // j % kAStages (j0 is a multiple)
        if (j >= kAStages && !mbar_wait_warp(smem_u32(&empty[s]), ((j / kAStages) - 1) & 1, a.polls)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag, 1); atomicOr(a.claim + 1, 1); }
          ok = false;
          break;
        }
        const long i = __shfl_sync(0xffffffffu, lane == 0 ? it[u] : 0L, 0);
        if (i < 0) {                                // the end: a stage without data
          if (lane == 0) {
            stage_i[s] = -1;
            mbar_arrive(smem_u32(&full[s]));
          }
          ended = true;
          break;
        }
        const long p = i / a.nchunks;               // row pair index: slot p/2, target or draft
        const int c = (int)(i % a.nchunks);
        const int n = min(kChunk, a.vocab - c * kChunk);
        // the item and its draft token go beside the stage before the
        // copy's arrival (release) makes the stage visible to the consumers
        if (lane == 0) {
          stage_x[s] = xs[u];
          stage_i[s] = (int)i;
        }
        __syncwarp();
        const T *src = MODE == kModeDraft   ? (const T *)a.draft + p * a.vocab + (long)c * kChunk
                       : MODE != kModeSample ? (const T *)a.target + p * a.vocab + (long)c * kChunk
                                             : (const T *)((p & 1) ? a.draft : a.target) +
                                                   (p >> 1) * a.vocab + (long)c * kChunk;
        copy_piece<T>(smem + s * kStage, ring + s * kStage, src, n, smem_u32(&full[s]), a.bulk, lane);
        issued = j + 1;
        if (lane == 0) {
          it[u] = ahead[u];
          xs[u] = token_of(it[u]);
          ahead[u] = -1;
          if (it[u] >= 0) {
            const long i2 = first_dyn + atomicAdd(a.claim, 1);
            ahead[u] = i2 < items ? i2 : -1;
          }
        }
      }
    }
  } else {
    for (long j = 0;; ++j) {
      const int s = (int)(j % kAStages);
      // a warp whose wait gave up neither reads nor releases the stage (its
      // copy may still land) and stops; the others are not held up by it
      if (!mbar_wait_warp(smem_u32(&full[s]), (j / kAStages) & 1, a.polls)) {
        if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag, 1); atomicOr(a.claim + 1, 1); }
        break;
      }
      const int i = stage_i[s];
      if (i < 0) break;                             // the end
      const long p = i / a.nchunks;
      const int c = i % a.nchunks;
      const int n = min(kChunk, a.vocab - c * kChunk);
      const uint4 *sv = reinterpret_cast<const uint4 *>(smem + s * kStage);
      const int v0 = warp * kWarpVecs;              // this warp's vectors: v0 + v * 32 + lane
      uint4 w[kV];
      if (n == kChunk) {                            // a whole chunk: no bound checks
#pragma unroll
        for (int v = 0; v < kV; ++v) w[v] = sv[v0 + v * 32 + lane];
      } else {
#pragma unroll
        for (int v = 0; v < kV; ++v) {
          const int idx = v0 + v * 32 + lane;
          w[v] = idx * N < n ? sv[idx] : Ld<T>::neg_inf();
        }
      }
      // the logit at the slot's draft token, if this warp's part holds it
      const int off = kToken ? stage_x[s] - c * kChunk : -1;
      if (off >= 0 && off < n && off / N >= v0 && off / N < v0 + kWarpVecs && (off / N - v0) % 32 == lane) {
        const int vx = (off / N - v0) / 32;
        uint4 wx = w[0];
#pragma unroll
        for (int v = 1; v < kV; ++v)
          if (v == vx) wx = w[v];
        a.xlogit[p] = pick<T>(wx, off % N);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      if (MODE == kModeGreedy) {
        // this warp's part: its largest value (NaN entries never count: the
        // maxima skip them, and a lane of NaN alone counts as -inf), then
        // the smallest index holding it -- searched only by the lanes whose
        // own maximum it is (usually one), vectors in order, entries past
        // the row excluded
        float lm = Ld<T>::vmax(w, kV);
        if (lm != lm) lm = -INFINITY;
        const uint32_t lu = __float_as_uint(lm);
        const uint32_t kl = __reduce_max_sync(0xffffffffu, (lu & 0x80000000u) ? ~lu : (lu | 0x80000000u));
        const float bv = __uint_as_float((kl & 0x80000000u) ? (kl & 0x7fffffffu) : ~kl);
        uint32_t cand = 0x7fffffffu;
        if (lm == bv) {
#pragma unroll
          for (int v = 0; v < kV; ++v) {
            float f[N];
            Ld<T>::unpack(w[v], f);
            const int base = (v0 + v * 32 + lane) * N;
#pragma unroll
            for (int e = 0; e < N; ++e)
              if (cand == 0x7fffffffu && f[e] == bv && base + e < n) cand = (uint32_t)(c * kChunk + base + e);
          }
        }
        const int bi = (int)__reduce_min_sync(0xffffffffu, cand);
        if (lane == 0)
          a.part4[(p * a.nchunks + c) * kAConsumerWarps + warp] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
        continue;
      }
      // this warp's part: its maximum, then its sum against a whole-number
      // reference (combined with the others' by exact powers of two)
      const float mx = Ld<T>::vmax(w, kV);
      const uint32_t mu = __float_as_uint(mx);
      const uint32_t km = __reduce_max_sync(0xffffffffu, (mu & 0x80000000u) ? ~mu : (mu | 0x80000000u));
      const float wmax = __uint_as_float((km & 0x80000000u) ? (km & 0x7fffffffu) : ~km);
      const float R = ref_of(wmax, a.ls);
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, below = 0.f;
      // sample matching: the entries below x, where x is in this part
      const int xo = MODE == kModeMatch ? stage_x[s] - c * kChunk : -1;
      const bool x_here = MODE == kModeMatch && xo > v0 * N && xo <= (v0 + kWarpVecs) * N;
      if (R != -INFINITY) {
#pragma unroll
        for (int v = 0; v < kV; ++v) {
          float f[N];
          Ld<T>::unpack(w[v], f);
#pragma unroll
          for (int e = 0; e < N; ++e) {
            const float m = rel_exp(f[e], R, a.ls);
            acc[(v * N + e) & 3] += m;
            if (x_here && (v0 + v * 32 + lane) * N + e < xo) below += m;
          }
        }
      }
      float sm = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      if (x_here)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) below += __shfl_xor_sync(0xffffffffu, below, o);
      if (lane == 0) {
        if (MODE == kModeDraft)
          a.part4[(p * a.nchunks + c) * kAConsumerWarps + warp] = make_float4(R, sm, wmax, 0.f);
        else if (MODE == kModeMatch)
          a.part4[(p * a.nchunks + c) * kAConsumerWarps + warp] = make_float4(R, sm, below, 0.f);
        else
          a.part[(p * a.nchunks + c) * kAConsumerWarps + warp] = make_float2(R, sm);
      }
    }
  }
  // after a wait that gave up the copies in flight land before the CTA
  // can exit (the flag is final after the barrier; the end took the stage
  // of item issued - kAStages, whose copy was consumed before)
  __syncthreads();
  if (producer && *(volatile int *)flag) {
    const long from = issued - (ended ? kAStages - 1 : kAStages);
    for (long j = from > 0 ? from : 0; j < issued; ++j)
      (void)mbar_wait_warp(smem_u32(&full[j % kAStages]), (j / kAStages) & 1);
  }
}

// The sampling rule's chunk pass for small batches: no ring, a warp per
// part (1/8 of a 32 KB chunk of one row) with its 16-byte loads issued at
// once, as many warps as the device holds looping over the parts -- so a
// batch of a few thousand parts is requested from memory in one go instead
// of three ring stages at a time per CTA.  Each warp reduces its part
// exactly as a consumer warp of the ring kernel does (the same loads, the
// same order of operations), so the partials are the same bits.
constexpr int kPartThreads = 256;

// five CTAs (40 warps, 40 parts in flight) per SM at 48 registers, no
// spills: the pass is bound by the bytes it has in flight
template <typename T>
__global__ void __launch_bounds__(kPartThreads, 5)
vocab_part_kernel(const __grid_constant__ ChunkParams a) {
  constexpr int N = Ld<T>::N;
  constexpr int kChunk = chunk_entries<T>();
  constexpr int kWarpVecs = kStageBytes / 16 / kAConsumerWarps;   // a part's vectors
  constexpr int kV = kWarpVecs / 32;
  grid_dep_launch();                           // the kernel after it may be scheduled
  if (a.zero != nullptr)                       // counters the kernel after it starts from
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero; i += gridDim.x * blockDim.x)
      a.zero[i] = 0;
  const int lane = threadIdx.x & 31;
  // fewer than 2^31 parts (the launch checks): 32-bit index arithmetic
  const unsigned parts = 2u * (unsigned)a.total_B * (unsigned)a.nchunks * kAConsumerWarps;
  const unsigned nwarps = gridDim.x * (kPartThreads / 32);
  const unsigned nch = (unsigned)a.nchunks;
#pragma unroll 1
  for (unsigned pi = blockIdx.x * (kPartThreads / 32) + (threadIdx.x >> 5); pi < parts; pi += nwarps) {
    const int pw = (int)(pi % kAConsumerWarps);                // the part within its chunk
    const unsigned i = pi / kAConsumerWarps;                   // the (row pair, chunk) item
    const unsigned p = i / nch;                                // row pair: slot p/2, target or draft
    const int c = (int)(i - p * nch);
    const int n = min(kChunk, a.vocab - c * kChunk);
    const T *src = (const T *)((p & 1) ? a.draft : a.target) + (size_t)(p >> 1) * a.vocab + (size_t)c * kChunk;
    const int v0 = pw * kWarpVecs;
    uint4 w[kV];
    if (n == kChunk && a.bulk != 0) {          // a whole chunk of 16-byte rows: no bound checks
#pragma unroll
      for (int v = 0; v < kV; ++v)
        w[v] = *reinterpret_cast<const uint4 *>(src + (v0 + v * 32 + lane) * N);
    } else {
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const int idx = v0 + v * 32 + lane;
        w[v] = idx * N < n ? Ld<T>::load(src + idx * N, n - idx * N, a.bulk != 0) : Ld<T>::neg_inf();
      }
    }
    // the logit at the slot's draft token, if this part holds it
    const int off = __ldg(a.draft_tokens + (p >> 1)) - c * kChunk;
    if (off >= 0 && off < n && off / N >= v0 && off / N < v0 + kWarpVecs && (off / N - v0) % 32 == lane) {
      const int vx = (off / N - v0) / 32;
      uint4 wx = w[0];
#pragma unroll
      for (int v = 1; v < kV; ++v)
        if (v == vx) wx = w[v];
      a.xlogit[p] = pick<T>(wx, off % N);
    }
    const float mx = Ld<T>::vmax(w, kV);
    const uint32_t mu = __float_as_uint(mx);
    const uint32_t km = __reduce_max_sync(0xffffffffu, (mu & 0x80000000u) ? ~mu : (mu | 0x80000000u));
    const float wmax = __uint_as_float((km & 0x80000000u) ? (km & 0x7fffffffu) : ~km);
    const float R = ref_of(wmax, a.ls);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (R != -INFINITY) {
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        float f[N];
        Ld<T>::unpack(w[v], f);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[(v * N + e) & 3] += rel_exp(f[e], R, a.ls);
      }
    }
    float sm = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) a.part[(p * a.nchunks + c) * kAConsumerWarps + pw] = make_float2(R, sm);
  }
}

// Parts per resident warp up to which the sampling rule's chunk pass takes
// the ring-free kernel above.  At five CTAs per SM, 16 x 1024 has 1.7 parts
// per warp, 8 x 32768 3.4 and 64 x 4096 13.5; an A/B on one GPU (ring-free
// against ring, step time): 59.4 -> 55.9 us, 230.3 -> 226.6 us and
// 288.3 -> 290.7 us, so the ring keeps the third.  The ring-free kernel has
// no bounded waits.
constexpr double kDirectPartsPerWarp = 6.0;

template <typename T>
cudaError_t launch_parts(const ChunkParams &c, cudaStream_t stream, bool *taken) {
  static std::mutex mu;
  static int resident[64] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (resident[dev] == 0) {
      int n = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, vocab_part_kernel<T>, kPartThreads, 0);
      if (e != cudaSuccess) return e;
      resident[dev] = n > 0 ? n : 1;
    }
    per_sm = resident[dev];
  }
  const long parts = 2L * c.total_B * c.nchunks * kAConsumerWarps;
  const long ctas = (long)per_sm * device_sm_count();
  *taken = (double)parts <= kDirectPartsPerWarp * (double)(ctas * (kPartThreads / 32)) &&
           parts < (1L << 31);
  if (!*taken) return cudaSuccess;
  const long grid = std::min<long>(ctas, (parts + kPartThreads / 32 - 1) / (kPartThreads / 32));
  vocab_part_kernel<T><<<(unsigned)grid, kPartThreads, 0, stream>>>(c);
  return cudaGetLastError();
}

// The cluster kernel's instance: consumer warps, ring stages, threads and
// shared memory.
template <int NW, int NS>
struct AccCfg {
  static constexpr int kNW = NW, kNS = NS, kThreadsPerCta = (NW + 1) * 32;
  static constexpr size_t kSmem = (size_t)NS * kStageBytes + sizeof(AccSharedT<NW>);
};
using CfgSingle = AccCfg<kConsumerWarps, kStages>;
static_assert(CfgSingle::kSmem <= 227 * 1024, "shared memory budget");

void mark(void *const *events, int i, cudaStream_t stream) {
  if (events != nullptr) record_event(events[i], stream);
}

template <typename C>
cudaLaunchConfig_t launch_config(int csize, int batch, cudaStream_t stream, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize, batch);
  cfg.blockDim = dim3(C::kThreadsPerCta);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Per device, instance and cluster size 1..kMaxCluster: clusters resident
// at once (queried once; the answer depends on the device only; -1 for a
// size the device cannot place).
template <typename T, typename C>
cudaError_t max_active_clusters(int dev, int csize, int *out) {
  static std::mutex mu;
  static int cache[64][kMaxCluster + 1] = {};
  auto kern = accept_kernel<T, C::kNW, C::kNS>;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][0] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    // sizes over 8 are optional: without the attribute they are skipped
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      (void)cudaGetLastError();
    cache[dev][0] = 1;
  }
  if (cache[dev][csize] == 0) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config<C>(csize, csize, nullptr, attr);
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
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

template <typename T, typename C>
cudaError_t launch_cfg(AcceptParams a, cudaStream_t stream) {
  const int dev = current_device();
  // Cluster size by a makespan estimate: clusters run in waves of the
  // resident count; a CTA's time is its share of the sequence's exponentials
  // at 16 per clock per SM (a round figure: the MUFU alone sustains ~24, the
  // whole streaming loop fewer) plus the fixed cost of the walk, residual
  // and draw phases.  Small batches get large clusters (every SM busy),
  // large batches small ones (fewer waves).  Never so small that a slice
  // needs more pieces than the kernel tracks.
  const int vec = 16 / (int)sizeof(T);
  const int piece = kStageBytes / (int)sizeof(T);
  const int64_t max_slice = (int64_t)kMaxPieces * piece;
  const double per_seq = (2.0 * a.total_B / a.batch + 2.0) * a.vocab;   // exponentials
  constexpr double kPhaseCycles = 20000.0;
  int csize = kMaxCluster;
  double best = 1e300;
  for (int c = kMaxCluster; c >= 1; --c) {
    if (((int64_t)a.vocab + c - 1) / c > max_slice) break;
    int n = 0;
    cudaError_t e = max_active_clusters<T, C>(dev, c, &n);
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
  const cudaLaunchConfig_t cfg = launch_config<C>(csize, a.batch, stream, attr);
  return cudaLaunchKernelEx(&cfg, accept_kernel<T, C::kNW, C::kNS>, a);
}

template <typename T>
cudaError_t launch(AcceptParams a, cudaStream_t stream) {
  return launch_cfg<T, CfgSingle>(a, stream);
}

// The chunk pass: as many CTAs as the device holds at once (queried once
// per device and dtype), never more than the items.
template <typename T, int MODE>
cudaError_t launch_chunks(const ChunkParams &c, cudaStream_t stream) {
  static std::mutex mu;
  static int resident[64] = {0};
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (resident[dev] == 0) {
      cudaError_t e = cudaFuncSetAttribute(vocab_chunk_kernel<T, MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)chunk_smem_bytes<T>());
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, vocab_chunk_kernel<T, MODE>, kAThreads,
                                                        chunk_smem_bytes<T>());
      if (e != cudaSuccess) return e;
      resident[dev] = n > 0 ? n : 1;
    }
    per_sm = resident[dev];
  }
  const long items = (MODE == kModeSample ? 2L : 1L) * c.total_B * c.nchunks;
  const long grid = std::min<long>(items, (long)per_sm * device_sm_count());
  vocab_chunk_kernel<T, MODE><<<(unsigned)grid, kAThreads, chunk_smem_bytes<T>(), stream>>>(c);
  return cudaGetLastError();
}

// ------------------------------------------------ greedy and matching finish
// After a greedy or matching chunk pass over the target rows: one CTA per
// sequence, a warp per slot.  Greedy: the row's argmax from the parts'
// candidates (largest value, smallest index); the step accepts iff the
// draft token is it, and a rejection emits it.  Matching: the row's
// reference M and normaliser S, the mass below the draft token x, Pre(x) =
// the parts before x's part plus the part's own mass below x, and x's mass
// m(x); with U = u S the step accepts iff Pre(x) <= U < Pre(x) + m(x).  A
// slot that rejects draws the target's own token at U at once (part_draw:
// the part holding U, then a column scan), so the walk -- warp 0, over
// every slot's outcome -- only picks the first rejected step's result.
constexpr int kRuleThreads = 512;
constexpr int kRuleWarps = kRuleThreads / 32;

struct RuleFinishParams {
  const void *target;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  const float4 *part4;      // [total_B][nchunks][kAConsumerWarps]
  const float *xlogit;      // [total_B] (matching)
  int *claim;               // the chunk pass's control words
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int vocab, total_B, B_max, nchunks, bulk;
  Scale ls;
};

template <typename T, int MODE>
__global__ void __launch_bounds__(kRuleThreads)
rule_finish_kernel(const __grid_constant__ RuleFinishParams a) {
  static_assert(MODE == kModeGreedy || MODE == kModeMatch, "the greedy and matching rules");
  constexpr int kChunk = chunk_entries<T>();
  constexpr int kPartLen = kChunk / kAConsumerWarps;   // entries of a part
  constexpr int kHeld = 4;                             // parts held per lane: 4 x 32
  __shared__ int acc_s[kMaxB], tok_s[kMaxB];
  __shared__ int fail_s;
  const int b = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  grid_dep_wait();                                     // the chunk pass's partials
  // the chunk pass's give-up flag, read by the last thread (checked at the
  // walk); the CTA whose ticket is the last zeroes the chunk pass's words
  const int flag_t = kRuleThreads - 1;
  int ticket = -1;
  if (t == flag_t) fail_s = chunk_flag_read(a.claim, &ticket);
  const int c0 = __ldg(a.cu_B + b), B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B;
  if (!valid) {                                        // malformed sequence: no walk
    if (t == 0) {
      a.n_accept[b] = 0;
      a.token[b] = -1;
      a.pos[b] = -1;
      raise_status(a.status, kStatusBadInput);
    }
    if (t == flag_t) chunk_flag_reset(a.claim, ticket, gridDim.x);
    return;
  }
  const Scale ls = a.ls;
  const int n_ent = a.nchunks * kAConsumerWarps;       // parts of a row
  for (int k = warp; k < B; k += kRuleWarps) {
    const float4 *pr = a.part4 + (long)(c0 + k) * n_ent;
    const int x = __ldg(a.draft_tokens + c0 + k);
    const bool xin = x >= 0 && x < a.vocab;
    float4 h[kHeld];
#pragma unroll
    for (int i = 0; i < kHeld; ++i)
      h[i] = lane + 32 * i < n_ent ? __ldcg(pr + lane + 32 * i)
                                   : make_float4(-INFINITY, MODE == kModeGreedy ? __int_as_float(0x7fffffff) : 0.f, 0.f, 0.f);
    if (MODE == kModeGreedy) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      auto take = [&](float4 v) {
        if (beats(v.x, __float_as_int(v.y), bv, bi)) { bv = v.x; bi = __float_as_int(v.y); }
      };
#pragma unroll
      for (int i = 0; i < kHeld; ++i) take(h[i]);
      for (int i = lane + 32 * kHeld; i < n_ent; i += 32) take(__ldcg(pr + i));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        const int am = bi == 0x7fffffff ? 0 : bi;   // no entry beat "none": a NaN row
        acc_s[k] = xin && x == am;
        tok_s[k] = am;
      }
    } else {
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < kHeld; ++i) M = fmaxf(M, h[i].x);
      for (int i = lane + 32 * kHeld; i < n_ent; i += 32) M = fmaxf(M, __ldcg(pr + i).x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      // S and Pre(x), in units of 2^M, as compensated pairs
      const int px = xin ? x / kPartLen : -1;        // x's part (parts are in vocabulary order)
      Ff S = ff_of(0.f), Pre = ff_of(0.f);
      auto add = [&](int i, float4 v) {
        const float w = (M != -INFINITY && v.x != -INFINITY) ? exp2_int(v.x - M) : 0.f;
        const float m = v.y > 0.f ? v.y * w : 0.f;
        S = ff_add(S, ff_of(m));
        if (i < px) Pre = ff_add(Pre, ff_of(m));
        else if (i == px && v.z > 0.f) Pre = ff_add(Pre, ff_of(v.z * w));
      };
#pragma unroll
      for (int i = 0; i < kHeld; ++i) add(lane + 32 * i, h[i]);
      for (int i = lane + 32 * kHeld; i < n_ent; i += 32) add(i, __ldcg(pr + i));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        S = ff_add(S, ff_shfl_xor(S, o));
        Pre = ff_add(Pre, ff_shfl_xor(Pre, o));
      }
      const int st = __ldg(a.tau + c0 + k);
      const float u = st >= 1 && st <= B ? __ldg(a.uniforms + (long)b * (a.B_max + 1) + st - 1) : 0.f;
      const float uh = u * S.hi;
      const Ff U = ff_add(Ff{uh, fmaf(u, S.hi, -uh)}, ff_of(u * S.lo));
      const float mx = xin ? rel_exp(__ldcg(a.xlogit + c0 + k), M, ls) : 0.f;   // m(x)
      const bool acc = mx > 0.f && !ff_gt(Pre, U) && ff_gt(ff_add(Pre, ff_of(mx)), U);
      int y = -1;
      if (!acc)                                      // warp-uniform: the target's own token at U
        y = part_draw<T, kHeld>(pr, h, n_ent, M, U, (const T *)a.target + (long)(c0 + k) * a.vocab,
                                a.vocab, kChunk, a.bulk != 0, ls, lane);
      if (lane == 0) {
        acc_s[k] = acc;
        tok_s[k] = y;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // the walk: the first rejected step over a permutation of 1..B
    const int tk = lane < B ? __ldg(a.tau + c0 + lane) : 0;
    const int x = lane < B ? __ldg(a.draft_tokens + c0 + lane) : 0;
    const uint32_t seen = __reduce_or_sync(0xffffffffu, lane < B && tk >= 1 && tk <= B ? 1u << (tk - 1) : 0u);
    const bool perm = seen == (B == 32 ? 0xffffffffu : (1u << B) - 1u);
    const bool rejects = lane < B && !acc_s[lane];
    const uint32_t rstep = __reduce_min_sync(0xffffffffu, rejects ? (uint32_t)tk : 0xffffffffu);
    const int last = rstep == 0xffffffffu ? B : (int)rstep;   // the walk's last step
    const bool badx = lane < B && tk <= last && (x < 0 || x >= a.vocab);
    const bool fail = fail_s != 0;
    const bool any_bad = __any_sync(0xffffffffu, badx);
    const unsigned rl = __ballot_sync(0xffffffffu, rejects && (uint32_t)tk == rstep);
    if (lane == 0) {
      if (!perm) raise_status(a.status, kStatusBadInput);
      else if (!fail && any_bad) raise_status(a.status, kStatusBadInput);
      if (!perm || fail) {                            // no walk
        a.n_accept[b] = 0;
        a.token[b] = -1;
        a.pos[b] = -1;
      } else if (rstep == 0xffffffffu) {              // every step accepted
        a.n_accept[b] = B;
        a.token[b] = -1;
        a.pos[b] = -1;
      } else {
        const int k = __ffs(rl) - 1;
        a.n_accept[b] = (int)rstep - 1;
        a.token[b] = tok_s[k];
        a.pos[b] = k;
      }
    }
  }
  if (t == flag_t) chunk_flag_reset(a.claim, ticket, gridDim.x);
}

template <typename T, int MODE>
cudaError_t launch_rule_finish(const RuleFinishParams &f, int batch, cudaStream_t stream) {
  return launch_pdl(rule_finish_kernel<T, MODE>, dim3(batch), dim3(kRuleThreads), 0, stream, f);
}

// ------------------------------------------------------------ sampling finish
// After the sampling rule's chunk pass, one launch (started early by
// programmatic dependent launch) of nsplit CTAs per sequence, CTA j owning
// the 32 KB chunks [j cpc, (j + 1) cpc) of the rows (nsplit from the batch:
// about two CTAs per SM in all):
//   1. the walk, in every CTA of the sequence alike (same inputs, same
//      order, so all agree): a warp per row merges the row's parts into its
//      reference and normaliser and p(x) or q(x); warp 0 walks the steps
//      (accept iff u[t-1] q(x) < p(x)); the first CTA writes n_accept and
//      pos (and token -1 when nothing is drawn);
//   2. on a rejection, a warp per sixteenth of each of its chunks (a "sub-
//      part": 2 KB of each of the rejected slot's two rows, one round of
//      loads): the residual mass, sum max(0, e_t - rho e_d), and the target
//      mass, sum e_t, as pairs in units of 2^Mt (rho = St / Sd);
//   3. the CTA that counts last for its sequence (a per-sequence counter in
//      the workspace, zeroed by the chunk pass) draws: the residual total
//      (the target total when the residual is empty), U = u[B] times it,
//      the sub-part holding U, then its entries in vocabulary order.
// So the whole GPU takes part in the residual pass (its rows come from L2
// when the chunk pass left them there), and the walk, the residual and the
// draw cost one launch after the chunk pass.
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kSubParts = kFinWarps;                 // sub-parts per chunk: a warp each

struct SampleFinishParams {
  const void *target;
  const void *draft;
  const int32_t *draft_tokens;
  const int32_t *tau;
  const int32_t *cu_B;
  const float *uniforms;
  const float2 *part;      // [2 total_B][nchunks][kAConsumerWarps]: the chunk pass's (R, s)
  const float *xlogit;     // [2 total_B]: the logits at the draft tokens
  float4 *res4;            // [batch][nchunks][kSubParts]: (residual pair, target pair)
  int *count;              // [batch]: CTAs whose residual sub-parts are written (the
                           // chunk pass zeroes them)
  int *claim;              // the chunk pass's control words
  int32_t *n_accept;
  int32_t *token;
  int32_t *pos;
  uint32_t *status;
  int batch, vocab, total_B, B_max, nchunks, bulk;
  int nsplit, cpc;         // CTAs per sequence, chunks per CTA
  Scale ls;
};

template <typename T>
__global__ void __launch_bounds__(kFinThreads, 2)
sample_finish_kernel(const __grid_constant__ SampleFinishParams a) {
  constexpr int N = Ld<T>::N;
  constexpr int kChunk = chunk_entries<T>();
  constexpr int kSubLen = kChunk / kSubParts;          // entries of a sub-part
  constexpr int kSubVecs = kSubLen / N;                // 16-byte vectors of a sub-part
  constexpr int kV = kSubVecs / 32;                    // per lane and row
  constexpr int kHeld = 4;                             // chunk-pass parts held per lane: 4 x 32
  static_assert(kV * 32 * N * kSubParts == kChunk, "sub-parts tile a chunk");
  __shared__ float4 nrm_s[2 * kMaxB];                  // per row (2k: target, 2k+1: draft): (M, S.hi, S.lo, p(x) or q(x))
  __shared__ float4 wsum_s[kFinWarps];                // the draw: per warp (residual pair, target pair)
  __shared__ int fail_s, rej_s, last_s;
  const int j = blockIdx.x, b = blockIdx.y, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // the inputs written before the chunk pass (the sections, labels and
  // uniforms; warp 0 holds lane l: tau, u[l], and u[B]) are read while it
  // finishes
  const int c0 = __ldg(a.cu_B + b), B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B;
  const int tk = valid && warp == 0 && lane < B ? __ldg(a.tau + c0 + lane) : 0;
  const float ul = valid && warp == 0 && lane <= B ? __ldg(a.uniforms + (long)b * (a.B_max + 1) + lane) : 0.f;
  const float uB = valid ? __ldg(a.uniforms + (long)b * (a.B_max + 1) + B) : 0.f;
  grid_dep_wait();                                     // the chunk pass's partials
  // the chunk pass's give-up flag (every CTA reads it; the last to count
  // zeroes the chunk pass's words at exit)
  const int flag_t = kFinThreads - 1;
  int ticket = -1;
  if (t == flag_t) fail_s = chunk_flag_read(a.claim, &ticket);
  const int ctas = gridDim.x * gridDim.y;
  if (!valid) {                                        // malformed sequence: no walk
    if (j == 0 && t == 0) {
      a.n_accept[b] = 0;
      a.token[b] = -1;
      a.pos[b] = -1;
      raise_status(a.status, kStatusBadInput);
    }
    if (t == flag_t) chunk_flag_reset(a.claim, ticket, ctas);
    return;
  }
  const Scale ls = a.ls;
  // -------------------------------------------------------- 1. the walk
  const int n_ent = a.nchunks * kAConsumerWarps;       // chunk-pass parts of a row
  // rows warp and warp + kFinWarps together (their loads in one round)
  for (int r0 = warp; r0 < 2 * B; r0 += 2 * kFinWarps) {
    float2 h[2][kHeld];
    float xl[2];
    bool xin[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int r = r0 + q * kFinWarps;
      const bool has = r < 2 * B;
      const float2 *pr = a.part + (long)(2 * c0 + r) * n_ent;
      const int x = has ? __ldg(a.draft_tokens + c0 + (r >> 1)) : 0;
      xin[q] = x >= 0 && x < a.vocab;
      xl[q] = has ? __ldcg(a.xlogit + 2 * c0 + r) : 0.f;
#pragma unroll
      for (int i = 0; i < kHeld; ++i)
        h[q][i] = has && lane + 32 * i < n_ent ? __ldcg(pr + lane + 32 * i) : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int r = r0 + q * kFinWarps;
      if (r >= 2 * B) break;                           // warp-uniform
      const float2 *pr = a.part + (long)(2 * c0 + r) * n_ent;
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < kHeld; ++i) M = fmaxf(M, h[q][i].x);
      for (int i = lane + 32 * kHeld; i < n_ent; i += 32) M = fmaxf(M, __ldcg(pr + i).x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      auto mass_of = [&](float2 v) {
        const float w = (M != -INFINITY && v.x != -INFINITY) ? exp2_int(v.x - M) : 0.f;
        return ff_of(v.y > 0.f ? v.y * w : 0.f);
      };
      Ff S = ff_of(0.f);
#pragma unroll
      for (int i = 0; i < kHeld; ++i) S = ff_add(S, mass_of(h[q][i]));
      for (int i = lane + 32 * kHeld; i < n_ent; i += 32) S = ff_add(S, mass_of(__ldcg(pr + i)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S = ff_add(S, ff_shfl_xor(S, o));
      if (lane == 0) {
        // p(x) or q(x); a token outside the vocabulary rejects
        nrm_s[r] = make_float4(M, S.hi, S.lo, xin[q] ? rel_exp(xl[q], M, ls) / (S.hi + S.lo) : 0.f);
        if (!xin[q] && (r & 1) == 0 && j == 0) raise_status(a.status, kStatusBadInput);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // the first rejected step over a permutation of 1..B
    const bool tin = lane < B && tk >= 1 && tk <= B;
    const uint32_t seen = __reduce_or_sync(0xffffffffu, tin ? 1u << (tk - 1) : 0u);
    const bool perm = seen == (B == 32 ? 0xffffffffu : (1u << B) - 1u);
    const float ut = __shfl_sync(0xffffffffu, ul, tin ? tk - 1 : 0);
    const bool rejects = tin && !(ut * nrm_s[2 * lane + 1].w < nrm_s[2 * lane].w);
    const uint32_t rstep = __reduce_min_sync(0xffffffffu, rejects ? (uint32_t)tk : 0xffffffffu);
    const unsigned rl = __ballot_sync(0xffffffffu, rejects && (uint32_t)tk == rstep);
    const bool walk = perm && !fail_s;
    if (lane == 0) {
      rej_s = walk && rstep != 0xffffffffu ? __ffs(rl) - 1 : -1;
      if (j == 0) {
        if (!perm) raise_status(a.status, kStatusBadInput);
        a.n_accept[b] = !walk ? 0 : rstep == 0xffffffffu ? B : (int)rstep - 1;
        a.pos[b] = walk && rstep != 0xffffffffu ? __ffs(rl) - 1 : -1;
        if (!walk || rstep == 0xffffffffu) a.token[b] = -1;   // else the draw writes it
      }
    }
  }
  __syncthreads();
  const int k = rej_s;
  if (k < 0) {
    if (t == flag_t) chunk_flag_reset(a.claim, ticket, ctas);
    return;
  }
  // ------------------------------------------------ 2. the residual sub-parts
  const float4 nt = nrm_s[2 * k], nd = nrm_s[2 * k + 1];
  const float Mt = nt.x, Md = nd.x;
  const Ff rho = ff_div(Ff{nt.y, nt.z}, Ff{nd.y, nd.z});
  const long row = c0 + k;
  const T *trow = (const T *)a.target + row * a.vocab;
  const T *drow = (const T *)a.draft + row * a.vocab;
  const int cend = min(a.nchunks, (j + 1) * a.cpc);
#pragma unroll 1
  for (int c = j * a.cpc; c < cend; ++c) {
    const int n = min(kChunk, a.vocab - c * kChunk);
    uint4 wt[kV], wd[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      const int e0 = (warp * kSubVecs + i * 32 + lane) * N;
      wt[i] = Ld<T>::load(trow + (long)c * kChunk + e0, n - e0, a.bulk != 0);
      wd[i] = Ld<T>::load(drow + (long)c * kChunk + e0, n - e0, a.bulk != 0);
    }
    float rs[4] = {0.f, 0.f, 0.f, 0.f}, ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      float ft[N], fd[N];
      Ld<T>::unpack(wt[i], ft);
      Ld<T>::unpack(wd[i], fd);
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const float et = rel_exp(ft[e], Mt, ls);
        rs[e & 3] += residual(et, draft_mass(fd[e], Md, rho, ls));
        ps[e & 3] += et;
      }
    }
    Ff fr = ff_add(ff_of(rs[0] + rs[1]), ff_of(rs[2] + rs[3]));
    Ff fp = ff_add(ff_of(ps[0] + ps[1]), ff_of(ps[2] + ps[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      fr = ff_add(fr, ff_shfl_xor(fr, o));
      fp = ff_add(fp, ff_shfl_xor(fp, o));
    }
    if (lane == 0)
      a.res4[((long)b * a.nchunks + c) * kSubParts + warp] = make_float4(fr.hi, fr.lo, fp.hi, fp.lo);
  }
  __syncthreads();                                     // every sub-part of this CTA written
  if (a.nsplit == 1) {
    if (t == 0) last_s = 1;                            // (written by this CTA alone)
  } else if (t == 0) {
    __threadfence();                                   // the sub-parts precede the count
    last_s = atomicAdd(a.count + b, 1) == a.nsplit - 1;
    if (last_s) __threadfence();                       // the others' sub-parts are visible
  }
  __syncthreads();
  if (last_s) {
    // ------------------------------------------------------- 3. the draw
    // warp w sums the sub-parts [w per, (w + 1) per); every warp finds, from
    // the same 16 warp totals in the same order, the warp whose range holds
    // U (the first whose running mass exceeds it, else the last with mass);
    // that warp finds the sub-part in its range and scans its entries
    const int n_sub = a.nchunks * kSubParts;
    const int per = (n_sub + kFinWarps - 1) / kFinWarps;
    const int s0 = min(n_sub, warp * per), s1 = min(n_sub, s0 + per);
    const float4 *pr = a.res4 + (long)b * n_sub;
    float4 h1[1];
    h1[0] = s0 + lane < s1 ? __ldcg(pr + s0 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    Ff Sr{h1[0].x, h1[0].y}, Sp{h1[0].z, h1[0].w};
    for (int i = s0 + 32 + lane; i < s1; i += 32) {
      const float4 v = __ldcg(pr + i);
      Sr = ff_add(Sr, Ff{v.x, v.y});
      Sp = ff_add(Sp, Ff{v.z, v.w});
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Sr = ff_add(Sr, ff_shfl_xor(Sr, o));
      Sp = ff_add(Sp, ff_shfl_xor(Sp, o));
    }
    if (lane == 0) wsum_s[warp] = make_float4(Sr.hi, Sr.lo, Sp.hi, Sp.lo);
    __syncthreads();
    float4 hw[1];
    hw[0] = lane < kFinWarps ? wsum_s[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    Ff Tr{hw[0].x, hw[0].y}, Tp{hw[0].z, hw[0].w};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Tr = ff_add(Tr, ff_shfl_xor(Tr, o));
      Tp = ff_add(Tp, ff_shfl_xor(Tp, o));
    }
    // U = u[B] S (the target's own mass when the residual is empty)
    const bool use_p = !(Tr.hi > 0.f);
    const Ff tot = use_p ? Tp : Tr;
    const float uh = uB * tot.hi;
    const Ff U = ff_add(Ff{uh, fmaf(uB, tot.hi, -uh)}, ff_of(uB * tot.lo));
    auto mass_of = [&](const float4 &v) { return use_p ? Ff{v.z, v.w} : Ff{v.x, v.y}; };
    Ff wstart;                                         // (16 totals, all held: wsum_s is not re-read)
    const int owner = locate_part<1>(wsum_s, hw, kFinWarps, U, mass_of, lane, &wstart);
    if (warp == owner) {
      const Ff U2 = ff_add(U, ff_neg(wstart));
      Ff base;
      const int sel = s0 + locate_part<1>(pr + s0, h1, s1 - s0, U2, mass_of, lane, &base);
      const int p0 = (sel / kSubParts) * kChunk + (sel % kSubParts) * kSubLen;
      const Ff D0 = ff_add(U2, ff_neg(base));
      const T *const rows[2] = {trow, drow};
      const int tok = scan_part<T, 2>(rows, p0, min(kSubLen, a.vocab - p0), kSubVecs, D0.hi + D0.lo,
                                      a.bulk != 0, lane, [&](const float (&f)[2][N], float (&m)[N]) {
#pragma unroll
                                        for (int e = 0; e < N; ++e) {
                                          const float et = rel_exp(f[0][e], Mt, ls);
                                          m[e] = use_p ? et : residual(et, draft_mass(f[1][e], Md, rho, ls));
                                        }
                                      });
      if (lane == 0) a.token[b] = tok;
    }
  }
  if (t == flag_t) chunk_flag_reset(a.claim, ticket, ctas);
}

// At most two CTAs per SM over the batch (one wave), each CTA whole chunks.
template <typename T>
cudaError_t launch_sample_finish(SampleFinishParams f, cudaStream_t stream) {
  const int want = 2 * device_sm_count() / f.batch;
  const int ns = std::max(1, std::min(want, f.nchunks));
  f.cpc = (f.nchunks + ns - 1) / ns;
  f.nsplit = (f.nchunks + f.cpc - 1) / f.cpc;
  return launch_pdl(sample_finish_kernel<T>, dim3(f.nsplit, f.batch), dim3(kFinThreads), 0, stream, f);
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
  const int32_t *decided;
  int vocab, total_B, B_max, csize, per, bulk;
};


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
  const int dcd = a.decided ? __ldg(a.decided + b) : 0;
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B && dcd >= 0 &&
                     dcd <= B;
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  if (valid) {
    for (int k = 0; k < B; ++k) {
      if (dcd > 0 && __ldg(a.tau + c0 + k) <= dcd) continue;   // decided: never tested
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
      uint32_t seen = 0;
      for (int k = 0; k < B; ++k) {
        const int tk = __ldg(a.tau + c0 + k);
        if (tk >= 1 && tk <= B) { seen |= 1u << (tk - 1); slot_of_step[tk - 1] = k; }
      }
      const bool perm = seen == (B == 32 ? 0xffffffffu : (1u << B) - 1u);
      if (!perm) raise_status(a.status, kStatusBadInput);
      int n = perm ? B : 0, tok = -1, ps = -1;
      for (int st = dcd + 1; perm && st <= B; ++st) {
        const int k = slot_of_step[st - 1];
        float v = -INFINITY;
        int am = 0x7fffffff;
        for (int r = 0; r < a.csize; ++r) {
          const float2 c = ld_dsmem2(dsmem(&cand[k], r));
          if (beats(c.x, __float_as_int(c.y), v, am)) { v = c.x; am = __float_as_int(c.y); }
        }
        if (am == 0x7fffffff) am = 0;               // no entry beat "none" (NaN row)
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
  const int32_t *decided;
  int vocab, total_B, B_max, csize, per, bulk;
  Scale ls;
};

struct __align__(16) MatchSlot {
  float R, xl;       // the slice's reference (log2 units) and l_x if x lies in it
  Ff s, pre;         // sum of 2^(l ls - R) over the slice, and over its entries below x
};

// (R, s, pre) += (R2, s2, pre2): both sums to the larger reference
__device__ __forceinline__ void match_merge(float &R, Ff &s, Ff &pre, float R2, Ff s2, Ff pre2) {
  const float M = fmaxf(R, R2);
  if (M == -INFINITY) return;
  const float a = exp2_int(R - M), b = exp2_int(R2 - M);
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
  const Scale ls = a.ls;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int dcd = a.decided ? __ldg(a.decided + b) : 0;
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B && dcd >= 0 &&
                     dcd <= B;
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  auto value_at = [&](const T *row, int e) { return Ld<T>::value(row[e]); };
  if (valid) {
    for (int k = 0; k < B; ++k) {
      if (dcd > 0 && __ldg(a.tau + c0 + k) <= dcd) continue;   // decided: never tested
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
        const float Rn = ref_of(mx, ls);
        if (Rn > R) {
          const float c = R == -INFINITY ? 0.f : exp2_int(R - Rn);
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
      uint32_t seen = 0;
      for (int k = 0; k < B; ++k) {
        const int tk = __ldg(a.tau + c0 + k);
        if (tk >= 1 && tk <= B) { seen |= 1u << (tk - 1); slot_of_step[tk - 1] = k; }
      }
      const bool perm = seen == (B == 32 ? 0xffffffffu : (1u << B) - 1u);
      if (!perm && rank == 0) raise_status(a.status, kStatusBadInput);
      int n = perm ? B : 0, rej = -1;
      for (int st = dcd + 1; perm && st <= B; ++st) {
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
            const float w = exp2_int(h.x - M);
            S = ff_add(S, Ff{h.z * w, h.w * w});
            Pre = ff_add(Pre, Ff{q.x * w, q.y * w});
          }
        const int x = __ldg(a.draft_tokens + c0 + k);
        if (x < 0 || x >= a.vocab) raise_status(a.status, kStatusBadInput);
        const float u = __ldg(a.uniforms + (long)b * (a.B_max + 1) + st - 1);
        const float uh = u * S.hi;
        const Ff U = ff_add(Ff{uh, fmaf(u, S.hi, -uh)}, ff_of(u * S.lo));
        const float px = (x >= 0 && x < a.vocab) ? rel_exp(xl, M, ls) : 0.f;   // mass of x
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
          const float w = h.x == -INFINITY ? 0.f : exp2_int(h.x - M);
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

// Workspace: the status word; for the chunked paths also the chunk pass's
// control words (beside the status word), the chunk partials and the
// draft-token logits.
// Sampling: partials [2 total_B][nchunks][8] (float2), logits [2 total_B],
// per-sequence counters [batch] (zeroed by the chunk pass) and the residual
// sub-parts [batch][nchunks][16] (float4);
// greedy and matching: partials [total_B][nchunks][8] (float4), logits
// [total_B].  A workspace of just the status word runs the single cluster
// kernel of the rule (the rows streamed per sequence), as do walks from
// decided steps (those kernels skip the decided slots' rows).
constexpr size_t kAcceptWorkspace = kAlign;
struct AcceptLayout {
  int nchunks;
  size_t off_part, off_xlogit, off_claim, off_count, off_res4, total;
};
AcceptLayout accept_layout(const simsd_accept_desc *d) {
  AcceptLayout L;
  const int chunk = kStageBytes / (d->dtype == SIMSD_BF16 ? 2 : 4);
  const bool pairs = d->rule == SIMSD_ACCEPT_SAMPLE;
  const size_t rows = (size_t)(pairs ? 2 : 1) * d->total_B;
  L.nchunks = (d->vocab + chunk - 1) / chunk;
  L.off_claim = kClaimOffset;                 // beside the status word
  L.off_part = kAcceptWorkspace;
  L.off_xlogit = align_up(L.off_part + rows * L.nchunks * kAConsumerWarps *
                                           (pairs ? sizeof(float2) : sizeof(float4)), kAlign);
  L.off_count = align_up(L.off_xlogit + rows * sizeof(float), kAlign);
  L.off_res4 = align_up(L.off_count + (pairs ? (size_t)d->batch * sizeof(int) : 0), kAlign);
  L.total = align_up(L.off_res4 + (pairs ? (size_t)d->batch * L.nchunks * kSubParts * sizeof(float4) : 0),
                     kAlign);
  return L;
}
size_t accept_workspace(const simsd_accept_desc *d) { return accept_layout(d).total; }

// Scratch of simsd_accept_noalloc: one static array per device, alive until
// the process exits.  Host code may not take its address directly (the
// name is a host-side stand-in there); static_scratch() looks the device
// address up once per device.
constexpr int kMaxDevices = 64;
static_assert(SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES % kAlign == 0, "scratch size");
static_assert(SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES >= kAcceptWorkspace, "scratch size");
static_assert(kClaimOffset >= sizeof(uint32_t) && kClaimOffset + kClaimBytes <= kAcceptWorkspace,
              "the control words sit beside the status word");
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
// simsd_read_status reads them).  ws_bytes: the workspace's size.
simsd_status run_accept(const simsd_accept_desc *d, char *ws, size_t ws_bytes,
                        cudaStream_t stream, void *const *events) {
  const int es = d->dtype == SIMSD_BF16 ? 2 : 4;
  const AcceptLayout L = accept_layout(d);
  const bool chunked = d->decided == nullptr && ws_bytes >= L.total;
  const bool bf16 = d->dtype == SIMSD_BF16;
  if (d->rule != SIMSD_ACCEPT_SAMPLE && chunked) {
    // the chunk pass over the target rows on every SM, then one CTA per sequence
    const bool greedy = d->rule == SIMSD_ACCEPT_GREEDY;
    ChunkParams c;
    c.target = d->target_logits;
    c.draft = nullptr;
    c.draft_tokens = d->draft_tokens;
    c.part = nullptr;
    c.xlogit = (float *)(ws + L.off_xlogit);
    c.part4 = (float4 *)(ws + L.off_part);
    c.claim = (int *)(ws + L.off_claim);
    c.zero = nullptr;
    c.n_zero = 0;
    c.status = (uint32_t *)ws;
    c.vocab = d->vocab;
    c.total_B = d->total_B;
    c.nchunks = L.nchunks;
    c.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits);
    c.polls = wait_polls_of(d->wait_polls);
    c.ls = scale_of(d->temperature > 0.f ? (double)d->temperature : 1.0);
    RuleFinishParams f;
    f.target = d->target_logits;
    f.draft_tokens = d->draft_tokens;
    f.tau = d->tau;
    f.cu_B = d->cu_B;
    f.uniforms = d->uniforms;
    f.part4 = c.part4;
    f.xlogit = c.xlogit;
    f.claim = c.claim;
    f.n_accept = d->n_accept;
    f.token = d->token;
    f.pos = d->pos;
    f.status = c.status;
    f.vocab = d->vocab;
    f.total_B = d->total_B;
    f.B_max = d->B_max;
    f.nchunks = L.nchunks;
    f.bulk = c.bulk;
    f.ls = c.ls;
    mark(events, 0, stream);
    cudaError_t e = greedy ? (bf16 ? launch_chunks<__nv_bfloat16, kModeGreedy>(c, stream)
                                   : launch_chunks<float, kModeGreedy>(c, stream))
                           : (bf16 ? launch_chunks<__nv_bfloat16, kModeMatch>(c, stream)
                                   : launch_chunks<float, kModeMatch>(c, stream));
    mark(events, 1, stream);
    if (e == cudaSuccess)
      e = greedy ? (bf16 ? launch_rule_finish<__nv_bfloat16, kModeGreedy>(f, d->batch, stream)
                         : launch_rule_finish<float, kModeGreedy>(f, d->batch, stream))
                 : (bf16 ? launch_rule_finish<__nv_bfloat16, kModeMatch>(f, d->batch, stream)
                         : launch_rule_finish<float, kModeMatch>(f, d->batch, stream));
    mark(events, 2, stream);
    return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
  }
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
    g.decided = d->decided;
    g.vocab = d->vocab;
    g.total_B = d->total_B;
    g.B_max = d->B_max;
    g.csize = 1;
    g.per = 0;
    g.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits);
    mark(events, 0, stream);
    const cudaError_t e = bf16 ? launch_greedy<__nv_bfloat16>(g, d->batch, stream)
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
    m.decided = d->decided;
    m.vocab = d->vocab;
    m.total_B = d->total_B;
    m.B_max = d->B_max;
    m.csize = 1;
    m.per = 0;
    m.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits);
    m.ls = scale_of(d->temperature > 0.f ? (double)d->temperature : 1.0);
    mark(events, 0, stream);
    const cudaError_t e = bf16 ? launch_match<__nv_bfloat16>(m, d->batch, stream)
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
  a.decided = d->decided;
  a.n_accept = d->n_accept;
  a.token = d->token;
  a.pos = d->pos;
  a.status = (uint32_t *)ws;
  a.batch = d->batch;
  a.vocab = d->vocab;
  a.B_max = d->B_max;
  a.total_B = d->total_B;
  a.polls = wait_polls_of(d->wait_polls);
  a.ls = scale_of(d->temperature > 0.f ? (double)d->temperature : 1.0);
  // slices of whole 16-byte vectors (set with the cluster size at launch);
  // a piece is one ring stage
  a.csize = kMaxCluster;
  a.per = 0;
  a.piece = 0;
  a.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->target_logits) &&
           aligned16(d->draft_logits);
  mark(events, 0, stream);
  cudaError_t e = cudaSuccess;
  if (chunked) {
    // the chunk pass over both rows of every slot on every SM, then the
    // walk, the residual parts and the draw
    ChunkParams c;
    c.target = d->target_logits;
    c.draft = d->draft_logits;
    c.draft_tokens = d->draft_tokens;
    c.part = (float2 *)(ws + L.off_part);
    c.xlogit = (float *)(ws + L.off_xlogit);
    c.claim = (int *)(ws + L.off_claim);
    c.part4 = nullptr;
    c.zero = (int *)(ws + L.off_count);
    c.n_zero = d->batch;
    c.status = a.status;
    c.vocab = d->vocab;
    c.total_B = d->total_B;
    c.nchunks = L.nchunks;
    c.bulk = a.bulk;
    c.polls = a.polls;
    c.ls = a.ls;
    SampleFinishParams f;
    f.target = d->target_logits;
    f.draft = d->draft_logits;
    f.draft_tokens = d->draft_tokens;
    f.tau = d->tau;
    f.cu_B = d->cu_B;
    f.uniforms = d->uniforms;
    f.part = c.part;
    f.xlogit = c.xlogit;
    f.count = (int *)(ws + L.off_count);
    f.res4 = (float4 *)(ws + L.off_res4);
    f.claim = c.claim;
    f.n_accept = d->n_accept;
    f.token = d->token;
    f.pos = d->pos;
    f.status = a.status;
    f.batch = d->batch;
    f.vocab = d->vocab;
    f.total_B = d->total_B;
    f.B_max = d->B_max;
    f.nchunks = L.nchunks;
    f.bulk = a.bulk;
    f.ls = a.ls;
    bool direct = false;
    e = bf16 ? launch_parts<__nv_bfloat16>(c, stream, &direct) : launch_parts<float>(c, stream, &direct);
    if (e == cudaSuccess && !direct)
      e = bf16 ? launch_chunks<__nv_bfloat16, kModeSample>(c, stream) : launch_chunks<float, kModeSample>(c, stream);
    mark(events, 1, stream);
    if (e == cudaSuccess)
      e = bf16 ? launch_sample_finish<__nv_bfloat16>(f, stream) : launch_sample_finish<float>(f, stream);
    mark(events, 2, stream);
    return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
  }
  mark(events, 1, stream);
  e = bf16 ? launch<__nv_bfloat16>(a, stream) : launch<float>(a, stream);
  mark(events, 2, stream);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

}  // namespace

int draft_chunk_entries(int esize) { return kStageBytes / esize; }

cudaError_t launch_draft_chunks(const simsd_draft_desc *d, float4 *part4, int *claim,
                                uint32_t *status, int nchunks, cudaStream_t stream) {
  ChunkParams c;
  c.target = nullptr;
  c.draft = d->draft_logits;
  c.draft_tokens = nullptr;
  c.part = nullptr;
  c.xlogit = nullptr;
  c.part4 = part4;
  c.claim = claim;
  c.zero = nullptr;
  c.n_zero = 0;
  c.status = status;
  c.vocab = d->vocab;
  c.total_B = d->total_B;
  c.nchunks = nchunks;
  const int es = d->dtype == SIMSD_BF16 ? 2 : 4;
  c.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->draft_logits);
  c.polls = kWaitPolls;
  c.ls = scale_of(d->temperature > 0.f ? (double)d->temperature : 1.0);
  return d->dtype == SIMSD_BF16 ? launch_chunks<__nv_bfloat16, kModeDraft>(c, stream)
                                : launch_chunks<float, kModeDraft>(c, stream);
}

}  // namespace simsd

using namespace simsd;

extern "C" {

size_t simsd_accept_workspace_size(const simsd_accept_desc *d) {
  if (accept_check(d) != SIMSD_OK) return 0;
  return accept_workspace(d);
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
  return run_accept(d, (char *)d->workspace, d->workspace_bytes, (cudaStream_t)stream_ptr, events);
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
  return run_accept(d, ws, SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES, (cudaStream_t)stream_ptr, nullptr);
}

}  // extern "C"
