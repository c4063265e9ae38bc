// attn_tc.cu -- K2 (bf16) on the 5th-generation tensor cores (tcgen05).
//
// SimSD section 2 "Temporal Attention Mask" and section 4 (one verification
// forward): every new row attends to the whole prompt; a slot row D~_i also
// to D_j with tau(j) < tau(i) and to D~_j with tau(j) >= tau(i); a data row
// D_i (convention) to D_j with tau(j) <= tau(i).  The mask is evaluated on
// the fly, only on blocks that reach the 2B new keys.
//
// One CTA per (key split, KV head x 128-row tile, sequence).  The query tile
// stacks the 2B tokens x G query heads of one KV head (row = token*G + head
// in group; rows past 2B*G are zero padding), so each key/value byte read
// from HBM serves every row.  The CTA's keys come in 64-key blocks dealt
// alternately to two independent streams, each with its own score tile S,
// two probability tiles P (so a stream's next softmax never waits for its
// previous P.V) and output accumulator O (and running max / sum); the two
// are merged in the epilogue.  Warp roles:
//   warp 0     TMA producer: K and V of each block (4 pages, one 2 KB box
//              per page and 64-column half, 128-byte swizzle) into a
//              5-stage ring;
//   warp 1     TMEM owner and MMA issuer (one thread): S = Q K^T into the
//              stream's TMEM tile (128 x 64 fp32), O += P V into the stream's
//              TMEM accumulator (128 x hd fp32); completion by commit;
//   warps 2-5  softmax of stream 0, warps 6-9 of stream 1, one thread per
//              query row: S from TMEM, scale, mask, running max with an 8
//              (log2) headroom -- O is rescaled in TMEM only when a row's
//              maximum outgrows it, which keeps the result exact (O and l
//              share the stale reference) -- and P as bf16 into a 128-byte
//              swizzled shared tile.
// Q lives in TMEM as the score MMA's A operand (loaded once by the stream-0
// softmax warps, a row per thread), which leaves shared memory to the P
// tiles and a 5-stage K/V ring.
// Every mbarrier wait is bounded; a wait that runs out sets the status word
// and the CTA drains and returns.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace simsd {
namespace {

constexpr int kRows = 128;           // query rows per CTA: the MMA's M
constexpr int kKeys = 64;            // keys per block: S width, P.V depth
constexpr int kPagesPerBlock = kKeys / kPage;
constexpr int kStages = 5;
constexpr int kStreams = 2;
constexpr int kWarps = 2 + 4 * kStreams;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kColO = kStreams * kKeys;   // O accumulators after the S tiles
constexpr int kBoxBytes = kPage * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kHeadroom = 8.f;     // log2 units a row max may grow before O is rescaled

constexpr int kPBufs = 2;            // P tiles per stream (double buffered)

enum { kBarKvFull = 0, kBarKvEmpty = kBarKvFull + kStages, kBarSFull = kBarKvEmpty + kStages,
       kBarSEmpty = kBarSFull + kStreams, kBarPFull = kBarSEmpty + kStreams,
       kBarPvDone = kBarPFull + kStreams * kPBufs, kBarQReady = kBarPvDone + kStreams * kPBufs,
       kNumBars = kBarQReady + 1 };

template <int HD>
struct TcSmem {
  static constexpr int kHalves = HD / 64;
  static constexpr int kHalfRows = kRows * 128;        // one 64-column half of a 128-row tile
  static constexpr int kP = kHalfRows;                  // 64 keys: one half
  static constexpr int kKvHalf = kKeys * 128;           // 64 keys x 64 columns
  static constexpr int kKv = kHalves * kKvHalf;         // K or V tile of a block
  static constexpr int kStage = 2 * kKv;
  static constexpr int kOffP = 0;                       // kStreams x kPBufs tiles
  static constexpr int kOffKv = kOffP + kStreams * kPBufs * kP;
  static constexpr int kOffBar = kOffKv + kStages * kStage;
  static constexpr int kOffTau = kOffBar + kNumBars * 8;
  static constexpr int kOffMl = kOffTau + 2 * kMaxB * 4;    // stream 1's (m, l) per row
  static constexpr int kOffMisc = kOffMl + kRows * 8;       // tmem address, error flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;              // 1024-byte alignment slack
  static constexpr uint32_t kColQ = kColO + kStreams * HD;  // Q: hd bf16 = hd/2 columns
  static constexpr uint32_t kTmemCols = (kColQ + HD / 2) <= 256 ? 256 : 512;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..7) of `row` in a 128-byte
  // swizzled tile whose base is 1024-byte aligned
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// 2^x on the MUFU (approximate; subnormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Visibility of key `key` (0..Lk-1) for a new row (token index tok of the
// 2B, slot row or data row, step label ti); tau of the new tokens in tau_s.
__device__ __forceinline__ bool visible(int key, int P, int B, const int *tau_s, bool row_slot,
                                        int ti) {
  if (key < P) return true;
  const int jj = key - P;
  const int tj = tau_s[jj];
  const bool key_slot = jj >= B;
  return row_slot ? (key_slot ? tj >= ti : tj < ti) : (!key_slot && tj <= ti);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ AttnParams a) {
  using L = TcSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sb = smem_raw + (base - raw);
  const uint32_t sP = base + L::kOffP, sKv = base + L::kOffKv;
  auto bar = [&](int i) { return base + L::kOffBar + 8u * i; };
  int *tau_s = reinterpret_cast<int *>(sb + L::kOffTau);
  float2 *ml_s = reinterpret_cast<float2 *>(sb + L::kOffMl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + L::kOffMisc);
  int *flag_s = reinterpret_cast<int *>(sb + L::kOffMisc + 4);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y % a.Hkv;
  const int rtile = blockIdx.y / a.Hkv;
  const int b = blockIdx.z;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int P = __ldg(a.lens + b);
  const int Lk = P + 2 * B;
  if (B < 1 || B > kMaxSection || P < 0 || (long)Lk > (long)a.max_pages_per_seq * kPage) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) raise_status(a.status, kStatusBadInput);
    return;
  }
  const int M = 2 * B * a.G;
  const int row0 = rtile * kRows;
  const int k_begin = split * a.chunk;
  if (row0 >= M || k_begin >= Lk) return;   // uniform: nothing to do here
  const int k_end = min(Lk, k_begin + a.chunk);
  const int n_blocks = (k_end - k_begin + kKeys - 1) / kKeys;
  const int n_splits_b = (Lk + a.chunk - 1) / a.chunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();                         // the split merge may be scheduled

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), 1);
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    for (int i = 0; i < kStreams; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), 4);
    }
    for (int i = 0; i < kStreams * kPBufs; ++i) {
      mbar_init(bar(kBarPFull + i), 4);
      mbar_init(bar(kBarPvDone + i), 1);
    }
    mbar_init(bar(kBarQReady), 4 * kStreams + 1);
    *flag_s = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc::relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (warp != 0) {
    // tau, the P tiles zeroed once (padding rows are never written again),
    // and Q into TMEM -- one row per thread of the stream-0 softmax warps,
    // two bf16 per column -- while the producer already streams K and V;
    // then arrive on the Q barrier
    const int t = threadIdx.x - 32, nt = kThreads - 32;
    for (int j = t; j < 2 * B; j += nt) tau_s[j] = __ldg(a.tau + c0 + (j < B ? j : j - B));
    for (int e = t; e < kStreams * kPBufs * L::kP / 16; e += nt)
      reinterpret_cast<uint4 *>(sb + L::kOffP)[e] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp >= 2 && warp < 6) {
      grid_dep_wait();                       // rotated q comes from the rotation kernel
      const int q4 = warp & 3, r = 32 * q4 + lane, grow = row0 + r;
      const uint4 *qrow = nullptr;
      if (grow < M)
        qrow = reinterpret_cast<const uint4 *>((const __nv_bfloat16 *)a.q_rot +
                                               ((2L * c0 + grow / a.G) * a.Hq + kvh * a.G + grow % a.G) * HD);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {     // 64 bf16 = 32 columns per store
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 v = qrow ? __ldg(qrow + 8 * c + e) : make_uint4(0, 0, 0, 0);
          w[4 * e] = v.x; w[4 * e + 1] = v.y; w[4 * e + 2] = v.z; w[4 * e + 3] = v.w;
        }
        tc::st32(tmem + ((uint32_t)(32 * q4) << 16) + L::kColQ + 32 * c, w);
      }
      tc::wait_st();
      tc::fence_before_sync();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarQReady));
    // every consumer needs the whole Q tile, tau and zeroed P tiles
    if (!mbar_wait_warp(bar(kBarQReady), 0)) {
      if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
    }
  }

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) { prefetch_tmap(&tmK); prefetch_tmap(&tmV); }
    const int32_t *bt = a.block_table + (long)b * a.max_pages_per_seq;
    int issued = 0;
    bool dep_done = false;
    for (int j = 0; j < n_blocks; ++j) {
      const int s = j % kStages;
      const int kb = k_begin + j * kKeys;
      if (!dep_done && kb + kKeys > P) {     // the block holds new keys K1 writes
        grid_dep_wait();
        dep_done = true;
      }
      const int n_pages = (min(kKeys, k_end - kb) + kPage - 1) / kPage;
      const int page = lane < n_pages ? __ldg(bt + kb / kPage + lane) : 0;   // before the wait
      if (j >= kStages && !mbar_wait_warp(bar(kBarKvEmpty + s), ((j / kStages) - 1) & 1)) {
        if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar(kBarKvFull + s), n_pages * L::kHalves * 2 * kBoxBytes);
      __syncwarp();
      if (lane < n_pages) {
        const uint32_t kt = sKv + s * L::kStage, vt = kt + L::kKv;
#pragma unroll
        for (int hh = 0; hh < L::kHalves; ++hh) {
          const uint32_t off = hh * L::kKvHalf + lane * kBoxBytes;
          tma_load_4d(kt + off, &tmK, bar(kBarKvFull + s), hh * 64, 0, kvh, page);
          tma_load_4d(vt + off, &tmV, bar(kBarKvFull + s), hh * 64, 0, kvh, page);
        }
      }
      issued = j + 1;
    }
    if (*(volatile int *)flag_s) {
      // let copies already in flight land before the CTA can exit
      for (int j = max(0, issued - kStages); j < issued; ++j)
        (void)mbar_wait_warp(bar(kBarKvFull + j % kStages), (j / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // One thread schedules both MMA kinds as their inputs become ready, so
    // a P.V never waits behind a later block's K load: S of block ns needs
    // its K/V stage and its stream's score tile free; P.V of block np needs
    // its P tile.  P.V goes in block order.
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kRows, kKeys, 0);
      constexpr uint32_t idO = tc::idesc_bf16(kRows, HD, 1);
      int ns = 0, np = 0;
      uint32_t idle = 0;
      while (np < n_blocks) {
        bool progressed = false;
        if (ns < n_blocks) {
          const int s = ns % kStages, st = ns & 1;
          if (mbar_test(bar(kBarKvFull + s), (ns / kStages) & 1) &&
              (ns < kStreams || mbar_test(bar(kBarSEmpty + st), ((ns >> 1) - 1) & 1))) {
            tc::fence_after_sync();
            const uint32_t kt = sKv + s * L::kStage;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const uint32_t ka = kt + (kk >> 2) * L::kKvHalf + (kk & 3) * 32;
              tc::mma_bf16_ts(tmem + st * kKeys, tmem + L::kColQ + kk * 8,
                              tc::smem_desc_sw128(ka, 16, 1024), idS, kk > 0);
            }
            tc::commit(bar(kBarSFull + st));
            ++ns;
            progressed = true;
          }
        }
        if (np < ns) {
          const int st = np & 1, s = np % kStages;
          const int ib = np >> 1;                 // block index within the stream
          const int pb = st * kPBufs + (ib & 1);  // its P tile
          if (mbar_test(bar(kBarPFull + pb), (ib >> 1) & 1)) {
            tc::fence_after_sync();
            const int kb = k_begin + np * kKeys;
            const int valid = min(kKeys, k_end - kb);
            const int loaded = (valid + kPage - 1) & ~(kPage - 1);
            const uint32_t vt = sKv + s * L::kStage + L::kKv;
            if (kb + valid == Lk && loaded > valid) {
              // slots past the sequence end in its last page hold arbitrary
              // data; P is 0 there, but 0 * NaN would poison O: zero V rows
              constexpr int CH = HD / 8;
              for (int e = 0; e < (loaded - valid) * CH; ++e) {
                const int r = valid + e / CH, c = e % CH;
                *reinterpret_cast<uint4 *>(sb + (vt - base) + (c >> 3) * L::kKvHalf + swz(r, c & 7)) =
                    make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
            }
            const uint32_t pt = sP + pb * L::kP;
            for (int kk = 0; kk < loaded / 16; ++kk)
              tc::mma_bf16(tmem + kColO + st * HD, tc::smem_desc_sw128(pt + kk * 32, 16, 1024),
                           tc::smem_desc_sw128(vt + kk * 2048, L::kKvHalf, 1024), idO,
                           (np >= kStreams || kk > 0));
            tc::commit(bar(kBarPvDone + pb));
            tc::commit(bar(kBarKvEmpty + s));
            ++np;
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > (kWaitPolls << 4)) {  // bounded: give up, flag, drain
          raise_status(a.status, kStatusTimeout);
          atomicOr(flag_s, 1);
          break;
        }
      }
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int st = (warp - 2) >> 2;          // stream of this warpgroup
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = 32 * q4 + lane;            // query row within the tile
    const int grow = row0 + r;
    const bool row_valid = grow < M;
    const bool warp_valid = row0 + 32 * q4 < M;
    const int tok = row_valid ? grow / a.G : 0;
    const bool row_slot = tok >= B;
    const int row_tau = tau_s[tok];
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t tS = trow + st * kKeys, tO = trow + kColO + st * HD;
    const float scale = a.sm_scale * kLog2e;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    int i = 0;                               // blocks of this stream so far
    for (int j = st; j < n_blocks; j += kStreams, ++i) {
      if (!mbar_wait_warp(bar(kBarSFull + st), i & 1)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sr[kKeys];
      if (warp_valid) {
        tc::ld32(tS, sr);
        tc::ld32(tS + 32, sr + 32);
        tc::wait_ld();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + st));
      const int kb = k_begin + j * kKeys;
      float mx = -INFINITY;                  // block max of the raw scores
      if (warp_valid) {
        if (kb + kKeys > min(P, k_end)) {
          // the block reaches past the prompt or the split's end: mask it
          uint64_t vis = 0;
          for (int c = 0; c < kKeys; ++c) {
            const int key = kb + c;
            if (key < k_end && visible(key, P, B, tau_s, row_slot, row_tau)) vis |= 1ull << c;
          }
#pragma unroll
          for (int c = 0; c < kKeys; ++c)
            if (!((vis >> c) & 1ull)) sr[c] = __float_as_uint(-INFINITY);
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kKeys; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sr[c]));
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale;   // scale > 0
      }
      // reference maximum: moves only when this block's max outgrows it
      const bool move = row_valid && mx > m_ref + kHeadroom;
      const float m_new = move ? mx : m_ref;
      const float alpha = move ? ex2(m_ref - m_new) : 1.f;     // m_ref = -inf -> 0
      const int pb = st * kPBufs + (i & 1);
      if (i >= kPBufs) {
        // the P.V that read this P tile two blocks ago must be done
        if (!mbar_wait_warp(bar(kBarPvDone + pb), ((i >> 1) - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
      }
      if (i > 0 && __any_sync(0xffffffffu, move)) {
        // rescaling O needs the stream's previous P.V (the latest) done
        const int pp = st * kPBufs + ((i - 1) & 1);
        if (!mbar_wait_warp(bar(kBarPvDone + pp), ((i - 1) >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        {
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tc::ld32(tO + 32 * c, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st32(tO + 32 * c, o);
          }
          tc::wait_st();
        }
      }
      l *= alpha;
      m_ref = m_new;
      if (row_valid) {
        // P row (bf16) into the swizzled tile: keys are the K dimension
        // p = 2^(s * scale - m_ref): one fma and the MUFU per score
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        uint8_t *prow = sb + L::kOffP + pb * L::kP;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kKeys / 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = ex2(fmaf(__uint_as_float(sr[8 * c + 2 * e]), scale, -mu));
            const float p1 = ex2(fmaf(__uint_as_float(sr[8 * c + 2 * e + 1]), scale, -mu));
            rs4[e] += p0 + p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4 *>(prow + swz(r, c)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + pb));
    }
    if (ok && i > 0 &&
        !mbar_wait_warp(bar(kBarPvDone + st * kPBufs + ((i - 1) & 1)), ((i - 1) >> 1) & 1))
      ok = false;
    if (!ok && lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
    tc::fence_after_sync();
    // -------------------------------------------------------- epilogue
    // stream 1 hands its (m, l) to stream 0, which merges the two O tiles
    if (st == 1) ml_s[r] = make_float2(m_ref, l);
    tc::fence_before_sync();                 // stream 1's O reads/waits before the sync
    named_sync(1, 4 * kStreams * 32);
    tc::fence_after_sync();
    const bool failed = *(volatile int *)flag_s != 0;
    if (st == 0 && warp_valid) {
      const bool has1 = n_blocks > 1;        // stream 1 saw at least one block
      const float2 ml1 = has1 ? ml_s[r] : make_float2(-INFINITY, 0.f);
      const float mm = fmaxf(m_ref, ml1.x);
      const float mu = mm == -INFINITY ? 0.f : mm;
      const float f0 = exp2f(m_ref - mu), f1 = has1 ? exp2f(ml1.x - mu) : 0.f;
      const float lt = l * f0 + ml1.y * f1;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const long orow = (2L * c0 + tok) * a.Hq + kvh * a.G + (row_valid ? grow % a.G : 0);
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o0[32], o1[32];
        tc::ld32(trow + kColO + 32 * c, o0);
        if (has1) tc::ld32(trow + kColO + HD + 32 * c, o1);
        tc::wait_ld();
        if (!row_valid || failed) continue;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          v[e] = __uint_as_float(o0[e]) * f0 + (has1 ? __uint_as_float(o1[e]) * f1 : 0.f);
        if (n_splits_b == 1) {
          uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)a.out + orow * HD + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(pack_bf16x2(v[8 * e] * inv, v[8 * e + 1] * inv),
                                pack_bf16x2(v[8 * e + 2] * inv, v[8 * e + 3] * inv),
                                pack_bf16x2(v[8 * e + 4] * inv, v[8 * e + 5] * inv),
                                pack_bf16x2(v[8 * e + 6] * inv, v[8 * e + 7] * inv));
        } else {
          const long prow = (long)split * a.T * a.Hq + orow;
          float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * HD + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          if (c == 0) a.ml_part[prow] = make_float2(mm, lt);
        }
      }
    }
  }
  // -------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(tmem, L::kTmemCols);
  }
}

static_assert(TcSmem<128>::kAlloc <= 227 * 1024, "shared memory budget");

template <int HD>
cudaError_t launch_hd(const CUtensorMap &mk, const CUtensorMap &mv, const AttnParams &a,
                      dim3 grid, cudaStream_t stream) {
  auto kern = attn_tc_kernel<HD>;
  const int smem = TcSmem<HD>::kAlloc;
  static std::atomic<uint64_t> configured{0};   // one bit per device
  const int dev = current_device();
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, mk, mv, a);
}

}  // namespace

cudaError_t launch_attn_tc(const simsd_verify_desc *d, const VerifyPlan &p,
                           const AttnParams &a, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, d->k_cache, d->num_pages, d->num_kv_heads, d->head_dim) ||
      !make_cache_map(&mv, d->v_cache, d->num_pages, d->num_kv_heads, d->head_dim))
    return cudaErrorInvalidValue;
  dim3 grid(p.n_splits, d->num_kv_heads * p.row_tiles, d->batch);
  if (d->head_dim == 128) return launch_hd<128>(mk, mv, a, grid, stream);
  return launch_hd<64>(mk, mv, a, grid, stream);
}

}  // namespace simsd
