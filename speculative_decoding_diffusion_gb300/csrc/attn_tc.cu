// attn_tc.cu -- K2 (bf16) on the 5th-generation tensor cores (tcgen05).
//
// SimSD section 2 "Temporal Attention Mask" and section 4 (one verification
// forward): every new row attends to the whole prompt; a slot row D~_i also
// to D_j with tau(j) < tau(i) and to D~_j with tau(j) >= tau(i); a data row
// D_i (convention) to D_j with tau(j) <= tau(i).  Each softmax thread
// builds its row's visibility of the 2B new keys once, as a bitmask; only
// blocks that reach the new keys (or the split's end) apply it.
//
// One CTA per (key split, KV head x 128-row tile, sequence).  The query tile
// stacks the 2B tokens x G query heads of one KV head (row = token*G + head
// in group; rows past 2B*G are zero padding), so each key/value byte read
// from HBM serves every row.  Keys come in 128-key blocks: an MMA
// instruction costs nearly the same at N = 64 as at N = 128, so wide score
// tiles halve the instructions per key.  Warp roles:
//   warps 0, 6 TMA producers: K (warp 0) and V (warp 6) of each block (8
//              pages, one 2 KB box per page and 64-column half, 128-byte
//              swizzle) into a 3-stage ring whose K and V halves are freed
//              separately -- a K half once the block's S = Q K^T is done,
//              so the next K copies start while the block's softmax and
//              P.V still run;
//   warp 1     TMEM owner and MMA issuer (one thread, never blocking on one
//              barrier): S = Q K^T into one of two TMEM score tiles (128 x
//              128 fp32), O += P V into the TMEM accumulator (128 x hd fp32)
//              with P read from TMEM as the A operand; completion by commit;
//   warps 2-5  softmax, one thread per query row: S from TMEM (a max pass,
//              then an exponent pass), scale, mask, running max with an 8
//              (log2) headroom -- O is rescaled in TMEM only when a row's
//              maximum outgrows it, which keeps the result exact (O and l
//              share the stale reference) -- and P as bf16 written back
//              over the score tile it came from.  Warps whose rows are all
//              padding sit out the key loop.
// Q lives in TMEM as the score MMA's A operand: the softmax warps rotate the
// raw queries themselves (a cos/sin table for the section's B positions in
// shared memory), so the kernel waits for the cache append only before the
// block holding the new keys.  Every mbarrier wait is
// bounded; a wait that runs out sets the status word and the CTA drains and
// returns.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "rope.cuh"
#include "tc.cuh"

namespace simsd {
namespace {

constexpr int kRows = 128;           // query rows per CTA: the MMA's M
constexpr int kKeys = 128;           // keys per block: S width, P.V depth
static_assert(kKeys == kBlockKeys, "split chunks are whole blocks");
constexpr int kStages = 3;
constexpr int kWarps = 7;                // producer K, MMA, 4 softmax, producer V
constexpr int kVWarp = 6;
constexpr int kThreads = kWarps * 32;
constexpr int kSoftmax = 4 * 32;     // softmax threads (warps 2-5)
constexpr int kBoxBytes = kPage * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kHeadroom = 8.f;     // log2 units a row max may grow before O is rescaled
constexpr uint32_t kColS = 0;        // two score / probability tiles: columns 0 and kKeys
constexpr uint32_t kColO = 2 * kKeys;

enum { kBarKFull = 0, kBarVFull = kBarKFull + kStages, kBarKEmpty = kBarVFull + kStages,
       kBarVEmpty = kBarKEmpty + kStages, kBarSFull = kBarVEmpty + kStages,
       kBarPFull = kBarSFull + 2, kBarPvDone = kBarPFull + 2,
       kBarQReady = kBarPvDone + 2, kNumBars = kBarQReady + 1 };

template <int HD>
struct TcSmem {
  static constexpr int kHalves = HD / 64;
  static constexpr int kKvHalf = kKeys * 128;           // 128 keys x 64 columns
  static constexpr int kKv = kHalves * kKvHalf;         // K or V tile of a block
  static constexpr int kStage = 2 * kKv;
  static constexpr int kOffKv = 0;
  static constexpr int kOffBar = kOffKv + kStages * kStage;
  static constexpr int kOffTau = kOffBar + kNumBars * 8;
  static constexpr int kOffCs = kOffTau + 2 * kMaxB * 4;     // [kMaxB][HD/2] (cos, sin)
  static constexpr int kOffMisc = kOffCs + kMaxB * (HD / 2) * 8;  // tmem address, error flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;              // 1024-byte alignment slack
  static constexpr uint32_t kColQ = kColO + HD;             // Q: hd bf16 = hd/2 columns
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColQ + HD / 2 <= kTmemCols, "TMEM budget");
  static_assert(4 * 32 * (HD + 4) * 4 <= kStages * kStage, "epilogue exchange fits the ring");
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

template <int V> struct IntC { static constexpr int value = V; };

// Word i (a compile-time constant after unrolling) of a 16-byte vector.
__device__ __forceinline__ uint32_t word4(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Visibility of new key jj (0..2B-1 past the prompt) for a new row (slot row
// or data row, step label ti); tau of the new tokens in tau_s.
__device__ __forceinline__ bool visible_new(int jj, int B, const int *tau_s, bool row_slot,
                                            int ti) {
  const int tj = tau_s[jj];
  const bool key_slot = jj >= B;
  return row_slot ? (key_slot ? tj >= ti : tj < ti) : (!key_slot && tj <= ti);
}

// bits [0, n) set (n clamped to 0..64)
__device__ __forceinline__ uint64_t low_bits(int n) {
  return n <= 0 ? 0ull : n >= 64 ? ~0ull : (1ull << n) - 1ull;
}
// x >> s for any s (negative: shift left); shifts of 64 or more give 0
__device__ __forceinline__ uint64_t shift_bits(uint64_t x, int s) {
  return s >= 64 || s <= -64 ? 0ull : s >= 0 ? x >> s : x << (-s);
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
  const uint32_t sKv = base + L::kOffKv;
  auto bar = [&](int i) { return base + L::kOffBar + 8u * i; };
  int *tau_s = reinterpret_cast<int *>(sb + L::kOffTau);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + L::kOffMisc);
  int *flag_s = reinterpret_cast<int *>(sb + L::kOffMisc + 4);

  // unit (sequence, KV head, row tile) and split of this CTA: units from
  // tail_from on run in s_tail splits of chunk_tail keys, the ones before
  // whole.  The split units' CTAs come last in the grid (they even out the
  // last wave), or first when the plan says so (tail_first: few full
  // waves, where their SMs then run the whole units offset by a split, so
  // the SMs' ramps at unit boundaries -- query rows, first copies -- no
  // longer fall at the same time and DRAM stays busy through them).
  const int ci = blockIdx.x;
  const int n_tail = (int)gridDim.x - a.tail_from;   // CTAs of split units
  const bool tail = a.tail_first ? ci < n_tail : ci >= a.tail_from;
  const int ti = a.tail_first ? ci : ci - a.tail_from;   // index among the split CTAs
  const int unit = tail ? a.tail_from + ti / a.s_tail : (a.tail_first ? ci - n_tail : ci);
  const int split = tail ? ti % a.s_tail : 0;
  const int chunk = tail ? a.chunk_tail : a.max_pages_per_seq * kPage;
  const int per_seq = a.Hkv * a.row_tiles;
  const int b = unit / per_seq;
  const int kvh = unit % per_seq % a.Hkv;
  const int rtile = unit % per_seq / a.Hkv;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int P = __ldg(a.lens + b);
  const int Lk = P + 2 * B;
  if (B < 1 || B > kMaxSection || B > a.B_max || c0 < 0 || c0 + B > a.total_B || P < 0 ||
      (long)Lk > (long)a.max_pages_per_seq * kPage ||
      (a.node_size > 0 && (2 * B) % a.node_size != 0)) {
    if (threadIdx.x == 0 && split == 0 && unit % per_seq == 0) raise_status(a.status, kStatusBadInput);
    return;
  }
  const int M = 2 * B * a.G;
  const int row0 = rtile * kRows;
  const int k_begin = split * chunk;
  if (row0 >= M || k_begin >= Lk) return;   // uniform: nothing to do here
  const int k_end = min(Lk, k_begin + chunk);
  const int n_blocks = (k_end - k_begin + kKeys - 1) / kKeys;
  const int n_splits_b = (Lk + chunk - 1) / chunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // copies of the tile's rows across the four TMEM lane quadrants (4 when
  // one 32-row group holds every real row, 2 for two groups, else 1), and
  // the softmax warps that own real rows (the others hold padding only)
  const int n_groups = min(4, (M - row0 + 31) / 32);
  const int R = n_groups == 1 ? 4 : n_groups == 2 ? 2 : 1;
  const int n_valid = R > 1 ? 4 : n_groups;
  grid_dep_launch();                         // the split merge may be scheduled
  // Producer lane i copies page i of a block (both halves of K and V).  The
  // page ids of the first kStages blocks are requested before the setup
  // below, later ones kStages blocks ahead into the same register slot
  // (the loop is unrolled by kStages: no register is moved while its load
  // is in flight), so no copy waits for a block-table round trip.
  const int32_t *bt = a.block_table + (long)b * a.max_pages_per_seq;
  auto block_page = [&](int jj) {
    if (jj >= n_blocks) return 0;
    const int kb = k_begin + jj * kKeys;
    return lane < (min(kKeys, k_end - kb) + kPage - 1) / kPage ? __ldg(bt + kb / kPage + lane) : 0;
  };
  int pages[kStages];
  if (warp == 0 || warp == kVWarp) {
    if (lane == 0) prefetch_tmap(warp == 0 ? &tmK : &tmV);
#pragma unroll
    for (int d = 0; d < kStages; ++d) pages[d] = block_page(d);
  }
  // softmax threads request their raw query row first, ahead of the K/V
  // stream the producer starts below (each thread one row of the tile)
  uint4 qv[HD / 8];
  const bool softmax_warp = warp >= 2 && warp < 6;
  if (softmax_warp) {
    const int qg = (warp & 3) % (4 / R), qrow_i = row0 + 32 * qg + lane;
    if (qrow_i < M) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          (const __nv_bfloat16 *)a.q + ((2L * c0 + qrow_i / a.G) * a.Hq + kvh * a.G + qrow_i % a.G) * HD);
#pragma unroll
      for (int e = 0; e < HD / 8; ++e) qv[e] = __ldg(src + e);
    } else {
#pragma unroll
      for (int e = 0; e < HD / 8; ++e) qv[e] = make_uint4(0, 0, 0, 0);
    }
  }
  // the section's step labels (softmax thread j < 2B: tau of new token j),
  // requested with the query rows, before the producer's copies fill the
  // memory system
  const int tsm = threadIdx.x - 64;
  const int tau_j = softmax_warp && a.node_size == 0 && tsm < 2 * B
                        ? __ldg(a.tau + c0 + (tsm < B ? tsm : tsm - B)) : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarKEmpty + i), 1);
      mbar_init(bar(kBarVEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarPFull + i), n_valid);
      mbar_init(bar(kBarPvDone + i), 1);
    }
    mbar_init(bar(kBarQReady), 4);
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
  int issued = 0;                            // producers: blocks whose loads were started

  if (warp == 0 || warp == kVWarp) {
    // --------------------------------------------------------- producers
    // warp 0 copies K, warp kVWarp copies V, each into its half of the
    // stage once the MMA issuer has released that half
    const bool kside = warp == 0;
    const CUtensorMap *tm = kside ? &tmK : &tmV;
    const int full0 = kside ? kBarKFull : kBarVFull, empty0 = kside ? kBarKEmpty : kBarVEmpty;
    bool dep_done = false, ok = true;
    for (int j0 = 0; ok && j0 < n_blocks; j0 += kStages) {
#pragma unroll
      for (int u = 0; u < kStages; ++u) {
        const int j = j0 + u;
        if (j >= n_blocks) break;
        const int s = u;                       // j % kStages (j0 is a multiple)
        const int kb = k_begin + j * kKeys;
        if (!dep_done && kb + kKeys > P) {   // the block holds new keys K1 writes
          grid_dep_wait();
          dep_done = true;
        }
        const int n_pages = (min(kKeys, k_end - kb) + kPage - 1) / kPage;
        const int page = pages[u];
        if (j >= kStages && !mbar_wait_warp(bar(empty0 + s), ((j / kStages) - 1) & 1, a.polls)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), n_pages * L::kHalves * kBoxBytes);
        __syncwarp();
        if (lane < n_pages) {
          const uint32_t t0 = sKv + s * L::kStage + (kside ? 0 : L::kKv);
#pragma unroll
          for (int hh = 0; hh < L::kHalves; ++hh)
            tma_load_4d(t0 + hh * L::kKvHalf + lane * kBoxBytes, tm, bar(full0 + s), hh * 64, 0, kvh, page);
        }
        issued = j + 1;
        pages[u] = block_page(j + kStages);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // One thread issues both MMA kinds as their inputs become ready: S of
    // block ns needs its K/V stage and its score tile free (the P.V that
    // read the tile two blocks ago done); P.V of block np needs its P.
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kRows, kKeys, 0);
      constexpr uint32_t idO = tc::idesc_bf16(kRows, HD, 1);
      bool ok = mbar_wait(bar(kBarQReady), 0, a.polls);
      int ns = 0, np = 0;
      uint64_t idle = 0;
      while (ok && np < n_blocks) {
        bool progressed = false;
        if (ns < n_blocks) {
          const int s = ns % kStages, tb = ns & 1;
          if (mbar_test(bar(kBarKFull + s), (ns / kStages) & 1) &&
              (ns < 2 || mbar_test(bar(kBarPvDone + tb), ((ns >> 1) - 1) & 1))) {
            tc::fence_after_sync();
            const uint32_t kt = sKv + s * L::kStage;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
              const uint32_t ka = kt + (kk >> 2) * L::kKvHalf + (kk & 3) * 32;
              tc::mma_bf16_ts(tmem + kColS + tb * kKeys, tmem + L::kColQ + kk * 8,
                              tc::smem_desc_sw128(ka, 16, 1024), idS, kk > 0);
            }
            tc::commit(bar(kBarSFull + tb));
            tc::commit(bar(kBarKEmpty + s));   // the K half is free once S is done
            ++ns;
            progressed = true;
          }
        }
        if (np < ns) {
          const int tb = np & 1, s = np % kStages;
          if (mbar_test(bar(kBarPFull + tb), (np >> 1) & 1) &&
              mbar_test(bar(kBarVFull + s), (np / kStages) & 1)) {
            tc::fence_after_sync();
            const int kb = k_begin + np * kKeys;
            const int valid = min(kKeys, k_end - kb);
            const int loaded = (valid + kPage - 1) & ~(kPage - 1);
            const uint32_t vt = sKv + s * L::kStage + L::kKv;
            for (int kk = 0; kk < loaded / 16; ++kk)
              tc::mma_bf16_ts(tmem + kColO, tmem + kColS + tb * kKeys + kk * 8,
                              tc::smem_desc_sw128(vt + kk * 2048, L::kKvHalf, 1024), idO,
                              (np > 0 || kk > 0));
            tc::commit(bar(kBarPvDone + tb));
            tc::commit(bar(kBarVEmpty + s));
            ++np;
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > ((uint64_t)a.polls << 4)) {  // bounded: give up, flag, drain
          ok = false;
        } else if (idle > 8) {
          // nothing ready for a while (usually: the softmax is on a block):
          // leave the issue slots to the softmax warp sharing this scheduler
          __nanosleep(32);
        }
      }
      if (!ok) {
        raise_status(a.status, kStatusTimeout);
        atomicOr(flag_s, 1);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax
    // With at most 64 real rows the tile's rows are replicated across the
    // four TMEM lane quadrants (R = 4 or 2 copies) and the copies split each
    // block's keys: every quadrant's warp handles 128/R keys of the same
    // rows with its own running reference, and writes P for its keys (zeros
    // elsewhere), so the P.V MMA leaves R partial outputs per row that the
    // epilogue merges to the largest reference.
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int groups = 4 / R;                // 32-row groups held per copy
    const int g = q4 % groups, kp = q4 / groups;
    const int r = 32 * g + lane;             // query row within the tile
    const int grow = row0 + r;
    const bool row_valid = grow < M;
    const bool warp_valid = row0 + 32 * g < M;
    const int tok = row_valid ? grow / a.G : 0;
    const bool row_slot = tok >= B;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    // tau of the section and the (cos, sin) table of its B positions, then
    // Q rotated into TMEM (one row per thread, two bf16 per column, zeros
    // for padding rows); then the issuer may start
    const int t = threadIdx.x - 64;
    const bool graph = a.node_size > 0;        // draft-graph nodes instead of D | D~
    const int npos = graph ? a.node_size : B;  // distinct positions of the new tokens
    float2 *cs_s = reinterpret_cast<float2 *>(sb + L::kOffCs);
    if (!graph)
      if (t < 2 * B) tau_s[t] = tau_j;      // 2B <= 64 <= kSoftmax
    for (int e = t; e < npos * (HD / 2); e += kSoftmax)
      cs_s[e] = rope_cs(a.tab, e % (HD / 2), P + e / (HD / 2));   // D~_k copies D_k's position
    named_sync(1, kSoftmax);
    {
      const int kq = !row_valid ? 0 : graph ? tok % a.node_size : (tok < B ? tok : tok - B);
      const float2 *cs = cs_s + kq * (HD / 2);
#pragma unroll
      for (int d0 = 0; d0 < HD / 2; d0 += 32) {
        // elements d0.. and d0 + hd/2.. of the row: y1 = x1 c - x2 s,
        // y2 = x2 c + x1 s, rounded to bf16 (rotate-half pairing); padding
        // rows are zero and stay zero
        uint32_t w1[16], w2[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t a1 = word4(qv[(d0 >> 3) + (e >> 2)], e & 3);
          const uint32_t a2 = word4(qv[((HD / 2 + d0) >> 3) + (e >> 2)], e & 3);
          const float x1l = __uint_as_float(a1 << 16), x1h = __uint_as_float(a1 & 0xffff0000u);
          const float x2l = __uint_as_float(a2 << 16), x2h = __uint_as_float(a2 & 0xffff0000u);
          const float2 cl = cs[d0 + 2 * e], ch = cs[d0 + 2 * e + 1];
          w1[e] = pack_bf16x2(x1l * cl.x - x2l * cl.y, x1h * ch.x - x2h * ch.y);
          w2[e] = pack_bf16x2(x2l * cl.x + x1l * cl.y, x2h * ch.x + x1h * ch.y);
        }
        tc::st16(trow + L::kColQ + d0 / 2, w1);
        tc::st16(trow + L::kColQ + (HD / 2 + d0) / 2, w2);
      }
      tc::wait_st();
      tc::fence_before_sync();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarQReady));
    // this row's visibility of the 2B new keys (bit jj: new key jj), built
    // while the first K/V stage is still in flight: the temporal mask, or
    // (draft-graph layout) the tokens of the row's own node
    uint64_t newvis = 0;
    if (graph) {
      newvis = low_bits(a.node_size) << ((tok / a.node_size) * a.node_size);
    } else {
      const int row_tau = tau_s[tok];
#pragma unroll 8
      for (int jj = 0; jj < 2 * B; ++jj)
        if (visible_new(jj, B, tau_s, row_slot, row_tau)) newvis |= 1ull << jj;
    }
    const uint32_t tO = trow + kColO;
    const float scale = a.sm_scale * kLog2e;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    int j = 0;
    // the key loop, compiled once per copy count (chunk loops unrolled)
    auto key_loop = [&](auto rc) {
      constexpr int RC = decltype(rc)::value;
      constexpr int KW = kKeys / RC;         // this warp's keys per block
      const int k_lo = kp * KW;
      for (; warp_valid && j < n_blocks; ++j) {
        const int tb = j & 1;
        const uint32_t tS = trow + kColS + tb * kKeys;
        if (!mbar_wait_warp(bar(kBarSFull + tb), (j >> 1) & 1, a.polls)) { ok = false; break; }
        tc::fence_after_sync();
        const int kb = k_begin + j * kKeys;
        // visibility of this warp's keys: prompt keys below the split's end
        // are visible; only blocks that reach the new keys or the end need
        // the bitmask (bit c: key kb + k_lo + c)
        uint64_t vis[(KW + 63) / 64];
#pragma unroll
        for (int h = 0; h < (KW + 63) / 64; ++h) vis[h] = ~0ull;
        if (kb + k_lo + KW > min(P, k_end)) {
          // prompt keys below the split's end, and new keys per newvis
          const int first_new = P - kb - k_lo, kend = k_end - kb - k_lo;
#pragma unroll
          for (int h = 0; h < (KW + 63) / 64; ++h)
            vis[h] = (low_bits(first_new - 64 * h) | shift_bits(newvis, 64 * h - first_new)) &
                     low_bits(kend - 64 * h);
        }
        // pass 1: the maximum of the raw scores over this warp's keys, 64
        // columns per TMEM round trip (the loop stays rolled: an unrolled
        // 128-key body overflows the instruction cache)
        constexpr int CB = KW < 64 ? KW : 64;
        float mx = -INFINITY;
#pragma unroll 1
        for (int ck = 0; ck < KW; ck += CB) {
          uint32_t sr[CB];
          const uint64_t vh = KW > 64 && ck >= 64 ? vis[KW > 64 ? 1 : 0] : vis[0];
#pragma unroll
          for (int q = 0; q < CB; q += 32) tc::ld32(tS + k_lo + ck + q, sr + q);
          tc::wait_ld();
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < CB; ++c) {
            const float v = ((vh >> ((ck & 63) + c)) & 1ull) ? __uint_as_float(sr[c]) : -INFINITY;
            m4[c & 3] = fmaxf(m4[c & 3], v);
          }
          mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
        }
        // (each copy of a replicated row keeps its own reference; the
        // epilogue merges the copies' (O, l, m) like splits)
        mx *= scale;                         // scale > 0
        // reference maximum: moves only when this block's max outgrows it
        const bool move = row_valid && mx > m_ref + kHeadroom;
        const float m_new = move ? mx : m_ref;
        const float alpha = move ? ex2(m_ref - m_new) : 1.f;     // m_ref = -inf -> 0
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          // rescaling O needs the previous block's P.V done
          if (!mbar_wait_warp(bar(kBarPvDone + (tb ^ 1)), ((j - 1) >> 1) & 1, a.polls)) { ok = false; break; }
          tc::fence_after_sync();
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
        l *= alpha;
        m_ref = m_new;
        // pass 2: p = 2^(s * scale - m_ref) as bf16 pairs into P columns
        // k_lo/2 .. (k_lo + KW)/2 of the score tile (the scores there are
        // read already or belong to other copies' keys), zeros in the rest
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int ck = 0; ck < KW; ck += CB) {
          uint32_t sr[CB], pw[CB / 2];
          const uint64_t vh = KW > 64 && ck >= 64 ? vis[KW > 64 ? 1 : 0] : vis[0];
#pragma unroll
          for (int q = 0; q < CB; q += 32) tc::ld32(tS + k_lo + ck + q, sr + q);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < CB / 2; ++e) {
            const int c = (ck & 63) + 2 * e;
            const float s0 = ((vh >> c) & 1ull) ? __uint_as_float(sr[2 * e]) : -INFINITY;
            const float s1 = ((vh >> (c + 1)) & 1ull) ? __uint_as_float(sr[2 * e + 1]) : -INFINITY;
            const float p0 = ex2(fmaf(s0, scale, -mu));
            const float p1 = ex2(fmaf(s1, scale, -mu));
            rs4[e & 3] += p0 + p1;
            pw[e] = pack_bf16x2(p0, p1);
          }
#pragma unroll
          for (int q = 0; q < CB / 2; q += 16) tc::st16(tS + (k_lo + ck) / 2 + q, pw + q);
        }
        if (RC > 1) {
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c = 0; c < kKeys / 2; c += 16)
            if (c < k_lo / 2 || c >= (k_lo + KW) / 2) tc::st16(tS + c, z);
        }
        tc::wait_st();
        l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        {
          // slots past the sequence end in its last page hold arbitrary
          // data; P is 0 there, but 0 * NaN would poison O: zero those V
          // rows (the stage landed before S was computed) before P.V reads
          const int valid = min(kKeys, k_end - kb);
          const int loaded = (valid + kPage - 1) & ~(kPage - 1);
          if (q4 == 0 && kb + valid == Lk && loaded > valid) {
            // the block's V half may still be landing: wait for it first
            if (!mbar_wait_warp(bar(kBarVFull + j % kStages), (j / kStages) & 1, a.polls)) { ok = false; break; }
            constexpr int CH = HD / 8;
            uint8_t *vt = sb + L::kOffKv + (j % kStages) * L::kStage + L::kKv;
            for (int e = lane; e < (loaded - valid) * CH; e += 32) {
              const int rr = valid + e / CH, c = e % CH;
              *reinterpret_cast<uint4 *>(vt + (c >> 3) * L::kKvHalf + swz(rr, c & 7)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + tb));
      }
    };
    if (R == 4) key_loop(IntC<4>{});
    else if (R == 2) key_loop(IntC<2>{});
    else key_loop(IntC<1>{});
    if (ok && j > 0 &&
        !mbar_wait_warp(bar(kBarPvDone + ((j - 1) & 1)), ((j - 1) >> 1) & 1, a.polls))
      ok = false;
    if (!ok && lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
    tc::fence_after_sync();
    // -------------------------------------------------------- epilogue
    const bool failed = *(volatile int *)flag_s != 0;
    const long orow = (2L * c0 + tok) * a.Hq + kvh * a.G + (row_valid ? grow % a.G : 0);
    // writes columns [c0c, c0c + n) of this thread's row from v (O sums,
    // unnormalised, relative to reference mr) with sum lt
    auto write_cols = [&](const float *v, int c0c, int n, float lt, float mr) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      if (n_splits_b == 1) {
        uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)a.out + orow * HD + c0c);
        for (int e = 0; e < n / 8; ++e)
          dst[e] = make_uint4(pack_bf16x2(v[8 * e] * inv, v[8 * e + 1] * inv),
                              pack_bf16x2(v[8 * e + 2] * inv, v[8 * e + 3] * inv),
                              pack_bf16x2(v[8 * e + 4] * inv, v[8 * e + 5] * inv),
                              pack_bf16x2(v[8 * e + 6] * inv, v[8 * e + 7] * inv));
      } else {
        const long prow = (long)split * a.T * a.Hq + orow;
        float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * HD + c0c);
        for (int e = 0; e < n / 4; ++e)
          dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        if (c0c == 0) a.ml_part[prow] = make_float2(mr, lt);   // O, l relative to mr
      }
    };
    if (R == 1) {
      if (warp_valid) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tc::ld32(tO + 32 * c, o);
          tc::wait_ld();
          if (!row_valid || failed) continue;
          write_cols(reinterpret_cast<const float *>(o), 32 * c, 32, l, m_ref);
        }
      }
    } else {
      // every copy puts its partial output, sum and reference in the (now
      // idle) K/V ring; then copy kp merges the R partials of columns
      // [kp * HD/R, ..) to the largest reference
      float *part = reinterpret_cast<float *>(sb + L::kOffKv);   // [R][groups][32][HD + 4]
      float *mine = part + ((kp * groups + g) * 32 + lane) * (HD + 4);
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tc::ld32(tO + 32 * c, o);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<float4 *>(mine + 32 * c + 4 * e) =
              make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                          __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
      }
      mine[HD] = l;
      mine[HD + 1] = m_ref;
      named_sync(1, kSoftmax);
      if (row_valid && !failed) {
        const int cw = HD / R, cb = kp * cw;    // 16, 32 or 64 columns
        float mt = -INFINITY;
        for (int c = 0; c < R; ++c) mt = fmaxf(mt, part[((c * groups + g) * 32 + lane) * (HD + 4) + HD + 1]);
        float wc[4], lt = 0.f;
        for (int c = 0; c < R; ++c) {
          const float *pc = part + ((c * groups + g) * 32 + lane) * (HD + 4);
          wc[c] = mt == -INFINITY ? 0.f : ex2(pc[HD + 1] - mt);   // -inf reference -> 0
          lt += wc[c] * pc[HD];
        }
        for (int q = 0; q < cw; q += 32) {
          const int n = min(32, cw - q);        // a multiple of 16
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
          for (int c = 0; c < R; ++c) {
            const float *src = part + ((c * groups + g) * 32 + lane) * (HD + 4) + cb + q;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (4 * e >= n) break;
              const float4 p4 = *reinterpret_cast<const float4 *>(src + 4 * e);
              v[4 * e] += wc[c] * p4.x; v[4 * e + 1] += wc[c] * p4.y;
              v[4 * e + 2] += wc[c] * p4.z; v[4 * e + 3] += wc[c] * p4.w;
            }
          }
          write_cols(v, cb + q, n, lt, mt);
        }
      }
    }
  }
  // -------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  // after a wait that gave up (any warp's: the flag is final here), the
  // copies still in flight land before the CTA can exit (default limit)
  if ((warp == 0 || warp == kVWarp) && *(volatile int *)flag_s)
    for (int j = max(0, issued - kStages); j < issued; ++j)
      (void)mbar_wait_warp(bar((warp == 0 ? kBarKFull : kBarVFull) + j % kStages), (j / kStages) & 1);
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
  dim3 grid(p.grid);
  if (d->head_dim == 128) return launch_hd<128>(mk, mv, a, grid, stream);
  return launch_hd<64>(mk, mv, a, grid, stream);
}

}  // namespace simsd
