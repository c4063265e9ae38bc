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
// from HBM serves every row.  Warp roles:
//   warp 0     TMA producer: 128-key blocks (8 pages) of K and V, one 2 KB
//              box per page and 64-column half (128-byte swizzle), into a
//              2-stage ring;
//   warp 1     TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into a
//              double-buffered TMEM tile (128 x 128 fp32), O += P_j V_j into
//              a TMEM accumulator (128 x hd fp32); completion by commit;
//   warps 2-5  softmax, one thread per query row: S_j from TMEM, scale,
//              mask, running max with an 8 (log2) headroom -- O is rescaled
//              in TMEM only when a row's maximum outgrows it, which keeps
//              the result exact (O and l share the stale reference) -- P_j as
//              bf16 into a 128B-swizzled shared tile, and the epilogue.
// Q is staged once into shared memory in the same swizzled K-major layout.
// Every mbarrier wait is bounded; a wait that runs out sets the status word
// and the CTA drains and returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace simsd {
namespace {

constexpr int kRows = 128;         // query rows per CTA: the MMA's M
constexpr int kKeys = kBlockKeys;  // keys per block: S width, P.V depth
constexpr int kStages = 2;
constexpr int kWarps = 6;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O [256,256+hd)
constexpr uint32_t kColO = 256;
constexpr int kBoxBytes = kPage * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kHeadroom = 8.f;   // log2 units a row max may grow before O is rescaled

enum { kBarKvFull = 0, kBarKvEmpty = 2, kBarSFull = 4, kBarSEmpty = 6, kBarPFull = 8,
       kBarPvDone = 9, kNumBars = 10 };

template <int HD>
struct TcSmem {
  static constexpr int kHalves = HD / 64;
  static constexpr int kHalfRows = kRows * 128;        // one 64-column half of Q or P
  static constexpr int kQ = kHalves * kHalfRows;
  static constexpr int kP = 2 * kHalfRows;              // 128 keys = two halves
  static constexpr int kKvHalf = kKeys * 128;
  static constexpr int kKv = kHalves * kKvHalf;         // K or V tile of a block
  static constexpr int kStage = 2 * kKv;
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = kOffQ + kQ;
  static constexpr int kOffKv = kOffP + kP;
  static constexpr int kOffBar = kOffKv + kStages * kStage;
  static constexpr int kOffTau = kOffBar + kNumBars * 8;
  static constexpr int kOffMisc = kOffTau + 2 * kMaxB * 4;  // tmem address, error flag
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;              // 1024-byte alignment slack
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..7) of `row` in a 128-byte
  // swizzled half tile whose base is 1024-byte aligned
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
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
  const uint32_t sQ = base + L::kOffQ, sP = base + L::kOffP, sKv = base + L::kOffKv;
  auto bar = [&](int i) { return base + L::kOffBar + 8u * i; };
  int *tau_s = reinterpret_cast<int *>(sb + L::kOffTau);
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), 1);
      mbar_init(bar(kBarKvEmpty + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), 4);
    }
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarPvDone), 1);
    *flag_s = 0;
    fence_barrier_init();
  }
  for (int j = threadIdx.x; j < 2 * B; j += kThreads)
    tau_s[j] = __ldg(a.tau + c0 + (j < B ? j : j - B));
  if (warp == 1) {
    tc::alloc(smem_u32(tmem_slot), kTmemCols);
    tc::relinquish();
  }
  // Q tile -> shared memory, K-major with the 128-byte swizzle
  {
    const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q_rot;
    constexpr int CH = HD / 8;
    for (int e = threadIdx.x; e < kRows * CH; e += kThreads) {
      const int r = e / CH, c = e % CH;
      const int grow = row0 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (grow < M) {
        const long qrow = (2L * c0 + grow / a.G) * a.Hq + kvh * a.G + grow % a.G;
        v = *reinterpret_cast<const uint4 *>(q + qrow * HD + c * 8);
      }
      *reinterpret_cast<uint4 *>(sb + L::kOffQ + (c >> 3) * L::kHalfRows + swz(r, c & 7)) = v;
    }
  }
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) { prefetch_tmap(&tmK); prefetch_tmap(&tmV); }
    const int32_t *bt = a.block_table + (long)b * a.max_pages_per_seq;
    int issued = 0;
    for (int j = 0; j < n_blocks; ++j) {
      const int s = j & 1;
      if (j >= kStages && !mbar_wait_warp(bar(kBarKvEmpty + s), ((j >> 1) - 1) & 1)) {
        if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
        break;
      }
      const int kb = k_begin + j * kKeys;
      const int n_pages = (min(kKeys, k_end - kb) + kPage - 1) / kPage;
      const int page = lane < n_pages ? __ldg(bt + kb / kPage + lane) : 0;
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
        (void)mbar_wait_warp(bar(kBarKvFull + (j & 1)), (j >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = tc::idesc_bf16(kRows, kKeys, 0);
    constexpr uint32_t idO = tc::idesc_bf16(kRows, HD, 1);
    bool ok = true;
    auto fail = [&]() {
      if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
      ok = false;
    };
    auto issue_s = [&](int j) {
      const int s = j & 1;
      if (!mbar_wait_warp(bar(kBarKvFull + s), (j >> 1) & 1)) { fail(); return; }
      if (j >= kStages && !mbar_wait_warp(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1)) { fail(); return; }
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t kt = sKv + s * L::kStage;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t qa = sQ + (kk >> 2) * L::kHalfRows + (kk & 3) * 32;
          const uint32_t ka = kt + (kk >> 2) * L::kKvHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + s * kKeys, tc::smem_desc_sw128(qa, 16, 1024),
                       tc::smem_desc_sw128(ka, 16, 1024), idS, kk > 0);
        }
        tc::commit(bar(kBarSFull + s));
      }
      __syncwarp();
    };
    issue_s(0);
    for (int j = 0; j < n_blocks && ok; ++j) {
      if (j + 1 < n_blocks) {
        issue_s(j + 1);
        if (!ok) break;
      }
      if (!mbar_wait_warp(bar(kBarPFull), j & 1)) { fail(); break; }
      tc::fence_after_sync();
      const int s = j & 1;
      const int kb = k_begin + j * kKeys;
      const int valid = min(kKeys, k_end - kb);
      const int loaded = (valid + kPage - 1) & ~(kPage - 1);
      const uint32_t vt = sKv + s * L::kStage + L::kKv;
      if (kb + valid == Lk && loaded > valid) {
        // slots past the sequence end in its last page hold arbitrary data;
        // P is 0 there, but 0 * NaN would poison O, so zero the V rows
        constexpr int CH = HD / 8;
        for (int e = lane; e < (loaded - valid) * CH; e += 32) {
          const int r = valid + e / CH, c = e % CH;
          *reinterpret_cast<uint4 *>(sb + (vt - base) + (c >> 3) * L::kKvHalf + swz(r, c & 7)) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        for (int kk = 0; kk < loaded / 16; ++kk) {
          const uint32_t pa = sP + (kk >> 2) * L::kHalfRows + (kk & 3) * 32;
          const uint32_t va = vt + kk * 2048;
          tc::mma_bf16(tmem + kColO, tc::smem_desc_sw128(pa, 16, 1024),
                       tc::smem_desc_sw128(va, L::kKvHalf, 1024), idO, (j > 0 || kk > 0));
        }
        tc::commit(bar(kBarPvDone));
        tc::commit(bar(kBarKvEmpty + s));
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int q4 = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = 32 * q4 + lane;            // query row within the tile
    const int grow = row0 + r;
    const bool row_valid = grow < M;
    const int tok = row_valid ? grow / a.G : 0;
    const bool row_slot = tok >= B;
    const int row_tau = tau_s[tok];
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const float scale = a.sm_scale * kLog2e;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_blocks; ++j) {
      const int s = j & 1;
      if (!mbar_wait_warp(bar(kBarSFull + s), (j >> 1) & 1)) {
        if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sr[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) tc::ld32(trow + s * kKeys + 32 * c, sr + 32 * c);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + s));
      const int kb = k_begin + j * kKeys;
      const bool no_mask = kb + kKeys <= min(P, k_end);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        float v = __uint_as_float(sr[c]) * scale;
        if (!no_mask) {
          const int key = kb + c;
          bool vis = key < k_end;
          if (vis && key >= P) {
            const int jj = key - P;            // 0..2B-1 among the new tokens
            const int tj = tau_s[jj];
            const bool key_slot = jj >= B;
            vis = row_slot ? (key_slot ? tj >= row_tau : tj < row_tau)
                           : (!key_slot && tj <= row_tau);
          }
          if (!vis) v = -INFINITY;
        }
        sr[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
      // reference maximum: moves only when this block's max outgrows it
      const bool move = row_valid && mx > m_ref + kHeadroom;
      const float m_new = move ? mx : m_ref;
      const float alpha = move ? exp2f(m_ref - m_new) : 1.f;   // m_ref = -inf -> 0
      if (j > 0) {
        // P_{j-1}.V must be done: P's buffer is reused and O may be rescaled
        if (!mbar_wait_warp(bar(kBarPvDone), (j - 1) & 1)) {
          if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, move)) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tc::ld32(trow + kColO + 32 * c, o);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::st32(trow + kColO + 32 * c, o);
          }
          tc::wait_st();
        }
      }
      l *= alpha;
      m_ref = m_new;
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      // P row (bf16) into the swizzled shared tile, keys as the K dimension
      uint8_t *prow = sb + L::kOffP;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float p0 = 0.f, p1 = 0.f;
          if (row_valid) {
            p0 = exp2f(__uint_as_float(sr[8 * c + 2 * i]) - mu);
            p1 = exp2f(__uint_as_float(sr[8 * c + 2 * i + 1]) - mu);
          }
          rs += p0 + p1;
          w[i] = pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4 *>(prow + (c >> 3) * L::kHalfRows + swz(r, c & 7)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      l += rs;
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
    }
    // -------------------------------------------------------- epilogue
    if (ok && !mbar_wait_warp(bar(kBarPvDone), (n_blocks - 1) & 1)) {
      if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
      ok = false;
    }
    tc::fence_after_sync();
    if (ok) {
      const bool failed = *(volatile int *)flag_s != 0;
      const long orow = (2L * c0 + tok) * a.Hq + kvh * a.G + (row_valid ? grow % a.G : 0);
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tc::ld32(trow + kColO + 32 * c, o);
        tc::wait_ld();
        if (!row_valid || failed) continue;
        if (n_splits_b == 1) {
          uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)a.out + orow * HD + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(
                pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
        } else {
          const long prow = (long)split * a.T * a.Hq + orow;
          float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * HD + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                 __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
          if (c == 0) a.ml_part[prow] = make_float2(m_ref, l);
        }
      }
    }
  }
  // -------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap &mk, const CUtensorMap &mv, const AttnParams &a,
                      dim3 grid, cudaStream_t stream) {
  auto kern = attn_tc_kernel<HD>;
  const int smem = TcSmem<HD>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(mk, mv, a);
  return cudaGetLastError();
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
