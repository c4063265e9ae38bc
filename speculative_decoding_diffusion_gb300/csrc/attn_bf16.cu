// attn_bf16.cu -- K2 (bf16): split-KV masked attention over the paged cache.
//
// SimSD section 2 "Temporal Attention Mask" and section 4 (one verification
// forward): every new row attends to the whole prompt; a slot row D~_i also
// to D_j with tau(j) < tau(i) and to D~_j with tau(j) >= tau(i); a data row
// D_i (convention) to D_j with tau(j) <= tau(i).  The mask is never stored:
// only the last 2B keys of a sequence need it and it is evaluated there
// from tau held in shared memory.
//
// Work decomposition: one CTA per (key split, KV head x row tile, sequence).
// The query tile stacks all 2B tokens x G query heads of one KV head (rows
// r = token * G + head_in_group), so every key/value byte streamed from HBM
// serves 2B*G rows.  8 consumer warps own 16 rows each; when the tile has
// fewer rows, the warps also split each stage's keys and merge at the end.
// A producer warp streams 128-key stages (8 pages) of K and V with TMA
// (128-byte swizzle, one 2 KB box per page and 64-column half) into a
// 3-stage shared-memory ring guarded by mbarriers.  Scores and P.V use
// mma.sync m16n8k16 bf16 -> fp32; the softmax is online in fp32 registers
// (log2 domain) with quad shuffles.  A split writes either the finished row
// (single-split sequences) or an unnormalised partial (O, m, l) for K3.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace simsd {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kBoxBytes = kPage * 128;  // one page x 64 bf16 columns
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct Smem {
  static constexpr int kHalves = HD / 64;
  static constexpr int kHalfBytes = kBlockKeys * 128;           // 16 KB
  static constexpr int kTileBytes = kHalves * kHalfBytes;       // K or V
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kTauOff = kBarOff + 2 * kStages * 8;
  static constexpr int kFlagOff = kTauOff + 2 * kMaxB * 4;
  static constexpr int kBytes = kFlagOff + 16;
  static constexpr int kAlloc = kBytes + 1024;                  // alignment slack
};

// Byte offset of 16-byte chunk c (0..HD/8-1) of key row r inside a K or V
// tile written by 128B-swizzled TMA boxes.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kBlockKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int HD, int KS>
__global__ void __launch_bounds__(kThreads, 1)
attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ AttnParams a) {
  using L = Smem<HD>;
  constexpr int RG = kConsumerWarps / KS;   // row groups of 16
  constexpr int KW = kBlockKeys / KS;       // keys per warp per stage
  constexpr int SUB = KW < 64 ? KW : 64;    // keys per score sub-block
  constexpr int NT = SUB / 8;               // score n-tiles per sub-block
  constexpr int OT = HD / 8;                // output n-tiles
  constexpr int QK = HD / 16;               // k-steps of q.k

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw);
  const uint32_t bar_full = base + L::kBarOff;
  const uint32_t bar_empty = bar_full + kStages * 8;
  int *tau_s = reinterpret_cast<int *>(sbase + L::kTauOff);
  int *flag_s = reinterpret_cast<int *>(sbase + L::kFlagOff);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y % a.Hkv;
  const int rtile = blockIdx.y / a.Hkv;
  const int b = blockIdx.z;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int P = __ldg(a.lens + b);
  const int Lk = P + 2 * B;                 // keys of this sequence
  const int M = 2 * B * a.G;                // query rows of this sequence
  const int row0 = rtile * a.rows_per_tile;
  const int k_begin = split * a.chunk;
  if (B < 1 || B > kMaxSection || P < 0 || (long)Lk > (long)a.max_pages_per_seq * kPage) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) raise_status(a.status, kStatusBadInput);
    return;                                  // malformed sequence
  }
  if (row0 >= M || k_begin >= Lk) return;   // uniform: nothing to do here
  const int k_end = min(Lk, k_begin + a.chunk);
  const int n_stages = (k_end - k_begin + kBlockKeys - 1) / kBlockKeys;
  const int n_splits_b = (Lk + a.chunk - 1) / a.chunk;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    *flag_s = 0;
    fence_barrier_init();
  }
  // tau of the 2B new tokens (D_j and D~_j share tau(j))
  for (int j = threadIdx.x; j < 2 * B; j += blockDim.x)
    tau_s[j] = __ldg(a.tau + c0 + (j < B ? j : j - B));
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    const int32_t *bt = a.block_table + (long)b * a.max_pages_per_seq;
    bool ok = true;
    for (int i = 0; i < n_stages && ok; ++i) {
      const int slot = i % kStages;
      if (i >= kStages && !mbar_wait_warp(bar_empty + 8 * slot, ((i / kStages) - 1) & 1)) {
        ok = false;
        if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
        break;
      }
      const int kb = k_begin + i * kBlockKeys;
      const int n_pages = (min(kBlockKeys, k_end - kb) + kPage - 1) / kPage;
      const int page = lane < n_pages ? __ldg(bt + kb / kPage + lane) : 0;
      if (lane == 0)
        mbar_arrive_expect_tx(bar_full + 8 * slot, n_pages * L::kHalves * 2 * kBoxBytes);
      __syncwarp();
      if (lane < n_pages) {
        const uint32_t kt = base + slot * L::kStageBytes;
        const uint32_t vt = kt + L::kTileBytes;
#pragma unroll
        for (int hh = 0; hh < L::kHalves; ++hh) {
          const uint32_t off = hh * L::kHalfBytes + lane * kBoxBytes;
          tma_load_4d(kt + off, &tmK, bar_full + 8 * slot, hh * 64, 0, kvh, page);
          tma_load_4d(vt + off, &tmV, bar_full + 8 * slot, hh * 64, 0, kvh, page);
        }
      }
    }
    if (!ok) {
      // let copies already in flight land before the CTA can exit
      const int issued = n_stages;
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = ((issued - 1 - s) / kStages) * kStages + s;
        (void)mbar_wait_warp(bar_full + 8 * s, (last / kStages) & 1);
      }
    }
    named_sync(2, kThreads);                // join the consumers' epilogue
    return;
  }

  // -------------------------------------------------------------- consumers
  const int rg = warp % RG, ks = warp / RG;
  const int g = lane >> 2, t4 = lane & 3;
  const int wrow = row0 + rg * 16;
  int row_tok[2], row_slot[2], row_tau[2], row_valid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = wrow + g + 8 * h;
    row_valid[h] = r < M;
    const int tok = row_valid[h] ? r / a.G : 0;
    row_tok[h] = tok;
    row_slot[h] = tok >= B;
    row_tau[h] = tau_s[tok];
  }
  // query fragments (rotated q, bf16) straight from global memory
  uint32_t qf[QK][4];
  {
    const __nv_bfloat16 *q = (const __nv_bfloat16 *)a.q_rot;
    const long tok_base = 2L * c0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = wrow + g + 8 * h;
      const __nv_bfloat16 *qrow =
          q + ((tok_base + row_tok[h]) * a.Hq + kvh * a.G + (r % a.G)) * HD;
#pragma unroll
      for (int kk = 0; kk < QK; ++kk) {
        uint32_t lo = 0, hi = 0;
        if (row_valid[h]) {
          lo = *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 2 * t4);
          hi = *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + 2 * t4);
        }
        qf[kk][h] = lo;       // a0 (row g) / a1 (row g+8)
        qf[kk][2 + h] = hi;   // a2 / a3
      }
    }
  }

  float o[OT][4];
#pragma unroll
  for (int n = 0; n < OT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const float scale = a.sm_scale * kLog2e;
  bool failed = false;

  for (int i = 0; i < n_stages; ++i) {
    const int slot = i % kStages;
    if (!failed && !mbar_wait_warp(bar_full + 8 * slot, (i / kStages) & 1)) {
      failed = true;
      if (lane == 0) { raise_status(a.status, kStatusTimeout); atomicOr(flag_s, 1); }
    }
    const int kb = k_begin + i * kBlockKeys;
    const int stage_valid = min(kBlockKeys, k_end - kb);
    const int stage_loaded = (stage_valid + kPage - 1) & ~(kPage - 1);
    const uint32_t kt = base + slot * L::kStageBytes;
    const uint32_t vt = kt + L::kTileBytes;
    const int wo = ks * KW;                 // this warp's first key in the stage
    if (!failed && wo < stage_loaded) {
      // Keys of the last page past the sequence end may hold anything; the
      // values there must be finite because P.V multiplies them by p = 0.
      if (kb + stage_loaded > Lk && kb + stage_valid == Lk) {
        const int first = Lk - kb, last = stage_loaded;   // rows [first, last)
        if (first >= wo && first < wo + KW) {
          for (int e = lane; e < (last - first) * (HD / 8); e += 32) {
            const int r = first + e / (HD / 8), c = e % (HD / 8);
            *reinterpret_cast<uint4 *>(sbase + (vt - base) + tile_off(r, c)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();  // the slot is refilled by TMA later
        }
        __syncwarp();
      }
      const bool no_mask = kb + kBlockKeys <= min(P, k_end);
#pragma unroll
      for (int sb = 0; sb < KW / SUB; ++sb) {
        const int k0 = wo + sb * SUB;       // first key of the sub-block in stage
        if (k0 >= stage_loaded) break;
        float s[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < QK; ++kk) {
#pragma unroll
          for (int np = 0; np < NT / 2; ++np) {
            if (k0 + np * 16 < stage_loaded) {
              const int mi = lane >> 3;
              const int r = k0 + np * 16 + ((mi >> 1) << 3) + (lane & 7);
              const int c = 2 * kk + (mi & 1);
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4(kt + tile_off(r, c), b0, b1, b2, b3);
              mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
              mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
            }
          }
        }
        // scale, mask, running max
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            float v = s[n][e] * scale;
            if (!no_mask) {
              const int key = kb + k0 + n * 8 + 2 * t4 + (e & 1);
              bool vis = key < k_end;
              if (vis && key >= P) {
                const int j = key - P;       // 0..2B-1 among the new tokens
                const int tj = tau_s[j];
                const bool key_slot = j >= B;
                vis = row_slot[h] ? (key_slot ? tj >= row_tau[h] : tj < row_tau[h])
                                  : (!key_slot && tj <= row_tau[h]);
              }
              if (!vis) v = -INFINITY;
            }
            s[n][e] = v;
            mx[h] = fmaxf(mx[h], v);
          }
        }
        float alpha[2], m_use[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          const float m_new = fmaxf(m_run[h], mx[h]);
          m_use[h] = m_new == -INFINITY ? 0.f : m_new;
          alpha[h] = exp2f(m_run[h] - m_use[h]);
          m_run[h] = m_new;
        }
        float rs[2] = {0.f, 0.f};
        uint32_t pf[NT / 2][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float p0 = exp2f(s[n][0] - m_use[0]);
          const float p1 = exp2f(s[n][1] - m_use[0]);
          const float p2 = exp2f(s[n][2] - m_use[1]);
          const float p3 = exp2f(s[n][3] - m_use[1]);
          rs[0] += p0 + p1;
          rs[1] += p2 + p3;
          pf[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(p0, p1);
          pf[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
#pragma unroll
        for (int n = 0; n < OT; ++n) {
          o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
          o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
        }
        // O += P V over this sub-block's loaded pages
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) {
          if (k0 + kk * 16 < stage_loaded) {
            // A fragment of P: rows g / g+8, keys 16kk + {2t4, 2t4+1, +8, +9}
            uint32_t pa[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
            for (int np = 0; np < OT / 2; ++np) {
              const int mi = lane >> 3;
              const int r = k0 + kk * 16 + ((mi & 1) << 3) + (lane & 7);
              const int c = 2 * np + (mi >> 1);
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4_trans(vt + tile_off(r, c), b0, b1, b2, b3);
              mma_bf16_16816(o[2 * np], pa, b0, b1);
              mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
  }

  // ---------------------------------------------------------------- epilogue
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  // all consumers are past the stage ring: it is free for the merge
  named_sync(1, kConsumerWarps * 32);
  const bool cta_failed = *(volatile int *)flag_s != 0;
  if (KS > 1) {
    float4 *mo = reinterpret_cast<float4 *>(sbase);    // [warp][OT][32]
    float4 *ml = mo + kConsumerWarps * OT * 32;          // [warp][32]
    if (ks > 0) {
#pragma unroll
      for (int n = 0; n < OT; ++n)
        mo[(warp * OT + n) * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
      ml[warp * 32 + lane] = make_float4(m_run[0], m_run[1], l_run[0], l_run[1]);
    }
    named_sync(1, kConsumerWarps * 32);
    if (ks == 0) {
#pragma unroll
      for (int p = 1; p < KS; ++p) {
        const int w2 = rg + p * RG;
        const float4 q = ml[w2 * 32 + lane];
        const float m2[2] = {q.x, q.y}, l2[2] = {q.z, q.w};
        float f1[2], f2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mm = fmaxf(m_run[h], m2[h]);
          const float mu = mm == -INFINITY ? 0.f : mm;
          f1[h] = exp2f(m_run[h] - mu);
          f2[h] = exp2f(m2[h] - mu);
          l_run[h] = l_run[h] * f1[h] + l2[h] * f2[h];
          m_run[h] = mm;
        }
#pragma unroll
        for (int n = 0; n < OT; ++n) {
          const float4 v = mo[(w2 * OT + n) * 32 + lane];
          o[n][0] = o[n][0] * f1[0] + v.x * f2[0];
          o[n][1] = o[n][1] * f1[0] + v.y * f2[0];
          o[n][2] = o[n][2] * f1[1] + v.z * f2[1];
          o[n][3] = o[n][3] * f1[1] + v.w * f2[1];
        }
      }
    }
  }
  if (ks == 0 && !cta_failed) {
    const long tok_base = 2L * c0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!row_valid[h]) continue;
      const int r = wrow + g + 8 * h;
      const long tok = tok_base + row_tok[h];
      const int head = kvh * a.G + (r % a.G);
      const long row = tok * a.Hq + head;
      if (n_splits_b == 1) {
        const float inv = 1.f / l_run[h];
        __nv_bfloat16 *out = (__nv_bfloat16 *)a.out + row * HD;
#pragma unroll
        for (int n = 0; n < OT; ++n)
          *reinterpret_cast<uint32_t *>(out + n * 8 + 2 * t4) =
              pack_bf16x2(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
      } else {
        const long prow = (long)split * a.T * a.Hq + row;
        float *op = a.o_part + prow * HD;
#pragma unroll
        for (int n = 0; n < OT; ++n)
          *reinterpret_cast<float2 *>(op + n * 8 + 2 * t4) =
              make_float2(o[n][2 * h], o[n][2 * h + 1]);
        if (t4 == 0) a.ml_part[prow] = make_float2(m_run[h], l_run[h]);
      }
    }
  }
  named_sync(2, kThreads);
}

template <int HD, int KS>
cudaError_t launch_variant(const CUtensorMap &mk, const CUtensorMap &mv,
                           const AttnParams &a, dim3 grid, cudaStream_t stream) {
  auto kern = attn_bf16_kernel<HD, KS>;
  const int smem = Smem<HD>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(mk, mv, a);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap &mk, const CUtensorMap &mv,
                      const AttnParams &a, int ks, dim3 grid, cudaStream_t stream) {
  switch (ks) {
    case 1: return launch_variant<HD, 1>(mk, mv, a, grid, stream);
    case 2: return launch_variant<HD, 2>(mk, mv, a, grid, stream);
    case 4: return launch_variant<HD, 4>(mk, mv, a, grid, stream);
    default: return launch_variant<HD, 8>(mk, mv, a, grid, stream);
  }
}

}  // namespace

cudaError_t launch_attn_bf16(const simsd_verify_desc *d, const VerifyPlan &p,
                             const AttnParams &a, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, d->k_cache, d->num_pages, d->num_kv_heads, d->head_dim) ||
      !make_cache_map(&mv, d->v_cache, d->num_pages, d->num_kv_heads, d->head_dim))
    return cudaErrorInvalidValue;
  dim3 grid(p.n_splits, d->num_kv_heads * p.row_tiles, d->batch);
  if (d->head_dim == 128) return launch_hd<128>(mk, mv, a, p.key_splits, grid, stream);
  return launch_hd<64>(mk, mv, a, p.key_splits, grid, stream);
}

}  // namespace simsd
