// loop.cu -- the two steps around the verification in the blockwise loop:
// the draft-side step (SimSD section 4, "Drafting": the draft proposes the
// section's tokens and their temporal order) and the commit (section 4,
// "Acceptance": the longest accepted prefix is committed and the process
// repeats; "Contributions": KV cache and blockwise decoding).
//
// Draft step.  One thread-block cluster of C CTAs per sequence, CTA r owning
// vocabulary slice r of every row.  For each open slot k (decided slots keep
// their token and label):
//   1. the slice's (reference, sum of exponentials) of draft row k / T, then
//      a cluster barrier;
//   2. every CTA merges the C slice partials of every open slot through
//      distributed shared memory, in rank order (so all CTAs agree): the
//      normaliser S_k, U_k = u_k S_k and the slice whose running mass first
//      exceeds U_k;
//   3. the CTA owning that slice scans it in vocabulary order (one
//      contiguous chunk per thread, compensated running sums) for the first
//      entry whose running mass exceeds U_k;
//   4. CTA 0 orders the open slots by their largest probability (that of
//      the row's largest logit; largest first, equal ones in position
//      order) after the decided labels.
// The order depends on the draft rows only: ordering on the drawn tokens'
// own probabilities would select on the samples and bias the walk.
//
// Commit.  One thread per sequence applies the walk's outcome to the
// block state (tokens, decided count, prompt length); see simsd.h.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "vocab.cuh"

namespace simsd {
namespace {

using namespace vocab;

constexpr int kDraftThreads = 512;
constexpr int kDraftWarps = kDraftThreads / 32;
constexpr int kDraftUnroll = 8;
constexpr int kDraftCluster = 8;
constexpr int kMaxVocabDraft = 1 << 21;

struct DraftParams {
  const void *draft;
  const int32_t *cu_B;
  const float *uniforms;
  const int32_t *decided;
  const int32_t *tau_prev;
  int32_t *tokens;
  int32_t *tau;
  float *confidence;
  uint32_t *status;
  int vocab, total_B, B_max, csize, per, bulk;
  Scale ls;
};

struct __align__(16) SlicePart {
  float R, xm;    // reference (log2 units) of the slice, -inf if empty; its largest logit
  Ff s;           // sum of 2^(l ls - R) over the slice
};

struct __align__(16) SlotPick {
  Ff S, base;     // the row's normaliser; the mass before the chosen slice
  Ff U;           // u S
  float M;        // the row's reference
  float xm;       // the row's largest logit
  int ch;         // the slice holding U
};

// (R, s) += (R2, s2), both to the larger reference
__device__ __forceinline__ void part_merge(float &R, Ff &s, float R2, Ff s2) {
  const float M = fmaxf(R, R2);
  if (M == -INFINITY) return;
  const float a = exp2_int(R - M), b = exp2_int(R2 - M);
  s = ff_add(Ff{s.hi * a, s.lo * a}, Ff{s2.hi * b, s2.lo * b});
  R = M;
}

template <typename T>
__global__ void __launch_bounds__(kDraftThreads)
draft_kernel(const __grid_constant__ DraftParams a) {
  constexpr int N = Ld<T>::N;
  __shared__ SlicePart part[kMaxB];
  __shared__ SlicePart wpart[kDraftWarps];
  __shared__ SlotPick pick_s[kMaxB];
  __shared__ Ff wsum[kDraftWarps];
  __shared__ int best_s, last_s;
  const int rank = blockIdx.x, b = blockIdx.y;    // the cluster spans x
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const Scale ls = a.ls;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  const int dcd = a.decided ? __ldg(a.decided + b) : 0;
  bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B && dcd >= 0 && dcd <= B;
  // open slots: a bit per slot (the same in every CTA)
  uint32_t open = 0;
  if (valid) {
    uint32_t seen = 0;
    for (int k = 0; k < B; ++k) {
      const int tp = a.decided ? __ldg(a.tau_prev + c0 + k) : B;
      if (tp >= 1 && tp <= B) seen |= 1u << (tp - 1);
      if (!a.decided || tp > dcd) open |= 1u << k;
    }
    if (a.decided && seen != (B == 32 ? 0xffffffffu : (1u << B) - 1u)) valid = false;
  }
  if (!valid && rank == 0 && t == 0) raise_status(a.status, kStatusBadInput);
  const int s0 = min(a.vocab, rank * a.per);
  const int len = min(a.vocab, s0 + a.per) - s0;
  auto row_of = [&](int k) { return (const T *)a.draft + (long)(c0 + k) * a.vocab + s0; };

  // ---------------------------------------------------------- 1. slices
  if (valid) {
    for (uint32_t m = open; m; m &= m - 1) {
      const int k = __ffs(m) - 1;
      const T *row = row_of(k);
      float R = -INFINITY, sm = 0.f, xm = -INFINITY;
      const int nu = a.bulk ? len / N : len;
      for (int i0 = t; i0 < nu; i0 += kDraftUnroll * kDraftThreads) {
        float f[kDraftUnroll][N];
#pragma unroll
        for (int u = 0; u < kDraftUnroll; ++u) {
          const int i = i0 + u * kDraftThreads;
          if (a.bulk) {
            Ld<T>::unpack(i < nu ? __ldg(reinterpret_cast<const uint4 *>(row) + i) : Ld<T>::neg_inf(), f[u]);
          } else {
#pragma unroll
            for (int e = 0; e < N; ++e) f[u][e] = (e == 0 && i < nu) ? Ld<T>::value(row[i]) : -INFINITY;
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kDraftUnroll; ++u)
#pragma unroll
          for (int e = 0; e < N; ++e) mx = fmaxf(mx, f[u][e]);
        xm = fmaxf(xm, mx);
        const float Rn = ref_of(mx, ls);
        if (Rn > R) {
          sm = R == -INFINITY ? 0.f : sm * exp2_int(R - Rn);
          R = Rn;
        }
        if (R == -INFINITY) continue;
#pragma unroll
        for (int u = 0; u < kDraftUnroll; ++u)
#pragma unroll
          for (int e = 0; e < N; ++e) sm += rel_exp(f[u][e], R, ls);
      }
      Ff s2 = ff_of(sm);
      float Rw = R;
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) {
        const float R2 = __shfl_xor_sync(0xffffffffu, Rw, o);
        part_merge(Rw, s2, R2, ff_shfl_xor(s2, o));
        xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, o));
      }
      if (lane == 0) wpart[warp] = SlicePart{Rw, xm, s2};
      __syncthreads();
      if (t == 0) {
        SlicePart c = wpart[0];
        for (int w = 1; w < kDraftWarps; ++w) {
          part_merge(c.R, c.s, wpart[w].R, wpart[w].s);
          c.xm = fmaxf(c.xm, wpart[w].xm);
        }
        part[k] = c;
      }
      __syncthreads();
    }
  }
  cluster_sync();                                   // B1: every slice's partials are in place

  // ---------------------------------------------------------- 2. merge
  // warp w merges open slot number w, w + 16, ...: lane r reads slice r
  if (valid) {
    int idx = 0;
    for (uint32_t m = open; m; m &= m - 1, ++idx) {
      if (idx % kDraftWarps != warp) continue;
      const int k = __ffs(m) - 1;
      SlicePart v{-INFINITY, -INFINITY, ff_of(0.f)};
      if (lane < a.csize) {
        const float4 h = ld_dsmem4(dsmem(&part[k], lane));
        v = SlicePart{h.x, h.y, Ff{h.z, h.w}};
      }
      float M = v.R, xm = v.xm;
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) {
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, o));
      }
      const float wgt = (M != -INFINITY && v.R != -INFINITY) ? exp2_int(v.R - M) : 0.f;
      const Ff mass{v.s.hi * wgt, v.s.lo * wgt};      // slice mass in units of 2^M
      Ff S = mass;
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) S = ff_add(S, ff_shfl_xor(S, o));
      const float u = __ldg(a.uniforms + (long)b * a.B_max + k);
      const float uh = u * S.hi;
      const Ff U = ff_add(Ff{uh, fmaf(u, S.hi, -uh)}, ff_of(u * S.lo));
      // inclusive scan of the slice masses in rank order
      Ff inc = mass;
#pragma unroll 1
      for (int d = 1; d < 32; d <<= 1) {
        const Ff y = ff_shfl_up(inc, d);
        if (lane >= d) inc = ff_add(y, inc);
      }
      const bool has = mass.hi > 0.f;
      const unsigned cross = __ballot_sync(0xffffffffu, has && ff_gt(inc, U));
      const unsigned nz = __ballot_sync(0xffffffffu, has);
      const int ch = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : 0);
      const Ff base = ff_shfl(ff_add(inc, ff_neg(mass)), ch);
      if (lane == 0) pick_s[k] = SlotPick{S, base, U, M, xm, ch};
    }
  }
  __syncthreads();

  // ---------------------------------------------------------- 3. scans
  if (valid) {
    for (uint32_t m = open; m; m &= m - 1) {
      const int k = __ffs(m) - 1;
      const SlotPick pk = pick_s[k];
      if (pk.ch != rank) continue;                  // uniform across the CTA
      const T *row = row_of(k);
      const int chunk = (len + kDraftThreads - 1) / kDraftThreads;
      const int e0 = min(len, t * chunk), e1 = min(len, e0 + chunk);
      float part_m = 0.f;
      int last = -1;
      for (int e = e0; e < e1; ++e) {
        const float q = rel_exp(Ld<T>::value(row[e]), pk.M, ls);
        part_m += q;
        if (q > 0.f) last = s0 + e;
      }
      if (t == 0) { best_s = 0x7fffffff; last_s = -1; }
      Ff inc = ff_of(part_m);
#pragma unroll 1
      for (int d = 1; d < 32; d <<= 1) {
        const Ff y = ff_shfl_up(inc, d);
        if (lane >= d) inc = ff_add(y, inc);
      }
      if (lane == 31) wsum[warp] = inc;
      __syncthreads();
      Ff start = pk.base;
      for (int w = 0; w < warp; ++w) start = ff_add(start, wsum[w]);
      start = ff_add(start, ff_add(inc, ff_of(-part_m)));
      const Ff D = ff_add(pk.U, ff_neg(start));
      const float dd = D.hi + D.lo;                 // U - this chunk's start
      int first = 0x7fffffff;
      if (dd < part_m) {
        float run = 0.f;
        for (int e = e0; e < e1; ++e) {
          const float q = rel_exp(Ld<T>::value(row[e]), pk.M, ls);
          run += q;
          if (q > 0.f && run > dd) { first = s0 + e; break; }
        }
      }
      if (first != 0x7fffffff) atomicMin(&best_s, first);
      if (last >= 0) atomicMax(&last_s, last);
      __syncthreads();
      if (t == 0) a.tokens[c0 + k] = best_s != 0x7fffffff ? best_s : last_s;
      __syncthreads();
    }
  }

  // ---------------------------------------------------------- 4. the order
  if (valid && rank == 0 && t < B) {
    const int k = t;
    if ((open >> k) & 1u) {
      const SlotPick pk = pick_s[k];
      // the row's largest probability, in the kernel's own arithmetic
      const float ck = rel_exp(pk.xm, pk.M, ls) / (pk.S.hi + pk.S.lo);
      int before = 0;
      for (uint32_t m = open; m; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const SlotPick pj = pick_s[j];
        const float cj = rel_exp(pj.xm, pj.M, ls) / (pj.S.hi + pj.S.lo);
        if (cj > ck || (cj == ck && j < k)) ++before;
      }
      a.tau[c0 + k] = dcd + 1 + before;
      if (a.confidence) a.confidence[c0 + k] = ck;
    } else {
      a.tau[c0 + k] = __ldg(a.tau_prev + c0 + k);
      if (a.confidence) a.confidence[c0 + k] = -1.f;
    }
  }
  cluster_sync();                                   // B2: no CTA leaves while others read it
}

// The draft step over a chunk pass (no decided slots; a full workspace).
// The chunk pass (accept.cu) left, per (row, 32 KB chunk, part of 1/8
// chunk), the part's reference, sum of 2^(l ls - reference) and largest
// logit; parts in (chunk, part) order are contiguous vocabulary ranges in
// vocabulary order.  One CTA per sequence, a warp per slot: the row's
// normaliser S and largest logit (exact merge by powers of two), U = u S,
// the first part whose running mass exceeds U (else the last with mass),
// then that part read again column by column in vocabulary order (an fp32
// scan relative to the part's start) for the first entry whose running
// mass exceeds U; then the slots ordered by their largest probability.
constexpr int kFinishThreads = 512;
constexpr int kFinishWarps = kFinishThreads / 32;
constexpr int kParts = 8;                         // parts per chunk (the chunk pass's warps)

struct FinishParams {
  const void *draft;
  const int32_t *cu_B;
  const float *uniforms;
  const float4 *part4;      // [total_B][nchunks][kParts]
  int *claim;               // the chunk pass's control words, zeroed here
  int32_t *tokens;
  int32_t *tau;
  float *confidence;
  uint32_t *status;
  int vocab, total_B, B_max, nchunks, chunk, bulk;
  Scale ls;
};

template <typename T>
__global__ void __launch_bounds__(kFinishThreads)
draft_finish_kernel(const __grid_constant__ FinishParams a) {
  __shared__ float conf_s[kMaxB];
  const int b = blockIdx.x, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  __shared__ int tok_s[kMaxB];
  __shared__ int fail_s;
  grid_dep_wait();                                  // the chunk pass's partials
  // the chunk pass's give-up flag, read by the last thread (checked before
  // any output is written); the CTA whose ticket is the last zeroes the
  // chunk pass's words
  const int flag_t = kFinishThreads - 1;
  int ticket = -1;
  if (t == flag_t) fail_s = chunk_flag_read(a.claim, &ticket);
  const int c0 = __ldg(a.cu_B + b), B = __ldg(a.cu_B + b + 1) - c0;
  const bool valid = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B;
  if (!valid) {                                     // tokens and tau are left unwritten
    if (t == 0) raise_status(a.status, kStatusBadInput);
    if (t == flag_t) chunk_flag_reset(a.claim, ticket, gridDim.x);
    return;
  }
  const Scale ls = a.ls;
  const int n_ent = a.nchunks * kParts;             // parts of a row
  for (int k = warp; k < B; k += kFinishWarps) {
    const float4 *pr = a.part4 + (long)(c0 + k) * n_ent;
    // the row: M, S, largest logit (the first 4 x 32 parts held)
    constexpr int kHeld = 4;
    float4 h[kHeld];
#pragma unroll
    for (int i = 0; i < kHeld; ++i)
      h[i] = lane + 32 * i < n_ent ? __ldcg(pr + lane + 32 * i) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    float M = -INFINITY, xm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kHeld; ++i) { M = fmaxf(M, h[i].x); xm = fmaxf(xm, h[i].z); }
    for (int i = lane + 32 * kHeld; i < n_ent; i += 32) {
      const float4 v = __ldcg(pr + i);
      M = fmaxf(M, v.x);
      xm = fmaxf(xm, v.z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, o));
    }
    auto mass_of = [&](float4 v) {
      const float w = (M != -INFINITY && v.x != -INFINITY) ? exp2_int(v.x - M) : 0.f;
      return v.y > 0.f ? v.y * w : 0.f;
    };
    Ff S = ff_of(0.f);
#pragma unroll
    for (int i = 0; i < kHeld; ++i) S = ff_add(S, ff_of(mass_of(h[i])));
    for (int i = lane + 32 * kHeld; i < n_ent; i += 32) S = ff_add(S, ff_of(mass_of(__ldcg(pr + i))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S = ff_add(S, ff_shfl_xor(S, o));
    const float u = __ldg(a.uniforms + (long)b * a.B_max + k);
    const float uh = u * S.hi;
    const Ff U = ff_add(Ff{uh, fmaf(u, S.hi, -uh)}, ff_of(u * S.lo));
    const int tok = part_draw<T, kHeld>(pr, h, n_ent, M, U, (const T *)a.draft + (long)(c0 + k) * a.vocab,
                                        a.vocab, a.chunk, a.bulk != 0, ls, lane);
    if (lane == 0) {
      tok_s[k] = tok;
      // the row's largest probability, in the kernel's own arithmetic
      conf_s[k] = rel_exp(xm, M, ls) / (S.hi + S.lo);
    }
  }
  __syncthreads();
  // a chunk pass whose wait gave up (its status bit is set): tokens and
  // tau are left unwritten
  if (t < B && !fail_s) {                           // largest first, equal ones in position order
    const float ck = conf_s[t];
    int before = 0;
    for (int j = 0; j < B; ++j) {
      const float cj = conf_s[j];
      if (cj > ck || (cj == ck && j < t)) ++before;
    }
    a.tokens[c0 + t] = tok_s[t];
    a.tau[c0 + t] = 1 + before;
    if (a.confidence) a.confidence[c0 + t] = ck;
  }
  if (t == flag_t) chunk_flag_reset(a.claim, ticket, gridDim.x);
}

template <typename T>
cudaError_t launch_finish(const FinishParams &f, int batch, cudaStream_t stream) {
  return launch_pdl(draft_finish_kernel<T>, dim3(batch), dim3(kFinishThreads), 0, stream, f);
}

// The commit: one thread per sequence.
struct CommitParams {
  const int32_t *cu_B, *tau, *n_accept, *token, *pos;
  int32_t *tokens, *decided, *lens, *done;
  uint32_t *status;
  int batch, total_B, B_max;
};

__global__ void __launch_bounds__(128) commit_kernel(const __grid_constant__ CommitParams a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.batch) return;
  const int c0 = __ldg(a.cu_B + b);
  const int B = __ldg(a.cu_B + b + 1) - c0;
  bool ok = B >= 1 && B <= a.B_max && c0 >= 0 && c0 + B <= a.total_B;
  const int n = ok ? __ldg(a.n_accept + b) : -1;
  const int p = ok ? __ldg(a.pos + b) : -1;
  ok = ok && n >= 0 && n <= B && (p >= 0 ? (p < B && n < B) : n == B);
  if (ok && p >= 0) ok = __ldg(a.tau + c0 + p) == n + 1;   // the walk's next step
  if (!ok) {
    raise_status(a.status, kStatusBadInput);
    a.done[b] = 0;
    return;
  }
  if (p >= 0) {
    a.tokens[c0 + p] = __ldg(a.token + b);
    a.decided[b] = n + 1;
    a.done[b] = 0;
  } else {
    a.lens[b] += B;
    a.decided[b] = 0;
    a.done[b] = 1;
  }
}

template <typename T>
cudaError_t launch_draft(DraftParams a, int batch, cudaStream_t stream) {
  const int vec = 16 / (int)sizeof(T);
  a.csize = max(1, min(kDraftCluster, device_sm_count() / max(1, batch)));
  a.per = ((a.vocab + a.csize - 1) / a.csize + vec - 1) / vec * vec;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.csize, batch);
  cfg.blockDim = dim3(kDraftThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, draft_kernel<T>, a);
}

simsd_status draft_check(const simsd_draft_desc *d) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (d->dtype != SIMSD_F32 && d->dtype != SIMSD_BF16) return SIMSD_ERR_DTYPE;
  if (d->batch < 1 || d->batch > 65535 || d->vocab < 1 || d->vocab > kMaxVocabDraft ||
      d->B_max < 1 || d->B_max > kMaxB || d->total_B < d->batch ||
      (int64_t)d->total_B > (int64_t)d->batch * d->B_max ||
      !(d->temperature >= 0.f && d->temperature <= 3.0e38f))
    return SIMSD_ERR_SHAPE;
  return SIMSD_OK;
}

constexpr size_t kStatusWorkspace = kAlign;

bool workspace_ok(void *ws, size_t bytes) {
  return ws != nullptr && ((uintptr_t)ws % kAlign) == 0 && bytes >= kStatusWorkspace;
}

}  // namespace
}  // namespace simsd

using namespace simsd;

extern "C" {

// The chunked path's workspace: status word and the chunk pass's control
// words | chunk partials.
struct DraftLayout {
  int nchunks, chunk;
  size_t off_part, off_claim, total;
};
DraftLayout draft_layout(const simsd_draft_desc *d) {
  DraftLayout L;
  L.chunk = draft_chunk_entries(d->dtype == SIMSD_BF16 ? 2 : 4);
  L.nchunks = (d->vocab + L.chunk - 1) / L.chunk;
  L.off_claim = kClaimOffset;                 // beside the status word
  L.off_part = kStatusWorkspace;
  L.total = align_up(L.off_part + (size_t)d->total_B * L.nchunks * kParts * sizeof(float4), kAlign);
  return L;
}

size_t simsd_draft_workspace_size(const simsd_draft_desc *d) {
  return draft_check(d) == SIMSD_OK ? draft_layout(d).total : 0;
}

simsd_status simsd_draft_step(const simsd_draft_desc *d, void *stream_ptr) {
  simsd_status st = draft_check(d);
  if (st != SIMSD_OK) return st;
  if (!d->draft_logits || !d->cu_B || !d->uniforms || !d->tokens || !d->tau ||
      (d->decided && !d->tau_prev))
    return SIMSD_ERR_NULL;
  if (!workspace_ok(d->workspace, d->workspace_bytes)) return SIMSD_ERR_WORKSPACE;
  const int es = d->dtype == SIMSD_BF16 ? 2 : 4;
  DraftParams a;
  a.draft = d->draft_logits;
  a.cu_B = d->cu_B;
  a.uniforms = d->uniforms;
  a.decided = d->decided;
  a.tau_prev = d->tau_prev;
  a.tokens = d->tokens;
  a.tau = d->tau;
  a.confidence = d->confidence;
  a.status = (uint32_t *)d->workspace;
  a.vocab = d->vocab;
  a.total_B = d->total_B;
  a.B_max = d->B_max;
  a.csize = 1;
  a.per = 0;
  a.bulk = ((size_t)d->vocab * es) % 16 == 0 && aligned16(d->draft_logits);
  a.ls = scale_of(d->temperature > 0.f ? (double)d->temperature : 1.0);
  const cudaStream_t stream = (cudaStream_t)stream_ptr;
  const DraftLayout L = draft_layout(d);
  if (d->decided == nullptr && d->workspace_bytes >= L.total) {
    // the chunk pass over every SM, then one CTA per sequence
    char *ws = (char *)d->workspace;
    FinishParams f;
    f.draft = d->draft_logits;
    f.cu_B = d->cu_B;
    f.uniforms = d->uniforms;
    f.part4 = (const float4 *)(ws + L.off_part);
    f.claim = (int *)(ws + L.off_claim);
    f.tokens = d->tokens;
    f.tau = d->tau;
    f.confidence = d->confidence;
    f.status = a.status;
    f.vocab = d->vocab;
    f.total_B = d->total_B;
    f.B_max = d->B_max;
    f.nchunks = L.nchunks;
    f.chunk = L.chunk;
    f.bulk = a.bulk;
    f.ls = a.ls;
    cudaError_t e = launch_draft_chunks(d, (float4 *)(ws + L.off_part), f.claim, a.status, L.nchunks, stream);
    if (e == cudaSuccess)
      e = d->dtype == SIMSD_BF16 ? launch_finish<__nv_bfloat16>(f, d->batch, stream)
                                 : launch_finish<float>(f, d->batch, stream);
    return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
  }
  // the single cluster kernel (a workspace of only the status word, or
  // decided slots)
  const cudaError_t e = d->dtype == SIMSD_BF16
                            ? launch_draft<__nv_bfloat16>(a, d->batch, stream)
                            : launch_draft<float>(a, d->batch, stream);
  return e == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

size_t simsd_commit_workspace_size(const simsd_commit_desc *d) {
  if (d == nullptr || d->batch < 1 || d->B_max < 1 || d->B_max > kMaxB ||
      d->total_B < d->batch || (int64_t)d->total_B > (int64_t)d->batch * d->B_max)
    return 0;
  return kStatusWorkspace;
}

simsd_status simsd_commit(const simsd_commit_desc *d, void *stream_ptr) {
  if (d == nullptr) return SIMSD_ERR_NULL;
  if (simsd_commit_workspace_size(d) == 0) return SIMSD_ERR_SHAPE;
  if (!d->cu_B || !d->tau || !d->n_accept || !d->token || !d->pos || !d->tokens ||
      !d->decided || !d->lens || !d->done)
    return SIMSD_ERR_NULL;
  if (!workspace_ok(d->workspace, d->workspace_bytes)) return SIMSD_ERR_WORKSPACE;
  CommitParams a;
  a.cu_B = d->cu_B;
  a.tau = d->tau;
  a.n_accept = d->n_accept;
  a.token = d->token;
  a.pos = d->pos;
  a.tokens = d->tokens;
  a.decided = d->decided;
  a.lens = d->lens;
  a.done = d->done;
  a.status = (uint32_t *)d->workspace;
  a.batch = d->batch;
  a.total_B = d->total_B;
  a.B_max = d->B_max;
  commit_kernel<<<(d->batch + 127) / 128, 128, 0, (cudaStream_t)stream_ptr>>>(a);
  return cudaGetLastError() == cudaSuccess ? SIMSD_OK : SIMSD_ERR_CUDA;
}

}  // extern "C"
