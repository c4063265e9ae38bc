"""Seeded synthetic inputs for the SimSD verification step.

This module only draws random arrays; it holds none of the method's
arithmetic (no layout, mask, RoPE, attention or acceptance rule).  Both the
fp64 oracle (through the tests) and the CUDA library (through the tests and
the benchmark) take their inputs from here, so the two sides see identical
values.  Floating-point arrays for bf16 workloads are returned as bf16 bit
patterns (uint16); ``to_f64`` widens them exactly.

Workload shapes follow an SDAR-8B-like verification step (32 query heads,
8 KV heads, head dim 128, vocabulary 151,936, RoPE base 1e6) and a tiny fp32
case; see ``CONFIGS``.  Draw order for a seed (numpy ``default_rng``):
  1 prompt lengths, 2 section lengths B_b, 3 step labels tau_b
  (a permutation of 1..B_b), 4 physical page order, 5 q, 6 prompt keys
  (raw for the tiny case, otherwise drawn directly in the rotated frame:
  a rotation keeps an iid normal vector iid normal), 7 prompt values,
  8 new keys, 9 new values, 10 target logits, 11 per-sequence draft noise
  scale, 12 draft noise, 13 draft tokens (inverse CDF of the draft softmax),
  14 acceptance uniforms (fp32 in [0,1), B_max+1 per sequence).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE = 16  # tokens per KV-cache page


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    prompt: object            # int, or (lo, hi) inclusive for a ragged mix
    B: object                 # int, or tuple of choices per sequence
    Hq: int = 32
    Hkv: int = 8
    hd: int = 128
    dtype: str = "bf16"       # "bf16" or "f32" (storage of q/k/v and logits)
    rope_base: float = 1.0e6
    vocab: int = 151936
    qkv_sd: float = 1.0       # sd of k, v (and q before q_scale)
    q_scale: float = 1.0 / math.sqrt(128.0)
    logit_sd: float = 3.0
    noise_sd: object = 1.0    # float, or (lo, hi) drawn per sequence
    shuffled_pages: bool = False
    raw_prompt_keys: bool = False
    sm_scale: float = 1.0
    slug: str = ""            # short file-name form of the name


CONFIGS = {
    0: Spec("tiny: 1 seq, P=64, B=4, Hq4/Hkv2/hd64, fp32, V=512", batch=1,
            prompt=64, B=4, Hq=4, Hkv=2, hd=64, dtype="f32", rope_base=1.0e4,
            vocab=512, qkv_sd=1.0 / 8.0, q_scale=1.0, logit_sd=2.0,
            noise_sd=0.5, raw_prompt_keys=True, slug="tiny_1x64_B4"),
    1: Spec("sdar8b-verify: 16 seq, P=1024, B=4", batch=16, prompt=1024, B=4,
            slug="sdar8b_16x1024_B4"),
    2: Spec("sdar8b-verify: 64 seq, P=4096, B=8", batch=64, prompt=4096, B=8,
            slug="sdar8b_64x4096_B8"),
    3: Spec("long-prefix: 8 seq, P=32768, B=16, shuffled pages", batch=8,
            prompt=32768, B=16, shuffled_pages=True, slug="longprefix_8x32768_B16"),
    4: Spec("ragged-mix: 256 seq, P~U[256,8192], B in {4,8}", batch=256,
            prompt=(256, 8192), B=(4, 8), noise_sd=(0.25, 2.0),
            shuffled_pages=True, slug="ragged_256xU256-8192_B4-8"),
}


@dataclasses.dataclass
class Workload:
    spec: Spec
    seed: int
    lens: np.ndarray          # int32[batch]      prompt KV length P_b
    Bs: np.ndarray            # int32[batch]      section length B_b
    cu_B: np.ndarray          # int32[batch+1]    prefix sums of B_b
    tau: np.ndarray           # int32[sum B]      step labels
    num_pages: int
    max_pages: int
    block_table: np.ndarray   # int32[batch, max_pages]
    q: np.ndarray             # [sum 2B, Hq, hd]   raw queries
    k_prompt: np.ndarray      # [sum P, Hkv, hd]   (rotated unless raw_prompt_keys)
    v_prompt: np.ndarray      # [sum P, Hkv, hd]
    k_new: np.ndarray         # [sum 2B, Hkv, hd]  raw
    v_new: np.ndarray         # [sum 2B, Hkv, hd]
    target: Optional[np.ndarray]        # [sum B, V]
    draft: Optional[np.ndarray]         # [sum B, V]
    draft_tokens: Optional[np.ndarray]  # int32[sum B]
    uniforms: Optional[np.ndarray]      # float32[batch, B_max+1]

    @property
    def B_max(self) -> int:
        return int(self.Bs.max())

    @property
    def total_B(self) -> int:
        return int(self.cu_B[-1])

    @property
    def prompt_offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lens, dtype=np.int64)])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = u + (((u >> 16) & 1) + np.uint32(0x7FFF))
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of a stored array (bf16 bits or fp32) to fp64."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _normal(rng, shape, sd, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sd != 1.0:
        x *= np.float32(sd)
    return _store(x, dtype)


def make(spec: Spec, seed: int, with_logits: bool = True,
         lens=None, Bs=None, taus=None) -> Workload:
    """Draw one workload.  lens / Bs / taus override the drawn values (they
    are still drawn, so the stream stays aligned) for edge-case tests."""
    rng = np.random.default_rng(seed)
    n = spec.batch
    # 1 prompt lengths
    if isinstance(spec.prompt, tuple):
        d_lens = rng.integers(spec.prompt[0], spec.prompt[1] + 1, size=n)
    else:
        d_lens = np.full(n, spec.prompt)
    # 2 section lengths
    if isinstance(spec.B, tuple):
        d_Bs = rng.choice(np.asarray(spec.B), size=n)
    else:
        d_Bs = np.full(n, spec.B)
    lens_a = np.asarray(d_lens if lens is None else lens, np.int32)
    Bs_a = np.asarray(d_Bs if Bs is None else Bs, np.int32)
    assert len(lens_a) == n and len(Bs_a) == n
    cu_B = np.zeros(n + 1, np.int32)
    cu_B[1:] = np.cumsum(Bs_a)
    # 3 step labels
    tau = np.empty(int(cu_B[-1]), np.int32)
    for b in range(n):
        t = rng.permutation(int(Bs_a[b])) + 1
        if taus is not None and taus[b] is not None:
            t = np.asarray(taus[b])
        tau[cu_B[b]:cu_B[b + 1]] = t
    # 4 pages: each sequence needs ceil((P + 2B) / PAGE) pages
    pages = (lens_a + 2 * Bs_a + PAGE - 1) // PAGE
    num_pages = int(pages.sum())
    max_pages = int(pages.max())
    phys = rng.permutation(num_pages) if spec.shuffled_pages else np.arange(num_pages)
    block_table = np.zeros((n, max_pages), np.int32)
    o = 0
    for b in range(n):
        block_table[b, :pages[b]] = phys[o:o + pages[b]]
        o += int(pages[b])
    T = 2 * int(cu_B[-1])
    sumP = int(lens_a.sum())
    dt = spec.dtype
    # 5..9 activations
    q = _normal(rng, (T, spec.Hq, spec.hd), spec.qkv_sd * spec.q_scale, dt)
    k_prompt = _normal(rng, (sumP, spec.Hkv, spec.hd), spec.qkv_sd, dt)
    v_prompt = _normal(rng, (sumP, spec.Hkv, spec.hd), spec.qkv_sd, dt)
    k_new = _normal(rng, (T, spec.Hkv, spec.hd), spec.qkv_sd, dt)
    v_new = _normal(rng, (T, spec.Hkv, spec.hd), spec.qkv_sd, dt)
    target = draft = draft_tokens = uniforms = None
    if with_logits:
        nB = int(cu_B[-1])
        V = spec.vocab
        # 10 target logits
        t32 = rng.standard_normal(size=(nB, V), dtype=np.float32)
        t32 *= np.float32(spec.logit_sd)
        target = _store(t32, dt)
        # 11 per-sequence draft noise scale
        if isinstance(spec.noise_sd, tuple):
            sig = rng.uniform(spec.noise_sd[0], spec.noise_sd[1], size=n)
        else:
            sig = np.full(n, float(spec.noise_sd))
        sig_slot = np.repeat(sig, Bs_a).astype(np.float32)
        # 12 draft = target + noise (on the stored target values)
        noise = rng.standard_normal(size=(nB, V), dtype=np.float32)
        noise *= sig_slot[:, None]
        noise += (bf16_bits_to_f32(target) if dt == "bf16" else target)
        draft = _store(noise, dt)
        del noise, t32
        # 13 draft tokens: inverse CDF of the draft softmax with rng uniforms
        u_draft = rng.random(size=nB)
        draft_tokens = np.empty(nB, np.int32)
        d64 = to_f64(draft)
        for s in range(nB):
            row = d64[s]
            w = np.exp(row - row.max())
            c = np.cumsum(w)
            draft_tokens[s] = min(int(np.searchsorted(c, u_draft[s] * c[-1], side="right")), V - 1)
        del d64
        # 14 acceptance uniforms, fp32 in [0, 1)
        uniforms = rng.random(size=(n, int(Bs_a.max()) + 1), dtype=np.float32)
    return Workload(spec, seed, lens_a, Bs_a, cu_B, tau, num_pages, max_pages,
                    block_table, q, k_prompt, v_prompt, k_new, v_new, target,
                    draft, draft_tokens, uniforms)


def head(w: Workload, n: int) -> Workload:
    """The first n sequences of w as a workload of their own (array slices
    and the matching prefix of the block table; pages keep their ids)."""
    n = min(n, len(w.lens))
    off = w.prompt_offsets
    nB, T, nP = int(w.cu_B[n]), 2 * int(w.cu_B[n]), int(off[n])
    spec = dataclasses.replace(w.spec, batch=n)
    return Workload(spec, w.seed, w.lens[:n], w.Bs[:n], w.cu_B[:n + 1], w.tau[:nB],
                    w.num_pages, w.max_pages,
                    w.block_table[:n], w.q[:T], w.k_prompt[:nP], w.v_prompt[:nP],
                    w.k_new[:T], w.v_new[:T],
                    None if w.target is None else w.target[:nB],
                    None if w.draft is None else w.draft[:nB],
                    None if w.draft_tokens is None else w.draft_tokens[:nB],
                    None if w.uniforms is None else w.uniforms[:n])


def config(i: int, **kw) -> Workload:
    """Workload of configuration i with seed i."""
    return make(CONFIGS[i], seed=i, **kw)


def paged(w: Workload, x_prompt: np.ndarray) -> np.ndarray:
    """Scatter prompt rows [sum P, Hkv, hd] into a zero-filled physical cache
    [num_pages, Hkv, PAGE, hd] through the block table (slots past P stay 0)."""
    Hkv, hd = x_prompt.shape[1], x_prompt.shape[2]
    cache = np.zeros((w.num_pages, Hkv, PAGE, hd), x_prompt.dtype)
    off = w.prompt_offsets
    for b in range(len(w.lens)):
        P = int(w.lens[b])
        for p0 in range(0, P, PAGE):
            n_tok = min(PAGE, P - p0)
            page = w.block_table[b, p0 // PAGE]
            rows = x_prompt[off[b] + p0: off[b] + p0 + n_tok]      # [n, Hkv, hd]
            cache[page, :, :n_tok, :] = rows.transpose(1, 0, 2)
    return cache
