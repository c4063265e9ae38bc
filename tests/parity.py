"""Shared helpers of the GPU parity tests: oracle results for a synthetic
workload and the comparison rules.

Tolerances (from the stated targets): attention rows agree within a max
relative error of 2e-2 with bf16 inputs/outputs and 1e-4 with fp32, where a
row's error is max|o_gpu - o_ref| / max|o_ref| over its head dimension.
Acceptance decisions are compared exactly except in the tie zone, where
fp32 rounding on the GPU may legitimately flip them:
  - a step whose oracle margin |u q(x) - p(x)| / p(x) is below TIE_ACCEPT
    (the GPU's p(x), q(x) carry up to ~1.5e-6 relative error: exponent
    argument rounding up to half an ulp of |x - max| log2 e <= ~40, exp2f's
    2 ulp, the normaliser);
  - a residual draw whose threshold u*S lies within TIE_RESIDUAL (absolute
    probability mass) of a bin edge of the oracle's fp64 CDF (each residual
    entry carries ~3e-7 relative error weighted by mass, so the GPU's CDF is
    within ~6e-7 of the exact one; fp64 sums add nothing comparable).
Inside the tie zone the GPU's result must still be valid: an accepted length
consistent with the steps decided outside the zone, and a drawn token with
positive residual mass whose CDF bin lies within TIE_RESIDUAL of u*S.
"""
import numpy as np

import oracle
import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}
TIE_ACCEPT = 5e-6
TIE_RESIDUAL = 2e-6


def prompt_keys_f64(w, b):
    """Rotated prompt keys of sequence b in fp64 (rotating raw keys with the
    oracle when the workload stores them raw)."""
    off = w.prompt_offsets
    kp = synth.to_f64(w.k_prompt[off[b]:off[b + 1]])
    if w.spec.raw_prompt_keys and len(kp):
        kp = oracle.rope(kp, np.arange(len(kp)), w.spec.rope_base)
    return kp


def oracle_seq(w, b, rows=None):
    """Oracle attention of sequence b: every row ([2B, Hq, hd]) or the given
    (token, head) pairs ([n, hd])."""
    off = w.prompt_offsets
    t0, t1 = 2 * int(w.cu_B[b]), 2 * int(w.cu_B[b + 1])
    P = int(w.lens[b])
    kp = prompt_keys_f64(w, b)
    vp = synth.to_f64(w.v_prompt[off[b]:off[b + 1]])
    return oracle.verify_attn_seq(
        synth.to_f64(w.q[t0:t1]), kp if P else None, vp if P else None,
        synth.to_f64(w.k_new[t0:t1]), synth.to_f64(w.v_new[t0:t1]),
        w.tau[w.cu_B[b]:w.cu_B[b + 1]], w.spec.rope_base, w.spec.sm_scale,
        rows=rows)


def oracle_all(w, n_threads=0):
    if not w.spec.raw_prompt_keys:
        return oracle.verify_attn(w.lens, w.cu_B, synth.to_f64(w.q), synth.to_f64(w.k_prompt),
                                  synth.to_f64(w.v_prompt), synth.to_f64(w.k_new),
                                  synth.to_f64(w.v_new), w.tau, w.spec.rope_base,
                                  w.spec.sm_scale, n_threads=n_threads)
    return np.concatenate([oracle_seq(w, b) for b in range(len(w.lens))], 0)


def row_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref).max(-1) / np.abs(ref).max(-1)


def check_attention(got, ref, dtype):
    err = row_errors(got, ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert err.max() <= TOL[dtype], "max row rel err %.3g > %g" % (err.max(), TOL[dtype])
    return err


def oracle_accept(w, temperature=1.0):
    return oracle.accept(w.cu_B, synth.to_f64(w.target), synth.to_f64(w.draft),
                         w.draft_tokens, w.tau, w.uniforms, temperature=temperature)


def check_accept(w, ref, n_accept, token, pos, temperature=1.0):
    """Exact agreement outside the tie zone; validity inside it.
    Returns (accept-step ties, residual-draw ties, residual draws)."""
    am = ref["accept_margin"]
    V = w.spec.vocab
    step_ties = draw_ties = draws = 0
    for b in range(len(w.lens)):
        s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
        B = s1 - s0
        tested = am[s0:s1]
        if ((tested >= 0) & (tested < TIE_ACCEPT)).any():
            step_ties += 1
            assert 0 <= n_accept[b] <= B
            if pos[b] >= 0:
                assert n_accept[b] < B and 0 <= token[b] < V
            continue
        assert n_accept[b] == ref["n_accept"][b], (b, n_accept[b], ref["n_accept"][b])
        assert pos[b] == ref["pos"][b], (b, pos[b], ref["pos"][b])
        if ref["pos"][b] < 0:
            assert token[b] == -1
            continue
        draws += 1
        k = s0 + int(ref["pos"][b])
        r, S = oracle.residual(synth.to_f64(w.target[k]) / temperature,
                               synth.to_f64(w.draft[k]) / temperature)
        C = np.cumsum(r)
        U = float(w.uniforms[b, B]) * S
        v = int(ref["token"][b])
        lo = C[v - 1] if v > 0 else 0.0
        if min(U - lo, C[v] - U) >= TIE_RESIDUAL:
            assert token[b] == v, (b, token[b], v)
            continue
        draw_ties += 1
        g = int(token[b])
        assert 0 <= g < V and r[g] > 0, (b, g)
        glo = C[g - 1] if g > 0 else 0.0
        assert glo - TIE_RESIDUAL <= U < C[g] + TIE_RESIDUAL, (b, g, v, U, glo, C[g])
    return step_ties, draw_ties, draws
