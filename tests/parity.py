"""Shared helpers of the GPU parity tests: oracle results for a synthetic
workload and the comparison rules.

Tolerances (from the stated targets): attention rows agree within a max
relative error of 2e-2 with bf16 inputs/outputs and 1e-4 with fp32, where a
row's error is max|o_gpu - o_ref| / max|o_ref| over its head dimension.
Acceptance decisions are compared exactly except in the tie zone: a step
whose oracle margin |u q(x) - p(x)| / p(x) is below 1e-5, or a residual draw
whose inverse-CDF threshold lies within 1e-5 (relative to the residual
mass) of a bin edge, may flip under fp32 rounding; there the GPU result is
only checked for validity.
"""
import numpy as np

import oracle
import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}
TIE = 1e-5


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


def oracle_accept(w):
    return oracle.accept(w.cu_B, synth.to_f64(w.target), synth.to_f64(w.draft),
                         w.draft_tokens, w.tau, w.uniforms)


def check_accept(w, ref, n_accept, token, pos):
    """Exact agreement outside the tie zone; validity inside it.
    Returns the number of sequences decided in the tie zone."""
    ties = 0
    am, rm = ref["accept_margin"], ref["resample_margin"]
    for b in range(len(w.lens)):
        s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
        B = s1 - s0
        tested = am[s0:s1]
        tie_step = (tested >= 0) & (tested < TIE)
        if tie_step.any():
            ties += 1
            assert 0 <= n_accept[b] <= B
            continue
        assert n_accept[b] == ref["n_accept"][b], (b, n_accept[b], ref["n_accept"][b])
        assert pos[b] == ref["pos"][b], (b, pos[b], ref["pos"][b])
        if ref["pos"][b] < 0:
            assert token[b] == -1
            continue
        if 0 <= rm[b] < TIE:
            ties += 1
            assert 0 <= token[b] < w.spec.vocab
            continue
        assert token[b] == ref["token"][b], (b, token[b], ref["token"][b])
    return ties
