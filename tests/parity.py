"""Shared helpers of the GPU parity tests: oracle results for a synthetic
workload and the comparison rules.

Tolerances (from the stated targets): attention rows agree within a max
relative error of 2e-2 with bf16 inputs/outputs and 1e-4 with fp32, where a
row's error is max|o_gpu - o_ref| / max|o_ref| over its head dimension.
Acceptance decisions are compared exactly except in the tie zone, where
fp32 rounding on the GPU may legitimately flip them:
  - a step whose oracle margin |u q(x) - p(x)| / p(x) is below TIE_ACCEPT
    (the GPU's p(x), q(x) carry up to ~1.5e-6 relative error: exponent
    argument rounding up to half an ulp of |x - max| log2 e <= ~40, exp2's
    approximation, the normaliser);
  - an inverse-CDF draw (the residual draw, sample matching's draw, the
    draft step's draw) whose threshold lies within TIE_RESIDUAL (absolute
    probability mass) of a bin edge of the oracle's fp64 CDF.  What can move
    the GPU's CDF against the exact one by a consistent amount is what
    every entry shares: the logit scale log2(e)/T (carried as a float pair,
    ~1e-15 relative) and the normalisers (the residual is drawn in
    target-mass units with the ratio of the normalisers as a pair, so none
    is rounded into the entries).  Per-entry rounding (the exponent
    argument, exp2's approximation, products; ~3e-7 relative each) is
    uncorrelated across entries: over a CDF of n entries of mass m_v it
    moves a sum by ~3e-7 sqrt(sum m_v^2), below 1e-9 for these rows.  The
    running sums are compensated fp32 pairs.  1e-8 leaves a margin of ten
    over that; measured on the five workloads, the GPU agreed with the
    oracle on every draw, down to a distance of 1.1e-9 from a bin edge.
Inside the tie zone the GPU's result must still be valid: an accepted length
consistent with the steps decided outside the zone, and a drawn token with
positive residual mass whose CDF bin lies within TIE_RESIDUAL of u*S.
"""
import numpy as np

import oracle
import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}
TIE_ACCEPT = 5e-6
TIE_RESIDUAL = 1e-8


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


def oracle_full_size(w, seqs_per_call=32, n_threads=0):
    """Oracle attention of every row of a large workload, in bounded memory:
    batches of sequences through the OpenMP oracle (parallel over
    sequences); workloads with fewer sequences than threads split each
    sequence's rows over a thread pool instead (ctypes calls release the
    interpreter lock)."""
    import concurrent.futures
    nt = n_threads or oracle.default_threads()
    if len(w.lens) >= nt:
        outs = []
        for b0 in range(0, len(w.lens), seqs_per_call):
            b1 = min(len(w.lens), b0 + seqs_per_call)
            sub = synth.head(w, b1) if b1 < len(w.lens) else w
            off = sub.prompt_offsets
            t0, t1 = 2 * int(sub.cu_B[b0]), 2 * int(sub.cu_B[b1])
            lens = sub.lens[b0:b1]
            cu = (sub.cu_B[b0:b1 + 1] - sub.cu_B[b0]).astype(np.int32)
            outs.append(oracle.verify_attn(
                lens, cu, synth.to_f64(sub.q[t0:t1]),
                synth.to_f64(sub.k_prompt[off[b0]:off[b1]]),
                synth.to_f64(sub.v_prompt[off[b0]:off[b1]]),
                synth.to_f64(sub.k_new[t0:t1]), synth.to_f64(sub.v_new[t0:t1]),
                sub.tau[sub.cu_B[b0]:sub.cu_B[b1]], w.spec.rope_base, w.spec.sm_scale,
                n_threads=nt))
        return np.concatenate(outs, 0)
    Hq = w.spec.Hq
    outs = []
    with concurrent.futures.ThreadPoolExecutor(nt) as ex:
        for b in range(len(w.lens)):
            twoB = 2 * int(w.Bs[b])
            rows = [(t, h) for t in range(twoB) for h in range(Hq)]
            chunks = [rows[i:i + 8] for i in range(0, len(rows), 8)]
            off = w.prompt_offsets
            t0, t1 = 2 * int(w.cu_B[b]), 2 * int(w.cu_B[b + 1])
            P = int(w.lens[b])
            kp = prompt_keys_f64(w, b)
            vp = synth.to_f64(w.v_prompt[off[b]:off[b + 1]])
            q = synth.to_f64(w.q[t0:t1])
            kn, vn = synth.to_f64(w.k_new[t0:t1]), synth.to_f64(w.v_new[t0:t1])
            tau = w.tau[w.cu_B[b]:w.cu_B[b + 1]]
            parts = list(ex.map(lambda rs: oracle.verify_attn_seq(
                q, kp if P else None, vp if P else None, kn, vn, tau, w.spec.rope_base,
                w.spec.sm_scale, rows=rs), chunks))
            outs.append(np.concatenate(parts, 0).reshape(twoB, Hq, -1))
    return np.concatenate(outs, 0)


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


def check_accept(w, ref, n_accept, token, pos, temperature=1.0, stats=None):
    """Exact agreement outside the tie zone; validity inside it.
    Returns (accept-step ties, residual-draw ties, residual draws).
    stats (a list, optional) receives (distance of u*S to the nearest edge
    of the oracle's bin in absolute mass, GPU token == oracle token) for
    every residual draw."""
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
        if stats is not None:
            stats.append((min(U - lo, C[v] - U), int(token[b]) == v))
        if min(U - lo, C[v] - U) >= TIE_RESIDUAL:
            assert token[b] == v, (b, token[b], v)
            continue
        draw_ties += 1
        g = int(token[b])
        assert 0 <= g < V and r[g] > 0, (b, g)
        glo = C[g - 1] if g > 0 else 0.0
        assert glo - TIE_RESIDUAL <= U < C[g] + TIE_RESIDUAL, (b, g, v, U, glo, C[g])
    return step_ties, draw_ties, draws


def max_ties(decisions):
    """Tie-zone decisions a test allows: 2% of the decisions, at least one."""
    return max(1, int(0.02 * decisions))


def tie_report(stats):
    """Summary of check_accept's per-draw stats: draws, the smallest edge
    distance at which the GPU disagreed (inf if never), and how many draws
    fall within each distance."""
    d = np.array([x[0] for x in stats]) if stats else np.zeros(0)
    agree = np.array([x[1] for x in stats], bool) if stats else np.zeros(0, bool)
    worst = float(d[~agree].max()) if (~agree).any() else float("inf")
    near = {t: int((d < t).sum()) for t in (1e-8, 3e-8, 1e-7, 3e-7, 1e-6, 2e-6)}
    return dict(draws=int(d.size), disagree=int((~agree).sum()), worst_disagree=worst,
                min_dist=float(d.min()) if d.size else float("inf"), near=near)
