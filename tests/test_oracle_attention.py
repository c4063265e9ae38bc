"""Pins for the oracle's RoPE and masked verification attention.

Pinned against: closed forms of the rotation (angle, norm, composition,
relative-position property), a textbook library routine (torch's
scaled_dot_product_attention in fp64 on the CPU, with the mask built from a
decoding simulation and RoPE written as complex multiplication), and the
invariances the temporal mask implies.
"""
import numpy as np
import pytest
import torch

import oracle


def complex_rope(x, pos, base):
    """Rotate-half RoPE as complex multiplication: z_d = x_d + i x_{d+hd/2}
    times exp(i pos base^(-2d/hd)) -- an independent route to the rotation."""
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    d = np.arange(half)
    ang = np.asarray(pos, np.float64)[:, None] * (float(base) ** (-2.0 * d / hd))[None, :]
    z = z * np.exp(1j * ang)[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_angle_closed_form():
    # hd = 2: a single pair rotated by exactly pos radians
    x = np.array([[[1.0, 0.0]], [[1.0, 0.0]], [[0.0, 1.0]]])
    pos = np.array([0, 1, 5])
    y = oracle.rope(x, pos, 10000.0)
    np.testing.assert_allclose(y[0, 0], [1.0, 0.0], atol=0)
    np.testing.assert_allclose(y[1, 0], [np.cos(1.0), np.sin(1.0)], rtol=1e-15)
    np.testing.assert_allclose(y[2, 0], [-np.sin(5.0), np.cos(5.0)], rtol=1e-15)
    # hd = 4: the second pair turns at pos * base^(-1/2)
    x = np.zeros((1, 1, 4)); x[0, 0, 1] = 1.0
    y = oracle.rope(x, [7], 100.0)
    np.testing.assert_allclose(y[0, 0], [0, np.cos(0.7), 0, np.sin(0.7)], atol=1e-15)


def test_rope_matches_complex_form_norm_and_composition():
    rng = np.random.default_rng(0)
    for hd, base in ((64, 1e4), (128, 1e6)):
        x = rng.standard_normal((9, 3, hd))
        pos = rng.integers(0, 40000, 9)
        y = oracle.rope(x, pos, base)
        # angles up to 4e4 rad carry ~1e-12 rad of fp64 rounding in either route
        np.testing.assert_allclose(y, complex_rope(x, pos, base), rtol=0, atol=1e-10)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
        a, b = rng.integers(0, 1000, 9), rng.integers(0, 1000, 9)
        np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, base), b, base),
                                   oracle.rope(x, a + b, base), rtol=1e-10, atol=1e-10)
        # relative position: <R(m) q, R(n) k> depends on m - n only
        q, k = rng.standard_normal((1, 1, hd)), rng.standard_normal((1, 1, hd))
        d1 = (oracle.rope(q, [100], base) * oracle.rope(k, [37], base)).sum()
        d2 = (oracle.rope(q, [1063], base) * oracle.rope(k, [1000], base)).sum()
        assert abs(d1 - d2) < 1e-10


def mask_from_simulation(P, B, tau):
    """Visible-column mask of the 2B new rows, by walking the decode steps."""
    L = P + 2 * B
    m = np.zeros((2 * B, L), bool)
    m[:, :P] = True
    revealed = set()
    for s in range(1, B + 1):
        (i,) = [j for j in range(B) if tau[j] == s]
        for j in revealed:
            m[B + i, P + j] = True
        for j in range(B):
            if tau[j] >= s:
                m[B + i, P + B + j] = True
        revealed.add(i)
        for j in revealed:
            m[i, P + j] = True
    return m


def sdpa_reference(q, kp, vp, kn, vn, tau, base, scale):
    """torch SDPA (fp64, CPU) on the paired layout."""
    twoB, Hq, hd = q.shape
    B = twoB // 2
    P, Hkv = kp.shape[0], kn.shape[1]
    new_pos = np.concatenate([P + np.arange(B), P + np.arange(B)])
    qr = complex_rope(q, new_pos, base)
    knr = complex_rope(kn, new_pos, base)
    K = np.concatenate([kp, knr], 0)            # [L, Hkv, hd]
    V = np.concatenate([vp, vn], 0)
    G = Hq // Hkv
    K = np.repeat(K, G, axis=1).transpose(1, 0, 2)  # [Hq, L, hd]
    V = np.repeat(V, G, axis=1).transpose(1, 0, 2)
    Q = qr.transpose(1, 0, 2)                       # [Hq, 2B, hd]
    mask = torch.from_numpy(mask_from_simulation(P, B, tau))
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=mask, scale=scale)
    return out.numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("P,B,Hq,Hkv,hd", [(0, 1, 2, 1, 8), (5, 3, 4, 2, 16),
                                          (37, 4, 4, 2, 64), (20, 8, 8, 2, 32)])
def test_attention_matches_library_sdpa(P, B, Hq, Hkv, hd):
    rng = np.random.default_rng(P * 100 + B)
    tau = rng.permutation(B) + 1
    q = rng.standard_normal((2 * B, Hq, hd))
    kp, vp = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((P, Hkv, hd))
    kn, vn = rng.standard_normal((2 * B, Hkv, hd)), rng.standard_normal((2 * B, Hkv, hd))
    scale = 1.0 / np.sqrt(hd)
    got = oracle.verify_attn_seq(q, kp if P else None, vp if P else None, kn, vn,
                                 tau, 1e4, scale)
    ref = sdpa_reference(q, kp, vp, kn, vn, tau, 1e4, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    # selected rows agree with the full computation
    rows = [(t, h) for t in range(2 * B) for h in range(Hq)][::3]
    sel = oracle.verify_attn_seq(q, kp if P else None, vp if P else None, kn, vn,
                                 tau, 1e4, scale, rows=rows)
    np.testing.assert_array_equal(sel, np.array([got[t, h] for t, h in rows]))


def test_masked_keys_do_not_matter():
    """Perturbing D_j with tau(j) >= tau(i) or D~_j with tau(j) < tau(i) leaves
    slot i's output bit-identical; perturbing a visible key changes it."""
    rng = np.random.default_rng(11)
    P, B, Hq, Hkv, hd = 9, 6, 4, 2, 16
    tau = rng.permutation(B) + 1
    q = rng.standard_normal((2 * B, Hq, hd))
    kp, vp = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((P, Hkv, hd))
    kn, vn = rng.standard_normal((2 * B, Hkv, hd)), rng.standard_normal((2 * B, Hkv, hd))
    base = oracle.verify_attn_seq(q, kp, vp, kn, vn, tau, 1e4, 0.25)
    for i in range(B):
        for j in range(B):
            for tok, hidden in ((j, tau[j] >= tau[i]), (B + j, tau[j] < tau[i])):
                kn2, vn2 = kn.copy(), vn.copy()
                kn2[tok] += 3.0
                vn2[tok] -= 2.0
                out = oracle.verify_attn_seq(q, kp, vp, kn2, vn2, tau, 1e4, 0.25)
                if hidden:
                    np.testing.assert_array_equal(out[B + i], base[B + i])
                else:
                    assert np.abs(out[B + i] - base[B + i]).max() > 1e-6


def test_single_visible_key_and_equal_keys():
    rng = np.random.default_rng(5)
    Hq, Hkv, hd = 2, 1, 8
    # P = 0, B = 1: D_1 sees only itself and D~_1 sees only itself
    q = rng.standard_normal((2, Hq, hd))
    kn, vn = rng.standard_normal((2, Hkv, hd)), rng.standard_normal((2, Hkv, hd))
    out = oracle.verify_attn_seq(q, None, None, kn, vn, [1], 1e4, 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], vn[0, 0], rtol=1e-15)
        np.testing.assert_allclose(out[1, h], vn[1, 0], rtol=1e-15)
    # equal (zero) keys: every visible value weighs the same
    P, B = 5, 3
    tau = np.array([2, 3, 1])
    q = rng.standard_normal((2 * B, Hq, hd))
    kp = np.zeros((P, Hkv, hd)); kn = np.zeros((2 * B, Hkv, hd))
    vp, vn = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((2 * B, Hkv, hd))
    out = oracle.verify_attn_seq(q, kp, vp, kn, vn, tau, 1e4, 1.0)
    _, m = oracle.layout(P, tau)
    allv = np.concatenate([vp, vn], 0)[:, 0, :]
    for r in range(2 * B):
        np.testing.assert_allclose(out[r, 0], allv[m[r].astype(bool)].mean(0), rtol=1e-13)


def test_position_shift_invariance():
    """Adding one offset to every position (prompt keys rotated at the
    shifted positions too) leaves every output unchanged."""
    rng = np.random.default_rng(2)
    P, B, Hq, Hkv, hd, base = 12, 4, 4, 2, 32, 1e4
    tau = rng.permutation(B) + 1
    q = rng.standard_normal((2 * B, Hq, hd))
    kp_raw, vp = rng.standard_normal((P, Hkv, hd)), rng.standard_normal((P, Hkv, hd))
    kn, vn = rng.standard_normal((2 * B, Hkv, hd)), rng.standard_normal((2 * B, Hkv, hd))
    outs = []
    for s in (0, 17, 4000):
        kp = oracle.rope(kp_raw, s + np.arange(P), base)
        outs.append(oracle.verify_attn_seq(q, kp, vp, kn, vn, tau, base, 0.2, pos_offset=s))
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-9, atol=1e-11)


def test_batch_matches_per_sequence():
    rng = np.random.default_rng(4)
    lens = np.array([3, 0, 10]); Bs = np.array([2, 1, 4])
    cu = np.concatenate([[0], np.cumsum(Bs)])
    Hq, Hkv, hd = 4, 2, 8
    T = 2 * cu[-1]
    q = rng.standard_normal((T, Hq, hd))
    kp, vp = rng.standard_normal((lens.sum(), Hkv, hd)), rng.standard_normal((lens.sum(), Hkv, hd))
    kn, vn = rng.standard_normal((T, Hkv, hd)), rng.standard_normal((T, Hkv, hd))
    tau = np.concatenate([rng.permutation(b) + 1 for b in Bs])
    out = oracle.verify_attn(lens, cu, q, kp, vp, kn, vn, tau, 1e4, 0.3, n_threads=2)
    po = np.concatenate([[0], np.cumsum(lens)])
    for b in range(3):
        t0, t1 = 2 * cu[b], 2 * cu[b + 1]
        ref = oracle.verify_attn_seq(q[t0:t1], kp[po[b]:po[b + 1]] if lens[b] else None,
                                     vp[po[b]:po[b + 1]] if lens[b] else None,
                                     kn[t0:t1], vn[t0:t1], tau[cu[b]:cu[b + 1]], 1e4, 0.3)
        np.testing.assert_array_equal(out[t0:t1], ref)
