"""Pins for the oracle's draft-graph verification (Spiffy, "Metodologia:
Spiffy": several draft candidates verified in parallel under a custom
blockwise attention mask; reading: each node a complete candidate state of
the block, attending to the prompt and to its own node).

Pinned against: the mask's closed form, a textbook library routine (torch's
scaled_dot_product_attention in fp64, unmasked, on one node at a time, RoPE
written as complex multiplication), and the invariances the block-diagonal
mask implies (node independence, identical nodes, shift of all positions).
"""
import numpy as np
import torch

import oracle
from test_oracle_attention import complex_rope


def rand(rng, *shape):
    return rng.standard_normal(shape) / 4.0


def test_mask_closed_form():
    for P, N, S in ((0, 1, 1), (3, 2, 4), (17, 5, 3), (1, 4, 8)):
        m = oracle.graph_mask(P, N, S)
        assert m.shape == (N * S, P + N * S)
        assert (m[:, :P] == 1).all()
        new = m[:, P:]
        np.testing.assert_array_equal(new, np.kron(np.eye(N, dtype=np.uint8), np.ones((S, S), np.uint8)))
        assert (m.sum(1) == P + S).all()            # every row: the prompt and its node


def sdpa_one_node(q, kp, vp, kn, vn, P, S, base, scale):
    """One node by the library routine: rotated q and keys at positions
    P + k (complex form), no mask over [prompt | node]."""
    pos = P + np.arange(S)
    qr = complex_rope(q, pos, base)
    kr = complex_rope(kn, pos, base)
    K = np.concatenate([kp, kr]) if P else kr
    Vv = np.concatenate([vp, vn]) if P else vn
    Hq, Hkv = q.shape[1], kn.shape[1]
    G = Hq // Hkv
    Kt = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), G, 0))     # [Hq, L, hd]
    Vt = torch.from_numpy(np.repeat(Vv.transpose(1, 0, 2), G, 0))
    Qt = torch.from_numpy(qr.transpose(1, 0, 2))                      # [Hq, S, hd]
    o = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, scale=scale)
    return o.numpy().transpose(1, 0, 2)


def test_each_node_is_plain_attention_over_prompt_and_itself():
    rng = np.random.default_rng(70)
    for P, N, S, Hq, Hkv, hd in ((0, 1, 5, 2, 1, 8), (9, 3, 4, 4, 2, 16), (33, 4, 8, 8, 2, 64)):
        base, scale = 1e4, 0.7
        kp = complex_rope(rand(rng, P, Hkv, hd), np.arange(P), base) if P else None
        vp = rand(rng, P, Hkv, hd) if P else None
        q, kn, vn = rand(rng, N * S, Hq, hd), rand(rng, N * S, Hkv, hd), rand(rng, N * S, Hkv, hd)
        out = oracle.verify_attn_graph_seq(q, kp, vp, kn, vn, S, base, scale)
        for n in range(N):
            sl = slice(n * S, (n + 1) * S)
            ref = sdpa_one_node(q[sl], kp, vp, kn[sl], vn[sl], P, S, base, scale)
            np.testing.assert_allclose(out[sl], ref, rtol=1e-11, atol=1e-13)


def test_nodes_do_not_see_each_other():
    """Changing one node's keys and values leaves every other node's rows
    bit-identical (masked keys contribute exact zeros)."""
    rng = np.random.default_rng(71)
    P, N, S, Hq, Hkv, hd = 20, 4, 6, 4, 2, 32
    kp, vp = rand(rng, P, Hkv, hd), rand(rng, P, Hkv, hd)
    q, kn, vn = rand(rng, N * S, Hq, hd), rand(rng, N * S, Hkv, hd), rand(rng, N * S, Hkv, hd)
    base = oracle.verify_attn_graph_seq(q, kp, vp, kn, vn, S, 1e6, 1.0)
    for m in range(N):
        kn2, vn2 = kn.copy(), vn.copy()
        kn2[m * S:(m + 1) * S] += 3.0
        vn2[m * S:(m + 1) * S] -= 2.0
        got = oracle.verify_attn_graph_seq(q, kp, vp, kn2, vn2, S, 1e6, 1.0)
        for n in range(N):
            sl = slice(n * S, (n + 1) * S)
            if n == m:
                assert np.abs(got[sl] - base[sl]).max() > 1e-3
            else:
                np.testing.assert_array_equal(got[sl], base[sl])


def test_identical_nodes_give_identical_rows():
    rng = np.random.default_rng(72)
    P, N, S, Hq, Hkv, hd = 11, 3, 5, 2, 2, 16
    kp, vp = rand(rng, P, Hkv, hd), rand(rng, P, Hkv, hd)
    q1, k1, v1 = rand(rng, S, Hq, hd), rand(rng, S, Hkv, hd), rand(rng, S, Hkv, hd)
    out = oracle.verify_attn_graph_seq(np.tile(q1, (N, 1, 1)), kp, vp, np.tile(k1, (N, 1, 1)),
                                       np.tile(v1, (N, 1, 1)), S, 1e4, 0.5)
    for n in range(1, N):
        np.testing.assert_array_equal(out[n * S:(n + 1) * S], out[:S])


def test_shift_of_all_positions_changes_nothing():
    """Rotating the prompt keys from position s on instead of 0 (and the
    nodes from P + s) leaves the outputs unchanged: RoPE sees only the
    differences of positions."""
    rng = np.random.default_rng(73)
    P, N, S, Hq, Hkv, hd, b = 15, 2, 4, 2, 1, 32, 1e4
    kraw, vp = rand(rng, P, Hkv, hd), rand(rng, P, Hkv, hd)
    q, kn, vn = rand(rng, N * S, Hq, hd), rand(rng, N * S, Hkv, hd), rand(rng, N * S, Hkv, hd)
    a = oracle.verify_attn_graph_seq(q, oracle.rope(kraw, np.arange(P), b), vp, kn, vn, S, b, 1.0)
    # the same layout shifted by s: the prompt keys and every node's q and
    # keys rotated at +s, attention written out directly
    s = 1000
    kp_s = oracle.rope(kraw, s + np.arange(P), b)
    qs = oracle.rope(q, s + np.tile(P + np.arange(S), N), b)
    ks = oracle.rope(kn, s + np.tile(P + np.arange(S), N), b)
    for n in range(N):
        sl = slice(n * S, (n + 1) * S)
        K = np.concatenate([kp_s, ks[sl]])
        V = np.concatenate([vp, vn[sl]])
        sc = np.einsum("thd,lhd->thl", qs[sl], np.repeat(K, Hq // Hkv, 1))
        w = np.exp(sc - sc.max(-1, keepdims=True))
        w /= w.sum(-1, keepdims=True)
        ref = np.einsum("thl,lhd->thd", w, np.repeat(V, Hq // Hkv, 1))
        np.testing.assert_allclose(a[sl], ref, rtol=1e-9, atol=1e-11)
