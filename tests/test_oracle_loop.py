"""Pins of the blockwise loop in the oracle (draft step -> acceptance ->
commit, repeated): hand-walked passes, the loop's invariants, and the
distribution of a finished block's tokens.

SimSD "Speculative Decoding Pipeline": the longest accepted prefix is
committed and the process repeats; the reading of a pass is in
oracle/loop.py.
"""
import numpy as np

import oracle
from oracle import loop

NEG = np.log(1e-300)   # a logit whose probability is negligible (not -inf)


def rows_of(probs):
    p = np.asarray(probs, np.float64)
    return np.where(p > 0, np.log(np.maximum(p, 1e-300)), NEG)


def test_two_passes_by_hand():
    """B = 4, V = 4.  Pass 1: the draft's tokens are 0, 1, 2, 2 with
    confidences 0.9, 0.6, 1.0, 0.25, so tau = (2, 3, 1, 4); step 1 (slot 2,
    p = q) accepts; step 2 (slot 0: p(0) = 0.45, q(0) = 0.9, u = 0.7)
    rejects and draws from max(0, p - q) = (0, 0.45, 0, 0): token 1 at
    slot 0, two positions decided.  Pass 2: slots 1 and 3 are open (tokens
    3 and 1, confidences 1 and 0.5: labels 3 and 4); the walk starts at
    step 3 and accepts both; nothing is drawn, so the block closes and lens
    advances by B."""
    cu = np.array([0, 4], np.int32)
    st = loop.initial_state(cu, [10])
    d1 = rows_of([[0.9, 0.1, 0, 0], [0, 0.6, 0.4, 0], [0, 0, 1, 0], [0.25] * 4])
    t1 = rows_of([[0.45, 0.55, 0, 0], [0, 0.6, 0.4, 0], [0, 0, 1, 0], [0.25] * 4])
    ud1 = np.array([[0.5, 0.3, 0.5, 0.6]], np.float32)
    ua1 = np.array([[0.2, 0.7, 0.1, 0.1, 0.5]], np.float32)
    st, r1 = loop.blockwise_pass(cu, st, d1, t1, ud1, ua1)
    np.testing.assert_array_equal(r1["draft_tokens"], [0, 1, 2, 2])
    np.testing.assert_array_equal(r1["tau"], [2, 3, 1, 4])
    assert (r1["n_accept"][0], r1["pos"][0], r1["token"][0]) == (1, 0, 1)
    np.testing.assert_array_equal(st["block_tokens"], [1, 1, 2, 2])
    assert st["decided"][0] == 2 and st["lens"][0] == 10 and r1["done"][0] == 0
    d2 = rows_of([[0.25] * 4, [0, 0, 0, 1], [0.25] * 4, [0.5, 0.5, 0, 0]])
    t2 = rows_of([[0.25] * 4, [0, 0, 0, 1], [0.25] * 4, [0.5, 0.5, 0, 0]])
    ud2 = np.array([[0.99, 0.5, 0.99, 0.7]], np.float32)
    ua2 = np.array([[0.99, 0.99, 0.5, 0.5, 0.5]], np.float32)
    st, r2 = loop.blockwise_pass(cu, st, d2, t2, ud2, ua2)
    # decided slots 0 and 2 keep tokens and labels; u there is never read
    np.testing.assert_array_equal(r2["draft_tokens"], [1, 3, 2, 1])
    np.testing.assert_array_equal(r2["tau"], [2, 3, 1, 4])
    assert r2["first_step"][0] == 3
    assert (r2["n_accept"][0], r2["pos"][0], r2["token"][0]) == (4, -1, -1)
    assert r2["done"][0] == 1 and st["lens"][0] == 14 and st["decided"][0] == 0
    np.testing.assert_array_equal(r2["block_tokens"], [1, 3, 2, 1])
    assert r2["confidence"][0] == -1 and r2["confidence"][2] == -1


def test_block_finished_by_a_draw_takes_a_closing_pass():
    """B = 2: pass 1 accepts step 1 and rejects step 2, deciding both
    positions by a draw; the block is not closed (the cache holds the
    draft's token there) until a pass that tests nothing (first step 3)."""
    cu = np.array([0, 2], np.int32)
    st = loop.initial_state(cu, [0])
    d = rows_of([[1, 0, 0], [0.5, 0.5, 0]])
    t = rows_of([[1, 0, 0], [0, 0, 1]])
    ud = np.array([[0.5, 0.2]], np.float32)      # slot 1 drafts token 0
    ua = np.array([[0.5, 0.5, 0.5]], np.float32)
    st, r1 = loop.blockwise_pass(cu, st, d, t, ud, ua)
    np.testing.assert_array_equal(r1["tau"], [1, 2])
    assert (r1["n_accept"][0], r1["pos"][0], r1["token"][0]) == (1, 1, 2)
    assert st["decided"][0] == 2 and r1["done"][0] == 0 and st["lens"][0] == 0
    st, r2 = loop.blockwise_pass(cu, st, d, t, ud, ua)
    assert r2["first_step"][0] == 3 and r2["n_accept"][0] == 2 and r2["pos"][0] == -1
    assert r2["done"][0] == 1 and st["lens"][0] == 2
    np.testing.assert_array_equal(r2["block_tokens"], [0, 2])


def test_loop_invariants():
    """Random blocks (B = 1..8): every pass either decides at least one more
    position or closes the block; decided positions keep their tokens and
    labels; tau stays a permutation; a block closes within B + 1 passes with
    every position decided."""
    rng = np.random.default_rng(40)
    n, V = 300, 12
    Bs = rng.integers(1, 9, n)
    cu = np.concatenate([[0], np.cumsum(Bs)]).astype(np.int32)
    st = loop.initial_state(cu, rng.integers(0, 50, n))
    closed = np.zeros(n, bool)
    passes = np.zeros(n, int)
    for it in range(10):
        dl = rng.standard_normal((int(cu[-1]), V)) * 2
        tl = dl + rng.standard_normal(dl.shape) * rng.uniform(0.2, 3)
        prev = {k: v.copy() for k, v in st.items()}
        st, r = loop.blockwise_pass(cu, st, dl, tl, rng.random((n, 8), dtype=np.float32),
                                    rng.random((n, 9), dtype=np.float32))
        for b in range(n):
            if closed[b]:
                continue
            s0, s1 = cu[b], cu[b + 1]
            B = s1 - s0
            tau = r["tau"][s0:s1]
            assert sorted(tau) == list(range(1, B + 1))
            d0 = prev["decided"][b]
            keep = prev["tau"][s0:s1] <= d0
            np.testing.assert_array_equal(tau[keep], prev["tau"][s0:s1][keep])
            np.testing.assert_array_equal(r["draft_tokens"][s0:s1][keep],
                                          prev["block_tokens"][s0:s1][keep])
            assert r["n_accept"][b] >= d0
            passes[b] += 1
            if r["done"][b]:
                closed[b] = True
                assert st["lens"][b] == prev["lens"][b] + B
                assert r["pos"][b] == -1 and r["n_accept"][b] == B
            else:
                assert st["decided"][b] > d0 and st["lens"][b] == prev["lens"][b]
                assert (r["block_tokens"][s0:s1] >= 0).all()
    assert closed.all()
    assert (passes <= Bs + 1).all()


def test_finished_block_follows_the_target():
    """Losslessness of the whole loop: with target rows that do not change
    from pass to pass (the positions are independent here), the tokens of a
    closed block are distributed as the product of the target's per-position
    distributions, whatever the draft proposes at each pass (fresh draft rows
    every pass).  B = 2, V = 3, 200,000 blocks; chi-square over the 9 cells."""
    rng = np.random.default_rng(41)
    n, B, V = 200_000, 2, 3
    cu = np.arange(0, B * n + 1, B, dtype=np.int32)
    tl1 = np.array([[0.3, -0.8, 1.1], [1.5, 0.2, -0.4]])
    p = np.exp(tl1 - tl1.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    tl = np.tile(tl1, (n, 1))
    st = loop.initial_state(cu, np.zeros(n))
    final = np.full((n, B), -1)
    for it in range(B + 1):
        dl = np.tile(rng.standard_normal((B, V)) * 1.5, (n, 1))
        st, r = loop.blockwise_pass(cu, st, dl, tl, rng.random((n, B), dtype=np.float32),
                                    rng.random((n, B + 1), dtype=np.float32))
        newly = (r["done"] == 1) & (final[:, 0] < 0)
        final[newly] = r["block_tokens"].reshape(n, B)[newly]
    assert (final >= 0).all()
    obs = np.bincount(final[:, 0] * V + final[:, 1], minlength=V * V)
    exp = np.outer(p[0], p[1]).reshape(-1) * n
    chi2 = ((obs - exp) ** 2 / exp).sum()
    assert chi2 < 30.0, chi2          # 8 degrees of freedom: p ~ 2e-4 at 30
