"""Pins for the oracle's acceptance walk (rejection sampling in tau order).

Pinned against: the mathematics of standard speculative sampling -- the
emitted token at each reached step follows the target distribution p
(losslessness), a step accepts with probability sum_v min(p, q), the walk
reaches step t with probability prod_{s<=t} alpha_s -- checked on the
oracle's own decisions by brute force over deterministic grids of uniforms
and by a fixed-seed Monte Carlo against exact enumeration; plus the special
cases p = q, u = 0 and a one-hot draft.
"""
import numpy as np
import pytest

import oracle
from oracle import exact


def softmax(x):
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def test_exact_module_closed_forms():
    """exact.py enumerates paths; its totals must meet the closed forms."""
    rng = np.random.default_rng(1)
    B, V = 3, 6
    p = softmax(rng.standard_normal((B, V)) * 2)
    q = softmax(rng.standard_normal((B, V)) * 2)
    tau = [2, 3, 1]
    d = exact.outcome_distribution(p, q, tau)
    assert abs(sum(d.values()) - 1.0) < 1e-12
    alpha = np.minimum(p, q).sum(1)
    order = [tau.index(t) for t in (1, 2, 3)]
    reach = 1.0
    for t, k in enumerate(order):
        r = np.maximum(p[k] - q[k], 0)
        for v in range(V):
            np.testing.assert_allclose(d.get((t, v), 0.0), reach * r[v], atol=1e-14)
        reach *= alpha[k]
    np.testing.assert_allclose(d[(B, -1)], reach, rtol=1e-12)
    for k in range(B):
        np.testing.assert_allclose(exact.step_emission(p[k], q[k]), p[k], atol=1e-14)


def run_single_slot(logit_t, logit_d, xs, u0s, u1s):
    """Many B = 1 sequences sharing one slot's logits."""
    n = len(xs)
    V = len(logit_t)
    target = np.broadcast_to(logit_t, (n, V))
    draft = np.broadcast_to(logit_d, (n, V))
    cu = np.arange(n + 1, dtype=np.int32)
    uni = np.stack([u0s, u1s], 1).astype(np.float32)
    return oracle.accept(cu, target, draft, xs, np.ones(n, np.int32), uni, n_threads=4)


def test_lossless_single_step_by_grid():
    """Emitted token distribution, integrated over midpoint grids of both
    uniforms using the oracle's decisions, equals p within grid error."""
    rng = np.random.default_rng(5)
    V, N = 8, 2000
    lt, ld = rng.standard_normal(V) * 1.5, rng.standard_normal(V) * 1.5
    p, q = softmax(lt), softmax(ld)
    grid = ((np.arange(N) + 0.5) / N).astype(np.float32)
    emit = np.zeros(V)
    for x in range(V):
        # (a) acceptance probability of draft token x over the u0 grid
        res = run_single_slot(lt, ld, np.full(N, x), grid, np.full(N, 0.5, np.float32))
        acc = (res["n_accept"] == 1).mean()
        assert abs(acc - min(1.0, p[x] / q[x])) <= 1.0 / N + 1e-7
        emit[x] += q[x] * acc
        if acc < 1.0:
            # (b) the residual draw over the u1 grid, forced rejection
            res = run_single_slot(lt, ld, np.full(N, x), np.full(N, 0.99999, np.float32), grid)
            assert (res["n_accept"] == 0).all() and (res["pos"] == 0).all()
            hist = np.bincount(res["token"], minlength=V) / N
            r = np.maximum(p - q, 0); r /= r.sum()
            assert np.abs(np.cumsum(hist) - np.cumsum(r)).max() <= 1.0 / N + 1e-9
            emit += q[x] * (1 - acc) * hist
    assert np.abs(emit - p).max() < 3.0 / N


def test_walk_distribution_monte_carlo():
    """V = 8, B = 3: fixed-seed Monte Carlo of the whole walk through the
    oracle against the exact outcome distribution (chi-square)."""
    rng = np.random.default_rng(12)
    V, B, n = 8, 3, 200_000
    lt = rng.standard_normal((B, V)) * np.array([[0.5], [2.0], [1.0]])
    ld = lt + rng.standard_normal((B, V)) * np.array([[0.3], [2.5], [1.0]])
    p, q = softmax(lt), softmax(ld)
    tau = np.array([3, 1, 2])
    xs = np.stack([rng.choice(V, size=n, p=q[k]) for k in range(B)], 1)
    uni = rng.random((n, B + 1), dtype=np.float32)
    cu = np.arange(0, B * n + 1, B, dtype=np.int32)
    res = oracle.accept(cu, np.tile(lt, (n, 1)), np.tile(ld, (n, 1)), xs.reshape(-1),
                        np.tile(tau, n), uni, n_threads=4)
    d = exact.outcome_distribution(p, q, tau)
    keys = sorted(d)
    idx = {k: i for i, k in enumerate(keys)}
    obs = np.zeros(len(keys))
    order = [list(tau).index(t) for t in (1, 2, 3)]
    for na, tok, pos in zip(res["n_accept"], res["token"], res["pos"]):
        obs[idx[(int(na), int(tok))]] += 1
        assert pos == (order[na] if na < B else -1)
    exp_counts = np.array([d[k] for k in keys]) * n
    keep = exp_counts > 5
    chi2 = (((obs - exp_counts) ** 2 / exp_counts)[keep]).sum()
    dof = keep.sum() - 1
    # chi-square upper quantile ~ dof + 4 sqrt(2 dof) is far beyond alpha=1e-3
    assert chi2 < dof + 4.0 * np.sqrt(2.0 * dof) + 10, (chi2, dof)
    assert obs[~keep].sum() < 50


def test_special_cases():
    rng = np.random.default_rng(9)
    V, B, n = 32, 5, 300
    lt = rng.standard_normal((n * B, V))
    tau = np.concatenate([rng.permutation(B) + 1 for _ in range(n)])
    xs = rng.integers(0, V, n * B)
    cu = np.arange(0, B * n + 1, B, dtype=np.int32)
    uni = (rng.random((n, B + 1), dtype=np.float32) * np.float32(0.999)).astype(np.float32)
    # p == q: every step accepted
    res = oracle.accept(cu, lt, lt, xs, tau, uni)
    assert (res["n_accept"] == B).all() and (res["token"] == -1).all() and (res["pos"] == -1).all()
    # u == 0: accepted whenever p(x) > 0, even when q(x) >> p(x)
    ld = lt + rng.standard_normal((n * B, V)) * 4
    res = oracle.accept(cu, lt, ld, xs, tau, np.zeros((n, B + 1), np.float32))
    assert (res["n_accept"] == B).all()
    # p(x) = 0 (logit -inf): that step always rejects
    lt2 = lt.copy()
    k = 2
    lt2[k::B][np.arange(n), xs[k::B]] = -np.inf
    res = oracle.accept(cu, lt2, ld, xs, tau, np.zeros((n, B + 1), np.float32))
    assert (res["pos"] == k).all()
    assert (res["n_accept"] == tau[k::B] - 1).all()
    assert (res["token"] != xs[k::B]).all()


def test_one_hot_draft():
    """q one-hot on a, draft token a: accept with probability p(a); on
    rejection the token follows p restricted to v != a, renormalised."""
    rng = np.random.default_rng(4)
    V, N, a = 10, 4000, 3
    lt = rng.standard_normal(V)
    ld = np.full(V, -np.inf); ld[a] = 0.0
    p = softmax(lt)
    grid = ((np.arange(N) + 0.5) / N).astype(np.float32)
    res = run_single_slot(lt, ld, np.full(N, a), grid, np.full(N, 0.5, np.float32))
    assert abs((res["n_accept"] == 1).mean() - p[a]) <= 1.0 / N + 1e-7
    res = run_single_slot(lt, ld, np.full(N, a), np.full(N, 0.99999, np.float32), grid)
    hist = np.bincount(res["token"], minlength=V) / N
    want = p.copy(); want[a] = 0; want /= want.sum()
    assert hist[a] == 0
    assert np.abs(np.cumsum(hist) - np.cumsum(want)).max() <= 1.0 / N + 1e-9


def test_margins_and_errors():
    V = 4
    lt = np.log(np.array([[0.4, 0.3, 0.2, 0.1]]))
    ld = np.log(np.array([[0.1, 0.2, 0.3, 0.4]]))
    # p(x=3) = 0.1, q = 0.4: accept iff u < 0.25; u = 0.25 exactly sits on the boundary
    res = oracle.accept([0, 1], lt, ld, [3], [1], np.array([[0.25, 0.5]], np.float32))
    assert res["accept_margin"][0] < 1e-6
    res = oracle.accept([0, 1], lt, ld, [3], [1], np.array([[0.75, 0.5]], np.float32))
    assert res["n_accept"][0] == 0 and res["pos"][0] == 0
    # residual r = (0.3, 0.1, 0, 0)/0.4: u = 0.5 -> U = 0.2 -> token 0, margin 0.25
    assert res["token"][0] == 0
    assert abs(res["resample_margin"][0] - 0.25) < 1e-12
    with pytest.raises(oracle.OracleError):
        oracle.accept([0, 2], np.zeros((2, 4)), np.zeros((2, 4)), [0, 1], [1, 1],
                      np.zeros((1, 3), np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.accept([0, 1], np.zeros((1, 4)), np.zeros((1, 4)), [4], [1],
                      np.zeros((1, 2), np.float32))


# ------------------------------------------------------------------ variants
def test_greedy_rule():
    """Greedy verification: accept iff the draft token is the target's argmax
    (first index among equal maxima); the first rejection emits the argmax.
    Expected values from numpy's argmax and a hand walk over tau."""
    rng = np.random.default_rng(21)
    B, V = 5, 40
    tau = np.array([3, 1, 5, 2, 4], np.int32)
    target = np.round(rng.standard_normal((B, V)) * 4) / 4      # ties occur
    target[1, 7] = target[1, 30] = target[1].max() + 1.0          # a tie at the top
    a = target.argmax(1)
    assert a[1] == 7
    cu = np.array([0, B], np.int32)
    # every draft token is the argmax: all accepted
    r = oracle.accept_greedy(cu, target, a.astype(np.int32), tau)
    assert r["n_accept"][0] == B and r["token"][0] == -1 and r["pos"][0] == -1
    # the slot tested third (tau = 3 -> k = 0) proposes another token
    x = a.astype(np.int32).copy()
    x[0] = (a[0] + 1) % V
    r = oracle.accept_greedy(cu, target, x, tau)
    assert r["n_accept"][0] == 2 and r["token"][0] == a[0] and r["pos"][0] == 0
    # the tied row: the later maximum is rejected in favour of the first
    x = a.astype(np.int32).copy()
    x[1] = 30
    r = oracle.accept_greedy(cu, target, x, tau)
    assert r["n_accept"][0] == 0 and r["token"][0] == 7 and r["pos"][0] == 1


def test_greedy_is_the_zero_temperature_limit():
    """Sampling at temperature -> 0 concentrates p and q on their argmax:
    a step accepts iff x = argmax p, and the residual max(0, p - q) is the
    point mass at argmax p.  The sampling oracle at T = 1e-6 must therefore
    agree with the greedy oracle (tie-free logits, any uniforms)."""
    rng = np.random.default_rng(22)
    n, B, V = 200, 4, 64
    target = rng.permutation(V * n * B).reshape(n * B, V) * 0.01       # distinct values
    draft = target + rng.standard_normal((n * B, V))
    cu = np.arange(0, n * B + 1, B, dtype=np.int32)
    tau = np.concatenate([rng.permutation(B) + 1 for _ in range(n)]).astype(np.int32)
    a = target.argmax(1)
    # half of the draft tokens are the target argmax, the rest random
    x = np.where(rng.random(n * B) < 0.7, a, rng.integers(0, V, n * B)).astype(np.int32)
    uni = rng.random((n, B + 1), dtype=np.float32)
    s = oracle.accept(cu, target, draft, x, tau, uni, temperature=1e-6)
    g = oracle.accept_greedy(cu, target, x, tau)
    np.testing.assert_array_equal(s["n_accept"], g["n_accept"])
    np.testing.assert_array_equal(s["pos"], g["pos"])
    np.testing.assert_array_equal(s["token"], g["token"])


def test_temperature_scales_both_rows():
    """Temperature T divides both rows' logits: at T = 2 the one-step outcome
    distribution (exact enumeration over the uniforms' grid of the oracle's
    own decisions) follows softmax(l / 2), not softmax(l)."""
    rng = np.random.default_rng(23)
    V, N = 6, 400
    lt = rng.standard_normal(V) * 2
    ld = lt + rng.standard_normal(V)
    T = 2.0
    grid = (np.arange(N) + 0.5) / N
    u0, u1 = np.meshgrid(grid, grid, indexing="ij")
    u0, u1 = u0.ravel(), u1.ravel()
    p = softmax(lt / T)
    q = softmax(ld / T)
    expected = np.zeros(V)
    for x in range(V):
        n = len(u0)
        cu = np.arange(n + 1, dtype=np.int32)
        r = oracle.accept(cu, np.broadcast_to(lt, (n, V)), np.broadcast_to(ld, (n, V)),
                          np.full(n, x, np.int32), np.ones(n, np.int32),
                          np.stack([u0, u1], 1).astype(np.float32), n_threads=4,
                          temperature=T)
        emitted = np.where(r["n_accept"] == 1, x, r["token"])
        expected += q[x] * np.bincount(emitted, minlength=V) / n
    # losslessness at temperature T: the emitted token follows p = softmax(l / T)
    np.testing.assert_allclose(expected, p, atol=3e-3)
    assert np.abs(expected - softmax(lt)).max() > 2e-2


def test_sample_matching_rule():
    """Sample matching: over a midpoint grid of u, a single step accepts with
    probability p(x) and the emitted token (x when accepted, the target's
    sample otherwise) follows p; a point-mass target accepts its token always
    and rejects every other one, emitting the point."""
    rng = np.random.default_rng(24)
    V, N = 7, 4000
    lt = rng.standard_normal(V) * 1.5
    p = softmax(lt)
    u = ((np.arange(N) + 0.5) / N).astype(np.float32)[:, None]
    cu = np.arange(N + 1, dtype=np.int32)
    for x in range(V):
        r = oracle.accept_match(cu, np.broadcast_to(lt, (N, V)), np.full(N, x, np.int32),
                                np.ones(N, np.int32), u)
        acc = r["n_accept"] == 1
        np.testing.assert_allclose(acc.mean(), p[x], atol=2.0 / N)
        emitted = np.where(acc, x, r["token"])
        np.testing.assert_allclose(np.bincount(emitted, minlength=V) / N, p, atol=2.0 / N)
        assert (r["pos"][~acc] == 0).all() and (r["token"][acc] == -1).all()
    point = np.full(V, -np.inf)
    point[3] = 0.0
    for x, want in ((3, 1), (5, 0)):
        r = oracle.accept_match(np.array([0, 1], np.int32), point[None], np.array([x], np.int32),
                                np.ones(1, np.int32), np.array([[0.99]], np.float32))
        assert r["n_accept"][0] == want and r["token"][0] == (-1 if want else 3)


def test_sample_matching_walk_order():
    """The walk follows tau: the steps use u[0], u[1], ... in temporal order
    and stop at the first mismatch (hand-built three-slot case)."""
    V = 4
    target = np.log(np.array([[0.1, 0.2, 0.3, 0.4],      # slot 0: tested second
                              [0.7, 0.1, 0.1, 0.1],      # slot 1: tested first
                              [0.25, 0.25, 0.25, 0.25]]))  # slot 2: tested third
    tau = np.array([2, 1, 3], np.int32)
    cu = np.array([0, 3], np.int32)
    # step 1 (slot 1): u = 0.5 -> token 0; step 2 (slot 0): u = 0.65 -> token 3
    u = np.array([[0.5, 0.65, 0.1, 0.0]], np.float32)
    r = oracle.accept_match(cu, target, np.array([3, 0, 0], np.int32), tau, u)
    assert r["n_accept"][0] == 3 and r["token"][0] == -1
    r = oracle.accept_match(cu, target, np.array([2, 0, 0], np.int32), tau, u)
    assert r["n_accept"][0] == 1 and r["pos"][0] == 0 and r["token"][0] == 3
    r = oracle.accept_match(cu, target, np.array([3, 1, 0], np.int32), tau, u)
    assert r["n_accept"][0] == 0 and r["pos"][0] == 1 and r["token"][0] == 0


# ------------------------------------------------------------------ draft side
def test_draft_step_samples_the_draft_distribution():
    """Over a midpoint grid of u, the draft-side step's token for a slot
    follows q = softmax(draft row) (exact up to the grid), and its confidence
    is the row's largest probability, whatever token was drawn."""
    rng = np.random.default_rng(25)
    V, N = 9, 3000
    ld = rng.standard_normal(V) * 1.2
    q = softmax(ld)
    cu = np.arange(N + 1, dtype=np.int32)
    u = ((np.arange(N) + 0.5) / N).astype(np.float32)[:, None]
    r = oracle.draft_step(cu, np.broadcast_to(ld, (N, V)), u)
    np.testing.assert_allclose(np.bincount(r["draft_tokens"], minlength=V) / N, q, atol=2.0 / N)
    np.testing.assert_allclose(r["confidence"], q.max(), rtol=1e-12)
    assert (r["tau"] == 1).all()


def test_draft_step_orders_by_confidence():
    """tau is a permutation ordering the slots by the draft's largest
    probability in each row, most confident first, equal ones in position
    order (hand-built: slot 2 certain, slots 0 and 3 tied at 0.5, slot 1
    least sure at 0.3 -- although its sampled token has 0.2)."""
    V = 4
    rows = np.log(np.array([[0.5, 0.5, 1e-300, 1e-300],    # slot 0: either token, q = 0.5
                            [0.3, 0.3, 0.2, 0.2],          # slot 1: q <= 0.3
                            [1.0, 1e-300, 1e-300, 1e-300],  # slot 2: q = 1
                            [1e-300, 0.5, 0.5, 1e-300]]))  # slot 3: q = 0.5
    cu = np.array([0, 4], np.int32)
    u = np.array([[0.2, 0.7, 0.9, 0.8]], np.float32)
    r = oracle.draft_step(cu, rows, u)
    np.testing.assert_array_equal(r["draft_tokens"], [0, 2, 0, 2])
    np.testing.assert_allclose(r["confidence"], [0.5, 0.3, 1.0, 0.5], rtol=1e-9)
    np.testing.assert_array_equal(r["tau"], [2, 4, 1, 3])
    rng = np.random.default_rng(26)
    B, n = 6, 50
    cu = np.arange(0, B * n + 1, B, dtype=np.int32)
    r = oracle.draft_step(cu, rng.standard_normal((B * n, 20)) * 2,
                          rng.random((n, B), dtype=np.float32))
    for b in range(n):
        t = r["tau"][b * B:(b + 1) * B]
        c = r["confidence"][b * B:(b + 1) * B]
        assert sorted(t) == list(range(1, B + 1))
        by_step = c[np.argsort(t)]
        assert (np.diff(by_step) <= 0).all()
