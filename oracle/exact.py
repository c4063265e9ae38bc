"""Exact outcome distribution of the acceptance walk -- TEST INFRASTRUCTURE.

SimSD (gist.science, paper 2606.02544), "Speculative Decoding Pipeline":
standard rejection sampling along the draft-induced temporal order, longest
accepted prefix committed.  This module does not run that procedure on
sampled inputs; it computes, by brute force over every draft-token vector
x in V^B (drawn x_k ~ q_k independently) and exact integration over the
uniforms, the probability of every outcome (n_accept, token).  Step t tests
the slot k with tau(k) = t and accepts with probability min(1, p_k(x_k) /
q_k(x_k)); at the first rejection the token follows max(0, p_k - q_k)
normalised (p_k itself when that is empty).

For tiny V and B only (pure Python loops).
"""
import itertools

import numpy as np


def residual(p, q):
    """norm(max(0, p - q)); p itself when p == q everywhere."""
    r = np.maximum(p - q, 0.0)
    s = r.sum()
    if s == 0.0:
        return p / p.sum()
    return r / s


def outcome_distribution(p, q, tau):
    """p, q: [B, V] probabilities; tau: [B] labels 1..B.
    Returns {(n_accept, token): probability}; token is -1 for n_accept == B."""
    p = np.asarray(p, np.float64)
    q = np.asarray(q, np.float64)
    B, V = p.shape
    order = [list(tau).index(t) for t in range(1, B + 1)]
    res = [residual(p[k], q[k]) for k in range(B)]
    dist = {}
    for x in itertools.product(range(V), repeat=B):
        w = 1.0
        for k in range(B):
            w *= q[k, x[k]]
        if w == 0.0:
            continue
        reach = w
        for t, k in enumerate(order):
            a = min(1.0, p[k, x[k]] / q[k, x[k]])
            rej = reach * (1.0 - a)
            if rej > 0.0:
                for v in range(V):
                    if res[k][v] > 0.0:
                        key = (t, v)
                        dist[key] = dist.get(key, 0.0) + rej * res[k][v]
            reach *= a
            if reach == 0.0:
                break
        if reach > 0.0:
            dist[(B, -1)] = dist.get((B, -1), 0.0) + reach
    return dist


def step_emission(p, q):
    """Distribution of the token emitted at one step that is reached:
    the draft token when accepted, the residual draw when rejected.
    p, q: [V].  Brute force over the draft token x ~ q."""
    p = np.asarray(p, np.float64)
    q = np.asarray(q, np.float64)
    r = residual(p, q)
    out = np.zeros_like(p)
    for x in range(len(p)):
        if q[x] == 0.0:
            continue
        a = min(1.0, p[x] / q[x])
        out[x] += q[x] * a
        out += q[x] * (1.0 - a) * r
    return out
