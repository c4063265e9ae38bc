"""fp64 CPU oracle for the SimSD verification step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
it imports nothing from the CUDA library: the two sides meet only through
the seeded generators in ``synth.py``.

The arithmetic lives in plain C (``layout.c``, ``attention.c``,
``accept.c``; see ``simsd_oracle.h`` for the passages each follows).  This
module only marshals numpy arrays through ctypes.  ``exact.py`` holds the
closed-form distribution of the acceptance walk used to pin ``accept``.

Parity unpinned: the RoPE pairing convention and the softmax scale (the
pages fix neither).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

ORACLE_OK, ORACLE_ERR_ARG, ORACLE_ERR_TAU = 0, 1, 2


class OracleError(RuntimeError):
    pass


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        I, D, P = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_tau_is_permutation.argtypes = [I, P]
        lib.oracle_mask_entry.argtypes = [I, I, P, I, I]
        lib.oracle_layout.argtypes = [I, I, P, P, P]
        lib.oracle_rope.argtypes = [P, I, I, I, P, D, P]
        lib.oracle_rope.restype = None
        lib.oracle_verify_attn_seq.argtypes = [I, I, I, I, I, D, D, I, P, P, P,
                                               P, P, P, I, P, P, P]
        lib.oracle_verify_attn.argtypes = [I, P, P, I, I, I, D, D, P, P, P, P,
                                           P, P, P, I]
        lib.oracle_accept.argtypes = [I, I, P, P, P, P, P, P, I, P, P, P, P,
                                      P, P, I]
        lib.oracle_accept_greedy.argtypes = [I, I, P, P, P, P, P, P, P, P]
        lib.oracle_accept_match.argtypes = [I, I, P, P, P, P, P, I, P, P, P, P]
        lib.oracle_draft_step.argtypes = [I, I, P, P, P, I, P, P, P, P, P]
        lib.oracle_commit.argtypes = [I, P, P, P, P, P, P, P, P, P]
        lib.oracle_graph_mask_entry.argtypes = [I, I, I, I, I]
        lib.oracle_verify_attn_graph_seq.argtypes = [I, I, I, I, I, I, D, D, P, P, P, P, P,
                                                     P]
        lib.oracle_residual.argtypes = [I, P, P, P]
        lib.oracle_residual.restype = D
        _LIB = lib
    return _LIB


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != ORACLE_OK:
        raise OracleError("%s failed with code %d" % (what, rc))


def tau_is_permutation(tau):
    tau = _c(tau, np.int32)
    return bool(_lib().oracle_tau_is_permutation(len(tau), _p(tau)))


def layout(P, tau, with_mask=True):
    """positions int32[P+2B], mask uint8[2B, P+2B] (or None)."""
    tau = _c(tau, np.int32)
    B = len(tau)
    positions = np.zeros(P + 2 * B, np.int32)
    mask = np.zeros((2 * B, P + 2 * B), np.uint8) if with_mask else None
    _check(_lib().oracle_layout(P, B, _p(tau), _p(positions), _p(mask)),
           "oracle_layout")
    return positions, mask


def rope(x, pos, base):
    """x [n_tok, n_heads, hd] fp64 rotated at pos[n_tok]."""
    x = _c(x, np.float64)
    pos = _c(pos, np.int32)
    n_tok, n_heads, hd = x.shape
    out = np.empty_like(x)
    _lib().oracle_rope(_p(x), n_tok, n_heads, hd, _p(pos), float(base), _p(out))
    return out


def verify_attn_seq(q, k_prompt, v_prompt, k_new, v_new, tau, rope_base,
                    sm_scale, pos_offset=0, rows=None):
    """One sequence.  q [2B,Hq,hd] raw; k_prompt/v_prompt [P,Hkv,hd] (keys
    already rotated); k_new/v_new [2B,Hkv,hd] raw; tau [B].
    rows: None for every row (returns [2B,Hq,hd]) or a list of
    (token, head) pairs (returns [n,hd])."""
    q = _c(q, np.float64)
    k_new, v_new = _c(k_new, np.float64), _c(v_new, np.float64)
    tau = _c(tau, np.int32)
    twoB, Hq, hd = q.shape
    Hkv = k_new.shape[1]
    P = 0 if k_prompt is None else k_prompt.shape[0]
    kp = None if P == 0 else _c(k_prompt, np.float64)
    vp = None if P == 0 else _c(v_prompt, np.float64)
    if rows is None:
        out = np.empty((twoB, Hq, hd), np.float64)
        n, rt, rh = -1, None, None
    else:
        rows = np.asarray(rows, np.int32).reshape(-1, 2)
        n = len(rows)
        rt, rh = _c(rows[:, 0], np.int32), _c(rows[:, 1], np.int32)
        out = np.empty((n, hd), np.float64)
    _check(_lib().oracle_verify_attn_seq(
        P, len(tau), Hq, Hkv, hd, float(rope_base), float(sm_scale),
        int(pos_offset), _p(tau), _p(q), _p(kp), _p(vp), _p(k_new), _p(v_new),
        n, _p(rt), _p(rh), _p(out)), "oracle_verify_attn_seq")
    return out


def verify_attn(lens, cu_B, q, k_prompt, v_prompt, k_new, v_new, tau,
                rope_base, sm_scale, n_threads=0):
    """Whole batch, sequences back to back (see simsd_oracle.h)."""
    lens, cu_B, tau = _c(lens, np.int32), _c(cu_B, np.int32), _c(tau, np.int32)
    q = _c(q, np.float64)
    k_new, v_new = _c(k_new, np.float64), _c(v_new, np.float64)
    k_prompt, v_prompt = _c(k_prompt, np.float64), _c(v_prompt, np.float64)
    T, Hq, hd = q.shape
    Hkv = k_new.shape[1]
    out = np.empty_like(q)
    _check(_lib().oracle_verify_attn(
        len(lens), _p(lens), _p(cu_B), Hq, Hkv, hd, float(rope_base),
        float(sm_scale), _p(tau), _p(q), _p(k_prompt), _p(v_prompt),
        _p(k_new), _p(v_new), _p(out), int(n_threads)), "oracle_verify_attn")
    return out


def _first(first_step, batch):
    return None if first_step is None else _c(first_step, np.int32).reshape(batch)


def accept(cu_B, target, draft, draft_tokens, tau, uniforms, n_threads=0, temperature=1.0,
           first_step=None):
    """Returns dict(n_accept, token, pos, accept_margin, resample_margin).
    target/draft [sum B, V] (any float dtype, taken exactly to fp64);
    uniforms [batch, u_stride] float32.  temperature T: p = softmax(target / T),
    q = softmax(draft / T) (the logits divided in fp64).  first_step [batch]
    (optional): the walk's first step per sequence (earlier steps decided)."""
    cu_B = _c(cu_B, np.int32)
    target, draft = _c(target, np.float64), _c(draft, np.float64)
    if temperature != 1.0:
        target = np.ascontiguousarray(target / float(temperature))
        draft = np.ascontiguousarray(draft / float(temperature))
    draft_tokens, tau = _c(draft_tokens, np.int32), _c(tau, np.int32)
    uniforms = _c(uniforms, np.float32)
    batch = len(cu_B) - 1
    V = target.shape[1]
    n_accept = np.zeros(batch, np.int32)
    token = np.zeros(batch, np.int32)
    pos = np.zeros(batch, np.int32)
    am = np.zeros(int(cu_B[-1]), np.float64)
    rm = np.zeros(batch, np.float64)
    fs = _first(first_step, batch)
    _check(_lib().oracle_accept(
        batch, V, _p(cu_B), _p(target), _p(draft), _p(draft_tokens), _p(tau),
        _p(uniforms), uniforms.shape[1], _p(fs), _p(n_accept), _p(token), _p(pos),
        _p(am), _p(rm), int(n_threads)), "oracle_accept")
    return dict(n_accept=n_accept, token=token, pos=pos, accept_margin=am,
                resample_margin=rm)


def accept_greedy(cu_B, target, draft_tokens, tau, first_step=None):
    """Greedy verification: dict(n_accept, token, pos); target [sum B, V]."""
    cu_B = _c(cu_B, np.int32)
    target = _c(target, np.float64)
    draft_tokens, tau = _c(draft_tokens, np.int32), _c(tau, np.int32)
    batch = len(cu_B) - 1
    n_accept = np.zeros(batch, np.int32)
    token = np.zeros(batch, np.int32)
    pos = np.zeros(batch, np.int32)
    fs = _first(first_step, batch)
    _check(_lib().oracle_accept_greedy(
        batch, target.shape[1], _p(cu_B), _p(target), _p(draft_tokens), _p(tau), _p(fs),
        _p(n_accept), _p(token), _p(pos)), "oracle_accept_greedy")
    return dict(n_accept=n_accept, token=token, pos=pos)


def accept_match(cu_B, target, draft_tokens, tau, uniforms, first_step=None):
    """Sample matching: dict(n_accept, token, pos); uniforms [batch, >= B]."""
    cu_B = _c(cu_B, np.int32)
    target = _c(target, np.float64)
    draft_tokens, tau = _c(draft_tokens, np.int32), _c(tau, np.int32)
    uniforms = _c(uniforms, np.float32)
    batch = len(cu_B) - 1
    n_accept = np.zeros(batch, np.int32)
    token = np.zeros(batch, np.int32)
    pos = np.zeros(batch, np.int32)
    fs = _first(first_step, batch)
    _check(_lib().oracle_accept_match(
        batch, target.shape[1], _p(cu_B), _p(target), _p(draft_tokens), _p(tau),
        _p(uniforms), uniforms.shape[1], _p(fs), _p(n_accept), _p(token), _p(pos)),
        "oracle_accept_match")
    return dict(n_accept=n_accept, token=token, pos=pos)


def draft_step(cu_B, draft, uniforms, temperature=1.0, decided=None, tau_prev=None,
               tokens_prev=None):
    """The draft-side step: dict(draft_tokens, tau, confidence) per slot;
    draft [sum B, V] logits (divided by the temperature), uniforms
    [batch, >= B] (u[k] samples slot k).  Within a block: decided [batch]
    steps already decided keep their labels (tau_prev) and tokens
    (tokens_prev); confidence is -1 there."""
    cu_B = _c(cu_B, np.int32)
    draft = _c(draft, np.float64)
    if temperature != 1.0:
        draft = np.ascontiguousarray(draft / float(temperature))
    uniforms = _c(uniforms, np.float32)
    n = int(cu_B[-1])
    batch = len(cu_B) - 1
    toks = np.zeros(n, np.int32) if tokens_prev is None else _c(tokens_prev, np.int32).copy()
    tau = np.zeros(n, np.int32)
    conf = np.zeros(n, np.float64)
    dec = None if decided is None else _c(decided, np.int32).reshape(batch)
    tp = None if tau_prev is None else _c(tau_prev, np.int32)
    _check(_lib().oracle_draft_step(batch, draft.shape[1], _p(cu_B), _p(draft),
                                    _p(uniforms), uniforms.shape[1], _p(dec), _p(tp),
                                    _p(toks), _p(tau), _p(conf)), "oracle_draft_step")
    return dict(draft_tokens=toks, tau=tau, confidence=conf)


def commit(cu_B, tau, n_accept, token, pos, block_tokens, decided, lens):
    """Commit after a pass of the blockwise loop; returns dict(block_tokens,
    decided, lens, done) (new arrays; the inputs are not modified)."""
    cu_B, tau = _c(cu_B, np.int32), _c(tau, np.int32)
    batch = len(cu_B) - 1
    bt = _c(block_tokens, np.int32).copy()
    dec = _c(decided, np.int32).copy()
    ln = _c(lens, np.int32).copy()
    done = np.zeros(batch, np.int32)
    _check(_lib().oracle_commit(batch, _p(cu_B), _p(tau), _p(_c(n_accept, np.int32)),
                                _p(_c(token, np.int32)), _p(_c(pos, np.int32)), _p(bt),
                                _p(dec), _p(ln), _p(done)), "oracle_commit")
    return dict(block_tokens=bt, decided=dec, lens=ln, done=done)


def graph_mask(P, n_nodes, node_size):
    """The draft-graph verification mask of the new rows, uint8
    [n_nodes * node_size, P + n_nodes * node_size], entry by entry."""
    T = n_nodes * node_size
    m = np.zeros((T, P + T), np.uint8)
    f = _lib().oracle_graph_mask_entry
    for r in range(T):
        for c in range(P + T):
            m[r, c] = f(P, n_nodes, node_size, r, c)
    return m


def verify_attn_graph_seq(q, k_prompt, v_prompt, k_new, v_new, node_size, rope_base,
                          sm_scale):
    """Attention of one sequence's candidate nodes (see simsd_oracle.h):
    q [T, Hq, hd], k_new / v_new [T, Hkv, hd] raw, node-major; prompt keys
    rotated.  Returns [T, Hq, hd]."""
    q = _c(q, np.float64)
    k_new, v_new = _c(k_new, np.float64), _c(v_new, np.float64)
    T, Hq, hd = q.shape
    if T % node_size:
        raise ValueError("the rows are not whole nodes")
    P = 0 if k_prompt is None else k_prompt.shape[0]
    kp = None if P == 0 else _c(k_prompt, np.float64)
    vp = None if P == 0 else _c(v_prompt, np.float64)
    out = np.empty_like(q)
    _check(_lib().oracle_verify_attn_graph_seq(
        P, T // node_size, node_size, Hq, k_new.shape[1], hd, float(rope_base),
        float(sm_scale), _p(q), _p(kp), _p(vp), _p(k_new), _p(v_new), _p(out)),
        "oracle_verify_attn_graph_seq")
    return out


def residual(target_row, draft_row):
    """(r, S): r = max(0, p - q) of one slot in fp64 (p when empty)."""
    t = _c(target_row, np.float64)
    d = _c(draft_row, np.float64)
    r = np.empty_like(t)
    S = _lib().oracle_residual(len(t), _p(t), _p(d), _p(r))
    return r, S


def library_path():
    return _build.LIB


def default_threads():
    return len(os.sched_getaffinity(0))
