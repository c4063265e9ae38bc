"""GPU parity of simsd_accept (K4) against the fp64 oracle.

Decisions (accepted length, rejected position, drawn token) must match the
oracle exactly on the same logits and uniforms, except for tie-zone
decisions (see parity.py), which are only checked for validity.  Plus the
special cases with a known answer, a Monte Carlo of 10^6 walks on V = 8,
B = 3 against the exact outcome distribution, and vocabularies whose rows
are not 16-byte multiples.
"""
import numpy as np
import pytest
import torch

import parity
import synth
import oracle
from oracle import exact
from speculative_decoding_diffusion_gb300 import binding
from speculative_decoding_diffusion_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu


PATHS = ["two-kernel", "single-launch"]


def run_accept(w, path="two-kernel"):
    """simsd_accept with the workspace size the library asks for (the
    two-kernel path: chunk pass, then the per-sequence cluster kernel) or
    one of just the status word (the single cluster kernel streaming the
    rows itself)."""
    dw = DeviceWorkload(w, with_verify=False)
    if path == "single-launch":
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        binding.accept(dw.target, dw.draft, dw.draft_tokens, dw.tau, dw.cu_B, dw.uniforms,
                       dw.n_accept, dw.token, dw.pos, ws, dw.total_B, dw.B_max)
    else:
        ws = dw.accept_ws
        dw.accept()
    torch.cuda.synchronize()
    assert binding.read_status(ws) == 0
    return (dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy())


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_configs_match_oracle(cfg, path):
    w = synth.config(cfg)
    n, tok, pos = run_accept(w, path)
    ref = parity.oracle_accept(w)
    stats = []
    step_ties, draw_ties, draws = parity.check_accept(w, ref, n, tok, pos, stats=stats)
    rep = parity.tie_report(stats)
    print("cfg%d %s: %d sequences, %d residual draws, %d draw ties, %d step ties; %s"
          % (cfg, path, len(w.lens), draws, draw_ties, step_ties, rep))
    assert step_ties == 0
    assert draw_ties <= 0.02 * draws, (draw_ties, draws)


def tiny_accept_spec(**kw):
    base = dict(name="acc", batch=64, prompt=0, B=(1, 2, 5, 8, 32), Hq=1, Hkv=1, hd=64,
                dtype="bf16", vocab=1003, logit_sd=2.0, noise_sd=(0.1, 3.0))
    base.update(kw)
    return synth.Spec(**base)


@pytest.mark.parametrize("dtype,vocab", [("bf16", 1003), ("bf16", 4096 + 8), ("f32", 777),
                                         ("f32", 2048), ("bf16", 9)])
@pytest.mark.parametrize("path", PATHS)
def test_odd_vocab_and_mixed_B(dtype, vocab, path):
    w = synth.make(tiny_accept_spec(dtype=dtype, vocab=vocab), seed=vocab)
    n, tok, pos = run_accept(w, path)
    parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)


@pytest.mark.parametrize("dtype,vocab,batch,B", [("bf16", 151936, 2, 32), ("bf16", 65539, 3, 32),
                                                 ("f32", 100003, 4, 17), ("bf16", 151936, 5, 1),
                                                 ("f32", 1 << 21, 2, 2), ("bf16", 1 << 21, 2, 3)])
@pytest.mark.parametrize("path", PATHS)
def test_few_sequences_large_clusters(dtype, vocab, batch, B, path):
    """Few sequences get the largest clusters (up to 16 CTAs each): slices
    of 1/16 of the vocabulary, the slice merge in 16-lane groups and, at
    B = 32, in two rounds of pairs; element copies where rows are not
    16-byte multiples.  The largest vocabulary (2^21) gives the chunked
    path's merges and part searches more parts than a warp holds."""
    w = synth.make(tiny_accept_spec(batch=batch, B=B, dtype=dtype, vocab=vocab), seed=vocab + B)
    n, tok, pos = run_accept(w, path)
    parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)


@pytest.mark.parametrize("dtype,vocab", [("bf16", 40000), ("f32", 777), ("bf16", 1003)])
def test_batches_over_twice_the_sm_count(dtype, vocab):
    """More sequences than two per SM: the finishing kernel runs one CTA per
    sequence (all chunks each) in more than one wave.  Against the oracle,
    on 16-byte-aligned rows and on element-copied ones."""
    w = synth.make(tiny_accept_spec(batch=400, dtype=dtype, vocab=vocab), seed=vocab + 400)
    n, tok, pos = run_accept(w, "two-kernel")
    step_ties, draw_ties, draws = parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)
    print("%s V=%d: %d sequences, %d draws, %d draw ties, %d step ties"
          % (dtype, vocab, len(w.lens), draws, draw_ties, step_ties))
    assert draw_ties <= parity.max_ties(draws)
    assert draws > 100


def test_invalid_token_rejects_and_empty_residual_draws_from_p():
    """A draft token outside the vocabulary rejects its step and sets the
    status word's bad-input bit; with identical target and draft rows the
    residual max(0, p - q) is empty, so the token is drawn from p itself
    (the fallback the pages' rule needs when p <= q everywhere)."""
    w = synth.make(tiny_accept_spec(batch=8, B=3, vocab=5000), seed=11)
    w.draft = w.target.copy()
    V, B = w.spec.vocab, 3
    first = []
    for b in range(len(w.lens)):
        s0 = int(w.cu_B[b])
        k = int(np.nonzero(w.tau[s0:s0 + B] == 1)[0][0])   # the slot tested first
        w.draft_tokens[s0 + k] = -1 if b % 2 else V
        first.append(k)
    dw = DeviceWorkload(w, with_verify=False)
    dw.accept()
    torch.cuda.synchronize()
    assert binding.read_status(dw.accept_ws) == 2             # the bad-input bit
    n, tok, pos = dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()
    for b, k in enumerate(first):
        assert n[b] == 0 and pos[b] == k
        s0 = int(w.cu_B[b])
        r, S = oracle.residual(synth.to_f64(w.target[s0 + k]), synth.to_f64(w.draft[s0 + k]))
        C = np.cumsum(r)                  # r = p: the residual is empty
        U = float(w.uniforms[b, B]) * S
        v = int(np.searchsorted(C, U, side="right"))
        lo = C[v - 1] if v > 0 else 0.0
        if v < V and min(U - lo, C[v] - U) >= parity.TIE_RESIDUAL:
            assert tok[b] == v, (b, tok[b], v)
        else:
            g = int(tok[b])
            assert 0 <= g < V and r[g] > 0
            glo = C[g - 1] if g > 0 else 0.0
            assert glo - parity.TIE_RESIDUAL <= U < C[g] + parity.TIE_RESIDUAL


def test_p_equals_q_accepts_everything():
    w = synth.make(tiny_accept_spec(), seed=1)
    w.draft = w.target.copy()
    w.uniforms = np.minimum(w.uniforms, np.float32(0.999))
    n, tok, pos = run_accept(w)
    assert np.array_equal(n, w.Bs) and (tok == -1).all() and (pos == -1).all()


def test_zero_uniforms_accept_everything():
    w = synth.make(tiny_accept_spec(), seed=2)
    w.uniforms[:] = 0
    n, tok, pos = run_accept(w)
    assert np.array_equal(n, w.Bs)


def test_certain_rejection_position():
    # target logit of the draft token at slot k = -inf: the walk stops at
    # step tau(k) (or earlier), and never draws the draft token there
    w = synth.make(tiny_accept_spec(dtype="f32"), seed=3)
    k_of = []
    for b in range(len(w.lens)):
        s0, B = int(w.cu_B[b]), int(w.Bs[b])
        k = B // 2
        w.target[s0 + k, w.draft_tokens[s0 + k]] = -np.inf
        k_of.append(k)
    n, tok, pos = run_accept(w)
    ref = parity.oracle_accept(w)
    parity.check_accept(w, ref, n, tok, pos)
    for b, k in enumerate(k_of):
        s0 = int(w.cu_B[b])
        assert n[b] <= w.tau[s0 + k] - 1
        if pos[b] == k:
            assert tok[b] != w.draft_tokens[s0 + k]


def test_walk_distribution_monte_carlo():
    """10^6 walks on V = 8, B = 3 through the GPU kernels; chi-square of the
    (n_accept, token) histogram against the exact enumeration."""
    rng = np.random.default_rng(2024)
    V, B, n = 8, 3, 1_000_000
    lt = (rng.standard_normal((B, V)) * np.array([[0.5], [2.0], [1.0]])).astype(np.float32)
    ld = (lt + rng.standard_normal((B, V)) * np.array([[0.3], [2.5], [1.0]])).astype(np.float32)
    p = np.exp(lt - lt.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    q = np.exp(ld - ld.max(1, keepdims=True)); q /= q.sum(1, keepdims=True)
    tau = np.array([2, 3, 1], np.int32)
    xs = np.stack([rng.choice(V, size=n, p=q[k]) for k in range(B)], 1).astype(np.int32)
    dev = "cuda"
    target = torch.from_numpy(np.tile(lt, (n, 1))).to(dev)
    draft = torch.from_numpy(np.tile(ld, (n, 1))).to(dev)
    toks = torch.from_numpy(xs.reshape(-1)).to(dev)
    taus = torch.from_numpy(np.tile(tau, n)).to(dev)
    cu = torch.arange(0, B * n + 1, B, dtype=torch.int32, device=dev)
    uni = torch.from_numpy(rng.random((n, B + 1), dtype=np.float32)).to(dev)
    n_acc = torch.empty(n, dtype=torch.int32, device=dev)
    tok = torch.empty_like(n_acc)
    pos = torch.empty_like(n_acc)
    # rows of this test: B * n = 3e6 > 65535 slots per launch, so split it
    chunk = 20000
    res_n, res_t, res_p = [], [], []
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        c = cu[s:e + 1] - cu[s]
        args = (target[B * s:B * e], draft[B * s:B * e], toks[B * s:B * e], taus[B * s:B * e],
                c, uni[s:e], n_acc[s:e], tok[s:e], pos[s:e], B * (e - s), B)
        ws = torch.zeros(binding.accept_workspace_size(*args), dtype=torch.uint8, device=dev)
        binding.accept(*args[:9], ws, *args[9:])
    torch.cuda.synchronize()
    na, tk, ps = n_acc.cpu().numpy(), tok.cpu().numpy(), pos.cpu().numpy()
    d = exact.outcome_distribution(p.astype(np.float64), q.astype(np.float64), tau)
    keys = sorted(d)
    idx = {k: i for i, k in enumerate(keys)}
    obs = np.zeros(len(keys))
    codes = na.astype(np.int64) * (V + 1) + (tk + 1)
    uniq, cnt = np.unique(codes, return_counts=True)
    order = [list(tau).index(t) for t in (1, 2, 3)]
    for c_, k_ in zip(uniq, cnt):
        key = (int(c_ // (V + 1)), int(c_ % (V + 1)) - 1)
        assert key in idx, key
        obs[idx[key]] += k_
    assert np.array_equal(ps[na < B], np.array(order)[na[na < B]])
    assert (ps[na == B] == -1).all()
    expc = np.array([d[k] for k in keys]) * n
    keep = expc > 5
    chi2 = (((obs - expc) ** 2 / expc)[keep]).sum()
    dof = keep.sum() - 1
    assert chi2 < dof + 4.0 * np.sqrt(2.0 * dof) + 10, (chi2, dof)


# ------------------------------------------------------------------ variants
# The greedy and matching rules have two paths too: a chunk pass over the
# target rows then one CTA per sequence (the full workspace), or one cluster
# per sequence streaming its rows (a workspace of just the status word).
RULE_PATHS = ["chunked", "cluster"]


def rule_workspace(dw, path):
    return dw.accept_ws if path == "chunked" else torch.zeros(256, dtype=torch.uint8, device="cuda")


def run_rule(w, rule, temperature=1.0, path="chunked"):
    dw = DeviceWorkload(w, with_verify=False)
    ws = rule_workspace(dw, path)
    greedy = rule == binding.SIMSD_ACCEPT_GREEDY
    binding.accept(dw.target, None if greedy else dw.draft, dw.draft_tokens, dw.tau, dw.cu_B,
                   None if greedy else dw.uniforms, dw.n_accept, dw.token, dw.pos,
                   ws, dw.total_B, dw.B_max, rule=rule, temperature=temperature)
    torch.cuda.synchronize()
    assert binding.read_status(ws) == 0
    return (dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy())


def variant_case(name):
    if name == "sdar8b":
        return synth.config(1)
    dtype, vocab, batch = {"bf16-1003": ("bf16", 1003, 64), "f32-777": ("f32", 777, 64),
                           "bf16-few": ("bf16", 151936, 3), "f32-odd": ("f32", 100003, 5),
                           "f32-max": ("f32", 1 << 21, 2)}[name]
    return synth.make(tiny_accept_spec(batch=batch, dtype=dtype, vocab=vocab), seed=vocab + batch)


@pytest.mark.parametrize("path", RULE_PATHS)
@pytest.mark.parametrize("name", ["sdar8b", "bf16-1003", "f32-777", "bf16-few", "f32-odd", "f32-max"])
def test_greedy_matches_oracle(name, path):
    """The greedy rule: accepted lengths, positions and tokens bit-exact
    against the oracle (argmax over the same bf16 / fp32 values, the
    smallest index among equal maxima).  70% of the draft tokens are made the
    target argmax so the walks get past their first step."""
    w = variant_case(name)
    a = synth.to_f64(w.target).argmax(1).astype(np.int32)
    rng = np.random.default_rng(7)
    w.draft_tokens = np.where(rng.random(len(a)) < 0.7, a, w.draft_tokens).astype(np.int32)
    n, tok, pos = run_rule(w, binding.SIMSD_ACCEPT_GREEDY, path=path)
    ref = oracle.accept_greedy(w.cu_B, synth.to_f64(w.target), w.draft_tokens, w.tau)
    np.testing.assert_array_equal(n, ref["n_accept"])
    np.testing.assert_array_equal(pos, ref["pos"])
    np.testing.assert_array_equal(tok, ref["token"])
    assert (n > 0).any() and (n < w.Bs).any()


# temperatures are floats in the ABI: values a float holds exactly, so that
# the oracle divides by the same number
@pytest.mark.parametrize("name,T", [("sdar8b", 0.5), ("sdar8b", 2.0), ("f32-777", 0.75),
                                    ("bf16-1003", 1.5)])
def test_temperature_matches_oracle(name, T):
    """Sampling at temperature T: p = softmax(target / T), q = softmax(draft / T);
    decisions exact outside the tie zone, valid inside."""
    w = variant_case(name)
    n, tok, pos = run_rule(w, binding.SIMSD_ACCEPT_SAMPLE, T)
    step_ties, draw_ties, draws = parity.check_accept(w, parity.oracle_accept(w, T), n, tok,
                                                      pos, T)
    print("%s T=%g: %d draws, %d draw ties, %d step ties" % (name, T, draws, draw_ties, step_ties))
    assert step_ties == 0 and draw_ties <= parity.max_ties(draws)


def check_match(w, n, tok, pos, temperature=1.0, tie=parity.TIE_RESIDUAL):
    """Sample matching against the oracle, decision by decision: exact unless
    u lies within `tie` of a bin edge the decision depends on (then validity)."""
    ref = oracle.accept_match(w.cu_B, synth.to_f64(w.target) / temperature, w.draft_tokens,
                              w.tau, w.uniforms)
    V = w.spec.vocab
    ties = 0
    for b in range(len(w.lens)):
        s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
        B = s1 - s0
        order = [int(np.nonzero(w.tau[s0:s1] == t)[0][0]) for t in range(1, B + 1)]
        near = False
        for t, k in enumerate(order[:int(ref["n_accept"][b]) + 1]):
            lt = synth.to_f64(w.target[s0 + k]) / temperature
            p = np.exp(lt - lt.max()); p /= p.sum()
            C = np.cumsum(p)
            u = float(w.uniforms[b, t])
            y = min(int(np.searchsorted(C, u, side="right")), V - 1)
            edges = [C[y - 1] if y > 0 else 0.0, C[y]]
            if min(abs(u - e) for e in edges) < tie:
                near = True
        if near:
            ties += 1
            assert 0 <= n[b] <= B
            if pos[b] >= 0:
                assert n[b] < B and 0 <= tok[b] < V
            continue
        assert n[b] == ref["n_accept"][b], (b, n[b], ref["n_accept"][b])
        assert pos[b] == ref["pos"][b], (b, pos[b], ref["pos"][b])
        assert tok[b] == ref["token"][b], (b, tok[b], ref["token"][b])
    return ties


@pytest.mark.parametrize("path", RULE_PATHS)
@pytest.mark.parametrize("name,T", [("sdar8b", 1.0), ("bf16-1003", 1.0), ("f32-777", 0.875),
                                    ("bf16-few", 1.0), ("f32-odd", 1.25), ("f32-max", 1.0)])
def test_sample_matching_matches_oracle(name, T, path):
    """Sample matching (accept iff the target's own inverse-CDF sample at
    u[t-1] equals the draft token; the rejection emits that sample): exact
    against the oracle outside the tie zone.  Half of the draft tokens are
    the target's own samples so that walks get past their first step."""
    w = variant_case(name)
    rng = np.random.default_rng(8)
    tl = synth.to_f64(w.target) / T
    for b in range(len(w.lens)):
        s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
        for k in range(s1 - s0):
            if rng.random() < 0.5:
                t = int(w.tau[s0 + k]) - 1
                p = np.exp(tl[s0 + k] - tl[s0 + k].max()); p /= p.sum()
                y = int(np.searchsorted(np.cumsum(p), float(w.uniforms[b, t]), side="right"))
                w.draft_tokens[s0 + k] = min(y, w.spec.vocab - 1)
    n, tok, pos = run_rule(w, binding.SIMSD_ACCEPT_MATCH, T, path)
    ties = check_match(w, n, tok, pos, T)
    print("%s T=%g %s: %d sequences, %d with a tie-zone draw" % (name, T, path, len(w.lens), ties))
    assert ties <= parity.max_ties(len(w.lens))
    assert (n > 0).any()


def test_rules_alternate_on_one_workspace():
    """Sampling, greedy, matching and sampling again on one workspace (the
    chunk pass's control words and counters shared between the calls):
    every call equals the same call on a fresh zeroed workspace."""
    w = variant_case("bf16-1003")
    dw = DeviceWorkload(w, with_verify=False)
    shared = torch.zeros_like(dw.accept_ws)

    def call(rule, ws):
        greedy = rule == binding.SIMSD_ACCEPT_GREEDY
        for t in (dw.n_accept, dw.token, dw.pos):
            t.fill_(-7)
        binding.accept(dw.target, dw.draft if rule == binding.SIMSD_ACCEPT_SAMPLE else None,
                       dw.draft_tokens, dw.tau, dw.cu_B, None if greedy else dw.uniforms,
                       dw.n_accept, dw.token, dw.pos, ws, dw.total_B, dw.B_max, rule=rule)
        torch.cuda.synchronize()
        return [t.cpu().numpy().copy() for t in (dw.n_accept, dw.token, dw.pos)]

    # (the shared workspace's status is read only at the end: reading it
    # would also clear the control words the calls must reset themselves)
    for rule in (binding.SIMSD_ACCEPT_SAMPLE, binding.SIMSD_ACCEPT_GREEDY, binding.SIMSD_ACCEPT_MATCH,
                 binding.SIMSD_ACCEPT_SAMPLE):
        got = call(rule, shared)
        fresh = torch.zeros_like(dw.accept_ws)
        ref = call(rule, fresh)
        assert binding.read_status(fresh) == 0
        for g, r in zip(got, ref):
            np.testing.assert_array_equal(g, r)
    assert binding.read_status(shared) == 0
