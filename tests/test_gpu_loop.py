"""GPU parity of the blockwise loop's steps against the oracle: the
draft-side step (simsd_draft_step), the walk from the decided steps
(simsd_accept with `decided`), the commit (simsd_commit), and several
passes of the whole loop (draft step -> verification -> acceptance ->
commit) with the cache advancing as blocks close.

Decisions are compared exactly, except where fp32 rounding may flip them
(an inverse-CDF draw whose u lies within parity.TIE_RESIDUAL of a bin
edge; two open slots whose confidences are within TIE_CONF of each other):
there the GPU's choice is checked for validity.  The loop is checked pass
by pass from the GPU's own state, so one tie cannot derail the rest.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import parity
import synth
from oracle import loop
from speculative_decoding_diffusion_gb300 import binding
from speculative_decoding_diffusion_gb300.staging import DeviceWorkload, to_device

pytestmark = pytest.mark.gpu

TIE_CONF = 1e-6        # relative difference of two confidences (fp32 on the GPU)


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to("cuda")


def ws():
    return torch.zeros(256, dtype=torch.uint8, device="cuda")


def softmax64(row):
    p = np.exp(row - row.max())
    return p / p.sum()


def draft_on_gpu(w, draft_dev, u, decided=None, tau_prev=None, tokens_prev=None, T=1.0,
                 chunked=False):
    """chunked: the workspace the library asks for (the chunk pass and one
    CTA per sequence); else only the status word (the cluster kernel)."""
    n = w.total_B
    tokens = dev_i32(np.zeros(n) if tokens_prev is None else tokens_prev)
    tau = torch.zeros(n, dtype=torch.int32, device="cuda")
    conf = torch.zeros(n, dtype=torch.float32, device="cuda")
    wsp = ws() if not chunked else torch.zeros(
        binding.draft_workspace_size(draft_dev, dev_i32(w.cu_B), w.total_B, w.B_max, T),
        dtype=torch.uint8, device="cuda")
    binding.draft_step(draft_dev, dev_i32(w.cu_B), torch.from_numpy(u).to("cuda"), tokens, tau,
                       wsp, w.total_B, w.B_max,
                       decided=None if decided is None else dev_i32(decided),
                       tau_prev=None if tau_prev is None else dev_i32(tau_prev),
                       confidence=conf, temperature=T)
    torch.cuda.synchronize()
    st = binding.read_status(wsp)
    return st, tokens.cpu().numpy(), tau.cpu().numpy(), conf.cpu().numpy()


def check_draft(w, draft_rows64, u, got_tok, got_tau, got_conf, ref, decided=None, T=1.0):
    """Exact tokens and labels outside the tie zones; validity inside.
    Returns (token ties, order ties)."""
    tok_ties = ord_ties = 0
    V = draft_rows64.shape[1]
    for b in range(len(w.lens)):
        s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
        d = 0 if decided is None else int(decided[b])
        open_k = [k for k in range(s1 - s0) if ref["confidence"][s0 + k] >= 0]
        for k in open_k:
            q = softmax64(draft_rows64[s0 + k] / T)
            C = np.cumsum(q)
            U = float(u[b, k])
            v = int(ref["draft_tokens"][s0 + k])
            lo = C[v - 1] if v > 0 else 0.0
            np.testing.assert_allclose(got_conf[s0 + k], ref["confidence"][s0 + k], rtol=2e-6)
            if min(U - lo, C[v] - U) >= parity.TIE_RESIDUAL:
                assert got_tok[s0 + k] == v, (b, k, got_tok[s0 + k], v)
            else:
                tok_ties += 1
                g = int(got_tok[s0 + k])
                assert 0 <= g < V and q[g] > 0
                glo = C[g - 1] if g > 0 else 0.0
                assert glo - parity.TIE_RESIDUAL <= U < C[g] + parity.TIE_RESIDUAL
        for k in range(s1 - s0):
            if ref["confidence"][s0 + k] < 0:       # decided: label and token kept
                assert got_tau[s0 + k] == ref["tau"][s0 + k]
                assert got_tok[s0 + k] == ref["draft_tokens"][s0 + k]
        c = np.array([ref["confidence"][s0 + k] for k in open_k])
        close = any(abs(c[i] - c[j]) <= TIE_CONF * max(c[i], c[j])
                    for i in range(len(c)) for j in range(i + 1, len(c)))
        labels = [int(got_tau[s0 + k]) for k in open_k]
        assert sorted(labels) == list(range(d + 1, s1 - s0 + 1))
        if close:
            ord_ties += 1
            continue
        for k in open_k:
            assert got_tau[s0 + k] == ref["tau"][s0 + k], (b, k)
    return tok_ties, ord_ties


@pytest.mark.parametrize("path", ["cluster", "chunked"])
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_draft_step_matches_oracle(cfg, path):
    w = synth.config(cfg)
    u = np.random.default_rng(600 + cfg).random((len(w.lens), w.B_max), dtype=np.float32)
    st, tok, tau, conf = draft_on_gpu(w, to_device(w.draft, "cuda"), u, chunked=path == "chunked")
    assert st == 0
    d64 = synth.to_f64(w.draft)
    ref = oracle.draft_step(w.cu_B, d64, u)
    ties = check_draft(w, d64, u, tok, tau, conf, ref)
    print("cfg%d %s: %d slots, token ties %d, order ties %d" % (cfg, path, w.total_B, *ties))
    assert ties[0] <= parity.max_ties(w.total_B) and ties[1] <= parity.max_ties(len(w.lens))


def loop_spec(**kw):
    base = dict(name="loop", batch=24, prompt=(0, 300), B=(1, 3, 4, 8, 16, 32), Hq=8, Hkv=2,
                hd=128, dtype="bf16", vocab=1000, logit_sd=2.0, noise_sd=(0.2, 2.5),
                shuffled_pages=True)
    base.update(kw)
    return synth.Spec(**base)


@pytest.mark.parametrize("dtype,vocab,T", [("bf16", 1000, 1.0), ("f32", 777, 0.75),
                                           ("bf16", 151936, 1.0), ("bf16", 4096 + 8, 1.25),
                                           ("f32", 40000, 1.0), ("bf16", 9, 1.0)])
def test_draft_step_chunked_mixed_B_and_vocab(dtype, vocab, T):
    """The chunked path on sections of 1 to 32 slots, vocabularies that end
    inside a chunk or a part, rows that are not 16-byte multiples (element
    copies), and temperatures other than 1."""
    w = synth.make(loop_spec(dtype=dtype, vocab=vocab, batch=12), seed=vocab + 5)
    u = np.random.default_rng(vocab + 6).random((len(w.lens), w.B_max), dtype=np.float32)
    st, tok, tau, conf = draft_on_gpu(w, to_device(w.draft, "cuda"), u, T=T, chunked=True)
    assert st == 0
    d64 = synth.to_f64(w.draft)
    ref = oracle.draft_step(w.cu_B, d64, u, temperature=T)
    ties = check_draft(w, d64, u, tok, tau, conf, ref, T=T)
    assert ties[0] <= parity.max_ties(w.total_B) and ties[1] <= parity.max_ties(len(w.lens))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_step_chunked_largest_vocabulary(dtype):
    """The largest vocabulary (2^21): more parts per row than a warp holds
    in the merge and in the part search."""
    vocab = 1 << 21
    w = synth.make(loop_spec(dtype=dtype, vocab=vocab, batch=2, B=(2, 5)), seed=33)
    u = np.random.default_rng(34).random((len(w.lens), w.B_max), dtype=np.float32)
    st, tok, tau, conf = draft_on_gpu(w, to_device(w.draft, "cuda"), u, chunked=True)
    assert st == 0
    d64 = synth.to_f64(w.draft)
    ref = oracle.draft_step(w.cu_B, d64, u)
    ties = check_draft(w, d64, u, tok, tau, conf, ref)
    assert ties[0] <= parity.max_ties(w.total_B) and ties[1] <= parity.max_ties(len(w.lens))


@pytest.mark.parametrize("dtype,vocab,T", [("bf16", 1000, 1.0), ("f32", 777, 0.75),
                                           ("bf16", 151936, 1.0), ("bf16", 4096 + 8, 1.25)])
def test_draft_step_with_decided_slots(dtype, vocab, T):
    """Slots whose labels are at most decided[b] keep their tokens and
    labels; the open ones are drawn and ordered after them."""
    w = synth.make(loop_spec(dtype=dtype, vocab=vocab, batch=12), seed=vocab)
    rng = np.random.default_rng(vocab + 1)
    decided = np.array([rng.integers(0, int(B) + 1) for B in w.Bs], np.int32)
    tokens_prev = rng.integers(0, vocab, w.total_B).astype(np.int32)
    u = rng.random((len(w.lens), w.B_max), dtype=np.float32)
    st, tok, tau, conf = draft_on_gpu(w, to_device(w.draft, "cuda"), u, decided, w.tau,
                                      tokens_prev, T)
    assert st == 0
    d64 = synth.to_f64(w.draft)
    ref = oracle.draft_step(w.cu_B, d64, u, temperature=T, decided=decided, tau_prev=w.tau,
                            tokens_prev=tokens_prev)
    check_draft(w, d64, u, tok, tau, conf, ref, decided, T)


@pytest.mark.parametrize("rule", [binding.SIMSD_ACCEPT_SAMPLE, binding.SIMSD_ACCEPT_GREEDY,
                                  binding.SIMSD_ACCEPT_MATCH])
def test_accept_from_decided_steps(rule):
    """The walk starts at step decided[b] + 1 (all decided: nothing is
    tested and n_accept = B)."""
    w = synth.make(loop_spec(batch=40), seed=77)
    rng = np.random.default_rng(78)
    decided = np.array([rng.integers(0, int(B) + 1) for B in w.Bs], np.int32)
    dw = DeviceWorkload(w, with_verify=False)
    greedy = rule == binding.SIMSD_ACCEPT_GREEDY
    if greedy:   # make walks pass their first steps now and then
        a = synth.to_f64(w.target).argmax(1).astype(np.int32)
        w.draft_tokens = np.where(rng.random(len(a)) < 0.7, a, w.draft_tokens).astype(np.int32)
        dw.draft_tokens.copy_(dev_i32(w.draft_tokens))
    binding.accept(dw.target, dw.draft if rule == binding.SIMSD_ACCEPT_SAMPLE else None,
                   dw.draft_tokens, dw.tau, dw.cu_B, None if greedy else dw.uniforms,
                   dw.n_accept, dw.token, dw.pos, dw.accept_ws, dw.total_B, dw.B_max, rule=rule,
                   decided=dev_i32(decided))
    torch.cuda.synchronize()
    assert binding.read_status(dw.accept_ws) == 0
    n, tok, pos = dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()
    first = decided + 1
    assert (n >= decided).all()
    assert ((decided == w.Bs) <= (n == w.Bs)).all()
    if rule == binding.SIMSD_ACCEPT_SAMPLE:
        ref = oracle.accept(w.cu_B, synth.to_f64(w.target), synth.to_f64(w.draft),
                            w.draft_tokens, w.tau, w.uniforms, first_step=first)
        parity.check_accept(w, ref, n, tok, pos)
    elif greedy:
        ref = oracle.accept_greedy(w.cu_B, synth.to_f64(w.target), w.draft_tokens, w.tau,
                                   first_step=first)
        np.testing.assert_array_equal(n, ref["n_accept"])
        np.testing.assert_array_equal(pos, ref["pos"])
        np.testing.assert_array_equal(tok, ref["token"])
    else:
        ref = oracle.accept_match(w.cu_B, synth.to_f64(w.target), w.draft_tokens, w.tau,
                                  w.uniforms, first_step=first)
        np.testing.assert_array_equal(n, ref["n_accept"])
        np.testing.assert_array_equal(pos, ref["pos"])
        np.testing.assert_array_equal(tok, ref["token"])


def test_commit_matches_oracle_and_rejects_inconsistent_walks():
    rng = np.random.default_rng(90)
    Bs = rng.integers(1, 33, 300).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(Bs)]).astype(np.int32)
    tau = np.concatenate([rng.permutation(int(B)) + 1 for B in Bs]).astype(np.int32)
    n = np.array([rng.integers(0, int(B) + 1) for B in Bs], np.int32)
    pos = np.array([-1 if n[b] == Bs[b] else int(np.nonzero(tau[cu[b]:cu[b + 1]] == n[b] + 1)[0][0])
                    for b in range(len(Bs))], np.int32)
    token = np.where(pos >= 0, rng.integers(0, 5000, len(Bs)), -1).astype(np.int32)
    tokens = rng.integers(0, 5000, int(cu[-1])).astype(np.int32)
    decided = np.minimum(n, rng.integers(0, 33, len(Bs))).astype(np.int32)
    lens = rng.integers(0, 9000, len(Bs)).astype(np.int32)
    ref = oracle.commit(cu, tau, n, token, pos, tokens, decided, lens)
    # two inconsistent walks: a rejection at a slot that is not the next step,
    # and n < B without a rejection
    bad_pos, bad_n = pos.copy(), n.copy()
    b1 = int(np.nonzero(pos >= 0)[0][0])
    bad_pos[b1] = (pos[b1] + 1) % Bs[b1] if Bs[b1] > 1 else 5
    b2 = int(np.nonzero((pos >= 0) & (np.arange(len(Bs)) != b1))[0][0])
    bad_pos[b2] = -1
    args = [dev_i32(x) for x in (cu, tau, bad_n, token, bad_pos)]
    t_d, dec_d, lens_d = dev_i32(tokens), dev_i32(decided), dev_i32(lens)
    done_d = torch.full((len(Bs),), 7, dtype=torch.int32, device="cuda")
    wsp = ws()
    binding.commit(*args, t_d, dec_d, lens_d, done_d, wsp, int(cu[-1]), int(Bs.max()))
    torch.cuda.synchronize()
    assert binding.read_status(wsp) == 2
    got = dict(block_tokens=t_d.cpu().numpy(), decided=dec_d.cpu().numpy(),
               lens=lens_d.cpu().numpy(), done=done_d.cpu().numpy())
    good = np.ones(len(Bs), bool)
    good[[b1, b2]] = False
    for k in ("decided", "lens", "done"):
        np.testing.assert_array_equal(got[k][good], ref[k][good], err_msg=k)
    for b in (b1, b2):       # left unchanged
        assert got["decided"][b] == decided[b] and got["lens"][b] == lens[b] and got["done"][b] == 0
    for b in np.nonzero(good)[0]:
        np.testing.assert_array_equal(got["block_tokens"][cu[b]:cu[b + 1]],
                                      ref["block_tokens"][cu[b]:cu[b + 1]])


class Model:
    """A stand-in for the models around one attention layer: embedding
    tables (a token's query, key and value rows; index V is [MASK]) and,
    per pass, fixed target / draft logit rows and uniforms.  The loop's
    decisions depend on these and on the block state only."""

    def __init__(self, w, passes, seed):
        rng = np.random.default_rng(seed)
        s, V = w.spec, w.spec.vocab
        bf = synth.f32_to_bf16_bits
        self.Eq = bf(rng.standard_normal((V + 1, s.Hq, s.hd), dtype=np.float32) / np.float32(np.sqrt(s.hd)))
        self.Ek = bf(rng.standard_normal((V + 1, s.Hkv, s.hd), dtype=np.float32))
        self.Ev = bf(rng.standard_normal((V + 1, s.Hkv, s.hd), dtype=np.float32))
        n = w.total_B
        self.TL = [bf(rng.standard_normal((n, V), dtype=np.float32) * np.float32(2.0))
                   for _ in range(passes)]
        self.DL = [bf(synth.bf16_bits_to_f32(t) + rng.standard_normal((n, V), dtype=np.float32)
                      * np.float32(rng.uniform(0.3, 2.0))) for t in self.TL]
        self.UD = [rng.random((len(w.lens), w.B_max), dtype=np.float32) for _ in range(passes)]
        self.UA = [rng.random((len(w.lens), w.B_max + 1), dtype=np.float32) for _ in range(passes)]

    def rows(self, w, tokens):
        """q, k, v of the 2B new tokens of every sequence (D: the tokens,
        D~: [MASK]), in the library's token order."""
        V = w.spec.vocab
        idx = []
        for b in range(len(w.lens)):
            s0, s1 = int(w.cu_B[b]), int(w.cu_B[b + 1])
            idx += list(tokens[s0:s1]) + [V] * (s1 - s0)
        idx = np.asarray(idx)
        return self.Eq[idx], self.Ek[idx], self.Ev[idx]


def test_blockwise_loop_passes():
    """Eight passes of the loop over 24 sequences (B from 1 to 32, prompts
    of 0 to 300 tokens), each step checked against the oracle run on the
    GPU's own inputs to that step: the draft step from the block state, the
    walk from the drafted tokens and labels, the commit from the walk, and
    each pass's attention rows over the cache as it stands (earlier closed
    blocks included: their data-section keys at their own positions)."""
    passes = 8
    spec = loop_spec()
    w0 = synth.make(spec, seed=5, with_logits=False)
    # block tables wide enough for a closed block per pass
    rng = np.random.default_rng(6)
    cap = (w0.lens + 2 * w0.Bs + passes * w0.Bs + 15) // 16
    num_pages = int(cap.sum())
    phys = rng.permutation(num_pages)
    bt = np.zeros((len(w0.lens), int(cap.max())), np.int32)
    o = 0
    for b in range(len(w0.lens)):
        bt[b, :cap[b]] = phys[o:o + cap[b]]
        o += int(cap[b])
    w = dataclasses.replace(w0, block_table=bt, num_pages=num_pages, max_pages=int(cap.max()))
    model = Model(w, passes, seed=7)
    dw = DeviceWorkload(w, with_accept=False)
    n, batch = w.total_B, len(w.lens)
    cu_d = dw.cu_B
    tokens = torch.zeros(n, dtype=torch.int32, device="cuda")
    tau = dev_i32(loop.initial_state(w.cu_B, w.lens)["tau"])
    conf = torch.zeros(n, dtype=torch.float32, device="cuda")
    decided = torch.zeros(batch, dtype=torch.int32, device="cuda")
    lens = dw.lens
    n_acc = torch.zeros(batch, dtype=torch.int32, device="cuda")
    tok, pos, done = torch.zeros_like(n_acc), torch.zeros_like(n_acc), torch.zeros_like(n_acc)
    wsd, wsa, wsc = ws(), ws(), ws()
    # the oracle's copy of each sequence's cached prompt: rotated keys, values
    off = w.prompt_offsets
    kp = [synth.to_f64(w.k_prompt[off[b]:off[b + 1]]) for b in range(batch)]
    vp = [synth.to_f64(w.v_prompt[off[b]:off[b + 1]]) for b in range(batch)]
    closed = 0
    for it in range(passes):
        state = dict(block_tokens=tokens.cpu().numpy(), tau=tau.cpu().numpy(),
                     decided=decided.cpu().numpy(), lens=lens.cpu().numpy())
        TL, DL = model.TL[it], model.DL[it]
        TL64, DL64 = synth.to_f64(TL), synth.to_f64(DL)
        tl_d, dl_d = to_device(TL, "cuda"), to_device(DL, "cuda")
        ud, ua = model.UD[it], model.UA[it]
        # 1. draft step (decided slots kept; tau rewritten in place)
        binding.draft_step(dl_d, cu_d, torch.from_numpy(ud).to("cuda"), tokens, tau, wsd,
                           n, w.B_max, decided=decided, tau_prev=tau, confidence=conf)
        drafted = tokens.clone()
        # 2. verification over the block's layout
        q, kn, vn = model.rows(w, drafted.cpu().numpy())
        dw.q.copy_(to_device(q, "cuda"))
        dw.k_new.copy_(to_device(kn, "cuda"))
        dw.v_new.copy_(to_device(vn, "cuda"))
        binding.verify_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.k_new, dw.v_new,
                            tau, lens, cu_d, dw.out, dw.verify_ws, n, w.B_max, w.spec.rope_base,
                            w.spec.sm_scale)
        # 3. the walk from the decided steps
        binding.accept(tl_d, dl_d, tokens, tau, cu_d, torch.from_numpy(ua).to("cuda"), n_acc,
                       tok, pos, wsa, n, w.B_max, decided=decided)
        walk = [x.clone() for x in (n_acc, tok, pos)]
        # 4. commit
        binding.commit(cu_d, tau, n_acc, tok, pos, tokens, decided, lens, done, wsc, n, w.B_max)
        torch.cuda.synchronize()
        for wsx in (wsd, dw.verify_ws, wsa, wsc):
            assert binding.read_status(wsx) == 0
        g_tok, g_tau = drafted.cpu().numpy(), tau.cpu().numpy()
        g_n, g_t, g_p = (x.cpu().numpy() for x in walk)
        # draft step vs the oracle from the block state
        ref_d = oracle.draft_step(w.cu_B, DL64, ud, decided=state["decided"],
                                  tau_prev=state["tau"], tokens_prev=state["block_tokens"])
        check_draft(w, DL64, ud, g_tok, g_tau, conf.cpu().numpy(), ref_d, state["decided"])
        # the walk vs the oracle on the GPU's drafted tokens and labels
        wp = dataclasses.replace(w, target=TL, draft=DL, draft_tokens=g_tok, tau=g_tau,
                                 uniforms=ua)
        ref_a = oracle.accept(w.cu_B, TL64, DL64, g_tok, g_tau, ua,
                              first_step=state["decided"] + 1)
        st_ties, _, _ = parity.check_accept(wp, ref_a, g_n, g_t, g_p)
        assert st_ties == 0
        # commit vs the oracle on the GPU's walk
        ref_c = oracle.commit(w.cu_B, g_tau, g_n, g_t, g_p, g_tok, state["decided"], state["lens"])
        np.testing.assert_array_equal(tokens.cpu().numpy(), ref_c["block_tokens"])
        np.testing.assert_array_equal(decided.cpu().numpy(), ref_c["decided"])
        np.testing.assert_array_equal(lens.cpu().numpy(), ref_c["lens"])
        np.testing.assert_array_equal(done.cpu().numpy(), ref_c["done"])
        # attention of this pass against the oracle over the cache as it was
        out = dw.out.float().cpu().numpy()
        for b in range(batch):
            t0, t1 = 2 * int(w.cu_B[b]), 2 * int(w.cu_B[b + 1])
            P = int(state["lens"][b])
            assert len(kp[b]) == P
            ref = oracle.verify_attn_seq(
                synth.to_f64(q[t0:t1]), kp[b] if P else None, vp[b] if P else None,
                synth.to_f64(kn[t0:t1]), synth.to_f64(vn[t0:t1]), g_tau[w.cu_B[b]:w.cu_B[b + 1]],
                w.spec.rope_base, w.spec.sm_scale)
            parity.check_attention(out[t0:t1], ref, "bf16")
        # a closed block's data-section keys (rotated at their positions)
        # and values join the oracle's prompt
        for b in np.nonzero(ref_c["done"])[0]:
            B, t0, P = int(w.Bs[b]), 2 * int(w.cu_B[b]), int(state["lens"][b])
            kr = oracle.rope(synth.to_f64(kn[t0:t0 + B]), P + np.arange(B), w.spec.rope_base)
            kp[b] = np.concatenate([kp[b].reshape(-1, *kr.shape[1:]), kr])
            vp[b] = np.concatenate([vp[b].reshape(-1, *kr.shape[1:]), synth.to_f64(vn[t0:t0 + B])])
            closed += 1
    assert closed >= batch        # blocks closed along the way
