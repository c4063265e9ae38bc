"""Device-side failure handling on the GPU, without faulting it.

- Descriptors whose device arrays disagree with the host-side sizes (a
  cu_B beyond total_B, a section longer than B_max) and step labels that are
  not a permutation: the kernels set the status word's bad-input bit, skip
  the sequence and report its outputs as "no walk" (n_accept 0, token -1,
  pos -1), reading nothing out of range.  The buffers are over-allocated so
  that even an unguarded read would stay inside memory.
- The bounded waits: with wait_polls < 0 every wait gives up at once; the
  call returns, the status word's timeout bit is set, the cache is left
  untouched, the acceptance reports "no walk", and the next call on the
  same context is correct again.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import synth
from speculative_decoding_diffusion_gb300 import binding
from speculative_decoding_diffusion_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu

BAD_INPUT, TIMEOUT = 2, 1


def accept_spec(**kw):
    base = dict(name="acc", batch=3, prompt=0, B=4, Hq=1, Hkv=1, hd=64, dtype="bf16",
                vocab=4096, logit_sd=2.0, noise_sd=1.0)
    base.update(kw)
    return synth.Spec(**base)


# every rule has a chunked path (the full workspace) and a single-launch
# cluster path (a workspace of the status word alone)
PATHS = ["chunked", "cluster"]


def run_rule(dw, rule, cu_B_dev, tau_dev, total_B, B_max, path="chunked", wait_polls=0):
    for t in (dw.n_accept, dw.token, dw.pos):
        t.fill_(-7)
    ws = dw.accept_ws if path == "chunked" else torch.zeros(256, dtype=torch.uint8, device="cuda")
    greedy = rule == binding.SIMSD_ACCEPT_GREEDY
    binding.accept(dw.target, None if rule != binding.SIMSD_ACCEPT_SAMPLE else dw.draft,
                   dw.draft_tokens, tau_dev, cu_B_dev, None if greedy else dw.uniforms,
                   dw.n_accept, dw.token, dw.pos, ws, total_B, B_max, rule=rule,
                   wait_polls=wait_polls)
    torch.cuda.synchronize()
    st = binding.read_status(ws)
    return st, dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()


def big_accept_workload():
    # 16 rows of logits behind a descriptor that claims 12 (3 x 4)
    w = synth.make(accept_spec(batch=4), seed=31)
    dw = DeviceWorkload(w, with_verify=False)
    return w, dw


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("rule", [binding.SIMSD_ACCEPT_SAMPLE, binding.SIMSD_ACCEPT_GREEDY,
                                  binding.SIMSD_ACCEPT_MATCH])
def test_accept_cu_B_beyond_descriptor(rule, path):
    w, dw = big_accept_workload()
    # the descriptor says 3 sequences, total_B 12, B_max 4; the device cu_B
    # gives sequence 1 a section of 6 (> B_max) and sequence 2 rows 10..13
    # (past total_B); only sequence 0 is well formed
    cu = torch.tensor([0, 4, 10, 14], dtype=torch.int32, device="cuda")
    st, n, tok, pos = run_rule(dw, rule, cu, dw.tau, 12, 4, path)
    assert st & BAD_INPUT
    for b in (1, 2):
        assert (n[b], tok[b], pos[b]) == (0, -1, -1), (b, n[b], tok[b], pos[b])
    ref_w = synth.make(accept_spec(batch=4), seed=31)
    if rule == binding.SIMSD_ACCEPT_GREEDY:
        ref = oracle.accept_greedy(ref_w.cu_B[:2], synth.to_f64(ref_w.target[:4]),
                                   ref_w.draft_tokens[:4], ref_w.tau[:4])
        assert (n[0], tok[0], pos[0]) == (ref["n_accept"][0], ref["token"][0], ref["pos"][0])
    else:
        assert 0 <= n[0] <= 4


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("rule", [binding.SIMSD_ACCEPT_SAMPLE, binding.SIMSD_ACCEPT_GREEDY,
                                  binding.SIMSD_ACCEPT_MATCH])
def test_accept_tau_not_a_permutation(rule, path):
    w, dw = big_accept_workload()
    tau = w.tau.copy()
    tau[4:8] = [1, 1, 2, 3]                  # sequence 1: label 4 missing, 1 twice
    tau[8:12] = [1, 2, 3, 5]                 # sequence 2: a label outside 1..4
    tau_dev = torch.from_numpy(tau).to("cuda")
    st, n, tok, pos = run_rule(dw, rule, dw.cu_B, tau_dev, w.total_B, w.B_max, path)
    assert st & BAD_INPUT
    for b in (1, 2):
        assert (n[b], tok[b], pos[b]) == (0, -1, -1), (b, n[b], tok[b], pos[b])
    for b in (0, 3):                         # untouched sequences still walk
        assert 0 <= n[b] <= 4 and (pos[b] == -1) == (n[b] == 4)


@pytest.mark.parametrize("path", PATHS)
def test_greedy_rows_without_a_larger_entry_give_index_zero(path):
    """A target row of -inf everywhere (or NaN everywhere) has no entry
    larger than another: the argmax is index 0, as in the oracle."""
    w = synth.make(accept_spec(batch=2, dtype="f32", vocab=1000), seed=5)
    s0 = int(w.cu_B[1])
    order = np.argsort(w.tau[s0:s0 + 4])     # slots in step order
    w.target[s0 + order[0]] = -np.inf
    w.target[int(w.cu_B[0]) + int(np.argsort(w.tau[:4])[0])] = np.nan
    w.draft_tokens[:] = 5                    # not index 0: both first steps reject
    dw = DeviceWorkload(w, with_verify=False)
    st, n, tok, pos = run_rule(dw, binding.SIMSD_ACCEPT_GREEDY, dw.cu_B, dw.tau, w.total_B, 4, path)
    assert st == 0
    ref = oracle.accept_greedy(w.cu_B, synth.to_f64(w.target), w.draft_tokens, w.tau)
    np.testing.assert_array_equal(n, ref["n_accept"])
    np.testing.assert_array_equal(tok, ref["token"])
    np.testing.assert_array_equal(pos, ref["pos"])
    assert (tok == 0).all() and (n == 0).all()


def small_verify_workload(seed=41):
    spec = synth.Spec(name="small", batch=2, prompt=64, B=4, Hq=8, Hkv=2, hd=128,
                      dtype="bf16", rope_base=1e6, vocab=1000, shuffled_pages=True)
    return synth.make(spec, seed=seed, with_logits=False, lens=[300, 80], Bs=[4, 4])


def test_verify_cu_B_beyond_descriptor():
    w = small_verify_workload()
    dw = DeviceWorkload(w, with_accept=False, extra_pages=4)
    dw.out.fill_(7.0)
    k0 = dw.k_cache.clone()
    cu = torch.tensor([0, 4, 13], dtype=torch.int32, device="cuda")   # B_1 = 9 > B_max 4
    binding.verify_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.k_new, dw.v_new,
                        dw.tau, dw.lens, cu, dw.out, dw.verify_ws, dw.total_B, dw.B_max,
                        dw.rope_base, dw.sm_scale)
    torch.cuda.synchronize()
    assert binding.read_status(dw.verify_ws) & BAD_INPUT
    out = dw.out.float().cpu().numpy()
    assert (out[8:] == 7.0).all()            # sequence 1's rows: skipped
    ref = parity.oracle_seq(w, 0)
    parity.check_attention(out[:8], ref, "bf16")
    # sequence 1's cache slots were not written
    k1 = dw.k_cache
    P1 = int(w.lens[1])
    for j in range(8):
        slot = P1 + j
        page = int(w.block_table[1, slot // 16])
        assert torch.equal(k1[page, :, slot % 16], k0[page, :, slot % 16])


def test_verify_wait_that_gives_up_returns_a_status():
    w = small_verify_workload(seed=43)
    dw = DeviceWorkload(w, with_accept=False)
    k0, v0 = dw.k_cache.clone(), dw.v_cache.clone()
    args = (dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.k_new, dw.v_new, dw.tau,
            dw.lens, dw.cu_B, dw.out, dw.verify_ws, dw.total_B, dw.B_max, dw.rope_base,
            dw.sm_scale)
    binding.verify_attn(*args, wait_polls=-1)
    torch.cuda.synchronize()
    st = binding.read_status(dw.verify_ws)
    assert st & TIMEOUT, st
    assert torch.equal(dw.k_cache, k0) and torch.equal(dw.v_cache, v0)
    # the context is still usable: the next call is correct
    binding.verify_attn(*args)
    torch.cuda.synchronize()
    assert binding.read_status(dw.verify_ws) == 0
    parity.check_attention(dw.out.float().cpu().numpy(), parity.oracle_all(w), "bf16")


def test_accept_wait_that_gives_up_returns_a_status():
    # a batch whose sampling chunk pass runs the ring (the ring-free pass
    # for small batches has no bounded waits)
    w = synth.make(accept_spec(batch=64, B=8, vocab=151936), seed=2)
    dw = DeviceWorkload(w, with_verify=False)
    args = (dw.target, dw.draft, dw.draft_tokens, dw.tau, dw.cu_B, dw.uniforms,
            dw.n_accept, dw.token, dw.pos, dw.accept_ws, dw.total_B, dw.B_max)
    for t in (dw.n_accept, dw.token, dw.pos):
        t.fill_(-7)
    binding.accept(*args, wait_polls=-1)
    torch.cuda.synchronize()
    assert binding.read_status(dw.accept_ws) & TIMEOUT
    n, tok, pos = dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()
    assert (n == 0).all() and (tok == -1).all() and (pos == -1).all()
    binding.accept(*args)
    torch.cuda.synchronize()
    assert binding.read_status(dw.accept_ws) == 0
    n, tok, pos = dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()
    parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)


def test_small_sampling_batches_have_no_bounded_waits():
    """The sampling rule's chunk pass for small batches loads each part
    directly (no ring, no waits) and the finishing kernel waits on nothing
    either: with every wait set to give up at once, the call still returns
    the oracle's decisions and no timeout bit."""
    w = synth.config(1)
    dw = DeviceWorkload(w, with_verify=False)
    binding.accept(dw.target, dw.draft, dw.draft_tokens, dw.tau, dw.cu_B, dw.uniforms,
                   dw.n_accept, dw.token, dw.pos, dw.accept_ws, dw.total_B, dw.B_max, wait_polls=-1)
    torch.cuda.synchronize()
    assert binding.read_status(dw.accept_ws) == 0
    n, tok, pos = dw.n_accept.cpu().numpy(), dw.token.cpu().numpy(), dw.pos.cpu().numpy()
    parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)


@pytest.mark.parametrize("rule,batch,vocab", [(binding.SIMSD_ACCEPT_GREEDY, 6, 40000),
                                              (binding.SIMSD_ACCEPT_MATCH, 6, 40000),
                                              (binding.SIMSD_ACCEPT_SAMPLE, 200, 151936)])
def test_chunk_pass_that_gives_up_means_no_walk(rule, batch, vocab):
    """The chunked path with every wait giving up at once: the chunk pass
    raises its give-up flag, so the kernel after it reports "no walk" for
    every sequence (whatever stale partials the workspace holds) and sets
    the timeout bit; it puts the chunk pass's control words back to zero, so
    the next call on the same workspace is correct (also with more
    sequences than SMs: one finishing CTA per sequence).  The sampling case
    is a batch large enough for the ring."""
    w = synth.make(accept_spec(batch=batch, B=(1, 3, 4), vocab=vocab), seed=17)
    dw = DeviceWorkload(w, with_verify=False)
    # a correct call first leaves real partials in the workspace
    st, n0, tok0, pos0 = run_rule(dw, rule, dw.cu_B, dw.tau, w.total_B, w.B_max)
    assert st == 0
    st, n, tok, pos = run_rule(dw, rule, dw.cu_B, dw.tau, w.total_B, w.B_max, wait_polls=-1)
    assert st & TIMEOUT, st
    assert (n == 0).all() and (tok == -1).all() and (pos == -1).all(), (n, tok, pos)
    for _ in range(2):
        st, n, tok, pos = run_rule(dw, rule, dw.cu_B, dw.tau, w.total_B, w.B_max)
        assert st == 0
        np.testing.assert_array_equal(n, n0)
        np.testing.assert_array_equal(tok, tok0)
        np.testing.assert_array_equal(pos, pos0)
