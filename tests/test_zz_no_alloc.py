"""simsd_accept_noalloc: acceptance for callers that cannot allocate.

Serving loops with a fixed device-memory budget, or plugins whose host
framework owns all device memory, cannot hand the library a workspace from
cudaMalloc.  The no-allocation entry point keeps its scratch in a static
device array instead.  Its decisions must equal those of simsd_accept on a
workspace of the same size (the same kernel on the same inputs, so integers
compare exactly), and agree with simsd_accept's default path within the
tie zone of the other acceptance tests, on two calls in a row -- the second
call sees the first call's leftovers in the shared array -- and the static
array covers the single-launch scratch of every valid size (one status
word), while invalid sizes are refused before anything runs.

This file is named to be collected last: it must pass both on its own in a
fresh process and after every other test.
"""
import numpy as np
import pytest
import torch

import parity
import synth
from speculative_decoding_diffusion_gb300 import binding
from speculative_decoding_diffusion_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu


def _outputs(dw):
    return (dw.n_accept.cpu().numpy().copy(), dw.token.cpu().numpy().copy(),
            dw.pos.cpu().numpy().copy())


def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row.  The static scratch holds the status word, so the
    no-allocation call runs the single-launch kernel: its decisions equal
    simsd_accept's on a workspace of the same size (the same kernel), and
    agree with the oracle -- and so with simsd_accept's default two-kernel
    path -- exactly outside the tie zone the other acceptance tests use."""
    w = synth.config(1)                       # 16 x vocab 151936, bf16
    dw = DeviceWorkload(w, with_verify=False)
    args = (dw.target, dw.draft, dw.draft_tokens, dw.tau, dw.cu_B, dw.uniforms,
            dw.n_accept, dw.token, dw.pos, dw.total_B, dw.B_max)
    status_ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(77)
    for call in range(2):
        if call == 1:   # second call: other uniforms, same shared scratch
            w.uniforms = rng.random(tuple(dw.uniforms.shape), dtype=np.float32)
            dw.uniforms.copy_(torch.from_numpy(w.uniforms))
        binding.accept(*args[:9], status_ws, *args[9:])
        torch.cuda.synchronize()
        same_kernel = _outputs(dw)
        dw.accept()
        torch.cuda.synchronize()
        default = _outputs(dw)
        for t in (dw.n_accept, dw.token, dw.pos):
            t.fill_(-7)
        binding.accept_noalloc(*args)
        torch.cuda.synchronize()
        got = _outputs(dw)
        for g, r in zip(got, same_kernel):
            np.testing.assert_array_equal(g, r)
        assert (got[0] >= 0).all()
        ref = parity.oracle_accept(w)
        parity.check_accept(w, ref, *got)
        parity.check_accept(w, ref, *default)


def test_noalloc_scratch_covers_every_size_and_refuses_bad_ones():
    lib = binding.lib()
    d = binding.AcceptDesc()
    for k, v in dict(batch=4096, vocab=1 << 21, total_B=4096 * 32, B_max=32,
                     dtype=binding.SIMSD_F32).items():
        setattr(d, k, v)
    # the largest valid sizes: every rule's two-kernel path asks for more
    # than the array holds, so the no-allocation entry point runs the
    # single-launch path there, whose scratch is the status word alone
    for rule in (binding.SIMSD_ACCEPT_SAMPLE, binding.SIMSD_ACCEPT_GREEDY,
                 binding.SIMSD_ACCEPT_MATCH):
        d.rule = rule
        assert lib.simsd_accept_workspace_size(d) > 4096
    d.rule = binding.SIMSD_ACCEPT_SAMPLE
    fake = 1 << 40   # never dereferenced: every call below returns before launching
    for f in ("target_logits", "draft_logits", "draft_tokens", "tau", "cu_B",
              "uniforms", "n_accept", "token", "pos"):
        setattr(d, f, fake)
    d.vocab = (1 << 21) + 1                          # beyond the vocabulary limit
    assert lib.simsd_accept_workspace_size(d) == 0
    assert lib.simsd_accept_noalloc(d, None) == 2    # SIMSD_ERR_SHAPE
    d.vocab = 1000
    d.target_logits = None
    assert lib.simsd_accept_noalloc(d, None) == 1    # SIMSD_ERR_NULL


def test_noalloc_chunked_path_at_small_sizes_in_turn():
    """Small calls whose chunk partials fit the static array take the
    two-kernel path there.  Calls of other sizes and rules in turn put their
    partials at other offsets of the same array; the chunk pass's control
    words sit at one fixed offset beside the status word, so every call
    starts from zeros and matches the oracle (greedy exactly, sampling and
    matching outside the tie zone)."""
    import oracle
    cases = [("bf16", 1003, 2, 2, binding.SIMSD_ACCEPT_SAMPLE),
             ("f32", 777, 3, 1, binding.SIMSD_ACCEPT_GREEDY),
             ("bf16", 4104, 2, 3, binding.SIMSD_ACCEPT_MATCH),
             ("bf16", 1003, 2, 2, binding.SIMSD_ACCEPT_GREEDY),
             ("f32", 777, 3, 1, binding.SIMSD_ACCEPT_SAMPLE)]
    for dtype, vocab, batch, B, rule in cases:
        spec = synth.Spec(name="na", batch=batch, prompt=0, B=B, Hq=1, Hkv=1, hd=64, dtype=dtype,
                          vocab=vocab, logit_sd=2.0, noise_sd=1.0)
        w = synth.make(spec, seed=vocab + batch + rule)
        dw = DeviceWorkload(w, with_verify=False)
        probe = binding.accept_workspace_size(dw.target, dw.draft, dw.draft_tokens, dw.tau,
                                              dw.cu_B, dw.uniforms, dw.n_accept, dw.token,
                                              dw.pos, dw.total_B, dw.B_max, rule=rule)
        assert probe <= binding.SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES, (dtype, vocab, probe)
        greedy = rule == binding.SIMSD_ACCEPT_GREEDY
        if greedy:   # most draft tokens the argmax, so walks get past step 1
            a = synth.to_f64(w.target).argmax(1).astype(np.int32)
            w.draft_tokens = np.where(np.arange(len(a)) % 3 != 0, a, w.draft_tokens).astype(np.int32)
            dw.draft_tokens.copy_(torch.from_numpy(w.draft_tokens))
        for t in (dw.n_accept, dw.token, dw.pos):
            t.fill_(-7)
        binding.accept_noalloc(dw.target, None if rule != binding.SIMSD_ACCEPT_SAMPLE else dw.draft,
                               dw.draft_tokens, dw.tau, dw.cu_B, None if greedy else dw.uniforms,
                               dw.n_accept, dw.token, dw.pos, dw.total_B, dw.B_max, rule=rule)
        torch.cuda.synchronize()
        n, tok, pos = _outputs(dw)
        if greedy:
            ref = oracle.accept_greedy(w.cu_B, synth.to_f64(w.target), w.draft_tokens, w.tau)
            np.testing.assert_array_equal(n, ref["n_accept"])
            np.testing.assert_array_equal(pos, ref["pos"])
            np.testing.assert_array_equal(tok, ref["token"])
        elif rule == binding.SIMSD_ACCEPT_SAMPLE:
            parity.check_accept(w, parity.oracle_accept(w), n, tok, pos)
        else:
            from test_gpu_accept import check_match
            assert check_match(w, n, tok, pos) <= parity.max_ties(len(w.lens))
