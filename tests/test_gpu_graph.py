"""GPU parity of the draft-graph verification layout (simsd_verify_attn
with node_size > 0) against the oracle: each sequence's new tokens are
candidate states of the block (Spiffy's draft-graph nodes), a row attends
to the prompt and to its own node, every node's token k sits at position
lens + k.  Every output row is compared (bf16 I/O: 2e-2, fp32: 1e-4), and
the cache slots written are checked as for the paired layout.
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


def graph_spec(**kw):
    base = dict(name="graph", batch=1, prompt=64, B=4, Hq=8, Hkv=2, hd=128, dtype="bf16",
                rope_base=1e6, vocab=1000, shuffled_pages=True)
    base.update(kw)
    return synth.Spec(**base)


def run_graph(w, node_size):
    dw = DeviceWorkload(w, with_accept=False)
    binding.verify_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_table, dw.k_new, dw.v_new,
                        None, dw.lens, dw.cu_B, dw.out, dw.verify_ws, dw.total_B, dw.B_max,
                        w.spec.rope_base, w.spec.sm_scale, node_size=node_size)
    torch.cuda.synchronize()
    st = binding.read_status(dw.verify_ws)
    return st, dw, dw.out.float().cpu().numpy()


def oracle_graph(w, node_size):
    outs = []
    off = w.prompt_offsets
    for b in range(len(w.lens)):
        t0, t1 = 2 * int(w.cu_B[b]), 2 * int(w.cu_B[b + 1])
        P = int(w.lens[b])
        kp = parity.prompt_keys_f64(w, b)
        vp = synth.to_f64(w.v_prompt[off[b]:off[b + 1]])
        outs.append(oracle.verify_attn_graph_seq(
            synth.to_f64(w.q[t0:t1]), kp if P else None, vp if P else None,
            synth.to_f64(w.k_new[t0:t1]), synth.to_f64(w.v_new[t0:t1]), node_size,
            w.spec.rope_base, w.spec.sm_scale))
    return np.concatenate(outs, 0)


# (node size, section B): 2B new tokens = 2B / node_size nodes
CASES = [(4, 4), (8, 16), (16, 16), (32, 32), (1, 4), (3, 3), (6, 9), (32, 16)]


@pytest.mark.parametrize("hd", [128, 64])
@pytest.mark.parametrize("node_size,B", CASES)
def test_graph_layout_matches_oracle(node_size, B, hd):
    spec = graph_spec(batch=5, hd=hd, B=B)
    w = synth.make(spec, seed=node_size * 100 + B, with_logits=False, lens=[0, 1, 17, 300, 1000])
    st, _, got = run_graph(w, node_size)
    assert st == 0
    parity.check_attention(got, oracle_graph(w, node_size), "bf16")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 2), (32, 8)])
def test_graph_head_groupings(Hq, Hkv):
    spec = graph_spec(batch=3, Hq=Hq, Hkv=Hkv, B=8, prompt=(50, 700))
    w = synth.make(spec, seed=Hq + Hkv, with_logits=False)
    st, _, got = run_graph(w, 4)
    assert st == 0
    parity.check_attention(got, oracle_graph(w, 4), "bf16")


@pytest.mark.parametrize("hd", [128, 64])
def test_graph_fp32(hd):
    spec = graph_spec(batch=3, hd=hd, dtype="f32", Hq=4, Hkv=2, qkv_sd=0.125, q_scale=1.0,
                      raw_prompt_keys=True, rope_base=1e4, B=6)
    w = synth.make(spec, seed=9, with_logits=False, lens=[0, 37, 200])
    st, _, got = run_graph(w, 4)
    assert st == 0
    parity.check_attention(got, oracle_graph(w, 4), "f32")


def test_graph_sdar_sized():
    """16 sequences x 1024-token prompts, 4 candidate nodes of 8 tokens each
    (32 new tokens per sequence), 32 / 8 heads, head dim 128."""
    w = synth.make(synth.CONFIGS[1], seed=11, with_logits=False, Bs=[16] * 16)
    st, _, got = run_graph(w, 8)
    assert st == 0
    parity.check_attention(got, oracle_graph(w, 8), "bf16")


def test_graph_cache_positions():
    """Token k of every node is written to its own cache slot, rotated at
    position lens + k: equal raw keys in two nodes give bit-identical keys."""
    spec = graph_spec(batch=2, B=8)
    w = synth.make(spec, seed=3, with_logits=False, lens=[30, 64])
    S = 4
    for b in range(2):
        t0 = 2 * int(w.cu_B[b])
        for n in range(1, 4):            # nodes 1..3 copy node 0's raw keys
            w.k_new[t0 + n * S:t0 + (n + 1) * S] = w.k_new[t0:t0 + S]
    st, dw, _ = run_graph(w, S)
    assert st == 0
    k = dw.k_cache.view(torch.int16).cpu().numpy()
    for b in range(2):
        P = int(w.lens[b])
        for n in range(1, 4):
            for kk in range(S):
                s1, s2 = P + kk, P + n * S + kk
                np.testing.assert_array_equal(k[w.block_table[b, s1 // 16], :, s1 % 16],
                                              k[w.block_table[b, s2 // 16], :, s2 % 16])


def test_graph_sections_not_whole_nodes_are_flagged():
    spec = graph_spec(batch=2, B=5)                 # 10 new tokens: not whole nodes of 4
    w = synth.make(spec, seed=4, with_logits=False, lens=[40, 50])
    st, _, _ = run_graph(w, 4)
    assert st & 2
