"""GPU parity of simsd_verify_attn (K1 + K2 + K3) against the fp64 oracle.

Every case calls the library through the C ABI on seeded synthetic inputs
and is compared on every output row, the full-size workloads included.  Also checked: the
cache slots K1 writes (placement bit-exact, values within bf16 rounding of
the oracle's rotation), that nothing else in the cache changes, the RoPE
copy (equal raw inputs at D_k and D~_k give bit-identical cached keys),
invariance of slot outputs to keys the mask hides, and run-to-run
determinism.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import parity
import synth
from speculative_decoding_diffusion_gb300 import binding
from speculative_decoding_diffusion_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu


def small_spec(**kw):
    base = dict(name="small", batch=1, prompt=64, B=4, Hq=8, Hkv=2, hd=128,
                dtype="bf16", rope_base=1e6, vocab=1000, shuffled_pages=True)
    base.update(kw)
    return synth.Spec(**base)


def run(w):
    dw = DeviceWorkload(w, with_accept=False)
    dw.verify()
    torch.cuda.synchronize()
    assert binding.read_status(dw.verify_ws) == 0
    return dw, dw.out.float().cpu().numpy()


def test_tiny_fp32_all_rows():
    w = synth.config(0, with_logits=False)
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "f32")


def test_sdar_b4_all_rows():
    w = synth.config(1, with_logits=False)
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "bf16")


RAGGED = [
    # lens, Bs: empty prompt, one-token prompt, page-aligned and ragged tails
    ([0, 1, 17, 300, 1000], [1, 3, 4, 8, 16]),
    ([15, 16, 127, 128, 129], [2, 5, 7, 1, 4]),
    ([4096, 33, 2049], [8, 8, 3]),
]


@pytest.mark.parametrize("hd", [128, 64])
@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_ragged_bf16(hd, case):
    lens, Bs = RAGGED[case]
    spec = small_spec(batch=len(lens), hd=hd)
    w = synth.make(spec, seed=100 + case, with_logits=False, lens=lens, Bs=Bs)
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "bf16")


@pytest.mark.parametrize("Hq,Hkv,B", [(8, 8, 4), (16, 2, 8), (8, 2, 32), (4, 4, 32)])
def test_head_groupings_and_long_sections(Hq, Hkv, B):
    # G = 1, G = 8, and B = 32 (256 query rows: two row tiles)
    spec = small_spec(batch=2, Hq=Hq, Hkv=Hkv, B=B, prompt=(100, 700))
    w = synth.make(spec, seed=7 + B, with_logits=False)
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "bf16")


@pytest.mark.parametrize("hd", [128, 64])
def test_fp32_ragged(hd):
    spec = small_spec(batch=3, hd=hd, dtype="f32", Hq=4, Hkv=2, qkv_sd=0.125,
                      q_scale=1.0, raw_prompt_keys=True, rope_base=1e4)
    w = synth.make(spec, seed=9, with_logits=False, lens=[0, 37, 200], Bs=[1, 4, 6])
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "f32")


def test_scaled_softmax():
    spec = small_spec(batch=2, q_scale=1.0, sm_scale=float(1 / np.sqrt(128)))
    w = synth.make(spec, seed=5, with_logits=False, lens=[500, 80], Bs=[4, 8])
    _, got = run(w)
    parity.check_attention(got, parity.oracle_all(w), "bf16")


def _cache_views(dw):
    return dw.k_cache.float().cpu().numpy(), dw.v_cache.float().cpu().numpy()


def test_cache_append_placement():
    spec = small_spec(batch=3, dtype="bf16")
    w = synth.make(spec, seed=21, with_logits=False, lens=[5, 16, 40], Bs=[3, 8, 2])
    dw = DeviceWorkload(w, with_accept=False, extra_pages=3)
    k0, v0 = _cache_views(dw)
    dw.verify()
    torch.cuda.synchronize()
    k1, v1 = _cache_views(dw)
    touched = np.zeros(k0.shape[0] * 16, bool).reshape(k0.shape[0], 16)
    for b in range(3):
        P, B = int(w.lens[b]), int(w.Bs[b])
        t0 = 2 * int(w.cu_B[b])
        pos_new = np.concatenate([P + np.arange(B), P + np.arange(B)])
        ref_k = oracle.rope(synth.to_f64(w.k_new[t0:t0 + 2 * B]), pos_new, w.spec.rope_base)
        for j in range(2 * B):
            slot = P + j
            page = w.block_table[b, slot // 16]
            touched[page, slot % 16] = True
            got_k = k1[page, :, slot % 16, :]
            got_v = v1[page, :, slot % 16, :]
            np.testing.assert_array_equal(got_v, synth.to_f64(w.v_new[t0 + j]))
            # one bf16 rounding of the rotated key
            np.testing.assert_allclose(got_k, ref_k[j], rtol=2 ** -8, atol=1e-6)
    # every other slot is untouched, bit for bit
    mask = ~touched
    for before, after in ((k0, k1), (v0, v1)):
        a = before.transpose(0, 2, 1, 3)[mask]
        c = after.transpose(0, 2, 1, 3)[mask]
        np.testing.assert_array_equal(a, c)


def test_rope_copy_pairs_bit_identical():
    spec = small_spec(batch=2)
    w = synth.make(spec, seed=3, with_logits=False, lens=[30, 64], Bs=[4, 5])
    for b in range(2):   # make D~_k's raw key equal to D_k's
        t0, B = 2 * int(w.cu_B[b]), int(w.Bs[b])
        w.k_new[t0 + B:t0 + 2 * B] = w.k_new[t0:t0 + B]
    dw, _ = run(w)
    k = dw.k_cache.view(torch.int16).cpu().numpy()
    for b in range(2):
        P, B = int(w.lens[b]), int(w.Bs[b])
        for kk in range(B):
            s1, s2 = P + kk, P + B + kk
            a = k[w.block_table[b, s1 // 16], :, s1 % 16]
            c = k[w.block_table[b, s2 // 16], :, s2 % 16]
            np.testing.assert_array_equal(a, c)


def test_hidden_keys_do_not_change_slot_rows():
    spec = small_spec(batch=1, Hq=4, Hkv=1)
    B = 6
    w = synth.make(spec, seed=13, with_logits=False, lens=[50], Bs=[B])
    tau = w.tau[:B]
    _, base = run(w)
    G = 4
    for j in range(B):
        w2 = dataclasses.replace(w, k_new=w.k_new.copy(), v_new=w.v_new.copy())
        w2.k_new[j] = synth.f32_to_bf16_bits(np.full(w.k_new[j].shape, 3.0, np.float32))
        w2.v_new[j] = synth.f32_to_bf16_bits(np.full(w.v_new[j].shape, -2.0, np.float32))
        _, got = run(w2)
        for i in range(B):
            if tau[j] >= tau[i]:      # D_j not yet revealed for slot i: hidden
                np.testing.assert_array_equal(got[B + i], base[B + i])
            else:
                assert np.abs(got[B + i] - base[B + i]).max() > 0


def test_deterministic():
    w = synth.config(1, with_logits=False)
    dw = DeviceWorkload(w, with_accept=False)
    outs = []
    for _ in range(3):
        dw.verify()
        outs.append(dw.out.view(torch.int16).cpu().numpy().copy())
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_all_rows(cfg):
    """Every output row of the 64 x 4096, 8 x 32768 (shuffled pages) and
    256-sequence ragged workloads, in the bench's launch configuration,
    against the fp64 oracle."""
    w = synth.config(cfg, with_logits=False)
    _, got = run(w)
    assert np.isfinite(got).all()
    ref = parity.oracle_full_size(w)
    err = parity.check_attention(got, ref, "bf16")
    print("cfg%d: %d rows, max row rel err %.3g, mean %.3g"
          % (cfg, err.size, err.max(), err.mean()))
