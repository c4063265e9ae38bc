"""Host-side checks of libsimsd.so (no GPU needed, no kernel launched).

- the library loads and exports every function include/simsd.h declares;
- simsd_layout matches the oracle bit for bit (positions and mask) over all
  orders for B <= 6 and random orders up to B = 32;
- argument errors come back as status codes before anything is launched.
"""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_diffusion_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_diffusion_gb300 import build
    build.build()
    return binding.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(simsd_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert lib.simsd_version() >= 100
    for code in range(9):
        assert binding.status_string(code) != "unknown status"


def test_layout_matches_oracle_all_orders(lib):
    for B in range(1, 7):
        for P in (0, 3):
            for perm in itertools.permutations(range(1, B + 1)):
                pos, m = binding.layout(P, perm)
                opos, om = oracle.layout(P, np.array(perm))
                assert np.array_equal(pos.numpy(), opos)
                assert np.array_equal(m.numpy(), om)


def test_layout_matches_oracle_random(lib):
    rng = np.random.default_rng(0)
    for _ in range(200):
        B = int(rng.integers(1, 33))
        P = int(rng.integers(0, 300))
        tau = rng.permutation(B) + 1
        pos, m = binding.layout(P, tau.tolist())
        opos, om = oracle.layout(P, tau)
        assert np.array_equal(pos.numpy(), opos)
        assert np.array_equal(m.numpy(), om)
        pos2, none = binding.layout(P, tau.tolist(), with_mask=False)
        assert none is None and np.array_equal(pos2.numpy(), opos)


@pytest.mark.parametrize("tau,codes", [([1, 1, 2], (3,)), ([0, 1, 2], (3,)), ([1, 2, 4], (3,)),
                                       ([], (1, 2)), (list(range(1, 34)), (2,))])
def test_layout_errors(lib, tau, codes):
    with pytest.raises(binding.SimsdError) as e:
        binding.layout(4, tau)
    assert e.value.code in codes


def _desc(**kw):
    d = binding.VerifyDesc()
    base = dict(batch=2, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                num_pages=300, max_pages_per_seq=150, total_B=8, B_max=4,
                dtype=binding.SIMSD_BF16, rope_base=1e6, sm_scale=1.0)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


def test_verify_workspace_size_and_shape_errors(lib):
    n = lib.simsd_verify_workspace_size(ctypes.byref(_desc()))
    # at least the rotated queries: T * Hq * hd * 2 bytes
    assert n >= 16 * 32 * 128 * 2 and n % 256 == 0
    for bad in (dict(head_dim=96), dict(num_q_heads=30), dict(page_size=32),
                dict(B_max=33), dict(total_B=1), dict(total_B=9), dict(batch=0),
                dict(dtype=7), dict(num_pages=0)):
        d = _desc(**bad)
        assert lib.simsd_verify_workspace_size(ctypes.byref(d)) == 0, bad
        code = lib.simsd_verify_attn(ctypes.byref(d), None)
        assert code in (2, 4), (bad, code)
    # valid sizes but NULL pointers
    assert lib.simsd_verify_attn(ctypes.byref(_desc()), None) == 1
    assert lib.simsd_verify_attn(None, None) == 1


def test_verify_workspace_errors(lib):
    d = _desc()
    fake = 1 << 40     # never dereferenced: the call returns before launching
    for f in ("q", "k_cache", "v_cache", "block_table", "k_new", "v_new", "tau",
              "lens", "cu_B", "out"):
        setattr(d, f, fake)
    d.workspace = None
    assert lib.simsd_verify_attn(ctypes.byref(d), None) == 5
    d.workspace = fake + 8                      # misaligned
    d.workspace_bytes = 1 << 40
    assert lib.simsd_verify_attn(ctypes.byref(d), None) == 5
    d.workspace = fake
    d.workspace_bytes = lib.simsd_verify_workspace_size(ctypes.byref(d)) - 1
    assert lib.simsd_verify_attn(ctypes.byref(d), None) == 5
    # value arrays off a 16-byte boundary are refused before the workspace
    for f in ("q", "k_cache", "v_cache", "k_new", "v_new", "out"):
        setattr(d, f, fake + 8)
        assert lib.simsd_verify_attn(ctypes.byref(d), None) == 8, f
        setattr(d, f, fake)


def test_accept_errors(lib):
    d = binding.AcceptDesc()
    for k, v in dict(batch=4, vocab=1000, total_B=16, B_max=4, dtype=1).items():
        setattr(d, k, v)
    n = lib.simsd_accept_workspace_size(ctypes.byref(d))
    assert n > 0 and n % 256 == 0
    assert lib.simsd_accept(ctypes.byref(d), None) == 1
    fake = 1 << 40
    for f in ("target_logits", "draft_logits", "draft_tokens", "tau", "cu_B",
              "uniforms", "n_accept", "token", "pos"):
        setattr(d, f, fake)
    assert lib.simsd_accept(ctypes.byref(d), None) == 5
    for bad in (dict(B_max=0), dict(B_max=33), dict(total_B=17), dict(vocab=0),
                dict(dtype=3), dict(batch=0)):
        for k, v in bad.items():
            setattr(d, k, v)
        assert lib.simsd_accept_workspace_size(ctypes.byref(d)) == 0
        assert lib.simsd_accept(ctypes.byref(d), None) in (2, 4)
        for k, v in dict(batch=4, vocab=1000, total_B=16, B_max=4, dtype=1).items():
            setattr(d, k, v)


def test_append_errors(lib):
    d = binding.AppendDesc()
    assert lib.simsd_prompt_append(ctypes.byref(d), None) == 2
    assert lib.simsd_prompt_append(None, None) == 1
    fake = 1 << 40
    for k, v in dict(batch=1, num_kv_heads=2, head_dim=128, page_size=16, num_pages=4,
                     max_pages_per_seq=4, total_n=3, dtype=1, rope_base=1e4).items():
        setattr(d, k, v)
    for f in ("k", "v", "start", "cu_n", "k_cache", "v_cache", "block_table"):
        setattr(d, f, fake)
    d.k = fake + 4
    assert lib.simsd_prompt_append(ctypes.byref(d), None) == 8


def test_verify_row_bytes_limit(lib):
    # (Hq + 2 Hkv) * hd * 4 bytes above 192 KiB: one token's rows cannot be staged
    assert lib.simsd_verify_workspace_size(ctypes.byref(_desc(num_q_heads=376, num_kv_heads=8,
                                                              dtype=binding.SIMSD_F32))) == 0
    assert lib.simsd_verify_workspace_size(ctypes.byref(_desc(num_q_heads=376, num_kv_heads=8))) > 0


def test_accept_rule_and_temperature_checks(lib):
    """The rule and the temperature are checked before any launch; the greedy
    rule needs neither draft logits nor uniforms (so with those NULL the call
    gets as far as the workspace check)."""
    d = binding.AcceptDesc()
    for k, v in dict(batch=4, vocab=1000, total_B=16, B_max=4, dtype=1).items():
        setattr(d, k, v)
    fake = 1 << 40
    for f in ("target_logits", "draft_logits", "draft_tokens", "tau", "cu_B",
              "uniforms", "n_accept", "token", "pos"):
        setattr(d, f, fake)
    assert lib.simsd_accept_workspace_size(ctypes.byref(d)) > 0   # zero-filled: rule 0, T -> 1
    for rule, temp in ((3, 1.0), (-1, 1.0), (0, -0.5), (0, float("nan")), (0, float("inf")),
                       (1, -1.0), (2, -2.0)):
        d.rule, d.temperature = rule, temp
        assert lib.simsd_accept_workspace_size(ctypes.byref(d)) == 0, (rule, temp)
        assert lib.simsd_accept(ctypes.byref(d), None) == 2, (rule, temp)
        assert lib.simsd_accept_noalloc(ctypes.byref(d), None) == 2, (rule, temp)
    d.rule, d.temperature = binding.SIMSD_ACCEPT_GREEDY, 0.0
    d.draft_logits = None
    d.uniforms = None
    assert lib.simsd_accept(ctypes.byref(d), None) == 5          # reached the workspace check
    d.target_logits = None
    assert lib.simsd_accept(ctypes.byref(d), None) == 1
    d.target_logits = fake
    d.rule, d.temperature = binding.SIMSD_ACCEPT_SAMPLE, 0.7
    assert lib.simsd_accept(ctypes.byref(d), None) == 1          # sampling needs both
    d.rule = binding.SIMSD_ACCEPT_MATCH                          # matching needs the uniforms
    assert lib.simsd_accept(ctypes.byref(d), None) == 1
    d.uniforms = fake
    assert lib.simsd_accept(ctypes.byref(d), None) == 5          # but no draft logits


def test_descriptor_layouts_match_the_header(tmp_path):
    """The binding's ctypes descriptors have the header's field offsets and
    sizes (a C program compiled against include/simsd.h prints them)."""
    import shutil
    import subprocess
    from speculative_decoding_diffusion_gb300 import binding
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"simsd_verify_desc": binding.VerifyDesc, "simsd_accept_desc": binding.AcceptDesc,
               "simsd_append_desc": binding.AppendDesc}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "simsd.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append('  printf("%s sizeof %%zu\\n", sizeof(%s));' % (cname, cname))
        for f, _ in py._fields_:
            lines.append('  printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(ROOT, "include")
    subprocess.run([cc, "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        a, b, c = line.split()
        got[(a, b)] = int(c)
    for cname, py in structs.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


@pytest.mark.parametrize("dtype,vocab,batch,total_B", [(binding.SIMSD_BF16, 151936, 16, 64),
                                                       (binding.SIMSD_F32, 777, 3, 7),
                                                       (binding.SIMSD_BF16, 1 << 21, 5, 160),
                                                       (binding.SIMSD_F32, 100003, 256, 1536)])
def test_accept_workspace_size_is_the_header_formula(lib, dtype, vocab, batch, total_B):
    """simsd_accept_workspace_size equals the sum the header states, term by
    term rounded up to 256 bytes, for every rule; and simsd_draft_workspace_size
    equals its own."""
    def r(x):
        return -(-x // 256) * 256
    E = 16384 if dtype == binding.SIMSD_BF16 else 8192
    C = -(-vocab // E)
    d = binding.AcceptDesc()
    for k, v in dict(batch=batch, vocab=vocab, total_B=total_B, B_max=32, dtype=dtype).items():
        setattr(d, k, v)
    want = {binding.SIMSD_ACCEPT_SAMPLE: 256 + r(2 * total_B * C * 64) + r(2 * total_B * 4) +
            r(batch * 4) + r(batch * C * 256),
            binding.SIMSD_ACCEPT_GREEDY: 256 + r(total_B * C * 128) + r(total_B * 4),
            binding.SIMSD_ACCEPT_MATCH: 256 + r(total_B * C * 128) + r(total_B * 4)}
    for rule, n in want.items():
        d.rule = rule
        assert lib.simsd_accept_workspace_size(ctypes.byref(d)) == n, rule
    dd = binding.DraftDesc()
    for k, v in dict(batch=batch, vocab=vocab, total_B=total_B, B_max=32, dtype=dtype).items():
        setattr(dd, k, v)
    assert lib.simsd_draft_workspace_size(ctypes.byref(dd)) == 256 + r(total_B * C * 128)


def _verify_ws_bytes(T, Hq, hd, n_splits):
    # the workspace carve-up of simsd_verify_attn (bf16): status word, one
    # int4 per new token, then, when the plan splits, the fp32 partial
    # outputs and the (max, sum) pairs of every split; each region 256-byte
    # aligned
    up = lambda n: (n + 255) // 256 * 256
    total = up(4) + up(T * 16)
    if n_splits > 1:
        total += up(n_splits * T * Hq * hd * 4) + up(n_splits * T * Hq * 8)
    return total


@pytest.mark.parametrize("batch,P,B,splits", [
    (16, 1024, 4, 1),      # 128 units of 9 blocks: one wave, no split
    (64, 4096, 8, 2),      # 512 units: three full waves, the last 56 units in 2 splits
    (8, 32768, 16, 2),     # 64 units of 257 blocks: every unit in 2 (one wave of 128 CTAs)
    (1, 32768, 4, 19),     # 8 units: 19 splits of 14 blocks fill one wave of 152 CTAs
])
def test_verify_split_plan(lib, batch, P, B, splits):
    """The key-split plan the host makes for a 152-SM device (the library's
    count when no device is visible), read back from the workspace size."""
    if torch.cuda.is_available():
        pytest.skip("the plan follows the visible device's SM count")
    max_pages = (P + 2 * B + 15) // 16
    d = _desc(batch=batch, num_pages=batch * max_pages, max_pages_per_seq=max_pages,
              total_B=batch * B, B_max=B)
    got = lib.simsd_verify_workspace_size(ctypes.byref(d))
    T = 2 * batch * B
    assert got == _verify_ws_bytes(T, 32, 128, splits), \
        [(s, _verify_ws_bytes(T, 32, 128, s)) for s in (1, 2, 3, splits)] + [got]


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """With no built library the binding raises on the first call: there is
    no other path to the results."""
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libsimsd.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()
    with pytest.raises(RuntimeError, match="not built"):
        binding.layout(4, [2, 1, 3])


@pytest.mark.parametrize("dtype,batch,P,B,merges", [
    (binding.SIMSD_BF16, 16, 1024, 4, 0), (binding.SIMSD_BF16, 64, 4096, 8, 1),
    (binding.SIMSD_BF16, 8, 32768, 16, 1), (binding.SIMSD_BF16, 1, 32768, 4, 1),
    (binding.SIMSD_F32, 1, 64, 4, 0), (binding.SIMSD_F32, 2, 4096, 4, 1)])
def test_bench_counts_the_merge_from_the_plan(lib, dtype, batch, P, B, merges):
    """bench.py counts the split merge's launch from the workspace size the
    library plans (the merge runs iff some unit's keys are split)."""
    import types
    import bench
    max_pages = (P + 2 * B + 15) // 16
    d = _desc(batch=batch, num_pages=batch * max_pages, max_pages_per_seq=max_pages,
              total_B=batch * B, B_max=B, dtype=dtype)
    ws = lib.simsd_verify_workspace_size(ctypes.byref(d))
    w = types.SimpleNamespace(cu_B=np.arange(batch + 1) * B,
                              spec=types.SimpleNamespace(dtype="bf16" if dtype == binding.SIMSD_BF16
                                                         else "f32", Hq=32, hd=128))
    assert bench.merge_launches(w, ws) == merges
