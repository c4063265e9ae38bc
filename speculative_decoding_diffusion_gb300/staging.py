"""Device staging of a verification workload (memory movement only).

Takes host arrays shaped like the C ABI's inputs -- bf16 values as uint16
bit patterns or fp32 -- and lays them out in device memory: the paged KV
cache [num_pages][Hkv][16][hd] filled through the block table, the new
tokens, the logits, the index arrays, the outputs and the workspaces.  No
arithmetic of the method happens here; the prompt keys of a workload whose
prompt keys are raw are rotated by the library (simsd_prompt_append).
"""
import numpy as np
import torch

from . import binding

PAGE = 16


def to_device(a, device):
    """uint16 arrays are bf16 bit patterns; everything else keeps its dtype."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceWorkload:
    """Everything one verification step needs, resident on `device`.

    `w` provides: lens, Bs, cu_B, tau, num_pages, max_pages, block_table,
    q, k_prompt, v_prompt, k_new, v_new, (target, draft, draft_tokens,
    uniforms), prompt_offsets, spec (Hq, Hkv, hd, rope_base, sm_scale,
    raw_prompt_keys)."""

    def __init__(self, w, device="cuda", with_accept=True, extra_pages=0,
                 with_verify=True):
        self.w = w
        spec = w.spec
        dev = torch.device(device)
        self.device = dev
        self.rope_base = spec.rope_base
        self.sm_scale = spec.sm_scale
        self.total_B = int(w.cu_B[-1])
        self.B_max = int(w.Bs.max())
        self.lens = torch.from_numpy(w.lens.astype(np.int32)).to(dev)
        self.cu_B = torch.from_numpy(w.cu_B.astype(np.int32)).to(dev)
        self.tau = torch.from_numpy(w.tau.astype(np.int32)).to(dev)
        self.block_table = torch.from_numpy(w.block_table.astype(np.int32)).to(dev)
        if with_verify:
            self.q = to_device(w.q, dev)
            self.k_new = to_device(w.k_new, dev)
            self.v_new = to_device(w.v_new, dev)
            dt = self.q.dtype
            n_pages = w.num_pages + extra_pages
            self.k_cache = torch.zeros((n_pages, spec.Hkv, PAGE, spec.hd), dtype=dt, device=dev)
            self.v_cache = torch.zeros_like(self.k_cache)
            self._fill_prompt(w, spec)
            self.out = torch.empty_like(self.q)
            nbytes = binding.verify_workspace_size(*self._verify_args())
            self.verify_ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        if with_accept and w.target is not None:
            self.target = to_device(w.target, dev)
            self.draft = to_device(w.draft, dev)
            self.draft_tokens = torch.from_numpy(w.draft_tokens.astype(np.int32)).to(dev)
            self.uniforms = torch.from_numpy(np.ascontiguousarray(w.uniforms, np.float32)).to(dev)
            batch = len(w.lens)
            self.n_accept = torch.empty(batch, dtype=torch.int32, device=dev)
            self.token = torch.empty(batch, dtype=torch.int32, device=dev)
            self.pos = torch.empty(batch, dtype=torch.int32, device=dev)
            nbytes = binding.accept_workspace_size(*self._accept_args())
            self.accept_ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    # ------------------------------------------------------------ prompt
    def _fill_prompt(self, w, spec):
        P = w.lens.astype(np.int64)
        if P.sum() == 0:
            return
        kp = to_device(w.k_prompt, self.device)
        vp = to_device(w.v_prompt, self.device)
        if spec.raw_prompt_keys:
            start = torch.zeros(len(P), dtype=torch.int32, device=self.device)
            cu_n = torch.from_numpy(np.concatenate([[0], np.cumsum(P)]).astype(np.int32)).to(self.device)
            binding.prompt_append(kp, vp, start, cu_n, self.k_cache, self.v_cache,
                                  self.block_table, self.rope_base)
            return
        seq = np.repeat(np.arange(len(P)), P)
        posn = np.arange(int(P.sum())) - np.repeat(w.prompt_offsets[:-1], P)
        page = w.block_table[seq, posn // PAGE].astype(np.int64)
        slot = (posn % PAGE).astype(np.int64)
        pi = torch.from_numpy(page).to(self.device)
        si = torch.from_numpy(slot).to(self.device)
        self.k_cache.permute(0, 2, 1, 3)[pi, si] = kp
        self.v_cache.permute(0, 2, 1, 3)[pi, si] = vp

    # ------------------------------------------------------------ calls
    def _verify_args(self):
        return (self.q, self.k_cache, self.v_cache, self.block_table, self.k_new,
                self.v_new, self.tau, self.lens, self.cu_B, self.out, self.total_B,
                self.B_max, self.rope_base, self.sm_scale)

    def verify(self, stream=None, events=None):
        (q, kc, vc, bt, kn, vn, tau, lens, cu, out, tb, bm, rb, sc) = self._verify_args()
        binding.verify_attn(q, kc, vc, bt, kn, vn, tau, lens, cu, out, self.verify_ws,
                            tb, bm, rb, sc, stream=stream, events=events)

    def _accept_args(self):
        return (self.target, self.draft, self.draft_tokens, self.tau, self.cu_B,
                self.uniforms, self.n_accept, self.token, self.pos, self.total_B,
                self.B_max)

    def accept(self, stream=None, events=None, rule=binding.SIMSD_ACCEPT_SAMPLE,
               temperature=1.0):
        (t, d, x, tau, cu, u, n, tok, pos, tb, bm) = self._accept_args()
        if rule != binding.SIMSD_ACCEPT_SAMPLE:      # greedy and matching read no draft logits
            d = None
        if rule == binding.SIMSD_ACCEPT_GREEDY:      # greedy reads no uniforms either
            u = None
        binding.accept(t, d, x, tau, cu, u, n, tok, pos, self.accept_ws, tb, bm,
                       stream=stream, events=events, rule=rule, temperature=temperature)
