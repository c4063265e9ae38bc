"""ctypes binding of libsimsd.so (C ABI: include/simsd.h).

Argument marshalling only: every step of the verification path runs in the
library's CUDA kernels.  Tensors are torch tensors (device memory and the
current stream come from torch); the binding passes their pointers and
sizes through the descriptors of the C ABI.  There is no fallback: if the
library is missing or cannot be loaded, every call raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsimsd.so")

SIMSD_F32, SIMSD_BF16 = 0, 1
SIMSD_ACCEPT_SAMPLE, SIMSD_ACCEPT_GREEDY, SIMSD_ACCEPT_MATCH = 0, 1, 2
STATUS = {0: "SIMSD_OK", 1: "SIMSD_ERR_NULL", 2: "SIMSD_ERR_SHAPE",
          3: "SIMSD_ERR_TAU", 4: "SIMSD_ERR_DTYPE", 5: "SIMSD_ERR_WORKSPACE",
          6: "SIMSD_ERR_CUDA", 7: "SIMSD_ERR_TIMEOUT", 8: "SIMSD_ERR_ALIGN"}

_i32, _f32, _vp, _sz = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class VerifyDesc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("num_q_heads", _i32), ("num_kv_heads", _i32),
                ("head_dim", _i32), ("page_size", _i32), ("num_pages", _i32),
                ("max_pages_per_seq", _i32), ("total_B", _i32), ("B_max", _i32),
                ("dtype", ctypes.c_int), ("rope_base", _f32), ("sm_scale", _f32),
                ("q", _vp), ("k_cache", _vp), ("v_cache", _vp), ("block_table", _vp),
                ("k_new", _vp), ("v_new", _vp), ("tau", _vp), ("lens", _vp),
                ("cu_B", _vp), ("out", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("wait_polls", _i32), ("node_size", _i32)]


class AppendDesc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("page_size", _i32), ("num_pages", _i32), ("max_pages_per_seq", _i32),
                ("total_n", _i32), ("dtype", ctypes.c_int), ("rope_base", _f32),
                ("k", _vp), ("v", _vp), ("start", _vp), ("cu_n", _vp),
                ("k_cache", _vp), ("v_cache", _vp), ("block_table", _vp)]


class AcceptDesc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("vocab", _i32), ("total_B", _i32), ("B_max", _i32),
                ("dtype", ctypes.c_int), ("target_logits", _vp), ("draft_logits", _vp),
                ("draft_tokens", _vp), ("tau", _vp), ("cu_B", _vp), ("uniforms", _vp),
                ("n_accept", _vp), ("token", _vp), ("pos", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("rule", ctypes.c_int), ("temperature", ctypes.c_float),
                ("wait_polls", _i32), ("decided", _vp)]


class DraftDesc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("vocab", _i32), ("total_B", _i32), ("B_max", _i32),
                ("dtype", ctypes.c_int), ("temperature", _f32), ("draft_logits", _vp),
                ("cu_B", _vp), ("uniforms", _vp), ("decided", _vp), ("tau_prev", _vp),
                ("tokens", _vp), ("tau", _vp), ("confidence", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz)]


class CommitDesc(ctypes.Structure):
    _fields_ = [("batch", _i32), ("total_B", _i32), ("B_max", _i32), ("cu_B", _vp),
                ("tau", _vp), ("n_accept", _vp), ("token", _vp), ("pos", _vp),
                ("tokens", _vp), ("decided", _vp), ("lens", _vp), ("done", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz)]


class SimsdError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s failed: %s (%d)" % (what, STATUS.get(code, "?"), code))
        self.code = code


_LIB = None


def lib():
    """The loaded library; raises if it was not built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsimsd.so is not built (run __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        L.simsd_status_string.restype = ctypes.c_char_p
        L.simsd_status_string.argtypes = [ctypes.c_int]
        L.simsd_version.restype = ctypes.c_int
        L.simsd_layout.restype = ctypes.c_int
        L.simsd_layout.argtypes = [_i32, _i32, _vp, _vp, _vp]
        L.simsd_verify_workspace_size.restype = _sz
        L.simsd_verify_workspace_size.argtypes = [ctypes.POINTER(VerifyDesc)]
        L.simsd_verify_attn.restype = ctypes.c_int
        L.simsd_verify_attn.argtypes = [ctypes.POINTER(VerifyDesc), _vp]
        L.simsd_prompt_append.restype = ctypes.c_int
        L.simsd_prompt_append.argtypes = [ctypes.POINTER(AppendDesc), _vp]
        L.simsd_accept_workspace_size.restype = _sz
        L.simsd_accept_workspace_size.argtypes = [ctypes.POINTER(AcceptDesc)]
        L.simsd_accept.restype = ctypes.c_int
        L.simsd_accept.argtypes = [ctypes.POINTER(AcceptDesc), _vp]
        L.simsd_verify_attn_timed.restype = ctypes.c_int
        L.simsd_verify_attn_timed.argtypes = [ctypes.POINTER(VerifyDesc), _vp, ctypes.POINTER(_vp)]
        L.simsd_accept_timed.restype = ctypes.c_int
        L.simsd_accept_timed.argtypes = [ctypes.POINTER(AcceptDesc), _vp, ctypes.POINTER(_vp)]
        L.simsd_accept_noalloc.restype = ctypes.c_int
        L.simsd_accept_noalloc.argtypes = [ctypes.POINTER(AcceptDesc), _vp]
        L.simsd_draft_workspace_size.restype = _sz
        L.simsd_draft_workspace_size.argtypes = [ctypes.POINTER(DraftDesc)]
        L.simsd_draft_step.restype = ctypes.c_int
        L.simsd_draft_step.argtypes = [ctypes.POINTER(DraftDesc), _vp]
        L.simsd_commit_workspace_size.restype = _sz
        L.simsd_commit_workspace_size.argtypes = [ctypes.POINTER(CommitDesc)]
        L.simsd_commit.restype = ctypes.c_int
        L.simsd_commit.argtypes = [ctypes.POINTER(CommitDesc), _vp]
        L.simsd_read_status.restype = ctypes.c_int
        L.simsd_read_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
        _LIB = L
    return _LIB


def _check(code, what):
    if code != 0:
        raise SimsdError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SIMSD_BF16
    if t.dtype == torch.float32:
        return SIMSD_F32
    raise TypeError("unsupported dtype %s" % t.dtype)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def status_string(code):
    return lib().simsd_status_string(int(code)).decode()


def layout(prompt_len, tau, with_mask=True):
    """Host call.  tau: sequence of ints.  Returns (positions, mask) as
    int32 / uint8 torch CPU tensors (mask None when with_mask is False)."""
    B = len(tau)
    t = torch.tensor(list(tau), dtype=torch.int32)
    positions = torch.empty(prompt_len + 2 * B, dtype=torch.int32)
    mask = torch.empty((2 * B, prompt_len + 2 * B), dtype=torch.uint8) if with_mask else None
    _check(lib().simsd_layout(prompt_len, B, _ptr(t), _ptr(positions), _ptr(mask)),
           "simsd_layout")
    return positions, mask


def _verify_desc(q, k_cache, v_cache, block_table, k_new, v_new, tau, lens, cu_B,
                 out, total_B, B_max, rope_base, sm_scale, workspace=None, wait_polls=0,
                 node_size=0):
    d = VerifyDesc()
    d.wait_polls = int(wait_polls)
    d.node_size = int(node_size)
    d.batch = lens.shape[0]
    d.num_q_heads = q.shape[1]
    d.num_kv_heads = k_new.shape[1]
    d.head_dim = q.shape[2]
    d.page_size = k_cache.shape[2]
    d.num_pages = k_cache.shape[0]
    d.max_pages_per_seq = block_table.shape[1]
    d.total_B = int(total_B)
    d.B_max = int(B_max)
    d.dtype = _dtype_code(q)
    d.rope_base = float(rope_base)
    d.sm_scale = float(sm_scale)
    d.q, d.k_cache, d.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
    d.block_table, d.k_new, d.v_new = _ptr(block_table), _ptr(k_new), _ptr(v_new)
    d.tau, d.lens, d.cu_B, d.out = _ptr(tau), _ptr(lens), _ptr(cu_B), _ptr(out)
    if workspace is not None:
        d.workspace = _ptr(workspace)
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    return d


def verify_workspace_size(q, k_cache, v_cache, block_table, k_new, v_new, tau,
                          lens, cu_B, out, total_B, B_max, rope_base, sm_scale, node_size=0):
    d = _verify_desc(q, k_cache, v_cache, block_table, k_new, v_new, tau, lens,
                     cu_B, out, total_B, B_max, rope_base, sm_scale, node_size=node_size)
    n = lib().simsd_verify_workspace_size(ctypes.byref(d))
    if n == 0:
        raise SimsdError(2, "simsd_verify_workspace_size")
    return int(n)


def _events(evs, n):
    arr = (_vp * n)()
    for i, e in enumerate(evs):
        arr[i] = None if e is None else e.cuda_event
    return arr


def verify_attn(q, k_cache, v_cache, block_table, k_new, v_new, tau, lens, cu_B,
                out, workspace, total_B, B_max, rope_base, sm_scale, stream=None,
                events=None, wait_polls=0, node_size=0):
    """simsd_verify_attn on the current (or given) torch stream.  events:
    optional 4 recorded torch.cuda.Event objects (see simsd_verify_attn_timed).
    wait_polls: the descriptor field (0: default limit; < 0: give up at once).
    node_size > 0: the draft-graph layout (tau may be None)."""
    d = _verify_desc(q, k_cache, v_cache, block_table, k_new, v_new, tau, lens,
                     cu_B, out, total_B, B_max, rope_base, sm_scale, workspace, wait_polls,
                     node_size)
    if events is None:
        _check(lib().simsd_verify_attn(ctypes.byref(d), _stream(stream)), "simsd_verify_attn")
    else:
        _check(lib().simsd_verify_attn_timed(ctypes.byref(d), _stream(stream), _events(events, 4)),
               "simsd_verify_attn_timed")


def prompt_append(k, v, start, cu_n, k_cache, v_cache, block_table, rope_base,
                  stream=None):
    d = AppendDesc()
    d.batch = start.shape[0]
    d.num_kv_heads = k.shape[1]
    d.head_dim = k.shape[2]
    d.page_size = k_cache.shape[2]
    d.num_pages = k_cache.shape[0]
    d.max_pages_per_seq = block_table.shape[1]
    d.total_n = k.shape[0]
    d.dtype = _dtype_code(k)
    d.rope_base = float(rope_base)
    d.k, d.v, d.start, d.cu_n = _ptr(k), _ptr(v), _ptr(start), _ptr(cu_n)
    d.k_cache, d.v_cache, d.block_table = _ptr(k_cache), _ptr(v_cache), _ptr(block_table)
    _check(lib().simsd_prompt_append(ctypes.byref(d), _stream(stream)), "simsd_prompt_append")


def _accept_desc(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token,
                 pos, total_B, B_max, workspace=None, rule=SIMSD_ACCEPT_SAMPLE, temperature=1.0,
                 wait_polls=0, decided=None):
    d = AcceptDesc()
    d.wait_polls = int(wait_polls)
    d.decided = _ptr(decided)
    d.rule = int(rule)
    d.temperature = float(temperature)
    d.batch = cu_B.shape[0] - 1
    d.vocab = target.shape[1]
    d.total_B = int(total_B)
    d.B_max = int(B_max)
    d.dtype = _dtype_code(target)
    d.target_logits = _ptr(target)
    d.draft_logits = None if draft is None else _ptr(draft)
    d.draft_tokens, d.tau, d.cu_B = _ptr(draft_tokens), _ptr(tau), _ptr(cu_B)
    d.uniforms = None if uniforms is None else _ptr(uniforms)
    d.n_accept, d.token, d.pos = _ptr(n_accept), _ptr(token), _ptr(pos)
    if workspace is not None:
        d.workspace = _ptr(workspace)
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    return d


def accept_workspace_size(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept,
                          token, pos, total_B, B_max, rule=SIMSD_ACCEPT_SAMPLE):
    """simsd_accept_workspace_size: the two-kernel path's workspace for `rule`
    (the sampling rule's is the largest of the three)."""
    d = _accept_desc(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token,
                     pos, total_B, B_max, rule=rule)
    n = lib().simsd_accept_workspace_size(ctypes.byref(d))
    if n == 0:
        raise SimsdError(2, "simsd_accept_workspace_size")
    return int(n)


def accept(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token, pos,
           workspace, total_B, B_max, stream=None, events=None, rule=SIMSD_ACCEPT_SAMPLE,
           temperature=1.0, wait_polls=0, decided=None):
    """simsd_accept; events: optional 3 recorded torch.cuda.Event objects;
    rule SIMSD_ACCEPT_GREEDY takes draft = uniforms = None; wait_polls as for
    verify_attn; decided: int32 [batch] steps decided in earlier passes."""
    d = _accept_desc(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token,
                     pos, total_B, B_max, workspace, rule, temperature, wait_polls, decided)
    if events is None:
        _check(lib().simsd_accept(ctypes.byref(d), _stream(stream)), "simsd_accept")
    else:
        _check(lib().simsd_accept_timed(ctypes.byref(d), _stream(stream), _events(events, 3)),
               "simsd_accept_timed")


# the static scratch of simsd_accept_noalloc (include/simsd.h)
SIMSD_ACCEPT_NOALLOC_SCRATCH_BYTES = 4096


def accept_noalloc(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token,
                   pos, total_B, B_max, stream=None, rule=SIMSD_ACCEPT_SAMPLE, temperature=1.0):
    """simsd_accept_noalloc: acceptance with the library's static scratch, for
    callers that may not allocate device memory (no workspace argument)."""
    d = _accept_desc(target, draft, draft_tokens, tau, cu_B, uniforms, n_accept, token,
                     pos, total_B, B_max, None, rule, temperature)
    _check(lib().simsd_accept_noalloc(ctypes.byref(d), _stream(stream)),
           "simsd_accept_noalloc")


def _status_ws(workspace):
    return _ptr(workspace), (0 if workspace is None else workspace.numel() * workspace.element_size())


def draft_workspace_size(draft, cu_B, total_B, B_max, temperature=1.0):
    """simsd_draft_workspace_size: the chunked path's workspace (a workspace
    of only the status word runs the single cluster kernel)."""
    d = DraftDesc()
    d.batch = cu_B.shape[0] - 1
    d.vocab = draft.shape[1]
    d.total_B, d.B_max = int(total_B), int(B_max)
    d.dtype = _dtype_code(draft)
    d.temperature = float(temperature)
    n = lib().simsd_draft_workspace_size(ctypes.byref(d))
    if n == 0:
        raise SimsdError(2, "simsd_draft_workspace_size")
    return int(n)


def draft_step(draft, cu_B, uniforms, tokens, tau, workspace, total_B, B_max, decided=None,
               tau_prev=None, confidence=None, temperature=1.0, stream=None):
    """simsd_draft_step: tokens (in/out) and tau (out) of every sequence's
    open slots; uniforms float32 [batch, B_max]."""
    d = DraftDesc()
    d.batch = cu_B.shape[0] - 1
    d.vocab = draft.shape[1]
    d.total_B, d.B_max = int(total_B), int(B_max)
    d.dtype = _dtype_code(draft)
    d.temperature = float(temperature)
    d.draft_logits, d.cu_B, d.uniforms = _ptr(draft), _ptr(cu_B), _ptr(uniforms)
    d.decided, d.tau_prev = _ptr(decided), _ptr(tau_prev)
    d.tokens, d.tau, d.confidence = _ptr(tokens), _ptr(tau), _ptr(confidence)
    d.workspace, d.workspace_bytes = _status_ws(workspace)
    _check(lib().simsd_draft_step(ctypes.byref(d), _stream(stream)), "simsd_draft_step")


def commit(cu_B, tau, n_accept, token, pos, tokens, decided, lens, done, workspace,
           total_B, B_max, stream=None):
    """simsd_commit: applies a pass's walk to the block state (tokens,
    decided, lens in/out; done out)."""
    d = CommitDesc()
    d.batch = cu_B.shape[0] - 1
    d.total_B, d.B_max = int(total_B), int(B_max)
    d.cu_B, d.tau, d.n_accept, d.token, d.pos = (_ptr(cu_B), _ptr(tau), _ptr(n_accept),
                                                  _ptr(token), _ptr(pos))
    d.tokens, d.decided, d.lens, d.done = _ptr(tokens), _ptr(decided), _ptr(lens), _ptr(done)
    d.workspace, d.workspace_bytes = _status_ws(workspace)
    _check(lib().simsd_commit(ctypes.byref(d), _stream(stream)), "simsd_commit")


def read_status(workspace, stream=None):
    """Synchronises the stream; returns the workspace status word."""
    w = ctypes.c_uint32(0)
    code = lib().simsd_read_status(_ptr(workspace), _stream(stream), ctypes.byref(w))
    if code not in (0, 7):
        raise SimsdError(code, "simsd_read_status")
    return int(w.value)
