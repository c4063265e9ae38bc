"""Benchmark of the SimSD verification step on GB300.

One step = the whole hot path over one batch: simsd_verify_attn (K1 RoPE-copy
+ paged append, K2 masked attention, K3 merge of split units) and
simsd_accept (K4a: a chunk pass over every SM computes each 32 KB chunk's
normaliser partials; K4b: one thread-block cluster per sequence merges
them, walks the steps along tau and draws the residual token at a
rejection).  Default workload: the ragged serving mix (256
sequences, prompt KV lengths uniform in [256, 8192], B in {4, 8}, 32/8
heads, head dim 128, vocabulary 151,936, bf16, shuffled 16-token pages),
the largest of the SDAR-8B-shaped workloads; --workload 1 is the
16 x 1024, B = 4 step.  Seeded synthetic data.

Prints ONE JSON line.  `value`: verified candidate tokens/s (sum of B over
the batch / step time) with inputs resident in HBM: the step's library calls
are captured once into a CUDA graph (the library allocates nothing and never
synchronises, so the calls capture as they are) and replayed; each replay is
timed with CUDA events on the launching stream, with L2 flushed (a 512 MB
write) before it.  Per-kernel times come from a second graph of the same
calls with the library's event marks as event-record nodes (those nodes sit
between kernels, so that graph forgoes the overlap of consecutive kernels
that the timed graph keeps).  `e2e`: the same metric through
the C ABI called directly from Python each step with host buffers (pinned
host -> device copies of the step's inputs and device -> host copies of its
results inside the timed region, the logits' copies on a second stream
overlapping the attention; host launch cost included); `e2e_graph`
captures those copies and calls in a graph as well.  `roofline`: the
attention kernel K2 (the dominant one), algorithmic bytes per launch over
its mean event-timed duration.
`next_rows`: the blockwise loop's draft-side step and commit and the
greedy and sample-matching acceptance rules on the same workload, each
replayed alone (event-timed, L2 flushed), outside the step's timed region.
`cpu_baseline`: the fp64 oracle on a bounded sample of the same workload
(its first sequences, as many as take about a second per pass), timed on
this host's cores.

--accept greedy / match times the other acceptance rules (the greedy rule,
sample matching), --temperature T sampling at temperature T; the default is
rejection sampling at T = 1.

--impl reference runs the oracle as the reference arm.  Multi-GPU (torchrun):
each rank runs its own replica batch (sequences are independent; no
collective on the data path), rank 0 prints the aggregate.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verified candidate tokens/s (attn+accept)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", type=int, default=4,
                    help="synthetic configuration index (4 = 256-sequence ragged mix, "
                         "1 = 16 x 1024 SDAR-8B verify step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--accept", default="sample", choices=["sample", "greedy", "match"],
                    help="acceptance rule: rejection sampling (default), greedy, or "
                         "sample matching")
    ap.add_argument("--temperature", type=float, default=1.0,
                    help="sampling temperature (rejection sampling only)")
    ap.add_argument("--accept-path", default="auto", choices=["auto", "single"],
                    help="acceptance (rejection sampling): the full workspace (auto: the "
                         "chunk pass and the cluster kernel), or only the status word "
                         "(single: the cluster kernel streaming the rows itself)")
    return ap.parse_args()


def rule_code(args):
    return {"sample": 0, "greedy": 1, "match": 2}[args.accept]


# ---------------------------------------------------------------- the next rows
def time_next_rows(w, dw, flush, reps, peak):
    """The loop's other steps and the acceptance variants on the same
    workload, each captured alone in a CUDA graph and replayed with L2
    flushed before each replay (event-timed): the draft-side step over every
    slot's draft row, the commit, the greedy rule and sample matching.
    Algorithmic bytes: the draft rows once (draft step), the target rows
    once (greedy, matching)."""
    import torch
    from speculative_decoding_diffusion_gb300 import binding
    dev = dw.target.device
    batch, B_max, total_B = len(w.lens), int(w.Bs.max()), int(w.cu_B[-1])
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    u_draft = torch.rand(batch, B_max, generator=g, device=dev, dtype=torch.float32)
    tokens = torch.zeros(total_B, dtype=torch.int32, device=dev)
    tau_out = torch.zeros(total_B, dtype=torch.int32, device=dev)
    ws = torch.zeros(binding.draft_workspace_size(dw.draft, dw.cu_B, total_B, B_max),
                     dtype=torch.uint8, device=dev)
    dw.accept()                               # the walk the commit applies
    c_tokens = dw.draft_tokens.clone()
    c_decided = torch.zeros(batch, dtype=torch.int32, device=dev)
    c_lens = dw.lens.clone()
    c_done = torch.zeros(batch, dtype=torch.int32, device=dev)
    cws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    calls = {
        "draft_step": lambda: binding.draft_step(dw.draft, dw.cu_B, u_draft, tokens, tau_out, ws,
                                                 total_B, B_max),
        "commit": lambda: binding.commit(dw.cu_B, dw.tau, dw.n_accept, dw.token, dw.pos, c_tokens,
                                         c_decided, c_lens, c_done, cws, total_B, B_max),
        "greedy": lambda: dw.accept(rule=binding.SIMSD_ACCEPT_GREEDY),
        "match": lambda: dw.accept(rule=binding.SIMSD_ACCEPT_MATCH),
    }
    es = 2 if w.spec.dtype == "bf16" else 4
    row_bytes = total_B * w.spec.vocab * es
    out = {}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, call in calls.items():
        call()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            call()
        ms = []
        for _ in range(reps):
            flush.zero_()
            t0.record()
            gr.replay()
            t1.record()
            torch.cuda.synchronize()
            ms.append(t0.elapsed_time(t1))
        us = float(np.mean(ms)) * 1e3
        rec = {"us": round(us, 2)}
        if name != "commit":
            gbs = row_bytes / (us / 1e6) / 1e9
            rec.update({"GBps": round(gbs, 1), "frac": round(gbs / peak, 3)})
        out[name] = rec
    st = binding.read_status(ws) | binding.read_status(cws)
    out["status_word"] = st
    return out


# ---------------------------------------------------------------- algorithmic bytes
def attn_bytes(w):
    """K+V of every prompt key, the 2B new keys/values read once and written
    once, q read once and the output written once."""
    s = w.spec
    es = 2 if s.dtype == "bf16" else 4
    T = 2 * int(w.cu_B[-1])
    kv_prompt = int(w.lens.sum()) * 2 * s.Hkv * s.hd * es
    kv_new = T * 2 * s.Hkv * s.hd * es * 2
    q_out = T * s.Hq * s.hd * es * 2
    return kv_prompt + kv_new + q_out


def k2_bytes(w):
    """What K2 alone must move: every key/value of the cache range (prompt and
    new) once, the rotated q once, the output once."""
    s = w.spec
    es = 2 if s.dtype == "bf16" else 4
    T = 2 * int(w.cu_B[-1])
    keys = int(w.lens.sum()) + T
    return keys * 2 * s.Hkv * s.hd * es + T * s.Hq * s.hd * es * 2


def accept_bytes(w, target_only=False):
    """Logits read once per slot: both rows, or the target row alone (greedy,
    sample matching)."""
    es = 2 if w.spec.dtype == "bf16" else 4
    return int(w.cu_B[-1]) * (1 if target_only else 2) * w.spec.vocab * es


# ---------------------------------------------------------------- peaks / clocks
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ncu traffic record
def traffic_record_path(spec):
    return os.path.join(ROOT, "profiles", "k2_traffic_%s.json" % spec.slug)


def recorded_traffic(spec):
    """DRAM bytes per K2 launch from the committed ncu summary of this
    workload, valid only while the kernel source is unchanged (hash recorded
    with the counters)."""
    src = os.path.join(ROOT, "speculative_decoding_diffusion_gb300", "csrc", "attn_tc.cu")
    rec = traffic_record_path(spec)
    if not os.path.exists(rec):
        return None
    try:
        d = json.load(open(rec))
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if d.get("source_sha256") == h and d.get("workload") == spec.name:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------- CPU oracle
# sequences of the bounded CPU sample: about a second of oracle work per pass
CPU_SAMPLE_SEQS = {0: 1, 1: 16, 2: 16, 3: 2, 4: 32}


def cpu_sample(w, index):
    """The first sequences of the workload (all of the small ones)."""
    import synth
    n = CPU_SAMPLE_SEQS.get(index, 16)
    return synth.head(w, n) if n < len(w.lens) else w


def sample_text(sub, w, reps, el):
    return ("the first %d of %d sequences of %s (%d candidate tokens, prompt KV %d), "
            "%d pass(es) in %.1f s" % (len(sub.lens), len(w.lens), w.spec.name,
                                       int(sub.cu_B[-1]), int(sub.lens.sum()), reps, el))


def oracle_step_sample(w, seconds, threads, rule="sample", temperature=1.0):
    """Time the oracle (attention + acceptance) over whole batches of the
    workload w until `seconds` have passed; returns (tokens/s, seconds, passes)."""
    import oracle
    import synth
    q = synth.to_f64(w.q)
    kp, vp = synth.to_f64(w.k_prompt), synth.to_f64(w.v_prompt)
    if w.spec.raw_prompt_keys:   # the oracle takes rotated prompt keys
        off = w.prompt_offsets
        kp = np.concatenate([oracle.rope(kp[off[b]:off[b + 1]], np.arange(int(w.lens[b])),
                                         w.spec.rope_base) for b in range(len(w.lens))])
    kn, vn = synth.to_f64(w.k_new), synth.to_f64(w.v_new)
    tl, dl = synth.to_f64(w.target), synth.to_f64(w.draft)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_attn(w.lens, w.cu_B, q, kp, vp, kn, vn, w.tau, w.spec.rope_base,
                           w.spec.sm_scale, n_threads=threads)
        if rule == "greedy":
            oracle.accept_greedy(w.cu_B, tl, w.draft_tokens, w.tau)
        elif rule == "match":
            oracle.accept_match(w.cu_B, tl / temperature, w.draft_tokens, w.tau, w.uniforms)
        else:
            oracle.accept(w.cu_B, tl, dl, w.draft_tokens, w.tau, w.uniforms, n_threads=threads,
                          temperature=temperature)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    toks = reps * int(w.cu_B[-1])
    return toks / el, el, reps


def merge_launches(w, ws_bytes):
    """1 when the verify plan splits some unit's keys (K3 runs), else 0: the
    workspace then holds split partials beyond the status word, the rotated
    queries (fp32 path) and one int4 per new token, each 256-byte aligned."""
    up = lambda n: (n + 255) // 256 * 256
    T = 2 * int(w.cu_B[-1])
    base = up(4) + up(T * 16)
    if w.spec.dtype != "bf16":
        base += up(T * w.spec.Hq * w.spec.hd * 4)
    return 1 if ws_bytes > base else 0


def cpu_threads():
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    from oracle import build as obuild
    obuild.build()
    w = synth.config(args.workload)
    sub = cpu_sample(w, args.workload)
    threads = cpu_threads()
    per_step = []
    per = max(1.0, min(8.0, 60.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        v, el, reps = oracle_step_sample(sub, per, threads, args.accept, args.temperature)
        if i >= args.warmup:
            per_step.append(el / reps)
    ms = float(np.mean(per_step)) * 1e3
    value = int(sub.cu_B[-1]) / (ms / 1e3)
    sample = ("the first %d of %d sequences of %s per pass, passes repeated for >= %.1f s "
              "per step" % (len(sub.lens), len(w.lens), w.spec.name, per))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, args):
    s = w.spec
    return {"workload": s.name, "global_batch": len(w.lens) * max(1, args.gpus),
            "seq_len": int(w.lens.max()), "B": int(w.Bs.max()), "q_heads": s.Hq,
            "kv_heads": s.Hkv, "head_dim": s.hd, "vocab": s.vocab,
            "parallelism": "replicas x%d" % max(1, args.gpus),
            "l2": "flushed (512 MB write) before every timed step",
            "accept": args.accept + ("" if args.accept == "greedy" or args.temperature == 1.0
                                     else " at temperature %g" % args.temperature)
                      + ("" if args.accept_path == "auto" else " (%s path)" % ACCEPT_PATHS[args.accept_path])}


ACCEPT_PATHS = {"auto": "two-kernel", "single": "single-launch cluster"}


# ---------------------------------------------------------------- multi-rank helpers
def max_over_ranks(dist, x, device):
    """The largest rank's value of x (x itself on a single rank): the job's
    time is its slowest rank's."""
    if not dist:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(tokens_per_rank_step, world, total_ms, steps):
    """Whole-job tokens/s: every rank's tokens of a step over the step time
    (the slowest rank's total over the steps)."""
    return tokens_per_rank_step * world / (total_ms / steps / 1e3)


# ---------------------------------------------------------------- GPU arm
def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import synth
    from speculative_decoding_diffusion_gb300 import build as libbuild
    from speculative_decoding_diffusion_gb300 import binding
    from speculative_decoding_diffusion_gb300.staging import DeviceWorkload
    libbuild.build()
    w = synth.config(args.workload)
    dw = DeviceWorkload(w, device="cuda:%d" % local)
    if args.accept_path == "single":
        dw.accept_ws = torch.zeros(256, dtype=torch.uint8, device="cuda:%d" % local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    vev = [ev() for _ in range(4)]
    aev = [ev() for _ in range(3)]
    for e in vev + aev:
        e.record()       # create the underlying CUDA events
    torch.cuda.synchronize()

    def step(timed):
        dw.verify(events=vev if timed else None)
        dw.accept(events=aev if timed else None, rule=rule_code(args),
                  temperature=args.temperature)

    # warm-up outside any graph (builds device-side caches and attributes)
    for _ in range(args.warmup):
        flush.zero_()
        step(False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()           # the timed step
    with torch.cuda.graph(graph):
        step(False)
    kgraph = torch.cuda.CUDAGraph()          # the same step with per-kernel marks
    with torch.cuda.graph(kgraph):
        step(True)
    for _ in range(3):
        flush.zero_()
        graph.replay()
        flush.zero_()
        kgraph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    t_start, t_end = ev(), ev()
    step_ms, k_ms = [], {n: [] for n in ("K1", "K2", "K3", "K4", "K4a", "K4b")}
    for _ in range(args.steps):
        flush.zero_()
        t_start.record()
        graph.replay()
        t_end.record()
        torch.cuda.synchronize()
        step_ms.append(t_start.elapsed_time(t_end))
    for _ in range(max(10, args.steps // 4)):
        flush.zero_()
        kgraph.replay()
        torch.cuda.synchronize()
        v = [vev[i].elapsed_time(vev[i + 1]) for i in range(3)]
        for n, t in zip(("K1", "K2", "K3"), v):
            k_ms[n].append(t)
        k_ms["K4"].append(aev[0].elapsed_time(aev[2]))
        k_ms["K4a"].append(aev[0].elapsed_time(aev[1]))
        k_ms["K4b"].append(aev[1].elapsed_time(aev[2]))
    torch.cuda.synchronize()
    dev_total_ms = max_over_ranks(dist, float(np.sum(step_ms)), "cuda")

    # ---- end to end through the C ABI with host buffers
    def pin(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                             else np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).pin_memory()

    host_in = {
        "q": pin(w.q), "k_new": pin(w.k_new), "v_new": pin(w.v_new),
        "target": pin(w.target), "draft": pin(w.draft),
        "draft_tokens": pin(w.draft_tokens.astype(np.int32)), "tau": pin(w.tau),
        "uniforms": pin(w.uniforms), "lens": pin(w.lens), "cu_B": pin(w.cu_B),
        "block_table": pin(w.block_table)}
    if args.accept != "sample":              # greedy and matching read no draft logits,
        del host_in["draft"]                 # greedy no uniforms either
    if args.accept == "greedy":
        del host_in["uniforms"]
    dev_of = {"q": dw.q, "k_new": dw.k_new, "v_new": dw.v_new, "target": dw.target,
              "draft": dw.draft, "draft_tokens": dw.draft_tokens, "tau": dw.tau,
              "uniforms": dw.uniforms, "lens": dw.lens, "cu_B": dw.cu_B,
              "block_table": dw.block_table}
    host_out = {"out": torch.empty(dw.out.shape, dtype=dw.out.dtype).pin_memory(),
                "n_accept": torch.empty(len(w.lens), dtype=torch.int32).pin_memory(),
                "token": torch.empty(len(w.lens), dtype=torch.int32).pin_memory(),
                "pos": torch.empty(len(w.lens), dtype=torch.int32).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    # The logits (most of the bytes) are copied on a second stream while the
    # attention inputs are copied and the attention runs; the acceptance
    # waits for them.  (Host-to-device copies top out near 210 GB/s on this
    # box whatever the number of streams, so overlap is what is left.)
    side = torch.cuda.Stream()
    late = [k for k in ("target", "draft") if k in host_in]

    def e2e_body():
        cur = torch.cuda.current_stream()
        for k, h in host_in.items():              # the attention's inputs first
            if k not in late:
                dev_of[k].copy_(h, non_blocking=True)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            for k in late:
                dev_of[k].copy_(host_in[k], non_blocking=True)
        dw.verify()
        cur.wait_stream(side)
        dw.accept(rule=rule_code(args), temperature=args.temperature)
        host_out["out"].copy_(dw.out, non_blocking=True)
        host_out["n_accept"].copy_(dw.n_accept, non_blocking=True)
        host_out["token"].copy_(dw.token, non_blocking=True)
        host_out["pos"].copy_(dw.pos, non_blocking=True)

    def e2e_step():
        e2e_body()
        stream.synchronize()

    for _ in range(3):
        flush.zero_()
        e2e_step()
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_total = float(np.sum(e2e_ms))
    # the same copies and calls replayed as one graph
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        e2e_body()
    g2.replay()
    torch.cuda.synchronize()
    e2eg_ms = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g2.replay()
        stream.synchronize()
        e2eg_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_total = max_over_ranks(dist, e2e_total, "cuda")
    e2eg_total = max_over_ranks(dist, float(np.sum(e2eg_ms)), "cuda")
    peak, peak_kind = hbm_peak()
    next_rows = time_next_rows(w, dw, flush, max(10, args.steps // 4), peak)
    clk = clocks.stop()
    status = binding.read_status(dw.verify_ws) | binding.read_status(dw.accept_ws)

    ms_per_step = dev_total_ms / args.steps
    value = throughput(int(w.cu_B[-1]), world, dev_total_ms, args.steps)
    e2e_value = throughput(int(w.cu_B[-1]), world, e2e_total, args.steps)
    e2eg_value = throughput(int(w.cu_B[-1]), world, e2eg_total, args.steps)
    k2_mean = float(np.mean(k_ms["K2"]))
    achieved = k2_bytes(w) / (k2_mean / 1e3) / 1e9
    traffic = recorded_traffic(w.spec)
    # K1, K2, K3 (only where a sequence's keys are split), and the
    # acceptance: on the chunked path the chunk pass (K4a) and the one
    # finishing kernel of the rule (K4b), else one cluster launch (K4a and
    # K4b are reported only on the chunked path)
    chunked = args.accept_path == "auto"
    n_launch = 2 + merge_launches(w, dw.verify_ws.numel()) + (2 if chunked else 1)
    if not chunked:
        del k_ms["K4a"], k_ms["K4b"]
    kernels = {n: {"ms": float(np.mean(t))} for n, t in k_ms.items()}
    attn_ms = sum(kernels[n]["ms"] for n in ("K1", "K2", "K3"))
    acc_ms = kernels["K4"]["ms"]
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.spec.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_of(w, args),
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d * world,
                    "d2h_bytes_per_step": d2h * world},
            "e2e_graph": {"value": e2eg_value, "unit": UNIT, "h2d_bytes_per_step": h2d * world,
                          "d2h_bytes_per_step": d2h * world},
            "gpu_launches": n_launch * args.steps,
            "roofline": {"kernel": "K2 split-KV masked attention", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic,
                         "algorithmic_bytes_per_launch": k2_bytes(w)},
            "verify_attn_GBps": attn_bytes(w) / (attn_ms / 1e3) / 1e9,
            "accept_GBps": accept_bytes(w, args.accept != "sample") / (acc_ms / 1e3) / 1e9,
            "accept_frac": accept_bytes(w, args.accept != "sample") / (acc_ms / 1e3) / 1e9 / peak,
            "kernels_ms": {n: round(k["ms"], 5) for n, k in kernels.items()},
            "next_rows": next_rows,
            "clocks": clk, "status_word": status}
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import build as obuild
        obuild.build()
        threads = cpu_threads()
        sub = cpu_sample(w, args.workload)
        v, el, reps = oracle_step_sample(sub, args.cpu_seconds, threads, args.accept,
                                         args.temperature)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": sample_text(sub, w, reps, el)
                                          + " (attention + acceptance)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
