"""Benchmark of the C2KV composed-cache hot path on one GB300 (or N replicas).

One step = one full request of the workload: compose the documents'
compressed pre-RoPE segments from the pinned host store into HBM (a kernel
reads them over the host link and re-rotates K), prefill the question on
every layer, then
decode every answer token on every layer.  Consecutive requests overlap as
in a serving loop: request r+1 is composed on a second stream, into its own
cache, while request r decodes.  Headline value: answer tokens per second
over the timed requests.  Prefill and decode are replayed from CUDA graphs
captured once (the graphs hold only this library's kernels).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
                       [--impl ours|reference] [--workload NAME]
Under torchrun (N > 1) every rank serves its own replica of the workload;
value = all ranks' tokens / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "composed-cache decode tok/s + attention HBM GB/s vs peak; compose+TTFT ms"
DEFAULT_WORKLOAD = "llama8b_32x4096_k4_b4"


# ------------------------------------------------------------------ oracle leg

def _oracle_worker(workload: str, wid: int, cmd_q, out_q) -> None:
    """One spawned, single-threaded worker of the CPU oracle: it draws one
    layer of the workload's first request once, then, for every budget it
    receives, repeats one layer of compose, one layer of question prefill
    (if the workload has a question) and one decode step of that layer until
    the budget is spent, and reports the median time of each part."""
    import numpy as np
    import oracle.c2kv_oracle as O
    from compressed_composable_kv_gb300 import synth as S

    w = S.WORKLOADS[workload]
    g = w.geom
    docs_meta, reqs = S.make_requests(w)
    req = reqs[0]
    st = {}
    for i in set(req.doc_ids):
        n, s = docs_meta[i]
        d = S.make_document(g, i, n, w.k, w.seed, n_slots=s, layers=1)
        st[i] = (n, s, d.k_pre, d.v)
    inp = S.make_step_inputs(w, layers=1, decode_steps=1)
    out_q.put(("ready", wid))
    while True:
        budget_s = cmd_q.get()
        if budget_s is None:
            return
        t_comp, t_pre, t_dec = [], [], []
        t_start = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            pos, lt, kr, vr = O.compose(st, req.doc_ids, req.order, w.k, g.rope_theta)
            t1 = time.perf_counter()
            kc, vc = kr[0], vr[0]
            if w.q_len:
                _, kq = O.attend_new_tokens(inp.q_pre[0, 0], inp.kq_pre[0, 0], inp.vq[0, 0], kc, vc, lt,
                                            g.rope_theta)
                kc = np.concatenate([kc, kq], axis=1)
                vc = np.concatenate([vc, inp.vq[0, 0].transpose(1, 0, 2)], axis=1)
            t2 = time.perf_counter()
            O.attend_new_tokens(inp.qd_pre[0:1, 0, 0], inp.kd_pre[0:1, 0, 0], inp.vd[0:1, 0, 0], kc, vc,
                                lt + w.q_len, g.rope_theta)
            t3 = time.perf_counter()
            t_comp.append(t1 - t0)
            t_pre.append(t2 - t1)
            t_dec.append(t3 - t2)
            if time.perf_counter() - t_start >= budget_s:
                break
        out_q.put(("done", wid, statistics.median(t_comp), statistics.median(t_pre),
                   statistics.median(t_dec), len(t_comp), len(pos)))


class OraclePool:
    """The CPU oracle on the host's cores: one spawned single-threaded worker
    per core of the process's affinity set.  The request's work is split over
    (layer, decode step) units -- L layers of compose (+ question prefill) and
    L x T decode steps per sequence -- which are independent, so C cores take
    1/C of them each; every worker times the same one-layer units while all C
    run at once (so the measured unit times include the cores' contention).
    The oracle's arithmetic is not changed."""

    def __init__(self, workload: str, cores: int = 0):
        import multiprocessing as mp
        self.workload = workload
        self.cores = cores or len(os.sched_getaffinity(0))
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.out_q = ctx.Queue()
            self.cmd_qs = [ctx.Queue() for _ in range(self.cores)]
            self.procs = [ctx.Process(target=_oracle_worker, args=(workload, i, self.cmd_qs[i], self.out_q),
                                      daemon=True) for i in range(self.cores)]
            for p in self.procs:
                p.start()
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        # every worker reports ready; one that died on start ends the wait
        # instead of the timeout
        import queue
        ready, t_end = 0, time.monotonic() + 900
        while ready < self.cores:
            try:
                msg = self.out_q.get(timeout=2)
            except queue.Empty:
                dead = [p.exitcode for p in self.procs if p.exitcode is not None]
                if dead or time.monotonic() > t_end:
                    self.close()
                    raise RuntimeError(f"oracle workers did not start (exit codes {dead})")
                continue
            assert msg[0] == "ready", msg
            ready += 1

    def sample(self, budget_s: float) -> dict:
        from compressed_composable_kv_gb300 import synth as S
        w = S.WORKLOADS[self.workload]
        t0 = time.perf_counter()
        for q in self.cmd_qs:
            q.put(budget_s)
        res = [self.out_q.get(timeout=budget_s * 20 + 600) for _ in range(self.cores)]
        wall = time.perf_counter() - t0
        comp = statistics.median(r[2] for r in res)
        pre = statistics.median(r[3] for r in res)
        dec = statistics.median(r[4] for r in res)
        reps = sum(r[5] for r in res)
        L, T, B = w.geom.n_layers, w.decode_steps, w.batch
        # B sequences x (L layers of compose + prefill, L x T decode steps), over C cores
        request_s = B * (L * (comp + pre) + L * T * dec) / self.cores
        return {
            "request_s": request_s,
            "tok_s": B * T / request_s,
            "wall_s": wall,
            "cores": self.cores,
            "kind": "oracle",
            "sample": (f"{self.workload}, request 0: 1 layer compose ({res[0][6]} slots)"
                       + (f" + 1 layer question prefill ({w.q_len} tokens)" if w.q_len else "")
                       + f" + 1 decode step, timed {reps} times in all on {self.cores} single-threaded "
                         f"processes at once ({wall:.1f} s); the request's {L} layers x (compose"
                       + (" + prefill" if w.q_len else "") + f") and {L} x {T} decode steps x {B} "
                         f"sequences divided over the {self.cores} cores (extrapolated)"),
        }

    def close(self) -> None:
        for q in self.cmd_qs:
            q.put(None)
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()


def run_oracle_sample(workload: str, budget_s: float) -> dict:
    pool = OraclePool(workload)
    try:
        return pool.sample(budget_s)
    finally:
        pool.close()


# ------------------------------------------------------------------ helpers

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def sources_sha(srcs: str) -> str:
    """sha256[:16] over the comma-separated source files, in order."""
    h = hashlib.sha256()
    for src in srcs.split(","):
        h.update(open(os.path.join(ROOT, src), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """dram bytes per key-row of `kernel` from the committed ncu summary, if the
    kernel's sources are unchanged since the capture (sha256 over them)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for ln in lines:
        if ln.startswith("#") or not ln.strip():
            continue
        name, srcs, sha, per_unit = ln.split()[:4]
        if name != kernel:
            continue
        return float(per_unit) if sources_sha(srcs) == sha else None
    return None


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise max of per-rank timings (replicas finish when the slowest
    does).  world == 1 returns the values unchanged."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def init_ranks(backend=None) -> None:
    """Process group of the replicas (env:// rendezvous), with a bounded
    timeout (C2KV_RANK_TIMEOUT_S, default 300 s): a rank that dies makes the
    others' next barrier or timing reduction fail instead of waiting on it."""
    import datetime
    import torch
    import torch.distributed as dist
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    timeout = datetime.timedelta(seconds=float(os.environ.get("C2KV_RANK_TIMEOUT_S", "300")))
    dist.init_process_group(backend, timeout=timeout)


def replica_tokens(batch: int, decode_steps: int, steps: int, world: int) -> int:
    """Answer tokens all ranks produce in `steps` requests each (weak scaling)."""
    return batch * decode_steps * steps * world


# ------------------------------------------------------------------ our arm

def run_ours(args, rank: int, world: int) -> dict:
    import numpy as np
    import torch
    import compressed_composable_kv_gb300 as P
    from compressed_composable_kv_gb300 import synth as S

    w = S.WORKLOADS[args.workload]
    g = w.geom
    L, Bn, Q, T = g.n_layers, w.batch, w.q_len, w.decode_steps
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda")

    # -------- setup (untimed): pinned store, caches, inputs, graphs
    docs_meta, reqs = S.make_requests(w)
    used = sorted({d for r in reqs for d in r.doc_ids})
    seg_bytes = {i: 2 * g.n_layers * g.n_kv_heads * docs_meta[i][1] * g.head_dim * 2 for i in used}
    # Each document is drawn, stored in the pinned pool and dropped in turn,
    # so the host holds one document's arrays at a time besides the pool.
    store = P.c2kv_store_create(g, sum(seg_bytes[i] + 512 for i in used) + (1 << 20))
    for i in used:
        d = S.make_document(g, i, docs_meta[i][0], w.k, w.seed, n_slots=docs_meta[i][1])
        P.c2kv_store_segments(store, [i], [d.n_tokens], [d.n_slots], w.k, [d.k_pre], [d.v])
        del d
    compose_bytes = sum(seg_bytes[d] for r in reqs for d in r.doc_ids)
    # Two request states (caches, tables, scratch, graphs): request r uses
    # state r % 2, and request r+1 is composed on a second stream while
    # request r decodes, as a serving loop would.  Every request does all of
    # its work inside the timed region.
    specs = [P.RequestSpec(r.doc_ids, r.order) for r in reqs]
    bts = [P.RequestBatch(store, g, specs, w.k, Q, T) for _ in range(2)]
    bt = bts[0]
    inp = S.make_step_inputs(w)
    names = ["q_pre", "kq_pre", "vq", "qd_pre", "kd_pre", "vd"]
    host = {}
    dev_ins = [{}, {}]   # per request state, so a request's inputs can land while the other decodes
    for n in names:
        a = getattr(inp, n)
        if a.size == 0:
            continue
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        host[n] = t.pin_memory()
        for d_in in dev_ins:
            d_in[n] = host[n].to(dev)
    h2d_bytes = sum(t.numel() * 2 for t in host.values())
    pre_out = torch.empty((L, Bn, Q, g.n_q_heads, g.head_dim), dtype=torch.bfloat16, device=dev) if Q else None
    dec_out = torch.empty((T, L, Bn, g.n_q_heads, g.head_dim), dtype=torch.bfloat16, device=dev)
    res_host = torch.empty((T, Bn, g.n_q_heads, g.head_dim), dtype=torch.bfloat16).pin_memory()
    d2h_bytes = res_host.numel() * 2

    stream = torch.cuda.Stream()    # prefill and decode
    cstream = torch.cuda.Stream()   # compose of the next request
    torch.cuda.synchronize()

    # Compose and prefill are layer-pipelined: layer group i is composed
    # (its copies queue behind group i-1's on the store's copy stream), then
    # its question prefill is enqueued, so the prefill of early layers runs
    # while later layers are still crossing the host link.
    n_groups = min(L, 8)
    groups = [(i * L // n_groups, (i + 1) * L // n_groups) for i in range(n_groups)]

    def prefill_layers(i, l0, l1):
        b, d_in = bts[i], dev_ins[i]
        for l in range(l0, l1):
            b.prefill(l, d_in["q_pre"][l], d_in["kq_pre"][l], d_in["vq"][l], pre_out[l], stream)

    def decode_all(i, steps=T):
        b, d_in = bts[i], dev_ins[i]
        for t in range(steps):
            for l in range(L):
                b.decode(l, d_in["qd_pre"][t, l], d_in["kd_pre"][t, l], d_in["vd"][t, l], dec_out[t, l], stream)
            b.advance(stream)

    # Warm the launch paths eagerly once per state (one decode step is enough
    # to set the kernels' attributes), then capture.
    g_pre = [[torch.cuda.CUDAGraph() for _ in groups] if Q else None for _ in bts]
    g_dec = [torch.cuda.CUDAGraph() for _ in bts]
    for i, b in enumerate(bts):
        with torch.cuda.stream(stream):
            b.compose(stream)
            if Q:
                prefill_layers(i, 0, L)
            b.reset_decode(stream)
            decode_all(i, 1)
        torch.cuda.synchronize()
        # the library's launch counter around the captures: launches per replay
        n0 = P.c2kv_kernel_launches()
        with torch.cuda.stream(stream):
            if Q:
                for gr, (l0, l1) in zip(g_pre[i], groups):
                    with torch.cuda.graph(gr, stream=stream):
                        prefill_layers(i, l0, l1)
            n1 = P.c2kv_kernel_launches()
            with torch.cuda.graph(g_dec[i], stream=stream):
                decode_all(i)
        torch.cuda.synchronize()
        graph_launches = (n1 - n0, P.c2kv_kernel_launches() - n1)   # (prefill, decode) per request
    assert P.c2kv_device_error() == P.C2KV_OK

    def isolated_request(e):
        """One request alone on the stream: compose layer-pipelined with the
        prefill, then decode (the time-to-first-token measurement)."""
        with torch.cuda.stream(stream):
            e[0].record(stream)
            for gi, (l0, l1) in enumerate(groups):
                bt.compose_layers(l0, l1, stream)
                if gi == len(groups) - 1:
                    e[1].record(stream)   # the whole cache is composed
                if Q:
                    g_pre[0][gi].replay()
            bt.reset_decode(stream)
            e[2].record(stream)
            g_dec[0].replay()
            e[3].record(stream)

    ev_grp = [[torch.cuda.Event() for _ in groups] for _ in bts]
    ev_free = [torch.cuda.Event() for _ in bts]
    ev_go = torch.cuda.Event()

    def enqueue_compose(i, with_host=False):
        with torch.cuda.stream(cstream):
            cstream.wait_event(ev_free[i])   # the state's previous request has decoded
            if with_host:                    # this request's inputs, from pinned host memory
                for n, d in dev_ins[i].items():
                    d.copy_(host[n], non_blocking=True)
            for gi, (l0, l1) in enumerate(groups):
                bts[i].compose_layers(l0, l1, cstream)
                ev_grp[i][gi].record(cstream)

    def run_request(i, e=None, with_host=False):
        with torch.cuda.stream(stream):
            for gi in range(len(groups)):
                stream.wait_event(ev_grp[i][gi])
                if Q:
                    g_pre[i][gi].replay()
            bts[i].reset_decode(stream)
            if e:
                e[0].record(stream)
            g_dec[i].replay()
            if e:
                e[1].record(stream)
            ev_free[i].record(stream)
            if with_host:
                res_host.copy_(dec_out[:, L - 1], non_blocking=True)

    def pipeline(n, evs=None, with_host=False):
        """n requests; request r+1's compose overlaps request r's decode."""
        ev_go.record(stream)
        cstream.wait_event(ev_go)
        enqueue_compose(0, with_host)
        for r in range(n):
            run_request(r % 2, evs[r] if evs else None, with_host)
            if r + 1 < n:
                enqueue_compose((r + 1) % 2, with_host)

    # pinned host->device copy bandwidth, the denominator of the compose
    # copies: a 1 GiB copy from pinned memory right before each isolated
    # compose below, so that both see the host link (shared with the other
    # GPUs and jobs on the same host) in the same state
    big = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    big_d = torch.empty_like(big, device=dev)

    def pinned_copy_s():
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            big_d.copy_(big, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        return a.elapsed_time(b_) / 1e3

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # time to first token and the phases of one request alone (untimed region)
    iso = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(3)]
    pinned_s = []
    for i, e in enumerate([iso[0]] + iso):
        t_pin = pinned_copy_s()
        if i > 0:
            pinned_s.append(t_pin)
        isolated_request(e)
        torch.cuda.synchronize()
    pinned_s += [pinned_copy_s() for _ in range(3)]
    # the link's rate: the best of the copies timed around the composes (the
    # host side of the link is shared, so single copies vary)
    pinned_gbs = big.numel() / min(pinned_s) / 1e9
    del big, big_d
    comp = statistics.mean(e[0].elapsed_time(e[1]) for e in iso) / 1e3
    pre = statistics.mean(e[1].elapsed_time(e[2]) for e in iso) / 1e3
    dec_iso = statistics.mean(e[2].elapsed_time(e[3]) for e in iso) / 1e3

    pipeline(args.warmup)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_idx = torch.cuda.current_device()
    with ClockSampler(gpu_idx) as clk:
        n_eager = P.c2kv_kernel_launches()
        t_beg.record(stream)
        pipeline(args.steps, ev)
        t_end.record(stream)
        n_eager = P.c2kv_kernel_launches() - n_eager   # the composition launches
        torch.cuda.synchronize()
    # kernels of this library launched in the timed region, per request
    launches_per_step = n_eager / args.steps + sum(graph_launches)
    barrier()
    torch.cuda.synchronize()
    elapsed = t_beg.elapsed_time(t_end) / 1e3
    err = P.c2kv_device_error()
    assert err == P.C2KV_OK, f"device error {err}"
    dec = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3   # decode phase in the timed region
    # between one request's decode and the next one's: that request's question
    # prefill (its compose ran during the decode before)
    gaps = [ev[r - 1][1].elapsed_time(ev[r][0]) / 1e3 for r in range(1, args.steps)]

    # e2e: the same requests with inputs copied from pinned host memory and
    # the answer read back, all inside the timed region
    pipeline(1, with_host=True)
    torch.cuda.synchronize()
    barrier()
    e_beg, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_beg.record(stream)
    pipeline(args.steps, with_host=True)
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_elapsed = e_beg.elapsed_time(e_end) / 1e3

    model = run_model_step(P, S, g, bts[0], stream, comp, peaks=measured_peaks()) if is_llama(g) else None

    elapsed, e2e_elapsed = max_over_ranks([elapsed, e2e_elapsed], world, dev)
    toks = replica_tokens(Bn, T, args.steps, world)
    # algorithmic decode bytes: every key row (K and V) of every sequence,
    # layer and step, plus q/out/new k,v rows
    keys = sum((n + Q + t + 1) for n in bt.n_slots for t in range(T))
    row = g.n_kv_heads * g.head_dim * 2 * 2
    small = Bn * (2 * g.n_q_heads + 2 * g.n_kv_heads) * g.head_dim * 2
    dec_bytes_layer = keys * row + T * small
    dec_launches = T * L
    bytes_per_launch = dec_bytes_layer / T
    avg_launch_s = dec / dec_launches
    achieved = bytes_per_launch / avg_launch_s / 1e9
    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0
    per_key = profiled_traffic("decode_tc_kernel" if g.head_dim == 128 else "decode_kernel")
    traffic = None if per_key is None else per_key * (keys / T)
    clocks = clk.summary()
    ttft = comp + pre + dec_iso / T
    out = {
        "metric": METRIC,
        "value": toks / elapsed,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, world),
        "compose_ms": comp * 1e3,
        "prefill_ms": pre * 1e3,
        "decode_ms": dec * 1e3,
        "ttft_ms": ttft * 1e3,
        "phases": ("compose_ms, prefill_ms and ttft_ms: a request alone on the GPU (compose layer-"
                   "pipelined with its prefill), mean of 3; decode_ms: mean decode phase of the timed "
                   "requests"),
        "decode_only_tok_s": Bn * T / dec,
        "decode_ms_range": [min(e[0].elapsed_time(e[1]) for e in ev), max(e[0].elapsed_time(e[1]) for e in ev)],
        "between_decodes_ms": statistics.mean(gaps) * 1e3 if gaps else None,
        "attention_hbm_gbs": achieved,
        "h2d": {"compose_bytes": compose_bytes, "achieved_gbs": compose_bytes / comp / 1e9,
                "pinned_copy_gbs": pinned_gbs, "frac": compose_bytes / comp / 1e9 / pinned_gbs,
                "compose_ms_runs": [e[0].elapsed_time(e[1]) for e in iso],
                "note": ("compose = reading the segments over the host link + re-rotation, wall time on the stream; "
                         "pinned_copy_gbs = the best of 1 GiB pinned copies timed right before each of the 3 "
                         "timed composes and 3 after them")},
        "roofline": {"kernel": "decode_tc_kernel" if g.head_dim == 128 else "decode_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (hbm_gbs, burst)",
                     "launch_time": "decode-phase time / attention launches (includes the per-step "
                                    "length-advance kernel and launch gaps)"},
        "e2e": {"value": toks / e2e_elapsed, "unit": "tok/s", "h2d_bytes_per_step": h2d_bytes + compose_bytes,
                "d2h_bytes_per_step": d2h_bytes},
        "clocks": clocks,
        "gpu_launches": int(round(launches_per_step * args.steps)),
    }
    if model is not None:
        out["model_tok_s"] = model["tok_s"]
        out["model"] = model
    torch.cuda.synchronize()
    P.c2kv_store_destroy(store)
    return out


def is_llama(g) -> bool:
    """The decoder step is the Llama-3.1-8B layer (the attention geometry of
    the Llama workloads)."""
    return (g.n_q_heads, g.n_kv_heads, g.head_dim) == (32, 8, 128)


def run_model_step(P, S, g, rb, stream, compose_s: float, peaks: dict, steps: int = 8) -> dict:
    """The whole model's decode rate on the composed batch `rb`: seeded
    synthetic weights of every Llama-3.1-8B layer and the LM head on the
    device, `steps` decode steps (each: every layer's norms, projections,
    attention over the composed cache and MLP, then the LM head) replayed from
    a CUDA graph; and the same steps' linear layers and norms alone, against
    the HBM roofline of their weight bytes.  Runs after the timed region."""
    import torch
    shape = S.LLAMA31_8B_MODEL
    gen = torch.Generator(device="cuda").manual_seed(0xDEC0DE)
    d, dim, F = g.head_dim, shape.dim, shape.ffn
    nq, nkv = g.n_q_heads * d, g.n_kv_heads * d

    def mat(rows, cols):
        return (torch.randn((rows, cols), device="cuda", generator=gen) * cols ** -0.5).to(torch.bfloat16)

    def norm():
        return (1.0 + 0.1 * torch.randn(dim, device="cuda", generator=gen)).to(torch.bfloat16)

    weights = {"layers": [{"attn_norm": norm(), "qkv": mat(nq + 2 * nkv, dim), "o": mat(dim, nq),
                           "mlp_norm": norm(), "gate_up": mat(2 * F, dim), "down": mat(dim, F)}
                          for _ in range(g.n_layers)],
               "final_norm": norm(), "lm_head": mat(shape.vocab, dim)}
    m = P.DecoderModel(g, shape, weights, batch=rb.batch)
    m.x.copy_(torch.randn(m.x.shape, device="cuda", generator=gen).to(torch.bfloat16))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):   # eager once (kernel attributes), then capture
        rb.reset_decode(stream)
        m.decode_step(rb, stream)
        m.linears_only(stream)
    torch.cuda.synchronize()
    g_step, g_lin = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_step, stream=stream):
            for _ in range(steps):
                m.decode_step(rb, stream)
        with torch.cuda.graph(g_lin, stream=stream):
            for _ in range(steps):
                m.linears_only(stream)

    def timed(graph):
        ts = []
        for _ in range(4):
            with torch.cuda.stream(stream):
                rb.reset_decode(stream)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                graph.replay()
                b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        return statistics.median(ts[1:]) / steps

    t_step = timed(g_step)
    t_lin = timed(g_lin)
    assert P.c2kv_device_error() == P.C2KV_OK
    wbytes = m.weight_bytes()
    peak = peaks.get("hbm_gbs") or 6800.0
    out = {
        "tok_s": rb.batch / t_step,
        "ms_per_step": t_step * 1e3,
        "ttft_ms": (compose_s + t_step) * 1e3,
        "linear": {"kernel": "linear_tc_kernel + rmsnorm_kernel", "bound": "hbm",
                   "ms_per_step": t_lin * 1e3, "weight_bytes": wbytes,
                   "achieved_gbs": wbytes / t_lin / 1e9, "peak": peak, "frac": wbytes / t_lin / 1e9 / peak},
        "note": (f"Llama-3.1-8B decoder ({g.n_layers} layers, dim {dim}, MLP {F}, vocabulary {shape.vocab}) with "
                 f"seeded synthetic weights over the composed caches: {steps} decode steps x {rb.batch} sequences "
                 "from a CUDA graph (norms, fused QKV, attention with the append, O projection, SwiGLU MLP, LM "
                 "head); linear = the same steps' projections and norms alone, weight bytes / time"),
    }
    del m, weights, g_step, g_lin
    torch.cuda.synchronize()
    return out


def workload_config(w, world: int) -> dict:
    """The `config` object of both arms' lines (host-side sizes only)."""
    from compressed_composable_kv_gb300 import synth as S
    g = w.geom
    docs_meta, reqs = S.make_requests(w)
    n_groups = min(g.n_layers, 8)
    return {
        "workload": w.name,
        "geometry": f"{g.n_layers} layers, {g.n_q_heads} q / {g.n_kv_heads} kv heads, head_dim {g.head_dim}, "
                    f"rope_theta {g.rope_theta:g}",
        "k": w.k, "batch": w.batch,
        "composed_slots": [sum(docs_meta[d][1] for d in r.doc_ids) for r in reqs],
        "original_tokens": [sum(docs_meta[d][0] for d in r.doc_ids) for r in reqs],
        "question_tokens": w.q_len, "decode_steps": w.decode_steps,
        "l2": "inputs larger than L2 (composed cache per request > 1 GB; 129 MB L2)",
        "graphs": "prefill and decode replayed from CUDA graphs of this library's kernels",
        "ttft_pipeline": (f"compose and prefill layer-pipelined in {n_groups} groups: compose_ms = "
                          "until the whole cache is composed (prefill of earlier groups overlaps it), "
                          "prefill_ms = the rest of the prefill"),
        "request_pipeline": ("consecutive requests: request r+1 is composed (host->device reads and "
                             "re-rotation by the composition kernel, second stream, its own cache) while "
                             "request r decodes"),
        "parallelism": f"replicas x{world}",
        "attention_only": ("value: attention over the composed cache only (no projection/MLP weights)"
                           + ("; model_tok_s: the whole Llama-3.1-8B decoder step with synthetic weights"
                              if is_llama(g) else "")),
    }


def run_sweep(args) -> None:
    """Decode time per token over a composed cache of 16k..128k original
    tokens, compressed at k=16, 8, 4 vs uncompressed (k=1), batch 4, Llama3.1-8B
    attention geometry (C2KV explainer, section "results": the full cache's
    per-token decode time grows ~linearly with context, the compressed one
    reads a quarter of the bytes).  Only decode attention is timed: each
    step is the 32 layers' decode launches replayed from a CUDA graph; the
    caches are filled with N(0,1) bf16 on the device outside the timed region.
    Prints one JSON line per (context, k)."""
    import torch
    import compressed_composable_kv_gb300 as P
    from compressed_composable_kv_gb300 import synth as S

    g = S.LLAMA31_8B
    L, H, D, B = g.n_layers, g.n_kv_heads, g.head_dim, 4
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    stream = torch.cuda.Stream()
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    for ctx in (16384, 32768, 65536, 131072):
        for k in (16, 8, 4, 1):
            n = ctx // k
            steps = 16
            cap = n + steps + 32
            kc = [torch.randn((L, H, cap, D), device="cuda").to(torch.bfloat16) for _ in range(B)]
            vc = [torch.randn((L, H, cap, D), device="cuda").to(torch.bfloat16) for _ in range(B)]
            tab_bytes = P.c2kv_rope_table_bytes(g, cap)
            tabs = [torch.empty(tab_bytes // 4, dtype=torch.float32, device="cuda") for _ in range(B)]
            pos = torch.arange(cap, dtype=torch.int32, device="cuda")
            for t in tabs:
                P.c2kv_rope_table(g, pos, t)
            n_dev = torch.full((B,), n, dtype=torch.int32, device="cuda")
            max_keys = n + steps
            ws = torch.zeros(P.c2kv_attend_workspace_size(g, B, 1, max_keys), dtype=torch.uint8, device="cuda")
            q = torch.randn((steps, L, B, g.n_q_heads, D), device="cuda").to(torch.bfloat16)
            kn = torch.randn((steps, L, B, H, D), device="cuda").to(torch.bfloat16)
            out = torch.empty((steps, L, B, g.n_q_heads, D), dtype=torch.bfloat16, device="cuda")

            def decode_all():
                for t in range(steps):
                    for l in range(L):
                        P.c2kv_attend_decode(g, l, kc, vc, tabs, cap, n_dev, max_keys, q[t, l], kn[t, l], kn[t, l],
                                             out[t, l], ws, stream, P.C2KV_DECODE_OVERLAP_PREVIOUS if l else 0)
                    P.c2kv_seq_advance(n_dev, 1, stream)

            torch.cuda.synchronize()   # the caches, tables and lengths above were made on torch's stream
            with torch.cuda.stream(stream):
                decode_all()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    decode_all()
            times = []
            for rep in range(args.warmup + args.steps):
                with torch.cuda.stream(stream):
                    n_dev.fill_(n)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                e1.synchronize()
                if rep >= args.warmup:
                    times.append(e0.elapsed_time(e1) / 1e3)
            assert P.c2kv_device_error() == P.C2KV_OK
            t_step = statistics.median(times) / steps            # all layers, one token
            keys = sum(n + i + 1 for i in range(steps)) / steps
            gbs = B * keys * H * D * 2 * 2 * L / t_step / 1e9
            print(json.dumps({"sweep": "decode_vs_context", "original_tokens": ctx, "k": k, "cache_rows": n,
                              "batch": B, "layers": L, "ms_per_token": t_step * 1e3,
                              "tok_s": B / t_step, "attention_hbm_gbs": gbs, "frac_of_hbm_peak": gbs / peak}))
            del kc, vc, tabs, graph, ws, q, kn, out
            torch.cuda.empty_cache()


def run_kernel_probe(args) -> None:
    """The attention launches of --workload alone, on a small device
    footprint (the case its kernel profiles are taken on): the workload's
    geometry with --probe-layers layers, its batch and composed lengths, caches
    and question filled with N(0,1) on the device, every row's RoPE table at
    its index.  Runs one eager question prefill per layer (if the workload has
    a question) and one eager decode step over every layer, then replays
    --steps decode steps over the layers from a CUDA graph and times them.
    Prints one JSON line."""
    import torch
    import compressed_composable_kv_gb300 as P
    from compressed_composable_kv_gb300 import synth as S

    w = S.WORKLOADS[args.workload]
    g0 = w.geom
    g = S.Geometry(args.probe_layers, g0.n_q_heads, g0.n_kv_heads, g0.head_dim, g0.rope_theta)
    docs, reqs = S.make_requests(w)
    lens = [sum(docs[d][1] for d in r.doc_ids) for r in reqs]
    L, H, D, B, Q, T = g.n_layers, g.n_kv_heads, g.head_dim, len(lens), w.q_len, args.steps
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(5)
    cap = max(lens) + Q + T + 32

    def rnd(*shape):
        return torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16)

    kc = [rnd(L, H, cap, D) for _ in range(B)]
    vc = [rnd(L, H, cap, D) for _ in range(B)]
    tabs = [torch.empty(P.c2kv_rope_table_bytes(g, cap) // 4, dtype=torch.float32, device="cuda") for _ in range(B)]
    idx = torch.arange(cap, dtype=torch.int32, device="cuda")
    for t in tabs:
        P.c2kv_rope_table(g, idx, t)
    start = torch.tensor([n + Q for n in lens], dtype=torch.int32, device="cuda")
    n_dev = start.clone()
    max_keys = max(lens) + Q + T
    ws_bytes = P.c2kv_attend_workspace_size(g, B, 1, max_keys)
    if Q:
        ws_bytes = max(ws_bytes, P.c2kv_attend_workspace_size(g, B, Q, max(lens) + Q))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    qd, kd = rnd(T, L, B, g.n_q_heads, D), rnd(T, L, B, H, D)
    outd = torch.empty_like(qd)
    torch.cuda.synchronize()
    prefill = None
    with torch.cuda.stream(stream):
        if Q:
            qp, kp = rnd(L, B, Q, g.n_q_heads, D), rnd(L, B, Q, H, D)
            outp = torch.empty_like(qp)
            for l in range(L):
                P.c2kv_attend_prefill(g, l, kc, vc, tabs, cap, lens, qp[l], kp[l], kp[l], outp[l], ws, stream)
    if Q:
        # the question prefill of every layer from a graph, timed: each call
        # appends the question at rows [n, n + Q) again, so replays are alike
        gp = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gp, stream=stream):
                for l in range(L):
                    P.c2kv_attend_prefill(g, l, kc, vc, tabs, cap, lens, qp[l], kp[l], kp[l], outp[l], ws, stream)
        pts = []
        for _ in range(args.warmup + 3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                gp.replay()
                e1.record(stream)
            e1.synchronize()
            pts.append(e0.elapsed_time(e1) / 1e3)
        t_pre = statistics.median(pts[args.warmup:]) / L
        # 4 d flops per visible (q row, key) pair: QK^T and PV, each 2 d
        pairs = sum(g.n_q_heads * (n + i + 1) for n in lens for i in range(Q))
        flops = 4 * D * pairs
        peaks = measured_peaks()
        tf_peak = peaks.get("bf16_tflops") or 1900.0
        byts = sum((n + Q) for n in lens) * H * D * 4
        prefill = {"us_per_layer": t_pre * 1e6, "tflops": flops / t_pre / 1e12,
                   "frac_of_bf16_peak": flops / t_pre / 1e12 / tf_peak,
                   "roofline_us": max(byts / ((peaks.get("hbm_gbs") or 6800.0) * 1e9), flops / (tf_peak * 1e12)) * 1e6,
                   "note": "per layer: append + prefill launches from a graph; flops = 4 d per visible (q row, key) "
                           "pair (the hi/lo q split runs QK^T twice on the tensor cores: 1.5x these flops)"}
        for l in range(L):
            P.c2kv_attend_decode(g, l, kc, vc, tabs, cap, n_dev, max_keys, qd[0, l], kd[0, l], kd[0, l],
                                 outd[0, l], ws, stream, 0)

    def decode_all():
        for t in range(T):
            for l in range(L):
                P.c2kv_attend_decode(g, l, kc, vc, tabs, cap, n_dev, max_keys, qd[t, l], kd[t, l], kd[t, l],
                                     outd[t, l], ws, stream, P.C2KV_DECODE_OVERLAP_PREVIOUS if l else 0)
            P.c2kv_seq_advance(n_dev, 1, stream)

    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            decode_all()
    times = []
    for _ in range(args.warmup + 3):
        with torch.cuda.stream(stream):
            n_dev.copy_(start)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    assert P.c2kv_device_error() == P.C2KV_OK
    t_launch = statistics.median(times[args.warmup:]) / (T * L)
    keys = sum(n + Q + t + 1 for n in lens for t in range(T)) / T
    gbs = keys * H * D * 4 / t_launch / 1e9
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    line = {"kernel_probe": w.name, "layers": L, "batch": B, "composed_slots": lens, "question_tokens": Q,
            "decode_us_per_launch": t_launch * 1e6, "decode_attention_gbs": gbs,
            "decode_frac_of_hbm_peak": gbs / peak,
            "note": (f"{L} layers of random caches; eager: {L if Q else 0} prefill + {L} decode launches, "
                     f"then {T} decode steps x {L} layers from a graph (timed)")}
    del kc, vc, tabs, graph
    torch.cuda.empty_cache()
    if prefill is not None:
        line["prefill"] = prefill
    if is_llama(g0):
        line["linear"] = probe_linears(P, S, B, stream, peak)
    print(json.dumps(line))


def probe_linears(P, S, tokens: int, stream, peak: float, sets: int = 4) -> dict:
    """Each projection of the Llama-3.1-8B layer (and the LM head) for `tokens`
    tokens: `sets` distinct seeded weights of each (so every call reads its
    weights from HBM), called back to back from a CUDA graph; per call time and
    weight bytes / time against the HBM peak.  The first eager calls are the
    launches the linear kernel's profile is taken on.  Then the layer's four
    projections in layer order (`layer_chain`), `sets` layers of them from a
    graph: per layer time and weight bytes / time."""
    import torch
    shape = S.LLAMA31_8B_MODEL
    dim, F = shape.dim, shape.ffn
    kinds = {"qkv": (6144, dim, P.C2KV_LINEAR_SPLIT3), "o": (dim, dim, P.C2KV_LINEAR_ADD),
             "gate_up": (2 * F, dim, P.C2KV_LINEAR_SWIGLU), "down": (dim, F, P.C2KV_LINEAR_ADD),
             "lm_head": (shape.vocab, dim, P.C2KV_LINEAR_STORE)}
    gen = torch.Generator(device="cuda").manual_seed(11)
    ws = torch.zeros(P.c2kv_linear_workspace_size(tokens, shape.vocab), dtype=torch.uint8, device="cuda")
    P.c2kv_workspace_init(ws)
    out = {}
    layer = {}

    def timed_graph(fn) -> float:
        """One eager run, then a CUDA graph of `fn` replayed 5 times; the median
        of the last 4 replays, in seconds."""
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                fn()
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                graph.replay()
                b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) / 1e3)
        del graph
        return statistics.median(ts[1:])

    for name, (n, k, epi) in kinds.items():
        wts = [(torch.randn((n, k), device="cuda", generator=gen) * k ** -0.5).to(torch.bfloat16)
               for _ in range(sets)]
        x = torch.randn((tokens, k), device="cuda", generator=gen).to(torch.bfloat16)
        width = {P.C2KV_LINEAR_SPLIT3: 4096, P.C2KV_LINEAR_SWIGLU: n // 2}.get(epi, n)
        y = torch.zeros((tokens, width), device="cuda", dtype=torch.bfloat16)
        y2 = torch.zeros((tokens, 1024), device="cuda", dtype=torch.bfloat16)
        y3 = torch.zeros((tokens, 1024), device="cuda", dtype=torch.bfloat16)

        def call(wt, x=x, y=y, y2=y2, y3=y3, epi=epi):
            kw = {}
            if epi == P.C2KV_LINEAR_SPLIT3:
                kw = dict(y2=y2, y3=y3, split1=4096, split2=5120)
            elif epi == P.C2KV_LINEAR_ADD:
                kw = dict(residual=y)
            P.c2kv_linear(x, wt, y, ws, epi, stream=stream, flags=P.C2KV_LINEAR_OVERLAP_PREVIOUS, **kw)

        def run():
            for wt in wts:
                call(wt)

        t = timed_graph(run) / sets
        out[name] = {"us": t * 1e6, "weight_bytes": n * k * 2, "gbs": n * k * 2 / t / 1e9,
                     "frac_of_hbm_peak": n * k * 2 / t / 1e9 / peak}
        if name != "lm_head":
            layer[name] = (call, wts)
        else:
            del wts
        torch.cuda.empty_cache()

    def run_chain():
        for s_ in range(sets):
            for name in ("qkv", "o", "gate_up", "down"):
                call_, wts_ = layer[name]
                call_(wts_[s_])

    t = timed_graph(run_chain) / sets
    byts = sum(kinds[n][0] * kinds[n][1] * 2 for n in ("qkv", "o", "gate_up", "down"))
    out["layer_chain"] = {"us": t * 1e6, "weight_bytes": byts, "gbs": byts / t / 1e9,
                          "frac_of_hbm_peak": byts / t / 1e9 / peak}
    layer.clear()
    torch.cuda.empty_cache()
    assert P.c2kv_device_error() == P.C2KV_OK
    return out


def run_extract(args) -> None:
    """Extraction-side attention at full size (section "structured information
    flow"): one document of 4000 tokens followed by its 1000 slots (k=4),
    Llama3.1-8B attention geometry, one c2kv_attend_masked call per layer for
    32 layers, under the structured mask, the anchor-token mask of the
    ablation (section "results") and, for comparison, the plain causal mask
    over the same 5000 tokens (which skips nothing).  achieved TFLOP/s counts
    4*d flops per visible (query head, key) pair."""
    import torch
    import compressed_composable_kv_gb300 as P
    from compressed_composable_kv_gb300 import synth as S

    g = S.LLAMA31_8B
    L, n_doc, k = g.n_layers, 4000, 4
    n_slot = -(-n_doc // k)
    N = n_doc + n_slot
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    stream = torch.cuda.Stream()
    gen = torch.Generator(device="cuda").manual_seed(7)
    q = torch.randn((L, N, g.n_q_heads, g.head_dim), device="cuda", generator=gen).to(torch.bfloat16)
    kk = torch.randn((L, N, g.n_kv_heads, g.head_dim), device="cuda", generator=gen).to(torch.bfloat16)
    v = torch.randn((L, N, g.n_kv_heads, g.head_dim), device="cuda", generator=gen).to(torch.bfloat16)
    out = torch.empty_like(q)
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    peak = measured_peaks().get("bf16_tflops") or 1900.0
    # visible (query, key) pairs: documents causal; slot i sees the sink, its
    # own block (the union when they coincide) and slots 0..i
    doc_pairs = n_doc * (n_doc + 1) // 2
    slot_pairs = sum(len(set(range(min(k, n_doc))) | set(range(i * k, min((i + 1) * k, n_doc)))) + i + 1
                     for i in range(n_slot))
    # anchor mask: the causal pairs plus every (document, anchor) pair
    anchor_pairs = N * (N + 1) // 2 + n_doc * n_slot
    names = {P.C2KV_MASK_STRUCTURED: "structured", P.C2KV_MASK_ANCHOR: "anchor", P.C2KV_MASK_CAUSAL: "causal"}
    for mask, n_d, n_s, pairs in ((P.C2KV_MASK_STRUCTURED, n_doc, n_slot, doc_pairs + slot_pairs),
                                  (P.C2KV_MASK_ANCHOR, n_doc, n_slot, anchor_pairs),
                                  (P.C2KV_MASK_CAUSAL, N, 0, N * (N + 1) // 2)):
        def run_layers():
            for l in range(L):
                P.c2kv_attend_masked(g, mask, n_d, n_s, k, q[l], kk[l], v[l], out[l], ws, stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                run_layers()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                run_layers()
                e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) / 1e3)
        assert P.c2kv_device_error() == P.C2KV_OK
        t = statistics.median(times)
        flops = L * g.n_q_heads * pairs * 4 * g.head_dim
        print(json.dumps({"extract": names[mask],
                          "doc_tokens": n_doc, "slots": n_s, "k": k, "layers": L,
                          "ms_per_document": t * 1e3, "tokens_per_s": N / t,
                          "visible_pairs_per_head": pairs, "achieved_tflops": flops / t / 1e12,
                          "peak_tflops": peak, "frac_of_bf16_peak": flops / t / 1e12 / peak,
                          "note": "one c2kv_attend_masked call per layer (rotation, append, tcgen05 attention)"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work (on every core) behind cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=1.0,
                    help="seconds of oracle work per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="decode time vs context (16k..128k), compressed k=16/8/4 vs uncompressed")
    ap.add_argument("--kernel-probe", action="store_true",
                    help="the workload's prefill and decode launches alone, on --probe-layers layers of random caches")
    ap.add_argument("--probe-layers", type=int, default=2)
    ap.add_argument("--extract", action="store_true",
                    help="extraction-side attention (structured, anchor and causal masks), "
                         "4000-token document + 1000 slots")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.extract:
        run_extract(args)
        return
    if args.kernel_probe:
        run_kernel_probe(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        # The reference arm is the CPU oracle on the host's cores; only rank 0 runs it.
        if rank != 0:
            return
        from compressed_composable_kv_gb300 import synth as S
        pool = OraclePool(args.workload)
        try:
            samples = []
            for i in range(args.warmup + args.steps):
                r = pool.sample(args.ref_budget)
                if i >= args.warmup:
                    samples.append(r)
        finally:
            pool.close()
        tok_s = statistics.mean(s["tok_s"] for s in samples)
        line = {
            "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            # the time of the work each step actually ran (one bounded sample)
            "ms_per_step": statistics.mean(s["wall_s"] for s in samples) * 1e3,
            "extrapolated_request_s": statistics.mean(s["request_s"] for s in samples),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(S.WORKLOADS[args.workload], world),
            "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": samples[0]["cores"], "kind": "oracle",
                             "sample": samples[0]["sample"] + "; one sample per step"},
            "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_oracle_sample(args.workload, args.cpu_budget)
    if world > 1:
        init_ranks()
    out = run_ours(args, rank, world)
    if cpu is not None:
        out["cpu_baseline"] = {"value": cpu["tok_s"], "unit": "tok/s", "cores": cpu["cores"],
                               "kind": "oracle", "sample": cpu["sample"]}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
