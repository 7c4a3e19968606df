"""Benchmark of the paged GQA attention hot path on GB300.

One step = one decode step of the 70B-shaped batch (32 sequences, 64 query / 8 kv
heads, head_dim 128, contexts uniform on [1024, 4096], 16-token blocks shuffled over
the pool, bf16 cache): append the new token's K/V into the paged cache and run paged
decode attention over every cached token, as one fused launch. The metric is decode
KV-read GB/s: the K and V bytes of every cached token of every kv-head, read once
per step, divided by the step time.

Every other decode workload is measured the same way and reported beside it (the
Llama-3-8B batch, the 70B batch over an E4M3 cache, the prefix-sharing batch), each
with an element-by-element oracle check of one step; then the varlen prefill and
the rows past it (chunked prefill, speculative verification, sliding-window decode,
E4M3 prefill).

Three block-table sets over disjoint physical blocks (or three disjoint caches)
rotate from launch to launch, so each reads data that the previous two did not touch
(> the 129 MB L2): the decode and cached-prefix numbers are HBM numbers, not L2
numbers.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same per-GPU batch (weak scaling, no
data-path collective); rank 0 prints one JSON line.
"""
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

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged GQA decode KV-read GB/s (% of HBM peak); prefill TFLOP/s (% peak)"
DATA = "synthetic (seeded N(0,1) bf16 q/K/V, seeded shuffled block tables)"
ROTATIONS = 2  # extra disjoint table sets -> 3 in rotation


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def _kernel_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DECODE_FILES = ["paged_kv_gqa_10_gb300/csrc/decode.cu", "paged_kv_gqa_10_gb300/csrc/ptx.cuh"]
PREFILL_FILES = ["paged_kv_gqa_10_gb300/csrc/prefill.cu", "paged_kv_gqa_10_gb300/csrc/tc.cuh",
                 "paged_kv_gqa_10_gb300/csrc/ptx.cuh"]
KV_WRITE_FILES = ["paged_kv_gqa_10_gb300/csrc/kv_cache.cu", "paged_kv_gqa_10_gb300/csrc/ptx.cuh"]


def _profile_traffic(name, files):
    """Per-launch DRAM bytes from a committed ncu summary, if its kernel hash
    still matches the sources (else None: the counters are stale)."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != _kernel_hash(files):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        mhz, max_mhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                max_mhz = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, rank, local, world
    return None, rank, local, world


def reduce_max(res, keys, dist, device):
    """Every rank's timings replaced by their maximum over the ranks (the slowest rank
    sets the whole job's time)."""
    for k in keys:
        t = torch.tensor([float(res[k])], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        res[k] = float(t.item())
    return res


def job_value(bytes_per_rank, world, ms):
    """Whole-job GB/s: every rank streams its own replica of the batch (weak scaling)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def _finite(x):
    """A float for the JSON line (NaN / inf as their names: strict JSON has neither)."""
    x = float(x)
    return x if x == x and abs(x) != float("inf") else str(x)


def _parity_summary(gpu_res, ref_out, ref_lse):
    """One decode step's GPU output against the oracle's, element by element, with the
    parity tolerance: out within 1e-2 + 1e-2 |ref|, lse within 1e-3."""
    import numpy as np
    if isinstance(gpu_res, str):
        return {"error": gpu_res}
    out, lse = gpu_res
    err = np.abs(np.asarray(out, np.float64) - ref_out)
    ratio = err / (1e-2 + 1e-2 * np.abs(ref_out))
    gl = np.asarray(lse, np.float64)
    same_inf = np.isinf(gl) & np.isinf(ref_lse) & (np.sign(gl) == np.sign(ref_lse))
    lerr = np.abs(np.where(same_inf, 0.0, gl) - np.where(same_inf, 0.0, ref_lse))
    ok = bool(np.all(ratio <= 1.0) and np.all(lerr <= 1e-3))
    return {"rows": int(ref_lse.size), "out_max_abs_err": _finite(err.max()),
            "out_max_err_over_tolerance": _finite(ratio.max()),
            "lse_max_abs_err": _finite(lerr.max()), "within_tolerance": ok}


def _cpu_baseline(inp, target_s=10.0, gpu_res=None):
    """The oracle, as it stands, on the host cores: the whole batch over its cache with
    the step's new rows appended, repeated until about target_s seconds of CPU work
    have been timed. The first result is also compared with the GPU's output of the
    same step (gpu_res: (out, lse) as arrays, or the text of the error that kept the
    GPU side from producing it)."""
    import oracle
    cores = oracle.default_threads()
    dt = oracle.E4M3 if inp.cache_dtype == "e4m3" else oracle.BF16
    kc, vc = oracle.kv_cache_write(inp.step_key, inp.step_value, inp.step_slots, inp.k_cache,
                                   inp.v_cache, dtype=dt, k_scale=inp.k_scale,
                                   v_scale=inp.v_scale)
    args = (inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale)
    kw = dict(threads=cores, dtype=dt, k_scale=inp.k_scale, v_scale=inp.v_scale)
    t0 = time.perf_counter()
    ref_out, ref_lse = oracle.paged_decode(*args, **kw)
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_decode(*args, **kw)
    dt_s = (time.perf_counter() - t0) / reps
    gbs = workloads.kv_read_bytes(inp) / dt_s / 1e9
    res = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": f"the whole batch ({inp.num_seqs} sequences, "
                     f"{int(inp.context_lens.sum())} cached tokens, the step's new rows "
                     f"appended) x {reps} repetitions, fp64 C oracle, OpenMP over "
                     f"(sequence, kv-head), {dt_s * reps:.1f} s"}
    if gpu_res is not None:
        res["parity"] = _parity_summary(gpu_res, ref_out, ref_lse)
    return res


DECODE_WORKLOADS = {
    "70b_bf16": (lambda: workloads.llama70b_decode(rotations=ROTATIONS),
                 "70B decode: B=32, Hq=64, Hkv=8, D=128, block 16, ctx U[1024,4096], bf16 cache"),
    "llama3_8b": (lambda: workloads.llama3_8b_decode(rotations=ROTATIONS),
                  "Llama-3-8B decode: B=64, Hq=32, Hkv=8, D=128, block 16, ctx U[256,1024], "
                  "pool 8192"),
    "70b_e4m3": (lambda: workloads.llama70b_decode(cache_dtype="e4m3", rotations=ROTATIONS),
                 "70B decode: B=32, Hq=64, Hkv=8, D=128, block 16, ctx U[1024,4096], E4M3 cache "
                 "with per-kv-head scales"),
    "prefix": (lambda: workloads.prefix_sharing_decode(rotations=ROTATIONS),
               "prefix-sharing decode: B=16, ctx 8192, Hq=32, Hkv=8, D=128, block 16, groups of 4 "
               "share the blocks of their first 4096 tokens"),
}
# the headline first (the largest single-GPU bf16 decode configuration), then the others
DECODE_ORDER = ["70b_bf16", "llama3_8b", "70b_e4m3", "prefix"]


def decode_config(name, inp):
    """The static description of a decode workload, identical in both bench arms."""
    B, Hq, D = inp.q.shape
    kvb = workloads.kv_read_bytes(inp)
    return {"workload": DECODE_WORKLOADS[name][1], "batch": B, "q_heads": Hq,
            "kv_heads": inp.num_kv_heads, "head_dim": D, "block_size": inp.block_size,
            "cache_dtype": inp.cache_dtype, "kv_bytes_per_step": kvb,
            "unique_kv_bytes_per_step": workloads.kv_read_bytes(inp, unique=True),
            "step": "the new token of every sequence appended at position L-1 and attention "
                    "over the whole context",
            "l2": f"{ROTATIONS + 1} rotating block-table sets over disjoint blocks "
                  f"({(ROTATIONS + 1) * kvb / 1e6:.0f} MB > 129 MB L2)",
            "parallelism": "replica per GPU"}


def run_reference(args):
    """The oracle as the reference arm: the headline decode workload, metric and unit,
    timed on the host cores (each step = the whole batch through the fp64 oracle, over
    the cache with the step's new rows appended once before timing)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import oracle
    inp = DECODE_WORKLOADS[args.workload][0]()
    cores = oracle.default_threads()
    dt = oracle.E4M3 if inp.cache_dtype == "e4m3" else oracle.BF16
    kc, vc = oracle.kv_cache_write(inp.step_key, inp.step_value, inp.step_slots, inp.k_cache,
                                   inp.v_cache, dtype=dt, k_scale=inp.k_scale,
                                   v_scale=inp.v_scale)
    a = (inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale)
    kw = dict(threads=cores, dtype=dt, k_scale=inp.k_scale, v_scale=inp.v_scale)
    for _ in range(args.warmup):
        oracle.paged_decode(*a, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_decode(*a, **kw)
    dt_s = (time.perf_counter() - t0) / max(args.steps, 1)
    v = workloads.kv_read_bytes(inp) / dt_s / 1e9
    sample = (f"whole batch per step ({inp.num_seqs} sequences, "
              f"{int(inp.context_lens.sum())} cached tokens, the step's new rows appended)")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA, "config": decode_config(args.workload, inp),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class DecodeBench:
    """Device state of one decode workload and its step: the new token's K/V appended
    and attention over the whole context, as one fused launch
    (pgqa_paged_attention_decode_append) or, with fused=False, as two calls
    (pgqa_kv_cache_write, then pgqa_paged_attention_decode)."""

    def __init__(self, inp, dev):
        import paged_kv_gqa_10_gb300 as pgqa
        self.pgqa, self.inp, self.dev = pgqa, inp, dev
        self.tables = [inp.block_tables] + inp.rotations
        self.slots = [inp.step_slots] + inp.rotation_slots
        self.R = len(self.tables)
        B, Hq, D = inp.q.shape
        self.kc, self.vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
        self.ks = None if inp.k_scale is None else inp.k_scale.to(dev)
        self.vs = None if inp.v_scale is None else inp.v_scale.to(dev)
        self.q = inp.q.to(dev)
        self.cl = inp.context_lens.to(dev)
        self.bts = [t.to(dev) for t in self.tables]
        self.sls = [t.to(dev) for t in self.slots]
        self.nk, self.nv = inp.step_key.to(dev), inp.step_value.to(dev)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.ws_n = pgqa.decode_workspace_size(B, Hq, inp.num_kv_heads, D, inp.max_context_len)
        self.ws = torch.zeros(max(self.ws_n, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.kv_bytes = workloads.kv_read_bytes(inp)
        nblk = int(((inp.context_lens + 15) // 16).sum())
        # one decode launch reads every cached KV byte once, q, the table entries and
        # lengths, and writes out and lse
        self.alg_bytes = (self.kv_bytes + self.q.numel() * 2 + self.out.numel() * 2 +
                          self.lse.numel() * 4 + nblk * 4 + B * 4)
        # the fused launch also reads the new rows and writes them into the cache
        self.alg_bytes_fused = self.alg_bytes + 2 * 2 * self.nk.numel() * 2
        self.graphs = None
        self.fused = True

    def append(self, r, slots=None, key=None, value=None):
        self.pgqa.kv_cache_write(self.nk if key is None else key, self.nv if value is None else value,
                                 self.sls[r] if slots is None else slots, self.kc, self.vc,
                                 k_scale=self.ks, v_scale=self.vs, dev_status=self.status)

    def decode(self, r, table=None):
        self.pgqa.paged_attention_decode(
            self.out, self.lse, self.q, self.kc, self.vc, self.bts[r] if table is None else table,
            self.cl, self.inp.scale, self.inp.max_context_len, k_scale=self.ks, v_scale=self.vs,
            workspace=self.ws if self.ws_n else None, dev_status=self.status)

    def decode_append(self, r, table=None):
        self.pgqa.paged_attention_decode_append(
            self.out, self.lse, self.q, self.nk, self.nv, self.kc, self.vc,
            self.bts[r] if table is None else table, self.cl, self.inp.scale,
            self.inp.max_context_len, k_scale=self.ks, v_scale=self.vs,
            workspace=self.ws if self.ws_n else None, dev_status=self.status)

    def step(self, i):
        r = i % self.R
        if self.fused:
            self.decode_append(r)
        else:
            self.append(r)
            self.decode(r)

    def capture(self):
        """One CUDA graph per rotation, each holding one step (append + decode), and one
        graph holding the R steps of a full rotation back to back (no launch gap between
        steps)."""
        self.graphs = []
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for r in range(self.R):  # warm the capture stream
                self.step(r)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for r in range(self.R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(r)
            self.graphs.append(g)
        self.rotation_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.rotation_graph):
            for r in range(self.R):
                self.step(r)
        torch.cuda.synchronize()

    def run_steps(self, first, n):
        """Exactly n steps starting at step `first` (whole rotations as one replay)."""
        i = 0
        while i < n:
            if (first + i) % self.R == 0 and n - i >= self.R:
                self.rotation_graph.replay()
                i += self.R
            else:
                self.graphs[(first + i) % self.R].replay()
                i += 1

    def check(self):
        torch.cuda.synchronize()
        st = int(self.status.item())
        assert st == 0, f"device status {st}"


def _elapsed(fn, n):
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(n):
        fn(i)
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def measure_decode(inp, args, dev, dist=None, clocks_index=None, full=True):
    """Step time (CUDA-graph replays over the rotating table sets) and the step kernel's
    time (a graph of back-to-back launches); with full=True also the eager step, the
    same step as two calls, and the end-to-end step through the public API."""
    b = DecodeBench(inp, dev)
    for i in range(args.warmup):
        b.step(i)
    b.check()
    b.capture()
    for i in range(args.warmup):
        b.graphs[i % b.R].replay()
    b.check()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = None
    first = -(-args.warmup // b.R) * b.R  # start the timed steps on a whole rotation
    if clocks_index is not None:
        with ClockSampler(clocks_index) as cs:
            ms_graph = _elapsed(lambda i: b.run_steps(first, args.steps) if i == 0 else None, 1)
        clocks = cs.summary()
    else:
        ms_graph = _elapsed(lambda i: b.run_steps(first, args.steps) if i == 0 else None, 1)
    if dist:
        dist.barrier()
    b.check()
    if full:
        ms_eager = _elapsed(lambda i: b.step(args.warmup + i), args.steps)
        # the same steps as two calls (cache write, then decode), for comparison
        b.fused = False
        b.capture()
        b.run_steps(first, b.R)
        b.check()
        ms_two = _elapsed(lambda i: b.run_steps(first, args.steps) if i == 0 else None, 1)
        b.check()
        b.fused = True
    # the step's kernel alone: one CUDA graph of back-to-back fused launches cycling
    # over the disjoint block-table sets (no launch finds the previous one's pages in
    # L2), timed with events on the launching stream; every launch appends the same
    # rows again, so the launches compute exactly what the step does
    n_rep = 4 * b.R
    g_dec = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec):
        for i in range(n_rep):
            b.decode_append(i % b.R)
    g_dec.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    reps = max(1, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g_dec.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    dec_ms = e0.elapsed_time(e1) / (reps * n_rep)
    b.check()
    if not full:
        res = {"bench": b, "ms_graph": ms_graph / args.steps, "dec_ms": dec_ms,
               "clocks": clocks}
        if dist:
            reduce_max(res, ("ms_graph", "dec_ms"), dist, dev)
        return res

    # end to end through the public API, eager calls: the step's inputs (q, the new K/V
    # rows, the lengths and the block table) packed in one pinned host buffer per
    # block-table set and copied in with one transfer; out and lse share one device
    # buffer, read back with one transfer (a second stream with events to overlap the
    # transfers with the kernels cost more host time than it hid)
    import paged_kv_gqa_10_gb300 as pgqa
    al = lambda n: (n + 255) // 256 * 256
    parts = [inp.q, inp.step_key, inp.step_value, inp.context_lens]
    sizes = [t.numel() * t.element_size() for t in parts + [b.tables[0]]]
    offs = [sum(al(n) for n in sizes[:k]) for k in range(len(sizes))]
    total = offs[-1] + al(sizes[-1])
    h_in = []
    for tab in b.tables:
        h = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for t, o, n in zip(parts + [tab], offs, sizes):
            h[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        h_in.append(h)
    d_in = torch.empty(total, dtype=torch.uint8, device=dev)
    view = lambda buf, o, n, like: buf[o:o + n].view(like.dtype).view(like.shape)
    d_q, d_k, d_v, d_cl, d_bt = (view(d_in, o, n, t) for t, o, n in
                                 zip(parts + [b.tables[0]], offs, sizes))
    ob, lb = b.out.numel() * 2, b.lse.numel() * 4
    d_res = torch.empty(al(ob) + lb, dtype=torch.uint8, device=dev)
    d_out, d_lse = view(d_res, 0, ob, b.out), view(d_res, al(ob), lb, b.lse)
    h_res = torch.empty(al(ob) + lb, dtype=torch.uint8).pin_memory()

    # the C-ABI call itself, its arguments marshalled once (the buffers do not move)
    import ctypes
    fn = pgqa._handle().pgqa_paged_attention_decode_append
    vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    NB, Hkv, bs, D = b.kc.shape
    B, Hq, _ = inp.q.shape
    ws = b.ws if b.ws_n else None
    c_args = (vp(d_out), vp(d_lse), vp(d_q), vp(d_k), vp(d_v), vp(b.kc), vp(b.vc), vp(d_bt),
              ctypes.c_int(d_bt.shape[1]), vp(d_cl), ctypes.c_int(B), ctypes.c_int(Hq),
              ctypes.c_int(Hkv), ctypes.c_int(D), ctypes.c_int(NB), ctypes.c_int(bs),
              ctypes.c_float(inp.scale), ctypes.c_int(pgqa._cache_dtype(b.kc)), vp(b.ks),
              vp(b.vs), ctypes.c_int(inp.max_context_len), vp(ws),
              ctypes.c_size_t(0 if ws is None else ws.numel()), vp(b.status),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    def e2e_step(i):
        d_in.copy_(h_in[i % b.R], non_blocking=True)
        rc = fn(*c_args)
        if rc != 0:
            raise RuntimeError(f"paged_attention_decode_append: {pgqa.status_string(rc)}")
        h_res.copy_(d_res, non_blocking=True)

    h2d = total
    d2h = h_res.numel()
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = _elapsed(lambda i: e2e_step(args.warmup + i), args.steps)
    b.check()
    res = {"bench": b, "ms_graph": ms_graph / args.steps, "ms_eager": ms_eager / args.steps,
           "ms_two": ms_two / args.steps, "dec_ms": dec_ms, "e2e_ms": e2e_ms / args.steps, "h2d": h2d, "d2h": d2h,
           "clocks": clocks}
    if dist:
        reduce_max(res, ("ms_graph", "ms_eager", "ms_two", "dec_ms", "e2e_ms"), dist, dev)
    return res


def measure_prefill(args, dev):
    """Varlen causal prefill workload: KV write of every prompt token, then prefill.
    The inputs (q 35.6 MB, K/V 71 MB written and read, out 35.6 MB) exceed the L2."""
    import paged_kv_gqa_10_gb300 as pgqa
    inp = workloads.varlen_prefill()
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    q, key, value = inp.q.to(dev), inp.key.to(dev), inp.value.to(dev)
    slots, bt, cu = inp.slot_mapping.to(dev), inp.block_tables.to(dev), inp.cu_seqlens.to(dev)
    T, Hq, D = inp.q.shape
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, inp.max_seqlen),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def write():
        pgqa.kv_cache_write(key, value, slots, kc, vc, dev_status=status)

    def prefill():
        pgqa.paged_prefill_varlen(out, lse, q, kc, vc, bt, cu, inp.max_seqlen, inp.scale,
                                  workspace=ws, dev_status=status)

    for _ in range(args.warmup):
        write()
        prefill()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n = max(20, args.steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        write()
        ev[i][1].record(stream)
        prefill()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    w_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    p_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / n
    flops = workloads.causal_flops(inp.seq_lens, Hq, D)
    tflops = flops / (p_ms * 1e-3) / 1e12
    _, bf16_peak, kind = _peaks()
    kv_bytes = 2 * 2 * (key.numel() * 2)  # K and V: read from the input, written to the cache
    return {
        "workload": "varlen causal prefill: 16 seqs, L U[128,2048] (T=%d), Hq=32, Hkv=8, D=128" % T,
        "value": tflops, "unit": "TFLOP/s", "ms": p_ms, "launches_timed": n,
        "timing": "CUDA events around each launch, each after the cache write of the batch",
        "flops": flops, "flops_rule": "4*Hq*D*L(L+1)/2 per sequence (unmasked pairs only)",
        "roofline": {"bound": "tensor", "kernel": "paged_prefill_kernel<128>", "achieved": tflops,
                     "peak": bf16_peak, "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                     "peak_kind": kind + " bf16 burst (cuBLAS)",
                     "traffic": _profile_traffic("prefill_varlen.json", PREFILL_FILES)},
        "kv_cache_write": {"ms": w_ms, "bytes": kv_bytes,
                           "GB/s": kv_bytes / (w_ms * 1e-3) / 1e9,
                           "traffic": _profile_traffic("kv_cache_write.json", KV_WRITE_FILES)},
    }


def measure_cached_prefix(args, dev, names=("chunked_prefill", "speculative_verify")):
    """The rows past prefill and decode: prefill over a cached prefix (chunked prefill)
    and speculative verification (5 tokens per sequence), each through
    pgqa_paged_prefill_varlen_kv. The K/V are written once into the cache, which is then
    copied to ROTATIONS more caches at other addresses; a CUDA graph of back-to-back
    launches cycling over the copies is timed with events, so no launch finds the
    previous one's K/V in L2."""
    import paged_kv_gqa_10_gb300 as pgqa
    hbm, bf16_peak, kind = _peaks()
    res = {}
    makers = {"chunked_prefill": workloads.chunked_prefill,
              "speculative_verify": workloads.speculative_verify}
    for name in names:
        inp = makers[name]()
        kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
        q, bt = inp.q.to(dev), inp.block_tables.to(dev)
        cu, lk = inp.cu_seqlens_q.to(dev), inp.seq_lens_k.to(dev)
        T, Hq, D = inp.q.shape
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, inp.max_seqlen_q),
                         dtype=torch.uint8, device=dev)
        pgqa.kv_cache_write(inp.key.to(dev), inp.value.to(dev), inp.slot_mapping.to(dev), kc, vc,
                            dev_status=status)
        caches = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(ROTATIONS)]
        R = len(caches)
        if name == "speculative_verify":
            # every sequence verifies the same number of draft tokens: the multi-token
            # decode, whose (sequence, kv-head) query rows share each page read
            B, nq = inp.num_seqs, inp.max_seqlen_q
            q4, out4, lse4 = q.view(B, nq, Hq, D), out.view(B, nq, Hq, D), lse.view(B, nq, Hq)
            ws = torch.zeros(pgqa.decode_multi_workspace_size(B, nq, Hq, inp.key.shape[1], D),
                             dtype=torch.uint8, device=dev)

            def call(r):
                pgqa.paged_attention_decode_multi(out4, lse4, q4, caches[r][0], caches[r][1], bt,
                                                  lk, inp.scale, inp.max_seqlen_k,
                                                  workspace=ws, dev_status=status)
        else:
            def call(r):
                pgqa.paged_prefill_varlen_kv(out, lse, q, caches[r][0], caches[r][1], bt, cu, lk,
                                             inp.max_seqlen_q, inp.max_seqlen_k, inp.scale,
                                             workspace=ws, dev_status=status)

        for i in range(args.warmup):
            call(i % R)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        reps = 4 * R
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                call(i % R)
        g.replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(2, args.steps // 10)
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ms = e0.elapsed_time(e1) / (n * reps)
        flops = workloads.chunked_flops(inp)
        kvb = workloads.chunked_kv_bytes(inp)
        tflops = flops / (ms * 1e-3) / 1e12
        gbs = kvb / (ms * 1e-3) / 1e9
        fn = ("pgqa_paged_attention_decode_multi" if name == "speculative_verify"
              else "pgqa_paged_prefill_varlen_kv")
        entry = {"workload": inp.name, "ms": ms, "flops": flops, "TFLOP/s": tflops,
                 "kv_bytes": kvb, "KV GB/s": gbs, "launches_timed": n * reps,
                 "call": f"{fn}, a CUDA graph of back-to-back launches "
                         f"cycling over {R} copies of the cache at different addresses "
                         f"({R} x {kvb / 1e6:.0f} MB of K/V > 129 MB L2)"}
        if name == "chunked_prefill":
            entry["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": bf16_peak,
                                 "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                                 "peak_kind": kind + " bf16 burst (cuBLAS)",
                                 "traffic": _profile_traffic("prefill_chunked.json",
                                                             PREFILL_FILES)}
        else:
            entry["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                 "frac": gbs / hbm, "peak_kind": kind,
                                 "traffic": _profile_traffic("decode_spec_verify.json",
                                                             DECODE_FILES)}
        res[name] = entry
        del caches
        torch.cuda.empty_cache()
    return res


def measure_e4m3_prefill(args, dev):
    """The varlen causal prefill workload over an E4M3 cache (per-kv-head scales
    amax / 448, written once by the cache-write kernel), timed per launch with events
    like the bf16 prefill."""
    import paged_kv_gqa_10_gb300 as pgqa
    _, bf16_peak, kind = _peaks()
    inp = workloads.varlen_prefill()
    kc, vc, ks, vs = (t.to(dev) for t in workloads.e4m3_prefill_cache(inp))
    q, bt, cu = inp.q.to(dev), inp.block_tables.to(dev), inp.cu_seqlens.to(dev)
    T, Hq, D = inp.q.shape
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, inp.max_seqlen),
                     dtype=torch.uint8, device=dev)
    pgqa.kv_cache_write(inp.key.to(dev), inp.value.to(dev), inp.slot_mapping.to(dev), kc, vc,
                        k_scale=ks, v_scale=vs, dev_status=status)

    def call():
        pgqa.paged_prefill_varlen_e4m3(out, lse, q, kc, vc, bt, cu, None, inp.max_seqlen, 0,
                                       inp.scale, ks, vs, workspace=ws, dev_status=status)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    stream = torch.cuda.current_stream()
    n = max(20, args.steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    flops = workloads.causal_flops(inp.seq_lens, Hq, D)
    tflops = flops / (ms * 1e-3) / 1e12
    return {"workload": inp.name + ", E4M3 cache", "ms": ms, "flops": flops,
            "TFLOP/s": tflops, "launches_timed": n,
            "call": "pgqa_paged_prefill_varlen_e4m3, events around each launch",
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                         "peak_kind": kind + " bf16 burst (cuBLAS); the MMAs run on f16 "
                                             "operands at the same nominal rate",
                         "traffic": _profile_traffic("prefill_e4m3_varlen.json", PREFILL_FILES)}}


def measure_window_decode(args, dev, window=2048):
    """Sliding-window decode on the 70B-shaped batch (contexts U[1024, 4096], window
    2048 keys): a CUDA graph of back-to-back launches cycling over the rotating table
    sets (no launch finds the previous one's pages in L2), KV bytes of the window."""
    import paged_kv_gqa_10_gb300 as pgqa
    inp = workloads.llama70b_decode(rotations=ROTATIONS)
    b = DecodeBench(inp, dev)
    for r in range(b.R):
        b.append(r)
    elem = 2
    row = inp.num_kv_heads * inp.head_dim * elem * 2
    kvb = sum(min(L, window) for L in inp.context_lens.tolist()) * row

    def call(r):
        pgqa.paged_attention_decode_window(b.out, b.lse, b.q, b.kc, b.vc, b.bts[r], b.cl,
                                           inp.scale, window, inp.max_context_len,
                                           workspace=b.ws, dev_status=b.status)

    for i in range(args.warmup):
        call(i % b.R)
    b.check()
    n_rep = 4 * b.R
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_rep):
            call(i % b.R)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, args.steps // 4)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    b.check()
    ms = e0.elapsed_time(e1) / (reps * n_rep)
    gbs = kvb / (ms * 1e-3) / 1e9
    hbm, _, kind = _peaks()
    return {"workload": f"sliding-window decode, window {window}: " + inp.name, "ms": ms,
            "kv_bytes": kvb, "KV GB/s": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_kind": kind,
                         "traffic": _profile_traffic("decode_window.json", DECODE_FILES)}}


def _oracle_parity(inp, gpu_res):
    """One decode step's GPU output (out, lse arrays, or the text of the error that kept
    the GPU side from producing it) against the oracle over the cache with the step's
    new rows appended."""
    import oracle
    if isinstance(gpu_res, str):
        return {"error": gpu_res}
    dt = oracle.E4M3 if inp.cache_dtype == "e4m3" else oracle.BF16
    kc, vc = oracle.kv_cache_write(inp.step_key, inp.step_value, inp.step_slots, inp.k_cache,
                                   inp.v_cache, dtype=dt, k_scale=inp.k_scale,
                                   v_scale=inp.v_scale)
    ref_out, ref_lse = oracle.paged_decode(inp.q, kc, vc, inp.block_tables, inp.context_lens,
                                           inp.scale, threads=oracle.default_threads(),
                                           dtype=dt, k_scale=inp.k_scale, v_scale=inp.v_scale)
    return _parity_summary(gpu_res, ref_out, ref_lse)


def _gpu_step_result(b):
    """One more fused step on the first block-table set, read back for the oracle."""
    try:
        b.decode_append(0)
        b.check()
        return (b.out.float().cpu().numpy(), b.lse.cpu().numpy())
    except Exception as e:  # reported in the line, never fatal to it
        return f"GPU step failed: {e!r}"


def decode_entry(name, inp, m, world):
    """The numbers of one decode workload: step and kernel time, GB/s, roofline."""
    b = m["bench"]
    hbm_peak, _, peak_kind = _peaks()
    kvb = b.kv_bytes
    unique = workloads.kv_read_bytes(inp, unique=True)
    shared = kvb - unique  # bytes of shared blocks read more than once (prefix sharing)
    alg = b.alg_bytes_fused - shared
    achieved = alg / (m["dec_ms"] * 1e-3) / 1e9
    D = inp.head_dim
    e = {"workload": DECODE_WORKLOADS[name][1],
         "ms_per_step": m["ms_graph"],
         "GB/s": job_value(kvb, world, m["ms_graph"]),
         "kernel_ms": m["dec_ms"],
         "roofline": {"bound": "hbm",
                      "kernel": f"paged_decode_kernel<{D},{inp.cache_dtype}> with the append",
                      "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                      "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                      "alg_bytes_per_launch": alg, "launch_ms": m["dec_ms"],
                      "traffic": _profile_traffic(f"decode_{name}.json", DECODE_FILES)}}
    if shared:
        e["unique_kv_bytes_per_step"] = unique
        e["unique GB/s"] = job_value(unique, world, m["ms_graph"])
        e["GB/s_note"] = ("GB/s counts every sequence's context (logical bytes, effective "
                          "with L2 serving the shared blocks); unique GB/s and the roofline "
                          "count each shared block once")
    return e


def run_ours(args):
    dist, rank, local, world = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    names = [args.workload] + ([] if args.only else
                               [n for n in DECODE_ORDER if n != args.workload])
    decode = {}
    head = None
    for name in names:
        inp = DECODE_WORKLOADS[name][0]()
        full = name == args.workload
        m = measure_decode(inp, args, dev, dist, clocks_index=local if full else None,
                           full=full)
        entry = decode_entry(name, inp, m, world)
        if rank == 0 and not args.no_cpu_baseline:
            gpu_res = _gpu_step_result(m["bench"])
            if full:
                cpu = _cpu_baseline(inp, args.cpu_seconds, gpu_res)
                entry["parity"] = cpu["parity"]
            else:
                entry["parity"] = _oracle_parity(inp, gpu_res)
        decode[name] = entry
        if full:
            head = (inp, m, cpu if rank == 0 and not args.no_cpu_baseline else None)
        else:
            del m
            torch.cuda.empty_cache()
    inp, m, cpu = head
    pref = None if args.no_prefill else measure_prefill(args, dev)
    nxt = None
    if not args.no_prefill and not args.only:
        nxt = measure_cached_prefix(args, dev)
        nxt["sliding_window_decode"] = measure_window_decode(args, dev)
        nxt["e4m3_prefill"] = measure_e4m3_prefill(args, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    b = m["bench"]
    kv_bytes = b.kv_bytes
    value = job_value(kv_bytes, world, m["ms_graph"])
    dt = "e4m3 KV, bf16 q/out" if inp.cache_dtype == "e4m3" else "bf16"
    config = decode_config(args.workload, inp)
    config["parallelism"] = f"replica per GPU x{world}"
    head_entry = decode[args.workload]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_graph"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dt,
        "data": DATA, "config": config,
        "step": {"launch": "one launch of paged_attention_decode_append per step, replayed as "
                           f"CUDA graphs of {b.R} steps (one per block-table set)",
                 "eager_ms_per_step": m["ms_eager"],
                 "two_call_ms_per_step": m["ms_two"],
                 "two_call_value": kv_bytes * world / (m["ms_two"] * 1e-3) / 1e9},
        "roofline": head_entry["roofline"],
        "e2e": {"value": kv_bytes * world / (m["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                "ms_per_step": m["e2e_ms"],
                "calls": "eager C-ABI call per step (arguments marshalled once); inputs packed "
                         "in one pinned buffer (one host-to-device copy), out and lse read back "
                         "with one copy"},
        "gpu_launches": args.steps,
        "clocks": m["clocks"],
        "decode": decode,
    }
    if pref is not None:
        line["prefill"] = pref
    if nxt is not None:
        line["next"] = nxt
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


ROWS = (["decode:" + n for n in DECODE_ORDER] +
        ["prefill", "chunked_prefill", "speculative_verify", "sliding_window_decode",
         "e4m3_prefill"])


def run_row(args):
    """One row of the bench alone, printed as one JSON line: a profiling aid (an ncu
    capture of one row's kernel runs only that row's launches)."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    r = args.row
    if r.startswith("decode:"):
        name = r.split(":", 1)[1]
        inp = DECODE_WORKLOADS[name][0]()
        res = decode_entry(name, inp, measure_decode(inp, args, dev, full=False), 1)
    elif r == "prefill":
        res = measure_prefill(args, dev)
    elif r in ("chunked_prefill", "speculative_verify"):
        res = measure_cached_prefix(args, dev, names=(r,))[r]
    elif r == "sliding_window_decode":
        res = measure_window_decode(args, dev)
    else:
        res = measure_e4m3_prefill(args, dev)
    print(json.dumps({"row": r, **res}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default=DECODE_ORDER[0], choices=sorted(DECODE_WORKLOADS),
                    help="the headline decode workload (timed end to end, with the oracle "
                         "baseline); the others are measured beside it")
    ap.add_argument("--only", action="store_true",
                    help="measure the headline decode workload and the prefill only")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--row", choices=ROWS,
                    help="run one row of the bench alone and print its numbers (profiling aid)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.row:
        return run_row(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
