"""Benchmark of the paged GQA attention hot path on GB300.

One step = one decode step of the Llama-3-8B-shaped batch (64 sequences, 32 query
/ 8 kv heads, head_dim 128, contexts uniform on [256, 1024], 16-token blocks
shuffled over an 8192-block pool): append the new token's K/V into the paged
cache (kv_cache_write) and run paged decode attention over every cached token.
The metric is decode KV-read GB/s: the K and V bytes of every cached token of
every kv-head, read once per step, divided by the step time.

Three block-table sets over disjoint physical blocks rotate from step to step, so
each step reads ~156 MB that the previous two steps did not touch (> the 129 MB
L2): the numbers are HBM numbers, not L2 numbers.

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
WORKLOAD = "Llama-3-8B decode: B=64, Hq=32, Hkv=8, D=128, block 16, ctx U[256,1024], pool 8192"
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


def _cpu_baseline(inp, target_s=10.0):
    """The oracle, as it stands, on the host cores: the whole batch, repeated
    until about target_s seconds of CPU work have been timed."""
    import oracle
    cores = oracle.default_threads()
    args = (inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    t0 = time.perf_counter()
    oracle.paged_decode(*args, threads=cores)
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_decode(*args, threads=cores)
    dt = (time.perf_counter() - t0) / reps
    gbs = workloads.kv_read_bytes(inp) / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the whole batch ({inp.num_seqs} sequences, "
                      f"{int(inp.context_lens.sum())} cached tokens) x {reps} repetitions, "
                      f"fp64 C oracle, OpenMP over (sequence, kv-head), {dt * reps:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm: the same workload, metric and unit, timed
    on the host cores (each step = the whole batch through the fp64 oracle)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import oracle
    inp = workloads.llama3_8b_decode()
    cores = oracle.default_threads()
    a = (inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    for _ in range(args.warmup):
        oracle.paged_decode(*a, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_decode(*a, threads=cores)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    v = workloads.kv_read_bytes(inp) / dt / 1e9
    sample = f"whole batch per step ({int(inp.context_lens.sum())} cached tokens)"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import paged_kv_gqa_10_gb300 as pgqa

    dist, rank, local, world = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    inp = workloads.llama3_8b_decode(rotations=ROTATIONS)
    tables = [inp.block_tables] + inp.rotations
    slots = [inp.step_slots] + inp.rotation_slots
    R = len(tables)
    B, Hq, D = inp.q.shape
    Hkv = inp.num_kv_heads
    kc, vc = inp.k_cache.to(dev), inp.v_cache.to(dev)
    q = inp.q.to(dev)
    cl = inp.context_lens.to(dev)
    bts = [t.to(dev) for t in tables]
    sls = [s.to(dev) for s in slots]
    nk, nv = inp.step_key.to(dev), inp.step_value.to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws_n = pgqa.decode_workspace_size(B, Hq, Hkv, D, inp.max_context_len)
    ws = torch.zeros(max(ws_n, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    maxctx = inp.max_context_len

    def step(i, ev=None):
        r = i % R
        pgqa.kv_cache_write(nk, nv, sls[r], kc, vc, dev_status=status)
        if ev is not None:
            ev[0].record(stream)
        pgqa.paged_attention_decode(out, lse, q, kc, vc, bts[r], cl, inp.scale, maxctx,
                                    workspace=ws if ws_n else None, dev_status=status)
        if ev is not None:
            ev[1].record(stream)

    kv_bytes = workloads.kv_read_bytes(inp)
    # algorithmic bytes of one decode launch: KV once + q + out + lse + table entries + lens
    nblk = int(((inp.context_lens + 15) // 16).sum())
    alg_bytes = kv_bytes + q.numel() * 2 + out.numel() * 2 + lse.numel() * 4 + nblk * 4 + B * 4

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i, kev[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    dec_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    ms_step = ms / args.steps
    value = kv_bytes * world / (ms_step * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers
    pin = lambda t: t.pin_memory()
    h_q, h_k, h_v, h_cl = pin(inp.q), pin(inp.step_key), pin(inp.step_value), pin(inp.context_lens)
    h_bt = [pin(t) for t in tables]
    h_sl = [pin(s) for s in slots]
    h_out = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    d_bt = torch.empty_like(bts[0])
    d_sl = torch.empty_like(sls[0])

    def e2e_step(i):
        r = i % R
        q.copy_(h_q, non_blocking=True)
        nk.copy_(h_k, non_blocking=True)
        nv.copy_(h_v, non_blocking=True)
        cl.copy_(h_cl, non_blocking=True)
        d_bt.copy_(h_bt[r], non_blocking=True)
        d_sl.copy_(h_sl[r], non_blocking=True)
        pgqa.kv_cache_write(nk, nv, d_sl, kc, vc, dev_status=status)
        pgqa.paged_attention_decode(out, lse, q, kc, vc, d_bt, cl, inp.scale, maxctx,
                                    workspace=ws if ws_n else None, dev_status=status)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_cl, h_bt[0], h_sl[0]))
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if dist:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = kv_bytes * world / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        return 0
    hbm_peak, _, peak_kind = _peaks()
    achieved = alg_bytes / (dec_ms * 1e-3) / 1e9
    dec_files = ["paged_kv_gqa_10_gb300/csrc/decode.cu", "paged_kv_gqa_10_gb300/csrc/ptx.cuh"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/K/V, seeded shuffled block tables)",
        "config": {"workload": WORKLOAD, "batch": B, "q_heads": Hq, "kv_heads": Hkv,
                   "head_dim": D, "block_size": 16, "kv_bytes_per_step": kv_bytes,
                   "step": "kv_cache_write(64 new tokens) + paged_attention_decode",
                   "l2": f"{R} rotating block-table sets over disjoint blocks "
                         f"({R * kv_bytes / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replica per GPU x{world}"},
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel<128,bf16>",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                     "alg_bytes_per_launch": alg_bytes, "launch_ms": dec_ms,
                     "traffic": _profile_traffic("decode_llama3_8b.json", dec_files)},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
