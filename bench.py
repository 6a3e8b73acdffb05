"""Benchmark: batched speculative-decoding verification on GB300.

Workload (the headline configuration): B=64 sequences, k=8 drafts,
V=128256, bf16 logits, temperature 0.7, stochastic verification (accept scan,
residual / bonus sampling).  Target logits ~ N(0, 4^2) - 1.1 ln(v+1), draft =
target + N(0, 1^2), draft tokens drawn from the draft softmax.  Synthetic,
seeded inputs; 279 MB of logits per step (larger than the 129 MB L2), and two
copies alternate between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is verified rows/s, B*(k+1) per step, from CUDA
events around K back-to-back calls (inputs resident in HBM); `e2e` repeats the
measurement through the public call with the inputs in pinned host memory,
the host->device copies and the device->host read of the result inside the
timed region.  `roofline` is for the dominant kernel (the row-statistics
pass), timed by events the library records around it on the launch stream.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead.

`--workload` selects a supplementary line for the other paths (one GPU):
c3_greedy (greedy on the C3 tensors), c3_greedy_match (the same with the
#Match outputs and stop-token truncation), c3_lenient (the headline with
lenience 2), c3_top_p / c3_top_k_top_p (the headline with consistent top-p
0.8, or top-k 50 then top-p 0.8), c4_guided (B=16 k=16 V=64000 greedy with a 24-token target
guide), c5_tree (B=8, 26-node trees, V=152064).  Inputs smaller than twice the
L2 rotate over enough device copies that every step reads from HBM.  These
steps are short next to the Python call that launches them, so they are
captured in a CUDA graph (the library launches on the capturing stream) and
the replays are timed.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified rows/s (B·(k+1)/s) and HBM GB/s vs GB300 peak, B=64 k=8 V=128256 bf16"
B, K, V, T, SEED, GEN_SEED = 64, 8, 128256, 0.7, 1234, 103
WORKLOAD = "C3 stochastic verification: B=64 k=8 V=128256 bf16 logits, T=0.7"
ELEM = 2  # bf16 bytes


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
            os.unlink(self.path)
        except Exception:
            return out
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=max(smax), reasons=sorted(reasons),
                       samples=len(sm))
        return out


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in ("spec_verify.cu", "spec_device.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_draft_online_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def captured_traffic():
    """DRAM bytes per row-pass launch from the committed ncu capture, or None when
    the kernel sources changed since that capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "row_pass_traffic.txt")) as f:
            fields = f.read().split()
        nbytes, sha = int(fields[2]), fields[4]
    except Exception:
        return None
    return nbytes if sha == kernel_source_hash() else None


def make_inputs():
    import workloads as wl
    return wl.c3(seed=GEN_SEED, verify_seed=SEED)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def _oracle_task(task):
    """One process of the oracle pool: verify sequences [lo, hi) of the stored workload."""
    paths, dtype, temperature, seed, lo, hi = task
    from oracle import verify as ov
    t, d, x = (np.load(q, mmap_mode="r") for q in paths)
    ov.verify_stochastic(np.asarray(t[lo:hi]), np.asarray(d[lo:hi]), np.asarray(x[lo:hi]), dtype, temperature, seed,
                         seq_offset=lo)
    return hi - lo


class OraclePool:
    """The oracle over sequences on all host cores: processes started with spawn
    (never forked from a process that holds a CUDA context), each reading the
    workload from .npy files it maps from a temporary folder."""

    def __init__(self, w):
        import multiprocessing
        self.w = w
        self.dir = tempfile.mkdtemp(prefix="oracle_")
        self.paths = []
        for name, a in (("t", w.target), ("d", w.draft), ("x", w.tokens)):
            q = os.path.join(self.dir, name + ".npy")
            np.save(q, a)
            self.paths.append(q)
        self.cores = os.cpu_count() or 1
        os.environ.setdefault("OMP_NUM_THREADS", "1")
        self.pool = multiprocessing.get_context("spawn").Pool(self.cores)
        self.pool.map(_oracle_task, [self.task(0, 1)] * self.cores)      # imports done in every process

    def task(self, lo, hi):
        return (self.paths, self.w.dtype, self.w.temperature, self.w.seed, lo, hi)

    def one_pass(self) -> int:
        """Every sequence of the workload once, one sequence per task; returns the sequences done."""
        return sum(self.pool.map(_oracle_task, [self.task(b, b + 1) for b in range(self.w.B)], chunksize=1))

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)


def cpu_oracle_run(w, seconds: float = 10.0):
    """Time the oracle on the host: all cores on whole passes over the workload's
    sequences (at least one, and up to about `seconds`), and one core on its
    first 8 sequences (about `seconds` / 2).  Returns the cpu_baseline object."""
    from oracle import verify as ov
    pool = OraclePool(w)
    try:
        seqs, t0 = 0, time.perf_counter()
        while True:
            seqs += pool.one_pass()
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    finally:
        pool.close()
    multi = seqs * (w.k + 1) / el
    nb = 8
    reps, t1 = 0, time.perf_counter()
    while True:
        ov.verify_stochastic(w.target[:nb], w.draft[:nb], w.tokens[:nb], w.dtype, w.temperature, w.seed)
        reps += 1
        el1 = time.perf_counter() - t1
        if el1 >= seconds / 2:
            break
    single = reps * nb * (w.k + 1) / el1
    return {"value": multi, "unit": "rows/s", "cores": pool.cores, "kind": "oracle",
            "sample": f"{seqs // w.B} passes over the workload's {w.B} sequences on {pool.cores} processes "
                      f"({el:.1f} s, fp64 numpy)",
            "single_core": {"value": single, "unit": "rows/s", "cores": 1,
                            "sample": f"{reps} x sequences 0..{nb - 1} in one process ({el1:.1f} s)"},
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args):
    """The CPU oracle as it stands, on the machine's host cores: each step verifies
    every sequence of the workload once, spread over all cores; the number of
    timed steps is capped so the whole run ends within about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = make_inputs()
    pool = OraclePool(w)
    try:
        for _ in range(min(args.warmup, 1)):
            pool.one_pass()
        t0 = time.perf_counter()
        pool.one_pass()
        per = time.perf_counter() - t0
        steps = max(1, min(args.steps, int(90.0 / max(per, 1e-3))))
        t_all = time.perf_counter()
        for _ in range(steps):
            pool.one_pass()
        el = time.perf_counter() - t_all
    finally:
        pool.close()
    value = steps * B * (K + 1) / el
    sample = (f"every sequence of the workload per step on {pool.cores} processes "
              f"({steps} of {args.steps} requested steps timed), fp64 numpy")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "k": K, "V": V, "temperature": T, "input_dtype": "bf16"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": pool.cores, "kind": "oracle", "sample": sample,
                         "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import speculative_decoding_draft_online_gb300 as sv

    w = make_inputs()
    tgt_np = w.target.view(np.int16)
    drf_np = w.draft.view(np.int16)
    copies = []
    for _ in range(2):
        copies.append((torch.from_numpy(tgt_np).to(dev).view(torch.bfloat16),
                       torch.from_numpy(drf_np).to(dev).view(torch.bfloat16)))
    tokens = torch.from_numpy(w.tokens).to(dev)
    stream = torch.cuda.current_stream(dev)
    ws = sv.workspace(B, K, V, sv.SPEC_BF16, dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)

    def step(i, events=None):
        t, d = copies[i & 1]
        # each replica draws the randomness of its own slice of an N*B-sequence batch
        sv.verify_ex(t, d, tokens, T, SEED, out_tokens=out, out_n=n, ws=ws, events=events,
                     sequence_offset=rank * B)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    n_host = n.cpu().numpy()
    resid_bytes = int(sum(2 * V * ELEM if nb < K else V * ELEM for nb in n_host))
    row_bytes = B * 2 * K * V * ELEM
    step_bytes = row_bytes + resid_bytes

    # --- device-timed region: K back-to-back calls (two launches each: the row
    # pass, then the sampling launch overlapping its tail)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    elapsed = start.elapsed_time(stop) / 1e3
    if world > 1:
        tt = torch.tensor([elapsed], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        elapsed = float(tt.item())
        torch.distributed.barrier()

    # --- per-kernel durations for the roofline: the library records events
    # before / after each launch (an event between the two launches also stops
    # them overlapping, so these steps are timed apart from the value above)
    nk = min(args.steps, 1000)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nk)]
    for evs in ev:                      # torch creates the CUDA event on first record
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(nk):
        step(i, ev[i])
    torch.cuda.synchronize()
    row_t = [e[0].elapsed_time(e[1]) for e in ev]
    call_t = [e[0].elapsed_time(e[3]) for e in ev]
    row_ms = statistics.mean(row_t)
    samp_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)

    def pct(xs):
        q = np.percentile(np.asarray(xs) * 1e3, [10, 50, 90])
        return {"p10_us": float(q[0]), "p50_us": float(q[1]), "p90_us": float(q[2])}
    rows_per_step = B * (K + 1)
    value = world * rows_per_step * args.steps / elapsed

    # --- end to end through the public call: pinned host inputs -> device -> verify -> host result
    h_t = torch.from_numpy(tgt_np).pin_memory()
    h_d = torch.from_numpy(drf_np).pin_memory()
    h_x = torch.from_numpy(w.tokens).pin_memory()
    h_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    d_t = torch.empty(tgt_np.shape, dtype=torch.int16, device=dev)
    d_d = torch.empty(drf_np.shape, dtype=torch.int16, device=dev)
    d_x = torch.empty(w.tokens.shape, dtype=torch.int32, device=dev)

    def e2e_step():
        d_t.copy_(h_t, non_blocking=True)
        d_d.copy_(h_d, non_blocking=True)
        d_x.copy_(h_x, non_blocking=True)
        sv.verify(d_t.view(torch.bfloat16), d_d.view(torch.bfloat16), d_x, T, SEED, out_tokens=out, out_n=n, ws=ws,
                  sequence_offset=rank * B)
        h_out.copy_(out, non_blocking=True)
        h_n.copy_(n, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    e2e_steps = max(5, min(50, args.steps // 20))
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_el = time.perf_counter() - t0
    if world > 1:
        tt = torch.tensor([e2e_el], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        e2e_el = float(tt.item())
    assert np.array_equal(h_n.numpy(), n_host), "e2e result differs from the device-resident run"
    h2d = h_t.numel() * 2 + h_d.numel() * 2 + h_x.numel() * 4
    d2h = h_out.numel() * 4 + h_n.numel() * 4

    peak, peak_kind = peaks()
    achieved = row_bytes / (row_ms / 1e3) / 1e9
    traffic = captured_traffic()

    line = None
    configs, probe = None, None
    if rank == 0 and world == 1 and not args.no_per_config:
        configs = per_config(dev, peaks()[0])
        probe = read_probe(dev)
    if rank == 0:
        cpu = cpu_oracle_run(w) if world == 1 and not args.no_cpu_baseline else None
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "k": K, "V": V, "temperature": T, "input_dtype": "bf16",
                       "l2": "inputs 279 MB > 129 MB L2; two copies alternate", "parallelism": f"replicas x{world}",
                       "step_bytes": step_bytes, "residual_bytes": resid_bytes,
                       "step_hbm_gbs": step_bytes / (elapsed / args.steps) / 1e9,
                       "row_pass_ms": row_ms, "sample_ms": samp_ms,
                       "row_pass_us_percentiles": pct(row_t), "evented_call_us_percentiles": pct(call_t),
                       "sample_bytes_l2_or_hbm": resid_bytes},
            "roofline": {"bound": "hbm", "kernel": "row_pass_kernel", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes": row_bytes},
            "e2e": {"value": rows_per_step * e2e_steps * world / e2e_el, "unit": "rows/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if configs is not None:
            line["config"]["per_config"] = configs
            line["roofline"]["read_probe_gbs"] = probe
            line["roofline"]["read_probe"] = ("spec_probe_read: the row pass's loads alone (persistent grid, "
                                              "16-byte no-L1 loads, 4 per thread in flight) over 2 GiB, best of 5")
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


L2_BYTES = 129 * 1024 * 1024


def graph_time(step, n_copies: int, target_steps: int = 480):
    """Seconds per step of `step(i)` (i = 0, 1, ...; the caller rotates n_copies
    input copies by i), captured in a CUDA graph of a multiple of n_copies steps
    and replayed until about target_steps steps; the library launches on the
    capturing stream.  Returns (seconds per step, steps timed)."""
    import torch
    for i in range(max(3, n_copies)):                  # warm, and the workspace prepared for these sizes
        step(i)
    torch.cuda.synchronize()
    per_graph = n_copies * max(1, 48 // n_copies)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    replays = max(1, target_steps // per_graph)
    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(replays):
        graph.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / 1e3 / (replays * per_graph), replays * per_graph


def per_config(dev, peak: float):
    """Device throughput of the five configurations: C1 tiny (fp32, stochastic and
    greedy), C2 (stochastic), C3 greedy (the headline tensors), C4 phrase drafts
    (a = 0.8, greedy) and C5 trees.  Each is a CUDA graph of consecutive calls
    over enough device copies of its inputs (target and draft alike) that every
    call reads its logits from HBM (more than twice the 129 MB L2 in total).
    `gbs` counts each call's algorithmic bytes: B*2k*V*s of row statistics plus
    the rows the draws read (2V*s per rejection, V*s per bonus, from the
    outputs) in stochastic mode, B*(k+1)*V*s greedy, B*(N+1)*V*s for trees."""
    import torch
    import speculative_decoding_draft_online_gb300 as sv
    import workloads as wl

    def dev_rows(a, dtype):
        a = np.ascontiguousarray(a)
        if dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    def measure(name, w, mode):
        elem = 2 if w.dtype == "bf16" else 4
        per_copy = w.target.nbytes + (w.draft.nbytes if mode == "stochastic" else 0)
        n_copies = max(2, -(-2 * L2_BYTES // per_copy) + 1)
        tgt = [dev_rows(w.target, w.dtype) for _ in range(n_copies)]
        drf = [dev_rows(w.draft, w.dtype) for _ in range(n_copies)] if mode == "stochastic" else None
        tokens = torch.from_numpy(np.ascontiguousarray(w.tokens)).to(dev)
        code = sv.SPEC_BF16 if w.dtype == "bf16" else sv.SPEC_FP32
        ws = sv.workspace(w.B, w.k, w.V, code, dev)
        parents = torch.from_numpy(w.parents).to(dev) if mode == "tree" else None
        out = torch.empty((w.B, w.k + 1), dtype=torch.int32, device=dev)
        n = torch.empty((w.B,), dtype=torch.int32, device=dev)

        def step(i):
            c = i % n_copies
            if mode == "stochastic":
                sv.verify(tgt[c], drf[c], tokens, w.temperature, w.seed, out_tokens=out, out_n=n, ws=ws)
            elif mode == "greedy":
                sv.verify(tgt[c], None, tokens, 0.0, 0, out_tokens=out, out_n=n, ws=ws)
            else:
                sv.verify_tree(tgt[c], tokens, parents, ws=ws)

        sec, steps = graph_time(step, n_copies)
        rows = w.B * (w.k + 1)
        if mode == "stochastic":
            sv.verify(tgt[0], drf[0], tokens, w.temperature, w.seed, out_tokens=out, out_n=n, ws=ws)
            torch.cuda.synchronize()
            nh = n.cpu().numpy()
            nbytes = w.B * 2 * w.k * w.V * elem + int(sum(2 * w.V * elem if x < w.k else w.V * elem for x in nh))
        else:
            nbytes = rows * w.V * elem
        gbs = nbytes / sec / 1e9
        del tgt, drf
        torch.cuda.empty_cache()
        return {"workload": name, "B": w.B, "k_or_N": w.k, "V": w.V, "dtype": w.dtype, "mode": mode,
                "us_per_step": sec * 1e6, "rows_per_s": rows / sec, "bytes_per_step": nbytes, "gbs": gbs,
                "frac_of_peak": gbs / peak, "steps": steps, "copies": n_copies}

    c3 = make_inputs()
    return [
        measure("C1 tiny B4 k4 V32000 fp32 T=1", wl.c1_tiny(), "stochastic"),
        measure("C1 tiny B4 k4 V32000 fp32, greedy", wl.c1_tiny(), "greedy"),
        measure("C2 B32 k5 V32000 bf16 T=1", wl.c2(), "stochastic"),
        measure("C3 B64 k8 V128256 bf16, greedy on the headline tensors", c3, "greedy"),
        measure("C4 B16 k16 V64000 bf16 greedy, a=0.8", wl.c4(0.8), "greedy"),
        measure("C5 B8 N26 V152064 bf16 greedy tree", wl.c5(), "tree"),
    ]


def read_probe(dev, nbytes: int = 2 << 30):
    """The read ceiling for the row pass's load pattern: the library's read
    probe (the row pass's loads and nothing else, as many CTAs as fit) over a
    2 GiB buffer, bytes / CUDA-event time, best of 5."""
    import torch
    import speculative_decoding_draft_online_gb300 as sv
    x = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev).uniform_()
    best = 0.0
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        sv.probe_read(x)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    del x
    torch.cuda.empty_cache()
    return best


VARIANTS = ("c3_greedy", "c3_greedy_match", "c3_lenient", "c3_top_p", "c3_top_k_top_p", "c4_guided", "c5_tree")


def run_variant(args):
    """A supplementary device-timed line for another path of the library."""
    import torch
    import speculative_decoding_draft_online_gb300 as sv
    import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = args.workload
    stops = None
    if name.startswith("c3"):
        w = make_inputs()
    elif name == "c4_guided":
        w, guide = wl.guided_drafts(0.8, 0.9, 24, seed=106)
    else:
        w = wl.c5()
    elem = 2 if w.dtype == "bf16" else 4
    rows = w.B * (w.k + 1)
    stochastic = name in ("c3_lenient", "c3_top_p", "c3_top_k_top_p")
    row_bytes = rows * w.V * elem if not stochastic else w.B * 2 * w.k * w.V * elem
    n_copies = max(2, -(-2 * L2_BYTES // max(1, w.target.nbytes)) + 1)

    def dev_logits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    copies = [dev_logits(w.target) for _ in range(n_copies)]
    draft = dev_logits(w.draft) if stochastic else None
    tokens = torch.from_numpy(w.tokens).to(dev)
    if name == "c3_greedy_match":
        stops = torch.tensor([2, 3, 128001], dtype=torch.int32, device=dev)
    if name == "c4_guided":
        guide_d = torch.from_numpy(guide).to(dev)
    if name == "c5_tree":
        parents = torch.from_numpy(w.parents).to(dev)

    ws = sv.workspace(w.B, w.k, w.V, sv.SPEC_BF16, dev)
    out = torch.empty((w.B, w.k + 1), dtype=torch.int32, device=dev)
    n = torch.empty((w.B,), dtype=torch.int32, device=dev)

    def step(i):
        t = copies[i % n_copies]
        if name == "c3_greedy":
            sv.verify(t, None, tokens, 0.0, 0, out_tokens=out, out_n=n, ws=ws)
        elif name == "c3_greedy_match":
            sv.verify_ex(t, None, tokens, 0.0, 0, out_tokens=out, out_n=n, ws=ws, match=True, committed=True,
                         stop_ids=stops)
        elif name == "c3_lenient":
            sv.verify_ex(t, draft, tokens, w.temperature, w.seed, out_tokens=out, out_n=n, ws=ws, lenience=2.0)
        elif name == "c3_top_p":
            sv.verify_ex(t, draft, tokens, w.temperature, w.seed, out_tokens=out, out_n=n, ws=ws, top_p=0.8)
        elif name == "c3_top_k_top_p":
            sv.verify_ex(t, draft, tokens, w.temperature, w.seed, out_tokens=out, out_n=n, ws=ws, top_k=50,
                         top_p=0.8)
        elif name == "c4_guided":
            sv.verify_guided(t, tokens, guide_d, ws=ws)
        else:
            sv.verify_tree(t, tokens, parents, ws=ws)

    for i in range(max(args.warmup, 3)):          # also leaves the workspace prepared for these sizes
        step(i)
    torch.cuda.synchronize()
    # one graph of n_copies * reps_per_graph steps, replayed until `steps` are done
    per_graph = n_copies * max(1, 48 // n_copies)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            step(i)
    replays = max(1, args.steps // per_graph)
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        start.record(stream)
        for _ in range(replays):
            graph.replay()
        stop.record(stream)
        torch.cuda.synchronize()
    elapsed = start.elapsed_time(stop) / 1e3
    args.steps = replays * per_graph
    peak, peak_kind = peaks()
    per_step = elapsed / args.steps
    gbs = row_bytes / per_step / 1e9
    line = {
        "metric": f"verified rows/s ({name})", "value": rows * args.steps / elapsed, "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "B": w.B, "k": w.k, "V": w.V, "input_dtype": w.dtype,
                   "timing": f"CUDA graph of {per_graph} steps, {replays} replays",
                   "l2": f"{n_copies} device copies rotate ({w.target.nbytes / 1e6:.1f} MB each)",
                   "row_bytes_per_step": row_bytes},
        "roofline": {"bound": "hbm", "kernel": "whole step" if stochastic else "row_pass_kernel",
                     "achieved": gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None, "algorithmic_bytes": row_bytes},
        "gpu_launches": (1 + stochastic + (name in ("c3_top_p", "c3_top_k_top_p"))) * args.steps,
        "clocks": clk.summary(),
        "supplementary": True,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-configuration lines")
    ap.add_argument("--workload", choices=("c3",) + VARIANTS, default="c3",
                    help="c3 is the headline; the others print a supplementary line (one GPU)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "c3":
        return run_variant(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
