"""Benchmark of the PLE n-gram row-id hash on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over
one batch, through the C ABI: each token's (request, offset) found from
cu_seqlens and the row-id hash of every layer, in one launch
(ple_row_ids_ex with req = local = NULL and cu_seqlens).  The same step as
two launches -- ple_build_token_index writing the index, then ple_row_ids
reading it -- is timed beside it.  The
workload is the large prefill: T=262144 tokens in 4 requests, ngram_size 4,
4 heads per order (12 heads), 8 layers, int64 ids, 20% adversarial boundary
runs.  Inputs are resident in HBM before the timed region; 64 distinct input
sets rotate (256 MiB of inputs) and two output buffers alternate (201 MB of
row ids written per step), so no step finds its inputs in the 126 MB L2.

Also measured, as extra keys: the row-id kernel's duration (the step's one
launch, CUDA events on its stream) against the HBM roofline, the end-to-end
rate with host buffers (pinned H2D of ids / cu_seqlens / context, the call,
D2H of all row ids), the decode B=1 device time per call (a CUDA graph of 300
calls, median of 7 replays), and the CPU oracle on the host cores.

--impl reference times the CPU oracle (the only reference this path has) on
bounded samples of the same workload.

Under torchrun (--gpus N > 1) every rank hashes its own seeded batch (weak
scaling, no collective on the data path); the step time is the max over
ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "row-ids/sec and % HBM roofline at large prefill; device µs/call at decode B=1"
UNIT = "row-ids/s"
L2_BYTES = 126 * 2 ** 20
ROTATE = 64
KERNEL_SOURCES = ["ple_rowids_common.cuh", "ple_rowids_fixed.cu", "ple_divmod.cuh", "ple_internal.h"]
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "row_ids_prefill_262144_traffic.json")


def _code_only(text: str) -> str:
    """The source without comments and blank lines: a comment edit leaves
    the kernel, and so its recorded traffic, unchanged."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "layer_gram_embedding_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def workload_config(batch: wl.Batch, extra=None):
    cfg = {
        "workload": (f"{batch.name}: T={batch.num_tokens} in {batch.num_requests} requests, "
                     f"ngram_size={batch.ngram_size}, heads_per_ngram={batch.heads_per_ngram} "
                     f"(H={batch.num_heads}), L={batch.num_layers} layers, "
                     f"{batch.ids.dtype.name} ids, 20% boundary runs"),
        "num_tokens": batch.num_tokens,
        "num_requests": batch.num_requests,
        "ngram_size": batch.ngram_size,
        "heads_per_ngram": batch.heads_per_ngram,
        "num_heads": batch.num_heads,
        "num_layers": batch.num_layers,
        "ids_dtype": batch.ids.dtype.name,
        "row_ids_per_step": batch.row_ids_per_call,
        "launches_per_step": 2,
    }
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_on(self):
        self.t_on = time.monotonic()

    def mark_off(self):
        self.t_off = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        window = [r for t, r in rows if self.t_on and self.t_off and self.t_on <= t <= self.t_off]
        used = window if window else [r for _, r in rows]
        sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(window)}


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling; no data-path collective)


class Dist:
    def __init__(self, backend: str | None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1 and backend:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline


def oracle_rate(batch: wl.Batch, budget_s: float):
    """Row ids/s of the oracle (index + hash) on the host, single-threaded:
    contiguous token samples of the workload (the whole batch when it is
    cheap enough), repeated until about budget_s seconds of CPU work."""
    import oracle

    def run(b):
        req, local = oracle.token_index(b.cu_seqlens, b.num_requests, b.num_tokens, b.is_decode)
        oracle.row_ids(b.ids, req, local, b.ngram_context, b.layer_multipliers, b.vocab_sizes,
                       b.offsets, b.ngram_size, b.heads_per_ngram, b.boundary_id)

    probe = wl.slice_batch(batch, 0, min(8192, batch.num_tokens))
    t = time.perf_counter()
    run(probe)
    per_token = max(time.perf_counter() - t, 1e-6) / probe.num_tokens
    n = int(min(batch.num_tokens, max(1024, budget_s / per_token)))
    sample = wl.slice_batch(batch, 0, n)
    reps, dt = 0, 0.0
    while dt < budget_s and reps < 1000:
        t = time.perf_counter()
        run(sample)
        dt += time.perf_counter() - t
        reps += 1
    return sample.row_ids_per_call * reps / dt, sample, dt, reps


_ALL_CORES_BARRIER = None


def _all_cores_init(barrier):
    global _ALL_CORES_BARRIER
    _ALL_CORES_BARRIER = barrier


def _oracle_slice_worker(job):
    """One host process of the all-cores oracle run: tokens [a, b) of the
    large prefill (a slice with its carried context), index + row ids
    repeated for about `budget` seconds after every process is ready.
    Returns (row ids hashed, seconds)."""
    a, b, budget = job
    import oracle

    s = wl.slice_batch(wl.prefill_262144(), a, b)
    _ALL_CORES_BARRIER.wait(timeout=120)  # a process that never starts breaks it
    rows, dt = 0, 0.0
    while dt < budget:
        t = time.perf_counter()
        req, local = oracle.token_index(s.cu_seqlens, s.num_requests, s.num_tokens, False)
        oracle.row_ids(s.ids, req, local, s.ngram_context, s.layer_multipliers, s.vocab_sizes,
                       s.offsets, s.ngram_size, s.heads_per_ngram, s.boundary_id)
        dt += time.perf_counter() - t
        rows += s.row_ids_per_call
    return rows, dt


def host_cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_rate_all_cores(batch: wl.Batch, budget_s: float, n_tok: int):
    """Row ids/s of the unchanged oracle on every host core at once: one
    process per core (spawned: the parent has used the GPU), each on an
    n_tok-token slice of the workload (spread over it when n_tok < T), all
    released together; the rate is the sum of the processes' rates while
    they ran side by side."""
    import multiprocessing as mp

    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    step = max(1, (batch.num_tokens - n_tok) // max(1, cores - 1))
    jobs = [(min(i * step, batch.num_tokens - n_tok), min(i * step, batch.num_tokens - n_tok) +
             n_tok, budget_s) for i in range(cores)]
    barrier = ctx.Barrier(cores)
    pool = ctx.Pool(cores, initializer=_all_cores_init, initargs=(barrier,))
    try:
        # bounded: a worker that cannot start must not stall the benchmark
        res = pool.map_async(_oracle_slice_worker, jobs, chunksize=1).get(
            timeout=180 + 4 * budget_s)
    except Exception as e:  # noqa: BLE001 -- reported, not raised
        pool.terminate()
        return None, f"{type(e).__name__}: {e}"
    pool.close()
    pool.join()
    return sum(r / dt for r, dt in res), cores


def reference_arm(args):
    dist = Dist(None)
    if dist.rank != 0:
        return 0
    batch = wl.prefill_262144()
    # calibrate the sample so that warmup + steps fit in about two minutes
    import oracle
    oracle.build()
    rate, _, _, _ = oracle_rate(batch, 0.5)
    per_step_s = min(30.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    n_tok = int(min(batch.num_tokens, max(256, per_step_s * rate / (batch.num_layers *
                                                                       batch.num_heads))))
    starts = [(i * 9973) % max(1, batch.num_tokens - n_tok + 1) for i in range(args.steps +
                                                                             args.warmup)]

    def step(i):
        s = wl.slice_batch(batch, starts[i], starts[i] + n_tok)
        req, local = oracle.token_index(s.cu_seqlens, s.num_requests, s.num_tokens, False)
        t = time.perf_counter()
        oracle.row_ids(s.ids, req, local, s.ngram_context, s.layer_multipliers, s.vocab_sizes,
                       s.offsets, s.ngram_size, s.heads_per_ngram, s.boundary_id)
        oracle.token_index(s.cu_seqlens, s.num_requests, s.num_tokens, False)
        return time.perf_counter() - t, s.row_ids_per_call

    for i in range(args.warmup):
        step(i)
    total_t, total_rows = 0.0, 0
    for i in range(args.warmup, args.warmup + args.steps):
        dt, rows = step(i)
        total_t += dt
        total_rows += rows
    value = total_rows / total_t
    sample = (f"{args.steps} contiguous samples of {n_tok} tokens of {batch.name} (carried "
              f"context at each cut), index build + row ids per sample")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": workload_config(batch, {"reference": "CPU oracle (plain C, single thread), "
                                                       "the only reference this path has",
                                          "sample_tokens_per_step": n_tok}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm


def our_arm(args):
    import torch

    import layer_gram_embedding_gb300 as ple
    from layer_gram_embedding_gb300 import build as lib_build

    dist = Dist("nccl")
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    lib_build.build()
    lib = ple.lib()
    stream = torch.cuda.current_stream(device)
    sh = ctypes.c_void_p(stream.cuda_stream)

    # ---- inputs, resident in HBM: ROTATE seeded batches sharing the model's parameters
    base = wl.prefill_262144(replay=1000 * dist.rank)
    batches = [base] + [wl.prefill_262144(replay=1000 * dist.rank + r) for r in range(1, ROTATE)]
    T, B, N, hpn, L, H = (base.num_tokens, base.num_requests, base.ngram_size,
                          base.heads_per_ngram, base.num_layers, base.num_heads)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    M, vocab, off = to_dev(base.layer_multipliers), to_dev(base.vocab_sizes), to_dev(base.offsets)
    sets = []
    for b in batches:
        sets.append(dict(ids=to_dev(b.ids), ctx=to_dev(b.ngram_context), cu=to_dev(b.cu_seqlens),
                         req=torch.empty(T, dtype=torch.int32, device=device),
                         local=torch.empty(T, dtype=torch.int32, device=device)))
    outs = [torch.empty((L, T, H), dtype=torch.int64, device=device) for _ in range(2)]
    P = ctypes.c_void_p
    idx_args, row_args, search_args = [], [], []
    for k, s in enumerate(sets):
        idx_args.append((P(s["cu"].data_ptr()), B, T, 0, P(s["req"].data_ptr()),
                         P(s["local"].data_ptr()), sh))
        row_args.append((P(s["ids"].data_ptr()), ple.PLE_I64, T, P(s["req"].data_ptr()),
                         P(s["local"].data_ptr()), P(s["ctx"].data_ptr()), B, N - 1,
                         P(M.data_ptr()), P(vocab.data_ptr()), P(off.data_ptr()), H, N, hpn, L,
                         base.boundary_id, P(outs[k % 2].data_ptr()), sh))
        # the whole step in one launch: req = local = NULL with cu_seqlens,
        # each token's request found in the kernel
        search_args.append((P(s["ids"].data_ptr()), ple.PLE_I64, T, None, None,
                            P(s["ctx"].data_ptr()), B, N - 1, P(M.data_ptr()),
                            P(vocab.data_ptr()), P(off.data_ptr()), H, N, hpn, L,
                            base.boundary_id, P(outs[k % 2].data_ptr()), ple.PLE_I64,
                            P(s["cu"].data_ptr()), None, None, sh))
    f_idx, f_rows, f_search = lib.ple_build_token_index, lib.ple_row_ids, lib.ple_row_ids_ex

    def step(i):
        if f_search(*search_args[i % ROTATE]):
            raise RuntimeError("library call failed")

    def step_with_index(i):
        k = i % ROTATE
        st = f_idx(*idx_args[k]) | f_rows(*row_args[k])
        if st:
            raise RuntimeError(f"library call failed: status {st}")

    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(visible.split(",")[dist.local_rank].strip() if visible else
                          str(dist.local_rank))
    clocks.start()
    for i in range(args.warmup):
        step(i)
        step_with_index(i)
    torch.cuda.synchronize(device)

    # ---- the timed region: K steps back to back, events only at its ends
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(device)
    clocks.mark_on()
    t_start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    dist.barrier()
    total_ms = t_start.elapsed_time(t_end)

    # ---- the step as two launches (ple_build_token_index, then ple_row_ids
    # reading the index), K steps back to back, for comparison
    w_start = torch.cuda.Event(enable_timing=True)
    w_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    w_start.record(stream)
    for i in range(args.steps):
        step_with_index(args.warmup + i)
    w_end.record(stream)
    torch.cuda.synchronize(device)
    with_index_ms = w_start.elapsed_time(w_end) / args.steps
    # the step's one kernel with an event pair around every launch, for
    # reference (an event between launches serialises them and adds its own
    # drain-and-launch gap to every launch)
    n_br = min(args.steps, 200)
    br = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_br)]
    for i in range(n_br):
        br[i][0].record(stream)
        step(i)
        br[i][1].record(stream)
    torch.cuda.synchronize(device)
    clocks.mark_off()
    bracketed_ms = float(np.median([a.elapsed_time(b) for a, b in br]))
    # the step is one launch, so the dominant kernel's average duration is the
    # step's, measured over the timed region on the launching stream
    kern_avg_ms = total_ms / args.steps
    total_ms = dist.max(total_ms, device)
    clk = clocks.stop()

    rows_per_step = base.row_ids_per_call
    value = dist.world * rows_per_step * args.steps / (total_ms / 1e3)
    idb = base.ids.dtype.itemsize
    # ids and cu_seqlens read, context and parameters read, row ids written
    kernel_bytes = (T * (idb + 8 * L * H) + 4 * (B + 1) + B * (N - 1) * idb +
                    8 * L * (N + 2 * H))
    peaks, peak_kind = measured_peaks()
    achieved = kernel_bytes / (kern_avg_ms / 1e3) / 1e9
    traffic = None
    try:
        with open(PROFILE_TRAFFIC) as fh:
            prof = json.load(fh)
        if prof.get("kernel_source_sha256_16") == kernel_source_hash():
            traffic = prof.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": "ple row_ids kernel (row_ids_fixed_kernel<int64, 4, 4>, requests "
                          "found from cu_seqlens in the kernel)",
                "algorithmic_bytes_per_launch": kernel_bytes,
                "kernel_ms_avg": kern_avg_ms,
                "kernel_timing": f"the timed region: {args.steps} one-launch steps back to back, "
                                 "CUDA events at its ends, on the launching stream",
                "kernel_ms_bracketed_median": bracketed_ms,
                "peak_kind": peak_kind}

    # ---- end to end through the public Python API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, ple, torch, device, stream, batches[:4], M, vocab, off)

    decode = None if args.no_decode else decode_latency(ple, torch, device)

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rate, sample, dt, reps = oracle_rate(base, args.cpu_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"tokens [0, {sample.num_tokens}) of {base.name}, index + row ids, "
                         f"{reps} runs, {dt:.1f} s on one thread", "host_cores": os.cpu_count(),
               "host_cpu": host_cpu_model()}
        if not args.no_all_cores:
            all_rate, cores = oracle_rate_all_cores(base, min(8.0, args.cpu_budget),
                                                    sample.num_tokens)
            if all_rate is None:
                cpu["all_cores"] = {"unavailable": cores}
            else:
                cpu["all_cores"] = {
                    "value": all_rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                    "sample": f"{cores} processes at once, each hashing a {sample.num_tokens}-token "
                              f"slice of {base.name} (index + row ids) for about "
                              f"{min(8.0, args.cpu_budget):.0f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": workload_config(base, {
            "l2": f"inputs rotate over {ROTATE} seeded sets ({ROTATE * (T * 16 + 64) >> 20} MiB) "
                  f"and 2 output buffers ({L * T * H * 8 / 1e6:.0f} MB written per step); "
                  "no step's data fits the 126 MB L2",
            "parallelism": f"replicas x{dist.world} (weak scaling, no collective)"}),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "step": "one launch: ple_row_ids_ex with req = local = NULL and cu_seqlens",
        "step_with_index_build": {
            "launches": 2, "ms_per_step": with_index_ms,
            "value": dist.world * rows_per_step / (with_index_ms / 1e3), "unit": UNIT,
            "what": "ple_build_token_index then ple_row_ids reading the index, back to back"},
        "clocks": clk,
        "decode_b1": decode,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def end_to_end(args, ple, torch, device, stream, batches, M, vocab, off):
    """The same metric through ple_row_ids (the Python binding; requests
    found from cu_seqlens in the kernel) with host buffers: every step copies
    its ids, cu_seqlens and context from pinned host memory, runs the call,
    and copies every row id back to pinned host memory.

    Steps are pipelined over two buffer slots, as a serving loop would run
    them: step i's device-to-host copy runs on a second stream while step
    i + 1's host-to-device copy and kernel run on the launching stream; a
    slot is reused only after its previous copy back has finished.  The
    timed region ends when the last step's rows are in host memory.  The
    same steps run one after another on one stream are reported beside it."""
    b0 = batches[0]
    T, B, L, H = b0.num_tokens, b0.num_requests, b0.num_layers, b0.num_heads
    host = []
    for b in batches:
        host.append(dict(ids=torch.from_numpy(b.ids).pin_memory(),
                         cu=torch.from_numpy(b.cu_seqlens).pin_memory(),
                         ctx=torch.from_numpy(np.ascontiguousarray(b.ngram_context)).pin_memory()))
    slots = []
    for _ in range(2):
        slots.append(dict(
            ids=torch.empty(T, dtype=torch.int64, device=device),
            cu=torch.empty(B + 1, dtype=torch.int32, device=device),
            ctx=torch.empty((B, b0.ngram_size - 1), dtype=torch.int64, device=device),
            out=torch.empty((L, T, H), dtype=torch.int64, device=device),
            h_out=torch.empty((L, T, H), dtype=torch.int64).pin_memory(),
            computed=torch.cuda.Event(), copied=torch.cuda.Event()))
    steps = max(3, min(args.steps, 100))
    h2d = T * 8 + (B + 1) * 4 + B * (b0.ngram_size - 1) * 8
    d2h = L * T * H * 8
    d2h_stream = torch.cuda.Stream(device)

    def run(i, pipelined):
        h, sl = host[i % len(host)], slots[i % 2 if pipelined else 0]
        if pipelined:
            stream.wait_event(sl["copied"])  # the slot's previous rows are in host memory
        sl["ids"].copy_(h["ids"], non_blocking=True)
        sl["cu"].copy_(h["cu"], non_blocking=True)
        sl["ctx"].copy_(h["ctx"], non_blocking=True)
        ple.ple_row_ids(sl["ids"], None, None, sl["ctx"], M, vocab, off, b0.ngram_size,
                        b0.heads_per_ngram, b0.boundary_id, out=sl["out"], cu_seqlens=sl["cu"])
        if pipelined:
            sl["computed"].record(stream)
            d2h_stream.wait_event(sl["computed"])
            with torch.cuda.stream(d2h_stream):
                sl["h_out"].copy_(sl["out"], non_blocking=True)
            sl["copied"].record(d2h_stream)
        else:
            sl["h_out"].copy_(sl["out"], non_blocking=True)

    def timed(pipelined):
        for i in range(3):
            run(i, pipelined)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            run(i, pipelined)
        if pipelined:
            stream.wait_stream(d2h_stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1)

    ms_serial = timed(False)
    ms = timed(True)
    return {"value": b0.row_ids_per_call * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "method": "two buffer slots; each step's device-to-host copy overlaps the next "
                      "step's host-to-device copy and kernel",
            "serial_ms_per_step": ms_serial / steps,
            "serial_value": b0.row_ids_per_call * steps / (ms_serial / 1e3)}


def decode_latency(ple, torch, device):
    """Device µs per call of ple_row_ids at decode B=1: a CUDA graph of 300
    back-to-back calls, median of 7 replays (the page's 7 x 300 method).
    Measured without an index (req = local = NULL, one launch per step) and
    with a prebuilt index (the page's memoized index), each with the head
    constants derived in the call (the page's arguments) and prepared once
    by ple_prepare_heads (model parameters, fixed across steps)."""
    b = wl.decode(1)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    ids, ctx = to_dev(b.ids), to_dev(b.ngram_context)
    M, vocab, off = to_dev(b.layer_multipliers), to_dev(b.vocab_sizes), to_dev(b.offsets)
    req, local = ple.ple_build_token_index(None, 1, 1, True, device=device)
    heads = ple.ple_prepare_heads(vocab, off)
    out = torch.empty((1, 1, 4), dtype=torch.int64, device=device)
    res = {"launches_per_call": 1, "method": "CUDA graph of 300 calls, median of 7 replays"}
    for name, (rq, lc, hd) in (("device_us_per_call", (None, None, None)),
                               ("device_us_per_call_with_index", (req, local, None)),
                               ("device_us_per_call_prepared_heads", (None, None, heads)),
                               ("device_us_per_call_with_index_prepared_heads",
                                (req, local, heads))):
        def call():
            ple.ple_row_ids(ids, rq, lc, ctx, M, vocab, off, 3, 2, b.boundary_id, out=out,
                            heads=hd)

        s = torch.cuda.Stream(device)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            call()
        torch.cuda.current_stream(device).wait_stream(s)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        calls = 300
        with torch.cuda.graph(g):
            for _ in range(calls):
                call()
        g.replay()
        torch.cuda.synchronize(device)
        per_call = []
        for _ in range(7):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize(device)
            per_call.append(1e3 * e0.elapsed_time(e1) / calls)
        res[name] = statistics.median(per_call)
        if name == "device_us_per_call":
            res["runs_us"] = per_call
    return res


def all_configs(args):
    """Every workload: device time per call of ple_row_ids and of a whole
    step (index + row ids), each from a CUDA graph of 300 back-to-back calls,
    median of 7 replays (the page's 7 x 300 method); one JSON object."""
    import torch

    import layer_gram_embedding_gb300 as ple
    from layer_gram_embedding_gb300 import build as lib_build

    lib_build.build()
    device = torch.device("cuda", 0)
    peaks, _ = measured_peaks()
    out = []
    for batch in wl.all_workloads():
        wname = batch.name + ("_i32" if batch.ids.dtype == np.int32 else "")
        if args.only and wname not in args.only:
            continue

        def to_dev(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        T, B, L, H = batch.num_tokens, batch.num_requests, batch.num_layers, batch.num_heads
        ids, ctx = to_dev(batch.ids), to_dev(batch.ngram_context)
        M, vocab, off = (to_dev(batch.layer_multipliers), to_dev(batch.vocab_sizes),
                         to_dev(batch.offsets))
        cu = to_dev(batch.cu_seqlens) if batch.cu_seqlens is not None else None
        req = torch.empty(T, dtype=torch.int32, device=device)
        local = torch.empty(T, dtype=torch.int32, device=device)
        o = torch.empty((L, T, H), dtype=torch.int64, device=device)
        o32 = torch.empty((L, T, H), dtype=torch.int32, device=device)
        # the row-id variants read a built index, as a serving step would
        ple.ple_build_token_index(cu, B, T, batch.is_decode, req=req, local=local)

        def rows():
            ple.ple_row_ids(ids, req, local, ctx, M, vocab, off, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, out=o)

        def rows_i32():
            ple.ple_row_ids(ids, req, local, ctx, M, vocab, off, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, out=o32,
                            out_dtype=torch.int32)

        def rows_no_index():
            ple.ple_row_ids(ids, None, None, ctx, M, vocab, off, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, out=o)

        heads = ple.ple_prepare_heads(vocab, off)

        def rows_prepared():
            ple.ple_row_ids(ids, req, local, ctx, M, vocab, off, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, out=o, heads=heads)

        def one_launch_step():
            # no index: a prefill's requests found from cu_seqlens in the
            # kernel, a decode's synthesised (req = t, local = 0)
            ple.ple_row_ids(ids, None, None, ctx, M, vocab, off, batch.ngram_size,
                            batch.heads_per_ngram, batch.boundary_id, out=o, cu_seqlens=cu)

        def step():
            ple.ple_build_token_index(cu, B, T, batch.is_decode, req=req, local=local)
            rows()

        res = {"workload": wname,
               "T": T, "B": B, "L": L, "H": H, "ngram_size": batch.ngram_size,
               "row_ids_per_call": batch.row_ids_per_call,
               "algorithmic_bytes": batch.algorithmic_bytes(), "launches_per_call": 1}
        variants = [("row_ids", rows), ("step", step), ("step_one_launch", one_launch_step),
                    ("row_ids_i32", rows_i32), ("row_ids_prepared_heads", rows_prepared)]
        if batch.is_decode:
            variants.append(("row_ids_no_index", rows_no_index))
        for name, fn in variants:
            s = torch.cuda.Stream(device)
            s.wait_stream(torch.cuda.current_stream(device))
            with torch.cuda.stream(s):
                fn()
            torch.cuda.current_stream(device).wait_stream(s)
            torch.cuda.synchronize(device)
            g = torch.cuda.CUDAGraph()
            calls = 300
            with torch.cuda.graph(g):
                for _ in range(calls):
                    fn()
            g.replay()
            torch.cuda.synchronize(device)
            runs = []
            for _ in range(7):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize(device)
                runs.append(1e3 * e0.elapsed_time(e1) / calls)
            us = statistics.median(runs)
            res[f"{name}_us"] = us
            del g
        res["row_ids_per_s"] = batch.row_ids_per_call / (res["step_us"] / 1e6)
        res["row_ids_per_s_one_launch"] = batch.row_ids_per_call / (res["step_one_launch_us"] / 1e6)
        res["kernel_gbs"] = batch.algorithmic_bytes() / (res["row_ids_us"] / 1e6) / 1e9
        res["kernel_frac_of_measured_hbm"] = res["kernel_gbs"] / peaks["hbm_gbs"]
        bytes32 = batch.algorithmic_bytes() - 4 * L * T * H
        res["i32_algorithmic_bytes"] = bytes32
        res["i32_kernel_gbs"] = bytes32 / (res["row_ids_i32_us"] / 1e6) / 1e9
        res["i32_kernel_frac_of_measured_hbm"] = res["i32_kernel_gbs"] / peaks["hbm_gbs"]
        out.append(res)
        print(json.dumps(res), file=sys.stderr, flush=True)
    print(json.dumps({"all_configs": out, "method": "CUDA graph of 300 back-to-back calls, "
                      "median of 7 replays; step = ple_build_token_index + ple_row_ids; "
                      "step_one_launch = ple_row_ids without an index (cu_seqlens searched in "
                      "the kernel for a prefill, req = t for a decode)"}))
    return 0


def embed_bench(args):
    """The fused table gather on the large-prefill shape: a 256-wide bfloat16
    table per layer with one row per head vocabulary entry (about 7.1 M rows,
    29 GB over 8 layers), one JSON line with the gather's HBM rate."""
    import torch

    import layer_gram_embedding_gb300 as ple
    from layer_gram_embedding_gb300 import build as lib_build

    lib_build.build()
    device = torch.device("cuda", 0)
    b = wl.prefill_262144()
    if args.embed_layers < b.num_layers:
        # fewer layers keep a profiling capture within a few GB of table
        k = max(1, args.embed_layers)
        b = wl.replace(b, layer_multipliers=b.layer_multipliers[:k], vocab_sizes=b.vocab_sizes[:k],
                       offsets=b.offsets[:k])
    T, B, L, H, N = b.num_tokens, b.num_requests, b.num_layers, b.num_heads, b.ngram_size
    D = args.embed_dim
    V = int(b.vocab_sizes.sum(axis=1).max())

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    gen = torch.Generator(device=device)
    gen.manual_seed(4000)
    table = torch.randn((L, V, D), dtype=torch.bfloat16, device=device, generator=gen)
    ids, ctx, cu = to_dev(b.ids), to_dev(b.ngram_context), to_dev(b.cu_seqlens)
    M, vocab, off = to_dev(b.layer_multipliers), to_dev(b.vocab_sizes), to_dev(b.offsets)
    req, local = ple.ple_build_token_index(cu, B, T, False)
    out = torch.empty((L, T, D), dtype=torch.float32, device=device)

    def call():
        ple.ple_row_embed(ids, req, local, ctx, M, vocab, off, N, b.heads_per_ngram,
                          b.boundary_id, table, out=out)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(device)
    steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    gather = L * T * H * D * 2
    written = L * T * D * 4
    total = gather + written + T * 16 + B * (N - 1) * 8 + 8 * L * (N + 2 * H)
    peaks, kind = measured_peaks()
    gbs = total / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "fused PLE table gather (hash + gather, row ids never written)",
        "workload": f"{b.name}: T={T}, L={L}, H={H}, D={D}, V={V} rows per layer, bf16 table "
                    f"{L * V * D * 2 / 1e9:.1f} GB, fp32 out",
        "ms_per_call": ms, "embeddings_per_s": L * T / (ms / 1e3),
        "algorithmic_bytes": total, "gather_bytes": gather, "out_bytes": written,
        "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
        "peak_kind": kind, "steps": steps, "launches_per_call": 1}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode B=1 latency")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="skip the all-cores oracle run beside the single-thread baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of single-thread oracle work for cpu_baseline")
    ap.add_argument("--embed", action="store_true",
                    help="time the fused table gather instead of the contract line")
    ap.add_argument("--embed-dim", type=int, default=256)
    ap.add_argument("--embed-layers", type=int, default=8,
                    help="layers of the large prefill the gather runs (default all 8)")
    ap.add_argument("--all-configs", action="store_true",
                    help="time every workload (graph of 300 calls) instead of the contract line")
    ap.add_argument("--only", nargs="+", default=None, metavar="WORKLOAD",
                    help="with --all-configs: only these workloads (e.g. mixed_8192)")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the decode B=1 latency (graph of 300 calls), one JSON object")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)
    if args.all_configs:
        return all_configs(args)
    if args.embed:
        return embed_bench(args)
    if args.decode_only:
        import torch

        import layer_gram_embedding_gb300 as ple
        from layer_gram_embedding_gb300 import build as lib_build

        lib_build.build()
        print(json.dumps({"decode_b1": decode_latency(ple, torch, torch.device("cuda", 0))}))
        return 0
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
