"""Benchmark of the PLE n-gram row-id hash on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--shard]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over
one batch, through the C ABI: each token's (request, offset) found from
cu_seqlens and the row-id hash of every layer, in one launch
(ple_row_ids_ex with req = local = NULL and cu_seqlens).  The workload is the
large prefill: T=262144 tokens in 4 requests, ngram_size 4, 4 heads per order
(12 heads), 8 layers, int64 ids, 20% adversarial boundary runs.  Inputs are
resident in HBM before the timed region; 64 distinct input sets rotate (256
MiB of inputs) and two output buffers alternate (201 MB of row ids written
per step), so no step finds its inputs in the 126 MB L2.

The timed region is exactly K steps back to back, bracketed by a barrier and
a device synchronisation on both sides, with CUDA events at its ends on the
launching stream.  It is repeated until at least --min-timed-ms of steps have
been timed; the step time is the median over the repeats (their spread is
reported), and the SM clocks are sampled across them.

Also measured, as extra keys:
  roofline     the step's one kernel against the HBM copy bandwidth;
  configs      every workload of the path (the 512-token prefill, decode
               B=1/4/8, the 16-request ragged prefill, the 48-layer mixed
               batch in both index forms, the large prefill with int32 ids
               and with int32 row ids, the fused table gather), device time
               per call from CUDA graphs of back-to-back calls (median of 7
               replays), each with its own clock record;
  e2e          the same metric with host buffers (pinned H2D of the step's
               inputs, D2H of its rows), and beside it the int32-row and
               gather variants, which return fewer or different bytes;
  decode_b1    device time per call, with and without programmatic
               dependent launch;
  cpu_baseline the CPU oracle on the host cores.

--impl reference times the CPU oracle (the only reference this path has) on
bounded samples of the same workload.

Under torchrun (--gpus N > 1) every rank hashes its own seeded batch (weak
scaling, no collective on the data path); the step time is the max over
ranks.  With --shard the ranks split ONE batch by token range instead
(ple_shard_plan / ple_shard_inputs: strong scaling, still no exchange).
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
KERNEL_SOURCES = ["ple_rowids_common.cuh", "ple_rowids_headlane.cu", "ple_divmod.cuh",
                  "ple_internal.h"]
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


def workload_config(batch: wl.Batch):
    """The workload, identical in both arms' lines."""
    return {
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
        "launches_per_step": 1,
        "step": "index found from cu_seqlens + row-id hash of every layer, one call",
    }


def call_bytes(batch: wl.Batch, mode: str, out_bytes: int = 8, prepared: bool = False,
               embed_dim: int = 0) -> int:
    """Algorithmic bytes of one row-id (or gather) call: ids read, the index
    read (mode "index"), cu_seqlens read (mode "cu"), nothing for a decode
    without an index (mode "decode"), context and parameters read, row ids
    written -- or, for the gather, the table rows read and the embeddings
    written."""
    idb = batch.ids.dtype.itemsize
    T, B, L, H, N = (batch.num_tokens, batch.num_requests, batch.num_layers, batch.num_heads,
                     batch.ngram_size)
    index = {"index": 8 * T, "cu": 4 * (B + 1), "decode": 0}[mode]
    params = 8 * L * N + (48 * L * H if prepared else 16 * L * H)
    out = L * T * H * out_bytes if not embed_dim else L * T * H * embed_dim * 2 + L * T * embed_dim * 4
    return T * idb + index + B * (N - 1) * idb + params + out


# ---------------------------------------------------------------------------
# clocks during the timed regions


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.windows = {}

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

    def mark(self, name: str, on: bool):
        w = self.windows.setdefault(name, [None, None])
        w[0 if on else 1] = time.monotonic()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def record(self, name: str):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        t_on, t_off = self.windows.get(name, (None, None))
        rows = []
        for t, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append((t, parts))
        window = [r for t, r in rows if t_on and t_off and t_on <= t <= t_off]
        # a window shorter than the sampling period: the samples around it
        if not window and t_on and t_off:
            near = sorted(rows, key=lambda tr: min(abs(tr[0] - t_on), abs(tr[0] - t_off)))[:2]
            used = [r for _, r in near]
        else:
            used = window
        sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        reasons = sorted({self.REASONS[i] for r in used for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(window)}


# ---------------------------------------------------------------------------
# distributed plumbing (no data-path collective)


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
        t = time.perf_counter()
        req, local = oracle.token_index(s.cu_seqlens, s.num_requests, s.num_tokens, False)
        oracle.row_ids(s.ids, req, local, s.ngram_context, s.layer_multipliers, s.vocab_sizes,
                       s.offsets, s.ngram_size, s.heads_per_ngram, s.boundary_id)
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
        "config": workload_config(batch),
        "config_notes": {"reference": "CPU oracle (plain C, single thread), the only "
                                      "reference this path has",
                         "sample_tokens_per_step": n_tok},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# device timing helpers


def graph_us_per_call(torch, device, calls_fns, calls: int, replays: int = 7):
    """Median device µs per call of a CUDA graph of `calls` back-to-back calls
    (cycling over calls_fns), over `replays` replays after one warm replay:
    the page's 7 x 300 method.  Returns (median, runs)."""
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for fn in calls_fns:
            fn()
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(calls):
            calls_fns[i % len(calls_fns)]()
    g.replay()
    torch.cuda.synchronize(device)
    runs = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize(device)
        runs.append(1e3 * e0.elapsed_time(e1) / calls)
    del g
    return statistics.median(runs), runs


def timed_regions(torch, device, stream, dist, step, first: int, steps: int, min_ms: float,
                  max_regions: int = 5000):
    """Repeats the timed region -- exactly `steps` steps back to back,
    bracketed by a barrier and a device synchronisation on both sides, CUDA
    events at its ends on the launching stream -- until min_ms of steps have
    been timed.  Returns the per-region milliseconds (max over ranks)."""
    out, total, i = [], 0.0, first
    while (total < min_ms or len(out) < 3) and len(out) < max_regions:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(steps):
            step(i)
            i += 1
        e1.record(stream)
        torch.cuda.synchronize(device)
        dist.barrier()
        ms = dist.max(e0.elapsed_time(e1), device)
        out.append(ms)
        total += ms
    return out


def spread(per_step_ms):
    a = np.asarray(per_step_ms)
    return {"regions": int(a.size), "median": float(np.median(a)), "min": float(a.min()),
            "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "max": float(a.max())}


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
    seed0 = 0 if args.shard else 1000 * dist.rank
    base = wl.prefill_262144(replay=seed0)
    batches = [base] + [wl.prefill_262144(replay=seed0 + r) for r in range(1, ROTATE)]
    T, B, N, hpn, L, H = (base.num_tokens, base.num_requests, base.ngram_size,
                          base.heads_per_ngram, base.num_layers, base.num_heads)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    M, vocab, off = to_dev(base.layer_multipliers), to_dev(base.vocab_sizes), to_dev(base.offsets)
    P = ctypes.c_void_p
    C = N - 1
    if args.shard:
        # one batch split by token range over the ranks: this rank's share
        plans = [ple.ple_shard_plan(b.cu_seqlens, B, T, dist.world, dist.rank) for b in batches]
        span = max(p[1] - p[0] for p in plans)
    sets = []
    for b in batches:
        s = dict(ids=to_dev(b.ids), ctx=to_dev(b.ngram_context), cu=to_dev(b.cu_seqlens),
                 req=torch.empty(T, dtype=torch.int32, device=device),
                 local=torch.empty(T, dtype=torch.int32, device=device))
        if args.shard:
            s["scu"] = torch.empty(B + 1, dtype=torch.int32, device=device)
            s["sctx"] = torch.empty((B, C), dtype=torch.int64, device=device)
        sets.append(s)
    T_out = span if args.shard else T
    outs = [torch.empty((L, T_out, H), dtype=torch.int64, device=device) for _ in range(2)]
    idx_args, row_args, search_args, shard_args = [], [], [], []
    for k, s in enumerate(sets):
        idx_args.append((P(s["cu"].data_ptr()), B, T, 0, P(s["req"].data_ptr()),
                         P(s["local"].data_ptr()), sh))
        row_args.append((P(s["ids"].data_ptr()), ple.PLE_I64, T, P(s["req"].data_ptr()),
                         P(s["local"].data_ptr()), P(s["ctx"].data_ptr()), B, C,
                         P(M.data_ptr()), P(vocab.data_ptr()), P(off.data_ptr()), H, N, hpn, L,
                         base.boundary_id, P(outs[k % 2].data_ptr()), sh))
        # the whole step in one launch: req = local = NULL with cu_seqlens,
        # each token's request found in the kernel
        search_args.append((P(s["ids"].data_ptr()), ple.PLE_I64, T, None, None,
                            P(s["ctx"].data_ptr()), B, C, P(M.data_ptr()),
                            P(vocab.data_ptr()), P(off.data_ptr()), H, N, hpn, L,
                            base.boundary_id, P(outs[k % 2].data_ptr()), ple.PLE_I64,
                            P(s["cu"].data_ptr()), None, None, sh))
        if args.shard:
            tb, te, rb, rc = plans[k]
            shard_args.append((
                (P(s["ids"].data_ptr()), ple.PLE_I64, P(s["cu"].data_ptr()),
                 P(s["ctx"].data_ptr()), B, T, C, tb, te, rb, rc, P(s["scu"].data_ptr()),
                 P(s["sctx"].data_ptr()), sh),
                (P(s["ids"].data_ptr() + 8 * tb), ple.PLE_I64, te - tb, None, None,
                 P(s["sctx"].data_ptr()), rc, C, P(M.data_ptr()), P(vocab.data_ptr()),
                 P(off.data_ptr()), H, N, hpn, L, base.boundary_id, P(outs[k % 2].data_ptr()),
                 ple.PLE_I64, P(s["scu"].data_ptr()), None, None, sh)))
    f_idx, f_rows, f_search = lib.ple_build_token_index, lib.ple_row_ids, lib.ple_row_ids_ex
    f_shard = lib.ple_shard_inputs

    def step(i):
        if f_search(*search_args[i % ROTATE]):
            raise RuntimeError("library call failed")

    def step_shard(i):
        a, r = shard_args[i % ROTATE]
        if f_shard(*a) | f_search(*r):
            raise RuntimeError("library call failed")

    def step_with_index(i):
        k = i % ROTATE
        st = f_idx(*idx_args[k]) | f_rows(*row_args[k])
        if st:
            raise RuntimeError(f"library call failed: status {st}")

    main_step = step_shard if args.shard else step
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(visible.split(",")[dist.local_rank].strip() if visible else
                          str(dist.local_rank))
    clocks.start()
    for i in range(args.warmup):
        main_step(i)
        if not args.shard:
            step_with_index(i)
    torch.cuda.synchronize(device)
    # beyond the W warm-up steps, untimed steps for --prewarm-ms of device
    # time, so that an idle GPU's clocks have ramped before the first timed
    # region (a run timed straight after start-up read twice the step time)
    t_end = time.perf_counter() + args.prewarm_ms / 1e3
    i = args.warmup
    while time.perf_counter() < t_end:
        for _ in range(50):
            main_step(i)
            i += 1
        torch.cuda.synchronize(device)

    # ---- the timed regions: K steps back to back each, repeated
    clocks.mark("headline", True)
    regions = timed_regions(torch, device, stream, dist, main_step, args.warmup, args.steps,
                            args.min_timed_ms)
    clocks.mark("headline", False)
    per_step = [ms / args.steps for ms in regions]
    step_ms = statistics.median(per_step)
    clk = clocks.record("headline")

    # ---- the step as two launches (ple_build_token_index, then ple_row_ids
    # reading the index), for comparison
    with_index = None
    bracketed_ms = None
    if not args.shard:
        w_regions = timed_regions(torch, device, stream, dist, step_with_index, args.warmup,
                                  args.steps, args.min_timed_ms / 4)
        with_index_ms = statistics.median([ms / args.steps for ms in w_regions])
        with_index = {
            "launches": 2, "ms_per_step": with_index_ms,
            "value": dist.world * base.row_ids_per_call / (with_index_ms / 1e3), "unit": UNIT,
            "what": "ple_build_token_index then ple_row_ids reading the index, back to back",
            "timed_regions": len(w_regions)}
        # the step's one kernel with an event pair around every launch, for
        # reference (an event between launches serialises them and adds its
        # own drain-and-launch gap to every launch)
        n_br = 200
        br = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_br)]
        for i in range(n_br):
            br[i][0].record(stream)
            step(i)
            br[i][1].record(stream)
        torch.cuda.synchronize(device)
        bracketed_ms = float(np.median([a.elapsed_time(b) for a, b in br]))

    rows_total = base.row_ids_per_call if args.shard else dist.world * base.row_ids_per_call
    value = rows_total / (step_ms / 1e3)
    peaks, peak_kind = measured_peaks()
    if args.shard:
        kernel_bytes = None
        roofline = None
    else:
        # ids and cu_seqlens read, context and parameters read, row ids written
        kernel_bytes = call_bytes(base, "cu")
        achieved = kernel_bytes / (step_ms / 1e3) / 1e9
        traffic = None
        try:
            with open(PROFILE_TRAFFIC) as fh:
                prof = json.load(fh)
            if prof.get("kernel_source_sha256_16") == kernel_source_hash():
                traffic = prof.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            pass
        sm_med = clk.get("sm_mhz")
        roofline = {
            "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
            "kernel": "ple row_ids kernel (row_ids_headlane_kernel<int64 ids, 4, 4, int64 rows, "
                      "block-shared constants>, requests found from cu_seqlens in the kernel)",
            "algorithmic_bytes_per_launch": kernel_bytes,
            "kernel_ms_avg": step_ms,
            "kernel_timing": f"median over {len(regions)} timed regions of {args.steps} "
                             "one-launch steps back to back, CUDA events at each region's ends "
                             "on the launching stream",
            "kernel_ms_bracketed_median": bracketed_ms,
            "kernel_ms_x_sm_mhz": step_ms * sm_med if sm_med else None,
            "peak_kind": peak_kind}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": workload_config(base),
        "config_notes": {
            "l2": f"inputs rotate over {ROTATE} seeded sets ({ROTATE * (T * 16 + 64) >> 20} MiB) "
                  f"and 2 output buffers ({L * T * H * 8 / 1e6:.0f} MB written per step); "
                  "no step's data fits the 126 MB L2",
            "parallelism": (f"token-range shards x{dist.world} of one batch (ple_shard_plan + "
                            "ple_shard_inputs + the row-id call per rank; no collective)"
                            if args.shard else
                            f"replicas x{dist.world} (weak scaling, no collective)")},
        "timed_regions": spread(per_step),
        "roofline": roofline,
        "gpu_launches": args.steps * (2 if args.shard else 1),
        "gpu_launches_note": "per timed region (each region is exactly --steps steps)",
        "step_with_index_build": with_index,
        "clocks": clk,
    }

    if dist.world == 1 and not args.shard:
        if not args.no_configs:
            line["configs"] = all_configs(args, ple, torch, device, clocks, peaks)
        if not args.no_e2e:
            line["e2e"] = end_to_end(args, ple, torch, device, stream, batches[:4], M, vocab, off)
            line["e2e_variants"] = e2e_variants(args, ple, torch, device, stream, batches[:4],
                                                M, vocab, off)
        if not args.no_decode:
            line["decode_b1"] = decode_latency(ple, torch, device)
    clocks.stop()

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
        line["cpu_baseline"] = cpu
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def end_to_end(args, ple, torch, device, stream, batches, M, vocab, off, out_dtype=None):
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
    out_dtype = out_dtype or torch.int64
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
            out=torch.empty((L, T, H), dtype=out_dtype, device=device),
            h_out=torch.empty((L, T, H), dtype=out_dtype).pin_memory(),
            computed=torch.cuda.Event(), copied=torch.cuda.Event()))
    steps = max(3, min(args.steps, 100))
    h2d = T * 8 + (B + 1) * 4 + B * (b0.ngram_size - 1) * 8
    d2h = L * T * H * slots[0]["out"].element_size()
    d2h_stream = torch.cuda.Stream(device)

    def run(i, pipelined):
        h, sl = host[i % len(host)], slots[i % 2 if pipelined else 0]
        if pipelined:
            stream.wait_event(sl["copied"])  # the slot's previous rows are in host memory
        sl["ids"].copy_(h["ids"], non_blocking=True)
        sl["cu"].copy_(h["cu"], non_blocking=True)
        sl["ctx"].copy_(h["ctx"], non_blocking=True)
        ple.ple_row_ids(sl["ids"], None, None, sl["ctx"], M, vocab, off, b0.ngram_size,
                        b0.heads_per_ngram, b0.boundary_id, out=sl["out"], cu_seqlens=sl["cu"],
                        out_dtype=out_dtype)
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
            "row_ids_dtype": str(out_dtype).replace("torch.", ""),
            "method": "two buffer slots; each step's device-to-host copy overlaps the next "
                      "step's host-to-device copy and kernel",
            "serial_ms_per_step": ms_serial / steps,
            "serial_value": b0.row_ids_per_call * steps / (ms_serial / 1e3)}


def e2e_variants(args, ple, torch, device, stream, batches, M, vocab, off):
    """End to end for the variants that return fewer bytes: int32 row ids
    (half the device-to-host bytes), and the fused gather, whose result is the
    embeddings ([L, T, D] fp32, D = --embed-dim) instead of row ids."""
    res = {"int32_row_ids": end_to_end(args, ple, torch, device, stream, batches, M, vocab, off,
                                       out_dtype=torch.int32)}
    b0 = batches[0]
    T, B, L, H, N = b0.num_tokens, b0.num_requests, b0.num_layers, b0.num_heads, b0.ngram_size
    D = args.embed_dim
    V = int(b0.vocab_sizes.sum(axis=1).max())
    gen = torch.Generator(device=device)
    gen.manual_seed(4000)
    table = torch.randn((L, V, D), dtype=torch.bfloat16, device=device, generator=gen)
    host = [dict(ids=torch.from_numpy(b.ids).pin_memory(),
                 cu=torch.from_numpy(b.cu_seqlens).pin_memory(),
                 ctx=torch.from_numpy(np.ascontiguousarray(b.ngram_context)).pin_memory())
            for b in batches]
    ids = torch.empty(T, dtype=torch.int64, device=device)
    cu = torch.empty(B + 1, dtype=torch.int32, device=device)
    ctx = torch.empty((B, N - 1), dtype=torch.int64, device=device)
    out = torch.empty((L, T, D), dtype=torch.float32, device=device)
    h_out = torch.empty((L, T, D), dtype=torch.float32).pin_memory()

    def run(i):
        h = host[i % len(host)]
        ids.copy_(h["ids"], non_blocking=True)
        cu.copy_(h["cu"], non_blocking=True)
        ctx.copy_(h["ctx"], non_blocking=True)
        ple.ple_row_embed(ids, None, None, ctx, M, vocab, off, N, b0.heads_per_ngram,
                          b0.boundary_id, table, out=out, cu_seqlens=cu)
        h_out.copy_(out, non_blocking=True)

    for i in range(2):
        run(i)
    torch.cuda.synchronize(device)
    steps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        run(i)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    res["row_embed"] = {
        "value": L * T / (ms / 1e3), "unit": "embeddings/s", "ms_per_step": ms, "steps": steps,
        "h2d_bytes_per_step": T * 8 + (B + 1) * 4 + B * (N - 1) * 8,
        "d2h_bytes_per_step": L * T * D * 4,
        "row_ids_per_s_equivalent": b0.row_ids_per_call / (ms / 1e3),
        "method": f"one stream: H2D of ids / cu_seqlens / context, ple_row_embed (D={D}, bf16 "
                  f"table of {L * V * D * 2 / 1e9:.1f} GB resident), D2H of every embedding"}
    del table
    torch.cuda.empty_cache()
    return res


def decode_latency(ple, torch, device):
    """Device µs per call of ple_row_ids at decode B=1: a CUDA graph of 300
    back-to-back calls, median of 7 replays (the page's 7 x 300 method).
    Measured without an index (req = local = NULL, one launch per step) and
    with a prebuilt index (the page's memoized index), each with the head
    constants derived in the call (the page's arguments) and prepared once
    by ple_prepare_heads (model parameters, fixed across steps); and without
    an index with programmatic dependent launch off, so that no call's launch
    overlaps the one before it."""
    b = wl.decode(1)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    ids, ctx = to_dev(b.ids), to_dev(b.ngram_context)
    M, vocab, off = to_dev(b.layer_multipliers), to_dev(b.vocab_sizes), to_dev(b.offsets)
    req, local = ple.ple_build_token_index(None, 1, 1, True, device=device)
    heads = ple.ple_prepare_heads(vocab, off)
    out = torch.empty((1, 1, 4), dtype=torch.int64, device=device)
    res = {"launches_per_call": 1, "method": "CUDA graph of 300 calls, median of 7 replays"}
    for name, (rq, lc, hd, pdl) in (
            ("device_us_per_call", (None, None, None, True)),
            ("device_us_per_call_with_index", (req, local, None, True)),
            ("device_us_per_call_prepared_heads", (None, None, heads, True)),
            ("device_us_per_call_with_index_prepared_heads", (req, local, heads, True)),
            ("device_us_per_call_no_programmatic_launch", (None, None, None, False)),
            ("device_us_per_call_prepared_heads_no_programmatic_launch",
             (None, None, heads, False))):
        def call():
            ple.ple_row_ids(ids, rq, lc, ctx, M, vocab, off, 3, 2, b.boundary_id, out=out,
                            heads=hd)

        prev = ple.set_programmatic_launch(pdl)
        try:
            us, runs = graph_us_per_call(torch, device, [call], 300)
        finally:
            ple.set_programmatic_launch(prev)
        res[name] = us
        if name == "device_us_per_call":
            res["runs_us"] = runs
    return res


def all_configs(args, ple, torch, device, clocks, peaks):
    """Every workload of the path, device µs per call from a CUDA graph of
    back-to-back calls, median of 7 replays (the page's 7 x 300 method), each
    with the clocks sampled while it ran.  Workloads whose data fits in L2
    reuse one input set (as the page's method does); the large ones cycle
    over 16 input sets (ids rolled) and two output buffers."""
    entries = {}
    hbm = peaks["hbm_gbs"]

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    def entry(key, batch, variants, sets=1):
        """variants: (name, mode, out_dtype, prepared, index_build, pdl)."""
        if args.only and key not in args.only:
            return
        T, B, L, H = batch.num_tokens, batch.num_requests, batch.num_layers, batch.num_heads
        M, vocab, off = (to_dev(batch.layer_multipliers), to_dev(batch.vocab_sizes),
                         to_dev(batch.offsets))
        heads = ple.ple_prepare_heads(vocab, off)
        ins = []
        for r in range(sets):
            ids = batch.ids if r == 0 else np.roll(batch.ids, 977 * r)
            d = dict(ids=to_dev(ids), ctx=to_dev(batch.ngram_context),
                     cu=to_dev(batch.cu_seqlens) if batch.cu_seqlens is not None else None)
            d["req"], d["local"] = ple.ple_build_token_index(d["cu"], B, T, batch.is_decode,
                                                             device=device)
            ins.append(d)
        res = {"workload": batch.name, "T": T, "B": B, "L": L, "H": H,
               "ngram_size": batch.ngram_size, "ids_dtype": batch.ids.dtype.name,
               "row_ids_per_call": batch.row_ids_per_call}
        calls = 300
        for name, mode, odt, prepared, build_index, pdl in variants:
            if args.forms and name not in args.forms:
                continue
            outs = [torch.empty((L, T, H), dtype=odt, device=device)
                    for _ in range(2 if sets > 1 else 1)]
            fns = []
            for r, d in enumerate(ins):
                o = outs[r % len(outs)]

                def fn(d=d, o=o):
                    if build_index:
                        ple.ple_build_token_index(d["cu"], B, T, batch.is_decode, req=d["req"],
                                                  local=d["local"])
                    idx = mode == "index"
                    ple.ple_row_ids(d["ids"], d["req"] if idx else None,
                                    d["local"] if idx else None, d["ctx"], M, vocab, off,
                                    batch.ngram_size, batch.heads_per_ngram, batch.boundary_id,
                                    out=o, out_dtype=odt, heads=heads if prepared else None,
                                    cu_seqlens=d["cu"] if mode == "cu" else None)
                fns.append(fn)
            prev = ple.set_programmatic_launch(pdl)
            clocks.mark(key + name, True)
            try:
                us, _ = graph_us_per_call(torch, device, fns, calls)
            finally:
                clocks.mark(key + name, False)
                ple.set_programmatic_launch(prev)
            nb = call_bytes(batch, mode, 4 if odt == torch.int32 else 8, prepared)
            v = {"us_per_call": us, "launches_per_call": 2 if build_index else 1,
                 "row_ids_per_s": batch.row_ids_per_call / (us / 1e6),
                 "clocks": clocks.record(key + name)}
            if not build_index:
                v["algorithmic_bytes"] = nb
                v["achieved_gbs"] = nb / (us / 1e6) / 1e9
                v["frac_of_measured_hbm"] = v["achieved_gbs"] / hbm
            res[name] = v
        res["method"] = (f"CUDA graph of {calls} back-to-back calls over {sets} input set(s), "
                         "median of 7 replays")
        entries[key] = res
        print(json.dumps({key: res}), file=sys.stderr, flush=True)

    I64, I32 = torch.int64, torch.int32
    # (name, mode, out dtype, prepared heads, index build in the call, programmatic launch)
    one = ("one_launch", "cu", I64, False, False, True)
    two = ("two_launch_step", "index", I64, False, True, True)
    idx = ("row_ids_reading_index", "index", I64, False, False, True)
    entry("prefill_512", wl.prefill_512(), [one, two, idx])
    for Bd in (1, 4, 8):
        entry(f"decode_b{Bd}", wl.decode(Bd), [
            ("one_launch", "decode", I64, False, False, True),
            ("one_launch_prepared_heads", "decode", I64, True, False, True),
            ("one_launch_no_programmatic_launch", "decode", I64, False, False, False),
            ("two_launch_step", "index", I64, False, True, True)])
    entry("ragged_16", wl.ragged_16(), [one, two, idx])
    entry("mixed_8192", wl.mixed_8192(), [
        one, idx, two,
        ("one_launch_prepared_heads", "cu", I64, True, False, True),
        ("row_ids_reading_index_prepared_heads", "index", I64, True, False, True),
        ("one_launch_int32_row_ids", "cu", I32, False, False, True)], sets=16)
    entry("prefill_262144_int32_ids", wl.prefill_262144(ids_dtype=np.int32), [one], sets=16)
    entry("prefill_262144_int32_row_ids", wl.prefill_262144(), [
        ("one_launch", "cu", I32, False, False, True),
        ("row_ids_reading_index", "index", I32, False, False, True)], sets=16)
    if not args.no_embed:
        for b in (wl.prefill_262144(), wl.prefill_262144_lowrep()):
            if not args.only or "row_embed_" + b.name in args.only:
                entries["row_embed_" + b.name] = embed_entry(args, ple, torch, device, clocks,
                                                             b, peaks)
    return entries


def configs_only(args):
    """Only the per-workload figures (all, or --only KEY ...), one JSON
    object; a small process for profiling one workload's kernels."""
    import torch

    import layer_gram_embedding_gb300 as ple
    from layer_gram_embedding_gb300 import build as lib_build

    lib_build.build()
    device = torch.device("cuda", 0)
    peaks, _ = measured_peaks()
    clocks = ClockSampler("0")
    clocks.start()
    out = {}
    if not args.only or "decode_b1_latency" in args.only:
        out["decode_b1"] = decode_latency(ple, torch, device)
    out["configs"] = all_configs(args, ple, torch, device, clocks, peaks)
    clocks.stop()
    print(json.dumps(out))
    return 0


def embed_entry(args, ple, torch, device, clocks, b, peaks):
    """The fused table gather (ple_row_embed, requests found from cu_seqlens)
    on one workload: a D-wide bfloat16 table per layer with one row per head
    vocabulary entry; device time per call from a graph of 20 calls, median
    of 7 replays."""
    if args.embed_layers < b.num_layers:
        k = max(1, args.embed_layers)
        b = wl.replace(b, layer_multipliers=b.layer_multipliers[:k],
                       vocab_sizes=b.vocab_sizes[:k], offsets=b.offsets[:k])
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
    out = torch.empty((L, T, D), dtype=torch.float32, device=device)

    def call():
        ple.ple_row_embed(ids, None, None, ctx, M, vocab, off, N, b.heads_per_ngram,
                          b.boundary_id, table, out=out, cu_seqlens=cu)

    key = "embed_" + b.name
    clocks.mark(key, True)
    us, _ = graph_us_per_call(torch, device, [call], 20)
    clocks.mark(key, False)
    nb = call_bytes(b, "cu", embed_dim=D)
    gbs = nb / (us / 1e6) / 1e9
    del table
    torch.cuda.empty_cache()
    return {"workload": b.name, "T": T, "L": L, "H": H, "D": D, "V": V,
            "table_gb": L * V * D * 2 / 1e9, "us_per_call": us,
            "embeddings_per_s": L * T / (us / 1e6), "algorithmic_bytes": nb,
            "gather_bytes": L * T * H * D * 2, "out_bytes": L * T * D * 4,
            "achieved_gbs": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
            "launches_per_call": 1, "clocks": clocks.record(key),
            "method": "CUDA graph of 20 calls, median of 7 replays"}


def embed_bench(args):
    """The fused table gather alone on one workload, one JSON line (for
    profiling: --embed-layers 1 keeps the table to a few GB)."""
    import torch

    import layer_gram_embedding_gb300 as ple
    from layer_gram_embedding_gb300 import build as lib_build

    lib_build.build()
    device = torch.device("cuda", 0)
    peaks, _ = measured_peaks()
    b = wl.prefill_262144_lowrep() if args.embed_workload == "lowrep" else wl.prefill_262144()
    clocks = ClockSampler("0")
    clocks.start()
    res = embed_entry(args, ple, torch, device, clocks, b, peaks)
    clocks.stop()
    print(json.dumps(res))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--shard", action="store_true",
                    help="split one batch by token range over the ranks (strong scaling)")
    ap.add_argument("--prewarm-ms", type=float, default=200.0,
                    help="untimed steps for this long after the warm-up steps (clock ramp)")
    ap.add_argument("--min-timed-ms", type=float, default=250.0,
                    help="repeat the K-step timed region until this much has been timed")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload figures")
    ap.add_argument("--no-embed", action="store_true", help="skip the gather in the configs")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurements")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode B=1 latency")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="skip the all-cores oracle run beside the single-thread baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of single-thread oracle work for cpu_baseline")
    ap.add_argument("--configs-only", action="store_true",
                    help="only the per-workload figures (one JSON object)")
    ap.add_argument("--only", nargs="+", default=None, metavar="KEY",
                    help="with --configs-only: these entries only (e.g. mixed_8192, "
                         "decode_b1, decode_b1_latency, row_embed_prefill_262144_lowrep)")
    ap.add_argument("--forms", nargs="+", default=None, metavar="NAME",
                    help="with --configs-only: only these call forms of each workload "
                         "(e.g. one_launch_int32_row_ids), for profiling one launch kind")
    ap.add_argument("--embed", action="store_true",
                    help="time only the fused table gather (one JSON line)")
    ap.add_argument("--embed-workload", choices=["runs", "lowrep"], default="runs")
    ap.add_argument("--embed-dim", type=int, default=256)
    ap.add_argument("--embed-layers", type=int, default=8,
                    help="layers of the large prefill the gather runs (default all 8)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)
    if args.embed:
        return embed_bench(args)
    if args.configs_only:
        return configs_only(args)
    return our_arm(args)


if __name__ == "__main__":
    sys.exit(main())
