"""Benchmark of the paged GQA decode step (KV append + split decode + combine).

Default workload: the Mistral-7B-v0.3-shaped serving batch (256 rows, 32 query
/ 8 kv heads, head_dim 128, contexts ~ U[1024, 32768], 64-position pages in
one shuffled pool of ~18 GB per K and V), the largest of the five workloads.
One step = one append of each row's new K/V at its page slot, then grouped
decode attention of every row over its pages: one paged_decode_step call (the
append inside the decode launch), or with --two-calls kv_append_paged then
paged_decode_attention.  Inputs are resident in HBM and
much larger than L2 (129 MB), so no flush is needed between steps; smaller
workloads (--workload) are timed step by step with an L2 flush between steps,
outside the timed spans (see L2Flush).

Prints one JSON line.  `value` is achieved HBM GB/s of the whole step over
all ranks (algorithmic bytes: every attended K/V row read once, q read, out
written, the append's read and write); `row_tokens_per_s` is rows decoded per
second.  On the default workload the line also carries `workloads`: the
other four decode workloads (Qwen2.5-shaped small and serving batches,
gpt-oss full-context and sliding-window layers), each measured the same way
in the same process.  `cpu_baseline` times the fp64 CPU oracle on the rows of
the batch and compares its output with the timed step's (`parity`).
`--impl reference` times the oracle on the host's cores on a bounded sample
of the same workload instead.

Multi-GPU: one process per GPU under torchrun; rows are independent, so each
rank decodes its own batch (weak scaling) and no collective touches the data
path; the ranks only meet at the barriers around the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from pgd_inputs import WORKLOADS, Workload, bf16_bits, make_batch  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak); row-tokens/s"
DEFAULT_WORKLOAD = "mistral_serve"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


class PackedInputs:
    """A step's inputs in one pinned host buffer and one device buffer, each
    tensor at a 256-byte-aligned offset, so that one copy uploads them all
    (as a serving loop would send a step's inputs); `views` are the device
    tensors the API is called with.  Several device buffers can share one
    host buffer (`host`)."""

    def __init__(self, tensors: dict, device, host=None):
        offs, total = {}, 0
        for k, t in tensors.items():
            n = t.numel() * t.element_size()
            offs[k] = (total, n)
            total = (total + n + 255) // 256 * 256
        if host is None:
            host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
            for k, t in tensors.items():
                o, n = offs[k]
                host[o:o + n].copy_(t.detach().cpu().reshape(-1).view(torch.uint8))
        self.host = host
        self.dev = torch.empty(total, dtype=torch.uint8, device=device)
        self.views = {k: self.dev[o:o + n].view(t.dtype).view(t.shape)
                      for k, t in tensors.items() for o, n in [offs[k]]}
        self.bytes = total

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


class L2Flush:
    """Between timed steps: write a 1 GiB buffer (evicting everything the step
    left in L2), then read a 512 MiB one, so that L2 holds clean lines of an
    unrelated buffer.  After the write alone L2 would be full of dirty lines,
    and the next step would pay for writing them back to HBM as it reads
    (11 us of a 62 us decode call on the gpt-oss full-context workload)."""

    label = "1 GiB write + 512 MiB read flush of L2 between steps"

    def __init__(self, device):
        self.dirty = torch.empty(2 ** 30, dtype=torch.uint8, device=device)
        self.clean = torch.ones(2 ** 27, dtype=torch.float32, device=device)

    def __call__(self, i: int):
        self.dirty.fill_(i & 0xFF)
        self.clean.sum()


# --------------------------------------------------------------------------- bytes


def algorithmic_bytes(wl: Workload, positions: np.ndarray) -> dict:
    """Bytes one step must move at least once.  K/V: every attended (position,
    kv head) row of K and of V, read once.  q read and out written once.  The
    append reads k_new and v_new and writes them into the pool.  Sinks, the
    table and positions are negligible and not counted.  Attended positions
    per active row: min(window, n + 1) with a window, n + 1 without."""
    n = positions.astype(np.int64)
    active = n >= 0
    attended = np.where(active, n + 1, 0)
    if wl.window > 0:
        attended = np.minimum(attended, wl.window)
    row_bytes = 2 * wl.kv_heads * wl.head_dim * 2
    kv = int(attended.sum()) * row_bytes
    q_out = 2 * len(n) * wl.q_heads * wl.head_dim * 2
    append = 2 * int(active.sum()) * row_bytes
    return {"kv": kv, "q_out": q_out, "decode": kv + q_out, "append": append,
            "step": kv + q_out + append}


def describe(wl: Workload) -> str:
    win = f"window {wl.window}" if wl.window > 0 else "full window"
    sink = "fp32 sinks" if wl.sinks else "no sink"
    return (f"{wl.name}: {wl.rows} rows, {wl.q_heads}q/{wl.kv_heads}kv, d{wl.head_dim}, "
            f"ctx U[{wl.ctx_lo},{wl.ctx_hi}], page {wl.page_size}, {sink}, {win}")


# --------------------------------------------------------------------------- env


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(wl: Workload, rank: int) -> int:
    """Each rank decodes its own batch: the workload's seed offset by rank."""
    return 1000 + list(WORKLOADS).index(wl.name) + 7919 * rank


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def measured_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples; only those taken inside
    the timed region (by their timestamps) are summarised."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device: torch.device):
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.gpu = str(device.index)
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1 + 0.1]
        use = inside or rows
        if not use:
            return None
        reasons = sorted({n for r in use for n, f in zip(self.NAMES, r[3]) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "in_timed_region": bool(inside)}


def kernel_traffic(source_digest: str, workload: str):
    """DRAM bytes per decode call (split + combine) from the committed ncu
    summary, if it was taken on the current kernel sources and this
    workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_digest") != source_digest or rec.get("workload") != workload:
        return None
    return rec.get("decode_bytes_per_launch")


def source_digest() -> str:
    """Digest of the sources the decode step is built from (the prefill
    kernel's own files excluded)."""
    csrc = os.path.join(ROOT, "paged_gqa_decode_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.startswith("paged_prefill"):
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- oracle timing


def oracle_rows_timing(batch, rows, window, nthreads=None, result=False):
    """Seconds the oracle takes for append + decode of `rows` of the batch
    (and its output for those rows when `result`)."""
    from tests.oracle_side import oracle_step, snapshot_rows
    host = snapshot_rows(batch, rows)
    t0 = time.perf_counter()
    want, _, _ = oracle_step(batch, host, window=window, sinks=batch.sinks,
                             scale=batch.wl.scale, nthreads=nthreads)
    elapsed = time.perf_counter() - t0
    return (elapsed, want) if result else elapsed


# The tolerance the parity tests hold the CUDA path to (bf16 output from fp32
# accumulation): max abs 1e-2 and max rel 2e-2, rel where |oracle| >= 1e-3.
ABS_TOL, REL_TOL, REL_FLOOR = 1e-2, 2e-2, 1e-3


def parity_stats(got: torch.Tensor, want: np.ndarray) -> dict:
    g = got.float().cpu().numpy().astype(np.float64)
    diff = np.abs(g - want)
    big = np.abs(want) >= REL_FLOOR
    rel = diff[big] / np.abs(want[big]) if big.any() else np.zeros(1)
    max_abs, max_rel = float(diff.max(initial=0.0)), float(rel.max(initial=0.0))
    finite = bool(np.all(np.isfinite(g)))
    return {"max_abs": max_abs, "max_rel": max_rel, "finite": finite,
            "within_tolerance": finite and max_abs <= ABS_TOL and max_rel <= REL_TOL,
            "tolerance": {"abs": ABS_TOL, "rel": REL_TOL, "rel_where_abs_oracle_ge": REL_FLOOR}}


def cpu_baseline(batch, out: torch.Tensor | None = None, max_rows: int = 256) -> dict:
    """The oracle (append + decode) on up to `max_rows` seeded rows of the
    batch, on all host cores.  With `out` (the GPU output of the timed step
    on the same batch), the oracle's result for those rows is also compared
    with it element by element."""
    import oracle
    wl = batch.wl
    pos = batch.layout.positions
    order = np.random.default_rng(0).permutation(wl.rows)
    rows = np.sort(order[:min(max_rows, wl.rows)])
    elapsed, want = oracle_rows_timing(batch, rows, wl.window, result=True)
    by = algorithmic_bytes(wl, pos[rows])
    line = {"value": by["step"] / elapsed / 1e9, "unit": "GB/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "row_tokens_per_s": len(rows) / elapsed,
            "sample": f"{len(rows)} of {wl.rows} rows of {wl.name} (seeded choice), "
                      f"append + decode, {elapsed:.2f} s"}
    if out is not None:
        idx = torch.as_tensor(rows, device=out.device)
        line["parity"] = {"rows_checked": int(len(rows)), "of_rows": int(wl.rows),
                          "against": "output of the last timed step",
                          **parity_stats(out.index_select(0, idx), want)}
    return line


# --------------------------------------------------------------------------- arms


def run_reference(args, wl: Workload):
    """The oracle as it stands, on the host's cores: each step is a bounded
    sample (a few rows) of the workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(wl.name), device="cpu"
                       if not torch.cuda.is_available() else "cuda:0")
    pos = batch.layout.positions
    order = np.random.default_rng(0).permutation(wl.rows)
    rows_per_step = args.reference_rows
    times, total_bytes, total_rows = [], 0, 0
    for step in range(args.warmup + args.steps):
        rows = order[(step * rows_per_step) % wl.rows:][:rows_per_step]
        if len(rows) < rows_per_step:
            rows = order[:rows_per_step]
        t = oracle_rows_timing(batch, rows, wl.window)
        if step >= args.warmup:
            times.append(t)
            total_bytes += algorithmic_bytes(wl, pos[rows])["step"]
            total_rows += len(rows)
    elapsed = sum(times)
    value = total_bytes / elapsed / 1e9
    sample = f"{rows_per_step} rows of {wl.name} per step (seeded), append + decode"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "rows_per_step": rows_per_step},
        "row_tokens_per_s": total_rows / elapsed,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.default_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_pgd(args, wl: Workload):
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    line = measure_decode(args, wl, world, rank, device, main=True)
    # The other decode workloads, each measured the same way in this process
    # (the headline line stays on the default, largest one).
    if not args.only and args.rows == 0 and wl.name == DEFAULT_WORKLOAD:
        extra = {}
        for name, other in WORKLOADS.items():
            if name == wl.name:
                continue
            r = measure_decode(args, other, world, rank, device, main=False)
            if r is not None:
                extra[name] = {k: r[k] for k in (
                    "value", "unit", "ms_per_step", "row_tokens_per_s", "decode_ms_per_step",
                    "latency_back_to_back", "e2e", "clocks", "gpu_launches")}
                extra[name]["workload"] = r["config"]["workload"]
                extra[name]["l2"] = r["config"]["l2"]
                extra[name]["roofline"] = {k: r["roofline"][k] for k in (
                    "bound", "achieved", "peak", "peak_kind", "unit", "frac")}
                if "cpu_baseline" in r:
                    extra[name]["cpu_baseline"] = r["cpu_baseline"]
        if line is not None:
            line["workloads"] = extra
    if line is not None:
        print(json.dumps(line), flush=True)


def measure_decode(args, wl: Workload, world: int, rank: int, device, main: bool):
    """One decode workload: timed steps, per-call spans, back-to-back latency,
    end-to-end with host copies, clocks, and (rank 0, N = 1) the oracle on
    its rows compared with the timed step's output.  Returns rank 0's line
    (None on the other ranks)."""
    import paged_gqa_decode_gb300 as pgd
    batch = make_batch(wl, seed=rank_seed(wl, rank), device=device)
    lay = batch.layout
    dims = pgd.make_dims(rows=wl.rows, num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                         head_dim=wl.head_dim, num_pages=lay.num_pages,
                         max_pages_per_row=batch.table.shape[1])
    ws = torch.empty(max(16, pgd.paged_decode_workspace_bytes(dims, args.pages_per_split)),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(batch.q)
    stream = torch.cuda.current_stream()
    by = algorithmic_bytes(wl, lay.positions)
    flush = None
    if by["step"] < 4 * L2_BYTES:
        flush = L2Flush(device)

    q_rot = batch.q.clone() if args.rope else None
    # one call per step (the append inside the decode launch) unless the two
    # calls are asked for or the append also rotates q and k
    fused = not (args.two_calls or args.rope)

    def append():
        if fused:  # the append runs inside the decode launch (paged_decode_step)
            return
        if args.rope:   # rope_rows on q and k fused into the append (base 1e6)
            q_rot.copy_(batch.q)
            pgd.rope_append_paged(q_rot, batch.k_new, batch.v_new, batch.table,
                                  batch.positions, batch.k_pool, batch.v_pool, theta=1e6)
        else:
            pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions,
                                batch.k_pool, batch.v_pool)

    def decode():
        if fused:
            pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                  batch.table, batch.positions, batch.sinks, wl.window, wl.scale,
                                  num_kv_heads=wl.kv_heads, out=out, workspace=ws,
                                  pages_per_split=args.pages_per_split,
                                  kernel=KERNEL_IDS[args.kernel])
            return
        pgd.paged_decode_attention(q_rot if args.rope else batch.q, batch.k_pool, batch.v_pool, batch.table,
                                   batch.positions, batch.sinks, wl.window, wl.scale,
                                   num_kv_heads=wl.kv_heads, out=out, workspace=ws,
                                   pages_per_split=args.pages_per_split,
                                   kernel=KERNEL_IDS[args.kernel])

    for _ in range(args.warmup):
        append()
        decode()
    status = pgd.get_device_error()
    if status != pgd.OK:
        raise RuntimeError(f"device error during warm-up: {pgd.status_string(status)}")

    # Small workloads run between L2 flushes; their calls are captured once
    # as CUDA graphs so host-side call overhead cannot land inside the timed
    # device spans.  Large ones are called directly (the host runs far ahead).
    step_append, step_decode, step_whole = append, decode, None
    if flush is not None:
        # the whole step (append + decode, launched back to back so each kernel
        # overlaps its predecessor's tail) and each call alone, as graphs
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graphs = []

        def whole():
            append()
            decode()

        with torch.cuda.stream(side):
            # with the append fused the step is the decode call alone
            for fn in ((decode, whole) if fused else (append, decode, whole)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    fn()
                graphs.append(g)
        torch.cuda.synchronize()
        if fused:
            graphs.insert(0, None)
        step_append, step_decode, step_whole = (g.replay if g else append for g in graphs)
        for _ in range(3):
            step_whole()
        torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark_start()
    for i in range(args.steps):
        if flush is not None:      # whole steps between flushes
            flush(i)
            ev[i][0].record(stream)
            step_whole()
            ev[i][2].record(stream)
        else:                      # back to back, a span per call
            ev[i][0].record(stream)
            step_append()
            ev[i][1].record(stream)
            step_decode()
            ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(world)
    clk = clocks.stop()
    status = pgd.get_device_error()
    if status != pgd.OK:
        raise RuntimeError(f"device error in the timed region: {pgd.status_string(status)}")
    if flush is None:
        append_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
        decode_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
        step_ms = ev[0][0].elapsed_time(ev[-1][2])
    else:
        step_ms = sum(e[0].elapsed_time(e[2]) for e in ev)
        # each call alone, for the per-kernel spans (outside the step timing)
        spans = {"append": 0.0, "decode": 0.0}
        for i in range(args.steps):
            for name, fn in ((("decode", step_decode),) if fused else
                             (("append", step_append), ("decode", step_decode))):
                flush(i)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                z.record(stream)
                torch.cuda.synchronize()
                spans[name] += a.elapsed_time(z)
        append_ms, decode_ms = spans["append"], spans["decode"]
    latency = None
    if flush is not None:
        # the step as a serving latency: whole-step graph replays back to
        # back, no flush between them (the working set stays in L2)
        reps = 50
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            step_whole()
        z.record(stream)
        torch.cuda.synchronize()
        latency = {"us_per_step": a.elapsed_time(z) * 1e3 / reps, "reps": reps,
                   "timing": "CUDA graph replays back to back, L2 warm (no flush)"}
    step_ms = max_over_ranks(step_ms, world, device)
    decode_ms = max_over_ranks(decode_ms, world, device)
    total_bytes = sum_over_ranks(by["step"] * args.steps, world, device)
    total_rows = sum_over_ranks(wl.rows * args.steps, world, device)
    value = total_bytes / (step_ms * 1e-3) / 1e9

    # End to end through the public API with host buffers: per step the
    # inputs go host -> device from pinned memory (packed in one buffer, one
    # copy), the step runs on them, and the output comes back.
    names = ["q", "k_new", "v_new", "table", "positions"] + (
        ["sinks"] if batch.sinks is not None else [])
    packed = PackedInputs({k: getattr(batch, k) for k in names}, device)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = packed.bytes
    d2h = host_out.numel() * host_out.element_size()

    def run_step(inp, o):
        """One step on the input tensors `inp`, output into `o`."""
        kw = dict(num_kv_heads=wl.kv_heads, out=o, workspace=ws,
                  pages_per_split=args.pages_per_split, kernel=KERNEL_IDS[args.kernel])
        if fused:
            pgd.paged_decode_step(inp["q"], inp["k_new"], inp["v_new"], batch.k_pool,
                                  batch.v_pool, inp["table"], inp["positions"], inp.get("sinks"),
                                  wl.window, wl.scale, **kw)
            return
        qq = inp["q"]
        if args.rope:
            q_rot.copy_(inp["q"])
            pgd.rope_append_paged(q_rot, inp["k_new"], inp["v_new"], inp["table"],
                                  inp["positions"], batch.k_pool, batch.v_pool, theta=1e6)
            qq = q_rot
        else:
            pgd.kv_append_paged(inp["k_new"], inp["v_new"], inp["table"], inp["positions"],
                                batch.k_pool, batch.v_pool)
        pgd.paged_decode_attention(qq, batch.k_pool, batch.v_pool, inp["table"],
                                   inp["positions"], inp.get("sinks"), wl.window, wl.scale, **kw)

    def e2e_step():
        packed.upload()
        run_step(packed.views, out)
        host_out.copy_(out, non_blocking=True)

    # Back-to-back steps (inputs larger than L2) are pipelined as a serving
    # loop would run them: step i + 1's inputs go up on a copy stream into a
    # second set of device buffers while step i computes, and step i's output
    # comes down while step i + 1 computes; every copy is inside the timed
    # region.  (Steps between L2 flushes run one at a time.)
    pipelined = flush is None and fused
    if pipelined:
        bufs = [packed, PackedInputs({k: getattr(batch, k) for k in names}, device,
                                     host=packed.host)]
        outs = [torch.empty_like(out) for _ in range(2)]
        copy = torch.cuda.Stream(device)
        ready = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer j are up
        freed = [torch.cuda.Event() for _ in range(2)]   # the step on buffer j is done

        def upload(j):
            with torch.cuda.stream(copy):
                copy.wait_event(freed[j])
                bufs[j].upload()
                ready[j].record(copy)

        def compute(j):
            stream.wait_event(ready[j])
            run_step(bufs[j].views, outs[j])
            freed[j].record(stream)

        def download(j):
            with torch.cuda.stream(copy):
                copy.wait_event(freed[j])
                host_out.copy_(outs[j], non_blocking=True)

        def e2e_run(n, start):
            copy.wait_event(start)
            upload(0)
            for i in range(n):
                j = i % 2
                compute(j)
                if i + 1 < n:
                    upload(1 - j)
                download(j)
            last = torch.cuda.Event()
            last.record(copy)
            stream.wait_event(last)

    if pipelined:
        warm = torch.cuda.Event()
        warm.record(stream)
        e2e_run(2, warm)
    else:
        for _ in range(2):
            e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    if pipelined:
        e0.record(stream)
        e2e_run(args.steps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
    elif flush is None:
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
    else:
        for i in range(args.steps):
            flush(i)
            e0.record(stream)
            e2e_step()
            e1.record(stream)
            torch.cuda.synchronize()
            e2e_ms += e0.elapsed_time(e1)
    barrier(world)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    decode_s = decode_ms * 1e-3 / args.steps
    # the decode call's algorithmic bytes; with the append fused in, its
    # read and write are part of the call
    call_bytes = by["decode"] + (by["append"] if fused else 0)
    achieved = call_bytes / decode_s / 1e9
    digest = source_digest()
    traffic = kernel_traffic(digest, wl.name)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(wl), "rows_per_gpu": wl.rows,
                   "pool_pages_per_gpu": lay.num_pages,
                   "pool_gb_per_gpu": 2 * lay.num_pages * wl.kv_heads * 64 * wl.head_dim * 2 / 1e9,
                   "l2": "inputs larger than L2" if flush is None else L2Flush.label,
                   "timing": "direct calls, back to back" if flush is None
                   else "CUDA graph replay of each whole step; each call alone for its span",
                   "pages_per_split": args.pages_per_split or "auto",
                   "kernel": args.kernel, "rope": bool(args.rope), "fused_append": bool(fused),
                   "parallelism": f"replicas over rows x{world}"},
        "row_tokens_per_s": total_rows / (step_ms * 1e-3),
        "pct_of_nominal_8tbs": 100.0 * value / world / NOMINAL_HBM_GBS,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "latency_back_to_back": latency,
        "append_ms_per_step": None if fused else append_ms / args.steps,
        "decode_ms_per_step": decode_ms / args.steps,
        "bytes_per_step_per_gpu": by,
        "roofline": {"bound": "hbm",
                     "kernel": "paged_decode_step (the decode call with the append fused in)"
                     if fused else "paged_decode_attention (the decode call)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic, "algorithmic_bytes_per_launch": call_bytes},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                "copies": ("inputs packed in one pinned buffer, one upload per step; "
                           + ("overlapped with the neighbouring steps' compute (two buffer sets)"
                              if pipelined else "in line with each step"))},
        "gpu_launches": ((0 if fused else 1) + pgd.attention_kernel_count(
            dims, 0, wl.window, args.pages_per_split, KERNEL_IDS[args.kernel])) * args.steps,
        "clocks": clk,
        "kernel_source_digest": digest,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batch, out)
    del batch, ws
    torch.cuda.empty_cache()
    return line


def prefill_work(wl, b) -> dict:
    """Algorithmic work of one prefill step.  Bytes: per row, the K/V of the
    union of its tokens' attended positions, read once; q read, out written;
    the tokens' K/V read and written into the pool.  FLOPs: per token and
    query head, 2 * D for each attended key in Q.K^T and again in P.V."""
    pos = b.positions_np.astype(np.int64)
    lo = np.maximum(pos - wl.window + 1, 0) if wl.window > 0 else np.zeros_like(pos)
    attended = pos - lo + 1
    row_bytes = 2 * wl.kv_heads * wl.head_dim * 2
    kv = 0
    for r in np.unique(b.rows_np):
        sel = b.rows_np == r
        # the union of the tokens' ranges [lo, pos]: merge them in order of lo
        covered, end = 0, -1
        for a, z in sorted(zip(lo[sel].tolist(), pos[sel].tolist())):
            if z > end:
                covered += z - max(a, end + 1) + 1
                end = z
        kv += covered * row_bytes
    tokens = len(pos)
    q_out = 2 * tokens * wl.q_heads * wl.head_dim * 2
    writes = 2 * tokens * row_bytes
    flops = int(attended.sum()) * wl.q_heads * wl.head_dim * 4
    return {"kv": kv, "q_out": q_out, "writes": writes, "bytes": kv + q_out + writes,
            "flops": flops, "tokens": tokens}


# --kernel names -> PGD_KERNEL_* values
KERNEL_IDS = {"auto": 0, "tensor": 1, "cuda": 2, "tiled": 3, "umma": 4, "pair": 5}


def measured_tensor_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def run_prefill(args, wl):
    """Prefill step over the packed chunks (one GPU): one paged_prefill_step
    call (the tokens' writes, then the attention), or with --two-calls
    page_slots + kv_write_slots + paged_prefill_attention."""
    import paged_gqa_decode_gb300 as pgd
    from pgd_inputs import PREFILL_WORKLOADS, make_prefill_batch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    b = make_prefill_batch(wl, 2000 + list(PREFILL_WORKLOADS).index(wl.name), device)
    work = prefill_work(wl, b)
    opts = dict(num_kv_heads=wl.kv_heads, pages_per_split=args.pages_per_split,
                kernel=KERNEL_IDS[args.kernel])
    out = torch.empty_like(b.q)
    dims = pgd.make_dims(rows=work["tokens"], num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                         head_dim=wl.head_dim, num_pages=b.num_pages,
                         max_pages_per_row=b.table.shape[1])
    ws = torch.empty(max(16, pgd.paged_decode_workspace_bytes(dims, args.pages_per_split)),
                     dtype=torch.uint8, device=device)
    slots = torch.empty(work["tokens"], dtype=torch.int32, device=device)

    def attention():
        pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                    b.sinks, wl.window, wl.scale, out=out, workspace=ws, **opts)

    def step():
        if not args.two_calls:
            pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.table, b.rows,
                                   b.positions, b.sinks, wl.window, wl.scale, out=out,
                                   workspace=ws, **opts)
            return
        s_ = pgd.page_slots(b.table, b.positions, b.rows, num_pages=b.num_pages)
        pgd.kv_write_slots(b.k_new, b.v_new, s_, b.k_pool, b.v_pool)
        attention()

    for _ in range(args.warmup):
        step()
    assert pgd.get_device_error() == pgd.OK
    flush = L2Flush(device)
    e = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush(i)
        e[i][0].record(stream)
        step()
        e[i][1].record(stream)
    torch.cuda.synchronize()
    assert pgd.get_device_error() == pgd.OK
    ms = sum(a.elapsed_time(z) for a, z in e) / args.steps
    # the attention call alone (its kernels: the block-order pass and the
    # attention kernel), between the same flushes, for the roofline
    spans = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush(i)
        spans[i][0].record(stream)
        attention()
        spans[i][1].record(stream)
    torch.cuda.synchronize()
    assert pgd.get_device_error() == pgd.OK
    attn_ms = sum(a.elapsed_time(z) for a, z in spans) / args.steps
    del slots
    hbm, hbm_kind = measured_peak()
    tf, tf_kind = measured_tensor_peak()
    gbs = work["bytes"] / (ms * 1e-3) / 1e9
    tflops = work["flops"] / (ms * 1e-3) / 1e12
    attn_tflops = work["flops"] / (attn_ms * 1e-3) / 1e12
    attn_gbs = (work["kv"] + work["q_out"]) / (attn_ms * 1e-3) / 1e9
    bound = "tensor" if work["flops"] / (tf * 1e12) > work["bytes"] / (hbm * 1e9) else "hbm"
    line = {
        "metric": "paged prefill attention: tokens/s (achieved GB/s, TFLOP/s)",
        "value": work["tokens"] / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "f32", "storage_dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {wl.rows} rows, {wl.q_heads}q/{wl.kv_heads}kv, "
                               f"d{wl.head_dim}, prefix U[{wl.prefix_lo},{wl.prefix_hi}], "
                               f"chunk {wl.chunk}, window {wl.window}, sinks {wl.sinks}",
                   "tokens": work["tokens"], "l2": L2Flush.label,
                   "kernel": args.kernel,
                   "step": "page_slots + kv_write_slots + paged_prefill_attention"
                   if args.two_calls else "paged_prefill_step (writes, then attention)"},
        "gbs": gbs, "tflops": tflops, "attention_ms_per_step": attn_ms,
        "roofline": {"bound": bound,
                     "kernel": "paged_prefill_attention (the attention call: block-order "
                               "pass and attention kernel), timed alone between flushes",
                     "achieved": attn_tflops if bound == "tensor" else attn_gbs,
                     "peak": tf if bound == "tensor" else hbm,
                     "peak_kind": tf_kind if bound == "tensor" else hbm_kind,
                     "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                     "frac": attn_tflops / tf if bound == "tensor" else attn_gbs / hbm,
                     "algorithmic_flops_per_launch": work["flops"]},
        "work": work,
        # the step's kernels: page_slots + kv_write_slots + the attention
        # call's, or the prefill step's
        "gpu_launches": ((2 + pgd.attention_kernel_count(
            dims, b.table.shape[0], wl.window, args.pages_per_split, KERNEL_IDS[args.kernel]))
            if args.two_calls else pgd.prefill_step_kernel_count(
                dims, b.table.shape[0], wl.window, args.pages_per_split,
                KERNEL_IDS[args.kernel])) * args.steps,
    }
    print(json.dumps(line), flush=True)


def run_rows(args, wl):
    """decode_rows step over dense per-row caches: write_rows + decode."""
    import paged_gqa_decode_gb300 as pgd
    from pgd_inputs import ROWS_WORKLOADS, make_rows_batch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    b = make_rows_batch(wl, 3000 + list(ROWS_WORKLOADS).index(wl.name), device)
    by = algorithmic_bytes(wl, b.positions_np)
    out = torch.empty_like(b.q)
    kernel = KERNEL_IDS[args.kernel]

    def step():
        if not args.two_calls:   # the append inside the decode launch
            pgd.decode_rows_step(b.q, b.k_new, b.v_new, b.cache_k, b.cache_v, b.positions,
                                 b.sinks, wl.window, wl.scale, out=out,
                                 pages_per_split=args.pages_per_split, kernel=kernel)
            return
        pgd.kv_append_rows(b.k_new, b.v_new, b.positions, b.cache_k, b.cache_v)
        pgd.decode_rows_attention(b.q, b.cache_k, b.cache_v, b.positions, b.sinks, wl.window,
                                  wl.scale, out=out, pages_per_split=args.pages_per_split,
                                  kernel=kernel)

    for _ in range(args.warmup):
        step()
    assert pgd.get_device_error() == pgd.OK
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.synchronize()
    flush = L2Flush(device)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush(i)
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert pgd.get_device_error() == pgd.OK
    ms = sum(a.elapsed_time(z) for a, z in ev) / args.steps
    peak, kind = measured_peak()
    gbs = by["step"] / (ms * 1e-3) / 1e9
    line = {
        "metric": "decode_rows attention (dense per-row caches): achieved HBM GB/s; row-tokens/s",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "storage_dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{describe(wl)}, dense caches MaxSeq {b.max_seq}",
                   "l2": L2Flush.label,
                   "timing": "CUDA graph replay per step (write_rows + decode" + (", two calls)" if args.two_calls else " in one launch)")},
        "row_tokens_per_s": wl.rows / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "peak_kind": kind,
                     "unit": "GB/s", "frac": gbs / peak},
        "bytes_per_step": by,
        "gpu_launches": ((1 if args.two_calls else 0) + pgd.attention_kernel_count(
            pgd._dense_dims(b.cache_k, wl.rows, wl.q_heads), 0, wl.window,
            args.pages_per_split, kernel)) * args.steps,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pgd", "reference"], default="pgd")
    ap.add_argument("--path", choices=["decode", "prefill", "rows"], default="decode",
                    help="decode step over pages (default), packed prefill chunks, or "
                         "decode_rows over dense per-row caches")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help=f"decode: {', '.join(WORKLOADS)}; prefill: mistral_prefill, "
                         "gptoss_prefill_sliding")
    ap.add_argument("--pages-per-split", type=int, default=0)
    ap.add_argument("--kernel", choices=list(KERNEL_IDS), default="auto",
                    help="kernel variant: decode tensor-core or CUDA-core products; prefill "
                         "also the token-block kernels (mma.sync 'tiled', tcgen05 'umma', tcgen05 on "
                         "pairs of SMs 'pair')")
    ap.add_argument("--two-calls", action="store_true",
                    help="kv_append_paged and paged_decode_attention as two calls (default: "
                         "one paged_decode_step call, the append inside the decode launch); "
                         "with --path prefill, page_slots + kv_write_slots + "
                         "paged_prefill_attention instead of one paged_prefill_step call")
    ap.add_argument("--rope", action="store_true",
                    help="decode path: fuse rope_rows (base 1e6) into the append")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's row count (small profiling cases)")
    ap.add_argument("--reference-rows", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="decode path: measure only --workload (by default the headline "
                         "workload's line also carries the other four under 'workloads')")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.path == "prefill":
        from pgd_inputs import PREFILL_WORKLOADS
        name = args.workload if args.workload in PREFILL_WORKLOADS else "mistral_prefill"
        wl = PREFILL_WORKLOADS[name]
        if args.rows > 0:
            wl = wl.replace(rows=args.rows)
        run_prefill(args, wl)
        return
    if args.path == "rows":
        from pgd_inputs import ROWS_WORKLOADS
        name = args.workload if args.workload in ROWS_WORKLOADS else "gptoss_rows_serve"
        wl = ROWS_WORKLOADS[name]
        if args.rows > 0:
            wl = wl.replace(rows=args.rows)
        run_rows(args, wl)
        return
    if args.workload not in WORKLOADS:
        ap.error(f"unknown decode workload {args.workload}")
    wl = WORKLOADS[args.workload]
    if args.rows > 0:
        wl = wl.replace(rows=args.rows)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_pgd(args, wl)
    world, _, _ = dist_env()
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
