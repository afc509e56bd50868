#!/usr/bin/env python
"""Benchmark of the communication-fused TP GEMM on GB300.

``python bench.py --gpus N --steps K --warmup W [--workload NAME] [--impl dg|reference]``

One step = one fused run of the whole problem (every virtual rank, every
rotation step, all shard transfers) on one GPU.  With N > 1 (torchrun, one
process per GPU) every GPU runs its own replica of the problem: the path is
emulated on one GPU and has no exchange between GPUs, so scaling is weak and
``value`` is the sum over replicas (N x flops / slowest rank's time).

Prints one JSON line (rank 0).  ``metric``/``unit``: TFLOP/s of the fused
run; ``roofline``: the fused kernel against the measured dense-bf16 peak;
``copy_hidden_fraction``: clamp((t_copy + t_gemm - t_fused) / t_copy, 0, 1)
with t_copy = t_serial - t_gemm; ``e2e``: the same metric with inputs copied
from pinned host memory and D copied back inside the timed region;
``cpu_baseline``: the CPU oracle on a bounded sample of the same problem.

``--impl reference`` times the CPU oracle (the slow reference program) on the
same workload and prints its own line (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from reduce_scatter_gb300 import configs  # noqa: E402

METRIC = "fused TP-GEMM TFLOP/s and % of GB300 BF16 peak; copy-hidden fraction"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAK_TFLOPS = 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["dg", "reference"], default="dg")
    ap.add_argument("--workload", choices=sorted(configs.WORKLOADS), default=configs.DEFAULT)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-e2e-pipelined", action="store_true")
    ap.add_argument("--no-modes", action="store_true", help="skip the GEMM_ONLY / SERIAL timings")
    ap.add_argument("--mode", choices=["fused", "gemm_only", "serial"], default="fused",
                    help="mode of the timed loop (gemm_only/serial for profilers that serialize streams)")
    ap.add_argument("--copy-streams", type=int, default=0, help="0 = the library default")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="extra plan option, e.g. L2_HINT=9 (names of dg.OPT_*)")
    ap.add_argument("--cpu-sample-rows", type=int, default=1024)
    ap.add_argument("--cpu-sample-cols", type=int, default=4096)
    ap.add_argument("--parity-rows", type=int, default=128,
                    help="rows of the sampled parity check on ranks other than 0 (rank 0 at N=1 checks the "
                         "CPU baseline's sample)")
    ap.add_argument("--parity-cols", type=int, default=1024)
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="store the DRAM bytes of an ncu --csv capture (dram__bytes_read.sum, "
                         "dram__bytes_write.sum, gpu__time_duration.sum of one dg_gemm launch) in "
                         "profiles/dram_traffic.json for --workload, tagged with the kernel source hash, "
                         "and exit")
    ap.add_argument("--record-command", default="", help="the ncu command line the CSV came from")
    ap.add_argument("--record-note", default="", help="a note stored with the record")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_PEAK_TFLOPS}, "fallback"


def kernel_source_hash() -> str:
    # the kernel and the host code that picks its variant and options
    h = hashlib.sha256()
    for name in ("dg_kernel.cuh", "dg_geom.h", "dg.cu"):
        with open(os.path.join(ROOT, "reduce_scatter_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


_UNIT = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
         "ns": 1.0, "nsecond": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}


def record_traffic(workload: str, csv_path: str, command: str, note: str) -> dict:
    """Parse one dg_gemm launch from an ncu --csv log and store it for the
    bench's roofline.traffic (only trusted while the kernel source is unchanged)."""
    import csv

    metrics, kernel = {}, None
    with open(csv_path, newline="") as f:
        rows = [r for r in csv.reader(line for line in f if line.startswith('"'))]
    head = rows[0]
    col = {name: i for i, name in enumerate(head)}
    for r in rows[1:]:
        if "dg_gemm" not in r[col["Kernel Name"]]:
            continue
        if kernel is not None and r[col["ID"]] != kernel[0]:
            break  # first captured launch only
        kernel = (r[col["ID"]], r[col["Kernel Name"]])
        val = float(r[col["Metric Value"]].replace(",", "")) * _UNIT.get(r[col["Metric Unit"]], float("nan"))
        metrics[r[col["Metric Name"]]] = val
    need = ("dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum")
    if kernel is None or any(k not in metrics for k in need):
        raise SystemExit(f"{csv_path}: no dg_gemm launch with {need}")
    rd, wr = int(metrics[need[0]]), int(metrics[need[1]])
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    rec[workload] = {"bytes_per_launch": rd + wr, "dram_bytes_read": rd, "dram_bytes_write": wr,
                     "kernel": kernel[1], "kernel_source_hash": kernel_source_hash(),
                     "gpu__time_duration_ns": int(metrics[need[2]]), "command": command, "note": note}
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec[workload]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open("/tmp/dg_clocks_%d.csv" % os.getpid(), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(loaded), "reasons": reasons}


def sample_indices(w, rows: int, cols: int):
    """Rows and columns of batch 0 of D that the oracle evaluates: spread
    evenly over every shard (and so over every rank's output)."""
    import numpy as np

    rows = min(rows, w.m)
    cols = min(cols, w.n)
    ridx = np.linspace(0, w.m - 1, rows).astype(np.int64)
    cidx = np.linspace(0, w.n - 1, cols).astype(np.int64)
    return ridx, cidx


def cpu_oracle_sample(w, rows: int, cols: int, keep_entries: bool = False):
    """Time the CPU oracle on rows x cols entries of D (all of K); with
    ``keep_entries`` also return the entries (for the parity check)."""
    import numpy as np

    from oracle import gemm as og
    from reduce_scatter_gb300 import synth

    LM, LN = w.l * w.m, w.l * w.n
    ridx, cidx = sample_indices(w, rows, cols)
    rows, cols = len(ridx), len(cidx)
    batch = 0
    if w.in_type == "bf16":
        a = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_A, (LM, w.k), ridx, w.dist_a))
        b = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_B, (LN, w.k), cidx, w.dist_b))
    else:
        a = og.fp8_bits_to_f64(synth.rows_fp8_bits_np(w.seed, synth.STREAM_A, (LM, w.k), ridx, w.dist_a,
                                                      w.in_type), w.in_type)
        b = og.fp8_bits_to_f64(synth.rows_fp8_bits_np(w.seed, synth.STREAM_B, (LN, w.k), cidx, w.dist_b,
                                                      w.in_type), w.in_type)
    c = None
    if w.beta != 0:
        crow = synth.rows_bits_np(w.seed, synth.STREAM_C, (LM, w.n), ridx, w.dist_c)[:, cidx - batch * w.n]
        c = og.bf16_bits_to_f64(crow)
    t0 = time.perf_counter()
    entries = og.gemm_entries(a, b, c, w.alpha * w.scale_a * w.scale_b, w.beta)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * cols * w.k
    try:
        from threadpoolctl import threadpool_info

        cores = max((i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"),
                    default=os.cpu_count())
    except Exception:
        cores = os.cpu_count()
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "seconds": dt,
           "sample": f"{rows} rows x {cols} columns of D (all K={w.k}) of {w.name}, fp64 numpy matmul; "
                     f"{flops:.3e} flop"}
    if keep_entries:
        out["entries"] = entries
    return out


PARITY_TOL = 2e-2  # max|D - D_oracle| <= PARITY_TOL * max|D_oracle| (bf16 inputs, fp32 accumulation)


def parity_check(d_sample, entries, rows, cols):
    """The timed run's D on the sampled entries against the oracle's."""
    import numpy as np

    got = np.asarray(d_sample, dtype=np.float64)
    finite = bool(np.isfinite(got).all())
    scale = float(max(np.abs(entries).max(), 1e-30))
    err = float(np.abs(got - entries).max() / scale) if finite else float("inf")
    return {"max_rel_err": err, "tol": PARITY_TOL, "rows": rows, "cols": cols, "ok": finite and err <= PARITY_TOL,
            "against": "oracle (fp64) on sampled entries of the timed run's D"}


# ------------------------------------------------------------ multi-rank


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of per-rank timings (ms) over all ranks.

    Every rank runs its own replica; the job is as slow as its slowest rank.
    """
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_replica: float, world: int, ms_slowest: float) -> float:
    """TFLOP/s of the whole job: every replica's work over the slowest rank's time."""
    return world * flops_per_replica / (ms_slowest * 1e-3) / 1e12


# ------------------------------------------------------------------ dg arm


def make_inputs(w, device):
    import torch

    from reduce_scatter_gb300 import synth

    chunk = 1 << 28  # fewer, larger generator launches
    if w.in_type == "bf16":
        A = synth.tensor_bits_torch(w.seed, synth.STREAM_A, (w.l, w.m, w.k), w.dist_a, device=device,
                                    chunk=chunk).view(torch.bfloat16)
        B = synth.tensor_bits_torch(w.seed, synth.STREAM_B, (w.l, w.n, w.k), w.dist_b, device=device,
                                    chunk=chunk).view(torch.bfloat16)
    else:  # fp8 bytes
        A = synth.tensor_fp8_bits_torch(w.seed, synth.STREAM_A, (w.l, w.m, w.k), w.dist_a, w.in_type,
                                        device=device, chunk=chunk)
        B = synth.tensor_fp8_bits_torch(w.seed, synth.STREAM_B, (w.l, w.n, w.k), w.dist_b, w.in_type,
                                        device=device, chunk=chunk)
    C = None
    if w.beta != 0:
        C = synth.tensor_bits_torch(w.seed, synth.STREAM_C, (w.l, w.m, w.n), w.dist_c, device=device,
                                    chunk=chunk).view(torch.bfloat16)
    return A, B, C


def input_bytes(w) -> int:
    """Bytes of A, B (and C when beta != 0) of a workload."""
    esz = 2 if w.in_type == "bf16" else 1
    return (w.l * w.m * w.k + w.l * w.n * w.k) * esz + (w.l * w.m * w.n * 2 if w.beta != 0 else 0)


def flushes_l2(w) -> bool:
    """Inputs smaller than twice the L2: the bench flushes L2 between steps."""
    return input_bytes(w) < 2 * L2_BYTES


def workload_config(w, world: int) -> dict:
    """The line's ``config``, the same for both arms."""
    return dict(w.describe(), parallelism=f"tp{w.tp} virtual ranks on 1 GPU" + (
        f", {world} replicas" if world > 1 else ""),
        l2="flushed between steps" if flushes_l2(w) else "inputs larger than L2 (no flush)")


def timed_loop(run, steps, warmup, stream, flush=None):
    """Per-step CUDA events on ``stream``; returns mean ms per step."""
    import torch

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.nvtx.range_push("timed loop")
    for s, e in ev:
        if flush is not None:
            flush()
        s.record(stream)
        run()
        e.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    return sum(s.elapsed_time(e) for s, e in ev) / steps


def copy_in_pieces(dst, src, piece_bytes=64 << 20):
    """dst.copy_(src) as copies of at most ``piece_bytes`` (flat views): copy engines take
    copies in issue order, so one multi-GB host copy would hold up the shard transfers."""
    d, s_ = dst.view(-1), src.view(-1)
    step = max(1, piece_bytes // d.element_size())
    for i in range(0, d.numel(), step):
        d[i:i + step].copy_(s_[i:i + step], non_blocking=True)


def e2e_pipelined(plan, ws, main, copy, A_h, B_h, C_h, A0, B0, C0, D0, steps):
    """End-to-end with two buffer sets: every step uploads its inputs from
    pinned host memory, runs, and downloads its D, but step i+1's upload and
    step i-1's download overlap step i's run (different copy engines and the
    two directions of the host link).  Returns ms per step over `steps`."""
    import torch

    dev = A0.device
    bufs = [(A0, B0, C0, D0), (torch.empty_like(A0), torch.empty_like(B0),
                               None if C0 is None else torch.empty_like(C0), torch.empty_like(D0))]
    D_h = [torch.empty(D0.shape, dtype=D0.dtype).pin_memory() for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ran = [ev(), ev()]      # step on buffer set b finished (inputs and D free after download)
    landed = [ev(), ev()]   # inputs of buffer set b uploaded
    fetched = [ev(), ev()]  # D of buffer set b downloaded
    for e in ran + fetched:
        e.record(main)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for i in range(steps):
        b = i & 1
        A, B, C, D = bufs[b]
        up.wait_event(ran[b])
        with torch.cuda.stream(up):
            copy_in_pieces(A, A_h)
            copy_in_pieces(B, B_h)
            if C is not None:
                copy_in_pieces(C, C_h)
        landed[b].record(up)
        main.wait_event(landed[b])
        main.wait_event(fetched[b])
        plan.run(A, B, C, D, ws, main, copy)
        ran[b].record(main)
        down.wait_event(ran[b])
        with torch.cuda.stream(down):
            copy_in_pieces(D_h[b], D)
        fetched[b].record(down)
    main.wait_event(fetched[0])
    main.wait_event(fetched[1])
    end.record(main)
    torch.cuda.synchronize()
    return {"ms_per_step": start.elapsed_time(end) / steps, "steps": steps,
            "mode": "two buffer sets: step i+1 upload and step i-1 download overlap step i"}


def run_dg(args, rank, world, dist):
    import torch

    from reduce_scatter_gb300 import dg

    w = configs.WORKLOADS[args.workload]
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    A, B, C = make_inputs(w, dev)
    D = torch.empty((w.l, w.m, w.n), dtype=torch.bfloat16, device=dev)
    plan = dg.Plan(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta, w.in_type, w.in_type, w.scale_a,
                   w.scale_b)
    if args.copy_streams > 0:
        plan.set_option(dg.OPT_COPY_STREAMS, args.copy_streams)
    for opt in args.option:
        name, val = opt.split("=")
        plan.set_option(getattr(dg, "OPT_" + name.upper()), int(val))
    ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    in_bytes = (A.numel() * A.element_size() + B.numel() * B.element_size()
                + (C.numel() * 2 if C is not None else 0))
    assert in_bytes == input_bytes(w)
    flush_buf = None
    if flushes_l2(w):
        flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush = (lambda: flush_buf.fill_(1.0)) if flush_buf is not None else None

    def run():
        plan.run(A, B, C, D, ws, main, copy)

    def barrier():
        if dist is not None:
            dist.barrier()

    mode = {"fused": dg.MODE_FUSED, "gemm_only": dg.MODE_GEMM_ONLY, "serial": dg.MODE_SERIAL}[args.mode]
    # correctness guard before timing: one run, device status must be clean.
    # GEMM_ONLY needs filled receive slots: fill them with a SERIAL run.
    plan.set_mode(dg.MODE_SERIAL if mode == dg.MODE_GEMM_ONLY else mode)
    run()
    plan.check(ws, main)
    plan.set_mode(mode)

    barrier()
    with ClockSampler(local) as clk:
        barrier()
        ms_fused = timed_loop(run, args.steps, args.warmup, main, flush)
        barrier()
    plan.check(ws, main)
    clocks = clk.summary()
    # the timed runs' D: the sampled entries for the oracle check, and (AG) all of it for the bit
    # comparison with the same kernel unsharded
    rows, cols = (args.cpu_sample_rows, args.cpu_sample_cols) if world == 1 else (args.parity_rows,
                                                                                  args.parity_cols)
    ridx, cidx = sample_indices(w, rows, cols)
    ri, ci = torch.from_numpy(ridx).to(dev), torch.from_numpy(cidx).to(dev)
    d_sample = D[0].index_select(0, ri).index_select(1, ci).float().cpu().numpy()
    ag = w.schedule in (dg.AG_ROTATING_A, dg.AG_ROTATING_B)
    D_fused = D.clone() if ag and w.tp > 1 and not args.no_modes and mode == dg.MODE_FUSED else None

    # latency-bound sizes: the same run replayed from a CUDA graph (one launch
    # of the whole captured run instead of its host-side enqueue)
    ms_graph = None
    if not args.no_modes and mode == dg.MODE_FUSED and ms_fused < 1.0:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plan.run(A, B, C, D, ws, torch.cuda.current_stream(), copy)
        ms_graph = timed_loop(graph.replay, args.steps, args.warmup, main, flush)
        plan.check(ws, main)
        del graph

    ms_gemm = ms_serial = None
    if (not args.no_modes and mode == dg.MODE_FUSED and w.schedule in (dg.AG_ROTATING_A, dg.AG_ROTATING_B)
            and w.tp > 1):
        plan.set_mode(dg.MODE_GEMM_ONLY)
        ms_gemm = timed_loop(run, max(3, args.steps // 2), 2, main, flush)
        plan.set_mode(dg.MODE_SERIAL)
        ms_serial = timed_loop(run, max(3, args.steps // 2), 2, main, flush)
        plan.set_mode(mode)
        plan.check(ws, main)

    # the same kernel on the unsharded problem (tp=1), and for the RS
    # schedules the non-fused baseline (per-rank partial GEMMs, then a
    # separate reduction kernel)
    ms_tp1 = ms_nonfused = None
    bit_exact = None
    if not args.no_modes and mode == dg.MODE_FUSED and w.tp > 1:
        p1 = dg.Plan(w.m, w.n, w.k, w.l, 1, w.schedule, w.alpha, w.beta, w.in_type, w.in_type, w.scale_a,
                     w.scale_b)
        ws1 = torch.zeros(max(p1.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
        ms_tp1 = timed_loop(lambda: p1.run(A, B, C, D, ws1, main, copy), max(3, args.steps // 2), 2, main, flush)
        p1.check(ws1, main)
        del ws1, p1
        if D_fused is not None:
            # AG keeps every output element's K order: the fused run equals tp = 1 bit for bit
            bit_exact = bool(torch.equal(D_fused.view(torch.int16), D.view(torch.int16)))
            del D_fused
            D_fused = None
        if w.schedule in (dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C):
            ps = dg.Plan(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta, w.in_type, w.in_type,
                         w.scale_a, w.scale_b)
            ps.set_mode(dg.MODE_SERIAL)
            wss = torch.zeros(max(ps.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
            ms_nonfused = timed_loop(lambda: ps.run(A, B, C, D, wss, main, main), max(3, args.steps // 2), 2,
                                     main, flush)
            ps.check(wss, main)
            del wss, ps

    e2e = None
    if not args.no_e2e:
        A_h = A.cpu().pin_memory()
        B_h = B.cpu().pin_memory()
        C_h = C.cpu().pin_memory() if C is not None else None
        D_h = torch.empty(D.shape, dtype=D.dtype).pin_memory()

        def run_e2e():
            # one C-ABI call with host buffers: uploads, the run and the download of D
            plan.run_host(A_h, B_h, C_h, None, D_h, A, B, C, D, ws, main, copy)

        e2e_steps = max(2, min(args.steps, 5))
        with ClockSampler(local) as clk_e2e:
            ms_e2e = timed_loop(run_e2e, e2e_steps, 3, main)
            plan.check(ws, main)
            # the device-only run right after, in the same thermal and power state: what the
            # end-to-end call adds beyond the kernel is the host link's share
            ms_dev_after = timed_loop(run, e2e_steps, 0, main)
            plan.check(ws, main)
        # the machine's host link on these buffers (it differs between boxes and sets the e2e floor)
        link = {}
        for name, dst, src in (("h2d_gbs", B, B_h), ("d2h_gbs", D_h, D)):
            t = timed_loop(lambda: dst.copy_(src, non_blocking=True), 3, 1, main)
            link[name] = round(src.numel() * src.element_size() / t / 1e6, 1)
        e2e = {"value": None, "unit": "TFLOP/s", "ms_per_step": ms_e2e, "steps": e2e_steps,
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": D.numel() * D.element_size(), "link": link,
               "clocks": clk_e2e.summary(), "device_ms_after": round(ms_dev_after, 4),
               "mode": "one dg_run_host call per step: inputs uploaded and D downloaded inside the call "
                       "(per-rank uploads gate the kernel's tiles, finished D blocks download during the run)"}
        if not args.no_e2e_pipelined:
            e2e["pipelined"] = e2e_pipelined(plan, ws, main, copy, A_h, B_h, C_h, A, B, C, D, e2e_steps + 2)
            plan.check(ws, main)
        del A_h, B_h, C_h, D_h

    # parity of the timed D on sampled entries: at N = 1 against the CPU baseline's own sample (main),
    # with N > 1 every rank checks a smaller sample of its replica
    parity = None
    if world > 1:
        ent = cpu_oracle_sample(w, rows, cols, keep_entries=True)["entries"]
        parity = parity_check(d_sample, ent, len(ridx), len(cidx))
        err_max, bad = max_over_ranks([parity["max_rel_err"], 0.0 if parity["ok"] else 1.0], dist, dev)
        parity.update(max_rel_err=err_max, ok=bad == 0.0, ranks=world)
    if parity is not None:
        parity["bit_exact_vs_tp1"] = bit_exact

    # max over ranks
    ms_fused, ms_gemm_m, ms_serial_m, ms_e2e, ms_tp1_m, ms_nonfused_m, ms_pipe = max_over_ranks(
        [ms_fused, ms_gemm or 0.0, ms_serial or 0.0, (e2e or {}).get("ms_per_step", 0.0), ms_tp1 or 0.0,
         ms_nonfused or 0.0, (e2e or {}).get("pipelined", {}).get("ms_per_step", 0.0)], dist, dev)
    if e2e is not None and "pipelined" in e2e:
        e2e["pipelined"]["ms_per_step"] = ms_pipe
    ms_tp1 = ms_tp1_m if ms_tp1 is not None else None
    ms_nonfused = ms_nonfused_m if ms_nonfused is not None else None
    if rank != 0:
        return None, None
    ms_gemm = ms_gemm_m if ms_gemm is not None else None
    ms_serial = ms_serial_m if ms_serial is not None else None

    peaks, peak_kind = measured_peaks()
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAK_TFLOPS))
    peak_sust = float(peaks.get("bf16_tflops_sustained", peak_burst))
    if w.in_type != "bf16":
        # fp8 dense peak: the measured bf16 peak x the nominal fp8 / bf16 ratio (4.5 / 2.25)
        peak_burst, peak_sust = 2.0 * peak_burst, 2.0 * peak_sust
    # The denominator matches how the kernel was timed: a timed region of back-to-back runs that
    # lasts long enough for the power limit to act (>= 0.5 s) is held to the sustained peak (the
    # GEMM measured back to back for seconds under the power cap); a short one to the burst peak.
    long_run = args.steps * ms_fused >= 500.0
    peak = peak_sust if long_run else peak_burst
    peak_note = "%s bf16 %s%s" % (peak_kind, "sustained" if long_run else "burst",
                                  "" if w.in_type == "bf16" else " x 2 (nominal fp8 / bf16 dense ratio)")
    if long_run:
        peak_note += " (timed region: %.2f s of back-to-back runs)" % (args.steps * ms_fused / 1e3)
    per_gpu = w.flops / (ms_fused * 1e-3) / 1e12
    value = whole_job_tflops(w.flops, world, ms_fused)
    hidden = None
    if ms_gemm is not None and ms_serial is not None:
        t_copy = ms_serial - ms_gemm
        hidden = max(0.0, min(1.0, (t_copy + ms_gemm - ms_fused) / t_copy)) if t_copy > 0 else None
    if e2e is not None:
        e2e["ms_per_step"] = ms_e2e
        e2e["value"] = whole_job_tflops(w.flops, world, ms_e2e)
        if "pipelined" in e2e:
            e2e["pipelined"]["value"] = whole_job_tflops(w.flops, world, e2e["pipelined"]["ms_per_step"])
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_fused, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.in_type == "bf16" else w.in_type + " inputs, fp32 accumulation, bf16 output",
        "data": "synthetic (seeded SplitMix64 inputs with the workload's distributions)",
        "mode": args.mode,
        "options": args.option,
        "config": workload_config(w, world),
        "pct_of_peak": round(100.0 * per_gpu / peak, 2),
        "ms_gemm_only": None if ms_gemm is None else round(ms_gemm, 4),
        "ms_serial": None if ms_serial is None else round(ms_serial, 4),
        "copy_hidden_fraction": None if hidden is None else round(hidden, 4),
        "fused_over_gemm_only": None if ms_gemm is None else round(ms_fused / ms_gemm, 4),
        "ms_unsharded_tp1": None if ms_tp1 is None else round(ms_tp1, 4),
        "ms_graph_replay": None if ms_graph is None else round(ms_graph, 4),
        "ms_rs_nonfused_baseline": None if ms_nonfused is None else round(ms_nonfused, 4),
        "fused_speedup_vs_nonfused": None if ms_nonfused is None else round(ms_nonfused / ms_fused, 4),
        "roofline": {"bound": "tensor", "achieved": round(per_gpu, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(per_gpu / peak, 4), "peak_source": peak_note,
                     "frac_of_burst": round(per_gpu / peak_burst, 4),
                     "frac_of_sustained": round(per_gpu / peak_sust, 4),
                     "traffic": recorded_traffic(w.name), "kernel": "dg::dg_gemm_kernel"},
        "clocks": clocks,
        "gpu_launches": args.steps,  # one dg_gemm_kernel launch per fused step
        "e2e": e2e,
        "parity": parity,
    }
    return line, (d_sample, bit_exact, len(ridx), len(cidx))


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = configs.WORKLOADS[args.workload]

    if args.record_traffic:
        print(json.dumps(record_traffic(args.workload, args.record_traffic, args.record_command, args.record_note)))
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        steps = []
        for _ in range(max(1, args.warmup)):
            cpu_oracle_sample(w, max(64, args.cpu_sample_rows // 4), max(256, args.cpu_sample_cols // 4))
        for _ in range(args.steps):
            steps.append(cpu_oracle_sample(w, max(64, args.cpu_sample_rows // 4), max(256, args.cpu_sample_cols // 4)))
        secs = sum(s["seconds"] for s in steps) / len(steps)
        val = sum(s["value"] for s in steps) / len(steps)
        line = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(w, world),
                "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": steps[0]["cores"],
                                 "kind": "oracle", "sample": steps[0]["sample"]},
                "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch.distributed as tdist

        backend = "nccl"
        tdist.init_process_group(backend=backend)
        dist = tdist
    line, sample = run_dg(args, rank, world, dist)
    ok = True
    if line is not None:
        if world == 1:
            # the CPU baseline's timed oracle entries double as the parity check of the timed D
            d_sample, bit_exact, rows, cols = sample
            base = cpu_oracle_sample(w, args.cpu_sample_rows, args.cpu_sample_cols, keep_entries=True)
            line["parity"] = parity_check(d_sample, base.pop("entries"), rows, cols)
            line["parity"]["bit_exact_vs_tp1"] = bit_exact
            base.pop("seconds", None)
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = base
        ok = line["parity"]["ok"] and line["parity"].get("bit_exact_vs_tp1") is not False
        print(json.dumps(line), flush=True)
        if not ok:
            print("bench: the timed run's D fails the parity check", file=sys.stderr)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())
