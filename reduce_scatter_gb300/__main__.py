"""Command-line runner in the manner of the Distributed GEMM example.

    python -m reduce_scatter_gb300 --m=16384 --n=106496 --k=16384 --warmup-iterations=10 --iterations=100

Runs one plan (all TP ranks on this GPU) on seeded synthetic inputs, checks D
against a single-device GEMM, and prints the disposition, the average runtime
and the throughput.  The flags follow the example's (Distributed GEMM README,
"Getting started": --m --n --k --l --alpha --beta --iterations
--warmup-iterations --eps), plus --tp and --schedule, which the example fixes
at build time, --mode (fused, or the GEMM-only and serial copy-then-GEMM
timings), --seed and --dist.

The single-device reference is the same kernel run unsharded (tp = 1): the
AllGather schedules keep every output's K order, so they match it bit for bit
(eps 0); the ReduceScatter schedules sum the K-slabs in another order and
match within a tolerance.  The check is

    max |D - D_ref| <= eps * max |D_ref|

(eps = 0: bit-identical).  Inputs from the package's seeded generator: A, B
and (when beta != 0) C drawn from --dist, uniform in [-1, 1) by default.
"""

from __future__ import annotations

import argparse
import sys


def parse(argv=None):
    from reduce_scatter_gb300 import dg

    ap = argparse.ArgumentParser(prog="python -m reduce_scatter_gb300",
                                 description="Distributed GEMM on one GB300: all TP ranks emulated on this GPU.")
    ap.add_argument("--m", type=int, default=16384, help="M extent of the GEMM")
    ap.add_argument("--n", type=int, default=106496, help="N extent of the GEMM")
    ap.add_argument("--k", type=int, default=16384, help="K extent of the GEMM")
    ap.add_argument("--l", type=int, default=1, help="L extent (batch) of the GEMM")
    ap.add_argument("--alpha", type=float, default=1.0, help="epilogue scalar alpha")
    ap.add_argument("--beta", type=float, default=0.0, help="epilogue scalar beta")
    ap.add_argument("--iterations", type=int, default=100, help="profiling iterations")
    ap.add_argument("--warmup-iterations", type=int, default=10, help="warmup iterations before profiling")
    ap.add_argument("--eps", type=float, default=0.0, help="threshold for the error against the reference GEMM")
    ap.add_argument("--tp", type=int, default=8, choices=[1, 2, 4, 8], help="tensor-parallel ranks")
    ap.add_argument("--schedule", default="AllGather1D_TilingCD_RotatingA", choices=sorted(dg.SCHEDULE_BY_NAME),
                    help="distributed GEMM schedule")
    ap.add_argument("--mode", default="fused", choices=["fused", "gemm_only", "serial"],
                    help="fused (transfers overlapping the kernel), gemm_only (transfers skipped, "
                         "slots pre-filled) or serial (transfers, then the kernel)")
    ap.add_argument("--seed", type=int, default=1, help="seed of the synthetic inputs")
    ap.add_argument("--dist", default="uniform:-1:1",
                    help="input distribution: uniform:LO:HI or normal:MEAN:STD (default uniform:-1:1)")
    a = ap.parse_args(argv)
    for name in ("m", "n", "k", "l"):
        if getattr(a, name) < 1:
            ap.error(f"--{name} must be >= 1")
    if a.iterations < 1 or a.warmup_iterations < 0:
        ap.error("--iterations must be >= 1 and --warmup-iterations >= 0")
    if a.eps < 0:
        ap.error("--eps must be >= 0")
    try:
        kind, x, y = a.dist.split(":")
        a.dist = (kind, float(x), float(y))
        if kind not in ("uniform", "normal") or (kind == "uniform" and not a.dist[1] < a.dist[2]) or \
                (kind == "normal" and not a.dist[2] > 0):
            raise ValueError
    except ValueError:
        ap.error("--dist must be uniform:LO:HI (LO < HI) or normal:MEAN:STD (STD > 0)")
    return a


def main(argv=None) -> int:
    a = parse(argv)
    import torch

    from reduce_scatter_gb300 import dg, synth

    if not torch.cuda.is_available():
        print("no CUDA device", file=sys.stderr)
        return 2
    sched = dg.SCHEDULE_BY_NAME[a.schedule]
    dev = torch.device("cuda", torch.cuda.current_device())

    def draw(stream, shape):
        return synth.tensor_bits_torch(a.seed, stream, shape, a.dist, device=dev).view(torch.bfloat16)

    A = draw(synth.STREAM_A, (a.l, a.m, a.k))
    B = draw(synth.STREAM_B, (a.l, a.n, a.k))  # stored N x K (its transpose), K innermost
    C = draw(synth.STREAM_C, (a.l, a.m, a.n)) if a.beta != 0 else None
    D = torch.empty((a.l, a.m, a.n), dtype=torch.bfloat16, device=dev)

    plan = dg.Plan(a.m, a.n, a.k, a.l, a.tp, sched, a.alpha, a.beta)
    modes = {"fused": dg.MODE_FUSED, "gemm_only": dg.MODE_GEMM_ONLY, "serial": dg.MODE_SERIAL}
    info = plan.info()
    ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
    main_s = torch.cuda.current_stream(dev)
    copy_s = torch.cuda.Stream(dev)

    # one fused run first: it fills the receive slots GEMM_ONLY reads
    plan.run(A, B, C, D, ws, main_s, copy_s)
    plan.check(ws, main_s)
    plan.set_mode(modes[a.mode])
    if a.mode == "serial":  # an RS plan's serial baseline needs the larger workspace, sized in that mode
        ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
    for _ in range(a.warmup_iterations):
        plan.run(A, B, C, D, ws, main_s, copy_s)
    plan.check(ws, main_s)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main_s)
    for _ in range(a.iterations):
        plan.run(A, B, C, D, ws, main_s, copy_s)
    stop.record(main_s)
    plan.check(ws, main_s)
    ms = start.elapsed_time(stop) / a.iterations

    # single-device reference: the same GEMM unsharded
    ref_sched = sched if sched in (dg.AG_ROTATING_A, dg.AG_ROTATING_B) else dg.AG_ROTATING_A
    ref_plan = dg.Plan(a.m, a.n, a.k, a.l, 1, ref_sched, a.alpha, a.beta)
    ref_ws = torch.zeros(max(ref_plan.workspace_bytes(), 256), dtype=torch.uint8, device=dev)
    D_ref = torch.empty_like(D)
    ref_plan.run(A, B, C, D_ref, ref_ws, main_s, main_s)
    ref_plan.check(ref_ws, main_s)
    scale = D_ref.float().abs().max().item()
    err = (D.float() - D_ref.float()).abs().max().item()
    if a.eps == 0:
        passed = torch.equal(D.view(torch.int16), D_ref.view(torch.int16))
    else:
        passed = err <= a.eps * scale
    flops = 2.0 * a.m * a.n * a.k * a.l
    tflops = flops / (ms * 1e-3) / 1e12
    print(f"  Schedule: {a.schedule}, TP={a.tp} (all ranks on one GPU), mode {a.mode}")
    print(f"  Problem size: {a.m} x {a.n} x {a.k} x {a.l}")
    print(f"  Local GEMM problem size: {info['local_m']} x {info['local_n']} x {info['local_k']} x {a.l}")
    print(f"  Disposition (eps: {a.eps:g}): {'Passed' if passed else 'Failed'}"
          f" (max |D - D_ref| / max |D_ref| = {err / max(scale, 1e-30):.3e})")
    print(f"  Avg runtime: {ms:.5f} ms")
    print(f"  TFLOPS: {tflops:.2f} (the whole problem on this GPU; {tflops / a.tp:.2f} per emulated rank)")
    return 0 if passed else 1


if __name__ == "__main__":
    sys.exit(main())
