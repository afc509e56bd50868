"""Named workloads: the problem sizes, schedules and input distributions of
the pages' benchmarks, as synthetic inputs.

* ``ag_a_tp2_256``: AllGather RotatingA, TP=2, 256^3 (latency / parity case).
* ``ag_a_tp2_blog``: the all_gather+matmul blog's 8192^2-per-rank,
  world_size=2 shape (gathered M = 16384, N = K = 8192), U[0,1) inputs
  (the blog uses torch.rand), here in bf16.
* ``ag_a_tp8_pr``: the Distributed GEMM pull request's TP=8 benchmark,
  16384 x 106496 x 16384; activations N(0,1), weights N(0,0.02).
* ``rs_a_tp8``: ReduceScatter TilingA RotatingC, TP=8, 16384 x 8192 x 28672
  (K split 8 x 3584); A N(0,1), B N(0,0.02).
* ``ag_b_tp4_batched`` / ``rs_b_tp4_batched``: RotatingB / TilingB RotatingC,
  TP=4, 8192 x 53248 x 8192, L=2, alpha=0.5, beta=1, C N(0,1).
* ``rs_b_tp4_quarter`` / ``rs_b_tp4_half``: rs_b_tp4_batched with N / 4 (N / 2)
  and L = 1, for profiler captures.
* ``ag_a_tp8_pr_small``: ag_a_tp8_pr with M / 2 and N / 8, for profiler
  captures of the headline kernel.
* ``ag_a_tp8_pr_e4m3`` / ``rs_a_tp8_e4m3``: the TP=8 problems with e4m3
  operands (the scaled variant): both drawn N(0,1) and rounded to e4m3, the
  weight's 0.02 standard deviation carried by scale_b.

A is the activation (M x K), B the weight stored N x K, C the epilogue input.
"""

from __future__ import annotations

from dataclasses import dataclass

U11 = ("uniform", -1.0, 1.0)
U01 = ("uniform", 0.0, 1.0)
N1 = ("normal", 0.0, 1.0)
N002 = ("normal", 0.0, 0.02)


@dataclass(frozen=True)
class Workload:
    name: str
    schedule: int
    tp: int
    m: int
    n: int
    k: int
    l: int = 1
    alpha: float = 1.0
    beta: float = 0.0
    dist_a: tuple = U11
    dist_b: tuple = U11
    dist_c: tuple = N1
    seed: int = 1
    in_type: str = "bf16"  # A and B element type: bf16, e4m3 or e5m2
    scale_a: float = 1.0
    scale_b: float = 1.0

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k * self.l

    def describe(self) -> dict:
        from . import dg

        return {"workload": self.name, "schedule": dg.SCHEDULE_NAMES[self.schedule], "tp": self.tp,
                "m": self.m, "n": self.n, "k": self.k, "l": self.l, "alpha": self.alpha, "beta": self.beta,
                "dist_a": list(self.dist_a), "dist_b": list(self.dist_b),
                "dist_c": list(self.dist_c) if self.beta else None, "seed": self.seed,
                "in_type": self.in_type, "scale_a": self.scale_a, "scale_b": self.scale_b}


WORKLOADS = {
    w.name: w
    for w in [
        Workload("ag_a_tp2_256", 0, 2, 256, 256, 256, dist_a=U11, dist_b=U11),
        Workload("ag_a_tp2_blog", 0, 2, 16384, 8192, 8192, dist_a=U01, dist_b=U01),
        Workload("ag_a_tp8_pr", 0, 8, 16384, 106496, 16384, dist_a=N1, dist_b=N002),
        Workload("rs_a_tp8", 2, 8, 16384, 8192, 28672, dist_a=N1, dist_b=N002),
        Workload("ag_b_tp4_batched", 1, 4, 8192, 53248, 8192, l=2, alpha=0.5, beta=1.0, dist_a=N1,
                 dist_b=N002, dist_c=N1),
        Workload("rs_b_tp4_batched", 3, 4, 8192, 53248, 8192, l=2, alpha=0.5, beta=1.0, dist_a=N1,
                 dist_b=N002, dist_c=N1),
        # ag_a_tp8_pr with M / 2 and N / 8: the same full-K (16384) tiles and wave regime,
        # about 2.6 GB on the device, for full profiler captures
        Workload("ag_a_tp8_pr_small", 0, 8, 8192, 13312, 16384, dist_a=N1, dist_b=N002),
        # fp8 versions of the TP=8 workloads: e4m3 operands drawn N(0,1), the weight's
        # N(0,0.02) scale carried by the per-tensor scale_b
        Workload("ag_a_tp8_pr_e4m3", 0, 8, 16384, 106496, 16384, dist_a=N1, dist_b=N1, in_type="e4m3",
                 scale_b=0.02),
        Workload("rs_a_tp8_e4m3", 2, 8, 16384, 8192, 28672, dist_a=N1, dist_b=N1, in_type="e4m3", scale_b=0.02),
        # ag_a_tp8_pr_small in e4m3 (about 1.3 GB on the device), for full profiler captures
        Workload("ag_a_tp8_pr_small_e4m3", 0, 8, 8192, 13312, 16384, dist_a=N1, dist_b=N1, in_type="e4m3",
                 scale_b=0.02),
        # a quarter of rs_b_tp4_batched's N and one batch: small enough (about 1 GB on the
        # device) for a full profiler capture, same per-tile work
        Workload("rs_b_tp4_quarter", 3, 4, 8192, 13312, 8192, l=1, alpha=0.5, beta=1.0, dist_a=N1,
                 dist_b=N002, dist_c=N1),
        # half of its N and one batch (about 2.3 GB on the device): enough column waves per
        # raster group for the rotating partial's L2 traffic to matter, still capturable
        Workload("rs_b_tp4_half", 3, 4, 8192, 26624, 8192, l=1, alpha=0.5, beta=1.0, dist_a=N1,
                 dist_b=N002, dist_c=N1),
    ]
}

DEFAULT = "ag_a_tp8_pr"
