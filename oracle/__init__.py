"""CPU oracle of the communication-fused tensor-parallel GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The device
path never imports it and shares no code with it.

* ``oracle.gemm``: the plain fp64 definition D = alpha*A*B + beta*C.
* ``oracle.schedules``: the four schedules restated rank by rank and step by
  step on small inputs.
"""

from . import gemm, schedules  # noqa: F401
