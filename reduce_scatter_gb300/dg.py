"""ctypes binding of the C ABI in ``include/dg.h`` (argument marshalling only).

Every computation runs in ``_lib/libdg.so``.  If the library has not been
built, importing works but the first call raises ``RuntimeError``: there is
no fallback path.

Pointers are accepted as ``torch.Tensor`` (its ``data_ptr()``), plain ints or
``None``; streams as ``torch.cuda.Stream`` or raw ``cudaStream_t`` ints.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libdg.so")

AG_ROTATING_A = 0
AG_ROTATING_B = 1
RS_TILING_A_ROTATING_C = 2
RS_TILING_B_ROTATING_C = 3
SCHEDULE_NAMES = {
    AG_ROTATING_A: "AllGather1D_TilingCD_RotatingA",
    AG_ROTATING_B: "AllGather1D_TilingCD_RotatingB",
    RS_TILING_A_ROTATING_C: "ReduceScatter1D_TilingA_RotatingC",
    RS_TILING_B_ROTATING_C: "ReduceScatter1D_TilingB_RotatingC",
}
SCHEDULE_BY_NAME = {v: k for k, v in SCHEDULE_NAMES.items()}

TYPE_BF16 = 0
TYPE_E4M3 = 1
TYPE_E5M2 = 2
TYPE_F32 = 3  # output (D) only
TYPE_NAMES = {TYPE_BF16: "bf16", TYPE_E4M3: "e4m3", TYPE_E5M2: "e5m2", TYPE_F32: "f32"}
TYPE_BY_NAME = {v: k for k, v in TYPE_NAMES.items()}

REDUCE_SUM = 0
REDUCE_AVG = 1
REDUCE_BY_NAME = {"sum": REDUCE_SUM, "avg": REDUCE_AVG}

MODE_FUSED = 0
MODE_GEMM_ONLY = 1
MODE_SERIAL = 2

OK = 0
ERR_ARG = -1
ERR_SHAPE = -2
ERR_UNSUPPORTED = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5
ERR_HANG = -6
ERR_STATE = -7

OPT_TIMEOUT_MS = 0
OPT_CHUNK_TILES = 1
OPT_FAULT_SKIP_FLAG = 2
OPT_FAULT_DELAY_MS = 3
OPT_GRID = 4
OPT_COPY_STREAMS = 5
OPT_CTA_GROUP = 6
OPT_EPILOGUE = 7
OPT_L2_HINT = 8
OPT_WAVE_SYNC = 9
OPT_RS_CE_PARTIALS = 10
OPT_OUT_TYPE = 11
OPT_REDUCE_OP = 12
OPT_COPY_PACE = 13
OPT_COPY_KIND = 14
OPT_HOST_OVERLAP = 15
OPT_TILE_ORDER = 16
OPT_RS_CE_BANDS = 17
OPT_GROUP_M = 18
OPT_RS_REDUCE = 19
OPT_MULTICAST = 20

# Every symbol include/dg.h declares.
EXPORTS = ("dg_plan", "dg_workspace_bytes", "dg_run_mode", "dg_set_option", "dg_run", "dg_check",
           "dg_plan_info_get", "dg_plan_tile", "dg_destroy", "dg_last_error", "dg_run_static",
           "dg_plan_scaled", "dg_run_ex", "dg_run_host", "dg_set_result_scale")

# Size of the library's built-in workspace used by dg_run_static.
STATIC_WORKSPACE_BYTES = 32 << 20


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64), ("l", ctypes.c_int64),
        ("tp", ctypes.c_int32), ("schedule", ctypes.c_int32),
        ("local_m", ctypes.c_int64), ("local_n", ctypes.c_int64), ("local_k", ctypes.c_int64),
        ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
        ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64),
        ("total_tiles", ctypes.c_int64),
        ("chunk_tiles", ctypes.c_int64), ("chunks_per_shard", ctypes.c_int64),
        ("n_flags", ctypes.c_int64),
        ("ws_bytes", ctypes.c_size_t),
        ("off_status", ctypes.c_size_t), ("off_flags", ctypes.c_size_t), ("off_slots", ctypes.c_size_t),
        ("off_partial", ctypes.c_size_t), ("off_serial", ctypes.c_size_t),
        ("slot_bytes", ctypes.c_size_t),
        ("copies_per_run", ctypes.c_int64),
        ("a_type", ctypes.c_int32), ("b_type", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
        ("out_type", ctypes.c_int32), ("reduce_op", ctypes.c_int32),
        ("epilogue", ctypes.c_int32), ("flag_parts", ctypes.c_int32), ("multicast", ctypes.c_int32),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class Tile(ctypes.Structure):
    _fields_ = [
        ("step", ctypes.c_int32), ("rank", ctypes.c_int32), ("slab", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("a_map", ctypes.c_int32), ("b_map", ctypes.c_int32),
        ("a_row", ctypes.c_int64), ("b_row", ctypes.c_int64),
        ("out_row", ctypes.c_int64), ("out_col", ctypes.c_int64),
        ("rows_valid", ctypes.c_int32), ("cols_valid", ctypes.c_int32),
        ("k_blocks", ctypes.c_int32),
        ("flag", ctypes.c_int64), ("tile_flag", ctypes.c_int64),
        ("src", ctypes.c_int32), ("dst", ctypes.c_int32),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class DGError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"dg error {code}: {msg}")
        self.code = code


_LIB = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.dg_plan.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i64, i32, i32, ctypes.c_float, ctypes.c_float]
        L.dg_plan.restype = i32
        L.dg_plan_scaled.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i64, i32, i32, ctypes.c_float,
                                     ctypes.c_float, i32, i32, ctypes.c_float, ctypes.c_float]
        L.dg_plan_scaled.restype = i32
        L.dg_workspace_bytes.argtypes = [vp]
        L.dg_workspace_bytes.restype = ctypes.c_size_t
        L.dg_run_mode.argtypes = [vp, i32]
        L.dg_run_mode.restype = i32
        L.dg_set_option.argtypes = [vp, i32, i64]
        L.dg_set_option.restype = i32
        L.dg_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.dg_run.restype = i32
        L.dg_run_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.dg_run_ex.restype = i32
        L.dg_set_result_scale.argtypes = [vp, ctypes.c_float]
        L.dg_set_result_scale.restype = i32
        L.dg_run_host.argtypes = [vp] * 13
        L.dg_run_host.restype = i32
        L.dg_run_static.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.dg_run_static.restype = i32
        L.dg_check.argtypes = [vp, vp, vp]
        L.dg_check.restype = i32
        L.dg_plan_info_get.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.dg_plan_info_get.restype = i32
        L.dg_plan_tile.argtypes = [vp, i64, ctypes.POINTER(Tile)]
        L.dg_plan_tile.restype = i32
        L.dg_destroy.argtypes = [vp]
        L.dg_destroy.restype = None
        L.dg_last_error.argtypes = []
        L.dg_last_error.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def last_error() -> str:
    return lib().dg_last_error().decode()


def _check(rc: int):
    if rc != OK:
        raise DGError(rc, last_error())
    return rc


def ptr(x) -> int | None:
    """Device address of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def stream_handle(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


class Plan:
    """One problem (m, n, k, l, tp, schedule, alpha, beta) behind ``dg_plan``.

    ``out_type`` (TYPE_BF16 / TYPE_F32 or "bf16" / "f32") and ``reduce_op``
    (REDUCE_SUM / REDUCE_AVG or "sum" / "avg") are set through
    ``dg_set_option`` right after planning."""

    def __init__(self, m, n, k, l, tp, schedule, alpha=1.0, beta=0.0, a_type=TYPE_BF16, b_type=TYPE_BF16,
                 scale_a=1.0, scale_b=1.0, out_type=TYPE_BF16, reduce_op=REDUCE_SUM, result_scale=1.0):
        if isinstance(schedule, str):
            schedule = SCHEDULE_BY_NAME[schedule]
        a_type = TYPE_BY_NAME.get(a_type, a_type)
        b_type = TYPE_BY_NAME.get(b_type, b_type)
        h = ctypes.c_void_p()
        if a_type == TYPE_BF16 and b_type == TYPE_BF16 and scale_a == 1.0 and scale_b == 1.0:
            _check(lib().dg_plan(ctypes.byref(h), m, n, k, l, tp, schedule, alpha, beta))
        else:
            _check(lib().dg_plan_scaled(ctypes.byref(h), m, n, k, l, tp, schedule, alpha, beta, a_type, b_type,
                                        scale_a, scale_b))
        self.a_type, self.b_type, self.scale_a, self.scale_b = a_type, b_type, scale_a, scale_b
        self._h = h
        self.out_type = TYPE_BY_NAME.get(out_type, out_type)
        self.reduce_op = REDUCE_BY_NAME.get(reduce_op, reduce_op)
        if self.out_type != TYPE_BF16:
            self.set_option(OPT_OUT_TYPE, self.out_type)
        if self.reduce_op != REDUCE_SUM:
            self.set_option(OPT_REDUCE_OP, self.reduce_op)
        if result_scale != 1.0:
            self.set_result_scale(result_scale)
        self.m, self.n, self.k, self.l, self.tp, self.schedule = m, n, k, l, tp, schedule
        self.alpha, self.beta = alpha, beta

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            lib().dg_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self) -> int:
        return int(lib().dg_workspace_bytes(self._h))

    def set_mode(self, mode: int):
        _check(lib().dg_run_mode(self._h, mode))

    def set_option(self, opt: int, value: int):
        _check(lib().dg_set_option(self._h, opt, value))

    def set_result_scale(self, scale: float):
        """``dg_set_result_scale``: multiplier before rounding to an fp8 D."""
        _check(lib().dg_set_result_scale(self._h, float(scale)))

    def info(self) -> dict:
        inf = PlanInfo()
        _check(lib().dg_plan_info_get(self._h, ctypes.byref(inf)))
        return inf.as_dict()

    def tile(self, t: int) -> dict:
        tl = Tile()
        _check(lib().dg_plan_tile(self._h, t, ctypes.byref(tl)))
        return tl.as_dict()

    def run(self, A, B, C, D, workspace, main_stream=None, copy_stream=None, raise_on_error=True) -> int:
        rc = lib().dg_run(self._h, ptr(A), ptr(B), ptr(C), ptr(D), ptr(workspace),
                          stream_handle(main_stream), stream_handle(copy_stream))
        if raise_on_error:
            _check(rc)
        return rc

    def run_ex(self, A, B, C, bias, D, workspace, main_stream=None, copy_stream=None, raise_on_error=True) -> int:
        """``dg_run_ex``: an optional per-column bf16 bias; D of the plan's output type."""
        rc = lib().dg_run_ex(self._h, ptr(A), ptr(B), ptr(C), ptr(bias), ptr(D), ptr(workspace),
                             stream_handle(main_stream), stream_handle(copy_stream))
        if raise_on_error:
            _check(rc)
        return rc

    def run_host(self, A_host, B_host, C_host, bias, D_host, A_dev, B_dev, C_dev, D_dev, workspace, main_stream=None,
                 copy_stream=None, raise_on_error=True) -> int:
        """``dg_run_host``: inputs copied from host memory, D copied back (host tensors' data_ptr)."""
        rc = lib().dg_run_host(self._h, ptr(A_host), ptr(B_host), ptr(C_host), ptr(bias), ptr(D_host), ptr(A_dev),
                               ptr(B_dev), ptr(C_dev), ptr(D_dev), ptr(workspace), stream_handle(main_stream),
                               stream_handle(copy_stream))
        if raise_on_error:
            _check(rc)
        return rc

    def run_static(self, A, B, C, D, main_stream=None, copy_stream=None, raise_on_error=True) -> int:
        """``dg_run_static``: the library's built-in workspace instead of a caller one."""
        rc = lib().dg_run_static(self._h, ptr(A), ptr(B), ptr(C), ptr(D), stream_handle(main_stream),
                                 stream_handle(copy_stream))
        if raise_on_error:
            _check(rc)
        return rc

    def check(self, workspace, stream=None, raise_on_error=True) -> int:
        rc = lib().dg_check(self._h, ptr(workspace), stream_handle(stream))
        if raise_on_error:
            _check(rc)
        return rc
