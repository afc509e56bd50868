"""The C ABI without a GPU: the library loads and exports every declared
symbol; the planner validates shapes; the tile order it decodes visits every
(output element, K range) exactly once, in the rotation the oracle states."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import schedules as osch
from reduce_scatter_gb300 import dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCHED_NAME = {dg.AG_ROTATING_A: osch.AG_ROTATING_A, dg.AG_ROTATING_B: osch.AG_ROTATING_B,
              dg.RS_TILING_A_ROTATING_C: osch.RS_TILING_A_ROTATING_C,
              dg.RS_TILING_B_ROTATING_C: osch.RS_TILING_B_ROTATING_C}


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(dg.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    return dg.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "dg.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(dg.EXPORTS), names
    for name in names:
        assert hasattr(L, name), name


def test_struct_sizes_match_header(L):
    # the ctypes mirrors must have the C layout: probe through the ABI
    p = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A)
    info = p.info()
    assert info["m"] == 256 and info["tp"] == 2 and info["schedule"] == 0
    assert info["ws_bytes"] == p.workspace_bytes()


@pytest.mark.parametrize("args,code", [
    ((-1, 8, 8, 1, 1, 0), dg.ERR_ARG),
    ((8, 8, 8, 1, 3, 0), dg.ERR_ARG),
    ((8, 8, 8, 1, 2, 7), dg.ERR_ARG),
    ((8, 8, 12, 1, 1, 0), dg.ERR_SHAPE),          # K % 8
    ((8, 12, 8, 1, 1, 0), dg.ERR_SHAPE),          # N % 8
    ((10, 16, 8, 1, 4, dg.AG_ROTATING_A), dg.ERR_SHAPE),   # M % tp
    ((10, 16, 8, 1, 4, dg.AG_ROTATING_B), dg.ERR_SHAPE),   # M % tp (B rotates, M still sharded)
    ((12, 16, 64, 1, 8, dg.RS_TILING_A_ROTATING_C), dg.ERR_SHAPE),  # M % tp
    ((16, 16, 24, 1, 2, dg.RS_TILING_A_ROTATING_C), dg.ERR_SHAPE),  # (K/tp) % 8
    ((16, 16, 36, 1, 8, dg.RS_TILING_B_ROTATING_C), dg.ERR_SHAPE),  # K % 8
])
def test_plan_rejects(L, args, code):
    h = ctypes.c_void_p()
    rc = L.dg_plan(ctypes.byref(h), *args, 1.0, 0.0)
    assert rc == code
    assert dg.last_error()


def test_null_and_bad_options(L):
    assert L.dg_plan(None, 8, 8, 8, 1, 1, 0, 1.0, 0.0) == dg.ERR_ARG
    p = dg.Plan(16, 16, 16, 1, 1, 0)
    with pytest.raises(dg.DGError):
        p.set_mode(9)
    with pytest.raises(dg.DGError):
        p.set_option(99, 1)
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_TIMEOUT_MS, 0)
    with pytest.raises(dg.DGError):
        p.tile(p.info()["total_tiles"])


def test_run_argument_checks_without_gpu(L):
    # argument checks come before any CUDA call
    p = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A, 1.0, 0.5)
    assert p.run(16, 16, None, 16, 256, raise_on_error=False) == dg.ERR_ARG  # C NULL with beta != 0
    p2 = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A)
    assert p2.run(16, 24, None, 16, 256, raise_on_error=False) == dg.ERR_ARG  # misaligned B
    assert p2.run(None, 16, None, 16, 256, raise_on_error=False) == dg.ERR_ARG
    assert p2.run(16, 16, None, 16, 128, raise_on_error=False) == dg.ERR_ARG  # workspace alignment


def test_empty_problem_is_a_noop(L):
    for m, n, k, l in [(0, 16, 16, 1), (16, 0, 16, 1), (16, 16, 16, 0)]:
        p = dg.Plan(m, n, k, l, 1, dg.AG_ROTATING_A)
        assert p.info()["total_tiles"] == 0
        assert p.run(None, None, None, None, None, raise_on_error=False) == dg.OK


def test_local_sizes_match_pr_printout(L, golden_dir):
    with open(os.path.join(golden_dir, "pr1907_distgemm_printout.json")) as f:
        g = json.load(f)
    for run in g["runs"]:
        m, n, k, l = run["problem"]
        info = dg.Plan(m, n, k, l, run["tp"], dg.AG_ROTATING_A).info()
        assert (info["local_m"], info["local_n"], info["local_k"], info["l"]) == tuple(run["local_problem"])


def _simulate(plan, m, n, k, l, tp, sched):
    """Walk the decoded order; check coverage and rotation against the oracle."""
    info = plan.info()
    T = info["total_tiles"]
    name = SCHED_NAME[sched]
    cover = np.zeros((l, m, n), dtype=np.int64)    # (output element, k-slab) visits via k ranges
    kcover = np.zeros((l, m, n, tp if sched >= 2 else 1), dtype=np.int64)
    last_step = {}
    prev_block_end = -1
    for t in range(T):
        tl = plan.tile(t)
        s, r, j, b = tl["step"], tl["rank"], tl["slab"], tl["batch"]
        assert j == osch.slab_index(name, tp, r, s)
        blk = osch.step_blocks(name, m, n, k, tp, r, s)
        rows = slice(tl["out_row"] - b * m, tl["out_row"] - b * m + tl["rows_valid"])
        cols = slice(tl["out_col"], tl["out_col"] + tl["cols_valid"])
        # the tile lies inside the oracle's block for (r, s)
        assert blk["rows"].start <= rows.start and rows.stop <= blk["rows"].stop
        assert blk["cols"].start <= cols.start and cols.stop <= blk["cols"].stop
        cover[b, rows, cols] += 1
        if sched >= 2:
            kcover[b, rows, cols, r] += 1
            want_src = (1 if info and plan.beta != 0 else 0) if s == 0 else 2
            assert tl["src"] == want_src
            assert tl["dst"] == (0 if s == tp - 1 else 1)
            assert tl["a_map"] == r and tl["b_map"] == r
            assert tl["k_blocks"] == -(-(k // tp) // 64)
            key = (b, rows.start, cols.start)
            assert last_step.get(key, -1) == s - 1, "steps of one tile in order"
            last_step[key] = s
        else:
            assert tl["k_blocks"] == -(-k // 64)
            local = (blk["recv"] is None)
            assert (tl["flag"] < 0) == local
            if sched == dg.AG_ROTATING_A:
                assert tl["a_map"] == (0 if local else 1)
                assert tl["b_row"] == b * n + tl["out_col"]
                if local:
                    assert tl["a_row"] == tl["out_row"]
            else:
                assert tl["b_map"] == (0 if local else 1)
                assert tl["a_row"] == tl["out_row"]
            if not local:
                assert 0 <= tl["flag"] < info["n_flags"]
        # step-major order
        blk_id = s * tp + r
        assert blk_id >= prev_block_end
        prev_block_end = blk_id
    if sched >= 2:
        assert np.all(kcover == 1)
        assert tp == 1 or all(v == tp - 1 for v in last_step.values())
    assert np.all(cover == (tp if sched >= 2 else 1))


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", [0, 1, 2, 3])
@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("shape", [(256, 512, 128, 1), (1024, 768, 512, 2), (136, 272, 80, 1)])
def test_tile_order_simulator(L, sched, tp, shape, cg):
    m, n, k, l = shape
    if sched in (2, 3) and (k % tp or (k // tp) % 8):
        k = 64 * tp
    if (sched in (0, 1, 2) and m % tp) or (sched != 2 and n % tp):
        pytest.skip("not divisible")
    plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.5)
    plan.set_option(dg.OPT_CTA_GROUP, cg)
    assert plan.info()["tile_m"] == 128 * cg
    _simulate(plan, m, n, k, l, tp, sched)
    if sched >= 2 and tp > 1:
        info = plan.info()
        assert info["flag_parts"] == (4 if info["epilogue"] in (2, 4) else 1)
        assert info["n_flags"] == l * tp * info["tiles_m"] * info["tiles_n"] * cg * info["flag_parts"]


def test_ag_flag_indices_follow_copy_order(L):
    # chunk flags are laid out in the order the copies are enqueued:
    # step-major, then rank, batch, chunk
    m, n, k, l, tp = 2048, 1024, 1024, 2, 4
    plan = dg.Plan(m, n, k, l, tp, dg.AG_ROTATING_A)
    plan.set_option(dg.OPT_CHUNK_TILES, 2)
    info = plan.info()
    nch = info["chunks_per_shard"]
    assert nch == -(-info["tiles_m"] // 2)
    seen = set()
    for t in range(info["total_tiles"]):
        tl = plan.tile(t)
        if tl["flag"] < 0:
            continue
        s, r, b = tl["step"], tl["rank"], tl["batch"]
        mt = (tl["a_row"] % (m // tp)) // info["tile_m"]
        assert tl["flag"] == ((r * (tp - 1) + s - 1) * l + b) * nch + mt // 2
        seen.add(tl["flag"])
    assert seen == set(range(info["n_flags"]))
    assert info["copies_per_run"] == info["n_flags"]


def test_workspace_layout_sizes(L):
    m, n, k, l, tp = 4096, 2048, 1024, 1, 8
    pa = dg.Plan(m, n, k, l, tp, dg.AG_ROTATING_A).info()
    assert pa["slot_bytes"] == (m // tp) * k * 2
    assert pa["ws_bytes"] >= pa["off_slots"] + tp * (tp - 1) * l * pa["slot_bytes"]
    pr = dg.Plan(m, n, k, l, tp, dg.RS_TILING_A_ROTATING_C)
    ir = pr.info()
    assert ir["ws_bytes"] >= ir["off_partial"] + l * m * n * 4
    pr.set_mode(dg.MODE_SERIAL)
    assert pr.workspace_bytes() >= ir["off_serial"] + tp * l * m * n * 4
    p1 = dg.Plan(m, n, k, l, 1, dg.AG_ROTATING_A).info()
    assert p1["n_flags"] == 0 and p1["copies_per_run"] == 0


def test_scaled_plan_rules(L):
    h = ctypes.c_void_p()
    # mixed 16-bit / 8-bit operands are refused; unknown types too
    assert L.dg_plan_scaled(ctypes.byref(h), 64, 64, 64, 1, 1, 0, 1.0, 0.0, dg.TYPE_BF16, dg.TYPE_E4M3,
                            1.0, 1.0) == dg.ERR_UNSUPPORTED
    assert L.dg_plan_scaled(ctypes.byref(h), 64, 64, 64, 1, 1, 0, 1.0, 0.0, 7, 7, 1.0, 1.0) == dg.ERR_ARG
    # fp8 rows need 16-byte pitch: K % 16, and (K/tp) % 16 for RS
    assert L.dg_plan_scaled(ctypes.byref(h), 64, 64, 40, 1, 1, 0, 1.0, 0.0, dg.TYPE_E4M3, dg.TYPE_E4M3,
                            1.0, 1.0) == dg.ERR_SHAPE
    assert L.dg_plan_scaled(ctypes.byref(h), 64, 64, 64, 1, 8, 2, 1.0, 0.0, dg.TYPE_E4M3, dg.TYPE_E4M3,
                            1.0, 1.0) == dg.ERR_SHAPE
    p = dg.Plan(1024, 1024, 640, 1, 4, dg.AG_ROTATING_A, a_type="e4m3", b_type="e5m2", scale_b=0.5)
    info = p.info()
    assert (info["a_type"], info["b_type"], info["elem_bytes"]) == (dg.TYPE_E4M3, dg.TYPE_E5M2, 1)
    assert info["slot_bytes"] == (1024 // 4) * 640          # one byte per element
    assert p.tile(0)["k_blocks"] == 5                        # 128 fp8 elements per K block
    pb = dg.Plan(1024, 1024, 640, 1, 4, dg.AG_ROTATING_A).info()
    assert pb["elem_bytes"] == 2 and pb["slot_bytes"] == 2 * info["slot_bytes"]


def test_ce_handoff_option_rules(L):
    p = dg.Plan(512, 512, 512, 1, 2, dg.AG_ROTATING_A)
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_RS_CE_PARTIALS, 1)          # AG plan
    p = dg.Plan(512, 1000, 512, 1, 8, dg.RS_TILING_B_ROTATING_C)
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_RS_CE_PARTIALS, 1)          # N/tp = 125, not a multiple of 8
    q = dg.Plan(2048, 1024, 1024, 2, 4, dg.RS_TILING_A_ROTATING_C)
    before = q.workspace_bytes()
    q.set_option(dg.OPT_RS_CE_PARTIALS, 1)
    info = q.info()
    slab = 2 * (2048 // 4) * 1024 * 4
    assert info["ws_bytes"] >= 3 * 4 * slab // 1 and info["ws_bytes"] > before
    assert info["n_flags"] == 4 * 4 * 2 * info["tiles_m"]
    for t in range(info["total_tiles"]):
        assert q.tile(t)["tile_flag"] == -1                # hand-offs go through the copy engine


@pytest.mark.parametrize("i", range(24))
def test_tile_order_simulator_random(L, i):
    rng = np.random.default_rng(500 + i)
    sched = int(rng.integers(0, 4))
    tp = int(rng.choice([1, 2, 4, 8]))
    l = int(rng.integers(1, 3))
    m = int(rng.integers(1, 6)) * 8 * tp
    n = int(rng.integers(1, 9)) * 8 * tp
    k = int(rng.integers(1, 5)) * 64 * tp
    plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.5 if rng.integers(0, 2) else 0.0)
    plan.set_option(dg.OPT_CTA_GROUP, int(rng.integers(1, 3)))
    _simulate(plan, m, n, k, l, tp, sched)


def test_output_type_and_reduce_op_rules(L):
    p = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A)
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_OUT_TYPE, 7)                   # no such type
    p.set_option(dg.OPT_OUT_TYPE, dg.TYPE_E4M3)            # fp8 D, with a result scale
    p.set_result_scale(0.25)
    with pytest.raises(dg.DGError):
        p.set_result_scale(float("nan"))
    assert p.run(16, 16, None, 16, 256, raise_on_error=False) == dg.ERR_STATE   # dg_run writes bf16 only
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_REDUCE_OP, dg.REDUCE_AVG)      # AG plans have no reduction
    p.set_option(dg.OPT_REDUCE_OP, dg.REDUCE_SUM)
    p.set_option(dg.OPT_OUT_TYPE, dg.TYPE_F32)
    info = p.info()
    assert (info["out_type"], info["reduce_op"]) == (dg.TYPE_F32, dg.REDUCE_SUM)
    # dg_run writes bf16 D only: an fp32-output plan is refused before any CUDA call
    assert p.run(16, 16, None, 16, 256, raise_on_error=False) == dg.ERR_STATE
    # dg_run_ex checks the bias alignment with the other pointers
    assert p.run_ex(16, 16, None, 24, 16, 256, raise_on_error=False) == dg.ERR_ARG
    q = dg.Plan(256, 256, 256, 1, 4, dg.RS_TILING_B_ROTATING_C, out_type="f32", reduce_op="avg")
    info = q.info()
    assert (info["out_type"], info["reduce_op"]) == (dg.TYPE_F32, dg.REDUCE_AVG)
    with pytest.raises(dg.DGError):
        q.set_option(dg.OPT_REDUCE_OP, 2)


def test_copy_pace_option_rules(L):
    p = dg.Plan(512, 512, 512, 1, 4, dg.AG_ROTATING_A)
    for v in (-1, 0, 1):
        p.set_option(dg.OPT_COPY_PACE, v)
    for v in (-2, 2):
        with pytest.raises(dg.DGError):
            p.set_option(dg.OPT_COPY_PACE, v)


def test_copy_kind_option_rules(L):
    p = dg.Plan(512, 512, 512, 1, 4, dg.AG_ROTATING_A)
    for v in (1, 2, 0, -1):
        p.set_option(dg.OPT_COPY_KIND, v)
    for v in (-2, 3):
        with pytest.raises(dg.DGError):
            p.set_option(dg.OPT_COPY_KIND, v)
    q = dg.Plan(512, 512, 512, 1, 4, dg.RS_TILING_A_ROTATING_C)
    for v in (0, 3, 1):
        q.set_option(dg.OPT_RS_CE_BANDS, v)
    with pytest.raises(dg.DGError):
        q.set_option(dg.OPT_RS_CE_BANDS, -1)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_upload_frontier_order_is_a_permutation_by_groups(L, sched, tp):
    # the same tiles as the step-major order, visited by (rank, shard) blocks in
    # groups g = max(r, j) that never go back, each group touching ranks 0..g only
    m, n, k, l = 1024, 1536, 256, 2
    ref = dg.Plan(m, n, k, l, tp, sched)
    fr = dg.Plan(m, n, k, l, tp, sched)
    fr.set_option(dg.OPT_TILE_ORDER, 1)
    T = ref.info()["total_tiles"]
    assert fr.info()["total_tiles"] == T
    key = lambda d: (d["step"], d["rank"], d["batch"], d["out_row"], d["out_col"], d["a_map"], d["a_row"],
                     d["b_map"], d["b_row"], d["flag"])  # noqa: E731
    a = sorted(key(ref.tile(t)) for t in range(T))
    tiles = [fr.tile(t) for t in range(T)]
    assert sorted(key(d) for d in tiles) == a
    groups = [max(d["rank"], d["slab"]) for d in tiles]
    assert groups == sorted(groups)
    per_block = T // (tp * tp)
    for t in range(0, T, per_block):
        blk = {(d["step"], d["rank"]) for d in tiles[t:t + per_block]}
        assert len(blk) == 1  # a block's tiles stay together
    for d in tiles:
        assert d["slab"] == (d["rank"] + d["step"]) % tp
    # group 0 is rank 0's step 0, its own inputs only
    assert (tiles[0]["rank"], tiles[0]["step"]) == (0, 0)


def test_tile_order_option_rules(L):
    p = dg.Plan(512, 512, 512, 1, 4, dg.AG_ROTATING_B)
    for v in (-1, 0, 1):
        p.set_option(dg.OPT_TILE_ORDER, v)
    for v in (-2, 2):
        with pytest.raises(dg.DGError):
            p.set_option(dg.OPT_TILE_ORDER, v)
    q = dg.Plan(512, 512, 512, 1, 4, dg.RS_TILING_A_ROTATING_C)
    q.set_option(dg.OPT_TILE_ORDER, 0)
    with pytest.raises(dg.DGError):
        q.set_option(dg.OPT_TILE_ORDER, 1)


def test_host_overlap_option_rules(L):
    p = dg.Plan(512, 512, 512, 1, 4, dg.AG_ROTATING_A)
    for v in (0, 1):
        p.set_option(dg.OPT_HOST_OVERLAP, v)
    for v in (-1, 2):
        with pytest.raises(dg.DGError):
            p.set_option(dg.OPT_HOST_OVERLAP, v)


def test_run_host_argument_checks_without_gpu(L):
    p = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A, 1.0, 0.5)
    # missing host or device buffers, C missing with beta != 0: refused before any CUDA call
    assert p.run_host(None, 16, None, None, 16, 16, 16, None, 16, 256, raise_on_error=False) == dg.ERR_ARG
    assert p.run_host(16, 16, None, None, 16, 16, 16, None, 16, 256, raise_on_error=False) == dg.ERR_ARG
    q = dg.Plan(256, 256, 256, 1, 2, dg.AG_ROTATING_A)
    assert q.run_host(16, 16, None, None, 16, None, 16, None, 16, 256, raise_on_error=False) == dg.ERR_ARG


@pytest.mark.parametrize("group_m", [1, 3, 8, 1000])
@pytest.mark.parametrize("sched", [0, 1, 2, 3])
def test_tile_order_simulator_raster_groups(L, sched, group_m):
    # any raster group height walks every tile of every block exactly once
    m, n, k, l, tp = 1280, 1536, 512, 2, 4
    plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.5)
    plan.set_option(dg.OPT_GROUP_M, group_m)
    _simulate(plan, m, n, k, l, tp, sched)
    with pytest.raises(dg.DGError):
        plan.set_option(dg.OPT_GROUP_M, -1)


def test_rs_reduce_and_epilogue_option_rules(L):
    assert dg.Plan(1024, 1024, 1024, 1, 8, dg.RS_TILING_A_ROTATING_C).info()["epilogue"] == 4   # alpha' = 2^0
    assert dg.Plan(1024, 1024, 1024, 1, 8, dg.RS_TILING_A_ROTATING_C, 0.75).info()["epilogue"] == 1  # not 2^e
    p = dg.Plan(1024, 1024, 1024, 1, 8, dg.RS_TILING_A_ROTATING_C)
    p.set_option(dg.OPT_EPILOGUE, 1)
    flags_staged = p.info()["n_flags"]
    p.set_option(dg.OPT_RS_REDUCE, 1)
    assert p.info()["n_flags"] == flags_staged
    p.set_option(dg.OPT_EPILOGUE, 2)                  # per-warp epilogue:
    assert p.info()["n_flags"] == 4 * flags_staged    # hand-offs are flagged per warp quarter
    with pytest.raises(dg.DGError):
        p.set_option(dg.OPT_RS_REDUCE, 2)
    p.set_option(dg.OPT_RS_REDUCE, -1)
    # the per-warp epilogue where at least half the steps load a source
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.RS_TILING_B_ROTATING_C, 0.5, 1.0).info()["epilogue"] == 2
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.RS_TILING_B_ROTATING_C, 0.5, 0.0).info()["epilogue"] == 4
    assert dg.Plan(1024, 1024, 1024, 1, 2, dg.RS_TILING_A_ROTATING_C).info()["epilogue"] == 2
    d = dg.Plan(1024, 1024, 1024, 1, 4, dg.RS_TILING_A_ROTATING_C)
    d.set_option(dg.OPT_EPILOGUE, 0)
    d.set_option(dg.OPT_RS_REDUCE, 1)                 # the reduction needs a staged epilogue
    assert d.info()["epilogue"] == 1
    q = dg.Plan(1024, 1024, 1024, 1, 4, dg.AG_ROTATING_A)
    with pytest.raises(dg.DGError):
        q.set_option(dg.OPT_RS_REDUCE, 1)
    for v in (0, 1, 2, 3, 4):
        q.set_option(dg.OPT_EPILOGUE, v)
    with pytest.raises(dg.DGError):
        q.set_option(dg.OPT_EPILOGUE, 5)


def test_multicast_eligibility(L):
    # tiles 2i and 2i + 1 must share their B rows inside one block
    for sched, shape, want in [(dg.AG_ROTATING_A, (16384, 106496, 16384, 1, 8), 1),
                               (dg.AG_ROTATING_B, (8192, 53248, 8192, 2, 4), 1),
                               (dg.RS_TILING_A_ROTATING_C, (16384, 8192, 28672, 1, 8), 0),   # AG only
                               (dg.RS_TILING_B_ROTATING_C, (8192, 53248, 8192, 2, 4), 0),
                               (dg.AG_ROTATING_A, (512, 512, 256, 1, 2), 0),      # one tile per block
                               (dg.AG_ROTATING_A, (1536, 512, 256, 1, 2), 0)]:    # three tile rows
        m, n, k, l, tp = shape
        p = dg.Plan(m, n, k, l, tp, sched)
        auto = want if sched in (dg.AG_ROTATING_A, dg.AG_ROTATING_B) and k >= 16384 else 0
        assert p.info()["multicast"] == auto              # automatic for AG with K >= 16384
        p.set_option(dg.OPT_MULTICAST, 0)
        assert p.info()["multicast"] == 0
        p.set_option(dg.OPT_MULTICAST, 1)
        assert p.info()["multicast"] == want, (sched, shape)
    p.set_option(dg.OPT_CTA_GROUP, 1)
    assert p.info()["multicast"] == 0                     # pair tiles only


def test_l2_hint_option_rules(L):
    p = dg.Plan(1024, 2048, 512, 1, 4, 2, 1.0, 0.0)
    for v in (0, 2, 9, 16, 32, 18, 42):
        p.set_option(dg.OPT_L2_HINT, v)
    for v in (-1, 3, 12, 48, 64):
        with pytest.raises(dg.DGError):
            p.set_option(dg.OPT_L2_HINT, v)


def test_ag_epilogue_defaults(L):
    # AG with beta == 0 reads no source: stores-only staging, bf16 and fp8 alike
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.AG_ROTATING_A).info()["epilogue"] == 3
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.AG_ROTATING_A, 1.0, 0.0, dg.TYPE_E4M3, dg.TYPE_E4M3).info()["epilogue"] == 3
    # with a source: staged for fp8 or long K, direct otherwise
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.AG_ROTATING_B, 1.0, 1.0, dg.TYPE_E4M3, dg.TYPE_E5M2).info()["epilogue"] == 1
    assert dg.Plan(1024, 1024, 16384, 1, 4, dg.AG_ROTATING_A, 1.0, 1.0).info()["epilogue"] == 1
    assert dg.Plan(1024, 1024, 1024, 1, 4, dg.AG_ROTATING_A, 1.0, 1.0).info()["epilogue"] == 0
