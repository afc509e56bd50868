/*
 * dg.h -- C ABI of the communication-fused tensor-parallel GEMM on one GB300.
 *
 * What it computes ("Distributed GEMM", CUTLASS example 65 README, section
 * "Getting started": the m, n, k, l (batch), alpha, beta problem):
 *
 *     D[l] = alpha * A[l] * B[l] + beta * C[l]          for l in [0, L)
 *
 * split over TP virtual ranks with one of the four schedules that README lists
 * under "Trying out other schedules".  All TP ranks are emulated on ONE GPU:
 * each rank's shards are views or receive slots in device memory, transfers
 * between ranks are copy-engine (two-dimensional device-to-device) copies on
 * side streams that each publish a ready flag, and one persistent kernel runs every rank's steps
 * in rotation order, waiting on a shard's flag before it loads that shard.
 *
 * Layouts (the pages do not fix them):
 *   A  bf16 (or fp8, dg_plan_scaled), L x M x K, row-major (K innermost)
 *   B  bf16 (or fp8), stored transposed: L x N x K, row-major (K innermost)
 *   C  bf16, L x M x N, row-major (read only when beta != 0)
 *   D  bf16 (or fp32, e4m3, e5m2: DG_OPT_OUT_TYPE), L x M x N, row-major
 *   bias  bf16, N values (dg_run_ex only; optional)
 * Every batch is densely packed after the previous one.  bf16 values are
 * passed as raw 16-bit patterns (dg_bf16_t).
 *
 * Shape rules: m, n, k, l >= 0; tp in {1, 2, 4, 8}; K % 8 == 0 and N % 8 == 0
 * (16-byte row pitch for the tensor-memory-access unit); the sharded extent
 * divides by tp (AG-RotatingA: M and N; AG-RotatingB: M and N;
 * RS-TilingA: M and K; RS-TilingB: N and K) and, for the RS schedules,
 * (K / tp) % 8 == 0.  Shards need not be multiples of the tile.
 *
 * Ownership: the caller owns A, B, C, D, the workspace and both streams.  The
 * plan owns only host state (geometry, events, cached tensor maps, the extra
 * copy streams it creates).  A workspace belongs to one plan at a time; the
 * first run of a plan with a given workspace clears the workspace's flag
 * words on the main stream.  Calls on one plan must not overlap in time
 * (different plans may be used from different threads); a plan's runs are
 * ordered on its main stream, and two runs of one plan must not share a
 * workspace while the first is still executing on another main stream.
 *
 * Concurrency on the GPU: the kernel is persistent, one CTA (pair) per SM,
 * and its transfers sit on copy streams behind stream waits.  Run dg runs one
 * after another (on one main stream, or with the next waiting for the
 * previous).  Two runs in flight on different streams can block each other:
 * CUDA multiplexes streams onto a limited number of hardware queues, so one
 * run's transfers may queue behind the other run's stream waits while the
 * other run's kernel holds every SM; the bounded waits then end the run with
 * DG_ERR_TIMEOUT (no hang).  An RS run's tiles also wait on tiles of other
 * CTAs of the same launch, so all of its CTAs must be resident together.
 *
 * Errors: every int-returning call returns DG_OK (0) or a negative dg_status;
 * dg_last_error() gives a message for the calling thread.
 */
#ifndef DG_H_
#define DG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dg_bf16_t;
typedef struct dg_plan_s* dg_plan_t;

/* The four schedules ("Distributed GEMM", CUTLASS example 65 README, section
 * "Trying out other schedules").  P = tp, rank r, step s:
 *   AG_ROTATING_A: rank r owns D[:, N_r]; step s computes D[M_j, N_r] with the
 *                  received A shard j = (r + s) mod P.
 *   AG_ROTATING_B: rank r owns D[M_r, :]; step s computes D[M_r, N_j] with the
 *                  received B shard j = (r + s) mod P.
 *   RS_TILING_A_ROTATING_C: rank r holds K-slab K_r; step s adds
 *                  alpha * A[M_j, K_r] B[K_r, :] into the rotating partial of
 *                  M-slab j = (r + s + 1) mod P, whose source at step 0 is
 *                  beta * C; the last step (j = r) writes D[M_r, :].
 *   RS_TILING_B_ROTATING_C: the same with N-slabs D[:, N_j].
 * The rotation follows _pipelined_all_gather_and_consume and
 * _pipelined_produce_and_all2all in torch/distributed/_symmetric_memory. */
enum dg_schedule {
  DG_AG_ROTATING_A = 0,
  DG_AG_ROTATING_B = 1,
  DG_RS_TILING_A_ROTATING_C = 2,
  DG_RS_TILING_B_ROTATING_C = 3
};

/* Run modes (how the AG shard transfers are issued):
 *   FUSED:     transfers on the copy stream, overlapped with the kernel, which
 *              waits per shard chunk on its ready flag.
 *   GEMM_ONLY: no transfers and no flag waits; the receive slots must already
 *              hold the shards (e.g. from an earlier FUSED run with the same A
 *              and B).  Measures the kernel alone.
 *   SERIAL:    all transfers on the main stream, then the kernel ("copy, then
 *              GEMM").  For the RS schedules SERIAL runs the non-fused
 *              baseline: one GEMM per rank into its own fp32 partial, then a
 *              separate reduction kernel; its workspace is larger (size the
 *              workspace after selecting the mode).
 * FUSED and GEMM_ONLY are the same kernel for the RS schedules (they move no
 * shards; the rotating partial lives in the workspace). */
enum dg_mode { DG_MODE_FUSED = 0, DG_MODE_GEMM_ONLY = 1, DG_MODE_SERIAL = 2 };

/* Element types.  A and B: BF16, E4M3 or E5M2 (C and the bias are always
 * bf16).  D: BF16 (default), F32, E4M3 or E5M2 (DG_OPT_OUT_TYPE), after the
 * out_dtype argument of the scaled fused ops in torch/distributed/_symmetric_memory;
 * an fp8 D holds result_scale * value (dg_set_result_scale) rounded to the
 * nearest code, ties to even, saturating at the largest finite value.
 * fp8 follows the OCP 8-bit formats: E4M3 is the variant without infinities
 * (largest finite 448), E5M2 the IEEE-like one (largest finite 57344); both
 * are passed as raw bytes. */
enum dg_type { DG_TYPE_BF16 = 0, DG_TYPE_E4M3 = 1, DG_TYPE_E5M2 = 2, DG_TYPE_F32 = 3 };

/* How the RS schedules combine the ranks' products (reduce_op of
 * fused_matmul_reduce_scatter in torch/distributed/_symmetric_memory: "sum"
 * is torch.sum over ranks, "avg" torch.mean).  With AVG every rank's product
 * and bias enter with weight 1/tp (exact, tp being a power of two); beta * C
 * still enters once. */
enum dg_reduce_op { DG_REDUCE_SUM = 0, DG_REDUCE_AVG = 1 };

enum dg_status {
  DG_OK = 0,
  DG_ERR_ARG = -1,         /* null/misaligned pointer, bad enum, negative extent */
  DG_ERR_SHAPE = -2,       /* extent not divisible by tp, or K/N pitch rule broken */
  DG_ERR_UNSUPPORTED = -3, /* device or driver lacks a needed feature */
  DG_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed */
  DG_ERR_TIMEOUT = -5,     /* a ready-flag wait ran out (device status word) */
  DG_ERR_HANG = -6,        /* an internal pipeline wait ran out; the kernel bailed out */
  DG_ERR_STATE = -7        /* call not valid in the plan's current state */
};

/* Options for dg_set_option. */
enum dg_option {
  DG_OPT_TIMEOUT_MS = 0,      /* ready-flag wait limit, ms (default 2000) */
  DG_OPT_CHUNK_TILES = 1,     /* tiles per shard transfer chunk (0 = auto, >= 16 MiB) */
  DG_OPT_FAULT_SKIP_FLAG = 2, /* test hook: drop the ready-flag write with this
                                 enqueue index (-1 = none, default) */
  DG_OPT_FAULT_DELAY_MS = 3,  /* test hook: hold the copy stream this long
                                 before the first transfer (default 0) */
  DG_OPT_GRID = 4,            /* persistent grid size in CTAs (0 = all co-resident) */
  DG_OPT_COPY_STREAMS = 5,    /* FUSED shard transfers spread round-robin over this many
                                 streams (1..8, default 2): the caller's copy stream plus
                                 streams the plan creates, so several copy engines run at once */
  DG_OPT_CTA_GROUP = 6,       /* tile configuration, before the first run: 2 (default) =
                                 256 x 256 tiles on an SM pair (tcgen05 cta_group::2),
                                 1 = 128 x 256 tiles on one SM */
  DG_OPT_EPILOGUE = 7,        /* epilogue, before the first run (all give the same bits, except
                                 in RS plans whose middle steps reduce with alpha * scale_a *
                                 scale_b not a power of two, DG_OPT_RS_REDUCE):
                                 1 = source and result chunks staged in shared memory and moved
                                 by TMA (default for AG plans with beta != 0 and fp8 inputs or
                                 K >= 16384, and for RS plans not covered below); 0 = direct
                                 per-row global accesses (one more operand stage; default for the
                                 other bf16 AG plans with beta != 0); 2 = staged per warp (each
                                 epilogue warp moves its own 32-row boxes, three source loads
                                 ahead, with no barrier between the warps; default for RS plans
                                 where at least half the steps load a source: tp <= 2, or
                                 tp <= 4 with beta != 0); 3 = result chunks staged, sources read
                                 directly (one more operand stage than 1; default for AG plans
                                 with beta == 0, which read no source); 4 = staged per warp
                                 with two slots, one load ahead, and one more operand stage
                                 (default for the other RS plans whose alpha * scale_a * scale_b
                                 is a power of two, where the middle steps load nothing,
                                 DG_OPT_RS_REDUCE) */
  DG_OPT_L2_HINT = 8,         /* L2 eviction policies of the kernel's TMA traffic: bits 0-1
                                 for the A loads, bits 2-3 for the B loads, bits 4-5 for the
                                 epilogue's (C / partial loads, partial / D stores and
                                 reductions); each 0 = none, 1 = evict first, 2 = evict last.
                                 Default 16 (the epilogue's traffic evict-first) on RS plans
                                 with bf16 operands, 0 otherwise */
  DG_OPT_RS_CE_PARTIALS = 10, /* RS plans with tp > 1, before the first run: 1 = hand the
                                 rotating partial from rank to rank by copy-engine transfers
                                 (each rank writes a send buffer; the copy streams wait on
                                 per-band completion counts, copy into the next rank's
                                 double-buffered receive buffer and publish a ready flag),
                                 0 (default) = the next rank reads the partial in place.
                                 Needs a copy stream distinct from the main stream. */
  DG_OPT_WAVE_SYNC = 9,       /* 1 = each CTA starts its i-th tile only after every CTA has
                                 issued the loads of its (i-1)-th (keeps the CTAs that share
                                 an operand strip in phase for L2 reuse; one counter word
                                 memset on the main stream per run), 0 = off, -1 (default) =
                                 on for AG plans whose per-wave operand strips exceed about
                                 96 MiB */
  DG_OPT_OUT_TYPE = 11,       /* element type of D: DG_TYPE_BF16 (default), DG_TYPE_F32,
                                 DG_TYPE_E4M3 or DG_TYPE_E5M2 (all but bf16 run through
                                 dg_run_ex; fp8 D is written by direct stores) */
  DG_OPT_REDUCE_OP = 12,      /* RS plans: dg_reduce_op, DG_REDUCE_SUM (default) or
                                 DG_REDUCE_AVG; AG plans accept only SUM */
  DG_OPT_COPY_PACE = 13,      /* AG FUSED runs with tp > 2: 1 = the shard transfers of step
                                 s >= 2 start only once the kernel has reached step s - 1
                                 (progress words the producers set; copy streams wait on them),
                                 so each step's transfers overlap the previous step's GEMM
                                 instead of all running at the start; paced transfers are
                                 enqueued after the kernel, so a layer that serializes launches
                                 (a profiler, CUDA_LAUNCH_BLOCKING) ends such a run with
                                 DG_ERR_TIMEOUT; 0 or -1 (default) = all transfers are issued
                                 at once, before the kernel */
  DG_OPT_COPY_KIND = 14,      /* how shard and partial transfers are issued: -1 (default) = auto,
                                 0 for the AG shard transfers and 2 for the RS hand-off copies;
                                 0 = two-dimensional device-to-device copies in the operand's own
                                 rows, which run on a copy engine beside a kernel that fills
                                 every SM (~1.0 TB/s on GB300); 1 = one-dimensional
                                 cudaMemcpyAsync, which on GB300 runs as a copy kernel on SMs
                                 and so only progresses where the GEMM kernel leaves an SM
                                 registers to spare (~3.2 TB/s when it gets SMs, but it
                                 competes with the GEMM for them); 2 = two-dimensional copies
                                 reshaped to at least 65,536 rows (the bytes are contiguous,
                                 so the row width is free), which the copy engines move at
                                 ~1.8 TB/s on GB300 for copies of 32 MiB or more (slower than 0
                                 below ~16 MiB), at the price of more HBM bandwidth taken from
                                 a GEMM running beside them */
  DG_OPT_HOST_OVERLAP = 15,   /* dg_run_host in FUSED mode with pinned host buffers: 1 (default) =
                                 launch the kernel at once and overlap the transfers with it
                                 (rank r's tiles wait for rank r's uploaded inputs; each
                                 finished (step, rank) block of D is downloaded while later
                                 steps run); 0 = upload everything, run, then download */
  DG_OPT_TILE_ORDER = 16,     /* order of the (rank, step) blocks of tiles: 0 = step-major (every
                                 rank's step s before any step s + 1); 1 = upload frontier, AG
                                 plans only: blocks (rank r, shard j) in groups g = max(r, j),
                                 so group g needs the inputs of ranks 0..g alone (copy pacing
                                 off); -1 (default) = 1 for AG runs of dg_run_host that overlap
                                 their uploads, else 0.  Results are bit-identical either way */
  DG_OPT_RS_CE_BANDS = 17,    /* RS with DG_OPT_RS_CE_PARTIALS: 256-row bands per hand-off copy
                                 (consecutive bands of one rank, step and batch go as one copy
                                 once all are complete, then each band's ready flag); 0
                                 (default) = auto, enough bands for >= 32 MiB per copy */
  DG_OPT_GROUP_M = 18,        /* raster of the tiles inside one (step, rank, batch) block: groups
                                 of this many tile rows, each swept column by column (so the
                                 tiles in flight share operand strips in L2); 0 (default) = auto */
  DG_OPT_RS_REDUCE = 19,      /* RS plans, before the first run: how the tiles of the middle steps
                                 (0 < s < tp - 1) update the rotating partial.  1 = add
                                 alpha' * product into it by TMA reductions (fp32 adds performed
                                 at the L2; alpha' = alpha * scale_a * scale_b, / tp for the
                                 mean) instead of loading it and storing fmaf(alpha', product,
                                 partial); needs a staged epilogue (selects it if the direct one
                                 is set); chunks that are not whole and the copy-engine hand-off
                                 still load, fmaf and store.  The product is rounded before the
                                 add, so where alpha' is not a power of two (or with a bias) the
                                 partial takes two roundings per step and the bits differ from
                                 0's in the last places (and between epilogue variants).
                                 0 = load, fmaf, store.  -1 (default) = 1 without a bias, else 0 */
  DG_OPT_MULTICAST = 20       /* AG plans with 256 x 256 pair tiles: 1 = clusters of two CTA pairs that take
                                 vertically adjacent tiles and share their B rows, each CTA
                                 loading half of its B rows for both pairs (TMA multicast), a
                                 quarter less operand traffic from L2 into shared memory; where
                                 the tile order allows it (every pair of consecutive tiles in one
                                 block with the same B rows), else as 0; same bits either way.
                                 0 = independent pairs.  -1 (default) = 1 for AG plans with
                                 K >= 16384, else 0 */
};

/* Plan geometry and workspace layout, for callers and tests. */
typedef struct dg_plan_info {
  int64_t m, n, k, l;
  int32_t tp, schedule;
  int64_t local_m, local_n, local_k; /* per-rank, per-step GEMM extents */
  int32_t tile_m, tile_n, tile_k;
  int64_t tiles_m, tiles_n;          /* tiles per (step, rank, batch) block */
  int64_t total_tiles;               /* all ranks, all steps */
  int64_t chunk_tiles, chunks_per_shard;
  int64_t n_flags;                   /* flag words in the workspace */
  size_t ws_bytes;
  size_t off_status, off_flags, off_slots, off_partial, off_serial;
  size_t slot_bytes;                 /* one receive slot (one shard, one batch) */
  int64_t copies_per_run;            /* transfer enqueues per FUSED/SERIAL run */
  int32_t a_type, b_type;            /* dg_type of A and B */
  int32_t elem_bytes;                /* bytes per A / B element (2 bf16, 1 fp8) */
  int32_t out_type;                  /* dg_type of D */
  int32_t reduce_op;                 /* dg_reduce_op */
  int32_t epilogue;                  /* DG_OPT_EPILOGUE in effect: 0 direct, 1 staged, 2 staged per warp */
  int32_t flag_parts;                /* RS hand-off flags per CTA half tile (4 with the per-warp epilogue) */
  int32_t multicast;                 /* DG_OPT_MULTICAST in effect and the step-major tile order allows it */
} dg_plan_info;

/* One tile of the step-major rotation order (host decoder, for tests). */
typedef struct dg_tile {
  int32_t step, rank, slab, batch;
  int32_t a_map, b_map;     /* tensor map index: AG 0 = home, 1 = receive slots;
                               RS = rank (its K-slab) */
  int64_t a_row, b_row;     /* first row loaded from that map */
  int64_t out_row, out_col; /* first D (or partial) element: row in L*M, column in N */
  int32_t rows_valid, cols_valid;
  int32_t k_blocks;
  int64_t flag;             /* AG ready-flag index (-1 = local shard) */
  int64_t tile_flag;        /* RS rotating-partial flag index (-1 = none) */
  int32_t src;              /* epilogue source: 0 none, 1 beta*C, 2 rotating partial */
  int32_t dst;              /* 0 = D (the plan's output type), 1 = rotating partial (fp32) */
} dg_tile;

/* Validate a problem and build a plan.  Host only: no CUDA call is made, so
 * this works without a GPU.  alpha/beta as in the README's --alpha/--beta. */
int dg_plan(dg_plan_t* out, int64_t m, int64_t n, int64_t k, int64_t l, int tp, int schedule,
            float alpha, float beta);

/* The scaled variant: A and B of dg_type a_type / b_type (both bf16, or both
 * fp8 in either format) with per-tensor scales, after the scaled all-gather /
 * reduce-scatter matmuls of torch/distributed/_symmetric_memory
 * (fused_all_gather_scaled_matmul and fused_scaled_matmul_reduce_scatter,
 * which pass A_scale and B_scale to a scaled matmul):
 *     D = alpha * scale_a * scale_b * A * B + beta * C
 * The three factors are folded into one fp32 multiplier (alpha*scale_a*scale_b
 * rounded to fp32) applied to the fp32 accumulator.  For fp8 inputs K must be
 * a multiple of 16 (and K/tp for the RS schedules); each K block holds 128
 * elements.  dg_plan is this call with bf16 inputs and unit scales. */
int dg_plan_scaled(dg_plan_t* out, int64_t m, int64_t n, int64_t k, int64_t l, int tp, int schedule,
                   float alpha, float beta, int a_type, int b_type, float scale_a, float scale_b);

/* Workspace bytes the plan needs in its current mode (0 is possible). */
size_t dg_workspace_bytes(dg_plan_t plan);

/* Select the run mode for later dg_run calls (dg_mode). */
int dg_run_mode(dg_plan_t plan, int mode);

/* Set a dg_option. */
int dg_set_option(dg_plan_t plan, int option, int64_t value);

/* Enqueue one run.  A and B hold the plan's input type (bf16 or fp8 bytes).
 * A, B, D, workspace: device pointers, 16-byte aligned
 * (workspace 256-byte aligned), workspace of dg_workspace_bytes(plan) bytes.
 * C may be NULL iff beta == 0.  main_stream / copy_stream: cudaStream_t
 * handles (copy_stream may equal main_stream; it is used only in FUSED mode
 * of the AG schedules).  Asynchronous: returns after enqueueing; the work is
 * ordered after prior work on main_stream and later work on main_stream is
 * ordered after all of it (copies included).  Device-side failures are
 * reported by dg_check.  The call may be captured into a CUDA graph on
 * main_stream (the copy streams join the capture through events); the graph
 * then clears the workspace's status and flag words at the start of every
 * replay, and replays must keep A, B, C, D and the workspace at the captured
 * addresses.  dg_check reports a replay's device status only until the plan
 * runs again outside the graph.  Make one run outside capture first (it sets
 * up the kernels' attributes). */
int dg_run(dg_plan_t plan, const void* A, const void* B, const dg_bf16_t* C,
           dg_bf16_t* D, void* workspace, void* main_stream, void* copy_stream);

/* dg_run with the epilogue extras of the scaled fused ops in
 * torch/distributed/_symmetric_memory (fused_all_gather_scaled_matmul and
 * fused_scaled_matmul_reduce_scatter pass bias and out_dtype to a scaled
 * matmul on every rank):
 *   bias  NULL, or N bf16 values (16-byte aligned) added to every row of
 *         every rank's product.  The AG schedules therefore add it once; the
 *         RS schedules once per rank before the reduction (tp copies with
 *         DG_REDUCE_SUM, their mean -- one copy -- with DG_REDUCE_AVG), as
 *         the module's reference composition (a scaled matmul with the bias
 *         on each rank, then reduce_scatter_tensor) does.
 *   D     elements of the plan's output type (DG_OPT_OUT_TYPE): bf16 or fp32.
 * The epilogue computes fmaf(alpha', acc, src) + w * bias in fp32, with
 * alpha' = alpha * scale_a * scale_b * w and w = 1 (or 1/tp for AVG), then
 * rounds to D's type.  Everything else is as for dg_run, which is this call
 * with bias = NULL on a bf16-output plan (dg_run refuses fp32-output plans
 * with DG_ERR_STATE). */
int dg_run_ex(dg_plan_t plan, const void* A, const void* B, const dg_bf16_t* C, const dg_bf16_t* bias,
              void* D, void* workspace, void* main_stream, void* copy_stream);

/* dg_run_ex with host-resident operands, for callers whose data lives in
 * host memory: copies A and B (and C when beta != 0) from host memory into
 * the caller's device buffers, runs the plan on them, and copies D back into
 * host memory.  Sizes follow the plan: A L*M*K elements, B L*N*K (both of the
 * plan's input type), C L*M*N bf16, D L*M*N of the output type.  bias, if not
 * NULL, is a device pointer.  The device buffers follow dg_run's rules.
 *
 * In FUSED mode with every host buffer page-locked (cudaHostAlloc or
 * cudaHostRegister) and DG_OPT_HOST_OVERLAP on (the default), the transfers
 * overlap the kernel: it is launched at once; plan-owned streams upload the
 * inputs in P units in the kernel's order (AG: rank r's home shards of A and
 * B and the part of C its tiles read; RS: the operand every tile reads whole,
 * then row slabs of the other operand and of C in the order the steps need
 * them), and each tile waits (bounded, like the shard flags) for the unit
 * holding its inputs; AG runs also take their blocks in the upload-frontier
 * order (DG_OPT_TILE_ORDER); each (step, rank) block of D is copied back as
 * soon as the kernel has finished it.  Otherwise (another mode,
 * pageable memory, or the option off) the call uploads everything on
 * main_stream, runs, then downloads: pageable memory works with
 * host-synchronous copies.  Either way the call is one operation on
 * main_stream: it starts after the work already enqueued there, and returns
 * after enqueueing; D_host is valid once main_stream has reached that point
 * (e.g. after dg_check).  Until then the host inputs must stay allocated and
 * unchanged (the uploads read them asynchronously, as cudaMemcpyAsync does),
 * and D_host and the device buffers must not be touched by other work.  The call can be captured into a CUDA graph on
 * main_stream like dg_run (the plan's own streams join the capture); a replay
 * reads the host buffers' contents at replay time. */
int dg_run_host(dg_plan_t plan, const void* A_host, const void* B_host, const dg_bf16_t* C_host,
                const dg_bf16_t* bias, void* D_host, void* A_dev, void* B_dev, dg_bf16_t* C_dev, void* D_dev,
                void* workspace, void* main_stream, void* copy_stream);

/* Multiplier applied to the result before it is rounded to an fp8 D (the
 * result_scale of the scaled fused ops; default 1).  Ignored for bf16 and
 * fp32 D.  DG_ERR_ARG for NaN. */
int dg_set_result_scale(dg_plan_t plan, float scale);

/* Synchronize `stream` and read the workspace status word of the plan's last
 * run: DG_OK, DG_ERR_TIMEOUT or DG_ERR_HANG (with the flag index in the
 * message), or DG_ERR_CUDA on a CUDA error.  workspace NULL: the built-in
 * array if the plan's last run was dg_run_static, else only the
 * synchronization is checked. */
int dg_check(dg_plan_t plan, void* workspace, void* stream);

/* Geometry and workspace layout. */
int dg_plan_info_get(dg_plan_t plan, dg_plan_info* info);

/* Decode tile t (0 <= t < total_tiles) of the rotation order on the host. */
int dg_plan_tile(dg_plan_t plan, int64_t t, dg_tile* out);

/* No-allocation variant of dg_run.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot call cudaMalloc (or
 * anything that allocates device memory) at the point where they run the
 * GEMM -- for example code inside an application whose device memory is all
 * owned and budgeted by a host framework, or a plug-in that is not allowed
 * to grow the process's device footprint after start-up.
 *
 * Instead of a caller-supplied workspace it uses one file-scope device array
 * of DG_STATIC_WORKSPACE_BYTES bytes inside this library.  Every GPU that
 * loads the library holds that array until the process exits, whether or not
 * this function is ever called.  The caller still passes A, B, C, D and the
 * streams exactly as for dg_run.
 *
 * Limits and rules:
 *   - The plan's dg_workspace_bytes() must be <= DG_STATIC_WORKSPACE_BYTES;
 *     larger plans are rejected with DG_ERR_SHAPE before any GPU work.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once; make that first call before starting any
 *     stream capture on that device.
 *   - All calls in the process share the one array, and it keeps the last
 *     call's contents.  The flag and status words that must start at zero are
 *     cleared on the main stream whenever a different plan used the array
 *     last.  Calls whose GPU work overlaps (on different streams, or from
 *     several threads) race on the array: serialize them.
 *   - main_stream must belong to the current device (DG_ERR_ARG otherwise):
 *     the array's address differs from device to device.
 *   - It makes no device-memory allocation or free (no cudaMalloc/cudaFree,
 *     no allocating library call).
 * dg_check(plan, NULL, stream) reports the plan's last dg_run_static call
 * like any run: it reads the device status word from the shared array
 * (DG_ERR_TIMEOUT when a ready-flag wait ran out; D is then undefined), as
 * long as no other call has used the array since. */
#define DG_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)
int dg_run_static(dg_plan_t plan, const dg_bf16_t* A, const dg_bf16_t* B, const dg_bf16_t* C,
                  dg_bf16_t* D, void* main_stream, void* copy_stream);

void dg_destroy(dg_plan_t plan);

/* Message of the calling thread's last error ("" if none). */
const char* dg_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
