// dg_geom.h -- problem geometry and the step-major rotation order of tiles.
//
// Shared by the host planner (which validates and describes the order) and
// the persistent kernel (whose producer, MMA and epilogue warps all walk the
// same order).  Plain integers only.
//
// Order: tile t = ((s * P + r) * TB) + u, with s the step, r the virtual rank
// and u the tile inside the (s, r) block of TB = L * tiles_m * tiles_n tiles.
// Every step of every rank comes before any tile of the next step, so the
// shard transfers for step s have all of the steps before it to arrive
// (step 0 is local for every rank).  Inside a block, tiles go batch-major and
// then in groups of GROUP_M tile rows swept column by column, so that the
// CTAs in flight share A rows and B columns in L2.
//
// A second order for the AllGather schedules (Geom::order = 1, "upload
// frontier"), used when the inputs are still arriving from the host rank by
// rank: the (rank r, shard j) blocks go in groups g = max(r, j) = 0..P-1, so a
// group needs nothing beyond the first g + 1 ranks' inputs.  Inside group g:
// (g, g) (step 0, no transfer), then (g, j < g), then (r < g, g).  The step of
// a block is s = (j - r) mod P.
//
// Which shard/slab a rank handles at a step (the rotation) follows
// _pipelined_all_gather_and_consume (AG: j = (r + s) mod P, local shard first)
// and _pipelined_produce_and_all2all (RS: j = (r + s + 1) mod P, own slab last)
// in torch/distributed/_symmetric_memory.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DG_HD __host__ __device__ __forceinline__
#else
#define DG_HD inline
#endif

namespace dg {

enum : int { SCHED_AG_A = 0, SCHED_AG_B = 1, SCHED_RS_A = 2, SCHED_RS_B = 3 };
// Non-fused ReduceScatter baseline: every rank's full partial product over its
// own K-slab, written to its own fp32 buffer (stacked rank-major); a separate
// reduction then sums them.  Tile order: rank-major, one step.
enum : int { SCHED_PARTIAL = 4 };
enum : int { SRC_NONE = 0, SRC_C = 1, SRC_X = 2 };
enum : int { DST_D = 0, DST_X = 1 };
enum : int { MAP_HOME = 0, MAP_SLOT = 1 };

struct Geom {
  int32_t sched, P;
  int64_t M, N, K, L;
  int32_t BM, BN, BK;
  int32_t group_m;
  int64_t blk_m, blk_n;     // rows / cols of one (step, rank) output block
  int64_t shard;            // rows of one transferred shard (AG) : M/P or N/P
  int64_t Ks;               // K extent per step (K for AG, K/P for RS)
  int64_t tiles_m, tiles_n; // tiles of one block
  int64_t tiles_block;      // L * tiles_m * tiles_n
  int64_t total_tiles;      // P * P * tiles_block
  int64_t chunk_tiles;      // AG: tiles of the rotated dim per transfer chunk
  int64_t nchunks;          // AG: chunks per shard
  int32_t beta_nonzero;
  int32_t ce_partials;  // RS: partials handed on by copy-engine transfers between rank buffers
  int32_t order;        // AG block order: 0 step-major, 1 upload frontier
};

struct Tile {
  int32_t s, r, j, l;
  int32_t a_map, b_map;
  int64_t a_row, b_row;
  int64_t out_row, out_col;
  int32_t rows_valid, cols_valid;
  int32_t k_blocks;
  int64_t flag;       // AG chunk flag, -1 if local
  int64_t tile_flag;  // RS tile flag, -1 if none
  int32_t src, dst;
  // RS with copy-engine hand-off: position in the rank's send / receive buffers
  int32_t band;       // tile row (m-tile) inside the slab
  int64_t xs_row;     // first row in the send buffer (rank-major, slab-local rows)
  int64_t xr_row;     // first row in the receive buffer of this step (double-buffered)
  int64_t x_col;      // first column inside the slab
};

DG_HD int64_t dg_min64(int64_t a, int64_t b) { return a < b ? a : b; }
DG_HD int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Block b (0 <= b < P * P) of the upload-frontier order: its rank r and shard j.
DG_HD void frontier_block(int64_t b, int64_t* r, int64_t* j) {
  int64_t g = 0;
  while ((g + 1) * (g + 1) <= b) ++g;  // groups 0..g-1 hold g * g blocks
  const int64_t i = b - g * g;          // 0 .. 2g
  if (i == 0) {
    *r = g, *j = g;
  } else if (i <= g) {
    *r = g, *j = i - 1;
  } else {
    *r = i - g - 1, *j = g;
  }
}

DG_HD Tile decode_tile(const Geom& g, int64_t t) {
  Tile o;
  const int64_t P = g.P;
  int64_t s, r, u;
  if (g.order == 1) {
    const int64_t b = t / g.tiles_block;
    u = t - b * g.tiles_block;
    int64_t jb;
    frontier_block(b, &r, &jb);
    s = (jb - r + P) % P;
  } else {
    const int64_t per_step = P * g.tiles_block;
    s = t / per_step;
    const int64_t rem = t - s * per_step;
    r = rem / g.tiles_block;
    u = rem - r * g.tiles_block;
  }
  const int64_t per_batch = g.tiles_m * g.tiles_n;
  const int64_t l = u / per_batch;
  const int64_t v = u - l * per_batch;
  // grouped raster: GROUP_M tile rows, swept column by column
  const int64_t gsz = (int64_t)g.group_m * g.tiles_n;
  const int64_t grp = v / gsz;
  const int64_t in = v - grp * gsz;
  const int64_t gm = dg_min64((int64_t)g.group_m, g.tiles_m - grp * g.group_m);
  const int64_t mt = grp * g.group_m + in % gm;
  const int64_t nt = in / gm;

  const bool ag = g.sched == SCHED_AG_A || g.sched == SCHED_AG_B;
  // (SCHED_PARTIAL has one step: total_tiles = P * tiles_block, so s = 0.)
  const int64_t j = ag ? (r + s) % P : (r + s + 1) % P;
  o.s = (int32_t)s;
  o.r = (int32_t)r;
  o.j = (int32_t)j;
  o.l = (int32_t)l;
  o.k_blocks = (int32_t)cdiv(g.Ks, g.BK);
  o.flag = -1;
  o.tile_flag = -1;
  o.band = 0;
  o.xs_row = o.xr_row = o.x_col = 0;
  const int64_t mrow = mt * g.BM;  // inside the block
  const int64_t ncol = nt * g.BN;
  o.rows_valid = (int32_t)dg_min64(g.BM, g.blk_m - mrow);
  o.cols_valid = (int32_t)dg_min64(g.BN, g.blk_n - ncol);
  // receive-slot index of (rank r, step s >= 1), batch l
  const int64_t slot = ((r * (P - 1) + (s - 1)) * g.L + l);

  if (g.sched == SCHED_AG_A) {
    // rank r owns D[:, N_r]; step s: rows of A shard j
    o.out_row = l * g.M + j * g.blk_m + mrow;
    o.out_col = r * g.blk_n + ncol;
    o.b_map = MAP_HOME;
    o.b_row = l * g.N + r * g.blk_n + ncol;
    if (s == 0) {
      o.a_map = MAP_HOME;
      o.a_row = o.out_row;
    } else {
      o.a_map = MAP_SLOT;
      o.a_row = slot * g.shard + mrow;
      o.flag = slot * g.nchunks + mt / g.chunk_tiles;
    }
    o.src = g.beta_nonzero ? SRC_C : SRC_NONE;
    o.dst = DST_D;
  } else if (g.sched == SCHED_AG_B) {
    // rank r owns D[M_r, :]; step s: columns of B shard j
    o.out_row = l * g.M + r * g.blk_m + mrow;
    o.out_col = j * g.blk_n + ncol;
    o.a_map = MAP_HOME;
    o.a_row = o.out_row;
    if (s == 0) {
      o.b_map = MAP_HOME;
      o.b_row = l * g.N + j * g.blk_n + ncol;
    } else {
      o.b_map = MAP_SLOT;
      o.b_row = slot * g.shard + ncol;
      o.flag = slot * g.nchunks + nt / g.chunk_tiles;
    }
    o.src = g.beta_nonzero ? SRC_C : SRC_NONE;
    o.dst = DST_D;
  } else if (g.sched == SCHED_PARTIAL) {
    o.out_row = (r * g.L + l) * g.M + mrow;  // row of the stacked partial buffers
    o.out_col = ncol;
    o.a_map = (int32_t)r;
    o.b_map = (int32_t)r;
    o.a_row = l * g.M + mrow;
    o.b_row = l * g.N + ncol;
    o.src = SRC_NONE;
    o.dst = DST_X;
  } else {
    // RS: rank r contributes its K-slab to output slab j
    const bool rs_a = g.sched == SCHED_RS_A;
    const int64_t row0 = rs_a ? j * g.blk_m : 0;
    const int64_t col0 = rs_a ? 0 : j * g.blk_n;
    o.out_row = l * g.M + row0 + mrow;
    o.out_col = col0 + ncol;
    o.a_map = (int32_t)r;
    o.b_map = (int32_t)r;
    o.a_row = o.out_row;
    o.b_row = l * g.N + o.out_col;
    const int64_t tiles_slab = g.tiles_m * g.tiles_n;
    const int64_t tf = ((l * P + j) * tiles_slab) + mt * g.tiles_n + nt;
    o.tile_flag = P > 1 && !g.ce_partials ? tf : -1;
    o.band = (int32_t)mt;
    o.x_col = ncol;
    o.xs_row = (r * g.L + l) * g.blk_m + mrow;
    o.xr_row = ((2 * r + (s & 1)) * g.L + l) * g.blk_m + mrow;
    o.src = s == 0 ? (g.beta_nonzero ? SRC_C : SRC_NONE) : SRC_X;
    o.dst = s == P - 1 ? DST_D : DST_X;
  }
  return o;
}

}  // namespace dg
