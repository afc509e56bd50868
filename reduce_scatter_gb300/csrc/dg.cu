// dg.cu -- C ABI (include/dg.h): planner, workspace layout, tensor maps,
// copy-engine shard mover and the launch of the persistent kernel.
//
// Emulation of TP ranks on one GPU ("Distributed GEMM", CUTLASS pull request
// #1907 description: point-to-point transfers, "a memcopy branch" beside the
// GEMM kernels, which only add barriers at their start, leaving the SMs to the
// GEMM and the copy engine to communication):
//   * rank r's home shards are views of the caller's A / B;
//   * rank r's receive slot for step s >= 1 is a workspace region; the copy
//     streams fill it in chunks with two-dimensional device-to-device copies,
//     which run on a copy engine, and after each chunk write the run's epoch
//     into that chunk's ready flag with a stream memory operation (no SM
//     involved);
//   * one persistent kernel runs every rank's steps in rotation order and its
//     producer waits on a chunk's flag before loading from the slot.
// The RS schedules move no shards: by default the rotating partial X_j lives
// in the workspace and each tile's hand-off from step s to s + 1 is a release
// / acquire on a per-tile flag; with DG_OPT_RS_CE_PARTIALS the partial moves
// between rank send and receive buffers by copy-engine copies (run_rs_ce).
// dg_run_host adds plan-owned upload and download streams around a run
// (enqueue_uploads / enqueue_downloads).

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include "dg.h"
#include "dg_kernel.cuh"

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DG_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
typedef CUresult (*WaitValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct Driver {
  EncodeTiledFn encode = nullptr;
  WriteValue32Fn write32 = nullptr;
  WaitValue32Fn wait32 = nullptr;
};

int get_driver(Driver* d) {
  static std::mutex mu;
  static Driver cached;
  static bool done = false;
  std::lock_guard<std::mutex> lk(mu);
  if (!done) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(DG_ERR_UNSUPPORTED, "driver entry point cuTensorMapEncodeTiled not found");
    cached.encode = reinterpret_cast<EncodeTiledFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(DG_ERR_UNSUPPORTED, "driver entry point cuStreamWriteValue32 not found");
    cached.write32 = reinterpret_cast<WriteValue32Fn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return fail(DG_ERR_UNSUPPORTED, "driver entry point cuStreamWaitValue32 not found");
    cached.wait32 = reinterpret_cast<WaitValue32Fn>(fn);
    done = true;
  }
  *d = cached;
  return DG_OK;
}

// Workspace -> owning plan, so a workspace reused by another plan gets its
// flag words cleared before its epochs are trusted.
std::mutex g_ws_mu;
std::unordered_map<const void*, uint64_t> g_ws_owner;
uint64_t g_next_plan_id = 1;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// NVTX range over a host-side call (a no-op unless a profiler is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Layout of the 256-byte status area: [0, 8) status word, [64, 68) wave
// counter, [128, 128 + 4 * tp) copy-pacing progress words, [192, 192 + 4 * tp)
// per-rank upload flags of runs that take host buffers.
constexpr size_t kProgressOffset = 128;
constexpr size_t kUpOffset = 192;

}  // namespace

struct dg_plan_s {
  dg::Geom g{};
  int64_t m = 0, n = 0, k = 0, l = 0;
  int tp = 1, schedule = 0;
  float alpha = 1.f, beta = 0.f;
  int a_type = DG_TYPE_BF16, b_type = DG_TYPE_BF16;  // input element types
  int esz = 2;                                       // bytes per A / B element
  float scale_a = 1.f, scale_b = 1.f;                // per-tensor scales (scaled GEMM)
  int out_type = DG_TYPE_BF16;                       // element type of D (DG_OPT_OUT_TYPE)
  float result_scale = 1.f;                          // fp8 D: multiplier before rounding
  int reduce_op = DG_REDUCE_SUM;                     // RS: sum or mean over ranks (DG_OPT_REDUCE_OP)
  int mode = DG_MODE_FUSED;
  int64_t timeout_ms = 2000;
  int64_t chunk_tiles_req = 0;
  int64_t fault_skip = -1;
  int64_t fault_delay_ms = 0;
  int64_t grid_req = 0;
  int cg = 2;  // CTA group of the tile config: 1 = 128 x 256 per SM, 2 = 256 x 256 per SM pair
  bool cep = false;  // RS: hand partials on by copy-engine transfers (DG_OPT_RS_CE_PARTIALS)
  size_t off_done = 0, off_send = 0, off_recv = 0;
  int epi = 0;  // epilogue: 0 direct, 1 staged through shared memory with TMA (default: RS, fp8, K >= 16384)
  uint32_t l2_hint = 0;  // L2 policies of the TMA traffic (DG_OPT_L2_HINT)
  int wave_sync = -1;  // DG_OPT_WAVE_SYNC: -1 auto, 0 off, 1 on
  int copy_pace = -1;  // DG_OPT_COPY_PACE: -1 auto, 0 off, 1 on
  int copy_kind = -1;  // DG_OPT_COPY_KIND: -1 auto (AG shards 0, RS hand-off 2), 0 copy engine (2D
                       // copies in the operand's rows), 1 one-dimensional cudaMemcpyAsync, 2 copy
                       // engine (tall 2D copies)
  int host_overlap = 1;  // DG_OPT_HOST_OVERLAP: dg_run_host overlaps its transfers with the kernel
  int tile_order = -1;   // DG_OPT_TILE_ORDER: -1 auto, 0 step-major, 1 upload frontier (AG)
  int64_t ce_bands = 0;  // DG_OPT_RS_CE_BANDS: 256-row bands per hand-off copy, 0 auto
  int64_t group_m_req = 0;  // DG_OPT_GROUP_M: tile rows per raster group, 0 auto
  int multicast = -1;       // DG_OPT_MULTICAST: two CTA pairs per cluster share their B rows (-1 auto)
  int mc_ok[2] = {-1, -1};  // per block order: every tile pair (2i, 2i + 1) may share (-1 not yet known)
  int max_quads = 0;        // co-resident clusters of four of the CG = 2 kernels
  bool map_mc = false;      // the cached B maps have the multicast boxes
  int rs_reduce = -1;       // DG_OPT_RS_REDUCE: middle RS steps add into the partial by TMA reduction
                            // (-1 auto: where that gives the same bits as load, fmaf, store)
  uint64_t id = 0;
  uint32_t epoch = 0;
  int static_dev = -1;  // device whose built-in workspace the plan's last run used (dg_run_static), or -1
  bool serial_ws = false;
  // layout
  int64_t n_flags = 0;
  size_t off_status = 0, off_flags = 0, off_slots = 0, off_partial = 0, off_serial = 0;
  size_t off_ddone = 0;  // per (step, rank) counters of finished D half tiles (dg_run_host)
  size_t slot_bytes = 0, ws_bytes_base = 0, ws_bytes_serial = 0;
  int64_t copies = 0;
  // runtime state
  bool rt = false;
  int device = -1;
  int num_sms = 0;
  int max_pairs = 0;  // co-resident CTA pairs of the CG = 2 kernel
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // extra copy streams (FUSED transfers spread round-robin over the caller's
  // copy stream and these, so that several copy engines move shards at once)
  int copy_streams = 2;
  int n_extra = 0;
  cudaStream_t extra[7] = {};
  cudaEvent_t extra_done[7] = {};
  // dg_run_host with overlapped transfers: host-to-device and device-to-host
  // streams, the fork point on the main stream, one event per rank's upload
  bool io_rt = false;
  cudaStream_t up_st = nullptr, down_st = nullptr;
  cudaEvent_t ev_io = nullptr, ev_up[8] = {}, ev_up_done = nullptr, ev_down_done = nullptr;
  dg::KParams kp;
  dg::Geom gser{};   // RS SERIAL baseline: per-rank partial GEMMs (SCHED_PARTIAL)
  dg::KParams kser;  // its kernel parameters
  const void* map_key[3] = {nullptr, nullptr, nullptr};
  int n_maps = 0;
};

namespace {

bool is_ag(int s) { return s == DG_AG_ROTATING_A || s == DG_AG_ROTATING_B; }

// Epilogue variant: 0 direct, 1 staged per CTA, 2 staged per warp, 3 stores
// staged only, 4 staged per warp with two slots.  The per-warp epilogues hand
// partials on, and count finished tiles, per warp quarter of a CTA's half tile.
bool epi_per_warp(const dg_plan_s* p) { return p->epi == 2 || p->epi == 4; }
int epi_parts(const dg_plan_s* p) { return epi_per_warp(p) ? dg::EPI_WARPS : 1; }
int epi_box_rows(const dg_plan_s* p) { return epi_per_warp(p) ? dg::WROWS : dg::ROWS_PER_CTA; }

int layout(dg_plan_s* p) {
  dg::Geom& g = p->g;
  p->mc_ok[0] = p->mc_ok[1] = -1;
  const int64_t P = p->tp;
  g.sched = p->schedule;
  g.P = (int32_t)P;
  g.M = p->m;
  g.N = p->n;
  g.K = p->k;
  g.L = p->l;
  g.BM = p->cg == 2 ? dg::Cfg<2>::TILE_M : dg::Cfg<1>::TILE_M;
  g.BN = dg::TILE_N;
  g.BK = dg::KROW_BYTES / p->esz;  // 64 bf16 or 128 fp8 elements: 128 bytes per row
  g.group_m = (int32_t)(p->group_m_req > 0 ? p->group_m_req : 16);
  g.beta_nonzero = p->beta != 0.f;
  g.order = p->tile_order == 1 ? 1 : 0;
  switch (p->schedule) {
    case DG_AG_ROTATING_A:
      g.blk_m = p->m / P, g.blk_n = p->n / P, g.shard = p->m / P, g.Ks = p->k;
      break;
    case DG_AG_ROTATING_B:
      g.blk_m = p->m / P, g.blk_n = p->n / P, g.shard = p->n / P, g.Ks = p->k;
      break;
    case DG_RS_TILING_A_ROTATING_C:
      g.blk_m = p->m / P, g.blk_n = p->n, g.shard = 0, g.Ks = p->k / P;
      break;
    default:
      g.blk_m = p->m, g.blk_n = p->n / P, g.shard = 0, g.Ks = p->k / P;
      break;
  }
  g.tiles_m = dg::cdiv(g.blk_m, g.BM);
  g.tiles_n = dg::cdiv(g.blk_n, g.BN);
  g.tiles_block = g.L * g.tiles_m * g.tiles_n;
  g.total_tiles = P * P * g.tiles_block;
  g.chunk_tiles = 1;
  g.nchunks = 0;
  p->n_flags = 0;
  p->copies = 0;
  if (is_ag(p->schedule)) {
    const int64_t rot_tiles = p->schedule == DG_AG_ROTATING_A ? g.tiles_m : g.tiles_n;
    const int64_t tile_rows = p->schedule == DG_AG_ROTATING_A ? g.BM : g.BN;
    int64_t ct = p->chunk_tiles_req;
    if (ct <= 0) {
      const int64_t bytes = tile_rows * std::max<int64_t>(p->k, 1) * p->esz;
      // >= 16 MiB per transfer: per-copy overhead dominates smaller chunks
      // (8-tile chunks moved RotatingB shards ~3x faster than 1-tile ones)
      ct = std::max<int64_t>(1, dg::cdiv(int64_t(16) << 20, bytes));
    }
    g.chunk_tiles = std::max<int64_t>(1, std::min<int64_t>(ct, std::max<int64_t>(rot_tiles, 1)));
    g.nchunks = dg::cdiv(rot_tiles, g.chunk_tiles);
    if (P > 1) {
      p->n_flags = P * (P - 1) * g.L * g.nchunks;
      p->copies = p->n_flags;
    }
  } else if (P > 1 && p->cep) {
    // copy-engine hand-off: one ready flag per (receiving rank, step, batch, band)
    p->n_flags = P * P * g.L * g.tiles_m;
  } else if (P > 1) {
    // one flag per tile and CTA of the group (each CTA hands on its own half),
    // or per warp quarter of it (per-warp epilogue)
    p->n_flags = g.L * P * g.tiles_m * g.tiles_n * p->cg * epi_parts(p);
  }
  g.ce_partials = p->cep ? 1 : 0;
  // RS SERIAL baseline geometry: every rank's full M x N partial over its K-slab
  p->gser = g;
  p->gser.sched = dg::SCHED_PARTIAL;
  p->gser.ce_partials = 0;  // the baseline writes its own partial buffers, no hand-off
  p->gser.blk_m = p->m;
  p->gser.blk_n = p->n;
  p->gser.tiles_m = dg::cdiv(p->m, g.BM);
  p->gser.tiles_n = dg::cdiv(p->n, g.BN);
  p->gser.tiles_block = g.L * p->gser.tiles_m * p->gser.tiles_n;
  p->gser.total_tiles = P * p->gser.tiles_block;
  p->off_status = 0;
  p->off_flags = 256;
  p->off_ddone = round_up(p->off_flags + (size_t)p->n_flags * 4, 256);
  size_t off = round_up(p->off_ddone + (size_t)(P * P) * 4, 1024);
  p->off_slots = off;
  p->slot_bytes = is_ag(p->schedule) ? (size_t)g.shard * (size_t)p->k * (size_t)p->esz : 0;
  if (is_ag(p->schedule) && P > 1) off = round_up(off + (size_t)(P * (P - 1) * g.L) * p->slot_bytes, 1024);
  p->off_partial = off;
  p->off_done = p->off_send = p->off_recv = off;
  if (!is_ag(p->schedule) && P > 1 && p->cep) {
    // done counters (per rank, step, batch, band), send buffers (one slab per
    // rank) and double-buffered receive buffers
    const size_t slab = (size_t)(g.L * g.blk_m * g.blk_n) * 4;
    p->off_done = off;
    off = round_up(off + (size_t)(P * P * g.L * g.tiles_m) * 4, 1024);
    p->off_send = off;
    off = round_up(off + (size_t)P * slab, 1024);
    p->off_recv = off;
    off = round_up(off + (size_t)(2 * P) * slab, 1024);
  } else if (!is_ag(p->schedule) && P > 1) {
    off = round_up(off + (size_t)(g.L * p->m * p->n) * 4, 1024);
  }
  p->off_serial = off;
  p->ws_bytes_base = off;
  p->ws_bytes_serial = off;
  if (!is_ag(p->schedule))
    p->ws_bytes_serial = round_up(off + (size_t)(P * g.L * p->m * p->n) * 4, 1024);
  return DG_OK;
}

// Wave gate (auto): AG plans whose wave of co-resident tiles touches more
// full-K operand strips than about three quarters of L2 holds, or more than
// about three eighths when a wave spans every tile row of its block (then
// every wave re-reads all of the block's row strips).  Tiles that share a
// strip otherwise drift apart by more than its L2 lifetime unless the CTAs
// start each wave together.
bool wave_sync_on(const dg_plan_s* p) {
  if (p->wave_sync >= 0) return p->wave_sync == 1;
  if (!is_ag(p->schedule)) return false;
  const dg::Geom& g = p->g;
  const int64_t units = p->cg == 2 ? p->max_pairs : p->num_sms;
  if (units <= 0 || g.tiles_m <= 0) return false;
  const double wm = (double)std::min<int64_t>(g.group_m, g.tiles_m);
  const double wn = std::min((double)g.tiles_n * g.L, (double)units / wm);
  const double strip = (double)g.BN * (double)p->k * (double)p->esz;  // 256 rows x K elements
  const double footprint = (wm + wn) * strip;
  const double mib = 1024.0 * 1024.0;
  return footprint > 96.0 * mib || (g.tiles_m <= g.group_m && footprint > 48.0 * mib);
}

// Multicast of B rows between the two CTA pairs of a cluster of four: the
// pairs take tiles 2i and 2i + 1 of the order, so every such pair of tiles
// must lie in one (step, rank, batch) block and read the same B rows (the
// grouped raster sweeps even-height groups of tile rows column by column).
//
// AG plans only: the two pairs of a cluster run their operand stages in step,
// so a pair's MMAs depend on the other pair's epilogue having freed its
// accumulator; an RS epilogue may wait there for a hand-off that the other
// pair's epilogue still holds.
bool multicast_ok(dg_plan_s* p, const dg::Geom& g) {
  int& ok = p->mc_ok[g.order == 1 ? 1 : 0];
  if (ok < 0) {
    ok = p->cg == 2 && is_ag(p->schedule) && g.total_tiles % 2 == 0 && g.tiles_block % 2 == 0;
    for (int64_t i = 0; ok && i < g.total_tiles / 2; ++i) {
      const dg::Tile a = dg::decode_tile(g, 2 * i), b = dg::decode_tile(g, 2 * i + 1);
      ok = a.s == b.s && a.r == b.r && a.l == b.l && a.b_map == b.b_map && a.b_row == b.b_row &&
           a.k_blocks == b.k_blocks && (g.sched != dg::SCHED_AG_B || a.flag == b.flag);
    }
  }
  return ok == 1;
}

// Automatic for AG plans with K >= 16384: their long tiles keep the two pairs
// of a cluster in step cheaply, and their long runs are held to the power
// limit, where a quarter less L2-to-SM traffic buys clock (+1.5 % on the TP=8
// AG workloads) that outweighs the SMs clusters of four leave idle (the TP=2
// shape and the RS plans measured 2-7 % slower with it).
bool multicast_wanted(const dg_plan_s* p) {
  return p->multicast == 1 || (p->multicast < 0 && is_ag(p->schedule) && p->k >= 16384);
}

int rt_init(dg_plan_s* p) {
  if (p->rt) return DG_OK;
  int dev = 0;
  DG_CUDA(cudaGetDevice(&dev));
  int major = 0, minor = 0;
  DG_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  DG_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (major != 10)
    return fail(DG_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                major, minor);
  DG_CUDA(cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev));
#define DG_SMEM_ATTR(CG, EPI, F8)                                                                  \
  DG_CUDA(cudaFuncSetAttribute(dg::dg_gemm_kernel<CG, EPI, F8>,                                   \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dg::Cfg<CG, EPI>::SMEM_BYTES))
  DG_SMEM_ATTR(1, 0, 0);
  DG_SMEM_ATTR(1, 1, 0);
  DG_SMEM_ATTR(2, 0, 0);
  DG_SMEM_ATTR(2, 1, 0);
  DG_SMEM_ATTR(1, 0, 1);
  DG_SMEM_ATTR(1, 1, 1);
  DG_SMEM_ATTR(2, 0, 1);
  DG_SMEM_ATTR(2, 1, 1);
  DG_SMEM_ATTR(1, 2, 0);
  DG_SMEM_ATTR(2, 2, 0);
  DG_SMEM_ATTR(1, 2, 1);
  DG_SMEM_ATTR(2, 2, 1);
  DG_SMEM_ATTR(1, 3, 0);
  DG_SMEM_ATTR(2, 3, 0);
  DG_SMEM_ATTR(1, 3, 1);
  DG_SMEM_ATTR(2, 3, 1);
  DG_SMEM_ATTR(1, 4, 0);
  DG_SMEM_ATTR(2, 4, 0);
  DG_SMEM_ATTR(1, 4, 1);
  DG_SMEM_ATTR(2, 4, 1);
#undef DG_SMEM_ATTR
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 256, 1, 1);
    cfg.blockDim = dim3(dg::NUM_THREADS, 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl0 = 0, ncl1 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 0>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&ncl0, dg::dg_gemm_kernel<2, 0, 0>, &cfg));
    cfg.dynamicSmemBytes = dg::Cfg<2, 1>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&ncl1, dg::dg_gemm_kernel<2, 1, 0>, &cfg));
    int ncl2 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 2>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&ncl2, dg::dg_gemm_kernel<2, 2, 0>, &cfg));
    int ncl3 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 3>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&ncl3, dg::dg_gemm_kernel<2, 3, 0>, &cfg));
    int ncl4 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 4>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&ncl4, dg::dg_gemm_kernel<2, 4, 0>, &cfg));
    p->max_pairs = std::min(std::min(std::min(ncl0, ncl1), std::min(ncl2, ncl3)), ncl4);
    attr[0].val.clusterDim.x = 4;
    cfg.gridDim = dim3(4 * 256, 1, 1);
    int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 0>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&q0, dg::dg_gemm_kernel<2, 0, 0>, &cfg));
    cfg.dynamicSmemBytes = dg::Cfg<2, 1>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&q1, dg::dg_gemm_kernel<2, 1, 0>, &cfg));
    cfg.dynamicSmemBytes = dg::Cfg<2, 2>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&q2, dg::dg_gemm_kernel<2, 2, 0>, &cfg));
    cfg.dynamicSmemBytes = dg::Cfg<2, 3>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&q3, dg::dg_gemm_kernel<2, 3, 0>, &cfg));
    int q4 = 0;
    cfg.dynamicSmemBytes = dg::Cfg<2, 4>::SMEM_BYTES;
    DG_CUDA(cudaOccupancyMaxActiveClusters(&q4, dg::dg_gemm_kernel<2, 4, 0>, &cfg));
    p->max_quads = std::min(std::min(std::min(q0, q1), std::min(q2, q3)), q4);
  }
  DG_CUDA(cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming));
  DG_CUDA(cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming));
  p->device = dev;
  p->rt = true;
  return DG_OK;
}

// Operand map: `rows` rows of `inner` elements (row pitch `pitch_elems`), box
// of one 128-byte K block x `box_rows` rows, 128-byte swizzle.  esz = 2 (bf16)
// or 1 (fp8, moved as bytes).
int encode_map(const Driver& drv, CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
               int64_t pitch_elems, int box_rows, int esz) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch_elems * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(dg::KROW_BYTES / esz), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = drv.encode(map, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %lld x %lld pitch %lld", (int)r,
                (long long)inner, (long long)rows, (long long)pitch_elems);
  return DG_OK;
}

// Epilogue chunk map: `rows` x `cols` elements (fp32 or bf16) with a row pitch
// of `cols`, box of 32 columns x `box_rows` rows (128: a CTA's chunk, staged
// epilogue; 32: a warp's, per-warp epilogue), swizzle matching the 32-column
// chunk's row bytes (128 B for fp32, 64 B for bf16).
int encode_epi_map(const Driver& drv, CUtensorMap* map, const void* base, bool f32, int64_t cols,
                   int64_t rows, int box_rows) {
  const int64_t esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esz)};
  cuuint32_t box[2] = {(cuuint32_t)dg::XCOLS, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = drv.encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the %s epilogue map %lld x %lld", (int)r,
                f32 ? "fp32" : "bf16", (long long)rows, (long long)cols);
  return DG_OK;
}

// Maps of the staged epilogue (caller pointers may change from run to run).
int build_epi_maps(dg_plan_s* p, const Driver& drv, const void* C, void* D, uint8_t* ws) {
  std::memset(&p->kp.tmX, 0, sizeof(CUtensorMap));
  std::memset(&p->kp.tmC, 0, sizeof(CUtensorMap));
  std::memset(&p->kp.tmD, 0, sizeof(CUtensorMap));
  if (p->epi == 0) return DG_OK;
  const int64_t rows = p->l * p->m;
  const int br = epi_box_rows(p);
  int rc = DG_OK;
  if (p->out_type == DG_TYPE_BF16 || p->out_type == DG_TYPE_F32) {  // fp8 D: direct stores only
    rc = encode_epi_map(drv, &p->kp.tmD, D, p->out_type == DG_TYPE_F32, p->n, rows, br);
    if (rc) return rc;
  }
  if (C && p->beta != 0.f) {
    rc = encode_epi_map(drv, &p->kp.tmC, C, false, p->n, rows, br);
    if (rc) return rc;
  }
  std::memset(&p->kp.tmS, 0, sizeof(CUtensorMap));
  std::memset(&p->kp.tmR, 0, sizeof(CUtensorMap));
  if (!is_ag(p->schedule) && p->tp > 1 && p->cep) {
    const dg::Geom& g = p->g;
    rc = encode_epi_map(drv, &p->kp.tmS, ws + p->off_send, true, g.blk_n, p->tp * g.L * g.blk_m, br);
    if (rc) return rc;
    rc = encode_epi_map(drv, &p->kp.tmR, ws + p->off_recv, true, g.blk_n, 2 * p->tp * g.L * g.blk_m, br);
    if (rc) return rc;
  } else if (!is_ag(p->schedule) && p->tp > 1) {
    rc = encode_epi_map(drv, &p->kp.tmX, ws + p->off_partial, true, p->n, rows, br);
    if (rc) return rc;
  }
  return DG_OK;
}

int build_maps(dg_plan_s* p, const Driver& drv, const void* A, const void* B, uint8_t* ws, bool mc) {
  if (p->map_key[0] == A && p->map_key[1] == B && p->map_key[2] == ws && p->map_mc == mc) return DG_OK;
  std::memset(p->kp.tmA, 0, sizeof(p->kp.tmA));
  std::memset(p->kp.tmB, 0, sizeof(p->kp.tmB));
  const dg::Geom& g = p->g;
  const int64_t P = p->tp;
  int rc = DG_OK;
  p->n_maps = 0;
  // each CTA loads its own rows of the tile: 128 of A; 256 (CG = 1) or 128 (CG = 2) of B
  const int a_box = dg::Cfg<1>::A_ROWS;
  // (with multicast each CTA loads half of its B rows for both pairs)
  const int b_box = mc ? dg::Cfg<2>::B_ROWS / 2 : p->cg == 2 ? dg::Cfg<2>::B_ROWS : dg::Cfg<1>::B_ROWS;
  static_assert(dg::Cfg<2, 0>::B_ROWS == dg::Cfg<2, 1>::B_ROWS, "box rows do not depend on the epilogue");
  if (p->k > 0) {
    if (is_ag(p->schedule)) {
      rc = encode_map(drv, &p->kp.tmA[0], A, p->k, g.L * p->m, p->k, a_box, p->esz);
      if (rc) return rc;
      rc = encode_map(drv, &p->kp.tmB[0], B, p->k, g.L * p->n, p->k, b_box, p->esz);
      if (rc) return rc;
      p->n_maps = 1;
      if (P > 1) {
        const int64_t slot_rows = P * (P - 1) * g.L * g.shard;
        if (p->schedule == DG_AG_ROTATING_A) {
          rc = encode_map(drv, &p->kp.tmA[1], ws + p->off_slots, p->k, slot_rows, p->k, a_box, p->esz);
          p->kp.tmB[1] = p->kp.tmB[0];
        } else {
          rc = encode_map(drv, &p->kp.tmB[1], ws + p->off_slots, p->k, slot_rows, p->k, b_box, p->esz);
          p->kp.tmA[1] = p->kp.tmA[0];
        }
        if (rc) return rc;
        p->n_maps = 2;
      }
    } else {
      const auto* a8 = static_cast<const uint8_t*>(A);  // byte addressing: K-slab offsets
      const auto* b8 = static_cast<const uint8_t*>(B);
      for (int64_t r = 0; r < P; ++r) {
        rc = encode_map(drv, &p->kp.tmA[r], a8 + r * g.Ks * p->esz, g.Ks, g.L * p->m, p->k, a_box, p->esz);
        if (rc) return rc;
        rc = encode_map(drv, &p->kp.tmB[r], b8 + r * g.Ks * p->esz, g.Ks, g.L * p->n, p->k, b_box, p->esz);
        if (rc) return rc;
      }
      p->n_maps = (int)P;
    }
  }
  p->map_key[0] = A;
  p->map_key[1] = B;
  p->map_key[2] = ws;
  p->map_mc = mc;
  return DG_OK;
}

// Device-to-device transfer of `rows` contiguous rows of `row_bytes` bytes.
//
// kind 0 (the AG shard transfers' default): a two-dimensional copy in the
// operand's own rows (pitch = row bytes).  Two-dimensional copies run on a copy engine beside a kernel
// that fills every SM, ~1.0 TB/s on GB300 (several such copies on separate
// streams share that rate).
// kind 1: one-dimensional cudaMemcpyAsync, which runs as a copy kernel on the
// SMs and so only starts where the persistent GEMM kernel leaves registers
// free (such copies stall until the kernel exits when it holds 47 K of an
// SM's 64 K registers, and move 3.2 TB/s when they get SMs).
// kind 2: a two-dimensional copy reshaped to at least kTallRows rows.  On
// GB300 a copy of 65,536 rows or more moves 1.8-2.1 TB/s where the same bytes
// in fewer, wider rows move ~1.0 TB/s.  The bytes are contiguous on both
// sides, so any row width that divides them gives the same result; the widest
// power of two that keeps kTallRows rows is taken and a remainder shorter than
// one row goes as a one-row copy.  The default for the RS hand-off, whose
// merged band copies (>= 32 MiB) it moves ~1.8 TB/s (RS-TilingB 12% faster
// than in rows); for the AG shard transfers it takes more of the HBM
// bandwidth and power beside the GEMM kernel, and those fused runs measured no
// faster (AG-RotatingB a few percent slower).  Below ~16 MiB the rows it needs
// get narrow (128 B at 8 MiB) and it is slower than kind 0.
constexpr size_t kTallRows = 65536;
constexpr size_t kMinTallWidth = 128;

cudaError_t ce_copy(void* dst, const void* src, size_t row_bytes, size_t rows, cudaStream_t st, int kind) {
  const size_t bytes = row_bytes * rows;
  if (kind == 1) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  if (kind == 2 && rows < kTallRows && bytes >= kTallRows * kMinTallWidth) {
    size_t w = kMinTallWidth;
    while (w * 2 * kTallRows <= bytes) w *= 2;
    const size_t h = bytes / w, body = h * w;
    cudaError_t e = cudaMemcpy2DAsync(dst, w, src, w, w, h, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess || body == bytes) return e;
    const size_t rest = bytes - body;
    return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + body, rest, static_cast<const uint8_t*>(src) + body, rest,
                             rest, 1, cudaMemcpyDeviceToDevice, st);
  }
  return cudaMemcpy2DAsync(dst, row_bytes, src, row_bytes, row_bytes, rows, cudaMemcpyDeviceToDevice, st);
}

void CUDART_CB sleep_cb(void* ms) {
  std::this_thread::sleep_for(std::chrono::milliseconds((int64_t)(intptr_t)ms));
}

// Plan-owned copy streams beyond the caller's (created on first use, each with
// an event the main stream joins on).
int ensure_extra_streams(dg_plan_s* p, int want) {
  while (p->n_extra < want) {
    DG_CUDA(cudaStreamCreateWithFlags(&p->extra[p->n_extra], cudaStreamNonBlocking));
    DG_CUDA(cudaEventCreateWithFlags(&p->extra_done[p->n_extra], cudaEventDisableTiming));
    p->n_extra++;
  }
  return DG_OK;
}

// The (step, rank) blocks of steps >= first_step in the order the kernel's
// tiles visit them: step-major, or for the upload-frontier order by groups of
// max(rank, shard).
struct Block {
  int64_t s, r;
};
std::vector<Block> consumption_order(const dg::Geom& g, int64_t first_step) {
  std::vector<Block> out;
  const int64_t P = g.P;
  if (g.order == 1) {
    for (int64_t b = 0; b < P * P; ++b) {
      int64_t r = 0, j = 0;
      dg::frontier_block(b, &r, &j);
      const int64_t s = (j - r + P) % P;
      if (s >= first_step) out.push_back({s, r});
    }
  } else {
    for (int64_t s = first_step; s < P; ++s)
      for (int64_t r = 0; r < P; ++r) out.push_back({s, r});
  }
  return out;
}

// Shard transfers of every rank and step s in [s_lo, s_hi] (s >= 1), each
// chunk followed by its ready-flag write on the same stream, in the order the
// kernel consumes them.  Chunks are dealt round-robin over `ns` streams;
// `*idx` is the enqueue index of the first chunk (and on return of the next),
// so that a run enqueued in two parts deals and numbers its chunks as one.
// With `wait_up` (inputs uploaded by the same call) a stream first waits for
// the upload of the rank whose home shard it copies.
int enqueue_copies(dg_plan_s* p, const Driver& drv, const void* A, const void* B, uint8_t* ws,
                   cudaStream_t* streams, int ns, bool pace, bool wait_up, int64_t s_lo, int64_t s_hi,
                   int64_t* idx_io) {
  NvtxRange range("dg_enqueue_copies");
  auto* progress = reinterpret_cast<uint32_t*>(ws + p->off_status + kProgressOffset);
  const dg::Geom& g = p->g;
  const int64_t P = p->tp;
  if (p->fault_delay_ms > 0 && *idx_io == 0)
    for (int i = 0; i < ns; ++i)
      DG_CUDA(cudaLaunchHostFunc(streams[i], sleep_cb, (void*)(intptr_t)p->fault_delay_ms));
  const bool rot_a = p->schedule == DG_AG_ROTATING_A;
  const auto* home = static_cast<const uint8_t*>(rot_a ? A : B);
  const int64_t row_bytes = p->k * p->esz;
  const int64_t outer = rot_a ? p->m : p->n;  // rows of one batch of the rotated operand
  const int64_t tile_rows = rot_a ? g.BM : g.BN;
  const int64_t chunk_rows = g.chunk_tiles * tile_rows;
  auto* slots = ws + p->off_slots;
  auto* flags = reinterpret_cast<uint32_t*>(ws + p->off_flags);
  uint32_t up_waited[8] = {};  // per stream: ranks whose upload it already waits for
  int64_t idx = *idx_io;
  int64_t last_s = 0;
  for (const Block& bk : consumption_order(p->kp.g, 1)) {
    const int64_t s = bk.s, r = bk.r;
    if (s < s_lo || s > s_hi) continue;
    if (pace && s >= 2 && s != last_s)
      // step s's shards move while the kernel computes step s - 1
      for (int i = 0; i < ns; ++i) {
        CUresult rc = drv.wait32((CUstream)streams[i], (CUdeviceptr)(progress + (s - 1)), 1u,
                                 CU_STREAM_WAIT_VALUE_GEQ);
        if (rc != CUDA_SUCCESS)
          return fail(rc == CUDA_ERROR_NOT_SUPPORTED ? DG_ERR_UNSUPPORTED : DG_ERR_CUDA,
                      "cuStreamWaitValue32 failed (%d)", (int)rc);
      }
    last_s = s;
    const int64_t j = (r + s) % P;
    for (int64_t l = 0; l < g.L; ++l) {
      const int64_t slot = (r * (P - 1) + (s - 1)) * g.L + l;
      for (int64_t c = 0; c < g.nchunks; ++c, ++idx) {
        cudaStream_t st = streams[idx % ns];
        if (wait_up && !((up_waited[idx % ns] >> j) & 1u)) {
          DG_CUDA(cudaStreamWaitEvent(st, p->ev_up[j], 0));
          up_waited[idx % ns] |= 1u << j;
        }
        const int64_t row0 = c * chunk_rows;
        const int64_t rows = std::min(chunk_rows, g.shard - row0);
        if (rows > 0 && row_bytes > 0) {  // K = 0: nothing to move, the flag still goes
          const uint8_t* src = home + (l * outer + j * g.shard + row0) * row_bytes;
          uint8_t* dst = slots + (slot * g.shard + row0) * row_bytes;
          DG_CUDA(ce_copy(dst, src, (size_t)row_bytes, (size_t)rows, st, p->copy_kind < 0 ? 0 : p->copy_kind));
        }
        if (idx != p->fault_skip) {
          CUresult rc = drv.write32((CUstream)st, (CUdeviceptr)(flags + slot * g.nchunks + c),
                                    p->epoch, 0);
          if (rc != CUDA_SUCCESS)
            return fail(rc == CUDA_ERROR_NOT_SUPPORTED ? DG_ERR_UNSUPPORTED : DG_ERR_CUDA,
                        "cuStreamWriteValue32 failed (%d)", (int)rc);
        }
      }
    }
  }
  *idx_io = idx;
  return DG_OK;
}

int launch_kp(dg_plan_s* p, const dg::KParams& kp, cudaStream_t st) {
  const int64_t tiles = kp.g.total_tiles;
  if (p->cg == 1) {
    int64_t grid = p->grid_req > 0 ? p->grid_req : p->num_sms;
    grid = std::min<int64_t>(grid, tiles);
    if (grid <= 0) return DG_OK;
    const bool f8 = p->esz == 1;
    if (p->epi == 4 && f8)
      dg::dg_gemm_kernel<1, 4, 1><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 4>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 4)
      dg::dg_gemm_kernel<1, 4, 0><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 4>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 3 && f8)
      dg::dg_gemm_kernel<1, 3, 1><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 3>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 3)
      dg::dg_gemm_kernel<1, 3, 0><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 3>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 2 && f8)
      dg::dg_gemm_kernel<1, 2, 1><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 2>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 2)
      dg::dg_gemm_kernel<1, 2, 0><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 2>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 1 && f8)
      dg::dg_gemm_kernel<1, 1, 1><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 1>::SMEM_BYTES, st>>>(kp);
    else if (p->epi == 1)
      dg::dg_gemm_kernel<1, 1, 0><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 1>::SMEM_BYTES, st>>>(kp);
    else if (f8)
      dg::dg_gemm_kernel<1, 0, 1><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 0>::SMEM_BYTES, st>>>(kp);
    else
      dg::dg_gemm_kernel<1, 0, 0><<<(unsigned)grid, dg::NUM_THREADS, dg::Cfg<1, 0>::SMEM_BYTES, st>>>(kp);
    DG_CUDA(cudaGetLastError());
    return DG_OK;
  }
  // CTA pairs: every pair must be co-resident (RS tiles wait on earlier tiles).
  // With multicast, clusters of two pairs, each cluster taking two tiles at a time.
  const int csize = kp.mc ? 4 : 2;
  int64_t units = p->grid_req > 0 ? p->grid_req / csize : (kp.mc ? p->max_quads : p->max_pairs);
  units = std::min<int64_t>(std::min<int64_t>(units, kp.mc ? p->max_quads : p->max_pairs), kp.mc ? tiles / 2 : tiles);
  if (units <= 0) return tiles > 0 ? fail(DG_ERR_UNSUPPORTED, "no co-resident CTA cluster") : DG_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(csize * units), 1, 1);
  cfg.blockDim = dim3(dg::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = p->epi == 4   ? dg::Cfg<2, 4>::SMEM_BYTES
                         : p->epi == 3 ? dg::Cfg<2, 3>::SMEM_BYTES
                         : p->epi == 2 ? dg::Cfg<2, 2>::SMEM_BYTES
                         : p->epi == 1 ? dg::Cfg<2, 1>::SMEM_BYTES
                                       : dg::Cfg<2, 0>::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool f8 = p->esz == 1;
  if (p->epi == 4 && f8)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 4, 1>, kp));
  else if (p->epi == 4)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 4, 0>, kp));
  else if (p->epi == 3 && f8)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 3, 1>, kp));
  else if (p->epi == 3)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 3, 0>, kp));
  else if (p->epi == 2 && f8)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 2, 1>, kp));
  else if (p->epi == 2)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 2, 0>, kp));
  else if (p->epi == 1 && f8)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 1, 1>, kp));
  else if (p->epi == 1)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 1, 0>, kp));
  else if (f8)
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 0, 1>, kp));
  else
    DG_CUDA(cudaLaunchKernelEx(&cfg, dg::dg_gemm_kernel<2, 0, 0>, kp));
  return DG_OK;
}

// Pacing of the AG shard transfers: the copies of step s >= 2 wait until the
// kernel has reached step s - 1 (progress words in the status area).  Off
// unless asked for: it measured neutral, and paced copies can only be
// enqueued after the kernel, so under a layer that serializes launches
// (a profiler, CUDA_LAUNCH_BLOCKING) they could not run before it.
bool copy_pace_on(const dg_plan_s* p) { return p->copy_pace == 1; }

int launch(dg_plan_s* p, cudaStream_t st, uint32_t wait_flags) {
  p->kp.wait_flags = wait_flags;
  return launch_kp(p, p->kp, st);
}

// ReduceScatter with copy-engine hand-off of the rotating partial (the
// "memcopy branch" form of RotatingC).  Rank r writes its step-s partial to
// its send buffer S_r; the kernel counts, per (rank, step, batch, band of 256
// rows), the half tiles written; a copy stream waits until the band is
// complete (and until the receiver has finished reading the same receive
// slot two steps earlier), copies it into the receiving rank's
// double-buffered receive buffer R_{r-1}[(s+1) & 1] and writes the band's
// ready flag, which rank r-1's epilogue waits on at step s+1.  The copies are
// enqueued step-major, so a copy waits only for tiles of its own step or the
// one before, and every tile only for copies of the step before.
int run_rs_ce(dg_plan_s* p, const Driver& drv, uint8_t* ws, cudaStream_t ms, cudaStream_t cs) {
  const dg::Geom& g = p->g;
  const int64_t P = p->tp, L = g.L, TM = g.tiles_m;
  const size_t ndone = (size_t)(P * P * L * TM);
  DG_CUDA(cudaMemsetAsync(ws + p->off_done, 0, ndone * 4, ms));
  const int ns = p->copy_streams;
  int rc = ensure_extra_streams(p, ns - 1);
  if (rc) return rc;
  cudaStream_t streams[8];
  streams[0] = cs;
  for (int i = 1; i < ns; ++i) streams[i] = p->extra[i - 1];
  DG_CUDA(cudaEventRecord(p->ev_fork, ms));
  rc = launch(p, ms, 0);
  if (rc) return rc;
  for (int i = 0; i < ns; ++i) DG_CUDA(cudaStreamWaitEvent(streams[i], p->ev_fork, 0));
  if (p->fault_delay_ms > 0)
    for (int i = 0; i < ns; ++i)
      DG_CUDA(cudaLaunchHostFunc(streams[i], sleep_cb, (void*)(intptr_t)p->fault_delay_ms));
  auto* done = reinterpret_cast<uint32_t*>(ws + p->off_done);
  auto* flags = reinterpret_cast<uint32_t*>(ws + p->off_flags);
  const uint32_t target = (uint32_t)(g.tiles_n * p->cg * epi_parts(p));  // half (quarter) tiles per band
  const size_t row_bytes = (size_t)g.blk_n * 4;
  auto idx = [&](int64_t q, int64_t s, int64_t l, int64_t b) { return ((q * P + s) * L + l) * TM + b; };
  auto check = [&](CUresult r, const char* what) {
    return r == CUDA_SUCCESS ? DG_OK
                             : fail(r == CUDA_ERROR_NOT_SUPPORTED ? DG_ERR_UNSUPPORTED : DG_ERR_CUDA, "%s failed (%d)",
                                    what, (int)r);
  };
  // Bands per copy: consecutive bands of one (rank, step, batch) are contiguous
  // in the send and receive buffers, so G of them go as one copy once all G
  // are counted complete (then G ready flags).  Auto: enough bands for >= 32
  // MiB, the size from which a copy reshaped to >= 65,536 rows reaches the
  // copy engines' full rate on GB300.
  const size_t band_bytes = row_bytes * (size_t)g.BM;
  int64_t G = p->ce_bands > 0 ? p->ce_bands : (int64_t)((size_t(32) << 20) + band_bytes - 1) / (int64_t)band_bytes;
  G = std::max<int64_t>(1, std::min<int64_t>(G, TM));
  int64_t n = 0;
  for (int64_t s = 0; s + 1 < P; ++s)
    for (int64_t r = 0; r < P; ++r) {
      const int64_t q = (r + P - 1) % P;  // the ring neighbour that adds the next K-slab
      for (int64_t l = 0; l < L; ++l)
        for (int64_t b0 = 0; b0 < TM; b0 += G, ++n) {
          const int64_t nb = std::min<int64_t>(G, TM - b0);
          cudaStream_t st = streams[n % ns];
          for (int64_t b = b0; b < b0 + nb; ++b) {
            rc = check(drv.wait32((CUstream)st, (CUdeviceptr)(done + idx(r, s, l, b)), target,
                                  CU_STREAM_WAIT_VALUE_GEQ),
                       "cuStreamWaitValue32");
            if (rc) return rc;
            if (s >= 1) {
              rc = check(drv.wait32((CUstream)st, (CUdeviceptr)(done + idx(q, s - 1, l, b)), target,
                                    CU_STREAM_WAIT_VALUE_GEQ),
                         "cuStreamWaitValue32");
              if (rc) return rc;
            }
          }
          const int64_t rows = std::min<int64_t>(nb * g.BM, g.blk_m - b0 * g.BM);
          const uint8_t* src = ws + p->off_send + (size_t)((r * L + l) * g.blk_m + b0 * g.BM) * row_bytes;
          uint8_t* dst = ws + p->off_recv + (size_t)(((2 * q + ((s + 1) & 1)) * L + l) * g.blk_m + b0 * g.BM) * row_bytes;
          DG_CUDA(ce_copy(dst, src, row_bytes, (size_t)rows, st, p->copy_kind < 0 ? 2 : p->copy_kind));
          for (int64_t b = b0; b < b0 + nb; ++b) {
            if (n == p->fault_skip && b == b0) continue;
            rc = check(drv.write32((CUstream)st, (CUdeviceptr)(flags + idx(q, s + 1, l, b)), p->epoch, 0),
                       "cuStreamWriteValue32");
            if (rc) return rc;
          }
        }
    }
  // After the kernel, raise every count: no copy-stream wait outlives a kernel
  // that stopped early (in a normal run every copy has already run by then).
  DG_CUDA(cudaMemsetAsync(ws + p->off_done, 0x7F, ndone * 4, ms));
  for (int i = 1; i < ns; ++i) {
    DG_CUDA(cudaEventRecord(p->extra_done[i - 1], streams[i]));
    DG_CUDA(cudaStreamWaitEvent(cs, p->extra_done[i - 1], 0));
  }
  DG_CUDA(cudaEventRecord(p->ev_join, cs));
  DG_CUDA(cudaStreamWaitEvent(ms, p->ev_join, 0));
  return DG_OK;
}

// Non-fused ReduceScatter baseline ("GEMM, then reduce"): one launch computes
// every rank's full partial over its K-slab into its own fp32 buffer; a
// separate kernel sums the partials, adds beta*C and writes D.
int run_rs_serial(dg_plan_s* p, const Driver& drv, const void* C, void* D, uint8_t* ws, cudaStream_t st) {
  p->kser = p->kp;
  p->kser.g = p->gser;
  p->kser.mc = 0;
  p->kser.rs_reduce = 0;
  p->kser.X = reinterpret_cast<float*>(ws + p->off_serial);
  p->kser.wait_flags = 0;
  std::memset(&p->kser.tmX, 0, sizeof(CUtensorMap));
  if (p->epi != 0) {
    int rc = encode_epi_map(drv, &p->kser.tmX, ws + p->off_serial, true, p->n, p->tp * p->l * p->m,
                            epi_box_rows(p));
    if (rc) return rc;
  }
  int rc = launch_kp(p, p->kser, st);
  if (rc) return rc;
  const int64_t n4 = p->l * p->m * p->n / 4;
  int64_t blocks = std::min<int64_t>((int64_t)p->num_sms * 8, (n4 + 255) / 256);
  if (blocks < 1) blocks = 1;
  dg::dg_reduce_partials_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      reinterpret_cast<const float*>(ws + p->off_serial), p->tp, n4,
      reinterpret_cast<const __nv_bfloat16*>(C), p->beta, D, p->out_type == DG_TYPE_F32 ? 1 : 0,
      p->out_type == DG_TYPE_E4M3 ? 1 : p->out_type == DG_TYPE_E5M2 ? 2 : 0, p->result_scale);
  DG_CUDA(cudaGetLastError());
  return DG_OK;
}

// --------------------------------------------------- runs with host buffers
//
// dg_run_host with DG_OPT_HOST_OVERLAP (default) in FUSED mode, with pinned
// host buffers: the kernel is launched at once and its tiles wait for their
// own inputs instead of for the whole upload, and D leaves the device one
// (step, rank) block at a time while later steps still run.
//   upload stream:   for f = 0..P-1: upload unit f (AG: rank f's home operand
//                    shards and C's row band M_f; RS: row slabs, see
//                    enqueue_upload_unit), then up_flags[f] = epoch (the
//                    producers and C-reading epilogues of the tiles that need
//                    unit f wait on it) and an event (AG shard transfers of
//                    rank f's home shard wait on it)
//   download stream: for every (step, rank) block that writes D, wait until
//                    the kernel has counted all its half tiles, then copy the
//                    block to the host
// The main stream joins both at the end, so the call stays one stream-ordered
// operation like the sequential form.

struct HostIO {
  const void* A;
  const void* B;
  const void* C;
  void* D;
};

int ensure_io(dg_plan_s* p) {
  if (p->io_rt) return DG_OK;
  DG_CUDA(cudaStreamCreateWithFlags(&p->up_st, cudaStreamNonBlocking));
  DG_CUDA(cudaStreamCreateWithFlags(&p->down_st, cudaStreamNonBlocking));
  DG_CUDA(cudaEventCreateWithFlags(&p->ev_io, cudaEventDisableTiming));
  DG_CUDA(cudaEventCreateWithFlags(&p->ev_up_done, cudaEventDisableTiming));
  DG_CUDA(cudaEventCreateWithFlags(&p->ev_down_done, cudaEventDisableTiming));
  for (int i = 0; i < 8; ++i) DG_CUDA(cudaEventCreateWithFlags(&p->ev_up[i], cudaEventDisableTiming));
  p->io_rt = true;
  return DG_OK;
}

// `rows` rows of `width` bytes at row pitch `pitch` (the same on both sides),
// as copies of at most kHostCopyBytes each.  Copy engines take copies in the
// order they were issued, so a shard transfer (or a download) queued behind
// one host copy of hundreds of MB waits for all of it while the kernel waits
// for that transfer; bounded pieces let the others in between.
constexpr size_t kHostCopyBytes = size_t(64) << 20;

int copy_rows(void* dst, const void* src, size_t pitch, size_t width, size_t rows, cudaMemcpyKind kind,
              cudaStream_t st) {
  if (width == 0 || rows == 0) return DG_OK;
  const size_t step = std::max<size_t>(1, kHostCopyBytes / std::max<size_t>(pitch, 1));
  for (size_t r0 = 0; r0 < rows; r0 += step) {
    const size_t n = std::min(step, rows - r0);
    DG_CUDA(cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + r0 * pitch, pitch,
                              static_cast<const uint8_t*>(src) + r0 * pitch, pitch, width, n, kind, st));
  }
  return DG_OK;
}

// Host-to-device copies of upload unit f, the inputs the tiles waiting on
// flag f need:
//   AG-RotatingA   rank f: A rows M_f, B rows N_f, C rows M_f (read by the
//                  tiles of shard f, which wait on unit f for their C)
//   AG-RotatingB   rank f: A rows M_f, B rows N_f, C rows M_f
//   RS-TilingA     B whole (unit 0 only), then A rows M_j and C rows M_j
//   RS-TilingB     A and C whole (unit 0 only), then B rows N_j
// with j = (f + 1) mod P, every batch l, C only when beta != 0.  An RS tile
// (s, r) works on slab (r + s + 1) mod P for every step, so it waits on unit
// (r + s) mod P (dg::upload_unit in the kernel).  Every copy is contiguous in
// host memory: row slabs rather than each rank's K columns or C's column
// blocks, and TilingB's C (whose slabs are column blocks) whole; strided host
// copies ran at a fraction of the link's rate.
int enqueue_upload_unit(dg_plan_s* p, const HostIO& io, const void* A, const void* B, void* C, int64_t f,
                        cudaStream_t st) {
  const dg::Geom& g = p->g;
  const int64_t L = g.L, M = p->m, N = p->n, K = p->k, P = p->tp;
  const size_t es = (size_t)p->esz, rowA = (size_t)K * es, rowC = (size_t)N * 2;
  auto* a_d = static_cast<uint8_t*>(const_cast<void*>(A));
  auto* b_d = static_cast<uint8_t*>(const_cast<void*>(B));
  auto* c_d = static_cast<uint8_t*>(C);
  const auto* a_h = static_cast<const uint8_t*>(io.A);
  const auto* b_h = static_cast<const uint8_t*>(io.B);
  const auto* c_h = static_cast<const uint8_t*>(io.C);
  const bool with_c = p->beta != 0.f;
  const auto H2D = cudaMemcpyHostToDevice;
  int rc = DG_OK;
  if (is_ag(p->schedule)) {
    for (int64_t l = 0; l < L && !rc; ++l) {
      const size_t a0 = (size_t)(l * M + f * g.blk_m) * rowA, b0 = (size_t)(l * N + f * g.blk_n) * rowA;
      rc = copy_rows(a_d + a0, a_h + a0, rowA, rowA, (size_t)g.blk_m, H2D, st);
      if (!rc) rc = copy_rows(b_d + b0, b_h + b0, rowA, rowA, (size_t)g.blk_n, H2D, st);
    }
    if (rc || !with_c) return rc;
    for (int64_t l = 0; l < L && !rc; ++l) {
      const size_t c0 = (size_t)(l * M + f * g.blk_m) * rowC;
      rc = copy_rows(c_d + c0, c_h + c0, rowC, rowC, (size_t)g.blk_m, H2D, st);
    }
    return rc;
  }
  const bool rs_a = p->schedule == DG_RS_TILING_A_ROTATING_C;
  const int64_t j = (f + 1) % P;
  if (f == 0) {  // the operand every tile reads whole (and TilingB's C)
    rc = rs_a ? copy_rows(b_d, b_h, rowA, rowA, (size_t)(L * N), H2D, st)
              : copy_rows(a_d, a_h, rowA, rowA, (size_t)(L * M), H2D, st);
    if (!rc && !rs_a && with_c) rc = copy_rows(c_d, c_h, rowC, rowC, (size_t)(L * M), H2D, st);
    if (rc) return rc;
  }
  for (int64_t l = 0; l < L && !rc; ++l) {
    const size_t o = rs_a ? (size_t)(l * M + j * g.blk_m) * rowA : (size_t)(l * N + j * g.blk_n) * rowA;
    rc = rs_a ? copy_rows(a_d + o, a_h + o, rowA, rowA, (size_t)g.blk_m, H2D, st)
              : copy_rows(b_d + o, b_h + o, rowA, rowA, (size_t)g.blk_n, H2D, st);
  }
  if (rc || !with_c || !rs_a) return rc;
  for (int64_t l = 0; l < L && !rc; ++l) {
    const size_t c0 = (size_t)(l * M + j * g.blk_m) * rowC;
    rc = copy_rows(c_d + c0, c_h + c0, rowC, rowC, (size_t)g.blk_m, H2D, st);
  }
  return rc;
}

// Uploads of every unit on the upload stream, after everything already on the
// main stream (which may still read the device inputs).
int enqueue_uploads(dg_plan_s* p, const Driver& drv, const HostIO& io, const void* A, const void* B, void* C,
                    uint8_t* ws) {
  auto* up = reinterpret_cast<uint32_t*>(ws + p->off_status + kUpOffset);
  if (p->fault_delay_ms > 0)
    DG_CUDA(cudaLaunchHostFunc(p->up_st, sleep_cb, (void*)(intptr_t)p->fault_delay_ms));
  for (int64_t r = 0; r < p->tp; ++r) {
    int rc = enqueue_upload_unit(p, io, A, B, C, r, p->up_st);
    if (rc) return rc;
    CUresult cr = drv.write32((CUstream)p->up_st, (CUdeviceptr)(up + r), p->epoch, 0);
    if (cr != CUDA_SUCCESS)
      return fail(cr == CUDA_ERROR_NOT_SUPPORTED ? DG_ERR_UNSUPPORTED : DG_ERR_CUDA, "cuStreamWriteValue32 failed (%d)",
                  (int)cr);
    DG_CUDA(cudaEventRecord(p->ev_up[r], p->up_st));
  }
  DG_CUDA(cudaEventRecord(p->ev_up_done, p->up_st));
  return DG_OK;
}

// Downloads of D, block by block as the kernel finishes them.  RS-TilingB
// writes all of D in its last step and its blocks are column blocks, so it
// waits for every block of that step and copies D whole (contiguous).
int enqueue_downloads(dg_plan_s* p, const Driver& drv, const HostIO& io, const void* D, uint8_t* ws) {
  const dg::Geom& g = p->g;
  const int64_t P = p->tp, L = g.L, M = p->m;
  const size_t de = p->out_type == DG_TYPE_F32 ? 4 : (p->out_type == DG_TYPE_BF16 ? 2 : 1);
  const size_t pitch = (size_t)p->n * de;
  auto* done = reinterpret_cast<uint32_t*>(ws + p->off_ddone);
  const uint32_t target = (uint32_t)(g.tiles_block * p->cg * epi_parts(p));  // half (quarter) tiles of a block
  const auto* d_d = static_cast<const uint8_t*>(D);
  auto* d_h = static_cast<uint8_t*>(io.D);
  const auto D2H = cudaMemcpyDeviceToHost;
  const bool ag = is_ag(p->schedule);
  for (const Block& bk : consumption_order(p->kp.g, ag ? 0 : P - 1)) {
    const int64_t s = bk.s, r = bk.r;
    CUresult cr = drv.wait32((CUstream)p->down_st, (CUdeviceptr)(done + s * P + r), target,
                             CU_STREAM_WAIT_VALUE_GEQ);
    if (cr != CUDA_SUCCESS)
      return fail(cr == CUDA_ERROR_NOT_SUPPORTED ? DG_ERR_UNSUPPORTED : DG_ERR_CUDA,
                  "cuStreamWaitValue32 failed (%d)", (int)cr);
    const int64_t j = ag ? (r + s) % P : r;  // the RS block of the last step is the rank's own slab
    int rc = DG_OK;
    if (p->schedule == DG_RS_TILING_B_ROTATING_C) {
      if (r == P - 1) rc = copy_rows(d_h, d_d, pitch, pitch, (size_t)(L * M), D2H, p->down_st);
    } else {
      for (int64_t l = 0; l < L && !rc; ++l) {
        int64_t row0, col0, cols;
        if (p->schedule == DG_AG_ROTATING_A) row0 = j * g.blk_m, col0 = r * g.blk_n, cols = g.blk_n;
        else if (p->schedule == DG_AG_ROTATING_B) row0 = r * g.blk_m, col0 = j * g.blk_n, cols = g.blk_n;
        else row0 = j * g.blk_m, col0 = 0, cols = p->n;
        const size_t o = (size_t)(l * M + row0) * pitch + (size_t)col0 * de;
        rc = copy_rows(d_h + o, d_d + o, pitch, (size_t)cols * de, (size_t)g.blk_m, D2H, p->down_st);
      }
    }
    if (rc) return rc;
  }
  return DG_OK;
}

bool pinned_host(const void* q) {
  if (!q) return false;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

int dispatch_run(dg_plan_s* p, const Driver& drv, const void* A, const void* B, const dg_bf16_t* C, void* D,
                 uint8_t* ws, cudaStream_t ms, cudaStream_t cs, bool rs_serial, bool pace, bool wait_up);

int run_impl(dg_plan_s* p, const void* A, const void* B, const dg_bf16_t* C, const dg_bf16_t* bias, void* D,
             void* workspace, void* main_stream, void* copy_stream, const HostIO* io) {
  NvtxRange range("dg_run");
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  p->static_dev = -1;
  if (p->g.total_tiles == 0) return DG_OK;  // empty output
  if (!A || !B || !D) return fail(DG_ERR_ARG, "A, B and D must be non-NULL");
  if (p->beta != 0.f && !C) return fail(DG_ERR_ARG, "C is NULL but beta != 0");
  auto misaligned = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) != 0; };
  if (misaligned(A, 16) || misaligned(B, 16) || misaligned(D, 16) || (C && misaligned(C, 16)) ||
      (bias && misaligned(bias, 16)))
    return fail(DG_ERR_ARG, "A, B, C, D and bias must be 16-byte aligned");
  // bytes this run uses (no side effect on the plan's SERIAL sizing record)
  const size_t need =
      (!is_ag(p->schedule) && p->mode == DG_MODE_SERIAL) ? p->ws_bytes_serial : p->ws_bytes_base;
  if (need > 0 && (!workspace || misaligned(workspace, 256)))
    return fail(DG_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
  const bool rs_serial = !is_ag(p->schedule) && p->mode == DG_MODE_SERIAL;
  if (rs_serial && !p->serial_ws)
    return fail(DG_ERR_STATE, "RS SERIAL needs the larger workspace: size it with dg_workspace_bytes in SERIAL mode");
  int rc = rt_init(p);
  if (rc) return rc;
  Driver drv;
  rc = get_driver(&drv);
  if (rc) return rc;
  auto ms = static_cast<cudaStream_t>(main_stream);
  auto cs = static_cast<cudaStream_t>(copy_stream);
  auto* ws = static_cast<uint8_t*>(workspace);

  // Epochs grow per plan across all of its workspaces, so flag words left in
  // any workspace by this plan's earlier runs stay below the current epoch.
  // A workspace new to this plan starts from zeroed flags.  Only when the
  // epoch would overflow is it restarted, and then every other workspace of
  // this plan is forgotten so that it is cleared again on its next use.
  bool clear = false;
  const bool wrap = (uint64_t)(p->epoch + 2) * (uint64_t)p->tp >= 0x7FFFFFFFull;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (wrap)
      for (auto it = g_ws_owner.begin(); it != g_ws_owner.end();)
        it = it->second == p->id ? g_ws_owner.erase(it) : std::next(it);
    auto it = g_ws_owner.find(workspace);
    if (it == g_ws_owner.end() || it->second != p->id) {
      g_ws_owner[workspace] = p->id;
      clear = true;
    }
  }
  // Under stream capture the run's epoch is frozen into the graph, so every
  // replay must start from zeroed status and flag words: clear them in the
  // graph itself (one memset node).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  DG_CUDA(cudaStreamIsCapturing(ms, &cap));
  if (cap == cudaStreamCaptureStatusActive) clear = true;
  if (clear) DG_CUDA(cudaMemsetAsync(ws, 0, p->off_flags + (size_t)p->n_flags * 4, ms));
  if (wrap) p->epoch = 0;
  p->epoch += 1;

  dg::KParams& kp = p->kp;
  kp.g = p->g;
  // Upload-frontier block order (AG): asked for, or automatic when this run
  // uploads its inputs rank by rank.
  kp.g.order = is_ag(p->schedule) && (p->tile_order == 1 || (p->tile_order < 0 && io)) ? 1 : 0;
  // B multicast between pairs (not for the RS baseline's per-rank GEMMs)
  const bool mc = multicast_wanted(p) && !rs_serial && p->max_quads > 0 && multicast_ok(p, kp.g);
  kp.mc = mc ? 1u : 0u;
  rc = build_maps(p, drv, A, B, ws, mc);
  if (rc) return rc;
  rc = build_epi_maps(p, drv, C, D, ws);
  if (rc) return rc;
  kp.C = reinterpret_cast<const __nv_bfloat16*>(C);
  kp.D = D;
  kp.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  kp.out_f32 = p->out_type == DG_TYPE_F32 ? 1u : 0u;
  kp.out_fp8 = p->out_type == DG_TYPE_E4M3 ? 1u : p->out_type == DG_TYPE_E5M2 ? 2u : 0u;
  kp.result_scale = p->result_scale;
  kp.X = reinterpret_cast<float*>(ws + p->off_partial);
  kp.flags = reinterpret_cast<uint32_t*>(ws + p->off_flags);
  kp.status = reinterpret_cast<unsigned long long*>(ws + p->off_status);
  kp.epoch = p->epoch;
  // scaled GEMM: alpha * scale_a * scale_b folded into one fp32 factor; the
  // mean over ranks weighs every rank's product and bias by 1/P (exact: P is a
  // power of two)
  const float w = p->reduce_op == DG_REDUCE_AVG ? 1.f / (float)p->tp : 1.f;
  kp.alpha = p->alpha * p->scale_a * p->scale_b * w;
  kp.bias_scale = w;
  kp.beta = p->beta;
  {
    const int tm = p->cg == 2 ? dg::Cfg<2>::TILE_M : dg::Cfg<1>::TILE_M;
    const uint32_t fa = p->esz == 1 ? (p->a_type == DG_TYPE_E5M2 ? 1u : 0u) : 1u;
    const uint32_t fb = p->esz == 1 ? (p->b_type == DG_TYPE_E5M2 ? 1u : 0u) : 1u;
    kp.idesc = dg::idesc_f32acc(tm, dg::TILE_N, fa, fb);
  }
  kp.n_maps = p->n_maps;
  kp.l2_hint = p->l2_hint;
  kp.done = reinterpret_cast<uint32_t*>(ws + p->off_done);
  kp.S = reinterpret_cast<float*>(ws + p->off_send);
  kp.R = reinterpret_cast<const float*>(ws + p->off_recv);
  kp.wave_sync = wave_sync_on(p) ? 1u : 0u;
  {
    // Middle RS steps may add alpha' * acc into the partial by TMA reduction
    // (a round-to-nearest fp32 add at the L2) instead of loading the partial
    // and storing fmaf(alpha', acc, partial).  That rounds the product, then
    // the sum.  With alpha' a power of two (or zero) the product is exact and
    // both give the same bits; otherwise they differ in the last bits of the
    // partial.  Automatic without a bias (the product is then all that is
    // added); chunks that are not whole, the direct epilogue and the
    // copy-engine hand-off still load, fmaf and store.
    const bool want = p->rs_reduce == 1 || (p->rs_reduce < 0 && bias == nullptr);
    kp.rs_reduce = want && p->epi != 0 && !is_ag(p->schedule) && !p->cep ? 1u : 0u;
  }
  kp.wave_ctr = reinterpret_cast<uint32_t*>(ws + p->off_status + 64);
  if (kp.wave_sync) DG_CUDA(cudaMemsetAsync(ws + p->off_status + 64, 0, 4, ms));
  const bool pace = copy_pace_on(p) && kp.g.order == 0 && is_ag(p->schedule) && p->tp > 2 &&
                    p->mode == DG_MODE_FUSED && cs != ms && cs != nullptr;
  kp.progress = pace ? reinterpret_cast<uint32_t*>(ws + p->off_status + kProgressOffset) : nullptr;
  if (pace) DG_CUDA(cudaMemsetAsync(ws + p->off_status + kProgressOffset, 0, (size_t)p->tp * 4, ms));
  kp.timeout_ns = (uint64_t)p->timeout_ms * 1000000ull;
  kp.hang_ns = kp.timeout_ns * 4 + 1000000000ull;
  kp.up_flags = nullptr;
  kp.d_done = nullptr;
  if (io) {
    rc = ensure_io(p);
    if (rc) return rc;
    kp.up_flags = reinterpret_cast<const uint32_t*>(ws + p->off_status + kUpOffset);
    kp.d_done = reinterpret_cast<uint32_t*>(ws + p->off_ddone);
    DG_CUDA(cudaMemsetAsync(ws + p->off_ddone, 0, (size_t)(p->tp * p->tp) * 4, ms));
    DG_CUDA(cudaEventRecord(p->ev_io, ms));
    DG_CUDA(cudaStreamWaitEvent(p->up_st, p->ev_io, 0));
    DG_CUDA(cudaStreamWaitEvent(p->down_st, p->ev_io, 0));
    rc = enqueue_uploads(p, drv, *io, A, B, const_cast<dg_bf16_t*>(C), ws);
    if (rc) return rc;
  }
  rc = dispatch_run(p, drv, A, B, C, D, ws, ms, cs, rs_serial, pace, io != nullptr);
  if (io) {
    const int rc_down = rc ? rc : enqueue_downloads(p, drv, *io, D, ws);
    // Raise every count once the kernel is done (one that stopped early leaves
    // blocks unfinished): no download wait outlives the kernel.  Then join.
    DG_CUDA(cudaMemsetAsync(ws + p->off_ddone, 0x7F, (size_t)(p->tp * p->tp) * 4, ms));
    DG_CUDA(cudaEventRecord(p->ev_down_done, p->down_st));
    DG_CUDA(cudaStreamWaitEvent(ms, p->ev_up_done, 0));
    DG_CUDA(cudaStreamWaitEvent(ms, p->ev_down_done, 0));
    if (!rc) rc = rc_down;
  }
  return rc;
}

// The launch (and, for AG FUSED, the shard transfers around it) of one run
// whose parameters are set.
int dispatch_run(dg_plan_s* p, const Driver& drv, const void* A, const void* B, const dg_bf16_t* C, void* D,
                 uint8_t* ws, cudaStream_t ms, cudaStream_t cs, bool rs_serial, bool pace, bool wait_up) {
  int rc = DG_OK;
  if (rs_serial) return run_rs_serial(p, drv, C, D, ws, ms);
  if (!is_ag(p->schedule) && p->tp > 1 && p->cep) {
    if (cs == ms || cs == nullptr)
      return fail(DG_ERR_ARG, "copy-engine hand-off needs a copy stream distinct from the main stream");
    return run_rs_ce(p, drv, ws, ms, cs);
  }
  if (is_ag(p->schedule) && p->tp > 1) {
    int mode = p->mode;
    if (mode == DG_MODE_FUSED && (cs == ms || cs == nullptr)) mode = DG_MODE_SERIAL;
    if (mode == DG_MODE_FUSED) {
      const int ns = p->copy_streams;
      rc = ensure_extra_streams(p, ns - 1);
      if (rc) return rc;
      cudaStream_t streams[8];
      streams[0] = cs;
      for (int i = 1; i < ns; ++i) streams[i] = p->extra[i - 1];
      DG_CUDA(cudaEventRecord(p->ev_fork, ms));
      for (int i = 0; i < ns; ++i) DG_CUDA(cudaStreamWaitEvent(streams[i], p->ev_fork, 0));
      // Transfers that wait on nothing the kernel does are enqueued before
      // it: every one without pacing, the first step's with it.  A layer
      // that serializes work in issue order (a profiler, CUDA_LAUNCH_BLOCKING)
      // then completes them before the kernel starts, instead of leaving the
      // kernel to wait for copies queued behind it.  Paced transfers wait on
      // the kernel's progress words, so they follow the launch.
      const int64_t P = p->tp;
      int64_t idx = 0;
      rc = enqueue_copies(p, drv, A, B, ws, streams, ns, pace, wait_up, 1, pace ? 1 : P - 1, &idx);
      if (rc) return rc;
      rc = launch(p, ms, 1);
      if (rc) return rc;
      if (pace) {
        rc = enqueue_copies(p, drv, A, B, ws, streams, ns, pace, wait_up, 2, P - 1, &idx);
        if (rc) return rc;
      }
      // Release every pacing wait still pending (a kernel that stopped early
      // never reaches the later steps): no copy-stream wait outlives the kernel.
      if (pace) DG_CUDA(cudaMemsetAsync(ws + p->off_status + kProgressOffset, 0x01, (size_t)p->tp * 4, ms));
      for (int i = 1; i < ns; ++i) {
        DG_CUDA(cudaEventRecord(p->extra_done[i - 1], streams[i]));
        DG_CUDA(cudaStreamWaitEvent(cs, p->extra_done[i - 1], 0));
      }
      DG_CUDA(cudaEventRecord(p->ev_join, cs));
      DG_CUDA(cudaStreamWaitEvent(ms, p->ev_join, 0));
    } else if (mode == DG_MODE_SERIAL) {
      int64_t idx = 0;
      rc = enqueue_copies(p, drv, A, B, ws, &ms, 1, false, wait_up, 1, p->tp - 1, &idx);
      if (rc) return rc;
      rc = launch(p, ms, 1);
      if (rc) return rc;
    } else {
      rc = launch(p, ms, 0);
      if (rc) return rc;
    }
  } else {
    rc = launch(p, ms, 0);
    if (rc) return rc;
  }
  return DG_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// No-allocation entry point.
//
// Some callers cannot allocate device memory where they run the GEMM (their
// host framework owns and budgets all of it, or they are a plug-in that must
// not grow the process's device footprint).  For them the workspace can live
// in this one file-scope device array instead.  Its size is fixed at build
// time, every GPU that loads this library holds it until the process exits,
// and all calls share it.
//
// In host code `dg_static_workspace` only names a host-side stand-in for the
// array, not a device address: its device address is looked up once per
// device with cudaGetSymbolAddress (with that device current) and then
// passed to the kernel like any caller workspace.
static __device__ __align__(256) unsigned char dg_static_workspace[DG_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxStaticDevices] = {};
}  // namespace


extern "C" {

const char* dg_last_error(void) { return g_err.c_str(); }

int dg_plan_scaled(dg_plan_t* out, int64_t m, int64_t n, int64_t k, int64_t l, int tp, int schedule,
                   float alpha, float beta, int a_type, int b_type, float scale_a, float scale_b) {
  if (!out) return fail(DG_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (m < 0 || n < 0 || k < 0 || l < 0) return fail(DG_ERR_ARG, "negative extent");
  if (tp != 1 && tp != 2 && tp != 4 && tp != 8) return fail(DG_ERR_ARG, "tp must be 1, 2, 4 or 8 (got %d)", tp);
  if (schedule < 0 || schedule > 3) return fail(DG_ERR_ARG, "unknown schedule %d", schedule);
  auto known = [](int t) { return t == DG_TYPE_BF16 || t == DG_TYPE_E4M3 || t == DG_TYPE_E5M2; };
  if (!known(a_type) || !known(b_type)) return fail(DG_ERR_ARG, "unknown input type (%d, %d)", a_type, b_type);
  if ((a_type == DG_TYPE_BF16) != (b_type == DG_TYPE_BF16))
    return fail(DG_ERR_UNSUPPORTED, "A and B must both be bf16 or both fp8");
  const int esz = a_type == DG_TYPE_BF16 ? 2 : 1;
  const int64_t kq = 16 / esz;  // K elements per 16 bytes (TMA row pitch and K-slab starts)
  if (k % kq || n % 8)
    return fail(DG_ERR_SHAPE, "K must be a multiple of %lld and N of 8 (K=%lld N=%lld)", (long long)kq,
                (long long)k, (long long)n);
  const bool rs = !is_ag(schedule);
  const bool need_m = schedule == DG_AG_ROTATING_A || schedule == DG_AG_ROTATING_B ||
                      schedule == DG_RS_TILING_A_ROTATING_C;
  const bool need_n = schedule != DG_RS_TILING_A_ROTATING_C;
  if (need_m && m % tp) return fail(DG_ERR_SHAPE, "M=%lld not divisible by tp=%d", (long long)m, tp);
  if (need_n && n % tp) return fail(DG_ERR_SHAPE, "N=%lld not divisible by tp=%d", (long long)n, tp);
  if (rs && k % tp) return fail(DG_ERR_SHAPE, "K=%lld not divisible by tp=%d", (long long)k, tp);
  if (rs && (k / tp) % kq)
    return fail(DG_ERR_SHAPE, "K/tp=%lld must be a multiple of %lld", (long long)(k / tp), (long long)kq);
  if (l * m > (int64_t(1) << 31) || l * n > (int64_t(1) << 31) || k > (int64_t(1) << 31))
    return fail(DG_ERR_SHAPE, "extent too large");
  auto* p = new dg_plan_s();
  p->m = m, p->n = n, p->k = k, p->l = l;
  p->tp = tp, p->schedule = schedule;
  p->alpha = alpha, p->beta = beta;
  p->a_type = a_type, p->b_type = b_type, p->esz = esz;
  p->scale_a = scale_a, p->scale_b = scale_b;
  // Staged epilogue by default for RS, for fp8 and for long K (where a tile's
  // mainloop is long and one fewer operand stage costs least); direct otherwise.
  // RS plans in which at least half the steps load a source chunk per tile
  // (the last step the partial, the first beta * C) take the per-warp staged
  // epilogue, whose loads run further ahead; with fewer such steps the
  // per-CTA one, whose larger boxes store the others' results faster.
  // AG plans with beta = 0 read no source at all: staging for the stores alone
  // leaves room for one more operand stage.  RS plans, whose middle steps add
  // by TMA reduction, load a source only at the last step and, with beta, the
  // first: with fewer than half the steps loading, two slots per warp and one
  // more operand stage where alpha * scale_a * scale_b is a power of two, the
  // per-CTA staging otherwise (measured faster on the fp8 plans, whose scales
  // rarely multiply to a power of two).
  const float a_eff = alpha * scale_a * scale_b;
  int a_exp = 0;
  const float a_fr = std::frexp(a_eff, &a_exp);
  const bool exact_red = a_eff == 0.f || a_fr == 0.5f || a_fr == -0.5f;
  const int loading = 1 + (beta != 0.f ? 1 : 0);
  if (is_ag(schedule) && beta == 0.f)
    p->epi = 3;
  else if (is_ag(schedule))
    p->epi = (esz == 1 || k >= 16384) ? 1 : 0;
  else if (loading * 2 >= tp)
    p->epi = 2;
  else
    p->epi = exact_red ? 4 : 1;
  // The RS epilogue streams the rotating partial (read once, written once per
  // step, far more bytes than L2 holds): with bf16 operands, evict it first,
  // so that the operand rows stay in L2 across the tiles that share them (fp8
  // operand tiles are half the bytes; there the policy measured slower).
  p->l2_hint = !is_ag(schedule) && esz == 2 ? 16u : 0u;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    p->id = g_next_plan_id++;
  }
  layout(p);
  *out = p;
  return DG_OK;
}

int dg_plan(dg_plan_t* out, int64_t m, int64_t n, int64_t k, int64_t l, int tp, int schedule,
            float alpha, float beta) {
  return dg_plan_scaled(out, m, n, k, l, tp, schedule, alpha, beta, DG_TYPE_BF16, DG_TYPE_BF16, 1.f, 1.f);
}

size_t dg_workspace_bytes(dg_plan_t p) {
  if (!p) return 0;
  if (p->mode == DG_MODE_SERIAL && !is_ag(p->schedule)) {
    p->serial_ws = true;
    return p->ws_bytes_serial;
  }
  return p->ws_bytes_base;
}

int dg_run_mode(dg_plan_t p, int mode) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  if (mode < DG_MODE_FUSED || mode > DG_MODE_SERIAL) return fail(DG_ERR_ARG, "unknown mode %d", mode);
  p->mode = mode;
  return DG_OK;
}

int dg_set_option(dg_plan_t p, int option, int64_t value) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  switch (option) {
    case DG_OPT_TIMEOUT_MS:
      if (value <= 0) return fail(DG_ERR_ARG, "timeout must be > 0");
      p->timeout_ms = value;
      return DG_OK;
    case DG_OPT_CHUNK_TILES:
      if (value < 0) return fail(DG_ERR_ARG, "chunk tiles must be >= 0");
      p->chunk_tiles_req = value;
      layout(p);
      return DG_OK;
    case DG_OPT_FAULT_SKIP_FLAG:
      p->fault_skip = value;
      return DG_OK;
    case DG_OPT_FAULT_DELAY_MS:
      if (value < 0) return fail(DG_ERR_ARG, "delay must be >= 0");
      p->fault_delay_ms = value;
      return DG_OK;
    case DG_OPT_GRID:
      if (value < 0) return fail(DG_ERR_ARG, "grid must be >= 0");
      p->grid_req = value;
      return DG_OK;
    case DG_OPT_COPY_STREAMS:
      if (value < 1 || value > 8) return fail(DG_ERR_ARG, "copy streams must be 1..8");
      p->copy_streams = (int)value;
      return DG_OK;
    case DG_OPT_RS_CE_PARTIALS:
      if (value != 0 && value != 1) return fail(DG_ERR_ARG, "RS copy-engine hand-off must be 0 or 1");
      if (p->epoch != 0) return fail(DG_ERR_STATE, "the hand-off is fixed after the first run");
      if (value == 1) {
        if (is_ag(p->schedule) || p->tp < 2)
          return fail(DG_ERR_UNSUPPORTED, "copy-engine hand-off is for RS plans with tp > 1");
        if (p->schedule == DG_RS_TILING_B_ROTATING_C && (p->n / p->tp) % 8)
          return fail(DG_ERR_UNSUPPORTED, "copy-engine hand-off needs N/tp %% 8 == 0");
        if (p->epi == 0) p->epi = 1;  // the hand-off runs through a staged epilogue
      }
      p->cep = value == 1;
      layout(p);
      return DG_OK;
    case DG_OPT_COPY_KIND:
      if (value < -1 || value > 2)
        return fail(DG_ERR_ARG,
                    "copy kind must be -1 (auto), 0 (copy engine), 1 (1D memcpy) or 2 (copy engine, tall copies)");
      p->copy_kind = (int)value;
      return DG_OK;
    case DG_OPT_MULTICAST:
      if (value < -1 || value > 1) return fail(DG_ERR_ARG, "multicast must be -1 (auto), 0 or 1");
      p->multicast = (int)value;
      return DG_OK;
    case DG_OPT_RS_REDUCE:
      if (value < -1 || value > 1) return fail(DG_ERR_ARG, "RS reduction must be -1 (auto), 0 or 1");
      if (p->epoch != 0) return fail(DG_ERR_STATE, "the RS reduction is fixed after the first run");
      if (value == 1) {
        if (is_ag(p->schedule)) return fail(DG_ERR_UNSUPPORTED, "the reduction is for the RS schedules");
        if (p->epi == 0) p->epi = 1;  // it runs in a staged epilogue
      }
      p->rs_reduce = (int)value;
      return DG_OK;
    case DG_OPT_GROUP_M:
      if (value < 0 || value > (1 << 20)) return fail(DG_ERR_ARG, "raster group must be 0 (auto) or positive");
      p->group_m_req = value;
      layout(p);
      return DG_OK;
    case DG_OPT_RS_CE_BANDS:
      if (value < 0 || value > (1 << 20)) return fail(DG_ERR_ARG, "bands per hand-off copy must be 0 (auto) or positive");
      p->ce_bands = value;
      return DG_OK;
    case DG_OPT_TILE_ORDER:
      if (value < -1 || value > 1) return fail(DG_ERR_ARG, "tile order must be -1 (auto), 0 or 1");
      if (value == 1 && !is_ag(p->schedule))
        return fail(DG_ERR_UNSUPPORTED, "the upload-frontier order is for the AllGather schedules");
      p->tile_order = (int)value;
      layout(p);
      return DG_OK;
    case DG_OPT_HOST_OVERLAP:
      if (value != 0 && value != 1) return fail(DG_ERR_ARG, "host overlap must be 0 or 1");
      p->host_overlap = (int)value;
      return DG_OK;
    case DG_OPT_COPY_PACE:
      if (value < -1 || value > 1) return fail(DG_ERR_ARG, "copy pacing must be -1 (auto), 0 or 1");
      p->copy_pace = (int)value;
      return DG_OK;
    case DG_OPT_WAVE_SYNC:
      if (value < -1 || value > 1) return fail(DG_ERR_ARG, "wave sync must be -1 (auto), 0 or 1");
      p->wave_sync = (int)value;
      return DG_OK;
    case DG_OPT_L2_HINT:
      if (value < 0 || value > 63 || (value & 3) == 3 || ((value >> 2) & 3) == 3 || ((value >> 4) & 3) == 3)
        return fail(DG_ERR_ARG, "L2 hint: three 2-bit fields (A, B, epilogue), each 0, 1 or 2");
      p->l2_hint = (uint32_t)value;
      return DG_OK;
    case DG_OPT_EPILOGUE:
      if (value < 0 || value > 4)
        return fail(DG_ERR_ARG,
                    "epilogue must be 0 (direct), 1 (staged), 2 (staged per warp), 3 (staged stores only) "
                    "or 4 (staged per warp, two slots)");
      if (p->epoch != 0) return fail(DG_ERR_STATE, "the epilogue is fixed after the first run");
      p->epi = (int)value;
      layout(p);
      return DG_OK;
    case DG_OPT_OUT_TYPE:
      if (value != DG_TYPE_BF16 && value != DG_TYPE_F32 && value != DG_TYPE_E4M3 && value != DG_TYPE_E5M2)
        return fail(DG_ERR_ARG, "output type must be DG_TYPE_BF16, DG_TYPE_F32, DG_TYPE_E4M3 or DG_TYPE_E5M2");
      p->out_type = (int)value;
      return DG_OK;
    case DG_OPT_REDUCE_OP:
      if (value != DG_REDUCE_SUM && value != DG_REDUCE_AVG)
        return fail(DG_ERR_ARG, "reduce op must be DG_REDUCE_SUM or DG_REDUCE_AVG");
      if (value == DG_REDUCE_AVG && is_ag(p->schedule))
        return fail(DG_ERR_UNSUPPORTED, "the reduce op applies to the RS schedules");
      p->reduce_op = (int)value;
      return DG_OK;
    case DG_OPT_CTA_GROUP:
      if (value != 1 && value != 2) return fail(DG_ERR_ARG, "CTA group must be 1 or 2");
      if (p->epoch != 0) return fail(DG_ERR_STATE, "the tile configuration is fixed after the first run");
      p->cg = (int)value;
      layout(p);
      return DG_OK;
    default:
      return fail(DG_ERR_ARG, "unknown option %d", option);
  }
}

int dg_plan_info_get(dg_plan_t p, dg_plan_info* o) {
  if (!p || !o) return fail(DG_ERR_ARG, "NULL argument");
  std::memset(o, 0, sizeof(*o));
  const dg::Geom& g = p->g;
  o->m = p->m, o->n = p->n, o->k = p->k, o->l = p->l;
  o->tp = p->tp, o->schedule = p->schedule;
  o->local_m = g.blk_m, o->local_n = g.blk_n, o->local_k = g.Ks;
  o->tile_m = g.BM, o->tile_n = g.BN, o->tile_k = g.BK;
  o->tiles_m = g.tiles_m, o->tiles_n = g.tiles_n;
  o->total_tiles = g.total_tiles;
  o->chunk_tiles = g.chunk_tiles, o->chunks_per_shard = g.nchunks;
  o->n_flags = p->n_flags;
  o->ws_bytes = dg_workspace_bytes(p);
  o->off_status = p->off_status, o->off_flags = p->off_flags, o->off_slots = p->off_slots;
  o->off_partial = p->off_partial, o->off_serial = p->off_serial;
  o->slot_bytes = p->slot_bytes;
  o->copies_per_run = p->copies;
  o->a_type = p->a_type, o->b_type = p->b_type, o->elem_bytes = p->esz;
  o->out_type = p->out_type, o->reduce_op = p->reduce_op;
  o->epilogue = p->epi, o->flag_parts = epi_parts(p);
  o->multicast = multicast_wanted(p) && multicast_ok(p, p->g) ? 1 : 0;
  return DG_OK;
}

int dg_plan_tile(dg_plan_t p, int64_t t, dg_tile* o) {
  if (!p || !o) return fail(DG_ERR_ARG, "NULL argument");
  if (t < 0 || t >= p->g.total_tiles) return fail(DG_ERR_ARG, "tile %lld out of range", (long long)t);
  const dg::Tile tl = dg::decode_tile(p->g, t);
  o->step = tl.s, o->rank = tl.r, o->slab = tl.j, o->batch = tl.l;
  o->a_map = tl.a_map, o->b_map = tl.b_map;
  o->a_row = tl.a_row, o->b_row = tl.b_row;
  o->out_row = tl.out_row, o->out_col = tl.out_col;
  o->rows_valid = tl.rows_valid, o->cols_valid = tl.cols_valid;
  o->k_blocks = tl.k_blocks;
  o->flag = tl.flag, o->tile_flag = tl.tile_flag;
  o->src = tl.src, o->dst = tl.dst;
  return DG_OK;
}

int dg_run(dg_plan_t p, const void* A, const void* B, const dg_bf16_t* C, dg_bf16_t* D,
           void* workspace, void* main_stream, void* copy_stream) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  if (p->out_type != DG_TYPE_BF16) return fail(DG_ERR_STATE, "the plan writes fp32 or fp8 D: run it with dg_run_ex");
  return dg_run_ex(p, A, B, C, nullptr, D, workspace, main_stream, copy_stream);
}

int dg_run_ex(dg_plan_t p, const void* A, const void* B, const dg_bf16_t* C, const dg_bf16_t* bias, void* D,
              void* workspace, void* main_stream, void* copy_stream) {
  return run_impl(p, A, B, C, bias, D, workspace, main_stream, copy_stream, nullptr);
}

int dg_run_host(dg_plan_t p, const void* A_host, const void* B_host, const dg_bf16_t* C_host, const dg_bf16_t* bias,
                void* D_host, void* A_dev, void* B_dev, dg_bf16_t* C_dev, void* D_dev, void* workspace,
                void* main_stream, void* copy_stream) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  if (p->g.total_tiles == 0) return DG_OK;  // empty output
  if (!A_host || !B_host || !D_host) return fail(DG_ERR_ARG, "A_host, B_host and D_host must be non-NULL");
  if (p->beta != 0.f && (!C_host || !C_dev)) return fail(DG_ERR_ARG, "C_host and C_dev are needed when beta != 0");
  if (!A_dev || !B_dev || !D_dev) return fail(DG_ERR_ARG, "A_dev, B_dev and D_dev must be non-NULL");
  auto ms = static_cast<cudaStream_t>(main_stream);
  const size_t a_bytes = (size_t)(p->l * p->m * p->k) * (size_t)p->esz;
  const size_t b_bytes = (size_t)(p->l * p->n * p->k) * (size_t)p->esz;
  const size_t c_bytes = (size_t)(p->l * p->m * p->n) * 2;
  const size_t d_elem = p->out_type == DG_TYPE_F32 ? 4 : (p->out_type == DG_TYPE_BF16 ? 2 : 1);
  const size_t d_bytes = (size_t)(p->l * p->m * p->n) * d_elem;
  const bool overlap = p->host_overlap && p->mode == DG_MODE_FUSED && pinned_host(A_host) && pinned_host(B_host) &&
                       pinned_host(D_host) && (p->beta == 0.f || pinned_host(C_host));
  if (overlap) {
    const HostIO io{A_host, B_host, C_host, D_host};
    return run_impl(p, A_dev, B_dev, p->beta != 0.f ? C_dev : nullptr, bias, D_dev, workspace, main_stream,
                    copy_stream, &io);
  }
  // sequential: host to device on the main stream, the run, device to host
  DG_CUDA(cudaMemcpyAsync(A_dev, A_host, a_bytes, cudaMemcpyHostToDevice, ms));
  DG_CUDA(cudaMemcpyAsync(B_dev, B_host, b_bytes, cudaMemcpyHostToDevice, ms));
  if (p->beta != 0.f) DG_CUDA(cudaMemcpyAsync(C_dev, C_host, c_bytes, cudaMemcpyHostToDevice, ms));
  int rc = dg_run_ex(p, A_dev, B_dev, p->beta != 0.f ? C_dev : nullptr, bias, D_dev, workspace, main_stream,
                     copy_stream);
  if (rc) return rc;
  DG_CUDA(cudaMemcpyAsync(D_host, D_dev, d_bytes, cudaMemcpyDeviceToHost, ms));
  return DG_OK;
}

int dg_set_result_scale(dg_plan_t p, float scale) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  if (!(scale == scale)) return fail(DG_ERR_ARG, "result scale is NaN");
  p->result_scale = scale;
  return DG_OK;
}

int dg_check(dg_plan_t p, void* workspace, void* stream) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (!workspace && p->static_dev >= 0) {
    // the last run used the built-in array (dg_run_static): its status word is there
    std::lock_guard<std::mutex> lk(g_static_mu);
    workspace = g_static_ptr[p->static_dev];
  }
  if (!workspace || p->epoch == 0) return DG_OK;
  unsigned long long st = 0;
  e = cudaMemcpy(&st, static_cast<uint8_t*>(workspace) + p->off_status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if ((uint32_t)(st >> 32) != p->epoch) return DG_OK;
  const uint32_t code = (uint32_t)(st >> 24) & 0xFF;
  const uint32_t info = (uint32_t)st & 0xFFFFFF;
  if (code == dg::DEV_TIMEOUT && (info & 0xF00000u) == dg::UP_FLAG_INFO)
    return fail(DG_ERR_TIMEOUT, "upload wait ran out (upload unit %u, run %u)", info & 0xFFu, p->epoch);
  if (code == dg::DEV_TIMEOUT)
    return fail(DG_ERR_TIMEOUT, "ready-flag wait ran out (flag %u, run %u)", info, p->epoch);
  if (code == dg::DEV_HANG)
    return fail(DG_ERR_HANG, "pipeline wait ran out (barrier 0x%06x, run %u)", info, p->epoch);
  return fail(DG_ERR_STATE, "unknown device status 0x%llx", st);
}

void dg_destroy(dg_plan_t p) {
  if (!p) return;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto it = g_ws_owner.begin(); it != g_ws_owner.end();)
      it = it->second == p->id ? g_ws_owner.erase(it) : std::next(it);
  }
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  for (int i = 0; i < p->n_extra; ++i) {
    cudaStreamDestroy(p->extra[i]);
    cudaEventDestroy(p->extra_done[i]);
  }
  if (p->io_rt) {
    cudaStreamDestroy(p->up_st);
    cudaStreamDestroy(p->down_st);
    cudaEventDestroy(p->ev_io);
    cudaEventDestroy(p->ev_up_done);
    cudaEventDestroy(p->ev_down_done);
    for (int i = 0; i < 8; ++i) cudaEventDestroy(p->ev_up[i]);
  }
  delete p;
}

}  // extern "C"

extern "C" int dg_run_static(dg_plan_t p, const dg_bf16_t* A, const dg_bf16_t* B, const dg_bf16_t* C,
                             dg_bf16_t* D, void* main_stream, void* copy_stream) {
  if (!p) return fail(DG_ERR_ARG, "plan is NULL");
  const size_t need = dg_workspace_bytes(p);
  if (need > DG_STATIC_WORKSPACE_BYTES)
    return fail(DG_ERR_SHAPE,
                "dg_run_static: plan needs %zu workspace bytes, the built-in array holds %zu; "
                "use dg_run with a caller workspace",
                need, (size_t)DG_STATIC_WORKSPACE_BYTES);
  if (p->g.total_tiles == 0) return DG_OK;
  // The array's address is per device: take the device the main stream runs
  // on, which must be the current one (the kernel launches there).
  int dev = 0;
  DG_CUDA(cudaGetDevice(&dev));
  int sdev = dev;
  DG_CUDA(cudaStreamGetDevice(static_cast<cudaStream_t>(main_stream), &sdev));
  if (sdev != dev)
    return fail(DG_ERR_ARG, "dg_run_static: the main stream belongs to device %d but device %d is current", sdev,
                dev);
  if (dev < 0 || dev >= kMaxStaticDevices) return fail(DG_ERR_UNSUPPORTED, "device index %d too large", dev);
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
      void* addr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&addr, dg_static_workspace);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(dg_static_workspace)");
      g_static_ptr[dev] = addr;
    }
    ws = g_static_ptr[dev];
  }
  // The flag and status words that must start at zero are cleared by dg_run
  // on the main stream whenever another plan used this array last.
  const int rc = dg_run(p, A, B, C, D, ws, main_stream, copy_stream);
  // dg_check(plan, NULL, stream) reads this run's status word from the array
  if (rc == DG_OK) p->static_dev = dev;
  return rc;
}
