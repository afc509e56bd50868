// dg_kernel.cuh -- persistent tcgen05 GEMM with shard-rotation tile order,
// flag-gated TMA producer and rotating-partial (RotatingC) epilogue, sm_103a.
//
// One CTA per SM, 192 threads; with CG = 2 the two CTAs of a pair share each
// 256 x 256 tile (the even CTA issues the MMAs for both SMs), and with
// multicast two pairs form a cluster of four that take vertically adjacent
// tiles, each CTA loading half of its B rows for both pairs:
//   warp 0      TMA producer: for each tile, waits (acquire, bounded) on the
//               ready flag of the shard chunk the tile reads (and, in runs that
//               upload their inputs, on the flag of the upload unit holding
//               them), then streams 128-byte K blocks (64 bf16 or 128 fp8
//               elements) of its 128 rows of A and its rows of B into a ring of
//               shared-memory stages (128-byte swizzle).
//   warp 1      MMA issuer (even CTA): 2 x 256 TMEM columns per CTA (two fp32
//               accumulators of 128 lanes x 256 columns), issues
//               tcgen05.mma.cta_group::{1,2}.kind::f16 (bf16) or kind::f8f6f4
//               (e4m3 / e5m2), four instructions per K block, and commits
//               stage-release and accumulator-full barriers (to both CTAs of a
//               pair).
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp owns the 32
//               TMEM lanes of its warp id mod 4), d = alpha*acc + source (+ the
//               bias), where the source is beta*C (AG, RS step 0), the rotating
//               fp32 partial (RS later steps) or nothing; writes D (bf16, fp32
//               or fp8) or the fp32 partial (in place, or into the rank's send
//               buffer for the copy-engine hand-off); counts finished D tiles
//               when the host downloads D block by block.
//
// Ordering across proxies:
//   copy engine -> shard data, then stream write of the ready flag;
//   producer: ld.acquire.gpu(flag) -> fence.proxy.async.global -> TMA loads.
//   RS epilogue: partial stores (or TMA reductions into it) complete ->
//   fence.proxy.async.global / fence (gpu) -> named barrier or warp sync ->
//   st.release.gpu(tile flag); the next step's epilogue acquires the flag
//   and reads the partial by TMA (or L1-bypassing loads).
//
// Every wait is bounded: flag waits by a timeout (on expiry the kernel records
// DG timeout in the workspace status word and carries on with whatever the
// buffer holds, so the pipeline drains normally); pipeline barrier waits by a
// longer limit, after which the kernel records a hang, stops issuing work,
// waits (bounded) for its own copies and MMAs in flight, frees its TMEM and
// exits.  Nothing traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dg_geom.h"

namespace dg {

constexpr int BK = 64;            // K elements per block for bf16 inputs (128 for fp8)
constexpr int KROW_BYTES = 128;   // bytes of one operand row per K block (the 128B swizzle span)
constexpr int MAX_MAPS = 9;  // RS: one K-slab map per rank (P <= 8); AG: home + slots
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int ROWS_PER_CTA = 128;  // accumulator rows (TMEM lanes) per CTA
constexpr int TILE_N = 256;        // accumulator columns
constexpr uint32_t TMEM_COLS = 2 * TILE_N;  // two accumulators

// Epilogue variants.
//   EPI = 0 (direct): each thread writes its accumulator row straight to
//           global memory (and reads its source row the same way).
//   EPI = 1 (staged): 32-column chunks of the source (beta*C or the fp32
//           rotating partial) are TMA-loaded into swizzled shared memory ahead
//           of use, and full destination chunks are staged in shared memory and
//           TMA-stored, so every global access is a coalesced bulk transfer.
//           Costs one operand stage of the ring (64 KB of staging).
constexpr int XCOLS = 32;                            // columns per epilogue chunk
constexpr uint32_t XBUF = ROWS_PER_CTA * XCOLS * 4;  // 16 KB: one fp32 chunk
//   EPI = 2 (per-warp staged): each epilogue warp moves its own 32 rows of a
//           chunk (32 x 32 boxes, 4 KB in fp32) through WSLOTS slots of its
//           own in shared memory: the source is TMA-loaded WPRE chunks ahead
//           into a slot, the result is written back into the same slot and
//           TMA-stored from it.  No barrier couples the four warps; the
//           rotating-partial hand-off is flagged per warp quarter of a tile.
constexpr int EPI_WARPS = 4;
constexpr int WROWS = ROWS_PER_CTA / EPI_WARPS;   // 32 rows per warp
constexpr uint32_t WBUF = WROWS * XCOLS * 4;      // 4 KB: one fp32 box
constexpr int WSLOTS = 4;                         // slots per warp (64 KB in all)
constexpr int WPRE = 3;                           // source loads issued ahead
//   EPI = 3 (staged stores): as 1 without source staging, for plans that
//           read no source; one more operand stage.
//   EPI = 4 (per-warp staged, two slots): as 2 with two slots per warp and one
//           load ahead, for RS plans whose middle steps load nothing (TMA
//           reductions); one more operand stage.

// Tile configuration per CTA group.
//   CG = 1: one SM, tile 128 x 256, tcgen05.mma.cta_group::1 (M=128, N=256).
//   CG = 2: an SM pair (cluster of 2), tile 256 x 256, tcgen05.mma.cta_group::2
//           (M=256, N=256) issued by the even CTA; each CTA stages its 128
//           rows of A and its 128 rows of B, and its TMEM holds its 128 rows.
template <int CG, int EPI = 0>
struct Cfg {
  static constexpr int TILE_M = 128 * CG;
  static constexpr int A_ROWS = 128;           // rows of A per CTA and stage
  static constexpr int B_ROWS = TILE_N / CG;   // rows of (N x K) B per CTA and stage
  static constexpr uint32_t A_BYTES = A_ROWS * KROW_BYTES;
  static constexpr uint32_t B_BYTES = B_ROWS * KROW_BYTES;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  // EPI = 3 (staged stores only): the staged epilogue without its source
  // chunks (plans that read no source: AG with beta = 0), which gives their
  // 32 KB back to the operand ring.
  // EPI = 4: the per-warp epilogue with two slots per warp (one load ahead),
  // which also leaves room for one more operand stage.
  static constexpr bool SRC_STAGING = EPI == 1 || EPI == 2;
  static constexpr int STAGES = CG == 1 ? (SRC_STAGING ? 3 : 4) : (SRC_STAGING ? 5 : 6);
  static constexpr uint32_t STAGING_BYTES =
      SRC_STAGING ? 4 * XBUF : (EPI == 3 || EPI == 4 ? 2 * XBUF : 0);  // [2 source +] 2 destination chunks
  static constexpr int WSL = EPI == 4 ? 2 : WSLOTS;  // per-warp slots in use
  static constexpr int WPR = WSL - 1;                // per-warp source loads ahead
  static constexpr uint32_t SMEM_BYTES =
      STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 512 /*barriers*/;
};

// Device status word: (epoch << 32) | (code << 24) | (info & 0xffffff).
constexpr uint32_t DEV_TIMEOUT = 1;  // a ready-flag wait ran out
constexpr uint32_t UP_FLAG_INFO = 0x600000u;  // status info of an upload-flag wait: | upload unit
constexpr uint32_t DEV_HANG = 2;     // a pipeline wait ran out

struct KParams {
  CUtensorMap tmA[MAX_MAPS];
  CUtensorMap tmB[MAX_MAPS];
  // staged epilogue: fp32 partial (box 32 x 128, 128B swizzle), bf16 C
  // (box 32 x 128, 64B swizzle), D in its output type (bf16 like C, fp32 like
  // the partial)
  CUtensorMap tmX, tmC, tmD;
  // RS with copy-engine hand-off: rank send buffers and (double-buffered)
  // receive buffers, fp32, slab-local rows and columns
  CUtensorMap tmS, tmR;
  uint32_t* done;       // per (rank, step, batch, band): half-tiles written to the send buffer
  float* S;             // send buffers (plain-store address of tmS)
  const float* R;       // receive buffers (plain-load address of tmR)
  Geom g;
  const __nv_bfloat16* C;
  void* D;                    // bf16, fp32 when out_f32, fp8 when out_fp8
  const __nv_bfloat16* bias;  // per-column bias (N values), or null
  float* X;
  uint32_t* flags;  // AG chunk flags or RS tile flags
  unsigned long long* status;
  uint32_t epoch;
  uint32_t wait_flags;  // AG: 1 = wait on chunk flags
  int32_t n_maps;       // tensor maps in use (each of tmA / tmB)
  uint32_t idesc;       // tcgen05 instruction descriptor (operand formats, M, N)
  uint32_t l2_hint;     // L2 policies: bits 0-1 A loads, bits 2-3 B loads, bits 4-5 the
                        // epilogue's TMA traffic (source loads, partial / D stores and
                        // reductions); each 0 none, 1 evict-first, 2 evict-last
  uint32_t wave_sync;   // producers start tile i only after every CTA issued tile i-1
  uint32_t* wave_ctr;   // per-run counter of tiles whose loads are issued (zeroed per run)
  uint32_t* progress;   // AG copy pacing: progress[s] set to 1 once a producer reaches step s, or null
  uint32_t rs_reduce;   // staged epilogues, in-place RS: middle steps add into the partial by TMA reduction
  uint32_t mc;          // CTA pairs in clusters of four: the two pairs take tiles 2i and 2i + 1, which
                        // share their B rows, and each CTA loads half of its B rows for both pairs
                        // (multicast); B maps then have 64-row boxes
  // Runs that upload their inputs and download D themselves (host buffers):
  // the inputs of a tile are on the device once up_flags[upload_unit(tile)]
  // >= epoch, and d_done[s * P + r] counts the half tiles of D finished for
  // step s, rank r.  Both null otherwise.
  const uint32_t* up_flags;
  uint32_t* d_done;
  float alpha, beta;
  float bias_scale;  // weight of the bias in every epilogue pass (1, or 1/P for the mean)
  uint32_t out_f32;  // D is fp32
  uint32_t out_fp8;  // D is fp8: 1 e4m3, 2 e5m2 (result_scale * value, nearest, saturating)
  float result_scale;
  uint64_t timeout_ns;
  uint64_t hang_ns;
};
static_assert(sizeof(KParams) <= 4096, "kernel parameters must fit the 4 KB parameter space");

// ------------------------------------------------------------------ PTX glue

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Count `bytes` of the barrier's current phase as arrived without a transfer
// (for a load that will never be issued).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait for the phase of parity `parity` of a barrier, with no status
// report (exit paths: wait for transfers in flight to land).
__device__ __forceinline__ void mbar_settle(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < 200000000ull) {
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Same loads with an L2 eviction policy (from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy(uint32_t kind) {
  uint64_t pol = 0;
  if (kind == 1)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Generic-proxy writes to shared memory made visible to a following TMA store.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The epilogue's L2 policy: `use` false leaves the default policy.
struct EpiPolicy {
  uint64_t pol;
  bool use;
};
__device__ __forceinline__ EpiPolicy epi_policy(const KParams& p) {
  const uint32_t kind = (p.l2_hint >> 4) & 3u;
  return EpiPolicy{kind ? l2_policy(kind) : 0ull, kind != 0};
}
// An epilogue TMA load (source chunk into shared memory) under that policy.
__device__ __forceinline__ void tma_load_2d_epi(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                int32_t y, EpiPolicy ep) {
  if (ep.use)
    tma_load_2d_hint(dst, map, bar, x, y, ep.pol);
  else
    tma_load_2d(dst, map, bar, x, y);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y,
                                             EpiPolicy ep) {
  if (ep.use)
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "l"(ep.pol)
                 : "memory");
  else
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
// Element-wise add of a shared-memory box into global memory (the reduction
// is performed at the L2; the map's element type, fp32 here, sets the add).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y,
                                                  EpiPolicy ep) {
  if (ep.use)
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "l"(ep.pol)
        : "memory");
  else
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk stores still read their shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N committed bulk stores are still incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset inside a 1024-byte-aligned tile written by TMA with the
// 128-byte (64-byte) swizzle: 16-byte unit bits [4,7) ([4,6)) XOR bits
// [7,10) ([7,9)) of the linear offset.
__device__ __forceinline__ uint32_t sw128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }
__device__ __forceinline__ uint32_t sw64(uint32_t off) { return off ^ (((off >> 7) & 3u) << 4); }

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// tcgen05 ---------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// CTA-pair (cta_group::2) forms -------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (here: the even CTA's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map,
                                                      uint32_t bar_cluster, int32_t x, int32_t y,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}
// The same load multicast to every CTA of `mask` (the same shared-memory
// offset in each); each destination's bytes are counted on the barrier at
// mbar's offset in that destination's even (MMA-issuing) CTA.
__device__ __forceinline__ void tma_load_2d_pair_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                    int32_t x, int32_t y, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on the mbarrier at this offset in every CTA of `mask` when
// the pair's earlier tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// fp8 operands (e4m3 / e5m2, formats in the instruction descriptor), fp32
// accumulator; one instruction covers K = 32 (32 bytes of each operand row).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread i of the warp gets lane (base+i),
// columns col..col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 64 bf16 (128 bytes) stored with the 128-byte swizzle, 8-row groups 1024
// bytes apart (the layout a TMA load with SWIZZLE_128B writes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                     // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator (bits 4-5 = 1), A format at bits
// 7-9 and B format at bits 10-12 (kind::f16: bf16 = 1; kind::f8f6f4:
// e4m3 = 0, e5m2 = 1), both operands K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f32acc(int m, int n, uint32_t a_fmt, uint32_t b_fmt) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) { return idesc_f32acc(m, n, 1, 1); }

// ---------------------------------------------------------------- status

__device__ __forceinline__ bool status_set(const KParams& p) {
  return (uint32_t)(ld_relaxed_u64(p.status) >> 32) == p.epoch;
}
__device__ __forceinline__ bool status_hang(const KParams& p) {
  unsigned long long v = ld_relaxed_u64(p.status);
  return (uint32_t)(v >> 32) == p.epoch && ((uint32_t)(v >> 24) & 0xFF) == DEV_HANG;
}
// First error of this epoch wins.
__device__ __noinline__ void status_record(const KParams& p, uint32_t code, uint32_t info) {
  unsigned long long want =
      ((unsigned long long)p.epoch << 32) | ((unsigned long long)(code & 0xFF) << 24) | (info & 0xFFFFFF);
  unsigned long long old = ld_relaxed_u64(p.status);
  while ((uint32_t)(old >> 32) != p.epoch) {
    unsigned long long seen = atomicCAS(p.status, old, want);
    if (seen == old) break;
    old = seen;
  }
}

// Wait until *f >= target.  false if it ran out (status recorded) or an
// earlier error of this run is already recorded (then it does not wait).
__device__ __noinline__ bool wait_flag_geq(const KParams& p, const uint32_t* f, uint32_t target,
                                           uint32_t info) {
  if (ld_acquire_u32(f) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (ld_acquire_u32(f) >= target) return true;
    if ((n & 31) == 0) {
      if (status_set(p)) return false;
      if (globaltimer() - t0 > p.timeout_ns) {
        status_record(p, DEV_TIMEOUT, info);
        return false;
      }
    }
    __nanosleep(128);
  }
}

// Bounded mbarrier wait.  false: this or another CTA ran out (hang recorded).
__device__ __forceinline__ bool mbar_wait(const KParams& p, uint32_t bar, uint32_t parity,
                                          uint32_t info) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255) == 0) {
      if (t0 == 0) t0 = globaltimer();
      if (status_hang(p)) return false;
      if (globaltimer() - t0 > p.hang_ns) {
        status_record(p, DEV_HANG, info);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------- epilogue math

struct alignas(16) F4 {
  float x, y, z, w;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// out += bias_scale * bias[gcol + i] for the ncols valid columns (the bias is
// shared by every row; all threads of the warp read the same bytes).
__device__ __forceinline__ void add_bias(const KParams& p, int64_t gcol, int ncols, float (&out)[32]) {
  const __nv_bfloat16* b = p.bias + gcol;
  if (ncols == 32 && (gcol & 7) == 0) {
    const uint4* b4 = reinterpret_cast<const uint4*>(b);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(b4 + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        out[q * 8 + 2 * h] = fmaf(p.bias_scale, bf16_bits_to_f32(w[h] & 0xFFFFu), out[q * 8 + 2 * h]);
        out[q * 8 + 2 * h + 1] = fmaf(p.bias_scale, bf16_bits_to_f32(w[h] >> 16), out[q * 8 + 2 * h + 1]);
      }
    }
  } else {
    const uint16_t* bs = reinterpret_cast<const uint16_t*>(b);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) out[i] = fmaf(p.bias_scale, bf16_bits_to_f32(__ldg(bs + i)), out[i]);
  }
}

// 32 consecutive results as fp8 bytes (result_scale applied, round to nearest
// even, saturating at the largest finite value), the ncols valid ones.
__device__ __forceinline__ void store_fp8_row(const KParams& p, uint8_t* d, int ncols, const float (&out)[32],
                                              bool vec) {
  const __nv_fp8_interpretation_t fmt = p.out_fp8 == 1 ? __NV_E4M3 : __NV_E5M2;
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(out[4 * q] * p.result_scale, out[4 * q + 1] * p.result_scale), __NV_SATFINITE, fmt);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(out[4 * q + 2] * p.result_scale, out[4 * q + 3] * p.result_scale), __NV_SATFINITE, fmt);
    w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  if (vec) {
    reinterpret_cast<uint4*>(d)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(d)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) d[i] = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
  }
}

// Plain stores of 32 consecutive fp32 values (the ncols valid ones).
__device__ __forceinline__ void store_f32_row(float* x, int ncols, const float (&out)[32], bool vec) {
  if (vec) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      __stcg(reinterpret_cast<float4*>(x) + q, make_float4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) __stcg(x + i, out[i]);
  }
}

// Source term (beta*C, the fp32 partial, or 0) for 32 consecutive columns of
// one output row, then d = alpha*acc + src (+ the bias), stored as D (bf16 or
// fp32) or as the fp32 partial.
// xsrc / xdst: where this row's 32 partial values are read / written (the
// shared partial X, or with the copy-engine hand-off the rank's receive and
// send buffers).
__device__ __forceinline__ void epilogue_row_chunk(const KParams& p, const Tile& tl, int64_t grow,
                                                   int64_t gcol, int ncols, float (&acc)[32], const float* xsrc,
                                                   float* xdst) {
  const int64_t N = p.g.N;
  const int64_t e0 = grow * N + gcol;  // element offset in C / D / X
  float src[32];
  if (tl.src == SRC_C) {
    const __nv_bfloat16* c = p.C + e0;
    if (ncols == 32 && (e0 & 7) == 0) {
      const uint4* c4 = reinterpret_cast<const uint4*>(c);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v = __ldg(c4 + q);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          src[q * 8 + 2 * h] = p.beta * bf16_bits_to_f32(w[h] & 0xFFFFu);
          src[q * 8 + 2 * h + 1] = p.beta * bf16_bits_to_f32(w[h] >> 16);
        }
      }
    } else {
      const uint16_t* cs = reinterpret_cast<const uint16_t*>(c);
#pragma unroll
      for (int i = 0; i < 32; ++i) src[i] = i < ncols ? p.beta * bf16_bits_to_f32(cs[i]) : 0.f;
    }
  } else if (tl.src == SRC_X) {
    const float* x = xsrc;
    if (ncols == 32 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v = __ldcg(reinterpret_cast<const float4*>(x) + q);
        src[4 * q] = v.x;
        src[4 * q + 1] = v.y;
        src[4 * q + 2] = v.z;
        src[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) src[i] = i < ncols ? __ldcg(x + i) : 0.f;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) src[i] = 0.f;
  }
  float out[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = fmaf(p.alpha, acc[i], src[i]);
  if (p.bias) add_bias(p, gcol, ncols, out);

  if (tl.dst == DST_D && p.out_fp8) {
    store_fp8_row(p, static_cast<uint8_t*>(p.D) + e0, ncols, out, ncols == 32 && (e0 & 15) == 0);
  } else if (tl.dst == DST_D && p.out_f32) {
    store_f32_row(static_cast<float*>(p.D) + e0, ncols, out, ncols == 32 && (e0 & 3) == 0);
  } else if (tl.dst == DST_D) {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.D) + e0;
    if (ncols == 32 && (e0 & 7) == 0) {
      uint4* d4 = reinterpret_cast<uint4*>(d);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16x2(out[8 * q + 0], out[8 * q + 1]);
        v.y = pack_bf16x2(out[8 * q + 2], out[8 * q + 3]);
        v.z = pack_bf16x2(out[8 * q + 4], out[8 * q + 5]);
        v.w = pack_bf16x2(out[8 * q + 6], out[8 * q + 7]);
        d4[q] = v;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncols) d[i] = __float2bfloat16_rn(out[i]);
    }
  } else {
    store_f32_row(xdst, ncols, out, ncols == 32 && (reinterpret_cast<uintptr_t>(xdst) & 15) == 0);
  }
}

// Masked direct store of 32 consecutive results of one output row (D at
// (grow, gcol); the partial at `x`).
__device__ __forceinline__ void store_row_chunk(const KParams& p, const Tile& tl, int64_t grow,
                                                int64_t gcol, int ncols, const float (&out)[32], float* x) {
  if (tl.dst == DST_D && p.out_fp8) {
    store_fp8_row(p, static_cast<uint8_t*>(p.D) + grow * p.g.N + gcol, ncols, out, false);
  } else if (tl.dst == DST_D && p.out_f32) {
    store_f32_row(static_cast<float*>(p.D) + grow * p.g.N + gcol, ncols, out, false);
  } else if (tl.dst == DST_D) {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.D) + grow * p.g.N + gcol;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) d[i] = __float2bfloat16_rn(out[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) __stcg(x + i, out[i]);
  }
}

// Row `row` (32 values) of a staged source chunk: fp32 with the 128-byte
// swizzle (the rotating partial) or bf16 with the 64-byte swizzle (C, scaled
// by beta).
__device__ __forceinline__ void staged_read_row(const uint8_t* buf, int row, bool f32, float beta,
                                                float (&src)[32]) {
  if (f32) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = *reinterpret_cast<const float4*>(buf + sw128((uint32_t)row * 128u + j * 16u));
      src[4 * j] = v.x;
      src[4 * j + 1] = v.y;
      src[4 * j + 2] = v.z;
      src[4 * j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(buf + sw64((uint32_t)row * 64u + j * 16u));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        src[8 * j + 2 * h] = beta * bf16_bits_to_f32(w[h] & 0xFFFFu);
        src[8 * j + 2 * h + 1] = beta * bf16_bits_to_f32(w[h] >> 16);
      }
    }
  }
}

// Row `row` of a staged destination chunk, in the layout its TMA store reads.
__device__ __forceinline__ void staged_write_row(uint8_t* buf, int row, bool f32, const float (&out)[32]) {
  if (f32) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(buf + sw128((uint32_t)row * 128u + j * 16u)) =
          make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 v;
      v.x = pack_bf16x2(out[8 * j + 0], out[8 * j + 1]);
      v.y = pack_bf16x2(out[8 * j + 2], out[8 * j + 3]);
      v.z = pack_bf16x2(out[8 * j + 4], out[8 * j + 5]);
      v.w = pack_bf16x2(out[8 * j + 6], out[8 * j + 7]);
      *reinterpret_cast<uint4*>(buf + sw64((uint32_t)row * 64u + j * 16u)) = v;
    }
  }
}

// Hand a rotating-partial half tile to the next step: the bulk stores that
// wrote it (all issued by this thread) complete, then the flag is released.
__device__ __forceinline__ void release_partial(const KParams& p, int64_t flag, uint32_t val) {
  bulk_wait<0>();
  fence_proxy_async_global();
  __threadfence();
  st_release_u32(p.flags + flag, val);
}

// TMA load of source chunk c of a tile half into staging buffer (idx & 1):
// the rotating partial (fp32, map `xmap` at column x_col0 / row x_row0) or
// beta*C (bf16, at the tile's output position).
__device__ __forceinline__ void staged_load_src(const KParams& p, const Tile& tl, int64_t row0, int c,
                                                uint32_t idx, uint32_t sbase, uint32_t bar_xfull,
                                                const CUtensorMap* xmap, int64_t x_col0, int64_t x_row0,
                                                EpiPolicy ep) {
  const uint32_t sb = idx & 1;
  const bool f32 = tl.src == SRC_X;
  mbar_arrive_expect_tx(bar_xfull + 8 * sb, f32 ? XBUF : XBUF / 2);
  if (f32)
    tma_load_2d_epi(sbase + sb * XBUF, xmap, bar_xfull + 8 * sb, (int32_t)(x_col0 + c * XCOLS), (int32_t)x_row0,
                    ep);
  else
    tma_load_2d_epi(sbase + sb * XBUF, &p.tmC, bar_xfull + 8 * sb, (int32_t)(tl.out_col + c * XCOLS),
                    (int32_t)row0, ep);
}

// Upload units whose flags a tile's inputs wait on (runs with host buffers).
// AG: unit f holds rank f's home shards and C's row band M_f (the C of
// AG-RotatingB's rank f; AG-RotatingA's tile (r, j) reads C[M_j, N_r]).  RS:
// unit f holds the row slab (f + 1) mod P of the sliced operand and of C
// (unit 0 also what every tile reads whole); tile (s, r) works on slab
// (r + s + 1) mod P.
__device__ __forceinline__ int32_t upload_unit(const Geom& g, const Tile& tl) {
  return (g.sched == SCHED_AG_A || g.sched == SCHED_AG_B) ? tl.r : (tl.r + tl.s) % g.P;
}
__device__ __forceinline__ int32_t upload_unit_c(const Geom& g, const Tile& tl) {
  return g.sched == SCHED_AG_A ? tl.j : upload_unit(g, tl);
}

// ------------------------------------------------------------------ kernel

template <int CG, int EPI, int F8>
__global__ void __launch_bounds__(NUM_THREADS, 1) dg_gemm_kernel(const __grid_constant__ KParams p) {
  using C = Cfg<CG, EPI>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // staged epilogue: source chunks [2] then destination chunks [2], 1024-aligned
  // (stores-only staging: destination chunks alone)
  uint8_t* xsrc = smem + STAGES * C::STAGE_BYTES;
  uint8_t* xdst = EPI == 3 ? xsrc : xsrc + 2 * XBUF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::STAGING_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, xfull[2], wfull[16]
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = smem_u32(bars + STAGES);
  const uint32_t bar_tfull = smem_u32(bars + 2 * STAGES);
  const uint32_t bar_tempty = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t bar_drain = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t bar_xfull = smem_u32(bars + 2 * STAGES + 5);
  const uint32_t bar_wfull = smem_u32(bars + 2 * STAGES + 7);  // [EPI_WARPS * WSLOTS] (EPI = 2)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 7 + EPI_WARPS * WSLOTS);
  volatile uint32_t* s_go = s_tmem + 1;  // [2] epilogue go/abort, by tile parity
  // [4] K-block loads each CTA of the cluster issued (kept in the even CTAs'
  // shared memory, for the exit: every load must land before its CTA exits)
  volatile uint32_t* s_kcnt = s_tmem + 3;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA rank in the cluster; `half`: which half of the pair's tile this CTA
  // holds (0 for CG = 1); the even CTA of a pair (`lead`) issues the MMAs.
  // With multicast (clusters of four) pair `pq` of the cluster takes tile
  // 2i + pq of the cluster's slot i.
  const uint32_t crank = CG == 2 ? cluster_ctarank() : 0u;
  const uint32_t half = crank & 1u;
  const uint32_t lead = crank & ~1u;
  const bool leader = half == 0;
  const bool mc = CG == 2 && p.mc != 0;
  const uint32_t pq = mc ? (crank >> 1) : 0u;
  const int64_t unit = mc ? (int64_t)(blockIdx.x >> 2) : CG == 2 ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
  const int64_t nunits = mc ? (int64_t)(gridDim.x >> 2) : CG == 2 ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, mc ? 2 : 1);  // with multicast both pairs free a stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_tfull + 8 * i, 1);
      mbar_init(bar_tempty + 8 * i, 4 * CG);  // one arrival per epilogue warp of the pair
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_xfull, 1);
    mbar_init(bar_xfull + 8, 1);
    for (int i = 0; i < EPI_WARPS * WSLOTS; ++i) mbar_init(bar_wfull + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if (CG == 2) {
      tmem_alloc_pair(smem_u32(s_tmem), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(s_tmem), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncwarp();
  if (CG == 2)
    cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  const int64_t T = p.g.total_tiles;
  const int64_t TI = mc ? T / 2 : T;  // tile slots (the host allows multicast only for even T)
  const uint32_t smem_base = smem_u32(smem);
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      for (int i = 0; i < p.n_maps; ++i) {
        prefetch_tmap(&p.tmA[i]);
        prefetch_tmap(&p.tmB[i]);
      }
      const int32_t kblk = p.g.BK;  // K elements per block: 128 bytes of a row
      const uint32_t hint_a = p.l2_hint & 3u, hint_b = (p.l2_hint >> 2) & 3u;
      const uint64_t pol_a = hint_a ? l2_policy(hint_a) : 0, pol_b = hint_b ? l2_policy(hint_b) : 0;
      uint32_t stage = 0, phase = 0;
      uint32_t nloads = 0;  // K-block loads issued: load n goes to stage n % STAGES, phase n / STAGES
      bool ok = true;
      uint32_t wave = 0;
      int32_t step_seen = -1;
      uint32_t up_ok = 0;  // ranks whose uploaded inputs this producer has seen
      for (int64_t i = unit; i < TI && ok; i += nunits, ++wave) {
        const int64_t t = mc ? 2 * i + pq : i;
        const Tile tl = decode_tile(p.g, t);
        if (p.progress && tl.s != step_seen) {
          // the copies of step s + 1 may start now (paced shard transfers);
          // set before any wait of this step, so it never depends on them
          step_seen = tl.s;
          st_relaxed_u32(p.progress + tl.s, 1u);
        }
        if (p.wave_sync && wave > 0) {
          // keep the CTAs in phase so that tiles sharing an operand strip read
          // it while it is still in L2 (a timing gate only: no data depends on it)
          const uint32_t want = wave * gridDim.x;
          const uint64_t t0 = globaltimer();
          while (ld_relaxed_u32(p.wave_ctr) < want) {
            if (globaltimer() - t0 > p.timeout_ns) break;
            __nanosleep(64);
          }
        }
        if (p.up_flags) {
          const int32_t uu = upload_unit(p.g, tl);
          if (!((up_ok >> uu) & 1u)) {
            // this tile's operands have been uploaded from the host
            wait_flag_geq(p, p.up_flags + uu, p.epoch, UP_FLAG_INFO | (uint32_t)uu);
            fence_proxy_async_global();
            up_ok |= 1u << uu;
          }
        }
        if (tl.flag >= 0 && p.wait_flags) {
          wait_flag_geq(p, p.flags + tl.flag, p.epoch, (uint32_t)tl.flag);
          fence_proxy_async_global();
        }
        const CUtensorMap* ma = &p.tmA[tl.a_map];
        const CUtensorMap* mb = &p.tmB[tl.b_map];
        const int32_t a_row = (int32_t)(tl.a_row + (int64_t)half * C::A_ROWS);
        const int32_t b_row = (int32_t)(tl.b_row + (int64_t)half * C::B_ROWS);
        for (int kb = 0; kb < tl.k_blocks; ++kb) {
          if (!mbar_wait(p, bar_empty + 8 * stage, phase ^ 1, 0x100000u | stage)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
          if (CG == 2) {
            const uint32_t fb_lead = mapa_shared(fb, lead);
            if (leader) mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);  // both CTAs' bytes
            if (hint_a)
              tma_load_2d_pair_hint(sa, ma, fb_lead, kb * kblk, a_row, pol_a);
            else
              tma_load_2d_pair(sa, ma, fb_lead, kb * kblk, a_row);
            if (mc)  // this pair's half of the CTA's B rows, for this CTA and its counterpart
              tma_load_2d_pair_mc(sa + C::A_BYTES + pq * (C::B_BYTES / 2), mb, fb_lead, kb * kblk,
                                  b_row + (int32_t)(pq * (C::B_ROWS / 2)),
                                  (uint16_t)((1u << crank) | (1u << (crank ^ 2u))));
            else if (hint_b)
              tma_load_2d_pair_hint(sa + C::A_BYTES, mb, fb_lead, kb * kblk, b_row, pol_b);
            else
              tma_load_2d_pair(sa + C::A_BYTES, mb, fb_lead, kb * kblk, b_row);
          } else {
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            if (hint_a)
              tma_load_2d_hint(sa, ma, fb, kb * kblk, a_row, pol_a);
            else
              tma_load_2d(sa, ma, fb, kb * kblk, a_row);
            if (hint_b)
              tma_load_2d_hint(sa + C::A_BYTES, mb, fb, kb * kblk, b_row, pol_b);
            else
              tma_load_2d(sa + C::A_BYTES, mb, fb, kb * kblk, b_row);
          }
          ++nloads;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (p.wave_sync) atomicAdd(p.wave_ctr, 1u);
      }
      if (!ok) aborted = true;
      if (CG == 1) {
        // every load issued must land before the CTA exits: the last phase of
        // each stage (phases of a stage complete in order)
        if (!ok)
          for (uint32_t n = nloads > (uint32_t)STAGES ? nloads - STAGES : 0u; n < nloads; ++n)
            mbar_settle(bar_full + 8 * (n % STAGES), (n / STAGES) & 1u);
      } else {
        // the loads landing in a pair are counted on its even CTA's barriers:
        // hand this CTA's count to the even CTA(s) its loads land in (they
        // wait for them before any CTA exits)
        st_shared_cluster_u32(mapa_shared(smem_u32((const void*)(s_kcnt + crank)), lead), nloads);
        if (mc) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)(s_kcnt + crank)), lead ^ 2u), nloads);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // --------------------------------------------------------------- MMA
      const uint32_t IDESC = p.idesc;
      uint32_t stage = 0, phase = 0, it = 0;
      bool ok = true;
      for (int64_t i = unit; i < TI && ok; i += nunits, ++it) {
        const int64_t t = mc ? 2 * i + pq : i;
        const Tile tl = decode_tile(p.g, t);
        const uint32_t buf = it & 1, use = it >> 1;
        if (!mbar_wait(p, bar_tempty + 8 * buf, (use & 1) ^ 1, 0x200000u | buf)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * TILE_N;
        for (int kb = 0; kb < tl.k_blocks; ++kb) {
          if (!mbar_wait(p, bar_full + 8 * stage, phase, 0x300000u | stage)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + C::A_BYTES);
#pragma unroll
          for (int kk = 0; kk < KROW_BYTES / 32; ++kk) {
            // +32 bytes per instruction inside the swizzled 128-byte row
            // (K = 16 bf16 or K = 32 fp8)
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            const uint64_t ad = da + (uint64_t)(2 * kk), bd = db + (uint64_t)(2 * kk);
            if (F8) {
              if (CG == 2)
                tc_mma_f8_pair(d_tmem, ad, bd, IDESC, acc);
              else
                tc_mma_f8(d_tmem, ad, bd, IDESC, acc);
            } else {
              if (CG == 2)
                tc_mma_bf16_pair(d_tmem, ad, bd, IDESC, acc);
              else
                tc_mma_bf16(d_tmem, ad, bd, IDESC, acc);
            }
          }
          if (CG == 2)  // the stage is free in both CTAs of the pair (of both pairs, with multicast)
            tc_commit_pair_mc(bar_empty + 8 * stage, mc ? (uint16_t)0xF : (uint16_t)(0x3u << lead));
          else
            tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if (CG == 2)
          tc_commit_pair_mc(bar_tfull + 8 * buf, (uint16_t)(0x3u << lead));
        else
          tc_commit(bar_tfull + 8 * buf);
      }
      if (!ok) {
        aborted = true;
        if (CG == 2)
          tc_commit_pair_mc(bar_drain, (uint16_t)(0x1u << lead));
        else
          tc_commit(bar_drain);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar_drain, 0) && globaltimer() - t0 < 200000000ull) {
        }
      }
    }
  } else if constexpr (EPI == 2 || EPI == 4) {
    // ------------------------------------------------- epilogue, per warp
    // Warp q owns TMEM lanes 32q..32q+31 (rows of the CTA's half tile).  Lane
    // 0 issues this warp's TMA loads and stores and its flag operations; the
    // chunk slots, their load barriers and the bulk groups are the warp's own.
    const int q = warp & 3;
    uint8_t* wb = xsrc + (uint32_t)q * (C::WSL * WBUF);
    const uint32_t wb_addr = smem_u32(wb);
    const uint32_t wbar = bar_wfull + 8u * (uint32_t)(C::WSL * q);
    uint32_t seq = 0;       // chunks of staged tiles so far: chunk g uses slot g % WSL and
                            // commits bulk group g (lane 0), so a slot's last store is a group index
    uint32_t ph = 0;        // per slot: parity of its next load completion
    uint32_t inflight = 0;  // slots whose load is issued and not yet consumed
    int64_t pend_flag = -1;  // quarter-tile flag whose release waits for this warp's bulk stores
    uint32_t pend_val = 0;
    uint32_t up_ok = 0;
    uint32_t it = 0;
    const EpiPolicy ep = epi_policy(p);
    for (int64_t i = unit; i < TI; i += nunits, ++it) {
      __syncwarp();  // every lane is done with the previous tile's slots before lane 0 reloads them
      const int64_t t = mc ? 2 * i + pq : i;
      const Tile tl = decode_tile(p.g, t);
      const uint32_t buf = it & 1, use = it >> 1;
      const int64_t tflag = tl.tile_flag >= 0 ? (tl.tile_flag * CG + half) * EPI_WARPS + q : -1;
      const int64_t wrow = (int64_t)half * ROWS_PER_CTA + q * WROWS;  // this warp's first row in the tile
      int rows_here = tl.rows_valid - (int)wrow;
      rows_here = rows_here < 0 ? 0 : (rows_here > WROWS ? WROWS : rows_here);
      const int64_t row0 = tl.out_row + wrow;
      const int nch = (tl.cols_valid + XCOLS - 1) / XCOLS;
      // TMA needs 16-byte aligned column coordinates (8 bf16); fp8 D goes out by direct stores
      const bool staged = (tl.out_col & 7) == 0 && !(p.out_fp8 && tl.dst == DST_D);
      const bool cep = p.g.ce_partials != 0;
      // a middle step of an in-place RS run may add its product into the
      // partial by TMA reduction instead of loading, adding and storing it
      const bool red = p.rs_reduce != 0 && staged && !cep && tl.src == SRC_X && tl.dst == DST_X;
      const bool has_src = staged && tl.src != SRC_NONE && rows_here > 0 && !red;
      const bool src_f32 = tl.src == SRC_X;
      const bool dst_f32 = tl.dst == DST_X || p.out_f32 != 0;
      const CUtensorMap* src_map = src_f32 ? (cep ? &p.tmR : &p.tmX) : &p.tmC;
      const CUtensorMap* dst_map = tl.dst == DST_X ? (cep ? &p.tmS : &p.tmX) : &p.tmD;
      const int64_t src_col0 = src_f32 && cep ? tl.x_col : tl.out_col;
      const int64_t src_row0 = src_f32 && cep ? tl.xr_row + wrow : row0;
      const int64_t dst_col0 = tl.dst == DST_X && cep ? tl.x_col : tl.out_col;
      const int64_t dst_row0 = tl.dst == DST_X && cep ? tl.xs_row + wrow : row0;
      const int64_t xd_pitch = cep ? p.g.blk_n : p.g.N;
      const int npre = has_src ? (nch < C::WPR ? nch : C::WPR) : 0;
      uint32_t go = 1;
      if (lane == 0) {
        if (cep && tl.s > 0) {
          const int64_t P = p.g.P;
          // the partial this step adds to has arrived in this rank's receive buffer
          const int64_t fsrc = ((tl.r * P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
          wait_flag_geq(p, p.flags + fsrc, p.epoch, (uint32_t)fsrc);
          if (tl.dst == DST_X) {
            // the send buffer's previous contents have been copied out
            const int64_t fsnd = ((((tl.r + P - 1) % P) * P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
            wait_flag_geq(p, p.flags + fsnd, p.epoch, (uint32_t)fsnd);
          }
        }
        const bool need_flag = tflag >= 0 && tl.s > 0;
        const uint32_t want = p.epoch * (uint32_t)p.g.P + (uint32_t)tl.s - 1;
        // never hold a deferred hand-off while waiting for one (a ring of
        // warps could each wait on the next one's)
        if (pend_flag >= 0 && need_flag && ld_acquire_u32(p.flags + tflag) < want) {
          release_partial(p, pend_flag, pend_val);
          pend_flag = -1;
        }
        if (need_flag) wait_flag_geq(p, p.flags + tflag, want, (uint32_t)tflag);
        if (p.up_flags && tl.src == SRC_C && !((up_ok >> upload_unit_c(p.g, tl)) & 1u)) {
          // C of this tile has been uploaded from the host
          const int32_t uu = upload_unit_c(p.g, tl);
          wait_flag_geq(p, p.up_flags + uu, p.epoch, UP_FLAG_INFO | (uint32_t)uu);
          fence_proxy_async_global();
          up_ok |= 1u << uu;
        }
        if (npre > 0) {
          // the source needs only the previous step: load it while the MMAs run.
          // Chunk seq + c reuses the slot of chunk seq + c - WSL, whose store
          // is bulk group seq + c - WSL of seq committed ones.
          fence_proxy_async_global();
          for (int c = 0; c < npre; ++c) {
            if (c == 0)
              bulk_wait_read<C::WSL - 1>();
            else if (c == 1)
              bulk_wait_read<(C::WSL >= 2 ? C::WSL - 2 : 0)>();
            else
              bulk_wait_read<(C::WSL >= 3 ? C::WSL - 3 : 0)>();
            const uint32_t sl = (seq + (uint32_t)c) % C::WSL;
            mbar_arrive_expect_tx(wbar + 8 * sl, src_f32 ? WBUF : WBUF / 2);
            tma_load_2d_epi(wb_addr + sl * WBUF, src_map, wbar + 8 * sl, (int32_t)(src_col0 + c * XCOLS),
                            (int32_t)src_row0, ep);
          }
        }
        // No warp blocks while it holds a deferred hand-off: the accumulator
        // depends on every warp of the pair having read the one before, and
        // one of those may wait for this very hand-off.  So the release is
        // deferred past this wait only when the accumulator is already full.
        if (pend_flag >= 0 && !mbar_try_wait(bar_tfull + 8 * buf, use & 1)) {
          release_partial(p, pend_flag, pend_val);
          pend_flag = -1;
        }
        go = mbar_wait(p, bar_tfull + 8 * buf, use & 1, 0x400000u | buf) ? 1u : 0u;
        if (pend_flag >= 0) {  // the previous tile's bulk stores have had a tile's time to complete
          release_partial(p, pend_flag, pend_val);
          pend_flag = -1;
        }
      }
      for (int c = 0; c < npre; ++c) inflight |= 1u << ((seq + (uint32_t)c) % C::WSL);
      go = __shfl_sync(0xffffffffu, go, 0);
      __syncwarp();  // lane 0's acquires are seen by the lanes that read C or the partial directly
      if (go == 0) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool row_ok = lane < rows_here;
      const int64_t grow = row0 + lane;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + buf * TILE_N;
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        float acc[32];
        if (tl.k_blocks > 0) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * XCOLS, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        }
        if (c == nch - 1) {
          // the accumulator has been read: hand the TMEM buffer back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (CG == 2)
              mbar_arrive_cluster(mapa_shared(bar_tempty + 8 * buf, lead));  // the even CTA's barrier
            else
              mbar_arrive(bar_tempty + 8 * buf);
          }
        }
        const int ncols = tl.cols_valid - c * XCOLS < XCOLS ? tl.cols_valid - c * XCOLS : XCOLS;
        if (!staged) {
          if (row_ok) {
            const float* xs = cep ? p.R + (src_row0 + lane) * p.g.blk_n + src_col0 + c * XCOLS
                                  : p.X + grow * p.g.N + tl.out_col + c * XCOLS;
            float* xd = (cep ? p.S : p.X) + (dst_row0 + lane) * xd_pitch + dst_col0 + c * XCOLS;
            epilogue_row_chunk(p, tl, grow, tl.out_col + c * XCOLS, ncols, acc, xs, xd);
          }
          continue;
        }
        const uint32_t g = seq + (uint32_t)c, sl = g % C::WSL;
        // a box whose rows and columns are all inside the tile (and its shard) goes out by TMA
        const bool tma_ok = rows_here == WROWS && ncols == XCOLS;
        float src[32];
        if (has_src) {
          mbar_wait(p, wbar + 8 * sl, (ph >> sl) & 1u, 0x500000u | (uint32_t)(q * C::WSL) | sl);
          ph ^= 1u << sl;
          inflight &= ~(1u << sl);
          staged_read_row(wb + sl * WBUF, lane, src_f32, p.beta, src);
        } else if (red && !tma_ok && row_ok) {
          // a ragged box of a reducing tile: load, add and store it directly
          const float* x = p.X + grow * p.g.N + tl.out_col + c * XCOLS;
#pragma unroll
          for (int i = 0; i < 32; ++i) src[i] = i < ncols ? __ldcg(x + i) : 0.f;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) src[i] = 0.f;
        }
        float out[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] = fmaf(p.alpha, acc[i], src[i]);
        if (p.bias) add_bias(p, tl.out_col + c * XCOLS, ncols, out);
        if (tma_ok) {
          // the slot is free: every lane has read its source row, or (no source)
          // the store of chunk g - WSL, bulk group g - WSL, has read it
          if (!has_src && lane == 0) bulk_wait_read<C::WSL - 1>();
          __syncwarp();
          staged_write_row(wb + sl * WBUF, lane, dst_f32, out);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (red)
              tma_reduce_add_2d(dst_map, wb_addr + sl * WBUF, (int32_t)(dst_col0 + c * XCOLS), (int32_t)dst_row0,
                                ep);
            else
              tma_store_2d(dst_map, wb_addr + sl * WBUF, (int32_t)(dst_col0 + c * XCOLS), (int32_t)dst_row0, ep);
          }
        } else if (row_ok) {
          float* xp = nullptr;  // the partial's plain-store address (send buffer or X)
          if (tl.dst == DST_X) xp = (cep ? p.S : p.X) + (dst_row0 + lane) * xd_pitch + dst_col0 + c * XCOLS;
          store_row_chunk(p, tl, grow, tl.out_col + c * XCOLS, ncols, out, xp);
        }
        if (lane == 0) bulk_commit();  // bulk group g (empty when the chunk went out by plain stores)
        if (has_src && c + C::WPR < nch) {
          // chunk c + WPR goes to the slot of chunk c - 1, whose store is the
          // group before the one just committed
          const uint32_t sn = (g + C::WPR) % C::WSL;
          __syncwarp();  // every lane has read chunk c - 1's source from that slot
          if (lane == 0) {
            bulk_wait_read<1>();
            mbar_arrive_expect_tx(wbar + 8 * sn, src_f32 ? WBUF : WBUF / 2);
            tma_load_2d_epi(wb_addr + sn * WBUF, src_map, wbar + 8 * sn,
                            (int32_t)(src_col0 + (c + C::WPR) * XCOLS), (int32_t)src_row0, ep);
          }
          inflight |= 1u << sn;
        }
      }
      if (staged) seq += (uint32_t)nch;
      if (p.d_done && tl.dst == DST_D) {
        // count this quarter tile of D as finished: its bulk and plain stores
        // complete and fenced first (the device-to-host stream waits on it)
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          bulk_wait<0>();
          fence_proxy_async_global();
          __threadfence();
          atomicAdd(p.d_done + (int64_t)tl.s * p.g.P + tl.r, 1u);
        }
      }
      if (cep && tl.dst == DST_X) {
        // count this quarter tile as written to the send buffer (the copy stream waits on it)
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          bulk_wait<0>();
          fence_proxy_async_global();
          __threadfence();
          const int64_t fd = ((tl.r * p.g.P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
          atomicAdd(p.done + fd, 1u);
        }
      }
      if (tflag >= 0 && tl.dst == DST_X) {
        const uint32_t val = p.epoch * (uint32_t)p.g.P + (uint32_t)tl.s;
        const bool all_bulk = staged && rows_here == WROWS && (tl.cols_valid % XCOLS) == 0;
        if (all_bulk) {
          // hand the partial on later, once the bulk stores are surely done
          pend_flag = tflag;
          pend_val = val;
        } else {
          // plain stores from the lanes: fence, gather, release now
          __threadfence();
          __syncwarp();
          if (lane == 0) {
            bulk_wait<0>();
            fence_proxy_async_global();
            st_release_u32(p.flags + tflag, val);
          }
        }
      }
    }
    if (lane == 0) {
      if (pend_flag >= 0) release_partial(p, pend_flag, pend_val);
      bulk_wait<0>();  // no bulk store may outlive the CTA
      if (aborted)     // nor a source load that was issued but never consumed
        for (uint32_t sl = 0; sl < (uint32_t)C::WSL; ++sl)
          if ((inflight >> sl) & 1u) mbar_settle(wbar + 8 * sl, (ph >> sl) & 1u);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;  // 0..127
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;    // accumulator row = TMEM lane
    const uint32_t xsrc_addr = smem_u32(xsrc);
    const uint32_t xdst_addr = smem_u32(xdst);
    int64_t pend_flag = -1;  // half-tile flag whose release waits for this CTA's bulk stores
    uint32_t pend_val = 0;
    uint32_t nload = 0;   // staged source chunks loaded so far (buffer idx & 1)
    uint32_t nsrc = 0;    // staged source loads issued (thread 0), for the exit
    uint32_t nstore = 0;  // staged destination chunks stored so far (buffer idx & 1)
    uint32_t up_ok = 0;   // ranks whose uploaded C this thread has seen (thread 0)
    uint32_t it = 0;
    const EpiPolicy ep = epi_policy(p);
    for (int64_t i = unit; i < TI; i += nunits, ++it) {
      const int64_t t = mc ? 2 * i + pq : i;
      const Tile tl = decode_tile(p.g, t);
      const uint32_t buf = it & 1, use = it >> 1;
      const int64_t tflag = tl.tile_flag >= 0 ? tl.tile_flag * CG + half : -1;
      const int rows_here = tl.rows_valid - (int)half * ROWS_PER_CTA;
      const int64_t row0 = tl.out_row + (int64_t)half * ROWS_PER_CTA;
      const int nch = (tl.cols_valid + XCOLS - 1) / XCOLS;
      // Staged tiles need 16-byte aligned TMA column coordinates (8 bf16); fp8
      // results go out by direct stores.
      // (stores-only staging takes no source: a tile with one goes the direct way)
      const bool staged = (EPI == 1 || (EPI == 3 && tl.src == SRC_NONE)) && (tl.out_col & 7) == 0 &&
                          !(p.out_fp8 && tl.dst == DST_D);
      // a middle step of an in-place RS run may add its product into the
      // partial by TMA reduction instead of loading, adding and storing it
      const bool red = p.rs_reduce != 0 && staged && p.g.ce_partials == 0 && tl.src == SRC_X && tl.dst == DST_X;
      const bool has_src = staged && tl.src != SRC_NONE && !red;
      // Where the rotating partial is read and written: the shared partial X
      // (in-place hand-off), or, with copy-engine hand-off, this rank's receive
      // and send buffers.
      const bool cep = p.g.ce_partials != 0;
      const CUtensorMap* src_map = cep ? &p.tmR : &p.tmX;
      const CUtensorMap* xdst_map = cep ? &p.tmS : &p.tmX;
      const int64_t src_col0 = cep ? tl.x_col : tl.out_col;
      const int64_t src_row0 = cep ? tl.xr_row + (int64_t)half * ROWS_PER_CTA : row0;
      const int64_t xd_col0 = cep ? tl.x_col : tl.out_col;
      const int64_t xd_row0 = cep ? tl.xs_row + (int64_t)half * ROWS_PER_CTA : row0;
      const int64_t xd_pitch = cep ? p.g.blk_n : p.g.N;
      if (et == 0) {
        if (cep && tl.s > 0) {
          const int64_t P = p.g.P;
          // the partial this step adds to has arrived in this rank's receive buffer
          const int64_t fsrc = ((tl.r * P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
          wait_flag_geq(p, p.flags + fsrc, p.epoch, (uint32_t)fsrc);
          if (tl.dst == DST_X) {
            // the send buffer's previous contents have been copied out
            const int64_t fsnd = ((((tl.r + P - 1) % P) * P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
            wait_flag_geq(p, p.flags + fsnd, p.epoch, (uint32_t)fsnd);
          }
        }
        const bool need_flag = tflag >= 0 && tl.s > 0;
        const uint32_t want = p.epoch * (uint32_t)p.g.P + (uint32_t)tl.s - 1;
        // Never hold a deferred hand-off while waiting for one: a ring of CTAs
        // could each wait on the next one's.  If this tile has to wait (its
        // previous step is not yet handed on, possibly by this very CTA),
        // release first.
        if (pend_flag >= 0 && need_flag && ld_acquire_u32(p.flags + tflag) < want) {
          release_partial(p, pend_flag, pend_val);
          pend_flag = -1;
        }
        if (need_flag) {
          // partial of this half tile from the previous step
          wait_flag_geq(p, p.flags + tflag, want, (uint32_t)tflag);
        }
        if (p.up_flags && tl.src == SRC_C && !((up_ok >> upload_unit_c(p.g, tl)) & 1u)) {
          // C of this tile has been uploaded from the host (the other threads
          // read it after the barrier below)
          const int32_t uu = upload_unit_c(p.g, tl);
          wait_flag_geq(p, p.up_flags + uu, p.epoch, UP_FLAG_INFO | (uint32_t)uu);
          fence_proxy_async_global();
          up_ok |= 1u << uu;
        }
        if (has_src) {
          // the source needs only the previous step: load it while the MMAs run
          fence_proxy_async_global();
          for (int c = 0; c < nch && c < 2; ++c)
            staged_load_src(p, tl, row0, c, nload + c, xsrc_addr, bar_xfull, src_map, src_col0, src_row0, ep);
          nsrc = nload + (uint32_t)(nch < 2 ? nch : 2);
        }
        bool go = mbar_wait(p, bar_tfull + 8 * buf, use & 1, 0x400000u | buf);
        if (pend_flag >= 0) {  // the previous tile's bulk stores have long completed
          release_partial(p, pend_flag, pend_val);
          pend_flag = -1;
        }
        s_go[it & 1] = go ? 1u : 0u;
      }
      named_bar_sync(1, EPI_THREADS);
      if (s_go[it & 1] == 0) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool row_ok = row < rows_here;
      const int64_t grow = row0 + row;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + buf * TILE_N;
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        float acc[32];
        if (tl.k_blocks > 0) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * XCOLS, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        }
        if (c == nch - 1) {
          // the accumulator has been read: hand the TMEM buffer back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (CG == 2)
              mbar_arrive_cluster(mapa_shared(bar_tempty + 8 * buf, lead));  // the even CTA's barrier
            else
              mbar_arrive(bar_tempty + 8 * buf);
          }
        }
        const int ncols = tl.cols_valid - c * XCOLS < XCOLS ? tl.cols_valid - c * XCOLS : XCOLS;
        if (!staged) {
          if (row_ok) {
            const float* xs = cep ? p.R + (src_row0 + row) * p.g.blk_n + src_col0 + c * XCOLS
                                  : p.X + grow * p.g.N + tl.out_col + c * XCOLS;
            float* xd = (cep ? p.S : p.X) + (xd_row0 + row) * xd_pitch + xd_col0 + c * XCOLS;
            epilogue_row_chunk(p, tl, grow, tl.out_col + c * XCOLS, ncols, acc, xs, xd);
          }
          continue;
        }
        // A whole chunk inside the tile (and inside its shard) goes out by TMA.
        const bool tma_ok = rows_here >= ROWS_PER_CTA && ncols == XCOLS;
        float src[32];
        if (has_src) {
          const uint32_t idx = nload + c, sb = idx & 1;
          mbar_wait(p, bar_xfull + 8 * sb, (idx >> 1) & 1, 0x500000u | sb);
          staged_read_row(xsrc + sb * XBUF, row, tl.src == SRC_X, p.beta, src);
        } else if (red && !tma_ok && row_ok) {
          // a ragged chunk of a reducing tile: load, add and store it directly
          const float* x = p.X + grow * p.g.N + tl.out_col + c * XCOLS;
#pragma unroll
          for (int i = 0; i < 32; ++i) src[i] = i < ncols ? __ldcg(x + i) : 0.f;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) src[i] = 0.f;
        }
        float out[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] = fmaf(p.alpha, acc[i], src[i]);
        if (p.bias) add_bias(p, tl.out_col + c * XCOLS, ncols, out);
        // barrier A: every thread is done with the source buffer, and the
        // store that used this destination buffer two chunks ago has read it
        if (et == 0 && tma_ok) bulk_wait_read<1>();
        named_bar_sync(1, EPI_THREADS);
        if (tma_ok) {
          const uint32_t db = nstore & 1;
          staged_write_row(xdst + db * XBUF, row, tl.dst == DST_X || p.out_f32 != 0, out);
          fence_proxy_async_smem();
          named_bar_sync(1, EPI_THREADS);  // barrier B: the chunk is complete in shared memory
          if (et == 0) {
            if (red)
              tma_reduce_add_2d(xdst_map, xdst_addr + db * XBUF, (int32_t)(xd_col0 + c * XCOLS), (int32_t)xd_row0,
                                ep);
            else if (tl.dst == DST_X)
              tma_store_2d(xdst_map, xdst_addr + db * XBUF, (int32_t)(xd_col0 + c * XCOLS), (int32_t)xd_row0, ep);
            else
              tma_store_2d(&p.tmD, xdst_addr + db * XBUF, (int32_t)(tl.out_col + c * XCOLS), (int32_t)row0, ep);
            bulk_commit();
          }
          ++nstore;
        } else if (row_ok) {
          float* xp = nullptr;  // the partial's plain-store address (send buffer or X)
          if (tl.dst == DST_X) xp = (cep ? p.S : p.X) + (xd_row0 + row) * xd_pitch + xd_col0 + c * XCOLS;
          store_row_chunk(p, tl, grow, tl.out_col + c * XCOLS, ncols, out, xp);
        }
        if (et == 0 && has_src && c + 2 < nch) {
          staged_load_src(p, tl, row0, c + 2, nload + c + 2, xsrc_addr, bar_xfull, src_map, src_col0, src_row0, ep);
          nsrc = nload + (uint32_t)c + 3;
        }
      }
      if (has_src) nload += (uint32_t)nch;
      if (p.d_done && tl.dst == DST_D) {
        // count this half tile of D as finished: its bulk and plain stores
        // complete and fenced first (the device-to-host stream waits on it)
        if (EPI != 0 && et == 0) bulk_wait<0>();
        __threadfence();
        named_bar_sync(1, EPI_THREADS);
        if (et == 0) {
          if (EPI != 0) fence_proxy_async_global();
          __threadfence();
          atomicAdd(p.d_done + (int64_t)tl.s * p.g.P + tl.r, 1u);
        }
      }
      if (cep && tl.dst == DST_X) {
        // count this half tile as written to the send buffer: its bulk and
        // plain stores complete and fenced first (the copy stream waits on it)
        if (et == 0) bulk_wait<0>();
        __threadfence();
        named_bar_sync(1, EPI_THREADS);
        if (et == 0) {
          fence_proxy_async_global();
          __threadfence();
          const int64_t fd = ((tl.r * p.g.P + tl.s) * p.g.L + tl.l) * p.g.tiles_m + tl.band;
          atomicAdd(p.done + fd, 1u);
        }
      }
      if (tflag >= 0 && tl.dst == DST_X) {
        const uint32_t val = p.epoch * (uint32_t)p.g.P + (uint32_t)tl.s;
        // every chunk left by TMA store (issued by thread 0 alone)?
        const bool all_bulk = staged && rows_here >= ROWS_PER_CTA && (tl.cols_valid % XCOLS) == 0;
        if (all_bulk) {
          // hand the partial on later, once the bulk stores are surely done
          pend_flag = tflag;
          pend_val = val;
        } else {
          // plain stores from every thread: fence, gather, release now
          if (EPI != 0 && et == 0) bulk_wait<0>();
          __threadfence();
          named_bar_sync(1, EPI_THREADS);
          if (et == 0) {
            if (EPI != 0) fence_proxy_async_global();
            st_release_u32(p.flags + tflag, val);
          }
        }
      }
    }
    if (et == 0 && pend_flag >= 0) release_partial(p, pend_flag, pend_val);
    if (EPI != 0 && et == 0) {
      bulk_wait<0>();  // no bulk store may outlive the CTA
      if (aborted)     // nor a source load that was issued but never consumed
        for (uint32_t idx = nsrc > 2u ? nsrc - 2u : 0u; idx < nsrc; ++idx)
          mbar_settle(bar_xfull + 8 * (idx & 1u), (idx >> 1) & 1u);
    }
  }

  if (CG == 2) {
    // The operand loads that land in a pair complete on its even CTA's
    // barriers: both CTAs' own loads, and with multicast the other pair's
    // halves of the B rows.  So each even CTA waits for all of them before any
    // CTA may exit.  After an abort the producers may have stopped at
    // different loads (at most one ring of stages apart: a load is issued only
    // once the MMAs consumed the stage's previous load, which needed every
    // contributor's bytes), so first the phases not every contributor loaded
    // are balanced: a phase the even CTA never armed is armed for the bytes
    // that were issued, a missing contribution to an armed phase is counted as
    // arrived.  Without an abort all counts are equal and every phase has
    // already completed.
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();  // the producers' counts are in the even CTAs' shared memory
    tc_fence_after();
    if (leader && warp == 0 && lane == 0) {
      const uint32_t own_bytes = mc ? C::A_BYTES + C::B_BYTES / 2 : C::STAGE_BYTES;
      const uint32_t oth_bytes = C::B_BYTES / 2;
      const uint32_t k0 = s_kcnt[lead], k1 = s_kcnt[lead + 1];
      const uint32_t k2 = mc ? s_kcnt[lead ^ 2u] : k0, k3 = mc ? s_kcnt[(lead ^ 2u) + 1] : k0;
      const uint32_t kmin = min(min(k0, k1), min(k2, k3)), kmax = max(max(k0, k1), max(k2, k3));
      auto bytes_in = [&](uint32_t n) {
        uint32_t b = (k0 > n ? own_bytes : 0u) + (k1 > n ? own_bytes : 0u);
        if (mc) b += (k2 > n ? oth_bytes : 0u) + (k3 > n ? oth_bytes : 0u);
        return b;
      };
      for (uint32_t n = kmin; n < kmax; ++n) {
        const uint32_t fb = bar_full + 8 * (n % STAGES), b = bytes_in(n);
        if (n < k0) {
          if (b < 2 * C::STAGE_BYTES) mbar_complete_tx(fb, 2 * C::STAGE_BYTES - b);
        } else if (b > 0) {
          mbar_arrive_expect_tx(fb, b);
        }
      }
      for (uint32_t n = kmax > (uint32_t)STAGES ? kmax - STAGES : 0u; n < kmax; ++n)
        if (n < k0 || bytes_in(n) > 0) mbar_settle(bar_full + 8 * (n % STAGES), (n / STAGES) & 1u);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (CG == 2)
    cluster_sync_all();  // no remote arrive may target a CTA that has exited
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (CG == 2)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Reduction of the non-fused ReduceScatter baseline:
//   D[e] = (X_0[e] + X_1[e] + ... + X_{P-1}[e]) + beta * C[e]   (bf16 or fp32 D)
// over the P stacked fp32 partials (each already scaled by alpha and carrying
// its bias), four elements per thread and iteration, grid-stride.  HBM-bound.
__global__ void __launch_bounds__(256) dg_reduce_partials_kernel(const float* __restrict__ X, int P,
                                                                 int64_t n4, const __nv_bfloat16* C,
                                                                 float beta, void* D, int out_f32, int out_fp8,
                                                                 float result_scale) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t plane = n4;  // float4 units per partial
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 acc = __ldcs(reinterpret_cast<const float4*>(X) + i);
    for (int r = 1; r < P; ++r) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(X) + r * plane + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (beta != 0.f) {
      const uint2 cw = __ldg(reinterpret_cast<const uint2*>(C) + i);
      acc.x += beta * bf16_bits_to_f32(cw.x & 0xFFFFu);
      acc.y += beta * bf16_bits_to_f32(cw.x >> 16);
      acc.z += beta * bf16_bits_to_f32(cw.y & 0xFFFFu);
      acc.w += beta * bf16_bits_to_f32(cw.y >> 16);
    }
    if (out_fp8) {
      const __nv_fp8_interpretation_t fmt = out_fp8 == 1 ? __NV_E4M3 : __NV_E5M2;
      const __nv_fp8x2_storage_t lo =
          __nv_cvt_float2_to_fp8x2(make_float2(acc.x * result_scale, acc.y * result_scale), __NV_SATFINITE, fmt);
      const __nv_fp8x2_storage_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(acc.z * result_scale, acc.w * result_scale), __NV_SATFINITE, fmt);
      reinterpret_cast<uint32_t*>(D)[i] = (uint32_t)lo | ((uint32_t)hi << 16);
    } else if (out_f32) {
      reinterpret_cast<float4*>(D)[i] = acc;
    } else {
      uint2 o;
      o.x = pack_bf16x2(acc.x, acc.y);
      o.y = pack_bf16x2(acc.z, acc.w);
      reinterpret_cast<uint2*>(D)[i] = o;
    }
  }
}

}  // namespace dg
