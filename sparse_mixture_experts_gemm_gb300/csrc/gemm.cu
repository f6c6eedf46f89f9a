// gemm.cu -- persistent grouped GEMM on the 5th-generation tensor cores.
//
// One kernel template serves the two grouped contractions of the block:
//   EPI_SWIGLU : for each expert group, gate and up projections of its rows in
//                one MMA (B tile = 128 gate rows over 128 up rows), epilogue
//                h = silu(gate) * up written once (section "Reduce
//                intermediate traffic and dispatch traffic": input
//                projections fused with the gated activation).  Routed A rows
//                are gathered from x by four extra warps (16-byte cp.async
//                into the swizzled tile, the token of each row from the
//                router's per-expert list or the slot permutation); the
//                shared expert's rows (x in order) come by TMA.
//   EPI_STORE  : the down projection of each group's rows, stored per slot.
// The tiles of both grouped GEMMs are derived on the device from the group
// sizes the routing left (section "Keep expert routing on the GPU": the
// block map of fixed-size blocks the grouped GEMM processes), so no host
// synchronisation is needed: every CTA scans ceil(rows / 128) over the groups
// and maps a tile index to (group, m, n) by binary search.  Tiles of one group
// are ordered with m innermost, so the CTAs that share a weight block run side
// by side and the weight block is read from HBM once.
//
// CTA layout: 192 threads (320 for the gate/up GEMM).  Warp 0 produces a
// shared-memory ring of 128-byte-swizzled K-major tiles (lane 0 issues the TMA
// tile loads; 4 stages); warp 1 allocates 2N TMEM
// columns (two 128 x N fp32 accumulators) and its lane 0 issues tcgen05.mma
// (M = 128, 32 bytes of K per instruction); warps 2-5 drain a finished
// accumulator with tcgen05.ld while the MMA fills the other; warps 6-9 of the
// gate/up GEMM gather its routed A rows.
// The grid is persistent: CTA c takes tile c, then claims tiles from a
// counter; in cluster-pair mode the clusters take work items in a fixed order.
// Every wait is bounded; a wait that runs out records a timeout in the status
// word, raises a CTA-wide abort flag, drains what it issued and returns.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <typename T, int BN>
struct Tile {
  static constexpr int BK = 128 / sizeof(T);  // K elements per 128-byte row
  static constexpr int A_BYTES = kBM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // as many stages as the tile budget holds, at most 8
  static constexpr int STAGES =
      (kStageBudget / STAGE_BYTES) < 8 ? (kStageBudget / STAGE_BYTES) : 8;
  static_assert(STAGES >= 2, "pipeline needs two stages");
};


}  // namespace

// Threads of one CTA: the gate/up GEMM adds four warps that gather the routed
// token rows of its A tiles.
template <int EPI>
constexpr int gemm_threads() { return EPI == EPI_SWIGLU ? kThreads + kGatherThreads : kThreads; }

template <typename T, int EPI, int BN, bool kPair>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const __grid_constant__ CUtensorMap tmB0s,
                const __grid_constant__ CUtensorMap tmB1s, const GemmParams p) {
  using C = Tile<T, BN>;
  constexpr bool kDual = (EPI == EPI_SWIGLU);  // B = gate rows over up rows
  constexpr bool kGather = (EPI == EPI_SWIGLU);  // routed A rows gathered by warps 6-9
  constexpr int kOutCols = (EPI == EPI_SWIGLU) ? BN / 2 : BN;
  constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint8_t *ctrl = sB + C::STAGES * C::B_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 512);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 516);
  int *s_off = reinterpret_cast<int *>(ctrl + 1536);        // [E + 1]
  int *s_mt = reinterpret_cast<int *>(ctrl + 1536 + 1040);  // [E + 2]
  int *s_it = reinterpret_cast<int *>(ctrl + 1536 + 2080);  // [E + 2], pair mode
  const TileRing ring{smem_u32(ctrl + 1056), smem_u32(ctrl + 1056 + 8 * kTileRing),
                      reinterpret_cast<volatile int *>(ctrl + 1024)};
  // readers of the ring: the MMA thread, 4 epilogue warps, 4 gather warps
  constexpr int kTileReaders = 1 + 4 + (EPI == EPI_SWIGLU ? 4 : 0);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::STAGES;
  const uint32_t tfull0 = empty0 + 8 * C::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long limit = MOE_WAIT_LIMIT_CYCLES;
  const GroupTable gt{s_off, s_mt};
  // pair mode: this CTA's rank in its cluster of two, the cluster's index
  // and count (items are taken in a fixed order: cluster c runs items
  // c, c + ncl, ...)
  const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const int cl = kPair ? static_cast<int>(blockIdx.x >> 1) : 0;
  const int ncl = kPair ? static_cast<int>(gridDim.x >> 1) : 1;
  constexpr uint16_t kBoth = 3;  // cluster mask of both CTAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // the TMA producer's expect-tx arrival, plus one per gather thread
      mbar_init(full0 + 8 * s, kGather ? 1 + kGatherThreads : 1);
      // pair mode: a stage is free when the MMAs of both CTAs are done with it
      // (the partner's producer writes half of the weight tile into it)
      mbar_init(empty0 + 8 * s, kPair ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    mbar_init(drain_bar, 1);
    for (int q = 0; q < kTileRing; ++q) {
      mbar_init(ring.full0 + 8 * q, 1);
      mbar_init(ring.empty0 + 8 * q, kTileReaders);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmAs);
    if (EPI == EPI_SWIGLU) {
      prefetch_tmap(&tmB1);
      prefetch_tmap(&tmB0s);
      prefetch_tmap(&tmB1s);
    }
    if (EPI == EPI_STORE) prefetch_tmap(kPair ? &tmB1s : &tmB0s);
    if (EPI == EPI_STORE && kPair) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // pair mode: both CTAs' barriers exist before either writes into the other
  if (kPair) cluster_sync_all();
  // Launched as a programmatic dependent, everything above overlaps the tail
  // of the previous kernel: none of it touches global memory.  The wait
  // returns once that kernel has completed and its writes are visible; the
  // next kernel may then be scheduled (its CTAs run their own prologue and
  // wait in turn).  Both are no-ops in an ordinary launch.
  pdl_wait();
  pdl_launch_dependents();
  build_group_table(p, s_off, s_mt, warp, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int ntiles = p.nt * s_mt[p.n_routed + 1];
  if (kPair) {
    build_item_table(p, s_mt, s_it, warp, lane);
    __syncthreads();
    ntiles = s_it[p.n_routed + 1];
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    uint32_t pend_mask = 0, pend_phase = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int ti = kPair ? cl + it * ncl : blockIdx.x + it * gridDim.x;
      if (!kPair) {
        int c_ok = 1;
        if (lane == 0) c_ok = claim_tile(ring, it, p.tile_ctr, ntiles, limit, abort_flag, ti) ? 1 : 0;
        ti = __shfl_sync(0xffffffffu, ti, 0);
        if (!__shfl_sync(0xffffffffu, c_ok, 0)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
      }
      if (ti >= ntiles) break;
      bool mc = false;
      const GemmTile tl = kPair ? decode_pair_item(gt, s_it, p, ti, rank, kOutCols, !kDual, mc)
                                : decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool sh = tl.group >= p.n_routed;
      const CUtensorMap *ma = sh ? &tmAs : &tmA;
      const CUtensorMap *mb0 = sh ? &tmB0s : &tmB0;
      const CUtensorMap *mb1 = sh ? &tmB1s : &tmB1;
      const int brow = sh ? tl.n0 : tl.group * p.b_rows_per_group + tl.n0;
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        const int kx = kb * C::BK;
        const uint32_t a_dst = smem_u32(sA + stage * C::A_BYTES);
        const uint32_t b_dst = smem_u32(sB + stage * C::B_BYTES);
        if (lane == 0) {
          // gate/up: routed A rows come from the gather warps, the shared
          // expert's (the tokens in order) from TMA like every B tile
          const bool a_tma = !kGather || sh;
          mbar_arrive_expect_tx(fb, a_tma ? C::STAGE_BYTES : C::B_BYTES);
          if (a_tma) tma_load_2d(a_dst, ma, fb, kx, tl.a_row, pol_a);
          if (kPair && mc) {
            // both CTAs multiply this weight tile: each loads one half into
            // both (gate/up: the gate rows or the up rows; down: 128 of the
            // 256 rows through the half-height map)
            const uint32_t hb = b_dst + rank * (C::B_BYTES / 2);
            if (kDual) tma_load_2d_mc(hb, rank ? mb1 : mb0, fb, kx, brow, kBoth, pol_w);
            else tma_load_2d_mc(hb, mb1, fb, kx, brow + rank * (BN / 2), kBoth, pol_w);
          } else if (kDual) {
            tma_load_2d(b_dst, mb0, fb, kx, brow, pol_w);
            tma_load_2d(b_dst + C::B_BYTES / 2, mb1, fb, kx, brow, pol_w);
          } else if (kPair) {
            tma_load_2d(b_dst, mb1, fb, kx, brow, pol_w);
            tma_load_2d(b_dst + C::B_BYTES / 2, mb1, fb, kx, brow + BN / 2, pol_w);
          } else {
            tma_load_2d(b_dst, mb0, fb, kx, brow, pol_w);
          }
        }
        pend_mask |= 1u << stage;
        pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (kPair && ok) {
      // the partner's MMA arrives on this CTA's stages: wait for its last
      // arrival on each, so none lands after the CTA has ended
      for (int j = 0; j < C::STAGES; ++j) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
          }
          break;
        }
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // copies already issued must land before the CTA's shared memory goes away
      for (int s = 0; s < C::STAGES; ++s)
        if (pend_mask & (1u << s))
          if (!mbar_wait(full0 + 8 * s, (pend_phase >> s) & 1, limit, nullptr))
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(kBM, BN, MmaKind<T>::ab_format);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int it = 0; ok; ++it) {
        int ti = kPair ? cl + it * ncl : blockIdx.x + it * gridDim.x;
        if (!kPair && !read_tile(ring, it, limit, abort_flag, ti)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
          ok = false;
          break;
        }
        if (ti >= ntiles) break;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          // gathered A rows were written by cp.async (generic proxy); the
          // barrier made them visible to this thread, the fence to the
          // tensor core's reads
          if (kGather) fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            MmaKind<T>::mma(d_tmem, sdesc_sw128(a0 + 32 * kk), sdesc_sw128(b0 + 32 * kk), idesc,
                            (kb | kk) != 0 ? 1u : 0u);
          // pair mode: the stage is released in both CTAs (the partner's
          // producer fills half of this CTA's weight tile)
          if (kPair) tc_commit_mc(empty0 + 8 * stage, kBoth);
          else tc_commit(empty0 + 8 * stage);
          issued = true;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // On the normal path the epilogue has waited for every accumulator, so
      // all MMAs are done.  After an abort, wait for the ones issued so far
      // before TMEM is released.
      if (!ok && issued) {
        tc_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0, limit, nullptr))
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
      }
    }
  } else if (kGather && warp >= 6) {
    // ------------------------------------------------------------ gather
    // Each routed A tile row (128 bytes of K per k-block, from the token row
    // perm[slot]) is copied by 8 threads, 16 bytes each, so one warp copies 4
    // whole rows per instruction; thread g takes chunk g % 8 of rows
    // g / 8 + 16 i.  Chunk c of row r goes where the 128-byte swizzle the MMA
    // descriptor expects puts it: c ^ (r % 8).  Rows past the tile's end are
    // left as they are: the epilogue never stores them.  Every gather thread
    // arrives on every stage's full barrier through cp.async.mbarrier.arrive,
    // which fires when the thread's copies so far have landed; the MMA thread
    // fences the proxy before the tensor core reads them.
    const int g = threadIdx.x - kThreads;
    const int c = g & 7, r0 = g >> 3;
    const int K = p.num_k_blocks * C::BK;
    const T *xg = static_cast<const T *>(p.x);
    constexpr int kChunk = 16 / static_cast<int>(sizeof(T));  // elements per 16 bytes
    constexpr int kRowsPer = kBM / (kGatherThreads / 8);      // rows per thread: 8
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int ti = cl + it * ncl, r_ok = 1;
      if (!kPair) {
        if (lane == 0) r_ok = read_tile(ring, it, limit, abort_flag, ti) ? 1 : 0;
        ti = __shfl_sync(0xffffffffu, ti, 0);
      }
      if (!__shfl_sync(0xffffffffu, r_ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
        }
        ok = false;
        break;
      }
      if (ti >= ntiles) break;
      bool mc = false;
      const GemmTile tl = kPair ? decode_pair_item(gt, s_it, p, ti, rank, kOutCols, !kDual, mc)
                                : decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool routed = tl.group < p.n_routed;
      const T *src[kRowsPer];
      int tok[kRowsPer];
      if (routed) gather_tokens<kRowsPer>(p, gt, tl, r0, tok);
#pragma unroll
      for (int i = 0; i < kRowsPer; ++i)
        src[i] = (routed && r0 + 16 * i < tl.rows)
                     ? xg + static_cast<long long>(tok[i]) * K + c * kChunk
                     : nullptr;
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t tile_dst = smem_u32(sA + stage * C::A_BYTES);
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          const int r = r0 + 16 * i;
          if (src[i] != nullptr)
            cp_async16(tile_dst + r * 128 + ((c ^ (r & 7)) << 4), src[i] + kb * C::BK);
        }
        cp_async_arrive(full0 + 8 * stage);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // copies in flight must land before the CTA's shared memory goes away
    cp_async_wait_all();
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;       // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;  // tile row == TMEM lane
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      int ti = kPair ? cl + it * ncl : blockIdx.x + it * gridDim.x;
      if (!kPair) {
        int r_ok = 1;
        if (lane == 0) r_ok = read_tile(ring, it, limit, abort_flag, ti) ? 1 : 0;
        ti = __shfl_sync(0xffffffffu, ti, 0);
        if (!__shfl_sync(0xffffffffu, r_ok, 0)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_EPI_TMEM_FULL);
          }
          break;
        }
      }
      if (ti >= ntiles) break;
      bool mc = false;
      const GemmTile tl = kPair ? decode_pair_item(gt, s_it, p, ti, rank, kOutCols, !kDual, mc)
                                : decode_tile(gt, p, ti, kOutCols, !kDual);
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_EPI_TMEM_FULL);
        }
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(wq * 32) << 16);
      const bool valid = r < tl.rows;

      if (EPI == EPI_SWIGLU) {
        T *hrow = reinterpret_cast<T *>(p.out) + static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          float g[32], u[32];
          tmem_ld32x2_sync(tb + c, tb + BN / 2 + c, g, u);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = silu(g[i]) * u[i];
            store32<T>(hrow + c, g);
          }
        }
      } else if (EPI == EPI_STORE) {
        T *yrow = reinterpret_cast<T *>(p.out) + static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32_sync(tb + c, v);
          if (valid) store32<T>(yrow + c, v);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (kPair) {
    // neither CTA ends while its partner may still write into it; after an
    // abort, copies the partner issued before it stopped get time to land
    cluster_sync_all();
    if (*abort_flag)
      for (int i = 0; i < 200; ++i) __nanosleep(1000);
  }
}

template <typename T, int EPI, int BN, bool kPair>
cudaError_t gemm_set_smem_attr() {
  return cudaFuncSetAttribute(gemm_kernel<T, EPI, BN, kPair>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
}

template <typename T, int EPI, int BN, bool kPair>
cudaError_t launch_gemm(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                        bool pdl) {
  if (grid <= 0) return cudaSuccess;
  if (kPair && (grid & 1)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemm_threads<EPI>());
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (kPair) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<T, EPI, BN, kPair>, maps.m[0], maps.m[1], maps.m[2],
                            maps.m[3], maps.m[4], maps.m[5], p);
}

int gemm_pair_clusters() {
  int best = 0;
  for (int e = 0; e < 2; ++e) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(e == 0 ? gemm_threads<EPI_SWIGLU>() : gemm_threads<EPI_STORE>());
    cfg.dynamicSmemBytes = kGemmSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t err =
        e == 0 ? cudaOccupancyMaxActiveClusters(&n, gemm_kernel<__nv_bfloat16, EPI_SWIGLU, kBN, true>,
                                                &cfg)
               : cudaOccupancyMaxActiveClusters(&n, gemm_kernel<__nv_bfloat16, EPI_STORE, kBN, true>,
                                                &cfg);
    if (err != cudaSuccess) return 0;
    best = e == 0 ? n : (n < best ? n : best);
  }
  return best;
}

template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_SWIGLU, kBN>();
template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_STORE, kBN>();
template cudaError_t gemm_set_smem_attr<float, EPI_SWIGLU, kBN>();
template cudaError_t gemm_set_smem_attr<float, EPI_STORE, kBN>();
template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_SWIGLU, kBN, true>();
template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_STORE, kBN, true>();
template cudaError_t launch_gemm<__nv_bfloat16, EPI_SWIGLU, kBN, true>(const GemmMaps &,
                                                                        const GemmParams &, int,
                                                                        cudaStream_t, bool);
template cudaError_t launch_gemm<__nv_bfloat16, EPI_STORE, kBN, true>(const GemmMaps &,
                                                                       const GemmParams &, int,
                                                                       cudaStream_t, bool);
template cudaError_t launch_gemm<__nv_bfloat16, EPI_SWIGLU, kBN>(const GemmMaps &, const GemmParams &,
                                                                  int, cudaStream_t, bool);
template cudaError_t launch_gemm<__nv_bfloat16, EPI_STORE, kBN>(const GemmMaps &, const GemmParams &,
                                                                 int, cudaStream_t, bool);
template cudaError_t launch_gemm<float, EPI_SWIGLU, kBN>(const GemmMaps &, const GemmParams &, int,
                                                          cudaStream_t, bool);
template cudaError_t launch_gemm<float, EPI_STORE, kBN>(const GemmMaps &, const GemmParams &, int,
                                                         cudaStream_t, bool);

// ---------------------------------------------------------------- test hook
// Waits on an mbarrier that nothing signals, with the same bounded wait the
// GEMM uses, then records the timeout and returns.
__global__ void debug_wait_kernel(int *status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait(smem_u32(&bar), 0, limit, nullptr))
      report_error(status, MOE_ERR_DEVICE_TIMEOUT, KID_DEBUG * 100 + SITE_DEBUG);
  }
}

cudaError_t launch_debug_wait(int *status, long long limit_cycles, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace moe
