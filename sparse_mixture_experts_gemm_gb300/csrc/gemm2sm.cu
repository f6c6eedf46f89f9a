// gemm2sm.cu -- the grouped GEMMs of large chunks on the two-CTA tensor-core
// MMA (tcgen05.mma.cta_group::2).
//
// A thread-block cluster of two CTAs (a CTA pair, one per SM of a pair)
// computes one 256 x 256 fp32 accumulator per work item: two consecutive
// 128-row M tiles of one expert group times one 256-row B tile (section
// "Match tile size to expert load": large groups take the large tile).  CTA r
// holds rows 128 r .. 128 r + 127 of the accumulator in its own TMEM, stages
// its own 128 A rows and one half of the B tile (gate/up: the 128 gate rows
// in CTA 0, the 128 up rows in CTA 1, so each CTA's accumulator is again
// [gate | up] for its rows; down: 128 of the 256 output columns each), and
// the MMA issued by CTA 0 reads both CTAs' halves.  Per SM and 64-element
// k-block this moves 16 KB of A and 16 KB of B into shared memory and reads
// 32 KB out of it; the one-CTA GEMM of the same 256-column tile moves 16 KB
// of A and 32 KB of B and reads 48 KB, more than shared memory delivers at
// the MMA's rate.
//
// Work items: group g with mt M tiles has nt * ceil(mt / 2) items, item
// (n, q) pairing M tiles 2 q and 2 q + 1 (the second may be past the group's
// end: that CTA still loads its B half, gathers no rows and stores nothing).
// Clusters take items in a fixed order (cluster c runs c, c + ncl, ...).
//
// Roles (both CTAs unless noted): warp 0 lane 0 issues the TMA loads of the
// CTA's A rows (shared expert, down projection) and B half; warp 1 allocates
// 512 TMEM columns in both CTAs (two accumulators); in CTA 0 its lane 0
// issues the MMAs, in CTA 1 (gate/up) it tells CTA 0 when the rows gathered
// into a stage have landed; warps 2-5
// drain the CTA's accumulator rows; warps 6-9 of the gate/up GEMM gather its
// routed A rows.  Barriers: full[s] in CTA 0 counts every byte of stage s in
// both CTAs (the TMA copies of both complete it directly) and the gather
// arrivals of CTA 0; CTA 1's gathered rows complete a local full[s], and its
// forwarder then adds 4 bytes to CTA 0's full[s] with an asynchronous remote
// store (a thread's remote mbarrier.arrive holds it for a round trip of about
// 1,500 cycles, longer than a stage's MMAs).  empty[s]
// and tfull[a] (both CTAs, arrived on by the MMA's multicast commit),
// tempty[a] (CTA 0 only: the four epilogue warps of each CTA have drained
// accumulator a).  Every wait is bounded; a wait that runs out records a
// timeout in the status word, raises the CTA's abort flag and stops its
// role; CTA 0 waits for the MMAs it issued, both CTAs meet at a cluster
// barrier before the TMEM is freed, and neither ends while the other may
// still write into it.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

// A stage holds 128 elements of K: two 128-byte column blocks of the CTA's
// 128 A rows and of its 128 B rows, each block a 16 KB tile in the 128-byte
// swizzle.  One barrier wait and one commit then cover 8 MMAs: the wait
// (about 90 cycles), the commit and the issue of each two-CTA MMA (about 80)
// are paid by one thread, and with 64-element stages that thread needed
// more cycles per stage than the MMAs took.
constexpr int kBK2 = 64;                                // bf16 K elements per 128-byte block
constexpr int kCB = 2;                                  // column blocks per stage
constexpr int kKS = kCB * kBK2;                         // K elements per stage
constexpr int kBlk = kBM * 128;                         // one 128-row column block: 16 KB
constexpr int kA2 = kCB * kBlk;                         // this CTA's A rows of a stage
constexpr int kB2 = kCB * kBlk;                         // this CTA's half of the B rows
constexpr int kStages2 = kStageBudget / (kA2 + kB2);  // 3
constexpr uint32_t kTmemCols2 = 2 * kBN;                // two accumulators
static_assert(kStages2 >= 2 && kStages2 <= 8, "stage count");

}  // namespace

template <int EPI>
constexpr int gemm2sm_threads() { return EPI == EPI_SWIGLU ? kThreads + kGatherThreads : kThreads; }

template <int EPI>
__global__ void __launch_bounds__(gemm2sm_threads<EPI>(), 1)
    gemm2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmB0s,
                   const __grid_constant__ CUtensorMap tmB1s, const GemmParams p) {
  using T = __nv_bfloat16;
  constexpr bool kDual = (EPI == EPI_SWIGLU);    // B = gate rows over up rows
  constexpr bool kGather = (EPI == EPI_SWIGLU);  // routed A rows gathered by warps 6-9
  constexpr int kOutCols = kDual ? kBN / 2 : kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages2 * kA2;
  uint8_t *ctrl = smem + kStageBudget;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 512);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 516);
  int *s_off = reinterpret_cast<int *>(ctrl + 1536);        // [E + 1]
  int *s_mt = reinterpret_cast<int *>(ctrl + 1536 + 1040);  // [E + 2]
  int *s_it = reinterpret_cast<int *>(ctrl + 1536 + 2080);  // [E + 2]
  uint32_t *s_pf = reinterpret_cast<uint32_t *>(ctrl + 1024);  // [kStages2] CTA 1's forwards

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages2;
  const uint32_t tfull0 = empty0 + 8 * kStages2;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long limit = MOE_WAIT_LIMIT_CYCLES;
  const GroupTable gt{s_off, s_mt};
  const int rank = static_cast<int>(cluster_ctarank());
  const int cl = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  constexpr uint16_t kBoth = 3;  // cluster mask of both CTAs

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      // CTA 0: its producer's expect-tx arrival and one per gather thread;
      // CTA 1: one per gather thread (gate/up; the down GEMM does not use it)
      mbar_init(full0 + 8 * s, rank == 0 ? 1 + (kGather ? kGatherThreads : 0)
                                         : (kGather ? kGatherThreads : 1));
      mbar_init(empty0 + 8 * s, 1);  // CTA 0's multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 8);  // four epilogue warps of each CTA
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmAs);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmB1s);
    if (kDual) {
      prefetch_tmap(&tmB0);
      prefetch_tmap(&tmB0s);
    }
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(tmem_slot), kTmemCols2);
    tmem_relinquish2();
  }
  // both CTAs' barriers exist before either arrives on the other's
  cluster_sync_all();
  // programmatic dependent launch: the prologue above overlaps the previous
  // kernel's tail; nothing before this wait touches global memory
  pdl_wait();
  pdl_launch_dependents();
  build_group_table(p, s_off, s_mt, warp, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  build_item_table(p, s_mt, s_it, warp, lane, true);
  __syncthreads();
  const int nitems = s_it[p.n_routed + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    uint32_t pend_mask = 0, pend_phase = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int ti = cl + it * ncl;
      if (ti >= nitems) break;
      const GemmTile tl = decode_2cta_item(gt, s_it, p, ti, rank, kOutCols, !kDual);
      const bool sh = tl.group >= p.n_routed;
      const CUtensorMap *ma = sh ? &tmAs : &tmA;
      // gate/up: the gate rows (CTA 0) or the up rows (CTA 1) of the N tile;
      // down: 128-row boxes, CTA r the rows n0 + 128 r
      const CUtensorMap *mb = (kDual && rank == 0) ? (sh ? &tmB0s : &tmB0) : (sh ? &tmB1s : &tmB1);
      const int brow =
          (sh ? tl.n0 : tl.group * p.b_rows_per_group + tl.n0) + (kDual ? 0 : rank * (kBN / 2));
      // A rows by TMA for the down GEMM and the gate/up GEMM's shared expert
      // (also in a CTA whose tile has no rows: the box is read as zeros or
      // ignored), otherwise by the gather warps.  CTA 0's full barrier
      // expects the bytes of both CTAs, plus the forward for gate/up.
      const bool a_tma = !kGather || sh;
      const uint32_t tx = 2 * (kB2 + (a_tma ? kA2 : 0)) + (kGather ? 4 : 0);
      const int nks = p.num_k_blocks / kCB;
      for (int ks = 0; ks < nks; ++ks) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0) {
          const uint32_t fb0 = cluster_map(fb, 0);
          if (rank == 0) mbar_arrive_expect_tx(fb, tx);
#pragma unroll
          for (int h = 0; h < kCB; ++h) {
            const int kx = ks * kKS + h * kBK2;
            if (a_tma)
              tma_load_2d_pair(smem_u32(sA + stage * kA2 + h * kBlk), ma, fb0, kx, tl.a_row, pol_a);
            tma_load_2d_pair(smem_u32(sB + stage * kB2 + h * kBlk), mb, fb0, kx, brow, pol_w);
          }
        }
        pend_mask |= 1u << stage;
        pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages2) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (ok) {
      // CTA 0's commits arrive on this CTA's stages: wait for the last
      // arrival on each, so none lands after the CTA has ended
      for (int j = 0; j < kStages2; ++j) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
          }
          break;
        }
        if (++stage == kStages2) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0 && rank == 0) {
      // copies already issued must land before the CTA's shared memory goes
      // away (CTA 1's copies complete on CTA 0, which waits for them; the
      // CTAs meet at the final cluster barrier)
      for (int s = 0; s < kStages2; ++s)
        if (pend_mask & (1u << s))
          if (!mbar_wait(full0 + 8 * s, (pend_phase >> s) & 1, limit, nullptr))
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(2 * kBM, kBN, MmaKind<T>::ab_format);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int it = 0; ok; ++it) {
        const int ti = cl + it * ncl;
        if (ti >= nitems) break;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        const int nks = p.num_k_blocks / kCB;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait(full0 + 8 * stage, phase, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          // gathered A rows were written by cp.async, the generic proxy: this
          // CTA's rows became visible to this thread through the full
          // barrier, the fence orders them before the tensor core's reads;
          // CTA 1's forwarder fenced its own rows before signalling.  (The
          // fence over all state spaces costs about 1,000 cycles here, more
          // than the stage's MMAs.)
          if (kGather) fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(sA + stage * kA2);
          const uint32_t b0 = smem_u32(sB + stage * kB2);
#pragma unroll
          for (int kk = 0; kk < 4 * kCB; ++kk) {
            const uint32_t off = (kk >> 2) * kBlk + 32 * (kk & 3);
            mma2_bf16(d_tmem, sdesc_sw128(a0 + off), sdesc_sw128(b0 + off), idesc,
                      (ks | kk) != 0 ? 1u : 0u);
          }
          tc_commit2_mc(empty0 + 8 * stage, kBoth);
          issued = true;
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit2_mc(tfull0 + 8 * acc, kBoth);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // On the normal path both epilogues have waited for every accumulator,
      // so all MMAs are done.  After an abort, wait for the ones issued so far
      // before either CTA frees its TMEM or shared memory.
      if (!ok && issued) {
        tc_commit2(drain_bar);
        if (!mbar_wait(drain_bar, 0, limit, nullptr))
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
      }
    }
  } else if (kGather && warp == 1) {
    // ------------------------------------------------------------ forwarder
    // CTA 1: the rows its gather warps copied into stage s are handed to
    // CTA 0's MMA issuer by an asynchronous 4-byte store that completes
    // CTA 0's full[s]
    if (lane == 0) {
      const uint32_t full_r = cluster_map(full0, 0);
      const uint32_t pf_r = cluster_map(smem_u32(s_pf), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int ti = cl + it * ncl;
        if (ti >= nitems) break;
        const int nks = p.num_k_blocks / kCB;
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait(full0 + 8 * stage, phase, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
            ok = false;
            break;
          }
          // the gathered rows (generic proxy) before the partner's MMA reads
          fence_proxy_async_smem();
          st_async_tx4(pf_r + 4 * stage, static_cast<uint32_t>(ks), full_r + 8 * stage);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (kGather && warp >= 6) {
    // ------------------------------------------------------------ gather
    // As in the one-CTA GEMM: thread g copies 16-byte chunk g % 8 of rows
    // g / 8 + 16 i of the CTA's A tile, at the chunk position the 128-byte
    // swizzle gives, and arrives on every stage's full barrier through
    // cp.async.mbarrier.arrive.
    const int g = threadIdx.x - kThreads;
    const int c = g & 7, r0 = g >> 3;
    const int K = p.num_k_blocks * kBK2;
    const T *xg = static_cast<const T *>(p.x);
    constexpr int kChunk = 8;                                // bf16 per 16 bytes
    constexpr int kRowsPer = kBM / (kGatherThreads / 8);     // rows per thread: 8
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int ti = cl + it * ncl;
      if (ti >= nitems) break;
      const GemmTile tl = decode_2cta_item(gt, s_it, p, ti, rank, kOutCols, !kDual);
      const bool routed = tl.group < p.n_routed;
      const T *src[kRowsPer];
      int tok[kRowsPer];
      if (routed) gather_tokens<kRowsPer>(p, gt, tl, r0, tok);
#pragma unroll
      for (int i = 0; i < kRowsPer; ++i)
        src[i] = (routed && r0 + 16 * i < tl.rows)
                     ? xg + static_cast<long long>(tok[i]) * K + c * kChunk
                     : nullptr;
      const int nks = p.num_k_blocks / kCB;
      for (int ks = 0; ks < nks; ++ks) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t tile_dst = smem_u32(sA + stage * kA2);
#pragma unroll
        for (int h = 0; h < kCB; ++h)
#pragma unroll
          for (int i = 0; i < kRowsPer; ++i) {
            const int r = r0 + 16 * i;
            if (src[i] != nullptr)
              cp_async16(tile_dst + h * kBlk + r * 128 + ((c ^ (r & 7)) << 4),
                         src[i] + ks * kKS + h * kBK2);
          }
        cp_async_arrive(full0 + 8 * stage);
        if (++stage == kStages2) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;       // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;  // tile row == TMEM lane
    const uint32_t tempty_r = cluster_map(tempty0, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      const int ti = cl + it * ncl;
      if (ti >= nitems) break;
      const GemmTile tl = decode_2cta_item(gt, s_it, p, ti, rank, kOutCols, !kDual);
      const bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_EPI_TMEM_FULL);
        }
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(wq * 32) << 16);
      const bool valid = r < tl.rows;
      T *orow = reinterpret_cast<T *>(p.out) + static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
      if (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 32) {
          float gv[32], uv[32];
          tmem_ld32x2_sync(tb + c, tb + kBN / 2 + c, gv, uv);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) gv[i] = silu(gv[i]) * uv[i];
            store32<T>(orow + c, gv);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          float v[32];
          tmem_ld32_sync(tb + c, v);
          if (valid) store32<T>(orow + c, v);
        }
      }
      // this warp's reads of the accumulator are done: one arrival per warp
      // on CTA 0's barrier
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty_r + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // no MMA of the pair is in flight and no arrival on the partner is pending
  // once both CTAs are here; then both free the TMEM together
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(tmem, kTmemCols2);
  // after an abort, copies the partner issued before it stopped get time to land
  if (*abort_flag)
    for (int i = 0; i < 200; ++i) __nanosleep(1000);
}

template <int EPI>
cudaError_t gemm2sm_set_smem_attr() {
  return cudaFuncSetAttribute(gemm2sm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kGemmSmem);
}

template <int EPI>
cudaError_t launch_gemm2sm(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                           bool pdl) {
  if (grid <= 0) return cudaSuccess;
  if (grid & 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(gemm2sm_threads<EPI>());
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = 2;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gemm2sm_kernel<EPI>, maps.m[0], maps.m[1], maps.m[2], maps.m[3],
                            maps.m[4], maps.m[5], p);
}

int gemm2sm_clusters() {
  int best = 0;
  for (int e = 0; e < 2; ++e) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(e == 0 ? gemm2sm_threads<EPI_SWIGLU>() : gemm2sm_threads<EPI_STORE>());
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
        e == 0 ? cudaOccupancyMaxActiveClusters(&n, gemm2sm_kernel<EPI_SWIGLU>, &cfg)
               : cudaOccupancyMaxActiveClusters(&n, gemm2sm_kernel<EPI_STORE>, &cfg);
    if (err != cudaSuccess) return 0;
    best = e == 0 ? n : (n < best ? n : best);
  }
  return best;
}

template cudaError_t gemm2sm_set_smem_attr<EPI_SWIGLU>();
template cudaError_t gemm2sm_set_smem_attr<EPI_STORE>();
template cudaError_t launch_gemm2sm<EPI_SWIGLU>(const GemmMaps &, const GemmParams &, int,
                                                cudaStream_t, bool);
template cudaError_t launch_gemm2sm<EPI_STORE>(const GemmMaps &, const GemmParams &, int,
                                               cudaStream_t, bool);

}  // namespace moe
