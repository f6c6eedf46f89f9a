// router.cu -- the router of the grouped path for bf16 tokens: logits, top-k,
// routing weights, ranks, per-expert token lists and histogram in one launch
// ("Optimizing on-device inference for Apple Silicon", sections "Qwen
// creates three distinct workload shapes": 256 experts, eight kept per
// token, and "Keep expert routing on the GPU": selection and the per-expert
// histogram stay on the device).
//
// One thread-block cluster of four CTAs per tile of 128 tokens.  CTA r
// multiplies the tokens' columns [r d/4, (r+1) d/4) with the same columns of
// all router rows on the tensor cores (M = 128 tokens, N = 256 experts, fp32
// accumulator in TMEM), so each CTA streams a quarter of the tile's tokens
// and of the router weights.  The four partial logit blocks are then
// exchanged through distributed shared memory: CTA r receives the partials
// of tokens 32 r .. 32 r + 31 from the other three CTAs into its (now idle)
// operand ring, each 4 KB block staged by the sending warp and moved by one
// bulk copy that completes a byte-counting barrier of the receiver; it sums
// the four partials in a fixed order (deterministic), adds the router bias and
// takes each token's top-k with eight threads per token: each sorts its 32
// experts' (logit, expert) keys in groups of 8 with bitonic networks and
// keeps the best 8, then three pairwise exchanges merge the lists.  The thread that ends with a token's list
// writes its experts and weights and claims each assignment's rank inside
// its expert group with one atomic per expert among the lanes of a warp.
//
// Warp 0 issues the TMA loads, warp 1 the MMAs, warps 2-9 drain TMEM into the
// owners' partial buffers and then select.  Every wait is bounded; a CTA that
// gave up tells the other CTAs of its cluster at the cluster barrier before
// the exchange, and then none of them exchanges or writes.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRSplit = 4;                    // CTAs per cluster: quarters of d
constexpr int kRN = 256;                      // experts per MMA (E <= 256)
constexpr int kRStages = 4;
constexpr int kRABytes = kBM * 128;           // 128 tokens x 64 columns
constexpr int kRBBytes = kRN * 128;           // 256 router rows x 64 columns
constexpr int kRStageBytes = kRABytes + kRBBytes;
constexpr int kRRows = kBM / kRSplit;         // tokens finished per CTA
// partial logits of one source CTA and 32 columns for the 32 tokens a CTA
// finishes: [32 rows][32 floats], 4 KB, the unit of the exchange
constexpr int kRBlock = kRRows * 32 * 4;
constexpr int kRRecvBytes = kRSplit * (kRN / 32) * kRBlock;  // [4 src][8 column blocks]
constexpr int kRStageSlot = kRBlock;                          // two per epilogue warp
static_assert(kRRecvBytes + 16 * kRStageSlot <= kRStages * kRStageBytes,
              "the exchange reuses the operand ring");
constexpr int kRThreads = 320;
constexpr int kREpiWarps = 8;
constexpr int kRCtrl = 2048;
constexpr int kRSmem = kRStages * kRStageBytes + 1024 + kRCtrl;

// Inside a block [32 rows][32 floats] of column block c, 16-byte chunk u of
// row j is kept at chunk u ^ ((j ^ c) % 8): a warp writing one chunk of all
// its rows, and the eight threads of a token reading chunk u of blocks
// c = 0..7, both spread over all 32 banks.
__device__ __forceinline__ int blk_off(int c, int j, int u) {
  return c * kRBlock + j * 128 + ((u ^ ((j ^ c) & 7)) << 4);
}

// Bulk copy of `bytes` of this CTA's shared memory into cluster CTA `rank`
// at the offset of `dst`, completing its barrier at the offset of `bar`.
__device__ __forceinline__ void bulk_s2s(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar,
                                         uint32_t rank) {
  uint32_t rdst, rbar;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rdst) : "r"(dst), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(bar), "r"(rank));
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(rdst), "r"(src), "r"(bytes), "r"(rbar)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the bulk copies this thread issued have read their source (all, or all
// but the last one)
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_but1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_s32(uint32_t local, uint32_t rank, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// A logit and its expert as one 64-bit key whose unsigned order is the
// selection order: larger logit first, then (for equal logits) the lower
// expert.  The float is mapped to an unsigned integer of the same order
// (sign bit set: all bits flipped; clear: sign bit set) above 255 - e, so a
// logit and its expert always move together.  Adding +0 first turns -0 into
// +0 (they compare equal as floats).
__device__ __forceinline__ unsigned long long logit_key(float v, int e) {
  const unsigned u = __float_as_uint(v + 0.0f);
  const unsigned o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | static_cast<unsigned>(255 - e);
}
__device__ __forceinline__ float key_logit(unsigned long long k) {
  const unsigned o = static_cast<unsigned>(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ int key_expert(unsigned long long k) {
  return 255 - static_cast<int>(k & 0xFFu);
}

// a >= b afterwards
__device__ __forceinline__ void cx(unsigned long long &a, unsigned long long &b) {
  const bool sw = a < b;
  const unsigned long long hi = sw ? b : a, lo = sw ? a : b;
  a = hi;
  b = lo;
}
// Sort 8 keys descending (bitonic network: 24 independent-per-stage
// compare-exchanges).
__device__ __forceinline__ void sort8(unsigned long long (&a)[8]) {
#pragma unroll
  for (int k = 2; k <= 8; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cx(a[i], a[l]);
          else cx(a[l], a[i]);
        }
      }
}
// a := the 8 largest of a and b (both sorted descending), sorted descending:
// the element-wise larger of a[i] and b[7 - i] are those 8 (a bitonic
// sequence), which three stages of compare-exchanges sort.
__device__ __forceinline__ void merge8(unsigned long long (&a)[8], const unsigned long long (&b)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = a[i] > b[7 - i] ? a[i] : b[7 - i];
#pragma unroll
  for (int j = 4; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int l = i ^ j;
      if (l > i) cx(a[i], a[l]);
    }
}

}  // namespace

__global__ void __launch_bounds__(kRThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kRStages * kRABytes;
  // after the MMAs: partials received [4 src][8 column blocks] at the
  // ring's start, then one staging block per epilogue warp
  uint8_t *recv = smem;
  uint8_t *stage_blk = smem + kRRecvBytes;
  uint8_t *ctrl = smem + kRStages * kRStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 256);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 260);
  volatile int *s_err = reinterpret_cast<volatile int *>(ctrl + 264);  // set by any cluster CTA
  float *s_bias = reinterpret_cast<float *>(ctrl + 1024);               // [256]

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kRStages;
  const uint32_t tfull = empty0 + 8 * kRStages;
  const uint32_t rbar = tfull + 8;  // the other CTAs' partials have landed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int tile = static_cast<int>(blockIdx.x) / kRSplit;
  const int nkb = a.d / (kRSplit * 64);  // K blocks of 64 columns per CTA
  const int kx0 = static_cast<int>(rank) * (a.d / kRSplit);
  const long long limit = MOE_WAIT_LIMIT_CYCLES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(rbar, 1);
    *abort_flag = 0;
    *s_err = 0;
    fence_mbar_init();
    // three CTAs each send this CTA 8 blocks
    mbar_arrive_expect_tx(rbar, (kRSplit - 1) * (kRN / 32) * kRBlock);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kRN);
    tmem_relinquish();
  }
  if (threadIdx.x >= 64)
    for (int e = threadIdx.x - 64; e < kRN; e += kRThreads - 64)
      s_bias[e] = e < a.E ? (a.bias ? a.bias[e] : 0.0f) : -INFINITY;
  // the tokens may be the previous kernel's output
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  // every CTA's error flag is initialised before any CTA may set it
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // tokens and router rows are read again
      uint32_t pend = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kRStages;
        if (kb >= kRStages && !mbar_wait(empty0 + 8 * s, ((kb / kRStages) - 1) & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        const int kx = kx0 + kb * 64;
        mbar_arrive_expect_tx(fb, kRStageBytes);
        tma_load_2d(smem_u32(sA + s * kRABytes), &tmX, fb, kx, tile * kBM, pol);
        tma_load_2d(smem_u32(sB + s * kRBBytes), &tmW, fb, kx, 0, pol);
        pend = kb;
      }
      if (!ok) {
        *abort_flag = 1;
        report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_ROUTER * 100 + SITE_PRODUCER_EMPTY);
        // copies already issued must land before the ring is reused
        for (int kb = pend > kRStages ? pend - kRStages + 1 : 0; kb <= static_cast<int>(pend); ++kb)
          if (!mbar_wait(full0 + 8 * (kb % kRStages), (kb / kRStages) & 1, limit, nullptr))
            report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_ROUTER * 100 + SITE_DRAIN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(kBM, kRN, MmaKind<__nv_bfloat16>::ab_format);
      bool issued = false;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kRStages;
        if (!mbar_wait(full0 + 8 * s, (kb / kRStages) & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kRABytes);
        const uint32_t b0 = smem_u32(sB + s * kRBBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          MmaKind<__nv_bfloat16>::mma(tmem, sdesc_sw128(a0 + 32 * kk), sdesc_sw128(b0 + 32 * kk),
                                      idesc, (kb | kk) != 0 ? 1u : 0u);
        tc_commit(empty0 + 8 * s);
        issued = true;
      }
      if (!ok) {
        *abort_flag = 1;
        report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_ROUTER * 100 + SITE_MMA_FULL);
      }
      // the epilogue waits for this arrival; after an abort it still comes
      // once the MMAs issued so far are done
      if (issued || ok) tc_commit(tfull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const bool w_ok = mbar_wait(tfull, 0, limit, abort_flag);
    if (!__all_sync(0xffffffffu, w_ok)) {
      ok = false;
      if (lane == 0) report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_ROUTER * 100 + SITE_EPI_TMEM_FULL);
    }
    tc_fence_after();
  }
  // a CTA that gave up tells every CTA of the cluster (its partials would be
  // missing or its ring still filling); the barrier also orders each CTA's
  // last MMA before any partial lands in its ring
  if (!ok || *abort_flag)
    for (uint32_t r = 0; r < kRSplit; ++r) st_cluster_s32(smem_u32(const_cast<int *>(s_err)), r, 1);
  __syncwarp();
  cluster_sync_all();
  const bool go = *s_err == 0;

  bool have = go;
  if (go && warp >= 2) {
    // TMEM lanes 32 (warp % 4) .. + 31 (tokens) belong to owner CTA warp % 4;
    // warps 2-5 hold column blocks 0-3, warps 6-9 blocks 4-7.  A block for
    // this CTA goes straight into its receive buffer; one for another CTA is
    // staged and sent by one bulk copy into that CTA's buffer.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * h + cc;
      float v[32];
      tmem_ld32_sync(tmem + (static_cast<uint32_t>(q * 32) << 16) + 32 * c, v);
      const bool mine = q == static_cast<int>(rank);
      // two staging slots per warp, used in turn
      uint8_t *slot = stage_blk + ((warp - 2) * 2 + (cc & 1)) * kRStageSlot;
      uint8_t *dst = mine ? recv + rank * (kRN / 32) * kRBlock : slot - c * kRBlock;
      if (!mine && cc >= 2) {
        // the copy that used this slot two blocks ago has read it
        if (lane == 0) bulk_wait_read_but1();
        __syncwarp();
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<float4 *>(dst + blk_off(c, lane, u)) =
            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      if (!mine) {
        fence_proxy_async_smem();  // the copy engine reads what the threads wrote
        __syncwarp();
        if (lane == 0)
          bulk_s2s(smem_u32(recv + (rank * (kRN / 32) + c) * kRBlock), smem_u32(slot), kRBlock,
                   rbar, q);
      }
    }
    if (lane == 0) bulk_wait_read();
    // this CTA's own blocks, written by all eight warps, then the others'
    named_bar_sync(1, kREpiWarps * 32);
    const bool r_ok = mbar_wait(rbar, 0, limit, nullptr);
    if (!__all_sync(0xffffffffu, r_ok)) {
      have = false;
      if (lane == 0) report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_ROUTER * 100 + SITE_DRAIN);
    }
  }

  if (have && warp >= 2) {
    // ------------------------------------------------------------ select
    // thread (j, s): token j of this CTA's 32, experts 32 s .. 32 s + 31
    const int t_loc = (warp - 2) * 32 + lane;
    const int j = t_loc >> 3, s = t_loc & 7;
    // each thread: the sorted top 8 of its 32 experts, in four groups of 8
    unsigned long long top[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      unsigned long long grp[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = 2 * g + h;
        const int off = blk_off(s, j, u);
        float4 acc = *reinterpret_cast<const float4 *>(recv + off);
#pragma unroll
        for (int src = 1; src < kRSplit; ++src) {
          const float4 p =
              *reinterpret_cast<const float4 *>(recv + src * (kRN / 32) * kRBlock + off);
          acc.x += p.x;
          acc.y += p.y;
          acc.z += p.z;
          acc.w += p.w;
        }
        const int e0 = 32 * s + 4 * u;
        grp[4 * h] = logit_key(acc.x + s_bias[e0], e0);
        grp[4 * h + 1] = logit_key(acc.y + s_bias[e0 + 1], e0 + 1);
        grp[4 * h + 2] = logit_key(acc.z + s_bias[e0 + 2], e0 + 2);
        grp[4 * h + 3] = logit_key(acc.w + s_bias[e0 + 3], e0 + 3);
      }
      sort8(grp);
      if (g == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) top[i] = grp[i];
      } else {
        merge8(top, grp);
      }
    }
    // the eight threads of a token exchange and merge their lists pairwise;
    // both threads of a pair end with the same list
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
      unsigned long long other[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) other[i] = __shfl_xor_sync(0xffffffffu, top[i], m);
      merge8(top, other);
    }
    float bv[kMaxTopK];
    int bi[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) {
      bv[i] = key_logit(top[i]);
      bi[i] = key_expert(top[i]);
    }
    const int t = tile * kBM + static_cast<int>(rank) * kRRows + j;
    if (s == 0 && t < a.T) {
      float ex[kMaxTopK];
      float sum = 0.0f;
#pragma unroll
      for (int i = 0; i < kMaxTopK; ++i) {
        ex[i] = (i < a.k) ? expf(bv[i] - bv[0]) : 0.0f;
        sum += ex[i];
      }
      const float inv_s = 1.0f / sum;
      // lanes of this warp that chose the same expert share one atomic on
      // its counter; all k atomics are issued before any result is used
      const unsigned act = __activemask();
      unsigned peers[kMaxTopK];
      int base[kMaxTopK];
#pragma unroll
      for (int i = 0; i < kMaxTopK; ++i) {
        base[i] = 0;
        peers[i] = 0;
        if (i < a.k) {
          const long long o = static_cast<long long>(t) * a.k + i;
          a.idx[o] = bi[i];
          a.w[o] = ex[i] * inv_s;
          peers[i] = __match_any_sync(act, bi[i]);
          if (lane == __ffs(peers[i]) - 1) {
            if (a.counts_direct) atomicAdd(a.counts_direct + bi[i], __popc(peers[i]));
            else base[i] = atomicAdd(a.counts + static_cast<long long>(bi[i]) * kCountStride,
                                     __popc(peers[i]));
          }
        }
      }
      if (!a.counts_direct) {
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i) {
          if (i < a.k) {
            const int rk = __shfl_sync(act, base[i], __ffs(peers[i]) - 1) +
                           __popc(peers[i] & ((1u << lane) - 1u));
            a.rank[static_cast<long long>(t) * a.k + i] = rk;
            // the token goes to place rk of its expert's list
            a.list[static_cast<long long>(bi[i]) * a.list_stride + rk] = t;
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kRN);
}

cudaError_t router_set_attr() {
  return cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
}

cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const RouterArgs &a,
                          cudaStream_t st, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  const int ntiles = (a.T + kBM - 1) / kBM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kRSplit * ntiles);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of whatever ran before: the prologue (barriers,
  // TMEM, the bias) overlaps it, the tokens are read after the wait
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, router_kernel, tm_x, tm_w, a);
}

}  // namespace moe
