// router.cu -- the router of the grouped path for bf16 tokens: logits, top-k,
// routing weights, ranks, per-expert token lists and histogram in one launch
// ("Optimizing on-device inference for Apple Silicon", sections "Qwen
// creates three distinct workload shapes": 256 experts, eight kept per
// token, and "Keep expert routing on the GPU": selection and the per-expert
// histogram stay on the device).
//
// One thread-block cluster of S CTAs per tile of 128 tokens (S = 4, or 2 for
// chunks whose 4-CTA clusters would not all be resident at once).  The
// tokens' columns are cut into quarters of d; CTA r multiplies quarters
// r 4/S .. (r + 1) 4/S - 1 with the same columns of all router rows on the
// tensor cores (M = 128 tokens, N = 256 experts), one fp32 accumulator per
// quarter in TMEM, so each CTA streams 1/S of the tile's tokens and of the
// router weights.  The partial logit blocks are then exchanged through
// distributed shared memory: CTA r receives the partials of tokens
// 128 r / S .. 128 (r + 1) / S - 1 from the other CTAs into its (now idle)
// operand ring, each 4 KB block staged by the sending warp and moved by one
// bulk copy that completes a byte-counting barrier of the receiver.  The
// logit is (q0 + q1) + (q2 + q3) over the quarter partials q, in fp32 and in
// this order with either S (with S = 2 each CTA adds its two quarters before
// sending), so the result does not depend on S; the receiver adds the
// router bias and takes each token's top-k with eight threads per token
// (32 tokens at a time): each sorts its 32
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

constexpr int kRN = 256;                      // experts per MMA (E <= 256)
constexpr int kRStages = 4;
constexpr int kRABytes = kBM * 128;           // 128 tokens x 64 columns
constexpr int kRBBytes = kRN * 128;           // 256 router rows x 64 columns
constexpr int kRStageBytes = kRABytes + kRBBytes;
// partial logits of one source CTA and 32 columns for 32 of the tokens a
// CTA finishes: [32 rows][32 floats], 4 KB, the unit of the exchange
constexpr int kRBlock = 32 * 32 * 4;
// [S sources][128 / S / 32 row blocks][8 column blocks]: 128 KB for either S
constexpr int kRRecvBytes = (kBM / 32) * (kRN / 32) * kRBlock;
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

template <int S>
__global__ void __launch_bounds__(kRThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const RouterArgs a) {
  constexpr int kRows = kBM / S;            // tokens this CTA finishes
  constexpr int kRB = kRows / 32;           // in row blocks of 32
  constexpr int kQ = 4 / S;                 // quarters of d this CTA multiplies
  constexpr uint32_t kCols = kQ * kRN;      // one accumulator per quarter
  static_assert(S == 2 || S == 4, "clusters of two or four CTAs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kRStages * kRABytes;
  // after the MMAs: partials received [S src][kRB row blocks][8 column
  // blocks] at the ring's start, then two staging blocks per epilogue warp
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
  const int tile = static_cast<int>(blockIdx.x) / S;
  const int nkb = a.d / (S * 64);  // K blocks of 64 columns per CTA
  const int nkq = a.d / (4 * 64);  // K blocks per quarter of d
  const int kx0 = static_cast<int>(rank) * (a.d / S);
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
    // every other CTA sends this CTA 8 column blocks per row block
    mbar_arrive_expect_tx(rbar, (S - 1) * kRB * (kRN / 32) * kRBlock);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kCols);
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
        // quarter kb / nkq of d goes to its own accumulator
        const int qk = kb % nkq;
        const uint32_t d_tmem = tmem + static_cast<uint32_t>((kb / nkq) * kRN);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          MmaKind<__nv_bfloat16>::mma(d_tmem, sdesc_sw128(a0 + 32 * kk), sdesc_sw128(b0 + 32 * kk),
                                      idesc, (qk | kk) != 0 ? 1u : 0u);
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
    for (uint32_t r = 0; r < S; ++r) st_cluster_s32(smem_u32(const_cast<int *>(s_err)), r, 1);
  __syncwarp();
  cluster_sync_all();
  const bool go = *s_err == 0;

  bool have = go;
  if (go && warp >= 2) {
    // TMEM lanes 32 (warp % 4) .. + 31 (tokens) are row block rb of owner
    // CTA (warp % 4) / kRB; warps 2-5 hold column blocks 0-3, warps 6-9
    // blocks 4-7.  With two quarters per CTA their partials are added here
    // (q0 + q1, or q2 + q3).  A block for this CTA goes straight into its
    // receive buffer; one for another CTA is staged and sent by one bulk copy
    // into that CTA's buffer, at [source = this CTA][rb][column block].
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int owner = q / kRB, rb = q % kRB;
    uint8_t *const my_blocks = recv + (rank * kRB + rb) * (kRN / 32) * kRBlock;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c = 4 * h + cc;
      const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + 32 * c;
      float v[32];
      if (kQ == 2) {
        float v1[32];
        tmem_ld32x2_sync(ta, ta + kRN, v, v1);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += v1[i];
      } else {
        tmem_ld32_sync(ta, v);
      }
      const bool mine = owner == static_cast<int>(rank);
      // two staging slots per warp, used in turn
      uint8_t *slot = stage_blk + ((warp - 2) * 2 + (cc & 1)) * kRStageSlot;
      uint8_t *dst = mine ? my_blocks : slot - c * kRBlock;
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
          bulk_s2s(smem_u32(my_blocks + c * kRBlock), smem_u32(slot), kRBlock, rbar,
                   static_cast<uint32_t>(owner));
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

  // ------------------------------------------------------------ select
  // thread (j, s): token j of row block rb of this CTA's tokens, experts
  // 32 s .. 32 s + 31
#pragma unroll 1
  for (int rb = 0; rb < kRB && have && warp >= 2; ++rb) {
    const int t_loc = (warp - 2) * 32 + lane;
    const int j = t_loc >> 3, s = t_loc & 7;
    // the partials of source CTA src for row block rb
    auto part = [&](int src, int off) {
      return *reinterpret_cast<const float4 *>(recv + (src * kRB + rb) * (kRN / 32) * kRBlock + off);
    };
    // each thread: the sorted top 8 of its 32 experts, in four groups of 8
    unsigned long long top[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      unsigned long long grp[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = 2 * g + h;
        const int off = blk_off(s, j, u);
        // (q0 + q1) + (q2 + q3): with S = 4 the sources are the quarters,
        // with S = 2 each source already holds its two quarters' sum
        float4 acc = part(0, off);
        const float4 p1 = part(1, off);
        acc.x += p1.x;
        acc.y += p1.y;
        acc.z += p1.z;
        acc.w += p1.w;
        if (S == 4) {
          float4 p23 = part(2, off);
          const float4 p3 = part(3, off);
          p23.x += p3.x;
          p23.y += p3.y;
          p23.z += p3.z;
          p23.w += p3.w;
          acc.x += p23.x;
          acc.y += p23.y;
          acc.z += p23.z;
          acc.w += p23.w;
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
    const int t = tile * kBM + static_cast<int>(rank) * kRows + rb * 32 + j;
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
  if (warp == 1) tmem_dealloc(tmem, kCols);
}

cudaError_t router_set_attr() {
  const cudaError_t e =
      cudaFuncSetAttribute(router_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
}

cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const RouterArgs &a,
                          cudaStream_t st, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  if (a.split != 2 && a.split != 4) return cudaErrorInvalidValue;
  const int ntiles = (a.T + kBM - 1) / kBM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.split * ntiles);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of whatever ran before: the prologue (barriers,
  // TMEM, the bias) overlaps it, the tokens are read after the wait
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return a.split == 2 ? cudaLaunchKernelEx(&cfg, router_kernel<2>, tm_x, tm_w, a)
                      : cudaLaunchKernelEx(&cfg, router_kernel<4>, tm_x, tm_w, a);
}

}  // namespace moe
