// gemm.cu -- persistent grouped GEMM on the 5th-generation tensor cores.
//
// One kernel template serves the three contractions of the block:
//   EPI_ROUTER : logits = x . Wr^T for 128 tokens x 256 experts, with the
//                softmax / top-k / renormalisation fused into the epilogue and
//                each assignment's rank inside its expert group claimed with an
//                atomic on the per-expert histogram; the last CTA scans the
//                histogram into group offsets ("Optimizing on-device inference
//                for Apple Silicon", sections "Qwen creates three distinct
//                workload shapes" and "Keep expert routing on the GPU").
//   EPI_SWIGLU : for each expert group, gate and up projections of its rows in
//                one MMA (B tile = 128 gate rows over 128 up rows), epilogue
//                h = silu(gate) * up written once (section "Reduce
//                intermediate traffic and dispatch traffic": input
//                projections fused with the gated activation).  Routed A rows
//                come from the permuted copy Xp (one 128-row TMA box per
//                stage); the shared expert reads x itself.
//   EPI_STORE  : the down projection of each group's rows, stored per slot.
// The tiles of both grouped GEMMs are derived on the device from the group
// offsets the routing wrote (section "Keep expert routing on the GPU": the
// block map of fixed-size blocks the grouped GEMM processes), so no host
// synchronisation is needed: every CTA scans ceil(rows / 128) over the groups
// and maps a tile index to (group, m, n) by binary search.  Tiles of one group
// are ordered with m innermost, so the CTAs that share a weight block run side
// by side and the weight block is read from HBM once.
//
// CTA layout: 192 threads.  Warp 0 produces a 4-stage shared-memory ring of
// 128-byte-swizzled K-major tiles (lane 0 issues the TMA tile loads); warp 1
// allocates 512
// TMEM columns (two 128 x 256 fp32 accumulators) and its lane 0 issues
// tcgen05.mma (M = 128, N = 256, 32 bytes of K per instruction); warps 2-5
// drain a finished accumulator with tcgen05.ld while the MMA fills the other.
// The grid is persistent: CTA c takes tiles c, c + gridDim.x, ...
// Every wait is bounded; a wait that runs out records a timeout in the status
// word, raises a CTA-wide abort flag, drains what it issued and returns.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <typename T>
struct Tile {
  static constexpr int BK = 128 / sizeof(T);  // K elements per 128-byte row
  static constexpr int A_BYTES = kBM * 128;
  static constexpr int B_BYTES = kBN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
};


__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

template <typename T>
__device__ __forceinline__ void store32(T *dst, const float (&v)[32]);
template <>
__device__ __forceinline__ void store32<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&v)[32]) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[q * 8 + 2 * j], v[q * 8 + 2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t *>(&b);
    }
    d[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
template <>
__device__ __forceinline__ void store32<float>(float *dst, const float (&v)[32]) {
  float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Keep the 8 largest (value, index) pairs, sorted descending; a candidate
// equal to a kept value goes after it, so ties favour the lower index when
// candidates arrive in increasing index order.
__device__ __forceinline__ void topk_insert(float (&bv)[kMaxTopK], int (&bi)[kMaxTopK], float v,
                                            int e) {
  if (!(v > bv[kMaxTopK - 1])) return;
  bv[kMaxTopK - 1] = v;
  bi[kMaxTopK - 1] = e;
#pragma unroll
  for (int j = kMaxTopK - 1; j > 0; --j) {
    if (bv[j] > bv[j - 1]) {
      const float tv = bv[j];
      bv[j] = bv[j - 1];
      bv[j - 1] = tv;
      const int ti = bi[j];
      bi[j] = bi[j - 1];
      bi[j - 1] = ti;
    }
  }
}

// Group table built by every CTA of a grouped GEMM: s_off[g] = first slot of
// group g (g <= E), s_mt[g] = first M tile of group g (g <= E + 1; group E is
// the shared expert).
struct GroupTable {
  const int *off;
  const int *mt;
};

__device__ __forceinline__ GemmTile decode_tile(const GroupTable &gt, const GemmParams &p, int i,
                                                int n_cols, bool down) {
  const int E = p.n_routed;
  int lo = 0, hi = E;  // largest g with nt * mt[g] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.nt * gt.mt[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int mtg = gt.mt[g + 1] - gt.mt[g];
  const int local = i - p.nt * gt.mt[g];
  const int n = local / mtg, m = local - (local / mtg) * mtg;
  GemmTile t;
  t.group = g;
  t.n0 = n * n_cols;
  t.pad[0] = t.pad[1] = t.pad[2] = 0;
  if (g < E) {
    const int cnt = gt.off[g + 1] - gt.off[g];
    t.a_row = gt.off[g] + m * kBM;
    t.out_row = t.a_row;
    t.rows = min(kBM, cnt - m * kBM);
  } else {
    t.rows = min(kBM, p.T - m * kBM);
    t.out_row = p.A + m * kBM;
    t.a_row = down ? t.out_row : m * kBM;  // gate/up reads tokens in order
  }
  return t;
}

__device__ __forceinline__ GemmTile router_tile(const GemmParams &p, int i) {
  GemmTile t;
  t.group = 0;
  t.a_row = i * kBM;
  t.out_row = i * kBM;
  t.rows = min(kBM, p.T - i * kBM);
  t.n0 = 0;
  t.pad[0] = t.pad[1] = t.pad[2] = 0;
  return t;
}

}  // namespace

template <typename T, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const __grid_constant__ CUtensorMap tmB0s,
                const __grid_constant__ CUtensorMap tmB1s, const GemmParams p) {
  using C = Tile<T>;
  constexpr bool kRouter = (EPI == EPI_ROUTER);
  constexpr bool kDual = (EPI == EPI_SWIGLU);  // B = gate rows over up rows
  constexpr int kOutCols = (EPI == EPI_SWIGLU) ? kBN / 2 : kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages * C::A_BYTES;
  uint8_t *ctrl = sB + kStages * C::B_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 512);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 516);
  int *s_last = reinterpret_cast<int *>(ctrl + 520);
  int *s_off = reinterpret_cast<int *>(ctrl + 1536);        // [E + 1]
  int *s_mt = reinterpret_cast<int *>(ctrl + 1536 + 1040);  // [E + 2]

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t tfull0 = empty0 + 8 * kStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long limit = MOE_WAIT_LIMIT_CYCLES;
  const GroupTable gt{s_off, s_mt};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmA);
    if (!kRouter) prefetch_tmap(&tmAs);
    if (EPI == EPI_SWIGLU) {
      prefetch_tmap(&tmB1);
      prefetch_tmap(&tmB0s);
      prefetch_tmap(&tmB1s);
    }
    if (EPI == EPI_STORE) prefetch_tmap(&tmB0s);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  int ntiles;
  if (kRouter) {
    ntiles = p.ntiles_host;
  } else {
    // group table: offsets, M tiles per group, exclusive scan (warp 2)
    const int E = p.n_routed;
    for (int g = threadIdx.x; g <= E; g += blockDim.x) s_off[g] = p.offsets[g];
    __syncthreads();
    for (int g = threadIdx.x; g <= E; g += blockDim.x) {
      const int rows = g < E ? s_off[g + 1] - s_off[g] : (p.n_shared ? p.T : 0);
      s_mt[g] = (rows + kBM - 1) / kBM;
    }
    __syncthreads();
    if (warp == 2) {
      const int n = E + 1;
      const int per = (n + 31) / 32;
      int sum = 0;
      for (int q = 0; q < per; ++q) {
        const int i = lane * per + q;
        if (i < n) sum += s_mt[i];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - sum;
      for (int q = 0; q < per; ++q) {
        const int i = lane * per + q;
        if (i < n) {
          const int v = s_mt[i];
          s_mt[i] = run;
          run += v;
        }
      }
      if (lane == 31) s_mt[n] = incl;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (!kRouter) ntiles = p.nt * s_mt[p.n_routed + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    uint32_t pend_mask = 0, pend_phase = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntiles && ok; ti += gridDim.x) {
      const GemmTile tl = kRouter ? router_tile(p, ti) : decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool sh = !kRouter && tl.group >= p.n_routed;
      const CUtensorMap *ma = sh ? &tmAs : &tmA;
      const CUtensorMap *mb0 = sh ? &tmB0s : &tmB0;
      const CUtensorMap *mb1 = sh ? &tmB1s : &tmB1;
      const int brow = kRouter ? 0 : (sh ? tl.n0 : tl.group * p.b_rows_per_group + tl.n0);
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
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(a_dst, ma, fb, kx, tl.a_row, pol_a);
          if (kDual) {
            tma_load_2d(b_dst, mb0, fb, kx, brow, pol_w);
            tma_load_2d(b_dst + C::B_BYTES / 2, mb1, fb, kx, brow, pol_w);
          } else {
            tma_load_2d(b_dst, mb0, fb, kx, brow, kRouter ? pol_a : pol_w);
          }
        }
        pend_mask |= 1u << stage;
        pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // copies already issued must land before the CTA's shared memory goes away
      for (int s = 0; s < kStages; ++s)
        if (pend_mask & (1u << s))
          if (!mbar_wait(full0 + 8 * s, (pend_phase >> s) & 1, limit, nullptr))
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(kBM, kBN, MmaKind<T>::ab_format);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int ti = blockIdx.x; ti < ntiles && ok; ti += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            MmaKind<T>::mma(d_tmem, sdesc_sw128(a0 + 32 * kk), sdesc_sw128(b0 + 32 * kk), idesc,
                            (kb | kk) != 0 ? 1u : 0u);
          tc_commit(empty0 + 8 * stage);
          issued = true;
          if (++stage == kStages) {
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;       // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;  // tile row == TMEM lane
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
      const GemmTile tl = kRouter ? router_tile(p, ti) : decode_tile(gt, p, ti, kOutCols, !kDual);
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
          tmem + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(wq * 32) << 16);
      const bool valid = r < tl.rows;

      if (EPI == EPI_SWIGLU) {
        T *hrow = reinterpret_cast<T *>(p.out) + static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 32) {
          float g[32], u[32];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + kBN / 2 + c, u);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = silu(g[i]) * u[i];
            store32<T>(hrow + c, g);
          }
        }
      } else if (EPI == EPI_STORE) {
        T *yrow = reinterpret_cast<T *>(p.out) + static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          float v[32];
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
          if (valid) store32<T>(yrow + c, v);
        }
      } else {
        float bv[kMaxTopK];
        int bi[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          bv[j] = -INFINITY;
          bi[j] = 0;
        }
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          float v[32];
          tmem_ld32(tb + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = c + i;
            if (e < p.E) topk_insert(bv, bi, v[i] + (p.bias ? p.bias[e] : 0.0f), e);
          }
        }
        if (valid) {
          const int t = tl.a_row + r;
          float ex[kMaxTopK];
          float s = 0.0f;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            ex[j] = (j < p.k) ? expf(bv[j] - bv[0]) : 0.0f;
            s += ex[j];
          }
          const float inv_s = 1.0f / s;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            if (j < p.k) {
              const long long o = static_cast<long long>(t) * p.k + j;
              p.idx[o] = bi[j];
              p.w[o] = ex[j] * inv_s;
              const int rk = atomicAdd(p.counts + bi[j], 1);
              if (p.rank) p.rank[o] = rk;
            }
          }
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
  if (warp == 1) tmem_dealloc(tmem, 512);

  if (kRouter && p.offsets_out) {
    // the last CTA to finish turns the histogram into group offsets
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = (atomicAdd(p.done, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (*s_last && warp == 0) {
      __threadfence();
      const int E = p.E;
      const int per = (E + 31) / 32;
      int sum = 0;
      for (int q = 0; q < per; ++q) {
        const int e = lane * per + q;
        if (e < E) sum += __ldcg(p.counts + e);
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - sum;
      for (int q = 0; q < per; ++q) {
        const int e = lane * per + q;
        if (e < E) {
          p.offsets_out[e] = run;
          run += __ldcg(p.counts + e);
        }
      }
      if (lane == 31) p.offsets_out[E] = incl;
    }
  }
}

template <typename T, int EPI>
cudaError_t gemm_set_smem_attr() {
  return cudaFuncSetAttribute(gemm_kernel<T, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kGemmSmem);
}

template <typename T, int EPI>
cudaError_t launch_gemm(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  gemm_kernel<T, EPI><<<grid, kThreads, kGemmSmem, st>>>(maps.m[0], maps.m[1], maps.m[2], maps.m[3],
                                                          maps.m[4], maps.m[5], p);
  return cudaGetLastError();
}

template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_SWIGLU>();
template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_STORE>();
template cudaError_t gemm_set_smem_attr<__nv_bfloat16, EPI_ROUTER>();
template cudaError_t gemm_set_smem_attr<float, EPI_SWIGLU>();
template cudaError_t gemm_set_smem_attr<float, EPI_STORE>();
template cudaError_t launch_gemm<__nv_bfloat16, EPI_SWIGLU>(const GemmMaps &, const GemmParams &, int,
                                                             cudaStream_t);
template cudaError_t launch_gemm<__nv_bfloat16, EPI_STORE>(const GemmMaps &, const GemmParams &, int,
                                                            cudaStream_t);
template cudaError_t launch_gemm<__nv_bfloat16, EPI_ROUTER>(const GemmMaps &, const GemmParams &, int,
                                                             cudaStream_t);
template cudaError_t launch_gemm<float, EPI_SWIGLU>(const GemmMaps &, const GemmParams &, int,
                                                     cudaStream_t);
template cudaError_t launch_gemm<float, EPI_STORE>(const GemmMaps &, const GemmParams &, int,
                                                    cudaStream_t);

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
