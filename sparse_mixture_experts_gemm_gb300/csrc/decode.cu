// decode.cu -- batch-1 path: one token through one MoE layer as three
// weight-streaming kernels.  "Optimizing on-device inference for Apple
// Silicon", section "Decode: minimise bytes moved per token" (with one row
// the weights are read once per token, so bytes moved set the speed),
// section "Optimise the single-row weight path" (row-parallel GEMV: a group of
// 32 threads cooperates on each output while reading different parts of the
// weight row), section "Reduce intermediate traffic and dispatch traffic"
// (gate/up projections fused with the activation; down projection fused with
// the routing score and the shared-expert result) and section "Let independent
// GPU work overlap" (work that does not depend on a result does not wait for
// it).
//
//   A  decode_router : router logits (one warp per expert) and, in other CTAs,
//                      the shared expert's gate/up rows, which do not depend on
//                      the routing.  Also prefetches the shared down matrix
//                      into L2.
//   B  decode_gateup : every CTA takes the top-k of the logits and the softmax
//                      over the chosen ones itself (one warp, two redux.sync
//                      per choice), then one warp per (chosen expert, row) pair
//                      computes h = silu(g) * u; prefetches the k chosen down
//                      matrices into L2.
//   C  decode_down   : the same top-k, then one warp per output element: sum
//                      over the routed slots of w_j * (Wd_j row . h_j), plus the
//                      shared slot.
// The kernels are chained with programmatic dependent launch.  Each one loads
// the static weights it can before griddepcontrol.wait (which waits for the
// previous kernel and makes its writes visible) and reads data produced by
// earlier kernels only after it.  Kernel C reads the logits before its wait:
// kernel A wrote them and had completed before kernel B passed its own wait
// and let C start.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "internal.h"
#include "ptx.cuh"
#include "decode_common.cuh"

namespace moe {

// ---------------------------------------------------------------- A: router
// CTAs [0, ceil(E/8)): one warp per expert logit.  CTAs after them: one warp
// per shared-expert intermediate row f (gate row and up row together).
template <typename T>
__global__ void __launch_bounds__(256) decode_router_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const int n_rt = (a.E + 7) / 8;
  extern __shared__ uint4 xs_a[];  // the token, one copy per CTA
  const uint4 *xv = xs_a;
  if (static_cast<int>(blockIdx.x) >= n_rt) {
    const int c = blockIdx.x - n_rt;
    const int f = c * 8 + warp;
    if (threadIdx.x == 0) {
      long long lo, hi;
      split16(static_cast<long long>(a.d) * a.F * sizeof(T), gridDim.x - n_rt, c, lo, hi);
      if (hi > lo) prefetch_l2(reinterpret_cast<const char *>(a.sd) + lo, static_cast<uint32_t>(hi - lo));
    }
    const uint4 *rg = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.sg) +
                                                      static_cast<long long>(f) * a.d);
    const uint4 *ru = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.su) +
                                                      static_cast<long long>(f) * a.d);
    RowPre pg, pu;
    if (f < a.F) {
      row_prefetch(pg, rg, nvec, lane);
      row_prefetch(pu, ru, nvec, lane);
    }
    pdl_launch_dependents();  // kernel B reads nothing of ours before its wait
    pdl_wait();
    load_token(xs_a, a.x, nvec);
    if (f >= a.F) return;
    float g = warp_sum(row_dot_pre<T>(pg, rg, xv, nvec, lane));
    float u = warp_sum(row_dot_pre<T>(pu, ru, xv, nvec, lane));
    if (lane == 0) a.h[static_cast<long long>(a.k) * a.F + f] = g / (1.0f + __expf(-g)) * u;
    return;
  }
  const int e = blockIdx.x * 8 + warp;
  const uint4 *row = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.wr) +
                                                     static_cast<long long>(e) * a.d);
  RowPre pr;
  if (e < a.E) row_prefetch(pr, row, nvec, lane);
  pdl_launch_dependents();  // kernel B reads nothing of ours before its wait
  pdl_wait();
  load_token(xs_a, a.x, nvec);
  if (e < a.E) {
    const float acc = warp_sum(row_dot_pre<T>(pr, row, xv, nvec, lane));
    if (lane == 0) a.logits[e] = acc + (a.bias ? a.bias[e] : 0.0f);
  }
}

// ---------------------------------------------------------------- B: gate / up
// TMA-fed split of the chosen experts' gate/up rows: tile t covers rows
// [rb * kRB, (rb + 1) * kRB) of slot s = t / (F / kRB); the CTA streams the
// tile's gate and up rows through a 4-stage ring of boxes of kRB rows x 512
// bytes (one box per matrix per stage, no swizzle), warp w (of 8) keeps partial
// dot products of rows 4w .. 4w+3 in registers across the k-blocks and writes
// h = silu(g) * u at the end.  Warp 8 lane 0 issues the copies.
constexpr int kRB = 32;
constexpr int kBStages = 4;
constexpr int kBBox = kRB * 512;  // bytes of one box

template <typename T>
__global__ void __launch_bounds__(288, 1)
    decode_gateup_kernel(const __grid_constant__ CUtensorMap tmG,
                         const __grid_constant__ CUtensorMap tmU, const DecodeArgs a) {
  constexpr int KB = 512 / static_cast<int>(sizeof(T));  // elements per box row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[kBStages], empty[kBStages];
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = a.d / KB;
  const int nrb = a.F / kRB;
  const int ntile = a.k * nrb;
  const long long limit = MOE_WAIT_LIMIT_CYCLES;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 8);
    }
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmG);
    prefetch_tmap(&tmU);
  }
  pdl_wait();
  if (warp == 0) warp_topk(a.logits, a.E, a.k, lane, s_sel, s_selw);
  uint4 *xs = reinterpret_cast<uint4 *>(dsm + kBStages * 2 * kBBox);
  const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
  for (int i = threadIdx.x; i < a.d * static_cast<int>(sizeof(T)) / 16; i += blockDim.x)
    xs[i] = ld_cg16(xg + i);
  __syncthreads();
  pdl_launch_dependents();
  if (blockIdx.x == 0) write_routing(a, s_sel, s_selw, threadIdx.x);
  if (warp == 8) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < ntile; t += gridDim.x) {
      const int s = t / nrb, rb = t - (t / nrb) * nrb;
      const int row = s_sel[s] * a.F + rb * kRB;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, limit, nullptr)) {
          report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_DECODE * 100 + SITE_PRODUCER_EMPTY);
          return;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        const uint32_t dst = smem_u32(dsm + stage * 2 * kBBox);
        mbar_arrive_expect_tx(fb, 2 * kBBox);
        tma_load_2d(dst, &tmG, fb, kb * KB, row, pol);
        tma_load_2d(dst + kBBox, &tmU, fb, kb * KB, row, pol);
        if (++stage == kBStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    return;
  }
  int stage = 0;
  uint32_t phase = 0;
  for (int t = blockIdx.x; t < ntile; t += gridDim.x) {
    const int s = t / nrb, rb = t - (t / nrb) * nrb;
    float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kb = 0; kb < nkb; ++kb) {
      const bool ok = mbar_wait(smem_u32(&full[stage]), phase, limit, nullptr);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_DECODE * 100 + SITE_MMA_FULL);
        return;
      }
      const uint4 *bg = reinterpret_cast<const uint4 *>(dsm + stage * 2 * kBBox);
      const uint4 *bu = bg + kBBox / 16;
      const uint4 xv = xs[kb * 32 + lane];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = 4 * warp + q;
        g[q] += V16<T>::dot(bg[r * 32 + lane], xv);
        u[q] += V16<T>::dot(bu[r * 32 + lane], xv);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
      if (++stage == kBStages) {
        stage = 0;
        phase ^= 1;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float gg = warp_sum(g[q]), uu = warp_sum(u[q]);
      if (lane == 0)
        a.h[static_cast<long long>(s) * a.F + rb * kRB + 4 * warp + q] = gg / (1.0f + __expf(-gg)) * uu;
    }
  }
}

// ---------------------------------------------------------------- C: down
// One warp per output element i.  The weight vectors of all k + 1 slots (up
// to 64 per row, two per lane) are requested before the wait for h.
template <typename T>
__device__ __forceinline__ const uint4 *down_row(const DecodeArgs &a, const int *sel, int s, int i) {
  const T *row = (s < a.k) ? reinterpret_cast<const T *>(a.wd) +
                                 (static_cast<long long>(sel[s]) * a.d + i) * a.F
                           : reinterpret_cast<const T *>(a.sd) + static_cast<long long>(i) * a.F;
  return reinterpret_cast<const uint4 *>(row);
}

template <typename T>
__global__ void __launch_bounds__(256, 2) decode_down_kernel(const DecodeArgs a) {
  extern __shared__ float4 s_h4[];  // [(k + n_shared) * F / 4]
  constexpr int NV = V16<T>::N;
  constexpr int kSlots = kMaxTopK + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  const int nslot = a.k + a.n_shared;
  const int nvec = a.F / NV;
  // the next kernel only loads static weights before its own wait
  pdl_launch_dependents();
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  if (warp == 0) warp_topk(a.logits, a.E, a.k, lane, s_sel, s_selw);
  __syncthreads();
  uint4 wv[kSlots][2];
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    if (s < nslot && i < a.d) {
      const uint4 *rp = down_row<T>(a, s_sel, s, i);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int v = q * 32 + lane;
        if (v < nvec) wv[s][q] = ld_stream16(rp + v);
      }
    }
  }
  pdl_wait();

  const int total4 = nslot * a.F / 4;
  for (int base = threadIdx.x; base < total4; base += 256 * 8) {
    float4 t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = base + u * 256;
      if (q < total4) t[u] = ld_cg_f32x4(a.h + 4 * q);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = base + u * 256;
      if (q < total4) s_h4[q] = t[u];
    }
  }
  __syncthreads();
  if (i >= a.d) return;
  const float *s_h = reinterpret_cast<const float *>(s_h4);
  float acc = 0.0f;
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    if (s < nslot) {
      const float *hs = s_h + s * a.F;
      float part = 0.0f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int v = q * 32 + lane;
        if (v < nvec) part += V16<T>::dotf(wv[s][q], hs + v * NV);
      }
      if (nvec > 64) {
        const uint4 *rp = down_row<T>(a, s_sel, s, i);
        for (int v = 64 + lane; v < nvec; v += 32) part += V16<T>::dotf(ld_stream16(rp + v), hs + v * NV);
      }
      acc = fmaf(s < a.k ? s_selw[s] : 1.0f, part, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) V16<T>::store(a.out, i, acc);
}

namespace {
template <typename K>
cudaError_t launch_ex(K kern, int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                      const DecodeArgs &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}
}  // namespace

template <typename T>
cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int grid = (a.E + 7) / 8 + (a.n_shared ? (a.F + 7) / 8 : 0);
  return launch_ex(decode_router_kernel<T>, grid, 256, static_cast<size_t>(a.d) * sizeof(T), st,
                   pdl, a);
}
template <typename T>
cudaError_t launch_decode_gateup(const DecodeArgs &a, const CUtensorMap &tmG, const CUtensorMap &tmU,
                                 cudaStream_t st, bool pdl) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const int ntile = a.k * (a.F / kRB);
  const int grid = ntile < sms ? ntile : sms;
  const size_t smem = 1024 + kBStages * 2 * kBBox + static_cast<size_t>(a.d) * sizeof(T);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(288);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_gateup_kernel<T>, tmG, tmU, a);
}
template <typename T>
cudaError_t launch_decode_down(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const size_t smem = sizeof(float) * (a.k + a.n_shared) * a.F;
  return launch_ex(decode_down_kernel<T>, (a.d + 7) / 8, 256, smem, st, pdl, a);
}

// Dynamic shared memory limit of the decode kernels (set once per device): the
// down kernel keeps h of all slots in shared memory.
template <typename T>
cudaError_t decode_set_smem_attr() {
  const cudaError_t e0 = cudaFuncSetAttribute(decode_router_kernel<T>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              16384 * static_cast<int>(sizeof(T)));
  if (e0 != cudaSuccess) return e0;
  const cudaError_t e = cudaFuncSetAttribute(
      decode_down_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (kMaxTopK + 1) * 4096 * static_cast<int>(sizeof(float)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_gateup_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              1024 + kBStages * 2 * kBBox + 16384 * static_cast<int>(sizeof(T)));
}
template cudaError_t decode_set_smem_attr<__nv_bfloat16>();
template cudaError_t decode_set_smem_attr<float>();

template cudaError_t launch_decode_router<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<__nv_bfloat16>(const DecodeArgs &, const CUtensorMap &,
                                                         const CUtensorMap &, cudaStream_t, bool);
template cudaError_t launch_decode_down<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_router<float>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<float>(const DecodeArgs &, const CUtensorMap &,
                                                 const CUtensorMap &, cudaStream_t, bool);
template cudaError_t launch_decode_down<float>(const DecodeArgs &, cudaStream_t, bool);

}  // namespace moe
