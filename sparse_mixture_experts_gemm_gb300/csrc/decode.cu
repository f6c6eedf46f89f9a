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
//                      the routing; the last router CTA takes the top-k and
//                      the softmax over the chosen logits.  Also prefetches the
//                      shared down matrix into L2.
//   B  decode_gateup : gate/up rows of the k chosen experts (one warp per row
//                      pair), h = silu(g) * u; prefetches the k chosen down
//                      matrices into L2.
//   C  decode_down   : one warp per output element: sum over the routed slots
//                      of w_j * (Wd_j row . h_j), plus the shared slot.
// The kernels are chained with programmatic dependent launch.  Each one loads
// the static weights it can before griddepcontrol.wait (which waits for the
// previous kernel and makes its writes visible) and reads data produced by
// earlier kernels only after it.  Kernel C reads the expert choice before its
// wait: it was written by kernel A, which had completed before kernel B passed
// its own wait and let C start.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <typename T>
struct V16;
template <>
struct V16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static float dot(const uint4 &w, const uint4 &x) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
    const uint32_t b[4] = {x.x, x.y, x.z, x.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16), s);
      s = fmaf(__uint_as_float(a[i] & 0xFFFF0000u), __uint_as_float(b[i] & 0xFFFF0000u), s);
    }
    return s;
  }
  // weights (8 bf16) against 8 fp32 values (h 16-byte aligned, two 16-byte reads)
  __device__ __forceinline__ static float dotf(const uint4 &w, const float *h) {
    const float4 h0 = reinterpret_cast<const float4 *>(h)[0];
    const float4 h1 = reinterpret_cast<const float4 *>(h)[1];
    float s = __uint_as_float(w.x << 16) * h0.x;
    s = fmaf(__uint_as_float(w.x & 0xFFFF0000u), h0.y, s);
    s = fmaf(__uint_as_float(w.y << 16), h0.z, s);
    s = fmaf(__uint_as_float(w.y & 0xFFFF0000u), h0.w, s);
    s = fmaf(__uint_as_float(w.z << 16), h1.x, s);
    s = fmaf(__uint_as_float(w.z & 0xFFFF0000u), h1.y, s);
    s = fmaf(__uint_as_float(w.w << 16), h1.z, s);
    s = fmaf(__uint_as_float(w.w & 0xFFFF0000u), h1.w, s);
    return s;
  }
  __device__ __forceinline__ static void store(void *out, int i, float v) {
    reinterpret_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
  }
};
template <>
struct V16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static float dot(const uint4 &w, const uint4 &x) {
    float s = __uint_as_float(w.x) * __uint_as_float(x.x);
    s = fmaf(__uint_as_float(w.y), __uint_as_float(x.y), s);
    s = fmaf(__uint_as_float(w.z), __uint_as_float(x.z), s);
    s = fmaf(__uint_as_float(w.w), __uint_as_float(x.w), s);
    return s;
  }
  __device__ __forceinline__ static float dotf(const uint4 &w, const float *h) {
    const float4 hv = *reinterpret_cast<const float4 *>(h);
    float s = __uint_as_float(w.x) * hv.x;
    s = fmaf(__uint_as_float(w.y), hv.y, s);
    s = fmaf(__uint_as_float(w.z), hv.z, s);
    s = fmaf(__uint_as_float(w.w), hv.w, s);
    return s;
  }
  __device__ __forceinline__ static void store(void *out, int i, float v) {
    reinterpret_cast<float *>(out)[i] = v;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Up to kPre 16-byte vectors of one row held in registers per lane: vector
// u * 32 + lane for u < kPre.  Loads issued before a dependency wait overlap
// the previous kernel's tail.
constexpr int kPre = 8;

struct RowPre {
  uint4 v[kPre];
};

__device__ __forceinline__ void row_prefetch(RowPre &r, const uint4 *row, int nvec, int lane) {
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = u * 32 + lane;
    if (i < nvec) r.v[u] = ld_stream16(row + i);
  }
}

// dot(row, x) for a row whose first 32 * kPre vectors are in r; the rest (rows
// longer than 256 vectors) are streamed here.
template <typename T>
__device__ __forceinline__ float row_dot_pre(const RowPre &r, const uint4 *row, const uint4 *xv,
                                             int nvec, int lane) {
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = u * 32 + lane;
    if (i < nvec) acc += V16<T>::dot(r.v[u], __ldg(xv + i));
  }
  for (int i = 32 * kPre + lane; i < nvec; i += 32) acc += V16<T>::dot(ld_stream16(row + i), __ldg(xv + i));
  return acc;
}

// Bring [p, p + bytes) into L2 without waiting; bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// This CTA's share [lo, hi) of a byte range split over n CTAs in 16-byte units.
__device__ __forceinline__ void split16(long long total, int n, int j, long long &lo,
                                        long long &hi) {
  const long long units = total / 16;
  lo = units * j / n * 16;
  hi = units * (j + 1) / n * 16;
}

}  // namespace

// ---------------------------------------------------------------- A: router
// CTAs [0, ceil(E/8)): one warp per expert logit.  CTAs after them: one warp
// per shared-expert intermediate row f (gate row and up row together).
template <typename T>
__global__ void __launch_bounds__(256) decode_router_kernel(const DecodeArgs a) {
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const int n_rt = (a.E + 7) / 8;
  const uint4 *xv = reinterpret_cast<const uint4 *>(a.x);
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
    pdl_wait();
    pdl_launch_dependents();
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
  pdl_wait();
  pdl_launch_dependents();
  if (e < a.E) {
    const float acc = warp_sum(row_dot_pre<T>(pr, row, xv, nvec, lane));
    if (lane == 0) a.logits[e] = acc + (a.bias ? a.bias[e] : 0.0f);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == static_cast<unsigned>(n_rt - 1)) ? 1 : 0;
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  // last CTA: top-k over the E logits, 8 per lane at most (E <= 256)
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ee = lane + 32 * i;
    v[i] = (ee < a.E) ? __ldcg(a.logits + ee) : -INFINITY;
  }
  float selv[kMaxTopK];
  int seli[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    selv[j] = -INFINITY;
    seli[j] = 0;
    if (j < a.k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ee = lane + 32 * i;
        if (v[i] > bv || (v[i] == bv && ee < bi)) {
          bv = v[i];
          bi = ee;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi >= a.E) bi = 0;  // only reachable with NaN logits; keeps every index in range
      selv[j] = bv;
      seli[j] = bi;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == bi) v[i] = -INFINITY;
    }
  }
  if (lane == 0) {
    float ex[kMaxTopK];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      ex[j] = (j < a.k) ? expf(selv[j] - selv[0]) : 0.0f;
      s += ex[j];
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < a.k) {
        a.sel[j] = seli[j];
        a.selw[j] = ex[j] / s;
      }
    *a.counter = 0u;
  }
}


// ---------------------------------------------------------------- B: gate / up
// One warp per (routed slot s, intermediate row f); thread 0 of each CTA
// prefetches its share of the k chosen down matrices into L2 for kernel C.
template <typename T>
__global__ void __launch_bounds__(256) decode_gateup_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + warp;
  const int s = gw / a.F, f = gw - (gw / a.F) * a.F;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    const long long per = static_cast<long long>(a.d) * a.F * sizeof(T);
    long long lo, hi;
    split16(per * a.k, gridDim.x, blockIdx.x, lo, hi);
    while (lo < hi) {
      const int j = static_cast<int>(lo / per);
      const long long off = lo - j * per;
      const long long n = (hi - lo) < (per - off) ? (hi - lo) : (per - off);
      prefetch_l2(reinterpret_cast<const char *>(a.wd) + a.sel[j] * per + off,
                  static_cast<uint32_t>(n));
      lo += n;
    }
  }
  if (s >= a.k) return;
  const int e = a.sel[s];
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const long long r = (static_cast<long long>(e) * a.F + f) * a.d;
  const uint4 *rg = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.wg) + r);
  const uint4 *ru = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.wu) + r);
  RowPre pg, pu;
  row_prefetch(pg, rg, nvec, lane);
  row_prefetch(pu, ru, nvec, lane);
  const uint4 *xv = reinterpret_cast<const uint4 *>(a.x);
  const float g = warp_sum(row_dot_pre<T>(pg, rg, xv, nvec, lane));
  const float u = warp_sum(row_dot_pre<T>(pu, ru, xv, nvec, lane));
  if (lane == 0) a.h[static_cast<long long>(s) * a.F + f] = g / (1.0f + __expf(-g)) * u;
}

// ---------------------------------------------------------------- C: down
// One warp per output element i.  The weight vectors of all k + 1 slots (up
// to 64 per row, two per lane) are requested before the wait for h.
template <typename T>
__device__ __forceinline__ const uint4 *down_row(const DecodeArgs &a, int s, int i) {
  const T *row = (s < a.k) ? reinterpret_cast<const T *>(a.wd) +
                                 (static_cast<long long>(a.sel[s]) * a.d + i) * a.F
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
  uint4 wv[kSlots][2];
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    if (s < nslot && i < a.d) {
      const uint4 *rp = down_row<T>(a, s, i);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int v = q * 32 + lane;
        if (v < nvec) wv[s][q] = ld_stream16(rp + v);
      }
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  const int total4 = nslot * a.F / 4;
  const float4 *hg = reinterpret_cast<const float4 *>(a.h);
  for (int base = threadIdx.x; base < total4; base += 256 * 8) {
    float4 t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = base + u * 256;
      if (q < total4) t[u] = __ldcg(hg + q);
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
        const uint4 *rp = down_row<T>(a, s, i);
        for (int v = 64 + lane; v < nvec; v += 32) part += V16<T>::dotf(ld_stream16(rp + v), hs + v * NV);
      }
      acc = fmaf(s < a.k ? a.selw[s] : 1.0f, part, acc);
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
  return launch_ex(decode_router_kernel<T>, grid, 256, 0, st, pdl, a);
}
template <typename T>
cudaError_t launch_decode_gateup(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  return launch_ex(decode_gateup_kernel<T>, (a.k * a.F + 7) / 8, 256, 0, st, pdl, a);
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
  return cudaFuncSetAttribute(decode_down_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (kMaxTopK + 1) * 4096 * static_cast<int>(sizeof(float)));
}
template cudaError_t decode_set_smem_attr<__nv_bfloat16>();
template cudaError_t decode_set_smem_attr<float>();

template cudaError_t launch_decode_router<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_down<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_router<float>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<float>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_down<float>(const DecodeArgs &, cudaStream_t, bool);

}  // namespace moe
