// decode.cu -- batch-1 path: one token through one MoE layer as three
// weight-streaming kernels.  "Optimizing on-device inference for Apple
// Silicon", section "Decode: minimise bytes moved per token" (with one row the
// weights are read once per token, so bytes moved set the speed), section
// "Optimise the single-row weight path" (row-parallel GEMV: a group of 32
// threads cooperates on each output while reading different parts of the
// weight row) and section "Reduce intermediate traffic and dispatch traffic"
// (gate/up projections fused with the activation; down projection fused with
// the routing score and the shared-expert result).
//
//   decode_router : one warp per expert logit (16-byte streaming loads of the
//                   router row, shuffle reduction); the last CTA to finish
//                   takes the top-k and the softmax over the chosen logits.
//   decode_gateup : one warp per (expert slot, intermediate row): gate and up
//                   rows streamed together, h = silu(g) * u.
//   decode_down   : one warp per output element: sum over the k routed slots
//                   of w_j * (Wd_j row . h_j), plus the shared slot.
// Each kernel may be launched with programmatic dependent launch: it calls
// griddepcontrol.wait before reading anything the previous kernel wrote and
// then lets its own dependents start.
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
  // weights (8 bf16) against 8 fp32 values
  __device__ __forceinline__ static float dotf(const uint4 &w, const float *h) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(a[i] << 16), h[2 * i], s);
      s = fmaf(__uint_as_float(a[i] & 0xFFFF0000u), h[2 * i + 1], s);
    }
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
    float s = __uint_as_float(w.x) * h[0];
    s = fmaf(__uint_as_float(w.y), h[1], s);
    s = fmaf(__uint_as_float(w.z), h[2], s);
    s = fmaf(__uint_as_float(w.w), h[3], s);
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

// dot(row, x) over nvec 16-byte vectors; lanes stride the row, 8 loads in
// flight per lane per round.
template <typename T>
__device__ __forceinline__ float row_dot(const uint4 *row, const uint4 *xv, int nvec, int lane) {
  float acc = 0.0f;
  for (int base = 0; base < nvec; base += 32 * 8) {
    uint4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) wv[u] = ld_stream16(row + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) acc += V16<T>::dot(wv[u], __ldg(xv + i));
    }
  }
  return acc;
}

}  // namespace

// ---------------------------------------------------------------- router
template <typename T>
__global__ void __launch_bounds__(256) decode_router_kernel(const DecodeArgs a) {
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  pdl_wait();
  pdl_launch_dependents();
  if (e < a.E) {
    const uint4 *row = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.wr) +
                                                       static_cast<long long>(e) * a.d);
    float acc = row_dot<T>(row, reinterpret_cast<const uint4 *>(a.x), nvec, lane);
    acc = warp_sum(acc);
    if (lane == 0) a.logits[e] = acc + (a.bias ? a.bias[e] : 0.0f);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1) ? 1 : 0;
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

// ---------------------------------------------------------------- gate / up
template <typename T>
__global__ void __launch_bounds__(256) decode_gateup_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + warp;
  const int s = gw / a.F, f = gw % a.F;
  const int nslot = a.k + a.n_shared;
  pdl_wait();
  pdl_launch_dependents();
  if (s >= nslot) return;
  const T *wg, *wu;
  if (s < a.k) {
    const int e = a.sel[s];
    wg = reinterpret_cast<const T *>(a.wg) + (static_cast<long long>(e) * a.F + f) * a.d;
    wu = reinterpret_cast<const T *>(a.wu) + (static_cast<long long>(e) * a.F + f) * a.d;
  } else {
    wg = reinterpret_cast<const T *>(a.sg) + static_cast<long long>(f) * a.d;
    wu = reinterpret_cast<const T *>(a.su) + static_cast<long long>(f) * a.d;
  }
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const uint4 *xv = reinterpret_cast<const uint4 *>(a.x);
  const uint4 *rg = reinterpret_cast<const uint4 *>(wg);
  const uint4 *ru = reinterpret_cast<const uint4 *>(wu);
  float g = 0.0f, u = 0.0f;
  for (int base = 0; base < nvec; base += 32 * 8) {
    uint4 vg[8], vu[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = base + q * 32 + lane;
      if (i < nvec) {
        vg[q] = ld_stream16(rg + i);
        vu[q] = ld_stream16(ru + i);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = base + q * 32 + lane;
      if (i < nvec) {
        const uint4 xx = __ldg(xv + i);
        g += V16<T>::dot(vg[q], xx);
        u += V16<T>::dot(vu[q], xx);
      }
    }
  }
  g = warp_sum(g);
  u = warp_sum(u);
  if (lane == 0) a.h[static_cast<long long>(s) * a.F + f] = g / (1.0f + __expf(-g)) * u;
}

// ---------------------------------------------------------------- down
template <typename T>
__global__ void __launch_bounds__(256) decode_down_kernel(const DecodeArgs a) {
  extern __shared__ float s_h[];  // [(k + n_shared)][F]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;  // output element
  const int nslot = a.k + a.n_shared;
  pdl_wait();
  pdl_launch_dependents();
  for (int q = threadIdx.x; q < nslot * a.F; q += blockDim.x) s_h[q] = a.h[q];
  __syncthreads();
  if (i >= a.d) return;
  constexpr int NV = V16<T>::N;
  const int nvec = a.F / NV;
  float acc = 0.0f;
  for (int s = 0; s < nslot; ++s) {
    const T *row;
    float ws;
    if (s < a.k) {
      row = reinterpret_cast<const T *>(a.wd) + (static_cast<long long>(a.sel[s]) * a.d + i) * a.F;
      ws = a.selw[s];
    } else {
      row = reinterpret_cast<const T *>(a.sd) + static_cast<long long>(i) * a.F;
      ws = 1.0f;
    }
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    const float *hs = s_h + s * a.F;
    float part = 0.0f;
    for (int base = 0; base < nvec; base += 32 * 4) {
      uint4 wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = base + q * 32 + lane;
        if (v < nvec) wv[q] = ld_stream16(rv + v);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = base + q * 32 + lane;
        if (v < nvec) part += V16<T>::dotf(wv[q], hs + v * NV);
      }
    }
    acc = fmaf(ws, part, acc);
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
  return launch_ex(decode_router_kernel<T>, (a.E + 7) / 8, 256, 0, st, pdl, a);
}
template <typename T>
cudaError_t launch_decode_gateup(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int warps = (a.k + a.n_shared) * a.F;
  return launch_ex(decode_gateup_kernel<T>, (warps + 7) / 8, 256, 0, st, pdl, a);
}
template <typename T>
cudaError_t launch_decode_down(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const size_t smem = sizeof(float) * (a.k + a.n_shared) * a.F;
  return launch_ex(decode_down_kernel<T>, (a.d + 7) / 8, 256, smem, st, pdl, a);
}

template <typename T>
cudaError_t decode_set_smem_attr(int bytes) {
  return cudaFuncSetAttribute(decode_down_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              bytes);
}
template cudaError_t decode_set_smem_attr<__nv_bfloat16>(int);
template cudaError_t decode_set_smem_attr<float>(int);

template <typename T>
cudaError_t decode_get_smem_attr(int *bytes) {
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, decode_down_kernel<T>);
  if (e == cudaSuccess) *bytes = fa.maxDynamicSharedSizeBytes;
  return e;
}
template cudaError_t decode_get_smem_attr<__nv_bfloat16>(int *);
template cudaError_t decode_get_smem_attr<float>(int *);

template cudaError_t launch_decode_router<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_down<__nv_bfloat16>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_router<float>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_gateup<float>(const DecodeArgs &, cudaStream_t, bool);
template cudaError_t launch_decode_down<float>(const DecodeArgs &, cudaStream_t, bool);

}  // namespace moe
