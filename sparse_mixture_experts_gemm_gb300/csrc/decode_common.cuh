// decode_common.cuh -- helpers shared by the batch-1 kernels: 16-byte weight
// vectors against the token, warp reductions, and the warp-wide top-k with
// softmax over the chosen logits.
#pragma once
#include <cuda_bf16.h>

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

// Order-preserving map of a float to an unsigned key (larger float, larger
// key; -0.0 sorts just below +0.0) and its inverse.
__device__ __forceinline__ unsigned fkey(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// One warp: the k largest of E <= 256 logits given as order-preserving keys
// (key[i] of expert lane + 32 i, 0 past E), ties to the lower index, and
// their softmax weights, into s_sel / s_selw (shared memory).  A round takes
// the warp maximum of the keys, then the lowest expert index holding it, with
// one redux.sync each.
__device__ __forceinline__ void topk_from_keys(unsigned (&key)[8], int E, int k, int lane,
                                               int *s_sel, float *s_selw) {
  float selv[kMaxTopK];
  int seli[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    selv[j] = -INFINITY;
    seli[j] = 0;
    if (j < k) {
      unsigned lm = key[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) lm = max(lm, key[i]);
      const unsigned gm = __reduce_max_sync(0xffffffffu, lm);
      int le = 0x7fffffff;
#pragma unroll
      for (int i = 7; i >= 0; --i)
        if (key[i] == gm) le = lane + 32 * i;
      int ge = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(le)));
      if (ge >= E) ge = 0;  // only reachable with NaN logits; keeps every index in range
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i == ge) key[i] = 0u;
      selv[j] = fkey_inv(gm);
      seli[j] = ge;
    }
  }
  if (lane == 0) {
    float ex[kMaxTopK];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      ex[j] = (j < k) ? expf(selv[j] - selv[0]) : 0.0f;
      sum += ex[j];
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        s_sel[j] = seli[j];
        s_selw[j] = ex[j] / sum;
      }
  }
}

// The same from logits in global memory (L2 reads: written by another kernel
// or CTA).
__device__ __forceinline__ void warp_topk(const float *logits, int E, int k, int lane, int *s_sel,
                                          float *s_selw) {
  unsigned key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? fkey(ld_cg_f32(logits + e)) : 0u;
  }
  topk_from_keys(key, E, k, lane, s_sel, s_selw);
}

// Thread j < k: entry j of the layer's routing (the choice the kernels use)
// into the caller's buffers, if it asked for them.  The k experts are
// distinct, so no two threads touch the same count.
__device__ __forceinline__ void write_routing(const DecodeArgs &a, const int *sel,
                                              const float *selw, int j) {
  if (j >= a.k) return;
  if (a.sel_idx) a.sel_idx[j] = sel[j];
  if (a.sel_w) a.sel_w[j] = selw[j];
  if (a.sel_counts) a.sel_counts[sel[j]] += 1;
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
// longer than 256 vectors) are streamed here.  xv: the token in shared memory.
template <typename T>
__device__ __forceinline__ float row_dot_pre(const RowPre &r, const uint4 *row, const uint4 *xv,
                                             int nvec, int lane) {
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = u * 32 + lane;
    if (i < nvec) acc += V16<T>::dot(r.v[u], xv[i]);
  }
  for (int i = 32 * kPre + lane; i < nvec; i += 32) acc += V16<T>::dot(ld_stream16(row + i), xv[i]);
  return acc;
}

// The token into shared memory (all threads; L2 reads, written by the kernel
// this one waited for), once per CTA rather than once per warp.
__device__ __forceinline__ void load_token(uint4 *xs, const void *x, int nvec) {
  const uint4 *xg = static_cast<const uint4 *>(x);
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) xs[i] = ld_cg16(xg + i);
  __syncthreads();
}

}  // namespace
}  // namespace moe
