// route.cu -- GPU-resident routing around the grouped GEMMs:
//   router_simt   fp32 router (one warp per token): logits, top-k, weights,
//                 and each assignment's rank inside its expert group, claimed
//                 with an atomic on the per-expert histogram;
//   offsets       exclusive prefix scan of the histogram into group offsets
//                 (the bf16 router does this in its last CTA instead);
//   place         slot = offset[expert] + rank for every assignment: the
//                 (token, choice) -> slot map read by the combine, and the
//                 slot -> token map the gate/up GEMM gathers rows with;
//   combine       out[t] = sum_j w[t][j] * Y[slot(t, j)] + Y_shared[t].
// Source: "Optimizing on-device inference for Apple Silicon", section "Keep
// expert routing on the GPU" (histogram, prefix scan into start offsets,
// scatter of rows into expert groups, all in one submission with no CPU
// synchronisation) and section "Reduce intermediate traffic and dispatch
// traffic" (routing score applied to the expert output, shared-expert result
// added).  The order of rows inside a group follows the atomics and may
// differ between runs; every output is independent of it, since each row of
// a group is computed on its own and the combine adds a token's terms in
// choice order.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Unpack a 16-byte vector into floats (8 bf16 or 4 fp32 values).
template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace

// ---------------------------------------------------------------- fp32 router
// One warp per token.  Logits in fp32 with lane-strided partial sums and a
// butterfly reduction; top-k by k rounds of warp arg-max (ties to the lower
// index); weights = softmax over the chosen logits.
template <typename T>
__global__ void __launch_bounds__(256) router_simt_kernel(const T *__restrict__ x,
                                                          const T *__restrict__ wr,
                                                          const float *__restrict__ bias, int T_tok,
                                                          int d, int E, int k, int32_t *idx,
                                                          float *w, int32_t *counts,
                                                          int32_t *rank) {
  extern __shared__ float s_logit[];  // [8 warps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T_tok) return;
  float *lg = s_logit + warp * E;
  const T *xr = x + static_cast<long long>(t) * d;
  for (int e = 0; e < E; ++e) {
    const T *wrow = wr + static_cast<long long>(e) * d;
    float acc = 0.0f;
    for (int i = lane; i < d; i += 32) acc = fmaf(to_f<T>(xr[i]), to_f<T>(wrow[i]), acc);
    acc = warp_sum(acc);
    if (lane == 0) lg[e] = acc + (bias ? bias[e] : 0.0f);
  }
  __syncwarp();
  float selv[kMaxTopK];
  int seli[kMaxTopK];
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = lg[e];
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
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
    if (bi >= E) bi = 0;  // only reachable with NaN logits; keeps every index in range
    selv[j] = bv;
    seli[j] = bi;
    __syncwarp();
    if (lane == 0) lg[bi] = -INFINITY;
    __syncwarp();
  }
  if (lane == 0) {
    float s = 0.0f;
    float ex[kMaxTopK];
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(selv[j] - selv[0]);
      s += ex[j];
    }
    for (int j = 0; j < k; ++j) {
      idx[static_cast<long long>(t) * k + j] = seli[j];
      w[static_cast<long long>(t) * k + j] = ex[j] / s;
      const int rk = atomicAdd(counts + seli[j], 1);
      if (rank) rank[static_cast<long long>(t) * k + j] = rk;
    }
  }
}

template <typename T>
cudaError_t launch_router_simt(const T *x, const T *wr, const float *bias, int T_tok, int d, int E,
                               int k, int32_t *idx, float *w, int32_t *counts, int32_t *rank,
                               cudaStream_t st) {
  const int grid = (T_tok + 7) / 8;
  const size_t smem = sizeof(float) * 8 * E;
  router_simt_kernel<T><<<grid, 256, smem, st>>>(x, wr, bias, T_tok, d, E, k, idx, w, counts, rank);
  return cudaGetLastError();
}
template cudaError_t launch_router_simt<float>(const float *, const float *, const float *, int, int,
                                               int, int, int32_t *, float *, int32_t *, int32_t *,
                                               cudaStream_t);
template cudaError_t launch_router_simt<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                                       const float *, int, int, int, int, int32_t *,
                                                       float *, int32_t *, int32_t *, cudaStream_t);

// ---------------------------------------------------------------- offsets
// offsets[e] = sum_{e' < e} counts[e'], offsets[E] = total; one warp.
// counts_out (may be null): each expert's count is added to it (the counts of
// a call's chunks sum up there).
__global__ void offsets_kernel(int32_t *counts, int E, int32_t *offsets, int32_t *counts_out,
                               int32_t *clear, int n_clear) {
  const int lane = threadIdx.x;
  const int per = (E + 31) / 32;
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int e = lane * per + q;
    if (e < E) sum += counts[e];
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
      offsets[e] = run;
      run += counts[e];
      if (counts_out) counts_out[e] += counts[e];
      counts[e] = 0;  // clear for the next call
    }
  }
  if (lane == 31) offsets[E] = incl;
  if (lane == 0)
    for (int q = 0; q < n_clear; ++q) clear[q * 32] = 0;
}

cudaError_t launch_offsets(int32_t *counts, int E, int32_t *offsets, int32_t *counts_out,
                           int32_t *clear, int n_clear, cudaStream_t st) {
  offsets_kernel<<<1, 32, 0, st>>>(counts, E, offsets, counts_out, clear, n_clear);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- place
// One thread per assignment i = t * k + j: slot = offsets[e] + rank, written
// over the rank in rank_inv[i]; perm[slot] = t names the token whose row the
// grouped gate/up GEMM gathers into that slot's tile row.
// idx, offsets and the ranks come from the router, the kernel this one
// waits for: read through L2 after the wait, never the non-coherent path.
__global__ void __launch_bounds__(256) place_kernel(const int32_t *idx, const int32_t *offsets,
                                                    int32_t *rank_inv, int32_t *perm, int A, int k,
                                                    int E, int *status) {
  // a programmatic dependent of the router: its outputs are read after the
  // wait; the grouped GEMM after it may then be scheduled
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= A) return;
  const int e = ld_cg_s32(idx + i);
  const int rank = ld_cg_s32(rank_inv + i);  // issued before e is used
  if (e < 0 || e >= E) {
    report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_PERMUTE * 100 + SITE_INDEX);
    return;
  }
  const int lo = ld_cg_s32(offsets + e), hi = ld_cg_s32(offsets + e + 1);
  const int slot = lo + rank;
  if (slot < lo || slot >= hi) {
    report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_PERMUTE * 100 + SITE_INDEX);
    return;
  }
  rank_inv[i] = slot;
  perm[slot] = i / k;
}

namespace {
cudaLaunchConfig_t pdl_config(int grid, int block, cudaStream_t st, bool pdl,
                              cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.stream = st;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}
}  // namespace

cudaError_t launch_place(const int32_t *idx, const int32_t *offsets, int32_t *rank_inv,
                         int32_t *perm, int A, int k, int E, int *status, cudaStream_t st,
                         bool pdl) {
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_config((A + 255) / 256, 256, st, pdl, &attr);
  return cudaLaunchKernelEx(&cfg, place_kernel, idx, offsets, rank_inv, perm, A, k, E, status);
}

// ---------------------------------------------------------------- combine
// One thread per 16-byte chunk of an output row; the k routed contributions
// are added in choice order (deterministic), then the shared expert's row.
// inv holds each assignment's slot (row of Y) or, when offsets is given, its
// rank inside its expert's group, to which the group's offset is added (the
// expert is idx's entry).  Y, the slots, ranks, offsets and weights were
// written by kernels earlier in the launch chain (Y by the one this kernel
// waits for): all are read after the wait (an asm with a memory clobber),
// never through the non-coherent path; Y without allocating in L1.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T *yp, const int32_t *inv,
                                                      const float *w, T *out, int T_tok, int k,
                                                      int d, int A_total, int n_shared,
                                                      int *status, const int32_t *idx,
                                                      const int32_t *offsets, int E,
                                                      int *clear_ctr) {
  // a programmatic dependent of the down GEMM (or GEMV): yp is read after
  // the wait
  pdl_wait();
  // the down GEMM has finished: its tile counter is free for the next call
  if (clear_ctr && blockIdx.x == 0 && threadIdx.x == 0) *clear_ctr = 0;
  constexpr int NV = Vec<T>::N;
  const int vpr = d / NV;  // vectors per row (a multiple of 32: a warp serves one token)
  // Grid-stride over the (token, vector) units: the grid is a few blocks per
  // SM (a ragged last wave of one-token blocks cost ~1 % of the step), and a
  // warp's 32 units always belong to one token.
  const long long total = static_cast<long long>(T_tok) * vpr;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; gid < total;
       gid += stride) {
    const int t = static_cast<int>(gid / vpr);
    const int c = static_cast<int>(gid % vpr);
    // the token's slots and weights: lanes j < k load slot j, lanes 16 + j
    // its weight, once per warp, and hand them to every lane; then every row
    // vector is requested, so all of the thread's loads are in flight
    // together; the sum keeps the fixed order
    int my_slot = 0;
    float my_w = 0.0f;
    bool bad = false;
    if (lane < k) {
      const long long o = static_cast<long long>(t) * k + lane;
      my_slot = inv[o];
      if (offsets) {
        const int e = idx[o];
        if (e < 0 || e >= E) bad = true;
        else my_slot += offsets[e];
      }
    }
    if (lane >= 16 && lane - 16 < k) my_w = w[static_cast<long long>(t) * k + lane - 16];
    int slot[kMaxTopK];
    float wt[kMaxTopK];
    bad = __any_sync(0xffffffffu, bad);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
      wt[j] = __shfl_sync(0xffffffffu, my_w, 16 + j);
      if (j < k) bad = bad || slot[j] < 0 || slot[j] >= A_total;
    }
    if (bad) {  // warp-uniform
      report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_COMBINE * 100 + SITE_INDEX);
      continue;
    }
    uint4 v[kMaxTopK + 1];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) v[j] = ld_na16(yp + static_cast<long long>(slot[j]) * d + c * NV);
    if (n_shared) v[kMaxTopK] = ld_na16(yp + static_cast<long long>(A_total + t) * d + c * NV);
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        float f[NV];
        Vec<T>::unpack(v[j], f);
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = fmaf(wt[j], f[i], acc[i]);
      }
    }
    if (n_shared) {
      float f[NV];
      Vec<T>::unpack(v[kMaxTopK], f);
#pragma unroll
      for (int i = 0; i < NV; ++i) acc[i] += f[i];
    }
    *reinterpret_cast<uint4 *>(out + static_cast<long long>(t) * d + c * NV) = Vec<T>::pack(acc);
  }
}

template <typename T>
cudaError_t launch_combine(const T *yp, const int32_t *inv, const float *w, T *out, int T_tok,
                           int k, int d, int A_total, int n_shared, int *status, int num_sms,
                           cudaStream_t st, bool pdl, const int32_t *idx, const int32_t *offsets,
                           int E, int *clear_ctr) {
  constexpr long long kBlocksPerSm = 4;  // 1,024 threads per SM, 8 loads of 16 bytes each in flight
  const long long threads = static_cast<long long>(T_tok) * (d / Vec<T>::N);
  const long long want = (threads + 255) / 256;
  const int grid = static_cast<int>(want < kBlocksPerSm * num_sms ? want : kBlocksPerSm * num_sms);
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_config(grid, 256, st, pdl, &attr);
  return cudaLaunchKernelEx(&cfg, combine_kernel<T>, yp, inv, w, out, T_tok, k, d, A_total,
                            n_shared, status, idx, offsets, E, clear_ctr);
}
template cudaError_t launch_combine<float>(const float *, const int32_t *, const float *, float *, int,
                                           int, int, int, int, int *, int, cudaStream_t, bool,
                                           const int32_t *, const int32_t *, int, int *);
template cudaError_t launch_combine<__nv_bfloat16>(const __nv_bfloat16 *, const int32_t *,
                                                   const float *, __nv_bfloat16 *, int, int, int, int,
                                                   int, int *, int, cudaStream_t, bool,
                                                   const int32_t *, const int32_t *, int, int *);

}  // namespace moe
