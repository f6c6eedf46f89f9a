// route.cu -- GPU-resident routing around the grouped GEMMs:
//   router_simt   fp32 router (one warp per token): logits, top-k, weights,
//                 per-128-token-block expert histogram;
//   permute       expert totals, exclusive prefix scan into group offsets, the
//                 per-expert tile lists ("block map") of both grouped GEMMs,
//                 and the stable token -> slot permutation;
//   gather        copies each assignment's token row into its expert group;
//   combine       out[t] = sum_j w[t][j] * Y[slot(t, j)] + Y_shared[t].
// Source: "Optimizing on-device inference for Apple Silicon", section "Keep
// expert routing on the GPU" (histogram, prefix scan into start offsets,
// scatter of rows into expert groups, block map of fixed-size blocks, all in
// one submission with no CPU synchronisation) and section "Reduce
// intermediate traffic and dispatch traffic" (routing score applied to the
// expert output, shared-expert result added).
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

// Inclusive scan of one int per thread over a 256-thread block.
__device__ __forceinline__ int block_incl_scan_256(int v, int *sbuf) {
  const int tid = threadIdx.x;
  sbuf[tid] = v;
  __syncthreads();
#pragma unroll
  for (int o = 1; o < 256; o <<= 1) {
    const int add = tid >= o ? sbuf[tid - o] : 0;
    __syncthreads();
    sbuf[tid] += add;
    __syncthreads();
  }
  const int r = sbuf[tid];
  __syncthreads();
  return r;
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
                                                          float *w, int32_t *blkcnt) {
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
      atomicAdd(blkcnt + static_cast<long long>(t / kBM) * E + seli[j], 1);
    }
  }
}

template <typename T>
cudaError_t launch_router_simt(const T *x, const T *wr, const float *bias, int T_tok, int d, int E,
                               int k, int32_t *idx, float *w, int32_t *blkcnt, int *status,
                               cudaStream_t st) {
  (void)status;
  const int grid = (T_tok + 7) / 8;
  const size_t smem = sizeof(float) * 8 * E;
  router_simt_kernel<T><<<grid, 256, smem, st>>>(x, wr, bias, T_tok, d, E, k, idx, w, blkcnt);
  return cudaGetLastError();
}
template cudaError_t launch_router_simt<float>(const float *, const float *, const float *, int, int,
                                               int, int, int32_t *, float *, int32_t *, int *,
                                               cudaStream_t);
template cudaError_t launch_router_simt<__nv_bfloat16>(const __nv_bfloat16 *, const __nv_bfloat16 *,
                                                       const float *, int, int, int, int, int32_t *,
                                                       float *, int32_t *, int *, cudaStream_t);

// ---------------------------------------------------------------- permute
// Grid: one CTA of 256 threads per 128-token block; thread e owns expert e.
// Every CTA recomputes the expert totals and its own block's prefix from the
// per-block histogram, so no grid-wide synchronisation is needed.  CTA 0 also
// writes counts, offsets and both tile lists; tiles of one expert are ordered
// (n, m) with m innermost so tiles sharing a weight block run side by side.
__global__ void __launch_bounds__(256) permute_kernel(
    const int32_t *__restrict__ idx, const int32_t *__restrict__ blkcnt, int T_tok, int k, int E,
    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, GemmTile *tiles1,
    GemmTile *tiles2, int *ntiles, int nt1, int nt2, int n_shared, int build_tiles, int *status) {
  __shared__ int s_scan[256];
  __shared__ int s_idx[kBM * kMaxTopK];
  const int e = threadIdx.x;
  const int b = blockIdx.x;
  const int nblk = (T_tok + kBM - 1) / kBM;
  int tot = 0, pre = 0;
  if (e < E) {
    for (int bb = 0; bb < nblk; ++bb) {
      const int c = blkcnt[static_cast<long long>(bb) * E + e];
      tot += c;
      if (bb < b) pre += c;
    }
  }
  const int off = block_incl_scan_256(tot, s_scan) - tot;
  const int A_total = T_tok * k;

  if (b == 0) {
    if (e < E) {
      if (counts) counts[e] = tot;
      if (offsets) offsets[e] = off;
      if (offsets && e == E - 1) offsets[E] = off + tot;
    }
    if (build_tiles) {
      const int mt = (e < E) ? (tot + kBM - 1) / kBM : 0;
      const int mt_off = block_incl_scan_256(mt, s_scan) - mt;
      for (int n = 0; n < nt1; ++n)
        for (int m = 0; m < mt; ++m) {
          GemmTile t;
          t.group = e;
          t.a_row = off + m * kBM;
          t.out_row = off + m * kBM;
          t.rows = min(kBM, tot - m * kBM);
          t.n0 = n * kBM;
          t.pad[0] = t.pad[1] = t.pad[2] = 0;
          tiles1[nt1 * mt_off + n * mt + m] = t;
        }
      for (int n = 0; n < nt2; ++n)
        for (int m = 0; m < mt; ++m) {
          GemmTile t;
          t.group = e;
          t.a_row = off + m * kBM;
          t.out_row = off + m * kBM;
          t.rows = min(kBM, tot - m * kBM);
          t.n0 = n * kBN;
          t.pad[0] = t.pad[1] = t.pad[2] = 0;
          tiles2[nt2 * mt_off + n * mt + m] = t;
        }
      // total routed M-tiles = last thread's inclusive value
      __shared__ int s_total_mt;
      if (e == 255) s_total_mt = mt_off + mt;
      __syncthreads();
      const int tmt = s_total_mt;
      const int mts = n_shared ? (T_tok + kBM - 1) / kBM : 0;
      for (int q = e; q < nt1 * mts; q += 256) {
        const int n = q / mts, m = q % mts;
        GemmTile t;
        t.group = E;
        t.a_row = m * kBM;                // rows of x
        t.out_row = A_total + m * kBM;    // shared rows follow the routed ones in H
        t.rows = min(kBM, T_tok - m * kBM);
        t.n0 = n * kBM;
        t.pad[0] = t.pad[1] = t.pad[2] = 0;
        tiles1[nt1 * tmt + q] = t;
      }
      for (int q = e; q < nt2 * mts; q += 256) {
        const int n = q / mts, m = q % mts;
        GemmTile t;
        t.group = E;
        t.a_row = A_total + m * kBM;
        t.out_row = A_total + m * kBM;
        t.rows = min(kBM, T_tok - m * kBM);
        t.n0 = n * kBN;
        t.pad[0] = t.pad[1] = t.pad[2] = 0;
        tiles2[nt2 * tmt + q] = t;
      }
      if (e == 0) {
        ntiles[0] = nt1 * (tmt + mts);
        ntiles[1] = nt2 * (tmt + mts);
      }
    }
  }

  // stable placement of this block's assignments: token order, then choice order
  const int t0 = b * kBM;
  const int nt = min(kBM, T_tok - t0);
  for (int i = e; i < nt * k; i += 256) s_idx[i] = idx[static_cast<long long>(t0) * k + i];
  __syncthreads();
  if (e < E) {
    int slot = off + pre;
    for (int i = 0; i < nt * k; ++i) {
      if (s_idx[i] == e) {
        perm[slot] = t0 + i / k;
        inv[static_cast<long long>(t0) * k + i] = slot;
        ++slot;
      }
    }
  }
  for (int i = e; i < nt * k; i += 256)
    if (s_idx[i] < 0 || s_idx[i] >= E)
      report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_PERMUTE * 100 + SITE_INDEX);
}

cudaError_t launch_permute(const int32_t *idx, const int32_t *blkcnt, int T_tok, int k, int E,
                           int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                           GemmTile *tiles1, GemmTile *tiles2, int *ntiles, int nt1, int nt2,
                           int n_shared, int build_tiles, int *status, cudaStream_t st) {
  const int nblk = (T_tok + kBM - 1) / kBM;
  permute_kernel<<<nblk, 256, 0, st>>>(idx, blkcnt, T_tok, k, E, counts, offsets, perm, inv, tiles1,
                                       tiles2, ntiles, nt1, nt2, n_shared, build_tiles, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- gather
// One warp per assignment slot: Xp[slot] = x[perm[slot]], 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256) gather_kernel(const T *__restrict__ x,
                                                     const int32_t *__restrict__ perm, T *xp, int A,
                                                     int d, int T_tok, int *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= A) return;
  const int t = perm[row];
  if (t < 0 || t >= T_tok) {
    if (lane == 0) report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_PERMUTE * 100 + SITE_INDEX);
    return;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(x + static_cast<long long>(t) * d);
  uint4 *dst = reinterpret_cast<uint4 *>(xp + static_cast<long long>(row) * d);
  const int nvec = d * static_cast<int>(sizeof(T)) / 16;
#pragma unroll 8
  for (int i = lane; i < nvec; i += 32) dst[i] = src[i];
}

template <typename T>
cudaError_t launch_gather(const T *x, const int32_t *perm, T *xp, int A, int d, int T_tok,
                          int *status, cudaStream_t st) {
  const int grid = (A + 7) / 8;
  gather_kernel<T><<<grid, 256, 0, st>>>(x, perm, xp, A, d, T_tok, status);
  return cudaGetLastError();
}
template cudaError_t launch_gather<float>(const float *, const int32_t *, float *, int, int, int,
                                          int *, cudaStream_t);
template cudaError_t launch_gather<__nv_bfloat16>(const __nv_bfloat16 *, const int32_t *,
                                                  __nv_bfloat16 *, int, int, int, int *,
                                                  cudaStream_t);

// ---------------------------------------------------------------- combine
// One thread per 16-byte chunk of an output row; the k routed contributions
// are added in choice order (deterministic), then the shared expert's row.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T *__restrict__ yp,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ w, T *out, int T_tok,
                                                      int k, int d, int A_total, int n_shared,
                                                      int *status) {
  constexpr int NV = Vec<T>::N;
  const int vpr = d / NV;  // vectors per row
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int t = static_cast<int>(gid / vpr);
  const int c = static_cast<int>(gid % vpr);
  if (t >= T_tok) return;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int slot = inv[static_cast<long long>(t) * k + j];
    if (slot < 0 || slot >= A_total) {
      report_error(status, MOE_ERR_DEVICE_BOUNDS, KID_COMBINE * 100 + SITE_INDEX);
      return;
    }
    const float wt = w[static_cast<long long>(t) * k + j];
    float f[NV];
    Vec<T>::unpack(*reinterpret_cast<const uint4 *>(yp + static_cast<long long>(slot) * d + c * NV), f);
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = fmaf(wt, f[i], acc[i]);
  }
  if (n_shared) {
    float f[NV];
    Vec<T>::unpack(
        *reinterpret_cast<const uint4 *>(yp + static_cast<long long>(A_total + t) * d + c * NV), f);
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] += f[i];
  }
  *reinterpret_cast<uint4 *>(out + static_cast<long long>(t) * d + c * NV) = Vec<T>::pack(acc);
}

template <typename T>
cudaError_t launch_combine(const T *yp, const int32_t *inv, const float *w, T *out, int T_tok,
                           int k, int d, int A_total, int n_shared, int *status, cudaStream_t st) {
  const long long threads = static_cast<long long>(T_tok) * (d / Vec<T>::N);
  const int grid = static_cast<int>((threads + 255) / 256);
  combine_kernel<T><<<grid, 256, 0, st>>>(yp, inv, w, out, T_tok, k, d, A_total, n_shared, status);
  return cudaGetLastError();
}
template cudaError_t launch_combine<float>(const float *, const int32_t *, const float *, float *, int,
                                           int, int, int, int, int *, cudaStream_t);
template cudaError_t launch_combine<__nv_bfloat16>(const __nv_bfloat16 *, const int32_t *,
                                                   const float *, __nv_bfloat16 *, int, int, int, int,
                                                   int, int *, cudaStream_t);

}  // namespace moe
