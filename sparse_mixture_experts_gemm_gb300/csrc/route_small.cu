// route_small.cu -- the whole routing step of a small batch (T <= 64 bf16
// tokens) in one launch: logits, top-k, weights, histogram, group offsets and
// the slot permutation.
//
// "Optimizing on-device inference for Apple Silicon", section "Match tile
// size to expert load" (the verification batches of speculative decoding,
// a handful of tokens, want their own path) and section "Keep expert routing
// on the GPU".  At a few tokens the tensor-core router is all latency (a K
// loop of 32 steps per tile, then candidate merges and a last-CTA scan across
// the grid); here one thread-block cluster of ceil(E / 16) CTAs does it: CTA
// c multiplies the router rows of experts 16 c .. 16 c + 15 with the batch's
// tokens (the small-batch main loop: its 16 warps split d, weights requested
// before the tokens arrive, warp-level MMAs; the tokens in passes of 16, the
// router rows coming from L2 after the first pass), and each logit goes
// straight into CTA 0's shared memory; after one cluster barrier CTA 0 takes each
// token's top-k (one warp per token), the
// rank of every assignment inside its expert's group (the number of earlier
// assignments, in (token, choice) order, to the same expert), the exclusive
// scan of the group sizes, and writes idx, w, inv (each assignment's slot),
// perm (each slot's token) and the offsets: the inputs of the grouped GEMMs
// and of the combine, with no histogram atomics in memory and no separate
// placement kernel.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "decode_common.cuh"
#include "gemv_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kRouteWarps = kGvWarps;

// logits of experts 16 u .. 16 u + 15 for the pass's tokens t0 .. t0 + T - 1
// (one unit per CTA)
struct RouterOp {
  const __nv_bfloat16 *x, *wr;
  const float *bias;
  uint4 *s_tok;
  float (*s_lg)[256];
  int T, t0, d, E, rs, nsteps, first, stride;
  __device__ void prepare() {
    first = blockIdx.x;
    stride = gridDim.x;
  }
  __device__ bool early(int u) const { return 16 * u < E; }
  __device__ void wait() {  // the tokens (no dependency): padded rows
    const int vr = d / 8;
    const uint4 *xg = reinterpret_cast<const uint4 *>(x);
    for (int i = threadIdx.x; i < T * vr; i += blockDim.x) {
      const int t = i / vr;
      s_tok[t * rs + (i - t * vr)] = __ldg(xg + i);
    }
    __syncthreads();
  }
  __device__ int count() const { return early(first) ? 1 : 0; }
  __device__ void rows(int u, int, const uint4 *&pa, const uint4 *&pb) const {
    const int g = (threadIdx.x & 31) >> 2, q = threadIdx.x & 3;
    pa = reinterpret_cast<const uint4 *>(wr + static_cast<long long>(min(16 * u + g, E - 1)) * d) + q;
    pb = reinterpret_cast<const uint4 *>(wr + static_cast<long long>(min(16 * u + g + 8, E - 1)) * d) + q;
  }
  __device__ int ncols(int) const { return T; }
  __device__ const uint4 *col(int, int nb) const {
    return s_tok + min(8 * nb + ((threadIdx.x & 31) >> 2), T - 1) * rs + (threadIdx.x & 3);
  }
  __device__ void epilogue(int u, const float *red) const {
    const int t = threadIdx.x;
    if (t >= 256) return;
    const int r = t & 15, m = t >> 4, e = 16 * u + r;
    if (m >= T || e >= E) return;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kGvWarps; ++w) v += red[w * 256 + gv_part(r, m)];
    st_cluster_f32(&s_lg[t0 + m][e], 0, v + (bias ? bias[e] : 0.0f));
  }
};
}  // namespace

__global__ void __launch_bounds__(kRouteWarps * 32, 1)
    route_small_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ wr,
                       const float *__restrict__ bias, int T, int d, int E, int k, int32_t *idx,
                       float *w, int32_t *inv, int32_t *perm, int32_t *offsets,
                       int32_t *counts_out, int32_t *clear, int n_clear) {
  // partial tiles, then [kSmallRoutePass][d / 8 + 4] tokens, then (read in
  // CTA 0) the logits [T][256]
  extern __shared__ uint4 s_dyn[];
  __shared__ int s_idx[kSmallRouteT][kMaxTopK];
  __shared__ float s_w[kSmallRouteT][kMaxTopK];
  __shared__ int s_rank[kSmallRouteT * kMaxTopK];
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next launch (the expert gate/up) may start its routing-independent
  // reads now: it waits for this grid before it reads any of its outputs
  pdl_launch_dependents();
  const int rs = d / 8 + 4;
  float(*s_lg)[256] =
      reinterpret_cast<float(*)[256]>(s_dyn + kGvRedBytes / 16 + kSmallRoutePass * rs);
  for (int t0 = 0; t0 < T; t0 += kSmallRoutePass) {
    RouterOp op;
    op.x = x + static_cast<long long>(t0) * d;
    op.wr = wr;
    op.bias = bias;
    op.s_tok = s_dyn + kGvRedBytes / 16;
    op.s_lg = s_lg;
    op.T = min(kSmallRoutePass, T - t0);
    op.t0 = t0;
    op.d = d;
    op.E = E;
    op.rs = rs;
    op.nsteps = d / 32;
    gv_run<1>(op, reinterpret_cast<float *>(s_dyn));
  }
  cluster_sync_all();  // every CTA of the cluster reaches this: no return above
  if (cluster_ctarank() != 0) return;

  // CTA 0: one warp per token takes its top-k and the softmax over them
  for (int t = warp; t < T; t += kRouteWarps) {
    unsigned key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ee = lane + 32 * i;
      key[i] = ee < E ? fkey(s_lg[t][ee]) : 0u;
    }
    topk_from_keys(key, E, k, lane, s_idx[t], s_w[t]);
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  // rank of assignment a = t k + j among the earlier ones with the same expert
  // (A = T k <= 512, the CTA's threads)
  const int A = T * k;
  const int a = threadIdx.x;
  int ea = 0;
  if (a < A) {
    const int ta = a / k;
    ea = s_idx[ta][a - ta * k];
    // a token's k experts are distinct: only earlier tokens can share ea
    int r = 0;
    for (int tq = 0; tq < ta; ++tq)
      for (int jq = 0; jq < k; ++jq) r += s_idx[tq][jq] == ea;
    s_rank[a] = r;
    atomicAdd(&s_cnt[ea], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the group sizes
    const int per = (E + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int i = lane * per + q;
      if (i < E) sum += s_cnt[i];
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
      if (i < E) {
        s_off[i] = run;
        run += s_cnt[i];
      }
    }
    if (lane == 31) s_off[E] = incl;
  }
  __syncthreads();
  if (a < A) {
    const int slot = s_off[ea] + s_rank[a];
    idx[a] = ea;
    w[a] = s_w[a / k][a % k];
    inv[a] = slot;
    perm[slot] = a / k;
  }
  for (int i = threadIdx.x; i <= E; i += blockDim.x) offsets[i] = s_off[i];
  if (counts_out)  // summed over the chunks of a call
    for (int i = threadIdx.x; i < E; i += blockDim.x) counts_out[i] += s_cnt[i];
  // the grouped GEMMs' tile counters start at zero
  if (threadIdx.x == 0)
    for (int q = 0; q < n_clear; ++q) clear[q * 32] = 0;
}

// one cluster: the whole grid (at most 16 CTAs for E <= 256)
cudaError_t launch_route_small(const void *x, const void *wr, const float *bias, int T, int d,
                               int E, int k, int32_t *idx, float *w, int32_t *inv, int32_t *perm,
                               int32_t *offsets, int32_t *counts_out, int32_t *clear, int n_clear,
                               cudaStream_t st) {
  const int ncta = (E + kRouteWarps - 1) / kRouteWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta);
  cfg.blockDim = dim3(kRouteWarps * 32);
  cfg.dynamicSmemBytes = kGvRedBytes + static_cast<size_t>(kSmallRoutePass) * (d / 8 + 4) * 16 +
                         static_cast<size_t>(T) * 256 * 4;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_small_kernel, static_cast<const __nv_bfloat16 *>(x),
                            static_cast<const __nv_bfloat16 *>(wr), bias, T, d, E, k, idx, w, inv,
                            perm, offsets, counts_out, clear, n_clear);
}

cudaError_t route_small_set_attr() {
  cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kGvRedBytes + kSmallRouteTokBytes + kSmallRoutePass * 64 +
                                           kSmallRouteT * 256 * 4);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

}  // namespace moe
