// decode_q4.cu -- the batch-1 path for 4-bit group-affine expert weights, and
// the quantiser that produces them.
//
// Format ("Optimizing on-device inference for Apple Silicon", section
// "Dequantise weights within matrix multiplication": 4-bit codes with one
// scale and one bias per group of 64 weights): a matrix [rows][cols] is codes
// [rows][cols / 2] (two per byte along the row, the even column in the low
// nibble) plus bf16 scales and biases [rows][cols / 64]; w = scale * q + bias.
// The pages' point is bytes: with one row per token every weight byte is read
// once (section "Decode: minimise bytes moved per token"), and this format
// reads 0.5625 bytes per weight instead of 2.
//
// The dequantisation is folded into the dot product: for one group of 64
// columns,  sum_c (s q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c,  and
// sum_c x_c is computed once per token (per group) in shared memory.  Each
// lane owns whole groups of a row (32 bytes of codes, one scale, one bias), so
// it reads the token (or h) from shared memory rows padded to 65 floats per
// group: lane g reads word g * 65 + e, bank (g + e) % 32, no conflicts.
//
// The three kernels mirror decode.cu (A router + shared gate/up, B routed
// gate/up, C down + combine), chained with programmatic dependent launch:
// static weights (the router rows, the shared expert's rows; C's rows once
// the choice is known) are requested before griddepcontrol.wait.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kPad = kQ4Group + 1;  // floats per padded group row in shared memory
constexpr int kMaxGroupsPerLane = 8;  // rows of up to 16384 columns

__device__ __forceinline__ float bf16f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Codes, scale and bias of the groups g = lane + 32 m of one row.
struct Q4Row {
  uint4 c[kMaxGroupsPerLane][2];
  uint16_t s[kMaxGroupsPerLane], b[kMaxGroupsPerLane];
};

__device__ __forceinline__ void q4_row_load(Q4Row &r, const Q4Mat &m, long long row, int cols,
                                            int lane) {
  const int G = cols / kQ4Group;
  const uint4 *cb = reinterpret_cast<const uint4 *>(m.c + row * (cols / 2));
  const uint16_t *sb = m.s + row * G, *bb = m.b + row * G;
#pragma unroll
  for (int q = 0; q < kMaxGroupsPerLane; ++q) {
    const int g = lane + 32 * q;
    if (g < G) {
      r.c[q][0] = ld_stream16(cb + 2 * g);
      r.c[q][1] = ld_stream16(cb + 2 * g + 1);
      r.s[q] = __ldg(sb + g);
      r.b[q] = __ldg(bb + g);
    }
  }
}

// sum over the 64 codes of a group of q_e * v_e (v: 64 floats in shared memory)
__device__ __forceinline__ float q4_group_dot(const uint4 &c0, const uint4 &c1, const float *v) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e)
      acc = fmaf(static_cast<float>((w[j] >> (4 * e)) & 15u), v[8 * j + e], acc);
  return acc;
}

// dot(row, v) for a row loaded into r; vp: padded groups of v, vs: group sums.
__device__ __forceinline__ float q4_row_dot(const Q4Row &r, int cols, const float *vp,
                                            const float *vs, int lane) {
  const int G = cols / kQ4Group;
  float acc = 0.0f;
#pragma unroll
  for (int q = 0; q < kMaxGroupsPerLane; ++q) {
    const int g = lane + 32 * q;
    if (g < G) {
      const float dq = q4_group_dot(r.c[q][0], r.c[q][1], vp + g * kPad);
      acc += bf16f(r.s[q]) * dq + bf16f(r.b[q]) * vs[g];
    }
  }
  return acc;
}

// The bf16 token into padded float groups vp[G][65] and group sums vs[G]
// (all threads of the CTA; L2 reads).
__device__ __forceinline__ void load_token_groups(float *vp, float *vs, const void *x, int d) {
  const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
  const uint32_t *xw = reinterpret_cast<const uint32_t *>(xb);
  for (int i = threadIdx.x; i < d / 2; i += blockDim.x) {
    const uint32_t v = __ldcg(xw + i);
    const int c = 2 * i, g = c / kQ4Group, e = c - g * kQ4Group;
    vp[g * kPad + e] = __uint_as_float(v << 16);
    vp[g * kPad + e + 1] = __uint_as_float(v & 0xFFFF0000u);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < d / kQ4Group; g += blockDim.x) {
    float s = 0.0f;
    for (int e = 0; e < kQ4Group; ++e) s += vp[g * kPad + e];
    vs[g] = s;
  }
  __syncthreads();
}

}  // namespace

// ---------------------------------------------------------------- A: router + shared gate/up
// CTAs [0, ceil(E / 8)): one warp per expert logit (bf16 router rows, as in
// decode.cu).  CTAs after them: one warp per shared-expert row f, its 4-bit
// gate and up rows loaded before the dependency wait.
__global__ void __launch_bounds__(256) decode_router_q4_kernel(const DecodeArgs a) {
  extern __shared__ uint4 sm4[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d;
  const int nvec = d * 2 / 16;
  const int n_rt = (a.E + 7) / 8;
  if (static_cast<int>(blockIdx.x) >= n_rt) {
    float *vp = reinterpret_cast<float *>(sm4);
    float *vs = vp + (d / kQ4Group) * kPad;
    const int f = (blockIdx.x - n_rt) * 8 + warp;
    Q4Row rg, ru;
    if (f < a.F) {
      q4_row_load(rg, a.q.sg, f, d, lane);
      q4_row_load(ru, a.q.su, f, d, lane);
    }
    pdl_launch_dependents();
    pdl_wait();
    load_token_groups(vp, vs, a.x, d);
    if (f >= a.F) return;
    const float g = warp_sum(q4_row_dot(rg, d, vp, vs, lane));
    const float u = warp_sum(q4_row_dot(ru, d, vp, vs, lane));
    if (lane == 0) a.h[static_cast<long long>(a.k) * a.F + f] = g / (1.0f + __expf(-g)) * u;
    return;
  }
  const int e = blockIdx.x * 8 + warp;
  const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.wr) +
                                                     static_cast<long long>(e) * d);
  RowPre pr;
  if (e < a.E) row_prefetch(pr, row, nvec, lane);
  pdl_launch_dependents();
  pdl_wait();
  load_token(sm4, a.x, nvec);
  if (e < a.E) {
    const float acc = warp_sum(row_dot_pre<__nv_bfloat16>(pr, row, sm4, nvec, lane));
    if (lane == 0) a.logits[e] = acc + (a.bias ? a.bias[e] : 0.0f);
  }
}

// ---------------------------------------------------------------- B: routed gate/up
// Tile t: 32 rows of slot s = t / (F / 32); warp w takes rows 4w .. 4w + 3,
// each a (gate row, up row) pair loaded whole into registers (one group per
// lane at d = 2048) before any is used.
constexpr int kQRB = 32;

__global__ void __launch_bounds__(256) decode_gateup_q4_kernel(const DecodeArgs a) {
  extern __shared__ float smf[];
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F;
  float *vp = smf;
  float *vs = vp + (d / kQ4Group) * kPad;
  const int nrb = F / kQRB;
  const int ntile = a.k * nrb;
  pdl_wait();
  if (warp == 0) warp_topk(a.logits, a.E, a.k, lane, s_sel, s_selw);
  load_token_groups(vp, vs, a.x, d);  // includes the barriers that publish s_sel
  pdl_launch_dependents();
  for (int t = blockIdx.x; t < ntile; t += gridDim.x) {
    const int s = t / nrb, rb = t - (t / nrb) * nrb;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int f = rb * kQRB + 4 * warp + q;
      const long long row = static_cast<long long>(s_sel[s]) * F + f;
      Q4Row rg, ru;
      q4_row_load(rg, a.q.g, row, d, lane);
      q4_row_load(ru, a.q.u, row, d, lane);
      const float g = warp_sum(q4_row_dot(rg, d, vp, vs, lane));
      const float u = warp_sum(q4_row_dot(ru, d, vp, vs, lane));
      if (lane == 0) a.h[static_cast<long long>(s) * F + f] = g / (1.0f + __expf(-g)) * u;
    }
  }
}

// ---------------------------------------------------------------- C: down + combine
// One warp per output element i.  The (slot, group) pairs of the row, k + 1
// slots of F / 64 groups, are spread over the lanes; their codes are loaded
// before the wait for h.
constexpr int kMaxPairsPerLane = 5;  // (8 + 1) slots x 16 groups (F = 1024) / 32

__global__ void __launch_bounds__(256) decode_down_q4_kernel(const DecodeArgs a) {
  extern __shared__ float smf[];
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F, GF = F / kQ4Group;
  const int nslot = a.k + a.n_shared;
  const int npair = nslot * GF;
  const int i = blockIdx.x * 8 + warp;
  pdl_launch_dependents();
  if (warp == 0) warp_topk(a.logits, a.E, a.k, lane, s_sel, s_selw);
  __syncthreads();
  uint4 c[kMaxPairsPerLane][2];
  uint16_t sc[kMaxPairsPerLane], bi[kMaxPairsPerLane];
#pragma unroll
  for (int m = 0; m < kMaxPairsPerLane; ++m) {
    const int p = lane + 32 * m;
    if (p < npair && i < d) {
      const int s = p / GF, g = p - s * GF;
      const Q4Mat &mat = s < a.k ? a.q.d : a.q.sd;
      const long long row = s < a.k ? static_cast<long long>(s_sel[s]) * d + i : i;
      const uint4 *cb = reinterpret_cast<const uint4 *>(mat.c + row * (F / 2));
      c[m][0] = ld_stream16(cb + 2 * g);
      c[m][1] = ld_stream16(cb + 2 * g + 1);
      sc[m] = __ldg(mat.s + row * GF + g);
      bi[m] = __ldg(mat.b + row * GF + g);
    }
  }
  pdl_wait();
  // h of every slot into padded groups, then the group sums
  float *hp = smf;
  float *hs = hp + npair * kPad;
  for (int q = threadIdx.x; q < nslot * F; q += blockDim.x) {
    const int p = q / kQ4Group, e = q - p * kQ4Group;
    hp[p * kPad + e] = __ldcg(a.h + q);
  }
  __syncthreads();
  for (int p = threadIdx.x; p < npair; p += blockDim.x) {
    float s = 0.0f;
    for (int e = 0; e < kQ4Group; ++e) s += hp[p * kPad + e];
    hs[p] = s;
  }
  __syncthreads();
  if (i >= d) return;
  float acc = 0.0f;
#pragma unroll
  for (int m = 0; m < kMaxPairsPerLane; ++m) {
    const int p = lane + 32 * m;
    if (p < npair) {
      const int s = p / GF;
      const float dq = q4_group_dot(c[m][0], c[m][1], hp + p * kPad);
      const float part = bf16f(sc[m]) * dq + bf16f(bi[m]) * hs[p];
      acc = fmaf(s < a.k ? s_selw[s] : 1.0f, part, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) reinterpret_cast<__nv_bfloat16 *>(a.out)[i] = __float2bfloat16_rn(acc);
}

// ---------------------------------------------------------------- quantiser
// One thread per group of 64 columns: bias = min and scale = (max - min) / 15,
// both rounded to bf16; q = nearest integer (ties to even) of (w - bias) /
// scale, clamped to 0..15; q = 0 when the scale is 0.
template <typename T>
__global__ void quantize_q4_kernel(const T *__restrict__ w, long long ngroups, int cols,
                                   uint8_t *codes, uint16_t *scales, uint16_t *biases) {
  const long long gi = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gi >= ngroups) return;
  const int G = cols / kQ4Group;
  const long long r = gi / G;
  const int g = static_cast<int>(gi - r * G);
  const T *src = w + r * cols + g * kQ4Group;
  float v[kQ4Group];
  float lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int e = 0; e < kQ4Group; ++e) {
    v[e] = static_cast<float>(src[e]);
    lo = fminf(lo, v[e]);
    hi = fmaxf(hi, v[e]);
  }
  const __nv_bfloat16 sb = __float2bfloat16_rn((hi - lo) / 15.0f);
  const __nv_bfloat16 bb = __float2bfloat16_rn(lo);
  const float s = __bfloat162float(sb), b = __bfloat162float(bb);
  uint32_t packed[kQ4Group / 8];
#pragma unroll
  for (int j = 0; j < kQ4Group / 8; ++j) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float q = s > 0.0f ? rintf((v[8 * j + e] - b) / s) : 0.0f;
      q = fminf(fmaxf(q, 0.0f), 15.0f);
      word |= static_cast<uint32_t>(q) << (4 * e);
    }
    packed[j] = word;
  }
  uint4 *dst = reinterpret_cast<uint4 *>(codes + (r * cols + g * kQ4Group) / 2);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  scales[gi] = *reinterpret_cast<const uint16_t *>(&sb);
  biases[gi] = *reinterpret_cast<const uint16_t *>(&bb);
}

// ---------------------------------------------------------------- launchers
namespace {
size_t tok_smem(int d) { return sizeof(float) * ((d / kQ4Group) * kPad + d / kQ4Group); }

template <typename K>
cudaError_t launch_q(K kern, int grid, size_t smem, cudaStream_t st, bool pdl,
                     const DecodeArgs &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
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

cudaError_t launch_decode_router_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int grid = (a.E + 7) / 8 + (a.n_shared ? (a.F + 7) / 8 : 0);
  size_t smem = tok_smem(a.d);
  if (smem < static_cast<size_t>(a.d) * 2) smem = static_cast<size_t>(a.d) * 2;
  return launch_q(decode_router_q4_kernel, grid, smem, st, pdl, a);
}
cudaError_t launch_decode_gateup_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const int ntile = a.k * (a.F / kQRB);
  return launch_q(decode_gateup_q4_kernel, ntile < sms ? ntile : sms, tok_smem(a.d), st, pdl, a);
}
cudaError_t launch_decode_down_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int npair = (a.k + a.n_shared) * (a.F / kQ4Group);
  const size_t smem = sizeof(float) * (static_cast<size_t>(npair) * kPad + npair);
  return launch_q(decode_down_q4_kernel, (a.d + 7) / 8, smem, st, pdl, a);
}

// The shared-memory limits of the three kernels for the largest supported
// shapes (d = 16384, F * (k + 1) = 4096 * 9 would not fit; the create call
// rejects layers whose h does not fit, see moe_create_q4).
cudaError_t decode_q4_set_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(decode_router_q4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tok_smem(16384)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_gateup_q4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tok_smem(16384)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_down_q4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              200 * 1024);
}

template <typename T>
cudaError_t launch_quantize_q4(const T *w, long long rows, int cols, uint8_t *codes,
                               uint16_t *scales, uint16_t *biases, cudaStream_t st) {
  const long long ngroups = rows * (cols / kQ4Group);
  if (ngroups == 0) return cudaSuccess;
  const long long grid = (ngroups + 127) / 128;
  quantize_q4_kernel<T><<<static_cast<unsigned>(grid), 128, 0, st>>>(w, ngroups, cols, codes,
                                                                     scales, biases);
  return cudaGetLastError();
}
template cudaError_t launch_quantize_q4<__nv_bfloat16>(const __nv_bfloat16 *, long long, int,
                                                       uint8_t *, uint16_t *, uint16_t *,
                                                       cudaStream_t);
template cudaError_t launch_quantize_q4<float>(const float *, long long, int, uint8_t *, uint16_t *,
                                               uint16_t *, cudaStream_t);

}  // namespace moe
