// gemv_small_q4.cu -- the small-batch grouped GEMV (T <= 32 bf16 tokens) on
// 4-bit group-affine expert weights.
//
// The same units and warps as the bf16 small-batch GEMV (gemv_small.cu: 16
// weight rows of one touched expert on the M side of an m16n8k16 MMA, the
// group's tokens or rows of h on the N side, gate/up units split over a pair
// of warps), with the weights arriving as codes: "Optimizing on-device
// inference for Apple Silicon", section "Dequantise weights within matrix
// multiplication" -- every weight is a 4-bit code q with one bf16 scale s
// and bias b per 64 weights of a row, w = s q + b, rebuilt in bf16 right
// before the product.
//
// Column mapping.  The MMA's k index is only summed over, so a lane may feed
// it any columns as long as the N side uses the same ones.  Here lane
// (g, c) takes, per 128-column super-step J, the 32 consecutive columns
// 128 J + 32 c .. of rows g and g + 8: one 16-byte load of codes per row and,
// since 32 aligned columns never straddle a 64-column group, one scale and
// one bias per row.  MMA step s of the super-step uses columns + 8 s .. + 7.
//
// Dequantisation (8 codes of a 32-bit word, two per byte, the even column in
// the low nibble): a byte permute of the word and the word shifted right by
// 4 puts the two nibbles of byte p in the low bytes of the two halves; masked
// and or-ed with 0x4300 they are the bf16 values 128 + q exactly; 128 is
// subtracted exactly, then one bf16x2 FMA with (s, s) and (b, b) gives the
// weights, each rounded once to bf16 (as in the 4-bit grouped GEMM).
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "gemm_common.cuh"
#include "gemv_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kWarps = 16;
constexpr int kPairs = kWarps / 2;
// super-steps in flight with NB 8-column blocks: fewer with more blocks
// (their accumulators take the registers)
template <int NB>
constexpr int pre_for() { return NB <= 2 ? 4 : 2; }
// the down kernel, whose N side (h) comes from global memory, holds two
template <int NB>
constexpr int pre_down() { return 2; }
// two buffers of [pair][4 NB values][32 lanes]
template <int NB>
constexpr int pair_bytes() { return 2 * kPairs * 4 * NB * 32 * 4; }

// 8 codes -> the 4 bf16x2 weight pairs of columns (0, 1), (2, 3), (4, 5), (6, 7)
__device__ __forceinline__ uint4 dq8(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 b2) {
  const uint32_t w4 = w >> 4;
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.0f, 128.0f);
  uint32_t r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t x = __byte_perm(w, w4, p | (p << 4) | ((4 + p) << 8) | ((4 + p) << 12));
    x = (x & 0x000F000Fu) | 0x43004300u;  // (128 + q_2p, 128 + q_2p+1)
    __nv_bfloat162 qv = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&x), k128);
    const __nv_bfloat162 wv = __hfma2(qv, s2, b2);
    r[p] = *reinterpret_cast<const uint32_t *>(&wv);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ __nv_bfloat162 bcast(uint16_t bits) {
  const __nv_bfloat16 v = __ushort_as_bfloat16(bits);
  return __halves2bfloat162(v, v);
}

// One row's codes and (scale, bias) for super-steps [J0, J0 + P).
template <int P>
struct RowQ {
  uint4 c[P];
  uint16_t s[P], b[P];
};
// codes: the row's codes offset to this lane's first super-step (uint4 index
// 4 J per super-step); sb: the row's scales / biases at this lane's group of
// super-step 0 (2 groups per super-step)
template <int P>
__device__ __forceinline__ void load_rowq(RowQ<P> &r, const uint4 *codes, const uint16_t *s,
                                          const uint16_t *b, int J0, int J1) {
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (J0 + i < J1) {
      r.c[i] = ld_stream16(codes + 4 * (J0 + i));
      r.s[i] = __ldg(s + 2 * (J0 + i));
      r.b[i] = __ldg(b + 2 * (J0 + i));
    }
}

// MMA steps of one super-step: rows g (ra) and g + 8 (rb) against the 32
// columns' N-side values x[nb] (uint4 per 8 columns, stride 1) of the
// column blocks nb < nblk; kGlobal: x in global memory (read through L2),
// else in shared memory.  The weights are rebuilt once for all blocks.
// the N-side pointers of a unit's column blocks
template <int NB>
struct Cols {
  const uint4 *p[NB];
};

template <bool kGlobal, int NB, int P>
__device__ __forceinline__ void superstep(float (&c)[NB][4], const RowQ<P> &ra, const RowQ<P> &rb,
                                          int i, const Cols<NB> xb, int off, int nblk) {
  const __nv_bfloat162 sa = bcast(ra.s[i]), ba = bcast(ra.b[i]);
  const __nv_bfloat162 sb = bcast(rb.s[i]), bb = bcast(rb.b[i]);
  const uint32_t wa[4] = {ra.c[i].x, ra.c[i].y, ra.c[i].z, ra.c[i].w};
  const uint32_t wb[4] = {rb.c[i].x, rb.c[i].y, rb.c[i].z, rb.c[i].w};
  if constexpr (NB <= 2) {
    // every N-side value first (h from global memory was written by the
    // gate/up kernel: coherent loads, all issued before the first MMA that
    // uses them), then the weights of each step, rebuilt once for the blocks
    uint4 v[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int s = 0; s < 4; ++s)
        if (nb < nblk) v[nb][s] = kGlobal ? ld_cg16(xb.p[nb] + off + s) : xb.p[nb][off + s];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint4 a = dq8(wa[s], sa, ba), b = dq8(wb[s], sb, bb);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        if (nb < nblk) gv_step(c[nb], a, b, v[nb][s]);
    }
  } else {
    // the weights of the super-step rebuilt once, then block by block its N
    // side (four loads issued together) and MMAs
    uint4 a[4], b[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      a[s] = dq8(wa[s], sa, ba);
      b[s] = dq8(wb[s], sb, bb);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      if (nb < nblk) {
        uint4 v[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) v[s] = kGlobal ? ld_cg16(xb.p[nb] + off + s) : xb.p[nb][off + s];
#pragma unroll
        for (int s = 0; s < 4; ++s) gv_step(c[nb], a[s], b[s], v[s]);
      }
    }
  }
}
}  // namespace

// gate/up: unit u = (touched group u / (F / 8), features 8 (u % (F / 8)) ..);
// pair p of CTA b takes units b + grid (p + 8 i); warp p takes the first half
// of d, warp p + 8 the second.  NB: 8-column blocks of a group, at most 4.
template <int NB>
__global__ void __launch_bounds__(kWarps * 32, 1) small_gateup_q4_kernel(SmallQ4Args qa) {
  constexpr int P = pre_for<NB>();
  const SmallArgs &a = qa.a;
  extern __shared__ uint4 s_dyn[];  // pair partials, then the tokens [T][d / 8 + 4]
  __shared__ int s_off[257], s_grp[257], s_ng;
  __shared__ int s_perm[kSmallGemvT * kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int pair = warp % kPairs, half = warp / kPairs;
  const int d = a.d, F = a.F, vr = d / 8, rs = vr + 4;
  const int fb = F / 8, nss = d / 256;  // super-steps per half of d
  const int col0 = half * (d / 2) + 32 * c;  // this lane's first column
  const int stride = gridDim.x * kPairs;
  float *s_part = reinterpret_cast<float *>(s_dyn);
  uint4 *s_tok = s_dyn + pair_bytes<NB>() / 16;
  const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
  for (int i = threadIdx.x; i < a.T * vr; i += blockDim.x) {
    const int t = i / vr;
    s_tok[t * rs + (i - t * vr)] = __ldg(xg + i);
  }
  pdl_wait();  // the routing step's offsets and permutation
  pdl_launch_dependents();
  touched_groups(a, s_off, s_grp, &s_ng, KID_GEMM_GATE_UP);
  for (int i = threadIdx.x; i < a.A; i += blockDim.x) {
    int t = ld_cg_s32(a.perm + i);
    if (t < 0 || t >= a.T) {
      report_error(a.status, MOE_ERR_DEVICE_BOUNDS, KID_GEMM_GATE_UP * 100 + SITE_INDEX);
      t = 0;
    }
    s_perm[i] = t;
  }
  __syncthreads();
  const int nunits = s_ng * fb;
  int it = 0;
  for (int u = blockIdx.x + gridDim.x * pair; u < nunits; u += stride, ++it) {
    const int gi = u / fb, f0 = (u - gi * fb) * 8, grp = s_grp[gi];
    const bool sh = grp == a.E;
    const int n = sh ? a.T : s_off[grp + 1] - s_off[grp];
    const int slot0 = sh ? a.A : s_off[grp];
    const Q4Mat &mg = sh ? qa.w.sg : qa.w.g, &mu = sh ? qa.w.su : qa.w.u;
    const long long row = (sh ? 0LL : static_cast<long long>(grp) * F) + f0 + g;
    const uint4 *cg = reinterpret_cast<const uint4 *>(mg.c + row * (d / 2) + col0 / 2);
    const uint4 *cu = reinterpret_cast<const uint4 *>(mu.c + row * (d / 2) + col0 / 2);
    const long long sbo = row * (d / 64) + col0 / 64;
    Cols<NB> xc;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = min(8 * nb + g, n - 1);
      xc.p[nb] = s_tok + (sh ? m : s_perm[slot0 + m]) * rs + col0 / 8;
    }
    const int nblk = (n + 7) / 8;
    float cacc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) cacc[nb][i] = 0.f;
    for (int J0 = 0; J0 < nss; J0 += P) {
      RowQ<P> ra, rb;
      load_rowq<P>(ra, cg, mg.s + sbo, mg.b + sbo, J0, nss);
      load_rowq<P>(rb, cu, mu.s + sbo, mu.b + sbo, J0, nss);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        if (J0 + i < nss) superstep<false, NB, P>(cacc, ra, rb, i, xc, 16 * (J0 + i), nblk);
      }
    }
    float *buf = s_part + ((it & 1) * kPairs + pair) * (4 * NB * 32) + lane;
    if (half == 1) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) buf[32 * (4 * nb + i)] = cacc[nb][i];
    }
    named_bar_sync(1 + pair, 64);
    if (half == 1) continue;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) cacc[nb][i] += buf[32 * (4 * nb + i)];
    __nv_bfloat16 *hp = a.h + static_cast<long long>(slot0) * F + f0 + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float *cc = cacc[nb];
      const int m = 8 * nb + 2 * c;
      if (m < n) hp[static_cast<long long>(m) * F] = __float2bfloat16_rn(silu(cc[0]) * cc[2]);
      if (m + 1 < n) hp[static_cast<long long>(m + 1) * F] = __float2bfloat16_rn(silu(cc[1]) * cc[3]);
    }
  }
}

// down: unit u = (touched group u / (d / 16), rows 16 (u % (d / 16)) ..);
// warp w of CTA b takes units b + grid (w + 16 i), each over the whole of F.
// NB: 8-column blocks of a group, at most 4.
template <int NB>
__global__ void __launch_bounds__(kWarps * 32, 1) small_down_q4_kernel(SmallQ4Args qa) {
  constexpr int P = pre_down<NB>();
  const SmallArgs &a = qa.a;
  __shared__ int s_off[257], s_grp[257], s_ng;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int d = a.d, F = a.F;
  const int rbk = d / 16, nss = F / 128, stride = gridDim.x * kWarps;
  // the offsets come from the routing step, which finished before the
  // gate/up launch let this one start; h is read only after the wait
  touched_groups(a, s_off, s_grp, &s_ng, KID_GEMM_DOWN);
  pdl_wait();  // h
  const int nunits = s_ng * rbk;
  for (int u = blockIdx.x + gridDim.x * warp; u < nunits; u += stride) {
    const int gi = u / rbk, r0 = (u - gi * rbk) * 16, grp = s_grp[gi];
    const bool sh = grp == a.E;
    const int n = sh ? a.T : s_off[grp + 1] - s_off[grp];
    const int slot0 = sh ? a.A : s_off[grp];
    const Q4Mat &md = sh ? qa.w.sd : qa.w.d;
    const long long ra0 = (sh ? 0LL : static_cast<long long>(grp) * d) + r0 + g;  // rows g, g + 8
    // lane c's 32 columns start 16 c bytes into each code row
    const uint4 *ca = reinterpret_cast<const uint4 *>(md.c + ra0 * (F / 2)) + c;
    const uint4 *cb = reinterpret_cast<const uint4 *>(md.c + (ra0 + 8) * (F / 2)) + c;
    const long long sa = ra0 * (F / 64) + c / 2, sb = (ra0 + 8) * (F / 64) + c / 2;
    Cols<NB> hc;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
      hc.p[nb] = reinterpret_cast<const uint4 *>(
                   a.h + static_cast<long long>(slot0 + min(8 * nb + g, n - 1)) * F) +
               4 * c;
    const int nblk = (n + 7) / 8;
    float cacc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) cacc[nb][i] = 0.f;
    for (int J0 = 0; J0 < nss; J0 += P) {
      RowQ<P> qa0, qb0;
      load_rowq<P>(qa0, ca, md.s + sa, md.b + sa, J0, nss);
      load_rowq<P>(qb0, cb, md.s + sb, md.b + sb, J0, nss);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        if (J0 + i < nss) superstep<true, NB, P>(cacc, qa0, qb0, i, hc, 16 * (J0 + i), nblk);
      }
    }
    __nv_bfloat16 *yp = a.y + static_cast<long long>(slot0) * d + r0 + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float *cc = cacc[nb];
      const int m = 8 * nb + 2 * c;
      if (m < n) {
        yp[static_cast<long long>(m) * d] = __float2bfloat16_rn(cc[0]);
        yp[static_cast<long long>(m) * d + 8] = __float2bfloat16_rn(cc[2]);
      }
      if (m + 1 < n) {
        yp[static_cast<long long>(m + 1) * d] = __float2bfloat16_rn(cc[1]);
        yp[static_cast<long long>(m + 1) * d + 8] = __float2bfloat16_rn(cc[3]);
      }
    }
  }
}

namespace {
template <typename K>
cudaError_t launch_q4(K kern, int grid, size_t smem, cudaStream_t st, bool pdl, const SmallQ4Args &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}
// the tokens of at most 16 (32) rows of d = 2048 and the pair partials of 2
// (4) column blocks (the bf16 small-batch GEMV's plan: small_gemv_fits
// decides for both)
constexpr size_t kTokBytes16 = 16 * (2048 / 8 + 4) * 16;
constexpr size_t kGateUpSmemMax2 = pair_bytes<2>() + kTokBytes16;
constexpr size_t kGateUpSmemMax4 = pair_bytes<4>() + 2 * kTokBytes16;
}  // namespace

cudaError_t launch_small_gateup_q4(const SmallQ4Args &a, int grid, cudaStream_t st, bool pdl) {
  const int T = a.a.T;
  const size_t tok = static_cast<size_t>(T) * (a.a.d / 8 + 4) * 16;
  return T <= 16 ? launch_q4(small_gateup_q4_kernel<2>, grid, pair_bytes<2>() + tok, st, pdl, a)
                 : launch_q4(small_gateup_q4_kernel<4>, grid, pair_bytes<4>() + tok, st, pdl, a);
}

cudaError_t launch_small_down_q4(const SmallQ4Args &a, int grid, cudaStream_t st, bool pdl) {
  return a.a.T <= 16 ? launch_q4(small_down_q4_kernel<2>, grid, 0, st, pdl, a)
                     : launch_q4(small_down_q4_kernel<4>, grid, 0, st, pdl, a);
}

cudaError_t small_gemv_q4_set_attr() {
  cudaError_t e = cudaFuncSetAttribute(small_gateup_q4_kernel<2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kGateUpSmemMax2));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_gateup_q4_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGateUpSmemMax4));
  return e;
}

}  // namespace moe
