// gemv_small.cu -- the expert projections of a small batch (T <= 32 bf16
// tokens): a grouped GEMV on warp-level tensor-core MMAs in which every SM
// streams weights.
//
// "Optimizing on-device inference for Apple Silicon", section "Match tile
// size to expert load": the tile shape should follow the number of rows an
// expert actually gets.  With a handful of tokens every touched expert holds
// one or two rows, so a 128 x 256 output tile per expert leaves most SMs idle
// (at T = 2, 17 groups make 68 gate/up tiles of 1 MB of weights each, while
// one SM streams ~40 GB/s).  Here the weights are the M side of an m16n8k16
// MMA and the group's columns (its tokens, or its rows of h) the N side (at
// most 16 in two 8-column blocks, or at most 32 in four for batches of 17 to
// 32 tokens, which hold fewer steps in registers), and a unit of work is 16 weight rows of one
// expert: 8 gate rows and the up rows of the same 8 features (gate/up, 64 KB
// at d = 2048), or 16 rows of W_down (down, 16 KB at F = 512).  Which units
// exist is decided on the device from the routing step's group offsets: at
// T = 2 there are 1,088 gate/up units and 2,176 down units, spread evenly
// over all SMs.
//
// Each unit belongs to warps that run on their own (no block-wide barrier):
// the weights go straight from HBM into registers, eight 32-column steps at a
// time, and the MMAs run as the loads land.  Lane (g, q) of a warp (g = lane
// / 4, q = lane % 4) reads, per step j, the 16 bytes at column 32 j + 8 q of
// rows g and g + 8; the MMA's k index is only summed over, so the lanes of a
// quad feed it their own columns (k = 2q, 2q + 1 from columns +0, +1 and
// k = 2q + 8, 2q + 9 from +2, +3; the step's second MMA takes +4..+7) and the
// N side is read with the same mapping: every product is formed once, in an
// fp32 accumulator.  A gate/up unit is shared by a pair of warps of one CTA,
// each taking half of d (so that at T = 2 all 16 warps of an SM stream), and
// the second warp's partial tile joins the first one's through shared memory
// under a two-warp barrier.
//
// Gate/up: rows g are gate rows f0 + g and rows g + 8 the up rows f0 + g, so
// a lane ends with gate and up values of the same (feature, token) pairs and
// writes h = silu(gate) * up as bf16 rows [slot][F] (the layout of the
// grouped GEMM's h).  Down: 16 rows of W_down against the group's rows of h,
// written as bf16 rows of Y [slot][d]; the common combine kernel then sums
// each token's top-k rows with its routing weights and adds the shared row.
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
// steps of 32 columns held in registers at once: fewer with more column
// blocks (their accumulators take the registers)
template <int NB>
constexpr int steps_for() { return NB <= 2 ? 8 : 6; }
// two buffers of [pair][4 NB values][32 lanes]
template <int NB>
constexpr int pair_bytes() { return 2 * kPairs * 4 * NB * 32 * 4; }

// weight pieces of steps [j0, j0 + S) of two rows (pointers already offset
// by this lane's q); steps at or past j1 are not read
template <int S>
__device__ __forceinline__ void load_rows(uint4 (&ra)[S], uint4 (&rb)[S], const uint4 *pa,
                                          const uint4 *pb, int j0, int j1) {
#pragma unroll
  for (int s = 0; s < S; ++s)
    if (j0 + s < j1) {
      ra[s] = ld_stream16(pa + 4 * (j0 + s));
      rb[s] = ld_stream16(pb + 4 * (j0 + s));
    }
}

}  // namespace

// gate/up: unit u = (touched group u / (F / 8), features 8 (u % (F / 8)) ..);
// pair p of CTA b takes units b + grid (p + 8 i); warp p takes the first half
// of d, warp p + 8 the second.  The shared expert's units come first and
// need no routing: their first weights are requested before the wait.
// NB: 8-column blocks of a group (its tokens), at most 4.
template <int NB>
__global__ void __launch_bounds__(kWarps * 32, 1) small_gateup_kernel(SmallArgs a) {
  constexpr int kSteps = steps_for<NB>();
  extern __shared__ uint4 s_dyn[];  // pair partials, then the tokens [T][d / 8 + 4]
  __shared__ int s_off[257], s_grp[257], s_ng;
  __shared__ int s_perm[kSmallGemvT * kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int pair = warp % kPairs, half = warp / kPairs;
  const int d = a.d, F = a.F, vr = d / 8, rs = vr + 4;
  const int fb = F / 8, nsteps = d / 32, j_lo = half * (nsteps / 2), j_hi = j_lo + nsteps / 2;
  const int stride = gridDim.x * kPairs;
  float *s_part = reinterpret_cast<float *>(s_dyn);
  uint4 *s_tok = s_dyn + pair_bytes<NB>() / 16;
  int u = blockIdx.x + gridDim.x * pair;
  uint4 ra[kSteps], rb[kSteps];
  bool pre = a.n_shared && u < fb;
  if (pre) {
    const long long r = static_cast<long long>(u * 8 + g) * d;
    load_rows<kSteps>(ra, rb, reinterpret_cast<const uint4 *>(a.sg + r) + q,
                      reinterpret_cast<const uint4 *>(a.su + r) + q, j_lo, j_hi);
  }
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
  for (int it = 0; u < nunits; u += stride, ++it, pre = false) {
    const int gi = u / fb, f0 = (u - gi * fb) * 8, grp = s_grp[gi];
    const bool sh = grp == a.E;
    const int n = sh ? a.T : s_off[grp + 1] - s_off[grp];
    const int slot0 = sh ? a.A : s_off[grp];
    const long long r = (sh ? 0LL : static_cast<long long>(grp) * F * d) +
                        static_cast<long long>(f0 + g) * d;
    const uint4 *pg = reinterpret_cast<const uint4 *>((sh ? a.sg : a.wg) + r) + q;
    const uint4 *pu = reinterpret_cast<const uint4 *>((sh ? a.su : a.wu) + r) + q;
    // this lane's columns g + 8 nb of the group (clamped: columns past n are
    // computed from a valid token and never stored)
    const uint4 *xc[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = min(8 * nb + g, n - 1);
      xc[nb] = s_tok + (sh ? m : s_perm[slot0 + m]) * rs + q;
    }
    float c[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nb][i] = 0.f;
    for (int j0 = j_lo; j0 < j_hi; j0 += kSteps) {
      if (!(pre && j0 == j_lo)) load_rows<kSteps>(ra, rb, pg, pu, j0, j_hi);
#pragma unroll
      for (int s = 0; s < kSteps; ++s) {
        if (j0 + s < j_hi) {
          const int cc = 4 * (j0 + s);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            if (8 * nb < n) gv_step(c[nb], ra[s], rb[s], xc[nb][cc]);
        }
      }
    }
    // the second half's partial tile joins the first's (two buffers: a
    // buffer is written again only after the next unit's barrier, which the
    // first warp passes after reading it)
    float *buf = s_part + ((it & 1) * kPairs + pair) * (4 * NB * 32) + lane;
    if (half == 1) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) buf[32 * (4 * nb + i)] = c[nb][i];
    }
    named_bar_sync(1 + pair, 64);
    if (half == 1) continue;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nb][i] += buf[32 * (4 * nb + i)];
    __nv_bfloat16 *hp = a.h + static_cast<long long>(slot0) * F + f0 + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = 8 * nb + 2 * q;
      if (m < n) hp[static_cast<long long>(m) * F] = __float2bfloat16_rn(silu(c[nb][0]) * c[nb][2]);
      if (m + 1 < n)
        hp[static_cast<long long>(m + 1) * F] = __float2bfloat16_rn(silu(c[nb][1]) * c[nb][3]);
    }
  }
}

// down: unit u = (touched group u / (d / 16), rows 16 (u % (d / 16)) ..);
// warp w of CTA b takes units b + grid (w + 16 i), each over the whole of F.
// NB: 8-column blocks of a group (its rows of h), at most 4.
template <int NB>
__global__ void __launch_bounds__(kWarps * 32, 1) small_down_kernel(SmallArgs a) {
  constexpr int kSteps = steps_for<NB>();
  __shared__ int s_off[257], s_grp[257], s_ng;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int d = a.d, F = a.F;
  const int rbk = d / 16, nsteps = F / 32, stride = gridDim.x * kWarps;
  // the offsets come from the routing step, which finished before the
  // gate/up launch let this one start; h is read only after the wait
  touched_groups(a, s_off, s_grp, &s_ng, KID_GEMM_DOWN);
  const int nunits = s_ng * rbk;
  int u = blockIdx.x + gridDim.x * warp;
  uint4 ra[kSteps], rb[kSteps];
  auto unit_rows = [&](int uu, const uint4 *&pa, const uint4 *&pb) {
    const int gi = uu / rbk, r0 = (uu - gi * rbk) * 16, grp = s_grp[gi];
    const bool sh = grp == a.E;
    const long long r = (sh ? 0LL : static_cast<long long>(grp) * d * F) +
                        static_cast<long long>(r0 + g) * F;
    pa = reinterpret_cast<const uint4 *>((sh ? a.sd : a.wd) + r) + q;
    pb = pa + F;  // row + 8: 8 F bf16 = F pieces of 16 B
  };
  bool pre = u < nunits;
  if (pre) {  // this warp's first weights load under the gate/up step
    const uint4 *pa, *pb;
    unit_rows(u, pa, pb);
    load_rows<kSteps>(ra, rb, pa, pb, 0, nsteps);
  }
  pdl_wait();  // h
  for (; u < nunits; u += stride, pre = false) {
    const int gi = u / rbk, r0 = (u - gi * rbk) * 16, grp = s_grp[gi];
    const bool sh = grp == a.E;
    const int n = sh ? a.T : s_off[grp + 1] - s_off[grp];
    const int slot0 = sh ? a.A : s_off[grp];
    const uint4 *pa, *pb;
    unit_rows(u, pa, pb);
    const uint4 *hq[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
      hq[nb] = reinterpret_cast<const uint4 *>(
                   a.h + static_cast<long long>(slot0 + min(8 * nb + g, n - 1)) * F) +
               q;
    float c[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nb][i] = 0.f;
    for (int j0 = 0; j0 < nsteps; j0 += kSteps) {
      if (!(pre && j0 == 0)) load_rows<kSteps>(ra, rb, pa, pb, j0, nsteps);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if (8 * nb < n) {
          // h was written by the gate/up kernel: coherent loads, all issued
          // before the first MMA that uses them
          uint4 hv[kSteps];
#pragma unroll
          for (int s = 0; s < kSteps; ++s)
            if (j0 + s < nsteps) hv[s] = ld_cg16(hq[nb] + 4 * (j0 + s));
#pragma unroll
          for (int s = 0; s < kSteps; ++s)
            if (j0 + s < nsteps) gv_step(c[nb], ra[s], rb[s], hv[s]);
        }
      }
    }
    __nv_bfloat16 *yp = a.y + static_cast<long long>(slot0) * d + r0 + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int m = 8 * nb + 2 * q;
      if (m < n) {
        yp[static_cast<long long>(m) * d] = __float2bfloat16_rn(c[nb][0]);
        yp[static_cast<long long>(m) * d + 8] = __float2bfloat16_rn(c[nb][2]);
      }
      if (m + 1 < n) {
        yp[static_cast<long long>(m + 1) * d] = __float2bfloat16_rn(c[nb][1]);
        yp[static_cast<long long>(m + 1) * d + 8] = __float2bfloat16_rn(c[nb][3]);
      }
    }
  }
}

namespace {
template <typename K>
cudaError_t launch_pdl(K kern, int grid, size_t smem, cudaStream_t st, bool pdl, const SmallArgs &a) {
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
// the tokens of at most 16 (32) rows of d = 2048 (4 KB each) and the pair
// partials of 2 (4) column blocks
constexpr size_t kTokBytes16 = 16 * (2048 / 8 + 4) * 16;
constexpr size_t kGateUpSmemMax2 = pair_bytes<2>() + kTokBytes16;
constexpr size_t kGateUpSmemMax4 = pair_bytes<4>() + 2 * kTokBytes16;
size_t gateup_smem(int T, int d) {
  return (T <= 16 ? pair_bytes<2>() : pair_bytes<4>()) + static_cast<size_t>(T) * (d / 8 + 4) * 16;
}
}  // namespace

bool small_gemv_fits(int T, int d, int F) {
  (void)F;
  return T >= 1 && T <= kSmallGemvT &&
         gateup_smem(T, d) <= (T <= 16 ? kGateUpSmemMax2 : kGateUpSmemMax4);
}

cudaError_t launch_small_gateup(const SmallArgs &a, int grid, cudaStream_t st, bool pdl) {
  const size_t smem = gateup_smem(a.T, a.d);
  return a.T <= 16 ? launch_pdl(small_gateup_kernel<2>, grid, smem, st, pdl, a)
                   : launch_pdl(small_gateup_kernel<4>, grid, smem, st, pdl, a);
}

cudaError_t launch_small_down(const SmallArgs &a, int grid, cudaStream_t st, bool pdl) {
  return a.T <= 16 ? launch_pdl(small_down_kernel<2>, grid, 0, st, pdl, a)
                   : launch_pdl(small_down_kernel<4>, grid, 0, st, pdl, a);
}

cudaError_t small_gemv_set_attr() {
  cudaError_t e = cudaFuncSetAttribute(small_gateup_kernel<2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kGateUpSmemMax2));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_gateup_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGateUpSmemMax4));
  return e;
}

}  // namespace moe
