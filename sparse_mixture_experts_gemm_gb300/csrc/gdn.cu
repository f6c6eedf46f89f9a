// gdn.cu -- the Gated DeltaNet recurrent scan (the C ABI in include/gdn.h).
//
// "Optimizing on-device inference for Apple Silicon", section "Keep the
// recurrent state on chip": the state matrix is split by columns, each
// column's slice loaded into registers once, carried through the whole scan
// and written back only at its end; partial results are exchanged by lane
// operations, not through shared memory; state and gate are 32-bit float,
// the activations bfloat16.  The pages give each column a whole SIMD group;
// here a column belongs to L lanes (L = 8: 16 fp32 entries per lane at
// d_k = 128, four columns per warp), which keeps all of the state's 2 MB
// (32 value heads x 128 x 128) in registers on ~7 warps per SM and needs 3
// shuffle rounds per reduction instead of 5 -- with one warp per column the
// per-token shuffles and scalar work would be issued for every column.
//
// Per token and column (lane part of the dot products, then a butterfly
// over the column's L lanes):
//     r = S . k_t,  p = S . q_t,  c = q_t . k_t (per token, computed once per CTA)
//     u = beta (v - alpha r)
//     o = alpha p + u c          (= q_t . S_new, without a second reduction)
//     S = alpha S + u k_t
// The recurrence's chain per token is the two reductions; everything that
// does not depend on the state is staged ahead: a CTA (4 warps, the 16
// columns of one value head) copies the bf16 q and k of its key head, its v
// columns and the gates of the next 32 tokens by cp.async while it scans the
// current 32, then converts them to fp32 once in shared memory for all of its
// columns and forms c.  Lane s of a column holds the entries 4 s + 32 i + 0..3
// (i = 0..3): the 8 lanes of a column read 128 contiguous bytes of k per
// instruction, so the shared-memory reads are free of bank conflicts.
#include <cuda_bf16.h>

#include "../../include/gdn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kDk = 128;       // d_k supported
constexpr int kLanes = 8;      // lanes per column
constexpr int kEpl = kDk / kLanes;       // state entries per lane
constexpr int kWarpsPerCta = 4;
constexpr int kCols = kWarpsPerCta * 32 / kLanes;  // columns per CTA
constexpr int kTb = 32;        // tokens per staged block

struct GdnArgs {
  const __nv_bfloat16 *q, *k, *v;
  const float *alpha, *beta, *s_in;
  float *s_out;
  __nv_bfloat16 *o;
  int T, Hk, Hv, dv;
};

struct GdnSmem {
  float kf[kTb][kDk], qf[kTb][kDk];  // fp32 activations of the current block
  float c[kTb];                       // q_t . k_t
  __nv_bfloat16 kr[kTb][kDk], qr[kTb][kDk];  // raw bf16 of the next block
  __nv_bfloat16 vr[kTb][kCols];
  float ar[kTb], br[kTb];
  __nv_bfloat16 vs[kTb][kCols];       // the current block's v, gate, strength
  float as[kTb], bs[kTb];
};

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// raw copies of tokens [t0, t0 + n) for this CTA (value head h, columns j0..)
__device__ __forceinline__ void stage_raw(GdnSmem &sm, const GdnArgs &a, int t0, int n, int h,
                                          int hk, int j0) {
  // q and k: 16 pieces of 16 B per token each
  for (int i = threadIdx.x; i < n * 32; i += blockDim.x) {
    const int t = i >> 5, p = i & 31, which = p >> 4, piece = p & 15;
    const long long src = (static_cast<long long>(t0 + t) * a.Hk + hk) * kDk + piece * 8;
    __nv_bfloat16 *dst = (which ? sm.qr[t] : sm.kr[t]) + piece * 8;
    cp_async16(smem_u32(dst), (which ? a.q : a.k) + src);
  }
  // v: kCols bf16 = 2 pieces per token; gate and strength: 4 B each
  for (int i = threadIdx.x; i < n * 4; i += blockDim.x) {
    const int t = i >> 2, p = i & 3;
    const long long tv = static_cast<long long>(t0 + t) * a.Hv + h;
    if (p < 2)
      cp_async16(smem_u32(&sm.vr[t][p * 8]), a.v + tv * a.dv + j0 + p * 8);
    else if (p == 2)
      cp_async4(&sm.ar[t], a.alpha + tv);
    else
      cp_async4(&sm.br[t], a.beta + tv);
  }
  cp_async_commit();
}

// raw block -> the fp32 block the scan reads; c_t = q_t . k_t (one warp per
// token, fixed order: lane-local sums of 4, then a butterfly)
__device__ __forceinline__ void convert_block(GdnSmem &sm, int n) {
  for (int i = threadIdx.x; i < n * kDk / 2; i += blockDim.x) {
    const int t = i / (kDk / 2), e = (i - t * (kDk / 2)) * 2;
    const float2 kk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&sm.kr[t][e]));
    const float2 qq = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&sm.qr[t][e]));
    sm.kf[t][e] = kk.x;
    sm.kf[t][e + 1] = kk.y;
    sm.qf[t][e] = qq.x;
    sm.qf[t][e + 1] = qq.y;
  }
  for (int i = threadIdx.x; i < n * kCols; i += blockDim.x) sm.vs[i / kCols][i % kCols] = sm.vr[i / kCols][i % kCols];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    sm.as[i] = sm.ar[i];
    sm.bs[i] = sm.br[i];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < n; t += kWarpsPerCta) {
    const float4 kk = reinterpret_cast<const float4 *>(sm.kf[t])[lane];
    const float4 qq = reinterpret_cast<const float4 *>(sm.qf[t])[lane];
    float s = kk.x * qq.x + kk.y * qq.y + kk.z * qq.z + kk.w * qq.w;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.c[t] = s;
  }
}
}  // namespace

// grid: (H_v * d_v) / kCols CTAs; CTA b scans columns kCols b .. of value head
// (kCols b) / d_v
__global__ void __launch_bounds__(kWarpsPerCta * 32) gdn_scan_kernel(GdnArgs a) {
  extern __shared__ __align__(16) uint8_t s_raw[];
  GdnSmem &sm = *reinterpret_cast<GdnSmem *>(s_raw);
  const int lane = threadIdx.x & 31, sub = lane % kLanes;
  const int col0 = blockIdx.x * kCols, h = col0 / a.dv, j0 = col0 - h * a.dv;
  const int hk = h / (a.Hv / a.Hk);
  const int cl = threadIdx.x / kLanes;  // column within the CTA
  const int j = j0 + cl;
  // this lane's state entries: 4 sub + 32 i + 0..3
  float s[kEpl];
  const long long sbase = (static_cast<long long>(h) * a.dv + j) * kDk;
  if (a.s_in) {
#pragma unroll
    for (int i = 0; i < kEpl / 4; ++i) {
      const float4 v4 = reinterpret_cast<const float4 *>(a.s_in + sbase)[sub + kLanes * i];
      s[4 * i] = v4.x;
      s[4 * i + 1] = v4.y;
      s[4 * i + 2] = v4.z;
      s[4 * i + 3] = v4.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kEpl; ++i) s[i] = 0.0f;
  }
  const int nblk = (a.T + kTb - 1) / kTb;
  if (nblk > 0) {
    stage_raw(sm, a, 0, min(kTb, a.T), h, hk, j0);
    cp_async_wait_all();
    __syncthreads();
    convert_block(sm, min(kTb, a.T));
    __syncthreads();
  }
  __nv_bfloat16 *orow = a.o + static_cast<long long>(h) * a.dv + j;
  const long long ostride = static_cast<long long>(a.Hv) * a.dv;
  for (int b = 0; b < nblk; ++b) {
    const int t0 = b * kTb, n = min(kTb, a.T - t0);
    if (b + 1 < nblk) stage_raw(sm, a, t0 + kTb, min(kTb, a.T - t0 - kTb), h, hk, j0);
    for (int tt = 0; tt < n; ++tt) {
      const float4 *kr = reinterpret_cast<const float4 *>(sm.kf[tt]) + sub;
      const float4 *qr = reinterpret_cast<const float4 *>(sm.qf[tt]) + sub;
      float4 k4[kEpl / 4];
      float r0 = 0.f, r1 = 0.f, p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int i = 0; i < kEpl / 4; ++i) {
        k4[i] = kr[kLanes * i];
        const float4 q4 = qr[kLanes * i];
        r0 = fmaf(s[4 * i], k4[i].x, r0);
        r1 = fmaf(s[4 * i + 1], k4[i].y, r1);
        r0 = fmaf(s[4 * i + 2], k4[i].z, r0);
        r1 = fmaf(s[4 * i + 3], k4[i].w, r1);
        p0 = fmaf(s[4 * i], q4.x, p0);
        p1 = fmaf(s[4 * i + 1], q4.y, p1);
        p0 = fmaf(s[4 * i + 2], q4.z, p0);
        p1 = fmaf(s[4 * i + 3], q4.w, p1);
      }
      float r = r0 + r1, p = p0 + p1;
#pragma unroll
      for (int o = kLanes / 2; o >= 1; o >>= 1) {
        r += __shfl_xor_sync(0xffffffffu, r, o);
        p += __shfl_xor_sync(0xffffffffu, p, o);
      }
      const float al = sm.as[tt], be = sm.bs[tt];
      const float u = be * (__bfloat162float(sm.vs[tt][cl]) - al * r);
      if (sub == 0) orow[(t0 + tt) * ostride] = __float2bfloat16_rn(fmaf(u, sm.c[tt], al * p));
#pragma unroll
      for (int i = 0; i < kEpl / 4; ++i) {
        s[4 * i] = fmaf(u, k4[i].x, al * s[4 * i]);
        s[4 * i + 1] = fmaf(u, k4[i].y, al * s[4 * i + 1]);
        s[4 * i + 2] = fmaf(u, k4[i].z, al * s[4 * i + 2]);
        s[4 * i + 3] = fmaf(u, k4[i].w, al * s[4 * i + 3]);
      }
    }
    if (b + 1 < nblk) {
      cp_async_wait_all();
      __syncthreads();  // every warp is done with this block's fp32 data
      convert_block(sm, min(kTb, a.T - t0 - kTb));
      __syncthreads();
    }
  }
  if (a.s_out) {
#pragma unroll
    for (int i = 0; i < kEpl / 4; ++i)
      reinterpret_cast<float4 *>(a.s_out + sbase)[sub + kLanes * i] =
          make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
  }
}

}  // namespace moe

extern "C" int gdn_scan(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *state_in, float *state_out, void *o, int T,
                        int n_k_heads, int n_v_heads, int d_k, int d_v, void *cuda_stream) {
  using namespace moe;
  if (T < 0 || n_k_heads <= 0 || n_v_heads <= 0 || d_k <= 0 || d_v <= 0) return MOE_ERR_INVALID_ARG;
  if (n_v_heads % n_k_heads != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !o)) return MOE_ERR_INVALID_ARG;
  if (d_k != kDk || d_v % kCols != 0) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(gdn_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(GdnSmem))) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!state_out && T == 0) return MOE_OK;
  GdnArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.k = static_cast<const __nv_bfloat16 *>(k);
  a.v = static_cast<const __nv_bfloat16 *>(v);
  a.alpha = alpha;
  a.beta = beta;
  a.s_in = state_in;
  a.s_out = state_out;
  a.o = static_cast<__nv_bfloat16 *>(o);
  a.T = T;
  a.Hk = n_k_heads;
  a.Hv = n_v_heads;
  a.dv = d_v;
  const int grid = n_v_heads * d_v / kCols;
  gdn_scan_kernel<<<grid, kWarpsPerCta * 32, sizeof(GdnSmem), static_cast<cudaStream_t>(cuda_stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
