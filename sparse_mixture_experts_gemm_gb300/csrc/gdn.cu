// gdn.cu -- the Gated DeltaNet recurrent scan (the C ABI in include/gdn.h).
//
// "Optimizing on-device inference for Apple Silicon", section "Keep the
// recurrent state on chip": the state matrix is split by columns, each
// column's slice loaded into registers once, carried through the whole scan
// and written back only at its end; partial results are exchanged by lane
// operations, not through shared memory; state and gate are 32-bit float,
// the activations bfloat16.
//
// Column split.  The pages give each column a whole SIMD group; here a
// column belongs to L = 8 lanes (16 fp32 entries per lane at d_k = 128, four
// columns per warp), which keeps the whole state (2 MB for 32 value heads of
// 128 x 128) in registers on ~7 warps per SM with 3 shuffle rounds per
// reduction.  Lane s of a column holds the entries 4 s + 32 i + 0..3 (i =
// 0..3), so the 8 lanes of a column read 128 contiguous bytes of a key per
// instruction (no shared-memory bank conflicts).
//
// Token order.  Scanning token by token makes every token wait for a dot
// product, a cross-lane reduction and the update of the one before (measured
// ~550 cycles per token on one warp).  The scan therefore takes 8 tokens at a
// time in the equivalent block form of the same recurrence (S the state
// before the 8 tokens, A_i the product of the gates alpha_0..alpha_{i-1}
// inside the block, g(i, l) the product of alpha_{l+1}..alpha_{i-1}):
//     P_i = k_i . S,  Q_i = q_i . S                  (16 independent reductions)
//     r_i = A_i P_i + sum_{l<i} g(i, l) (k_i . k_l) u_l    (what S recalls at k_i)
//     u_i = beta_i (v_i - alpha_i r_i)
//     o_i = A_{i+1} Q_i + sum_{l<=i} g(i+1, l) (q_i . k_l) u_l
//     S  <- A_8 S + sum_l g(8, l) u_l k_l
// which is the token-by-token rule S <- alpha S + u k, o = S . q written out
// (no division, no rescaling: a zero gate makes the products zero).  Only
// the u_i form a chain (two dependent FMAs per token); the dot products, the
// reductions and the update are independent work.  The coefficient tables
// come once per CTA from the block's Gram products q_i . k_l and k_i . k_l,
// computed on warp-level bf16 MMAs (products of bf16 values are exact in
// fp32; fp32 accumulation).
//
// Staging.  A CTA (4 warps, the 16 columns of one value head) copies the bf16
// q and k of its key head, its v columns and the gates of the next 32 tokens
// by cp.async while it scans the current 32, then converts q and k to fp32
// once for all of its columns and builds the four 8-token blocks' tables.
#include <cuda_bf16.h>

#include <cstddef>

#include "../../include/gdn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kDk = 128;                    // d_k supported
constexpr int kLanes = 8;                   // lanes per column
constexpr int kEpl = kDk / kLanes;          // state entries per lane
constexpr int kCols = 16;                   // columns per CTA (one value head's)
constexpr int kWarpsPerCta = kCols * kLanes / 32;
constexpr int kTb = 32;                     // tokens per staged block
constexpr int kB = 8;                       // tokens per block of the recurrence
constexpr int kSub = kTb / kB;              // blocks of the recurrence per staged block
constexpr int kRawStride = kDk + 32;        // raw row: 320 B (rows g, g + 1 in other banks)
static_assert(kB <= 8 && kTb % kB == 0, "the Gram MMA covers at most 8 tokens");

struct GdnArgs {
  const __nv_bfloat16 *q, *k, *v;
  const float *alpha, *beta, *s_in;
  float *s_out;
  __nv_bfloat16 *o;
  int T, Hk, Hv, dv;
};

// Tables of one 8-token block (tokens i, l = 0..7 of the block), stored by
// l so that the chain reads one contiguous row per token.
struct BlockTab {
  float C[kB][kB];   // [l][i] = g(i, l) (k_i . k_l), l < i (0 elsewhere)
  float D[kB][kB];   // [l][i] = g(i + 1, l) (q_i . k_l), l <= i (0 elsewhere)
  float A[kB + 1];   // A_i = alpha_0 .. alpha_{i-1}
  float E[kB];       // g(8, l)
  float al[kB], be[kB];
};

// Every array that cp.async writes 16 bytes at a time, or that is read as
// float4 / uint4, starts on a 16-byte boundary (checked below).
struct GdnSmem {
  alignas(16) float kf[kTb][kDk];           // fp32 activations of the current block
  alignas(16) float qf[kTb][kDk];
  alignas(16) BlockTab tab[kSub];
  alignas(16) __nv_bfloat16 vs[kTb][kCols];   // the current block's v
  alignas(16) __nv_bfloat16 kr[kTb][kRawStride];  // raw bf16 of the next block
  alignas(16) __nv_bfloat16 qr[kTb][kRawStride];
  alignas(16) __nv_bfloat16 vr[kTb][kCols];
  alignas(16) float ar[kTb];
  alignas(16) float br[kTb];
};
static_assert(offsetof(GdnSmem, qf) % 16 == 0 && offsetof(GdnSmem, tab) % 16 == 0 &&
                  offsetof(GdnSmem, kr) % 16 == 0 && offsetof(GdnSmem, qr) % 16 == 0 &&
                  offsetof(GdnSmem, vr) % 16 == 0 && (kRawStride * 2) % 16 == 0 &&
                  (kCols * 2) % 16 == 0,
              "16-byte copies and vector reads need 16-byte aligned rows");

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// Raw copies of tokens [t0, t0 + n) for this CTA (value head h, columns j0..);
// the rows of the block past n are zeros with gate 1 and strength 0, so they
// leave the state unchanged.
__device__ __forceinline__ void stage_raw(GdnSmem &sm, const GdnArgs &a, int t0, int n, int h,
                                          int hk, int j0) {
  for (int i = threadIdx.x; i < kTb * 32; i += blockDim.x) {
    const int t = i >> 5, p = i & 31, which = p >> 4, piece = p & 15;
    __nv_bfloat16 *dst = (which ? sm.qr[t] : sm.kr[t]) + piece * 8;
    if (t < n) {
      const long long src = (static_cast<long long>(t0 + t) * a.Hk + hk) * kDk + piece * 8;
      cp_async16(smem_u32(dst), (which ? a.q : a.k) + src);
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  for (int i = threadIdx.x; i < kTb * 4; i += blockDim.x) {
    const int t = i >> 2, p = i & 3;
    const long long tv = static_cast<long long>(t0 + t) * a.Hv + h;
    if (t < n) {
      if (p < 2)
        cp_async16(smem_u32(&sm.vr[t][p * 8]), a.v + tv * a.dv + j0 + p * 8);
      else if (p == 2)
        cp_async4(&sm.ar[t], a.alpha + tv);
      else
        cp_async4(&sm.br[t], a.beta + tv);
    } else {
      if (p < 2)
        *reinterpret_cast<uint4 *>(&sm.vr[t][p * 8]) = make_uint4(0, 0, 0, 0);
      else if (p == 2)
        sm.ar[t] = 1.0f;
      else
        sm.br[t] = 0.0f;
    }
  }
  cp_async_commit();
}

// Warp w builds the tables of the staged block's 8-token block w.  Gram
// products on m16n8k16: A rows 0..7 = q_i, rows 8..15 = k_i; B columns =
// k_l.  The MMA's k index is only summed over, so lane (g, c4) feeds it the
// 8 columns 32 j + 8 c4 .. of its rows (k = 2 c4, 2 c4 + 1 from +0, +1;
// 2 c4 + 8, 2 c4 + 9 from +2, +3; the step's second MMA takes +4..+7) and the
// B side is read with the same mapping.
__device__ __forceinline__ void block_tables(GdnSmem &sm, int w, int lane) {
  const int g = lane >> 2, c4 = lane & 3, t = kB * w + min(g, kB - 1);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kDk / 32; ++j) {
    const uint4 qv = *reinterpret_cast<const uint4 *>(&sm.qr[t][32 * j + 8 * c4]);
    const uint4 kv = *reinterpret_cast<const uint4 *>(&sm.kr[t][32 * j + 8 * c4]);
    mma_bf16(acc, qv.x, kv.x, qv.y, kv.y, kv.x, kv.y);
    mma_bf16(acc, qv.z, kv.z, qv.w, kv.w, kv.z, kv.w);
  }
  // acc: (q_g . k_{2 c4}, q_g . k_{2 c4 + 1}, k_g . k_{2 c4}, k_g . k_{2 c4 + 1})
  BlockTab &tb = sm.tab[w];
  const float *al = &sm.ar[kB * w];  // this block's gates
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int l = 2 * c4 + e;
    if (g >= kB || l >= kB) continue;
    // g(i, l) = alpha_{l+1} .. alpha_{i-1}: for i = g (C) and i = g + 1 (D)
    float gi = 1.0f;
#pragma unroll
    for (int m = 0; m < kB; ++m)
      if (m > l && m < g) gi *= al[m];
    const float gi1 = (g > l) ? gi * sm.ar[t] : 1.0f;  // g(g + 1, l) (l <= g); alpha_g
    tb.C[l][g] = l < g ? gi * acc[2 + e] : 0.0f;
    tb.D[l][g] = l <= g ? gi1 * acc[e] : 0.0f;
  }
  if (lane <= kB) {  // A_i, i = lane
    float p = 1.0f;
#pragma unroll
    for (int m = 0; m < kB; ++m)
      if (m < lane) p *= al[m];
    tb.A[lane] = p;
  }
  if (lane < kB) {  // E_l = g(8, l), l = lane; gates and strengths
    float p = 1.0f;
#pragma unroll
    for (int m = 0; m < kB; ++m)
      if (m > lane) p *= al[m];
    tb.E[lane] = p;
    tb.al[lane] = al[lane];
    tb.be[lane] = sm.br[kB * w + lane];
  }
}

// raw block -> fp32 q, k and v for the scan; the tables of its 8-token blocks
__device__ __forceinline__ void convert_block(GdnSmem &sm) {
  static_assert(kTb * kDk / 4 % (kWarpsPerCta * 32) == 0, "whole passes");
#pragma unroll
  for (int i = threadIdx.x; i < kTb * kDk / 4; i += kWarpsPerCta * 32) {
    const int t = i / (kDk / 4), e = (i - t * (kDk / 4)) * 4;
    const uint2 kk = *reinterpret_cast<const uint2 *>(&sm.kr[t][e]);
    const uint2 qq = *reinterpret_cast<const uint2 *>(&sm.qr[t][e]);
    const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.x));
    const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kk.y));
    const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq.x));
    const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qq.y));
    *reinterpret_cast<float4 *>(&sm.kf[t][e]) = make_float4(k0.x, k0.y, k1.x, k1.y);
    *reinterpret_cast<float4 *>(&sm.qf[t][e]) = make_float4(q0.x, q0.y, q1.x, q1.y);
  }
  for (int i = threadIdx.x; i < kTb * kCols; i += blockDim.x)
    sm.vs[i / kCols][i % kCols] = sm.vr[i / kCols][i % kCols];
  for (int w = threadIdx.x >> 5; w < kSub; w += kWarpsPerCta) block_tables(sm, w, threadIdx.x & 31);
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
  // this lane's entries 4 sub + 32 c + 0..3 as pairs: s2[2 c] = (+0, +1), s2[2 c + 1] = (+2, +3)
  float2 s2[kEpl / 2];
  const long long sbase = (static_cast<long long>(h) * a.dv + j) * kDk;
  if (a.s_in) {
#pragma unroll
    for (int c = 0; c < kEpl / 4; ++c) {
      const float4 v4 = reinterpret_cast<const float4 *>(a.s_in + sbase)[sub + kLanes * c];
      s2[2 * c] = f2(v4.x, v4.y);
      s2[2 * c + 1] = f2(v4.z, v4.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < kEpl / 2; ++c) s2[c] = f2(0.0f, 0.0f);
  }
  const int nblk = (a.T + kTb - 1) / kTb;
  if (nblk > 0) {
    stage_raw(sm, a, 0, min(kTb, a.T), h, hk, j0);
    cp_async_wait_all();
    __syncthreads();
    convert_block(sm);
    __syncthreads();
  }
  __nv_bfloat16 *orow = a.o + static_cast<long long>(h) * a.dv + j;
  const long long ostride = static_cast<long long>(a.Hv) * a.dv;
  for (int b = 0; b < nblk; ++b) {
    const int t0 = b * kTb, n = min(kTb, a.T - t0);
    if (b + 1 < nblk) stage_raw(sm, a, t0 + kTb, min(kTb, a.T - t0 - kTb), h, hk, j0);
    for (int sb = 0; sb * kB < n; ++sb) {
      const BlockTab &tb = sm.tab[sb];
      const int tb0 = sb * kB;
      // P_i, Q_i: this lane's part (chunk by chunk, 16 independent
      // accumulator chains), then one butterfly for all 16
      float2 pk[kB], pqq[kB], pq[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        pk[i] = f2(0.f, 0.f);
        pqq[i] = f2(0.f, 0.f);
      }
#pragma unroll
      for (int c = 0; c < kEpl / 4; ++c) {
#pragma unroll
        for (int i = 0; i < kB; ++i) {
          const float4 k4 = reinterpret_cast<const float4 *>(sm.kf[tb0 + i])[sub + kLanes * c];
          const float4 q4 = reinterpret_cast<const float4 *>(sm.qf[tb0 + i])[sub + kLanes * c];
          pk[i] = __ffma2_rn(s2[2 * c], f2(k4.x, k4.y), pk[i]);
          pk[i] = __ffma2_rn(s2[2 * c + 1], f2(k4.z, k4.w), pk[i]);
          pqq[i] = __ffma2_rn(s2[2 * c], f2(q4.x, q4.y), pqq[i]);
          pqq[i] = __ffma2_rn(s2[2 * c + 1], f2(q4.z, q4.w), pqq[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) pq[i] = f2(pk[i].x + pk[i].y, pqq[i].x + pqq[i].y);
#pragma unroll
      for (int o = kLanes / 2; o >= 1; o >>= 1) {
#pragma unroll
        for (int i = 0; i < kB; ++i)
          pq[i] = __fadd2_rn(pq[i], f2(__shfl_xor_sync(0xffffffffu, pq[i].x, o),
                                       __shfl_xor_sync(0xffffffffu, pq[i].y, o)));
      }
      // the chain, right-looking: once u_l is known it enters every later
      // token's recall and every output at once (independent FMAs), so the
      // chain is the u_l alone
      float R[kB], O[kB], u[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        R[i] = tb.A[i] * pq[i].x;
        O[i] = tb.A[i + 1] * pq[i].y;
      }
#pragma unroll
      for (int l = 0; l < kB; ++l) {
        const float v = __bfloat162float(sm.vs[tb0 + l][cl]);
        u[l] = tb.be[l] * fmaf(-tb.al[l], R[l], v);
#pragma unroll
        for (int i = l + 1; i < kB; ++i) R[i] = fmaf(tb.C[l][i], u[l], R[i]);
#pragma unroll
        for (int i = l; i < kB; ++i) O[i] = fmaf(tb.D[l][i], u[l], O[i]);
      }
      if (sub == 0) {
#pragma unroll
        for (int i = 0; i < kB; ++i)
          if (tb0 + i < n) orow[(t0 + tb0 + i) * ostride] = __float2bfloat16_rn(O[i]);
      }
      // S <- A_8 S + sum_l g(8, l) u_l k_l
      const float a8 = tb.A[kB];
#pragma unroll
      for (int c = 0; c < kEpl / 2; ++c) s2[c] = __fmul2_rn(f2(a8, a8), s2[c]);
#pragma unroll
      for (int l = 0; l < kB; ++l) {
        const float w = tb.E[l] * u[l];
        const float4 *kr = reinterpret_cast<const float4 *>(sm.kf[tb0 + l]) + sub;
#pragma unroll
        for (int c = 0; c < kEpl / 4; ++c) {
          const float4 k4 = kr[kLanes * c];
          s2[2 * c] = __ffma2_rn(f2(w, w), f2(k4.x, k4.y), s2[2 * c]);
          s2[2 * c + 1] = __ffma2_rn(f2(w, w), f2(k4.z, k4.w), s2[2 * c + 1]);
        }
      }
    }
    if (b + 1 < nblk) {
      cp_async_wait_all();
      __syncthreads();  // every warp is done with this block's fp32 data and tables
      convert_block(sm);
      __syncthreads();
    }
  }
  if (a.s_out) {
#pragma unroll
    for (int c = 0; c < kEpl / 4; ++c)
      reinterpret_cast<float4 *>(a.s_out + sbase)[sub + kLanes * c] =
          make_float4(s2[2 * c].x, s2[2 * c].y, s2[2 * c + 1].x, s2[2 * c + 1].y);
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
