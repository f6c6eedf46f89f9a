// gdn.cu -- the Gated DeltaNet recurrent scan (the C ABI in include/gdn.h).
//
// "Optimizing on-device inference for Apple Silicon", section "Keep the
// recurrent state on chip": the state matrix is split by columns, each
// column's slice loaded into registers once, carried through the whole scan
// and written back only at its end; state and gate are 32-bit float, the
// activations bfloat16.
//
// Token order.  Scanning token by token makes every token wait for a dot
// product, a cross-lane reduction and the update of the one before (measured
// ~550 cycles per token on one warp).  The scan takes 8 tokens at a time in
// the equivalent block form of the same recurrence (S the state before the 8
// tokens, A_i the product of the gates alpha_0..alpha_{i-1} inside the block,
// g(i, l) the product of alpha_{l+1}..alpha_{i-1}):
//     P_i = k_i . S,  Q_i = q_i . S
//     r_i = A_i P_i + sum_{l<i} g(i, l) (k_i . k_l) u_l    (what S recalls at k_i)
//     u_i = beta_i (v_i - alpha_i r_i)
//     o_i = A_{i+1} Q_i + sum_{l<=i} g(i+1, l) (q_i . k_l) u_l
//     S  <- A_8 S + sum_l g(8, l) u_l k_l
// which is the token-by-token rule S <- alpha S + u k, o = S . q written out
// (no division or rescaling: a zero gate makes the products zero).
//
// Tensor cores.  P, Q and the rank-8 update are matrix products of the state
// (columns x d_k) with the block's keys and queries, so they run on m16n8k8
// TF32 MMAs: a warp owns 16 columns and keeps their state in registers in the
// MMA accumulator layout (lane (g, c) holds columns g and g + 8 at d_k
// positions 8 n + 2 c, 8 n + 2 c + 1 of each 8-wide chunk n: 64 fp32).  The
// update accumulates straight into those registers.  As an operand the state
// is split into two TF32 parts (hi = S rounded to TF32, lo = S - hi rounded
// to TF32), and the keys and queries, bf16, are exact in TF32, so every
// product keeps ~21 significant bits and sums in fp32: the 32-bit state the
// pages ask for, at tensor-core issue rates.  For the products with the
// state, the MMA's k index is only summed over, so lane (g, c) feeds it the
// state entries it already holds (k = c and c + 4 from positions 2 c and
// 2 c + 1) and the key rows are read with the same mapping.
//
// The chain.  Only the u_i form a chain; each lane runs it for its two
// columns (the four lanes of a quad alike, after an all-gather of P and Q),
// right-looking: once u_l is known it enters every later recall and every
// output at once.  The coefficient tables come from the block's Gram
// products q_i . k_l and k_i . k_l on bf16 MMAs (exact products, fp32 sums).
//
// Staging.  A CTA is one warp (one value head's 16 columns); it copies the
// bf16 q and k of its key head, its v columns and the gates of the next 32
// tokens by cp.async into the second of two buffers while it scans the
// current 32, and reads q and k for the MMAs straight from the bf16 rows.
#include <cuda_bf16.h>

#include <cstddef>

#include "../../include/gdn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kDk = 128;               // d_k supported
constexpr int kCols = 16;              // columns per warp (= per CTA)
constexpr int kChunks = kDk / 8;       // 8-wide d_k chunks of the accumulator layout
constexpr int kTb = 32;                // tokens per staged block
constexpr int kB = 8;                  // tokens per block of the recurrence
constexpr int kSub = kTb / kB;
constexpr int kRow = kDk + 8;          // staged bf16 row: 272 B (row g on bank 4 g)

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

struct Stage {
  alignas(16) __nv_bfloat16 k[kTb][kRow];
  alignas(16) __nv_bfloat16 q[kTb][kRow];
  alignas(16) __nv_bfloat16 v[kTb][kCols];
  alignas(16) float al[kTb];
  alignas(16) float be[kTb];
};

struct GdnSmem {
  Stage st[2];
  BlockTab tab[kSub];
};
static_assert(offsetof(Stage, q) % 16 == 0 && offsetof(Stage, v) % 16 == 0 &&
                  sizeof(Stage) % 16 == 0 && (kRow * 2) % 16 == 0,
              "16-byte copies need 16-byte aligned rows");

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 f2z() { return make_float2(0.0f, 0.0f); }

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo, both TF32
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}
// the two bf16 of a 32-bit word as fp32 bit patterns (exact in TF32)
__device__ __forceinline__ uint32_t bf16_lo(uint32_t w) { return w << 16; }
__device__ __forceinline__ uint32_t bf16_hi(uint32_t w) { return w & 0xffff0000u; }
__device__ __forceinline__ uint32_t bf16_bits(__nv_bfloat16 x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(x)) << 16;
}

// Raw copies of tokens [t0, t0 + n) for this CTA (value head h, columns j0..)
// into stage s; rows past n are zeros with gate 1 and strength 0 (they leave
// the state unchanged).  One commit group per call.
__device__ __forceinline__ void stage_block(Stage &s, const GdnArgs &a, int t0, int n, int h,
                                            int hk, int j0, int lane) {
  for (int i = lane; i < kTb * 32; i += 32) {
    const int t = i >> 5, p = i & 31, which = p >> 4, piece = p & 15;
    __nv_bfloat16 *dst = (which ? s.q[t] : s.k[t]) + piece * 8;
    if (t < n)
      cp_async16(smem_u32(dst), (which ? a.q : a.k) +
                                    (static_cast<long long>(t0 + t) * a.Hk + hk) * kDk + piece * 8);
    else
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int i = lane; i < kTb * 4; i += 32) {
    const int t = i >> 2, p = i & 3;
    const long long tv = static_cast<long long>(t0 + t) * a.Hv + h;
    if (t < n) {
      if (p < 2)
        cp_async16(smem_u32(&s.v[t][p * 8]), a.v + tv * a.dv + j0 + p * 8);
      else if (p == 2)
        cp_async4(&s.al[t], a.alpha + tv);
      else
        cp_async4(&s.be[t], a.beta + tv);
    } else {
      if (p < 2)
        *reinterpret_cast<uint4 *>(&s.v[t][p * 8]) = make_uint4(0, 0, 0, 0);
      else if (p == 2)
        s.al[t] = 1.0f;
      else
        s.be[t] = 0.0f;
    }
  }
  cp_async_commit();
}

// Tables of 8-token block w of stage s.  Gram products on m16n8k16: A rows
// 0..7 = q_i, rows 8..15 = k_i; B columns = k_l; lane (g, c) feeds the MMA
// the 8 columns 32 j + 8 c .. of its rows (k = 2 c, 2 c + 1 from +0, +1;
// 2 c + 8, 2 c + 9 from +2, +3; the step's second MMA takes +4..+7) and the
// B side is read with the same mapping.
__device__ __forceinline__ void block_tables(const Stage &s, BlockTab &tb, int w, int lane) {
  const int g = lane >> 2, c4 = lane & 3, t = kB * w + g;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kDk / 32; ++j) {
    const uint4 qv = *reinterpret_cast<const uint4 *>(&s.q[t][32 * j + 8 * c4]);
    const uint4 kv = *reinterpret_cast<const uint4 *>(&s.k[t][32 * j + 8 * c4]);
    mma_bf16(acc, qv.x, kv.x, qv.y, kv.y, kv.x, kv.y);
    mma_bf16(acc, qv.z, kv.z, qv.w, kv.w, kv.z, kv.w);
  }
  // acc: (q_g . k_{2 c}, q_g . k_{2 c + 1}, k_g . k_{2 c}, k_g . k_{2 c + 1})
  const float *al = &s.al[kB * w];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int l = 2 * c4 + e;
    float gi = 1.0f;  // g(g, l) = alpha_{l+1} .. alpha_{g-1}
#pragma unroll
    for (int m = 0; m < kB; ++m)
      if (m > l && m < g) gi *= al[m];
    const float gi1 = (g > l) ? gi * al[g] : 1.0f;  // g(g + 1, l), l <= g
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
    tb.be[lane] = s.be[kB * w + lane];
  }
}
}  // namespace

// grid: (H_v * d_v) / kCols CTAs of one warp; CTA b scans columns kCols b ..
// of value head (kCols b) / d_v.  Lane (g, c) = (lane / 4, lane % 4) holds
// columns j0 + g and j0 + g + 8.
__global__ void __launch_bounds__(32) gdn_scan_kernel(GdnArgs a) {
  extern __shared__ __align__(16) uint8_t s_raw[];
  GdnSmem &sm = *reinterpret_cast<GdnSmem *>(s_raw);
  const int lane = threadIdx.x, g = lane >> 2, c = lane & 3;
  const int col0 = blockIdx.x * kCols, h = col0 / a.dv, j0 = col0 - h * a.dv;
  const int hk = h / (a.Hv / a.Hk);
  // st[n] = (S[g][8n + 2c], S[g][8n + 2c + 1], S[g + 8][8n + 2c], S[g + 8][8n + 2c + 1])
  float st[kChunks][4];
  const long long sb0 = (static_cast<long long>(h) * a.dv + j0 + g) * kDk + 2 * c;
  const long long sb8 = sb0 + 8LL * kDk;
#pragma unroll
  for (int n = 0; n < kChunks; ++n) {
    float2 x = f2z(), y = f2z();
    if (a.s_in) {
      x = *reinterpret_cast<const float2 *>(a.s_in + sb0 + 8 * n);
      y = *reinterpret_cast<const float2 *>(a.s_in + sb8 + 8 * n);
    }
    st[n][0] = x.x;
    st[n][1] = x.y;
    st[n][2] = y.x;
    st[n][3] = y.y;
  }
  const int nblk = (a.T + kTb - 1) / kTb;
  __nv_bfloat16 *ob = a.o + static_cast<long long>(h) * a.dv + j0 + g;
  const long long ostride = static_cast<long long>(a.Hv) * a.dv;
  if (nblk > 0) stage_block(sm.st[0], a, 0, min(kTb, a.T), h, hk, j0, lane);
  for (int b = 0; b < nblk; ++b) {
    const int t0 = b * kTb, n = min(kTb, a.T - t0);
    if (b + 1 < nblk)
      stage_block(sm.st[(b + 1) & 1], a, t0 + kTb, min(kTb, a.T - t0 - kTb), h, hk, j0, lane);
    else
      cp_async_commit();  // an empty group keeps the count below uniform
    cp_async_wait_group<1>();  // this block's copies have landed
    __syncwarp();
    const Stage &S = sm.st[b & 1];
#pragma unroll 1
    for (int w = 0; w < kSub; ++w) block_tables(S, sm.tab[w], w, lane);
    __syncwarp();
#pragma unroll 1
    for (int sb = 0; sb * kB < n; ++sb) {
      const BlockTab &tb = sm.tab[sb];
      const int tb0 = sb * kB;
      // P = S K^T, Q = S Q^T over the block's 8 tokens (hi and lo parts of
      // the state, even and odd chunks in separate accumulators)
      float acc[2][4][4];  // [chunk parity][P hi, P lo, Q hi, Q lo][fragment]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[x][y][z] = 0.0f;
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_tf32(st[ch][e], hi[e], lo[e]);
        const uint32_t kw = *reinterpret_cast<const uint32_t *>(&S.k[tb0 + g][8 * ch + 2 * c]);
        const uint32_t qw = *reinterpret_cast<const uint32_t *>(&S.q[tb0 + g][8 * ch + 2 * c]);
        float(&A)[4][4] = acc[ch & 1];
        // a0 = (g, k c) <- entry 2c, a1 = (g + 8, k c), a2 = (g, k c + 4) <- entry 2c + 1, a3 = (g + 8, k c + 4)
        mma_tf32(A[0], hi[0], hi[2], hi[1], hi[3], bf16_lo(kw), bf16_hi(kw));
        mma_tf32(A[1], lo[0], lo[2], lo[1], lo[3], bf16_lo(kw), bf16_hi(kw));
        mma_tf32(A[2], hi[0], hi[2], hi[1], hi[3], bf16_lo(qw), bf16_hi(qw));
        mma_tf32(A[3], lo[0], lo[2], lo[1], lo[3], bf16_lo(qw), bf16_hi(qw));
      }
      // this lane: P, Q of columns g, g + 8 at tokens 2c, 2c + 1
      float pf[4], qf[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pf[e] = (acc[0][0][e] + acc[0][1][e]) + (acc[1][0][e] + acc[1][1][e]);
        qf[e] = (acc[0][2][e] + acc[0][3][e]) + (acc[1][2][e] + acc[1][3][e]);
      }
      // all 8 tokens for both columns from the quad
      float p0[kB], p1[kB], q0[kB], q1[kB];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int src = (lane & ~3) | s;
        p0[2 * s] = __shfl_sync(0xffffffffu, pf[0], src);
        p0[2 * s + 1] = __shfl_sync(0xffffffffu, pf[1], src);
        p1[2 * s] = __shfl_sync(0xffffffffu, pf[2], src);
        p1[2 * s + 1] = __shfl_sync(0xffffffffu, pf[3], src);
        q0[2 * s] = __shfl_sync(0xffffffffu, qf[0], src);
        q0[2 * s + 1] = __shfl_sync(0xffffffffu, qf[1], src);
        q1[2 * s] = __shfl_sync(0xffffffffu, qf[2], src);
        q1[2 * s + 1] = __shfl_sync(0xffffffffu, qf[3], src);
      }
      // the chain, right-looking, for columns g (0) and g + 8 (1)
      float R0[kB], R1[kB], O0[kB], O1[kB], u0[kB], u1[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        R0[i] = tb.A[i] * p0[i];
        R1[i] = tb.A[i] * p1[i];
        O0[i] = tb.A[i + 1] * q0[i];
        O1[i] = tb.A[i + 1] * q1[i];
      }
#pragma unroll
      for (int l = 0; l < kB; ++l) {
        const float al = tb.al[l], be = tb.be[l];
        u0[l] = be * fmaf(-al, R0[l], __bfloat162float(S.v[tb0 + l][g]));
        u1[l] = be * fmaf(-al, R1[l], __bfloat162float(S.v[tb0 + l][g + 8]));
#pragma unroll
        for (int i = l + 1; i < kB; ++i) {
          R0[i] = fmaf(tb.C[l][i], u0[l], R0[i]);
          R1[i] = fmaf(tb.C[l][i], u1[l], R1[i]);
        }
#pragma unroll
        for (int i = l; i < kB; ++i) {
          O0[i] = fmaf(tb.D[l][i], u0[l], O0[i]);
          O1[i] = fmaf(tb.D[l][i], u1[l], O1[i]);
        }
      }
      // lane c writes tokens 2c, 2c + 1 of both columns
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if ((i >> 1) == c && tb0 + i < n) {
          const long long off = (t0 + tb0 + i) * ostride;
          ob[off] = __float2bfloat16_rn(O0[i]);
          ob[off + 8] = __float2bfloat16_rn(O1[i]);
        }
      }
      // S <- A_8 S + W K with W[col][l] = g(8, l) u_l: A operand rows g, g + 8,
      // k = token c and c + 4
      float w0 = 0.f, w1 = 0.f, w4 = 0.f, w5 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i == c) {
          w0 = tb.E[i] * u0[i];
          w1 = tb.E[i] * u1[i];
          w4 = tb.E[i + 4] * u0[i + 4];
          w5 = tb.E[i + 4] * u1[i + 4];
        }
      }
      uint32_t wh[4], wl[4];
      split_tf32(w0, wh[0], wl[0]);  // a0 = (g, k c)
      split_tf32(w1, wh[1], wl[1]);  // a1 = (g + 8, k c)
      split_tf32(w4, wh[2], wl[2]);  // a2 = (g, k c + 4)
      split_tf32(w5, wh[3], wl[3]);  // a3 = (g + 8, k c + 4)
      const float a8 = tb.A[kB];
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
        for (int e = 0; e < 4; ++e) st[ch][e] *= a8;
        // b0 = (k = token c, column g of the chunk), b1 = (token c + 4, column g)
        const uint32_t b0 = bf16_bits(S.k[tb0 + c][8 * ch + g]);
        const uint32_t b1 = bf16_bits(S.k[tb0 + c + 4][8 * ch + g]);
        mma_tf32(st[ch], wh[0], wh[1], wh[2], wh[3], b0, b1);
        mma_tf32(st[ch], wl[0], wl[1], wl[2], wl[3], b0, b1);
      }
    }
    __syncwarp();  // done with this stage before it is refilled
  }
  cp_async_wait_group<0>();
  if (a.s_out) {
#pragma unroll
    for (int n = 0; n < kChunks; ++n) {
      *reinterpret_cast<float2 *>(a.s_out + sb0 + 8 * n) = make_float2(st[n][0], st[n][1]);
      *reinterpret_cast<float2 *>(a.s_out + sb8 + 8 * n) = make_float2(st[n][2], st[n][3]);
    }
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
  gdn_scan_kernel<<<grid, 32, sizeof(GdnSmem), static_cast<cudaStream_t>(cuda_stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
