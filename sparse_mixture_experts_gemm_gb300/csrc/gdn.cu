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
// TF32 MMAs.  A group of 16 columns is held by 4 warps that split d_k: warp
// w keeps the state of all 16 columns at d_k chunks 4 w .. 4 w + 3 in
// registers in the MMA accumulator layout (lane (g, c) holds columns g and
// g + 8 at d_k positions 8 n + 2 c, 8 n + 2 c + 1 of chunk n: 16 fp32).  A
// CTA owns one group, or two (8 warps) when one group per CTA would leave
// two CTAs on some SM.  The update
// accumulates straight into those registers.  As an operand the state is
// split into two TF32 parts (hi = the top 11 significant bits of S, lo the
// top 11 of S - hi), and the keys and queries, bf16, are exact in TF32, so
// every product keeps ~22 significant bits and sums in fp32: the 32-bit
// state the pages ask for, at tensor-core issue rates.  For the products
// with the state, the MMA's k index is only summed over, so lane (g, c) feeds
// it the state entries it already holds (k = c and c + 4 from positions 2 c
// and 2 c + 1) and the key rows are read with the same mapping.
//
// The chain.  The warps' partial P and Q meet in shared memory (two buffers);
// warp 0 alone sums them, runs the chain for the CTA's columns, one column
// per lane (right-looking: once u_l is known it enters every later recall and
// every output at once; only the u_i form a chain), writes the outputs and
// leaves g(8, l) u_l in shared memory for the update, which every warp then
// applies to its quarter (two barriers per 8 tokens).  Running the chain in
// one warp instead of four halves the instructions the CTA issues.
//
// Staging.  The CTA copies the bf16 q and k of its key head, its v columns
// and the gates of the next 32 tokens by cp.async into the second of two
// buffers while it scans the current 32, and reads q and k for the MMAs
// straight from the bf16 rows.
#include <cuda_bf16.h>

#include <cstddef>

#include "../../include/gdn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kDk = 128;               // d_k supported
constexpr int kCols = 16;              // columns per group (the MMAs' M)
constexpr int kGMax = 2;               // column groups per CTA: 2, or 1 where d_v is not a multiple of 32
constexpr int kWarps = 4;              // warps per column group, each a quarter of d_k
constexpr int kChunks = kDk / 8 / kWarps;  // 8-wide d_k chunks per warp
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
// l so that the chain reads whole rows (16-byte vectors; the zeros outside
// the triangles make the full-row updates exact).
struct alignas(16) BlockTab {
  float C[kB][kB];   // [l][i] = g(i, l) (k_i . k_l), l < i (0 elsewhere)
  float D[kB][kB];   // [l][i] = g(i + 1, l) (q_i . k_l), l <= i (0 elsewhere)
  float A[kB + 4];   // A_i = alpha_0 .. alpha_{i-1}, i = 0..8 (then padding)
  float E[kB];       // g(8, l)
  float al[kB], be[kB];
};
static_assert(sizeof(BlockTab) % 16 == 0 && offsetof(BlockTab, A) % 16 == 0 &&
                  offsetof(BlockTab, E) % 16 == 0 && offsetof(BlockTab, al) % 16 == 0 &&
                  offsetof(BlockTab, be) % 16 == 0,
              "the chain reads the tables as 16-byte vectors");

__device__ __forceinline__ void ld8(const float *p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

struct Stage {
  alignas(16) __nv_bfloat16 k[kTb][kRow];
  alignas(16) __nv_bfloat16 q[kTb][kRow];
  alignas(16) __nv_bfloat16 v[kTb][kGMax * kCols];
  alignas(16) float al[kTb];
  alignas(16) float be[kTb];
};

struct GdnSmem {
  Stage st[2];
  BlockTab tab[2][kSub];  // by staged-block parity
  // [buffer][warp][P, Q][column][token] partial sums; rows of 12 floats so
  // that the 8 columns a quarter-warp reads start in different banks
  float part[2][kGMax * kWarps][2][kCols][kB + 4];
  alignas(16) float wu[kGMax * kCols][kB + 4];  // g(8, l) u_l of the CTA's columns (rows padded as part)
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

// x ~ hi + lo, both TF32 (the low 13 bits cleared): hi keeps the top 11
// significant bits of x, lo = x - hi exactly and then its own top 11, so the
// pair carries ~22 of x's 24 bits; two integer ops and one FADD, no
// conversion instruction
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}
// the two bf16 of a 32-bit word as fp32 bit patterns (exact in TF32)
__device__ __forceinline__ uint32_t bf16_lo(uint32_t w) { return w << 16; }
__device__ __forceinline__ uint32_t bf16_hi(uint32_t w) { return w & 0xffff0000u; }
__device__ __forceinline__ uint32_t bf16_bits(__nv_bfloat16 x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(x)) << 16;
}

// Raw copies of tokens [t0, t0 + n) for this CTA (value head h, G groups of
// 16 columns from j0) into stage s by the CTA's G * 128 threads; rows past n
// are zeros with gate 1 and strength 0 (they leave the state unchanged).  One
// commit group per call.
template <int G>
__device__ __forceinline__ void stage_block(Stage &s, const GdnArgs &a, int t0, int n, int h,
                                            int hk, int j0, int tid) {
  constexpr int nt = G * kWarps * 32, pv = 2 * G;  // threads; 16-byte pieces of v per token
  for (int i = tid; i < kTb * 32; i += nt) {
    const int t = i >> 5, p = i & 31, which = p >> 4, piece = p & 15;
    __nv_bfloat16 *dst = (which ? s.q[t] : s.k[t]) + piece * 8;
    if (t < n)
      cp_async16(smem_u32(dst), (which ? a.q : a.k) +
                                    (static_cast<long long>(t0 + t) * a.Hk + hk) * kDk + piece * 8);
    else
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int i = tid; i < kTb * (pv + 2); i += nt) {
    const int t = i / (pv + 2), p = i - t * (pv + 2);
    const long long tv = static_cast<long long>(t0 + t) * a.Hv + h;
    if (t < n) {
      if (p < pv)
        cp_async16(smem_u32(&s.v[t][p * 8]), a.v + tv * a.dv + j0 + p * 8);
      else if (p == pv)
        cp_async4(&s.al[t], a.alpha + tv);
      else
        cp_async4(&s.be[t], a.beta + tv);
    } else {
      if (p < pv)
        *reinterpret_cast<uint4 *>(&s.v[t][p * 8]) = make_uint4(0, 0, 0, 0);
      else if (p == pv)
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

// grid: (H_v * d_v) / (16 G) CTAs of 4 G warps; CTA b scans columns 16 G b ..
// of value head (16 G b) / d_v.  Lane (g, c) = (lane / 4, lane % 4) of warp w
// holds columns j0 + 16 (w / 4) + g and + 8 at d_k chunks 4 (w % 4) ..; lane
// l of warp 0 runs the chain of column j0 + l (with G = 1, lanes 16..31 repeat
// lanes 0..15).  Two groups per CTA give every lane of the chain warp a column
// of its own, and with d_v = 128 one CTA per SM for 32 value heads.
template <int G>
__global__ void __launch_bounds__(G * kWarps * 32, 1) gdn_scan_kernel(GdnArgs a) {
  constexpr int kColsCta = G * kCols;
  extern __shared__ __align__(16) uint8_t s_raw[];
  GdnSmem &sm = *reinterpret_cast<GdnSmem *>(s_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int jc = lane & (kColsCta - 1);  // the column this lane runs the chain for
  const int jg = jc >> 4, jl = jc & 15;  // its group and place in the group
  const int col0 = blockIdx.x * kColsCta, h = col0 / a.dv, j0 = col0 - h * a.dv;
  const int hk = h / (a.Hv / a.Hk);
  const int cg = warp / kWarps;               // this warp's column group
  const int ch0 = (warp % kWarps) * kChunks;  // this warp's first d_k chunk
  // st[n] = (S[g][8m + 2c], S[g][8m + 2c + 1], S[g + 8][8m + 2c], S[g + 8][8m + 2c + 1]), m = ch0 + n
  float st[kChunks][4];
  const long long sb0 =
      (static_cast<long long>(h) * a.dv + j0 + kCols * cg + g) * kDk + 8 * ch0 + 2 * c;
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
  __nv_bfloat16 *ob = a.o + static_cast<long long>(h) * a.dv + j0 + jc;
  const long long ostride = static_cast<long long>(a.Hv) * a.dv;
  int it = 0;  // 8-token blocks done (selects the partial-sum buffer)
  // The first staged block's copies and tables up front; those of block b + 1
  // during block b: its copies are issued at b's start, every thread waits
  // for its own before the first barrier of b's third 8-token block (every
  // block but the last is whole), and warps 1..3 build the tables while warp
  // 0 runs the chains of b's third and fourth 8-token blocks.
  if (nblk > 0) {
    stage_block<G>(sm.st[0], a, 0, min(kTb, a.T), h, hk, j0, tid);
    cp_async_wait_group<0>();
    __syncthreads();
    if (warp < kSub) block_tables(sm.st[0], sm.tab[0][warp], warp, lane);
    __syncthreads();
  }
  for (int b = 0; b < nblk; ++b) {
    const int t0 = b * kTb, n = min(kTb, a.T - t0);
    const bool next = b + 1 < nblk;
    if (next)
      stage_block<G>(sm.st[(b + 1) & 1], a, t0 + kTb, min(kTb, a.T - t0 - kTb), h, hk, j0, tid);
    const Stage &S = sm.st[b & 1];
#pragma unroll 1
    for (int sb = 0; sb * kB < n; ++sb, ++it) {
      const BlockTab &tb = sm.tab[b & 1][sb];
      const int tb0 = sb * kB;
      // this warp's part of P = S K^T and Q = S Q^T (hi and lo parts of the
      // state, even and odd chunks in separate accumulators)
      float acc[2][4][4];  // [chunk parity][P hi, P lo, Q hi, Q lo][fragment]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y)
#pragma unroll
          for (int z = 0; z < 4; ++z) acc[x][y][z] = 0.0f;
#pragma unroll
      for (int nn = 0; nn < kChunks; ++nn) {
        const int m = ch0 + nn;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_tf32(st[nn][e], hi[e], lo[e]);
        const uint32_t kw = *reinterpret_cast<const uint32_t *>(&S.k[tb0 + g][8 * m + 2 * c]);
        const uint32_t qw = *reinterpret_cast<const uint32_t *>(&S.q[tb0 + g][8 * m + 2 * c]);
        float(&A)[4][4] = acc[nn & 1];
        // a0 = (g, k c) <- entry 2c, a1 = (g + 8, k c), a2 = (g, k c + 4) <- entry 2c + 1, a3 = (g + 8, k c + 4)
        mma_tf32(A[0], hi[0], hi[2], hi[1], hi[3], bf16_lo(kw), bf16_hi(kw));
        mma_tf32(A[1], lo[0], lo[2], lo[1], lo[3], bf16_lo(kw), bf16_hi(kw));
        mma_tf32(A[2], hi[0], hi[2], hi[1], hi[3], bf16_lo(qw), bf16_hi(qw));
        mma_tf32(A[3], lo[0], lo[2], lo[1], lo[3], bf16_lo(qw), bf16_hi(qw));
      }
      // partials of columns g, g + 8 at tokens 2c, 2c + 1 into shared memory
      float(&pt)[kGMax * kWarps][2][kCols][kB + 4] = sm.part[it & 1];
#pragma unroll
      for (int pq = 0; pq < 2; ++pq) {
        const int y = 2 * pq;
        *reinterpret_cast<float2 *>(&pt[warp][pq][g][2 * c]) =
            make_float2((acc[0][y][0] + acc[0][y + 1][0]) + (acc[1][y][0] + acc[1][y + 1][0]),
                        (acc[0][y][1] + acc[0][y + 1][1]) + (acc[1][y][1] + acc[1][y + 1][1]));
        *reinterpret_cast<float2 *>(&pt[warp][pq][g + 8][2 * c]) =
            make_float2((acc[0][y][2] + acc[0][y + 1][2]) + (acc[1][y][2] + acc[1][y + 1][2]),
                        (acc[0][y][3] + acc[0][y + 1][3]) + (acc[1][y][3] + acc[1][y + 1][3]));
      }
      // (a block with a successor is whole: it has 8-token blocks 0..3)
      if (next && sb == 2) cp_async_wait_group<0>();  // block b + 1's copies, this thread's
      __syncthreads();
      if (next && sb >= 2 && warp > 0) {
        // the next block's tables, one per warp and 8-token block, while warp
        // 0 runs this block's chain: tables 0..3 now with two column groups,
        // else 0..2 now and 3 in the next one
        const int w = sb == 2 ? (warp <= kSub ? warp - 1 : -1) : (G == 1 && warp == 1 ? 3 : -1);
        if (w >= 0) block_tables(sm.st[(b + 1) & 1], sm.tab[(b + 1) & 1][w], w, lane);
      }
      if (warp == 0) {
        // P, Q of column jc at the 8 tokens, summed over the warps in order
        float p[kB], q[kB];
#pragma unroll
        for (int i = 0; i < kB; ++i) p[i] = q[i] = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float4 pv = *reinterpret_cast<const float4 *>(&pt[kWarps * jg + w][0][jl][4 * hf]);
            const float4 qv = *reinterpret_cast<const float4 *>(&pt[kWarps * jg + w][1][jl][4 * hf]);
            p[4 * hf] += pv.x;
            p[4 * hf + 1] += pv.y;
            p[4 * hf + 2] += pv.z;
            p[4 * hf + 3] += pv.w;
            q[4 * hf] += qv.x;
            q[4 * hf + 1] += qv.y;
            q[4 * hf + 2] += qv.z;
            q[4 * hf + 3] += qv.w;
          }
        }
        // the chain, right-looking, for column jc
        float R[kB], O[kB], u[kB], Av[kB], alv[kB], bev[kB], ev[kB];
        ld8(tb.A, Av);  // A_0 .. A_7
        const float a8v = reinterpret_cast<const float4 *>(tb.A + kB)->x;  // A_8 (16-byte aligned)
        ld8(tb.al, alv);
        ld8(tb.be, bev);
        ld8(tb.E, ev);
#pragma unroll
        for (int i = 0; i < kB; ++i) {
          R[i] = Av[i] * p[i];
          O[i] = (i + 1 < kB ? Av[i + 1] : a8v) * q[i];
        }
#pragma unroll
        for (int l = 0; l < kB; ++l) {
          u[l] = bev[l] * fmaf(-alv[l], R[l], __bfloat162float(S.v[tb0 + l][jc]));
          float cr[kB], dr[kB];
          ld8(tb.C[l], cr);
          ld8(tb.D[l], dr);
#pragma unroll
          for (int i = l + 1; i < kB; ++i) R[i] = fmaf(cr[i], u[l], R[i]);
#pragma unroll
          for (int i = l; i < kB; ++i) O[i] = fmaf(dr[i], u[l], O[i]);
        }
        if (lane < kColsCta) {
#pragma unroll
          for (int i = 0; i < kB; ++i)
            if (tb0 + i < n) ob[(t0 + tb0 + i) * ostride] = __float2bfloat16_rn(O[i]);
          float4 *dst = reinterpret_cast<float4 *>(&sm.wu[jc][0]);
          dst[0] = make_float4(ev[0] * u[0], ev[1] * u[1], ev[2] * u[2], ev[3] * u[3]);
          dst[1] = make_float4(ev[4] * u[4], ev[5] * u[5], ev[6] * u[6], ev[7] * u[7]);
        }
      }
      __syncthreads();  // the scaled deltas are in shared memory
      // S <- A_8 S + W K with W[col][l] = g(8, l) u_l: A operand rows g, g + 8,
      // k = token c and c + 4
      const int wr = kCols * cg + g;  // this lane's rows of W: columns wr, wr + 8
      const float w0 = sm.wu[wr][c], w1 = sm.wu[wr + 8][c], w4 = sm.wu[wr][c + 4], w5 = sm.wu[wr + 8][c + 4];
      const float a8 = reinterpret_cast<const float4 *>(tb.A + kB)->x;
      uint32_t wh[4], wl[4];
      split_tf32(w0, wh[0], wl[0]);  // a0 = (g, k c)
      split_tf32(w1, wh[1], wl[1]);  // a1 = (g + 8, k c)
      split_tf32(w4, wh[2], wl[2]);  // a2 = (g, k c + 4)
      split_tf32(w5, wh[3], wl[3]);  // a3 = (g + 8, k c + 4)
#pragma unroll
      for (int nn = 0; nn < kChunks; ++nn) {
        const int m = ch0 + nn;
#pragma unroll
        for (int e = 0; e < 4; ++e) st[nn][e] *= a8;
        // b0 = (k = token c, column g of the chunk), b1 = (token c + 4, column g)
        const uint32_t b0 = bf16_bits(S.k[tb0 + c][8 * m + g]);
        const uint32_t b1 = bf16_bits(S.k[tb0 + c + 4][8 * m + g]);
        mma_tf32(st[nn], wh[0], wh[1], wh[2], wh[3], b0, b1);
        mma_tf32(st[nn], wl[0], wl[1], wl[2], wl[3], b0, b1);
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
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
  // 16-byte copies of q, k, v rows; 8-byte state reads and writes; 4-byte gates
  auto misaligned = [](const void *ptr, uintptr_t n) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) % n) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(state_in, 8) ||
      misaligned(state_out, 8) || misaligned(alpha, 4) || misaligned(beta, 4) || misaligned(o, 2))
    return MOE_ERR_ALIGNMENT;
  if (cudaFuncSetAttribute(gdn_scan_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(GdnSmem))) != cudaSuccess ||
      cudaFuncSetAttribute(gdn_scan_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  // Two groups of 16 columns per CTA where a head's columns split into them
  // and one group per CTA would put two CTAs on some SM: the two groups'
  // state products then share an SM's tensor issue inside one CTA instead of
  // two CTAs' (measured 249 vs 257 us for 32 heads of 128 columns), while
  // with fewer columns one group per CTA keeps each CTA's chain shortest
  // (212 vs 262 us for a single head).
  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (d_v % (kGMax * kCols) == 0 && static_cast<long long>(n_v_heads) * d_v / kCols > sms)
    gdn_scan_kernel<kGMax><<<n_v_heads * d_v / (kGMax * kCols), kGMax * kWarps * 32, sizeof(GdnSmem), st>>>(a);
  else
    gdn_scan_kernel<1><<<n_v_heads * d_v / kCols, kWarps * 32, sizeof(GdnSmem), st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
