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
// The dequantisation is folded into the dot product: for the columns of one
// group,  sum_c (s q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c,  with the
// codes turned into the floats 128 + q by byte permutes (no integer-to-float
// conversion) and 128 * sum_c x_c taken back once per group.  The values x
// (the token, or h for the down projection) sit in registers; the codes,
// scales and biases come through shared memory.
//
// Kernels (chained with programmatic dependent launch): A the router as one
// thread-block cluster that publishes the layer's top-k once; B the gate/up
// rows of the k chosen experts and of the shared one; C the down rows and the
// combine.  Static weights (the shared expert's gate/up blocks, C's rows once
// the choice is known) are requested before griddepcontrol.wait.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf16f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Sum over the 8 codes of one 32-bit word (columns c .. c + 7: byte j holds
// column c + 2j in its low nibble, c + 2j + 1 in its high nibble) of
// (128 + q) * x.  Each code becomes the float 128 + q with one byte permute:
// the nibble, isolated in a byte, lands in bits 16..19 under the exponent byte
// 0x43 (128.0f), which is exact.  The caller removes 128 * sum(x) once per
// group, so no code is converted with an integer-to-float instruction.
__device__ __forceinline__ float q4_word_dot(uint32_t w, const float *x, float acc) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sel = 0x4055u | (static_cast<uint32_t>(j) << 8);
    acc = fmaf(__uint_as_float(__byte_perm(lo, 0x43u, sel)), x[2 * j], acc);
    acc = fmaf(__uint_as_float(__byte_perm(hi, 0x43u, sel)), x[2 * j + 1], acc);
  }
  return acc;
}

// s * sum q x + b * sum x for one group's share, given p = sum (128 + q) x and
// sx = sum x over the same columns.
__device__ __forceinline__ float q4_finish(float p, float sx, uint16_t s, uint16_t b) {
  const float sf = bf16f(s);
  return sf * p + fmaf(-128.0f, sf, bf16f(b)) * sx;
}

// Warp reduce-scatter of N partial sums (N a power of two, <= 32): returns
// the warp total of value lane >> (5 - log2 N).  N - 1 + (5 - log2 N)
// shuffles instead of 5 N.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int h = N / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const float send = up ? v[j] : v[j + h];
      const float keep = up ? v[j + h] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 / N; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// ---------------------------------------------------------------- gate/up rows
// Kernel B's items are (slot s, row f), item = s * F + f, over the k routed
// slots and the shared expert (slot k): h[item] = silu(gate . x) * (up . x).
// A CTA of 16 warps takes a block of n consecutive items (one slot; F is a
// multiple of n), whose code bytes, scales and biases are contiguous in both
// matrices.  A row of d columns is 2G chunks of 32 codes (16 bytes), G =
// d / 64; a team of ceil(2G / 32) warps shares a row, its lane slot q owning
// chunk q (consecutive lanes read consecutive 16 bytes: no bank conflicts)
// with the token's 32 values of that chunk in registers.  Each team takes
// kQB items of the block.
constexpr int kQB = 4;
constexpr int kGateUpWarps = 16;

struct XChunk {
  float x[32];
  float sx;
};

// 32 token values (one chunk) from the CTA's shared-memory copy of the token.
__device__ __forceinline__ void load_x_chunk(XChunk &xc, const uint4 *tok, int chunk) {
  const uint4 *p = tok + chunk * 4;
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = p[j];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      xc.x[8 * j + 2 * t] = __uint_as_float(u[t] << 16);
      xc.x[8 * j + 2 * t + 1] = __uint_as_float(u[t] & 0xFFFF0000u);
      s += xc.x[8 * j + 2 * t] + xc.x[8 * j + 2 * t + 1];
    }
  }
  xc.sx = s;
}

__device__ __forceinline__ float chunk_dot(const uint4 &c, const float (&x)[32]) {
  float p0 = q4_word_dot(c.x, x, 0.0f);
  float p1 = q4_word_dot(c.y, x + 8, 0.0f);
  p0 = q4_word_dot(c.z, x + 16, p0);
  p1 = q4_word_dot(c.w, x + 24, p1);
  return p0 + p1;
}

// Block of rows of one 4-bit matrix staged in shared memory.
struct QBlock {
  const uint4 *c;     // [rows][d / 32] chunks
  const uint16_t *s;  // [rows][G]
  const uint16_t *b;
};

// chunk q of row r against its token chunk: that chunk's share of the row's dot
__device__ __forceinline__ float qblock_chunk_dot(const QBlock &m, int r, int G, int q,
                                                  const XChunk &xc) {
  const int g = q >> 1;
  return q4_finish(chunk_dot(m.c[r * 2 * G + q], xc.x), xc.sx, m.s[r * G + g], m.b[r * G + g]);
}

// Team geometry of a kGateUpWarps-warp CTA for rows of d columns (the team
// count a power of two, so that the block size divides F).
struct Team {
  int wt, teams, team, tw, q;
  bool active;
  __device__ Team(int d, int warp, int lane) {
    const int chunks = 2 * (d / kQ4Group);
    wt = (chunks + 31) / 32;
    teams = 1;
    while (2 * teams * wt <= kGateUpWarps) teams *= 2;
    team = warp / wt;
    tw = warp - team * wt;
    q = tw * 32 + lane;
    active = team < teams && q < chunks;
  }
};

// Shared-memory plan of one block of n rows of a gate and an up matrix:
// codes, then scales and biases, then the token.
struct GateUpSmem {
  QBlock g, u;
  const uint4 *x;
  __device__ GateUpSmem(uint8_t *base, int n, int d) {
    const int G = d / kQ4Group;
    const int cb = n * d / 2, sb = n * G * 2;
    g.c = reinterpret_cast<const uint4 *>(base);
    u.c = reinterpret_cast<const uint4 *>(base + cb);
    g.s = reinterpret_cast<const uint16_t *>(base + 2 * cb);
    g.b = reinterpret_cast<const uint16_t *>(base + 2 * cb + sb);
    u.s = reinterpret_cast<const uint16_t *>(base + 2 * cb + 2 * sb);
    u.b = reinterpret_cast<const uint16_t *>(base + 2 * cb + 3 * sb);
    x = reinterpret_cast<const uint4 *>(base + 2 * cb + 4 * sb);
  }
};

__host__ __device__ constexpr size_t gateup_smem_bytes(int n, int d) {
  return static_cast<size_t>(n) * d + static_cast<size_t>(n) * (d / kQ4Group) * 8 +
         static_cast<size_t>(d) * 2;
}

// All threads: cp.async of bytes (a multiple of 16) from src to dst.
__device__ __forceinline__ void cp_async_range(uint8_t *dst, const void *src, int bytes) {
  const uint8_t *s8 = static_cast<const uint8_t *>(src);
  const uint32_t d0 = smem_u32(dst);
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) cp_async16(d0 + 16 * i, s8 + 16 * i);
}

// Stages of a block (rows row0 .. row0 + n - 1 of mg and mu): stage j holds
// rows j n / ns .. (j + 1) n / ns - 1.  The code bytes of a stage (16 KB per
// matrix at d >= 2048) go by one bulk copy per matrix, issued by thread 0
// with the stage's byte count; the scales and biases by cp.async from every
// thread, each thread arriving on the stage barrier once its copies landed
// (barrier count: blockDim.x + 1).  One bulk copy per 16 KB keeps the per-copy
// cost of the copy engine small against its transfer time, where thread
// copies of the whole block would stream far below the memory's rate.
__device__ __forceinline__ void gateup_issue(uint8_t *base, const Q4Mat &mg, const Q4Mat &mu,
                                             long long row0, int n, int d, int ns,
                                             uint64_t *bar) {
  const int G = d / kQ4Group;
  const int cb = n * d / 2, sb = n * G * 2;
  const int rows = n / ns;
  const int scb = rows * d / 2, ssb = rows * G * 2;  // per stage
  for (int j = 0; j < ns; ++j) {
    const long long r = row0 + static_cast<long long>(j) * rows;
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(smem_u32(&bar[j]), 2 * scb);
      bulk_g2s(base + j * scb, mg.c + r * (d / 2), scb, &bar[j]);
      bulk_g2s(base + cb + j * scb, mu.c + r * (d / 2), scb, &bar[j]);
    }
    cp_async_range(base + 2 * cb + j * ssb, mg.s + r * G, ssb);
    cp_async_range(base + 2 * cb + sb + j * ssb, mg.b + r * G, ssb);
    cp_async_range(base + 2 * cb + 2 * sb + j * ssb, mu.s + r * G, ssb);
    cp_async_range(base + 2 * cb + 3 * sb + j * ssb, mu.b + r * G, ssb);
    cp_async_arrive(smem_u32(&bar[j]));
  }
}

}  // namespace

// ---------------------------------------------------------------- A: router + top-k
// One cluster of ceil(E / 16) CTAs of 16 warps, one warp per expert logit
// (bf16 router rows requested before the dependency wait, the token copied
// once per CTA).  Every logit goes straight into CTA 0's shared memory; after
// one cluster barrier CTA 0 picks the layer's top-k (dsel).  No global
// round trip, fence or arrival counter sits between the logits and the
// choice.
constexpr int kRouterWarps = 16;

__global__ void __launch_bounds__(kRouterWarps * 32) decode_router_q4_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __shared__ float s_lg[256];  // CTA 0: the layer's logits
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d;
  const int nvec = d * 2 / 16;
  const int e = blockIdx.x * kRouterWarps + warp;
  const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.wr) +
                                                     static_cast<long long>(e) * d);
  RowPre pr;
  if (e < a.E) row_prefetch(pr, row, nvec, lane);
  pdl_launch_dependents();
  pdl_wait();
  uint4 *xs = reinterpret_cast<uint4 *>(qsm);
  load_token(xs, a.x, nvec);
  if (e < a.E) {
    const float acc = warp_sum(row_dot_pre<__nv_bfloat16>(pr, row, xs, nvec, lane));
    if (lane == 0) st_cluster_f32(&s_lg[e], 0, acc + (a.bias ? a.bias[e] : 0.0f));
  }
  cluster_sync_all();  // every CTA of the cluster reaches this: no return above
  if (cluster_ctarank() != 0 || warp != 0) return;
  unsigned key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ee = lane + 32 * i;
    key[i] = ee < a.E ? fkey(s_lg[ee]) : 0u;
  }
  topk_from_keys(key, a.E, a.k, lane, s_sel, s_selw);
  __syncwarp();
  if (lane < a.k) {
    for (int r = 0; r < kSelReplicas; ++r) {
      a.dsel[32 * r + lane] = s_sel[lane];
      a.dsel[32 * r + 8 + lane] = __float_as_int(s_selw[lane]);
    }
  }
  write_routing(a, s_sel, s_selw, lane);
}

// ---------------------------------------------------------------- B: gate/up
// Blocks of the shared expert's items (static rows) are copied before the
// dependency wait; routed blocks read their expert from dsel after it.
__global__ void __launch_bounds__(kGateUpWarps * 32) decode_gateup_q4_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ float red[kGateUpWarps][2 * kQB];
  __shared__ int s_row0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F, G = d / kQ4Group;
  const Team tm(d, warp, lane);
  const int n = tm.teams * kQB;
  // copy stages: the compute left after the last stage lands is 1 / ns of the
  // block (more stages issue more, smaller copies, and measured slower)
  const int ns = tm.teams >= 2 ? 2 : 1;
  const int it0 = blockIdx.x * n;
  const int s = it0 / F, f0 = it0 - s * F;
  const bool shared_blk = s >= a.k;
  if (threadIdx.x == 0) {
    for (int j = 0; j < ns; ++j) mbar_init(smem_u32(&bar[j]), blockDim.x + 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (shared_blk) gateup_issue(qsm, a.q.sg, a.q.su, f0, n, d, ns, bar);
  pdl_wait();
  // kernel A is complete: kernel C may launch (it reads only the top-k)
  pdl_launch_dependents();
  // the token (the previous layer's output) and this block's expert, in one
  // round of L2 reads
  const GateUpSmem sm(qsm, n, d);
  uint4 *xs = const_cast<uint4 *>(sm.x);
  if (!shared_blk && threadIdx.x == 0)
    s_row0 = ld_cg_s32(a.dsel + 32 * (blockIdx.x % kSelReplicas) + s) * F + f0;
  const uint4 *xg = static_cast<const uint4 *>(a.x);
  for (int i = threadIdx.x; i < d * 2 / 16; i += blockDim.x) xs[i] = ld_cg16(xg + i);
  __syncthreads();
  if (!shared_blk) gateup_issue(qsm, a.q.g, a.q.u, s_row0, n, d, ns, bar);
  XChunk xc;
  if (tm.active) load_x_chunk(xc, sm.x, tm.q);
  // team j takes per = kQB / ns items of every stage, so all warps compute on
  // each stage as it lands: the team's item m = st per + jj is row
  // st n / ns + j per + jj of the block.  Threads outside a team read row 0
  // with a zero token.
  const int per = kQB / ns;
  const int team_c = tm.team < tm.teams ? tm.team : 0;
  const int q_c = tm.active ? tm.q : 0;
  if (!tm.active) {
#pragma unroll
    for (int c = 0; c < 32; ++c) xc.x[c] = 0.0f;
    xc.sx = 0.0f;
  }
  float v[2 * kQB];
  bool ok = true;
#pragma unroll
  for (int m = 0; m < kQB; ++m) {
    const int st = m / per, jj = m - st * per;
    if (jj == 0) ok = mbar_wait(smem_u32(&bar[st]), 0, MOE_WAIT_LIMIT_CYCLES, nullptr) && ok;
    const int r = st * (n / ns) + team_c * per + jj;
    v[2 * m] = qblock_chunk_dot(sm.g, r, G, q_c, xc);
    v[2 * m + 1] = qblock_chunk_dot(sm.u, r, G, q_c, xc);
  }
  if (!ok) {
#pragma unroll
    for (int m = 0; m < 2 * kQB; ++m) v[m] = 0.0f;
    if (lane == 0) report_error(a.status, MOE_ERR_DEVICE_TIMEOUT, KID_DECODE * 100 + SITE_STAGE);
  }
  const float t = warp_reduce_scatter<2 * kQB>(v, lane);
  if ((lane & 3) == 0) red[warp][lane >> 2] = t;
  __syncthreads();
  const int i = threadIdx.x;
  if (i < n) {
    const int st = i / (n / ns), rem = i - st * (n / ns);
    const int team = rem / per, jj = rem - team * per;
    const int m = st * per + jj;
    float g = 0.0f, u = 0.0f;
    for (int w = 0; w < tm.wt; ++w) {
      g += red[team * tm.wt + w][2 * m];
      u += red[team * tm.wt + w][2 * m + 1];
    }
    a.h[it0 + i] = g / (1.0f + __expf(-g)) * u;
  }
}

// ---------------------------------------------------------------- C: down + combine
// A CTA computes output rows i0 .. i0 + R - 1.  Their down-matrix rows of
// every slot (codes, scales, biases) are copied to shared memory with cp.async
// as soon as the top-k is known, before the wait for h.  Thread t owns CPL
// consecutive columns of one slot's h (slot t / (F / CPL)), those h values in
// registers; its partial for row r is weighted by the slot's routing weight,
// reduce-scattered over the warp and summed over the warps in shared memory.
constexpr int kQR = 16;  // output rows per CTA, at most

// All threads: cp.async of `bytes` from src to dst in pieces of `piece`
// bytes (4, 8 or 16; both addresses and bytes multiples of it).
__device__ __forceinline__ void cp_async_pieces(void *dst, const void *src, int bytes, int piece) {
  const uint8_t *s8 = static_cast<const uint8_t *>(src);
  const uint32_t d0 = smem_u32(dst);
  for (int o = threadIdx.x * piece; o < bytes; o += blockDim.x * piece) {
    if (piece == 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d0 + o), "l"(s8 + o)
                   : "memory");
    else if (piece == 8)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d0 + o), "l"(s8 + o)
                   : "memory");
    else
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d0 + o), "l"(s8 + o)
                   : "memory");
  }
}

__host__ __device__ constexpr size_t down_smem_bytes(int R, int nslot, int F) {
  return static_cast<size_t>(R) * nslot * (F / 2 + 2 * (F / 32));
}

template <int CPL>
__global__ void __launch_bounds__(640) decode_down_q4_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __shared__ int s_sel[kMaxTopK];
  __shared__ float s_selw[kMaxTopK];
  __shared__ float acc_s[20][kQR];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F, GF = F / kQ4Group;
  const int sps = F / CPL;  // slices per slot
  const int nslot = a.k + a.n_shared;
  const int slot = threadIdx.x / sps, sl = threadIdx.x - slot * sps;
  const bool active = slot < nslot;
  const int R = a.c_rows;
  const int i0 = blockIdx.x * R;
  const int nr = (d - i0) < R ? (d - i0) : R;  // rows of this CTA
  // shared memory: codes [nslot][R][F / 2], scales and biases [nslot][R][GF]
  // (a slot's rows i0 .. i0 + nr - 1 are consecutive rows of its matrix)
  uint8_t *cs = qsm;
  uint16_t *ss = reinterpret_cast<uint16_t *>(qsm + static_cast<size_t>(R) * nslot * (F / 2));
  uint16_t *bs = ss + R * nslot * GF;
  pdl_launch_dependents();
  // the layer's top-k (kernel A finished before kernel B let this kernel start)
  if (static_cast<int>(threadIdx.x) < a.k) {
    const int *rep = a.dsel + 32 * (blockIdx.x % kSelReplicas);
    s_sel[threadIdx.x] = ld_cg_s32(rep + threadIdx.x);
    s_selw[threadIdx.x] = __int_as_float(ld_cg_s32(rep + 8 + threadIdx.x));
  }
  __syncthreads();
  {
    const int sbp = F / 32 < 16 ? F / 32 : 16;  // scale/bias piece: 4, 8 or 16 bytes
    for (int sl_ = 0; sl_ < nslot; ++sl_) {
      const Q4Mat &mat = sl_ < a.k ? a.q.d : a.q.sd;
      const long long row = (sl_ < a.k ? static_cast<long long>(s_sel[sl_]) * d : 0) + i0;
      cp_async_pieces(cs + static_cast<size_t>(sl_) * R * (F / 2), mat.c + row * (F / 2),
                      nr * (F / 2), 16);
      cp_async_pieces(ss + sl_ * R * GF, mat.s + row * GF, nr * GF * 2, sbp);
      cp_async_pieces(bs + sl_ * R * GF, mat.b + row * GF, nr * GF * 2, sbp);
    }
    cp_async_commit();
  }
  pdl_wait();
  float hv[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) hv[j] = 0.0f;
  float sh = 0.0f, wslot = 0.0f;
  if (active) {
    const float *hp = a.h + slot * F + sl * CPL;
#pragma unroll
    for (int j = 0; j < CPL / 4; ++j) {
      const float4 v = ld_cg_f32x4(hp + 4 * j);
      hv[4 * j] = v.x;
      hv[4 * j + 1] = v.y;
      hv[4 * j + 2] = v.z;
      hv[4 * j + 3] = v.w;
      sh += (v.x + v.y) + (v.z + v.w);
    }
    wslot = slot < a.k ? s_selw[slot] : 1.0f;
  }
  cp_async_wait_all();
  __syncthreads();
  const int g = (active ? sl : 0) * CPL / kQ4Group;
  // Branch-free over the rows, so that their dependent FMA chains interleave:
  // rows past nr read row 0 and are zeroed; threads past the last slot read
  // slot 0 with h = 0 and weight 0.
  const int slot_c = active ? slot : 0, sl_c = active ? sl : 0;
  const float wuse = active ? wslot : 0.0f;
  float part[kQR];
#pragma unroll
  for (int r = 0; r < kQR; ++r) {
    const int rsi = slot_c * R + (r < nr ? r : 0);
    const uint32_t *cw = reinterpret_cast<const uint32_t *>(
        cs + static_cast<size_t>(rsi) * (F / 2) + sl_c * (CPL / 2));
    float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) {
      if (j & 1)
        p1 = q4_word_dot(cw[j], hv + 8 * j, p1);
      else
        p0 = q4_word_dot(cw[j], hv + 8 * j, p0);
    }
    const float v = q4_finish(p0 + p1, sh, ss[rsi * GF + g], bs[rsi * GF + g]);
    part[r] = r < nr ? wuse * v : 0.0f;
  }
  const float t = warp_reduce_scatter<kQR>(part, lane);
  if ((lane & 1) == 0) acc_s[warp][lane >> 1] = t;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  if (static_cast<int>(threadIdx.x) < nr) {
    float o = 0.0f;
    for (int w = 0; w < nw; ++w) o += acc_s[w][threadIdx.x];
    reinterpret_cast<__nv_bfloat16 *>(a.out)[i0 + threadIdx.x] = __float2bfloat16_rn(o);
  }
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
template <typename K>
cudaError_t launch_q(K kern, int grid, int threads, size_t smem, cudaStream_t st, bool pdl,
                     const DecodeArgs &a, int cluster = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

// Kernels B and C each take more than half of an SM's shared memory, so that
// no SM holds two CTAs of either: two CTAs of B on one SM share its copy
// engine and finish last, and the layer waits for them.
constexpr size_t kOnePerSm = 116 * 1024;
size_t one_per_sm(size_t bytes) { return bytes > kOnePerSm ? bytes : kOnePerSm; }

// items per kernel-B block: kQB per team, as the Team geometry counts teams
int items_per_cta(int d) {
  const int wt = (2 * (d / kQ4Group) + 31) / 32;
  int teams = 1;
  while (2 * teams * wt <= kGateUpWarps) teams *= 2;
  return teams * kQB;
}
size_t gateup_smem(int d) { return gateup_smem_bytes(items_per_cta(d), d); }

// columns of h per thread in kernel C: the fewest that keep the CTA within
// 640 threads (more warps hide more of the dependent-FMA latency)
int down_cpl(const DecodeArgs &a) {
  const int slots = a.k + a.n_shared;
  for (int cpl : {8, 16})
    if (slots * (a.F / cpl) <= 640) return cpl;
  return 0;
}
}  // namespace

// one cluster: the whole grid (at most 16 CTAs for E <= 256)
cudaError_t launch_decode_router_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int ncta = (a.E + kRouterWarps - 1) / kRouterWarps;
  return launch_q(decode_router_q4_kernel, ncta, kRouterWarps * 32, static_cast<size_t>(a.d) * 2,
                  st, pdl, a, ncta);
}
// one CTA per block of items; F is a multiple of the block
cudaError_t launch_decode_gateup_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int per = items_per_cta(a.d);
  const int grid = (a.k + a.n_shared) * a.F / per;
  return launch_q(decode_gateup_q4_kernel, grid, kGateUpWarps * 32, one_per_sm(gateup_smem(a.d)),
                  st, pdl, a);
}
cudaError_t launch_decode_down_q4(const DecodeArgs &a, cudaStream_t st, bool pdl) {
  const int sms = sm_count();
  const int cpl = down_cpl(a);
  if (sms == 0 || cpl == 0) return cudaErrorInvalidValue;
  DecodeArgs b = a;
  int R = (a.d + sms - 1) / sms;
  R = R < 1 ? 1 : (R > kQR ? kQR : R);
  b.c_rows = R;
  const int nslot = a.k + a.n_shared;
  const int threads = (nslot * (a.F / cpl) + 31) / 32 * 32;
  const int grid = (a.d + R - 1) / R;
  const size_t smem = one_per_sm(down_smem_bytes(R, nslot, a.F));
  if (cpl == 8) return launch_q(decode_down_q4_kernel<8>, grid, threads, smem, st, pdl, b);
  return launch_q(decode_down_q4_kernel<16>, grid, threads, smem, st, pdl, b);
}

// Kernel B stages a block of gate/up rows and the token: at most 72 KB
// (n d = 64 K for every supported d, plus the scales and biases) + 32 KB.
// Kernel C stages at most 16 rows x (k + 1) F / 2 (+ 1/8) bytes: 90 KB.
// Both launch with kOnePerSm (116 KB), above either.  Kernel A runs as one
// cluster of up to 16 CTAs (above the portable 8).
cudaError_t decode_q4_set_smem_attr() {
  const int bytes = static_cast<int>(kOnePerSm);
  cudaError_t e = cudaFuncSetAttribute(decode_router_q4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_router_q4_kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_gateup_q4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_down_q4_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_down_q4_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
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
