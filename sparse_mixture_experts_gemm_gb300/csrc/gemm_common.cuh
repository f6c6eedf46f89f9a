// gemm_common.cuh -- pieces shared by the bf16 and the 4-bit grouped GEMMs:
// the epilogue's activation and row stores, the device-side group table and
// tile decoding, and the shared-memory ring that hands claimed tile ids from
// the producer to the other roles of a CTA.
#pragma once
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// silu(z) = z / (1 + e^-z) with the fast (approximate-reciprocal) division:
// relative error ~1e-7, far below the bf16 rounding of h; for z -> -inf the
// denominator overflows to inf and the quotient is 0, the function's limit.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 32 consecutive bytes from eight words (dst 32-byte aligned): a thread's
// store covers whole 32-byte sectors, so none reaches L2 as two halves
__device__ __forceinline__ void st_global_32b(void *dst, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 32 floats of one output row (dst 64-byte aligned for bf16, 128 for fp32)
template <typename T>
__device__ __forceinline__ void store32(T *dst, const float (&v)[32]);
template <>
__device__ __forceinline__ void store32<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[q * 16 + 2 * j], v[q * 16 + 2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t *>(&b);
    }
    st_global_32b(dst + q * 16, w);
  }
}
template <>
__device__ __forceinline__ void store32<float>(float *dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __float_as_uint(v[q * 8 + j]);
    st_global_32b(dst + q * 8, w);
  }
}

// Group table built by every CTA of a grouped GEMM: s_off[g] = first slot of
// group g (g <= E), s_mt[g] = first M tile of group g (g <= E + 1; group E is
// the shared expert).
struct GroupTable {
  const int *off;
  const int *mt;
};

// Tokens of the rows of routed tile tl that a gather thread copies: rows
// r0 + 16 i (i < kRows) that exist, -1 for the others.  The token comes from
// the router's per-expert list (tokens in rank order) or, without lists, from
// the slot permutation.  Both were written by kernels the GEMM waited for at
// griddepcontrol.wait (an asm with a memory clobber: no load moves above
// it): ordinary loads, so the 8 threads that share a row hit in L1, all
// issued together.
template <int kRows>
__device__ __forceinline__ void gather_tokens(const GemmParams &p, const GroupTable &gt,
                                              const GemmTile &tl, int r0, int (&tok)[kRows]) {
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int r = r0 + 16 * i;
    tok[i] = -1;
    if (r < tl.rows)
      tok[i] = p.list ? p.list[static_cast<long long>(tl.group) * p.list_stride +
                               (tl.a_row - gt.off[tl.group]) + r]
                      : p.perm[tl.a_row + r];
  }
}

__device__ __forceinline__ GemmTile decode_tile(const GroupTable &gt, const GemmParams &p, int i,
                                                int n_cols, bool down) {
  const int E = p.n_routed;
  int lo = 0, hi = E;  // largest g with nt * mt[g] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.nt * gt.mt[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int mtg = gt.mt[g + 1] - gt.mt[g];
  const int local = i - p.nt * gt.mt[g];
  const int n = local / mtg, m = local - (local / mtg) * mtg;
  GemmTile t;
  t.group = g;
  t.n0 = n * n_cols;
  t.pad[0] = t.pad[1] = t.pad[2] = 0;
  if (g < E) {
    const int cnt = gt.off[g + 1] - gt.off[g];
    t.a_row = gt.off[g] + m * kBM;
    t.out_row = t.a_row;
    t.rows = min(kBM, cnt - m * kBM);
  } else {
    t.rows = min(kBM, p.T - m * kBM);
    t.out_row = p.A + m * kBM;
    t.a_row = down ? t.out_row : m * kBM;  // gate/up reads tokens in order
  }
  return t;
}

// Every thread of the CTA: the group table (s_off[g] for g <= E, s_mt[g] =
// first M tile of group g for g <= E + 1, group E the shared expert), built
// from the offsets the routing wrote.  Warp 2 runs the exclusive scan.
__device__ __forceinline__ void build_group_table(const GemmParams &p, int *s_off, int *s_mt,
                                                  int warp, int lane) {
  const int E = p.n_routed;
  if (p.counts_in) {
    // the cluster router left only the histogram: scan it here
    for (int g = threadIdx.x; g < E; g += blockDim.x)
      s_off[g] = p.counts_in[static_cast<long long>(g) * kCountStride];
    __syncthreads();
    if (warp == 2) {
      const int per = (E + 31) / 32;
      int sum = 0;
      for (int q = 0; q < per; ++q) {
        const int i = lane * per + q;
        if (i < E) sum += s_off[i];
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
          const int c = s_off[i];
          if (blockIdx.x == 0 && p.counts_out) p.counts_out[i] += c;  // summed over a call's chunks
          s_off[i] = run;
          run += c;
        }
      }
      if (lane == 31) s_off[E] = incl;
    }
    __syncthreads();
    if (blockIdx.x == 0 && p.offsets_out)
      for (int g = threadIdx.x; g <= E; g += blockDim.x) p.offsets_out[g] = s_off[g];
  } else {
    for (int g = threadIdx.x; g <= E; g += blockDim.x) s_off[g] = p.offsets[g];
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    // the gate/up GEMM that read them has finished (this kernel waited for it)
    if (p.clear_counts)
      for (int g = threadIdx.x; g < E; g += blockDim.x)
        p.clear_counts[static_cast<long long>(g) * kCountStride] = 0;
    if (p.clear_ctr && threadIdx.x == 0) *p.clear_ctr = 0;
  }
  for (int g = threadIdx.x; g <= E; g += blockDim.x) {
    const int rows = g < E ? s_off[g + 1] - s_off[g] : (p.n_shared ? p.T : 0);
    s_mt[g] = (rows + kBM - 1) / kBM;
  }
  __syncthreads();
  if (warp == 2) {
    const int n = E + 1;
    const int per = (n + 31) / 32;
    int sum = 0;
    for (int q = 0; q < per; ++q) {
      const int i = lane * per + q;
      if (i < n) sum += s_mt[i];
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
      if (i < n) {
        const int v = s_mt[i];
        s_mt[i] = run;
        run += v;
      }
    }
    if (lane == 31) s_mt[n] = incl;
  }
}

// Work items of the grouped GEMMs in cluster-pair mode (two CTAs of a
// thread-block cluster run each item side by side, their stages in lockstep).
// Group g with mt M tiles and nt N tiles has nt * floor(mt / 2) pair items --
// M tiles 2q and 2q + 1 of one N tile, so both CTAs multiply the same weight
// tile, each loading half of it for both -- then, when mt is odd, ceil(nt / 2)
// items of its last M tile, N tiles 2q and 2q + 1 (each CTA its own weight
// tile).  With the two-CTA MMA (two_cta) every item is two consecutive M
// tiles of one N tile, the second possibly empty: nt * ceil(mt / 2) items.
// s_it[g] = first item of group g (g <= E + 1).  Warp 2 runs the scan over
// the finished s_mt prefix.
__device__ __forceinline__ void build_item_table(const GemmParams &p, const int *s_mt, int *s_it,
                                                 int warp, int lane, bool two_cta = false) {
  if (warp != 2) return;
  const int n = p.n_routed + 1;
  const int per = (n + 31) / 32;
  auto items = [&](int g) {
    const int mt = s_mt[g + 1] - s_mt[g];
    return two_cta ? p.nt * ((mt + 1) >> 1)
                   : p.nt * (mt >> 1) + (mt & 1) * ((p.nt + 1) >> 1);
  };
  int sum = 0;
  for (int q = 0; q < per; ++q) {
    const int i = lane * per + q;
    if (i < n) sum += items(i);
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
    if (i < n) {
      s_it[i] = run;
      run += items(i);
    }
  }
  if (lane == 31) s_it[n] = incl;
}

// The tile of cluster CTA `rank` (0 or 1) in pair-mode item i; mc is set when
// both CTAs share the weight tile (a pair item).  In the last-M-tile items of
// a group with an odd number of N tiles, rank 1 may have no N tile left: it
// then runs the previous N tile with no rows, so every stage still fills and
// empties in step with its partner but nothing is stored.
__device__ __forceinline__ GemmTile decode_pair_item(const GroupTable &gt, const int *s_it,
                                                     const GemmParams &p, int i, int rank,
                                                     int n_cols, bool down, bool &mc) {
  const int E = p.n_routed;
  int lo = 0, hi = E;  // largest g with s_it[g] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_it[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int mtg = gt.mt[g + 1] - gt.mt[g];
  const int pairs = mtg >> 1;
  int local = i - s_it[g];
  int m, n;
  bool idle = false;
  if (local < p.nt * pairs) {
    n = local / pairs;
    m = 2 * (local - n * pairs) + rank;
    mc = true;
  } else {
    local -= p.nt * pairs;
    n = 2 * local + rank;
    m = mtg - 1;
    mc = false;
    if (n >= p.nt) {
      n = p.nt - 1;
      idle = true;
    }
  }
  GemmTile t;
  t.group = g;
  t.n0 = n * n_cols;
  t.pad[0] = t.pad[1] = t.pad[2] = 0;
  if (g < E) {
    const int cnt = gt.off[g + 1] - gt.off[g];
    t.a_row = gt.off[g] + m * kBM;
    t.out_row = t.a_row;
    t.rows = min(kBM, cnt - m * kBM);
  } else {
    t.rows = min(kBM, p.T - m * kBM);
    t.out_row = p.A + m * kBM;
    t.a_row = down ? t.out_row : m * kBM;
  }
  if (idle) t.rows = 0;
  return t;
}

// Two-CTA-MMA work item i (two_cta items of build_item_table): group g,
// N tile n and pair q of its M tiles, m innermost (the clusters that share a
// weight tile run side by side); CTA `rank` of the cluster takes M tile
// 2 q + rank, with no rows when that tile is past the group's end.
__device__ __forceinline__ GemmTile decode_2cta_item(const GroupTable &gt, const int *s_it,
                                                     const GemmParams &p, int i, int rank,
                                                     int n_cols, bool down) {
  const int E = p.n_routed;
  int lo = 0, hi = E;  // largest g with s_it[g] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_it[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int pairs = (gt.mt[g + 1] - gt.mt[g] + 1) >> 1;
  const int local = i - s_it[g];
  const int n = local / pairs;
  const int m = 2 * (local - n * pairs) + rank;
  GemmTile t;
  t.group = g;
  t.n0 = n * n_cols;
  t.pad[0] = t.pad[1] = t.pad[2] = 0;
  if (g < E) {
    const int cnt = gt.off[g + 1] - gt.off[g];
    t.a_row = gt.off[g] + m * kBM;
    t.out_row = t.a_row;
    t.rows = max(0, min(kBM, cnt - m * kBM));
  } else {
    t.rows = max(0, min(kBM, p.T - m * kBM));
    t.out_row = p.A + m * kBM;
    t.a_row = down ? t.out_row : m * kBM;
  }
  return t;
}

// Tile sequence of a CTA of the grouped GEMMs: lane 0 of the producer warp
// claims tiles (its first is blockIdx.x, every later one comes from a global
// counter, so CTAs that drew cheap tiles take more of them) and publishes each
// id in a small shared ring; the MMA thread, the epilogue warps and the gather
// warps read the ids from the ring in the same order.  A claim past the last
// tile ends every role's loop.  The router keeps the static order (one tile
// per CTA at most sizes).
constexpr int kTileRing = 4;
struct TileRing {
  uint32_t full0, empty0;  // [kTileRing] mbarriers each
  volatile int *ids;       // [kTileRing]
};

// Lane 0 of the producer warp: claim the it-th tile.  False when the slot's
// readers did not release it in time (the abort flag is then set).
__device__ __forceinline__ bool claim_tile(const TileRing &r, int it, int *ctr, int ntiles,
                                           long long limit, volatile int *abort, int &ti) {
  const int slot = it % kTileRing;
  if (it >= kTileRing && !mbar_wait(r.empty0 + 8 * slot, ((it / kTileRing) - 1) & 1, limit, abort))
    return false;
  ti = it == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(ctr, 1);
  if (ti > ntiles) ti = ntiles;
  r.ids[slot] = ti;
  mbar_arrive(r.full0 + 8 * slot);  // release: the id is visible with the phase
  return true;
}

// One thread per reading role: the it-th tile id; false when it did not
// arrive in time.
__device__ __forceinline__ bool read_tile(const TileRing &r, int it, long long limit,
                                          volatile int *abort, int &ti) {
  const int slot = it % kTileRing;
  if (!mbar_wait(r.full0 + 8 * slot, (it / kTileRing) & 1, limit, abort)) return false;
  ti = r.ids[slot];
  mbar_arrive(r.empty0 + 8 * slot);
  return true;
}

}  // namespace
}  // namespace moe
