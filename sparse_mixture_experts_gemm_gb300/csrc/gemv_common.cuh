// gemv_common.cuh -- warp-level m16n8k16 MMA steps of a weight matrix times
// at most 16 columns (used by the small-batch kernels), and the block-wide
// main loop of the small-batch router's logits.
//
// Main loop.  Unit of work: one CTA takes a block of kR x 16 weight rows (a "unit") and
// its 16 warps split it: warp w owns row block w / S (S = 16 / kR) and the
// reduction steps j = w % S + S i (a step is 32 columns).  Lane (g, q) of a
// warp (g = lane / 4, q = lane % 4) reads, per step, the 16 bytes at column
// 32 j + 8 q of rows g and g + 8 of its block.  Because the MMA's k index is
// only summed over, each lane feeds it its own columns (k = 2q, 2q + 1 from
// columns +0, +1; k = 2q + 8, 2q + 9 from +2, +3; the second MMA of the step
// takes +4..+7), and the B operand (the columns: tokens, or rows of h) is read
// with the same mapping, so every product is formed once.  A step's weights
// sit in registers; a warp holds two sets of four steps and loads the next
// set while it multiplies the current one, across unit boundaries too.  At
// the end of a unit every warp leaves its fp32 partial tile in shared memory
// (two buffers, one barrier per unit) and the op's epilogue sums the S
// partials of each output.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "ptx.cuh"
#include "status.h"

namespace moe {
namespace {

constexpr int kGvWarps = 16;
constexpr int kGvSet = 4;                       // steps per register set
constexpr int kGvRed = kGvWarps * 32 * 8;       // floats of one partial buffer
constexpr int kGvRedBytes = 2 * kGvRed * 4;     // both buffers

__device__ __forceinline__ void gv_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one step: rows g (ra) and g + 8 (rb) against 8 columns (b: this lane's 8
// values of its column at the same offsets)
__device__ __forceinline__ void gv_step(float (&c)[4], const uint4 &ra, const uint4 &rb,
                                        const uint4 &b) {
  gv_mma(c, ra.x, rb.x, ra.y, rb.y, b.x, b.y);
  gv_mma(c, ra.z, rb.z, ra.w, rb.w, b.z, b.w);
}

// Where partial (row r of the 16-row block, column m) of a warp's tile sits
// in its [32 lanes][8] slice: lane 4 (r % 8) + (m % 8) / 2, register
// 4 (m / 8) + m % 2 + 2 (r / 8).
__device__ __forceinline__ int gv_part(int r, int m) {
  return (4 * (r & 7) + ((m & 7) >> 1)) * 8 + 4 * (m >> 3) + (m & 1) + 2 * (r >> 3);
}

// Op interface (device member functions of the op):
//   void prepare()                 block-wide, before anything: sets first and
//                                  stride (this CTA's units are first,
//                                  first + stride, ...)
//   int first, stride, nsteps      nsteps = reduction length / 32
//   bool early(int u)              unit u exists and its rows are known
//                                  before op.wait()
//   void wait()                    block-wide: dependency wait, staging, barrier
//   int count()                    after wait(): how many units this CTA takes
//   void rows(int u, int rb, const uint4 *&pa, const uint4 *&pb)
//                                  this lane's rows g and g + 8 of row block rb
//                                  (already offset by q 16-byte pieces)
//   int ncols(int u)               columns of unit u (1..16)
//   const uint4 *col(int u, int nb) this lane's column g + 8 nb in shared
//                                  memory (offset by q pieces; clamped to a
//                                  valid column: results past ncols are unused)
//   void epilogue(int u, const float *red)   block-wide, after the barrier;
//                                  red: [16 warps][32 lanes][8] partials
// The groups that got rows, in unit order: the shared expert (group E) first,
// then the routed experts in index order.  Copies the offsets; block-wide.
// An invalid partition is reported and leaves no groups.
template <class Args>
__device__ __forceinline__ void touched_groups(const Args &a, int *s_off, int *s_grp, int *s_ng,
                                               int kid) {
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = ld_cg_s32(a.offsets + i);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = a.n_shared ? 1 : 0;
    bool bad = s_off[0] != 0 || s_off[a.E] != a.A;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      const int rows = e < a.E ? s_off[e + 1] - s_off[e] : 0;
      bad = bad || rows < 0;
      const unsigned m = __ballot_sync(0xffffffffu, rows > 0);
      if (rows > 0) s_grp[n + __popc(m & ((1u << lane) - 1u))] = e;
      n += __popc(m);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (a.n_shared) s_grp[0] = a.E;
      *s_ng = bad ? 0 : n;
      if (bad && blockIdx.x == 0) report_error(a.status, MOE_ERR_DEVICE_BOUNDS, kid * 100 + SITE_INDEX);
    }
  }
  __syncthreads();
}
template <int kR, class Op>
__device__ __forceinline__ void gv_run(Op &op, float *red) {
  constexpr int S = kGvWarps / kR;
  const int warp = threadIdx.x >> 5;
  const int rb = warp / S, sl = warp % S;
  const int spw = (op.nsteps + S - 1) / S;  // steps per warp
  const int nbat = (spw + kGvSet - 1) / kGvSet;
  uint4 a0[kGvSet], b0[kGvSet], a1[kGvSet], b1[kGvSet];
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};

  auto load = [&](uint4(&ra)[kGvSet], uint4(&rbb)[kGvSet], int it) {
    const int u = op.first + op.stride * (it / nbat), bt = it % nbat;
    const uint4 *pa, *pb;
    op.rows(u, rb, pa, pb);
#pragma unroll
    for (int s = 0; s < kGvSet; ++s) {
      const int j = sl + S * (kGvSet * bt + s);
      if (j < op.nsteps) {
        ra[s] = ld_stream16(pa + 4 * j);
        rbb[s] = ld_stream16(pb + 4 * j);
      }
    }
  };
  int par = 0;
  auto compute = [&](const uint4(&ra)[kGvSet], const uint4(&rbb)[kGvSet], int it) {
    const int u = op.first + op.stride * (it / nbat), bt = it % nbat;
    const int nc = op.ncols(u);
    const uint4 *x0 = op.col(u, 0), *x1 = op.col(u, 1);
#pragma unroll
    for (int s = 0; s < kGvSet; ++s) {
      const int j = sl + S * (kGvSet * bt + s);
      if (j < op.nsteps) {
        gv_step(c0, ra[s], rbb[s], x0[4 * j]);
        if (nc > 8) gv_step(c1, ra[s], rbb[s], x1[4 * j]);
      }
    }
    if (bt == nbat - 1) {  // unit done: partials out, one barrier, epilogue
      float *buf = red + par * kGvRed + (warp * 32 + (threadIdx.x & 31)) * 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        buf[i] = c0[i];
        buf[4 + i] = c1[i];
        c0[i] = 0.f;
        c1[i] = 0.f;
      }
      __syncthreads();
      op.epilogue(u, red + par * kGvRed);
      par ^= 1;
    }
  };

  op.prepare();
  const bool pre = op.early(op.first);
  if (pre) load(a0, b0, 0);
  op.wait();
  const int items = op.count() * nbat;
  if (items > 0 && !pre) load(a0, b0, 0);
  for (int it = 0; it < items; it += 2) {
    if (it + 1 < items) load(a1, b1, it + 1);
    compute(a0, b0, it);
    if (it + 2 < items) load(a0, b0, it + 2);
    if (it + 1 < items) compute(a1, b1, it + 1);
  }
}

}  // namespace
}  // namespace moe
