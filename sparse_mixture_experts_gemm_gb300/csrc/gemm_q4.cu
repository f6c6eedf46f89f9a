// gemm_q4.cu -- the grouped GEMMs of the block with 4-bit group-affine expert
// weights, the dequantisation fused into the GEMM.
//
// "Optimizing on-device inference for Apple Silicon", section "Dequantise
// weights within matrix multiplication": the tensor operation takes bf16
// operands, so the 4-bit weights are rebuilt one small weight tile at a time
// in on-chip memory, right before the multiplication, accumulation in fp32 and
// bf16 output; the expanded weight matrix never goes to memory.  Format as in
// decode_q4.cu: codes two per byte along the row (the even column in the low
// nibble), one bf16 scale and one bf16 bias per 64 columns, w = s q + b.
//
// The structure is the bf16 grouped GEMM's (gemm.cu: persistent CTAs claiming
// tiles, tcgen05.mma from 128-byte-swizzled K-major shared-memory tiles into a
// double-buffered TMEM accumulator, the same epilogues), with the B operand
// made on the chip.  One K block is 64 columns, exactly one scale/bias group:
//   * the code producer (one warp, lane 0) streams the tile's code bytes
//     (BN rows x 32 bytes per K block) into a ring of 6 code stages, and the
//     scales and biases of 8 K blocks at a time into a ring of 2 chunks, by
//     TMA;
//   * 16 dequantising warps turn each code stage into the bf16 B tile of an
//     operand stage: w = s q + b with one bf16 rounding (q exact in bf16, one
//     bf16x2 FMA per pair), written in the 128-byte swizzle the MMA
//     descriptor expects, then a proxy fence and one arrival per warp;
//   * A comes as before (TMA for the shared expert's rows and for H, the
//     gather warps for routed token rows).
// A and B have rings of their own: 5 stages of A (the gathered token rows
// arrive from L2 with a latency of several MMA stages, so they need the
// depth) and 2 of B (dequantised on the chip, a short hop); the deep prefetch
// from HBM is the code ring's (6 stages).
// Every wait is bounded; a wait that runs out records a timeout, raises the
// CTA's abort flag, drains what it issued and returns.
#include <cuda_bf16.h>

#include "../../include/moe.h"
#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kAS = 5;            // A stages (token rows, 16 KB)
constexpr int kBS = 2;            // B stages (dequantised weights, 32 KB)
constexpr int kCode = 6;          // code stages
constexpr int kSb = 2;            // scale/bias chunks
constexpr int kSbGroups = 8;      // K blocks per scale/bias chunk
constexpr int kDqWarps = 16;      // dequantising warps
constexpr int kDqRows = kBN / kDqWarps;  // B rows per dequantising warp: 16
constexpr int kABytes = kBM * 128;
constexpr int kBBytes = kBN * 128;
constexpr int kCBytes = kBN * 32;                 // codes of one K block
constexpr int kSbBytes = 2 * kBN * kSbGroups * 2;  // scales [kBN][8], then biases
static_assert(kAS * kABytes + kBS * kBBytes + kCode * kCBytes + kSb * kSbBytes + 1024 + kGemmCtrl ==
                  kQ4GemmSmem,
              "shared-memory plan");

template <int EPI>
constexpr int gather_warps() { return EPI == EPI_SWIGLU ? kGatherThreads / 32 : 0; }
// warps: 0 A producer and tile claims, 1 MMA, 2-5 epilogue, [6-9 gather],
// then the dequantising warps, then the code producer
template <int EPI>
constexpr int q4_threads() { return 32 * (6 + gather_warps<EPI>() + kDqWarps + 1); }

// 8 codes of one 32-bit word (columns c .. c + 7, byte j holding column
// c + 2j in its low nibble) into 8 bf16 weights s q + b, in column order.
// With w4 = w >> 4, one byte permute puts byte j of w in byte 0 and byte j of
// w4 in byte 2; masking to 0x000F000F and setting 0x43004300 makes the bf16
// pair (128 + q_2j, 128 + q_2j+1), exact; subtracting 128 leaves q exactly;
// one bf16x2 FMA rounds s q + b once.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 b2) {
  const __nv_bfloat162 c128 = __floats2bfloat162_rn(128.0f, 128.0f);
  const uint32_t w4 = w >> 4;
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sel = (4u + j) << 12 | (4u + j) << 8 | static_cast<uint32_t>(j) << 4 | j;
    const uint32_t v = (__byte_perm(w, w4, sel) & 0x000F000Fu) | 0x43004300u;
    const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&v), c128);
    const __nv_bfloat162 o = __hfma2(q, s2, b2);
    r[j] = *reinterpret_cast<const uint32_t *>(&o);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// 16 floats to 16 bf16 (one 32-byte store; dst 32-byte aligned)
__device__ __forceinline__ void store16_bf16(__nv_bfloat16 *dst, const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t *>(&b);
  }
  st_global_32b(dst, w);
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(q4_threads<EPI>(), 1)
    gemm_q4_kernel(const __grid_constant__ Q4GemmMaps mp, const GemmParams p) {
  constexpr bool kDual = (EPI == EPI_SWIGLU);    // B = gate rows over up rows
  constexpr bool kGather = (EPI == EPI_SWIGLU);  // routed A rows gathered
  constexpr int kOutCols = kDual ? kBN / 2 : kBN;
  constexpr uint32_t kTmemCols = 2 * kBN;
  constexpr int kDq0 = 6 + gather_warps<EPI>();  // first dequantising warp
  constexpr int kCodeWarp = kDq0 + kDqWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + kAS * kABytes;
  uint8_t *sC = sB + kBS * kBBytes;
  uint8_t *sSB = sC + kCode * kCBytes;
  uint8_t *ctrl = sSB + kSb * kSbBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ctrl);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + 512);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + 516);
  int *s_off = reinterpret_cast<int *>(ctrl + 1536);        // [E + 1]
  int *s_mt = reinterpret_cast<int *>(ctrl + 1536 + 1040);  // [E + 2]
  const TileRing ring{smem_u32(ctrl + 1056), smem_u32(ctrl + 1056 + 8 * kTileRing),
                      reinterpret_cast<volatile int *>(ctrl + 1024)};
  // readers of the ring: MMA, 4 epilogue warps, gather warps, dequantising
  // warps, code producer
  constexpr int kTileReaders = 1 + 4 + gather_warps<EPI>() + kDqWarps + 1;

  const uint32_t full0 = smem_u32(bars);        // A stage full
  const uint32_t empty0 = full0 + 8 * kAS;      // A stage free (MMA commit)
  const uint32_t bfull0 = empty0 + 8 * kAS;     // B stage dequantised
  const uint32_t bempty0 = bfull0 + 8 * kBS;    // B stage free (MMA commit)
  const uint32_t cfull0 = bempty0 + 8 * kBS;    // code stage landed
  const uint32_t cempty0 = cfull0 + 8 * kCode;  // code stage read
  const uint32_t sbfull0 = cempty0 + 8 * kCode;
  const uint32_t sbempty0 = sbfull0 + 8 * kSb;
  const uint32_t tfull0 = sbempty0 + 8 * kSb;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long limit = MOE_WAIT_LIMIT_CYCLES;
  const GroupTable gt{s_off, s_mt};
  const int nkb = p.num_k_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAS; ++s) {
      // the A producer's arrival (with the A bytes when A comes by TMA) and
      // one per gather thread
      mbar_init(full0 + 8 * s, 1 + (kGather ? kGatherThreads : 0));
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int s = 0; s < kBS; ++s) {
      mbar_init(bfull0 + 8 * s, kDqWarps);
      mbar_init(bempty0 + 8 * s, 1);
    }
    for (int s = 0; s < kCode; ++s) {
      mbar_init(cfull0 + 8 * s, 1);
      mbar_init(cempty0 + 8 * s, kDqWarps);
    }
    for (int s = 0; s < kSb; ++s) {
      mbar_init(sbfull0 + 8 * s, 1);
      mbar_init(sbempty0 + 8 * s, kDqWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    mbar_init(drain_bar, 1);
    for (int q = 0; q < kTileRing; ++q) {
      mbar_init(ring.full0 + 8 * q, 1);
      mbar_init(ring.empty0 + 8 * q, kTileReaders);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kCodeWarp && lane == 0) {
    prefetch_tmap(&mp.a);
    for (int i = 0; i < 4; ++i) {
      prefetch_tmap(&mp.c[i]);
      prefetch_tmap(&mp.s[i]);
      prefetch_tmap(&mp.b[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // programmatic dependent launch: as in the bf16 GEMM, the prologue above
  // overlaps the previous kernel; its outputs are read only after the wait
  pdl_wait();
  pdl_launch_dependents();
  build_group_table(p, s_off, s_mt, warp, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = p.nt * s_mt[p.n_routed + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ A producer
    // claims the tiles; per K block: waits for a free operand stage and
    // loads A there by TMA (the shared expert's rows, H) or just arrives
    // (routed gate/up rows come from the gather warps)
    const uint64_t pol_a = policy_evict_last();
    uint32_t pend_mask = 0, pend_phase = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int ti = 0, c_ok = 1;
      if (lane == 0) c_ok = claim_tile(ring, it, p.tile_ctr, ntiles, limit, abort_flag, ti) ? 1 : 0;
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (!__shfl_sync(0xffffffffu, c_ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
        }
        ok = false;
        break;
      }
      if (ti >= ntiles) break;
      const GemmTile tl = decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool sh = tl.group >= p.n_routed;
      const bool a_tma = !kGather || sh;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0) {
          if (a_tma) {
            mbar_arrive_expect_tx(fb, kABytes);
            tma_load_2d(smem_u32(sA + stage * kABytes), &mp.a, fb, kb * 64, tl.a_row, pol_a);
          } else {
            mbar_arrive(fb);
          }
        }
        if (a_tma) {
          pend_mask |= 1u << stage;
          pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == kAS) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // copies already issued must land before the CTA's shared memory goes away
      for (int s = 0; s < kAS; ++s)
        if (pend_mask & (1u << s))
          if (!mbar_wait(full0 + 8 * s, (pend_phase >> s) & 1, limit, nullptr))
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
    }
  } else if (warp == kCodeWarp) {
    // ------------------------------------------------------------ code producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      uint32_t cpend = 0, cpend_ph = 0, spend = 0, spend_ph = 0;
      int cs = 0, sb = 0;
      uint32_t cph = 0, sbph = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int ti = 0;
        if (!read_tile(ring, it, limit, abort_flag, ti)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          ok = false;
          break;
        }
        if (ti >= ntiles) break;
        const GemmTile tl = decode_tile(gt, p, ti, kOutCols, !kDual);
        const bool sh = tl.group >= p.n_routed;
        const int m0 = sh ? 2 : 0;  // gate (or down) map; up is m0 + 1
        const int brow = sh ? tl.n0 : tl.group * p.b_rows_per_group + tl.n0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          if (kb % kSbGroups == 0) {
            if (!mbar_wait(sbempty0 + 8 * sb, sbph ^ 1, limit, abort_flag)) {
              *abort_flag = 1;
              report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
              ok = false;
              break;
            }
            const uint32_t fb = sbfull0 + 8 * sb;
            const uint32_t dst = smem_u32(sSB + sb * kSbBytes);
            constexpr uint32_t kHalf = kBN * kSbGroups * 2;  // one array: [kBN][8] bf16
            mbar_arrive_expect_tx(fb, kSbBytes);
            if (kDual) {
              constexpr uint32_t kRows = kBN / 2 * kSbGroups * 2;
              tma_load_2d(dst, &mp.s[m0], fb, kb, brow, pol_w);
              tma_load_2d(dst + kRows, &mp.s[m0 + 1], fb, kb, brow, pol_w);
              tma_load_2d(dst + kHalf, &mp.b[m0], fb, kb, brow, pol_w);
              tma_load_2d(dst + kHalf + kRows, &mp.b[m0 + 1], fb, kb, brow, pol_w);
            } else {
              tma_load_2d(dst, &mp.s[m0], fb, kb, brow, pol_w);
              tma_load_2d(dst + kHalf, &mp.b[m0], fb, kb, brow, pol_w);
            }
            spend |= 1u << sb;
            spend_ph = (spend_ph & ~(1u << sb)) | (sbph << sb);
          }
          if (!mbar_wait(cempty0 + 8 * cs, cph ^ 1, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
            ok = false;
            break;
          }
          const uint32_t fb = cfull0 + 8 * cs;
          const uint32_t dst = smem_u32(sC + cs * kCBytes);
          mbar_arrive_expect_tx(fb, kCBytes);
          if (kDual) {
            tma_load_2d(dst, &mp.c[m0], fb, kb * 32, brow, pol_w);
            tma_load_2d(dst + kCBytes / 2, &mp.c[m0 + 1], fb, kb * 32, brow, pol_w);
          } else {
            tma_load_2d(dst, &mp.c[m0], fb, kb * 32, brow, pol_w);
          }
          cpend |= 1u << cs;
          cpend_ph = (cpend_ph & ~(1u << cs)) | (cph << cs);
          if (++cs == kCode) {
            cs = 0;
            cph ^= 1;
          }
          if (kb % kSbGroups == kSbGroups - 1 || kb == nkb - 1) {
            if (++sb == kSb) {
              sb = 0;
              sbph ^= 1;
            }
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < kCode; ++s)
          if (cpend & (1u << s))
            if (!mbar_wait(cfull0 + 8 * s, (cpend_ph >> s) & 1, limit, nullptr))
              report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
        for (int s = 0; s < kSb; ++s)
          if (spend & (1u << s))
            if (!mbar_wait(sbfull0 + 8 * s, (spend_ph >> s) & 1, limit, nullptr))
              report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(kBM, kBN, MmaKind<__nv_bfloat16>::ab_format);
      int stage = 0, bstage = 0;
      uint32_t phase = 0, bphase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int it = 0; ok; ++it) {
        int ti = 0;
        if (!read_tile(ring, it, limit, abort_flag, ti)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
          ok = false;
          break;
        }
        if (ti >= ntiles) break;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_TMEM_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, limit, abort_flag) ||
              !mbar_wait(bfull0 + 8 * bstage, bphase, limit, abort_flag)) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          // gathered A rows were written by cp.async (generic proxy); the
          // barrier made them visible to this thread, the fence to the tensor
          // core's reads (the dequantising warps fence their own stores)
          if (kGather) fence_proxy_async_smem();
          const uint32_t a0 = smem_u32(sA + stage * kABytes);
          const uint32_t b0 = smem_u32(sB + bstage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            MmaKind<__nv_bfloat16>::mma(d_tmem, sdesc_sw128(a0 + 32 * kk), sdesc_sw128(b0 + 32 * kk),
                                        idesc, (kb | kk) != 0 ? 1u : 0u);
          tc_commit(empty0 + 8 * stage);
          tc_commit(bempty0 + 8 * bstage);
          issued = true;
          if (++stage == kAS) {
            stage = 0;
            phase ^= 1;
          }
          if (++bstage == kBS) {
            bstage = 0;
            bphase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok && issued) {
        tc_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0, limit, nullptr))
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_DRAIN);
      }
    }
  } else if (kGather && warp >= 6 && warp < kDq0) {
    // ------------------------------------------------------------ gather
    // as in the bf16 GEMM: 8 threads per 128-byte row, chunk c of row r at
    // c ^ (r % 8), completion through cp.async.mbarrier.arrive
    const int g = threadIdx.x - kThreads;
    const int c = g & 7, r0 = g >> 3;
    const int K = nkb * 64;
    const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(p.x);
    constexpr int kRowsPer = kBM / (kGatherThreads / 8);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int ti = 0, r_ok = 1;
      if (lane == 0) r_ok = read_tile(ring, it, limit, abort_flag, ti) ? 1 : 0;
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (!__shfl_sync(0xffffffffu, r_ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
        }
        ok = false;
        break;
      }
      if (ti >= ntiles) break;
      const GemmTile tl = decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool routed = tl.group < p.n_routed;
      const __nv_bfloat16 *src[kRowsPer];
      int tok[kRowsPer];
      if (routed) gather_tokens<kRowsPer>(p, gt, tl, r0, tok);
#pragma unroll
      for (int i = 0; i < kRowsPer; ++i)
        src[i] = (routed && r0 + 16 * i < tl.rows) ? xg + static_cast<long long>(tok[i]) * K + c * 8
                                                   : nullptr;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool w_ok = mbar_wait(empty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
          }
          ok = false;
          break;
        }
        const uint32_t tile_dst = smem_u32(sA + stage * kABytes);
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          const int r = r0 + 16 * i;
          if (src[i] != nullptr) cp_async16(tile_dst + r * 128 + ((c ^ (r & 7)) << 4), src[i] + kb * 64);
        }
        cp_async_arrive(full0 + 8 * stage);
        if (++stage == kAS) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp >= kDq0 && warp < kCodeWarp) {
    // ------------------------------------------------------------ dequantise
    // Warp w writes rows kDqRows w .. kDqRows (w + 1) - 1 of each B tile, 8
    // rows per pass:
    // lane (r, p) takes code words 2p and 2p + 1 of row r (16 codes, the
    // 16-byte chunks 2p and 2p + 1 of the bf16 row) with one scale and bias,
    // so a pass reads 256 contiguous code bytes and each store covers 8 rows
    // whose chunks land in distinct bank groups (rows in even/odd pairs).
    const int w = warp - kDq0;
    const int pr = lane & 3;
    int stage = 0, cs = 0, sb = 0;
    uint32_t phase = 0, cph = 0, sbph = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int ti = 0, r_ok = 1;
      if (lane == 0) r_ok = read_tile(ring, it, limit, abort_flag, ti) ? 1 : 0;
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (!__shfl_sync(0xffffffffu, r_ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_PRODUCER_EMPTY);
        }
        ok = false;
        break;
      }
      if (ti >= ntiles) break;
      for (int kb = 0; kb < nkb; ++kb) {
        bool w_ok = true;
        if (kb % kSbGroups == 0) w_ok = mbar_wait(sbfull0 + 8 * sb, sbph, limit, abort_flag);
        w_ok = w_ok && mbar_wait(cfull0 + 8 * cs, cph, limit, abort_flag);
        w_ok = w_ok && mbar_wait(bempty0 + 8 * stage, phase ^ 1, limit, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_MMA_FULL);
          }
          ok = false;
          break;
        }
        const uint8_t *code = sC + cs * kCBytes;
        const __nv_bfloat16 *ssc = reinterpret_cast<const __nv_bfloat16 *>(sSB + sb * kSbBytes);
        const __nv_bfloat16 *sbi = ssc + kBN * kSbGroups;
        uint8_t *bt = sB + stage * kBBytes;
        const int gcol = kb % kSbGroups;
#pragma unroll
        for (int i = 0; i < kDqRows / 8; ++i) {
          const int row = kDqRows * w + 8 * i + (lane >> 2);
          const uint2 words = *reinterpret_cast<const uint2 *>(code + row * 32 + pr * 8);
          const __nv_bfloat162 s2 = __bfloat162bfloat162(ssc[row * kSbGroups + gcol]);
          const __nv_bfloat162 b2 = __bfloat162bfloat162(sbi[row * kSbGroups + gcol]);
          uint8_t *rowp = bt + row * 128;
          *reinterpret_cast<uint4 *>(rowp + (((2 * pr) ^ (row & 7)) << 4)) = dequant8(words.x, s2, b2);
          *reinterpret_cast<uint4 *>(rowp + (((2 * pr + 1) ^ (row & 7)) << 4)) =
              dequant8(words.y, s2, b2);
        }
        // the tile is read by the tensor core (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bfull0 + 8 * stage);
          mbar_arrive(cempty0 + 8 * cs);
          if (kb % kSbGroups == kSbGroups - 1 || kb == nkb - 1) mbar_arrive(sbempty0 + 8 * sb);
        }
        if (++stage == kBS) {
          stage = 0;
          phase ^= 1;
        }
        if (++cs == kCode) {
          cs = 0;
          cph ^= 1;
        }
        if (kb % kSbGroups == kSbGroups - 1 || kb == nkb - 1) {
          if (++sb == kSb) {
            sb = 0;
            sbph ^= 1;
          }
        }
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;       // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;  // tile row == TMEM lane
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      int ti = 0, r_ok = 1;
      if (lane == 0) r_ok = read_tile(ring, it, limit, abort_flag, ti) ? 1 : 0;
      ti = __shfl_sync(0xffffffffu, ti, 0);
      if (!__shfl_sync(0xffffffffu, r_ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_EPI_TMEM_FULL);
        }
        break;
      }
      if (ti >= ntiles) break;
      const GemmTile tl = decode_tile(gt, p, ti, kOutCols, !kDual);
      const bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, limit, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.status, MOE_ERR_DEVICE_TIMEOUT, p.kid * 100 + SITE_EPI_TMEM_FULL);
        }
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(wq * 32) << 16);
      const bool valid = r < tl.rows;
      __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                            static_cast<long long>(tl.out_row + r) * p.ldo + tl.n0;
      // 16 columns at a time: this CTA runs many warps, registers are few
      if (kDual) {
#pragma unroll 1
        for (int c = 0; c < kBN / 2; c += 16) {
          float g[16], u[16];
          tmem_ld16x2_sync(tb + c, tb + kBN / 2 + c, g, u);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 16; ++i) g[i] = silu(g[i]) * u[i];
            store16_bf16(orow + c, g);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN; c += 16) {
          float v[16];
          tmem_ld16_sync(tb + c, v);
          if (valid) store16_bf16(orow + c, v);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int EPI>
cudaError_t gemm_q4_set_smem_attr() {
  return cudaFuncSetAttribute(gemm_q4_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kQ4GemmSmem);
}

template <int EPI>
cudaError_t launch_gemm_q4(const Q4GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                           bool pdl) {
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(q4_threads<EPI>());
  cfg.dynamicSmemBytes = kQ4GemmSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_q4_kernel<EPI>, maps, p);
}

template cudaError_t gemm_q4_set_smem_attr<EPI_SWIGLU>();
template cudaError_t gemm_q4_set_smem_attr<EPI_STORE>();
template cudaError_t launch_gemm_q4<EPI_SWIGLU>(const Q4GemmMaps &, const GemmParams &, int,
                                                cudaStream_t, bool);
template cudaError_t launch_gemm_q4<EPI_STORE>(const Q4GemmMaps &, const GemmParams &, int,
                                               cudaStream_t, bool);

}  // namespace moe
