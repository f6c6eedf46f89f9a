// status.h -- device status word layout and failure detail codes.
// The status word is two ints in device memory per handle: [0] = first error
// code (MOE_ERR_*), [1] = detail: kernel id * 100 + site id.
#pragma once

namespace moe {

enum KernelId {
  KID_ROUTER = 1,
  KID_PERMUTE = 2,
  KID_GEMM_GATE_UP = 3,
  KID_GEMM_DOWN = 4,
  KID_COMBINE = 5,
  KID_DECODE = 6,
  KID_DEBUG = 9,
};

enum WaitSite {
  SITE_PRODUCER_EMPTY = 1,  // TMA producer waiting for a free smem stage
  SITE_MMA_FULL = 2,        // MMA issuer waiting for a loaded smem stage
  SITE_MMA_TMEM_EMPTY = 3,  // MMA issuer waiting for the epilogue to drain TMEM
  SITE_EPI_TMEM_FULL = 4,   // epilogue waiting for a finished accumulator
  SITE_DRAIN = 5,           // final wait for in-flight copies / MMAs
  SITE_INDEX = 6,           // an index check failed
  SITE_DEBUG = 7,           // the test hook's never-signalled barrier
  SITE_STAGE = 8,           // a 4-bit batch-1 kernel waiting for its staged rows
};

}  // namespace moe
