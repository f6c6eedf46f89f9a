// internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// One output tile of a grouped GEMM: 128 rows x N columns of one group.
// Groups 0..E-1 are routed experts; group E is the shared expert.
struct GemmTile {
  int group;    // expert id, E for the shared expert
  int a_row;    // first row of the A operand (first slot, row of x, or row of H)
  int out_row;  // first output row (row of H or Yp)
  int rows;     // valid rows, 0..128 (0: a cluster-pair CTA that stores nothing)
  int n0;       // first output column; also the row offset inside the group's B
  int pad[3];
};
static_assert(sizeof(GemmTile) == 32, "tile record is 32 bytes");

enum Epilogue { EPI_SWIGLU = 0, EPI_STORE = 1 };

constexpr int kBM = 128;      // rows per tile (TMEM lanes)
constexpr int kBN = 256;      // MMA N: B rows per tile of the expert GEMMs
constexpr int kStageBudget = 4 * (kBM * 128 + kBN * 128);  // smem for the operand stages
constexpr int kThreads = 192; // warp 0 loads, warp 1 MMA, warps 2-5 epilogue
constexpr int kGatherThreads = 128;  // gate/up GEMM: warps 6-9 gather routed token rows
constexpr int kGemmCtrl = 5120;  // barriers, TMEM slot, tile ring, group and item tables
constexpr int kGemmSmem = kStageBudget + 1024 + kGemmCtrl;
constexpr int kCountStride = 32;  // router histogram: one counter per 128-byte line
constexpr int kMaxTopK = 8;

struct GemmParams {
  // grouped GEMMs: tiles derived from the group offsets
  const int32_t *offsets;  // [E + 1] first slot of each routed group (device)
  int T;                   // tokens of this chunk
  int A;                   // T * k routed assignments
  int n_shared;            // 0 or 1: group E = the shared expert over all T tokens
  int nt;                  // N tiles per group
  int num_k_blocks;        // K / (128 bytes / element size)
  int n_routed;            // E
  int b_rows_per_group;    // rows of one routed group's B matrix (F or d)
  // epilogue output
  void *out;               // H (gate/up) or Y (down)
  long long ldo;           // elements per output row
  int *status;             // device status word
  int kid;                 // KernelId for failure details
  int *tile_ctr;           // grouped GEMMs: tiles claimed after each CTA's first, zero before the launch
  // gate/up GEMM: routed A rows are gathered from the tokens, row r of group
  // g's M tile m from token list[g * list_stride + m * 128 + r] (the router's
  // per-expert token lists) or, with list null, perm[slot]
  const int32_t *perm;     // [A] token of each slot
  int32_t *list;           // [E][list_stride] tokens of each group in rank order
  long long list_stride;
  const void *x;           // [T][K] the chunk's tokens
  // grouped GEMMs after the cluster router: the group offsets come from its
  // line-padded histogram counts_in (CTA 0 also writes them to offsets_out
  // and adds the counts into counts_out, when given); the down GEMM's CTA 0
  // zeroes clear_counts (that histogram) and *clear_ctr (the gate/up GEMM's
  // tile counter) for the next call, both read only by the finished gate/up
  const int32_t *counts_in;
  int32_t *offsets_out;    // [E + 1]
  int32_t *counts_out;     // [E], summed over a call's chunks (may be null)
  int32_t *clear_counts;
  int *clear_ctr;
};

// Tensor maps: A routed, A shared, B0 routed, B1 routed, B0 shared, B1 shared.
struct GemmMaps {
  CUtensorMap m[6];
};

// gemm.cu
// pdl: launched as a programmatic dependent of the previous kernel on st.
// kPair (grouped GEMMs): thread-block clusters of two CTAs that run the
// pair-mode work items (gemm_common.cuh) in lockstep; grid even.  For
// EPI_STORE the B1 maps then hold 128-row boxes of the down weights.
template <typename T, int EPI, int BN, bool kPair = false>
cudaError_t launch_gemm(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                        bool pdl = false);
template <typename T, int EPI, int BN, bool kPair = false>
cudaError_t gemm_set_smem_attr();
// Clusters of two pair-mode CTAs that can be resident at once (0 on error).
int gemm_pair_clusters();

// gemm2sm.cu: the bf16 grouped GEMMs on the two-CTA MMA (clusters of two,
// grid even; the maps as for the pair mode of launch_gemm).
template <int EPI>
cudaError_t launch_gemm2sm(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                           bool pdl = false);
template <int EPI>
cudaError_t gemm2sm_set_smem_attr();
int gemm2sm_clusters();

// router.cu: the router of chunks of more than kSmallRouteT bf16 tokens.
// One cluster of `split` CTAs per 128 tokens (each 4 / split quarters of d,
// all experts; split 4, or 2 when four CTAs per tile would not all be
// resident at once).
// Writes idx [T][k], w [T][k]; then either adds each expert's count into
// counts_direct [E] (routing only) or claims ranks on the line-padded
// histogram counts [E * kCountStride] (zero before the launch), writing each
// assignment's rank into rank [T][k] and the token into list[e][rank].
struct RouterArgs {
  int T, d, E, k;
  const float *bias;       // [E] or null
  int32_t *idx;
  float *w;
  int32_t *counts;         // line-padded histogram (ranks)
  int32_t *counts_direct;  // [E] per-expert counts (no ranks, no lists)
  int32_t *rank;
  int32_t *list;
  long long list_stride;
  int *status;
  int split;  // CTAs per cluster: 4 or 2 (the same results either way)
};
cudaError_t router_set_attr();
// pdl: launched as a programmatic dependent of the previous kernel on st
cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const RouterArgs &a,
                          cudaStream_t st, bool pdl = false);
cudaError_t launch_debug_wait(int *status, long long limit_cycles, cudaStream_t st);

// route_small.cu: routing of batches of at most kSmallRouteT bf16 tokens
// (tokens in passes of kSmallRoutePass, a pass's tokens within
// kSmallRouteTokBytes) in one cluster launch: writes idx, w,
// inv (slots), perm, offsets and zeroes the n_clear words clear[32 q].
constexpr int kSmallRouteT = 64;
constexpr int kSmallRoutePass = 16;
constexpr int kSmallRouteTokBytes = 65536;
// gemv_small.cu: the grouped GEMVs take batches of at most kSmallGemvT tokens;
// by default bf16 layers use them up to kSmallGemvTBf16 tokens (the grouped
// GEMMs are as fast above), 4-bit layers up to kSmallGemvT
// (moe_set_option(MOE_OPT_GEMV_MAX_TOKENS) changes the limit)
constexpr int kSmallGemvT = 32;
constexpr int kSmallGemvTBf16 = 16;
// chunks of at least this many tokens run the bf16 grouped GEMMs on clusters
// of two CTAs (moe_set_option(MOE_OPT_PAIR_MIN_TOKENS) changes it)
constexpr long long kPairMinTokens = 8192;
// chunks of at least this many tokens run the gate/up GEMM, and of at least
// kMma2DownMinTokens the down GEMM, on the two-CTA MMA instead
// (moe_set_option(MOE_OPT_MMA2_MIN_TOKENS / MOE_OPT_MMA2_DOWN_MIN_TOKENS))
constexpr long long kMma2MinTokens = 8192;
constexpr long long kMma2DownMinTokens = 16384;
// counts_out (may be null): each expert's group size is added to it.
cudaError_t launch_route_small(const void *x, const void *wr, const float *bias, int T, int d,
                               int E, int k, int32_t *idx, float *w, int32_t *inv, int32_t *perm,
                               int32_t *offsets, int32_t *counts_out, int32_t *clear, int n_clear,
                               cudaStream_t st);
cudaError_t route_small_set_attr();

// gemv_small.cu: gate/up (h = silu(gate) * up as bf16 rows) and down (bf16
// rows of Y) of a small batch as a grouped GEMV on warp-level MMAs; the units
// (16 weight rows of one touched expert) are found on the device from the
// routing step's offsets.  Tokens T <= kSmallGemvT, bf16.
struct SmallArgs {
  const __nv_bfloat16 *x;                 // [T][d]
  const __nv_bfloat16 *wg, *wu, *wd;      // routed experts
  const __nv_bfloat16 *sg, *su, *sd;      // shared expert (n_shared == 1)
  const int32_t *offsets, *perm;          // routing step's output
  __nv_bfloat16 *h;                       // [A + T][F]
  __nv_bfloat16 *y;                       // [A + T][d]
  int T, d, F, E, A, n_shared;
  int *status;
};
// whether the kernels' shared memory plans fit (tokens and a ring of at
// least two stages)
bool small_gemv_fits(int T, int d, int F);
cudaError_t launch_small_gateup(const SmallArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_small_down(const SmallArgs &a, int grid, cudaStream_t st, bool pdl);
cudaError_t small_gemv_set_attr();

// gemm_q4.cu: the grouped GEMMs (EPI_SWIGLU, EPI_STORE; bf16 tokens) with
// 4-bit group-affine weights, dequantised into the MMA's B tiles.  Maps:
// a = the A operand by TMA (x for the shared expert's gate/up rows, H for the
// down GEMM); c, s, b = codes [rows][K / 2] u8 (boxes 32 bytes x rows), scales
// and biases [rows][K / 64] (boxes 8 groups x rows), indexed
// 2 * shared + half (half 0: gate or down, 1: up).
struct Q4GemmMaps {
  CUtensorMap a;
  CUtensorMap c[4], s[4], b[4];
};
constexpr int kQ4GemmSmem = 5 * (kBM * 128) + 2 * (kBN * 128) + 6 * (kBN * 32) +
                            2 * (2 * kBN * 8 * 2) + 1024 + kGemmCtrl;
template <int EPI>
cudaError_t launch_gemm_q4(const Q4GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t st,
                           bool pdl = false);
template <int EPI>
cudaError_t gemm_q4_set_smem_attr();

// noalloc.cu: device address of moe_decode_noalloc's status word on the
// current device (null if the lookup failed)
int *noalloc_status_word();

// moe.cu: tensor-map encoding (host only, no allocation)
bool encode_map_2d(CUtensorMap *m, const void *base, size_t esz, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// route.cu
template <typename T>
cudaError_t launch_router_simt(const T *x, const T *wr, const float *bias, int T_tok, int d, int E,
                               int k, int32_t *idx, float *w, int32_t *counts, int32_t *rank,
                               cudaStream_t st);
// also zeroes counts[0, E) and n_clear words clear[32 q] for the next call
// counts_out (may be null) accumulates the counts
cudaError_t launch_offsets(int32_t *counts, int E, int32_t *offsets, int32_t *counts_out,
                           int32_t *clear, int n_clear, cudaStream_t st);
cudaError_t launch_place(const int32_t *idx, const int32_t *offsets, int32_t *rank_inv,
                         int32_t *perm, int A, int k, int E, int *status, cudaStream_t st,
                         bool pdl = false);
// inv[t][j]: the slot (row of Y) of assignment (t, j); with offsets given,
// its rank inside the group of expert idx[t][j] (slot = offsets[e] + rank)
template <typename T>
cudaError_t launch_combine(const T *yp, const int32_t *inv, const float *w, T *out, int T_tok,
                           int k, int d, int A_total, int n_shared, int *status, int num_sms,
                           cudaStream_t st, bool pdl = false, const int32_t *idx = nullptr,
                           const int32_t *offsets = nullptr, int E = 0,
                           int *clear_ctr = nullptr);

// 4-bit group-affine matrix (codes two per byte, even column in the low
// nibble; one bf16 scale and bias per 64 columns of a row)
constexpr int kQ4Group = 64;
constexpr int kSelReplicas = 16;
struct Q4Mat {
  const uint8_t *c;   // [rows][cols / 2]
  const uint16_t *s;  // [rows][cols / 64]
  const uint16_t *b;  // [rows][cols / 64]
};
struct Q4Weights {
  Q4Mat g, u, d, sg, su, sd;
};

// gemv_small_q4.cu: the small-batch grouped GEMV on 4-bit expert weights
// (same arguments as the bf16 one; the weight pointers of a are unused)
struct SmallQ4Args {
  SmallArgs a;
  Q4Weights w;
};
cudaError_t launch_small_gateup_q4(const SmallQ4Args &a, int grid, cudaStream_t st, bool pdl);
cudaError_t launch_small_down_q4(const SmallQ4Args &a, int grid, cudaStream_t st, bool pdl);
cudaError_t small_gemv_q4_set_attr();

// decode.cu
struct DecodeArgs {
  const void *x;
  const void *wr, *wg, *wu, *wd, *sg, *su, *sd;
  const float *bias;
  int d, F, E, k, n_shared;
  float *logits;       // [E]
  float *h;            // [(k + 1)][F]
  void *out;           // [d]
  int *status;
  // launch shape, filled in by the launchers
  int rows_a;          // kernel A: router rows or shared items per CTA
  int ring;            // kernel B: ring slots per CTA
  int c_rows;          // kernel C: output rows per CTA (upper bound)
  Q4Weights q;         // 4-bit expert weights (decode_q4.cu), unused by the bf16 kernels
  // decode_q4.cu: the top-k picked once per layer by kernel A, in
  // kSelReplicas copies of 128 bytes (32 words: [0, 8) experts, [8, 16) their
  // weights as float bits), so that the many CTAs reading it share no line
  int *dsel;
  // the routing the kernels use, for a caller that asked for it (each may be
  // null): the k experts, their weights, and +1 on each chosen expert's count
  int32_t *sel_idx;
  float *sel_w;
  int32_t *sel_counts;
};

// decode_q4.cu: the batch-1 kernels for 4-bit expert weights (bf16 tokens,
// bf16 router) and the quantiser
cudaError_t launch_decode_router_q4(const DecodeArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_decode_gateup_q4(const DecodeArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_decode_down_q4(const DecodeArgs &a, cudaStream_t st, bool pdl);
cudaError_t decode_q4_set_smem_attr();
template <typename T>
cudaError_t launch_quantize_q4(const T *w, long long rows, int cols, uint8_t *codes,
                               uint16_t *scales, uint16_t *biases, cudaStream_t st);
template <typename T>
cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t st, bool pdl);
// tmG / tmU: w_gate / w_up as [E * F][d] with boxes of (512 bytes) x 32 rows, no swizzle
template <typename T>
cudaError_t launch_decode_gateup(const DecodeArgs &a, const CUtensorMap &tmG, const CUtensorMap &tmU,
                                 cudaStream_t st, bool pdl);
template <typename T>
cudaError_t launch_decode_down(const DecodeArgs &a, cudaStream_t st, bool pdl);
// Raise the dynamic shared memory limit of the three decode kernels (once per
// device, with the device current).
template <typename T>
cudaError_t decode_set_smem_attr();

}  // namespace moe
