// moe.cu -- host side of the C ABI declared in include/moe.h: argument
// validation, the one workspace allocation, TMA descriptors, and the kernel
// sequence of the prefill and decode paths.
//
// Prefill, per chunk of at most max_tokens tokens ("Optimizing on-device
// inference for Apple Silicon", section "Bound temporary memory with request
// chunking"), all on the caller's stream with no host synchronisation
// (section "Keep expert routing on the GPU"):
//   router (tcgen05 for bf16, SIMT + offsets for fp32) -> place (slot of
//   every assignment and token of every slot) -> grouped gate/up GEMM + SiLU
//   (routed rows gathered from x inside the kernel) -> grouped down GEMM ->
//   combine.
// Decode (T == 1, section "Optimise the single-row weight path"):
//   decode_router -> decode_gateup -> decode_down, chained with programmatic
//   dependent launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "internal.h"
#include "status.h"

using namespace moe;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// 2D map over a row-major [rows][cols] matrix with a box of box_cols x
// box_rows elements; 128-byte swizzle or none; out-of-range elements read as
// zero.  Host-only (encodes the descriptor, allocates nothing).
bool moe::encode_map_2d(CUtensorMap *m, const void *base, size_t esz, uint64_t rows, uint64_t cols,
                        uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  // 2-byte elements travel as bf16 (also the raw bits of 4-bit scales and
  // biases), 1-byte ones as u8 (4-bit codes, two per byte); TMA copies bits
  const CUtensorMapDataType dt = esz == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// The GEMM operand map: boxes of 128 bytes of columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, size_t esz, uint64_t rows, uint64_t cols,
              uint32_t box_rows) {
  return encode_map_2d(m, base, esz, rows, cols, static_cast<uint32_t>(128 / esz), box_rows, true);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};

}  // namespace

constexpr int kRouteCtlCounts = 256 * kCountStride;
// the router's histogram (one counter per 128-byte line), then a spare line,
// the gate/up and the down GEMM's tile counters, each on its own line
constexpr size_t kRouteCtlBytes = sizeof(int32_t) * (kRouteCtlCounts + 96);

struct moe_handle {
  moe_config cfg;
  int device = 0;
  int num_sms = 0;
  size_t esz = 2;
  int nt1 = 0, nt2 = 0;  // N tiles of the gate/up and down GEMMs
  // workspace (one allocation)
  void *ws = nullptr;
  int32_t *idx = nullptr, *inv = nullptr, *offsets = nullptr, *status = nullptr;
  // [256 * kCountStride] per-expert counts (line-padded for the bf16 router,
  // dense for the fp32 one), then the router's CTA ticket and the grouped
  // GEMMs' tile counters
  int32_t *route_ctl = nullptr;
  float *w = nullptr, *logits = nullptr, *hdec = nullptr;
  int32_t *dctl = nullptr;  // 4-bit batch-1 path: the layer's top-k (DecodeArgs::dsel)
  int32_t *perm = nullptr;  // [A] token of each slot
  int32_t *list = nullptr;  // [E][max_tokens] tokens of each expert group in rank order
  void *hbuf = nullptr, *yp = nullptr;
  // static tensor maps
  CUtensorMap tm_dg, tm_du;  // decode gate/up GEMV boxes
  CUtensorMap tm_h, tm_wg, tm_wu, tm_wd, tm_sg, tm_su, tm_sd;
  // cluster-pair grouped GEMMs (bf16): the down weights in 128-row boxes,
  // the grid (two CTAs per cluster, 0: not available) and the smallest
  // chunk that takes them
  CUtensorMap tm_wd2, tm_sd2;
  CUtensorMap tm_wr256;  // router rows in boxes of 256 rows (the cluster router)
  int pair_grid = 0;
  long long pair_min_tokens = kPairMinTokens;
  // two-CTA-MMA grouped GEMMs (bf16): grid and the smallest chunk for each
  int mma2_grid = 0;
  long long mma2_min_tokens = kMma2MinTokens;
  long long mma2_down_min_tokens = kMma2DownMinTokens;
  // the router's clusters of two CTAs: from the smallest chunk whose clusters
  // of four (4 CTAs of one SM each per 128 tokens) would not all be resident
  long long router_pair_min_tokens = 0;
  int gemv_max_tokens = -1;  // -1: by weight type (kSmallGemvTBf16 / kSmallGemvT)
  // 4-bit expert weights (moe_create_q4)
  bool q4 = false;
  bool q4_prefill = false;  // the grouped GEMMs support the layer's shape
  Q4Weights qw = {};
  Q4GemmMaps q4g = {}, q4d = {};  // gate/up and down GEMM maps (a set per call / once)
  // host-buffer calls (moe_forward_host): two device slots, each an input and
  // an output region of cap tokens, a copy-in and a copy-out stream, and per
  // slot the events that order the copies against the forward on the caller's
  // stream
  struct HostStage {
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t in_done[2] = {}, fwd_done[2] = {}, out_done[2] = {};
    bool used[2] = {false, false};
    char *buf = nullptr;
    size_t cap = 0;
    int next = 0, last = -1;
  } hs;
  // profiling
  bool prof = false;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
  size_t pool_used = 0;
  int32_t *counts() { return route_ctl; }
  int32_t *tile_ctr(int gemm) { return route_ctl + kRouteCtlCounts + 32 * (gemm + 1); }
};

namespace {

// q4: the expert weights come as 4-bit matrices (moe_create_q4), so the bf16
// expert pointers must be NULL.
int check_cfg(const moe_config *c, bool q4 = false) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->d_ff <= 0 || c->n_experts <= 0 || c->top_k <= 0 ||
      c->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_INVALID_ARG;
  if (!c->w_router) return MOE_ERR_INVALID_ARG;
  if (q4) {
    if (c->w_gate || c->w_up || c->w_down || c->s_gate || c->s_up || c->s_down)
      return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  } else {
    if (!c->w_gate || !c->w_up || !c->w_down) return MOE_ERR_INVALID_ARG;
    if (c->n_shared && (!c->s_gate || !c->s_up || !c->s_down)) return MOE_ERR_INVALID_ARG;
  }
  if (c->d_model % 256 != 0 || c->d_model > 16384) return MOE_ERR_UNSUPPORTED;
  if (c->d_ff % 128 != 0 || c->d_ff > 4096) return MOE_ERR_UNSUPPORTED;
  if (c->n_experts > 256 || c->top_k > kMaxTopK || c->top_k > c->n_experts)
    return MOE_ERR_UNSUPPORTED;
  if (c->max_tokens > 65536) return MOE_ERR_UNSUPPORTED;
  const void *ptrs[] = {c->w_router, c->w_gate, c->w_up, c->w_down,
                        c->s_gate,   c->s_up,   c->s_down, c->router_bias};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

cudaEvent_t prof_event(moe_handle *h) {
  if (h->pool_used == h->pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->pool.push_back(e);
  }
  return h->pool[h->pool_used++];
}

// Records an event pair around one launch when profiling is on.
struct ProfScope {
  moe_handle *h;
  int kind;
  cudaStream_t st;
  cudaEvent_t b = nullptr;
  ProfScope(moe_handle *h_, int kind_, cudaStream_t st_) : h(h_), kind(kind_), st(st_) {
    if (h->prof) {
      b = prof_event(h);
      if (b) cudaEventRecord(b, st);
    }
  }
  ~ProfScope() {
    if (h->prof && b) {
      cudaEvent_t e = prof_event(h);
      if (e) {
        cudaEventRecord(e, st);
        h->recs.push_back({kind, b, e});
      }
    }
  }
};

#define MOE_TRY(expr)                             \
  do {                                            \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// The bf16 router of chunks above the small-batch size: one cluster of four
// CTAs per 128 tokens, or of two CTAs from router_pair_min_tokens on
// (router.cu; the same results either way).  With counts_direct it writes the
// per-expert counts for the caller; otherwise it claims ranks on the
// handle's histogram and fills the per-expert token lists.
int launch_router_bf16(moe_handle *h, const void *x, int T, int32_t *idx, float *w,
                       int32_t *counts_direct, cudaStream_t st) {
  const moe_config &c = h->cfg;
  CUtensorMap tm_x;
  if (!make_map(&tm_x, x, 2, T, c.d_model, kBM)) return MOE_ERR_CUDA;
  RouterArgs a = {};
  a.T = T;
  a.d = c.d_model;
  a.E = c.n_experts;
  a.k = c.top_k;
  a.bias = c.router_bias;
  a.idx = idx;
  a.w = w;
  a.counts = h->counts();
  a.counts_direct = counts_direct;
  a.rank = h->inv;
  a.list = h->list;
  a.list_stride = c.max_tokens;
  a.status = h->status;
  a.split = T >= h->router_pair_min_tokens ? 2 : 4;
  MOE_TRY(launch_router(tm_x, h->tm_wr256, a, st, !h->prof));
  return MOE_OK;
}

// Where a forward puts the routing its kernels compute: idx [Tc][k] and
// w [Tc][k] of this chunk (null: the handle's workspace) and the per-expert
// counts of the call (null: not wanted; otherwise zeroed at the call's start
// and summed over its chunks).
struct RouteOut {
  int32_t *idx = nullptr;
  float *w = nullptr;
  int32_t *counts = nullptr;
};

// a chunk of Tc bf16 tokens routes in one cluster launch (tokens in passes
// of kSmallRoutePass, each pass staged in shared memory)
bool small_route_ok(int Tc, int d) {
  const int pass = Tc < kSmallRoutePass ? Tc : kSmallRoutePass;
  return Tc <= kSmallRouteT && static_cast<long long>(pass) * d * 2 <= kSmallRouteTokBytes;
}

// The small-batch router (routing and placement in one cluster launch, 16
// tokens per pass) serves the chunks that run the grouped GEMVs; every other
// bf16 chunk takes the cluster router, whose per-expert token lists feed the
// grouped GEMMs (at 32 and 64 tokens the small router's passes took 25 and
// 42 us, the cluster router ~20).
bool use_small_route(const moe_handle *h, int Tc) {
  const moe_config &c = h->cfg;
  if (c.dtype != MOE_BF16 || !small_route_ok(Tc, c.d_model) ||
      !small_gemv_fits(Tc, c.d_model, c.d_ff))
    return false;
  const int gemv_max = h->gemv_max_tokens >= 0 ? h->gemv_max_tokens
                                                : (h->q4 ? kSmallGemvT : kSmallGemvTBf16);
  return Tc <= gemv_max || (h->q4 && !h->q4_prefill);
}

template <typename T>
int run_prefill_chunk(moe_handle *h, const T *x, int Tc, T *out, const RouteOut &ro,
                      cudaStream_t st) {
  const moe_config &c = h->cfg;
  const int d = c.d_model, F = c.d_ff, E = c.n_experts, k = c.top_k;
  const int A = Tc * k;
  const int BK = static_cast<int>(128 / sizeof(T));
  // the chunk's routing: written by the router, read by place and combine
  int32_t *idx = ro.idx ? ro.idx : h->idx;
  float *wts = ro.w ? ro.w : h->w;

  // route_ctl is zero here: create cleared it; the small-batch and fp32
  // routers clear the GEMMs' tile counters when they are done, and after the
  // bf16 cluster router the down GEMM clears its histogram and the gate/up
  // tile counter, the combine the down tile counter
  const bool small = sizeof(T) == 2 && use_small_route(h, Tc);
  if (small) {
    // a few tokens: routing and placement in one cluster launch
    ProfScope ps(h, MOE_KERNEL_ROUTER, st);
    MOE_TRY(launch_route_small(x, c.w_router, c.router_bias, Tc, d, E, k, idx, wts, h->inv,
                               h->perm, h->offsets, ro.counts, h->tile_ctr(0), 2, st));
  } else {
    ProfScope ps(h, MOE_KERNEL_ROUTER, st);
    if (sizeof(T) == 2) {
      // tokens into per-expert lists, ranks into inv, the histogram: no
      // placement step (the gate/up GEMM scans the histogram into the group
      // offsets, the combine adds each assignment's group offset to its rank)
      const int rc = launch_router_bf16(h, x, Tc, idx, wts, nullptr, st);
      if (rc != MOE_OK) return rc;
    } else {
      MOE_TRY(launch_router_simt<T>(x, static_cast<const T *>(c.w_router), c.router_bias, Tc, d, E,
                                    k, idx, wts, h->counts(), h->inv, st));
      MOE_TRY(launch_offsets(h->counts(), E, h->offsets, ro.counts, h->tile_ctr(0), 2, st));
    }
  }
  // the kernels after the router run as programmatic dependents, each
  // waiting for its predecessor inside (event records between kernels would
  // break the chain, so not while profiling)
  const bool pdl = !h->prof;
  // the tensor-core router writes per-expert token lists, from which the
  // gate/up GEMM gathers its rows; the fp32 router's ranks become slots and
  // a slot permutation in a placement step
  const bool lists = sizeof(T) == 2 && !small;
  if (!small && !lists) {
    ProfScope ps(h, MOE_KERNEL_PERMUTE, st);
    MOE_TRY(launch_place(idx, h->offsets, h->inv, h->perm, A, k, E, h->status, st, pdl));
  }
  // grouped GEMV up to the handle's limit; 4-bit shapes the 4-bit GEMMs do
  // not take always (forward_shape_ok admitted only chunks that fit it):
  // exactly the chunks use_small_route sent to the small-batch router
  if (small) {
    // a few tokens: every touched expert gets a few rows, grouped GEMV over
    // all SMs (the tensor-core tiles of 128 rows would stay mostly empty and
    // leave most SMs idle)
    SmallArgs sa;
    sa.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    sa.wg = static_cast<const __nv_bfloat16 *>(c.w_gate);
    sa.wu = static_cast<const __nv_bfloat16 *>(c.w_up);
    sa.wd = static_cast<const __nv_bfloat16 *>(c.w_down);
    sa.sg = static_cast<const __nv_bfloat16 *>(c.s_gate);
    sa.su = static_cast<const __nv_bfloat16 *>(c.s_up);
    sa.sd = static_cast<const __nv_bfloat16 *>(c.s_down);
    sa.offsets = h->offsets;
    sa.perm = h->perm;
    sa.h = static_cast<__nv_bfloat16 *>(h->hbuf);
    sa.y = static_cast<__nv_bfloat16 *>(h->yp);
    sa.T = Tc;
    sa.d = d;
    sa.F = F;
    sa.E = E;
    sa.A = A;
    sa.n_shared = c.n_shared;
    sa.status = h->status;
    SmallQ4Args qa;
    qa.a = sa;
    qa.w = h->qw;
    {
      ProfScope ps(h, MOE_KERNEL_GEMV_GATE_UP, st);
      MOE_TRY(h->q4 ? launch_small_gateup_q4(qa, h->num_sms, st, pdl)
                    : launch_small_gateup(sa, h->num_sms, st, pdl));
    }
    {
      ProfScope ps(h, MOE_KERNEL_GEMV_DOWN, st);
      MOE_TRY(h->q4 ? launch_small_down_q4(qa, h->num_sms, st, pdl)
                    : launch_small_down(sa, h->num_sms, st, pdl));
    }
    ProfScope ps(h, MOE_KERNEL_COMBINE, st);
    MOE_TRY(launch_combine<T>(static_cast<const T *>(h->yp), h->inv, wts, out, Tc, k, d, A,
                              c.n_shared, h->status, h->num_sms, st, pdl));
    return MOE_OK;
  }
  // large chunks: the grouped GEMMs on clusters of two CTAs, either on the
  // two-CTA MMA (256 x 256 tiles) or as pairs of one-CTA MMAs that share each
  // weight tile of a group's consecutive M tiles; the gate/up and the down
  // GEMM choose independently (every mode produces the same bits)
  const bool bf16 = sizeof(T) == 2 && !h->q4;
  const bool mma2 = bf16 && h->mma2_grid > 0 && Tc >= h->mma2_min_tokens;
  const bool mma2_down = bf16 && h->mma2_grid > 0 && Tc >= h->mma2_down_min_tokens;
  const bool pair_ok = bf16 && h->pair_grid > 0 && Tc >= h->pair_min_tokens;
  const bool pair = !mma2 && pair_ok;
  const bool pair_down = !mma2_down && pair_ok;
  GemmParams base = {};
  base.offsets = h->offsets;
  base.T = Tc;
  base.A = A;
  base.n_shared = c.n_shared;
  base.n_routed = E;
  base.status = h->status;
  {
    ProfScope ps(h, MOE_KERNEL_GEMM_GATE_UP, st);
    GemmMaps m;
    // routed rows are gathered from x by the kernel; the shared expert's
    // rows (x in token order) come through this map
    if (!make_map(&m.m[1], x, sizeof(T), Tc, d, kBM)) return MOE_ERR_CUDA;
    m.m[0] = m.m[1];
    m.m[2] = h->tm_wg;
    m.m[3] = h->tm_wu;
    m.m[4] = c.n_shared ? h->tm_sg : h->tm_wg;
    m.m[5] = c.n_shared ? h->tm_su : h->tm_wu;
    GemmParams p = base;
    p.nt = h->nt1;
    p.num_k_blocks = d / BK;
    p.b_rows_per_group = F;
    p.out = h->hbuf;
    p.ldo = F;
    p.kid = KID_GEMM_GATE_UP;
    p.tile_ctr = h->tile_ctr(0);
    p.perm = h->perm;
    p.list = lists ? h->list : nullptr;
    p.list_stride = c.max_tokens;
    p.x = x;
    if (lists) {
      // the cluster router left the histogram: this GEMM scans it into the
      // group offsets (for itself, the down GEMM and the combine) and adds it
      // to the caller's counts
      p.counts_in = h->counts();
      p.offsets_out = h->offsets;
      p.counts_out = ro.counts;
    }
    if (h->q4) {  // 4-bit weights (bf16 tokens): dequantised in the GEMM
      Q4GemmMaps mq = h->q4g;
      mq.a = m.m[1];
      MOE_TRY(launch_gemm_q4<EPI_SWIGLU>(mq, p, h->num_sms, st, pdl));
    } else if (mma2) {
      MOE_TRY(launch_gemm2sm<EPI_SWIGLU>(m, p, h->mma2_grid, st, pdl));
    } else if (pair) {
      MOE_TRY((launch_gemm<__nv_bfloat16, EPI_SWIGLU, kBN, true>(m, p, h->pair_grid, st, pdl)));
    } else {
      MOE_TRY((launch_gemm<T, EPI_SWIGLU, kBN>(m, p, h->num_sms, st, pdl)));
    }
  }
  {
    ProfScope ps(h, MOE_KERNEL_GEMM_DOWN, st);
    GemmMaps m;
    m.m[0] = m.m[1] = h->tm_h;
    m.m[2] = m.m[3] = h->tm_wd;
    m.m[4] = m.m[5] = c.n_shared ? h->tm_sd : h->tm_wd;
    GemmParams p = base;
    p.nt = h->nt2;
    p.num_k_blocks = F / BK;
    p.b_rows_per_group = d;
    p.out = h->yp;
    p.ldo = d;
    p.kid = KID_GEMM_DOWN;
    p.tile_ctr = h->tile_ctr(1);
    // the finished gate/up GEMM read these: clear them for the next call
    p.clear_counts = lists ? h->counts() : nullptr;
    p.clear_ctr = h->tile_ctr(0);
    if (h->q4) {
      MOE_TRY(launch_gemm_q4<EPI_STORE>(h->q4d, p, h->num_sms, st, pdl));
    } else if (pair_down || mma2_down) {
      // 128-row boxes of the down weights
      m.m[3] = h->tm_wd2;
      m.m[5] = c.n_shared ? h->tm_sd2 : h->tm_wd2;
      if (mma2_down) MOE_TRY(launch_gemm2sm<EPI_STORE>(m, p, h->mma2_grid, st, pdl));
      else MOE_TRY((launch_gemm<__nv_bfloat16, EPI_STORE, kBN, true>(m, p, h->pair_grid, st, pdl)));
    } else {
      MOE_TRY((launch_gemm<T, EPI_STORE, kBN>(m, p, h->num_sms, st, pdl)));
    }
  }
  {
    ProfScope ps(h, MOE_KERNEL_COMBINE, st);
    MOE_TRY(launch_combine<T>(static_cast<const T *>(h->yp), h->inv, wts, out, Tc, k, d, A,
                              c.n_shared, h->status, h->num_sms, st, pdl, lists ? idx : nullptr,
                              lists ? h->offsets : nullptr, E, h->tile_ctr(1)));
  }
  return MOE_OK;
}

template <typename T>
int run_decode(moe_handle *h, const T *x, T *out, const RouteOut &ro, cudaStream_t st) {
  const moe_config &c = h->cfg;
  DecodeArgs a = {};
  a.sel_idx = ro.idx;
  a.sel_w = ro.w;
  a.sel_counts = ro.counts;
  a.x = x;
  a.wr = c.w_router;
  a.wg = c.w_gate;
  a.wu = c.w_up;
  a.wd = c.w_down;
  a.sg = c.s_gate;
  a.su = c.s_up;
  a.sd = c.s_down;
  a.bias = c.router_bias;
  a.d = c.d_model;
  a.F = c.d_ff;
  a.E = c.n_experts;
  a.k = c.top_k;
  a.n_shared = c.n_shared;
  a.logits = h->logits;
  a.h = h->hdec;
  a.out = out;
  a.status = h->status;
  const bool pdl = !h->prof;  // event records between kernels would break the chain
  if (h->q4) {
    a.q = h->qw;
    a.dsel = h->dctl;
    {
      ProfScope ps(h, MOE_KERNEL_DECODE_ROUTER, st);
      MOE_TRY(launch_decode_router_q4(a, st, pdl));
    }
    {
      ProfScope ps(h, MOE_KERNEL_DECODE_GATE_UP, st);
      MOE_TRY(launch_decode_gateup_q4(a, st, pdl));
    }
    {
      ProfScope ps(h, MOE_KERNEL_DECODE_DOWN, st);
      MOE_TRY(launch_decode_down_q4(a, st, pdl));
    }
    return MOE_OK;
  }
  {
    ProfScope ps(h, MOE_KERNEL_DECODE_ROUTER, st);
    MOE_TRY(launch_decode_router<T>(a, st, pdl));
  }
  {
    ProfScope ps(h, MOE_KERNEL_DECODE_GATE_UP, st);
    MOE_TRY(launch_decode_gateup<T>(a, h->tm_dg, h->tm_du, st, pdl));
  }
  {
    ProfScope ps(h, MOE_KERNEL_DECODE_DOWN, st);
    MOE_TRY(launch_decode_down<T>(a, st, pdl));
  }
  return MOE_OK;
}

template <typename T>
int set_attrs(const moe_config &c) {
  if (gemm_set_smem_attr<T, EPI_SWIGLU, kBN>() != cudaSuccess) return MOE_ERR_CUDA;
  if (gemm_set_smem_attr<T, EPI_STORE, kBN>() != cudaSuccess) return MOE_ERR_CUDA;
  if (decode_set_smem_attr<T>() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_ALIGNMENT: return "pointer or pitch not 16-byte aligned";
    case MOE_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case MOE_ERR_DEVICE_BOUNDS: return "a device index check failed";
    case MOE_ERR_OUT_OF_MEMORY: return "workspace allocation failed";
    default: return "unknown error";
  }
}

}  // extern "C"

namespace {

// Checks of one 4-bit matrix [rows][cols]: present and 16-byte aligned.
int check_q4(const moe_q4_matrix &m) {
  if (!m.codes || !m.scales || !m.biases) return MOE_ERR_INVALID_ARG;
  if (!aligned16(m.codes) || !aligned16(m.scales) || !aligned16(m.biases)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

Q4Mat q4mat(const moe_q4_matrix &m) { return Q4Mat{m.codes, m.scales, m.biases}; }

// Grouped-GEMM maps of one 4-bit matrix [rows][K]: codes in boxes of 32
// bytes (one 64-column K block) x box_rows, scales and biases in boxes of 8
// groups x box_rows.  K a multiple of 512 (16-byte scale/bias row pitch).
bool make_q4_maps(Q4GemmMaps &q, int i, const moe_q4_matrix &m, uint64_t rows, int K,
                  uint32_t box_rows) {
  return encode_map_2d(&q.c[i], m.codes, 1, rows, K / 2, 32, box_rows, false) &&
         encode_map_2d(&q.s[i], m.scales, 2, rows, K / kQ4Group, 8, box_rows, false) &&
         encode_map_2d(&q.b[i], m.biases, 2, rows, K / kQ4Group, 8, box_rows, false);
}

int create_impl(const moe_config *cfg, const moe_q4_weights *q4, moe_handle **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_cfg(cfg, q4 != nullptr);
  if (rc != MOE_OK) return rc;
  if (q4) {
    const moe_q4_matrix *ms[] = {&q4->gate, &q4->up, &q4->down, &q4->s_gate, &q4->s_up,
                                 &q4->s_down};
    for (int i = 0; i < (cfg->n_shared ? 6 : 3); ++i)
      if ((rc = check_q4(*ms[i])) != MOE_OK) return rc;
    // the batch-1 down kernel gives each thread at most 16 columns of one
    // slot's h, in a CTA of at most 640 threads
    if ((cfg->top_k + cfg->n_shared) * cfg->d_ff > 640 * 16) return MOE_ERR_UNSUPPORTED;
  }
  moe_handle *h = new (std::nothrow) moe_handle();
  if (!h) return MOE_ERR_OUT_OF_MEMORY;
  h->cfg = *cfg;
  const moe_config &c = h->cfg;
  h->esz = c.dtype == MOE_BF16 ? 2 : 4;
  h->nt1 = c.d_ff / kBM;
  h->nt2 = c.d_model / kBN;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
          cudaSuccess) {
    delete h;
    return MOE_ERR_CUDA;
  }
  h->router_pair_min_tokens = static_cast<long long>(kBM) * (h->num_sms / 4) + 1;
  const int d = c.d_model, F = c.d_ff, E = c.n_experts, k = c.top_k, Tm = c.max_tokens;
  const size_t A = static_cast<size_t>(Tm) * k;
  const size_t esz = h->esz;

  // carve the workspace
  struct Part {
    void **dst;
    size_t bytes;
  };
  std::vector<Part> parts = {
      {reinterpret_cast<void **>(&h->idx), sizeof(int32_t) * A},
      {reinterpret_cast<void **>(&h->w), sizeof(float) * A},
      {reinterpret_cast<void **>(&h->inv), sizeof(int32_t) * A},
      {reinterpret_cast<void **>(&h->route_ctl), kRouteCtlBytes},
      {reinterpret_cast<void **>(&h->offsets), sizeof(int32_t) * (E + 1)},
      {reinterpret_cast<void **>(&h->status), sizeof(int32_t) * 4},
      {reinterpret_cast<void **>(&h->logits), sizeof(float) * E},
      {reinterpret_cast<void **>(&h->hdec), sizeof(float) * (k + 1) * F},
      {reinterpret_cast<void **>(&h->dctl), sizeof(int32_t) * 32 * kSelReplicas},
      {reinterpret_cast<void **>(&h->perm), sizeof(int32_t) * A},
      {reinterpret_cast<void **>(&h->list), sizeof(int32_t) * E * static_cast<size_t>(Tm)},
      {&h->hbuf, esz * (A + Tm) * F},
      {&h->yp, esz * (A + Tm) * d},
  };
  size_t total = 0;
  for (auto &p : parts) total = align_up(total, 1024) + p.bytes;
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OUT_OF_MEMORY;
  }
  size_t off = 0;
  for (auto &p : parts) {
    off = align_up(off, 1024);
    *p.dst = static_cast<char *>(h->ws) + off;
    off += p.bytes;
  }
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    moe_destroy(h);
    return MOE_ERR_CUDA;
  }

  // tensor maps of the weights and the fixed workspace buffers
  bool ok = make_map(&h->tm_h, h->hbuf, esz, A + Tm, F, kBM) &&
            make_map(&h->tm_wr256, c.w_router, esz, E, d, 256);
  if (ok && !q4)
    ok = encode_map_2d(&h->tm_dg, c.w_gate, esz, static_cast<uint64_t>(E) * F, d,
                       static_cast<uint32_t>(512 / esz), 32, false) &&
         encode_map_2d(&h->tm_du, c.w_up, esz, static_cast<uint64_t>(E) * F, d,
                       static_cast<uint32_t>(512 / esz), 32, false) &&
         make_map(&h->tm_wg, c.w_gate, esz, static_cast<uint64_t>(E) * F, d, kBM) &&
         make_map(&h->tm_wu, c.w_up, esz, static_cast<uint64_t>(E) * F, d, kBM) &&
         make_map(&h->tm_wd, c.w_down, esz, static_cast<uint64_t>(E) * d, F, kBN) &&
         make_map(&h->tm_wd2, c.w_down, esz, static_cast<uint64_t>(E) * d, F, kBN / 2);
  if (ok && !q4 && c.n_shared)
    ok = make_map(&h->tm_sg, c.s_gate, esz, F, d, kBM) &&
         make_map(&h->tm_su, c.s_up, esz, F, d, kBM) && make_map(&h->tm_sd, c.s_down, esz, d, F, kBN) &&
         make_map(&h->tm_sd2, c.s_down, esz, d, F, kBN / 2);
  if (q4) {
    h->q4 = true;
    h->qw.g = q4mat(q4->gate);
    h->qw.u = q4mat(q4->up);
    h->qw.d = q4mat(q4->down);
    if (c.n_shared) {
      h->qw.sg = q4mat(q4->s_gate);
      h->qw.su = q4mat(q4->s_up);
      h->qw.sd = q4mat(q4->s_down);
    }
    if (ok && decode_q4_set_smem_attr() != cudaSuccess) ok = false;
    // the grouped GEMMs (T >= 2) take K blocks of 64 columns with scale and
    // bias rows of 16-byte pitch: d and F multiples of 512
    h->q4_prefill = d % 512 == 0 && F % 512 == 0;
    if (ok && h->q4_prefill) {
      const uint64_t EF = static_cast<uint64_t>(E) * F, Ed = static_cast<uint64_t>(E) * d;
      ok = make_q4_maps(h->q4g, 0, q4->gate, EF, d, kBN / 2) &&
           make_q4_maps(h->q4g, 1, q4->up, EF, d, kBN / 2) &&
           make_q4_maps(h->q4d, 0, q4->down, Ed, F, kBN);
      if (ok && c.n_shared)
        ok = make_q4_maps(h->q4g, 2, q4->s_gate, F, d, kBN / 2) &&
             make_q4_maps(h->q4g, 3, q4->s_up, F, d, kBN / 2) &&
             make_q4_maps(h->q4d, 2, q4->s_down, d, F, kBN);
      if (ok && !c.n_shared) {  // never used; valid descriptors all the same
        h->q4g.c[2] = h->q4g.c[0], h->q4g.s[2] = h->q4g.s[0], h->q4g.b[2] = h->q4g.b[0];
        h->q4g.c[3] = h->q4g.c[1], h->q4g.s[3] = h->q4g.s[1], h->q4g.b[3] = h->q4g.b[1];
        h->q4d.c[2] = h->q4d.c[0], h->q4d.s[2] = h->q4d.s[0], h->q4d.b[2] = h->q4d.b[0];
      }
      if (ok) {  // the down GEMM has no "up" matrix
        h->q4d.c[1] = h->q4d.c[0], h->q4d.s[1] = h->q4d.s[0], h->q4d.b[1] = h->q4d.b[0];
        h->q4d.c[3] = h->q4d.c[2], h->q4d.s[3] = h->q4d.s[2], h->q4d.b[3] = h->q4d.b[2];
        h->q4d.a = h->tm_h;
        h->q4g.a = h->tm_h;  // replaced by the tokens' map at every call
      }
      if (ok && (gemm_q4_set_smem_attr<EPI_SWIGLU>() != cudaSuccess ||
                 gemm_q4_set_smem_attr<EPI_STORE>() != cudaSuccess))
        ok = false;
    }
  }
  if (!ok) {
    moe_destroy(h);
    return MOE_ERR_CUDA;
  }
  rc = c.dtype == MOE_BF16 ? set_attrs<__nv_bfloat16>(c) : set_attrs<float>(c);
  if (rc == MOE_OK && c.dtype == MOE_BF16 &&
      (router_set_attr() != cudaSuccess || route_small_set_attr() != cudaSuccess || small_gemv_set_attr() != cudaSuccess ||
       small_gemv_q4_set_attr() != cudaSuccess))
    rc = MOE_ERR_CUDA;
  if (rc == MOE_OK && c.dtype == MOE_BF16 && !q4) {
    // cluster-pair grouped GEMMs: as many clusters of two as fit at once
    if (gemm_set_smem_attr<__nv_bfloat16, EPI_SWIGLU, kBN, true>() != cudaSuccess ||
        gemm_set_smem_attr<__nv_bfloat16, EPI_STORE, kBN, true>() != cudaSuccess)
      rc = MOE_ERR_CUDA;
    const int ncl = rc == MOE_OK ? gemm_pair_clusters() : 0;
    cudaGetLastError();
    h->pair_grid = 2 * std::min(ncl, h->num_sms / 2);
    // the same for the two-CTA MMA
    if (rc == MOE_OK && (gemm2sm_set_smem_attr<EPI_SWIGLU>() != cudaSuccess ||
                         gemm2sm_set_smem_attr<EPI_STORE>() != cudaSuccess))
      rc = MOE_ERR_CUDA;
    const int ncl2 = rc == MOE_OK ? gemm2sm_clusters() : 0;
    cudaGetLastError();
    h->mma2_grid = 2 * std::min(ncl2, h->num_sms / 2);
  }
  if (rc != MOE_OK) {
    moe_destroy(h);
    return rc;
  }
  *out = h;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_create(const moe_config *cfg, moe_handle **out) { return create_impl(cfg, nullptr, out); }

int moe_create_q4(const moe_config *cfg, const moe_q4_weights *w, moe_handle **out) {
  if (!w) {
    if (out) *out = nullptr;
    return MOE_ERR_INVALID_ARG;
  }
  return create_impl(cfg, w, out);
}

int moe_quantize_q4(const void *w, moe_dtype dtype, long long rows, int cols, uint8_t *codes,
                    uint16_t *scales, uint16_t *biases, void *cuda_stream) {
  if (rows < 0 || cols <= 0 || cols % kQ4Group) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!w || !codes || !scales || !biases) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(biases))
    return MOE_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (dtype == MOE_BF16)
    MOE_TRY(launch_quantize_q4(static_cast<const __nv_bfloat16 *>(w), rows, cols, codes, scales,
                               biases, st));
  else
    MOE_TRY(launch_quantize_q4(static_cast<const float *>(w), rows, cols, codes, scales, biases, st));
  return MOE_OK;
}

int moe_destroy(moe_handle *h) {
  if (!h) return MOE_OK;
  for (cudaEvent_t e : h->pool) cudaEventDestroy(e);
  int rc = MOE_OK;
  moe_handle::HostStage &hs = h->hs;
  for (cudaStream_t s : {hs.cin, hs.cout})
    if (s && cudaStreamSynchronize(s) != cudaSuccess) rc = MOE_ERR_CUDA;
  for (int i = 0; i < 2; ++i)
    for (cudaEvent_t e : {hs.in_done[i], hs.fwd_done[i], hs.out_done[i]})
      if (e) cudaEventDestroy(e);
  for (cudaStream_t s : {hs.cin, hs.cout})
    if (s) cudaStreamDestroy(s);
  if (hs.buf && cudaFree(hs.buf) != cudaSuccess) rc = MOE_ERR_CUDA;
  if (h->ws && cudaFree(h->ws) != cudaSuccess) rc = MOE_ERR_CUDA;
  delete h;
  return rc;
}

int moe_route(moe_handle *h, const void *x, int T, int32_t *topk_idx, float *topk_w,
              int32_t *counts, void *cuda_stream) {
  if (!h || T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !topk_idx || !topk_w || !counts) return MOE_ERR_INVALID_ARG;
  if (T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x)) return MOE_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const moe_config &c = h->cfg;
  const int d = c.d_model, E = c.n_experts, k = c.top_k;
  ProfScope ps(h, MOE_KERNEL_ROUTER, st);
  if (c.dtype == MOE_BF16) {
    // the router adds each expert's assignments to counts
    MOE_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st));
    if (use_small_route(h, T))
      return launch_route_small(x, c.w_router, c.router_bias, T, d, E, k, topk_idx, topk_w, h->inv,
                                h->perm, h->offsets, counts, h->tile_ctr(0), 2, st) == cudaSuccess
                 ? MOE_OK
                 : MOE_ERR_CUDA;
    return launch_router_bf16(h, x, T, topk_idx, topk_w, counts, st);
  }
  MOE_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st));
  MOE_TRY(launch_router_simt<float>(static_cast<const float *>(x),
                                    static_cast<const float *>(c.w_router), c.router_bias, T, d, E,
                                    k, topk_idx, topk_w, counts, nullptr, st));
  return MOE_OK;
}

namespace {

// 4-bit layers whose d or F the grouped GEMMs do not take run batches only
// where every chunk takes the small-batch kernels
int forward_shape_ok(const moe_handle *h, int T) {
  if (h->q4 && T != 1 && !h->q4_prefill) {
    // 4-bit shapes the grouped GEMMs do not take: every chunk (full ones of
    // max_tokens, then the rest) must run on the small-batch kernels
    const int d = h->cfg.d_model, F = h->cfg.d_ff;
    const int c0 = std::min(T, h->cfg.max_tokens), rest = T % c0;
    for (const int Tc : {c0, rest})
      if (Tc > 0 && !(small_route_ok(Tc, d) && small_gemv_fits(Tc, d, F)))
        return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// The copy streams and events of the host-buffer calls, made on first use.
int host_stage_init(moe_handle *h) {
  moe_handle::HostStage &s = h->hs;
  if (s.cout) return MOE_OK;
  for (int i = 0; i < 2; ++i)
    for (cudaEvent_t *e : {&s.in_done[i], &s.fwd_done[i], &s.out_done[i]})
      if (!*e) MOE_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  if (!s.cin) MOE_TRY(cudaStreamCreateWithFlags(&s.cin, cudaStreamNonBlocking));
  MOE_TRY(cudaStreamCreateWithFlags(&s.cout, cudaStreamNonBlocking));
  return MOE_OK;
}

// Grows both slots to T tokens.  Earlier calls may still be using them, so
// the copy streams and the caller's stream are drained before the old
// buffer is freed.
int host_stage_reserve(moe_handle *h, size_t T, cudaStream_t st) {
  moe_handle::HostStage &s = h->hs;
  if (T <= s.cap) return MOE_OK;
  MOE_TRY(cudaStreamSynchronize(s.cin));
  MOE_TRY(cudaStreamSynchronize(s.cout));
  MOE_TRY(cudaStreamSynchronize(st));
  if (s.buf) MOE_TRY(cudaFree(s.buf));
  s.buf = nullptr;
  s.cap = 0;
  const size_t row = h->esz * h->cfg.d_model;
  if (cudaMalloc(&s.buf, 4 * T * row) != cudaSuccess) {
    s.buf = nullptr;
    cudaGetLastError();
    return MOE_ERR_OUT_OF_MEMORY;
  }
  s.cap = T;
  return MOE_OK;
}

}  // namespace

}  // extern "C"

namespace {

// moe_forward and moe_forward_routed: validation, then the batch-1 path or
// the chunk loop; idx / w / counts as for moe_forward_routed (each may be null).
int forward_impl(moe_handle *h, const void *x, int T, void *out, int32_t *idx, float *w,
                 int32_t *counts, void *cuda_stream) {
  if (!h || T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
  const size_t row = h->esz * h->cfg.d_model;
  const char *xb = static_cast<const char *>(x);
  char *ob = static_cast<char *>(out);
  if (xb < ob + row * T && ob < xb + row * T) return MOE_ERR_INVALID_ARG;  // overlap
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (const int rc = forward_shape_ok(h, T); rc != MOE_OK) return rc;
  // the kernels add to the counts
  if (counts)
    MOE_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * h->cfg.n_experts, st));
  const int k = h->cfg.top_k;
  if (T == 1) {
    const RouteOut ro{idx, w, counts};
    return h->cfg.dtype == MOE_BF16
               ? run_decode<__nv_bfloat16>(h, static_cast<const __nv_bfloat16 *>(x),
                                           static_cast<__nv_bfloat16 *>(out), ro, st)
               : run_decode<float>(h, static_cast<const float *>(x), static_cast<float *>(out),
                                   ro, st);
  }
  for (int c0 = 0; c0 < T; c0 += h->cfg.max_tokens) {
    const int Tc = (T - c0) < h->cfg.max_tokens ? (T - c0) : h->cfg.max_tokens;
    const long long o = static_cast<long long>(c0) * k;
    const RouteOut ro{idx ? idx + o : nullptr, w ? w + o : nullptr, counts};
    int rc;
    if (h->cfg.dtype == MOE_BF16)
      rc = run_prefill_chunk<__nv_bfloat16>(
          h, reinterpret_cast<const __nv_bfloat16 *>(xb + row * c0), Tc,
          reinterpret_cast<__nv_bfloat16 *>(ob + row * c0), ro, st);
    else
      rc = run_prefill_chunk<float>(h, reinterpret_cast<const float *>(xb + row * c0), Tc,
                                    reinterpret_cast<float *>(ob + row * c0), ro, st);
    if (rc != MOE_OK) return rc;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_forward(moe_handle *h, const void *x, int T, void *out, void *cuda_stream) {
  return forward_impl(h, x, T, out, nullptr, nullptr, nullptr, cuda_stream);
}

int moe_forward_routed(moe_handle *h, const void *x, int T, void *out, int32_t *topk_idx,
                       float *topk_w, int32_t *counts, void *cuda_stream) {
  return forward_impl(h, x, T, out, topk_idx, topk_w, counts, cuda_stream);
}

int moe_forward_host(moe_handle *h, const void *x_host, int T, void *out_host,
                     void *cuda_stream) {
  if (!h || T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  const size_t row = h->esz * h->cfg.d_model, bytes = row * T;
  const char *xb = static_cast<const char *>(x_host);
  char *ob = static_cast<char *>(out_host);
  if (xb < ob + bytes && ob < xb + bytes) return MOE_ERR_INVALID_ARG;  // overlap
  if (const int rc = forward_shape_ok(h, T); rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (const int rc = host_stage_init(h); rc != MOE_OK) return rc;
  if (const int rc = host_stage_reserve(h, T, st); rc != MOE_OK) return rc;
  moe_handle::HostStage &s = h->hs;
  const int k = s.next;
  char *xs = s.buf + (2 * k) * s.cap * row, *os = s.buf + (2 * k + 1) * s.cap * row;
  // copy-in: the slot's input is free once the forward two calls back is done
  if (s.used[k]) MOE_TRY(cudaStreamWaitEvent(s.cin, s.fwd_done[k], 0));
  MOE_TRY(cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, s.cin));
  MOE_TRY(cudaEventRecord(s.in_done[k], s.cin));
  // forward: after its input arrived and the slot's previous result left
  MOE_TRY(cudaStreamWaitEvent(st, s.in_done[k], 0));
  if (s.used[k]) MOE_TRY(cudaStreamWaitEvent(st, s.out_done[k], 0));
  if (const int rc = moe_forward(h, xs, T, os, cuda_stream); rc != MOE_OK) return rc;
  MOE_TRY(cudaEventRecord(s.fwd_done[k], st));
  // copy-out
  MOE_TRY(cudaStreamWaitEvent(s.cout, s.fwd_done[k], 0));
  MOE_TRY(cudaMemcpyAsync(out_host, os, bytes, cudaMemcpyDeviceToHost, s.cout));
  MOE_TRY(cudaEventRecord(s.out_done[k], s.cout));
  s.used[k] = true;
  s.last = k;
  s.next = k ^ 1;
  return MOE_OK;
}

int moe_host_join(moe_handle *h, void *cuda_stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  // the copy-out stream runs in order: its last event covers every copy-out
  if (h->hs.last >= 0)
    MOE_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(cuda_stream),
                                h->hs.out_done[h->hs.last], 0));
  return MOE_OK;
}

int moe_status(moe_handle *h, void *cuda_stream, int *detail) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int s[2] = {0, 0};
  if (cudaMemcpy(s, h->status, sizeof s, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(h->status, 0, sizeof s) != cudaSuccess) return MOE_ERR_CUDA;
  // an aborted launch can leave the router's histogram or the GEMMs' tile
  // counters behind
  if (s[0] != MOE_OK && cudaMemset(h->route_ctl, 0, kRouteCtlBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (detail) *detail = s[1];
  return s[0];
}

int moe_set_option(moe_handle *h, int option, long long value) {
  if (!h || value < 0) return MOE_ERR_INVALID_ARG;
  switch (option) {
    case MOE_OPT_PAIR_MIN_TOKENS: h->pair_min_tokens = value; return MOE_OK;
    case MOE_OPT_MMA2_MIN_TOKENS: h->mma2_min_tokens = value; return MOE_OK;
    case MOE_OPT_MMA2_DOWN_MIN_TOKENS: h->mma2_down_min_tokens = value; return MOE_OK;
    case MOE_OPT_ROUTER_PAIR_MIN_TOKENS: h->router_pair_min_tokens = value; return MOE_OK;
    case MOE_OPT_GEMV_MAX_TOKENS:
      if (value > kSmallGemvT) return MOE_ERR_INVALID_ARG;
      h->gemv_max_tokens = static_cast<int>(value);
      return MOE_OK;
    default: return MOE_ERR_INVALID_ARG;
  }
}

int moe_profile(moe_handle *h, int enable) {
  if (!h) return MOE_ERR_INVALID_ARG;
  h->prof = enable != 0;
  if (h->prof) {
    h->recs.clear();
    h->pool_used = 0;
  }
  return MOE_OK;
}

int moe_profile_read(moe_handle *h, float *ms, int64_t *launches, int n) {
  if (!h || n < 0) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (ms) ms[i] = 0.0f;
    if (launches) launches[i] = 0;
  }
  if (!h->recs.empty() && cudaEventSynchronize(h->recs.back().b) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (const ProfRec &r : h->recs) {
    if (r.kind >= n) continue;
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return MOE_ERR_CUDA;
    if (ms) ms[r.kind] += t;
    if (launches) launches[r.kind] += 1;
  }
  return MOE_OK;
}

int moe_debug_wait_timeout(moe_handle *h, int wait_us, void *cuda_stream) {
  if (wait_us < 1 || wait_us > 2000000) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (h) {
    dev = h->device;
  } else if (cudaGetDevice(&dev) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  // no handle: the status word of the allocation-free entry point
  int *status = h ? h->status : noalloc_status_word();
  if (!status) return MOE_ERR_CUDA;
  int clk_khz = 0;
  if (cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  const long long cycles = static_cast<long long>(clk_khz) * wait_us / 1000;
  MOE_TRY(launch_debug_wait(status, cycles, static_cast<cudaStream_t>(cuda_stream)));
  return MOE_OK;
}

}  // extern "C"
