// noalloc.cu -- batch-1 forward of one MoE layer that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's memory manager (the allocator owns the whole device pool), code
// that must not allocate after start-up (real-time or certified serving
// loops), or a plugin that is only handed device pointers.  moe_create
// allocates the workspace of a handle, so such callers cannot use it.  This
// entry point needs no handle: the caller passes the layer description,
// the input token and the output row, and the decode kernels' scratch lives
// in one file-scope device array below that every GPU loading this library
// holds until the process exits.
//
// Scratch layout (4-byte words): [0, 256) router logits, [256, 256 +
// kNoAllocMaxH) the intermediate h of the k routed experts and the shared
// one, then 4 ints: the status word (first error code, detail) that the
// kernels' bounded waits report into.  Within a call every logit and h value
// is written before it is read, so they need no clearing between calls; the
// status word starts at zero (static storage) and is cleared when
// moe_noalloc_status reads it.  The pages describe no allocation-free mode;
// this has no counterpart there.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxH = 16384;                  // (top_k + n_shared) * d_ff at most
constexpr int kNoAllocStatus = 256 + kNoAllocMaxH;   // first word of the status
constexpr int kNoAllocFloats = kNoAllocStatus + 4;   // 66,576 bytes

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: the device address of the
// scratch array.  In host code the array's name is only a host-side stand-in;
// a kernel must be given this address instead.
int setup_device(int dev, float **out) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // the decode kernels stage weight rows in dynamic shared memory
    if (decode_set_smem_attr<__nv_bfloat16>() != cudaSuccess ||
        decode_set_smem_attr<float>() != cudaSuccess)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The status word inside the scratch array of the current device (device
// address), for the failure-path test hook; null when the lookup failed.
int *noalloc_status_word() {
  int dev = 0;
  float *s = nullptr;
  if (cudaGetDevice(&dev) != cudaSuccess || setup_device(dev, &s) != MOE_OK) return nullptr;
  return reinterpret_cast<int *>(s + kNoAllocStatus);
}

}  // namespace moe

using namespace moe;

extern "C" int moe_noalloc_status(void *cuda_stream, int *detail) {
  int *w = noalloc_status_word();
  if (!w) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int s[2] = {0, 0};
  if (cudaMemcpy(s, w, sizeof s, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(w, 0, sizeof s) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = s[1];
  return s[0];
}

extern "C" int moe_decode_noalloc(const moe_config *c, const void *x, void *out,
                                  void *cuda_stream) {
  if (!c || !x || !out) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->d_ff <= 0 || c->n_experts <= 0 || c->top_k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_INVALID_ARG;
  if (!c->w_router || !c->w_gate || !c->w_up || !c->w_down) return MOE_ERR_INVALID_ARG;
  if (c->n_shared && (!c->s_gate || !c->s_up || !c->s_down)) return MOE_ERR_INVALID_ARG;
  if (c->d_model % 256 != 0 || c->d_model > 16384 || c->d_ff % 128 != 0 || c->d_ff > 4096 ||
      c->n_experts > 256 || c->top_k > kMaxTopK || c->top_k > c->n_experts)
    return MOE_ERR_UNSUPPORTED;
  // the static scratch holds h for at most kNoAllocMaxH values
  if ((c->top_k + c->n_shared) * c->d_ff > kNoAllocMaxH) return MOE_ERR_UNSUPPORTED;
  const void *ptrs[] = {x, out, c->w_router, c->w_gate, c->w_up, c->w_down,
                        c->s_gate, c->s_up, c->s_down, c->router_bias};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  const size_t row = static_cast<size_t>(c->d_model) * (c->dtype == MOE_BF16 ? 2 : 4);
  const char *xb = static_cast<const char *>(x);
  const char *ob = static_cast<const char *>(out);
  if (xb < ob + row && ob < xb + row) return MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  float *s = nullptr;
  const int rc = setup_device(dev, &s);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

  DecodeArgs a = {};
  a.x = x;
  a.wr = c->w_router;
  a.wg = c->w_gate;
  a.wu = c->w_up;
  a.wd = c->w_down;
  a.sg = c->s_gate;
  a.su = c->s_up;
  a.sd = c->s_down;
  a.bias = c->router_bias;
  a.d = c->d_model;
  a.F = c->d_ff;
  a.E = c->n_experts;
  a.k = c->top_k;
  a.n_shared = c->n_shared;
  a.logits = s;
  a.h = s + 256;
  a.out = out;
  a.status = reinterpret_cast<int *>(s + kNoAllocStatus);
  const bool bf16 = c->dtype == MOE_BF16;
  if ((bf16 ? launch_decode_router<__nv_bfloat16>(a, st, false)
            : launch_decode_router<float>(a, st, false)) != cudaSuccess)
    return MOE_ERR_CUDA;
  // tensor maps of the gate/up weights for the streaming kernel (host-side
  // descriptors passed by value; nothing is allocated)
  const size_t esz = bf16 ? 2 : 4;
  CUtensorMap tmG, tmU;
  if (!encode_map_2d(&tmG, c->w_gate, esz, static_cast<uint64_t>(c->n_experts) * c->d_ff,
                     c->d_model, static_cast<uint32_t>(512 / esz), 32, false) ||
      !encode_map_2d(&tmU, c->w_up, esz, static_cast<uint64_t>(c->n_experts) * c->d_ff,
                     c->d_model, static_cast<uint32_t>(512 / esz), 32, false))
    return MOE_ERR_CUDA;
  if ((bf16 ? launch_decode_gateup<__nv_bfloat16>(a, tmG, tmU, st, false)
            : launch_decode_gateup<float>(a, tmG, tmU, st, false)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if ((bf16 ? launch_decode_down<__nv_bfloat16>(a, st, false)
            : launch_decode_down<float>(a, st, false)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
