// moe_route_noalloc: the router entry point for callers that cannot allocate
// device memory when they call it -- e.g. a serving engine whose memory pool
// has reserved the whole device for weights and the KV cache up front, code
// that must not re-enter its own allocator, or a plain C caller with no
// device allocator at hand.  Its scratch (the router's token-block
// completion counters and, when needed, the fp32 logits) is a fixed array
// inside this library instead of a caller-provided workspace.
#include <string.h>

#include <mutex>

#include "moe.h"
#include "moe_internal.cuh"

namespace {

// Layout of the array: moe_route's workspace for the largest call it takes,
// [status 256 B][token-block counters][logits T*E fp32].
constexpr size_t kScratchBytes =
    moe::kRouteCntOffset + moe::kRouteCntBytes + moe::ws_align_up(4 * static_cast<size_t>(MOE_NOALLOC_MAX_LOGITS));

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_route_scratch on the current device, looked up once
// per device (the name is only a host-side stand-in in host code).
void* scratch_on_current_device(moe_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      *st = MOE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *st = MOE_OK;
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" moe_status moe_route_noalloc(const moe_bf16* x, int T, int H, const moe_bf16* gate,
                                        const float* router_bias, const float* expert_bias,
                                        const moe_recipe* recipe, float* logits_out, int32_t* topk_idx,
                                        float* topk_w, cudaStream_t stream) {
  // the checks moe_route makes, before anything touches the shared array
  moe_status st = moe::route_check_args(x, T, H, gate, recipe, topk_idx, topk_w);
  if (st != MOE_OK || T == 0) return st;
  // sizes beyond the fixed array are refused before anything runs
  if (T > MOE_NOALLOC_MAX_TOKENS || static_cast<long long>(T) * recipe->num_experts > MOE_NOALLOC_MAX_LOGITS)
    return MOE_ERR_UNSUPPORTED;
  void* scratch = scratch_on_current_device(&st);
  if (st != MOE_OK) return st;
  // the counters must start at zero; the array keeps the previous call's contents
  const size_t used = moe::kRouteCntOffset + moe::ws_align_up(4 * static_cast<size_t>(moe::ceil_div(T, 4) + 1));
  if (cudaMemsetAsync(scratch, 0, used, stream) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_route(x, T, H, gate, router_bias, expert_bias, recipe, logits_out, topk_idx, topk_w, scratch,
                   kScratchBytes, stream);
}
