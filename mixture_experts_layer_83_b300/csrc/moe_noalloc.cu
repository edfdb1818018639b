// Routing and dispatch tables without a caller-provided workspace.
//
// moe_route_from_keys needs a little device scratch (the per-chunk expert histogram of the
// dispatch).  Some callers cannot hand it any: code that runs where allocating device memory
// is not allowed or not available (inside a memory pool that is already fully carved up, a
// plugin whose host framework owns every allocation, or a C caller with no allocator wired
// up).  For them this entry point keeps that scratch in a fixed array compiled into the
// library, so a call needs only its inputs and outputs.
//
// The array lives in every GPU that loads the library until the process exits.  Its size is
// fixed (MOE_NOALLOC_SCRATCH_BYTES); shapes that need more are rejected.  All calls on a
// device share it, so calls whose work overlaps on the GPU (different streams, or different
// host threads) race on it and must be serialised by the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe_layer.h"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kScratchInts = MOE_NOALLOC_SCRATCH_BYTES / sizeof(int);

// Per-chunk expert histogram of the dispatch (chunks of kDispatchChunk assignments x E).
// Nothing in it needs to start at zero: every call's histogram kernel writes each entry the
// call later reads.
static __device__ __align__(256) int g_route_scratch[kScratchInts];

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The CUDA driver API's cuCtxGetCurrent, reached through the runtime (the library links no
// driver library directly).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// Device address of g_route_scratch on the current device.  Host code only sees a stand-in
// for the array, so the address is looked up with the device current and cached together with
// the context it belongs to: a reset of the device (a new primary context loads the module
// again, at a new address) makes the next call look it up again.
int scratch_address(int** out) {
  static std::mutex mu;
  static int* addr[kMaxDevices] = {nullptr};
  static CUcontext ctx_of[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;  // null until the runtime has made a context current
  if (get(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> g(mu);
  if (addr[dev] == nullptr || ctx == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    // the lookup makes the device's primary context current if none is
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MOE_ERR_CUDA;
    addr[dev] = static_cast<int*>(p);
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_route_from_keys_noalloc(const moe_shape* s, const float* sel_key,
                                           const float* gate_score, int* topk_idx,
                                           float* topk_w, int* expert_counts,
                                           int* expert_offsets, int* sorted_token,
                                           int* slot_pos, cudaStream_t stream) {
  using namespace moe;
  if (s == nullptr || s->T < 1 || s->E < 1 || s->k < 1 || s->k > s->E || s->k > 32 ||
      s->E > 1024 || (long long)s->T * s->k > INT_MAX / 2)
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {sel_key, gate_score, topk_idx, topk_w, expert_counts, expert_offsets,
                        sorted_token, slot_pos};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  const long long R = (long long)s->T * s->k;
  const long long chunks = (R + kDispatchChunk - 1) / kDispatchChunk;
  if (chunks * s->E > (long long)kScratchInts) return MOE_ERR_WORKSPACE;
  int* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  if (launch_topk(2, sel_key, gate_score, nullptr, s->T, s->E, s->k, 0, 0, topk_idx, topk_w, stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_dispatch(topk_idx, s->T, s->k, s->E, 256, 0, scratch, expert_counts, expert_offsets,
                      nullptr, 0, 0, nullptr, INT_MAX, nullptr, sorted_token, slot_pos, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
