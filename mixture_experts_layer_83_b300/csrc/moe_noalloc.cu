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

// Device address of g_route_scratch on the current device.  Host code only sees a stand-in
// for the array, so the address is looked up once per device (with that device current) and
// cached.
int scratch_address(int** out) {
  static std::mutex mu;
  static int* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> g(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    addr[dev] = static_cast<int*>(p);
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
  if (launch_dispatch(topk_idx, s->T, s->k, s->E, 256, scratch, expert_counts, expert_offsets,
                      nullptr, 0, 0, nullptr, INT_MAX, nullptr, sorted_token, slot_pos, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
