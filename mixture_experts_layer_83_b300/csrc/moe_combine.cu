// Combine: out[t] = sum_j w_tj * y[slot_pos[t][j]] (+ y[R + t] for the shared expert),
// accumulated in fp32 in the fixed order j = 0..k-1, then the shared row, rounded once.
// No atomics: each output element is owned by one thread, so the result is bit-identical
// from run to run.  This is the one-GPU form of the combine all-to-all: expert outputs are
// weighted, summed and put back in token order (page "Expert-Parallel MoE Inference:
// Serving Sparse Models at Scale", "Deeper Analysis"; page "MoE Expert Parallelism in
// Practice", "Core Principles" part 1).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4& v, float w) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}

// One warp per work item: a span of kChunkVec 16-byte vectors (2 KiB) of one token's output
// row, so a short batch still spreads over many warps (each output element keeps its fixed
// summation order, so the result does not depend on the split).  The warp stages the k (slot
// position, weight) pairs of its token in shared memory, then each lane owns the span's
// vectors lane, lane + 32, ...
constexpr int kChunkVec = 128;

__global__ void __launch_bounds__(256) combine_bf16_kernel(
    const uint4* __restrict__ y, const int* __restrict__ slot_pos, const float* __restrict__ w,
    int T, int k, int nvec, int R, int has_shared, uint4* __restrict__ out) {
  __shared__ int s_pos[8][32];
  __shared__ float s_w[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  const int chunks = (nvec + kChunkVec - 1) / kChunkVec;
  const long long items = (long long)T * chunks;
  for (long long it = (long long)blockIdx.x * wpb + warp; it < items; it += (long long)gridDim.x * wpb) {
    const int t = static_cast<int>(it / chunks);
    const int c = static_cast<int>(it - (long long)t * chunks);
    if (lane < k) {
      s_pos[warp][lane] = slot_pos[(size_t)t * k + lane];
      s_w[warp][lane] = w[(size_t)t * k + lane];
    }
    __syncwarp();
    const int v_end = min(nvec, (c + 1) * kChunkVec);
    for (int v = c * kChunkVec + lane; v < v_end; v += 32) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; ++j)
        if (s_pos[warp][j] >= 0)  // an assignment dropped at capacity contributes nothing
          acc_bf16x8(acc, __ldg(y + (size_t)s_pos[warp][j] * nvec + v), s_w[warp][j]);
      if (has_shared) acc_bf16x8(acc, __ldg(y + (size_t)(R + t) * nvec + v), 1.f);
      uint4 o;
      __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) oh[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      out[(size_t)t * nvec + v] = o;
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(256) combine_f32_kernel(
    const float* __restrict__ y, const int* __restrict__ slot_pos, const float* __restrict__ w,
    int T, int k, int d, int R, int has_shared, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const int my_pos = lane < k ? slot_pos[(size_t)t * k + lane] : 0;
    const float my_w = lane < k ? w[(size_t)t * k + lane] : 0.f;
    for (int c0 = 0; c0 < d; c0 += 32) {
      const int c = c0 + lane;
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int p = __shfl_sync(kFull, my_pos, j);
        const float wj = __shfl_sync(kFull, my_w, j);
        if (c < d && p >= 0) acc = fmaf(wj, y[(size_t)p * d + c], acc);
      }
      if (c < d) {
        if (has_shared) acc += y[(size_t)(R + t) * d + c];
        out[(size_t)t * d + c] = acc;
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(const void* y, const int* slot_pos, const float* topk_w, int T, int k,
                           int d, int R, int has_shared, int bf16, void* out, cudaStream_t s) {
  const int threads = 256, wpb = threads / 32;
  int blocks = (T + wpb - 1) / wpb;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (bf16) {
    const long long items = (long long)T * ((d / 8 + kChunkVec - 1) / kChunkVec);
    const long long b16 = (items + wpb - 1) / wpb;
    combine_bf16_kernel<<<(int)(b16 < 148 * 32 ? b16 : 148 * 32), threads, 0, s>>>(
        static_cast<const uint4*>(y), slot_pos, topk_w, T, k, d / 8, R, has_shared,
        static_cast<uint4*>(out));
  } else {
    combine_f32_kernel<<<blocks, threads, 0, s>>>(static_cast<const float*>(y), slot_pos, topk_w,
                                                  T, k, d, R, has_shared, static_cast<float*>(out));
  }
  return cudaGetLastError();
}

}  // namespace moe
