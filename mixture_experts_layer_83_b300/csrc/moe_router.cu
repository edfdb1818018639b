// Router kernels: true-fp32 gate logits on CUDA cores (fp32 layers; bf16 layers compute the
// logits with the tensor-core GEMM) and the warp-per-token top-k with renormalisation.
//
// Page "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section "Deeper
// Analysis": a linear gate scores every expert for every token, a softmax is applied and the
// top-k are kept; their outputs are later combined weighted by the gate scores.
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>

#include "moe_internal.h"
#include "route_select.cuh"

namespace moe {
namespace {

__global__ void router_logits_f32_kernel(const float* __restrict__ x, const float* __restrict__ wr,
                                         int T, int d, int E, float* __restrict__ logits) {
  const size_t n = (size_t)T * E;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / E), e = (int)(i % E);
    const float* xr = x + (size_t)t * d;
    const float* wrow = wr + (size_t)e * d;
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(xr[c], wrow[c], acc);
    logits[i] = acc;
  }
}

// One warp per token: the token's keys are read (lane l holds experts l, l + 32, ...) and
// select_topk picks and renormalises its k experts (see route_select.cuh).
template <int NV, int SRC>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ a,
                                                   const float* __restrict__ b,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int k, int G, int M, int* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w, int kc) {
  const int ko = kc > k ? kc : k;  // outputs per token
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  float be[NV];  // this lane's experts' selection bias
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int e = lane + 32 * v;
    be[v] = bias != nullptr && e < E ? bias[e] : 0.f;
  }
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    float key[NV], val[NV];
    uint32_t taken = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int e = lane + 32 * v;
      key[v] = -INFINITY;
      val[v] = 0.f;
      if (e < E)
        select_key<SRC>(a[(size_t)t * E + e], SRC == 2 ? b[(size_t)t * E + e] : 0.f, be[v],
                        key[v], val[v]);
      else
        taken |= 1u << v;
    }
    select_topk<NV, SRC>(key, val, taken, E, k, G, M, topk_idx + (size_t)t * ko,
                         topk_w + (size_t)t * ko, kc);
  }
}

template <int NV>
cudaError_t launch_topk_nv(int src, const float* a, const float* b, const float* bias, int T,
                           int E, int k, int G, int M, int* idx, float* w, int kc, cudaStream_t s) {
  const int threads = 256, wpb = threads / 32;
  int blocks = (T + wpb - 1) / wpb;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (src == 0)
    topk_kernel<NV, 0><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w, kc);
  else if (src == 1)
    topk_kernel<NV, 1><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w, kc);
  else
    topk_kernel<NV, 2><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w, kc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits_f32(const float* x, const float* w_router, int T, int d, int E,
                                     float* logits, cudaStream_t s) {
  const size_t n = (size_t)T * E;
  size_t blocks = (n + 255) / 256;
  if (blocks > 148 * 64) blocks = 148 * 64;
  router_logits_f32_kernel<<<(int)blocks, 256, 0, s>>>(x, w_router, T, d, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_topk(int src, const float* a, const float* b, const float* bias, int T, int E,
                        int k, int G, int M, int* topk_idx, float* topk_w, cudaStream_t s, int kc) {
  const int nv = (E + 31) / 32;
  if (nv <= 1) return launch_topk_nv<1>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
  if (nv <= 2) return launch_topk_nv<2>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
  if (nv <= 4) return launch_topk_nv<4>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
  if (nv <= 8) return launch_topk_nv<8>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
  if (nv <= 16) return launch_topk_nv<16>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
  return launch_topk_nv<32>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, kc, s);
}

}  // namespace moe
