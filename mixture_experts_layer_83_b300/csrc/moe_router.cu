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

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

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

// Does (ka, ea) precede (kb, eb) in the selection order: larger key first, then lower id.
__device__ __forceinline__ bool before(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

// One warp per token.  Lane l holds experts l, l+32, ... (NV slots).  k rounds: every lane
// proposes its best untaken expert, a butterfly of shuffles agrees on the warp's best, the
// owning lane marks it taken and lane r keeps round r's winner.  A NaN key is treated as
// -inf, so the chosen ids are always distinct and in range.
//   SRC 0: a = logits, softmax weights over the chosen logits.
//   SRC 1: a = logits, key = sigmoid(logit), weights = renormalised sigmoids.
//   SRC 2: a = supplied keys, b = supplied scores, weights = renormalised scores.
// The optional bias is added to the key (SRC 0/1) and never to the weights.
// Group-limited routing (G > 0; page "Expert-Parallel MoE Inference", "Load imbalance and how
// to fight it": node-limited routing caps how many groups of experts a token may span): the
// experts form G contiguous groups of E / G; a group's score is its largest key; the M best
// groups are kept (equal scores: the lower group id) and the experts of the other groups are
// excluded before the k rounds.
template <int NV, int SRC>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ a,
                                                   const float* __restrict__ b,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int k, int G, int M, int* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    float key[NV], val[NV];
    uint32_t taken = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int e = lane + 32 * v;
      float kv = -INFINITY, vv = 0.f;
      if (e < E) {
        const float s = a[(size_t)t * E + e];
        if (SRC == 0) {
          kv = s;
          vv = s;
        } else if (SRC == 1) {
          vv = s;
          kv = 1.f / (1.f + expf(-s));
        } else {
          kv = s;
          vv = b[(size_t)t * E + e];
        }
        if (SRC != 2 && bias != nullptr) kv += bias[e];
        if (kv != kv) kv = -INFINITY;
      } else {
        taken |= 1u << v;
      }
      key[v] = kv;
      val[v] = vv;
    }
    if (G > 0) {
      const int gsz = E / G;
      float my_g = -INFINITY;  // lane g holds group g's score
      for (int g = 0; g < G; ++g) {
        float m = -INFINITY;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int e = lane + 32 * v;
          if (e < E && e / gsz == g) m = fmaxf(m, key[v]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
        if (lane == g) my_g = m;
      }
      uint32_t gsel = 0;
      for (int r = 0; r < M; ++r) {
        const bool cand = lane < G && !((gsel >> lane) & 1u);
        float bk = cand ? my_g : -INFINITY;
        int be = cand ? lane : INT_MAX;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ok = __shfl_xor_sync(kFull, bk, off);
          const int oe = __shfl_xor_sync(kFull, be, off);
          if (before(ok, oe, bk, be)) {
            bk = ok;
            be = oe;
          }
        }
        gsel |= 1u << be;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int e = lane + 32 * v;
        if (e < E && !((gsel >> (e / gsz)) & 1u)) taken |= 1u << v;
      }
    }
    int my_e = 0;
    float my_val = 0.f;
    for (int r = 0; r < k; ++r) {
      float bk = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int e = lane + 32 * v;
        if (!((taken >> v) & 1u) && before(key[v], e, bk, be)) {
          bk = key[v];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(kFull, bk, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (before(ok, oe, bk, be)) {
          bk = ok;
          be = oe;
        }
      }
      const int wl = be & 31, wv = be >> 5;
      float wval = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v)
        if (v == wv) wval = val[v];
      wval = __shfl_sync(kFull, wval, wl);
      if (lane == wl) taken |= 1u << wv;
      if (lane == r) {
        my_e = be;
        my_val = wval;
      }
    }
    float s;
    if (SRC == 0) {
      float m = lane < k ? my_val : -INFINITY;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      s = lane < k ? expf(my_val - m) : 0.f;
    } else if (SRC == 1) {
      s = lane < k ? 1.f / (1.f + expf(-my_val)) : 0.f;
    } else {
      s = lane < k ? my_val : 0.f;
    }
    float sum = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = s / sum;
    }
  }
}

template <int NV>
cudaError_t launch_topk_nv(int src, const float* a, const float* b, const float* bias, int T,
                           int E, int k, int G, int M, int* idx, float* w, cudaStream_t s) {
  const int threads = 256, wpb = threads / 32;
  int blocks = (T + wpb - 1) / wpb;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (src == 0)
    topk_kernel<NV, 0><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w);
  else if (src == 1)
    topk_kernel<NV, 1><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w);
  else
    topk_kernel<NV, 2><<<blocks, threads, 0, s>>>(a, b, bias, T, E, k, G, M, idx, w);
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
                        int k, int G, int M, int* topk_idx, float* topk_w, cudaStream_t s) {
  const int nv = (E + 31) / 32;
  if (nv <= 1) return launch_topk_nv<1>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
  if (nv <= 2) return launch_topk_nv<2>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
  if (nv <= 4) return launch_topk_nv<4>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
  if (nv <= 8) return launch_topk_nv<8>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
  if (nv <= 16) return launch_topk_nv<16>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
  return launch_topk_nv<32>(src, a, b, bias, T, E, k, G, M, topk_idx, topk_w, s);
}

}  // namespace moe
