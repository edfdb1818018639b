// Per-token expert selection shared by the routing kernels (the top-k kernel over stored keys
// and the fused router's epilogue): one warp per token, lane l holding experts l, l + 32, ...
//
// Page "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section "Deeper
// Analysis": a linear gate scores every expert, a softmax is applied and the top-k are kept;
// their outputs are later combined weighted by the gate scores.
#pragma once
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

namespace moe {

// Does (ka, ea) precede (kb, eb) in the selection order: larger key first, then lower id.
__device__ __forceinline__ bool select_before(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

// Selection key and gate value of one expert from its stored value(s).
//   SRC 0: a = logit; key = logit, value = logit (softmax over the chosen logits).
//   SRC 1: a = logit; key = sigmoid(logit), value = logit (renormalised sigmoids).
//   SRC 2: a = supplied key, b = supplied score.
// The expert's selection bias (0 when the layer has none) is added to the key (SRC 0/1) and
// never to the value.  A NaN key becomes -inf, so the chosen ids are always distinct and in
// range.
template <int SRC>
__device__ __forceinline__ void select_key(float a, float b, float bias_e, float& key, float& val) {
  if (SRC == 0) {
    key = a;
    val = a;
  } else if (SRC == 1) {
    val = a;
    key = 1.f / (1.f + expf(-a));
  } else {
    key = a;
    val = b;
  }
  if (SRC != 2) key += bias_e;
  if (key != key) key = -INFINITY;
}

// The warp's token: key[v] / val[v] hold experts lane + 32 v (bit v of `taken` set for experts
// past E).  Group-limited routing (G > 0; page "Expert-Parallel MoE Inference", "Load
// imbalance and how to fight it": node-limited routing caps how many groups of experts a token
// may span): the experts form G contiguous groups of E / G; a group's score is its largest
// key; the M best groups are kept (equal scores: the lower group id) and the experts of the
// other groups are excluded.  Then k rounds: every lane proposes its best untaken expert, a
// butterfly of shuffles agrees on the warp's best, the owning lane marks it taken and lane r
// keeps round r's winner.  Lanes r < k write expert r of the token (key-descending order) and
// its renormalised gate weight to out_idx[r], out_w[r].
// Candidate mode (kc > k, for rerouting at an expert capacity): kc rounds, and lanes r < kc
// write expert r and its raw value (no renormalisation) instead.
template <int NV, int SRC>
__device__ __forceinline__ void select_topk(const float (&key)[NV], const float (&val)[NV],
                                            uint32_t taken, int E, int k, int G, int M,
                                            int* out_idx, float* out_w, int kc = 0) {
  const bool cands = kc > k;
  const int rounds = cands ? kc : k;
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
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
        if (select_before(ok, oe, bk, be)) {
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
  for (int r = 0; r < rounds; ++r) {
    float bk = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int e = lane + 32 * v;
      if (!((taken >> v) & 1u) && select_before(key[v], e, bk, be)) {
        bk = key[v];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(kFull, bk, off);
      const int oe = __shfl_xor_sync(kFull, be, off);
      if (select_before(ok, oe, bk, be)) {
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
  if (cands) {
    if (lane < kc) {
      out_idx[lane] = my_e;
      out_w[lane] = my_val;
    }
    return;
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
    out_idx[lane] = my_e;
    out_w[lane] = s / sum;
  }
}

}  // namespace moe
