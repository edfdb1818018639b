// Expert SwiGLU FFN for fp32 layers, on CUDA cores in true fp32 (no TF32), one thread per
// output element.  Routed rows are the expert-contiguous gathered rows xs[0..R) whose expert
// is found from the segment offsets; the shared expert's rows read x directly and are
// stored after the routed ones (h_sh, and y rows R..R+T).  This path exists for fp32 layers;
// bf16 layers run the tensor-core grouped GEMM instead.
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {
namespace {

// Segment of a sorted row: the e with offsets[e] <= row < offsets[e+1] (empty segments skipped).
__device__ __forceinline__ int segment_of(const int* __restrict__ offsets, int E, int row) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= row) lo = mid;
    else hi = mid;
  }
  return lo;
}

__global__ void ffn_gateup_f32_kernel(const float* __restrict__ xs, const float* __restrict__ x,
                                      const int* __restrict__ offsets, int E, int R, int T_sh,
                                      int d, int F, int Fs, const float* __restrict__ wgu,
                                      const float* __restrict__ sh_wgu, float* __restrict__ h,
                                      float* __restrict__ h_sh) {
  const size_t n_routed = (size_t)R * F;
  const size_t n = n_routed + (size_t)T_sh * Fs;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const float* a;
    const float* wg;
    const float* wu;
    float* dst;
    if (i < n_routed) {
      const int row = (int)(i / F), f = (int)(i % F);
      if (row >= offsets[E]) continue;  // past the rows dispatched under a capacity
      const int e = segment_of(offsets, E, row);
      a = xs + (size_t)row * d;
      wg = wgu + ((size_t)e * 2 * F + f) * d;
      wu = wgu + ((size_t)e * 2 * F + F + f) * d;
      dst = h + i;
    } else {
      const size_t j = i - n_routed;
      const int row = (int)(j / Fs), f = (int)(j % Fs);
      a = x + (size_t)row * d;
      wg = sh_wgu + (size_t)f * d;
      wu = sh_wgu + (size_t)(Fs + f) * d;
      dst = h_sh + j;
    }
    float g = 0.f, u = 0.f;
    for (int c = 0; c < d; ++c) {
      g = fmaf(a[c], wg[c], g);
      u = fmaf(a[c], wu[c], u);
    }
    *dst = g / (1.f + expf(-g)) * u;
  }
}

__global__ void ffn_down_f32_kernel(const float* __restrict__ h, const float* __restrict__ h_sh,
                                    const int* __restrict__ offsets, int E, int R, int T_sh, int d,
                                    int F, int Fs, const float* __restrict__ wd,
                                    const float* __restrict__ sh_wd, float* __restrict__ y) {
  const size_t n = (size_t)(R + T_sh) * d;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / d), c = (int)(i % d);
    const float* a;
    const float* w;
    int K;
    if (row < R) {
      if (row >= offsets[E]) continue;  // past the rows dispatched under a capacity
      const int e = segment_of(offsets, E, row);
      a = h + (size_t)row * F;
      w = wd + ((size_t)e * d + c) * F;
      K = F;
    } else {
      a = h_sh + (size_t)(row - R) * Fs;
      w = sh_wd + (size_t)c * Fs;
      K = Fs;
    }
    float acc = 0.f;
    for (int f = 0; f < K; ++f) acc = fmaf(a[f], w[f], acc);
    y[i] = acc;
  }
}

int grid_for(size_t n) {
  size_t b = (n + 255) / 256;
  if (b > 148 * 64) b = 148 * 64;
  return (int)(b == 0 ? 1 : b);
}

}  // namespace

// stage 0: gate/up + SwiGLU into h / h_sh; stage 1: down projection into y.
cudaError_t launch_ffn_f32(const float* xs, const float* x, const int* offsets, int E, int R,
                           int T_sh, int d, int F, int Fs, const float* w_gate_up,
                           const float* w_down, const float* sh_gate_up, const float* sh_down,
                           float* h, float* h_sh, float* y, cudaStream_t s, int stage) {
  if (stage == 0) {
    const size_t n = (size_t)R * F + (size_t)T_sh * Fs;
    ffn_gateup_f32_kernel<<<grid_for(n), 256, 0, s>>>(xs, x, offsets, E, R, T_sh, d, F, Fs,
                                                      w_gate_up, sh_gate_up, h, h_sh);
  } else {
    const size_t n = (size_t)(R + T_sh) * d;
    ffn_down_f32_kernel<<<grid_for(n), 256, 0, s>>>(h, h_sh, offsets, E, R, T_sh, d, F, Fs, w_down,
                                                    sh_down, y);
  }
  return cudaGetLastError();
}

}  // namespace moe
