// Device twin of the seeded input generator in moe_inputs/host.py.
//
// Same recipe, same operation order: splitmix64 words, 53-bit uniforms, Marsaglia-Bray
// polar normals with a self-contained atanh-series logarithm, fp64 -> fp32 -> bf16 rounding
// (both round-to-nearest-even).  Every fp64 operation uses an explicitly rounded intrinsic
// (__dadd_rn, __dmul_rn, __ddiv_rn, __dsqrt_rn) so that no multiply-add is contracted and
// the results are bit-identical to the numpy twin.  Holds no arithmetic of the MoE layer.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kM2 = 0x94D049BB133111EBull;
constexpr int kAtanhTerms = 12;
constexpr int kMaxAttempts = 64;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * kM1;
  z = (z ^ (z >> 27)) * kM2;
  return z ^ (z >> 31);
}

__device__ inline uint64_t word(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * kG); }

__device__ inline double unit53(uint64_t w) {
  return __dmul_rn((double)(w >> 11), 0x1p-53);
}

__device__ double ln_series(double s) {
  const double kLn2 = 0x1.62e42fefa39efp-1;
  const double kSqrtHalf = 0x1.6a09e667f3bcdp-1;
  int e;
  double m = frexp(s, &e);
  if (m < kSqrtHalf) {
    m = __dmul_rn(m, 2.0);
    e -= 1;
  }
  double t = __ddiv_rn(__dadd_rn(m, -1.0), __dadd_rn(m, 1.0));
  double w = __dmul_rn(t, t);
  double p = __ddiv_rn(1.0, (double)(2 * kAtanhTerms + 1));
  for (int n = kAtanhTerms - 1; n >= 0; --n)
    p = __dadd_rn(__dmul_rn(p, w), __ddiv_rn(1.0, (double)(2 * n + 1)));
  return __dadd_rn(__dmul_rn((double)e, kLn2), __dmul_rn(__dmul_rn(2.0, t), p));
}

__device__ double normal_at(uint64_t key, uint64_t i) {
  for (int a = 0; a < kMaxAttempts; ++a) {
    uint64_t n1 = (i * (uint64_t)kMaxAttempts + (uint64_t)a) * 2ull;
    double u = __dadd_rn(__dmul_rn(2.0, unit53(word(key, n1))), -1.0);
    double v = __dadd_rn(__dmul_rn(2.0, unit53(word(key, n1 + 1))), -1.0);
    double s = __dadd_rn(__dmul_rn(u, u), __dmul_rn(v, v));
    if (s < 1.0 && s > 0.0) {
      double q = __ddiv_rn(__dmul_rn(-2.0, ln_series(s)), s);
      return __dmul_rn(u, __dsqrt_rn(q));
    }
  }
  return 0.0;
}

__global__ void fill_normal_kernel(void* dst, int is_bf16, uint64_t n, uint64_t key, double stdv) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float f = __double2float_rn(__dmul_rn(normal_at(key, i), stdv));
    if (is_bf16)
      reinterpret_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(f);
    else
      reinterpret_cast<float*>(dst)[i] = f;
  }
}

__global__ void fill_uniform_kernel(float* dst, uint64_t n, uint64_t key, double lo, double hi) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  double span = __dadd_rn(hi, -lo);
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = __double2float_rn(__dadd_rn(lo, __dmul_rn(span, unit53(word(key, i)))));
}

uint64_t stream_key(uint64_t seed, uint64_t tid) {
  uint64_t k0 = mix64((seed + 1) * kG);
  return mix64(k0 ^ ((tid + 1) * kG));
}

int grid_for(uint64_t n) {
  uint64_t blocks = (n + 255) / 256;
  return (int)(blocks > 148ull * 64 ? 148ull * 64 : (blocks == 0 ? 1 : blocks));
}

}  // namespace

extern "C" {

// Fill dst[0..n) with N(0, stdv^2) draws of tensor `tid` under `seed`; dtype 0 = fp32, 1 = bf16.
// dst is device memory owned by the caller.  Returns 0 or the cudaError_t of the launch.
int moegen_fill_normal(void* dst, int dtype, uint64_t n, uint64_t seed, uint64_t tid, double stdv,
                       cudaStream_t stream) {
  if (n == 0) return 0;
  fill_normal_kernel<<<grid_for(n), 256, 0, stream>>>(dst, dtype == 1, n, stream_key(seed, tid), stdv);
  return (int)cudaGetLastError();
}

// Fill dst[0..n) (fp32) with U(lo, hi) draws of tensor `tid` under `seed`.
int moegen_fill_uniform(float* dst, uint64_t n, uint64_t seed, uint64_t tid, double lo, double hi,
                        cudaStream_t stream) {
  if (n == 0) return 0;
  fill_uniform_kernel<<<grid_for(n), 256, 0, stream>>>(dst, n, stream_key(seed, tid), lo, hi);
  return (int)cudaGetLastError();
}

}  // extern "C"
