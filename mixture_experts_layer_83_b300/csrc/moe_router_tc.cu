// The fused router of the bf16 layer (E <= 256): gate GEMM on the tensor cores, then the
// score (softmax or sigmoid + selection bias), top-k and renormalisation in the GEMM's own
// epilogue, so the fp32 logits never travel through HBM (page "Expert-Parallel MoE Inference:
// Serving Sparse Models at Scale", section "Deeper Analysis": a linear gate scores every
// expert, a softmax is applied and the top-k are kept).
//
// A CTA pair (2-CTA cluster, tcgen05 cta_group::2) owns a block of N tokens: the MMA's M = 256
// rows are the experts (this CTA's 128 rows are experts 128 * rank .. + 127; rows past E are
// zero-filled by TMA and never selected), N = the block's tokens (each CTA holds N / 2 rows
// of x per stage).  Four producer warps stream weight and token tiles through a TMA ring (each
// owns every fourth stage), warp 1 of the even CTA issues the MMAs into tensor memory, warps
// 2..5 move the fp32 logits out of tensor memory.  CTA r selects for tokens r * N / 2 .. of
// the block, so each CTA's epilogue writes the logits of its 128 experts straight into the
// shared memory of the CTA that selects for the token ([token][256 experts], the peer's half
// through distributed shared memory).  Then every warp of both CTAs selects, one warp per
// token, from its own shared memory, and writes the token's k experts and gate weights.
//
// Short batches (decode) have too few token blocks to fill the GPU, so the reduction over d is
// split over S pairs per block: each writes its partial logits to the workspace, and the last
// CTA of the block to arrive (a per-block counter) sums the S partials in split order, so the
// result does not depend on which CTA arrives last, and selects for the whole block.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"
#include "route_select.cuh"

namespace moe {
namespace {

// warps 0, 6, 7, 8: producers; 1: MMA issuer; 2..5: epilogue; all nine select afterwards
constexpr int kRtWarps = 9;
constexpr int kRtProducers = 4;
constexpr int kRtThreads = 32 * kRtWarps;
constexpr int kRtABytes = 128 * 128;  // this CTA's 128 expert rows x 64 K, bf16
constexpr int kRtMaxStages = 12;
constexpr int kRtBarBytes = 8 * (2 * kRtMaxStages + 2);
constexpr size_t kRtSmemLimit = 232448;

__device__ bool rt_drain(uint64_t* full, const int* armed, int stages) {
  const uint64_t t0 = globaltimer_ns();
  for (int s = 0; s < stages; ++s) {
    if (armed[s] == 0) continue;
    const uint32_t a = smem_u32(&full[s]);
    const uint32_t parity = static_cast<uint32_t>(armed[s] - 1) & 1u;
    while (!mbar_try_wait(a, parity))
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

template <int SRC, int NV>
__global__ void __launch_bounds__(kRtThreads, 1) router_tc_kernel(const __grid_constant__ RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  if (cluster_nctarank() != 2) {  // launched without its clusters: record and leave
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrLaunchShape);
    return;
  }
  const long long clk0 = clock64();
  const long long ns0 = static_cast<long long>(globaltimer_ns());
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int stage_bytes = kRtABytes + p.b_stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
  uint64_t* empty = full + kRtMaxStages;
  uint64_t* tfull = empty + kRtMaxStages;
  uint64_t* drain = tfull + 1;
  int* misc = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + kRtBarBytes);
  volatile int* abort_flag = misc + 1;
  volatile int* is_last = misc + 2;
  // [N / 2][256] logits of the tokens this CTA selects for, over the ring once it is idle
  float* L = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int item = static_cast<int>(cluster_id_x());
  const int block = item / p.splits, split = item % p.splits;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kblocks, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;
  // Every pair reads the same gate weights; starting each pair's walk over its k-blocks at a
  // different block (and wrapping around) spreads those reads over the L2 slices instead of
  // having all pairs request the same lines at once.  The order is fixed per work item, so
  // the result is reproducible.
  const int kstart = nkb > 0 ? (item * 7) % nkb : 0;
  const int N = p.N, half = N >> 1;
  const int t0 = block * N;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *is_last = 0;
    fence_mbarrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 0) {
    tmem_alloc<2>(reinterpret_cast<uint32_t*>(misc), 256);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);

  bool ok = true;
  const int pid = warp == 0 ? 0 : (warp >= 6 ? warp - 5 : -1);
  if (pid >= 0) {
    // ------------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();   // the gate weights are read by every pair
      const uint64_t pol_x = l2_policy_evict_first();  // a token row is read by S pairs at most
      int armed[kRtMaxStages];
      for (int s = 0; s < kRtMaxStages; ++s) armed[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int ki = 0; ki < nkb; ++ki) {
        const int kb = kb0 + (kstart + ki) % nkb;
        if (stage % kRtProducers != pid) {  // another producer's stage
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, kErrProducerWait)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + (size_t)stage * stage_bytes;
        if (leader) {
          mbar_arrive_expect_tx(&full[stage], 2u * static_cast<uint32_t>(stage_bytes));
          ++armed[stage];
        }
        const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
        tma_load_2d_pair(sA, &p.tmA, fb, kb * 64, rank * 128, pol_w);
        tma_load_2d_pair(sA + kRtABytes, &p.tmB, fb, kb * 64, t0 + rank * half, pol_x);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok && leader && !rt_drain(full, armed, S)) atomicCAS(p.err, 0, kErrDrainWait);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(256, N);
      int stage = 0;
      uint32_t phase = 0;
      for (int ki = 0; ki < nkb; ++ki) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.err, kErrMmaWait)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_k_sw128(smem_u32(smem + (size_t)stage * stage_bytes));
        const uint64_t bd = sdesc_k_sw128(smem_u32(smem + (size_t)stage * stage_bytes + kRtABytes));
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_bf16<2>(tmem_base, ad + 2ull * j, bd + 2ull * j, idesc, (ki > 0 || j > 0) ? 1u : 0u);
        mma_commit<2>(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit<2>(tfull);
      // every MMA this thread issued completes before tensor memory is released
      mma_commit<2>(drain, 1);
      const uint32_t da = smem_u32(drain);
      const uint64_t w0 = globaltimer_ns();
      while (!mbar_try_wait(da, 0u)) {
        if (globaltimer_ns() - w0 > kWaitLimitNs) {
          atomicCAS(p.err, 0, kErrDrainWait);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    // warp w reads tensor-memory lanes 32 (w % 4) .. : experts 128 rank + 32 (w % 4) + lane
    const int q = warp & 3;
    const bool got = mbar_wait(tfull, 0u, abort_flag, p.err, kErrEpilogueWait);
    __syncwarp();
    if (__any_sync(0xFFFFFFFFu, !got || *abort_flag != 0)) {  // one decision for the warp
      ok = false;
    } else {
      tc_fence_after();
      const int el = q * 32 + lane;         // expert within this CTA's 128
      const int e = rank * 128 + el;
      // token i of the block is selected by CTA i / half, at row i % half of its buffer
      const uint32_t Lme = smem_u32(L) + static_cast<uint32_t>(e * 4);
      const uint32_t Lpeer = mapa_shared(Lme, static_cast<uint32_t>(rank ^ 1));
      for (int c = 0; c < (N + 31) >> 5; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 32), v);
        if (p.splits == 1) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int i = c * 32 + j;
            if (i < N) {
              const int owner = i >= half ? 1 : 0;
              const uint32_t off = static_cast<uint32_t>((i - owner * half) * 256 * 4);
              if (owner == rank)
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(Lme + off), "r"(v[j]) : "memory");
              else
                asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(Lpeer + off), "r"(v[j]) : "memory");
            }
          }
        } else if (e < p.E) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int t = t0 + c * 32 + j;
            if (c * 32 + j < N && t < p.T)
              p.partial[((size_t)split * p.T + t) * p.E + e] = __uint_as_float(v[j]);
          }
        }
      }
      tc_fence_before();
    }
  }
  __syncthreads();

  // ------------------------------------------------------------------ selection
  const int ko = p.kc > p.k ? p.kc : p.k;  // outputs per token
  float be[NV];  // this lane's experts' selection bias
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) {
    const int e = lane + 32 * vv;
    be[vv] = p.bias != nullptr && e < p.E ? p.bias[e] : 0.f;
  }
  if (p.splits == 1) {
    cluster_sync();  // every logit of this CTA's tokens is in its shared memory
    if (*abort_flag == 0) {
      for (int il = warp; il < half; il += kRtWarps) {
        const int t = t0 + rank * half + il;
        if (t >= p.T) break;
        float key[NV], val[NV];
        uint32_t taken = 0;
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) {
          const int e = lane + 32 * vv;
          key[vv] = -INFINITY;
          val[vv] = 0.f;
          if (e < p.E) select_key<SRC>(L[il * 256 + e], 0.f, be[vv], key[vv], val[vv]);
          else taken |= 1u << vv;
        }
        select_topk<NV, SRC>(key, val, taken, p.E, p.k, p.G, p.M, p.topk_idx + (size_t)t * ko,
                             p.topk_w + (size_t)t * ko, p.kc);
      }
    }
  } else {
    // the last CTA of the block to arrive sums the partials in split order and selects
    if (*abort_flag == 0) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0)
        *is_last = atomicAdd(&p.counters[block], 1) == 2 * p.splits - 1 ? 1 : 0;
      __syncthreads();
      if (*is_last) {
        __threadfence();
        for (int i = warp; i < N; i += kRtWarps) {
          const int t = t0 + i;
          if (t >= p.T) break;
          // sums in split order; the loads of four splits are in flight together
          float lg[NV];
#pragma unroll
          for (int vv = 0; vv < NV; ++vv) lg[vv] = 0.f;
          for (int s0 = 0; s0 < p.splits; s0 += 4) {
            float part[4][NV];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int vv = 0; vv < NV; ++vv) {
                const int e = lane + 32 * vv;
                part[j][vv] = s0 + j < p.splits && e < p.E
                                  ? __ldcg(p.partial + ((size_t)(s0 + j) * p.T + t) * p.E + e)
                                  : 0.f;
              }
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int vv = 0; vv < NV; ++vv)
                if (s0 + j < p.splits) lg[vv] += part[j][vv];
          }
          float key[NV], val[NV];
          uint32_t taken = 0;
#pragma unroll
          for (int vv = 0; vv < NV; ++vv) {
            const int e = lane + 32 * vv;
            key[vv] = -INFINITY;
            val[vv] = 0.f;
            if (e < p.E) select_key<SRC>(lg[vv], 0.f, be[vv], key[vv], val[vv]);
            else taken |= 1u << vv;
          }
          select_topk<NV, SRC>(key, val, taken, p.E, p.k, p.G, p.M, p.topk_idx + (size_t)t * ko,
                               p.topk_w + (size_t)t * ko, p.kc);
        }
      }
    }
  }

  __syncthreads();
  // no CTA of the pair leaves (or frees tensor memory) while its peer may still read its
  // shared memory or the pair's MMAs may still run
  cluster_sync();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<2>(tmem_base, 256);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) record_clocks(p.err, 0, clk0, ns0);
}

template <int SRC, int NV>
cudaError_t launch_rt(const RouterParams& p, size_t smem, cudaStream_t s) {
  static std::mutex mu;
  static unsigned long long configured = 0;  // bit per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 64 || !((configured >> dev) & 1ull)) {
      err = cudaFuncSetAttribute(router_tc_kernel<SRC, NV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kRtSmemLimit));
      if (err != cudaSuccess) return err;
      if (dev < 64) configured |= 1ull << dev;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * p.blocks * p.splits), 1, 1);
  cfg.blockDim = dim3(kRtThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, router_tc_kernel<SRC, NV>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int SRC>
cudaError_t launch_rt_src(const RouterParams& p, size_t smem, cudaStream_t s) {
  const int nv = (p.E + 31) / 32;
  if (nv <= 1) return launch_rt<SRC, 1>(p, smem, s);
  if (nv <= 2) return launch_rt<SRC, 2>(p, smem, s);
  if (nv <= 4) return launch_rt<SRC, 4>(p, smem, s);
  return launch_rt<SRC, 8>(p, smem, s);
}

}  // namespace

size_t router_tc_smem_bytes(const RouterParams& p) {
  return 1024 + (size_t)p.stages * (kRtABytes + p.b_stage_bytes) + kRtBarBytes + 64;
}

int router_tc_plan(int T, int d, int E, int sms, int max_partial_rows, RouterParams& p) {
  if (E < 1 || E > 256 || d % 64 != 0 || T < 1) return -1;
  const int pairs = sms / 2;
  if (pairs < 1) return -1;
  p.T = T;
  p.E = E;
  p.d = d;
  p.kblocks = d / 64;
  // about one block per pair, 16 to 256 tokens
  int n = 16 * ((T + 16 * pairs - 1) / (16 * pairs));
  p.N = n > 256 ? 256 : n;
  p.blocks = (T + p.N - 1) / p.N;
  // few blocks: split the reduction over d so that about every pair has work, at least four
  // 64-wide k-blocks a split, partials within the workspace's bound
  int splits = 1;
  if (2 * p.blocks <= pairs) {
    splits = pairs / p.blocks;
    if (splits > p.kblocks / 4) splits = p.kblocks / 4;
    while (splits > 1 && (long long)splits * T > max_partial_rows) --splits;
    if (splits < 1) splits = 1;
  }
  p.kb_per_split = (p.kblocks + splits - 1) / splits;
  p.splits = (p.kblocks + p.kb_per_split - 1) / p.kb_per_split;
  p.b_stage_bytes = (p.N / 2) * 128;
  const int stage = kRtABytes + p.b_stage_bytes;
  int stages = static_cast<int>((kRtSmemLimit - 1024 - kRtBarBytes - 64) / stage);
  stages = stages > kRtMaxStages ? kRtMaxStages : stages;
  stages -= stages % kRtProducers;  // each producer owns every fourth stage
  p.stages = stages;
  // the logits buffer [N][128] fp32 reuses the ring
  if (stages < kRtProducers || (size_t)stages * stage < (size_t)p.N * 128 * 4) return -1;
  return 0;
}

cudaError_t launch_router_tc(int score_fn, const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_tc_smem_bytes(p);
  if (smem > kRtSmemLimit) return cudaErrorInvalidConfiguration;
  return score_fn == 0 ? launch_rt_src<0>(p, smem, s) : launch_rt_src<1>(p, smem, s);
}

}  // namespace moe
