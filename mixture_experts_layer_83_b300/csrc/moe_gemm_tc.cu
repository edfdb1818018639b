// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// Computes D = A * B^T per tile, A = 128 weight rows (the MMA's M), B = up to 256 token rows
// (the MMA's N, any multiple of 16), K in 64-element blocks; bf16 operands, fp32 accumulation
// in tensor memory.  Putting the weights on M and the tokens on N ("swap AB") lets a tile
// follow an expert's token count with 16-row granularity, so a ragged expert segment wastes
// at most 15 rows -- the same kernel serves 256-row prefill segments and 4-row decode
// segments.  The experts run as one grouped GEMM over the expert segments (page "Tensor vs
// Expert vs Data Parallelism for MoE Serving", Figure 2: experts run grouped GEMMs).
//
// Roles (224 threads, one CTA per SM, persistent over a static tile stride):
//   warp 0 lane 0   weight producer: TMA of the 128 x 64 weight block of each k-step into
//                   the weight ring (16 KiB stages, up to 12 deep): weights come from HBM
//                   and need the longest look-ahead
//   warp 6 lane 0   token producer: TMA of the N x 64 token block into the token ring (a few
//                   stages: token tiles are L2 hits, re-read by every weight tile)
//   warp 1 lane 0   MMA issuer: 4 x tcgen05.mma (K=16) per k-step into one of two TMEM
//                   accumulators (256 columns each); commits release ring stages and hand
//                   finished accumulators to the epilogue
//   warps 2..5      epilogue: tcgen05.ld, then per mode
//                     router : fp32 logits [T][E]
//                     gate/up: rows 0..63 of A are gate rows, 64..127 the matching up rows;
//                              both are staged token-major in shared memory, then each thread
//                              forms h = silu(gate) * up for 8 features of one token and
//                              stores them as one 16-byte bf16 vector
//                     down   : y staged token-major (bf16), stored as full 16-byte rows
// The tile scheduler reads the segment offsets and the n-tile prefix the dispatch scan wrote,
// so nothing crosses to the host.  Tile order within a segment is (m-group, m, n-tile), so the
// CTAs running at the same time share weight tiles (all n-tiles of an m) and token tiles (a
// group of m) through L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace moe {
namespace {

constexpr int kThreads = 224;
constexpr int kMaxStagesA = 12;
constexpr int kMaxStagesB = 4;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;
constexpr int kABytes = 128 * 128;       // weight stage: 128 rows x 64 bf16
constexpr int kStageLdF = 68;            // fp32 row of the gate/up staging (64 + pad)
constexpr int kStageLdH = 136;           // bf16 row of the down staging (128 + pad)
constexpr int kXchgFloats = 2 * 16 * kStageLdF;  // 8704 B, also holds 32 x kStageLdH bf16
static_assert(32 * kStageLdH * 2 <= kXchgFloats * 4, "down staging fits the epilogue buffer");
constexpr int kBarBytes = 512;           // 2 * (12 + 4) + 5 mbarriers, rounded
constexpr int kMiscBytes = 128;
constexpr size_t kSmemLimit = 232448;    // 227 KiB opt-in per CTA
constexpr size_t kSmemFloor = 120 * 1024;  // keeps a second CTA (and TMEM demand) off the SM

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// Wait for every load a producer armed on its ring (used when unwinding after an abort).
__device__ void drain_ring(uint64_t* full, const int* armed, int stages, int* err) {
  for (int s = 0; s < stages; ++s)
    if (armed[s] > 0 && !drain_wait(&full[s], static_cast<uint32_t>(armed[s] - 1) & 1u))
      atomicCAS(err, 0, kErrDrainWait);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int SA = p.stages_a, SB = p.stages_b;
  uint8_t* ring_a = smem;
  uint8_t* ring_b = smem + (size_t)SA * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring_b + (size_t)SB * p.b_stage_bytes);
  uint64_t* full_a = bars;
  uint64_t* empty_a = full_a + kMaxStagesA;
  uint64_t* full_b = empty_a + kMaxStagesA;
  uint64_t* empty_b = full_b + kMaxStagesB;
  uint64_t* tfull = empty_b + kMaxStagesB;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  int* misc = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);
  volatile int* abort_flag = misc + 1;
  float* xchg = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(misc) + kMiscBytes);
  int* s_seg = reinterpret_cast<int*>(xchg + kXchgFloats);
  const int n_seg0 = p.prob[0].seg_off != nullptr ? p.prob[0].n_seg : 0;
  int* s_ntp = s_seg + (n_seg0 + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < p.n_prob; ++i) {
      tma_prefetch_desc(&p.prob[i].tmA);
      for (int b = 0; b < 4; ++b) tma_prefetch_desc(&p.prob[i].tmB[b]);
    }
  }
  if (warp == 0) {
    tmem_alloc(reinterpret_cast<uint32_t*>(misc), kTmemCols);
    tmem_relinquish();
  }
  if (n_seg0 > 0) {
    for (int i = threadIdx.x; i <= n_seg0; i += kThreads) {
      s_seg[i] = p.prob[0].seg_off[i];
      s_ntp[i] = p.prob[0].ntp[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);

  const int tiles0 = (n_seg0 > 0 ? s_ntp[n_seg0] : p.prob[0].nt) * p.prob[0].m_tiles;
  const int tiles1 = p.n_prob > 1 ? p.prob[1].nt * p.prob[1].m_tiles : 0;
  const int total = tiles0 + tiles1;

  if (warp == 0) {
    // ---------------------------------------------------------------- weight producer
    if (lane == 0) {
      // weights read by one tile only stream through L2 (evict first); weights a neighbouring
      // n-tile reads again stay at normal priority
      const uint64_t pol_once = l2_policy_evict_first();
      const uint64_t pol_shared = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int armed[kMaxStagesA];
      for (int s = 0; s < kMaxStagesA; ++s) armed[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const int arow = tl.seg * P.a_seg_stride + tl.m * P.a_m_stride;
        const bool box1 = tile_has_box1(P, tl);
        const uint64_t pol = tl.nt > 1 ? pol_shared : pol_once;
        const uint32_t bytes = static_cast<uint32_t>((box1 ? 2 : 1) * P.a_box_rows * 128);
        const int kblocks = P.K >> 6;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_a[stage], phase ^ 1u, abort_flag, p.err, kErrProducerWait)) {
            ok = false;
            break;
          }
          uint8_t* sA = ring_a + (size_t)stage * kABytes;
          mbar_arrive_expect_tx(&full_a[stage], bytes);
          ++armed[stage];
          tma_load_2d(sA, &P.tmA, &full_a[stage], kb * 64, arow, pol);
          if (box1) tma_load_2d(sA + 64 * 128, &P.tmA, &full_a[stage], kb * 64, arow + P.a_box1_off, pol);
          if (++stage == SA) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) drain_ring(full_a, armed, SA, p.err);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ---------------------------------------------------------------- token producer
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_last();  // re-read by every weight tile
      int stage = 0;
      uint32_t phase = 0;
      int armed[kMaxStagesB];
      for (int s = 0; s < kMaxStagesB; ++s) armed[s] = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const uint32_t bytes = static_cast<uint32_t>(tl.ncols * 128);
        const int kblocks = P.K >> 6;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_b[stage], phase ^ 1u, abort_flag, p.err, kErrProducerWait)) {
            ok = false;
            break;
          }
          uint8_t* sB = ring_b + (size_t)stage * p.b_stage_bytes;
          mbar_arrive_expect_tx(&full_b[stage], bytes);
          ++armed[stage];
          const int kx = kb * 64;
          int off = 0, rem = tl.ncols;
          while (rem >= 128) {
            tma_load_2d(sB + off * 128, &P.tmB[0], &full_b[stage], kx, tl.row0 + off, pol_x);
            off += 128;
            rem -= 128;
          }
          if (rem & 64) {
            tma_load_2d(sB + off * 128, &P.tmB[1], &full_b[stage], kx, tl.row0 + off, pol_x);
            off += 64;
          }
          if (rem & 32) {
            tma_load_2d(sB + off * 128, &P.tmB[2], &full_b[stage], kx, tl.row0 + off, pol_x);
            off += 32;
          }
          if (rem & 16) tma_load_2d(sB + off * 128, &P.tmB[3], &full_b[stage], kx, tl.row0 + off, pol_x);
          if (++stage == SB) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) drain_ring(full_b, armed, SB, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      int acc_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const int buf = acc_i & 1;
        const uint32_t use = static_cast<uint32_t>(acc_i >> 1);
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p.err, kErrMmaWait)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kAccCols);
        const uint32_t idesc = idesc_bf16_f32(128, tl.ncols);
        const int kblocks = P.K >> 6;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full_a[sa], pa, abort_flag, p.err, kErrMmaWait) ||
              !mbar_wait(&full_b[sb], pb, abort_flag, p.err, kErrMmaWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k_sw128(smem_u32(ring_a + (size_t)sa * kABytes));
          const uint64_t bd = sdesc_k_sw128(smem_u32(ring_b + (size_t)sb * p.b_stage_bytes));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16(d_tmem, ad + 2ull * j, bd + 2ull * j, idesc, (kb | j) != 0 ? 1u : 0u);
          mma_commit(&empty_a[sa]);
          mma_commit(&empty_b[sb]);
          if (++sa == SA) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sb == SB) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[buf]);
        ++acc_i;
      }
      // every MMA this thread issued completes before tensor memory is released
      mma_commit(drain);
      if (!drain_wait(drain, 0)) atomicCAS(p.err, 0, kErrDrainWait);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    int acc_i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile tl;
      decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
      const TcProblem& P = p.prob[tl.prob];
      const int buf = acc_i & 1;
      const uint32_t use = static_cast<uint32_t>(acc_i >> 1);
      const bool ok = mbar_wait(&tfull[buf], use & 1u, abort_flag, p.err, kErrEpilogueWait);
      __syncwarp();
      if (named_bar_or(1, 128, !ok || *abort_flag != 0)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * kAccCols);
      const int nchunks = (tl.valid + 31) >> 5;
      const int ep = threadIdx.x - 64;  // 0..127 across the four epilogue warps
      if (MODE == kModeGateUp) {
        // Rows 0..63 of the accumulator are gate features, 64..127 the matching up features.
        // Per 16 tokens: every warp stages its 32 features x 16 tokens (fp32) token-major in
        // shared memory, then each thread computes 8 consecutive h features of one token and
        // stores them as one 16-byte vector (a warp writes four full 128-byte h rows).
        float* gs = xchg;                // [16 tokens][kStageLdF] gate
        float* us = xchg + 16 * kStageLdF;  // [16 tokens][kStageLdF] up
        float* mine = q < 2 ? gs : us;
        const int fl = (q & 1) * 32 + lane;  // this lane's feature within the tile's 64
        const int tt = ep >> 3, fg = ep & 7;
        __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(P.out);
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c * 32), v);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int col0 = c * 32 + half * 16;
            if (col0 >= tl.valid) break;  // uniform over the 128 epilogue threads
#pragma unroll
            for (int j = 0; j < 16; ++j) mine[j * kStageLdF + fl] = __uint_as_float(v[half * 16 + j]);
            named_bar_sync(2, 128);
            const int col = col0 + tt;
            if (col < tl.valid) {
              const float4* g4 = reinterpret_cast<const float4*>(gs + tt * kStageLdF + fg * 8);
              const float4* u4 = reinterpret_cast<const float4*>(us + tt * kStageLdF + fg * 8);
              const float4 ga = g4[0], gb = g4[1], ua = u4[0], ub = u4[1];
              const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
              const float u[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
              uint4 o;
              __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float h0 = __fdividef(g[2 * i] * u[2 * i], 1.f + __expf(-g[2 * i]));
                const float h1 =
                    __fdividef(g[2 * i + 1] * u[2 * i + 1], 1.f + __expf(-g[2 * i + 1]));
                oh[i] = __floats2bfloat162_rn(h0, h1);
              }
              *reinterpret_cast<uint4*>(hout + (size_t)(P.out_row_base + tl.row0 + col) * P.out_ld +
                                        tl.m * 64 + fg * 8) = o;
            }
            named_bar_sync(2, 128);
          }
        }
      } else if (MODE == kModeDown) {
        // Per 32 tokens: each lane writes its channel's 32 values (bf16) token-major into
        // shared memory; then the 128 threads store full 256-byte y rows in 16-byte vectors.
        __nv_bfloat16* ys = reinterpret_cast<__nv_bfloat16*>(xchg);  // [32][kStageLdH]
        const int chl = q * 32 + lane;
        __nv_bfloat16* yout = static_cast<__nv_bfloat16*>(P.out);
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j) ys[j * kStageLdH + chl] = __float2bfloat16_rn(__uint_as_float(v[j]));
          named_bar_sync(2, 128);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = i * 128 + ep;
            const int tok = idx >> 4, part = idx & 15;
            const int col = c * 32 + tok;
            const int ch0 = tl.m * 128 + part * 8;
            if (col < tl.valid && ch0 < P.out_valid_m)
              *reinterpret_cast<uint4*>(yout + (size_t)(P.out_row_base + tl.row0 + col) * P.out_ld +
                                        ch0) =
                  *reinterpret_cast<const uint4*>(ys + tok * kStageLdH + part * 8);
          }
          named_bar_sync(2, 128);
        }
      } else {
        const int e = tl.m * 128 + q * 32 + lane;
        const bool e_ok = e < P.out_valid_m;
        float* lout = static_cast<float*>(P.out);
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = c * 32 + j;
            if (e_ok && col < tl.valid)
              lout[(size_t)(tl.row0 + col) * P.out_ld + e] = __uint_as_float(v[j]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
      ++acc_i;
    }
  }

  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t fixed_smem_bytes(int n_seg) {
  return 1024 + kBarBytes + kMiscBytes + sizeof(float) * kXchgFloats +
         2 * sizeof(int) * (size_t)(n_seg + 1);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

template <int MODE>
cudaError_t launch_mode(const TcParams& p, int grid, size_t smem, cudaStream_t s) {
  static std::mutex mu;
  static unsigned configured = 0;  // bit per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 32 && !((configured >> dev) & 1u)) {
      err = cudaFuncSetAttribute(gemm_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
      if (err != cudaSuccess) return err;
      configured |= 1u << dev;
    } else if (dev >= 32) {
      err = cudaFuncSetAttribute(gemm_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLimit));
      if (err != cudaSuccess) return err;
    }
  }
  gemm_tc_kernel<MODE><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Ring depths for an n-tile cap: the token ring holds a few stages (its loads hit L2), the
// weight ring takes the rest of shared memory (its loads come from HBM).
void gemm_tc_plan(int bn, int n_seg, TcParams& p) {
  p.b_stage_bytes = bn * 128;
  p.stages_b = bn >= 128 ? 3 : 4;
  const size_t avail = kSmemLimit - fixed_smem_bytes(n_seg) - (size_t)p.stages_b * p.b_stage_bytes;
  int sa = static_cast<int>(avail / kABytes);
  p.stages_a = sa > kMaxStagesA ? kMaxStagesA : sa;
}

size_t gemm_tc_smem_bytes(const TcParams& p) {
  const int n_seg = p.prob[0].seg_off != nullptr ? p.prob[0].n_seg : 0;
  size_t b = fixed_smem_bytes(n_seg) + (size_t)p.stages_a * kABytes +
             (size_t)p.stages_b * p.b_stage_bytes;
  return b < kSmemFloor ? kSmemFloor : b;
}

int encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return -1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

cudaError_t launch_gemm_tc(int mode, const TcParams& p, int grid, cudaStream_t s) {
  const size_t smem = gemm_tc_smem_bytes(p);
  if (smem > kSmemLimit || p.stages_a < 2 || p.stages_b < 2 || p.stages_a > kMaxStagesA ||
      p.stages_b > kMaxStagesB)
    return cudaErrorInvalidConfiguration;
  switch (mode) {
    case kModeRouter: return launch_mode<kModeRouter>(p, grid, smem, s);
    case kModeGateUp: return launch_mode<kModeGateUp>(p, grid, smem, s);
    default: return launch_mode<kModeDown>(p, grid, smem, s);
  }
}

}  // namespace moe
