// Dispatch: group the T*k (token, slot) assignments by expert with token order kept inside
// each expert -- the one-GPU form of the dispatch all-to-all (page "Expert-Parallel MoE
// Inference: Serving Sparse Models at Scale", section "The all-to-all dispatch and combine,
// step by step"; page "MoE Expert Parallelism in Practice", "Core Principles" part 1).
//
// A deterministic stable counting sort, no atomic return value is ever used as a position:
//   1. dispatch_count: per chunk of kDispatchChunk assignments, a shared-memory histogram.
//   2. dispatch_scan (one block): per expert, exclusive scan over chunks; expert_counts;
//      offsets = exclusive scan over experts; the n-tile prefix the grouped GEMM schedules by.
//   3. dispatch_scatter: per chunk, per warp: counts of each expert by warp (match_any), a scan
//      over the warps, then position = offsets[e] + chunk base + warp base + rank among the
//      earlier equal lanes.  Assignment i = t*k + j, so the order is token order.
//   4. gather: xs[p] = x[sorted_token[p]], one warp per row, 16-byte vectors.
// With an expert capacity (page "Expert-Parallel MoE Inference", section "Capacity factor and
// token dropping"), an assignment whose rank among its expert's assignments (token order) is
// capacity or more is dropped: slot_pos = -1, no row in the permutation; expert_counts,
// offsets and the tile prefixes count the dispatched assignments only.
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "tile_sched.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__global__ void dispatch_count_kernel(const int* __restrict__ topk_idx, int R, int E,
                                      int* __restrict__ chunk_counts) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kDispatchChunk;
  const int n = min(kDispatchChunk, R - base);
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&hist[topk_idx[base + i]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Inclusive block scan of one value per thread (blockDim.x == 1024).
__device__ int block_inclusive_scan(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, w, off);
      if (lane >= off) w += o;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  const int add = warp > 0 ? scratch[warp - 1] : 0;
  __syncthreads();
  return v + add;
}

// ntp / ntp2: prefixes of the tile units per expert (seg_units) for n-tile caps bn / bn2 and
// tall-tile limits tall / tall2 (the two grouped GEMMs may tile the token rows differently);
// either may be null.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int* __restrict__ chunk_counts,
                                                             int nchunks, int E, int bn, int tall,
                                                             int* __restrict__ expert_counts,
                                                             int* __restrict__ offsets,
                                                             int* __restrict__ ntp, int bn2,
                                                             int tall2, int* __restrict__ ntp2,
                                                             int capacity, int* __restrict__ dropped) {
  __shared__ int scratch[32];
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      const size_t o = (size_t)c * E + e;
      const int v = chunk_counts[o];
      chunk_counts[o] = tot;
      tot += v;
    }
  }
  const int routed = tot;
  tot = tot < capacity ? tot : capacity;  // dispatched assignments
  const int nt = seg_units(tot, bn, tall);
  const int nt2 = bn2 > 0 ? seg_units(tot, bn2, tall2) : 0;
  const int inc_rows = block_inclusive_scan(tot, scratch);
  const int inc_nt = block_inclusive_scan(nt, scratch);
  const int inc_nt2 = block_inclusive_scan(nt2, scratch);
  const int inc_drop = block_inclusive_scan(routed - tot, scratch);
  if (dropped != nullptr && e == 1023) *dropped = inc_drop;
  if (e < E) {
    expert_counts[e] = tot;
    offsets[e] = inc_rows - tot;
    if (ntp) ntp[e] = inc_nt - nt;
    if (ntp2) ntp2[e] = inc_nt2 - nt2;
    if (e == E - 1) {
      offsets[E] = inc_rows;
      if (ntp) ntp[E] = inc_nt;
      if (ntp2) ntp2[E] = inc_nt2;
    }
  }
}

__global__ void __launch_bounds__(kDispatchWarps * 32) dispatch_scatter_kernel(
    const int* __restrict__ topk_idx, int R, int E, int k, const int* __restrict__ chunk_base,
    const int* __restrict__ offsets, int capacity, int* __restrict__ sorted_token,
    int* __restrict__ slot_pos) {
  extern __shared__ int wcount[];  // [kDispatchWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) wcount[i] = 0;
  __syncthreads();
  constexpr int kPerWarp = kDispatchChunk / kDispatchWarps;
  const int base = blockIdx.x * kDispatchChunk + warp * kPerWarp;
  int* mine = wcount + warp * E;
  for (int r = 0; r < kPerWarp; r += 32) {
    const int i = base + r + lane;
    const int e = i < R ? topk_idx[i] : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
    if (i < R && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per expert and warp: the rank (token order) of the warp's first assignment of the expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kDispatchWarps; ++w) {
      const int c = wcount[w * E + e];
      wcount[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int r = 0; r < kPerWarp; r += 32) {
    const int i = base + r + lane;
    const int e = i < R ? topk_idx[i] : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
    if (i < R) {
      const int rank = mine[e] + __popc(peers & lt);
      if (rank < capacity) {
        const int pos = offsets[e] + rank;
        slot_pos[i] = pos;
        sorted_token[pos] = i / k;
      } else {
        slot_pos[i] = -1;  // dropped at the expert's capacity
      }
    }
    __syncwarp();
    if (i < R && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per destination row; 16-byte vectors, four loads in flight per lane per step.  The
// row count is *rows_dev when given (rows dispatched under a capacity), else R.
__global__ void gather_rows_v16_kernel(const uint4* __restrict__ x, const int* __restrict__ sorted_token,
                                       int R, const int* __restrict__ rows_dev, int row_vecs,
                                       uint4* __restrict__ xs) {
  if (rows_dev != nullptr) R = *rows_dev;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int p = gw; p < R; p += nw) {
    const uint4* src = x + (size_t)sorted_token[p] * row_vecs;
    uint4* dst = xs + (size_t)p * row_vecs;
    int v = lane;
    for (; v + 96 < row_vecs; v += 128) {
      const uint4 a0 = __ldg(src + v), a1 = __ldg(src + v + 32), a2 = __ldg(src + v + 64),
                  a3 = __ldg(src + v + 96);
      dst[v] = a0;
      dst[v + 32] = a1;
      dst[v + 64] = a2;
      dst[v + 96] = a3;
    }
    for (; v < row_vecs; v += 32) dst[v] = __ldg(src + v);
  }
}

__global__ void gather_rows_w4_kernel(const uint32_t* __restrict__ x, const int* __restrict__ sorted_token,
                                      int R, const int* __restrict__ rows_dev, int row_words,
                                      uint32_t* __restrict__ xs) {
  if (rows_dev != nullptr) R = *rows_dev;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int p = gw; p < R; p += nw) {
    const uint32_t* src = x + (size_t)sorted_token[p] * row_words;
    uint32_t* dst = xs + (size_t)p * row_words;
    for (int v = lane; v < row_words; v += 32) dst[v] = src[v];
  }
}

}  // namespace

cudaError_t launch_dispatch(const int* topk_idx, int T, int k, int E, int bn, int tall,
                            int* chunk_counts, int* expert_counts, int* offsets, int* ntp, int bn2,
                            int tall2,
                            int* ntp2, int capacity, int* dropped, int* sorted_token,
                            int* slot_pos, cudaStream_t s) {
  const int R = T * k;
  const int nchunks = (R + kDispatchChunk - 1) / kDispatchChunk;
  dispatch_count_kernel<<<nchunks, 256, E * sizeof(int), s>>>(topk_idx, R, E, chunk_counts);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  dispatch_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, nchunks, E, bn, tall, expert_counts, offsets, ntp,
                                          bn2, tall2, ntp2, capacity, dropped);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  dispatch_scatter_kernel<<<nchunks, kDispatchWarps * 32, kDispatchWarps * E * sizeof(int), s>>>(
      topk_idx, R, E, k, chunk_counts, offsets, capacity, sorted_token, slot_pos);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, const int* sorted_token, int R, const int* rows_dev,
                          int d, int elt_bytes, void* xs, cudaStream_t s) {
  const size_t row_bytes = (size_t)d * elt_bytes;
  const int threads = 256;
  int blocks = (R + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (row_bytes % 16 == 0)
    gather_rows_v16_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint4*>(x), sorted_token, R,
                                                      rows_dev, (int)(row_bytes / 16),
                                                      static_cast<uint4*>(xs));
  else
    gather_rows_w4_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint32_t*>(x), sorted_token, R,
                                                     rows_dev, (int)(row_bytes / 4),
                                                     static_cast<uint32_t*>(xs));
  return cudaGetLastError();
}

}  // namespace moe
