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
// offsets and the tile prefixes count the dispatched assignments only.  A negative expert id
// (a slot that rerouting left without an expert) is dispatched nowhere either.
//
// Rerouting at capacity (the same section: overflow tokens are rerouted to their next-best
// expert) runs in rounds over each token's kc candidates (its top-kc experts in selection
// order): in round 0 slot j proposes candidate j; experts accept proposals in token order while
// they have room; each rejected slot takes its token's next unused candidate for the next
// round; a slot whose candidates run out is dropped.  A round is a histogram of the proposals,
// a scan that compares them with each expert's room, a ranking that accepts or rejects each
// proposal and a per-token step to the next candidates: the same stable counting sort as the
// dispatch, so the outcome is deterministic.
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
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = topk_idx[base + i];
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
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

// Per expert e < E: rewrites the chunk histogram chunk_counts[c][e] (c < nchunks) as exclusive
// prefixes over the chunks (token order) and leaves the expert's total in tot_s[e].  The
// block's 1024 threads split into G = 1024 / E' threads per expert (E' = E rounded up to a
// power of two), each over a contiguous run of chunks: the loads of a run are independent of
// one another, and the only serial step is a scan over the G partial sums in shared memory.
// part and tot_s hold 1024 ints each.
__device__ void chunk_scan(int* __restrict__ chunk_counts, int nchunks, int E, int* part, int* tot_s) {
  int ep = 1;
  while (ep < E) ep <<= 1;
  const int G = 1024 / ep;
  const int g = threadIdx.x / ep, e = threadIdx.x % ep;
  const int per = (nchunks + G - 1) / G;
  const int c0 = g * per, c1 = min(nchunks, c0 + per);
  const bool active = e < E && g < G;
  if (active) {
    int sum = 0;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) sum += chunk_counts[(size_t)c * E + e];
    part[g * ep + e] = sum;
  }
  __syncthreads();
  if (active && g == 0) {
    int run = 0;
    for (int x = 0; x < G; ++x) {
      const int v = part[x * ep + e];
      part[x * ep + e] = run;
      run += v;
    }
    tot_s[e] = run;
  }
  __syncthreads();
  if (active) {
    int run = part[g * ep + e];
    for (int c = c0; c < c1; c += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c + j < c1 ? chunk_counts[(size_t)(c + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c + j < c1) {
          chunk_counts[(size_t)(c + j) * E + e] = run;
          run += v[j];
        }
    }
  }
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
  __shared__ int part[1024], tot_s[1024];
  chunk_scan(chunk_counts, nchunks, E, part, tot_s);
  const int e = threadIdx.x;
  int tot = e < E ? tot_s[e] : 0;
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
    const int e0 = i < R ? topk_idx[i] : -1;
    const int e = e0 >= 0 ? e0 : -1 - lane;  // no expert: a key no other lane holds
    const unsigned peers = __match_any_sync(kFull, e);
    if (e0 >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
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
    const int e0 = i < R ? topk_idx[i] : -1;
    const int e = e0 >= 0 ? e0 : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
    if (i < R && e0 < 0) {
      slot_pos[i] = -1;  // a slot without an expert
    } else if (i < R) {
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
    if (e0 >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ rerouting rounds
// prop[i]: candidate index slot i proposes (-1: none, -2: rejected this round); assign_c[i]:
// the accepted candidate index or -1; next_c[t]: the token's next unused candidate.
__global__ void reroute_init_kernel(int T, int k, int E, int* __restrict__ prop,
                                    int* __restrict__ assign_c, int* __restrict__ next_c,
                                    int* __restrict__ fill) {
  const int R = T * k;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x) {
    prop[i] = i % k;
    assign_c[i] = -1;
    if (i % k == 0) next_c[i / k] = k;
    if (i < E) fill[i] = 0;
  }
  if (blockIdx.x == 0)
    for (int e = R + threadIdx.x; e < E; e += blockDim.x) fill[e] = 0;
}

// The expert a slot proposes: its token's candidate prop[i], or -1.
__device__ __forceinline__ int proposed_expert(const int* cand, const int* prop, int i, int k,
                                               int kc) {
  const int c = prop[i];
  return c >= 0 ? cand[(size_t)(i / k) * kc + c] : -1;
}

__global__ void reroute_count_kernel(const int* __restrict__ cand, int kc,
                                     const int* __restrict__ prop, int R, int k, int E,
                                     int* __restrict__ chunk_counts) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kDispatchChunk;
  const int n = min(kDispatchChunk, R - base);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = proposed_expert(cand, prop, base + i, k, kc);
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Per expert: the chunk bases of this round's proposals (in place), the room before the round
// (left) and the slots filled after it.
__global__ void __launch_bounds__(1024) reroute_scan_kernel(int* __restrict__ chunk_counts,
                                                            int nchunks, int E, int capacity,
                                                            int* __restrict__ fill,
                                                            int* __restrict__ left) {
  __shared__ int part[1024], tot_s[1024];
  chunk_scan(chunk_counts, nchunks, E, part, tot_s);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int tot = tot_s[e];
    const int room = capacity - fill[e] > 0 ? capacity - fill[e] : 0;
    left[e] = room;
    fill[e] += tot < room ? tot : room;
  }
}

// A proposal is accepted when its rank among the round's proposals to its expert (token order)
// is below the expert's room.
__global__ void __launch_bounds__(kDispatchWarps * 32) reroute_accept_kernel(
    const int* __restrict__ cand, int kc, int* __restrict__ prop, int R, int k, int E,
    const int* __restrict__ chunk_base, const int* __restrict__ left, int* __restrict__ assign_c) {
  extern __shared__ int wcount[];  // [kDispatchWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) wcount[i] = 0;
  __syncthreads();
  constexpr int kPerWarp = kDispatchChunk / kDispatchWarps;
  const int base = blockIdx.x * kDispatchChunk + warp * kPerWarp;
  int* mine = wcount + warp * E;
  for (int r = 0; r < kPerWarp; r += 32) {
    const int i = base + r + lane;
    const int e0 = i < R ? proposed_expert(cand, prop, i, k, kc) : -1;
    const int e = e0 >= 0 ? e0 : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
    if (e0 >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
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
    const int e0 = i < R ? proposed_expert(cand, prop, i, k, kc) : -1;
    const int e = e0 >= 0 ? e0 : -1 - lane;
    const unsigned peers = __match_any_sync(kFull, e);
    if (e0 >= 0) {
      if (mine[e] + __popc(peers & lt) < left[e]) {
        assign_c[i] = prop[i];
        prop[i] = -1;
      } else {
        prop[i] = -2;
      }
    }
    __syncwarp();
    if (e0 >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
}

// Each rejected slot of a token, in slot order, takes the token's next unused candidate.
__global__ void reroute_advance_kernel(int T, int k, int kc, int* __restrict__ prop,
                                       int* __restrict__ next_c) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    int nc = next_c[t];
    for (int j = 0; j < k; ++j) {
      const size_t i = (size_t)t * k + j;
      if (prop[i] != -2) continue;
      prop[i] = nc < kc ? nc++ : -1;
    }
    next_c[t] = nc;
  }
}

// The serving expert of every slot (-1: dropped) and the gate weights renormalised over the
// serving experts (softmax over their logits, or renormalised sigmoids); one warp per token.
__global__ void reroute_finish_kernel(int T, int k, int kc, int src, const int* __restrict__ cand,
                                      const float* __restrict__ cand_val,
                                      const int* __restrict__ assign_c, int* __restrict__ topk_idx,
                                      float* __restrict__ topk_w, int* __restrict__ dropped) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const int c = lane < k ? assign_c[(size_t)t * k + lane] : -1;
    const bool served = c >= 0;
    const float v = served ? cand_val[(size_t)t * kc + c] : -INFINITY;
    float s;
    if (src == 0) {
      float m = v;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      s = served ? expf(v - m) : 0.f;
    } else {
      s = served ? 1.f / (1.f + expf(-v)) : 0.f;
    }
    float sum = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = served ? cand[(size_t)t * kc + c] : -1;
      topk_w[(size_t)t * k + lane] = served ? s / sum : 0.f;
    }
    const unsigned miss = __ballot_sync(kFull, lane < k && !served);
    if (dropped != nullptr && lane == 0 && miss != 0) atomicAdd(dropped, __popc(miss));
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

cudaError_t launch_reroute(const int* cand, const float* cand_val, int T, int k, int kc, int E,
                           int capacity, int src, int* chunk_counts, int* prop, int* assign_c,
                           int* next_c, int* fill, int* left, int* topk_idx, float* topk_w,
                           int* dropped, cudaStream_t s) {
  const int R = T * k;
  const int nchunks = (R + kDispatchChunk - 1) / kDispatchChunk;
  int blocks = (R + 255) / 256;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (blocks < 1) blocks = 1;
  reroute_init_kernel<<<blocks, 256, 0, s>>>(T, k, E, prop, assign_c, next_c, fill);
  cudaError_t err = cudaGetLastError();
  // round 0 proposes the top-k; each later round at least one more candidate per token that
  // still has a rejected slot, so kc - k + 1 rounds settle every slot
  for (int round = 0; round <= kc - k && err == cudaSuccess; ++round) {
    reroute_count_kernel<<<nchunks, 256, E * sizeof(int), s>>>(cand, kc, prop, R, k, E, chunk_counts);
    reroute_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, nchunks, E, capacity, fill, left);
    reroute_accept_kernel<<<nchunks, kDispatchWarps * 32, kDispatchWarps * E * sizeof(int), s>>>(
        cand, kc, prop, R, k, E, chunk_counts, left, assign_c);
    reroute_advance_kernel<<<(T + 255) / 256, 256, 0, s>>>(T, k, kc, prop, next_c);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  if (dropped != nullptr && (err = cudaMemsetAsync(dropped, 0, sizeof(int), s)) != cudaSuccess) return err;
  int wblocks = (T + 7) / 8;
  if (wblocks > 148 * 32) wblocks = 148 * 32;
  reroute_finish_kernel<<<wblocks, 256, 0, s>>>(T, k, kc, src, cand, cand_val, assign_c, topk_idx,
                                                topk_w, dropped);
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
