// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// Computes D = A * B^T per tile, A = weight rows (the MMA's M), B = token rows (the MMA's N,
// any multiple of 16 up to 256 per MMA; a wide tile runs two MMAs over up to 512), K in
// 64-element blocks; bf16 operands, fp32 accumulation in tensor memory.  Putting the weights on M and the tokens on N ("swap AB") lets a tile follow
// an expert's token count with 16-row granularity, so a ragged expert segment wastes at most
// 15 rows -- the same kernel serves 256-row prefill segments and 4-row decode segments.  The
// experts run as one grouped GEMM over the expert segments (page "Tensor vs Expert vs Data
// Parallelism for MoE Serving", Figure 2: experts run grouped GEMMs).
//
// Two forms, chosen by the template argument CG:
//   CG = 1  one CTA per tile: M = 128 weight rows, the CTA holds all N token rows.
//   CG = 2  a CTA pair (a 2-CTA cluster on the two SMs of a TPC, tcgen05 cta_group::2) per
//           tile: M = 256 weight rows, each CTA holds its own 128 weight rows and half of the
//           N token rows, and each CTA's tensor memory receives its 128 rows x N.  Per SM
//           this moves a third less operand data per FLOP (16 KB of weights + N/2 x 128 B of
//           tokens per k-block instead of 16 KB + N x 128 B), which is what the expert GEMMs
//           of a prefill batch are limited by.  Both CTAs' TMA loads count their bytes on the
//           even CTA's barriers; its MMA issuer runs the pair and its commits arrive on both
//           CTAs' barriers (multicast).
//
// Roles (persistent over a static tile stride; warps 0..6, plus warps 7..11 for a wide pair,
// plus extra producer warps for the pair forms; warp 7 of a wide pair is the second MMA
// issuer and warps 8..11 the second epilogue group, each owning one accumulator half):
//   warp 0 lane 0   weight producer: TMA of the 128 x 64 weight block of each k-step into
//                   the weight ring (16 KiB stages, up to 12 deep): weights come from HBM
//                   and need the longest look-ahead
//   warp 6 lane 0   token producer: TMA of this CTA's N (or N/2) x 64 token block into the
//                   token ring (token tiles are L2 hits, re-read by every weight tile)
//   warp 1 lane 0   MMA issuer (even CTA of a pair only): 4 x tcgen05.mma (K=16) per k-step
//                   into a TMEM accumulator (two 256-column buffers for the one-CTA form, one
//                   per pair otherwise); commits release ring stages and hand finished
//                   accumulators to the epilogues.  The two issuers of a wide pair share
//                   each token stage; they share the weight stage of a wide tile, while on a
//                   tall tile each reads, waits for and releases a weight stage of its own
//   warps 2..5      epilogue: tcgen05.ld, then per mode
//                     router : fp32 logits [T][E]
//                     gate/up: rows 0..63 of the CTA's A are gate rows, 64..127 the matching
//                              up rows; both are staged token-major in shared memory, then
//                              each thread forms h = silu(gate) * up for 8 features of one
//                              token and stores them as one 16-byte bf16 vector
//                     down   : y (bf16) stored from registers, a warp's 32 channels of one
//                              token per store
// The tile scheduler reads the segment offsets and the n-tile prefix the dispatch scan wrote,
// so nothing crosses to the host.  Tile order within a segment is (m-group, m, n-tile), so the
// CTAs running at the same time share weight tiles (all n-tiles of an m) and token tiles (a
// group of m) through L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace moe {
namespace {

constexpr int kMaxStagesA = 12;
constexpr int kMaxStagesB = 8;
constexpr int kAccCols = 256;  // one accumulator: 128 lanes x up to 256 fp32 columns
// Three forms share this kernel:
//   one CTA (CG = 1, router): one CTA per SM, accumulator double-buffered in 512 TMEM columns.
//   narrow pair (CG = 2, both expert GEMMs at decode-sized segments, n-tile cap under 256
//     rows): two pairs per TPC (two CTAs per SM), one 256-column accumulator each; the second
//     pair keeps the tensor cores busy while the first drains its accumulator, and two MMA
//     issuers per SM halve the per-instruction issue cost (about 125 cycles per tcgen05.mma
//     from one thread) that otherwise bounds MMAs with N < 256.
//   wide pair (CG = 2, WIDE, both expert GEMMs at prefill-sized segments): one pair per TPC,
//     n-tiles of up to 512 token rows in one 512-column accumulator, split over two MMA
//     issuers (one per 256-column half) and two epilogue groups.  An expert's whole token
//     segment (up to 512 rows) shares one pass over its weights, so each weight tile is
//     streamed from HBM once.  A segment of at most 256 rows runs as a tall tile instead: two
//     scheduled m-tiles over all of its rows, each issuer and epilogue group taking one m-tile,
//     so both issuers still run MMAs with N = the segment's rows.
// Producer threads per ring.  One thread's TMA issue bounds the stream it keeps in flight, so
// the pair forms spread each ring over several producer warps.  Producer pid owns the ring
// stages s with s % producers == pid and fills their rounds in order: every stage keeps a
// single producer, so a producer can never be two rounds ahead on a stage (where the parity
// of an mbarrier wait would no longer tell the rounds apart).  Ring depths are multiples of
// the producer counts.
template <int CG, int WIDE> constexpr int producers_a() { return CG == 2 ? 2 : 1; }
template <int CG, int WIDE> constexpr int producers_b() { return WIDE ? 4 : (CG == 2 ? 2 : 1); }
// The gate/up GEMM gathers its token rows itself (the fused dispatch): its token producers
// load the rows of x that the dispatch permutation names with TMA tile::gather4 (four rows
// per instruction), so no permuted copy of x is ever written.
template <int MODE> constexpr bool gathers() { return MODE == kModeGateUp; }
// Warps 0..6 (0..11 for a wide pair) have fixed roles; the extra producers follow them.
template <int WIDE> constexpr int base_warps() { return WIDE ? 12 : 7; }
template <int MODE, int CG, int WIDE> constexpr int warps_of() {
  return base_warps<WIDE>() + producers_a<CG, WIDE>() - 1 + producers_b<CG, WIDE>() - 1;
}
template <int MODE, int CG, int WIDE> constexpr int threads_of() {
  return 32 * warps_of<MODE, CG, WIDE>();
}
template <int CG, int WIDE> constexpr int acc_bufs() { return CG == 1 ? 2 : 1; }
template <int CG, int WIDE> constexpr uint32_t tmem_cols() { return CG == 2 && !WIDE ? 256u : 512u; }
template <int CG, int WIDE> constexpr int ctas_per_sm() { return CG == 2 && !WIDE ? 2 : 1; }

// Token columns of the two MMAs of a wide tile: n0 = the first half rounded up to 16 rows
// (all of a tile that fits one accumulator half), n1 = the rest.
struct NSplit {
  int n0, n1;
};
template <int WIDE>
__device__ __forceinline__ NSplit n_split(int ncols) {
  if (!WIDE || ncols <= kAccCols) return NSplit{ncols, 0};
  const int n0 = (((ncols >> 4) + 1) >> 1) << 4;
  return NSplit{n0, ncols - n0};
}
constexpr int kABytes = 128 * 128;       // weight stage: 128 rows x 64 bf16
constexpr int kStageLdF = 68;            // fp32 row of the gate/up staging (64 + pad)
constexpr int kXchgFloats = 2 * 16 * kStageLdF;  // 8704 B: gate and up, 16 tokens each
constexpr int kBarBytes = 512;           // 2 * (12 + 8) + 6 mbarriers, rounded
static_assert(8 * (2 * (kMaxStagesA + kMaxStagesB) + 6) <= kBarBytes, "mbarriers fit");
constexpr int kMiscBytes = 128;
constexpr size_t kSmemLimit = 232448;    // 227 KiB opt-in per CTA
constexpr size_t kSmemLimitPair = 112 * 1024;  // two per SM with room to spare in its 228 KiB
constexpr size_t kSmemFloor = 120 * 1024;  // keeps a second one-CTA kernel (and its TMEM demand) off the SM
size_t smem_limit(int cg, int wide) { return cg == 2 && !wide ? kSmemLimitPair : kSmemLimit; }

// One lane's output channel for up to 32 tokens (rows ld apart), fp32 accumulators to bf16.
__device__ __forceinline__ void store_down_chunk(__nv_bfloat16* y, int ld, int n, const uint32_t (&v)[32]) {
  if (n >= 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) y[(size_t)j * ld] = __float2bfloat16_rn(__uint_as_float(v[j]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) y[(size_t)j * ld] = __float2bfloat16_rn(__uint_as_float(v[j]));
  }
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// Wait for every load a producer armed on its ring (used when unwinding after an abort).  One
// wall-clock limit covers the whole ring.
__device__ void drain_ring(uint64_t* full, const int* armed, int stages, int* err) {
  const uint64_t t0 = globaltimer_ns();
  for (int s = 0; s < stages; ++s) {
    if (armed[s] == 0) continue;
    const uint32_t a = smem_u32(&full[s]);
    const uint32_t parity = static_cast<uint32_t>(armed[s] - 1) & 1u;
    while (!mbar_try_wait(a, parity)) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(err, 0, kErrDrainWait);
        return;
      }
    }
  }
}

template <int MODE, int CG, int WIDE>
__global__ void __launch_bounds__(threads_of<MODE, CG, WIDE>(), ctas_per_sm<CG, WIDE>())
    gemm_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  if constexpr (CG == 2) {
    // a pair kernel launched without 2-CTA clusters: record it and leave before any shared
    // state exists (the condition is uniform over the grid)
    if (cluster_nctarank() != 2) {
      if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrLaunchShape);
      return;
    }
  }
  const long long clk0 = clock64();
  const long long ns0 = static_cast<long long>(globaltimer_ns());
  // the gate/up GEMM gathers its token rows unless the host staged them in a permuted copy
  const bool gather = gathers<MODE>() && p.gather != 0;
  constexpr int kGroups = WIDE ? 2 : 1;           // epilogue groups of four warps
  constexpr int kIssuers = WIDE ? 2 : 1;          // MMA issuing threads
  constexpr int kBufs = acc_bufs<CG, WIDE>();
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
  uint64_t* drain = tempty + 2;  // one per issuer
  int* misc = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);
  volatile int* abort_flag = misc + 1;
  float* xchg0 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(misc) + kMiscBytes);
  int* s_seg = reinterpret_cast<int*>(xchg0 + kGroups * kXchgFloats);
  const int n_seg0 = p.prob[0].seg_off != nullptr ? p.prob[0].n_seg : 0;
  int* s_ntp = s_seg + (n_seg0 + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rank within the pair (the even CTA issues the MMAs) and this CTA's stream of tiles
  const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int unit0 = CG == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int nunits = CG == 2 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    // every ring stage and accumulator is released by each MMA issuer once
    for (int s = 0; s < SA; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&empty_a[s], kIssuers);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], kIssuers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], kIssuers);
      mbar_init(&tempty[b], 4 * kGroups * CG);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < p.n_prob; ++i) {
      tma_prefetch_desc(&p.prob[i].tmA);
      for (int b = 0; b < (gather ? 1 : 5); ++b) tma_prefetch_desc(&p.prob[i].tmB[b]);
    }
  }
  if (warp == 0) {
    tmem_alloc<CG>(reinterpret_cast<uint32_t*>(misc), tmem_cols<CG, WIDE>());
    tmem_relinquish<CG>();
  }
  if (n_seg0 > 0) {
    for (int i = threadIdx.x; i <= n_seg0; i += threads_of<MODE, CG, WIDE>()) {
      s_seg[i] = p.prob[0].seg_off[i];
      s_ntp[i] = p.prob[0].ntp[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before any remote arrival or TMA completion
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);

  const int tiles0 = n_seg0 > 0 ? s_ntp[n_seg0] * tiles_per_unit(p.prob[0])
                                : p.prob[0].nt * p.prob[0].m_tiles;
  const int tiles1 = p.n_prob > 1 ? p.prob[1].nt * p.prob[1].m_tiles : 0;
  const int total = tiles0 + tiles1;

  constexpr int kProdA = producers_a<CG, WIDE>(), kProdB = producers_b<CG, WIDE>();
  // producer ids: weight ring (warp 0, then the first extra warps), token ring (warp 6, then the
  // rest)
  int a_pid = -1, b_pid = -1;
  if (warp == 0) {
    a_pid = 0;
  } else if (warp == 6) {
    b_pid = 0;
  } else if (warp >= base_warps<WIDE>()) {
    const int x = warp - base_warps<WIDE>();
    if (x < kProdA - 1) a_pid = x + 1;
    else b_pid = x - (kProdA - 1) + 1;
  }
  if (a_pid >= 0) {
    // ---------------------------------------------------------------- weight producer(s)
    const int pid = a_pid;
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
      for (int t = unit0; t < total && ok; t += nunits) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const uint64_t pol = tl.nt > 1 ? pol_shared : pol_once;
        // a tall tile's k-step fills two weight stages, one per scheduled m-tile (and issuer)
        const int parts = tl.tall ? 2 : 1;
        const int kblocks = P.K >> 6;
        for (int kb = 0; kb < kblocks && ok; ++kb) {
          for (int part = 0; part < parts; ++part) {
            if (stage % kProdA != pid) {  // another producer's stage
              if (++stage == SA) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            const int mp = tl.tall ? 2 * tl.m + part : tl.m;  // scheduled m-tile
            const int mc = CG == 2 ? 2 * mp + rank : mp;        // this CTA's weight tile
            const int arow = tl.seg * P.a_seg_stride + mc * P.a_m_stride;
            const bool box1 = a_has_box1(P, mc);
            // the even CTA's barrier counts the bytes of both CTAs of a pair
            const uint32_t bytes = CG == 2 ? a_block_bytes(P, 2 * mp) + a_block_bytes(P, 2 * mp + 1)
                                           : a_block_bytes(P, mc);
            if (!mbar_wait(&empty_a[stage], phase ^ 1u, abort_flag, p.err, kErrProducerWait)) {
              ok = false;
              break;
            }
            uint8_t* sA = ring_a + (size_t)stage * kABytes;
            if (leader) {
              mbar_arrive_expect_tx(&full_a[stage], bytes);
              ++armed[stage];
            }
            if constexpr (CG == 2) {
              const uint32_t fb = mapa_shared(smem_u32(&full_a[stage]), 0);
              tma_load_2d_pair(sA, &P.tmA, fb, kb * 64, arow, pol);
              if (box1) tma_load_2d_pair(sA + 64 * 128, &P.tmA, fb, kb * 64, arow + P.a_box1_off, pol);
            } else {
              tma_load_2d(sA, &P.tmA, &full_a[stage], kb * 64, arow, pol);
              if (box1) tma_load_2d(sA + 64 * 128, &P.tmA, &full_a[stage], kb * 64, arow + P.a_box1_off, pol);
            }
            if (++stage == SA) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) drain_ring(full_a, armed, SA, p.err);
    }
    __syncwarp();
  } else if (b_pid >= 0) {
    // ---------------------------------------------------------------- token producer(s)
    // Tiles of token rows by TMA.  The gathering GEMM (the fused dispatch) instead loads B row
    // r of a routed tile from row sorted_token[r] of x (the shared expert's tile from row r)
    // with tile::gather4, four rows per instruction, spread over the warp's 32 lanes; rows past
    // the segment point past the end of x and read zeros (their columns are never stored).
    // Either way the data lands in the 128-byte-swizzled layout the MMA descriptors expect and
    // its bytes are counted on the pair leader's full barrier.
    const int pid = b_pid;
    if (gather || lane == 0) {
      const uint64_t pol_x = l2_policy_evict_last();  // re-read by every weight tile
      int stage = 0;
      uint32_t phase = 0;
      int armed[kMaxStagesB];
      for (int s = 0; s < kMaxStagesB; ++s) armed[s] = 0;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += nunits) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const NSplit ns = n_split<WIDE>(tl.ncols);
        const uint32_t bytes = static_cast<uint32_t>(tl.ncols * 128);
        const int kblocks = P.K >> 6;
        // gathering: this CTA's rows of MMA 0 and MMA 1 (stage rows [0, rows0) and
        // [rows0, rows0 + rows1)), their first rows in the tile, the end of the segment
        const int rows0 = CG == 2 ? ns.n0 >> 1 : ns.n0;
        const int rows1 = CG == 2 ? ns.n1 >> 1 : ns.n1;
        const int g00 = tl.row0 + rank * rows0, g10 = tl.row0 + ns.n0 + rank * rows1;
        const int end = tl.row0 + tl.valid;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (stage % kProdB != pid) {  // another producer's stage
            if (++stage == SB) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          bool freed = true;
          if (lane == 0)
            freed = mbar_wait(&empty_b[stage], phase ^ 1u, abort_flag, p.err, kErrProducerWait);
          if (gather) freed = __shfl_sync(0xFFFFFFFFu, freed ? 1 : 0, 0) != 0;
          if (!freed) {
            ok = false;
            break;
          }
          uint8_t* sB = ring_b + (size_t)stage * p.b_stage_bytes;
          if (leader && lane == 0) {
            mbar_arrive_expect_tx(&full_b[stage], bytes);
            ++armed[stage];
          }
          const uint32_t fb = CG == 2 ? mapa_shared(smem_u32(&full_b[stage]), 0) : 0u;
          const int kx = kb * 64;
          if (gathers<MODE>() && gather) {
            for (int i = lane; i < (rows0 + rows1) >> 2; i += 32) {
              int src[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int r = 4 * i + j;
                const int g = r < rows0 ? g00 + r : g10 + (r - rows0);
                src[j] = g < end ? (P.gidx != nullptr ? __ldg(P.gidx + g) : g) : P.grows;
              }
              if constexpr (CG == 2)
                tma_gather4_pair(sB + i * 512, &P.tmB[0], fb, kx, src, pol_x);
              else
                tma_gather4(sB + i * 512, &P.tmB[0], &full_b[stage], kx, src, pol_x);
            }
            if (++stage == SB) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          // each MMA's N token rows are split over a pair: the even CTA holds the first half,
          // the odd one the second (N is a multiple of 16, so each half is a multiple of 8);
          // a wide tile's second MMA follows the first in the stage
          int soff = 0;  // shared-memory row of this CTA's stage
#pragma unroll 1
          for (int h = 0; h < kIssuers; ++h) {
            const int nh = h == 0 ? ns.n0 : ns.n1;
            const int rows = CG == 2 ? nh >> 1 : nh;
            const int g0 = tl.row0 + (h == 0 ? 0 : ns.n0) + rank * rows;
            int off = 0;
            // boxes of 128, 64, 32, 16 and 8 rows cover any multiple of 8
#pragma unroll 1
            for (int b = 0, box = 128; b < 5; ++b, box >>= 1) {
              const int nbox = b == 0 ? (rows - off) >> 7 : ((rows - off) >= box ? 1 : 0);
              for (int i = 0; i < nbox; ++i) {
                if constexpr (CG == 2)
                  tma_load_2d_pair(sB + (soff + off) * 128, &P.tmB[b], fb, kx, g0 + off, pol_x);
                else
                  tma_load_2d(sB + (soff + off) * 128, &P.tmB[b], &full_b[stage], kx, g0 + off, pol_x);
                off += box;
              }
            }
            soff += rows;
          }
          if (++stage == SB) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader && lane == 0) drain_ring(full_b, armed, SB, p.err);
    }
    __syncwarp();
  } else if (warp == 1 || (WIDE && warp == 7)) {
    // ---------------------------------------------------------------- MMA issuer(s)
    // Issuer h owns MMAs over token columns [h ? n0 : 0, +n_h) into accumulator columns
    // [h * 256, +n_h); both wait for every stage and release it after their MMAs.
    const int h = warp == 1 ? 0 : 1;
    if (lane == 0 && leader) {
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      int acc_i = 0;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += nunits) {
        Tile tl;
        decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
        const TcProblem& P = p.prob[tl.prob];
        const NSplit ns = n_split<WIDE>(tl.ncols);
        // a wide tile splits its token columns over the issuers; a tall tile gives each issuer
        // all of them against its own weight stage
        const int nh = tl.tall ? tl.ncols : (h == 0 ? ns.n0 : ns.n1);
        const int brow = tl.tall || h == 0 ? 0 : (CG == 2 ? ns.n0 >> 1 : ns.n0);  // B stage row
        const int parts = tl.tall ? 2 : 1;
        const int buf = acc_i % kBufs;
        const uint32_t use = static_cast<uint32_t>(acc_i / kBufs);
        // a pair's accumulator is free once the epilogues of both CTAs have read it
        const bool freed =
            CG == 2 ? mbar_wait_cluster(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p.err, kErrMmaWait)
                    : mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p.err, kErrMmaWait);
        if (!freed) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kAccCols + h * kAccCols);
        const uint32_t idesc = idesc_bf16_f32(128 * CG, nh > 0 ? nh : 16);
        const int kblocks = P.K >> 6;
        for (int kb = 0; kb < kblocks; ++kb) {
          // the issuers share the token stage; a wide tile's weight stage too, while a tall tile
          // gives each issuer a weight stage of its own, which it alone waits for and releases
          // (committing twice: a weight stage's empty barrier counts one arrival per issuer)
          int ast[2];
          uint32_t aph[2];
          for (int x = 0; x < parts; ++x) {
            ast[x] = sa;
            aph[x] = pa;
            if (++sa == SA) {
              sa = 0;
              pa ^= 1u;
            }
          }
          const int own = WIDE && tl.tall ? h : 0;  // the weight stage this issuer reads
          const bool got = mbar_wait(&full_b[sb], pb, abort_flag, p.err, kErrMmaWait) &&
                           mbar_wait(&full_a[ast[own]], aph[own], abort_flag, p.err, kErrMmaWait);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (nh > 0) {
            const uint64_t ad = sdesc_k_sw128(smem_u32(ring_a + (size_t)ast[own] * kABytes));
            const uint64_t bd =
                sdesc_k_sw128(smem_u32(ring_b + (size_t)sb * p.b_stage_bytes + (size_t)brow * 128));
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_bf16<CG>(d_tmem, ad + 2ull * j, bd + 2ull * j, idesc, (kb | j) != 0 ? 1u : 0u);
          }
          mma_commit<CG>(&empty_a[ast[own]]);
          if (WIDE && tl.tall) mma_commit<CG>(&empty_a[ast[own]]);
          mma_commit<CG>(&empty_b[sb]);
          if (++sb == SB) {
            sb = 0;
            pb ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit<CG>(&tfull[buf]);
        ++acc_i;
      }
      // every MMA this thread issued completes before tensor memory is released
      mma_commit<CG>(&drain[h], 1);
      if (!drain_wait(&drain[h], 0)) atomicCAS(p.err, 0, kErrDrainWait);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    // Group g (warps 2..5, and 8..11 of a wide tile) reads accumulator half g; each warp may
    // only access its tensor-memory lane quarter (warp % 4).
    const int g = warp >= 8 ? 1 : 0;
    const int q = warp & 3;
    const int ep = threadIdx.x - (g == 0 ? 64 : 256);  // 0..127 within the group
    const int bar_or = 1 + 2 * g, bar_sync = 2 + 2 * g;
    float* xchg = xchg0 + g * kXchgFloats;
    const uint32_t tempty_lead[2] = {
        CG == 2 ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u,
        CG == 2 ? mapa_shared(smem_u32(&tempty[1]), 0) : 0u};
    int acc_i = 0;
    for (int t = unit0; t < total; t += nunits) {
      Tile tl;
      decode_tile(p, s_seg, s_ntp, tiles0, t, tl);
      const TcProblem& P = p.prob[tl.prob];
      // this group's scheduled m-tile (a tall tile's group g takes the g-th of its two) and this
      // CTA's 128-row weight tile within it
      const int mp = tl.tall ? 2 * tl.m + g : tl.m;
      tl.m = CG == 2 ? 2 * mp + rank : mp;
      const NSplit ns = n_split<WIDE>(tl.ncols);
      const int buf = acc_i % kBufs;
      const uint32_t use = static_cast<uint32_t>(acc_i / kBufs);
      const bool ok = mbar_wait(&tfull[buf], use & 1u, abort_flag, p.err, kErrEpilogueWait);
      __syncwarp();
      if (named_bar_or(bar_or, 128, !ok || *abort_flag != 0)) break;
      tc_fence_after();
      // this group's token columns: [c0, c0 + valid) of the tile, at accumulator column acol
      const int c0 = tl.tall || g == 0 ? 0 : ns.n0;
      const int width = tl.tall ? tl.ncols : (g == 0 ? ns.n0 : ns.n1);
      int valid = tl.valid - c0;
      valid = valid < 0 ? 0 : (valid > width ? width : valid);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * kAccCols + g * kAccCols);
      const int nchunks = (valid + 31) >> 5;
      const int rowb = P.out_row_base + tl.row0 + c0;  // output row of this group's column 0
      if (tl.m >= P.m_cta || valid == 0) {
        // the second tile of a pair past the end of the weight rows, or no columns here
      } else if (MODE == kModeGateUp) {
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
            if (col0 >= valid) break;  // uniform over the group's 128 threads
#pragma unroll
            for (int j = 0; j < 16; ++j) mine[j * kStageLdF + fl] = __uint_as_float(v[half * 16 + j]);
            named_bar_sync(bar_sync, 128);
            const int col = col0 + tt;
            if (col < valid) {
              const float4* g4 = reinterpret_cast<const float4*>(gs + tt * kStageLdF + fg * 8);
              const float4* u4 = reinterpret_cast<const float4*>(us + tt * kStageLdF + fg * 8);
              const float4 ga = g4[0], gb = g4[1], ua = u4[0], ub = u4[1];
              const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
              const float uv[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
              uint4 o;
              __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float h0 = __fdividef(gv[2 * i] * uv[2 * i], 1.f + __expf(-gv[2 * i]));
                const float h1 =
                    __fdividef(gv[2 * i + 1] * uv[2 * i + 1], 1.f + __expf(-gv[2 * i + 1]));
                oh[i] = __floats2bfloat162_rn(h0, h1);
              }
              *reinterpret_cast<uint4*>(hout + (size_t)(rowb + col) * P.out_ld + tl.m * 64 + fg * 8) = o;
            }
            named_bar_sync(bar_sync, 128);
          }
        }
      } else if (MODE == kModeDown) {
        // Lane = output channel, register j = token 32c + j: for each token the warp stores its
        // 32 consecutive channels (64 contiguous bytes) straight from registers, with no
        // shared-memory transpose and no group barrier.  The tensor-memory load of the next
        // chunk is in flight while one is stored.
        const int ch = tl.m * 128 + q * 32 + lane;
        __nv_bfloat16* ycol = static_cast<__nv_bfloat16*>(P.out) + (size_t)rowb * P.out_ld + ch;
        const bool ch_ok = ch < P.out_valid_m;
        uint32_t va[32], vb[32];
        tmem_ld_32x32b_x32_issue(tbase, va);
        tmem_ld_wait(va);
        for (int c = 0; c < nchunks; c += 2) {  // nchunks is uniform over the group
          const bool more = c + 1 < nchunks;
          if (more) tmem_ld_32x32b_x32_issue(tbase + static_cast<uint32_t>((c + 1) * 32), vb);
          if (ch_ok) store_down_chunk(ycol + (size_t)(c * 32) * P.out_ld, P.out_ld, valid - c * 32, va);
          if (more) {
            tmem_ld_wait(vb);
            const bool again = c + 2 < nchunks;
            if (again) tmem_ld_32x32b_x32_issue(tbase + static_cast<uint32_t>((c + 2) * 32), va);
            if (ch_ok)
              store_down_chunk(ycol + (size_t)((c + 1) * 32) * P.out_ld, P.out_ld, valid - (c + 1) * 32, vb);
            if (again) tmem_ld_wait(va);
          }
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
            if (e_ok && col < valid) lout[(size_t)(rowb + col) * P.out_ld + e] = __uint_as_float(v[j]);
          }
        }
      }
      // this warp's reads of the accumulator are done: one arrival per warp on the (even
      // CTA's) accumulator-empty barrier
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) mbar_arrive_remote(tempty_lead[buf]);
        else mbar_arrive(&tempty[buf]);
      }
      ++acc_i;
    }
  }

  __syncthreads();
  // no CTA of a pair leaves (or frees tensor memory) while the pair's MMAs, TMA completions or
  // remote arrivals may still touch it
  if constexpr (CG == 2) cluster_sync();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, tmem_cols<CG, WIDE>());
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) record_clocks(p.err, MODE, clk0, ns0);
}

size_t fixed_smem_bytes(int n_seg, int wide) {
  return 1024 + kBarBytes + kMiscBytes + sizeof(float) * kXchgFloats * (wide ? 2 : 1) +
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

// Opt-in shared memory of a kernel instance, set once per device.
template <int MODE, int CG, int WIDE>
cudaError_t configure(int dev) {
  static std::mutex mu;
  static unsigned long long configured = 0;  // bit per device
  std::lock_guard<std::mutex> g(mu);
  if (dev < 64 && ((configured >> dev) & 1ull)) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(gemm_tc_kernel<MODE, CG, WIDE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_limit(CG, WIDE)));
  // the whole unified L1/shared array as shared memory: two pair CTAs per SM need it
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(gemm_tc_kernel<MODE, CG, WIDE>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  if (err == cudaSuccess && dev < 64) configured |= 1ull << dev;
  return err;
}

template <int MODE>
cudaError_t launch_single(const TcParams& p, int sms, size_t smem, cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if ((err = configure<MODE, 1, 0>(dev)) != cudaSuccess) return err;
  gemm_tc_kernel<MODE, 1, 0><<<sms, threads_of<MODE, 1, 0>(), smem, s>>>(p);
  return cudaGetLastError();
}

cudaLaunchConfig_t pair_config(int grid, int threads, size_t smem, cudaStream_t s,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// CTA pairs resident at once: the persistent grid.  A pair CTA's shared-memory budget (at most
// kSmemLimitPair) leaves room for two of them per SM, so two pairs run on each TPC.  The
// occupancy queries of the runtime report one cluster per TPC for this kernel, yet a grid of
// two pairs per TPC measures almost twice the MMA rate of one, so the count is taken from the
// budget.  Were it ever too high the extra pairs would only wait for a free TPC (the tiles are
// statically strided over pairs and no pair waits for another), costing time, not results.
int resident_pairs(int sms, size_t smem, int wide) {
  const int per_sm = !wide && smem <= kSmemLimitPair ? 2 : 1;
  return per_sm * (sms / 2);
}

template <int MODE, int WIDE>
cudaError_t launch_pair(const TcParams& p, int sms, size_t smem, cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if ((err = configure<MODE, 2, WIDE>(dev)) != cudaSuccess) return err;
  const int pairs = resident_pairs(sms, smem, WIDE);
  if (pairs < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(2 * pairs, threads_of<MODE, 2, WIDE>(), smem, s, attr);
  err = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<MODE, 2, WIDE>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

__global__ void wait_timeout_kernel(int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  // nothing arrives on the barrier, so its first phase never completes
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, err, kErrDiagWait, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_pair_unclustered(int* err, cudaStream_t s) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.err = err;
  gemm_tc_kernel<kModeDown, 2, 1><<<2, threads_of<kModeDown, 2, 1>(), 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

// Ring depths for an n-tile cap: the token ring holds a few stages (its loads hit L2), the
// weight ring takes the rest of shared memory (its loads come from HBM).  A CTA of a pair
// holds half of each token tile and shares its SM with a second pair CTA, so it has half the
// shared memory.
void gemm_tc_plan(int bn, int n_seg, TcParams& p) {
  const int rows = p.cg == 2 ? bn / 2 : bn;
  p.b_stage_bytes = rows * 128;
  const int pa = p.cg == 1 ? producers_a<1, 0>() : (p.wide ? producers_a<2, 1>() : producers_a<2, 0>());
  const int pb = p.cg == 1 ? producers_b<1, 0>() : (p.wide ? producers_b<2, 1>() : producers_b<2, 0>());
  if (p.cg == 2 && !p.wide) p.stages_b = bn >= 128 ? 2 : kMaxStagesB;
  else p.stages_b = bn >= 128 ? (p.wide ? 4 : 3) : 4;
  p.stages_b -= p.stages_b % pb;
  const size_t avail = smem_limit(p.cg, p.wide) - fixed_smem_bytes(n_seg, p.wide) -
                       (size_t)p.stages_b * p.b_stage_bytes;
  int sa = static_cast<int>(avail / kABytes);
  sa = sa > kMaxStagesA ? kMaxStagesA : sa;
  p.stages_a = sa - sa % pa;
}

size_t gemm_tc_smem_bytes(const TcParams& p) {
  const int n_seg = p.prob[0].seg_off != nullptr ? p.prob[0].n_seg : 0;
  size_t b = fixed_smem_bytes(n_seg, p.wide) + (size_t)p.stages_a * kABytes +
             (size_t)p.stages_b * p.b_stage_bytes;
  return p.cg == 1 && b < kSmemFloor ? kSmemFloor : b;
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

cudaError_t launch_gemm_tc(int mode, const TcParams& p, int sms, cudaStream_t s) {
  const size_t smem = gemm_tc_smem_bytes(p);
  const int pa = p.cg == 1 ? producers_a<1, 0>() : (p.wide ? producers_a<2, 1>() : producers_a<2, 0>());
  const int pb = p.cg == 1 ? producers_b<1, 0>() : (p.wide ? producers_b<2, 1>() : producers_b<2, 0>());
  if (smem > smem_limit(p.cg, p.wide) || p.stages_a < 2 || p.stages_b < 2 ||
      p.stages_a > kMaxStagesA || p.stages_b > kMaxStagesB || p.stages_a % pa != 0 ||
      p.stages_b % pb != 0)
    return cudaErrorInvalidConfiguration;
  // the forms this library uses: router on one CTA, gate/up on wide pairs, down on pairs
  if (mode == kModeRouter && p.cg == 1 && !p.wide) return launch_single<kModeRouter>(p, sms, smem, s);
  if (mode != kModeGateUp && p.gather != 0) return cudaErrorInvalidConfiguration;
  // tall tiles need the two MMA issuers of the wide pair form
  if ((p.prob[0].tall_rows > 0 || p.prob[1].tall_rows > 0) && !(p.cg == 2 && p.wide))
    return cudaErrorInvalidConfiguration;
  if (mode == kModeGateUp && p.cg == 2 && p.wide && p.bn <= 2 * kAccCols)
    return launch_pair<kModeGateUp, 1>(p, sms, smem, s);
  if (mode == kModeGateUp && p.cg == 2 && !p.wide && p.bn <= kAccCols)
    return launch_pair<kModeGateUp, 0>(p, sms, smem, s);
  if (mode == kModeDown && p.cg == 2 && !p.wide && p.bn <= kAccCols)
    return launch_pair<kModeDown, 0>(p, sms, smem, s);
  if (mode == kModeDown && p.cg == 2 && p.wide && p.bn <= 2 * kAccCols)
    return launch_pair<kModeDown, 1>(p, sms, smem, s);
  return cudaErrorInvalidConfiguration;
}

}  // namespace moe
