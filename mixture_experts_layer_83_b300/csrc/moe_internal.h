// Host-side declarations shared by the kernel files and the C ABI layer (moe_api.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Codes a kernel records in the workspace status word when it gives up on a wait.
enum DeviceErr {
  kErrNone = 0,
  kErrProducerWait = 1,
  kErrMmaWait = 2,
  kErrEpilogueWait = 3,
  kErrDrainWait = 4,
  kErrLaunchShape = 5,  // a CTA-pair kernel was launched without 2-CTA clusters
  kErrDiagWait = 6,     // the diagnostic wait of moe_debug_wait_timeout ran out (its purpose)
};

// Epilogues of the tensor-core grouped GEMM.
enum GemmMode { kModeRouter = 0, kModeGateUp = 1, kModeDown = 2 };

// Clock records in the status block: CTA 0 of each tensor-core kernel writes {clock64 at start,
// %globaltimer at start, clock64 at end, %globaltimer at end} to slot (router 0, gate/up 1,
// down 2), 64 bit each, starting kClockOffset bytes after the status word.
constexpr int kClockOffset = 64;
__device__ __forceinline__ void record_clocks(int* status, int slot, long long c0, long long t0) {
  long long t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  long long* r = reinterpret_cast<long long*>(reinterpret_cast<char*>(status) + kClockOffset) + 4 * slot;
  r[0] = c0;
  r[1] = t0;
  r[2] = clock64();
  r[3] = t1;
}

// Assignments handled per block by the dispatch histogram / permutation kernels.
constexpr int kDispatchChunk = 1024;
constexpr int kDispatchWarps = 8;

// One operand set of the persistent grouped GEMM.  "A" is always a weight matrix (the
// MMA's M dimension, 128 rows per tile), "B" the token rows (the MMA's N dimension, a
// multiple of 16 up to the n-tile cap), both K-major bf16 read through TMA with 128-byte
// swizzle; the product is D = A * B^T accumulated in fp32 in tensor memory.
struct TcProblem {
  CUtensorMap tmA;     // weights [rows][K]: box 64 columns x a_box_rows rows
  CUtensorMap tmB[5];  // tokens  [rows][K]: boxes of 128 / 64 / 32 / 16 / 8 rows x 64 columns
  void* out;
  const int* seg_off;  // grouped: device [n_seg+1] first B row of each segment; null = single
  const int* ntp;      // grouped: device [n_seg+1] prefix of tile units per segment
  int tall_rows;       // grouped, pairs: segments of 1..tall_rows rows run as tall tiles (0: none)
  int K;               // reduction length, multiple of 64
  int m_tiles;         // scheduled m-tiles per segment: weight tiles of one CTA, or of a pair
  int m_cta;           // 128-row weight tiles per segment (a pair's second tile may be past it)
  int group;           // m-tiles scheduled together (divides m_tiles)
  int a_seg_stride;    // A rows between segments
  int a_m_stride;      // A rows between m-tiles
  int a_box1_off;      // A row offset of the second box of a tile
  int a_valid_rows;    // second box is loaded only if (m * a_m_stride + a_box1_off) < this
  int a_box_rows;      // rows per A box (64, or the whole A height when smaller)
  int n_seg;           // grouped: number of segments
  int rows;            // single segment: B rows
  int nt;              // single segment: n-tiles
  int out_ld;          // output row stride in elements
  int out_row_base;    // output row of B row 0
  int out_valid_m;     // weight rows that produce output (router: E, down: d)
  // Token rows gathered by the kernel itself (gate/up): B row r is row gidx[r] (row r when
  // gidx is null) of the grows-row tensor that tmB[0] maps with a one-row box.
  const int* gidx;
  int grows;
};

struct TcParams {
  TcProblem prob[2];
  int n_prob;
  int cg;             // CTAs per MMA: 1, or 2 (a CTA pair, tcgen05 cta_group::2, M = 256)
  int wide;           // pairs only: n-tiles up to 512 token rows, split over two MMA issuers
  int bn;             // n-tile cap: multiple of 16, at most 256 (512 for wide pairs)
  int stages_a;       // depth of the weight ring (16 KiB stages)
  int stages_b;       // depth of the token ring
  int b_stage_bytes;  // B rows one CTA holds per stage (bn, or bn / 2 for a pair) * 128 B
  int gather;         // 1: token rows are gathered by TMA tile::gather4 (gate/up), 0: tiles
  int* err;           // device status word
};

// Tensor-core GEMM (moe_gemm_tc.cu).
size_t gemm_tc_smem_bytes(const TcParams& p);
void gemm_tc_plan(int bn, int n_seg, TcParams& p);
// Launches one GEMM: `sms` CTAs (cg 1), or as many 2-CTA clusters as fit at once (cg 2).
cudaError_t launch_gemm_tc(int mode, const TcParams& p, int sms, cudaStream_t s);
int encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows);
// Diagnostics of the device error path: the CTA-pair GEMM launched as two plain CTAs (no
// cluster), which records kErrLaunchShape in *err and returns at once; and one CTA waiting on
// an mbarrier that nothing completes, with a wall-clock limit of limit_ns, which records
// kErrDiagWait in *err when the limit runs out and returns.
cudaError_t launch_pair_unclustered(int* err, cudaStream_t s);
cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t s);

// Fused router of bf16 layers with E <= 256 (moe_router_tc.cu): gate GEMM on CTA pairs, score,
// top-k and renormalisation in its epilogue.
struct RouterParams {
  CUtensorMap tmA;  // w_router [E][d]: box 64 columns x 128 rows
  CUtensorMap tmB;  // x [T][d]: box 64 columns x N / 2 rows
  const float* bias;
  int* topk_idx;
  float* topk_w;
  float* partial;   // split reduction: [splits][T][E] fp32 partial logits
  int* counters;    // split reduction: [blocks] arrivals, zero when the kernel starts
  int* err;         // device status word
  int T, E, k, G, M, d;
  int kc;           // > k: candidate mode ([T][kc] experts and raw values, for rerouting)
  int N;            // tokens per block: multiple of 16, at most 256
  int blocks, splits, kb_per_split, kblocks;
  int stages, b_stage_bytes;
};
// Geometry for T tokens (-1: the shape does not fit this router).  max_partial_rows bounds
// splits * T.
int router_tc_plan(int T, int d, int E, int sms, int max_partial_rows, RouterParams& p);
size_t router_tc_smem_bytes(const RouterParams& p);
// score_fn: 0 softmax, 1 sigmoid.
cudaError_t launch_router_tc(int score_fn, const RouterParams& p, cudaStream_t s);

// Router (moe_router.cu).
cudaError_t launch_router_logits_f32(const float* x, const float* w_router, int T, int d, int E,
                                     float* logits, cudaStream_t s);
// src: 0 = logits + softmax, 1 = logits + sigmoid, 2 = supplied key (a) and score (b).
// G > 0: group-limited, M of G contiguous expert groups kept per token (G = 0: plain top-k).
// kc > k: candidate mode, [T][kc] experts in selection order and their raw values.
cudaError_t launch_topk(int src, const float* a, const float* b, const float* bias, int T, int E,
                        int k, int G, int M, int* topk_idx, float* topk_w, cudaStream_t s,
                        int kc = 0);

// Dispatch (moe_dispatch.cu).
// ntp / ntp2 (either may be null): per-expert prefixes of tile units (seg_units) for n-tile
// caps bn / bn2 and tall-tile limits tall / tall2.
// capacity: per-expert limit of dispatched assignments (INT_MAX: dropless); *dropped (may be
// null) receives the number dropped; a dropped assignment gets slot_pos -1.
cudaError_t launch_dispatch(const int* topk_idx, int T, int k, int E, int bn, int tall,
                            int* chunk_counts, int* expert_counts, int* offsets, int* ntp, int bn2,
                            int tall2,
                            int* ntp2, int capacity, int* dropped, int* sorted_token,
                            int* slot_pos, cudaStream_t s);
// Rerouting at capacity: from cand [T][kc] (experts in selection order) and their raw values,
// rounds of proposals up to each expert's capacity; writes the serving expert of every slot
// (-1: dropped) to topk_idx [T][k], the weights renormalised over the serving experts to
// topk_w (src: 0 softmax logits, 1 sigmoid logits) and the number of dropped slots to *dropped
// (may be null).  Scratch: chunk_counts as for the dispatch, prop / assign_c [T*k], next_c [T],
// fill / left [E].
cudaError_t launch_reroute(const int* cand, const float* cand_val, int T, int k, int kc, int E,
                           int capacity, int src, int* chunk_counts, int* prop, int* assign_c,
                           int* next_c, int* fill, int* left, int* topk_idx, float* topk_w,
                           int* dropped, cudaStream_t s);
// rows_dev (may be null): device row count replacing R (rows dispatched under a capacity).
cudaError_t launch_gather(const void* x, const int* sorted_token, int R, const int* rows_dev,
                          int d, int elt_bytes, void* xs, cudaStream_t s);

// fp32 expert FFN on CUDA cores (moe_ffn_simt.cu).
cudaError_t launch_ffn_f32(const float* xs, const float* x, const int* offsets, int E, int R,
                           int T_sh, int d, int F, int Fs, const float* w_gate_up,
                           const float* w_down, const float* sh_gate_up, const float* sh_down,
                           float* h, float* h_sh, float* y, cudaStream_t s, int stage);

// Combine (moe_combine.cu).
cudaError_t launch_combine(const void* y, const int* slot_pos, const float* topk_w, int T, int k,
                           int d, int R, int has_shared, int bf16, void* out, cudaStream_t s);

}  // namespace moe
