// C ABI of the MoE layer (declared in include/moe_layer.h): argument checks, the workspace
// layout, tensor-map encoding and the launch sequence on the caller's stream.
//
// Sequence of one forward pass (all on `stream`, no host synchronisation):
//   router GEMM -> top-k -> histogram / scan / stable permutation -> gather -> gate/up grouped
//   GEMM (+SwiGLU) -> down grouped GEMM -> combine.
// bf16 layers run the three GEMMs on the tensor cores (moe_gemm_tc.cu); fp32 layers run them
// in true fp32 on CUDA cores (moe_router.cu, moe_ffn_simt.cu).  Routing, dispatch and combine
// kernels are shared by both.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/moe_layer.h"
#include "moe_internal.h"
#include "tile_sched.h"

namespace moe {
namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The CUDA error behind this thread's latest MOE_ERR_CUDA (moe_last_cuda_error_name).
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

int cuda_failed(cudaError_t e) {
  t_last_cuda_error = e;
  return MOE_ERR_CUDA;
}

// The status block: the device status word, then the fused router's per-block arrival
// counters; cleared at the start of every forward pass.
constexpr size_t kStatusBytes = 2048;
constexpr int kCounterInts = 256;
constexpr size_t kCounterOffset = 512;
// Rows of partial logits the fused router may write when it splits the reduction over d.
constexpr int kRouterPartialRows = 2048;

// Whether a layer runs the fused router (tensor-core gate GEMM with the top-k in its epilogue).
bool fused_router(const moe_shape& s) { return s.dtype == MOE_DTYPE_BF16 && s.E <= 256; }

struct Layout {
  size_t status, logits, partial, topk_idx, topk_w, chunk, offsets, ntp, ntp2, sorted, slot,
      cand, cand_val, prop, assign_c, next_c, fill, left, xs_y, h, h_sh, total;
};

// Workspace carve-up.  xs (gathered rows) and y (expert outputs, routed rows then the shared
// expert's rows) share one region: xs is dead once the gate/up GEMM has consumed it.
Layout layout_of(const moe_shape& s) {
  const size_t elt = s.dtype == MOE_DTYPE_BF16 ? 2 : 4;
  const size_t R = (size_t)s.T * s.k;
  const size_t nch = (R + kDispatchChunk - 1) / kDispatchChunk;
  const size_t tsh = s.Fs > 0 ? (size_t)s.T : 0;
  Layout w;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  w.status = take(kStatusBytes);
  w.logits = take(fused_router(s) ? 0 : (size_t)s.T * s.E * 4);
  w.partial = take(fused_router(s) ? (size_t)kRouterPartialRows * s.E * 4 : 0);
  w.topk_idx = take(R * 4);
  w.topk_w = take(R * 4);
  w.chunk = take(nch * s.E * 4);
  w.offsets = take((size_t)(s.E + 1) * 4);
  w.ntp = take((size_t)(s.E + 1) * 4);
  w.ntp2 = take((size_t)(s.E + 1) * 4);
  w.sorted = take(R * 4);
  w.slot = take(R * 4);
  // rerouting at capacity: up to 32 candidates per token and the rounds' state
  w.cand = take((size_t)s.T * 32 * 4);
  w.cand_val = take((size_t)s.T * 32 * 4);
  w.prop = take(R * 4);
  w.assign_c = take(R * 4);
  w.next_c = take((size_t)s.T * 4);
  w.fill = take((size_t)s.E * 4);
  w.left = take((size_t)s.E * 4);
  w.xs_y = take((R + tsh) * s.d * elt);
  w.h = take(R * s.F * elt);
  w.h_sh = take(tsh * (size_t)s.Fs * elt);
  w.total = o;
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const moe_shape* s, bool routing_only) {
  if (s == nullptr) return MOE_ERR_INVALID_ARG;
  if (s->T < 1 || s->E < 1 || s->k < 1 || s->k > s->E || s->k > kMaxK || s->E > kMaxE)
    return MOE_ERR_INVALID_ARG;
  if ((long long)s->T * s->k > INT_MAX / 2) return MOE_ERR_INVALID_ARG;
  if (routing_only) return MOE_OK;
  if (s->d < 1 || s->F < 1 || s->Fs < 0) return MOE_ERR_INVALID_ARG;
  if (s->dtype != MOE_DTYPE_F32 && s->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  const long long R = (long long)s->T * s->k;
  if ((R + s->T) * (long long)s->d > (1LL << 40) || R * (long long)s->F > (1LL << 40))
    return MOE_ERR_INVALID_ARG;
  if ((long long)s->E * 2 * s->F > INT_MAX || (long long)s->E * s->d > INT_MAX)
    return MOE_ERR_INVALID_ARG;
  if (s->dtype == MOE_DTYPE_BF16 && (s->d % 64 != 0 || s->F % 64 != 0 || s->Fs % 64 != 0))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Group-limited routing: G contiguous groups of E / G experts (G <= 32), M kept per token, with
// room for k experts in the kept groups.  G = 0: plain top-k.
int check_groups(const moe_shape& s, int G, int M) {
  if (G == 0 && M == 0) return MOE_OK;
  if (G < 1 || G > 32 || s.E % G != 0 || M < 1 || M > G || M * (s.E / G) < s.k)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Expert capacity for a capacity factor: ceil(factor * T * k / E) dispatched assignments per
// expert, INT_MAX for a factor of 0 (dropless).  -1: an invalid factor.
int capacity_of(const moe_shape& s, double factor) {
  if (factor == 0.0) return INT_MAX;
  if (!(factor > 0.0) || !isfinite(factor)) return -1;
  const double c = ceil(factor * ((double)s.T * (double)s.k / (double)s.E));
  return c >= (double)INT_MAX ? INT_MAX : (int)c;
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> g(mu);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

int largest_group(int m_tiles) {
  for (int g = 16; g > 1; g >>= 1)
    if (m_tiles % g == 0) return g;
  return 1;
}

// n-tile cap of the down GEMM: twice the mean rows per expert, 32..256.
int expert_bn(const moe_shape& s) {
  const long long R = (long long)s.T * s.k;
  const int avg = (int)((R + s.E - 1) / s.E);
  int bn = pow2_at_least(avg * 2 > 32 ? avg * 2 : 32);
  return bn > 256 ? 256 : bn;
}

// Whether the gate/up GEMM runs on wide pairs: when experts average more than 64 rows (a
// prefill batch), a segment of up to twice the mean rows then shares one pass over the
// expert's weights.  Smaller segments (decode) stream weights with more producers per SM on
// two narrow pairs per TPC instead.
bool gateup_wide(const moe_shape& s) { return expert_bn(s) >= 256; }

// Segments run on wide pairs as tall tiles: two scheduled m-tiles (512 weight rows per pair)
// over up to 256 of the segment's rows, one per MMA issuer, which halves the token traffic
// per FLOP against a 256-row weight tile and gives both issuers full-width MMAs.  Needs an
// even number of scheduled m-tiles.
int gateup_tall_rows(const moe_shape& s) {
  const int pairs = (s.F / 64 + 1) / 2;
  return gateup_wide(s) && pairs % 2 == 0 ? 256 : 0;
}

// Whether every segment runs as tall n-tiles (ceil(rows / 256) of them, rows split evenly):
// the n-tile cap is then the tall-tile limit.  Chosen when experts average 384 rows or more:
// long segments then stream each token stage once per 512 weight rows instead of 256
// (measured on one B300, same box: Mixtral-shaped layer 2.10 ms against 2.24 ms with wide
// tiles); at about 256 rows per expert (the DeepSeek-V3 prefill layer) the wide tiles of up
// to 384 rows are faster (7.39 ms against 7.96 ms).
bool gateup_all_tall(const moe_shape& s) {
  const long long R = (long long)s.T * s.k;
  return gateup_tall_rows(s) > 0 && (R + s.E - 1) / s.E >= 384;
}

// n-tile cap of the expert GEMMs on wide pairs: the tall-tile limit when every tile is tall;
// else 512 token rows when experts average 384 rows or more (two full 256-column MMA halves
// per tile), else 384 (segments near the mean still fit one tile, and the smaller token stages
// leave shared memory for a six-deep weight ring); the narrow cap otherwise.
int gateup_bn(const moe_shape& s) {
  if (!gateup_wide(s)) return expert_bn(s);
  if (gateup_all_tall(s)) return gateup_tall_rows(s);
  const long long R = (long long)s.T * s.k;
  return (R + s.E - 1) / s.E >= 384 ? 512 : 384;
}

// Whether the gate/up GEMM gathers its token rows from x itself (TMA tile::gather4 through
// the dispatch permutation: the fused dispatch) instead of reading a permuted copy of x that a
// separate gather kernel writes.  It does on narrow pairs (decode-sized segments), where the
// gathers cost nothing measurable and the gather launch goes away.  Wide pairs need a token
// stage of up to 256 rows per CTA every k-step, 64 four-row gathers against 2 box loads, and
// the TMA unit's gather rate then bounds the GEMM below its tensor rate (measured on one B300,
// same box, DeepSeek-V3 prefill: gate/up 4.93 ms gathering against 4.28 ms + 0.25 ms for the
// separate gather).
bool gateup_gathers(const moe_shape& s) { return !gateup_wide(s); }

// The down GEMM runs on wide pairs exactly when gate/up does; its tall tiles need an even
// number of scheduled m-tiles whenever gate/up has tall tiles, else it stays on narrow pairs
// (measured on the DeepSeek-V3 prefill layer: 2.19-2.25 ms on wide pairs with tall tiles
// against 2.57-2.59 ms on narrow pairs).
bool down_wide(const moe_shape& s) {
  const int pairs = ((s.d + 127) / 128 + 1) / 2;
  return gateup_wide(s) && (pairs % 2 == 0 || gateup_tall_rows(s) == 0);
}
// (A double-buffered form, every tile two weight tiles over at most 128 rows so that two
// accumulators fit the 512 TMEM columns, measured 3.16 ms against 2.28 ms here: 128-row MMAs
// cannot keep the tensor pipe busy.)
int down_bn(const moe_shape& s) { return down_wide(s) ? gateup_bn(s) : expert_bn(s); }
int down_tall_rows(const moe_shape& s) {
  const int pairs = ((s.d + 127) / 128 + 1) / 2;
  return down_wide(s) && pairs % 2 == 0 ? gateup_tall_rows(s) : 0;
}

// n-tile cap of the router GEMM: about one tile per SM.
int router_bn(const moe_shape& s, int sms) {
  const int m_tiles = (s.E + 127) / 128;
  const int nt_target = (sms + m_tiles - 1) / m_tiles;
  int per = (s.T + nt_target - 1) / nt_target;
  int bn = pow2_at_least(per < 16 ? 16 : per);
  return bn > 256 ? 256 : bn;
}

int encode_tokens(TcProblem& P, const void* base, int rows, int cols) {
  const uint32_t boxes[5] = {128, 64, 32, 16, 8};
  for (int b = 0; b < 5; ++b)
    if (encode_tmap_bf16(&P.tmB[b], base, (uint64_t)rows, (uint64_t)cols, boxes[b]) != 0) return -1;
  return 0;
}

struct Plan {
  TcParams router, gateup, down;
};

// Tile geometry of the three GEMMs of a bf16 layer (everything but pointers and tensor maps).
void geometry_router(const moe_shape& s, int sms, TcParams& p) {
  memset(&p, 0, sizeof(p));
  TcProblem& P = p.prob[0];
  p.n_prob = 1;
  p.cg = 1;
  p.bn = router_bn(s, sms);
  P.a_box_rows = s.E < 64 ? s.E : 64;
  P.K = s.d;
  P.m_cta = (s.E + 127) / 128;
  P.m_tiles = P.m_cta;
  P.group = largest_group(P.m_tiles);
  P.a_seg_stride = 0;
  P.a_m_stride = 128;
  P.a_box1_off = 64;
  P.a_valid_rows = s.E;
  P.rows = s.T;
  P.nt = (s.T + p.bn - 1) / p.bn;
  P.out_ld = s.E;
  P.out_valid_m = s.E;
  gemm_tc_plan(p.bn, 0, p);
}

// The expert GEMMs run on CTA pairs: a scheduled m-tile is two 128-row weight tiles.
void set_m_tiles(TcProblem& P, int m_cta, int cg) {
  P.m_cta = m_cta;
  P.m_tiles = cg == 2 ? (m_cta + 1) / 2 : m_cta;
  P.group = largest_group(P.m_tiles);
}

void geometry_gateup(const moe_shape& s, TcParams& p) {
  memset(&p, 0, sizeof(p));
  const int bn = gateup_bn(s);
  p.n_prob = s.Fs > 0 ? 2 : 1;
  p.cg = 2;
  p.wide = gateup_wide(s) ? 1 : 0;
  p.bn = bn;
  p.gather = gateup_gathers(s) ? 1 : 0;
  TcProblem& P = p.prob[0];
  P.a_box_rows = 64;
  P.n_seg = s.E;
  P.K = s.d;
  P.grows = s.T;
  set_m_tiles(P, s.F / 64, p.cg);
  P.tall_rows = gateup_tall_rows(s);
  P.a_seg_stride = 2 * s.F;
  P.a_m_stride = 64;
  P.a_box1_off = s.F;
  P.a_valid_rows = INT_MAX;
  P.out_ld = s.F;
  P.out_valid_m = INT_MAX;
  if (s.Fs > 0) {
    TcProblem& Q = p.prob[1];
    Q.a_box_rows = 64;
    Q.K = s.d;
    Q.grows = s.T;
    set_m_tiles(Q, s.Fs / 64, p.cg);
    Q.a_seg_stride = 0;
    Q.a_m_stride = 64;
    Q.a_box1_off = s.Fs;
    Q.a_valid_rows = INT_MAX;
    Q.rows = s.T;
    Q.nt = (s.T + bn - 1) / bn;
    Q.out_ld = s.Fs;
    Q.out_valid_m = INT_MAX;
  }
  gemm_tc_plan(bn, s.E, p);
}

void geometry_down(const moe_shape& s, TcParams& p) {
  memset(&p, 0, sizeof(p));
  const int bn = down_bn(s);
  p.n_prob = s.Fs > 0 ? 2 : 1;
  p.cg = 2;
  p.wide = down_wide(s) ? 1 : 0;
  p.bn = bn;
  TcProblem& P = p.prob[0];
  P.a_box_rows = 64;
  P.n_seg = s.E;
  P.K = s.F;
  set_m_tiles(P, (s.d + 127) / 128, p.cg);
  P.tall_rows = down_tall_rows(s);
  P.a_seg_stride = s.d;
  P.a_m_stride = 128;
  P.a_box1_off = 64;
  P.a_valid_rows = s.d;
  P.out_ld = s.d;
  P.out_valid_m = s.d;
  if (s.Fs > 0) {
    TcProblem& Q = p.prob[1];
    Q.a_box_rows = 64;
    Q.K = s.Fs;
    set_m_tiles(Q, (s.d + 127) / 128, p.cg);
    Q.a_seg_stride = 0;
    Q.a_m_stride = 128;
    Q.a_box1_off = 64;
    Q.a_valid_rows = s.d;
    Q.rows = s.T;
    Q.nt = (s.T + bn - 1) / bn;
    Q.out_ld = s.d;
    Q.out_row_base = s.T * s.k;
    Q.out_valid_m = s.d;
  }
  gemm_tc_plan(bn, s.E, p);
}

// Geometry plus operand pointers and tensor maps.
int plan_bf16(const moe_shape& s, const void* x, const void* w_router, const void* w_gate_up,
              const void* w_down, const moe_shared_expert* sh, char* ws, const Layout& L,
              const int* sorted, int sms, Plan& pl) {
  const int T = s.T, d = s.d, E = s.E, F = s.F, Fs = s.Fs;
  const int R = T * s.k;
  int* status = reinterpret_cast<int*>(ws + L.status);
  int* offsets = reinterpret_cast<int*>(ws + L.offsets);
  int* ntp = reinterpret_cast<int*>(ws + L.ntp);
  int* ntp2 = reinterpret_cast<int*>(ws + L.ntp2);
  void* xs_y = ws + L.xs_y;
  void* h = ws + L.h;
  void* h_sh = ws + L.h_sh;

  TcParams& pr = pl.router;  // the router GEMM of layers without the fused router
  geometry_router(s, sms, pr);
  pr.err = status;
  pr.prob[0].out = ws + L.logits;
  if (!fused_router(s) &&
      (encode_tmap_bf16(&pr.prob[0].tmA, w_router, (uint64_t)E, (uint64_t)d,
                        (uint32_t)pr.prob[0].a_box_rows) != 0 ||
       encode_tokens(pr.prob[0], x, T, d) != 0))
    return -1;

  TcParams& pg = pl.gateup;
  geometry_gateup(s, pg);
  pg.err = status;
  pg.prob[0].out = h;
  pg.prob[0].seg_off = offsets;
  pg.prob[0].ntp = ntp2;  // gate/up tiles the segments with its own n-tile cap
  // gathering: routed rows x[sorted_token[r]] (the fused dispatch) through a one-row box map
  // of x; else tiles of the permuted copy xs
  pg.prob[0].gidx = sorted;
  if (encode_tmap_bf16(&pg.prob[0].tmA, w_gate_up, (uint64_t)E * 2 * F, (uint64_t)d, 64) != 0 ||
      (pg.gather ? encode_tmap_bf16(&pg.prob[0].tmB[0], x, (uint64_t)T, (uint64_t)d, 1)
                 : encode_tokens(pg.prob[0], xs_y, R, d)) != 0)
    return -1;
  if (Fs > 0) {
    pg.prob[1].out = h_sh;
    pg.prob[1].gidx = nullptr;  // the shared expert reads every token in order
    if (encode_tmap_bf16(&pg.prob[1].tmA, sh->w_gate_up, (uint64_t)2 * Fs, (uint64_t)d, 64) != 0 ||
        (pg.gather ? encode_tmap_bf16(&pg.prob[1].tmB[0], x, (uint64_t)T, (uint64_t)d, 1)
                   : encode_tokens(pg.prob[1], x, T, d)) != 0)
      return -1;
  }

  TcParams& pd = pl.down;
  geometry_down(s, pd);
  pd.err = status;
  pd.prob[0].out = xs_y;
  pd.prob[0].seg_off = offsets;
  pd.prob[0].ntp = ntp;  // the down GEMM's own tile-unit prefix
  if (encode_tmap_bf16(&pd.prob[0].tmA, w_down, (uint64_t)E * d, (uint64_t)F, 64) != 0 ||
      encode_tokens(pd.prob[0], h, R, F) != 0)
    return -1;
  if (Fs > 0) {
    pd.prob[1].out = xs_y;
    if (encode_tmap_bf16(&pd.prob[1].tmA, sh->w_down, (uint64_t)d, (uint64_t)Fs, 64) != 0 ||
        encode_tokens(pd.prob[1], h_sh, T, Fs) != 0)
      return -1;
  }
  return 0;
}

int check_forward_args(const moe_shape* s, const void* x, const void* w_router,
                       const void* w_gate_up, const void* w_down, int score_fn, const float* bias,
                       const moe_shared_expert* sh, const void* out, const int* expert_counts,
                       const void* workspace, size_t workspace_bytes, const int* topk_idx_out,
                       const float* topk_w_out, const int* sorted_token_out) {
  int rc = check_shape(s, false);
  if (rc != MOE_OK) return rc;
  if (!x || !w_router || !w_gate_up || !w_down || !out || !expert_counts || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (s->Fs > 0 && (sh == nullptr || sh->w_gate_up == nullptr || sh->w_down == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (s->Fs == 0 && sh != nullptr) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w_router, w_gate_up, w_down, out, expert_counts, workspace, bias,
                        topk_idx_out, topk_w_out, sorted_token_out,
                        sh ? sh->w_gate_up : nullptr, sh ? sh->w_down : nullptr};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < layout_of(*s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int forward_impl(const moe_shape* s, const void* x, const void* w_router, const void* w_gate_up,
                 const void* w_down, int score_fn, const float* bias,
                 const moe_shared_expert* sh, void* out, int* expert_counts, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream, int* topk_idx_out,
                 float* topk_w_out, int* sorted_token_out, const moe_forward_opts* opts) {
  int rc = check_forward_args(s, x, w_router, w_gate_up, w_down, score_fn, bias, sh, out,
                              expert_counts, workspace, workspace_bytes, topk_idx_out, topk_w_out,
                              sorted_token_out);
  if (rc != MOE_OK) return rc;
  const int n_groups = opts ? opts->n_groups : 0, topk_groups = opts ? opts->topk_groups : 0;
  rc = check_groups(*s, n_groups, topk_groups);
  if (rc != MOE_OK) return rc;
  const int capacity = capacity_of(*s, opts ? opts->capacity_factor : 0.0);
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  // rerouting: `reroute` candidates beyond the top-k, only with a capacity
  const int reroute = opts ? opts->reroute : 0;
  if (reroute < 0 || (reroute > 0 && capacity == INT_MAX) || s->k + reroute > kMaxK ||
      s->k + reroute > s->E)
    return MOE_ERR_INVALID_ARG;
  // under group-limited routing every candidate comes from the kept groups
  if (reroute > 0 && n_groups > 0 && s->k + reroute > topk_groups * (s->E / n_groups))
    return MOE_ERR_INVALID_ARG;
  const int kc = reroute > 0 ? s->k + reroute : 0;
  int* dropped = opts ? opts->dropped : nullptr;
  if (dropped != nullptr && !aligned16(dropped)) return MOE_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const moe_shape& S = *s;
  const Layout L = layout_of(S);
  char* ws = static_cast<char*>(workspace);
  const bool bf16 = S.dtype == MOE_DTYPE_BF16;
  const int R = S.T * S.k;
  const int tsh = S.Fs > 0 ? S.T : 0;
  int* status = reinterpret_cast<int*>(ws + L.status);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  int* tidx = topk_idx_out ? topk_idx_out : reinterpret_cast<int*>(ws + L.topk_idx);
  float* tw = topk_w_out ? topk_w_out : reinterpret_cast<float*>(ws + L.topk_w);
  int* chunk = reinterpret_cast<int*>(ws + L.chunk);
  int* offsets = reinterpret_cast<int*>(ws + L.offsets);
  int* ntp = reinterpret_cast<int*>(ws + L.ntp);
  int* ntp2 = reinterpret_cast<int*>(ws + L.ntp2);
  int* sorted = sorted_token_out ? sorted_token_out : reinterpret_cast<int*>(ws + L.sorted);
  int* slot = reinterpret_cast<int*>(ws + L.slot);
  int* cand = reinterpret_cast<int*>(ws + L.cand);
  float* cand_val = reinterpret_cast<float*>(ws + L.cand_val);
  // the router writes candidates when rerouting, else the top-k and its weights
  int* ridx = kc > 0 ? cand : tidx;
  float* rw = kc > 0 ? cand_val : tw;
  void* xs_y = ws + L.xs_y;

  Plan pl;
  RouterParams rp;
  const bool fused = fused_router(S);
  int bn = expert_bn(S);
  if (bf16) {
    if (plan_bf16(S, x, w_router, w_gate_up, w_down, sh, ws, L, sorted, sms, pl) != 0) return MOE_ERR_CUDA;
    if ((!fused && pl.router.stages_a < 2) || pl.gateup.stages_a < 2 || pl.down.stages_a < 2)
      return MOE_ERR_UNSUPPORTED;
  }
  if (fused) {
    memset(&rp, 0, sizeof(rp));
    if (router_tc_plan(S.T, S.d, S.E, sms, kRouterPartialRows, rp) != 0) return MOE_ERR_UNSUPPORTED;
    if (encode_tmap_bf16(&rp.tmA, w_router, (uint64_t)S.E, (uint64_t)S.d, 128) != 0 ||
        encode_tmap_bf16(&rp.tmB, x, (uint64_t)S.T, (uint64_t)S.d, (uint32_t)(rp.N / 2)) != 0)
      return MOE_ERR_CUDA;
    rp.bias = bias;
    rp.topk_idx = ridx;
    rp.topk_w = rw;
    rp.kc = kc;
    rp.partial = reinterpret_cast<float*>(ws + L.partial);
    rp.counters = status + kCounterOffset / sizeof(int);
    rp.err = status;
    rp.k = S.k;
    rp.G = n_groups;
    rp.M = topk_groups;
  }
  cudaEvent_t* ev = opts ? opts->stage_events : nullptr;
  auto mark = [&](int i) -> bool { return ev == nullptr || cudaEventRecord(ev[i], stream) == cudaSuccess; };
  cudaError_t err = cudaSuccess;
#define MOE_TRY(expr)                 \
  do {                                \
    err = (expr);                     \
    if (err != cudaSuccess) return cuda_failed(err); \
  } while (0)

  if (!mark(0)) return MOE_ERR_CUDA;
  // the status word, the kernels' clock records and the fused router's arrival counters
  MOE_TRY(cudaMemsetAsync(status, 0, kCounterOffset + kCounterInts * sizeof(int), stream));
  if (fused) {
    // gate GEMM, score, top-k and renormalisation in one kernel: no logits in HBM
    MOE_TRY(launch_router_tc(score_fn == MOE_SCORE_SOFTMAX ? 0 : 1, rp, stream));
    if (!mark(1) || !mark(2)) return MOE_ERR_CUDA;
  } else {
    if (bf16) MOE_TRY(launch_gemm_tc(kModeRouter, pl.router, sms, stream));
    else MOE_TRY(launch_router_logits_f32(static_cast<const float*>(x), static_cast<const float*>(w_router),
                                          S.T, S.d, S.E, logits, stream));
    if (!mark(1)) return MOE_ERR_CUDA;
    MOE_TRY(launch_topk(score_fn == MOE_SCORE_SOFTMAX ? 0 : 1, logits, nullptr, bias, S.T, S.E, S.k,
                        n_groups, topk_groups, ridx, rw, stream, kc));
    if (!mark(2)) return MOE_ERR_CUDA;
  }
  if (kc > 0)  // rerouting rounds: the serving expert of every slot and the served weights
    MOE_TRY(launch_reroute(cand, cand_val, S.T, S.k, kc, S.E, capacity,
                           score_fn == MOE_SCORE_SOFTMAX ? 0 : 1, chunk,
                           reinterpret_cast<int*>(ws + L.prop), reinterpret_cast<int*>(ws + L.assign_c),
                           reinterpret_cast<int*>(ws + L.next_c), reinterpret_cast<int*>(ws + L.fill),
                           reinterpret_cast<int*>(ws + L.left), tidx, tw, dropped, stream));
  MOE_TRY(launch_dispatch(tidx, S.T, S.k, S.E, bf16 ? down_bn(S) : bn, bf16 ? down_tall_rows(S) : 0,
                          chunk, expert_counts, offsets, ntp,
                          bf16 ? gateup_bn(S) : 0, bf16 ? gateup_tall_rows(S) : 0,
                          bf16 ? ntp2 : nullptr, kc > 0 ? INT_MAX : capacity,
                          kc > 0 ? nullptr : dropped, sorted, slot, stream));
  if (!mark(3)) return MOE_ERR_CUDA;
  // a gathering gate/up GEMM reads x through the permutation itself; otherwise (and for the
  // fp32 expert FFN) the permuted copy xs is written first
  if (!bf16 || !gateup_gathers(S))
    MOE_TRY(launch_gather(x, sorted, R, capacity == INT_MAX ? nullptr : offsets + S.E, S.d,
                          bf16 ? 2 : 4, xs_y, stream));
  if (!mark(4)) return MOE_ERR_CUDA;
  if (bf16) {
    MOE_TRY(launch_gemm_tc(kModeGateUp, pl.gateup, sms, stream));
    if (!mark(5)) return MOE_ERR_CUDA;
    MOE_TRY(launch_gemm_tc(kModeDown, pl.down, sms, stream));
  } else {
    MOE_TRY(launch_ffn_f32(static_cast<const float*>(xs_y), static_cast<const float*>(x), offsets,
                           S.E, R, tsh, S.d, S.F, S.Fs, static_cast<const float*>(w_gate_up),
                           static_cast<const float*>(w_down),
                           sh ? static_cast<const float*>(sh->w_gate_up) : nullptr,
                           sh ? static_cast<const float*>(sh->w_down) : nullptr,
                           reinterpret_cast<float*>(ws + L.h), reinterpret_cast<float*>(ws + L.h_sh),
                           nullptr, stream, 0));
    if (!mark(5)) return MOE_ERR_CUDA;
    MOE_TRY(launch_ffn_f32(nullptr, nullptr, offsets, S.E, R, tsh, S.d, S.F, S.Fs, nullptr,
                           static_cast<const float*>(w_down), nullptr,
                           sh ? static_cast<const float*>(sh->w_down) : nullptr,
                           reinterpret_cast<float*>(ws + L.h), reinterpret_cast<float*>(ws + L.h_sh),
                           static_cast<float*>(xs_y), stream, 1));
  }
  if (!mark(6)) return MOE_ERR_CUDA;
  MOE_TRY(launch_combine(xs_y, slot, tw, S.T, S.k, S.d, R, S.Fs > 0 ? 1 : 0, bf16 ? 1 : 0, out, stream));
  if (!mark(7)) return MOE_ERR_CUDA;
#undef MOE_TRY
  return MOE_OK;
}

int route_from_keys_impl(const moe_shape* s, const float* sel_key, const float* gate_score, int n_groups,
                         int topk_groups, int* topk_idx, float* topk_w, int* expert_counts,
                         int* expert_offsets, int* sorted_token, int* slot_pos, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_shape(s, true);
  if (rc != MOE_OK) return rc;
  rc = check_groups(*s, n_groups, topk_groups);
  if (rc != MOE_OK) return rc;
  const void* ptrs[] = {sel_key, gate_score, topk_idx, topk_w, expert_counts, expert_offsets,
                        sorted_token, slot_pos, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  // only the layout's leading tables (they depend on T, E and k alone) are used here
  moe_shape r = *s;
  r.d = 64;
  r.F = 64;
  r.Fs = 0;
  r.dtype = MOE_DTYPE_F32;
  const Layout L = layout_of(r);
  if (workspace_bytes < L.ntp + align256((size_t)(s->E + 1) * 4)) return MOE_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = launch_topk(2, sel_key, gate_score, nullptr, s->T, s->E, s->k, n_groups,
                              topk_groups, topk_idx, topk_w, stream);
  if (e == cudaSuccess)
    e = launch_dispatch(topk_idx, s->T, s->k, s->E, 256, 0, reinterpret_cast<int*>(ws + L.chunk),
                        expert_counts, expert_offsets, reinterpret_cast<int*>(ws + L.ntp), 0, 0,
                        nullptr, INT_MAX, nullptr, sorted_token, slot_pos, stream);
  return e == cudaSuccess ? MOE_OK : cuda_failed(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_layer_workspace_size(const moe_shape* s) {
  if (check_shape(s, false) != MOE_OK) return 0;
  return layout_of(*s).total;
}

int moe_layer_forward(const moe_shape* s, const void* x, const void* w_router,
                      const void* w_gate_up, const void* w_down, moe_score_fn score_fn,
                      const float* bias, const moe_shared_expert* shared_expert, void* out,
                      int* expert_counts, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream, int* topk_idx_out, float* topk_w_out,
                      int* sorted_token_out) {
  return forward_impl(s, x, w_router, w_gate_up, w_down, (int)score_fn, bias, shared_expert, out,
                      expert_counts, workspace, workspace_bytes, stream, topk_idx_out, topk_w_out,
                      sorted_token_out, nullptr);
}

int moe_layer_forward_ex(const moe_shape* s, const void* x, const void* w_router,
                         const void* w_gate_up, const void* w_down, moe_score_fn score_fn,
                         const float* bias, const moe_shared_expert* shared_expert, void* out,
                         int* expert_counts, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream, int* topk_idx_out, float* topk_w_out,
                         int* sorted_token_out, const moe_forward_opts* opts) {
  if (opts != nullptr && opts->stage_events != nullptr)
    for (int i = 0; i < MOE_NUM_STAGE_EVENTS; ++i)
      if (opts->stage_events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  return forward_impl(s, x, w_router, w_gate_up, w_down, (int)score_fn, bias, shared_expert, out,
                      expert_counts, workspace, workspace_bytes, stream, topk_idx_out, topk_w_out,
                      sorted_token_out, opts);
}

int moe_route_from_keys(const moe_shape* s, const float* sel_key, const float* gate_score,
                        int* topk_idx, float* topk_w, int* expert_counts, int* expert_offsets,
                        int* sorted_token, int* slot_pos, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return route_from_keys_impl(s, sel_key, gate_score, 0, 0, topk_idx, topk_w, expert_counts,
                              expert_offsets, sorted_token, slot_pos, workspace, workspace_bytes,
                              stream);
}

int moe_route_from_keys_grouped(const moe_shape* s, const float* sel_key,
                                const float* gate_score, int n_groups, int topk_groups,
                                int* topk_idx, float* topk_w, int* expert_counts,
                                int* expert_offsets, int* sorted_token, int* slot_pos,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (n_groups < 1) return MOE_ERR_INVALID_ARG;
  return route_from_keys_impl(s, sel_key, gate_score, n_groups, topk_groups, topk_idx, topk_w,
                              expert_counts, expert_offsets, sorted_token, slot_pos, workspace,
                              workspace_bytes, stream);
}

int moe_debug_gemm_tiles(const moe_shape* s, int which, int num_sms, const int* expert_counts,
                         int* tiles, int max_tiles, int* geometry) {
  if (check_shape(s, false) != MOE_OK || s->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (which < 0 || which > 2 || num_sms < 1) return MOE_ERR_INVALID_ARG;
  if (which > 0 && expert_counts == nullptr) return MOE_ERR_INVALID_ARG;
  TcParams p;
  if (which == 0) geometry_router(*s, num_sms, p);
  else if (which == 1) geometry_gateup(*s, p);
  else geometry_down(*s, p);
  int* seg = nullptr;
  int* ntp = nullptr;
  int tiles0;
  if (which > 0) {
    seg = new int[s->E + 1];
    ntp = new int[s->E + 1];
    seg[0] = 0;
    ntp[0] = 0;
    for (int e = 0; e < s->E; ++e) {
      if (expert_counts[e] < 0) {
        delete[] seg;
        delete[] ntp;
        return MOE_ERR_INVALID_ARG;
      }
      seg[e + 1] = seg[e] + expert_counts[e];
      ntp[e + 1] = ntp[e] + seg_units(expert_counts[e], p.bn, p.prob[0].tall_rows);
    }
    p.prob[0].seg_off = seg;
    p.prob[0].ntp = ntp;
    tiles0 = ntp[s->E] * tiles_per_unit(p.prob[0]);
  } else {
    tiles0 = p.prob[0].nt * p.prob[0].m_tiles;
  }
  const int total = tiles0 + (p.n_prob > 1 ? p.prob[1].nt * p.prob[1].m_tiles : 0);
  // one row per CTA tile: a pair's scheduled tile is two CTA tiles (the second one only when
  // it is inside the weight rows), exactly as the kernel's epilogue decides
  int n = 0;
  for (int t = 0; t < total; ++t) {
    Tile tl;
    decode_tile(p, seg, ntp, tiles0, t, tl);
    const TcProblem& P = p.prob[tl.prob];
    for (int x = 0; x < (tl.tall ? 2 : 1) * p.cg; ++x) {
      const int mp = tl.tall ? 2 * tl.m + x / p.cg : tl.m;  // scheduled m-tile
      const int r = x % p.cg;
      const int mc = p.cg == 2 ? 2 * mp + r : mp;
      if (mc >= P.m_cta) continue;
      if (tiles != nullptr && n < max_tiles) {
        int* o = tiles + 7 * (size_t)n;
        o[0] = tl.prob;
        o[1] = tl.seg;
        o[2] = mc;
        o[3] = tl.row0;
        o[4] = tl.ncols;
        o[5] = tl.valid;
        o[6] = a_has_box1(P, mc) ? 1 : 0;
      }
      ++n;
    }
  }
  if (geometry) {
    geometry[0] = p.bn;
    geometry[1] = p.stages_a;
    geometry[2] = p.stages_b;
    geometry[3] = (int)gemm_tc_smem_bytes(p);
    geometry[4] = p.prob[0].m_cta;
    geometry[5] = p.n_prob > 1 ? p.prob[1].m_cta : 0;
    geometry[6] = p.prob[0].group;
    geometry[7] = p.prob[0].K;
    geometry[8] = p.cg;
  }
  delete[] seg;
  delete[] ntp;
  return n;
}

int moe_debug_unclustered_pair(void* workspace, cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  int* status = static_cast<int*>(workspace);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = launch_pair_unclustered(status, stream);
  return e == cudaSuccess ? MOE_OK : cuda_failed(e);
}

int moe_debug_wait_timeout(void* workspace, unsigned long long limit_ns, cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  if (limit_ns < 1000ull || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  int* status = static_cast<int*>(workspace);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = launch_wait_timeout(status, limit_ns, stream);
  return e == cudaSuccess ? MOE_OK : cuda_failed(e);
}

int moe_layer_num_launches(const moe_shape* s) {
  if (check_shape(s, false) != MOE_OK) return -1;
  // router (fused with the top-k on bf16 layers of up to 256 experts, else a GEMM and a top-k
  // kernel), 3 dispatch kernels, [row gather], gate/up, down, combine: the row gather runs
  // unless the gate/up GEMM gathers its token rows itself
  const bool bf16 = s->dtype == MOE_DTYPE_BF16;
  return (fused_router(*s) ? 1 : 2) + 3 + (bf16 && gateup_gathers(*s) ? 0 : 1) + 3;
}

int moe_workspace_status(const void* workspace, int* status, int* detail) {
  if (workspace == nullptr || status == nullptr) return MOE_ERR_INVALID_ARG;
  int code = 0;
  if (cudaMemcpy(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  *status = code == 0 ? MOE_OK : MOE_ERR_DEVICE;
  if (detail) *detail = code;
  return MOE_OK;
}

int moe_workspace_kernel_clocks(const void* workspace, double* report) {
  if (workspace == nullptr || report == nullptr) return MOE_ERR_INVALID_ARG;
  long long r[12];
  if (cudaMemcpy(r, static_cast<const char*>(workspace) + kClockOffset, sizeof(r),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int k = 0; k < 3; ++k) {
    const long long dc = r[4 * k + 2] - r[4 * k], dt = r[4 * k + 3] - r[4 * k + 1];
    const bool valid = dc > 0 && dt > 0 && dt < 100000000000ll;
    report[2 * k] = valid ? static_cast<double>(dc) / static_cast<double>(dt) * 1e3 : 0.0;
    report[2 * k + 1] = valid ? static_cast<double>(dt) * 1e-6 : 0.0;
  }
  return MOE_OK;
}

const char* moe_last_cuda_error_name(void) { return cudaGetErrorName(t_last_cuda_error); }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or tensor-map error";
    case MOE_ERR_DEVICE: return "a kernel gave up on an internal wait";
    default: return "unknown status";
  }
}

}  // extern "C"
