/* moe_layer.h -- C ABI of the B300 (sm_103a) forward pass of one sparse Mixture-of-Experts
 * FFN layer, single GPU.
 *
 * The operation (one layer, T tokens of width d, E routed experts, top-k):
 *   1. router: logits = x * w_router^T, then a score per expert: softmax over the E logits,
 *      or a sigmoid of each logit.  Page "Expert-Parallel MoE Inference: Serving Sparse Models
 *      at Scale", section "Deeper Analysis: Routing, Balance, and a Capacity Worked Example":
 *      a linear gate scores every expert for every token, a softmax is applied and the top-k
 *      are kept.  The sigmoid form with a per-expert selection bias is the auxiliary-loss-free
 *      balancing named on page "Expert Parallelism for MoE Serving", section "The Future of
 *      Expert Parallelism for MoE Serving".
 *   2. top-k: the k largest selection keys per token (key = logit for softmax, sigmoid score
 *      for sigmoid, plus bias[e] when a bias is given); equal keys go to the lower expert id;
 *      the k gate weights are the unbiased scores of the chosen experts, renormalised to sum
 *      to one.
 *   3. dispatch: assignments grouped by expert, token order kept within an expert -- the
 *      one-GPU form of the dispatch all-to-all (page "Expert-Parallel MoE Inference", section
 *      "The all-to-all dispatch and combine, step by step"; page "MoE Expert Parallelism in
 *      Practice", "Core Principles" part 1).
 *   4. experts: each routed expert is a SwiGLU FFN, W_down (silu(W_gate x) * (W_up x)), run as
 *      a grouped GEMM over the expert segments (page "Tensor vs Expert vs Data Parallelism for
 *      MoE Serving", Figure 2: experts run grouped GEMMs).  An optional shared expert of inner
 *      width Fs sees every token with weight 1 (same page, "Context and Background": routed
 *      experts plus a shared expert).
 *   5. combine: out[t] = sum_j w_tj * y_(t,j) + y_shared[t], summed in a fixed order with no
 *      floating-point atomics, so the output is bit-reproducible from run to run (page "MoE
 *      Expert Parallelism in Practice", "Core Principles" part 1: outputs are combined and
 *      mapped back to the original token order).
 * The layer is drop-free unless the caller sets an expert capacity (moe_forward_opts): every
 * assignment is computed (page "Expert-Parallel MoE Inference", "Capacity factor and token
 * dropping": production inference prefers a drop-free path).
 *
 * Conventions for every entry point:
 *   - Every array pointer is DEVICE memory owned by the caller, 16-byte aligned, row-major.
 *     The library allocates no memory, keeps no per-call state and takes no ownership.
 *   - All work is enqueued on `stream`; no call synchronises with the host (except
 *     moe_workspace_status, which says so), so a forward pass can be captured in a CUDA graph.
 *   - Errors are returned before anything is enqueued: MOE_ERR_INVALID_ARG for a null
 *     required pointer, misaligned pointer or out-of-range size; MOE_ERR_UNSUPPORTED for a
 *     shape the kernels do not handle; MOE_ERR_WORKSPACE for a workspace smaller than
 *     moe_layer_workspace_size().  MOE_ERR_CUDA reports a failed launch or tensor-map
 *     encode.  Kernels that time out on an internal wait record a code that
 *     moe_workspace_status() returns as MOE_ERR_DEVICE (the kernel returns instead of
 *     hanging).
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;
typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,
  MOE_ERR_UNSUPPORTED = -2,
  MOE_ERR_WORKSPACE = -3,
  MOE_ERR_CUDA = -4,
  MOE_ERR_DEVICE = -5
};

/* Limits: 1 <= k <= 32, k <= E <= 1024, T * k < 2^31.  For MOE_DTYPE_BF16 (tensor-core
 * path, fp32 accumulation): d, F and Fs must be multiples of 64.  MOE_DTYPE_F32 runs every
 * product in true fp32 (no TF32) on CUDA cores and has no shape restriction. */
typedef struct {
  int T;   /* tokens */
  int d;   /* hidden width */
  int E;   /* routed experts */
  int k;   /* experts per token */
  int F;   /* routed expert inner width */
  int Fs;  /* shared expert inner width, 0 = no shared expert */
  moe_dtype dtype; /* element type of x, all weights, out */
} moe_shape;

typedef struct {
  const void* w_gate_up; /* [2*Fs][d]: rows 0..Fs-1 gate, rows Fs..2Fs-1 up (K-major) */
  const void* w_down;    /* [d][Fs] */
} moe_shared_expert;

/* Bytes of device workspace moe_layer_forward and moe_route_from_keys need for this shape
 * (worst case: the pass is drop-free, so R = T*k routed rows always fit).  0 if the shape is
 * invalid. */
size_t moe_layer_workspace_size(const moe_shape* s);

/* One forward pass of the layer.
 *   x         [T][d]          dtype
 *   w_router  [E][d]          dtype; row e scores expert e
 *   w_gate_up [E][2F][d]      dtype; per expert F gate rows then F up rows (K-major)
 *   w_down    [E][d][F]       dtype (K-major)
 *   score_fn  MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID
 *   bias      [E] fp32 or NULL; added to the selection key only (never to the weights)
 *   shared_expert  NULL when s->Fs == 0, else both pointers set
 *   out       [T][d]          dtype, written
 *   expert_counts [E] int32, written: tokens routed to each expert
 *   workspace / workspace_bytes: at least moe_layer_workspace_size(s) bytes; its contents
 *             are scratch between calls; calls that overlap on the GPU must not share it
 *   topk_idx_out [T][k] int32, topk_w_out [T][k] fp32, sorted_token_out [T*k] int32: optional
 *             (NULL to skip) copies of the routing (key-descending order) and of the dispatch
 *             permutation (for each expert in id order, its tokens in ascending order).
 * Returns MOE_OK or a negative MOE_ERR_* (see the conventions above). */
int moe_layer_forward(const moe_shape* s, const void* x, const void* w_router,
                      const void* w_gate_up, const void* w_down, moe_score_fn score_fn,
                      const float* bias, const moe_shared_expert* shared_expert, void* out,
                      int* expert_counts, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream, int* topk_idx_out, float* topk_w_out,
                      int* sorted_token_out);

/* Number of CUDA events moe_layer_forward_ex records when stage_events is given:
 * [0] start, [1] router GEMM, [2] top-k, [3] histogram/scan/permutation, [4] gather (fp32
 * layers only; a bf16 layer's gate/up GEMM gathers its token rows itself, so [4] == [3]),
 * [5] gate/up grouped GEMM, [6] down grouped GEMM, [7] combine (each after its kernels). */
#define MOE_NUM_STAGE_EVENTS 8

typedef struct {
  cudaEvent_t* stage_events; /* NULL, or MOE_NUM_STAGE_EVENTS events created by the caller */
  /* Group-limited (node-limited) routing, page "Expert-Parallel MoE Inference: Serving Sparse
   * Models at Scale", section "Load imbalance and how to fight it": node-limited routing caps
   * how many nodes a token's experts may span.  The experts form n_groups contiguous groups of
   * E / n_groups (an expert-parallel placement); a group's score is its largest selection key;
   * the topk_groups best groups are kept (equal scores: the lower group id) and the top-k runs
   * over their experts only.  0 / 0: plain top-k.  Otherwise 1 <= n_groups <= 32, E divisible
   * by n_groups, 1 <= topk_groups <= n_groups and topk_groups * E / n_groups >= k, else
   * MOE_ERR_INVALID_ARG. */
  int n_groups;
  int topk_groups;
  /* Expert capacity (same page, section "Capacity factor and token dropping"): each expert
   * takes at most capacity = ceil(capacity_factor * T * k / E) assignments; tokens claim an
   * expert's slots in token order and an assignment beyond the capacity is dropped: it skips
   * the expert FFN and contributes nothing to its token's output (the token's other weights
   * are not renormalised; the layer output carries no residual).  expert_counts then counts
   * the dispatched assignments.  0: dropless.  Negative, NaN or infinite: MOE_ERR_INVALID_ARG.
   * A double, so that a factor written in decimal (0.8) gives the capacity of its exact value
   * where factor * T * k / E is a whole number (a float 0.8 would round it up by one). */
  double capacity_factor;
  int* dropped; /* NULL, or a device int (16-byte aligned) receiving the dropped assignments */
  /* Rerouting instead of dropping (same section: overflow tokens are rerouted to their
   * next-best expert); needs capacity_factor > 0.  reroute = the candidates each token may
   * take beyond its top-k (its next-best experts in selection order; k + reroute <= 32 and
   * <= E; with group-limited routing the candidates come from the kept groups only, and
   * k + reroute <= topk_groups * E / n_groups).  In round 0 every token's k slots propose
   * its top-k; an expert accepts proposals in token order while it has room; each rejected
   * slot takes its token's next unused candidate and proposes it in the next round; a slot
   * whose candidates run out is dropped.  The gate
   * weights are renormalised over the experts that serve the token.  topk_idx_out then holds
   * the serving expert of every slot (-1: dropped) and topk_w_out those weights.  0: drop. */
  int reroute;
} moe_forward_opts;

/* moe_layer_forward with options (stage timing events, group-limited routing); opts may be
 * NULL. */
int moe_layer_forward_ex(const moe_shape* s, const void* x, const void* w_router,
                         const void* w_gate_up, const void* w_down, moe_score_fn score_fn,
                         const float* bias, const moe_shared_expert* shared_expert, void* out,
                         int* expert_counts, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream, int* topk_idx_out, float* topk_w_out,
                         int* sorted_token_out, const moe_forward_opts* opts);

/* Routing and dispatch tables from supplied fp32 selection keys and gate scores (steps 2-3
 * above with the scores given instead of computed), for bit-exact checks:
 *   sel_key [T][E], gate_score [T][E] fp32
 *   topk_idx [T][k], topk_w [T][k] = gate_score of the chosen, renormalised
 *   expert_counts [E], expert_offsets [E+1] (exclusive prefix sum, last = T*k)
 *   sorted_token [T*k], slot_pos [T][k] (position of assignment (t, j) in sorted order).
 * s->d, s->F, s->Fs and s->dtype are ignored.  Returns MOE_OK or MOE_ERR_*. */
int moe_route_from_keys(const moe_shape* s, const float* sel_key, const float* gate_score,
                        int* topk_idx, float* topk_w, int* expert_counts, int* expert_offsets,
                        int* sorted_token, int* slot_pos, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* moe_route_from_keys with group-limited routing (n_groups >= 1, topk_groups as in
 * moe_forward_opts); same outputs, workspace and errors. */
int moe_route_from_keys_grouped(const moe_shape* s, const float* sel_key,
                                const float* gate_score, int n_groups, int topk_groups,
                                int* topk_idx, float* topk_w, int* expert_counts,
                                int* expert_offsets, int* sorted_token, int* slot_pos,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_route_from_keys for callers that cannot allocate device memory (an allocator they do
 * not own, a pool that is already carved up, a C host with no allocator wired in).  The
 * pages have no counterpart: this is a convenience of this library.  Same arguments and
 * results as moe_route_from_keys without the workspace: the dispatch histogram lives in a
 * fixed array of MOE_NOALLOC_SCRATCH_BYTES inside the library, held on every GPU that loads
 * the library until the process exits.  Shapes whose histogram ((T*k + 1023)/1024 chunks x E
 * int32) does not fit are rejected with MOE_ERR_WORKSPACE before anything is enqueued.
 * The first call on a device looks up the array's device address (with that device
 * current); make that first call before any stream capture.  The address belongs to the
 * device's context: after a device reset the next call looks it up again, so make that call
 * before any capture too.  Every call on a device shares
 * the array, so calls whose work overlaps on the GPU race and must be serialised by the
 * caller.  No memory is allocated or freed. */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
int moe_route_from_keys_noalloc(const moe_shape* s, const float* sel_key,
                                const float* gate_score, int* topk_idx, float* topk_w,
                                int* expert_counts, int* expert_offsets, int* sorted_token,
                                int* slot_pos, cudaStream_t stream);

/* Diagnostics, host only (launches nothing): the tile schedule the bf16 grouped GEMM `which`
 * (0 = router, 1 = gate/up, 2 = down) would run for the given per-expert token counts
 * (host array [E]; ignored for the router) on a device with num_sms SMs.  Writes up to
 * max_tiles rows of 7 ints, one per CTA tile, {operand set (0 routed / 1 shared), segment,
 * 128-row weight tile m, first token row, token columns N (a multiple of 16; over 256 they are
 * split across two MMAs), rows that belong to the segment, loads second 64-row weight box}
 * into tiles (host; may be NULL), and 9 ints {n-tile cap,
 * weight-ring stages, token-ring stages, shared-memory bytes per CTA, weight tiles of set 0,
 * weight tiles of set 1, m-group, K of set 0, CTAs per MMA (1, or 2 for a CTA pair)} into
 * geometry (host, may be NULL).  In the CTA-pair GEMMs (gate/up and down) the two CTAs of a
 * pair hold weight tiles 2j and 2j + 1 over the same token rows; the second is listed only
 * when it exists.  A tall tile (a segment short enough for one n-tile, on the wide pair form)
 * covers two scheduled weight tiles: its CTA tiles 4j .. 4j + 3 are listed in that order.
 * Returns the number of CTA tiles (may exceed max_tiles) or a negative MOE_ERR_*. */
int moe_debug_gemm_tiles(const moe_shape* s, int which, int num_sms, const int* expert_counts,
                         int* tiles, int max_tiles, int* geometry);

/* Diagnostics of the device error path (the pages' "fixed buffers fail loudly", page "Tensor vs
 * Expert vs Data Parallelism for MoE Serving", section "Trade-offs, Gotchas, and What Goes
 * Wrong": a failure must surface as an error, never as a hang).  Both clear the status word at
 * the start of `workspace` (the word moe_workspace_status reads), then enqueue on `stream` one
 * launch that ends by itself and leaves the GPU usable:
 *   moe_debug_unclustered_pair: the CTA-pair expert GEMM launched as two plain CTAs (no 2-CTA
 *     cluster); it records code 5 and returns before touching shared or tensor memory.
 *   moe_debug_wait_timeout: one CTA waits on an mbarrier that nothing completes, with a
 *     wall-clock limit of limit_ns (1e3 .. 1e9 ns, else MOE_ERR_INVALID_ARG); when the limit
 *     runs out it records code 6 and returns.
 * Afterwards moe_workspace_status gives MOE_ERR_DEVICE with that code as the detail.  Device
 * codes: 1 a producer's wait, 2 an MMA issuer's wait, 3 an epilogue's wait, 4 the final drain
 * of in-flight copies ran out (limit 2 s each); 5 a pair kernel without clusters; 6 the
 * diagnostic wait. */
int moe_debug_unclustered_pair(void* workspace, cudaStream_t stream);
int moe_debug_wait_timeout(void* workspace, unsigned long long limit_ns, cudaStream_t stream);

/* Redundant-expert placement plan, HOST code: every pointer is HOST memory, nothing is
 * enqueued.  Pages "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section
 * "Load imbalance and how to fight it", and "Tensor vs Expert vs Data Parallelism for MoE
 * Serving", section "Load imbalance and EPLB": copies of hot experts in n_redundant extra slots
 * and an expert-to-GPU placement that evens the expected per-GPU load.
 *   expert_load [E] int32 >= 0, e.g. expert_counts summed over recent steps
 *   slot_expert [E + n_redundant], slot_gpu [E + n_redundant]: written; slot i holds a replica
 *     of expert slot_expert[i] on GPU slot_gpu[i]; GPU g owns slots g*P .. g*P + P - 1,
 *     P = (E + n_redundant) / n_gpus, filled in placement order
 *   gpu_load [n_gpus] fp64: written; the expected load of each GPU, a replica of expert e
 *     carrying expert_load[e] / (replicas of e)
 * The plan: each redundant slot goes to the expert with the largest load per replica (equal:
 * lower id); replicas, largest load per replica first (equal: lower expert, lower replica), go
 * to the least-loaded GPU with a free slot that does not yet hold the expert, else to the
 * least-loaded GPU with a free slot (equal load: lower GPU id).  Every expert gets at least one
 * slot and every GPU exactly P.  MOE_ERR_INVALID_ARG for a null pointer, E < 1, n_gpus < 1,
 * n_redundant < 0, E + n_redundant > 2^20 or not a multiple of n_gpus, or a negative load. */
int moe_eplb_plan(const int* expert_load, int E, int n_gpus, int n_redundant, int* slot_expert,
                  int* slot_gpu, double* gpu_load);

/* Load arithmetic, HOST code (host pointers, nothing enqueued).
 * moe_load_expectation: expected rows per expert under uniform routing when n_gpus GPUs each
 *   bring tokens_per_gpu tokens to one expert-parallel group (page "Tensor vs Expert vs Data
 *   Parallelism for MoE Serving", sections "Why sparsity demands a large batch" and "A
 *   back-of-envelope sizing helper"): *tokens_per_expert = tokens_per_gpu * n_gpus * k / E and
 *   *slots_per_gpu = (E + n_redundant) / n_gpus.  n_gpus = 1 gives one GPU's batch * k / E.
 * moe_load_report: from expert_counts [E] (e.g. a forward pass's, copied to the host), with
 *   the experts in n_groups contiguous groups (an expert-parallel placement; E divisible by
 *   n_groups): report[0] = mean rows per expert, report[1] = max / mean over experts,
 *   report[2] = max / mean over groups (page "Expert-Parallel MoE Inference: Serving Sparse
 *   Models at Scale", section "A capacity and throughput worked example": the busiest GPU's
 *   load over the mean), report[3] = experts with at least one row.
 * Both return MOE_OK, or MOE_ERR_INVALID_ARG for a null pointer, a size out of range (k > E,
 * a negative count) or E not divisible by n_groups. */
int moe_load_expectation(int tokens_per_gpu, int E, int k, int n_gpus, int n_redundant,
                         double* slots_per_gpu, double* tokens_per_expert);
int moe_load_report(const int* expert_counts, int E, int n_groups, double* report);

/* Kernel launches one moe_layer_forward makes for this shape (for launch accounting), without
 * options: group-limited routing and a capacity launch the same kernels; rerouting adds four
 * launches per round (reroute + 1 rounds), one to set up and one to finish (and a memset of
 * the dropped-assignment counter when one is given). */
int moe_layer_num_launches(const moe_shape* s);

/* Reads the device status word of a workspace after the caller's work on it has finished:
 * SYNCHRONOUS (cudaMemcpy).  *status = MOE_OK, or MOE_ERR_DEVICE if a kernel gave up on an
 * internal wait; *detail = the raw code the kernel recorded (0 if none). */
int moe_workspace_status(const void* workspace, int* status, int* detail);

/* Clock record of the latest forward pass on a workspace, SYNCHRONOUS (cudaMemcpy), for
 * telling a kernel's work from the clock it ran at (a board at its power limit lowers the SM
 * clock, and a sampled clock reading need not show it).  CTA 0 of each tensor-core kernel of
 * a bf16 layer records its SM clock counter and the global timer when it starts and ends;
 * report[2 i] = SM clock in MHz over that span, report[2 i + 1] = the span in ms, for i = 0
 * router, 1 gate/up GEMM, 2 down GEMM (0, 0 where no record was written: the forward pass
 * clears the records first, and fp32 layers' kernels do not record). */
int moe_workspace_kernel_clocks(const void* workspace, double* report);

/* Name of the CUDA error (e.g. "cudaErrorInvalidConfiguration") behind the latest
 * MOE_ERR_CUDA a launch returned on the calling host thread, "cudaSuccess" if none. */
const char* moe_last_cuda_error_name(void);

/* Static string for a status code. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H */
