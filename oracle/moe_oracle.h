/* moe_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, single-threaded, fp64 CPU reference of the forward pass of one sparse
 * Mixture-of-Experts FFN layer.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the product library never does, and this header shares
 * nothing with the CUDA path.
 *
 * What it computes (every sum in fp64, inputs converted exactly from fp32 / bf16):
 *   logits l[t][e] = sum_i x[t][i] * w_router[e][i]
 *   softmax: score = softmax over all E logits, key = logit (+ bias[e] if given)
 *   sigmoid: score = 1 / (1 + exp(-l)),        key = score (+ bias[e] if given)
 *   S_t = the k largest keys (ties -> lower expert id), in key-descending order
 *   w_tj = score[S_tj] / sum_j' score[S_tj']
 *   FFN_e(x) = W_down[e] (silu(W_gate[e] x) * (W_up[e] x)),  silu(g) = g / (1 + exp(-g))
 *   out[t] = sum_j w_tj FFN_{S_tj}(x_t) + FFN_shared(x_t)
 *
 * Sources (web pages on expert-parallel MoE serving):
 *   - "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section "Deeper
 *     Analysis: Routing, Balance, and a Capacity Worked Example": a linear gate scores every
 *     expert per token, a softmax is applied, the top-k are kept, and the k expert outputs are
 *     combined weighted by the gate scores.
 *   - "MoE Expert Parallelism in Practice", "Core Principles" part 1: router -> top-k ->
 *     dispatch -> expert FFN -> combine, mapped back to the original token order.
 *   - "Tensor vs Expert vs Data Parallelism for MoE Serving", "Context and Background":
 *     routed experts plus one shared expert, top-8.
 * Readings not fixed by the pages (renormalisation over the selected k, sigmoid scoring with
 * a selection-only bias, SwiGLU experts, lower-id tie-break, shared expert weight 1) follow
 * the layer specification the tests are written against.
 *
 * Conventions: dtype 0 = fp32 elements, 1 = bf16 elements (uint16 bit patterns).  All
 * arrays are row-major and owned by the caller.  Functions return 0 on success, -1 on an
 * invalid argument, -2 when a needed expert's weights were not supplied.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_SOFTMAX = 0, ORACLE_SIGMOID = 1 };

/* Stored element i of an fp32 / bf16 array as an exact double. */
double oracle_elem(const void* base, int dtype, size_t i);

/* Router logits, gate scores and selection keys for n_tok token rows.
 * x_rows [n_tok][d], w_router [E][d]; bias [E] fp32 or NULL (= 0): selection only.
 * logits, score, key: [n_tok][E] fp64, any may be NULL. */
int oracle_router_scores(int n_tok, int d, int E, int dtype, const void* x_rows,
                         const void* w_router, int score_fn, const float* bias,
                         double* logits, double* score, double* key);

/* Top-k selection and renormalisation for n_tok rows of keys/scores [n_tok][E].
 * topk_idx [n_tok][k] (key descending, ties -> lower id), topk_w [n_tok][k],
 * margin [n_tok] = k-th key minus (k+1)-th key (+inf when k == E); topk_w / margin may be NULL. */
int oracle_topk(int n_tok, int E, int k, const double* key, const double* score,
                int* topk_idx, double* topk_w, double* margin);

/* Group-limited top-k: experts in n_groups contiguous groups of E / n_groups; a group's score
 * is its largest key; the topk_groups best groups are kept (ties -> lower group id); the top-k
 * and renormalisation of oracle_topk then run over the kept groups' experts only.
 * margin [n_tok] = min(topk_groups-th group score minus the next group's, k-th key minus the
 * (k+1)-th key among the kept experts), +inf where there is no next. */
int oracle_topk_grouped(int n_tok, int E, int k, int n_groups, int topk_groups,
                        const double* key, const double* score, int* topk_idx, double* topk_w,
                        double* margin);

/* Dispatch tables of a routing (topk_idx [T][k]):
 *   counts[e] = number of tokens routed to e; offsets = exclusive prefix sum (E+1 entries);
 *   sorted_token[R] (R = T*k): for e = 0..E-1, the tokens routed to e in ascending order;
 *   slot_pos[T][k]: position of (t, j) in sorted_token. */
int oracle_dispatch(int T, int E, int k, const int* topk_idx, int* counts, int* offsets,
                    int* sorted_token, int* slot_pos);

/* Expert capacity: ceil(capacity_factor * T * k / E) (capacity_factor > 0), or -1. */
int oracle_capacity(int T, int E, int k, double capacity_factor);

/* Dispatch with an expert capacity: per expert, the first `capacity` assignments in token
 * order are dispatched and the rest dropped.  counts [E] = dispatched per expert, offsets
 * [E+1], sorted_token [dispatched total], slot_pos [T][k] = position or -1 (dropped),
 * *dropped = dropped assignments (any output except counts / offsets may be NULL). */
/* Capacity with rerouting of overflow to the next-best expert (rounds; see moe_oracle.c):
 * cand [T][kc] = each token's experts in selection order (kc >= k); outputs the serving expert
 * and candidate index of every slot (-1: dropped) and the dispatch tables of that assignment. */
int oracle_dispatch_reroute(int T, int E, int k, int kc, const int* cand, int capacity,
                            int* assign, int* assign_cand, int* counts, int* offsets,
                            int* sorted_token, int* slot_pos, int* dropped);

/* Weights renormalised over each token's serving experts (0 for a dropped slot). */
int oracle_served_weights(int T, int E, int k, const double* score, const int* assign, double* w);

int oracle_dispatch_capacity(int T, int E, int k, const int* topk_idx, int capacity,
                             int* counts, int* offsets, int* sorted_token, int* slot_pos,
                             int* dropped);

/* xs[p] = x[sorted_token[p]] for p < R (fp64 rows of width d). */
int oracle_gather(int R, int d, const int* sorted_token, const double* x, double* xs);

/* out[t] = sum_j topk_w[t][j] * ys[slot_pos[t][j]] (+ y_shared[t] if not NULL); a slot_pos
 * of -1 (an assignment dropped at capacity) contributes nothing. */
int oracle_combine(int T, int k, int d, const int* slot_pos, const double* topk_w,
                   const double* ys, const double* y_shared, double* out);

/* One SwiGLU expert on one fp64 row: w_gate_up [2F][d] (gate rows, then up rows),
 * w_down [d][F]; y [d]. */
int oracle_swiglu_ffn(int d, int F, int dtype, const double* xrow, const void* w_gate_up,
                      const void* w_down, double* y);

typedef struct {
  int d, E, k, F, Fs, dtype;
  const void* const* w_gate_up; /* [E] pointers to [2F][d]; an entry may be NULL if unused */
  const void* const* w_down;    /* [E] pointers to [d][F] */
  const void* sh_gate_up;       /* [2Fs][d] or NULL when Fs == 0 */
  const void* sh_down;          /* [d][Fs]  or NULL when Fs == 0 */
} oracle_layer;

/* Layer output rows for n_tok token rows x_rows [n_tok][d] under the given routing
 * (topk_idx [n_tok][k], topk_w [n_tok][k]); out [n_tok][d] fp64. */
int oracle_layer_rows(const oracle_layer* L, int n_tok, const void* x_rows, const int* topk_idx,
                      const double* topk_w, double* out);

/* Expert placement over n_gpus GPUs with n_redundant extra replicas of the hottest experts
 * (see moe_oracle.c): slot_expert / slot_gpu [E + n_redundant], gpu_load [n_gpus]. */
int oracle_eplb_plan(const int* load, int E, int n_gpus, int n_redundant, int* slot_expert,
                     int* slot_gpu, double* gpu_load);

#ifdef __cplusplus
}
#endif
#endif
