/* moe_oracle.c -- TEST INFRASTRUCTURE ONLY: plain fp64 reference of one MoE FFN layer.
 * The definitions and their sources are listed in moe_oracle.h.  No blocking, no fusion, no
 * reordering: each function is the textbook loop of the step it names. */
#include "moe_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

double oracle_elem(const void* base, int dtype, size_t i) {
  if (dtype == ORACLE_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

/* Linear gate followed by the score function.  Page "Expert-Parallel MoE Inference",
 * section "Deeper Analysis": a tiny linear gate scores every expert for every token and a
 * softmax is applied.  Sigmoid scoring with a selection-only bias is the alternative the
 * layer specification adds for the DeepSeek-V3-shaped workloads. */
int oracle_router_scores(int n_tok, int d, int E, int dtype, const void* x_rows,
                         const void* w_router, int score_fn, const float* bias,
                         double* logits, double* score, double* key) {
  if (n_tok < 0 || d < 1 || E < 1 || !x_rows || !w_router) return -1;
  if (score_fn != ORACLE_SOFTMAX && score_fn != ORACLE_SIGMOID) return -1;
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  double* s = (double*)malloc(sizeof(double) * (size_t)E);
  if (!l || !s) { free(l); free(s); return -1; }
  for (int t = 0; t < n_tok; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += oracle_elem(x_rows, dtype, (size_t)t * d + i) *
               oracle_elem(w_router, dtype, (size_t)e * d + i);
      l[e] = acc;
    }
    if (score_fn == ORACLE_SOFTMAX) {
      double mx = l[0];
      for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
      double den = 0.0;
      for (int e = 0; e < E; ++e) den += exp(l[e] - mx);
      for (int e = 0; e < E; ++e) s[e] = exp(l[e] - mx) / den;
    } else {
      for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-l[e]));
    }
    for (int e = 0; e < E; ++e) {
      size_t o = (size_t)t * E + e;
      if (logits) logits[o] = l[e];
      if (score) score[o] = s[e];
      if (key) {
        /* softmax is monotone in the logit, so the logit itself orders the experts */
        double base = score_fn == ORACLE_SOFTMAX ? l[e] : s[e];
        key[o] = base + (bias ? (double)bias[e] : 0.0);
      }
    }
  }
  free(l);
  free(s);
  return 0;
}

/* Keep the top-k experts (page "Expert-Parallel MoE Inference", "Deeper Analysis"), then
 * renormalise the kept scores to sum to one.  Selection: k times, take the unselected expert
 * with the largest key; among equal keys the lower id. */
int oracle_topk(int n_tok, int E, int k, const double* key, const double* score,
                int* topk_idx, double* topk_w, double* margin) {
  if (n_tok < 0 || E < 1 || k < 1 || k > E || !key || !topk_idx) return -1;
  if (topk_w && !score) return -1;
  char* taken = (char*)malloc((size_t)E);
  if (!taken) return -1;
  for (int t = 0; t < n_tok; ++t) {
    const double* kr = key + (size_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || kr[e] > kr[best]) best = e;  /* strict: equal keys keep the lower id */
      }
      taken[best] = 1;
      topk_idx[(size_t)t * k + j] = best;
    }
    if (margin) {
      int next = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (next < 0 || kr[e] > kr[next])) next = e;
      margin[t] = next < 0 ? INFINITY : kr[topk_idx[(size_t)t * k + k - 1]] - kr[next];
    }
    if (topk_w) {
      const double* sr = score + (size_t)t * E;
      double den = 0.0;
      for (int j = 0; j < k; ++j) den += sr[topk_idx[(size_t)t * k + j]];
      for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = sr[topk_idx[(size_t)t * k + j]] / den;
    }
  }
  free(taken);
  return 0;
}

/* Group-limited (node-limited) top-k.  Page "Expert-Parallel MoE Inference: Serving Sparse
 * Models at Scale", section "Load imbalance and how to fight it": node-limited routing caps how
 * many nodes (groups of experts) a token's experts may span.  The experts form n_groups
 * contiguous groups of E / n_groups.  The pages do not say how a group is scored; the reading
 * taken here: a group's score is the largest key among its experts.  The topk_groups groups
 * with the largest scores are kept (equal scores: the lower group id), then the top-k is taken
 * as in oracle_topk over the experts of the kept groups only, and renormalised the same way. */
int oracle_topk_grouped(int n_tok, int E, int k, int n_groups, int topk_groups,
                        const double* key, const double* score, int* topk_idx, double* topk_w,
                        double* margin) {
  if (n_tok < 0 || E < 1 || k < 1 || k > E || !key || !topk_idx) return -1;
  if (n_groups < 1 || E % n_groups != 0 || topk_groups < 1 || topk_groups > n_groups) return -1;
  const int gsize = E / n_groups;
  if (topk_groups * gsize < k) return -1;
  if (topk_w && !score) return -1;
  char* taken = (char*)malloc((size_t)E);
  char* allowed = (char*)malloc((size_t)E);
  char* gsel = (char*)malloc((size_t)n_groups);
  double* gscore = (double*)malloc(sizeof(double) * (size_t)n_groups);
  if (!taken || !allowed || !gsel || !gscore) {
    free(taken); free(allowed); free(gsel); free(gscore);
    return -1;
  }
  for (int t = 0; t < n_tok; ++t) {
    const double* kr = key + (size_t)t * E;
    /* group scores: the best key of each group */
    for (int g = 0; g < n_groups; ++g) {
      double best = kr[g * gsize];
      for (int i = 1; i < gsize; ++i)
        if (kr[g * gsize + i] > best) best = kr[g * gsize + i];
      gscore[g] = best;
    }
    /* keep topk_groups groups: each time the unkept group with the largest score */
    memset(gsel, 0, (size_t)n_groups);
    int last_kept = -1;
    for (int r = 0; r < topk_groups; ++r) {
      int bg = -1;
      for (int g = 0; g < n_groups; ++g) {
        if (gsel[g]) continue;
        if (bg < 0 || gscore[g] > gscore[bg]) bg = g;
      }
      gsel[bg] = 1;
      last_kept = bg;
    }
    double gmargin = INFINITY;
    for (int g = 0; g < n_groups; ++g)
      if (!gsel[g] && gscore[last_kept] - gscore[g] < gmargin) gmargin = gscore[last_kept] - gscore[g];
    for (int e = 0; e < E; ++e) allowed[e] = gsel[e / gsize];
    /* top-k over the allowed experts */
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (!allowed[e] || taken[e]) continue;
        if (best < 0 || kr[e] > kr[best]) best = e;
      }
      taken[best] = 1;
      topk_idx[(size_t)t * k + j] = best;
    }
    if (margin) {
      int next = -1;
      for (int e = 0; e < E; ++e)
        if (allowed[e] && !taken[e] && (next < 0 || kr[e] > kr[next])) next = e;
      const double emargin = next < 0 ? INFINITY : kr[topk_idx[(size_t)t * k + k - 1]] - kr[next];
      margin[t] = emargin < gmargin ? emargin : gmargin;
    }
    if (topk_w) {
      const double* sr = score + (size_t)t * E;
      double den = 0.0;
      for (int j = 0; j < k; ++j) den += sr[topk_idx[(size_t)t * k + j]];
      for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = sr[topk_idx[(size_t)t * k + j]] / den;
    }
  }
  free(taken);
  free(allowed);
  free(gsel);
  free(gscore);
  return 0;
}

/* Group the (token, slot) assignments by expert, token order preserved within an expert:
 * the single-GPU form of the dispatch all-to-all (page "Expert-Parallel MoE Inference",
 * "The all-to-all dispatch and combine, step by step"; page "MoE Expert Parallelism in
 * Practice", "Core Principles" part 1, "dispatch tokens to selected experts"). */
int oracle_dispatch(int T, int E, int k, const int* topk_idx, int* counts, int* offsets,
                    int* sorted_token, int* slot_pos) {
  if (T < 0 || E < 1 || k < 1 || !topk_idx || !counts || !offsets) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (size_t i = 0; i < (size_t)T * k; ++i) {
    int e = topk_idx[i];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  if (sorted_token || slot_pos) {
    int p = 0;
    for (int e = 0; e < E; ++e)
      for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j)
          if (topk_idx[(size_t)t * k + j] == e) {
            if (sorted_token) sorted_token[p] = t;
            if (slot_pos) slot_pos[(size_t)t * k + j] = p;
            ++p;
          }
  }
  return 0;
}

/* Expert capacity (page "Expert-Parallel MoE Inference: Serving Sparse Models at Scale",
 * section "Capacity factor and token dropping"): capacity = capacity_factor * (tokens * k /
 * experts) slots per expert, rounded up to a whole slot (the pages do not say how a fractional
 * capacity is rounded; up keeps at least the average load).  Each routed token checks whether
 * its expert still has a free slot: tokens claim slots in token order, the first `capacity`
 * assignments of an expert are dispatched and the rest are dropped (they skip the FFN).
 * counts[e] = dispatched assignments of e, offsets its exclusive prefix sum, sorted_token the
 * dispatched tokens expert by expert in token order, slot_pos[t][j] their positions or -1 when
 * dropped; *dropped = number of dropped assignments. */
int oracle_capacity(int T, int E, int k, double capacity_factor) {
  if (T < 0 || E < 1 || k < 1 || !(capacity_factor > 0.0)) return -1;
  return (int)ceil(capacity_factor * ((double)T * (double)k / (double)E));
}

int oracle_dispatch_capacity(int T, int E, int k, const int* topk_idx, int capacity,
                             int* counts, int* offsets, int* sorted_token, int* slot_pos,
                             int* dropped) {
  if (T < 0 || E < 1 || k < 1 || capacity < 0 || !topk_idx || !counts || !offsets) return -1;
  for (size_t i = 0; i < (size_t)T * k; ++i)
    if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;
  int ndrop = 0, p = 0;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    int claimed = 0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[(size_t)t * k + j] == e) {
          if (claimed < capacity) {
            if (sorted_token) sorted_token[p] = t;
            if (slot_pos) slot_pos[(size_t)t * k + j] = p;
            ++p;
            ++claimed;
          } else {
            if (slot_pos) slot_pos[(size_t)t * k + j] = -1;
            ++ndrop;
          }
        }
    counts[e] = claimed;
    offsets[e + 1] = offsets[e] + claimed;
  }
  if (dropped) *dropped = ndrop;
  return 0;
}

/* Capacity with rerouting (same page and section: overflow tokens are dropped or rerouted to
 * their next-best expert).  The pages give no procedure; the reading taken here runs in rounds.
 * Each token t has kc candidates cand[t][0..kc-1], its experts in selection order (its top-kc).
 * In round 0 slot j of every token proposes candidate j (its top-k).  In a round, proposals are
 * taken in token order (then slot order) and an expert accepts a proposal while it holds fewer
 * than `capacity` accepted slots.  After the round, each rejected slot of a token (in slot
 * order) takes the token's next unused candidate and proposes it in the next round; a slot
 * with no candidate left is dropped.  Rounds continue while a slot proposes.
 * assign[t][j] = the serving expert or -1 (dropped), assign_cand[t][j] = its candidate index or
 * -1; counts / offsets / sorted_token / slot_pos are the dispatch tables of the final
 * assignment (per expert, its tokens in ascending order); *dropped = dropped slots. */
int oracle_dispatch_reroute(int T, int E, int k, int kc, const int* cand, int capacity,
                            int* assign, int* assign_cand, int* counts, int* offsets,
                            int* sorted_token, int* slot_pos, int* dropped) {
  if (T < 0 || E < 1 || k < 1 || kc < k || kc > E || capacity < 0 || !cand || !assign ||
      !counts || !offsets)
    return -1;
  for (size_t i = 0; i < (size_t)T * kc; ++i)
    if (cand[i] < 0 || cand[i] >= E) return -1;
  const size_t R = (size_t)T * k;
  int* fill = (int*)calloc((size_t)E, sizeof(int));
  int* prop = (int*)malloc(R * sizeof(int));    /* proposing candidate index, -1 = none */
  int* rejected = (int*)malloc(R * sizeof(int));
  int* next = (int*)malloc((size_t)(T > 0 ? T : 1) * sizeof(int));
  if (!fill || !prop || !rejected || !next) {
    free(fill); free(prop); free(rejected); free(next);
    return -1;
  }
  for (int t = 0; t < T; ++t) {
    next[t] = k;
    for (int j = 0; j < k; ++j) {
      prop[(size_t)t * k + j] = j;
      assign[(size_t)t * k + j] = -1;
      if (assign_cand) assign_cand[(size_t)t * k + j] = -1;
    }
  }
  int proposing = T * k > 0;
  while (proposing) {
    for (size_t i = 0; i < R; ++i) rejected[i] = 0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        const size_t i = (size_t)t * k + j;
        if (prop[i] < 0) continue;
        const int e = cand[(size_t)t * kc + prop[i]];
        if (fill[e] < capacity) {
          ++fill[e];
          assign[i] = e;
          if (assign_cand) assign_cand[i] = prop[i];
        } else {
          rejected[i] = 1;
        }
        prop[i] = -1;
      }
    proposing = 0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        const size_t i = (size_t)t * k + j;
        if (!rejected[i] || next[t] >= kc) continue;
        prop[i] = next[t]++;
        proposing = 1;
      }
  }
  int ndrop = 0, p = 0;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    int n = 0;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (assign[(size_t)t * k + j] == e) {
          if (sorted_token) sorted_token[p] = t;
          if (slot_pos) slot_pos[(size_t)t * k + j] = p;
          ++p;
          ++n;
        }
    counts[e] = n;
    offsets[e + 1] = offsets[e] + n;
  }
  for (size_t i = 0; i < R; ++i)
    if (assign[i] < 0) {
      if (slot_pos) slot_pos[i] = -1;
      ++ndrop;
    }
  if (dropped) *dropped = ndrop;
  free(fill); free(prop); free(rejected); free(next);
  return 0;
}

/* Gate weights renormalised over the experts that serve each token (the renormalisation of the
 * top-k weights with the served experts in place of the top-k): w[t][j] = score[t][assign] /
 * sum over the token's served slots, 0 for a dropped slot. */
int oracle_served_weights(int T, int E, int k, const double* score, const int* assign, double* w) {
  if (T < 0 || E < 1 || k < 1 || !score || !assign || !w) return -1;
  for (int t = 0; t < T; ++t) {
    double den = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = assign[(size_t)t * k + j];
      if (e >= 0) den += score[(size_t)t * E + e];
    }
    for (int j = 0; j < k; ++j) {
      const int e = assign[(size_t)t * k + j];
      w[(size_t)t * k + j] = e >= 0 ? score[(size_t)t * E + e] / den : 0.0;
    }
  }
  return 0;
}

int oracle_gather(int R, int d, const int* sorted_token, const double* x, double* xs) {
  if (R < 0 || d < 1 || !sorted_token || !x || !xs) return -1;
  for (int p = 0; p < R; ++p)
    for (int c = 0; c < d; ++c) xs[(size_t)p * d + c] = x[(size_t)sorted_token[p] * d + c];
  return 0;
}

/* Weighted sum of the k expert outputs back in token order (page "Expert-Parallel MoE
 * Inference", "Deeper Analysis"; page "MoE Expert Parallelism in Practice", "Core
 * Principles" part 1, combine and map back to the original token order). */
int oracle_combine(int T, int k, int d, const int* slot_pos, const double* topk_w,
                   const double* ys, const double* y_shared, double* out) {
  if (T < 0 || k < 1 || d < 1 || !slot_pos || !topk_w || !ys || !out) return -1;
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        const int p = slot_pos[(size_t)t * k + j];
        if (p < 0) continue;  /* an assignment dropped at capacity contributes nothing */
        acc += topk_w[(size_t)t * k + j] * ys[(size_t)p * d + c];
      }
      if (y_shared) acc += y_shared[(size_t)t * d + c];
      out[(size_t)t * d + c] = acc;
    }
  return 0;
}

/* One expert: SwiGLU feed-forward block. */
int oracle_swiglu_ffn(int d, int F, int dtype, const double* xrow, const void* w_gate_up,
                      const void* w_down, double* y) {
  if (d < 1 || F < 1 || !xrow || !w_gate_up || !w_down || !y) return -1;
  double* h = (double*)malloc(sizeof(double) * (size_t)F);
  if (!h) return -1;
  for (int f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      g += xrow[i] * oracle_elem(w_gate_up, dtype, (size_t)f * d + i);
      u += xrow[i] * oracle_elem(w_gate_up, dtype, (size_t)(F + f) * d + i);
    }
    h[f] = g / (1.0 + exp(-g)) * u;
  }
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int f = 0; f < F; ++f) acc += h[f] * oracle_elem(w_down, dtype, (size_t)c * F + f);
    y[c] = acc;
  }
  free(h);
  return 0;
}

/* out[t] = sum_j w_tj FFN_{S_tj}(x_t) + FFN_shared(x_t), shared expert with weight 1
 * (page "Tensor vs Expert vs Data Parallelism for MoE Serving", "Context and Background":
 * routed experts plus a shared expert). */
int oracle_layer_rows(const oracle_layer* L, int n_tok, const void* x_rows, const int* topk_idx,
                      const double* topk_w, double* out) {
  if (!L || n_tok < 0 || !x_rows || !topk_idx || !topk_w || !out) return -1;
  if (L->d < 1 || L->E < 1 || L->k < 1 || L->k > L->E || L->F < 1 || L->Fs < 0) return -1;
  if (!L->w_gate_up || !L->w_down) return -1;
  if (L->Fs > 0 && (!L->sh_gate_up || !L->sh_down)) return -1;
  const int d = L->d;
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  if (!xr || !y) { free(xr); free(y); return -1; }
  int rc = 0;
  for (int t = 0; t < n_tok && rc == 0; ++t) {
    for (int i = 0; i < d; ++i) xr[i] = oracle_elem(x_rows, L->dtype, (size_t)t * d + i);
    double* o = out + (size_t)t * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j = 0; j < L->k; ++j) {
      int e = topk_idx[(size_t)t * L->k + j];
      if (e < 0 || e >= L->E) { rc = -1; break; }
      if (!L->w_gate_up[e] || !L->w_down[e]) { rc = -2; break; }
      oracle_swiglu_ffn(d, L->F, L->dtype, xr, L->w_gate_up[e], L->w_down[e], y);
      double w = topk_w[(size_t)t * L->k + j];
      for (int c = 0; c < d; ++c) o[c] += w * y[c];
    }
    if (rc == 0 && L->Fs > 0) {
      oracle_swiglu_ffn(d, L->Fs, L->dtype, xr, L->sh_gate_up, L->sh_down, y);
      for (int c = 0; c < d; ++c) o[c] += y[c];
    }
  }
  free(xr);
  free(y);
  return rc;
}

/* Expert placement with redundant experts (page "Expert-Parallel MoE Inference: Serving Sparse
 * Models at Scale", section "Load imbalance and how to fight it": redundant experts duplicate
 * the hottest experts so their load spreads; EPLB computes an expert-to-GPU placement that
 * equalises expected load).  The pages give the goal, not the algorithm; the plain reading:
 *   1. every expert has one replica; each of the n_redundant extra slots goes, one at a time, to
 *      the expert with the largest load per replica (equal: the lower expert id); a replica
 *      carries load / replicas;
 *   2. replicas are placed largest first (equal loads: lower expert id, then lower replica
 *      index), each on the GPU with the smallest load among those with a free slot and no
 *      replica of the same expert (if every GPU with a free slot already holds one, among all
 *      GPUs with a free slot); equal loads: the lower GPU id.  Each GPU has
 *      (E + n_redundant) / n_gpus slots.
 * slot_expert / slot_gpu [E + n_redundant]: slot s of GPU g is g * slots_per_gpu + (its order of
 * placement on g); gpu_load [n_gpus]. */
int oracle_eplb_plan(const int* load, int E, int n_gpus, int n_redundant, int* slot_expert,
                     int* slot_gpu, double* gpu_load) {
  if (!load || E < 1 || n_gpus < 1 || n_redundant < 0 || !slot_expert || !slot_gpu || !gpu_load)
    return -1;
  const int S = E + n_redundant;
  if (S % n_gpus != 0) return -1;
  const int per_gpu = S / n_gpus;
  int* rep = (int*)calloc((size_t)E, sizeof(int));
  int* item_e = (int*)malloc(sizeof(int) * (size_t)S);
  int* item_r = (int*)malloc(sizeof(int) * (size_t)S);
  char* used = (char*)calloc((size_t)S, 1);
  int* filled = (int*)calloc((size_t)n_gpus, sizeof(int));
  char* hosts = (char*)calloc((size_t)n_gpus * (size_t)E, 1);
  if (!rep || !item_e || !item_r || !used || !filled || !hosts) {
    free(rep); free(item_e); free(item_r); free(used); free(filled); free(hosts);
    return -1;
  }
  for (int e = 0; e < E; ++e) {
    if (load[e] < 0) { free(rep); free(item_e); free(item_r); free(used); free(filled); free(hosts); return -1; }
    rep[e] = 1;
  }
  for (int r = 0; r < n_redundant; ++r) {
    int best = 0;
    for (int e = 1; e < E; ++e)
      if ((double)load[e] / rep[e] > (double)load[best] / rep[best]) best = e;
    rep[best] += 1;
  }
  int n = 0;
  for (int e = 0; e < E; ++e)
    for (int r = 0; r < rep[e]; ++r) {
      item_e[n] = e;
      item_r[n] = r;
      ++n;
    }
  for (int g = 0; g < n_gpus; ++g) gpu_load[g] = 0.0;
  for (int placed = 0; placed < S; ++placed) {
    /* next item: the largest unplaced replica load; ties: lower expert, then lower replica */
    int it = -1;
    for (int i = 0; i < S; ++i) {
      if (used[i]) continue;
      if (it < 0) { it = i; continue; }
      const double li = (double)load[item_e[i]] / rep[item_e[i]];
      const double lt = (double)load[item_e[it]] / rep[item_e[it]];
      if (li > lt || (li == lt && (item_e[i] < item_e[it] ||
                                   (item_e[i] == item_e[it] && item_r[i] < item_r[it]))))
        it = i;
    }
    used[it] = 1;
    const int e = item_e[it];
    int g_best = -1;
    for (int pass = 0; pass < 2 && g_best < 0; ++pass)
      for (int g = 0; g < n_gpus; ++g) {
        if (filled[g] == per_gpu) continue;
        if (pass == 0 && hosts[(size_t)g * E + e]) continue;
        if (g_best < 0 || gpu_load[g] < gpu_load[g_best]) g_best = g;
      }
    const int slot = g_best * per_gpu + filled[g_best];
    slot_expert[slot] = e;
    slot_gpu[slot] = g_best;
    filled[g_best] += 1;
    hosts[(size_t)g_best * E + e] = 1;
    gpu_load[g_best] += (double)load[e] / rep[e];
  }
  free(rep); free(item_e); free(item_r); free(used); free(filled); free(hosts);
  return 0;
}
