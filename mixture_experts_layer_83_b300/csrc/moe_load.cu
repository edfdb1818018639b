// Load arithmetic of an MoE layer (host code, launches nothing).
//
// Expected load under uniform routing, page "Tensor vs Expert vs Data Parallelism for MoE
// Serving": section "Why sparsity demands a large batch" (top-k of E experts sends a batch of B
// tokens B * k / E rows per expert on average) and section "A back-of-envelope sizing helper"
// (with expert parallelism over G GPUs, each holding an equal share of E + redundant expert
// slots, every GPU contributes its tokens to the global batch, so an expert sees
// tokens_per_gpu * G * k / E rows per step).
//
// Measured load, page "MoE Expert Parallelism in Practice", section "Common Misconceptions"
// (per-expert token counts are a metric to watch) and page "Expert-Parallel MoE Inference:
// Serving Sparse Models at Scale", section "A capacity and throughput worked example" (the
// busiest GPU's load over the mean): max over mean of the per-expert counts and of the
// per-group sums, groups being contiguous blocks of experts (an expert-parallel placement).
#include "../../include/moe_layer.h"

extern "C" int moe_load_expectation(int tokens_per_gpu, int E, int k, int n_gpus,
                                    int n_redundant, double* slots_per_gpu,
                                    double* tokens_per_expert) {
  if (tokens_per_gpu < 0 || E < 1 || k < 1 || k > E || n_gpus < 1 || n_redundant < 0)
    return MOE_ERR_INVALID_ARG;
  if (slots_per_gpu == nullptr || tokens_per_expert == nullptr) return MOE_ERR_INVALID_ARG;
  *slots_per_gpu = (static_cast<double>(E) + n_redundant) / n_gpus;
  *tokens_per_expert = static_cast<double>(tokens_per_gpu) * n_gpus * k / E;
  return MOE_OK;
}

extern "C" int moe_load_report(const int* expert_counts, int E, int n_groups, double* report) {
  if (expert_counts == nullptr || report == nullptr || E < 1 || n_groups < 1 ||
      E % n_groups != 0)
    return MOE_ERR_INVALID_ARG;
  long long total = 0, max_e = 0, max_g = 0, group = 0;
  int touched = 0;
  const int per = E / n_groups;
  for (int e = 0; e < E; ++e) {
    const long long c = expert_counts[e];
    if (c < 0) return MOE_ERR_INVALID_ARG;
    total += c;
    touched += c > 0 ? 1 : 0;
    max_e = c > max_e ? c : max_e;
    group += c;
    if ((e + 1) % per == 0) {
      max_g = group > max_g ? group : max_g;
      group = 0;
    }
  }
  const double mean_e = static_cast<double>(total) / E;
  const double mean_g = static_cast<double>(total) / n_groups;
  report[0] = mean_e;
  report[1] = total > 0 ? max_e / mean_e : 0.0;
  report[2] = total > 0 ? max_g / mean_g : 0.0;
  report[3] = touched;
  return MOE_OK;
}
