// Redundant-expert placement plan (host code, launches nothing).
//
// Pages "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section "Load imbalance
// and how to fight it" (extra copies of the hottest experts; a balancer that places experts on
// GPUs so the expected load evens out), and "Tensor vs Expert vs Data Parallelism for MoE
// Serving", section "Load imbalance and EPLB" (a pool of E + redundant expert slots; the balancer
// minimises the largest per-GPU receive load).  The pages give the goal, not the algorithm; this
// is the plain greedy reading of it, in two passes:
//   1. replication: each redundant slot goes to the expert whose load per replica is currently
//      the largest (equal: the lower expert id);
//   2. placement: replicas in decreasing order of load per replica (equal: lower expert id, then
//      lower replica) each go to the least-loaded GPU that still has a free slot and does not
//      already hold that expert, else to the least-loaded GPU with a free slot (equal load: the
//      lower GPU id).  A replica carries load[e] / replicas[e].
// Loads per replica are compared exactly (int64 cross products), so no rounding decides a
// choice in step 1 or in the order of step 2; GPU loads are double sums, accumulated in
// placement order.
#include <algorithm>
#include <cstdint>
#include <queue>
#include <set>
#include <utility>
#include <vector>

#include "../../include/moe_layer.h"

namespace {

// load_a / n_a > load_b / n_b, exactly (n > 0; int32 loads and counts, so the products fit).
inline bool per_replica_greater(int64_t load_a, int64_t n_a, int64_t load_b, int64_t n_b) {
  return load_a * n_b > load_b * n_a;
}

constexpr int kMaxSlots = 1 << 20;

}  // namespace

extern "C" int moe_eplb_plan(const int* expert_load, int E, int n_gpus, int n_redundant,
                             int* slot_expert, int* slot_gpu, double* gpu_load) {
  if (expert_load == nullptr || slot_expert == nullptr || slot_gpu == nullptr ||
      gpu_load == nullptr || E < 1 || n_gpus < 1 || n_redundant < 0 ||
      n_redundant > kMaxSlots - E || (E + n_redundant) % n_gpus != 0)
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e)
    if (expert_load[e] < 0) return MOE_ERR_INVALID_ARG;
  const int slots = E + n_redundant, per_gpu = slots / n_gpus;

  // 1. replication: a max-heap on (load per replica, -expert id)
  std::vector<int> reps(E, 1);
  auto heap_less = [&](int a, int b) {  // true when a ranks below b
    if (per_replica_greater(expert_load[b], reps[b], expert_load[a], reps[a])) return true;
    if (per_replica_greater(expert_load[a], reps[a], expert_load[b], reps[b])) return false;
    return a > b;
  };
  std::priority_queue<int, std::vector<int>, decltype(heap_less)> heap(heap_less);
  for (int e = 0; e < E; ++e) heap.push(e);
  for (int r = 0; r < n_redundant; ++r) {
    const int e = heap.top();
    heap.pop();
    ++reps[e];
    heap.push(e);
  }

  // 2. placement order: experts by load per replica, descending; an expert's replicas are
  //    consecutive (they carry equal load)
  std::vector<int> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (per_replica_greater(expert_load[a], reps[a], expert_load[b], reps[b])) return true;
    if (per_replica_greater(expert_load[b], reps[b], expert_load[a], reps[a])) return false;
    return a < b;
  });

  // GPUs with a free slot, ordered by (load, id)
  std::set<std::pair<double, int>> open;
  std::vector<int> filled(n_gpus, 0);
  for (int g = 0; g < n_gpus; ++g) {
    gpu_load[g] = 0.0;
    open.emplace(0.0, g);
  }
  std::vector<std::vector<int>> holders(E);  // GPUs holding a replica of expert e
  for (const int e : order) {
    const double share = (double)expert_load[e] / reps[e];
    for (int r = 0; r < reps[e]; ++r) {
      auto pick = open.begin();
      for (auto it = open.begin(); it != open.end(); ++it)
        if (std::find(holders[e].begin(), holders[e].end(), it->second) == holders[e].end()) {
          pick = it;
          break;
        }
      const int g = pick->second;
      open.erase(pick);
      const int slot = g * per_gpu + filled[g]++;
      slot_expert[slot] = e;
      slot_gpu[slot] = g;
      holders[e].push_back(g);
      gpu_load[g] += share;
      if (filled[g] < per_gpu) open.emplace(gpu_load[g], g);
    }
  }
  return MOE_OK;
}
