"""Load arithmetic of the library (host code) against the numbers the pages work out:

* "Tensor vs Expert vs Data Parallelism for MoE Serving", section "Why sparsity demands a large
  batch": top-8 of 256 experts gives batch / 32 rows per expert (8 at a batch of 256, 64 at
  2,048) -- tests/golden/sparsity_batch_example.json;
* the same page, section "A back-of-envelope sizing helper": 128 decode tokens per GPU give
  about 32 rows per expert at EP8, 128 at EP32 and 576 at EP144, where each GPU holds 2 expert
  slots (32 redundant experts above EP8) -- tests/golden/sizing_helper_example.json;
* "Expert-Parallel MoE Inference: Serving Sparse Models at Scale", section "A capacity and
  throughput worked example": 512 tokens, top-8 of 256 experts over 16 GPUs give 16 rows per
  expert and 256 per GPU under even routing, and a busiest GPU at 1.6x the mean receives about
  410 -- tests/golden/capacity_worked_example.json.
"""
import json
import os

import numpy as np
import pytest

import mixture_experts_layer_83_b300 as moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    return json.load(open(os.path.join(GOLDEN, name)))


def test_tokens_per_expert_follow_the_sparsity_example():
    g = _golden("sparsity_batch_example.json")
    for row in g["expected"]:
        _, tpe = moe.moe_load_expectation(row["batch"], g["n_experts"], g["top_k"])
        assert tpe == row["tokens_per_expert"]


def test_sizing_helper_example():
    g = _golden("sizing_helper_example.json")
    for row in g["expected"]:
        slots, tpe = moe.moe_load_expectation(g["tokens_per_rank"], g["n_experts"], g["top_k"],
                                              row["ep"], row["redundant"])
        assert tpe == row["tokens_per_expert"]
        if "expert_slots_per_gpu" in row:
            assert slots == row["expert_slots_per_gpu"]
        assert slots == (g["n_experts"] + row["redundant"]) / row["ep"]


def test_load_report_on_the_capacity_worked_example():
    """Even routing of the worked example: every expert 16 rows, every 16-expert group 256;
    then one GPU made the busiest at 1.6x the mean: the report gives 1.6 and its load 410."""
    g = _golden("capacity_worked_example.json")
    E, ep, exp = g["n_experts"], g["ep_size"], g["expected"]
    even = np.full(E, exp["tokens_per_expert_uniform"], np.int32)
    r = moe.moe_load_report(even, ep)
    assert r["mean_rows_per_expert"] == exp["tokens_per_expert_uniform"]
    assert r["expert_max_over_mean"] == 1.0 and r["group_max_over_mean"] == 1.0
    assert r["experts_touched"] == E
    assert r["mean_rows_per_expert"] * E / ep == exp["token_experts_per_gpu_uniform"]
    # move rows from the other GPUs to GPU 0 until it holds 1.6x the mean (the total stays T*k)
    per = E // ep
    skew = even.copy()
    extra = int(round((exp["busiest_gpu_skew"] - 1.0) * exp["token_experts_per_gpu_uniform"]))
    skew[:per] += extra // per
    skew[:extra % per] += 1
    take = extra
    for e in range(E - 1, per - 1, -1):
        t = min(take, 1)
        skew[e] -= t
        take -= t
        if take == 0:
            break
    assert skew.sum() == g["tokens"] * g["top_k"]
    r = moe.moe_load_report(skew, ep)
    assert skew[:per].sum() == exp["busiest_gpu_token_experts_approx"]
    assert r["group_max_over_mean"] == pytest.approx(
        exp["busiest_gpu_token_experts_approx"] / exp["token_experts_per_gpu_uniform"])
    assert round(r["group_max_over_mean"], 2) == pytest.approx(exp["busiest_gpu_skew"], abs=0.01)


def test_load_report_hand_case_and_errors():
    r = moe.moe_load_report([0, 4, 2, 2, 0, 0], 2)   # groups [0,4,2] and [2,0,0]
    assert r == {"mean_rows_per_expert": 8 / 6, "expert_max_over_mean": 4 / (8 / 6),
                 "group_max_over_mean": 6 / 4, "experts_touched": 3}
    with pytest.raises(moe.MoeError):
        moe.moe_load_report([1, 2, 3], 2)
    with pytest.raises(moe.MoeError):
        moe.moe_load_report([1, -2], 1)
    with pytest.raises(moe.MoeError):
        moe.moe_load_expectation(128, 8, 9)
