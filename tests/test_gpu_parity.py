"""GPU parity through the C ABI against the fp64 oracle, at sizes the oracle finishes in
seconds but that span several tiles and ragged tails, plus the degenerate cases."""
import numpy as np
import pytest

import moe_inputs
import oracle
from moe_inputs import configs
from moe_inputs.configs import SIGMOID, SOFTMAX, make_shape

from layer_check import check_dispatch, full_check, gpu_forward, to_host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_83_b300 as moe
    moe.lib()


SMALL = {
    # several m-tiles, ragged expert segments, shared expert, sigmoid + bias
    "bf16_sigmoid_shared": make_shape(300, 256, 16, 4, 192, Fs=128, score=SIGMOID,
                                      bias_range=0.01, seed=11),
    # d % 128 == 64: the down GEMM's last weight tile is half empty
    "bf16_softmax_half_tile": make_shape(517, 192, 8, 2, 320, seed=12),
    # 256 experts, ~6 rows each (decode-like segments), E not a multiple of 128 in the router
    "bf16_many_experts": make_shape(200, 128, 200, 8, 64, Fs=64, score=SIGMOID, bias_range=0.01,
                                    seed=13),
    # segments longer than the 256-row n-tile cap
    "bf16_long_segments": make_shape(600, 384, 4, 2, 256, seed=17),
    "bf16_single_expert": make_shape(77, 128, 1, 1, 128, seed=14),
    "bf16_k_equals_E": make_shape(40, 64, 6, 6, 64, seed=15),
    "bf16_single_token": make_shape(1, 256, 32, 4, 128, Fs=64, score=SIGMOID, bias_range=0.01,
                                    seed=16),
    "bf16_k32": make_shape(50, 128, 64, 32, 64, seed=19),
    "f32_tiny_config": configs.CONFIGS[0],
    "f32_ragged": make_shape(99, 70, 5, 2, 33, Fs=17, dtype="f32", score=SIGMOID, bias_range=0.05,
                             seed=18),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_matches_oracle(name):
    stats = full_check(SMALL[name])
    print(name, stats)


def test_hot_experts_and_many_empty_experts():
    """A large bias sends every token to experts 2 and 5: two segments of T rows each, all
    other segments empty."""
    cfg = make_shape(700, 128, 12, 2, 128, Fs=64, score=SIGMOID, bias_range=0.01, seed=21)
    host = moe_inputs.host_inputs(cfg)
    host["bias"] = host["bias"].copy()
    host["bias"][[2, 5]] = 5.0
    stats = full_check(cfg, host=host)
    assert stats["excluded"] == 0


def test_output_is_bit_reproducible():
    cfg = SMALL["bf16_sigmoid_shared"]
    dev = moe_inputs.upload(cfg, moe_inputs.host_inputs(cfg))
    a = to_host(gpu_forward(cfg, dev))
    b = to_host(gpu_forward(cfg, dev))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_workspace_status_is_clean_after_a_pass():
    import mixture_experts_layer_83_b300 as moe
    cfg = SMALL["bf16_many_experts"]
    dev = moe_inputs.upload(cfg, moe_inputs.host_inputs(cfg))
    res = gpu_forward(cfg, dev)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(res["workspace"]) == (moe.MOE_OK, 0)


# ------------------------------------------------------------------ bit-exact routing
def _oracle_keys(T, E, score, seed, ties):
    """fp32 selection keys and gate scores derived from oracle fp64 logits of synthetic rows."""
    cfg = make_shape(T, 64, E, 1, 64, score=score, bias_range=0.01 if score == SIGMOID else 0.0,
                     seed=seed)
    x = moe_inputs.host_tensor(cfg, "x")
    wr = moe_inputs.host_tensor(cfg, "w_router")
    lg, sc, _ = oracle.router_scores(x, wr, score)
    if score == SIGMOID:
        b = moe_inputs.host_tensor(cfg, "bias")
        key = sc.astype(np.float32) + b            # fp32 key = fp32(sigma) + b, in fp32
    else:
        key = lg.astype(np.float32)
    if ties:
        key = (np.round(key * 8) / 8).astype(np.float32)
    return np.ascontiguousarray(key, np.float32), np.ascontiguousarray(sc, np.float32)


@pytest.mark.parametrize("T,E,k,score,ties", [(1000, 256, 8, SIGMOID, False),
                                              (4096, 8, 2, SOFTMAX, True),
                                              (333, 1024, 32, SIGMOID, True),
                                              (2500, 128, 8, SOFTMAX, True),
                                              (64, 32, 32, SOFTMAX, False),
                                              (3000, 33, 5, SIGMOID, True),
                                              (1, 7, 3, SOFTMAX, True)])
def test_route_from_keys_is_bit_exact(T, E, k, score, ties):
    import mixture_experts_layer_83_b300 as moe
    key, sc = _oracle_keys(T, E, score, seed=T + E + k, ties=ties)
    o_idx, o_w, _ = oracle.topk(key.astype(np.float64), sc.astype(np.float64), k)
    o_counts, o_off, o_st, o_sp = oracle.dispatch(o_idx, E)
    dev = "cuda"
    kk, ss = torch.from_numpy(key).to(dev), torch.from_numpy(sc).to(dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    st = torch.empty(T * k, dtype=torch.int32, device=dev)
    sp = torch.empty((T, k), dtype=torch.int32, device=dev)
    shape = moe.make_shape(T, 64, E, k, 64)
    ws = torch.empty(moe.moe_layer_workspace_size(shape), dtype=torch.uint8, device=dev)
    moe.moe_route_from_keys(shape, kk, ss, idx, w, counts, off, st, sp, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    np.testing.assert_array_equal(counts.cpu().numpy(), o_counts)
    np.testing.assert_array_equal(off.cpu().numpy(), o_off)
    np.testing.assert_array_equal(st.cpu().numpy(), o_st)
    np.testing.assert_array_equal(sp.cpu().numpy(), o_sp)
    np.testing.assert_allclose(w.cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,k,G,M,score,ties", [(1000, 256, 8, 8, 4, SIGMOID, False),
                                                  (2500, 128, 8, 8, 4, SOFTMAX, True),
                                                  (700, 64, 6, 4, 2, SOFTMAX, True),
                                                  (300, 40, 5, 5, 2, SIGMOID, True),
                                                  (100, 32, 4, 32, 4, SOFTMAX, True),
                                                  (50, 24, 3, 8, 1, SIGMOID, True)])
def test_route_from_keys_grouped_is_bit_exact(T, E, k, G, M, score, ties):
    """Group-limited routing on oracle-supplied fp32 keys: top-k sets and order, counts,
    offsets, permutation and slot positions equal to the oracle's group-limited top-k."""
    import mixture_experts_layer_83_b300 as moe
    key, sc = _oracle_keys(T, E, score, seed=T + E + k + G, ties=ties)
    o_idx, o_w, _ = oracle.topk_grouped(key.astype(np.float64), sc.astype(np.float64), k, G, M)
    o_counts, o_off, o_st, o_sp = oracle.dispatch(o_idx, E)
    dev = "cuda"
    kk, ss = torch.from_numpy(key).to(dev), torch.from_numpy(sc).to(dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    st = torch.empty(T * k, dtype=torch.int32, device=dev)
    sp = torch.empty((T, k), dtype=torch.int32, device=dev)
    shape = moe.make_shape(T, 64, E, k, 64)
    ws = torch.empty(moe.moe_layer_workspace_size(shape), dtype=torch.uint8, device=dev)
    moe.moe_route_from_keys_grouped(shape, kk, ss, G, M, idx, w, counts, off, st, sp, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    np.testing.assert_array_equal(counts.cpu().numpy(), o_counts)
    np.testing.assert_array_equal(off.cpu().numpy(), o_off)
    np.testing.assert_array_equal(st.cpu().numpy(), o_st)
    np.testing.assert_array_equal(sp.cpu().numpy(), o_sp)
    np.testing.assert_allclose(w.cpu().numpy(), o_w, rtol=2e-6, atol=1e-7)


GROUPED = {
    # 64 experts in 8 groups, 3 kept: sigmoid + bias with a shared expert
    "bf16_sigmoid_groups": dict(make_shape(500, 256, 64, 8, 128, Fs=64, score=SIGMOID,
                                           bias_range=0.01, seed=31), groups=8, topk_groups=3),
    # softmax, 4 groups of 8, 2 kept
    "bf16_softmax_groups": dict(make_shape(400, 192, 32, 4, 192, seed=32), groups=4,
                                topk_groups=2),
    # one group kept: every token's experts come from a single group of 8
    "bf16_one_group": dict(make_shape(300, 128, 64, 4, 64, seed=33), groups=8, topk_groups=1),
}


CAPACITY = {
    # skewed by a large bias on two experts: they overflow a capacity of 1.0 x the mean load
    "bf16_capacity_1.0": dict(make_shape(400, 256, 16, 4, 192, Fs=64, score=SIGMOID,
                                         bias_range=0.01, seed=41), capacity_factor=1.0),
    # softmax, fractional capacity (300 * 2 / 7 * 1.25 = 107.1 -> 108 slots)
    "bf16_capacity_1.25": dict(make_shape(300, 192, 7, 2, 128, seed=42), capacity_factor=1.25),
    # a tiny capacity: most assignments dropped, some tokens lose every expert
    "bf16_capacity_tiny": dict(make_shape(200, 128, 8, 2, 64, seed=43), capacity_factor=0.05),
    # fp32 layer with drops
    "f32_capacity": dict(make_shape(99, 70, 5, 2, 33, Fs=17, dtype="f32", score=SIGMOID,
                                    bias_range=0.05, seed=44), capacity_factor=0.8),
    # group-limited routing and a capacity together
    "bf16_groups_and_capacity": dict(make_shape(500, 256, 64, 8, 128, Fs=64, score=SIGMOID,
                                                bias_range=0.01, seed=45), groups=8,
                                     topk_groups=3, capacity_factor=1.1),
}


@pytest.mark.parametrize("name", list(CAPACITY))
def test_capacity_layer_matches_oracle(name):
    cfg = CAPACITY[name]
    host = moe_inputs.host_inputs(cfg)
    if name == "bf16_capacity_1.0":
        host["bias"] = host["bias"].copy()
        host["bias"][[3, 11]] = 0.5     # two hot experts
    stats = full_check(cfg, host=host)
    print(name, stats)


@pytest.mark.parametrize("name", list(GROUPED))
def test_group_limited_layer_matches_oracle(name):
    stats = full_check(GROUPED[name])
    print(name, stats)


def test_forward_dispatch_tables_match_oracle_for_gpu_routing():
    cfg = SMALL["bf16_many_experts"]
    dev = moe_inputs.upload(cfg, moe_inputs.host_inputs(cfg))
    res = to_host(gpu_forward(cfg, dev))
    counts, _ = check_dispatch(cfg, res["topk_idx"], res["counts"], res["sorted_token"])
    assert counts.sum() == cfg["T"] * cfg["k"]


def test_kernel_clock_records():
    """After a bf16 forward pass the router, gate/up and down kernels have recorded a plausible
    SM clock and duration; an fp32 pass (CUDA-core kernels) records none."""
    import mixture_experts_layer_83_b300 as moe
    c = make_shape(T=256, d=256, E=16, k=4, F=128, Fs=64, dtype="bf16", score=SIGMOID,
                   bias_range=0.01, seed=11, name="clocks")
    res = gpu_forward(c, moe_inputs.upload(c, moe_inputs.host_inputs(c)))
    torch.cuda.synchronize()
    kc = moe.moe_workspace_kernel_clocks(res["workspace"])
    for name, (mhz, ms) in kc.items():
        assert 300 < mhz < 2500 and 0 < ms < 100, (name, mhz, ms)
    c32 = dict(c, dtype="f32", name="clocks-f32")
    res = gpu_forward(c32, moe_inputs.upload(c32, moe_inputs.host_inputs(c32)))
    torch.cuda.synchronize()
    assert all(v == (0.0, 0.0) for v in moe.moe_workspace_kernel_clocks(res["workspace"]).values())


@pytest.mark.parametrize("score,k,extra,cf,Fs,seed", [(SOFTMAX, 2, 2, 1.0, 0, 201),
                                                      (SIGMOID, 4, 4, 1.0, 64, 228),
                                                      (SOFTMAX, 1, 3, 1.0, 0, 201),
                                                      (SIGMOID, 2, 6, 0.75, 64, 228),
                                                      (SOFTMAX, 4, 2, 0.8, 64, 201)])
def test_reroute_matches_oracle(score, k, extra, cf, Fs, seed):
    """Rerouting at capacity, bit-exact against the oracle on the same inputs: the serving
    expert of every slot (-1: dropped), expert counts, the permutation and the number dropped;
    the served weights and the layer output within tolerance.  The inputs are such that no
    token has a near-tie (1e-4) within its top-(k + extra + 1) keys, so both sides see the same
    candidate order."""
    import mixture_experts_layer_83_b300 as moe
    c = make_shape(T=300, d=256, E=16, k=k, F=128, Fs=Fs, dtype="bf16", score=score,
                   bias_range=0.01 if score == SIGMOID else 0.0, seed=seed, name="reroute")
    c.update(capacity_factor=cf, reroute=extra)
    host = moe_inputs.host_inputs(c)
    res = to_host(gpu_forward(c, moe_inputs.upload(c, host)))
    _, sc, key = oracle.router_scores(host["x"], host["w_router"], c["score"], host.get("bias"))
    kc = k + extra
    cand, _, _ = oracle.topk(key, sc, kc)
    srt = -np.sort(-key, axis=1)[:, :kc + 1]
    assert np.min(srt[:, :-1] - srt[:, 1:]) >= 1e-4, "inputs with a near-tie: pick another seed"
    cap = oracle.capacity(c["T"], c["E"], k, cf)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, c["E"], cap)
    np.testing.assert_array_equal(res["topk_idx"], assign)
    np.testing.assert_array_equal(res["counts"], counts)
    np.testing.assert_array_equal(res["sorted_token"][:offsets[-1]], st)
    assert int(res["dropped"][0]) == dropped
    w = oracle.served_weights(sc, assign)
    np.testing.assert_allclose(res["topk_w"], w, rtol=0, atol=2e-5)
    experts = {e: (host["w_gate_up"][e], host["w_down"][e]) for e in range(c["E"])}
    shared = (host["sh_gate_up"], host["sh_down"]) if Fs > 0 else None
    from layer_check import check_output, oracle_rows
    ref = oracle_rows(c, host["x"], np.where(assign >= 0, assign, 0), w, experts, shared, 4)
    print(check_output(c, res["out"], ref), "rerouted+dropped:", dropped, "counts max", counts.max(), cap)


@pytest.mark.parametrize("T,E,k,extra,cf,seed", [(48, 32, 4, 28, 0.5, 501),
                                                  (64, 8, 2, 6, 0.9, 501)])
def test_reroute_at_the_candidate_limits(T, E, k, extra, cf, seed):
    """Rerouting with the most candidates the options allow: k + extra = 32 (the selection's
    limit, 28 rounds after the first) and k + extra = E (every expert a candidate); bit-exact
    against the oracle on inputs whose candidate keys have no near-tie."""
    c = make_shape(T=T, d=128, E=E, k=k, F=64, Fs=0, dtype="bf16", score=SOFTMAX, seed=seed,
                   name="reroute")
    c.update(capacity_factor=cf, reroute=extra)
    host = moe_inputs.host_inputs(c)
    res = to_host(gpu_forward(c, moe_inputs.upload(c, host)))
    _, sc, key = oracle.router_scores(host["x"], host["w_router"], c["score"], host.get("bias"))
    kc = k + extra
    srt = -np.sort(-key, axis=1)[:, :kc + 1]
    assert np.min(srt[:, :-1] - srt[:, 1:]) >= 1e-4, "inputs with a near-tie: pick another seed"
    cand, _, _ = oracle.topk(key, sc, kc)
    cap = oracle.capacity(T, E, k, cf)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, E, cap)
    assert ((assign >= 0) & (assign != cand[:, :k])).any(), "no slot was rerouted"
    np.testing.assert_array_equal(res["topk_idx"], assign)
    np.testing.assert_array_equal(res["counts"], counts)
    np.testing.assert_array_equal(res["sorted_token"][:offsets[-1]], st)
    assert int(res["dropped"][0]) == dropped
    np.testing.assert_allclose(res["topk_w"], oracle.served_weights(sc, assign), rtol=0, atol=2e-5)


@pytest.mark.parametrize("dtype,score,T,E,cf,seed", [("f32", SOFTMAX, 300, 16, 1.0, 402),
                                                      ("bf16", SOFTMAX, 96, 272, 0.5, 402),
                                                      ("bf16", SIGMOID, 96, 272, 0.5, 509)])
def test_reroute_unfused_router_matches_oracle(dtype, score, T, E, cf, seed):
    """Rerouting where the candidates come from the top-k kernel rather than the fused router:
    the fp32 layer (CUDA-core router GEMM) and a bf16 layer with more than 256 experts (the
    tensor-core router GEMM writes logits); top-2 with 2 more candidates, bit-exact against the
    oracle on inputs with no near-tie among each token's top-5 keys."""
    k, extra = 2, 2
    c = make_shape(T=T, d=128, E=E, k=k, F=64, Fs=0, dtype=dtype, score=score,
                   bias_range=0.01 if score == SIGMOID else 0.0, seed=seed, name="reroute")
    c.update(capacity_factor=cf, reroute=extra)
    host = moe_inputs.host_inputs(c)
    res = to_host(gpu_forward(c, moe_inputs.upload(c, host)))
    _, sc, key = oracle.router_scores(host["x"], host["w_router"], c["score"], host.get("bias"))
    kc = k + extra
    srt = -np.sort(-key, axis=1)[:, :kc + 1]
    assert np.min(srt[:, :-1] - srt[:, 1:]) >= 1e-4, "inputs with a near-tie: pick another seed"
    cand, _, _ = oracle.topk(key, sc, kc)
    cap = oracle.capacity(T, E, k, cf)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, E, cap)
    assert ((assign >= 0) & (assign != cand[:, :k])).any(), "no slot was rerouted"
    np.testing.assert_array_equal(res["topk_idx"], assign)
    np.testing.assert_array_equal(res["counts"], counts)
    np.testing.assert_array_equal(res["sorted_token"][:offsets[-1]], st)
    assert int(res["dropped"][0]) == dropped
    w = oracle.served_weights(sc, assign)
    np.testing.assert_allclose(res["topk_w"], w, rtol=0, atol=2e-5)
    experts = {e: (host["w_gate_up"][e], host["w_down"][e]) for e in range(E)}
    from layer_check import check_output, oracle_rows
    ref = oracle_rows(c, host["x"], np.where(assign >= 0, assign, 0), w, experts, None, 4)
    print(check_output(c, res["out"], ref))


@pytest.mark.parametrize("score,k,extra,Fs,E,G,M,seed", [(SOFTMAX, 2, 2, 0, 16, 4, 2, 302),
                                                       (SIGMOID, 4, 3, 64, 32, 8, 3, 319)])
def test_reroute_with_groups_matches_oracle(score, k, extra, Fs, E, G, M, seed):
    """Rerouting under group-limited routing: the candidates are the token's top-(k + extra)
    experts of its kept groups, bit-exact against the oracle's grouped top-k and rounds.  The
    inputs have no near-tie (1e-4) among the kept groups' top-(k + extra + 1) keys nor between
    the M-th and (M+1)-th group scores."""
    c = make_shape(T=300, d=256, E=E, k=k, F=128, Fs=Fs, dtype="bf16", score=score,
                   bias_range=0.01 if score == SIGMOID else 0.0, seed=seed, name="reroute")
    c.update(capacity_factor=1.0, reroute=extra, groups=G, topk_groups=M)
    host = moe_inputs.host_inputs(c)
    res = to_host(gpu_forward(c, moe_inputs.upload(c, host)))
    _, sc, key = oracle.router_scores(host["x"], host["w_router"], c["score"], host.get("bias"))
    kc = k + extra
    gs = key.reshape(len(key), G, E // G).max(axis=2)
    gsrt = -np.sort(-gs, axis=1)
    assert np.min(gsrt[:, M - 1] - gsrt[:, M]) >= 1e-4, "group scores with a near-tie"
    cand, _, _ = oracle.topk_grouped(key, sc, kc + 1, G, M)
    kept = np.take_along_axis(key, cand.astype(np.int64), axis=1)
    assert np.min(kept[:, :-1] - kept[:, 1:]) >= 1e-4, "keys with a near-tie"
    cand = np.ascontiguousarray(cand[:, :kc])
    cap = oracle.capacity(c["T"], E, k, 1.0)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, E, cap)
    assert ((assign >= 0) & (assign != cand[:, :k])).any(), "no slot was rerouted"
    np.testing.assert_array_equal(res["topk_idx"], assign)
    np.testing.assert_array_equal(res["counts"], counts)
    np.testing.assert_array_equal(res["sorted_token"][:offsets[-1]], st)
    assert int(res["dropped"][0]) == dropped
    w = oracle.served_weights(sc, assign)
    np.testing.assert_allclose(res["topk_w"], w, rtol=0, atol=2e-5)
    experts = {e: (host["w_gate_up"][e], host["w_down"][e]) for e in range(E)}
    shared = (host["sh_gate_up"], host["sh_down"]) if Fs > 0 else None
    from layer_check import check_output, oracle_rows
    ref = oracle_rows(c, host["x"], np.where(assign >= 0, assign, 0), w, experts, shared, 4)
    print(check_output(c, res["out"], ref))
