"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names the mistake it is built to catch.  Sources of the definitions are in
oracle/moe_oracle.h.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
from moe_inputs import host

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def silu(g):
    return g * expit(g)


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------------ element decoding
def test_bf16_element_decoding():
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x4049, 0x0000, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 0.5, 3.140625, 0.0, -0.0]
    got = [oracle.lib().oracle_elem(bits.ctypes.data, oracle.BF16, i) for i in range(6)]
    assert got == want


# ------------------------------------------------------------------ hand-worked cases
def test_hand_case_softmax_router_and_swiglu():
    """d=2, E=4, k=2, F=1, x=[1,0], logits [2,1,0,-1].  Closed forms: S=(0,1),
    w0 = 1/(1+e^-1), w1 = 1/(1+e^1); expert e has gate weight a_e=e+1, up 1, down [1,0],
    so out = [w0*silu(1) + w1*silu(2), 0].  Catches: wrong softmax direction, missing
    renormalisation, gate/up swapped, wrong output row of W_down."""
    x = f32([[1, 0]])
    wr = f32([[2, 0], [1, 0], [0, 0], [-1, 0]])
    _, s, key = oracle.router_scores(x, wr, oracle.SOFTMAX)
    idx, w, margin = oracle.topk(key, s, 2)
    assert idx.tolist() == [[0, 1]]
    assert w[0, 0] == pytest.approx(1 / (1 + math.exp(-1)), abs=1e-15)
    assert w[0, 1] == pytest.approx(1 / (1 + math.exp(1)), abs=1e-15)
    assert margin[0] == pytest.approx(1.0)
    gu = {e: f32([[e + 1, 0], [1, 0]]) for e in range(4)}     # [2F][d]: gate row, up row
    dn = {e: f32([[1], [0]]) for e in range(4)}               # [d][F]
    out = oracle.layer_rows(x, idx, w, gu, dn)
    s1 = 1 / (1 + math.exp(-1))
    s2 = 2 / (1 + math.exp(-2))
    want = (1 / (1 + math.exp(-1))) * s1 + (1 / (1 + math.exp(1))) * s2
    assert out[0, 0] == pytest.approx(want, abs=1e-14)
    assert out[0, 0] == pytest.approx(1.0082122816, abs=1e-9)
    assert out[0, 1] == 0.0


def test_hand_case_tie_break_lower_id():
    """logits [1,1,1,0], k=2 -> S=(0,1), w=(1/2,1/2).  Catches a tie-break toward the
    higher id or an unstable selection."""
    x = f32([[1, 0]])
    wr = f32([[1, 0], [1, 0], [1, 0], [0, 0]])
    _, s, key = oracle.router_scores(x, wr, oracle.SOFTMAX)
    idx, w, margin = oracle.topk(key, s, 2)
    assert idx.tolist() == [[0, 1]]
    assert w.tolist() == [[0.5, 0.5]]
    assert margin[0] == 0.0


def test_hand_case_sigmoid_bias_selects_but_does_not_weight():
    """l=[0,.5,-.5,1], b=[0,-.6,.7,0]: keys sigma+b = [.5, .0225, 1.0775, .7311] -> S=(2,3);
    w from the UNBIASED sigma: sigma(-.5)/(sigma(-.5)+sigma(1)).  Catches weights taken
    from biased keys, bias ignored in selection, or a sign error in the sigmoid."""
    x = f32([[1, 0]])
    wr = f32([[0, 0], [0.5, 0], [-0.5, 0], [1, 0]])
    bias = f32([0, -0.6, 0.7, 0])
    _, s, key = oracle.router_scores(x, wr, oracle.SIGMOID, bias)
    idx, w, _ = oracle.topk(key, s, 2)
    assert idx.tolist() == [[2, 3]]
    sa, sb = 1 / (1 + math.exp(0.5)), 1 / (1 + math.exp(-1.0))
    assert w[0, 0] == pytest.approx(sa / (sa + sb), abs=1e-15)
    assert w[0, 0] == pytest.approx(0.3405564903, abs=1e-9)
    assert key[0, 1] == pytest.approx(1 / (1 + math.exp(-0.5)) + float(np.float32(-0.6)), abs=1e-15)


# ------------------------------------------------------------------ library / closed-form reductions
def test_logits_equal_library_matmul_and_softmax():
    """Logits = x W_r^T (numpy matmul), scores = scipy softmax / expit.  Non-square shapes
    catch a transposed operand; any dropped term changes the matmul."""
    rng = np.random.default_rng(1)
    x = f32(rng.standard_normal((7, 24)))
    wr = f32(rng.standard_normal((5, 24)) / 5)
    bias = f32(rng.uniform(-0.1, 0.1, 5))
    ref = x.astype(np.float64) @ wr.astype(np.float64).T
    lg, s, key = oracle.router_scores(x, wr, oracle.SOFTMAX)
    np.testing.assert_allclose(lg, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s, softmax(ref, axis=1), rtol=1e-13)
    np.testing.assert_array_equal(key, lg)
    lg2, s2, key2 = oracle.router_scores(x, wr, oracle.SIGMOID, bias)
    np.testing.assert_allclose(s2, expit(ref), rtol=1e-13)
    np.testing.assert_allclose(key2, expit(ref) + bias.astype(np.float64), rtol=1e-13)


def test_softmax_renorm_closed_form():
    """After renormalisation over the selected set, w_j = 1 / (1 + sum_{j' != j} e^(l_j' - l_j))."""
    rng = np.random.default_rng(2)
    l = rng.standard_normal((20, 16)) * 2
    s = softmax(l, axis=1)
    idx, w, _ = oracle.topk(l, s, 4)
    for t in range(20):
        sel = l[t, idx[t]]
        for j in range(4):
            want = 1.0 / (1.0 + sum(math.exp(sel[jj] - sel[j]) for jj in range(4) if jj != j))
            assert w[t, j] == pytest.approx(want, rel=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-15)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 4), (10, 3), (10, 10), (9, 8)])
def test_topk_brute_force_with_ties(E, k):
    """Against brute force over all C(E,k) subsets: the selected set is the unique subset
    whose every member beats every non-member (larger key, or equal key and lower id).
    Keys are quantised so ties are frequent.  Order: key descending, ties lower id."""
    rng = np.random.default_rng(E * 31 + k)
    key = np.round(rng.standard_normal((200, E)) * 2) / 2
    score = rng.uniform(0.1, 1.0, (200, E))
    idx, w, margin = oracle.topk(key, score, k)

    def beats(a, b, kr):
        return kr[a] > kr[b] or (kr[a] == kr[b] and a < b)

    for t in range(200):
        kr = key[t]
        valid = [S for S in itertools.combinations(range(E), k)
                 if all(beats(a, b, kr) for a in S for b in range(E) if b not in S)]
        assert len(valid) == 1
        assert sorted(idx[t].tolist()) == list(valid[0])
        order = sorted(valid[0], key=lambda e: (-kr[e], e))
        assert idx[t].tolist() == order
        sel = score[t, order]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=1e-15)
        if k < E:
            rest = max(kr[b] for b in range(E) if b not in valid[0])
            assert margin[t] == kr[order[-1]] - rest
        else:
            assert margin[t] == np.inf


# ------------------------------------------------------------------ group-limited top-k
def test_hand_case_group_limited_routing():
    """E=8 in 4 groups of 2, keep 2 groups, k=3; keys [0.9,0.1 | 0.2,0.15 | 0.85,0.8 | 0.3,0.95].
    Group scores (best key): 0.9, 0.2, 0.85, 0.95 -> groups 3 and 0 kept -> experts {0,1,6,7};
    top-3 by key: 7 (0.95), 0 (0.9), 6 (0.3).  Plain top-3 would take 4 (0.85) instead of 6.
    Catches: group scored by its mean or sum (sum keeps group 2), groups not limiting the choice."""
    key = np.array([[0.9, 0.1, 0.2, 0.15, 0.85, 0.8, 0.3, 0.95]])
    idx, w, margin = oracle.topk_grouped(key, key, 3, 4, 2)
    assert idx[0].tolist() == [7, 0, 6]
    np.testing.assert_allclose(w[0], np.array([0.95, 0.9, 0.3]) / 2.15, rtol=1e-15)
    # margins: kept groups' 2nd score 0.9 vs the best dropped 0.85 -> 0.05; experts: 0.3 vs 0.1
    assert margin[0] == pytest.approx(0.05, abs=1e-15)
    pidx, _, _ = oracle.topk(key, key, 3)
    assert pidx[0].tolist() == [7, 0, 4]


def test_group_limited_tie_breaks_to_lower_group():
    """Two groups with equal best keys and room for one: the lower group id is kept."""
    key = np.array([[0.5, 0.1, 0.5, 0.4, 0.2, 0.3]])   # 3 groups of 2, best keys 0.5, 0.5, 0.3
    idx, _, margin = oracle.topk_grouped(key, key, 2, 3, 1)
    assert idx[0].tolist() == [0, 1] and margin[0] == 0.0


@pytest.mark.parametrize("E,G,M,k", [(8, 4, 2, 3), (8, 2, 1, 4), (9, 3, 2, 4), (12, 4, 3, 5),
                                     (10, 5, 2, 2), (12, 6, 6, 6), (8, 8, 3, 3)])
def test_group_limited_brute_force_with_ties(E, G, M, k):
    """Against brute force: enumerate every set of M groups and every k-subset of their experts;
    the chosen groups are the unique M-set whose every member beats every non-member by group
    score (best key; ties -> lower group id), and the chosen experts the unique k-subset of the
    kept experts whose members beat every other kept expert.  Quantised keys make ties common."""
    rng = np.random.default_rng(E * 101 + G * 7 + M * 3 + k)
    key = np.round(rng.standard_normal((150, E)) * 2) / 2
    score = rng.uniform(0.1, 1.0, (150, E))
    idx, w, margin = oracle.topk_grouped(key, score, k, G, M)
    gs = E // G

    def beats(a, b, v):
        return v[a] > v[b] or (v[a] == v[b] and a < b)

    for t in range(150):
        kr = key[t]
        gscore = [max(kr[g * gs:(g + 1) * gs]) for g in range(G)]
        gsets = [S for S in itertools.combinations(range(G), M)
                 if all(beats(a, b, gscore) for a in S for b in range(G) if b not in S)]
        assert len(gsets) == 1
        allowed = [e for e in range(E) if e // gs in gsets[0]]
        esets = [S for S in itertools.combinations(allowed, k)
                 if all(beats(a, b, kr) for a in S for b in allowed if b not in S)]
        assert len(esets) == 1
        order = sorted(esets[0], key=lambda e: (-kr[e], e))
        assert idx[t].tolist() == order
        sel = score[t, order]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=1e-15)


def test_group_limited_reduces_to_plain_topk():
    """One group, or every group kept: the same routing as the plain top-k (itself pinned by
    brute force above)."""
    rng = np.random.default_rng(5)
    key = np.round(rng.standard_normal((300, 16)) * 2) / 2
    score = rng.uniform(0.1, 1.0, (300, 16))
    pidx, pw, pm = oracle.topk(key, score, 4)
    for G, M in ((1, 1), (4, 4), (16, 16)):
        idx, w, m = oracle.topk_grouped(key, score, 4, G, M)
        np.testing.assert_array_equal(idx, pidx)
        np.testing.assert_array_equal(w, pw)


def test_group_limited_rejects_bad_shapes():
    key = np.zeros((1, 8))
    for G, M, k in ((3, 1, 1), (4, 0, 1), (4, 5, 1), (4, 1, 3)):
        with pytest.raises(ValueError):
            oracle.topk_grouped(key, key, k, G, M)


# ------------------------------------------------------------------ dispatch tables
def _random_routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (100, 16, 5), (64, 64, 64)])
def test_dispatch_against_stable_sort_and_invariants(T, E, k):
    """Against Python's stable sort of (expert, token) pairs; invariants: sum counts = T*k,
    offsets = exclusive scan, segments ascending in t, slot_pos o sorted_token = identity."""
    idx = _random_routing(T, E, k, T + E + k)
    counts, offsets, st, sp = oracle.dispatch(idx, E)
    pairs = sorted(((int(idx[t, j]), t, j) for t in range(T) for j in range(k)))
    assert st.tolist() == [t for _, t, _ in pairs]
    for p, (_, t, j) in enumerate(pairs):
        assert sp[t, j] == p
    assert counts.sum() == T * k
    np.testing.assert_array_equal(np.bincount(idx.ravel(), minlength=E), counts)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    for e in range(E):
        seg = st[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    for t in range(T):
        for j in range(k):
            assert st[sp[t, j]] == t


def test_dispatch_reproduces_capacity_worked_example():
    """Page worked example: 512 decode tokens, top-8 of 256 experts, EP=16 -> 4096
    assignments, 16 per expert under perfectly even routing, 256 per 16-expert GPU."""
    g = json.load(open(os.path.join(GOLDEN, "capacity_worked_example.json")))
    T, E, k, ep = g["tokens"], g["n_experts"], g["top_k"], g["ep_size"]
    idx = np.array([[(8 * t + j) % E for j in range(k)] for t in range(T)], dtype=np.int32)
    counts, offsets, _, _ = oracle.dispatch(idx, E)
    assert offsets[-1] == g["expected"]["assignments"]
    assert set(counts.tolist()) == {g["expected"]["tokens_per_expert_uniform"]}
    per_gpu = counts.reshape(ep, E // ep).sum(1)
    assert set(per_gpu.tolist()) == {g["expected"]["token_experts_per_gpu_uniform"]}
    skew = g["expected"]["busiest_gpu_skew"]
    assert round(skew * per_gpu.mean()) == g["expected"]["busiest_gpu_token_experts_approx"]


# ------------------------------------------------------------------ expert capacity
def test_capacity_formula_on_the_worked_example():
    """Page formula capacity = capacity_factor * (tokens * k / experts): the worked example's
    512 decode tokens, top-8 of 256 experts give 16 slots at factor 1.0, 20 at 1.25 and 32 at
    2.0; a fractional capacity rounds up (200 / 7 = 28.57 -> 29)."""
    g = json.load(open(os.path.join(GOLDEN, "capacity_worked_example.json")))
    T, E, k = g["tokens"], g["n_experts"], g["top_k"]
    assert oracle.capacity(T, E, k, 1.0) == g["expected"]["tokens_per_expert_uniform"] == 16
    assert oracle.capacity(T, E, k, 1.25) == 20 and oracle.capacity(T, E, k, 2.0) == 32
    assert oracle.capacity(100, 7, 2, 1.0) == 29
    with pytest.raises(ValueError):
        oracle.capacity(10, 4, 2, 0.0)


def test_capacity_hand_case():
    """5 tokens, 2 experts, top-1, routed [0,0,0,1,0], capacity 2: expert 0 keeps tokens 0 and
    1, tokens 2 and 4 are dropped (slot -1), expert 1 keeps token 3."""
    counts, offsets, st, sp, dropped = oracle.dispatch_capacity(
        np.array([[0], [0], [0], [1], [0]]), 2, 2)
    assert counts.tolist() == [2, 1] and offsets.tolist() == [0, 2, 3]
    assert st.tolist() == [0, 1, 3] and sp[:, 0].tolist() == [0, 1, -1, 2, -1]
    assert dropped == 2


@pytest.mark.parametrize("T,E,k,cap", [(40, 6, 2, 5), (100, 16, 5, 20), (64, 8, 8, 64),
                                       (33, 4, 3, 1), (10, 3, 2, 0)])
def test_capacity_dispatch_invariants(T, E, k, cap):
    """Skewed random routings: kept per expert = min(routed, capacity); the kept assignments
    of an expert are its `capacity` lowest token ids; kept + dropped = T*k; kept slots are a
    bijection onto [0, kept total) consistent with sorted_token.  Catches: dropping by arrival
    slot j instead of token order, counts before capping, off-by-one at the capacity."""
    rng = np.random.default_rng(T * 7 + E + k + cap)
    p = rng.dirichlet(np.full(E, 0.3))
    idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    counts, offsets, st, sp, dropped = oracle.dispatch_capacity(idx, E, cap)
    routed = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(counts, np.minimum(routed, cap))
    assert counts.sum() + dropped == T * k
    for e in range(E):
        toks = sorted(t for t in range(T) if e in idx[t])
        kept = sorted(int(t) for t, j in zip(*np.where(idx == e)) if sp[t, j] >= 0)
        assert kept == toks[:cap]
        seg = st[offsets[e]:offsets[e + 1]].tolist()
        assert seg == kept
    kept_slots = sp[sp >= 0]
    assert sorted(kept_slots.tolist()) == list(range(counts.sum()))
    for t, j in zip(*np.where(sp >= 0)):
        assert st[sp[t, j]] == t


def test_capacity_large_enough_is_dropless():
    """A capacity of T (no expert can hold more) reproduces the dropless dispatch."""
    idx = _random_routing(80, 10, 3, 4)
    a = oracle.dispatch(idx, 10)
    b = oracle.dispatch_capacity(idx, 10, 80)
    for x, y in zip(a, b[:4]):
        np.testing.assert_array_equal(x, y)
    assert b[4] == 0


def test_combine_skips_dropped_assignments():
    """Identity experts with some assignments dropped: out[t] = (sum of the kept weights) x[t]."""
    rng = np.random.default_rng(9)
    T, E, k, d = 30, 5, 2, 4
    x = rng.standard_normal((T, d))
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), T)
    counts, offsets, st, sp, dropped = oracle.dispatch_capacity(idx, E, 7)
    assert dropped > 0
    ys = oracle.gather(st, x)
    out = oracle.combine(sp, w, ys)
    kept_w = np.where(sp >= 0, w, 0.0).sum(1)
    np.testing.assert_allclose(out, kept_w[:, None] * x, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ redundant-expert placement
def test_eplb_hand_cases():
    """8 experts with loads [10,1,...,1] on 2 GPUs.  No replicas: the largest goes first to GPU 0,
    GPU 1 fills its 4 slots with four 1s, GPU 0 takes the last three -> loads [13, 4].  Two
    redundant slots: expert 0 takes both (10/1, then 10/2 lead), three replicas of 10/3; GPU 1
    takes the second (GPU 0 already holds expert 0), the third goes back to GPU 0 (both hold one,
    equal load, lower id), GPU 1 then takes four 1s and GPU 0 the last three -> [29/3, 22/3]."""
    se, sg, gl = oracle.eplb_plan([10, 1, 1, 1, 1, 1, 1, 1], 2, 0)
    np.testing.assert_array_equal(gl, [13.0, 4.0])
    assert se.tolist() == [0, 5, 6, 7, 1, 2, 3, 4] and sg.tolist() == [0] * 4 + [1] * 4
    se, sg, gl = oracle.eplb_plan([10, 1, 1, 1, 1, 1, 1, 1], 2, 2)
    np.testing.assert_allclose(gl, [29 / 3, 22 / 3], rtol=1e-15)
    assert se.tolist() == [0, 0, 5, 6, 7, 0, 1, 2, 3, 4]


@pytest.mark.parametrize("E,G,R", [(16, 4, 0), (16, 4, 4), (128, 8, 8), (256, 16, 16), (10, 5, 5)])
def test_eplb_invariants(E, G, R):
    """Skewed random loads: every expert placed at least once, each GPU exactly (E+R)/G slots,
    load conserved, a GPU holds two replicas of an expert only if some GPU holds none of it is
    impossible (more replicas than GPUs), and the replicated experts are those the greedy
    favours: an expert a with n_a >= 2 replicas had the largest load per replica when it got its
    last one, i.e. load_a / (n_a - 1) >= load_b / n_b for every other expert b."""
    rng = np.random.default_rng(E + G + R)
    load = (rng.pareto(1.2, E) * 100).astype(np.int32)
    se, sg, gl = oracle.eplb_plan(load, G, R)
    S = E + R
    assert sorted(set(se.tolist())) == list(range(E))
    assert np.bincount(sg, minlength=G).tolist() == [S // G] * G
    n = np.bincount(se, minlength=E)
    np.testing.assert_allclose(gl.sum(), load.sum(), rtol=1e-12)
    per = load / n
    np.testing.assert_allclose(np.bincount(sg, weights=per[se], minlength=G), gl, rtol=1e-12)
    for a in np.where(n >= 2)[0]:
        assert load[a] / (n[a] - 1) >= (per[np.arange(E) != a]).max() - 1e-9
    for g in range(G):
        held = se[sg == g]
        for e in set(held.tolist()):
            if (held == e).sum() > 1:
                assert n[e] > G


def test_eplb_balances_a_skewed_load():
    """A Zipf-like load on 64 experts over 8 GPUs: the plan's max/mean GPU load is below the
    contiguous placement's and falls further with redundant slots."""
    load = (1000 * np.arange(1, 65) ** -1.2).astype(np.int32)
    contiguous = load.reshape(8, 8).sum(1)
    ratio = lambda gl: gl.max() / gl.mean()
    r0 = ratio(contiguous)
    r1 = ratio(oracle.eplb_plan(load, 8, 0)[2])
    r2 = ratio(oracle.eplb_plan(load, 8, 8)[2])
    assert r0 > r1 > r2 >= 1.0


def test_identity_experts_round_trip_returns_x():
    """Dispatch (gather) then combine with identity experts returns x (weights sum to 1)."""
    rng = np.random.default_rng(5)
    T, E, k, d = 50, 12, 3, 9
    x = rng.standard_normal((T, d))
    l = rng.standard_normal((T, E))
    idx, w, _ = oracle.topk(l, softmax(l, axis=1), k)
    _, _, st, sp = oracle.dispatch(idx, E)
    xs = oracle.gather(st, x)
    out = oracle.combine(sp, w, xs)
    np.testing.assert_allclose(out, x, atol=1e-12)
    shared = rng.standard_normal((T, d))
    np.testing.assert_allclose(oracle.combine(sp, w, xs, shared), x + shared, atol=1e-12)


def test_combine_against_einsum():
    rng = np.random.default_rng(6)
    T, k, d, R = 11, 3, 5, 40
    sp = rng.integers(0, R, (T, k)).astype(np.int32)
    w = rng.uniform(0, 1, (T, k))
    ys = rng.standard_normal((R, d))
    np.testing.assert_allclose(oracle.combine(sp, w, ys), np.einsum("tj,tjc->tc", w, ys[sp]),
                               rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ expert FFN
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_swiglu_against_library_matmul(dtype):
    """y = W_d (silu(W_g x) * (W_u x)) with numpy matmul and scipy expit; F != d catches a
    transposed weight, the asymmetric silu catches gate/up swapped."""
    rng = np.random.default_rng(7)
    d, F = 12, 20
    wgu = f32(rng.standard_normal((2 * F, d)) / math.sqrt(d))
    wd = f32(rng.standard_normal((d, F)) / math.sqrt(F))
    x = rng.standard_normal(d)
    if dtype == "bf16":
        wgu_s, wd_s = host.f32_to_bf16_bits(wgu), host.f32_to_bf16_bits(wd)
        wgu = host.bf16_bits_to_f32(wgu_s); wd = host.bf16_bits_to_f32(wd_s)
    else:
        wgu_s, wd_s = wgu, wd
    g = wgu[:F].astype(np.float64) @ x
    u = wgu[F:].astype(np.float64) @ x
    want = wd.astype(np.float64) @ (silu(g) * u)
    np.testing.assert_allclose(oracle.swiglu_ffn(x, wgu_s, wd_s), want, rtol=1e-12, atol=1e-13)


def test_single_expert_layer_is_dense_swiglu():
    """E = k = 1: the layer is one dense SwiGLU FFN (weight 1)."""
    rng = np.random.default_rng(8)
    T, d, F = 6, 16, 24
    x = f32(rng.standard_normal((T, d)))
    wr = f32(rng.standard_normal((1, d)))
    wgu = f32(rng.standard_normal((1, 2 * F, d)) / 4)
    wd = f32(rng.standard_normal((1, d, F)) / 5)
    _, s, key = oracle.router_scores(x, wr, oracle.SOFTMAX)
    idx, w, _ = oracle.topk(key, s, 1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    out = oracle.layer_rows(x, idx, w, wgu, wd)
    xd = x.astype(np.float64)
    want = (silu(xd @ wgu[0, :F].T.astype(np.float64)) * (xd @ wgu[0, F:].T.astype(np.float64))) \
        @ wd[0].T.astype(np.float64)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)


def test_identical_experts_make_output_routing_independent():
    """All experts equal -> out = dense FFN regardless of routing (weights sum to 1);
    the shared expert adds its own dense FFN."""
    rng = np.random.default_rng(9)
    T, d, E, k, F, Fs = 10, 8, 6, 3, 16, 8
    x = f32(rng.standard_normal((T, d)))
    one_gu = f32(rng.standard_normal((2 * F, d)) / 3)
    one_dn = f32(rng.standard_normal((d, F)) / 4)
    shg = f32(rng.standard_normal((2 * Fs, d)) / 3)
    shd = f32(rng.standard_normal((d, Fs)) / 3)
    wgu = np.stack([one_gu] * E); wd = np.stack([one_dn] * E)
    l = rng.standard_normal((T, E))
    idx, w, _ = oracle.topk(l, softmax(l, axis=1), k)
    out = oracle.layer_rows(x, idx, w, wgu, wd, shg, shd)
    xd = x.astype(np.float64)
    dense = (silu(xd @ one_gu[:F].T.astype(np.float64)) * (xd @ one_gu[F:].T.astype(np.float64))) \
        @ one_dn.T.astype(np.float64)
    shared = (silu(xd @ shg[:Fs].T.astype(np.float64)) * (xd @ shg[Fs:].T.astype(np.float64))) \
        @ shd.T.astype(np.float64)
    np.testing.assert_allclose(out, dense + shared, rtol=1e-12, atol=1e-12)
    idx2 = np.roll(idx, 1, axis=1)
    np.testing.assert_allclose(oracle.layer_rows(x, idx2, w, wgu, wd, shg, shd), out,
                               rtol=1e-12, atol=1e-12)


def test_missing_expert_weights_is_an_error():
    x = f32([[1.0, 2.0]])
    idx = np.array([[1]], dtype=np.int32)
    w = np.array([[1.0]])
    with pytest.raises(ValueError):
        oracle.layer_rows(x, idx, w, {0: f32([[1, 0], [0, 1]])}, {0: f32([[1], [1]])})


def test_softmax_bias_moves_selection_not_weights():
    """Softmax with a selection bias: key = logit + b selects, the weights stay the
    renormalised unbiased softmax.  l=[2,1,0], b=[0,0,2.5]: keys [2,1,2.5];
    k=2 -> (2, 0) with w = softmax([0, 2]) = (1/(1+e^2), 1/(1+e^-2))."""
    x = f32([[1, 0]])
    wr = f32([[2, 0], [1, 0], [0, 0]])
    bias = f32([0, 0, 2.5])
    _, s, key = oracle.router_scores(x, wr, oracle.SOFTMAX, bias)
    idx, w, _ = oracle.topk(key, s, 2)
    assert idx.tolist() == [[2, 0]]
    assert w[0, 0] == pytest.approx(1 / (1 + math.exp(2)), abs=1e-15)
    assert w[0, 1] == pytest.approx(1 / (1 + math.exp(-2)), abs=1e-15)


# ------------------------------------------------------------------ rerouting at capacity
def test_reroute_hand_case_overflow_moves_to_next_best():
    """4 tokens, 3 experts, top-1 with all 3 candidates, capacity 2.  Round 0: tokens 0 and 1
    fill expert 0, token 2 overflows, token 3 takes expert 1; round 1: token 2 moves to its
    next-best expert 1, which still has a slot."""
    cand = [[0, 1, 2], [0, 2, 1], [0, 1, 2], [1, 0, 2]]
    assign, ac, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, 1, 3, 2)
    assert assign[:, 0].tolist() == [0, 0, 1, 1] and ac[:, 0].tolist() == [0, 0, 1, 0]
    assert counts.tolist() == [2, 2, 0] and offsets.tolist() == [0, 2, 4, 4]
    assert st.tolist() == [0, 1, 2, 3] and sp[:, 0].tolist() == [0, 1, 2, 3] and dropped == 0


def test_reroute_hand_case_candidates_run_out():
    """Same candidates, capacity 1.  Round 0: token 0 -> 0, token 3 -> 1, tokens 1 and 2
    rejected; round 1: token 1 takes expert 2, token 2 finds expert 1 full; round 2: token 2
    finds expert 2 full and has no candidate left: dropped."""
    cand = [[0, 1, 2], [0, 2, 1], [0, 1, 2], [1, 0, 2]]
    assign, ac, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, 1, 3, 1)
    assert assign[:, 0].tolist() == [0, 2, -1, 1] and ac[:, 0].tolist() == [0, 1, -1, 0]
    assert counts.tolist() == [1, 1, 1] and st.tolist() == [0, 3, 1]
    assert sp[:, 0].tolist() == [0, 2, -1, 1] and dropped == 1


def test_reroute_hand_case_two_slots_take_successive_candidates():
    """Top-2 of 4 experts, capacity 1: token 0 fills experts 0 and 1; token 1's two rejected
    slots take its next candidates in slot order (slot 0 -> expert 3, slot 1 -> expert 2)."""
    cand = [[0, 1, 2, 3], [0, 1, 3, 2]]
    assign, ac, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, 2, 4, 1)
    assert assign.tolist() == [[0, 1], [3, 2]] and ac.tolist() == [[0, 1], [2, 3]]
    assert counts.tolist() == [1, 1, 1, 1] and st.tolist() == [0, 0, 1, 1]
    assert sp.tolist() == [[0, 1], [3, 2]] and dropped == 0


def _skewed_candidates(rng, T, E, kc):
    w = 1.0 / np.arange(1, E + 1) ** 1.5
    keys = np.log(w)[None, :] + rng.standard_normal((T, E))
    idx, _, _ = oracle.topk(keys, np.ones((T, E)), kc)
    return idx


@pytest.mark.parametrize("T,E,k,extra,cap", [(50, 8, 2, 2, 6), (200, 16, 4, 4, 30), (64, 8, 8, 0, 40),
                                             (100, 12, 3, 9, 20), (30, 6, 1, 5, 3)])
def test_reroute_invariants(T, E, k, extra, cap):
    """Random skewed candidate lists: no expert over capacity; served + dropped = T*k; each
    token's serving experts are distinct candidates of its own list; the tables are a stable
    counting sort of the assignment.  Catches: double-booking an expert, a token served twice
    by one expert, candidates taken out of order."""
    rng = np.random.default_rng(T + E + k)
    cand = _skewed_candidates(rng, T, E, k + extra)
    assign, ac, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, E, cap)
    assert counts.max() <= cap and counts.sum() + dropped == T * k
    for t in range(T):
        served = [(e, c) for e, c in zip(assign[t], ac[t]) if e >= 0]
        assert len({e for e, _ in served}) == len(served)
        for e, c in served:
            assert cand[t][c] == e
    want_st = [t for e in range(E) for t in range(T) for j in range(k) if assign[t, j] == e]
    assert st.tolist() == want_st
    for t in range(T):
        for j in range(k):
            assert (sp[t, j] < 0) == (assign[t, j] < 0)
            if sp[t, j] >= 0:
                assert st[sp[t, j]] == t and offsets[assign[t, j]] <= sp[t, j] < offsets[assign[t, j] + 1]


@pytest.mark.parametrize("T,E,k,cap", [(40, 6, 2, 5), (100, 16, 4, 20), (33, 4, 3, 1)])
def test_reroute_without_extra_candidates_is_capacity_dropping(T, E, k, cap):
    """With no candidate beyond the top-k the procedure is the capacity dispatch that drops."""
    rng = np.random.default_rng(7 * T + k)
    cand = _skewed_candidates(rng, T, E, k)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, k, E, cap)
    c2, o2, st2, sp2, d2 = oracle.dispatch_capacity(cand, E, cap)
    assert counts.tolist() == c2.tolist() and st.tolist() == st2.tolist()
    assert sp.tolist() == sp2.tolist() and dropped == d2
    assert np.array_equal(assign, np.where(sp2 >= 0, cand, -1))


def test_reroute_with_room_everywhere_is_dropless():
    """A capacity no expert can reach: the top-k of every token, dropless tables."""
    rng = np.random.default_rng(3)
    cand = _skewed_candidates(rng, 80, 10, 6)
    assign, _, counts, offsets, st, sp, dropped = oracle.dispatch_reroute(cand, 4, 10, 80 * 4)
    c2, o2, st2, sp2 = oracle.dispatch(cand[:, :4], 10)
    assert np.array_equal(assign, cand[:, :4]) and dropped == 0
    assert counts.tolist() == c2.tolist() and st.tolist() == st2.tolist() and sp.tolist() == sp2.tolist()


def test_served_weights_renormalise_over_serving_experts():
    score = np.array([[0.5, 0.3, 0.2], [0.1, 0.6, 0.3]])
    w = oracle.served_weights(score, np.array([[0, 2], [-1, -1]]))
    np.testing.assert_allclose(w, [[0.5 / 0.7, 0.2 / 0.7], [0.0, 0.0]], rtol=0, atol=1e-15)
    w = oracle.served_weights(score, np.array([[1, -1], [2, 1]]))
    np.testing.assert_allclose(w, [[1.0, 0.0], [0.3 / 0.9, 0.6 / 0.9]], rtol=0, atol=1e-15)
