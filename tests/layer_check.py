"""Parity helpers: run the layer through the C ABI on the GPU, compute the fp64 oracle on the
same inputs, and compare them the way the layer's correctness criteria read:

* routing: bit-exact top-k sets for every token whose k-th / (k+1)-th key margin (fp64 oracle
  keys) is at least ``MARGIN``; a token under the margin may pick either side of the near-tie,
  but its choice must be a valid top-k of the oracle keys up to ``MARGIN``;
* dispatch tables: bit-exact against the oracle's tables for the GPU's routing;
* group-limited routing (a workload with ``topk_groups`` > 0 keeps that many of its ``groups``
  expert groups per token): the same, against the oracle's group-limited top-k, whose margin
  also covers near-ties between groups;
* expert capacity (a workload with ``capacity_factor`` > 0): dispatch tables and the number
  dropped bit-exactly against the oracle's capacity dispatch of the GPU's routing, and the
  output against the oracle with the dropped assignments contributing nothing;
* output: max |err| <= 2e-2 * max |ref| and sum |err| / sum |ref| <= 5e-3 for bf16 (tighter
  for fp32), the oracle evaluated under the GPU's routing, so an accepted near-tie does not
  count as an output error.

Test infrastructure: imports the oracle.
"""
import numpy as np

import moe_inputs
import oracle
from moe_inputs import configs

MARGIN = 1e-4
TOL = {"bf16": dict(max_rel=2e-2, mean_rel=5e-3), "f32": dict(max_rel=1e-4, mean_rel=1e-5)}


def moe_dtype(cfg):
    import mixture_experts_layer_83_b300 as moe
    return moe.MOE_DTYPE_BF16 if cfg["dtype"] == "bf16" else moe.MOE_DTYPE_F32


def gpu_forward(cfg, dev, stream=None, workspace=None, stage_events=None):
    """Run the layer on device tensors ``dev`` (from moe_inputs.device_inputs / upload)."""
    import torch
    import mixture_experts_layer_83_b300 as moe
    c = configs.get(cfg)
    T, d, E, k = c["T"], c["d"], c["E"], c["k"]
    shape = moe.make_shape(T, d, E, k, c["F"], c["Fs"], moe_dtype(c))
    ws_bytes = moe.moe_layer_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev["x"].device)
    out = torch.empty_like(dev["x"])
    counts = torch.empty(E, dtype=torch.int32, device=out.device)
    tidx = torch.empty((T, k), dtype=torch.int32, device=out.device)
    tw = torch.empty((T, k), dtype=torch.float32, device=out.device)
    st = torch.empty(T * k, dtype=torch.int32, device=out.device)
    dropped = torch.zeros(4, dtype=torch.int32, device=out.device)
    shared = (dev["sh_gate_up"], dev["sh_down"]) if c["Fs"] > 0 else None
    cf = c.get("capacity_factor", 0.0)
    moe.moe_layer_forward(shape, dev["x"], dev["w_router"], dev["w_gate_up"], dev["w_down"],
                          c["score"], dev.get("bias"), shared, out, counts, workspace, ws_bytes,
                          stream, tidx, tw, st, stage_events=stage_events,
                          capacity_factor=cf, dropped=dropped if cf > 0 else None,
                          reroute=c.get("reroute", 0), **group_args(c))
    return dict(out=out, counts=counts, topk_idx=tidx, topk_w=tw, sorted_token=st,
                dropped=dropped[:1], workspace=workspace)


def to_host(res):
    import torch
    h = {}
    for key, v in res.items():
        if key == "workspace":
            continue
        if v.dtype == torch.bfloat16:
            h[key] = v.float().cpu().numpy().astype(np.float64)
        else:
            h[key] = v.cpu().numpy()
    return h


def group_args(cfg):
    """Group-limited routing options of a workload (none unless it sets topk_groups)."""
    c = configs.get(cfg)
    if c.get("topk_groups", 0) > 0:
        return dict(n_groups=c["groups"], topk_groups=c["topk_groups"])
    return {}


def oracle_routing(cfg, x, w_router, bias, threads=None):
    """fp64 oracle logits -> (key, score, topk_idx, margin) for all rows of x (host arrays)."""
    c = configs.get(cfg)
    g = group_args(c)

    def part(lo, hi):
        lg, sc, key = oracle.router_scores(x[lo:hi], w_router, c["score"], bias)
        if g:
            idx, _, margin = oracle.topk_grouped(key, sc, c["k"], g["n_groups"], g["topk_groups"])
        else:
            idx, _, margin = oracle.topk(key, sc, c["k"])
        return key, sc, idx, margin

    parts = oracle.parallel_rows(part, x.shape[0], threads=threads)
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(4))


def check_routing(cfg, key, score, margin, o_idx, g_idx, g_w):
    """Returns (n_excluded, oracle weights under the GPU's routing)."""
    c = configs.get(cfg)
    k = c["k"]
    T = g_idx.shape[0]
    assert g_idx.shape == (T, k)
    assert np.all((g_idx >= 0) & (g_idx < c["E"])), "expert id out of range"
    for t in range(T):
        assert len(set(g_idx[t].tolist())) == k, f"token {t}: repeated expert"
    excluded = margin < MARGIN
    same = np.sort(g_idx, 1) == np.sort(o_idx, 1)
    bad = np.where(~excluded & ~np.all(same, 1))[0]
    assert bad.size == 0, f"{bad.size} tokens with margin >= {MARGIN} routed differently, e.g. " \
        f"t={bad[0]} gpu={g_idx[bad[0]]} oracle={o_idx[bad[0]]} margin={margin[bad[0]]}"
    rows = np.arange(T)[:, None]
    sel_key = key[rows, g_idx]
    g = group_args(c)
    if g:
        # a group-limited choice spans at most topk_groups groups
        gs = c["E"] // g["n_groups"]
        spans = np.array([len(set((g_idx[t] // gs).tolist())) for t in range(T)])
        assert np.all(spans <= g["topk_groups"]), "routing spans too many groups"
    elif k < c["E"]:
        masked = key.copy()
        masked[rows, g_idx] = -np.inf
        gap = sel_key.min(1) - masked.max(1)
        assert np.all(gap >= -MARGIN), f"invalid near-tie choice, gap {gap.min()}"
    # GPU order: non-increasing oracle key up to the margin
    assert np.all(np.diff(sel_key, axis=1) <= MARGIN)
    sc = score[rows, g_idx]
    w_ref = sc / sc.sum(1, keepdims=True)
    np.testing.assert_allclose(g_w, w_ref, rtol=0, atol=2e-5)
    return int(excluded.sum()), w_ref


def check_dispatch(cfg, g_idx, g_counts, g_sorted, g_dropped=None):
    """Dispatch tables of the GPU's routing against the oracle's; returns (counts, kept mask
    [T][k]) -- the mask is all True for a dropless layer."""
    c = configs.get(cfg)
    cf = c.get("capacity_factor", 0.0)
    if cf > 0:
        cap = oracle.capacity(c["T"], c["E"], c["k"], cf)
        counts, offsets, st, sp, dropped = oracle.dispatch_capacity(g_idx.astype(np.int32),
                                                                    c["E"], cap)
        np.testing.assert_array_equal(g_counts, counts)
        np.testing.assert_array_equal(g_sorted[:offsets[-1]], st)
        assert g_dropped is not None and int(g_dropped[0]) == dropped
        return counts, sp >= 0
    counts, offsets, st, _ = oracle.dispatch(g_idx.astype(np.int32), c["E"])
    np.testing.assert_array_equal(g_counts, counts)
    np.testing.assert_array_equal(g_sorted, st)
    return counts, np.ones(g_idx.shape, dtype=bool)


def check_reroute(cfg, key, score, g_idx, g_counts, g_sorted, g_dropped):
    """Rerouting at capacity, checked on the GPU's own assignment (the rounds can cascade from
    one near-tie in a candidate order, so at full size the exact decisions are not compared):
    every serving expert is among its token's top-(k + reroute) oracle keys up to MARGIN, a
    token's serving experts are distinct, no expert is over capacity, served + dropped = T*k,
    and the dispatch tables are the stable counting sort of the assignment.  Returns the
    oracle weights renormalised over the GPU's serving experts."""
    c = configs.get(cfg)
    T, E, k = c["T"], c["E"], c["k"]
    kc = k + c["reroute"]
    cap = oracle.capacity(T, E, k, c["capacity_factor"])
    assert g_counts.max() <= cap
    assert int(g_counts.sum()) + int(g_dropped[0]) == T * k
    kth = -np.sort(-key, axis=1)[:, kc - 1]   # the kc-th largest oracle key of each token
    for t in range(T):
        served = g_idx[t][g_idx[t] >= 0]
        assert len(set(served.tolist())) == len(served), f"token {t}: expert served twice"
        assert np.all(key[t, served] >= kth[t] - MARGIN), f"token {t}: expert beyond its candidates"
    want = [t for e in range(E) for t in range(T) for j in range(k) if g_idx[t, j] == e]
    np.testing.assert_array_equal(g_sorted[:len(want)], want)
    np.testing.assert_array_equal(g_counts, np.bincount(g_idx[g_idx >= 0], minlength=E))
    return oracle.served_weights(score, g_idx)


def check_output(cfg, got, ref):
    c = configs.get(cfg)
    tol = TOL[c["dtype"]]
    err = np.abs(got - ref)
    max_ref = np.abs(ref).max()
    max_rel = err.max() / max_ref
    mean_rel = err.sum() / np.abs(ref).sum()
    assert np.all(np.isfinite(got)), "non-finite output"
    assert max_rel <= tol["max_rel"], f"max|err|/max|ref| = {max_rel:.3e}"
    assert mean_rel <= tol["mean_rel"], f"sum|err|/sum|ref| = {mean_rel:.3e}"
    return dict(max_rel=float(max_rel), mean_rel=float(mean_rel))


def oracle_rows(cfg, x_rows, idx, w, experts, shared, threads=None):
    """Oracle output rows under a routing; ``experts``: dict e -> (w_gate_up[e], w_down[e])."""
    gu = {e: v[0] for e, v in experts.items()}
    dn = {e: v[1] for e, v in experts.items()}
    shg, shd = shared if shared is not None else (None, None)

    def part(lo, hi):
        return oracle.layer_rows(x_rows[lo:hi], idx[lo:hi], w[lo:hi], gu, dn, shg, shd)

    return np.concatenate(oracle.parallel_rows(part, x_rows.shape[0], threads=threads, chunk=1))


def full_check(cfg, dev=None, host=None, threads=None):
    """Small shapes: GPU vs oracle on every token (host inputs uploaded byte-identically)."""
    c = configs.get(cfg)
    host = host if host is not None else moe_inputs.host_inputs(c)
    dev = dev if dev is not None else moe_inputs.upload(c, host)
    res = to_host(gpu_forward(c, dev))
    key, score, o_idx, margin = oracle_routing(c, host["x"], host["w_router"], host.get("bias"),
                                               threads)
    n_ex, w_ref = check_routing(c, key, score, margin, o_idx, res["topk_idx"], res["topk_w"])
    _, kept = check_dispatch(c, res["topk_idx"], res["counts"], res["sorted_token"],
                             res["dropped"])
    w_ref = np.where(kept, w_ref, 0.0)   # a dropped assignment contributes nothing
    experts = {e: (host["w_gate_up"][e], host["w_down"][e]) for e in range(c["E"])}
    shared = (host["sh_gate_up"], host["sh_down"]) if c["Fs"] > 0 else None
    ref = oracle_rows(c, host["x"], res["topk_idx"], w_ref, experts, shared, threads)
    stats = check_output(c, res["out"], ref)
    stats["excluded"] = n_ex
    return stats


def _host_elems(t):
    """Device tensor -> host array in the oracle's element format (bf16 bits / fp32)."""
    import torch
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _cta_box_edges(g0, rows):
    """Rows on both sides of each TMA box edge of one CTA's token rows [g0, g0 + rows): the
    kernel covers them with boxes of 128, 64, 32, 16 and 8 rows."""
    edges, off = [], 0
    for box in (128, 64, 32, 16, 8):
        n = (rows - off) // box if box == 128 else (1 if rows - off >= box else 0)
        for _ in range(n):
            off += box
            edges += [g0 + off - 1, g0 + off]
    return edges


def tile_edge_rows(row0, ncols, valid, wide):
    """Token rows of a GEMM tile where its index arithmetic changes: the first and last valid
    rows, the split of each MMA's N rows over the two CTAs of a pair, the split of a wide tile
    into its two MMAs (n0 = the first half rounded up to 16 rows) and the TMA box edges."""
    rows = [row0, row0 + valid - 1]
    if wide and ncols > 256:
        n0 = (((ncols >> 4) + 1) >> 1) << 4
        halves = [(row0, n0), (row0 + n0, ncols - n0)]
    else:
        halves = [(row0, ncols)]
    for start, n in halves:
        rows += [start - 1, start, start + n // 2 - 1, start + n // 2, start + n - 1]
        rows += _cta_box_edges(start, n // 2) + _cta_box_edges(start + n // 2, n // 2)
    return [r for r in rows if row0 <= r < row0 + valid]


def boundary_tokens(cfg, counts, sorted_token):
    """Tokens whose rows sit on tile edges of the two expert GEMMs, from the kernels' own tile
    decoder (moe_debug_gemm_tiles): every edge of every n-tile and tall tile of the hottest,
    the coldest and a median non-empty expert, the last row of every expert's segment, and the
    edges of the shared expert's first and last n-tiles.  Returns (tokens, description)."""
    import mixture_experts_layer_83_b300 as moe
    c = configs.get(cfg)
    shape = moe.make_shape(c["T"], c["d"], c["E"], c["k"], c["F"], c["Fs"], moe_dtype(c))
    counts = np.asarray(counts, dtype=np.int32)
    nz = np.where(counts > 0)[0]
    by_count = nz[np.argsort(counts[nz], kind="stable")]
    picked = {int(by_count[-1]), int(by_count[0]), int(by_count[len(by_count) // 2])}
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows, sh_tokens = set(), set()
    tiles_seen = 0
    for which in (1, 2):
        tiles, geo = moe.moe_debug_gemm_tiles(shape, which, counts)
        wide = geo["bn"] > 256
        for prob, seg, _m, row0, ncols, valid, _b in tiles.tolist():
            if prob == 0 and seg in picked:
                rows.update(tile_edge_rows(row0, ncols, valid, wide))
                tiles_seen += 1
        sh = tiles[tiles[:, 0] == 1]
        if sh.size:
            for row0 in (int(sh[:, 3].min()), int(sh[:, 3].max())):
                t = sh[sh[:, 3] == row0][0]
                sh_tokens.update(tile_edge_rows(int(t[3]), int(t[4]), int(t[5]), wide))
    rows.update(int(offsets[e + 1] - 1) for e in nz)      # each segment's last row
    toks = {int(sorted_token[r]) for r in rows} | sh_tokens
    desc = dict(experts=sorted(picked), tile_rows=len(rows), shared_rows=len(sh_tokens),
                tiles=tiles_seen)
    return toks, desc


def _oracle_expert_rows(dev, xs64, by_expert, threads):
    """ys[(i, j)] for every sampled (token row i, slot j) grouped by expert: each expert's
    weights are copied to the host once and its pairs are spread over host threads; an
    expert's host copy is released when its last pair is done."""
    import threading
    from concurrent.futures import ThreadPoolExecutor
    total = sum(len(v) for v in by_expert.values())
    chunk = max(1, -(-total // (4 * threads)))
    tasks = [(e, pairs[i:i + chunk]) for e, pairs in sorted(by_expert.items())
             for i in range(0, len(pairs), chunk)]
    left = {e: -(-len(p) // chunk) for e, p in by_expert.items()}
    cache, locks, mu = {}, {e: threading.Lock() for e in by_expert}, threading.Lock()
    out = {}

    def run(task):
        e, pairs = task
        with locks[e]:
            if e not in cache:
                cache[e] = (_host_elems(dev["w_gate_up"][e]), _host_elems(dev["w_down"][e]))
            wgu, wd = cache[e]
        res = [((i, j), oracle.swiglu_ffn(xs64[i], wgu, wd)) for i, j in pairs]
        with mu:
            out.update(res)
            left[e] -= 1
            if left[e] == 0:
                cache.pop(e, None)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, tasks))
    return out


def sampled_check(cfg, dev, n_sample=1024, threads=None, seed=0):
    """Full-size check: the whole layer runs on the GPU as bench.py runs it; routing is checked
    for every token, dispatch tables bit-exactly, outputs on a seeded sample of ``n_sample``
    tokens plus every token on a tile edge of the expert GEMMs (boundary_tokens) and, under a
    capacity, a token with a dropped assignment.  The oracle evaluates each sampled (token,
    expert) pair with its SwiGLU and sums them with its combine."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    c = configs.get(cfg)
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    res = to_host(gpu_forward(c, dev))
    x = _host_elems(dev["x"])
    wr = _host_elems(dev["w_router"])
    bias = dev["bias"].cpu().numpy() if "bias" in dev else None
    key, score, o_idx, margin = oracle_routing(c, x, wr, bias, threads)
    if c.get("reroute", 0) > 0:
        n_ex = 0
        w_ref = check_reroute(c, key, score, res["topk_idx"], res["counts"], res["sorted_token"],
                              res["dropped"])
        np.testing.assert_allclose(res["topk_w"], w_ref, rtol=0, atol=2e-5)
        counts, kept = res["counts"], res["topk_idx"] >= 0
        res["topk_idx"] = np.where(kept, res["topk_idx"], 0)   # weight 0: contributes nothing
    else:
        n_ex, w_ref = check_routing(c, key, score, margin, o_idx, res["topk_idx"], res["topk_w"])
        counts, kept = check_dispatch(c, res["topk_idx"], res["counts"], res["sorted_token"],
                                      res["dropped"])
        w_ref = np.where(kept, w_ref, 0.0)   # a dropped assignment contributes nothing
    T, k = c["T"], c["k"]
    edges = {}
    if n_sample >= T:
        sample = np.arange(T)
    else:
        rng = np.random.default_rng(seed)
        sample = set(rng.choice(T, n_sample, replace=False).tolist())
        forced = set()
        if c["dtype"] == "bf16":
            forced, edges = boundary_tokens(c, counts, res["sorted_token"])
        if not kept.all():   # and a token with a dropped assignment
            forced.add(int(np.where(~kept.all(1))[0][-1]))
        edges["forced_tokens"] = len(forced - sample)
        sample = np.array(sorted(sample | forced))
    n = sample.size
    g_idx = res["topk_idx"][sample]
    xs64 = as_float64(c, x[sample])
    by_expert = {}
    for i in range(n):
        for j in range(k):
            by_expert.setdefault(int(g_idx[i, j]), []).append((i, j))
    yd = _oracle_expert_rows(dev, xs64, by_expert, threads)
    ys = np.zeros((n * k, c["d"]))
    for (i, j), y in yd.items():
        ys[i * k + j] = y
    y_sh = None
    if c["Fs"] > 0:
        shg, shd = _host_elems(dev["sh_gate_up"]), _host_elems(dev["sh_down"])
        with ThreadPoolExecutor(max_workers=threads) as ex:
            y_sh = np.stack(list(ex.map(lambda i: oracle.swiglu_ffn(xs64[i], shg, shd),
                                        range(n))))
    slots = np.arange(n * k, dtype=np.int32).reshape(n, k)
    ref = oracle.combine(slots, w_ref[sample], ys, y_sh)
    stats = check_output(c, res["out"][sample], ref)
    stats.update(excluded=n_ex, sampled=int(n), experts_touched=int((counts > 0).sum()),
                 max_over_mean=float(counts.max() / counts.mean()),
                 dropped=int((~kept).sum()), edges=edges)
    return stats


def as_float64(cfg, arr):
    if arr.dtype == np.uint16:
        return (arr.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(arr, dtype=np.float64)
