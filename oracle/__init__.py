"""TEST INFRASTRUCTURE ONLY: ctypes wrapper of the fp64 C oracle (``moe_oracle.c``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
leg use this package.  The oracle itself is single-threaded C; ``parallel_map`` below only
spreads independent token ranges over host threads (ctypes releases the GIL), it does not
change what any call computes.
"""
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.c")
LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")

SOFTMAX, SIGMOID = 0, 1
F32, BF16 = 0, 1

_c_int_p = ctypes.POINTER(ctypes.c_int)
_c_dbl_p = ctypes.POINTER(ctypes.c_double)


class OracleLayer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("F", ctypes.c_int), ("Fs", ctypes.c_int), ("dtype", ctypes.c_int),
                ("w_gate_up", ctypes.POINTER(ctypes.c_void_p)),
                ("w_down", ctypes.POINTER(ctypes.c_void_p)),
                ("sh_gate_up", ctypes.c_void_p), ("sh_down", ctypes.c_void_p)]


def build(force=False):
    """Compile the oracle with gcc (plain IEEE fp64, no contraction, no fast-math)."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC):
        return LIB_PATH
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-Wall",
           "-o", LIB_PATH, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        l = ctypes.CDLL(LIB_PATH)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        l.oracle_elem.argtypes = [vp, ci, ctypes.c_size_t]
        l.oracle_elem.restype = ctypes.c_double
        l.oracle_router_scores.argtypes = [ci, ci, ci, ci, vp, vp, ci, vp, vp, vp, vp]
        l.oracle_topk.argtypes = [ci, ci, ci, vp, vp, vp, vp, vp]
        l.oracle_topk_grouped.argtypes = [ci, ci, ci, ci, ci, vp, vp, vp, vp, vp]
        l.oracle_dispatch.argtypes = [ci, ci, ci, vp, vp, vp, vp, vp]
        l.oracle_capacity.argtypes = [ci, ci, ci, ctypes.c_double]
        l.oracle_eplb_plan.argtypes = [vp, ci, ci, ci, vp, vp, vp]
        l.oracle_dispatch_capacity.argtypes = [ci, ci, ci, vp, ci, vp, vp, vp, vp, vp]
        l.oracle_dispatch_reroute.argtypes = [ci, ci, ci, ci, vp, ci, vp, vp, vp, vp, vp, vp, vp]
        l.oracle_served_weights.argtypes = [ci, ci, ci, vp, vp, vp]
        l.oracle_gather.argtypes = [ci, ci, vp, vp, vp]
        l.oracle_combine.argtypes = [ci, ci, ci, vp, vp, vp, vp, vp]
        l.oracle_swiglu_ffn.argtypes = [ci, ci, ci, vp, vp, vp, vp]
        l.oracle_layer_rows.argtypes = [ctypes.POINTER(OracleLayer), ci, vp, vp, vp, vp]
        for f in ("oracle_router_scores", "oracle_topk", "oracle_topk_grouped", "oracle_dispatch",
                  "oracle_capacity", "oracle_dispatch_capacity", "oracle_dispatch_reroute",
                  "oracle_served_weights", "oracle_eplb_plan",
                  "oracle_gather",
                  "oracle_combine", "oracle_swiglu_ffn", "oracle_layer_rows"):
            getattr(l, f).restype = ci
        _lib = l
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} returned {rc}")


def _dt(arr):
    return BF16 if arr.dtype == np.uint16 else F32


def _elems(a):
    a = np.ascontiguousarray(a)
    if a.dtype not in (np.uint16, np.float32):
        raise TypeError("oracle inputs are fp32 arrays or bf16 bit patterns (uint16)")
    return a


def router_scores(x_rows, w_router, score_fn, bias=None):
    x_rows, w_router = _elems(x_rows), _elems(w_router)
    n, d = x_rows.shape
    E = w_router.shape[0]
    logits = np.empty((n, E)); score = np.empty((n, E)); key = np.empty((n, E))
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _check(lib().oracle_router_scores(n, d, E, _dt(x_rows), _p(x_rows), _p(w_router), score_fn,
                                      _p(b), _p(logits), _p(score), _p(key)), "router_scores")
    return logits, score, key


def topk(key, score, k):
    key = np.ascontiguousarray(key, dtype=np.float64)
    score = np.ascontiguousarray(score, dtype=np.float64)
    n, E = key.shape
    idx = np.empty((n, k), dtype=np.int32); w = np.empty((n, k)); margin = np.empty(n)
    _check(lib().oracle_topk(n, E, k, _p(key), _p(score), _p(idx), _p(w), _p(margin)), "topk")
    return idx, w, margin


def topk_grouped(key, score, k, n_groups, topk_groups):
    """Group-limited top-k (see moe_oracle.h): (topk_idx, topk_w, margin)."""
    key = np.ascontiguousarray(key, dtype=np.float64)
    score = np.ascontiguousarray(score, dtype=np.float64)
    n, E = key.shape
    idx = np.empty((n, k), dtype=np.int32); w = np.empty((n, k)); margin = np.empty(n)
    _check(lib().oracle_topk_grouped(n, E, k, n_groups, topk_groups, _p(key), _p(score), _p(idx),
                                     _p(w), _p(margin)), "topk_grouped")
    return idx, w, margin


def dispatch(topk_idx, E):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, dtype=np.int32); offsets = np.empty(E + 1, dtype=np.int32)
    st = np.empty(T * k, dtype=np.int32); sp = np.empty((T, k), dtype=np.int32)
    _check(lib().oracle_dispatch(T, E, k, _p(topk_idx), _p(counts), _p(offsets), _p(st), _p(sp)),
           "dispatch")
    return counts, offsets, st, sp


def capacity(T, E, k, capacity_factor):
    c = lib().oracle_capacity(T, E, k, float(capacity_factor))
    if c < 0:
        raise ValueError("capacity: bad arguments")
    return c


def dispatch_capacity(topk_idx, E, cap):
    """Dispatch with an expert capacity (see moe_oracle.h):
    (counts, offsets, sorted_token, slot_pos with -1 for dropped, dropped)."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, dtype=np.int32); offsets = np.empty(E + 1, dtype=np.int32)
    st = np.empty(T * k, dtype=np.int32); sp = np.empty((T, k), dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    _check(lib().oracle_dispatch_capacity(T, E, k, _p(topk_idx), int(cap), _p(counts),
                                          _p(offsets), _p(st), _p(sp), _p(dropped)),
           "dispatch_capacity")
    return counts, offsets, st[:offsets[-1]], sp, int(dropped[0])


def dispatch_reroute(cand, k, E, cap):
    """Capacity with rerouting (see moe_oracle.c): cand [T][kc] candidates in selection order.
    Returns (assign [T][k] expert or -1, assign_cand [T][k], counts, offsets, sorted_token,
    slot_pos, dropped)."""
    cand = np.ascontiguousarray(cand, dtype=np.int32)
    T, kc = cand.shape
    assign = np.empty((T, k), dtype=np.int32); ac = np.empty((T, k), dtype=np.int32)
    counts = np.empty(E, dtype=np.int32); offsets = np.empty(E + 1, dtype=np.int32)
    st = np.empty(max(T * k, 1), dtype=np.int32); sp = np.empty((T, k), dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    _check(lib().oracle_dispatch_reroute(T, E, k, kc, _p(cand), int(cap), _p(assign), _p(ac),
                                         _p(counts), _p(offsets), _p(st), _p(sp), _p(dropped)),
           "dispatch_reroute")
    return assign, ac, counts, offsets, st[:offsets[-1]], sp, int(dropped[0])


def served_weights(score, assign):
    """Weights renormalised over each token's serving experts (0 for dropped slots)."""
    score = np.ascontiguousarray(score, dtype=np.float64)
    assign = np.ascontiguousarray(assign, dtype=np.int32)
    T, k = assign.shape
    w = np.empty((T, k))
    _check(lib().oracle_served_weights(T, score.shape[1], k, _p(score), _p(assign), _p(w)),
           "served_weights")
    return w


def eplb_plan(load, n_gpus, n_redundant):
    """Expert placement with redundant experts (see moe_oracle.c):
    (slot_expert, slot_gpu, gpu_load)."""
    load = np.ascontiguousarray(load, dtype=np.int32)
    S = load.size + n_redundant
    se = np.empty(S, dtype=np.int32); sg = np.empty(S, dtype=np.int32)
    gl = np.empty(n_gpus, dtype=np.float64)
    _check(lib().oracle_eplb_plan(_p(load), load.size, n_gpus, n_redundant, _p(se), _p(sg),
                                  _p(gl)), "eplb_plan")
    return se, sg, gl


def gather(sorted_token, x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    st = np.ascontiguousarray(sorted_token, dtype=np.int32)
    xs = np.empty((st.size, x.shape[1]))
    _check(lib().oracle_gather(st.size, x.shape[1], _p(st), _p(x), _p(xs)), "gather")
    return xs


def combine(slot_pos, topk_w, ys, y_shared=None):
    sp = np.ascontiguousarray(slot_pos, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float64)
    ys = np.ascontiguousarray(ys, dtype=np.float64)
    ysh = None if y_shared is None else np.ascontiguousarray(y_shared, dtype=np.float64)
    T, k = sp.shape
    out = np.empty((T, ys.shape[1]))
    _check(lib().oracle_combine(T, k, ys.shape[1], _p(sp), _p(w), _p(ys), _p(ysh), _p(out)),
           "combine")
    return out


def swiglu_ffn(xrow, w_gate_up, w_down):
    w_gate_up, w_down = _elems(w_gate_up), _elems(w_down)
    xrow = np.ascontiguousarray(xrow, dtype=np.float64)
    d = xrow.size
    F = w_gate_up.shape[0] // 2
    y = np.empty(d)
    _check(lib().oracle_swiglu_ffn(d, F, _dt(w_gate_up), _p(xrow), _p(w_gate_up), _p(w_down),
                                   _p(y)), "swiglu_ffn")
    return y


def layer_rows(x_rows, topk_idx, topk_w, w_gate_up, w_down, sh_gate_up=None, sh_down=None):
    """Layer output for token rows.  ``w_gate_up`` / ``w_down``: dict expert -> array, or a
    stacked array [E][...]; experts not routed to by these rows may be missing."""
    x_rows = _elems(x_rows)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float64)
    n, k = idx.shape
    if isinstance(w_gate_up, np.ndarray):
        E = w_gate_up.shape[0]
        gu = {e: w_gate_up[e] for e in range(E)}
        dn = {e: w_down[e] for e in range(E)}
    else:
        E = max(max(w_gate_up.keys()) + 1, int(idx.max()) + 1)
        gu, dn = w_gate_up, w_down
    keep = []
    gp = (ctypes.c_void_p * E)(); dp = (ctypes.c_void_p * E)()
    for e in range(E):
        if e in gu:
            a, b = _elems(gu[e]), _elems(dn[e])
            keep += [a, b]
            gp[e], dp[e] = a.ctypes.data, b.ctypes.data
    first = _elems(next(iter(gu.values())))
    F = first.shape[0] // 2
    Fs = 0
    shg = shd = None
    if sh_gate_up is not None:
        shg, shd = _elems(sh_gate_up), _elems(sh_down)
        Fs = shg.shape[0] // 2
    L = OracleLayer(x_rows.shape[1], E, k, F, Fs, _dt(x_rows), gp, dp, _p(shg), _p(shd))
    out = np.empty((n, x_rows.shape[1]))
    _check(lib().oracle_layer_rows(ctypes.byref(L), n, _p(x_rows), _p(idx), _p(w), _p(out)),
           "layer_rows")
    return out


def parallel_rows(fn, n, threads=None, chunk=None):
    """Run ``fn(lo, hi)`` over [0, n) split into ranges on host threads; concatenates."""
    threads = threads or max(1, (os.cpu_count() or 1))
    chunk = chunk or max(1, -(-n // (threads * 4)))
    ranges = [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda r: fn(*r), ranges))
    return parts
